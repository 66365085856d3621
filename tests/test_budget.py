"""Budget selection and the seeded load test (mixed_prefill_decode_gb300.budget).

Pinned by closed forms (a constant step time fixes every TTFT and gap), brute
force (the selection rule, the least-squares fit on exact data), the oracle
packer (replayed along a simulated stream, bit-exact batches and block tables)
and the numbers the pofe.ai "Chunked prefill" page prints from its own
simulator ("Simulated numbers: choosing the budget",
tests/golden/pofe_budget_sim.json), within tolerances since the page gives
neither its seeds nor its arrival rates.  Host only: no GPU."""

import json
import math
import os

import numpy as np
import pytest

from mixed_prefill_decode_gb300 import budget as BU
from mixed_prefill_decode_gb300 import step_model as SM
from oracle import packer as OP

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pofe_budget_sim.json")))
OPT = BU.analytic_step_time(SM.H100_CLASS, SM.LLAMA_8B)
PES = BU.analytic_step_time(SM.H100_CLASS, SM.LLAMA_8B, pessimistic=True)


def test_select_budget_matches_brute_force():
    rng = np.random.default_rng(5)
    for _ in range(200):
        Cs = sorted(rng.choice(np.arange(64, 16384), size=rng.integers(1, 8), replace=False).tolist())
        curve = {C: float(t) for C, t in zip(Cs, rng.uniform(0.001, 0.2, size=len(Cs)))}
        target = float(rng.uniform(0.0, 0.2))
        want = None
        for C in Cs:
            if curve[C] <= target:
                want = C
        assert BU.select_budget(curve, target) == want


def test_fit_recovers_exact_coefficients():
    rng = np.random.default_rng(6)
    true = BU.StepTimeFit(t0=2e-3, a=3e-6, b=4e-9, c=5e-12)
    batches = []
    for _ in range(12):
        rows = [(i, 1, int(k)) for i, k in enumerate(rng.integers(100, 30000, size=rng.integers(1, 200)))]
        q = int(rng.integers(2, 4000))
        rows.append((len(rows), q, q + int(rng.integers(0, 16000))))
        batches.append(rows)
    fit = BU.StepTimeFit.fit(batches, [true(r) for r in batches])
    for name in ("t0", "a", "b", "c"):
        assert getattr(fit, name) == pytest.approx(getattr(true, name), rel=1e-6)


@pytest.mark.parametrize("prompt,output,budget", [(1, 1, 512), (1000, 5, 256), (513, 3, 512), (8192, 10, 2048)])
def test_lone_request_closed_form(prompt, output, budget):
    t = 0.01
    res = BU.simulate(budget, [(0.0, prompt, output)], lambda rows: t)
    chunks = math.ceil(prompt / budget)
    assert res.iterations == chunks + output - 1
    assert res.ttft_s[0] == pytest.approx(chunks * t)
    assert len(res.tbt_s) == output - 1 and np.allclose(res.tbt_s, t)
    assert res.output_tokens == output


def test_constant_step_time_fixes_every_gap():
    # with a fixed iteration time every request that is decoding gets a token
    # every iteration (the packer schedules all decodes first), so each gap is t
    reqs = BU.draw_requests(BU.LoadSpec(rate=30, n_requests=300, seed=11))
    res = BU.simulate(4096, reqs, lambda rows: 0.02)
    assert np.allclose(res.tbt_s, 0.02)
    assert res.output_tokens == sum(o for _, _, o in reqs)
    assert np.all(res.ttft_s >= 0.02 - 1e-12)


def test_deterministic_and_budget_respected():
    reqs = BU.draw_requests(BU.LoadSpec(rate=20, n_requests=400, seed=3))
    a = BU.simulate(512, reqs, OPT, rate=20)
    b = BU.simulate(512, reqs, OPT, rate=20)
    assert a.summary() == b.summary()
    assert a.max_tokens_in_step <= 512
    assert BU.draw_requests(BU.LoadSpec(rate=20, n_requests=400, seed=3)) == reqs


def test_draws_follow_the_stated_distributions():
    reqs = BU.draw_requests(BU.LoadSpec(rate=10, n_requests=20000, seed=1))
    arr = np.array([a for a, _, _ in reqs])
    p = np.array([q for _, q, _ in reqs])
    o = np.array([q for _, _, q in reqs])
    assert np.mean(np.diff(arr)) == pytest.approx(0.1, rel=0.03)        # Poisson, 10 per second
    assert p.mean() == pytest.approx(1000, rel=0.04) and p.max() <= 8192 and p.min() >= 1
    assert o.mean() == pytest.approx(250, rel=0.04) and o.min() >= 1


def test_packer_matches_oracle_along_a_simulated_stream():
    log = []
    reqs = BU.draw_requests(BU.LoadSpec(rate=25, n_requests=250, seed=9))
    res = BU.simulate(768, reqs, OPT, max_seqs=64, chunk_cap=300, log=log)
    num_pages = sum((p + o + 15) // 16 + 1 for _, p, o in reqs) + 1
    ref = OP.Packer(768, 64, 300, list(range(num_pages)))
    n_pack = 0
    for ev in log:
        if ev[0] == "add":
            ref.add(ev[1], ev[2])
        elif ev[0] == "finish":
            ref.finish(ev[1])
        else:
            assert [(r[0], r[1], r[2], list(r[3])) for r in ref.pack()] == ev[1]
            n_pack += 1
    assert n_pack == res.iterations + sum(1 for e in log if e[0] == "pack" and not e[1])


def test_page_p99_gaps():
    reqs = BU.draw_requests(BU.LoadSpec(rate=16, n_requests=600, seed=1))
    for C, want in G["p99_tbt_ms_by_budget"].items():
        got = BU.simulate(int(C), reqs, OPT).summary()["p99_tbt_ms"]
        assert got == pytest.approx(want, rel=0.10), (C, got, want)


def test_page_saturated_throughput():
    reqs = BU.draw_requests(BU.LoadSpec(rate=200, n_requests=3000, seed=2))
    for C, want in G["optimistic_saturated_output_tok_s"].items():
        got = BU.simulate(int(C), reqs, OPT).summary()["output_tok_s"]
        assert got == pytest.approx(want, rel=0.06), (C, got, want)
    lo, hi = G["pessimistic_saturated_output_tok_s_range"]
    for C in (256, 512, 1024, 2048):
        got = BU.simulate(C, reqs, PES).summary()["output_tok_s"]
        assert lo * 0.96 <= got <= hi * 1.04, (C, got)


def test_page_goodput():
    slo = G["goodput_slo"]
    kw = dict(n_requests=1500, seed=3, tbt_slo=slo["p99_tbt_ms"] / 1e3, ttft_slo=slo["p99_ttft_ms"] / 1e3)
    for C, want in G["goodput_rps_pessimistic"].items():
        g, _ = BU.goodput(int(C), [want - 2, want, want + 2], PES, **kw)
        assert g == want, (C, g)
    for C, want in G["goodput_rps_optimistic"].items():
        g, _ = BU.goodput(int(C), [want - 4, want - 2, want, want + 2, want + 4], OPT, **kw)
        assert g is not None and abs(g - want) <= 2, (C, g)
    g, pts = BU.goodput(2048, [8, 16, 24], OPT, **kw)
    assert g is None and all(p["p99_tbt_ms"] > slo["p99_tbt_ms"] for p in pts)


def test_adaptive_policy_in_the_load_test_matches_oracle_packer():
    log = []
    reqs = BU.draw_requests(BU.LoadSpec(rate=25, n_requests=200, seed=21))
    BU.simulate(1024, reqs, OPT, max_seqs=64, adaptive=(64, 256, 2048, 8), log=log)
    num_pages = sum((p + o + 15) // 16 + 1 for _, p, o in reqs) + 1
    ref = OP.Packer(1024, 64, 0, list(range(num_pages)), adaptive=(64, 256, 2048, 8))
    for ev in log:
        if ev[0] == "add":
            ref.add(ev[1], ev[2])
        elif ev[0] == "finish":
            ref.finish(ev[1])
        else:
            assert [(r[0], r[1], r[2], list(r[3])) for r in ref.pack()] == ev[1]


def test_head_of_line_cap_lets_short_prompts_in():
    # a 100,000-token document arrives first, then short prompts: without a
    # cap it takes the whole prefill share for ~50 iterations (pofe.ai "Failure
    # modes and how to spot them"); with a per-request cap the short prompts
    # are admitted beside it
    reqs = [(0.0, 100000, 2)] + [(0.001 * i, 200, 2) for i in range(1, 21)]
    t = 0.01
    free = BU.simulate(2048, reqs, lambda rows: t)
    capped = BU.simulate(2048, reqs, lambda rows: t, chunk_cap=512)
    assert np.max(free.ttft_s[1:]) > 40 * t
    assert np.max(capped.ttft_s[1:]) < 5 * t
