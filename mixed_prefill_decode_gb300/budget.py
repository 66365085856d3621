"""Token-budget selection from a profiled step-time curve, and the seeded load
test that checks the choice by replaying requests through the packer.

pofe.ai "Chunked prefill":
  * "Tuning knobs": profile the iteration time against the number of tokens
    once for the model and GPU, set the budget to the largest value whose
    iteration time stays within the target time between tokens (TBT), then
    verify with a load test that replays the length distribution and read the
    p99, not the mean;
  * "Simulated numbers: choosing the budget": a seeded simulator whose
    scheduler takes decodes first, then partial prefills, then admissions,
    replaying Poisson arrivals with lognormal prompts (mean 1,000 tokens, up to
    8,192) and outputs (mean 250); it reports p99 TBT and TTFT, saturated
    throughput, and goodput: the highest arrival rate at which p99 TBT stays
    under 50 ms and p99 TTFT under 1 s.

The scheduler here is the library's packer (``mb_sched_*``, the same code that
builds the batches ``mb_step`` runs); the iteration time comes from a
``StepTimeFit`` to step times measured on the GPU (``bench.py --budget``) or
from the page's analytic models (``step_model``).

Readings where the page is silent:
  * lognormal shape sigma = 1 for prompts and outputs, with mu = ln(mean) -
    sigma^2 / 2 so that the stated mean is the law's mean; lengths are rounded
    to whole tokens, at least 1, at most 8,192 (the page's prompt cap, used for
    outputs too);
  * the iteration that schedules a prompt's last chunk emits the request's
    first token (TTFT = that iteration's end - arrival); every later iteration
    that schedules the request as a decode row emits one more (TBT = time
    between consecutive tokens of a request); a request leaves the packer when
    it has produced its output count;
  * an iteration starts when the previous one ends, at the latest arrival
    time if nothing was schedulable; requests that arrived by an iteration's
    start are offered to the packer before it packs;
  * percentiles are NumPy's default (linear interpolation).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import binding as mb
from . import step_model as SM

PAGE_TOKENS = 16
Row = Tuple[int, int, int]      # (request id, qo_len, kv_len) of one batch row


# --------------------------------------------------------------- step time
def row_features(rows: Sequence[Row]) -> Tuple[float, float, float]:
    """(tokens T, decode keys read, unmasked chunk-attention query-key pairs)
    of one batch: what the step time grows with."""
    T = kvd = pairs = 0.0
    for _, qo, kv in rows:
        T += qo
        if qo == 1:
            kvd += kv
        else:
            c = kv - qo
            pairs += qo * c + qo * (qo + 1) / 2
    return T, kvd, pairs


@dataclasses.dataclass
class StepTimeFit:
    """t = t0 + a T + b KVd + c pairs (seconds), least squares over profiled
    batches: the linear layers grow with the tokens, decode attention with the
    keys it streams, chunk attention with its query-key pairs."""
    t0: float
    a: float
    b: float
    c: float

    @classmethod
    def fit(cls, batches: Sequence[Sequence[Row]], seconds: Sequence[float]) -> "StepTimeFit":
        X = np.array([[1.0, *row_features(r)] for r in batches])
        y = np.asarray(seconds, dtype=np.float64)
        # columns scaled to unit norm so the solve is well conditioned
        scale = np.linalg.norm(X, axis=0)
        scale[scale == 0] = 1.0
        coef, *_ = np.linalg.lstsq(X / scale, y, rcond=None)
        coef = coef / scale
        return cls(*[float(v) for v in coef])

    def __call__(self, rows: Sequence[Row]) -> float:
        T, kvd, pairs = row_features(rows)
        return max(self.t0 + self.a * T + self.b * kvd + self.c * pairs, 0.0)


def analytic_step_time(machine: SM.Machine, model: SM.Model, pessimistic: bool = False) -> Callable:
    """The page's step-time models as a batch -> seconds function."""
    f = SM.iteration_time_pessimistic if pessimistic else SM.iteration_time

    def step(rows: Sequence[Row]) -> float:
        chunks = [(qo, kv - qo) for _, qo, kv in rows if qo > 1]
        decs = [kv - 1 for _, qo, kv in rows if qo == 1]
        return f(machine, model, chunks, decs)

    return step


def select_budget(curve: Dict[int, float], tbt_target: float) -> Optional[int]:
    """The largest profiled budget whose iteration time is within the TBT
    target ("Tuning knobs"); None if even the smallest misses it."""
    ok = [C for C, t in curve.items() if t <= tbt_target]
    return max(ok) if ok else None


# ------------------------------------------------------------- load test
@dataclasses.dataclass(frozen=True)
class LoadSpec:
    rate: float                 # arrivals per second (Poisson)
    n_requests: int
    prompt_mean: float = 1000.0
    output_mean: float = 250.0
    max_len: int = 8192
    sigma: float = 1.0
    seed: int = 0


def draw_requests(spec: LoadSpec) -> List[Tuple[float, int, int]]:
    """Seeded (arrival time s, prompt tokens, output tokens), by arrival."""
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    gaps = rng.exponential(1.0 / spec.rate, size=spec.n_requests)
    arr = np.cumsum(gaps) - gaps[0]

    def lengths(mean):
        mu = math.log(mean) - spec.sigma ** 2 / 2
        v = np.rint(rng.lognormal(mu, spec.sigma, size=spec.n_requests))
        return np.clip(v, 1, spec.max_len).astype(np.int64)

    prompts, outputs = lengths(spec.prompt_mean), lengths(spec.output_mean)
    return [(float(a), int(p), int(o)) for a, p, o in zip(arr, prompts, outputs)]


@dataclasses.dataclass
class LoadResult:
    budget: int
    rate: float
    iterations: int
    makespan_s: float
    output_tokens: int
    ttft_s: np.ndarray          # per request
    tbt_s: np.ndarray           # per token gap
    max_tokens_in_step: int

    def summary(self) -> dict:
        pct = lambda v, q: float(np.percentile(v, q)) if len(v) else float("nan")
        return {"budget": self.budget, "rate": self.rate, "iterations": self.iterations,
                "p50_tbt_ms": round(pct(self.tbt_s, 50) * 1e3, 3), "p99_tbt_ms": round(pct(self.tbt_s, 99) * 1e3, 3),
                "p50_ttft_ms": round(pct(self.ttft_s, 50) * 1e3, 3), "p99_ttft_ms": round(pct(self.ttft_s, 99) * 1e3, 3),
                "output_tok_s": round(self.output_tokens / self.makespan_s, 2) if self.makespan_s > 0 else 0.0}


def simulate(budget: int, requests: Sequence[Tuple[float, int, int]], step_time: Callable[[Sequence[Row]], float],
             max_seqs: int = 256, chunk_cap: int = 0, num_pages: Optional[int] = None, rate: float = float("nan"),
             log: Optional[list] = None, adaptive: Optional[Tuple[int, int, int, int]] = None) -> LoadResult:
    """Replay ``requests`` through the packer with the given budget; each
    iteration takes ``step_time(rows)`` seconds.  ``chunk_cap`` caps every
    prefill chunk (the head-of-line cap); ``adaptive`` = (min, base, max,
    decode pressure) sets the per-step chunk size from the decode load
    (``mb_sched_set_adaptive``).  ``log`` (if a list) receives
    the call sequence: ("add", id, prompt), ("pack", rows), ("finish", id)."""
    if num_pages is None:   # room for every request's whole context at once
        num_pages = sum((p + o + PAGE_TOKENS - 1) // PAGE_TOKENS + 1 for _, p, o in requests) + 1
    s = mb.mb_sched_create(budget, max_seqs, chunk_cap, list(range(num_pages)))
    try:
        if adaptive:
            mb.mb_sched_set_adaptive(s, *adaptive)
        n = len(requests)
        computed = [0] * n
        produced = [0] * n
        last_tok = [0.0] * n
        ttft = [math.nan] * n
        tbt: List[float] = []
        now = requests[0][0] if n else 0.0
        nxt = 0             # next request to offer
        live = 0
        iters = 0
        max_T = 0
        out_tokens = 0
        while nxt < n or live > 0:
            while nxt < n and requests[nxt][0] <= now:
                mb.mb_sched_add(s, nxt, requests[nxt][1], 0)
                if log is not None:
                    log.append(("add", nxt, requests[nxt][1]))
                nxt += 1
                live += 1
            qo_indptr, kv_len, bt_indptr, bt, req_ids = mb.mb_sched_pack(s)
            ids = [int(i) for i in req_ids]
            rows = [(ids[i], int(qo_indptr[i + 1] - qo_indptr[i]), int(kv_len[i])) for i in range(len(ids))]
            if log is not None:
                tables = [[int(x) for x in bt[bt_indptr[i]:bt_indptr[i + 1]]] for i in range(len(ids))]
                log.append(("pack", [(r[0], r[1], r[2], t) for r, t in zip(rows, tables)]))
            if not rows:
                if nxt < n:
                    now = max(now, requests[nxt][0])
                    continue
                raise RuntimeError("packer scheduled nothing with live requests (out of pages or sequence slots)")
            now += step_time(rows)
            iters += 1
            max_T = max(max_T, sum(r[1] for r in rows))
            for rid, qo, _ in rows:
                was = computed[rid]
                computed[rid] += qo
                prompt, out = requests[rid][1], requests[rid][2]
                if was < prompt and computed[rid] < prompt:
                    continue                       # a chunk that does not finish the prompt
                if was < prompt:
                    ttft[rid] = now - requests[rid][0]
                else:
                    tbt.append(now - last_tok[rid])
                last_tok[rid] = now
                produced[rid] += 1
                out_tokens += 1
                if produced[rid] >= out:
                    mb.mb_sched_finish(s, rid)
                    if log is not None:
                        log.append(("finish", rid))
                    live -= 1
        t0 = requests[0][0] if n else 0.0
        return LoadResult(budget, rate, iters, now - t0, out_tokens, np.array(ttft), np.array(tbt), max_T)
    finally:
        mb.mb_sched_destroy(s)


def goodput(budget: int, rates: Sequence[float], step_time: Callable, n_requests: int, seed: int = 0,
            tbt_slo: float = 0.050, ttft_slo: float = 1.0, **kw) -> Tuple[Optional[float], List[dict]]:
    """Highest of ``rates`` whose load test keeps p99 TBT <= tbt_slo and p99
    TTFT <= ttft_slo, with every tested point's summary."""
    best, points = None, []
    for r in sorted(rates):
        res = simulate(budget, draw_requests(LoadSpec(rate=r, n_requests=n_requests, seed=seed)), step_time,
                       rate=r, **kw)
        sm = res.summary()
        sm["meets_slo"] = bool(sm["p99_tbt_ms"] <= tbt_slo * 1e3 and sm["p99_ttft_ms"] <= ttft_slo * 1e3)
        points.append(sm)
        if sm["meets_slo"]:
            best = r
    return best, points
