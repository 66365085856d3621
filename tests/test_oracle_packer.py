"""Pins for the oracle packer: the worked example of the pofe.ai "Chunked
prefill" page and brute-force invariants over seeded random request streams.
CPU only."""

import json
import os

import numpy as np
import pytest

from oracle.packer import Packer, NoSpace, pages_for, rows_to_csr

GOLD = os.path.join(os.path.dirname(__file__), "golden", "pofe_packer_example.json")


def test_worked_example_eight_mixed_iterations():
    g = json.load(open(GOLD))
    pk = Packer(budget=g["budget"], max_seqs=1000, chunk_cap=0, free_order=range(100000))
    for i in range(g["running_decodes"]):
        pk.add(i, prompt_len=g["decode_context"], computed=g["decode_context"])
    pk.add(9999, prompt_len=g["prompt_len"])
    for it in range(g["mixed_iterations"]):
        rows = pk.pack()
        dec = [r for r in rows if r[1] == 1]
        pre = [r for r in rows if r[0] == 9999]
        assert len(dec) == g["running_decodes"]
        assert len(pre) == 1 and pre[0][1] == g["chunk_tokens_per_iteration"]
        assert pre[0][2] == (it + 1) * g["chunk_tokens_per_iteration"]
        assert sum(r[1] for r in rows) == g["budget"]
    rows = pk.pack()
    assert len(rows) == g["decodes_in_iteration_after_prompt"]
    assert all(r[1] == 1 for r in rows)
    assert rows[-1][0] == 9999 and rows[-1][2] == g["prompt_len"] + 1


def test_decodes_first_then_partials_then_admissions_fifo():
    pk = Packer(budget=20, max_seqs=10, chunk_cap=0, free_order=range(100))
    pk.add(1, 5, computed=5)      # running
    pk.add(2, 30, computed=10)    # partial
    pk.add(3, 4)                  # waiting
    pk.add(4, 100)                # waiting
    rows = pk.pack()
    assert [(r[0], r[1]) for r in rows] == [(1, 1), (2, 19)]
    rows = pk.pack()
    assert [(r[0], r[1]) for r in rows] == [(1, 1), (2, 1), (3, 4), (4, 14)]
    rows = pk.pack()   # 2 and 3 are decoding now
    assert [(r[0], r[1]) for r in rows] == [(1, 1), (2, 1), (3, 1), (4, 17)]


def test_decodes_never_exceed_budget():
    pk = Packer(budget=3, max_seqs=10, chunk_cap=0, free_order=range(100))
    for i in range(5):
        pk.add(i, 7, computed=7)
    rows = pk.pack()
    assert [r[0] for r in rows] == [0, 1, 2]


def test_chunk_cap_and_max_seqs_and_page_exhaustion():
    pk = Packer(budget=100, max_seqs=2, chunk_cap=30, free_order=range(4))
    pk.add(1, 50)
    pk.add(2, 50)
    pk.add(3, 50)
    rows = pk.pack()
    # cap 30 each; the third is refused by max_seqs; 2 + 2 pages used
    assert [(r[0], r[1]) for r in rows] == [(1, 30), (2, 30)]
    rows = pk.pack()
    # no page left: each partial keeps to its pages (32 tokens) -> 2 more each
    assert [(r[0], r[1], r[2]) for r in rows] == [(1, 2, 32), (2, 2, 32)]
    rows = pk.pack()
    assert rows == []
    pk.finish(1)
    rows = pk.pack()
    # 1's two pages go to 2 (which completes); 3 finds no page left for its chunk
    assert [(r[0], r[1], r[2]) for r in rows] == [(2, 18, 50)]
    rows = pk.pack()
    assert [(r[0], r[1], r[2]) for r in rows] == [(2, 1, 51)]
    pk.finish(2)
    rows = pk.pack()
    assert [(r[0], r[1], r[2], r[3]) for r in rows] == [(3, 30, 30, [2, 3])]


def test_admission_stops_at_first_failure():
    pk = Packer(budget=64, max_seqs=8, chunk_cap=0, free_order=range(2))
    pk.add(1, 40)   # needs 3 pages for 40 tokens -> refused, and blocks 2
    pk.add(2, 5)
    assert pk.pack() == []


def test_add_running_needs_pages():
    pk = Packer(budget=8, max_seqs=8, chunk_cap=0, free_order=range(2))
    with pytest.raises(NoSpace):
        pk.add(1, 40, computed=40)


def _random_stream(seed, steps=60):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(8, 200))
    pk = Packer(budget=int(rng.integers(1, 300)), max_seqs=int(rng.integers(1, 12)),
                chunk_cap=int(rng.choice([0, 0, 16, 100])), free_order=rng.permutation(P))
    nid = 0
    for _ in range(steps):
        if rng.random() < 0.5:
            pk.add(nid, int(rng.integers(1, 400)))
            nid += 1
        if pk.reqs and rng.random() < 0.2:
            pk.finish(int(rng.choice(sorted(pk.reqs))))
        before = {rid: r.computed for rid, r in pk.reqs.items()}
        running_before = [r.rid for r in pk.running]
        rows = pk.pack()
        yield pk, P, rows, before, running_before


@pytest.mark.parametrize("seed", range(25))
def test_invariants_random_streams(seed):
    for pk, P, rows, before, running_before in _random_stream(seed):
        total = sum(r[1] for r in rows)
        assert total <= pk.budget
        ids = [r[0] for r in rows]
        assert len(set(ids)) == len(ids)
        # decodes come first, in running order
        nd = sum(1 for rid in ids if rid in running_before)
        assert ids[:nd] == [rid for rid in running_before if rid in ids]
        # budget ran out before any running decode was skipped for budget
        if nd < len(running_before) and pk.budget >= len(running_before):
            assert len(pk.free) == 0 or any(
                pages_for(before[rid] + 1) - pages_for(before[rid]) > 0 for rid in running_before if rid not in ids)
        all_pages = []
        for rid, qo, kv, table in rows:
            assert qo >= 1 and kv == before[rid] + qo
            assert len(table) == pages_for(kv)
            all_pages.extend(table)
        assert len(set(all_pages)) == len(all_pages)
        # conservation of pages: held + free == pool
        held = [p for r in pk.reqs.values() for p in r.pages]
        assert sorted(held + list(pk.free)) == list(range(P))
        q, kvl, bti, bt, rid = rows_to_csr(rows)
        assert q[-1] == total and len(bt) == bti[-1]


def test_adaptive_chunk_closed_forms():
    # llm-stack-book 7.8 "Priority and Preemption Policies": defaults min 128,
    # base 512, max 4,096, pressure 16
    from oracle.packer import adaptive_chunk
    f = lambda d: adaptive_chunk(d, 128, 512, 4096, 16)
    assert f(0) == 4096                   # no decode running: full large chunks
    assert f(16) == 128 and f(500) == 128 # at and past the pressure threshold
    assert f(8) == 320                    # halfway: 512 - 0.5 * 384
    assert f(1) == 488                    # 512 - 384 / 16
    assert f(15) == 152                   # 512 - 15 * 24
    vals = [f(d) for d in range(1, 16)]
    assert all(a >= b for a, b in zip(vals, vals[1:]))   # monotone in the decode load


def test_adaptive_cap_bounds_every_prefill_chunk():
    from oracle.packer import adaptive_chunk
    rng = np.random.default_rng(77)
    pk = Packer(budget=2048, max_seqs=64, chunk_cap=0, free_order=range(20000), adaptive=(64, 256, 1024, 8))
    nid = 0
    for _ in range(120):
        if rng.random() < 0.6:
            pk.add(nid, int(rng.integers(1, 3000)))
            nid += 1
        if pk.running and rng.random() < 0.3:
            pk.finish(pk.running[0].rid)
        d = len(pk.running)
        cap = adaptive_chunk(d, 64, 256, 1024, 8)
        running = {r.rid for r in pk.running}
        for rid, qo, kv, table in pk.pack():
            if rid not in running:
                assert qo <= cap


def test_max_seqs_alone_stops_admission():
    # pages and budget to spare: only the sequence limit turns the third away
    pk = Packer(budget=100, max_seqs=2, chunk_cap=0, free_order=range(64))
    for rid in (1, 2, 3):
        pk.add(rid, 10)
    assert [(r[0], r[1]) for r in pk.pack()] == [(1, 10), (2, 10)]
    assert [(r[0], r[1]) for r in pk.pack()] == [(1, 1), (2, 1)]      # still two sequences
    pk.finish(1)
    assert [(r[0], r[1]) for r in pk.pack()] == [(2, 1), (3, 10)]


def test_decode_without_a_page_is_skipped_alone():
    # request 1 sits on a page boundary (16 cached: its next token needs a
    # second page), request 2 has room in its page; no page is free
    pk = Packer(budget=10, max_seqs=4, chunk_cap=0, free_order=range(2))
    pk.add(1, 16, computed=16)
    pk.add(2, 5, computed=5)
    assert len(pk.free) == 0
    assert [(r[0], r[1], r[2]) for r in pk.pack()] == [(2, 1, 6)]
    pk.finish(2)                                  # its page frees request 1
    assert [(r[0], r[1], r[2], r[3]) for r in pk.pack()] == [(1, 1, 17, [0, 1])]


def test_freed_pages_go_to_the_tail_of_the_free_list():
    pk = Packer(budget=16, max_seqs=4, chunk_cap=0, free_order=[2, 0, 1])
    pk.add(1, 16)
    assert pk.pack()[0][3] == [2]
    pk.finish(1)                                   # free list: 0, 1, 2
    pk.add(2, 16)
    assert pk.pack()[0][3] == [0]
    pk.add(3, 32)
    # 2's first decode crosses into a second page (1), then 3 takes the
    # remaining 15 tokens of the budget on the last free page (2)
    assert pk.pack() == [(2, 1, 17, [0, 1]), (3, 15, 15, [2])]


def test_adaptive_size_truncates_and_combines_with_the_fixed_cap():
    from oracle.packer import adaptive_chunk
    # llm-stack-book 7.8 "Priority and Preemption Policies": the line value is
    # truncated to an integer; 512 - (4/7) 384 = 292.57 -> 292
    assert adaptive_chunk(4, 128, 512, 4096, 7) == 292
    assert adaptive_chunk(2, 128, 512, 4096, 7) == 402     # 402.29
    # with a fixed per-request cap as well, the smaller of the two applies
    pk = Packer(budget=2048, max_seqs=8, chunk_cap=100, free_order=range(200), adaptive=(64, 256, 1024, 8))
    pk.add(1, 500)
    assert [(r[0], r[1]) for r in pk.pack()] == [(1, 100)]   # no decode: adaptive 1,024, cap 100
    pk = Packer(budget=2048, max_seqs=8, chunk_cap=1000, free_order=range(200), adaptive=(64, 256, 1024, 8))
    pk.add(1, 5, computed=5)
    pk.add(2, 500)
    assert [(r[0], r[1]) for r in pk.pack()] == [(1, 1), (2, 232)]   # one decode: 256 - 192/8, under cap 1,000


@pytest.mark.parametrize("seed", range(5))
def test_state_words_round_trip_and_resume(seed):
    # a packer rebuilt from its state words packs exactly what the original does
    from oracle.packer import state_words, from_state_words
    stream = _random_stream(seed, steps=50)
    for k, (pk, P, rows, before, running_before) in enumerate(stream):
        if k in (10, 30):
            words = state_words(pk)
            twin = from_state_words(words)
            assert state_words(twin) == words
            for _ in range(5):
                assert twin.pack() == pk.pack()
