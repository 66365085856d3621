"""Host-side checks of the C-ABI library that need no GPU: the library loads
and exports every entry point include/mb.h declares, the native packer agrees
bit for bit with the oracle packer, and descriptor validation rejects every
malformed batch before any device work."""

import numpy as np
import pytest
import torch

from oracle.packer import Packer, rows_to_csr
from mixed_prefill_decode_gb300 import workload as W


def test_exports_every_declared_symbol(mb):
    syms = mb.header_symbols()
    assert len(syms) >= 20
    missing = [s for s in syms if not hasattr(mb.lib(), s)]
    assert missing == []


def _drive_both(seed, steps=80):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(4, 300))
    budget = int(rng.integers(1, 600))
    max_seqs = int(rng.integers(1, 20))
    cap = int(rng.choice([0, 0, 8, 64, 256]))
    order = rng.permutation(P)
    return rng, P, budget, max_seqs, cap, order


@pytest.mark.parametrize("seed", range(40))
def test_native_packer_matches_oracle_bit_exactly(mb, seed):
    rng, P, budget, max_seqs, cap, order = _drive_both(seed)
    # seeds 30-39: adaptive chunk size on (min, base, max, pressure)
    adaptive = None
    if seed >= 30:
        mn = int(rng.integers(1, 64))
        base = mn + int(rng.integers(0, 300))
        adaptive = (mn, base, base + int(rng.integers(0, 600)), int(rng.integers(1, 12)))
    py = Packer(budget, max_seqs, cap, order, adaptive=adaptive)
    s = mb.mb_sched_create(budget, max_seqs, cap, order)
    if adaptive:
        mb.mb_sched_set_adaptive(s, *adaptive)
    try:
        nid = 0
        for step in range(80):
            if rng.random() < 0.45:
                plen = int(rng.integers(1, 500))
                comp = int(rng.choice([0, 0, 0, int(rng.integers(0, plen + 40))]))
                try:
                    py.add(nid, plen, comp)
                    ok_py = True
                except Exception:
                    ok_py = False
                try:
                    mb.mb_sched_add(s, nid, plen, comp)
                    ok_c = True
                except mb.MbError as e:
                    ok_c = False
                    assert e.status == mb.MB_ENOSPACE
                assert ok_py == ok_c
                nid += 1
            if py.reqs and rng.random() < 0.25:
                rid = int(rng.choice(sorted(py.reqs)))
                py.finish(rid)
                mb.mb_sched_finish(s, rid)
            rows = py.pack()
            qo, kv, bti, bt, ids = rows_to_csr(rows)
            cqo, ckv, cbti, cbt, cids = mb.mb_sched_pack(s)
            assert list(cqo) == qo
            assert list(ckv) == kv
            assert list(cbti) == bti
            assert list(cbt) == bt
            assert list(cids) == ids
            fr, run, par, wait = mb.mb_sched_counts(s)
            assert (fr, run, par, wait) == (len(py.free), len(py.running), len(py.partial), len(py.waiting))
    finally:
        mb.mb_sched_destroy(s)


# The hand-traced scripts of test_oracle_packer.py (sequence limit, a decode
# skipped for want of a page, freed pages at the tail of the free list, the
# adaptive size under a fixed cap), replayed on the native packer.
HAND_TRACES = {
    "max_seqs": ((100, 2, 0, range(64), None),
                 [("add", 1, 10, 0), ("add", 2, 10, 0), ("add", 3, 10, 0), ("pack",), ("pack",), ("finish", 1),
                  ("pack",)]),
    "decode_without_page": ((10, 4, 0, range(2), None),
                            [("add", 1, 16, 16), ("add", 2, 5, 5), ("pack",), ("finish", 2), ("pack",)]),
    "free_list_tail": ((16, 4, 0, [2, 0, 1], None),
                       [("add", 1, 16, 0), ("pack",), ("finish", 1), ("add", 2, 16, 0), ("pack",),
                        ("add", 3, 32, 0), ("pack",)]),
    "adaptive_under_cap": ((2048, 8, 100, range(200), (64, 256, 1024, 8)), [("add", 1, 500, 0), ("pack",)]),
    "adaptive_one_decode": ((2048, 8, 1000, range(200), (64, 256, 1024, 8)),
                            [("add", 1, 5, 5), ("add", 2, 500, 0), ("pack",)]),
}


@pytest.mark.parametrize("name", list(HAND_TRACES))
def test_native_packer_hand_traces(mb, name):
    (budget, max_seqs, cap, order, adaptive), ops = HAND_TRACES[name]
    order = list(order)
    py = Packer(budget, max_seqs, cap, order, adaptive=adaptive)
    s = mb.mb_sched_create(budget, max_seqs, cap, np.asarray(order))
    if adaptive:
        mb.mb_sched_set_adaptive(s, *adaptive)
    try:
        for op in ops:
            if op[0] == "add":
                py.add(*op[1:])
                mb.mb_sched_add(s, *op[1:])
            elif op[0] == "finish":
                py.finish(op[1])
                mb.mb_sched_finish(s, op[1])
            else:
                qo, kv, bti, bt, ids = rows_to_csr(py.pack())
                c = mb.mb_sched_pack(s)
                assert [list(x) for x in c] == [qo, kv, bti, bt, ids]
    finally:
        mb.mb_sched_destroy(s)


@pytest.mark.parametrize("seed", [3, 11, 17, 31, 35])
def test_native_checkpoint_matches_oracle_and_resumes(mb, seed):
    """Every 10 steps the native packer is replaced by one loaded from its own
    checkpoint; the words equal the oracle's state words, and the batches
    stay bit-identical to the oracle's for the whole stream."""
    from oracle.packer import state_words
    rng, P, budget, max_seqs, cap, order = _drive_both(seed)
    adaptive = (8, 64, 256, 4) if seed >= 30 else None
    py = Packer(budget, max_seqs, cap, order, adaptive=adaptive)
    s = mb.mb_sched_create(budget, max_seqs, cap, order)
    if adaptive:
        mb.mb_sched_set_adaptive(s, *adaptive)
    try:
        nid = 0
        for step in range(80):
            if step % 10 == 9:
                words = mb.mb_sched_save(s)
                assert list(words) == state_words(py)
                t = mb.mb_sched_load(words)
                mb.mb_sched_destroy(s)
                s = t
                assert list(mb.mb_sched_save(s)) == list(words)
            if rng.random() < 0.45:
                plen = int(rng.integers(1, 500))
                comp = int(rng.choice([0, 0, 0, int(rng.integers(0, plen + 40))]))
                try:
                    py.add(nid, plen, comp)
                    ok_py = True
                except Exception:
                    ok_py = False
                try:
                    mb.mb_sched_add(s, nid, plen, comp)
                    ok_c = True
                except mb.MbError:
                    ok_c = False
                assert ok_py == ok_c
                nid += 1
            if py.reqs and rng.random() < 0.25:
                rid = int(rng.choice(sorted(py.reqs)))
                py.finish(rid)
                mb.mb_sched_finish(s, rid)
            qo, kv, bti, bt, ids = rows_to_csr(py.pack())
            assert [list(x) for x in mb.mb_sched_pack(s)] == [qo, kv, bti, bt, ids]
    finally:
        mb.mb_sched_destroy(s)


# A hand-made state: 6 pages; free 3, 4, 5; running request 1 (prompt 10,
# 20 computed, pages 0, 1); partial request 2 (prompt 40, 16 computed, page
# 2); waiting request 3 (prompt 9).
GOOD_STATE = [0x4D4253434844, 1, 100, 4, 0, 6, 0, 0, 0, 0, 3, 3, 4, 5,
              1, 1, 10, 20, 2, 0, 1,
              1, 2, 40, 16, 1, 2,
              1, 3, 9, 0, 0]


def _edit(i, v):
    w = list(GOOD_STATE)
    w[i] = v
    return w


BAD_STATES = {
    "magic": _edit(0, 0x4D4253434845),
    "version": _edit(1, 2),
    "budget 0": _edit(2, 0),
    "adaptive half set": _edit(6, 5),
    "truncated": GOOD_STATE[:-1],
    "trailing word": GOOD_STATE + [0],
    "free page twice": _edit(12, 3),
    "page out of range": _edit(13, 6),
    "page held by no one": _edit(5, 7),
    "pages do not match computed": _edit(17, 40),
    "partial request past its prompt": _edit(24, 40),
    "waiting request with progress": _edit(30, 1),
    "duplicate request id": _edit(22, 1),
    "page in a table and free": _edit(26, 3),
    # 2^40 cached tokens with an empty table: a 32-bit page count would wrap to 0
    "computed past int32 with no pages": [GOOD_STATE[0], 1, 100, 4, 0, 6, 0, 0, 0, 0, 5, 0, 1, 3, 4, 5,
                                          1, 1, 10, 1 << 40, 0,
                                          1, 2, 40, 16, 1, 2,
                                          1, 3, 9, 0, 0],
}


def test_sched_load_accepts_a_valid_state_and_round_trips(mb):
    s = mb.mb_sched_load(GOOD_STATE)
    try:
        assert list(mb.mb_sched_save(s)) == GOOD_STATE
        assert mb.mb_sched_counts(s) == (3, 1, 1, 1)
        qo, kv, bti, bt, ids = mb.mb_sched_pack(s)
        # request 1 decodes (page 1 has room), 2 finishes its prompt with 24
        # tokens (40 need pages 2, 3, 4), 3 is admitted with 9 tokens (page 5)
        assert list(ids) == [1, 2, 3] and list(qo) == [0, 1, 25, 34] and list(kv) == [21, 40, 9]
        assert list(bt) == [0, 1, 2, 3, 4, 5]
    finally:
        mb.mb_sched_destroy(s)


@pytest.mark.parametrize("name", list(BAD_STATES))
def test_sched_load_rejects_bad_states(mb, name):
    with pytest.raises(mb.MbError) as e:
        mb.mb_sched_load(BAD_STATES[name])
    assert e.value.status == mb.MB_EINVAL


def test_sched_save_reports_its_size_and_refuses_a_short_buffer(mb):
    import ctypes
    s = mb.mb_sched_load(GOOD_STATE)
    try:
        n = ctypes.c_int64()
        assert mb.lib().mb_sched_save(s, None, 0, ctypes.byref(n)) == mb.MB_OK and n.value == len(GOOD_STATE)
        buf = np.full(len(GOOD_STATE) - 1, -7, dtype=np.int64)
        st = mb.lib().mb_sched_save(s, buf.ctypes.data_as(mb.c_int64_p), len(buf), ctypes.byref(n))
        assert st == mb.MB_ENOSPACE and n.value == len(GOOD_STATE) and np.all(buf == -7)
    finally:
        mb.mb_sched_destroy(s)


def test_native_packer_worked_example(mb):
    s = mb.mb_sched_create(576, 1000, 0, np.arange(20000))
    for i in range(64):
        mb.mb_sched_add(s, i, 1125, 1125)
    mb.mb_sched_add(s, 9999, 4096, 0)
    for it in range(8):
        qo, kv, bti, bt, ids = mb.mb_sched_pack(s)
        assert qo[-1] == 576 and len(ids) == 65 and ids[-1] == 9999
        assert kv[-1] == 512 * (it + 1)
    qo, kv, bti, bt, ids = mb.mb_sched_pack(s)
    assert len(ids) == 65 and qo[-1] == 65 and kv[-1] == 4097
    mb.mb_sched_destroy(s)


def test_sched_rejects_bad_config(mb):
    with pytest.raises(mb.MbError) as e:
        mb.mb_sched_create(0, 4, 0, np.arange(4))
    assert e.value.status == mb.MB_EINVAL
    with pytest.raises(mb.MbError):
        mb.mb_sched_create(8, 4, 0, [0, 0, 1])   # not a permutation
    s = mb.mb_sched_create(8, 4, 0, np.arange(2))
    with pytest.raises(mb.MbError) as e:
        mb.mb_sched_add(s, 1, 100, 100)          # needs 7 pages
    assert e.value.status == mb.MB_ENOSPACE
    mb.mb_sched_add(s, 1, 10, 0)
    with pytest.raises(mb.MbError):
        mb.mb_sched_add(s, 1, 10, 0)             # duplicate id
    with pytest.raises(mb.MbError):
        mb.mb_sched_finish(s, 77)
    mb.mb_sched_destroy(s)


def _good():
    b, P = W.make_batch([(30, 1), (0, 70), (5, 11)], seed=5)
    return b, P


def test_batch_validate_accepts_good_and_empty(mb):
    b, P = _good()
    mb.mb_batch_validate(mb.Batch.of(b), P, 1000)
    mb.mb_batch_validate(mb.Batch([0], [], [0], []), P, 1)


@pytest.mark.parametrize("bad", ["qo0", "qo_zero", "kv_lt_qo", "short_table", "page_range", "page_dup",
                                 "too_many_tokens", "neg_page"])
def test_batch_validate_rejects(mb, bad):
    b, P = _good()
    qo, kv, bti, bt = b.qo_indptr.copy(), b.kv_len.copy(), b.bt_indptr.copy(), b.bt.copy()
    maxT = 1000
    if bad == "qo0":
        qo = qo + 1
    elif bad == "qo_zero":
        qo[2] = qo[1]
    elif bad == "kv_lt_qo":
        kv[1] = 69
    elif bad == "short_table":
        bti[2] -= 1
        bt = np.delete(bt, bti[2])
        bti[3] -= 1
    elif bad == "page_range":
        bt[0] = P
    elif bad == "page_dup":
        bt[1] = bt[0]
    elif bad == "too_many_tokens":
        maxT = int(qo[-1]) - 1
    elif bad == "neg_page":
        bt[3] = -1
    with pytest.raises(mb.MbError) as e:
        mb.mb_batch_validate(mb.Batch(qo, kv, bti, bt), P, maxT)
    assert e.value.status == mb.MB_EINVAL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks behaviour without a GPU")
def test_compute_calls_fail_loudly_without_gpu(mb):
    with pytest.raises(mb.MbError) as e:
        mb.mb_gemm(16, 16, 16, None, 128, 128, 64, 0)
    assert e.value.status in (mb.MB_ECUDA, mb.MB_EUNSUPPORTED)
    sh = W.TINY.as_dict()
    with pytest.raises(mb.MbError) as e:
        mb.Layer(sh, {k: 16 for k in ("g_attn", "w_qkv", "w_o", "g_ffn", "w_gate_up", "w_down")}, 64, 8)
    assert e.value.status in (mb.MB_ECUDA, mb.MB_EUNSUPPORTED)
