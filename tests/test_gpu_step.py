"""GPU parity of the whole layer step (mb_step through the C ABI) against the
oracle, on the same seeded inputs:

* KV placement bit-exact: every slot the step must not touch keeps its input
  bits (cached prefix values and the sentinel), every written slot is within
  tolerance of the oracle's K / V;
* outputs and every intermediate within max|d| <= 2e-2 max|ref| per tensor;
* the attention alone, fed the GPU's own rotated q and KV pool, against the
  oracle's attention (isolates the attention kernels from upstream rounding).

Workloads: the pages' tiny, Llama-3-8B and Qwen3-14B configurations at full
size, oracle-sized GQA batches with ragged tails, and edge cases (kv_len 1,
page boundaries, two-token chunks, chunks of 129 rows)."""

import numpy as np
import pytest
import torch

from oracle import layer as OL
from mixed_prefill_decode_gb300 import workload as W
from gpu_util import to_dev, from_dev, dev_buffer_bits, assert_close, f64, rel_err

pytestmark = pytest.mark.gpu

BUFS = {"xn": 0, "qkv": 1, "q": 2, "o": 3, "h": 4, "hn": 5, "a": 6}


def _stream():
    return torch.cuda.current_stream().cuda_stream


class Run:
    def __init__(self, mb, wl: W.Workload, unit_gains=False):
        self.wl = wl
        self.shape = wl.shape
        self.wb, self.x, self.batch, self.pool = W.materialize(wl, unit_gains=unit_gains)
        self.dw = {k: to_dev(v) for k, v in self.wb.items()}
        self.dpool = to_dev(self.pool.reshape(-1))
        self.layer = mb.Layer(self.shape.as_dict(), self.dw, max_tokens=max(1, self.batch.num_tokens),
                              num_pages=self.pool.shape[0], kv_buf=self.dpool)
        self.mb = mb

    def step(self):
        dx = to_dev(self.x)
        dy = torch.empty_like(dx)
        self.layer.step(self.mb.Batch.of(self.batch), dx, dy, _stream())
        self.mb.mb_device_status(self.layer.handle, _stream())
        self.y = from_dev(dy)
        self.pool_after = from_dev(self.dpool).reshape(self.pool.shape)
        self.bufs = {k: dev_buffer_bits(*self.layer.buffer(i)) for k, i in BUFS.items()}
        return self

    def oracle(self):
        self.opool = f64(self.pool)
        self.ref = OL.layer_step(self.shape.as_dict(), OL.weights_to_f64(self.wb), self.opool,
                                 self.batch.qo_indptr, self.batch.kv_len, self.batch.bt_indptr, self.batch.bt,
                                 f64(self.x))
        return self

    def close(self):
        self.layer.close()


def check_kv(run: Run):
    """Bit-exact placement + values of the written slots."""
    sh = run.shape
    written = np.zeros(run.pool.shape[0] * 16, dtype=bool)
    for page, slot in run.ref["written"]:
        written[page * 16 + slot] = True
    before = run.pool.transpose(0, 3, 1, 2, 4).reshape(-1, 2 * sh.n_kv_heads * sh.head_dim)
    after = run.pool_after.transpose(0, 3, 1, 2, 4).reshape(-1, 2 * sh.n_kv_heads * sh.head_dim)
    untouched_equal = np.array_equal(before[~written], after[~written])
    assert untouched_equal, "a slot outside this step's (page, slot) set changed"
    ref = run.opool.transpose(0, 3, 1, 2, 4).reshape(-1, 2, sh.n_kv_heads * sh.head_dim)
    got = f64(after).reshape(-1, 2, sh.n_kv_heads * sh.head_dim)
    ek = assert_close("K appended", got[written, 0], ref[written, 0])
    ev = assert_close("V appended", got[written, 1], ref[written, 1])
    return ek, ev


def check_all(run: Run):
    T = run.batch.num_tokens
    sh = run.shape
    errs = {}
    errs["k"], errs["v"] = check_kv(run)
    errs["xn"] = assert_close("xn", f64(run.bufs["xn"]).reshape(T, -1), run.ref["xn"])
    errs["qkv"] = assert_close("qkv", f64(run.bufs["qkv"]).reshape(T, -1), run.ref["qkv"])
    errs["q"] = assert_close("q (rotated)", f64(run.bufs["q"]).reshape(T, sh.n_q_heads, sh.head_dim), run.ref["q"])
    errs["o"] = assert_close("attention o", f64(run.bufs["o"]).reshape(T, -1), run.ref["o"])
    errs["h"] = assert_close("h", f64(run.bufs["h"]).reshape(T, -1), run.ref["h"])
    errs["hn"] = assert_close("hn", f64(run.bufs["hn"]).reshape(T, -1), run.ref["hn"])
    errs["a"] = assert_close("a (SwiGLU)", f64(run.bufs["a"]).reshape(T, -1), run.ref["a"])
    errs["y"] = assert_close("y", f64(run.y).reshape(T, -1), run.ref["y"])
    return errs


def check_attention_isolated(run: Run):
    """Oracle attention on the GPU's own q and KV pool vs the GPU's o."""
    sh = run.shape
    T = run.batch.num_tokens
    q = f64(run.bufs["q"]).reshape(T, sh.n_q_heads, sh.head_dim)
    pool = f64(run.pool_after)
    b = run.batch
    o_ref = np.empty((T, sh.n_q_heads, sh.head_dim))
    for r in range(b.num_reqs):
        t0, t1 = b.qo_indptr[r], b.qo_indptr[r + 1]
        table = b.bt[b.bt_indptr[r]:b.bt_indptr[r + 1]]
        K, V = OL.gather_kv(pool, table, int(b.kv_len[r]))
        o_ref[t0:t1] = OL.attention_request(q[t0:t1], K, V, int(b.kv_len[r]) - (t1 - t0))
    got = f64(run.bufs["o"]).reshape(T, sh.n_q_heads, sh.head_dim)
    # decode rows and chunk rows separately, so that neither hides behind the other
    qo = b.qo_len()
    dec_rows = np.concatenate([np.arange(b.qo_indptr[r], b.qo_indptr[r + 1]) for r in range(b.num_reqs)
                               if qo[r] == 1] or [np.zeros(0, int)])
    chk_rows = np.concatenate([np.arange(b.qo_indptr[r], b.qo_indptr[r + 1]) for r in range(b.num_reqs)
                               if qo[r] > 1] or [np.zeros(0, int)])
    e = {}
    if len(dec_rows):
        e["decode"] = assert_close("decode attention", got[dec_rows], o_ref[dec_rows])
    if len(chk_rows):
        e["chunk"] = assert_close("chunk attention", got[chk_rows], o_ref[chk_rows])
    return e


WORKLOADS = {
    "tiny_T68": lambda: W.tiny_mixed(),
    "gqa4_small": lambda: W.small_mixed(W.SMALL_GQA, seed=101),
    "g5_qknorm_small": lambda: W.small_mixed(W.SMALL_G5_QKN, seed=102, n_dec=7, chunk=333, prefix=250),
    "gqa4_edges": lambda: W.Workload("edges", W.SMALL_GQA,
                                     [(0, 1), (1, 1), (14, 1), (15, 1), (16, 1), (63, 1), (64, 1), (128, 1),
                                      (0, 2), (15, 129), (0, 300), (127, 2), (1000, 1)], 104),
    "tiny_decode_only": lambda: W.Workload("dec", W.TINY, [(5, 1), (300, 1), (17, 1)], 105),
    "tiny_one_chunk": lambda: W.Workload("chunk", W.TINY, [(0, 256)], 106),
    # few chunk tiles over long prefixes: each tile's keys are split into
    # pieces merged by log-sum-exp (a 256-row tile, a tile of 44 rows, and a
    # 100-row chunk whose second query tile is empty)
    "gqa4_split_tiles": lambda: W.Workload("split", W.SMALL_GQA, [(3000, 1), (4000, 256), (5000, 1)], 107),
    "g5_qknorm_split_ragged": lambda: W.Workload("split5", W.SMALL_G5_QKN, [(2500, 300), (777, 1), (3100, 100)],
                                                 108),
}


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_step_parity_small(mb, name):
    run = Run(mb, WORKLOADS[name]()).step().oracle()
    try:
        errs = check_all(run)
        errs.update(check_attention_isolated(run))
        print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    finally:
        run.close()


@pytest.mark.parametrize("name", ["llama3_8b_T576"] + [f"qwen3_14b_P{p}" for p in (0, 1024, 2200)])
def test_step_parity_full_size(mb, name):
    wl = W.llama3_8b_mixed() if name.startswith("llama") else W.qwen3_14b_mixed(int(name.split("P")[1]))
    run = Run(mb, wl, unit_gains=True).step().oracle()
    try:
        errs = check_all(run)
        errs.update(check_attention_isolated(run))
        print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    finally:
        run.close()


def test_chunked_steps_match_oracle_and_repeat(mb):
    """A 300-token prompt fed as chunks 100 + 37 + 163 through three mb_step
    calls, alongside two decodes, matches the oracle run the same way; a
    repeated step gives bit-identical outputs."""
    sh = W.SMALL_GQA
    wb = W.make_weights(sh, 301)
    dw = {k: to_dev(v) for k, v in wb.items()}
    prompt = W.make_embeddings(300, sh.d_model, 302)
    dec_ctx = [40, 90]
    batches = []
    num_pages = 64
    perm = np.random.default_rng(303).permutation(num_pages).astype(np.int32)
    tables = {0: perm[:19], 1: perm[19:23], 2: perm[23:30]}
    pool = np.full((num_pages, 2, sh.n_kv_heads, 16, sh.head_dim), W.KV_SENTINEL, np.uint16)
    rng = np.random.default_rng(304)
    for i, c in enumerate(dec_ctx):
        for p in range(c):
            pool[tables[i + 1][p // 16], :, :, p % 16] = W.f32_to_bf16_bits(
                rng.standard_normal((2, sh.n_kv_heads, sh.head_dim), dtype=np.float32))
    dpool = to_dev(pool.reshape(-1))
    layer = mb.Layer(sh.as_dict(), dw, max_tokens=512, num_pages=num_pages, kv_buf=dpool)
    opool = f64(pool)
    ow = OL.weights_to_f64(wb)
    done = 0
    try:
        for step, n in enumerate([100, 37, 163]):
            kvs = [done + n, dec_ctx[0] + step + 1, dec_ctx[1] + step + 1]
            qo = [0, n, n + 1, n + 2]
            bti = [0]
            bt = []
            for r, kvl in enumerate(kvs):
                tbl = tables[r][: W.pages_for(kvl)]
                bt.extend(tbl)
                bti.append(len(bt))
            dec_x = W.make_embeddings(2, sh.d_model, 400 + step)
            x = np.concatenate([prompt[done:done + n], dec_x])
            dx = to_dev(x)
            dy = torch.empty_like(dx)
            batch = mb.Batch(qo, kvs, bti, bt)
            layer.step(batch, dx, dy, _stream())
            mb.mb_device_status(layer.handle, _stream())
            y1 = from_dev(dy)
            ref = OL.layer_step(sh.as_dict(), ow, opool, qo, kvs, bti, bt, f64(x))
            assert_close(f"chunked step {step} y", f64(y1), ref["y"])
            if step == 1:
                # the same step again rewrites the same slots with the same values
                layer.step(batch, dx, dy, _stream())
                mb.mb_device_status(layer.handle, _stream())
                assert np.array_equal(from_dev(dy), y1)
            done += n
        got_pool = f64(from_dev(dpool).reshape(pool.shape))
        for r in range(3):
            n_tok = [300, dec_ctx[0] + 3, dec_ctx[1] + 3][r]
            Kg, Vg = OL.gather_kv(got_pool, tables[r], n_tok)
            Kr, Vr = OL.gather_kv(opool, tables[r], n_tok)
            assert_close(f"kv of request {r}", np.stack([Kg, Vg]), np.stack([Kr, Vr]))
    finally:
        layer.close()


def test_empty_batch_is_noop(mb):
    sh = W.TINY
    wb = W.make_weights(sh, 5)
    dw = {k: to_dev(v) for k, v in wb.items()}
    layer = mb.Layer(sh.as_dict(), dw, max_tokens=16, num_pages=4)
    try:
        x = torch.zeros((1, sh.d_model), dtype=torch.bfloat16, device="cuda")
        y = torch.zeros_like(x)
        layer.step(mb.Batch([0], [], [0], []), x, y, _stream())
        mb.mb_device_status(layer.handle, _stream())
        assert mb.mb_layer_last_launches(layer.handle) == 0
    finally:
        layer.close()


def test_step_rejects_malformed_descriptor_before_launch(mb):
    sh = W.TINY
    wb = W.make_weights(sh, 6)
    dw = {k: to_dev(v) for k, v in wb.items()}
    layer = mb.Layer(sh.as_dict(), dw, max_tokens=16, num_pages=4)
    try:
        x = torch.zeros((2, sh.d_model), dtype=torch.bfloat16, device="cuda")
        y = torch.zeros_like(x)
        with pytest.raises(mb.MbError) as e:
            layer.step(mb.Batch([0, 2], [1], [0, 1], [0]), x, y, _stream())   # kv_len < qo_len
        assert e.value.status == mb.MB_EINVAL
        with pytest.raises(mb.MbError):
            layer.step(mb.Batch([0, 1], [1], [0, 1], [9]), x, y, _stream())   # page out of range
        with pytest.raises(mb.MbError):
            layer.step(mb.Batch([0, 17], [17], [0, 2], [0, 1]), x, y, _stream())  # T > max_tokens
    finally:
        layer.close()


@pytest.mark.parametrize("name", ["llama3_8b_T576", "qwen3_14b_P0", "qwen3_14b_P2200"])
def test_many_repeats_bit_identical(mb, name):
    """Several hundred back-to-back steps on one input: every output equals the
    first bit for bit and no kernel reports an error.  Rare pipeline races
    (a ring slot read before its copy lands, TMEM freed under an MMA) show up
    here as a mismatch or an error word long before a single step would."""
    wl = W.llama3_8b_mixed() if name.startswith("llama") else W.qwen3_14b_mixed(int(name.split("P")[1]))
    wb, x, batch, pool = W.materialize(wl, unit_gains=True)
    dw = {k: to_dev(v) for k, v in wb.items()}
    dpool = to_dev(pool.reshape(-1))
    layer = mb.Layer(wl.shape.as_dict(), dw, batch.num_tokens, pool.shape[0], kv_buf=dpool)
    try:
        cb = mb.Batch.of(batch)
        dx = to_dev(x)
        first = torch.empty_like(dx)
        dy = torch.empty_like(dx)
        layer.step(cb, dx, first, _stream())
        mismatches = torch.zeros((), dtype=torch.int64, device=dx.device)
        for _ in range(400):
            layer.step(cb, dx, dy, _stream())
            mismatches += (dy.view(torch.int16) != first.view(torch.int16)).any().to(torch.int64)
        mb.mb_device_status(layer.handle, _stream())
        assert int(mismatches) == 0, f"{int(mismatches)} of 400 repeated steps differ from the first"
    finally:
        layer.close()


@pytest.mark.parametrize("name,caps", [("llama3_8b_T576", (1, 5, 24, 0)), ("qwen3_14b_P2200", (3, 40, 0))])
def test_decode_sm_cap_is_bit_identical(mb, name, caps):
    """Capping the decode-worker CTAs (the decode SM partition) changes only
    which worker takes which decode item, not what an item computes: every
    cap gives the uncapped output bit for bit."""
    wl = W.llama3_8b_mixed() if name.startswith("llama") else W.qwen3_14b_mixed(int(name.split("P")[1]))
    wb, x, batch, pool = W.materialize(wl, unit_gains=True)
    dw = {k: to_dev(v) for k, v in wb.items()}
    dpool = to_dev(pool.reshape(-1))
    layer = mb.Layer(wl.shape.as_dict(), dw, batch.num_tokens, pool.shape[0], kv_buf=dpool)
    try:
        cb = mb.Batch.of(batch)
        dx = to_dev(x)
        ref = torch.empty_like(dx)
        layer.step(cb, dx, ref, _stream())
        for cap in caps:
            mb.mb_layer_set_decode_sms(layer.handle, cap)
            dy = torch.empty_like(dx)
            for _ in range(3):
                layer.step(cb, dx, dy, _stream())
            mb.mb_device_status(layer.handle, _stream())
            assert torch.equal(dy.view(torch.int16), ref.view(torch.int16)), f"decode SM cap {cap}"
        with pytest.raises(mb.MbError):
            mb.mb_layer_set_decode_sms(layer.handle, -1)
    finally:
        layer.close()


def test_two_micro_batches_on_two_streams(mb):
    """The decode rows and the chunk rows of one batch as two micro-batches,
    stepped by two layers over the same weights and KV pool, each with a GEMM
    workspace of its own, on two streams at once, under SM caps that add up to
    the SM count (the decode attention of one beside the GEMMs of the other,
    as ConfluxServe overlaps them): every row matches the oracle's full-batch
    step, and each micro-batch equals the same micro-batch run alone bit for
    bit (the schedules depend only on the shapes and caps)."""
    wl = W.small_mixed(W.SMALL_GQA, seed=121, n_dec=9, chunk=300, prefix=2500)
    wb, x, batch, pool = W.materialize(wl)
    sh = wl.shape
    ref = OL.layer_step(sh.as_dict(), OL.weights_to_f64(wb), f64(pool), batch.qo_indptr, batch.kv_len,
                        batch.bt_indptr, batch.bt, f64(x))
    qo = batch.qo_len()
    dec = [r for r in range(batch.num_reqs) if qo[r] == 1]
    chk = [r for r in range(batch.num_reqs) if qo[r] > 1]

    def sub(rs):
        rows = np.concatenate([np.arange(batch.qo_indptr[r], batch.qo_indptr[r + 1]) for r in rs])
        q = np.cumsum([0] + [int(qo[r]) for r in rs]).astype(np.int32)
        tabs = [batch.bt[batch.bt_indptr[r]:batch.bt_indptr[r + 1]] for r in rs]
        bti = np.cumsum([0] + [len(t) for t in tabs]).astype(np.int32)
        return rows, W.Batch(q, batch.kv_len[rs].astype(np.int32), bti, np.concatenate(tabs).astype(np.int32))

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    parts = {"decode": sub(dec), "chunk": sub(chk)}
    caps = {"decode": (sms // 6, sms // 6), "chunk": (sms - sms // 6, 0)}   # (GEMM CTAs, decode workers)
    dw = {k: to_dev(v) for k, v in wb.items()}
    dpool = to_dev(pool.reshape(-1))
    layers, ws, outs = {}, {}, {}
    try:
        for name, (rows, b) in parts.items():
            L = mb.Layer(sh.as_dict(), dw, b.num_tokens, pool.shape[0], kv_buf=dpool)
            ws[name] = torch.zeros(mb.mb_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
            mb.mb_layer_set_gemm_workspace(L.handle, ws[name])
            mb.mb_layer_set_gemm_sms(L.handle, caps[name][0])
            mb.mb_layer_set_decode_sms(L.handle, caps[name][1])
            layers[name] = L
        xs = {name: to_dev(x[rows]) for name, (rows, b) in parts.items()}
        alone = {}
        for name, (rows, b) in parts.items():   # each micro-batch alone, one stream
            y = torch.empty_like(xs[name])
            layers[name].step(mb.Batch.of(b), xs[name], y, _stream())
            mb.mb_device_status(layers[name].handle, _stream())
            alone[name] = from_dev(y)
        streams = {name: torch.cuda.Stream() for name in parts}
        start = torch.cuda.Event()
        start.record()
        for rep in range(3):
            for name, (rows, b) in parts.items():
                s = streams[name]
                s.wait_event(start)
                outs[name] = torch.empty_like(xs[name])
                with torch.cuda.stream(s):
                    layers[name].step(mb.Batch.of(b), xs[name], outs[name], s.cuda_stream)
            for name in parts:
                mb.mb_device_status(layers[name].handle, streams[name].cuda_stream)
                assert np.array_equal(from_dev(outs[name]), alone[name]), f"{name} on two streams, rep {rep}"
        for name, (rows, b) in parts.items():
            assert_close(f"{name} micro-batch y", f64(alone[name]).reshape(len(rows), -1), ref["y"][rows])
    finally:
        for L in layers.values():
            L.close()
