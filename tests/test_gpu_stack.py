"""GPU checks of the layer stack (several layers, one descriptor per step).

* A stack's output is bit-identical to chaining mb_step layer by layer (the
  same kernels in the same order), with and without CUDA graphs, including a
  graph replay after the descriptor's block tables changed.
* A small stack matches the oracle composed over its layers.
* The 40-layer Qwen3-14B-shaped stack with a 2,048-token chunk at prefix
  30,720 and 96 decodes: layers 0, 19 and 39 match the oracle fed the GPU's
  input to each (per-layer checks at full size), and the graph-replayed stack
  equals the chained steps bit for bit at that size.
* The 32-layer Llama-3-8B-shaped stack at the token-budget sweep's smallest
  point, checked layer by layer."""

import numpy as np
import pytest
import torch

from oracle import layer as OL
from mixed_prefill_decode_gb300 import workload as W
from gpu_util import to_dev, from_dev, assert_close, f64

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _small_stack(mb, n_layers=3, shape=W.SMALL_G5_QKN, seed=700):
    wl = W.small_mixed(shape, seed=seed, n_dec=6, chunk=230, prefix=140)
    batch, num_pages = W.make_batch(wl.reqs, seed + 1, spare_pages=4)
    x = W.make_embeddings(batch.num_tokens, shape.d_model, seed + 2)
    layers, pools, wbits = [], [], []
    for l in range(n_layers):
        wb = W.make_weights(shape, seed + 10 + l)
        pool = W.make_kv_pool(shape, num_pages, batch, seed + 20 + l)
        dw = {k: to_dev(v) for k, v in wb.items()}
        dpool = to_dev(pool.reshape(-1))
        layers.append(mb.Layer(shape.as_dict(), dw, batch.num_tokens, num_pages, kv_buf=dpool))
        pools.append((pool, dpool))
        wbits.append(wb)
    return wl, batch, x, layers, pools, wbits


def _chain(mb, layers, batch, x):
    cur = to_dev(x)
    for L in layers:
        out = torch.empty_like(cur)
        L.step(mb.Batch.of(batch), cur, out, _stream())
        cur = out
    mb.mb_device_status(layers[0].handle, _stream())
    return from_dev(cur)


@pytest.mark.parametrize("graphs", [False, True])
def test_stack_equals_chained_steps_and_oracle(mb, graphs):
    wl, batch, x, layers, pools, wbits = _small_stack(mb)
    try:
        ref_bits = _chain(mb, layers, batch, x)
        stack = mb.mb_stack_create([L.handle for L in layers], graphs)
        try:
            dx = to_dev(x)
            dy = torch.empty_like(dx)
            for rep in range(3):   # capture, then replays
                dy.fill_(float("nan"))
                mb.mb_stack_step(stack, [L.kv for L in layers], mb.Batch.of(batch), dx, dy, _stream())
                mb.mb_device_status(layers[0].handle, _stream())
                assert np.array_equal(from_dev(dy), ref_bits), f"stack differs from chained steps (rep {rep})"
            assert mb.mb_stack_last_launches(stack) == len(layers) * mb.mb_layer_last_launches(layers[0].handle)
        finally:
            mb.mb_stack_destroy(stack)
        # oracle over the layers (pools as they were before the GPU steps)
        h = f64(x)
        for l in range(len(layers)):
            r = OL.layer_step(wl.shape.as_dict(), OL.weights_to_f64(wbits[l]), f64(pools[l][0]),
                              batch.qo_indptr, batch.kv_len, batch.bt_indptr, batch.bt, h)
            h = r["y"]
        assert_close("3-layer stack y", f64(ref_bits).reshape(h.shape), h)
    finally:
        for L in layers:
            L.close()


def test_stack_graph_replay_after_descriptor_change(mb):
    """Same geometry, different block tables: the replayed graph reads the new
    descriptor and matches chained steps on the new tables."""
    wl, batch, x, layers, pools, wbits = _small_stack(mb, n_layers=2, shape=W.SMALL_GQA, seed=800)
    try:
        stack = mb.mb_stack_create([L.handle for L in layers], True)
        try:
            dx = to_dev(x)
            dy = torch.empty_like(dx)
            mb.mb_stack_step(stack, [L.kv for L in layers], mb.Batch.of(batch), dx, dy, _stream())
            # relabel every page id: same geometry, different tables
            num_pages = pools[0][0].shape[0]
            relabel = np.random.default_rng(5).permutation(num_pages).astype(np.int32)
            b2 = W.Batch(batch.qo_indptr, batch.kv_len, batch.bt_indptr, relabel[batch.bt])
            dy.fill_(float("nan"))
            mb.mb_stack_step(stack, [L.kv for L in layers], mb.Batch.of(b2), dx, dy, _stream())
            mb.mb_device_status(layers[0].handle, _stream())
            got = from_dev(dy)
            assert np.array_equal(got, _chain(mb, layers, b2, x))
        finally:
            mb.mb_stack_destroy(stack)
    finally:
        for L in layers:
            L.close()


def test_stack_graph_replay_over_a_growing_prefix(mb):
    """A prompt fed chunk by chunk through a graph-replayed stack: every step
    has the same geometry (decodes plus one 128-row chunk) but a longer block
    table for the chunk; each step equals the chained mb_step calls on the
    same descriptor bit for bit, and the last one matches the oracle."""
    sh = W.SMALL_GQA
    sw = W.PromptSweep("small_prompt", sh, 2, [40, 333, 900], 512, 128, 901)
    full, num_pages = sw.layout(spare_pages=4)
    pools0 = [W.make_kv_pool(sh, num_pages, full, 910 + l) for l in range(sw.n_layers)]
    wbits = [W.make_weights(sh, 920 + l) for l in range(sw.n_layers)]
    T = sw.batch_at(0, full).num_tokens

    def make_layers():
        out = []
        for l in range(sw.n_layers):
            dw = {k: to_dev(v) for k, v in wbits[l].items()}
            out.append((mb.Layer(sh.as_dict(), dw, T, num_pages, kv_buf=to_dev(pools0[l].reshape(-1))), dw))
        return out

    chained, stacked = make_layers(), make_layers()
    stack = mb.mb_stack_create([L.handle for L, _ in stacked], True)
    try:
        opools = [f64(p) for p in pools0]
        for k in range(sw.steps):
            b = sw.batch_at(k, full)
            x = W.make_embeddings(T, sh.d_model, 930 + k)
            want = _chain(mb, [L for L, _ in chained], b, x)
            dy = torch.empty_like(to_dev(x))
            mb.mb_stack_step(stack, [L.kv for L, _ in stacked], mb.Batch.of(b), to_dev(x), dy, _stream())
            mb.mb_device_status(stacked[0][0].handle, _stream())
            assert np.array_equal(from_dev(dy), want), f"graph replay at prefix {k * sw.chunk}"
            h = f64(x)
            for l in range(sw.n_layers):
                h = OL.layer_step(sh.as_dict(), OL.weights_to_f64(wbits[l]), opools[l], b.qo_indptr, b.kv_len,
                                  b.bt_indptr, b.bt, h)["y"]
            assert_close(f"stack at prefix {k * sw.chunk}", f64(want).reshape(h.shape), h)
    finally:
        mb.mb_stack_destroy(stack)
        for L, _ in chained + stacked:
            L.close()


def _chain_full_size(mb, wl, n_layers, weight_seed, pool_seed, check_layers):
    """Run an n_layers stack of full-size layers (weights and KV drawn on the
    device) as chained mb_step calls, keeping the input and output of the
    layers in check_layers; then the same layers as one stack (CUDA graph)
    must give the chain's output bit for bit.  Each checked layer is compared
    with the oracle fed the GPU's bf16 input to that layer."""
    sh = wl.shape
    batch, num_pages = W.make_batch(wl.reqs, wl.seed + 1, spare_pages=4)
    x = W.make_embeddings(batch.num_tokens, sh.d_model, wl.seed + 2)
    layers, dws = [], []
    errs = {}
    try:
        for l in range(n_layers):
            dw = W.device_weights(sh, weight_seed + l)
            dpool = W.device_kv_pool(sh, num_pages, pool_seed + l)
            layers.append(mb.Layer(sh.as_dict(), dw, batch.num_tokens, num_pages, kv_buf=dpool))
            dws.append((dw, dpool))
        cb = mb.Batch.of(batch)
        cur = to_dev(x)
        io = {}
        for l, L in enumerate(layers):
            out = torch.empty_like(cur)
            L.step(cb, cur, out, _stream())
            if l in check_layers:
                io[l] = (from_dev(cur), None)
                mb.mb_device_status(L.handle, _stream())
                io[l] = (io[l][0], from_dev(out))
            cur = out
        mb.mb_device_status(layers[0].handle, _stream())
        chain_out = from_dev(cur)
        stack = mb.mb_stack_create([L.handle for L in layers], True)
        try:
            y = torch.empty_like(cur)
            mb.mb_stack_step(stack, [L.kv for L in layers], cb, to_dev(x), y, _stream())
            mb.mb_device_status(layers[0].handle, _stream())
            assert np.array_equal(from_dev(y), chain_out), "stack (graph) differs from the chained steps"
        finally:
            mb.mb_stack_destroy(stack)
        for l in sorted(check_layers):
            xin, yout = io[l]
            wbits = {k: from_dev(v) for k, v in dws[l][0].items()}
            # the step's own slots are rewritten by the oracle before it attends;
            # every other slot is as the layer found it
            pool = f64(from_dev(dws[l][1]))
            r = OL.layer_step(sh.as_dict(), OL.weights_to_f64(wbits), pool, batch.qo_indptr, batch.kv_len,
                              batch.bt_indptr, batch.bt, f64(xin))
            del pool
            errs[l] = assert_close(f"{wl.name} layer {l} y", f64(yout).reshape(r["y"].shape), r["y"])
        return batch, errs
    finally:
        for L in layers:
            L.close()


def test_qwen3_14b_stack40_layers_match_oracle(mb):
    """The 40-layer Qwen3-14B-shaped stack, a 2,048-token chunk after 30,720
    cached tokens plus 96 decodes with contexts log-uniform in [1024, 8192]:
    layers 0, 19 and 39 each match the oracle fed the GPU's input to that
    layer, and the stack's graph equals the chained steps bit for bit."""
    wl, n_layers = W.qwen3_14b_stack(prefix=30720)
    batch, errs = _chain_full_size(mb, wl, n_layers, wl.seed + 100, wl.seed + 200, {0, 19, 39})
    print(f"{wl.name}: T={batch.num_tokens}", {l: f"{e:.2e}" for l, e in errs.items()})


def test_llama3_8b_stack32_smallest_sweep_point_layer_by_layer(mb):
    """The 32-layer Llama-3-8B-shaped stack at the sweep's smallest point
    (budget 256, one decode with a context log-uniform in [512, 32768] and a
    255-token chunk after a prefix uniform in [0, 16384]): every layer matches
    the oracle fed the GPU's input to it."""
    wl, n_layers = W.llama3_8b_stack(256, 1)
    batch, errs = _chain_full_size(mb, wl, n_layers, 5100, wl.seed + 200, set(range(n_layers)))
    print(f"{wl.name}: T={batch.num_tokens}, kv={list(batch.kv_len)}",
          f"max layer error {max(errs.values()):.2e}")
