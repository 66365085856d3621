"""GPU checks of the layer stack (several layers, one descriptor per step).

* A stack's output is bit-identical to chaining mb_step layer by layer (the
  same kernels in the same order), with and without CUDA graphs, including a
  graph replay after the descriptor's block tables changed.
* A small stack matches the oracle composed over its layers.
* The 40-layer Qwen3-14B-shaped stack with a 2,048-token chunk at prefix
  30,720 and 96 decodes: its last layer matches the oracle fed the GPU's input
  to that layer (per-layer check at full size)."""

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


def test_qwen3_14b_stack40_last_layer_matches_oracle(mb):
    wl, n_layers = W.qwen3_14b_stack(prefix=30720)
    sh = wl.shape
    batch, num_pages = W.make_batch(wl.reqs, wl.seed + 1, spare_pages=4)
    x = W.make_embeddings(batch.num_tokens, sh.d_model, wl.seed + 2)
    layers, dws = [], []
    try:
        for l in range(n_layers):
            dw = W.device_weights(sh, wl.seed + 100 + l)
            dpool = W.device_kv_pool(sh, num_pages, wl.seed + 200 + l)
            layers.append(mb.Layer(sh.as_dict(), dw, batch.num_tokens, num_pages, kv_buf=dpool))
            dws.append((dw, dpool))
        last_pool_before = dws[-1][1].clone()
        cb = mb.Batch.of(batch)
        dx = to_dev(x)
        # input of the last layer: the first 39 layers as a stack
        s39 = mb.mb_stack_create([L.handle for L in layers[:-1]], True)
        s40 = mb.mb_stack_create([L.handle for L in layers], True)
        try:
            x39 = torch.empty_like(dx)
            mb.mb_stack_step(s39, [L.kv for L in layers[:-1]], cb, dx, x39, _stream())
            y40 = torch.empty_like(dx)
            mb.mb_stack_step(s40, [L.kv for L in layers], cb, dx, y40, _stream())
            mb.mb_device_status(layers[0].handle, _stream())
        finally:
            mb.mb_stack_destroy(s39)
            mb.mb_stack_destroy(s40)
        wl_bits = {k: from_dev(v) for k, v in dws[-1][0].items()}
        r = OL.layer_step(sh.as_dict(), OL.weights_to_f64(wl_bits), f64(from_dev(last_pool_before)),
                          batch.qo_indptr, batch.kv_len, batch.bt_indptr, batch.bt, f64(from_dev(x39)))
        e = assert_close("stack40 layer 39 y", f64(from_dev(y40)).reshape(r["y"].shape), r["y"])
        print(f"stack40 last-layer error {e:.2e}, T={batch.num_tokens}")
    finally:
        for L in layers:
            L.close()
