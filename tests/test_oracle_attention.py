"""Pins for the oracle's paged attention and for the layer-level invariants the
pages fix.  CPU only.

* torch's scaled_dot_product_attention (float64, explicit boolean mask, KV
  heads expanded) on KV gathered into contiguous arrays: the library routine
  the masked-softmax definition of llm-stack-book 7.8 reduces to.
* kv_len = 1 gives o = v; identical keys give the mean of the visible values;
  a dominant key selects its value.
* Chunked prefill == one unchunked prefill, for the KV cache and the outputs
  (llm-stack-book 7.8, "Choosing the Chunk Size" and "Attention on Partial KV
  Caches"); a decode step == the last row of a prefill over the same tokens.
* Page permutation and batch composition do not change any request's result.
"""

import math

import numpy as np
import pytest
import torch

from oracle import layer as L
from mixed_prefill_decode_gb300 import workload as W


def _sdpa_reference(q, K, V, cached):
    """torch SDPA on contiguous KV with the chunk mask: row i sees j <= cached+i."""
    qo, Hq, hd = q.shape
    kv, Hkv, _ = K.shape
    group = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)                      # [Hq, qo, hd]
    kt = torch.from_numpy(K).repeat_interleave(group, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(V).repeat_interleave(group, dim=1).permute(1, 0, 2)
    mask = torch.arange(kv)[None, :] <= (cached + torch.arange(qo))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    return out.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv,hd,cached,qo", [
    (4, 4, 64, 0, 1), (4, 4, 64, 37, 1), (8, 2, 128, 100, 33), (10, 2, 128, 0, 50),
    (6, 3, 32, 17, 17), (5, 1, 16, 250, 1)])
def test_attention_matches_sdpa(Hq, Hkv, hd, cached, qo):
    rng = np.random.default_rng(Hq * 1000 + cached + qo)
    kv = cached + qo
    q = rng.standard_normal((qo, Hq, hd))
    K = rng.standard_normal((kv, Hkv, hd))
    V = rng.standard_normal((kv, Hkv, hd))
    got = L.attention_request(q, K, V, cached)
    ref = _sdpa_reference(q, K, V, cached)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_attention_single_key_returns_value():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 4, 64))
    K = rng.standard_normal((1, 2, 64))
    V = rng.standard_normal((1, 2, 64))
    o = L.attention_request(q, K, V, 0)
    for h in range(4):
        np.testing.assert_allclose(o[0, h], V[0, h // 2], rtol=0, atol=1e-15)


def test_attention_identical_keys_average_visible_values():
    rng = np.random.default_rng(2)
    cached, qo, hd = 9, 5, 16
    kv = cached + qo
    k = rng.standard_normal(hd)
    K = np.broadcast_to(k, (kv, 1, hd)).copy()
    V = rng.standard_normal((kv, 1, hd))
    q = rng.standard_normal((qo, 2, hd))
    o = L.attention_request(q, K, V, cached)
    for i in range(qo):
        vis = cached + i + 1
        for h in range(2):
            np.testing.assert_allclose(o[i, h], V[:vis, 0].mean(axis=0), rtol=1e-12, atol=1e-13)


def test_attention_dominant_key_selects_its_value_and_mask_hides_future():
    hd, kv = 8, 6
    K = np.zeros((kv, 1, hd))
    V = np.arange(kv * hd, dtype=np.float64).reshape(kv, 1, hd)
    q = np.zeros((3, 1, hd))
    q[:, 0, 0] = 200.0
    K[2, 0, 0] = 1.0      # key 2 dominates wherever it is visible
    K[5, 0, 0] = 2.0      # key 5 dominates more but is only visible to the last row
    o = L.attention_request(q, K, V, cached=3)    # rows at positions 3, 4, 5
    np.testing.assert_allclose(o[0, 0], V[2, 0], atol=1e-9)
    np.testing.assert_allclose(o[1, 0], V[2, 0], atol=1e-9)
    np.testing.assert_allclose(o[2, 0], V[5, 0], atol=1e-9)


def test_gather_through_block_table_is_page_order_independent():
    rng = np.random.default_rng(3)
    Hkv, hd, n = 2, 16, 45
    K = rng.standard_normal((n, Hkv, hd))
    V = rng.standard_normal((n, Hkv, hd))
    outs = []
    for seed in (0, 1):
        perm = np.random.default_rng(seed).permutation(10)
        table = perm[: W.pages_for(n)]
        pool = np.full((10, 2, Hkv, 16, hd), np.nan)
        for p in range(n):
            pool[table[p // 16], 0, :, p % 16] = K[p]
            pool[table[p // 16], 1, :, p % 16] = V[p]
        Kg, Vg = L.gather_kv(pool, table, n)
        np.testing.assert_array_equal(Kg, K)
        np.testing.assert_array_equal(Vg, V)
        outs.append(L.attention_request(rng.standard_normal((1, 4, hd)) * 0 + 1.0, Kg, Vg, n - 1))
    np.testing.assert_array_equal(outs[0], outs[1])


# --------------------------------------------------------------------------
# layer-level invariants
# --------------------------------------------------------------------------

def _run_steps(shape, w, x_all, steps, num_pages=64, seed=0):
    """Feed one request's tokens through consecutive layer steps.

    steps: list of token counts per step.  Returns (y rows concatenated in
    token order, pool, table)."""
    Hkv, hd = shape.n_kv_heads, shape.head_dim
    pool = np.zeros((num_pages, 2, Hkv, 16, hd))
    table = np.random.default_rng(seed).permutation(num_pages).astype(np.int64)
    ys, done = [], 0
    for n in steps:
        kv = done + n
        r = L.layer_step(shape.as_dict(), w, pool, [0, n], [kv], [0, W.pages_for(kv)],
                         table[: W.pages_for(kv)], x_all[done:done + n])
        ys.append(r["y"])
        done = kv
    return np.concatenate(ys), pool, table


def _f64_weights(shape, seed):
    return L.weights_to_f64(W.make_weights(shape, seed))


@pytest.mark.parametrize("shape", [W.TINY, W.SMALL_G5_QKN], ids=["tiny", "g5_qknorm"])
def test_chunked_prefill_equals_unchunked(shape):
    w = _f64_weights(shape, 11)
    n = 61
    x = L.bf16_bits_to_f64(W.make_embeddings(n, shape.d_model, 12))
    y1, pool1, table = _run_steps(shape, w, x, [n])
    y2, pool2, table2 = _run_steps(shape, w, x, [16, 7, 30, 8])
    assert np.array_equal(table, table2)
    np.testing.assert_allclose(y2, y1, rtol=1e-9, atol=1e-9)
    pages = table[: W.pages_for(n)]
    kv1 = np.stack([pool1[pages[p // 16], :, :, p % 16] for p in range(n)])
    kv2 = np.stack([pool2[pages[p // 16], :, :, p % 16] for p in range(n)])
    np.testing.assert_allclose(kv2, kv1, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("shape", [W.TINY, W.SMALL_GQA], ids=["tiny", "gqa4"])
def test_decode_equals_last_row_of_prefill(shape):
    w = _f64_weights(shape, 21)
    n = 40
    x = L.bf16_bits_to_f64(W.make_embeddings(n, shape.d_model, 22))
    y_full, _, _ = _run_steps(shape, w, x, [n])
    y_dec, _, _ = _run_steps(shape, w, x, [n - 1, 1])
    np.testing.assert_allclose(y_dec[-1], y_full[-1], rtol=1e-9, atol=1e-9)
    y_dec2, _, _ = _run_steps(shape, w, x, [n - 3, 1, 1, 1])
    np.testing.assert_allclose(y_dec2[-3:], y_full[-3:], rtol=1e-9, atol=1e-9)


def test_batch_composition_does_not_change_rows():
    """Rows of a mixed batch equal the rows of each request run alone (linear
    layers act per token; attention reads only the request's own pages)."""
    shape = W.SMALL_GQA
    wl = W.small_mixed(shape, seed=31, n_dec=3, chunk=40, prefix=20)
    wb, xb, batch, poolb = W.materialize(wl)
    w = L.weights_to_f64(wb)
    x = L.bf16_bits_to_f64(xb)
    pool = L.bf16_bits_to_f64(poolb)
    full = L.layer_step(shape.as_dict(), w, pool.copy(), batch.qo_indptr, batch.kv_len,
                        batch.bt_indptr, batch.bt, x)
    for r in range(batch.num_reqs):
        t0, t1 = batch.qo_indptr[r], batch.qo_indptr[r + 1]
        table = batch.bt[batch.bt_indptr[r]:batch.bt_indptr[r + 1]]
        alone = L.layer_step(shape.as_dict(), w, pool.copy(), [0, t1 - t0], [batch.kv_len[r]],
                             [0, len(table)], table, x[t0:t1])
        np.testing.assert_allclose(alone["y"], full["y"][t0:t1], rtol=1e-10, atol=1e-10)


def test_append_places_tokens_by_page_and_slot():
    shape = W.TINY
    wl = W.tiny_mixed()
    wb, xb, batch, poolb = W.materialize(wl)
    pool = L.bf16_bits_to_f64(poolb)
    r = L.layer_step(shape.as_dict(), L.weights_to_f64(wb), pool, batch.qo_indptr,
                     batch.kv_len, batch.bt_indptr, batch.bt, L.bf16_bits_to_f64(xb))
    cached = batch.cached()
    for req in range(batch.num_reqs):
        table = batch.bt[batch.bt_indptr[req]:batch.bt_indptr[req + 1]]
        for i, t in enumerate(range(batch.qo_indptr[req], batch.qo_indptr[req + 1])):
            p = cached[req] + i
            assert tuple(r["written"][t]) == (table[p // 16], p % 16)
    # untouched slots keep the sentinel (a NaN) and nothing else became NaN
    touched = np.zeros(pool.shape[0] * 16, bool)
    for req in range(batch.num_reqs):
        table = batch.bt[batch.bt_indptr[req]:batch.bt_indptr[req + 1]]
        for p in range(batch.kv_len[req]):
            touched[table[p // 16] * 16 + p % 16] = True
    slot_nan = np.isnan(pool).any(axis=(1, 2, 4)).reshape(-1)
    assert np.array_equal(slot_nan, ~touched)
