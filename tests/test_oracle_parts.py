"""Pins for the oracle's RoPE, RMSNorm, linear, SwiGLU and layer composition.
CPU only.  Each check uses a fact other than the oracle's own formula: a
library routine, a closed form, or an invariant."""

import math

import numpy as np
import pytest
import torch

from oracle import layer as L
from mixed_prefill_decode_gb300 import workload as W


# ---- RoPE ---------------------------------------------------------------

def _rope_complex(x, pos, theta):
    """RoPE as complex multiplication: z_i = x_i + i x_{i+hd/2} times
    exp(i pos theta^(-2i/hd))."""
    hd = x.shape[-1]
    half = hd // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = theta ** (-np.arange(half) * 2.0 / hd)
    z = z * np.exp(1j * np.asarray(pos)[..., None] * freq)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 3, 128))
    pos = rng.integers(0, 40000, size=(7, 1))
    np.testing.assert_allclose(L.rope(x, pos, 5e5), _rope_complex(x, pos, 5e5), rtol=1e-12, atol=1e-12)


def test_rope_position_zero_is_identity_and_preserves_pair_norms():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 64))
    np.testing.assert_array_equal(L.rope(x, np.zeros((5,)), 1e4), x)
    y = L.rope(x, np.arange(5) * 997, 1e4)
    n0 = x[:, :32] ** 2 + x[:, 32:] ** 2
    n1 = y[:, :32] ** 2 + y[:, 32:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p, pp, s in [(5, 2, 100), (1000, 17, 3), (0, 0, 31000)]:
        a = L.rope(q, np.array(p + s), 1e6) @ L.rope(k, np.array(pp + s), 1e6)
        b = L.rope(q, np.array(p), 1e6) @ L.rope(k, np.array(pp), 1e6)
        assert abs(a - b) < 1e-10 * (1 + abs(b))


def test_rope_first_pair_rotates_by_position():
    """Pair 0 has frequency 1: a unit vector on x_0 rotates by pos radians."""
    x = np.zeros(8)
    x[0] = 1.0
    y = L.rope(x, np.array(1.0), 1e4)
    assert abs(y[0] - math.cos(1.0)) < 1e-15 and abs(y[4] - math.sin(1.0)) < 1e-15


# ---- RMSNorm ------------------------------------------------------------

def test_rms_norm_matches_torch():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 256)) * 3
    g = 1 + 0.1 * rng.standard_normal(256)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (256,), torch.from_numpy(g), eps=1e-6)
    np.testing.assert_allclose(L.rms_norm(x, g, 1e-6), ref.numpy(), rtol=1e-12)


def test_rms_norm_scale_invariance_and_constant_rows():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 64))
    g = rng.standard_normal(64)
    np.testing.assert_allclose(L.rms_norm(7.5 * x, g, 0.0), L.rms_norm(x, g, 0.0), rtol=1e-12)
    c = np.full((1, 64), -2.0)
    np.testing.assert_allclose(L.rms_norm(c, g, 0.0), -g[None, :], rtol=1e-15)


# ---- linear / SwiGLU ----------------------------------------------------

def test_linear_one_hot_weight_selects_input_column():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 6))
    w = np.zeros((3, 6))
    w[0, 5] = 1.0
    w[2, 1] = 2.0
    y = L.linear(x, w)
    np.testing.assert_array_equal(y[:, 0], x[:, 5])
    np.testing.assert_array_equal(y[:, 1], 0.0)
    np.testing.assert_array_equal(y[:, 2], 2.0 * x[:, 1])


def test_silu_closed_forms():
    assert L.silu(np.array(0.0)) == 0.0
    assert abs(L.silu(np.array(40.0)) - 40.0) < 1e-12
    assert abs(L.silu(np.array(-40.0))) < 1e-15
    assert abs(L.silu(np.array(1.0)) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16


def _zero_layer(shape):
    w = L.weights_to_f64(W.make_weights(shape, 7))
    for k in ("w_qkv", "w_o", "w_gate_up", "w_down"):
        w[k] = np.zeros_like(w[k])
    return w


def _one_token_step(shape, w, x):
    Hkv, hd = shape.n_kv_heads, shape.head_dim
    pool = np.zeros((1, 2, Hkv, 16, hd))
    return L.layer_step(shape.as_dict(), w, pool, [0, 1], [1], [0, 1], [0], x)


def test_zero_weights_give_identity_layer():
    shape = W.TINY
    x = np.random.default_rng(8).standard_normal((1, shape.d_model))
    r = _one_token_step(shape, _zero_layer(shape), x)
    np.testing.assert_array_equal(r["y"], x)


def test_gate_up_order_and_swiglu():
    """Gate pre-activation 30 on feature 0, up 1.5: a_0 = silu(30) * 1.5 and
    the down projection routes a_0 to output 3 on top of the residual."""
    shape = W.TINY
    d, F = shape.d_model, shape.d_ff
    w = _zero_layer(shape)
    w["g_ffn"] = np.ones(d)
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    xn0 = 1.0 / math.sqrt(1.0 / d + shape.rms_eps)   # RMSNorm(x) at index 0
    w["w_gate_up"][0, 0] = 30.0 / xn0       # gate feature 0
    w["w_gate_up"][F + 0, 0] = 1.5 / xn0    # up feature 0
    w["w_down"][3, 0] = 1.0
    r = _one_token_step(shape, w, x)
    expect = 30.0 / (1.0 + math.exp(-30.0)) * 1.5
    assert abs(r["a"][0, 0] - expect) < 1e-9
    assert abs(r["y"][0, 3] - expect) < 1e-9
    np.testing.assert_allclose(np.delete(r["y"][0], 3), np.delete(x[0], 3), atol=1e-15)


def test_single_token_attention_path_is_value_projection():
    """With one key (kv_len = 1), o = v, so h = x + (xn W_v^T) W_o^T for a
    layer whose Q/K rows are random and FFN is zero."""
    shape = W.TINY
    d, hd, Hq, Hkv = shape.d_model, shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    w = L.weights_to_f64(W.make_weights(shape, 9))
    w["w_gate_up"] = np.zeros_like(w["w_gate_up"])
    x = np.random.default_rng(10).standard_normal((1, d))
    r = _one_token_step(shape, w, x)
    xn = x / np.sqrt(np.mean(x * x) + shape.rms_eps) * w["g_attn"]
    v = xn @ w["w_qkv"][(Hq + Hkv) * hd:].T          # [1, Hkv*hd]
    assert Hq == Hkv       # group 1: q head h reads v head h
    np.testing.assert_allclose(r["h"], x + v @ w["w_o"].T, rtol=1e-10, atol=1e-12)


def test_next_tokens_greedy_one_hot_and_ties():
    # LM head rows that are one-hot in d pick the coordinate of the largest
    # normalised activation; duplicated rows tie and the lower id wins
    from oracle.layer import next_tokens_greedy
    rng = np.random.default_rng(4)
    d, vocab = 16, 40
    x = rng.standard_normal((5, d))
    g = np.ones(d)
    W = np.zeros((vocab, d))
    for v in range(d):
        W[v, v] = 1.0
    W[30] = W[3]                    # a duplicate of row 3
    logits, ids = next_tokens_greedy(x, [4, 0, 2], g, W, 1e-6)
    for k, r in enumerate([4, 0, 2]):
        want = int(np.argmax(x[r]))
        assert ids[k] == want
        assert logits[k, 30] == logits[k, 3]
    x2 = np.zeros((1, d))
    x2[0, 3] = 5.0
    _, ids2 = next_tokens_greedy(x2, [0], g, W, 1e-6)
    assert ids2[0] == 3             # tie with row 30: the lower index


def test_ffn_half_reads_only_h():
    """Two inputs with the same attention residual h give the same y.

    With V = I, W_o = -1.5 I and one key per request (o = v), h = x - 1.5
    RMSNorm(x).  For u with rms 1, x = u and x = -2u both give h = -0.5 u, so
    the FFN half (RMSNorm(h), SwiGLU, down, residual h) must return the same
    y for both.  An FFN that normalised x, or added x as its residual, would
    not: the two inputs differ in sign and size."""
    shape = W.TINY.as_dict()
    shape["rms_eps"] = 0.0
    d, Hq, Hkv, hd = shape["d_model"], shape["n_q_heads"], shape["n_kv_heads"], shape["head_dim"]
    assert Hq == Hkv and Hkv * hd == d
    w = L.weights_to_f64(W.make_weights(W.TINY, 11))
    w["g_attn"] = np.ones(d)
    w["w_qkv"][(Hq + Hkv) * hd:] = np.eye(d)
    w["w_o"] = -1.5 * np.eye(d)
    z = np.random.default_rng(12).standard_normal(d)
    u = z / np.sqrt(np.mean(z * z))
    x = np.stack([u, -2.0 * u])
    pool = np.zeros((2, 2, Hkv, 16, hd))
    r = L.layer_step(shape, w, pool, [0, 1, 2], [1, 1], [0, 1, 2], [0, 1], x)
    np.testing.assert_allclose(r["h"], np.stack([-0.5 * u, -0.5 * u]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["y"][0], r["y"][1], rtol=0, atol=1e-12)
    assert np.max(np.abs(r["y"][0] - r["h"][0])) > 1e-3      # the FFN does contribute
    # the miswirings named above would separate the two rows by this much
    def ffn(t):
        gu = L.linear(L.rms_norm(t, w["g_ffn"], 0.0), w["w_gate_up"])
        return L.linear(L.silu(gu[:, :shape["d_ff"]]) * gu[:, shape["d_ff"]:], w["w_down"])
    assert np.max(np.abs(ffn(x[:1]) - ffn(x[1:]))) > 1e-3


def test_qk_norm_is_per_head_and_precedes_rope():
    """Qwen3 q/k-norm: RMSNorm over head_dim with its gains, then RoPE.

    x = e_0 and one-hot rows put sqrt(d) (up to eps) in element 0 of q head 0
    and k head 0 only.  Norm per head gives sqrt(hd) * g[0] there; RoPE at
    position p then moves it onto the pair (0, hd/2) as (cos p, sin p), both
    scaled by g[0].  Rotating first would scale the sin term by g[hd/2];
    normalising over all heads at once would give sqrt(Hq hd) instead."""
    shape = W.SMALL_G5_QKN.as_dict()
    d, Hq, Hkv, hd = shape["d_model"], shape["n_q_heads"], shape["n_kv_heads"], shape["head_dim"]
    eps = shape["rms_eps"]
    w = L.weights_to_f64(W.make_weights(W.SMALL_G5_QKN, 13))
    w["g_attn"] = np.ones(d)
    w["w_qkv"] = np.zeros_like(w["w_qkv"])
    w["w_qkv"][0, 0] = 1.0               # q head 0, element 0
    w["w_qkv"][Hq * hd, 0] = 1.0         # k head 0, element 0
    g_q, g_k = np.ones(hd), np.ones(hd)
    g_q[0], g_q[hd // 2] = 1.5, 0.5
    g_k[0], g_k[hd // 2] = 0.75, 2.0
    w["g_q"], w["g_k"] = g_q, g_k
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    p = 5                                # one decode after 5 cached tokens
    pool = np.zeros((1, 2, Hkv, 16, hd))
    r = L.layer_step(shape, w, pool, [0, 1], [p + 1], [0, 1], [0], x)
    pre = 1.0 / math.sqrt(1.0 / d + eps)                 # element 0 after the input norm
    mag = pre / math.sqrt(pre * pre / hd + eps)          # after the per-head norm
    for got, g in ((r["q"][0, 0], g_q[0]), (pool[0, 0, 0, p], g_k[0])):
        want = np.zeros(hd)
        want[0], want[hd // 2] = g * mag * math.cos(p), g * mag * math.sin(p)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.all(r["q"][0, 1:] == 0) and np.all(pool[0, 0, 1:, p] == 0)
