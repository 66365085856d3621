"""Oracle for one transformer-layer step over a mixed prefill+decode batch.

TEST INFRASTRUCTURE ONLY (see the package docstring): plain, slow, float64.

What it computes (one pre-norm decoder layer, no biases; the pages never write
the block out, so this is the plainest reading of a Llama-3 / Qwen3 layer):

    xn   = RMSNorm(x) * g_attn
    qkv  = xn W_qkv^T ;  q, k, v = split(qkv)            (rows of W_qkv: Q; K; V)
    q, k = RMSNorm_hd(q) * g_q, RMSNorm_hd(k) * g_k      (Qwen3 only)
    q, k = RoPE(q, pos), RoPE(k, pos),  pos = c_r + i
    append k, v of every new token to its page / slot    (append, then attend)
    o    = softmax(q K^T / sqrt(hd) + causal mask) V      per request and head
    h    = x + o W_o^T
    hn   = RMSNorm(h) * g_ffn
    a    = silu(hn W_gate^T) * (hn W_up^T)                (rows of W_gate_up: gate; up)
    y    = h + a W_down^T

Sources:
  * chunk attention mask, scale and GQA mapping: llm-stack-book 7.8 "Attention
    on Partial KV Caches" (query at position T_past + i sees keys 0..T_past + i)
    and its exercise 5 (GQA by repeat_interleave, so KV head = q_head // group);
  * qo_len / kv_len framing of a mixed batch: Perplexity "Disaggregated Prefill
    and Decode", section "Prefill versus Decode-prestaties";
  * append-then-attend inside one pass: pofe.ai "Chunked prefill", "How it
    works, step by step", step 4;
  * HND page layout [page][K/V][head][slot][hd]: Perplexity page, section
    "Gesharcde KV Cache Transfers";
  * KV tensor geometry [L, 2, T, n_kv_heads, d_head]: llm-stack-book 7.8,
    KV-cache size discussion.

Storage: every intermediate is float64; bf16 inputs are decoded exactly.  No
intermediate rounding (the CUDA path rounds to bf16 between kernels; the
acceptance tolerance absorbs that).
"""

from __future__ import annotations

import math
from typing import Dict

import numpy as np

PAGE_TOKENS = 16


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Building blocks
# --------------------------------------------------------------------------

def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis.  The pages name the
    Llama-3 / Qwen3 layers without writing their norm out; this is RMSNorm
    as published (Zhang and Sennrich, "Root Mean Square Layer
    Normalization", 2019), with the gain applied after the scaling."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T with W stored row-major [N, K].  Every token of the mixed
    batch, prefill or decode, is one row of the same product: a linear layer
    applies the same weights to every token (ConfluxServe, "Why can linear
    layers be batched but attention cannot?"; pofe.ai, "The bottleneck:
    prefill-decode interference": the decodes are extra rows of the prefill's
    matrix multiply)."""
    return x @ w.T


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x), the gate of the SwiGLU feed-forward block of Llama-3 /
    Qwen3 layers (Shazeer, "GLU Variants Improve Transformer", 2020); the
    pages name the block without writing it out."""
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE: element i pairs with i + hd/2, frequency
    theta^(-2i/hd), angle pos * frequency.  ``x`` is [..., hd]; ``pos``
    broadcasts against x.shape[:-1].  The pages give only the position a
    chunk's token takes (llm-stack-book 7.8, "Attention on Partial KV
    Caches": query i of a chunk sits at T_past + i); the rotation is the
    rotary embedding as published (Su et al., "RoFormer", 2021) in the
    half-split pairing of Llama-3 / Qwen3 layers."""
    hd = x.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / hd)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def page_slot(block_table: np.ndarray, p: int):
    """Token p of a request lives in page block_table[p // 16], slot p % 16:
    the paged KV cache indexed through a per-request block table
    (llm-stack-book 7.8, "Attention on Partial KV Caches"; pofe.ai, "How it
    works, step by step": the chunk's keys are read partly from the paged
    cache), with 16-token pages."""
    return int(block_table[p // PAGE_TOKENS]), p % PAGE_TOKENS


def gather_kv(pool: np.ndarray, block_table: np.ndarray, n: int):
    """Keys and values 0..n-1 of one request, read through its block table.
    pool is [P][2][Hkv][16][hd] (heads before slots, the HND order of the
    Perplexity page, "Gesharcde KV Cache Transfers"); returns K, V as
    [n, Hkv, hd]."""
    p = np.arange(n)
    pages = block_table[p // PAGE_TOKENS]
    slots = p % PAGE_TOKENS
    K = pool[pages, 0, :, slots, :]
    V = pool[pages, 1, :, slots, :]
    return K, V


def attention_request(q: np.ndarray, K: np.ndarray, V: np.ndarray, cached: int) -> np.ndarray:
    """Masked softmax attention for one request.

    q: [qo, Hq, hd] queries at positions cached + i;  K, V: [kv, Hkv, hd] with
    kv = cached + qo.  Query row i sees keys j <= cached + i.  Scale 1/sqrt(hd).
    GQA: q head h reads KV head h // (Hq / Hkv).  Follows llm-stack-book 7.8,
    "Attention on Partial KV Caches" (the mask over the cached prefix plus the
    chunk, and the scale) and its exercise 5 (GQA by repeating each KV head
    over its group); a decode row is the case qo = 1 (Perplexity page,
    "Prefill versus Decode-prestaties": qo_len 1 against a long kv_len).
    """
    qo, Hq, hd = q.shape
    kv, Hkv, _ = K.shape
    group = Hq // Hkv
    q_pos = cached + np.arange(qo)
    k_pos = np.arange(kv)
    allowed = k_pos[None, :] <= q_pos[:, None]          # [qo, kv]
    scale = 1.0 / math.sqrt(hd)
    out = np.empty((qo, Hq, hd))
    for h in range(Hq):
        hk = h // group
        s = (q[:, h, :] @ K[:, hk, :].T) * scale         # [qo, kv]
        s = np.where(allowed, s, -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        p = e / np.sum(e, axis=1, keepdims=True)
        out[:, h, :] = p @ V[:, hk, :]
    return out


# --------------------------------------------------------------------------
# The layer step
# --------------------------------------------------------------------------

def layer_step(shape: Dict, w: Dict[str, np.ndarray], pool: np.ndarray, qo_indptr, kv_len,
               bt_indptr, bt, x: np.ndarray) -> Dict[str, np.ndarray]:
    """One layer over a mixed batch.

    shape: d_model, n_q_heads, n_kv_heads, head_dim, d_ff, rms_eps, rope_theta,
           qk_norm.
    w:     float64 weights (see module docstring for layouts).
    pool:  float64 KV pool [P][2][Hkv][16][hd]; this step's K/V are written
           into it (in place) before attention.
    x:     float64 [T, d].
    Returns the intermediates and the output y, plus ``written``: the (page,
    slot) of every appended token in token order.
    """
    d = shape["d_model"]
    Hq, Hkv, hd = shape["n_q_heads"], shape["n_kv_heads"], shape["head_dim"]
    F = shape["d_ff"]
    eps = shape["rms_eps"]
    qo_indptr = np.asarray(qo_indptr)
    kv_len = np.asarray(kv_len)
    bt_indptr = np.asarray(bt_indptr)
    bt = np.asarray(bt)
    T = int(qo_indptr[-1])
    n_req = kv_len.shape[0]
    assert x.shape == (T, d)

    xn = rms_norm(x, w["g_attn"], eps)
    qkv = linear(xn, w["w_qkv"])
    q = qkv[:, : Hq * hd].reshape(T, Hq, hd)
    k = qkv[:, Hq * hd: (Hq + Hkv) * hd].reshape(T, Hkv, hd)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(T, Hkv, hd)
    if shape["qk_norm"]:
        q = rms_norm(q, w["g_q"], eps)
        k = rms_norm(k, w["g_k"], eps)

    pos = np.empty(T, dtype=np.int64)
    for r in range(n_req):
        t0, t1 = int(qo_indptr[r]), int(qo_indptr[r + 1])
        c = int(kv_len[r]) - (t1 - t0)
        pos[t0:t1] = c + np.arange(t1 - t0)
    q = rope(q, pos[:, None], shape["rope_theta"])
    k = rope(k, pos[:, None], shape["rope_theta"])

    # append this step's keys and values, then attend
    written = np.empty((T, 2), dtype=np.int64)
    for r in range(n_req):
        t0, t1 = int(qo_indptr[r]), int(qo_indptr[r + 1])
        table = bt[bt_indptr[r]:bt_indptr[r + 1]]
        for t in range(t0, t1):
            page, slot = page_slot(table, int(pos[t]))
            pool[page, 0, :, slot, :] = k[t]
            pool[page, 1, :, slot, :] = v[t]
            written[t] = (page, slot)

    o = np.empty((T, Hq, hd))
    for r in range(n_req):
        t0, t1 = int(qo_indptr[r]), int(qo_indptr[r + 1])
        table = bt[bt_indptr[r]:bt_indptr[r + 1]]
        n = int(kv_len[r])
        K, V = gather_kv(pool, table, n)
        o[t0:t1] = attention_request(q[t0:t1], K, V, n - (t1 - t0))
    o = o.reshape(T, Hq * hd)

    h = x + linear(o, w["w_o"])
    hn = rms_norm(h, w["g_ffn"], eps)
    gu = linear(hn, w["w_gate_up"])
    a = silu(gu[:, :F]) * gu[:, F:]
    y = h + linear(a, w["w_down"])
    return {"xn": xn, "qkv": qkv, "q": q, "k": k, "v": v, "o": o, "h": h, "hn": hn,
            "a": a, "y": y, "pos": pos, "written": written}


def weights_to_f64(w: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    return {kk: bf16_bits_to_f64(vv) for kk, vv in w.items()}


def next_tokens_greedy(x: np.ndarray, rows, g_final: np.ndarray, w_lm: np.ndarray, eps: float):
    """The tokens a pass samples (pofe.ai "Chunked prefill", "How it works,
    step by step", step 5: each decode row and the last row of a prompt whose
    last chunk ran sample in the same pass).  The pages leave the rule open;
    the greedy one: logits = RMSNorm(x[rows]) g_final W_lm^T, token = the
    argmax, the lowest index among equal maxima (NumPy's argmax returns the
    first).  Returns (logits float64 [n, vocab], ids int64 [n])."""
    y = rms_norm(np.asarray(x, dtype=np.float64)[np.asarray(rows, dtype=np.int64)], g_final, eps)
    logits = linear(y, w_lm)
    return logits, np.argmax(logits, axis=1)
