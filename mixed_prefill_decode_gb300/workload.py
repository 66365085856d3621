"""Seeded synthetic inputs for the mixed prefill+decode layer step.

This module only draws numbers and lays out batch descriptors.  It holds none
of the layer's arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  Every array it returns is plain NumPy: bf16 tensors are returned as
their raw 16-bit patterns (``np.uint16``), integer tables as ``np.int32``.

Shapes and distributions follow the workloads the pages describe:

* weights N(0, 0.02), token embeddings N(0, 1), rounded to bf16;
* 16-token KV pages handed out from a seeded random permutation, so that the
  block tables are scattered over the pool;
* batches of one prefill chunk (qo_len = chunk, kv_len = cached prefix + chunk)
  plus qo_len = 1 decode rows, decodes first (the scheduler on the pofe.ai
  "Chunked prefill" page, "How it works, step by step").
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

PAGE_TOKENS = 16
# Untouched KV slots carry this bf16 pattern (a quiet NaN with a marker
# payload) so that a write to the wrong slot is caught bit-exactly.
KV_SENTINEL = np.uint16(0x7FC1)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); return the bits."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    out = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return out.astype(np.uint16).reshape(a.shape)


# --------------------------------------------------------------------------
# Layer shapes
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LayerShape:
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    rms_eps: float
    rope_theta: float
    qk_norm: int

    @property
    def qkv_dim(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def kv_bytes_per_token(self) -> int:
        # K and V, bf16
        return 2 * self.n_kv_heads * self.head_dim * 2

    def as_dict(self) -> dict:
        return dataclasses.asdict(self)


TINY = LayerShape(d_model=256, n_q_heads=4, n_kv_heads=4, head_dim=64, d_ff=1024,
                  rms_eps=1e-6, rope_theta=1e4, qk_norm=0)
LLAMA3_8B = LayerShape(d_model=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                       d_ff=14336, rms_eps=1e-6, rope_theta=5e5, qk_norm=0)
QWEN3_14B = LayerShape(d_model=5120, n_q_heads=40, n_kv_heads=8, head_dim=128,
                       d_ff=17408, rms_eps=1e-6, rope_theta=1e6, qk_norm=1)
# A small shape with GQA (group 4, odd group 5 variant below) and qk-norm, used
# by tests that need several tiles and ragged tails at oracle-friendly sizes.
SMALL_GQA = LayerShape(d_model=512, n_q_heads=8, n_kv_heads=2, head_dim=128, d_ff=1536,
                       rms_eps=1e-6, rope_theta=5e5, qk_norm=0)
SMALL_G5_QKN = LayerShape(d_model=640, n_q_heads=10, n_kv_heads=2, head_dim=128, d_ff=1280,
                          rms_eps=1e-6, rope_theta=1e6, qk_norm=1)


# --------------------------------------------------------------------------
# Weights
# --------------------------------------------------------------------------

def make_weights(shape: LayerShape, seed: int, unit_gains: bool = False) -> Dict[str, np.ndarray]:
    """Random-init layer weights as bf16 bit patterns.

    Linear weights are row-major [N, K] (y = x W^T):
      w_qkv     [(Hq + 2 Hkv) hd, d]   rows = [Q; K; V]
      w_o       [d, Hq hd]
      w_gate_up [2 F, d]               rows = [gate; up]
      w_down    [d, F]
    Norm gains are 1 + N(0, 0.1) unless ``unit_gains`` (then exactly 1.0).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    d, hd, F = shape.d_model, shape.head_dim, shape.d_ff
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads

    def lin(n, k):
        return f32_to_bf16_bits(rng.standard_normal((n, k), dtype=np.float32) * np.float32(0.02))

    def gain(n):
        if unit_gains:
            return f32_to_bf16_bits(np.ones(n, dtype=np.float32))
        return f32_to_bf16_bits(1.0 + 0.1 * rng.standard_normal(n, dtype=np.float32))

    w = {
        "g_attn": gain(d),
        "w_qkv": lin((Hq + 2 * Hkv) * hd, d),
        "w_o": lin(d, Hq * hd),
        "g_ffn": gain(d),
        "w_gate_up": lin(2 * F, d),
        "w_down": lin(d, F),
    }
    if shape.qk_norm:
        w["g_q"] = gain(hd)
        w["g_k"] = gain(hd)
    return w


def make_embeddings(T: int, d: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return f32_to_bf16_bits(rng.standard_normal((T, d), dtype=np.float32))


# --------------------------------------------------------------------------
# Batch descriptors
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Batch:
    """CSR batch descriptor: request r owns tokens [qo_indptr[r], qo_indptr[r+1])
    of the step, has kv_len[r] keys after this step's append, and its pages are
    bt[bt_indptr[r] : bt_indptr[r+1]]."""
    qo_indptr: np.ndarray
    kv_len: np.ndarray
    bt_indptr: np.ndarray
    bt: np.ndarray

    @property
    def num_reqs(self) -> int:
        return int(self.kv_len.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.qo_indptr[-1])

    def qo_len(self) -> np.ndarray:
        return np.diff(self.qo_indptr)

    def cached(self) -> np.ndarray:
        return self.kv_len - self.qo_len()


def pages_for(n_tokens: int) -> int:
    return (n_tokens + PAGE_TOKENS - 1) // PAGE_TOKENS


def make_batch(reqs: Sequence[Tuple[int, int]], seed: int, spare_pages: int = 8,
               num_pages: Optional[int] = None) -> Tuple[Batch, int]:
    """Lay out a batch for requests given as (cached prefix c, new tokens qo).

    Pages are drawn in request order from a seeded permutation of the pool; the
    pool holds exactly the pages needed plus ``spare_pages`` that nobody owns.
    Returns (batch, num_pages).
    """
    need = [pages_for(c + q) for c, q in reqs]
    total = sum(need)
    if num_pages is None:
        num_pages = total + spare_pages
    if num_pages < total:
        raise ValueError("pool too small")
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(num_pages).astype(np.int32)
    qo_indptr = np.zeros(len(reqs) + 1, np.int32)
    bt_indptr = np.zeros(len(reqs) + 1, np.int32)
    kv_len = np.zeros(len(reqs), np.int32)
    for r, (c, q) in enumerate(reqs):
        if q < 1 or c < 0:
            raise ValueError("each request needs qo >= 1 and c >= 0")
        qo_indptr[r + 1] = qo_indptr[r] + q
        kv_len[r] = c + q
        bt_indptr[r + 1] = bt_indptr[r] + need[r]
    bt = perm[:total].copy()
    return Batch(qo_indptr, kv_len, bt_indptr, bt), num_pages


def make_kv_pool(shape: LayerShape, num_pages: int, batch: Batch, seed: int,
                 fill_all: bool = False) -> np.ndarray:
    """KV pool [P][2][Hkv][16][hd] as bf16 bits.

    Slots holding a request's cached prefix get N(0, 1) values; every other
    slot holds ``KV_SENTINEL``.  With ``fill_all`` every slot gets a value
    (timing runs, where the pool is larger than anything parity touches).
    """
    Hkv, hd = shape.n_kv_heads, shape.head_dim
    pool = np.full((num_pages, 2, Hkv, PAGE_TOKENS, hd), KV_SENTINEL, dtype=np.uint16)
    rng = np.random.Generator(np.random.PCG64(seed))
    if fill_all:
        pool[...] = f32_to_bf16_bits(rng.standard_normal(pool.shape, dtype=np.float32))
        return pool
    cached = batch.cached()
    for r in range(batch.num_reqs):
        c = int(cached[r])
        if c == 0:
            continue
        pages = batch.bt[batch.bt_indptr[r]:batch.bt_indptr[r + 1]]
        vals = f32_to_bf16_bits(rng.standard_normal((c, 2, Hkv, hd), dtype=np.float32))
        for p in range(c):
            pool[pages[p // PAGE_TOKENS], :, :, p % PAGE_TOKENS, :] = vals[p]
    return pool


# --------------------------------------------------------------------------
# The pages' workloads, at the sizes they state
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    shape: LayerShape
    reqs: List[Tuple[int, int]]   # (cached c, qo) per request, decodes first
    seed: int


def tiny_mixed(seed: int = 1000) -> Workload:
    """d_model 256 layer: one 64-token chunk on a 64-token prefix plus four
    decodes with contexts U[128, 256]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    dec = [(int(c), 1) for c in rng.integers(128, 256, size=4, endpoint=True)]
    return Workload("tiny_mixed_T68", TINY, dec + [(64, 64)], seed)


def llama3_8b_mixed(seed: int = 2000) -> Workload:
    """Llama-3-8B-shaped layer: 64 decodes at 1,125-token contexts plus one
    512-token chunk whose cached prefix is U[0, 4096]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    c = int(rng.integers(0, 4096, endpoint=True))
    return Workload("llama3_8b_mixed_T576", LLAMA3_8B, [(1125, 1)] * 64 + [(c, 512)], seed)


def qwen3_14b_mixed(prefill_tokens: int, seed: int = 3000) -> Workload:
    """Qwen3-14B-shaped layer: 16 decodes at 8,192-token contexts plus
    ``prefill_tokens`` (0, 1024 or 2200) piggybacked tokens of one prompt,
    prefix 0."""
    reqs = [(8192, 1)] * 16
    if prefill_tokens:
        reqs.append((0, prefill_tokens))
    return Workload(f"qwen3_14b_mixed_P{prefill_tokens}", QWEN3_14B, reqs,
                    seed + {0: 0, 1024: 1, 2200: 2}.get(prefill_tokens, 9))


def small_mixed(shape: LayerShape, seed: int, n_dec: int = 5, chunk: int = 200,
                prefix: int = 77) -> Workload:
    """Oracle-sized mixed batch with ragged tails everywhere: decodes at odd
    contexts, one chunk that spans several 128-row tiles."""
    rng = np.random.Generator(np.random.PCG64(seed))
    dec = [(int(c), 1) for c in rng.integers(1, 700, size=n_dec, endpoint=True)]
    reqs = dec + ([(prefix, chunk)] if chunk else [])
    return Workload(f"small_mixed_{shape.d_model}", shape, reqs, seed)


def materialize(w: Workload, unit_gains: bool = False, fill_all_kv: bool = False,
                spare_pages: int = 8):
    """All arrays for one workload: weights, x, batch, pool."""
    weights = make_weights(w.shape, w.seed + 1, unit_gains=unit_gains)
    batch, num_pages = make_batch(w.reqs, w.seed + 2, spare_pages=spare_pages)
    x = make_embeddings(batch.num_tokens, w.shape.d_model, w.seed + 3)
    pool = make_kv_pool(w.shape, num_pages, batch, w.seed + 4, fill_all=fill_all_kv)
    return weights, x, batch, pool


# --------------------------------------------------------------------------
# Stacks (many layers): generated on the device with torch's seeded CUDA
# generator, since tens of GB of random weights would take minutes on the
# host.  Returned as torch bf16 tensors; a test copies back the layers the
# oracle checks.
# --------------------------------------------------------------------------

def qwen3_14b_stack(prefix: int = 30720, seed: int = 4000, n_decodes: int = 96):
    """40-layer Qwen3-14B-shaped stack: one 2,048-token chunk after `prefix`
    cached tokens of a 32,768-token prompt, plus decodes with contexts
    log-uniform in [1024, 8192]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.exp(rng.uniform(np.log(1024), np.log(8192), size=n_decodes)).astype(np.int64)
    reqs = [(int(c), 1) for c in ctx] + [(prefix, 2048)]
    return Workload(f"qwen3_14b_stack40_P{prefix}", QWEN3_14B, reqs, seed + prefix), 40


@dataclasses.dataclass
class PromptSweep:
    """A long prompt fed through an n_layers stack as fixed-size chunks, one
    chunk per step, beside running decodes (pofe.ai "Chunked prefill": the
    scheduler gives a partial prompt the budget left after the decodes; the
    prompt's prefix grows by one chunk per step).  The decodes' positions are
    held from step to step (each rewrites its own slot), which leaves every
    step's work unchanged.  ``layout`` places the whole prompt's pages once;
    ``batch_at(k)`` is step k's descriptor: the decodes, then chunk k of the
    prompt (qo = chunk, kv = (k + 1) chunk) reading the first pages of the
    prompt's table."""
    name: str
    shape: LayerShape
    n_layers: int
    decodes: List[int]     # cached context of each decode
    prompt: int
    chunk: int
    seed: int

    @property
    def steps(self) -> int:
        return -(-self.prompt // self.chunk)

    def layout(self, spare_pages: int = 4) -> Tuple[Batch, int]:
        reqs = [(c, 1) for c in self.decodes] + [(0, self.prompt)]
        return make_batch(reqs, self.seed + 1, spare_pages=spare_pages)

    def batch_at(self, k: int, full: Batch, with_decodes: bool = True, with_chunk: bool = True) -> Batch:
        n_dec = len(self.decodes)
        rows = []
        if with_decodes:
            for r in range(n_dec):
                kv = self.decodes[r] + 1
                rows.append((1, kv, full.bt[full.bt_indptr[r]:full.bt_indptr[r] + pages_for(kv)]))
        if with_chunk:
            q0 = k * self.chunk
            qo = min(self.chunk, self.prompt - q0)
            kv = q0 + qo
            rows.append((qo, kv, full.bt[full.bt_indptr[n_dec]:full.bt_indptr[n_dec] + pages_for(kv)]))
        qo_indptr = np.cumsum([0] + [r[0] for r in rows]).astype(np.int32)
        kv_len = np.array([r[1] for r in rows], dtype=np.int32)
        bt_indptr = np.cumsum([0] + [len(r[2]) for r in rows]).astype(np.int32)
        bt = np.concatenate([r[2] for r in rows]).astype(np.int32)
        return Batch(qo_indptr, kv_len, bt_indptr, bt)


def qwen3_14b_prompt_sweep(seed: int = 4000, n_decodes: int = 96, prompt: int = 32768, chunk: int = 2048):
    """The 40-layer Qwen3-14B-shaped stack over a whole 32,768-token prompt fed
    as 2,048-token chunks (prefix 0, 2,048, ..., 30,720) beside 96 decodes
    with contexts log-uniform in [1024, 8192] (the same decodes as
    qwen3_14b_stack)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.exp(rng.uniform(np.log(1024), np.log(8192), size=n_decodes)).astype(np.int64)
    return PromptSweep(f"qwen3_14b_stack40_prompt{prompt}", QWEN3_14B, 40, [int(c) for c in ctx], prompt, chunk,
                       seed + 77)


def llama3_8b_stack(budget: int, n_decodes: int, seed: int = 5000):
    """32-layer Llama-3-8B-shaped stack for the token-budget sweep: n_decodes
    decodes with contexts log-uniform in [512, 32768] and one prefill chunk of
    budget - n_decodes tokens with a prefix uniform in [0, 16384] (no chunk if
    the decodes use the whole budget)."""
    rng = np.random.Generator(np.random.PCG64(seed + 31 * budget + n_decodes))
    ctx = np.exp(rng.uniform(np.log(512), np.log(32768), size=n_decodes)).astype(np.int64)
    reqs = [(int(c), 1) for c in ctx]
    if budget > n_decodes:
        reqs.append((int(rng.integers(0, 16384, endpoint=True)), budget - n_decodes))
    return Workload(f"llama3_8b_stack32_C{budget}_b{n_decodes}", LLAMA3_8B, reqs,
                    seed + 31 * budget + n_decodes), 32


def device_weights(shape: LayerShape, seed: int, device="cuda", unit_gains: bool = True):
    """Random-init layer weights drawn on the device (torch, seeded): linear
    weights N(0, 0.02), gains 1 (or 1 + N(0, 0.1)); bf16 tensors with the
    layouts of make_weights."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    d, hd, F = shape.d_model, shape.head_dim, shape.d_ff
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads

    def lin(n, k):
        return (torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)

    def gain(n):
        if unit_gains:
            return torch.ones(n, device=device, dtype=torch.bfloat16)
        return (1 + 0.1 * torch.randn(n, generator=g, device=device, dtype=torch.float32)).to(torch.bfloat16)

    w = {"g_attn": gain(d), "w_qkv": lin((Hq + 2 * Hkv) * hd, d), "w_o": lin(d, Hq * hd), "g_ffn": gain(d),
         "w_gate_up": lin(2 * F, d), "w_down": lin(d, F)}
    if shape.qk_norm:
        w["g_q"] = gain(hd)
        w["g_k"] = gain(hd)
    return w


def device_kv_pool(shape: LayerShape, num_pages: int, seed: int, device="cuda"):
    """A KV pool [P][2][Hkv][16][hd] bf16 filled with N(0, 1), on the device."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((num_pages, 2, shape.n_kv_heads, PAGE_TOKENS, shape.head_dim), generator=g,
                       device=device, dtype=torch.float32).to(torch.bfloat16)
