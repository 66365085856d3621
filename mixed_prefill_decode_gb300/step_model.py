"""Roofline step-time model of one serving iteration.

Host-side analytic model: ``bench.py`` reports it beside the measured step,
and ``budget.py`` can drive its load test with it (the page's own simulator
ran on it).  It holds none of the layer's arithmetic.

The pofe.ai "Chunked prefill" page ("The bottleneck: prefill-decode
interference" and "What chunking costs") models an iteration of P prompt tokens
and D decode tokens on an N-parameter 16-bit model with achievable bandwidth
B_W and compute F; its display formulas did not survive extraction.  The
reading below reproduces every number the page prints from the model (ridge
~221 tokens; 10.0 ms for 64 decodes at 1,125 tokens; 118 ms for a 4,096-token
prefill; 251 / 427 ms and +6.2 / 3.0 / 0.6 % for an 8,192-token prompt in one
shot / 128 / 256 / 512 / 2,048-token chunks; 16.2 -> 17.8 ms and 136 ms for the
worked example; 1.88 GB and 0.70 ms of repeated KV reads):

    T     = max(FLOPs / F, bytes / B_W) + t_iter
    FLOPs = 2 N (P + D) + 4 d L * pairs
    bytes = 2 N + kappa * (KV tokens read)

where a chunk of P tokens after a cached prefix c contributes
pairs = P c + P (P + 1) / 2 and reads c cached tokens, and a decode at context
c contributes c + 1 pairs and reads c + 1 tokens.  t_iter = 0.5 ms is the
per-iteration constant that the printed decode and mixed-iteration numbers
need (the page does not name it).
"""

from __future__ import annotations

import dataclasses
from typing import Iterable, Sequence, Tuple


@dataclasses.dataclass(frozen=True)
class Machine:
    flops: float        # achievable FLOP/s
    bandwidth: float    # achievable bytes/s
    t_iter: float = 0.5e-3


@dataclasses.dataclass(frozen=True)
class Model:
    n_params: float
    kappa: float        # KV bytes per token over all layers
    d_model: int
    n_layers: int


# The page's assumptions: 60 % of 989 TFLOP/s and 80 % of 3.35 TB/s, an 8B
# model with the Llama-3.1-8B KV geometry (kappa = 131,072 B/token).
H100_CLASS = Machine(flops=0.6 * 989e12, bandwidth=0.8 * 3.35e12)
LLAMA_8B = Model(n_params=8e9, kappa=131072.0, d_model=4096, n_layers=32)


def ridge_tokens(m: Machine) -> float:
    """P* = F / B_W: tokens per iteration at which weight reads and weight
    FLOPs take equal time (2N FLOPs and 2N bytes per token)."""
    return m.flops / m.bandwidth


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K and V for every layer: 2 * L * Hkv * hd * bytes."""
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes


def iteration_time(machine: Machine, model: Model, chunks: Sequence[Tuple[int, int]],
                   decode_ctx: Iterable[int]) -> float:
    """Seconds for one iteration with prefill ``chunks`` = [(P, cached c)] and
    decodes at contexts ``decode_ctx``."""
    decode_ctx = list(decode_ctx)
    tokens = sum(p for p, _ in chunks) + len(decode_ctx)
    pairs = sum(p * c + p * (p + 1) / 2 for p, c in chunks) + sum(c + 1 for c in decode_ctx)
    kv_read = sum(c for _, c in chunks) + sum(c + 1 for c in decode_ctx)
    flops = 2 * model.n_params * tokens + 4 * model.d_model * model.n_layers * pairs
    nbytes = 2 * model.n_params + model.kappa * kv_read
    return max(flops / machine.flops, nbytes / machine.bandwidth) + machine.t_iter


def iteration_time_pessimistic(machine: Machine, model: Model, chunks: Sequence[Tuple[int, int]],
                               decode_ctx: Iterable[int]) -> float:
    """The page's second model ("Simulated numbers: choosing the budget"):
    decode attention runs after the matrix multiplies and adds its full
    memory time instead of overlapping, i.e. the decodes' KV bytes leave the
    max() and are added on:  max(FLOPs / F, (2 N + kappa * chunk KV) / B_W)
    + kappa * decode KV / B_W + t_iter."""
    decode_ctx = list(decode_ctx)
    tokens = sum(p for p, _ in chunks) + len(decode_ctx)
    pairs = sum(p * c + p * (p + 1) / 2 for p, c in chunks) + sum(c + 1 for c in decode_ctx)
    kv_chunk = sum(c for _, c in chunks)
    kv_decode = sum(c + 1 for c in decode_ctx)
    flops = 2 * model.n_params * tokens + 4 * model.d_model * model.n_layers * pairs
    overlapped = max(flops / machine.flops, (2 * model.n_params + model.kappa * kv_chunk) / machine.bandwidth)
    return overlapped + model.kappa * kv_decode / machine.bandwidth + machine.t_iter


def chunked_prompt_time(machine: Machine, model: Model, prompt: int, chunk: int) -> float:
    """A prompt alone, processed in ``chunk``-token pieces."""
    t, c = 0.0, 0
    while c < prompt:
        p = min(chunk, prompt - c)
        t += iteration_time(machine, model, [(p, c)], [])
        c += p
    return t


def repeated_kv_bytes(model: Model, prompt: int, chunk: int) -> float:
    """Extra KV traffic from chunking: chunk k re-reads the k*c cached tokens,
    kappa * c * sum_k k = kappa * c * n (n - 1) / 2 with n = prompt / chunk."""
    n = prompt // chunk
    return model.kappa * chunk * n * (n - 1) / 2


def layer_flops(shape: dict, tokens: int) -> float:
    """Linear-layer FLOPs of one layer step: 2 T sum(N K) over QKV, O, gate/up
    and down."""
    d, hd, F = shape["d_model"], shape["head_dim"], shape["d_ff"]
    Hq, Hkv = shape["n_q_heads"], shape["n_kv_heads"]
    nk = (Hq + 2 * Hkv) * hd * d + d * Hq * hd + 2 * F * d + d * F
    return 2.0 * tokens * nk
