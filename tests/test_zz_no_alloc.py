"""The allocation-free GEMM entry point (mb_gemm_noalloc), for callers that
cannot allocate device memory: code running inside an allocator's hooks or
out-of-memory path, processes whose device memory is all handed out up front,
plugins limited to the buffers their host passes in.  Its scratch is a static
device array instead of a workspace.

Checked through the C ABI on two calls in a row (the second call reuses the
scratch the first one left behind), each followed by mb_device_status(NULL),
which reads the array's error word without allocating:

* against the oracle's linear layer (and its SwiGLU), within the tolerance of
  the other GPU tests;
* against the regular entry point (mb_gemm) on the same inputs;
* a split wait made to run out is reported as MB_EDEVICE by the next
  mb_device_status(NULL) even after a later call, and the call after that is
  correct again.

This file is collected last so that a run stopping at the first failure has
already run every other test."""

import numpy as np
import pytest
import torch

from oracle import layer as OL
from mixed_prefill_decode_gb300 import workload as W
from gpu_util import to_dev, from_dev, assert_close, f64

pytestmark = pytest.mark.gpu

CASES = [
    # M, N, K, epilogue: split shapes (fewer tiles than SMs) and an unsplit one
    (576, 4096, 4096, 1),
    (68, 768, 256, 0),
    (200, 1536, 512, 2),
    (1040, 5120, 5120, 0),
]


def _inputs(M, N, K, epi):
    rng = np.random.default_rng(M + N + K + epi)
    nb = 2 * N if epi == 2 else N
    A = W.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    B = W.f32_to_bf16_bits(rng.standard_normal((nb, K), dtype=np.float32) * np.float32(0.02))
    R = W.f32_to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if epi == 1 else None
    return A, B, R


def _oracle(A, B, R, N, epi):
    y = OL.linear(f64(A), f64(B))
    if epi == 2:
        return OL.silu(y[:, :N]) * y[:, N:]
    return y + (f64(R) if epi == 1 else 0.0)


@pytest.mark.parametrize("M,N,K,epi", CASES)
def test_noalloc_gemm_matches_oracle_and_regular_entry_point(mb, M, N, K, epi):
    A, B, R = _inputs(M, N, K, epi)
    dA, dB = to_dev(A), to_dev(B)
    dR = to_dev(R) if R is not None else None
    s = torch.cuda.current_stream().cuda_stream
    want = _oracle(A, B, R, N, epi)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mb.mb_gemm(dA, dB, ref, dR, M, N, K, epi, None, s)
    mb.mb_device_status(None, s)
    regular = f64(from_dev(ref))
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        mb.mb_gemm_noalloc(dA, dB, out, dR, M, N, K, epi, s)
        mb.mb_device_status(None, s)
        got = f64(from_dev(out))
        assert_close(f"noalloc call {call} {M}x{N}x{K} epi {epi} vs oracle", got, want)
        assert_close(f"noalloc call {call} {M}x{N}x{K} epi {epi} vs mb_gemm", got, regular)


def test_noalloc_gemm_reports_a_wait_that_ran_out(mb):
    """A split wait that runs out (the head piece also waits for a piece that
    no CTA writes, 1 ms limit) leaves its code in the static array; a second
    call does not clear it; mb_device_status(NULL) reports MB_EDEVICE once and
    resets the tickets; the next call is correct with a clean status."""
    M, N, K, epi = 576, 4096, 4096, 1
    A, B, R = _inputs(M, N, K, epi)
    dA, dB, dR = to_dev(A), to_dev(B), to_dev(R)
    s = torch.cuda.current_stream().cuda_stream
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mb.mb_gemm_set_split_wait(1_000_000, 1)
    try:
        mb.mb_gemm_noalloc(dA, dB, out, dR, M, N, K, epi, s)
    finally:
        mb.mb_gemm_set_split_wait(0, 0)
    mb.mb_gemm_noalloc(dA, dB, out, dR, M, N, K, epi, s)   # a clean call after the failed one
    with pytest.raises(mb.MbError) as e:
        mb.mb_device_status(None, s)
    assert e.value.status == mb.MB_EDEVICE
    mb.mb_device_status(None, s)   # reported once, then clear
    out.fill_(float("nan"))
    mb.mb_gemm_noalloc(dA, dB, out, dR, M, N, K, epi, s)
    mb.mb_device_status(None, s)
    assert_close("noalloc after a reported error", f64(from_dev(out)), _oracle(A, B, R, N, epi))


def test_noalloc_gemm_rejects_bad_arguments(mb):
    with pytest.raises(mb.MbError):
        mb.mb_gemm_noalloc(16, 16, 16, None, 128, 128, 60, 0)
