"""The allocation-free GEMM entry point (mb_gemm_noalloc), for callers that
cannot allocate device memory: code running inside an allocator's hooks or
out-of-memory path, processes whose device memory is all handed out up front,
plugins limited to the buffers their host passes in.  Its scratch is a static
device array instead of a workspace.

Checked through the C ABI against the regular entry point (mb_gemm) on the
same inputs, within the tolerance of the other GPU tests, on two calls in a
row (the second call reuses the scratch the first one left behind).  This file
is collected last so that a run stopping at the first failure has already
run every other test."""

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("M,N,K,epi", CASES)
def test_noalloc_gemm_matches_regular_entry_point(mb, M, N, K, epi):
    rng = np.random.default_rng(M + N + K + epi)
    nb = 2 * N if epi == 2 else N
    A = to_dev(W.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32)))
    B = to_dev(W.f32_to_bf16_bits(rng.standard_normal((nb, K), dtype=np.float32) * np.float32(0.02)))
    R = to_dev(W.f32_to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32))) if epi == 1 else None
    s = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    mb.mb_gemm(A, B, ref, R, M, N, K, epi, None, s)
    mb.mb_device_status(None, s)
    want = f64(from_dev(ref))
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        mb.mb_gemm_noalloc(A, B, out, R, M, N, K, epi, s)
        torch.cuda.synchronize()
        assert_close(f"noalloc call {call} {M}x{N}x{K} epi {epi}", f64(from_dev(out)), want)


def test_noalloc_gemm_rejects_bad_arguments(mb):
    with pytest.raises(mb.MbError):
        mb.mb_gemm_noalloc(16, 16, 16, None, 128, 128, 60, 0)
