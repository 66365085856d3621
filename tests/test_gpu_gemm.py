"""GPU parity of the token-batched tcgen05 GEMM (all three epilogues) against
the oracle's float64 linear layer, over shapes that span several tiles, ragged
M tails, stream-K splits and the layer shapes of the pages' workloads, in both
tile configurations (128-row tiles per CTA; 256-row tiles over CTA pairs)."""

import numpy as np
import pytest
import torch

from oracle import layer as OL
from mixed_prefill_decode_gb300 import workload as W
from gpu_util import to_dev, from_dev, assert_close, f64

pytestmark = pytest.mark.gpu

SHAPES = [
    # M, N, K
    (1, 256, 64), (68, 768, 256), (68, 256, 1024), (129, 640, 512), (200, 1536, 512),
    (300, 512, 1536), (576, 6144, 4096), (576, 4096, 4096), (16, 7168, 5120), (1040, 5120, 5120),
    (2216, 512, 128),
    # 256-row tiles over CTA pairs (from 1,024 tokens on): last pair tiles whose
    # second CTA has no rows (1100, 1300, 2144, 4100), grouped, split and
    # data-parallel schedules
    (1100, 1536, 512), (1300, 768, 1024), (2144, 2560, 2048), (4100, 512, 256),
    # pairs below 1,024 tokens (M mod 256 > 128): the second CTA of the last pair
    # tile holds 16, 60 and 104 rows
    (400, 768, 512), (700, 1536, 1024), (1000, 512, 256),
    # grouped schedule with every N-tile split along K (the down projection at
    # 576 tokens: 224 K steps over two groups)
    (576, 4096, 14336),
    # at least 192 K steps: stream-K covers only the last partial wave of pair
    # tiles (2144 x 5120: 180 tiles, two whole waves on 76 pairs); 1100 x 512
    # (five M-tiles) takes the grouped schedule, its N-tiles split along K
    (1100, 512, 12288), (2144, 5120, 12288),
    # at most 32 rows with split tiles: the head stages every piece at once
    # (7 rows: 18 pieces a round; 32 rows: 4) and sums them before TMEM
    (7, 5120, 17408), (25, 1536, 4096), (32, 4096, 14336),
]


def _inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = W.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    B = W.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    R = W.f32_to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    return A, B, R


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("epi", [0, 1])
def test_gemm_store_and_residual(mb, M, N, K, epi):
    A, B, R = _inputs(M, N, K, M * 7 + N + K + epi)
    dA, dB, dR = to_dev(A), to_dev(B), to_dev(R)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for rep in range(2):   # twice: stream-K tickets must reset themselves
        dD.fill_(float("nan"))
        mb.mb_gemm(dA, dB, dD, dR if epi == 1 else None, M, N, K, epi, None, torch.cuda.current_stream().cuda_stream)
        mb.mb_device_status(None, torch.cuda.current_stream().cuda_stream)
        ref = OL.linear(f64(A), f64(B)) + (f64(R) if epi == 1 else 0.0)
        assert_close(f"gemm{epi} {M}x{N}x{K}", f64(from_dev(dD)), ref)


@pytest.mark.parametrize("M,F,K", [(68, 1024, 256), (200, 1536, 512), (576, 14336, 4096), (16, 17408, 5120),
                                   (130, 128, 64), (1040, 1024, 512), (2216, 2048, 1024),
                                   (700, 1024, 512), (1030, 256, 12288), (20, 2048, 8192)])
def test_gemm_swiglu(mb, M, F, K):
    A, B, _ = _inputs(M, 2 * F, K, M + F + K)
    dA, dB = to_dev(A), to_dev(B)
    dD = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    dD.fill_(float("nan"))
    mb.mb_gemm(dA, dB, dD, None, M, F, K, 2, None, torch.cuda.current_stream().cuda_stream)
    mb.mb_device_status(None, torch.cuda.current_stream().cuda_stream)
    gu = OL.linear(f64(A), f64(B))
    ref = OL.silu(gu[:, :F]) * gu[:, F:]
    assert_close(f"swiglu {M}x{F}x{K}", f64(from_dev(dD)), ref)


def test_gemm_rejects_bad_shapes(mb):
    with pytest.raises(mb.MbError):
        mb.mb_gemm(16, 16, 16, None, 128, 128, 60, 0)      # K % 64
    with pytest.raises(mb.MbError):
        mb.mb_gemm(16, 16, 16, None, 128, 100, 64, 2)      # F % 128


def test_split_wait_expiry_reports_and_recovers(mb):
    """The bounded wait of a K-split tile's head piece, made to run out (it
    also waits for a piece that no CTA writes, with a 1 ms limit): the kernel
    unwinds instead of hanging, mb_device_status reports MB_EDEVICE and resets
    the tile tickets, and the GEMMs after it are correct with a clean status.
    The down projection at 576 tokens splits every N-tile along K."""
    M, N, K = 576, 4096, 14336
    A, B, R = _inputs(M, N, K, 4242)
    dA, dB, dR = to_dev(A), to_dev(B), to_dev(R)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    ref = OL.linear(f64(A), f64(B)) + f64(R)
    mb.mb_gemm_set_split_wait(1_000_000, 1)
    try:
        for rep in range(2):
            mb.mb_gemm(dA, dB, dD, dR, M, N, K, 1, None, s)
            with pytest.raises(mb.MbError) as e:
                mb.mb_device_status(None, s)
            assert e.value.status == mb.MB_EDEVICE, f"expiry {rep}: status {e.value.status}"
    finally:
        mb.mb_gemm_set_split_wait(0, 0)
    for rep in range(2):
        dD.fill_(float("nan"))
        mb.mb_gemm(dA, dB, dD, dR, M, N, K, 1, None, s)
        mb.mb_device_status(None, s)
        assert_close(f"after expiry {rep}", f64(from_dev(dD)), ref)
    with pytest.raises(mb.MbError):
        mb.mb_gemm_set_split_wait(0, -1)


def test_gemm_reads_b_written_by_the_kernel_just_before(mb):
    """A standalone call's B may come from the kernel just before it on the
    stream: B waits for that kernel like A does (only a layer's own weights
    are loaded before the grid-dependency wait).  B is rewritten on the device
    right before each call, and the result must follow the new B."""
    M, N, K = 576, 4096, 4096
    A, B0, _ = _inputs(M, N, K, 11)
    _, B1, _ = _inputs(M, N, K, 12)
    s = torch.cuda.current_stream().cuda_stream
    dA, dB, dB0, dB1 = to_dev(A), to_dev(B0), to_dev(B0), to_dev(B1)
    dD = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for src, Bh in ((dB1, B1), (dB0, B0), (dB1, B1)):
        torch.mul(src, 1, out=dB)   # an elementwise kernel writes B (exactly), then the GEMM at once
        mb.mb_gemm(dA, dB, dD, None, M, N, K, 0, None, s)
        mb.mb_device_status(None, s)
        assert_close(f"gemm after B rewritten {M}x{N}x{K}", f64(from_dev(dD)), OL.linear(f64(A), f64(Bh)))
