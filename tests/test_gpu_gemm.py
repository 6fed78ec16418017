"""Tensor-core (bf16) and CUDA-core (fp32) GEMM building block vs the plain
definition C[m, n] = Σ_k A[m, k]·B[n, k] in fp64, all operand layouts, tile
tails, multi-tile K."""

import numpy as np
import pytest
import torch

from _parity import f64

pytestmark = pytest.mark.gpu

SHAPES = [(128, 256, 64), (200, 264, 136), (384, 520, 1000), (8, 8, 8),
          (1000, 24, 72)]


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_bf16_layouts(tp, a_mn, b_mn, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = f64(A) @ f64(Bm).T
    dA = (A.t().contiguous() if a_mn else A).cuda()
    dB = (Bm.t().contiguous() if b_mn else Bm).cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    tp.gemm(dA, dB, C, a_mn_major=bool(a_mn), b_mn_major=bool(b_mn))
    tp.device_status()
    got = f64(C)
    assert np.isfinite(got).all()
    # bf16 output rounding (2^-8 relative) dominates fp32 accumulation error
    err = np.abs(got - ref).max()
    assert err <= 8e-3 * np.abs(ref).max() + 1e-3, err


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1)])
def test_gemm_f32(tp, a_mn, b_mn):
    M, N, K = 136, 72, 200
    g = torch.Generator().manual_seed(5)
    A = torch.randn(M, K, generator=g)
    Bm = torch.randn(N, K, generator=g)
    ref = f64(A) @ f64(Bm).T
    dA = (A.t().contiguous() if a_mn else A).cuda()
    dB = (Bm.t().contiguous() if b_mn else Bm).cuda()
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tp.gemm(dA, dB, C, a_mn_major=bool(a_mn), b_mn_major=bool(b_mn))
    tp.device_status()
    assert np.abs(f64(C) - ref).max() <= 1e-5 * np.abs(ref).max()


def test_gemm_large_k_many_tiles(tp):
    M, N, K = 512, 1024, 4096
    g = torch.Generator().manual_seed(11)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Bm = (torch.randn(N, K, generator=g) / 64).to(torch.bfloat16)
    ref = f64(A) @ f64(Bm).T
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tp.gemm(A.cuda(), Bm.cuda(), C)
    tp.device_status()
    assert np.abs(f64(C) - ref).max() <= 8e-3 * np.abs(ref).max()


def test_gemm_single_row(tp):
    # M = 1 (K-major A only: an MN-major A would need a leading dimension of 1)
    g = torch.Generator().manual_seed(3)
    A = torch.randn(1, 72, generator=g).to(torch.bfloat16)
    Bm = torch.randn(40, 72, generator=g).to(torch.bfloat16)
    C = torch.empty((1, 40), dtype=torch.bfloat16, device="cuda")
    tp.gemm(A.cuda(), Bm.cuda(), C)
    tp.device_status()
    ref = f64(A) @ f64(Bm).T
    assert np.abs(f64(C) - ref).max() <= 8e-3 * np.abs(ref).max()


def test_gemm_rejects_unaligned_leading_dim(tp):
    A = torch.zeros(8, 1, dtype=torch.bfloat16, device="cuda")  # [K, M=1]
    Bm = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(1, 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.gemm(A, Bm, C, a_mn_major=True)
    assert e.value.code == 2


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(2560, 2048, 192), (2504, 2000, 200)])
def test_gemm_partial_last_wave(tp, a_mn, b_mn, M, N, K):
    # 10 × 8 = 80 pair tiles: one full wave of the ≤ 76 resident pairs and a
    # last wave of a few tiles (the second shape also ragged in M, N and K)
    g = torch.Generator().manual_seed(M + N + K + 2 * a_mn + b_mn)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = f64(A) @ f64(Bm).T
    dA = (A.t().contiguous() if a_mn else A).cuda()
    dB = (Bm.t().contiguous() if b_mn else Bm).cuda()
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    tp.gemm(dA, dB, C, a_mn_major=bool(a_mn), b_mn_major=bool(b_mn))
    tp.device_status()
    got = f64(C)
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= 8e-3 * np.abs(ref).max() + 1e-3, err
