"""The tensor-core (tcgen05/TMA/TMEM) BF16 GEMM in isolation, against a float64 CPU matmul of the
same bf16 inputs (a textbook routine). Shapes span several tiles, ragged token counts and the
8B model's projection sizes."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _f64(t):
    return t.float().double().numpy()


@pytest.mark.parametrize("M,K,T", [(128, 64, 1), (256, 128, 100), (384, 256, 129), (512, 512, 256),
                                   (640, 320, 300), (6144, 4096, 512), (4096, 14336, 77)])
def test_gemm_store_and_add(M, K, T):
    from transformer_decode_kv_gb300.binding import debug_gemm_bf16
    W = _bf16((M, K), 1, 0.05)
    X = _bf16((T, K), 2)
    ref = oracle.linear(_f64(X), _f64(W))                       # [T][M]
    Wd, Xd = W.cuda(), X.cuda()
    Y = torch.full((T, M), float("nan"), device="cuda")
    assert debug_gemm_bf16(0, Wd, Xd, Y) == 0
    got = Y.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err < 2e-5, err
    base = torch.randn(T, M, device="cuda")
    Y2 = base.clone()
    assert debug_gemm_bf16(1, Wd, Xd, Y2) == 0
    err = np.max(np.abs((Y2 - base).cpu().double().numpy() - ref)) / np.max(np.abs(ref))
    assert err < 2e-5, err


@pytest.mark.parametrize("F,K,T", [(64, 64, 5), (192, 256, 200), (14336, 4096, 512)])
def test_gemm_swiglu(F, K, T):
    from transformer_decode_kv_gb300.binding import debug_gemm_bf16
    W = _bf16((2 * F, K), 3, 0.05)
    X = _bf16((T, K), 4)
    gu = oracle.linear(_f64(X), _f64(W))
    ref = oracle.swiglu(gu[:, :F], gu[:, F:])
    Y = torch.zeros((T, F), dtype=torch.bfloat16, device="cuda")
    assert debug_gemm_bf16(2, W.cuda(), X.cuda(), Y, F=F) == 0
    got = Y.cpu().double().numpy()
    # bf16 output: one rounding of the result (2^-9 relative) on top of the f32 sums
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err < 5e-3, err


def test_gemm_rejects_unsupported_shapes():
    from transformer_decode_kv_gb300.binding import debug_gemm_bf16
    W = torch.zeros((100, 64), dtype=torch.bfloat16, device="cuda")
    X = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((4, 100), device="cuda")
    assert debug_gemm_bf16(0, W, X, Y) == -1
