"""The token-major tensor-core GEMM of the prefill ubatches in isolation (f16 operands, tcgen05;
the two-CTA cta_group::2 kernel above 128 tokens, the one-CTA kernel at or below, and forced),
against a float64 CPU matmul of the same f16 inputs (a textbook routine). Shapes span ragged token
counts, split K and the 8B model's projection sizes; the second weight term (the form a Q8_0
weight's d*q takes) is multiplied in too."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _f16(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.float16)


def _f64(t):
    return t.double().numpy()


@pytest.mark.parametrize("M,K,T,splits", [(256, 64, 129, 1), (512, 256, 300, 1), (256, 128, 100, 1),
                                          (6144, 4096, 512, 1), (4096, 4096, 512, 2),
                                          (4096, 14336, 512, 2), (512, 1024, 257, 3)])
@pytest.mark.parametrize("one_cta", [False, True])
def test_gemm_tn_store_and_add(M, K, T, splits, one_cta):
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_f16
    W, X = _f16((M, K), 1, 0.05), _f16((T, K), 2)
    ref = oracle.linear(_f64(X), _f64(W))                       # [T][M]
    Wd, Xd = W.cuda(), X.cuda()
    Y = torch.zeros((T, M), device="cuda") if splits > 1 else torch.full((T, M), float("nan"), device="cuda")
    assert debug_gemm_tn_f16(0, Wd, Xd, Y, splits=splits, one_cta=one_cta) == 0
    got = Y.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < 2e-5
    base = torch.randn(T, M, device="cuda")
    Y2 = base.clone()
    assert debug_gemm_tn_f16(1, Wd, Xd, Y2, splits=splits, one_cta=one_cta) == 0
    err = np.max(np.abs((Y2 - base).cpu().double().numpy() - ref)) / np.max(np.abs(ref))
    assert err < 2e-5, err


@pytest.mark.parametrize("F,K,T", [(128, 64, 200), (256, 128, 257), (14336, 4096, 512)])
@pytest.mark.parametrize("one_cta", [False, True])
def test_gemm_tn_swiglu(F, K, T, one_cta):
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_f16
    W, X = _f16((2 * F, K), 3, 0.05), _f16((T, K), 4)
    gu = oracle.linear(_f64(X), _f64(W))
    ref = oracle.swiglu(gu[:, :F], gu[:, F:])
    Y = torch.zeros((T, F), dtype=torch.float16, device="cuda")
    assert debug_gemm_tn_f16(2, W.cuda(), X.cuda(), Y, F=F, one_cta=one_cta) == 0
    got = Y.cpu().double().numpy()
    # f16 output: one rounding of the result (2^-11 relative) on top of the f32 sums
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < 1e-3


def test_gemm_tn_two_weight_terms_and_kernels_agree():
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_f16
    M, K, T = 512, 512, 384
    W, Wl, X = _f16((M, K), 5, 0.05), _f16((M, K), 6, 0.05 / 2048), _f16((T, K), 7)
    ref = oracle.linear(_f64(X), _f64(W) + _f64(Wl))
    out = []
    for one in (False, True):
        Y = torch.full((T, M), float("nan"), device="cuda")
        assert debug_gemm_tn_f16(0, W.cuda(), X.cuda(), Y, W_lo=Wl.cuda(), one_cta=one) == 0
        out.append(Y.cpu().double().numpy())
        assert np.max(np.abs(out[-1] - ref)) / np.max(np.abs(ref)) < 2e-5
    # the same products in the same k order: the two kernels agree to float32 rounding
    assert np.max(np.abs(out[0] - out[1])) / np.max(np.abs(ref)) < 1e-6


def test_gemm_tn_rejects_unsupported_shapes():
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_f16
    W = torch.zeros((384, 64), dtype=torch.float16, device="cuda")
    X = torch.zeros((200, 64), dtype=torch.float16, device="cuda")
    assert debug_gemm_tn_f16(0, W, X, torch.zeros((200, 384), device="cuda")) == -1      # M % 256
