"""The token-major tensor-core GEMM over a Q8_0 weight as the library stores it (int8 quants and
fp16 block scales), dequantised inside the kernel into the exact f16 terms of d * q, against the
oracle: the weight decoded from its Q8_0 blocks ([P2] "llama.cpp Architecture", Example 2: an fp16
scale and 32 int8 quants per block, value d * q) and multiplied in float64 (MUL_MAT, Example 4).
Shapes span ragged and small token counts (a single 128-token tile runs on the pair with an empty
peer), split K, the 8B model's projection sizes and the SwiGLU epilogue."""
import numpy as np
import pytest
import torch

import oracle
from oracle.formats import Q8_0

pytestmark = pytest.mark.gpu
TOL = 2e-5          # max error relative to the largest value: f32 sums of exact products


def _q8(rows, K, seed, scale_sigma):
    """Random Q8_0 rows: (raw blocks uint8 [rows][K/32*34], quants int8 [rows][K], scales f16)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randint(-128, 128, (rows, K), generator=g, dtype=torch.int8)
    d = (torch.randn(rows, K // 32, generator=g).abs() * scale_sigma).to(torch.float16)
    blocks = np.zeros((rows, K // 32, 34), dtype=np.uint8)
    blocks[:, :, 0:2] = d.numpy().view(np.uint8).reshape(rows, K // 32, 2)
    blocks[:, :, 2:] = q.numpy().view(np.uint8).reshape(rows, K // 32, 32)
    return blocks.reshape(rows, -1), q, d


def _f16(shape, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.float16)


def _weight(raw, K):
    return oracle.decode_weight(raw, Q8_0, K)


@pytest.mark.parametrize("M,K,T,splits", [(256, 64, 129, 1), (512, 256, 300, 1), (256, 128, 100, 1),
                                          (256, 128, 1, 1), (6144, 4096, 512, 1), (4096, 4096, 512, 2),
                                          (4096, 14336, 512, 2), (512, 1024, 257, 3)])
def test_gemm_q8_store_and_add(M, K, T, splits):
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_q8
    raw, q, d = _q8(M, K, 10 + M + K, 0.01)
    X = _f16((T, K), 20 + T)
    ref = oracle.linear(X.double().numpy(), _weight(raw, K))                 # [T][M]
    qd, dd, Xd = q.cuda(), d.cuda(), X.cuda()
    Y = torch.zeros((T, M), device="cuda") if splits > 1 else torch.full((T, M), float("nan"), device="cuda")
    assert debug_gemm_tn_q8(0, qd, dd, Xd, Y, splits=splits) == 0
    got = Y.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err < TOL, err
    base = torch.randn(T, M, device="cuda")
    Y2 = base.clone()
    assert debug_gemm_tn_q8(1, qd, dd, Xd, Y2, splits=splits) == 0
    err = np.max(np.abs((Y2 - base).cpu().double().numpy() - ref)) / np.max(np.abs(ref))
    assert err < TOL, err


@pytest.mark.parametrize("F,K,T", [(128, 64, 200), (256, 128, 257), (128, 256, 40), (14336, 4096, 512)])
def test_gemm_q8_swiglu(F, K, T):
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_q8
    raw, q, d = _q8(2 * F, K, 30 + F, 0.01)
    X = _f16((T, K), 40 + T)
    gu = oracle.linear(X.double().numpy(), _weight(raw, K))
    ref = oracle.swiglu(gu[:, :F], gu[:, F:])
    Y = torch.zeros((T, F), dtype=torch.float16, device="cuda")
    assert debug_gemm_tn_q8(2, q.cuda(), d.cuda(), X.cuda(), Y, F=F) == 0
    got = Y.cpu().double().numpy()
    # f16 output: one rounding of the result (2^-11 relative) on top of the f32 sums
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < 1e-3


def test_gemm_q8_model_scales_with_subnormal_low_terms():
    """Scales of the size the synthetic 8B model draws (|N(0, 2e-4)|): the low f16 term of d * q
    falls in the f16 subnormal range, where it keeps fewer bits; the sums still hold the bar."""
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_q8
    M, K, T = 512, 4096, 300
    raw, q, d = _q8(M, K, 50, 2e-4)
    X = _f16((T, K), 51)
    ref = oracle.linear(X.double().numpy(), _weight(raw, K))
    Y = torch.full((T, M), float("nan"), device="cuda")
    assert debug_gemm_tn_q8(0, q.cuda(), d.cuda(), X.cuda(), Y) == 0
    err = np.max(np.abs(Y.cpu().double().numpy() - ref)) / np.max(np.abs(ref))
    assert err < TOL, err


def test_gemm_q8_rejects_unsupported_shapes():
    from transformer_decode_kv_gb300.binding import debug_gemm_tn_q8
    raw, q, d = _q8(128, 64, 60, 0.01)
    X = _f16((8, 64), 61).cuda()
    Y = torch.zeros((8, 128), device="cuda")
    assert debug_gemm_tn_q8(0, q.cuda(), d.cuda(), X, Y) == -1          # M % 256 != 0
