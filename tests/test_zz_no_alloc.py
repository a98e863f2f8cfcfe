"""The GEMM entry point that allocates no device memory (llm_gemm_bf16_noalloc), for callers that
cannot allocate: its results must match the allocating entry point (llm_debug_gemm_bf16) and the
oracle's matrix product on two calls in a row.

The error word it keeps in its fixed scratch array is planted with a nonzero value before the
second call, as a failed earlier call would leave it: the call must clear it and return 0.

Kept in a file pytest collects last; it passes alone in a fresh process (the first call sets up the
scratch address on the device) and after the other tests."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
TOL = 2e-5          # the tensor-core GEMM tests' bar (max error relative to the largest value)


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).cuda()


def _f64(t):
    return t.cpu().double().numpy()


def test_noalloc_gemm_matches_allocating_entry_point_and_oracle_twice():
    from transformer_decode_kv_gb300.binding import (debug_gemm_bf16, debug_noalloc_scratch_poke,
                                                     gemm_bf16_noalloc)
    # call 1: store epilogue, ragged token count
    W, X = _bf16((384, 256), 11, 0.05), _bf16((130, 256), 12)
    want = torch.zeros(130, 384, device="cuda")
    got = torch.full((130, 384), float("nan"), device="cuda")
    assert debug_gemm_bf16(0, W, X, want) == 0
    assert gemm_bf16_noalloc(0, W, X, got) == 0
    a, b = _f64(got), _f64(want)
    assert np.max(np.abs(a - b)) / np.max(np.abs(b)) <= TOL
    o = oracle.linear(_f64(X), _f64(W))                       # MUL_MAT in float64
    assert np.max(np.abs(a - o)) / np.max(np.abs(o)) <= TOL
    # call 2: SwiGLU epilogue on other inputs, straight after, with the error word left nonzero
    F = 128
    W2, X2 = _bf16((2 * F, 512), 13, 0.05), _bf16((300, 512), 14)
    want2 = torch.zeros(300, F, dtype=torch.bfloat16, device="cuda")
    got2 = torch.zeros(300, F, dtype=torch.bfloat16, device="cuda")
    assert debug_gemm_bf16(2, W2, X2, want2, F=F) == 0
    assert debug_noalloc_scratch_poke(0xDEAD) == 0
    assert gemm_bf16_noalloc(2, W2, X2, got2, F=F) == 0
    a, b = _f64(got2), _f64(want2)
    assert np.max(np.abs(a - b)) / np.max(np.abs(b)) <= TOL
    g2 = oracle.linear(_f64(X2), _f64(W2))
    o2 = oracle.swiglu(g2[:, :F], g2[:, F:])
    # the output is rounded to bf16 (8 significant bits): half an ulp of the largest value
    assert np.max(np.abs(a - o2)) / np.max(np.abs(o2)) <= 2.0 ** -8
    # an unsupported shape is refused, not run
    assert gemm_bf16_noalloc(0, _bf16((100, 64), 15), _bf16((4, 64), 16), torch.zeros(4, 100, device="cuda")) == -1
