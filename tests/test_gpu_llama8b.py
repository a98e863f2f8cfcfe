"""GPU parity on the Llama-3-8B-shaped BF16 workload at full size, through the C ABI, against the
oracle: the 512-token prompt prefilled as one ubatch (tensor-core GEMMs, bf16 operands) and two
greedy decode steps (GEMV path), logits within a max relative error of 2e-2 per row and greedy
tokens equal wherever the oracle's top-2 gap exceeds 1e-3.

The oracle decodes each weight matrix from its bf16 storage when used (float64, bounded host
memory), so one pass over the 8B model costs it tens of seconds on the host cores."""
import numpy as np
import pytest

import oracle
import synthetic as S
from tests import gpu_common as G

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
TOL = 2e-2
KEY = "llama8b_bf16_1seq"


def _oracle_ctx():
    w = S.WORKLOADS[KEY]
    ow = oracle.OracleWeights(cache=False, row_chunk=4096)
    for n, wt, sh, t in G.device_model(KEY):
        ow.add(n, wt, sh[0], G.to_numpy_raw(t))
    return oracle.OracleContext(w.hp, ow, n_ctx=w.n_ctx, type_k=w.type_kv, type_v=w.type_kv,
                                n_batch=w.n_batch, n_ubatch=w.n_ubatch)


def test_llama8b_bf16_prompt_and_two_greedy_steps():
    w = S.WORKLOADS[KEY]
    ctx = G.library_ctx(KEY)
    toks = G.prompts(KEY)[0]
    assert ctx.decode(toks) == 0, ctx.last_error()
    ora = _oracle_ctx()
    assert ora.decode(toks) == 0
    rep = G.greedy_compare(ctx, ora, 1, [w.n_prompt - 1], 2, TOL, {})
    print("8B bf16 parity:", rep)
    ctx.free()
