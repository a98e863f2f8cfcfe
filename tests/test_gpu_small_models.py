"""GPU parity on small BF16 and Q8_0 models whose shapes take every fast path of the library:
the tensor-core prefill GEMMs (BF16), the bulk-staged decode GEMVs with fused RMSNorm, RoPE + K/V
append, SwiGLU and logits/argmax epilogues (BF16 and Q8_0), and decode-step graph replay.
Against the oracle: logits within the 2e-2 bar of BF16 and Q8_0 weights (the prefill GEMMs take
f16 operands), greedy tokens gap-checked."""
import dataclasses

import numpy as np
import pytest

import oracle
import synthetic as S
from synthetic.configs import HParams, Workload
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

SMALL = HParams(n_layer=2, n_embd=512, n_head=8, n_head_kv=2, head_dim=64, n_ff=1024, n_vocab=1024,
                rope_freq_base=10000.0, rms_eps=1e-5)


def _workload(key, types, n_prompt, n_ubatch):
    return Workload(key, SMALL, types, S.F16, n_ctx=1024, n_seq=1, n_prompt=n_prompt, n_batch=512,
                    n_ubatch=n_ubatch, n_decode=8, weight_seed=3100 + len(key), prompt_seed=4100)


@pytest.mark.parametrize("key,types,tol", [
    ("small_bf16", {"embd": S.BF16, "linear": S.BF16}, 2e-2),
    ("small_q8_0", {"embd": S.F32, "linear": S.Q8_0}, 2e-2),     # prefill GEMMs take f16 operands
])
@pytest.mark.parametrize("n_prompt,n_ubatch", [(300, 512), (77, 32)])
def test_small_model_prefill_and_decode(key, types, tol, n_prompt, n_ubatch):
    wk = f"{key}_{n_prompt}_{n_ubatch}"
    S.WORKLOADS[wk] = _workload(wk, types, n_prompt, n_ubatch)
    G.device_model.cache_clear(); G.oracle_weights.cache_clear()
    ctx, ora = G.library_ctx(wk), G.oracle_ctx(wk)
    toks = G.prompts(wk)[0]
    assert ctx.decode(toks) == 0, ctx.last_error()
    assert ora.decode(toks) == 0
    rep = G.greedy_compare(ctx, ora, 1, [n_prompt - 1], 8, tol, {})
    assert rep.get("tokens_checked", 0) >= 4
    perf = ctx.perf()
    assert perf["n_graph_replays"] >= 7            # decode steps replay one captured graph
    ctx.free()
    del S.WORKLOADS[wk]
