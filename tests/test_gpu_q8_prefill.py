"""GPU parity of Q8_0 prefill on the tensor cores (the token-major tcgen05 GEMM reads each Q8_0
weight as stored and dequantises every k-step into two f16 terms, hi + lo, which hold d*q exactly;
activations one f16 term) on a 2-layer
model of the Llama-3-8B layer shape with Q8_0 linear weights and F32 embeddings/norms (the 8k
workload's types), through the C ABI.

A 512-token prompt (one ubatch: every GEMM on the tensor cores) then greedy steps (Q8_0 GEMVs),
against the oracle: every flagged logits row within the 2e-2 bar (expected ~1e-3: the f16
activations carry 11 significant bits)."""
import numpy as np
import pytest

import synthetic as S
from synthetic.configs import HParams, Workload
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

HP = HParams(n_layer=2, n_embd=4096, n_head=32, n_head_kv=8, head_dim=128, n_ff=14336,
             n_vocab=32000, rope_freq_base=500000.0, rms_eps=1e-5)
KEY = "llama8b_layers2_q8_0"
TOL = 2e-2


def test_q8_0_prefill_on_tensor_cores_matches_oracle():
    S.WORKLOADS[KEY] = Workload(KEY, HP, {"embd": S.F32, "linear": S.Q8_0}, S.F16, n_ctx=1024,
                                n_seq=1, n_prompt=512, n_batch=512, n_ubatch=512, n_decode=4,
                                weight_seed=3400, prompt_seed=4400)
    G.device_model.cache_clear()
    G.oracle_weights.cache_clear()
    ctx = G.library_ctx(KEY)
    ora = G.oracle_ctx(KEY)
    toks = G.prompts(KEY)[0]
    flags = np.zeros(512, dtype=np.int8)
    flags[[0, 100, 300, 511]] = 1
    assert ctx.decode(toks, logits=flags) == 0, ctx.last_error()
    assert ora.decode(toks, logits=flags) == 0
    assert ctx.perf()["n_ubatches"] == 1
    # the weights stay as stored (Q8_0: 34 bytes per 32 values), plus, for the prefill GEMMs, a
    # second copy of the linear layers' block scales in the per-k-step layout (2 bytes per 32)
    q8 = lambda rows, cols: rows * cols // 32 * (34 + 2)
    qkvw = (HP.n_head + 2 * HP.n_head_kv) * HP.head_dim
    per_layer = (q8(qkvw, HP.n_embd) + q8(HP.n_embd, HP.n_head * HP.head_dim) + q8(2 * HP.n_ff, HP.n_embd) +
                 q8(HP.n_embd, HP.n_ff))
    stored = HP.n_layer * per_layer + HP.n_vocab * HP.n_embd * 4 + HP.n_vocab * HP.n_embd // 32 * 34
    assert ctx.perf()["weight_device_bytes"] == stored
    errs = []
    for i in (0, 100, 300, 511):
        errs.append(G.rel_err(ctx.get_logits_ith(i), ora.get_logits_ith(i)))
    print("Q8_0 prefill rows:", errs)
    assert max(errs) <= TOL, errs
    assert max(errs) <= 5e-3, errs              # well inside the bar: exact weights, f16 activations
    rep = G.greedy_compare(ctx, ora, 1, [511], 4, TOL, {})
    print("Q8_0 steps:", rep)
    ctx.free()
