"""The prefill path of the Llama-3-8B layer shape (2 layers, BF16 or Q8_0 linear weights, F16
cache) over a prompt of two 512-token ubatches, where the Q/K/V GEMM's epilogue (the two-CTA
kernel's, or the Q8_0 kernel's transposed one) applies RoPE and writes K and V to their cache
cells: a cell index planted past the cache for the second ubatch is caught by that epilogue's
bounds check, llm_decode returns -3 and rolls the second ubatch back ("デコードループ",
エラーリカバリとステートロールバック), and decoding the rest afterwards gives the logits of a run that
never failed. The two runs agree to RUN_TOL, not bit for bit: the K splits of the output and down
projections add their partial sums in whichever order they finish, and the next layer rounds the
activations to f16 (11 significant bits), so a last-place difference can move an activation by one
f16 step (4.9e-4 relative)."""
import numpy as np
import pytest

import synthetic as S
from synthetic.configs import HParams, Workload
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

HP = HParams(n_layer=2, n_embd=4096, n_head=32, n_head_kv=8, head_dim=128, n_ff=14336,
             n_vocab=32000, rope_freq_base=500000.0, rms_eps=1e-5)
RUN_TOL = 2e-3


@pytest.mark.parametrize("wtype", ["bf16", "q8_0"])
def test_bad_cell_in_the_fused_qkv_epilogue_rolls_back_and_resumes(wtype):
    KEY = "llama8b_layers2_" + wtype
    lin = S.BF16 if wtype == "bf16" else S.Q8_0
    S.WORKLOADS[KEY] = Workload(KEY, HP, {"embd": S.BF16, "linear": lin}, S.F16, n_ctx=2048,
                                n_seq=1, n_prompt=1024, n_batch=1024, n_ubatch=512, n_decode=2,
                                weight_seed=3500, prompt_seed=4500)
    G.device_model.cache_clear()
    toks = G.prompts(KEY)[0]
    ref = G.library_ctx(KEY)
    assert ref.decode(toks) == 0, ref.last_error()
    want = ref.get_logits_ith(-1).astype(np.float64)
    ctx = G.library_ctx(KEY)
    ctx.inject_fault(1, 1)
    assert ctx.decode(toks) == -3
    assert ctx.seq_pos_max(0) == 511 and ctx.kv_used_cells() == 512
    assert ctx.get_logits_ith(-1) is None
    assert ctx.decode(toks[512:]) == 0, ctx.last_error()
    assert G.rel_err(ctx.get_logits_ith(-1), want) < RUN_TOL
    # and the next greedy step agrees (both fed the clean run's token)
    t = ref.get_argmax_ith(-1)
    assert ref.decode([t]) == 0 and ctx.decode([t]) == 0
    assert G.rel_err(ctx.get_logits_ith(-1), ref.get_logits_ith(-1).astype(np.float64)) < RUN_TOL
    ctx.free(); ref.free()
    del S.WORKLOADS[KEY]
    G.device_model.cache_clear()
