"""The tcgen05 prefill attention tiles (32 tokens x 4 query heads = 128 MMA rows, 128-cell steps,
scores and outputs in TMEM) on a 2-layer model of the Llama-3-8B layer shape (BF16 weights, F16
cache), through the C ABI, against the oracle:

  - a 1024-token prompt in two 512-token ubatches: flagged logits rows within the 2e-2 bar of
    BF16 weights (expected well inside it: ~5e-3, the f16 activations carry 11 significant bits);
  - the same prompt in 64-token ubatches, where each tile's cell list is split into several work
    items whose partial states are merged: the same logits to RUN_TOL (ubatch splitting does not
    change the result, "llama.cpp AI LLM Engine - Як це працює", Крок 12);
  - two sequences in one batch (sequence-major): each sees only its own cells, rows against the
    oracle."""
import numpy as np
import pytest

import synthetic as S
from synthetic.configs import HParams, Workload
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

HP = HParams(n_layer=2, n_embd=4096, n_head=32, n_head_kv=8, head_dim=128, n_ff=14336,
             n_vocab=32000, rope_freq_base=500000.0, rms_eps=1e-5)
KEY = "llama8b_layers2_bf16_attn"
TOL = 2e-2
RUN_TOL = 2e-3        # two runs of the library: f16 activations round 1 ulp apart at most here


@pytest.fixture(scope="module")
def model():
    S.WORKLOADS[KEY] = Workload(KEY, HP, {"embd": S.BF16, "linear": S.BF16}, S.F16, n_ctx=2048,
                                n_seq=2, n_prompt=1024, n_batch=2048, n_ubatch=512, n_decode=2,
                                weight_seed=3600, prompt_seed=4600)
    G.device_model.cache_clear()
    G.oracle_weights.cache_clear()
    yield KEY
    del S.WORKLOADS[KEY]
    G.device_model.cache_clear()
    G.oracle_weights.cache_clear()


ROWS = [0, 200, 511, 512, 777, 1023]


def test_tc_attention_prompt_matches_oracle_and_ubatch_split(model):
    toks = G.prompts(model)[0]
    flags = np.zeros(len(toks), dtype=np.int8)
    flags[ROWS] = 1
    ctx = G.library_ctx(model, n_seq_max=1)
    assert ctx.decode(toks, logits=flags) == 0, ctx.last_error()
    ora = G.oracle_ctx(model, n_seq_max=1)
    assert ora.decode(toks, logits=flags) == 0
    errs = [G.rel_err(ctx.get_logits_ith(i), ora.get_logits_ith(i)) for i in ROWS]
    print("tc attention rows vs oracle:", errs)
    assert max(errs) <= TOL, errs
    assert max(errs) <= 8e-3, errs
    want = [ctx.get_logits_ith(i).astype(np.float64) for i in ROWS]
    ctx.free()
    # 64-token ubatches: several work items per tile, merged
    small = G.library_ctx(model, n_seq_max=1, n_ubatch=64)
    assert small.decode(toks, logits=flags) == 0, small.last_error()
    errs = [G.rel_err(small.get_logits_ith(i), w) for i, w in zip(ROWS, want)]
    print("64-token ubatches vs 512:", errs)
    assert max(errs) <= RUN_TOL, errs
    small.free()


def test_tc_attention_two_sequences(model):
    ps = G.prompts(model)
    n = 300
    toks = np.concatenate([ps[0][:n], ps[1][:n]])
    seqs = [[0]] * n + [[1]] * n
    rows = [0, n - 1, n, 2 * n - 1]
    flags = np.zeros(2 * n, dtype=np.int8)
    flags[rows] = 1
    ctx = G.library_ctx(model)
    ora = G.oracle_ctx(model)
    assert ctx.decode(toks, seq_ids=seqs, logits=flags) == 0, ctx.last_error()
    assert ora.decode(toks, seq_id=seqs, n_seq_id=[1] * (2 * n), logits=flags) == 0
    errs = [G.rel_err(ctx.get_logits_ith(i), ora.get_logits_ith(i)) for i in rows]
    print("two sequences vs oracle:", errs)
    assert max(errs) <= 8e-3, errs
    ctx.free()
