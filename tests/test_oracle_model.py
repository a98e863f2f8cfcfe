"""The oracle's whole forward pass, pinned by analytic models and invariants.

The pages print no logits for a reproducible input, so whole-forward values are pinned by:
  * analytic models whose weights reduce the forward pass to a closed form (uniform attention is
    the mean of the visible value rows; zeroed projections leave the embedding on the residual);
  * invariants: cached decoding equals a no-cache forward of the whole sequence; the result does
    not depend on how a batch is split into ubatches; sequences batched together equal each
    sequence run alone.
"""
import numpy as np
import pytest

import oracle
from oracle.context import forward_no_cache
from synthetic.configs import HParams
from tests.helpers import MICRO, oracle_weights, tiny_weights

import synthetic as S


def _analytic_model(rng, d=4, V=5, F=2):
    """One layer, one head of size d: Wq = 0 (all scores equal), Wv = Wo = I, ffn_down = 0."""
    hp = HParams(n_layer=1, n_embd=d, n_head=1, n_head_kv=1, head_dim=d, n_ff=F, n_vocab=V,
                 rope_freq_base=10000.0, rms_eps=1e-6)
    E = rng.standard_normal((V, d)).astype(np.float32)
    Wout = rng.standard_normal((V, d)).astype(np.float32)
    mats = {
        "token_embd.weight": E, "output.weight": Wout,
        "output_norm.weight": np.ones((1, d), np.float32),
        "blk.0.attn_norm.weight": np.ones((1, d), np.float32),
        "blk.0.ffn_norm.weight": np.ones((1, d), np.float32),
        "blk.0.attn_q.weight": np.zeros((d, d), np.float32),
        "blk.0.attn_k.weight": rng.standard_normal((d, d)).astype(np.float32),
        "blk.0.attn_v.weight": np.eye(d, dtype=np.float32),
        "blk.0.attn_output.weight": np.eye(d, dtype=np.float32),
        "blk.0.ffn_gate.weight": rng.standard_normal((F, d)).astype(np.float32),
        "blk.0.ffn_up.weight": rng.standard_normal((F, d)).astype(np.float32),
        "blk.0.ffn_down.weight": np.zeros((d, F), np.float32),
    }
    w = oracle.OracleWeights()
    for k, m in mats.items():
        w.add(k, oracle.F32, m.shape[1], m)
    return hp, w, E.astype(np.float64), Wout.astype(np.float64)


def test_analytic_uniform_attention_is_mean_of_visible_values():
    rng = np.random.default_rng(5)
    hp, w, E, Wout = _analytic_model(rng)
    ctx = oracle.OracleContext(hp, w, n_ctx=256, n_seq_max=2, type_k=oracle.F32,
                               type_v=oracle.F32, n_batch=32, n_ubatch=3)
    toks = [1, 4, 2, 0, 3, 3, 1]
    seqs = [[0], [1], [0], [0], [1], [0], [1]]
    assert ctx.decode(toks, seq_id=seqs, n_seq_id=[1] * 7, logits=[1] * 7) == 0
    norm = lambda x: x / np.sqrt(np.mean(x * x) + hp.rms_eps)
    hist = {0: [], 1: []}
    for t, (tok, s) in enumerate(zip(toks, seqs)):
        vrow = norm(E[tok]).astype(np.float32).astype(np.float64)   # V row as the F32 cache holds it
        hist[s[0]].append(vrow)
        x = E[tok] + np.mean(hist[s[0]], axis=0)                    # mean of same-sequence rows so far
        want = norm(x) @ Wout.T
        assert np.allclose(ctx.get_logits_ith(t), want, rtol=1e-12, atol=1e-12)
    # a later single-token step sees the whole history of its sequence only
    assert ctx.decode([2], seq_id=[[1]], n_seq_id=[1]) == 0
    hist[1].append(norm(E[2]).astype(np.float32).astype(np.float64))
    want = norm(E[2] + np.mean(hist[1], axis=0)) @ Wout.T
    assert np.allclose(ctx.get_logits_ith(-1), want, rtol=1e-12, atol=1e-12)


def test_analytic_zero_projections_leave_the_embedding():
    rng = np.random.default_rng(6)
    hp, w, E, Wout = _analytic_model(rng)
    w.add("blk.0.attn_output.weight", oracle.F32, 4, np.zeros((4, 4), np.float32))
    ctx = oracle.OracleContext(hp, w, n_ctx=256, type_k=oracle.F16, type_v=oracle.F16)
    assert ctx.decode([3, 1, 4], logits=[1, 1, 1]) == 0
    for t, tok in enumerate([3, 1, 4]):
        x = E[tok]
        want = x / np.sqrt(np.mean(x * x) + hp.rms_eps) @ Wout.T
        assert np.allclose(ctx.get_logits_ith(t), want, rtol=1e-13, atol=1e-13)
    # tied output: without output.weight the embedding matrix is reused
    del w.raw["output.weight"]
    ctx = oracle.OracleContext(hp, w, n_ctx=256)
    assert ctx.decode([2]) == 0
    x = E[2]
    assert np.allclose(ctx.get_logits_ith(0), x / np.sqrt(np.mean(x * x) + hp.rms_eps) @ E.T)


@pytest.fixture(scope="module")
def micro():
    return oracle_weights(MICRO, 21, {"embd": S.F32, "linear": S.F32})


@pytest.mark.parametrize("tkv", [oracle.F32, oracle.F16])
def test_cached_decode_equals_no_cache_forward(micro, tkv):
    toks = S.prompt_tokens(31, 12, MICRO.n_vocab).numpy()
    full = forward_no_cache(micro, MICRO, toks, tkv, tkv)
    ctx = oracle.OracleContext(MICRO, micro, n_ctx=256, type_k=tkv, type_v=tkv, n_ubatch=5)
    assert ctx.decode(toks[:7], logits=[1] * 7) == 0
    got = [ctx.get_logits_ith(i) for i in range(7)]
    for t in toks[7:]:
        assert ctx.decode([t]) == 0
        got.append(ctx.get_logits_ith(-1))
    rtol = 1e-9 if tkv == oracle.F32 else 1e-4
    scale = np.max(np.abs(full), axis=1, keepdims=True)
    assert np.max(np.abs(np.array(got) - full) / scale) < rtol


def test_ubatch_split_does_not_change_logits(micro):
    toks = S.prompt_tokens(32, 32, MICRO.n_vocab).numpy()
    ref = None
    for nub in (1, 7, 32):
        ctx = oracle.OracleContext(MICRO, micro, n_ctx=256, type_k=oracle.F32,
                                   type_v=oracle.F32, n_ubatch=nub)
        assert ctx.decode(toks, logits=[1] * 32) == 0
        out = ctx.logits.copy()
        assert [len(u["slots"]) for u in ctx.last_ubatches][0] == min(nub, 32)
        if ref is None:
            ref = out
        else:
            assert np.allclose(out, ref, rtol=1e-11, atol=1e-11)


def test_sequences_batched_equal_each_alone(micro):
    n_seq, n = 3, 9
    prompts = [S.prompt_tokens(40 + s, n, MICRO.n_vocab).numpy() for s in range(n_seq)]
    # interleaved batch order: token i of every sequence, then i + 1 ...
    toks, seqs = [], []
    for i in range(n):
        for s in range(n_seq):
            toks.append(prompts[s][i]); seqs.append([s])
    ctx = oracle.OracleContext(MICRO, micro, n_ctx=256, n_seq_max=n_seq, type_k=oracle.F16,
                               type_v=oracle.F16, n_ubatch=4)
    assert ctx.decode(toks, seq_id=seqs, n_seq_id=[1] * len(toks), logits=[1] * len(toks)) == 0
    for s in range(n_seq):
        alone = oracle.OracleContext(MICRO, micro, n_ctx=256, type_k=oracle.F16, type_v=oracle.F16)
        assert alone.decode(prompts[s], logits=[1] * n) == 0
        for i in range(n):
            assert np.allclose(ctx.get_logits_ith(i * n_seq + s), alone.get_logits_ith(i),
                               rtol=1e-9, atol=1e-9)
    # seq_rm of one sequence leaves the others' next step unchanged, and its cells are reused
    ctx.seq_rm(1, 4, -1)
    freed = [c for c in range(ctx.n_ctx) if ctx.cells.pos[c] < 0][:2]
    assert ctx.decode([5, 6], seq_id=[[0], [1]], n_seq_id=[1, 1], logits=[1, 1]) == 0
    assert ctx.last_ubatches[0]["slots"] == freed
    assert ctx.seq_pos_max(1) == 4
    alone = oracle.OracleContext(MICRO, micro, n_ctx=256, type_k=oracle.F16, type_v=oracle.F16)
    assert alone.decode(np.append(prompts[0], 5), logits=[0] * n + [1]) == 0
    assert np.allclose(ctx.get_logits_ith(0), alone.get_logits_ith(-1), rtol=1e-9, atol=1e-9)


def test_tiny_model_cached_decode_equals_no_cache_forward():
    w = tiny_weights(1001)
    toks = S.prompt_tokens(2001, 6, S.TINY.n_vocab).numpy()
    full = forward_no_cache(w, S.TINY, toks, oracle.F32, oracle.F32)
    ctx = oracle.OracleContext(S.TINY, w, n_ctx=512, type_k=oracle.F32, type_v=oracle.F32)
    assert ctx.decode(toks[:4], logits=[0, 0, 0, 1]) == 0
    got = [ctx.get_logits_ith(-1)]
    for t in toks[4:]:
        assert ctx.decode([t]) == 0
        got.append(ctx.get_logits_ith(-1))
    assert np.allclose(np.array(got), full[3:], rtol=1e-9, atol=1e-9 * np.abs(full).max())
