"""GPU parity of the KV defrag (llm_memory_update with optimize), through the C ABI.

  - Every layer's K/V rows move with their cells, bit-exact: after the defrag, new cell i holds the
    bytes old cell src[i] held, src being the oracle's defrag map for the same cell state
    (F16 and Q8_0 caches; the Q8_0 blocks move with their scales).
  - Logits of the next step after the defrag: equal to a twin context that was not defragmented
    (up to float summation order, 1e-5) and to the oracle that defragmented too (1e-4, the F32
    model's bar).
"""
import numpy as np
import pytest

import oracle
import synthetic as S
from oracle.formats import F16, Q8_0
from tests import gpu_common as G

pytestmark = pytest.mark.gpu
KEY = "tiny_f32_8seq"
N_SEQ, N_PROMPT = 4, 40


def _decode(ctx, toks, seqs, logits):
    if isinstance(ctx, oracle.OracleContext):
        return ctx.decode(toks, seq_id=seqs, n_seq_id=[len(s) for s in seqs], logits=logits)
    return ctx.decode(toks, seq_ids=seqs, logits=logits)


def _fragment(ctx):
    """Interleaved prompts of N_SEQ sequences, then holes: sequence 1 cut at 10, sequence 3 loses
    positions 5..14, sequence 0 gets 6 more tokens into the first holes."""
    w = S.WORKLOADS[KEY]
    toks = np.concatenate([S.prompt_tokens(w.prompt_seed_of(s), N_PROMPT, w.hp.n_vocab).numpy()
                           for s in range(N_SEQ)])
    seqs = [[s] for s in range(N_SEQ) for _ in range(N_PROMPT)]
    order = np.argsort(np.tile(np.arange(N_PROMPT), N_SEQ), kind="stable")   # interleave
    toks, seqs = toks[order], [seqs[i] for i in order]
    assert _decode(ctx, toks, seqs, [0] * len(toks)) == 0
    ctx.seq_rm(1, 10, -1)
    ctx.seq_rm(3, 5, 15)
    extra = [int(t) for t in toks[:6]]
    assert _decode(ctx, extra, [[0]] * 6, [0] * 6) == 0


def _next(ctx):
    nxt = [11, 22, 33, 44]
    assert ctx.decode(nxt, seq_ids=[[s] for s in range(N_SEQ)], logits=[1] * N_SEQ) == 0, ctx.last_error()
    return [ctx.get_logits_ith(i).copy() for i in range(N_SEQ)]


@pytest.mark.parametrize("tkv", [F16, Q8_0])
def test_defrag_moves_rows_and_keeps_logits(tkv):
    w = S.WORKLOADS[KEY]
    hp = w.hp
    kw = dict(n_seq_max=N_SEQ, type_k=tkv, type_v=tkv)
    a, b = G.library_ctx(KEY, **kw), G.library_ctx(KEY, **kw)
    ora = G.oracle_ctx(KEY, **kw)
    for ctx in (a, b):
        _fragment(ctx)
    _fragment(ora)
    src = ora.cells.defrag_order()
    keep = src >= 0
    before = [[b.kv_cache(il, which).copy() for which in (0, 1)] for il in range(hp.n_layer)]
    assert b.memory_update(True) == 1
    assert ora.memory_update(True) is True
    assert b.memory_update(True) == 0
    for il in range(hp.n_layer):
        for which in (0, 1):
            after = b.kv_cache(il, which)
            assert np.array_equal(after[:, keep], before[il][which][:, src[keep]]), (il, which)
    la, lb = _next(a), _next(b)
    lo = [None] * N_SEQ
    assert ora.decode([11, 22, 33, 44], seq_id=[[s] for s in range(N_SEQ)], n_seq_id=[1] * N_SEQ,
                      logits=[1] * N_SEQ) == 0
    assert b.last_slots().tolist() == [s for u in ora.last_ubatches for s in u["slots"]]
    for s in range(N_SEQ):
        lo[s] = ora.get_logits_ith(s)
        assert G.rel_err(lb[s], la[s].astype(np.float64)) <= 1e-5, s
        tol = 1e-4 if tkv == F16 else 1e-3
        assert G.rel_err(lb[s], lo[s]) <= tol, s
    for c in (a, b):
        c.free()
