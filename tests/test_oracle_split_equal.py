"""Pins of the oracle's split cache (one stream per sequence, kv_unified = false) and its
ubatch splitter split_equal: hand-worked splits, invariants of the split on random batches, the
stream bounds (n_ctx_seq = n_ctx / n_seq_max), and results equal to the unified cache's."""
import numpy as np
import pytest

import oracle
import synthetic as S
from oracle.memory import DecodeStatus, split_equal, split_simple
from tests.helpers import MICRO, oracle_weights


def test_hand_worked_splits():
    # sequences 0,0,0,1,1,2 in ubatches of 4: one token of each live sequence per ubatch
    assert split_equal([0, 0, 0, 1, 1, 2], 4) == [[0, 3, 5], [1, 4], [2]]
    # equal shares: 2 sequences x 3 tokens fit 6; the longer one continues alone
    assert split_equal([0, 1, 0, 1, 0, 1, 0, 0], 6) == [[0, 2, 4, 1, 3, 5], [6, 7]]
    # "sequential": a gap in the ids ends the ubatch's sequence run
    assert split_equal([0, 2, 2], 8) == [[0], [1, 2]]
    # more live sequences than n_ubatch: the lowest n_ubatch of them
    assert split_equal([3, 2, 1, 0], 2) == [[3, 2], [1, 0]]


@pytest.mark.parametrize("seed", range(6))
def test_split_invariants(seed):
    rng = np.random.default_rng(seed)
    n, n_ub = int(rng.integers(1, 200)), int(rng.integers(1, 40))
    seqs = rng.integers(0, 7, size=n).tolist()
    ubs = split_equal(seqs, n_ub)
    flat = [i for u in ubs for i in u]
    assert sorted(flat) == list(range(n))                        # every token once
    for s in set(seqs):                                           # batch order within a sequence
        mine = [i for i in flat if seqs[i] == s]
        assert mine == sorted(mine)
    for u in ubs:
        assert 1 <= len(u) <= n_ub
        ss = [seqs[i] for i in u]
        ids = sorted(set(ss))
        assert ids == list(range(ids[0], ids[0] + len(ids)))      # consecutive ids
        counts = {s: ss.count(s) for s in ids}
        assert len(set(counts.values())) == 1                    # n_seq_tokens each
        assert ss == sorted(ss)                                   # sequence by sequence
    # one sequence: the same ubatches as split_simple
    assert split_equal([4] * n, n_ub) == [list(r) for r in split_simple(n, n_ub)]


def _ctx(w, unified, n_ctx=256, n_seq=4, n_ubatch=7):
    return oracle.OracleContext(MICRO, w, n_ctx=n_ctx, n_seq_max=n_seq, n_ubatch=n_ubatch,
                                kv_unified=unified)


@pytest.fixture(scope="module")
def micro():
    return oracle_weights(MICRO, 21, {"embd": S.F32, "linear": S.F32})


def test_streams_bound_the_slots():
    ctx = oracle.OracleContext(MICRO, None, n_ctx=256, n_seq_max=4, n_ubatch=16, kv_unified=False,
                               compute=False)
    assert ctx.cells.n_ctx_seq == 64
    seqs = [[i % 4] for i in range(20)]
    assert ctx.decode(list(range(1, 21)), seq_id=seqs, n_seq_id=[1] * 20) == 0
    for s in range(4):                                 # each sequence in its own 64 cells
        assert np.nonzero(ctx.cells.seq[:, s])[0].tolist() == list(range(64 * s, 64 * s + 5)), s
    # ubatches of 16: 4 sequences x 4 tokens, then 4 x 1
    assert [len(u["slots"]) for u in ctx.last_ubatches] == [16, 4]
    # a full stream refuses more tokens although other streams have room
    assert ctx.decode([1] * 59, seq_id=[[2]] * 59, n_seq_id=[1] * 59) == 0
    assert ctx.decode([1], seq_id=[[2]], n_seq_id=[1]) == int(DecodeStatus.NO_KV_SLOT)
    assert ctx.decode([1], seq_id=[[3]], n_seq_id=[1]) == 0
    # a token of two sequences cannot live in two streams
    assert ctx.decode([1], seq_id=[[0, 1]], n_seq_id=[2]) == int(DecodeStatus.INVALID_BATCH)


def _close(x, y):
    return np.max(np.abs(x - y)) <= 1e-12 * np.max(np.abs(x))


def test_split_cache_gives_the_unified_results(micro):
    a, b = _ctx(micro, True), _ctx(micro, False)
    rng = np.random.default_rng(5)
    toks = rng.integers(0, MICRO.n_vocab, size=40).tolist()
    seqs = [[int(s)] for s in rng.integers(0, 4, size=40)]
    flags = (rng.random(40) < 0.4).astype(int).tolist()
    flags[-1] = 1
    for ctx in (a, b):
        assert ctx.decode(toks, seq_id=seqs, n_seq_id=[1] * 40, logits=flags) == 0
    for i in range(40):
        ra, rb = a.get_logits_ith(i), b.get_logits_ith(i)
        assert (ra is None) == (rb is None), i
        if ra is not None:
            assert _close(ra, rb), i
    # output rows are in batch order although the split cache's ubatches reorder the tokens
    assert _close(a.get_logits_ith(-1), b.get_logits_ith(-1))
    assert np.array_equal(b.get_logits_ith(-1), b.get_logits_ith(39))
    assert np.array_equal(b.get_logits_ith(-2), b.get_logits_ith(int(np.nonzero(flags)[0][-2])))
    nxt = [[s] for s in range(4)]
    for ctx in (a, b):
        assert ctx.decode([1, 2, 3, 4], seq_id=nxt, n_seq_id=[1] * 4, logits=[1] * 4) == 0
    for i in range(4):
        assert _close(a.get_logits_ith(i), b.get_logits_ith(i)), i
