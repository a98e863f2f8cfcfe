"""Pins of the oracle's batch / KV-cell bookkeeping: hand-computed cases and brute force."""
import numpy as np
import pytest

import oracle
from oracle.memory import Cells, sanitize_batch, split_simple

V, NSEQ = 100, 4


def sb(token, pos=None, seq=None, logits=None, cells=None, n_batch=64, output_all=False):
    n_seq_id = None if seq is None else [len(s) for s in seq]
    return sanitize_batch(token, pos, n_seq_id, seq, logits, n_vocab=V, n_seq_max=NSEQ,
                          n_batch=n_batch, cells=cells, output_all=output_all)


def test_sanitize_defaults():
    b = sb([5, 6, 7])
    assert b.seq_id == [[0], [0], [0]]
    assert b.pos.tolist() == [0, 1, 2]
    assert b.output.tolist() == [False, False, True]
    assert sb([5, 6], output_all=True).output.tolist() == [True, True]
    # positions continue each sequence from the memory, in batch order, per sequence
    c = Cells(16)
    c.apply([0, 1, 2], [0, 1, 2], [[0], [0], [0]])
    c.apply([3], [0], [[2]])
    b = sb([1, 2, 3, 4, 5], seq=[[0], [1], [0], [2], [1]], cells=c)
    assert b.pos.tolist() == [3, 0, 4, 1, 1]
    # a token in two sequences advances both
    b = sb([1, 2, 3], seq=[[1, 3], [1], [3]], cells=None)
    assert b.pos.tolist() == [0, 1, 1]


def test_sanitize_rejects_invalid_batches():
    assert sb([]) is None
    assert sb([V]) is None and sb([-1]) is None
    assert sb([1], seq=[[NSEQ]]) is None
    assert sb(list(range(65))) is None                           # more than n_batch tokens
    c = Cells(8)
    c.apply([0, 1], [0, 1], [[0], [0]])
    assert sb([1], pos=[5], cells=c) is None                     # gap after seq_pos_max
    assert sb([1, 2], pos=[2, 2], cells=c) is None               # not consecutive
    assert sb([1, 2], pos=[2, 3], cells=c).pos.tolist() == [2, 3]


def test_split_simple_in_batch_order():
    assert [list(r) for r in split_simple(5, 2)] == [[0, 1], [2, 3], [4]]
    assert [list(r) for r in split_simple(3, 8)] == [[0, 1, 2]]


def test_slots_lowest_free_and_holes_reused():
    c = Cells(8)
    assert c.find_slots(3) == [0, 1, 2]
    c.apply([0, 1, 2, 3], [0, 1, 2, 3], [[0]] * 4)
    c.apply([4, 5], [0, 1], [[1]] * 2)
    c.seq_rm(0, 2, -1)                                           # frees cells 2 and 3
    assert c.pos.tolist() == [0, 1, -1, -1, 0, 1, -1, -1]
    assert c.find_slots(3) == [2, 3, 6]
    assert c.find_slots(5) is None
    assert c.seq_pos_max(0) == 1 and c.seq_pos_min(1) == 0 and c.seq_pos_max(3) == -1


def test_seq_rm_ranges_and_shared_cells():
    c = Cells(6)
    c.apply([0, 1, 2], [0, 1, 2], [[0, 1], [0, 1], [0]])
    c.seq_rm(1, 0, -1)                                           # shared cells keep seq 0
    assert c.pos.tolist()[:3] == [0, 1, 2] and c.seqs_of(0) == {0}
    c.seq_rm(0, 1, 2)                                            # [1, 2): only position 1
    assert c.pos.tolist()[:3] == [0, -1, 2]
    c.seq_rm(0, -5, -1)                                          # p0 < 0 -> 0
    assert c.pos.tolist()[:3] == [-1, -1, -1]
    c.apply([0, 1], [0, 0], [[2], [3]])
    c.seq_rm(-1, 0, -1)                                          # every sequence
    assert c.n_kv() == 0


def test_mask_brute_force_small_case():
    # cells: seq0 pos 0,1 ; seq1 pos 0 ; shared {0,1} pos 2 ; empty ; seq0 pos 3
    c = Cells(6)
    c.apply([0, 1, 2, 3, 5], [0, 1, 0, 2, 3], [[0], [0], [1], [0, 1], [0]])
    assert c.n_kv() == 6
    m = c.mask([3, 2, 1], [[0], [1], [1]], 6)
    assert m[0].tolist() == [True, True, False, True, False, True]   # seq0 @ pos 3
    assert m[1].tolist() == [False, False, True, True, False, False]  # seq1 @ pos 2
    assert m[2].tolist() == [False, False, True, False, False, False]  # seq1 @ pos 1
    # brute force against the rule on a random state
    rng = np.random.default_rng(0)
    c = Cells(40)
    for cell in rng.permutation(40)[:30]:
        c.pos[cell] = rng.integers(0, 20)
        c.seq[cell, rng.choice(NSEQ, size=rng.integers(1, 3), replace=False)] = True
    pos = rng.integers(0, 20, size=7)
    seqs = [[int(rng.integers(0, NSEQ))] for _ in range(7)]
    m = c.mask(pos, seqs, 40)
    for t in range(7):
        for cell in range(40):
            want = c.pos[cell] >= 0 and seqs[t][0] in c.seqs_of(cell) and c.pos[cell] <= pos[t]
            assert m[t, cell] == want


def _ctx(n_ctx=256, n_ubatch=4, n_seq=2):
    from tests.helpers import MICRO, oracle_weights
    w = oracle_weights(MICRO, 11, {"embd": 0, "linear": 0})
    return oracle.OracleContext(MICRO, w, n_ctx=n_ctx, n_seq_max=n_seq, type_k=0, type_v=0,
                                n_batch=64, n_ubatch=n_ubatch)


def test_full_cache_returns_1_and_leaves_state_unchanged():
    ctx = _ctx(n_ctx=256, n_ubatch=64)
    assert ctx.decode(list(range(60)), logits=None) == 0
    assert ctx.decode(list(range(60)), logits=None) == 0
    assert ctx.decode(list(range(60)), logits=None) == 0
    assert ctx.decode(list(range(60)), logits=None) == 0
    before = (ctx.cells.pos.copy(), ctx.cells.seq.copy(), [k.copy() for k in ctx.K])
    assert ctx.decode(list(range(17))) == 1                         # 240 used, 16 free
    assert np.array_equal(ctx.cells.pos, before[0]) and np.array_equal(ctx.cells.seq, before[1])
    assert all(np.array_equal(a, b) for a, b in zip(ctx.K, before[2]))
    assert ctx.decode(list(range(16))) == 0


def test_abort_and_compute_failure_roll_back_only_the_failing_ubatch():
    for code, hook in ((2, "abort"), (-3, "fail")):
        ctx = _ctx(n_ubatch=4)
        calls = []
        if hook == "abort":
            ctx.abort_callback = lambda: (calls.append(1), len(calls) == 3)[1]
        else:
            ctx.fail_at_ubatch = 2
        assert ctx.decode(list(range(10)), logits=[1] * 10) == code
        # ubatches 0 and 1 (positions 0..7) stay; ubatch 2 (8, 9) is rolled back
        assert ctx.seq_pos_max(0) == 7 and ctx.cells.n_kv() == 8
        assert ctx.get_logits_ith(0) is None and ctx.n_outputs == 0
        # decoding continues from position 8
        ctx.abort_callback, ctx.fail_at_ubatch = None, None
        assert ctx.decode([1, 2]) == 0 and ctx.seq_pos_max(0) == 9


def test_logits_index_resolution():
    ctx = _ctx()
    assert ctx.decode([3, 4, 5, 6, 7], logits=[0, 1, 0, 1, 1]) == 0
    assert ctx.n_outputs == 3
    assert ctx.get_logits_ith(0) is None and ctx.get_logits_ith(5) is None
    assert np.array_equal(ctx.get_logits_ith(1), ctx.get_logits_ith(-3))
    assert np.array_equal(ctx.get_logits_ith(4), ctx.get_logits_ith(-1))
    assert ctx.get_logits_ith(-4) is None
    assert ctx.get_argmax_ith(2) == -1
    assert ctx.get_argmax_ith(3) == int(np.argmax(ctx.get_logits_ith(3)))
    assert ctx.decode([9]) == 0 and ctx.n_outputs == 1 and ctx.get_logits_ith(4) is None


def test_invalid_batch_returns_minus_1():
    ctx = _ctx()
    assert ctx.decode([]) == -1
    assert ctx.decode([1000]) == -1
    assert ctx.decode([1], seq_id=[[5]], n_seq_id=[1]) == -1
    assert ctx.cells.n_kv() == 0
