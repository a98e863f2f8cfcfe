"""Pins of the oracle's KV defrag (memory_update with optimize): the figure the pages print,
invariants of a compaction on random fragmented caches, unchanged logits, and the one defrag
retry when no slot is found."""
import os

import numpy as np
import pytest

import oracle
import synthetic as S
from oracle.memory import Cells
from tests.helpers import MICRO, oracle_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "defrag_figure.txt")


def _figure():
    rows = {"before": {}, "after": {}}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, val = (x.strip() for x in line.split("="))
        side, cell = key.split()
        rows[side][int(cell)] = None if val == "-" else tuple(int(v) for v in val.split())
    return rows


def test_the_pages_figure():
    fig = _figure()
    c = Cells(8)
    used = {k: v for k, v in fig["before"].items() if v is not None}
    c.apply(list(used), [v[1] for v in used.values()], [[v[0]] for v in used.values()])
    c.move(c.defrag_order())
    for cell, want in fig["after"].items():
        if want is None:
            assert c.pos[cell] < 0, cell
        else:
            assert c.seqs_of(cell) == {want[0]} and c.pos[cell] == want[1], cell
    assert c.n_kv() == 5


def _random_cells(rng, n_ctx=200, n_seq=6):
    c = Cells(n_ctx)
    nxt = [0] * n_seq
    for _ in range(30):
        if rng.random() < 0.3:
            s = int(rng.integers(0, n_seq))
            c.seq_rm(s, int(rng.integers(0, 20)), -1)
            nxt[s] = c.seq_pos_max(s) + 1
            continue
        n = int(rng.integers(1, 12))
        sl = c.find_slots(n)
        if sl is None:
            break
        ss = rng.choice(n_seq, size=2 if rng.random() < 0.2 else 1, replace=False).tolist()
        p0 = max(nxt[s] for s in ss)
        c.apply(sl, list(range(p0, p0 + n)), [ss] * n)
        for s in ss:
            nxt[s] = p0 + n
    return c


@pytest.mark.parametrize("seed", range(5))
def test_compaction_invariants(seed):
    c = _random_cells(np.random.default_rng(seed))
    before = sorted((int(c.pos[i]), tuple(sorted(c.seqs_of(i)))) for i in range(c.size) if c.pos[i] >= 0)
    n_used = len(before)
    src = c.defrag_order()
    assert np.all(src[:n_used] >= 0) and np.all(src[n_used:] < 0)
    assert sorted(src[:n_used].tolist()) == [i for i in range(c.size) if c.pos[i] >= 0]
    c.move(src)
    after = sorted((int(c.pos[i]), tuple(sorted(c.seqs_of(i)))) for i in range(c.size) if c.pos[i] >= 0)
    assert after == before                                   # nothing lost, nothing invented
    assert np.all(c.pos[:n_used] >= 0) and np.all(c.pos[n_used:] < 0)
    assert c.n_kv() == n_used
    # cells of a sequence's lowest-id group are contiguous and in position order
    key = [(min(c.seqs_of(i)), int(c.pos[i])) for i in range(n_used)]
    assert key == sorted(key)
    assert c.is_defragged()                                          # idempotent


def test_defrag_keeps_logits():
    w = oracle_weights(MICRO, 21, {"embd": S.F32, "linear": S.F32})
    ctxs = [oracle.OracleContext(MICRO, w, n_ctx=256, n_seq_max=3, n_ubatch=8) for _ in range(2)]
    toks = S.prompt_tokens(41, 30, MICRO.n_vocab).numpy()
    for ctx in ctxs:
        assert ctx.decode(toks, seq_id=[[i % 3] for i in range(30)], n_seq_id=[1] * 30) == 0
        ctx.seq_rm(1, 4, -1)
        ctx.seq_rm(0, 2, 5)                      # a hole inside sequence 0 too
        assert ctx.decode(toks[:3], seq_id=[[2]] * 3, n_seq_id=[1] * 3) == 0
    assert ctxs[1].memory_update(True) is True
    assert ctxs[1].memory_update(True) is False
    assert ctxs[1].cells.n_kv() < ctxs[0].cells.n_kv()
    nxt = [5, 7, 9]
    for ctx in ctxs:
        assert ctx.decode(nxt, seq_id=[[0], [1], [2]], n_seq_id=[1] * 3, logits=[1] * 3) == 0
    for i in range(3):
        a, b = ctxs[0].get_logits_ith(i), ctxs[1].get_logits_ith(i)
        assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a)), i


def test_no_slot_tries_one_defrag():
    ctx = oracle.OracleContext(MICRO, None, n_ctx=256, n_seq_max=2, n_batch=256, compute=False)
    assert ctx.decode([1] * 200, seq_id=[[i % 2] for i in range(200)], n_seq_id=[1] * 200) == 0
    ctx.seq_rm(0, 50, -1)                        # frees the even cells from 100 on
    assert not ctx.cells.is_defragged()
    assert ctx.decode([1] * 200, seq_id=[[1]] * 200, n_seq_id=[1] * 200) == 1     # 106 free
    assert ctx.cells.is_defragged()
    assert ctx.decode([1] * 100, seq_id=[[1]] * 100, n_seq_id=[1] * 100) == 0


def test_streams_defrag_within_each_stream():
    c = Cells(16, n_stream=2)                    # cells 0-7 stream 0, 8-15 stream 1
    c.apply([0, 2, 5, 9, 12, 15], [0, 1, 2, 0, 1, 2], [[0], [0], [0], [1], [1], [1]])
    src = c.defrag_order()
    assert src.tolist() == [0, 2, 5, -1, -1, -1, -1, -1, 9, 12, 15, -1, -1, -1, -1, -1]
    c.move(src)
    assert c.pos.tolist() == [0, 1, 2, -1, -1, -1, -1, -1, 0, 1, 2, -1, -1, -1, -1, -1]
