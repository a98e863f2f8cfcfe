"""The C-ABI library on a machine without a GPU: it loads, exports every symbol include/llm.h
declares, and its host control plane (batch sanitising, ubatch split, slot search, cell
commit, seq_rm, visibility lists, rollback, return codes) matches the oracle bit for bit.

The library runs in host-only mode here (LLM_CTX_HOST_ONLY): no device memory, no kernels."""
import os
import re

import numpy as np
import pytest

import oracle
from synthetic.configs import HParams

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def T():
    from transformer_decode_kv_gb300 import build, binding
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding


def test_library_exports_every_declared_symbol(T):
    hdr = open(os.path.join(ROOT, "include", "llm.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    declared = set(re.findall(r"\b(llm_[a-z0-9_]+)\s*\(", hdr))
    assert len(declared) >= 20
    L = T.lib()
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert declared == set(T.SIGNATURES), declared ^ set(T.SIGNATURES)


HP = HParams(n_layer=2, n_embd=64, n_head=8, n_head_kv=2, head_dim=32, n_ff=96, n_vocab=50,
             rope_freq_base=10000.0, rms_eps=1e-6)


def test_context_parameter_derivation(T):
    c = T.Context(HP, n_ctx=100, n_batch=2048, n_ubatch=512, host_only=True)
    assert (c.n_ctx, c.n_batch, c.n_ubatch) == (256, 256, 256)
    c = T.Context(HP, n_ctx=8320, n_batch=8192, n_ubatch=512, host_only=True)
    assert (c.n_ctx, c.n_batch, c.n_ubatch) == (8448, 8192, 512)
    with pytest.raises(T.LlmError):
        T.Context(HP, n_ctx=256, n_seq_max=0, host_only=True)
    with pytest.raises(T.LlmError):
        T.Context(HParams(2, 64, 6, 4, 32, 96, 50, 1e4, 1e-6), n_ctx=256, host_only=True)


def _pair(T, n_ctx, n_seq, n_batch, n_ubatch, unified=True):
    lib = T.Context(HP, n_ctx=n_ctx, n_seq_max=n_seq, n_batch=n_batch, n_ubatch=n_ubatch,
                    host_only=True, kv_unified=unified)
    lib.debug_capture(True)
    ora = oracle.OracleContext(HP, None, n_ctx=n_ctx, n_seq_max=n_seq, n_batch=n_batch,
                               n_ubatch=n_ubatch, compute=False, kv_unified=unified)
    return lib, ora


def _same_state(lib, ora, n_seq):
    for s in range(n_seq):
        assert lib.seq_pos_max(s) == ora.seq_pos_max(s), s
        assert lib.seq_pos_min(s) == ora.seq_pos_min(s), s
    assert lib.kv_used_cells() == int(np.sum(ora.cells.pos >= 0))


def _decode_both(lib, ora, toks, seqs=None, pos=None, logits=None):
    n_seq_id = None if seqs is None else [len(s) for s in seqs]
    r_lib = lib.decode(toks, pos=pos, seq_ids=seqs, logits=logits)
    r_ora = ora.decode(toks, pos=pos, n_seq_id=n_seq_id, seq_id=seqs, logits=logits)
    assert r_lib == r_ora, (r_lib, r_ora, lib.last_error())
    if r_lib == 0:
        slots = [s for u in ora.last_ubatches for s in u["slots"]]
        assert lib.last_slots().tolist() == slots
        for k, u in enumerate(ora.last_ubatches):
            m = lib.ubatch_mask(k)
            assert m.shape == u["mask"].shape, (m.shape, u["mask"].shape)
            assert np.array_equal(m, u["mask"]), k
        assert lib.n_outputs == ora.n_outputs
    return r_lib


def test_bookkeeping_matches_oracle_scripted(T):
    lib, ora = _pair(T, n_ctx=256, n_seq=4, n_batch=64, n_ubatch=5)
    # interleaved multi-sequence prompt, one ubatch boundary inside each sequence
    toks = list(range(1, 21))
    seqs = [[i % 4] for i in range(20)]
    assert _decode_both(lib, ora, toks, seqs, logits=[1] * 20) == 0
    _same_state(lib, ora, 4)
    # a token shared by two sequences, then per-sequence steps
    assert _decode_both(lib, ora, [7], [[1, 3]]) == 0                 # both continue from 5
    assert _decode_both(lib, ora, [7], [[3]]) == 0
    assert _decode_both(lib, ora, [7], [[1, 3]]) == -1                # seq 3 would not be consecutive
    assert _decode_both(lib, ora, [7, 8, 9, 10], [[0], [1], [2], [3]]) == 0
    _same_state(lib, ora, 4)
    # seq_rm frees cells that are reused lowest-first
    lib.seq_rm(2, 2, -1); ora.seq_rm(2, 2, -1)
    lib.seq_rm(0, -1, 3); ora.seq_rm(0, -1, 3)
    _same_state(lib, ora, 4)
    assert _decode_both(lib, ora, [3, 4, 5], [[2], [2], [1]]) == 0
    _same_state(lib, ora, 4)
    # explicit positions: consecutive ok, gaps rejected
    p = ora.seq_pos_max(3) + 1
    assert _decode_both(lib, ora, [1, 2], [[3], [3]], pos=[p, p + 1]) == 0
    assert _decode_both(lib, ora, [1], [[3]], pos=[p + 5]) == -1
    # invalid batches
    assert _decode_both(lib, ora, [50]) == -1
    assert _decode_both(lib, ora, [1], [[4]]) == -1
    assert _decode_both(lib, ora, list(range(65))) == -1
    # negative logits indices resolve like the oracle's
    assert _decode_both(lib, ora, [1, 2, 3], [[1], [1], [1]], logits=[1, 0, 1]) == 0
    # seq_rm of everything empties the cache
    lib.seq_rm(-1, -1, -1); ora.seq_rm(-1, -1, -1)
    _same_state(lib, ora, 4)
    assert lib.kv_used_cells() == 0


def test_full_cache_returns_1_without_state_change(T):
    lib, ora = _pair(T, n_ctx=256, n_seq=2, n_batch=256, n_ubatch=64)
    assert _decode_both(lib, ora, [1] * 200, [[0]] * 200) == 0
    assert _decode_both(lib, ora, [1] * 57, [[1]] * 57) == 1          # 56 free
    _same_state(lib, ora, 2)
    assert lib.seq_pos_max(1) == -1
    assert _decode_both(lib, ora, [1] * 56, [[1]] * 56) == 0
    assert lib.kv_used_cells() == 256
    assert _decode_both(lib, ora, [1], [[0]]) == 1
    lib.seq_rm(0, 100, -1); ora.seq_rm(0, 100, -1)
    assert _decode_both(lib, ora, [2] * 30, [[1]] * 30) == 0          # reuses cells 100..129
    _same_state(lib, ora, 2)


def test_abort_rolls_back_only_the_current_ubatch(T):
    lib, ora = _pair(T, n_ctx=256, n_seq=2, n_batch=64, n_ubatch=4)
    n = {"lib": 0, "ora": 0}

    def mk(key):
        def cb():
            n[key] += 1
            return n[key] == 3
        return cb
    lib.set_abort_callback(mk("lib"))
    ora.abort_callback = mk("ora")
    assert _decode_both(lib, ora, list(range(10)), [[0]] * 5 + [[1]] * 5) == 2
    _same_state(lib, ora, 2)
    assert lib.seq_pos_max(0) == 4 and lib.seq_pos_max(1) == 2
    lib.set_abort_callback(None)
    ora.abort_callback = None
    assert _decode_both(lib, ora, [5, 6], [[1], [1]]) == 0
    _same_state(lib, ora, 2)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bookkeeping_matches_oracle_randomized(T, seed):
    rng = np.random.default_rng(seed)
    n_seq = 5
    lib, ora = _pair(T, n_ctx=512, n_seq=n_seq, n_batch=48, n_ubatch=int(rng.integers(1, 17)))
    codes = []
    for step in range(80):
        r = rng.random()
        if r < 0.15:
            s = int(rng.integers(-1, n_seq))
            p0 = int(rng.integers(-2, 40))
            p1 = int(rng.integers(-2, 60))
            assert lib.seq_rm(s, p0, p1) == 1
            ora.seq_rm(s, p0, p1)
        else:
            n = int(rng.integers(1, 40))
            seqs = []
            multi = rng.random() < 0.2
            for _ in range(n):
                k = 2 if multi and rng.random() < 0.3 else 1
                seqs.append(sorted(rng.choice(n_seq, size=k, replace=False).tolist()))
            toks = rng.integers(0, HP.n_vocab, size=n).tolist()
            logits = (rng.random(n) < 0.3).astype(int).tolist() if rng.random() < 0.5 else None
            codes.append(_decode_both(lib, ora, toks, seqs, logits=logits))
        _same_state(lib, ora, n_seq)
    # the scenario exercises success, full-cache and invalid-batch paths
    assert codes.count(0) >= 20 and (-1 in codes)


def _defrag_both(lib, ora):
    r_lib = lib.memory_update(True)
    r_ora = ora.memory_update(True)
    assert r_lib == int(r_ora), (r_lib, r_ora)
    return r_lib


def test_defrag_matches_oracle_figure_and_retry(T):
    # the pages' figure: S0P0, S0P1, -, S1P0, S0P2, -, S1P1 -> packed by sequence, then position
    lib, ora = _pair(T, n_ctx=256, n_seq=2, n_batch=64, n_ubatch=64)
    assert _decode_both(lib, ora, [1, 2, 3, 4, 5, 6, 7], [[0], [0], [0], [1], [0], [1], [1]]) == 0
    lib.seq_rm(0, 2, 3); ora.seq_rm(0, 2, 3)         # cell 2
    lib.seq_rm(1, 1, 2); ora.seq_rm(1, 1, 2)         # cell 5
    assert _defrag_both(lib, ora) == 1
    assert _defrag_both(lib, ora) == 0
    _same_state(lib, ora, 2)
    assert _decode_both(lib, ora, [8, 9], [[0], [1]], logits=[1, 1]) == 0
    # no free run: one defrag, then the search again (still 1 when the cache is full)
    lib, ora = _pair(T, n_ctx=256, n_seq=2, n_batch=256, n_ubatch=64)
    assert _decode_both(lib, ora, [1] * 200, [[i % 2] for i in range(200)]) == 0
    lib.seq_rm(0, 50, -1); ora.seq_rm(0, 50, -1)
    assert _decode_both(lib, ora, [1] * 200, [[1]] * 200) == 1
    assert lib.perf()["n_defrags"] == 1
    _same_state(lib, ora, 2)
    assert _decode_both(lib, ora, [1] * 100, [[1]] * 100) == 0
    _same_state(lib, ora, 2)


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_defrag_matches_oracle_randomized(T, seed):
    rng = np.random.default_rng(seed)
    n_seq = 6
    lib, ora = _pair(T, n_ctx=256, n_seq=n_seq, n_batch=64, n_ubatch=int(rng.integers(1, 33)))
    moved = 0
    for step in range(120):
        r = rng.random()
        if r < 0.2:
            s = int(rng.integers(-1, n_seq))
            p0, p1 = int(rng.integers(-2, 30)), int(rng.integers(-2, 60))
            lib.seq_rm(s, p0, p1)
            ora.seq_rm(s, p0, p1)
        elif r < 0.3:
            moved += _defrag_both(lib, ora)
        else:
            n = int(rng.integers(1, 30))
            seqs = []
            for _ in range(n):
                k = 2 if rng.random() < 0.1 else 1
                seqs.append(sorted(rng.choice(n_seq, size=k, replace=False).tolist()))
            toks = rng.integers(0, HP.n_vocab, size=n).tolist()
            _decode_both(lib, ora, toks, seqs, logits=[1] * n)
        _same_state(lib, ora, n_seq)
    assert moved >= 3


def test_split_cache_scripted(T):
    lib, ora = _pair(T, n_ctx=256, n_seq=4, n_batch=64, n_ubatch=6, unified=False)
    assert lib.n_ctx_seq == 64
    seqs = [[i % 4] for i in range(22)] + [[1]] * 5
    assert _decode_both(lib, ora, list(range(1, 28)), seqs, logits=[1] * 27) == 0
    assert [len(u["slots"]) for u in ora.last_ubatches] == [4, 4, 4, 4, 4, 2, 5]
    _same_state(lib, ora, 4)
    assert _decode_both(lib, ora, [1], [[0, 1]]) == -1           # one token, two streams
    assert _decode_both(lib, ora, [1] * 59, [[2]] * 59) == 0       # stream 2: 5 + 59 = 64 cells
    assert _decode_both(lib, ora, [1], [[2]]) == 1                 # full stream
    assert _decode_both(lib, ora, [1], [[3]]) == 0
    lib.seq_rm(2, 3, 10); ora.seq_rm(2, 3, 10)
    assert _defrag_both(lib, ora) == 1
    assert _decode_both(lib, ora, [1] * 7, [[2]] * 7) == 0
    _same_state(lib, ora, 4)


@pytest.mark.parametrize("seed", [6, 7, 8])
def test_split_cache_matches_oracle_randomized(T, seed):
    rng = np.random.default_rng(seed)
    n_seq = 5
    lib, ora = _pair(T, n_ctx=512, n_seq=n_seq, n_batch=64, n_ubatch=int(rng.integers(1, 20)),
                     unified=False)
    codes = []
    for step in range(100):
        r = rng.random()
        if r < 0.15:
            s = int(rng.integers(-1, n_seq))
            p0, p1 = int(rng.integers(-2, 30)), int(rng.integers(-2, 60))
            lib.seq_rm(s, p0, p1)
            ora.seq_rm(s, p0, p1)
        elif r < 0.22:
            _defrag_both(lib, ora)
        else:
            n = int(rng.integers(1, 40))
            seqs = [[int(rng.integers(0, n_seq))] for _ in range(n)]
            if rng.random() < 0.05:
                seqs[0] = [0, 1]
            toks = rng.integers(0, HP.n_vocab, size=n).tolist()
            codes.append(_decode_both(lib, ora, toks, seqs, logits=[1] * n))
        _same_state(lib, ora, n_seq)
    assert codes.count(0) >= 20 and 1 in codes


def test_literal_65536_cell_cache_of_the_32_sequence_workload(T):
    """The 32-sequence workload read literally: 32 prompts of 2048 tokens fill all 65536 cells, so
    the first decode step (one token per sequence) finds no cell and returns 1 with every cell
    holding what it held; seq_rm of the upper half of sequence 0 frees 1024 cells, which 32 steps
    of 32 tokens use up (lowest cells first), and the 33rd step returns 1 again, changing no
    sequence's positions. The failed search is retried once after a defrag, which may move cells
    (the second failure does: the freed cells sit between used ones), so what must stay is each
    sequence's set of positions, and the library's cells must equal the oracle's.
    ("Як це працює", Крок 11-12: no slot for a ubatch -> 1 before any ubatch is committed;
    "デコードループ", KVキャッシュの詳細 (FAILED_PREPARE -> defrag -> retry) and
    エラーリカバリとステートロールバック.)"""

    def content(o):
        return sorted((s, int(o.cells.pos[c])) for c in np.nonzero(o.cells.pos >= 0)[0]
                      for s in np.nonzero(o.cells.seq[c])[0])

    n_seq, n_p = 32, 2048
    lib, ora = _pair(T, n_ctx=65536, n_seq=n_seq, n_batch=2048, n_ubatch=512)
    for s in range(n_seq):
        flags = [0] * (n_p - 1) + [1]
        assert _decode_both(lib, ora, [s + 1] * n_p, [[s]] * n_p, logits=flags) == 0
    assert lib.kv_used_cells() == 65536
    seqs = [[s] for s in range(n_seq)]
    step = [5] * n_seq
    before = content(ora)
    assert _decode_both(lib, ora, step, seqs, logits=[1] * n_seq) == 1
    _same_state(lib, ora, n_seq)
    assert content(ora) == before
    assert all(lib.seq_pos_max(s) == n_p - 1 for s in range(n_seq))
    half = (lib.seq_pos_max(0) + 1) // 2
    assert lib.seq_rm(0, half, -1) == 1 and ora.seq_rm(0, half, -1)
    _same_state(lib, ora, n_seq)
    assert lib.kv_used_cells() == 65536 - 1024
    for i in range(32):
        assert _decode_both(lib, ora, step, seqs, logits=[1] * n_seq) == 0, i
        assert lib.last_slots().min() >= half      # the freed cells of sequence 0, lowest first
    assert lib.kv_used_cells() == 65536
    assert lib.seq_pos_max(0) == half + 31 and lib.seq_pos_max(1) == n_p + 31
    before = content(ora)
    assert _decode_both(lib, ora, step, seqs, logits=[1] * n_seq) == 1
    _same_state(lib, ora, n_seq)
    assert content(ora) == before
    # the library's cells after its defrag are the oracle's, cell by cell: the next batch that
    # fits takes the same slots on both sides
    lib.seq_rm(5, n_p, -1); ora.seq_rm(5, n_p, -1)
    assert _decode_both(lib, ora, [9] * 8, [[5]] * 8) == 0
