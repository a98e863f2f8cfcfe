"""GPU parity of a split KV cache (kv_unified = false: one stream of n_ctx / n_seq_max cells per
sequence, ubatches from split_equal), through the C ABI, against the oracle.

An interleaved four-sequence prompt batch (split_equal takes the tokens out of batch order), then
greedy steps: slots and masks bit-exact, every flagged logits row within 1e-4 (the tiny F32
model's bar) of the oracle's, rows addressed in batch order (also from the end, i < 0), and the
same logits as a unified cache up to float summation order."""
import numpy as np
import pytest

import synthetic as S
from tests import gpu_common as G

pytestmark = pytest.mark.gpu
KEY = "tiny_f32_8seq"
N_SEQ, N_PROMPT, TOL = 4, 24, 1e-4


def _batch():
    w = S.WORKLOADS[KEY]
    toks = np.concatenate([S.prompt_tokens(w.prompt_seed_of(s), N_PROMPT, w.hp.n_vocab).numpy()
                           for s in range(N_SEQ)])
    seqs = [[s] for s in range(N_SEQ) for _ in range(N_PROMPT)]
    order = np.argsort(np.tile(np.arange(N_PROMPT), N_SEQ), kind="stable")   # interleave
    toks, seqs = toks[order], [seqs[i] for i in order]
    flags = np.zeros(len(toks), dtype=np.int8)
    flags[::5] = 1
    flags[-N_SEQ:] = 1
    return toks, seqs, flags


def test_split_cache_prompt_and_greedy_steps():
    kw = dict(n_seq_max=N_SEQ, n_ubatch=16)
    lib = G.library_ctx(KEY, kv_unified=False, **kw)
    uni = G.library_ctx(KEY, **kw)
    ora = G.oracle_ctx(KEY, kv_unified=False, **kw)
    assert lib.n_ctx_seq == lib.n_ctx // N_SEQ
    lib.debug_capture(True)
    toks, seqs, flags = _batch()
    assert lib.decode(toks, seq_ids=seqs, logits=flags) == 0, lib.last_error()
    assert uni.decode(toks, seq_ids=seqs, logits=flags) == 0
    assert ora.decode(toks, seq_id=seqs, n_seq_id=[1] * len(toks), logits=flags) == 0
    assert lib.last_slots().tolist() == [s for u in ora.last_ubatches for s in u["slots"]]
    for k, u in enumerate(ora.last_ubatches):
        assert np.array_equal(lib.ubatch_mask(k), u["mask"]), k
    assert lib.n_outputs == ora.n_outputs == int(flags.sum())
    for i in list(np.nonzero(flags)[0]) + [-1, -2, -int(flags.sum())]:
        g, o, u = lib.get_logits_ith(int(i)), ora.get_logits_ith(int(i)), uni.get_logits_ith(int(i))
        assert G.rel_err(g, o) <= TOL, i
        assert G.rel_err(g, u.astype(np.float64)) <= 1e-5, i
        assert lib.get_argmax_ith(int(i)) == int(np.argmax(g)), i
    lib.debug_capture(False)
    rows = [len(toks) - N_SEQ + s for s in range(N_SEQ)]
    nxt_rows = [i for i in rows]
    rep = G.greedy_compare(lib, ora, N_SEQ, nxt_rows, 8, TOL, {})
    assert rep["tokens_checked"] >= 16
    for c in (lib, uni):
        c.free()
