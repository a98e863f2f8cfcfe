"""GPU parity of the decode path on the tiny-model workloads, through the C ABI, against the oracle.

Bar: logits within a max relative error of 1e-4 per row (F32 weights; the F16 KV cache is rounded
identically on both sides); greedy tokens equal wherever the oracle's top-2 gap exceeds 1e-3;
KV slot indices and attention masks bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from oracle.context import forward_layers
from oracle.formats import round_to_type
from tests import gpu_common as G

pytestmark = pytest.mark.gpu
TOL = 1e-4


def test_generator_is_device_independent():
    for name, shape, wt in (("blk.0.attn_q.weight", (256, 256), S.BF16),
                            ("blk.1.ffn_gate.weight", (256, 704), S.Q8_0),
                            ("output.weight", (256, 4096), S.F32)):
        a = S.weight_bytes(77, name, shape, wt, "cpu")
        b = S.weight_bytes(77, name, shape, wt, "cuda").cpu()
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    assert torch.equal(S.prompt_tokens(5, 999, 151936, "cpu"), S.prompt_tokens(5, 999, 151936, "cuda").cpu())


def test_tiny_1seq_prompt_and_32_greedy_steps():
    key = "tiny_f32_1seq"
    w = S.WORKLOADS[key]
    ctx, ora = G.library_ctx(key), G.oracle_ctx(key)
    toks = G.prompts(key)[0]
    assert ctx.decode(toks) == 0, ctx.last_error()
    assert ora.decode(toks) == 0
    assert ctx.last_slots().tolist() == list(range(w.n_prompt))
    rep = G.greedy_compare(ctx, ora, 1, [w.n_prompt - 1], w.n_decode, TOL, {})
    assert rep["tokens_checked"] >= w.n_decode // 2
    assert ctx.seq_pos_max(0) == w.n_prompt + w.n_decode - 1
    ctx.free()


def test_tiny_8seq_batched_prompt_and_greedy_steps():
    key = "tiny_f32_8seq"
    w = S.WORKLOADS[key]
    ctx, ora = G.library_ctx(key), G.oracle_ctx(key)
    ctx.debug_capture(True)
    toks, seqs, flags = G.prompt_batch(key)
    assert ctx.decode(toks, seq_ids=seqs, logits=flags) == 0, ctx.last_error()
    assert ora.decode(toks, seq_id=seqs, n_seq_id=[1] * len(toks), logits=flags) == 0
    assert ctx.n_outputs == w.n_seq
    slots = [s for u in ora.last_ubatches for s in u["slots"]]
    assert ctx.last_slots().tolist() == slots
    for k, u in enumerate(ora.last_ubatches):
        assert np.array_equal(ctx.ubatch_mask(k), u["mask"]), k
    rows = [(s + 1) * w.n_prompt - 1 for s in range(w.n_seq)]
    # the workload's whole run: 128 greedy steps of one token per sequence
    rep = G.greedy_compare(ctx, ora, w.n_seq, rows, w.n_decode, TOL, {})
    assert rep["tokens_checked"] >= 400
    assert all(ctx.seq_pos_max(s) == w.n_prompt + w.n_decode - 1 for s in range(w.n_seq))
    ctx.free()


def test_tiny_layer_outputs_match_oracle_layer_by_layer():
    key = "tiny_f32_1seq"
    w = S.WORKLOADS[key]
    hp = w.hp
    ctx = G.library_ctx(key)
    ctx.debug_capture(True)
    toks = G.prompts(key)[0][:20]
    assert ctx.decode(toks, logits=[1] * 20) == 0
    ow = G.oracle_weights(key)
    pos = np.arange(20)
    causal = np.tril(np.ones((20, 20), dtype=bool))
    x = ow.rows("token_embd.weight", toks)
    got = ctx.debug_tensor("embd").reshape(20, hp.n_embd)
    assert np.max(np.abs(got - x)) == 0.0
    for il in range(hp.n_layer):
        store = {}

        def kv_write(_il, k, v):
            store["kv"] = (round_to_type(k, w.type_kv), round_to_type(v, w.type_kv))

        def kv_read(_il):
            return store["kv"][0], store["kv"][1], causal
        x = forward_layers(ow, hp, x, pos, kv_write, kv_read, layers=[il])
        got = ctx.debug_tensor("l_out", il).reshape(20, hp.n_embd)
        e = np.max(np.abs(got - x)) / np.max(np.abs(x))
        assert e < 1e-5, (il, e)
    ctx.free()


def test_ubatch_split_and_sequence_isolation_on_gpu():
    key = "tiny_f32_8seq"
    w = S.WORKLOADS[key]
    toks, seqs, flags = G.prompt_batch(key)
    n = 2 * w.n_prompt
    ref = None
    for nub in (128, 37, 5):
        ctx = G.library_ctx(key, n_ubatch=nub)
        assert ctx.decode(toks[:n], seq_ids=seqs[:n], logits=[1] * n) == 0
        out = np.stack([ctx.get_logits_ith(i) for i in range(n)])
        if ref is None:
            ref = out
        else:
            assert np.max(np.abs(out - ref)) / np.max(np.abs(ref)) < TOL, nub
        ctx.free()
    # sequence 1 alone gives the same logits as inside the batch
    ctx = G.library_ctx(key)
    p1 = G.prompts(key)[1]
    assert ctx.decode(p1, logits=[1] * w.n_prompt) == 0
    alone = np.stack([ctx.get_logits_ith(i) for i in range(w.n_prompt)])
    assert np.max(np.abs(alone - ref[w.n_prompt:])) / np.max(np.abs(ref)) < TOL
    ctx.free()


def test_error_paths_on_gpu():
    key = "tiny_f32_1seq"
    ctx = G.library_ctx(key, n_ctx=256, n_batch=256, n_ubatch=16)
    toks = G.prompts(key)[0]
    # a bad cell index planted for ubatch 1: the kernel's bounds check reports it, -3, rollback
    ctx.inject_fault(1, 1)
    assert ctx.decode(toks) == -3
    assert ctx.seq_pos_max(0) == 15 and ctx.kv_used_cells() == 16
    assert ctx.get_logits_ith(-1) is None
    # the cache still works and continues from the kept ubatch
    assert ctx.decode(toks[16:]) == 0, ctx.last_error()
    ref = G.library_ctx(key, n_ctx=256, n_batch=256, n_ubatch=16)
    assert ref.decode(toks) == 0
    assert G.rel_err(ctx.get_logits_ith(-1), ref.get_logits_ith(-1).astype(np.float64)) < 1e-6
    # the same bounds check inside the fused decode-step kernels
    p = ctx.seq_pos_max(0)
    ctx.inject_fault(1, 0)
    assert ctx.decode([7]) == -3
    assert ctx.seq_pos_max(0) == p
    assert ctx.decode([7]) == 0 and ctx.seq_pos_max(0) == p + 1
    # abort before the second ubatch
    calls = []
    ref.set_abort_callback(lambda: (calls.append(1), len(calls) == 2)[1])
    assert ref.decode(toks[:20]) == 2
    assert ref.seq_pos_max(0) == 31 + 16
    ref.set_abort_callback(None)
    # a batch within n_batch that the cache cannot hold returns 1 and changes nothing
    used = ref.kv_used_cells()
    pmax = ref.seq_pos_max(0)
    assert ref.decode(np.zeros(256 - used + 1, dtype=np.int32)) == 1, ref.last_error()
    assert ref.kv_used_cells() == used and ref.seq_pos_max(0) == pmax
    assert ref.get_logits_ith(-1) is None
    assert ref.decode(np.zeros(256 - used, dtype=np.int32)) == 0      # exactly the free cells fit
    ctx.free(); ref.free()


@pytest.mark.parametrize("n_prompt", [1000, 2000, 2044, 3500])
@pytest.mark.parametrize("tkv", [oracle.F16, oracle.Q8_0])
def test_tiny_long_context_decode(tkv, n_prompt):
    """A long prompt then greedy steps, against the oracle; F16 and Q8_0 caches. The decode
    attention's 16 blocks per KV head take slices of about 63 and 125 cells (one and two passes
    of 64 cells); from 2048 cells on, two clusters of 16 share each KV head's list and merge
    through global partial rows: 2044 crosses that bound between the third and fourth step,
    3500 takes slices of about 110 cells."""
    key = "tiny_f32_1seq"
    over = dict(n_ctx=4096, n_batch=4096, n_ubatch=512, type_k=tkv, type_v=tkv)
    ctx, ora = G.library_ctx(key, **over), G.oracle_ctx(key, **over)
    toks = S.prompt_tokens(4242, n_prompt, S.WORKLOADS[key].hp.n_vocab).numpy()
    assert ctx.decode(toks) == 0, ctx.last_error()
    assert ora.decode(toks) == 0
    tol = TOL if tkv == oracle.F16 else 1e-3
    rep = G.greedy_compare(ctx, ora, 1, [len(toks) - 1], 6, tol, {})
    print("long context", tkv, rep)
    ctx.free()


@pytest.mark.parametrize("n_seq", [16, 48])
def test_tiny_many_sequence_decode_steps(n_seq):
    """Decode steps with one token for each of 16 or 48 sequences in one ubatch: the tensor-core
    decode attention runs with clusters of 4 and of 1 block per (token, KV head)."""
    key = "tiny_f32_8seq"
    w = S.WORKLOADS[key]
    over = dict(n_seq_max=n_seq, n_ctx=4096, n_batch=1024, n_ubatch=512)
    ctx, ora = G.library_ctx(key, **over), G.oracle_ctx(key, **over)
    n_p = 20
    toks = np.concatenate([S.prompt_tokens(900 + s, n_p, w.hp.n_vocab).numpy() for s in range(n_seq)])
    seqs = [[s] for s in range(n_seq) for _ in range(n_p)]
    flags = np.zeros(len(toks), dtype=np.int8)
    flags[[(s + 1) * n_p - 1 for s in range(n_seq)]] = 1
    assert ctx.decode(toks, seq_ids=seqs, logits=flags) == 0, ctx.last_error()
    assert ora.decode(toks, seq_id=seqs, n_seq_id=[1] * len(toks), logits=flags) == 0
    rows = [(s + 1) * n_p - 1 for s in range(n_seq)]
    rep = G.greedy_compare(ctx, ora, n_seq, rows, 3, TOL, {})
    assert rep["tokens_checked"] >= n_seq
    ctx.free()


def test_tiny_many_long_sequences_decode_steps():
    """16 sequences of 520 cells: clusters of 4 blocks per (token, KV head), each block walking 3
    passes of 64 cells."""
    key = "tiny_f32_8seq"
    w = S.WORKLOADS[key]
    n_seq, n_p = 16, 520
    over = dict(n_seq_max=n_seq, n_ctx=8448, n_batch=1024, n_ubatch=512)
    ctx, ora = G.library_ctx(key, **over), G.oracle_ctx(key, **over)
    for s in range(n_seq):
        toks = S.prompt_tokens(700 + s, n_p, w.hp.n_vocab).numpy()
        flags = np.zeros(n_p, dtype=np.int8)
        flags[-1] = 1
        assert ctx.decode(toks, seq_ids=[[s]] * n_p, logits=flags) == 0, ctx.last_error()
        assert ora.decode(toks, seq_id=[[s]] * n_p, n_seq_id=[1] * n_p, logits=flags) == 0
    # the last call's output row is sequence 15's; run one step of all sequences to compare
    nxt = [int(ctx.get_argmax_ith(-1))] * n_seq
    seqs = [[s] for s in range(n_seq)]
    assert ctx.decode(nxt, seq_ids=seqs, logits=[1] * n_seq) == 0, ctx.last_error()
    assert ora.decode(nxt, seq_id=seqs, n_seq_id=[1] * n_seq, logits=[1] * n_seq) == 0
    rep = G.greedy_compare(ctx, ora, n_seq, list(range(n_seq)), 2, TOL, {})
    assert rep["tokens_checked"] >= n_seq
    ctx.free()
