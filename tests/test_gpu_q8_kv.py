"""GPU parity of the Q8_0 KV cache (type_k = type_v = Q8_0), through the C ABI, against the oracle.

  - The quantiser, bit-exact: the float32 K/V rows the library handed to its cache write (the
    debug capture) quantised by the oracle give exactly the library's stored blocks (scale bits
    and quants), on the prompt path (one block per prompt token) and the one-token decode path.
  - Whole runs on the tiny model (one sequence, and eight sequences batched): logits within a max
    relative error of 1e-3 per row, greedy tokens equal where the oracle's top-2 gap exceeds 1e-3.
    The bar is wider than the F16 cache's 1e-4 because the two sides quantise K/V rows computed
    in different precisions (float32 here, float64 in the oracle): a value whose product lies
    within rounding of a half-integer lands one quantisation step (max|x| / 127 of its block)
    apart, which moves a logit by far more than float32 rounding does.
  - The f16 copy of the quants the tensor-core prefill tiles read (they apply the scales): every
    used cell's int8 quants, bit-exact.
  - The Llama-3-8B shape (head_dim 128) at full size: layers checked one by one on the library's
    own inputs and dequantised cache (the F16 path's 2e-2 bar).
"""
import numpy as np
import pytest

import oracle
import synthetic as S
from oracle.formats import Q8_0, q8_0_to_f64, quantize_q8_0
from tests import gpu_common as G

pytestmark = pytest.mark.gpu
TOL = 1e-3


def _check_blocks(ctx, T, slots):
    hp = ctx._hp
    Hkv, hd = hp.n_head_kv, hp.head_dim
    for il in range(hp.n_layer):
        for which, name in ((0, "k_in"), (1, "v_in")):
            rows = ctx.debug_tensor(name, il)
            assert rows is not None and rows.size == T * Hkv * hd
            want = quantize_q8_0(rows.reshape(T, Hkv, hd).astype(np.float64))
            got = ctx.kv_cache(il, which)[:, slots, :].transpose(1, 0, 2)
            assert got.shape == want.shape
            bad = np.argwhere(got != want)
            assert bad.size == 0, (il, name, bad[:5])


def test_quantiser_bit_exact_on_the_library_rows():
    key = "tiny_f32_1seq"
    ctx = G.library_ctx(key, type_k=Q8_0, type_v=Q8_0)
    ctx.debug_capture(True)
    toks = G.prompts(key)[0]
    assert ctx.decode(toks) == 0, ctx.last_error()
    _check_blocks(ctx, len(toks), ctx.last_slots())
    assert ctx.decode([int(ctx.get_argmax_ith(-1))]) == 0, ctx.last_error()
    _check_blocks(ctx, 1, ctx.last_slots())
    ctx.free()


def test_tiny_1seq_q8_0_cache_prompt_and_greedy_steps():
    key = "tiny_f32_1seq"
    w = S.WORKLOADS[key]
    ctx = G.library_ctx(key, type_k=Q8_0, type_v=Q8_0)
    ora = G.oracle_ctx(key, type_k=Q8_0, type_v=Q8_0)
    toks = G.prompts(key)[0]
    assert ctx.decode(toks) == 0, ctx.last_error()
    assert ora.decode(toks) == 0
    rep = G.greedy_compare(ctx, ora, 1, [w.n_prompt - 1], w.n_decode, TOL, {})
    print("tiny Q8_0 cache:", rep)
    assert rep["tokens_checked"] >= w.n_decode // 2
    ctx.free()


def test_tiny_8seq_q8_0_cache_batched():
    key = "tiny_f32_8seq"
    w = S.WORKLOADS[key]
    ctx = G.library_ctx(key, type_k=Q8_0, type_v=Q8_0)
    ora = G.oracle_ctx(key, type_k=Q8_0, type_v=Q8_0)
    toks, seqs, flags = G.prompt_batch(key)
    assert ctx.decode(toks, seq_ids=seqs, logits=flags) == 0, ctx.last_error()
    assert ora.decode(toks, seq_id=seqs, n_seq_id=[1] * len(toks), logits=flags) == 0
    rows = [(s + 1) * w.n_prompt - 1 for s in range(w.n_seq)]
    rep = G.greedy_compare(ctx, ora, w.n_seq, rows, 16, TOL, {})
    print("tiny 8-seq Q8_0 cache:", rep)
    assert rep["tokens_checked"] >= 50
    ctx.free()


def test_prefill_tiles_read_the_exact_quants():
    key = "tiny_f32_8seq"
    ctx = G.library_ctx(key, type_k=Q8_0, type_v=Q8_0)
    hp = ctx._hp
    Hkv, hd = hp.n_head_kv, hp.head_dim
    toks, seqs, flags = G.prompt_batch(key)
    assert ctx.decode(toks, seq_ids=seqs, logits=flags) == 0, ctx.last_error()
    used = np.unique(ctx.last_slots())
    for which in (0, 1):
        blocks = ctx.kv_cache(hp.n_layer - 1, which)            # the copy holds the last layer
        q = blocks.reshape(Hkv, -1, hd // 32, 34)[:, :, :, 2:].view(np.int8).reshape(Hkv, -1, hd)
        got = ctx.kv_f16_copy(which)[:, used]
        assert np.array_equal(got.astype(np.float64), q[:, used].astype(np.float64)), which
    ctx.free()


@pytest.mark.slow
def test_llama8b_shape_q8_0_cache_layerwise():
    key = "llama8b_bf16_1seq"
    w = S.WORKLOADS[key]
    hp, d = w.hp, w.hp.n_embd
    Hkv, hd = hp.n_head_kv, hp.head_dim
    ctx = G.library_ctx(key, type_k=Q8_0, type_v=Q8_0)
    ow = G.oracle_weights(key, cache=False)
    mirror = oracle.OracleContext(hp, None, n_ctx=w.n_ctx, type_k=Q8_0, type_v=Q8_0,
                                  n_batch=w.n_batch, n_ubatch=w.n_ubatch, compute=False)
    toks = G.prompts(key)[0]

    def cache(il):
        out = []
        for which in (0, 1):
            b = ctx.kv_cache(il, which)
            out.append(q8_0_to_f64(b.reshape(-1, hd // 32 * 34), hd).reshape(Hkv, -1, hd))
        return out

    def check(rows, pos, tag):
        slots = ctx.last_slots()
        vis = mirror.cells.mask(pos, [[0]] * len(pos), mirror.cells.n_kv())
        for il in (0, 1, hp.n_layer - 1):
            x_in, x_out = G.captured_rows(ctx, il, rows)
            kc, vc = cache(il)
            e = G.layer_check(ow, hp, il, x_in, x_out, pos, slots[rows], vis, kc, vc, Q8_0)
            print(tag, il, e)
            assert max(e.values()) <= 2e-2, (tag, il, e)

    ctx.debug_capture(True)
    assert ctx.decode(toks) == 0, ctx.last_error()
    assert mirror.decode(toks) == 0
    rows = [0, 255, 511]
    check(rows, np.array(rows), "prompt")
    x_last = ctx.debug_tensor("l_out", hp.n_layer - 1).reshape(-1, d)[[w.n_prompt - 1]]
    lc = G.logits_check(ow, hp, x_last, [ctx.get_logits_ith(-1)], [ctx.get_argmax_ith(-1)])
    assert lc["logits"] <= 2e-2, lc
    tok = ctx.get_argmax_ith(-1)
    assert ctx.decode([tok]) == 0, ctx.last_error()
    assert mirror.decode([tok]) == 0
    check([0], np.array([w.n_prompt]), "decode")
    ctx.free()
