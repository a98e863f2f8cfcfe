"""Pins of the oracle's building blocks against numbers the pages print and closed forms.

Each test fixes one fact that a plausible mistake in the oracle (a dropped term, a wrong sign or
index, a transposed operand) would break."""
import math
import os

import numpy as np
import pytest

import oracle
import synthetic as S
from oracle import formats as OF
from oracle.memory import derive_cparams, split_simple

GOLD = {}
with open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.txt")) as f:
    for line in f:
        line = line.split("#")[0].strip()
        if line:
            k, v = [s.strip() for s in line.split("=")]
            GOLD[k] = v

MiB = 1024.0 * 1024.0


def g(k):
    return float(GOLD[k])


# ---------------------------------------------------------------- sizes, layouts, parameters
def test_row_bytes_match_page_example_2():
    assert OF.type_row_bytes(OF.F32, 256) * 704 == int(g("row_bytes_ffn_gate_f32"))
    assert OF.type_row_bytes(OF.F16, 256) * 704 == int(g("row_bytes_ffn_gate_f16"))
    assert OF.type_row_bytes(OF.Q8_0, 256) == int(g("nb1_ffn_gate_q8_0"))
    assert OF.type_row_bytes(OF.Q8_0, 256) * 704 == int(g("row_bytes_ffn_gate_q8_0"))
    # the synthetic generator packs exactly that many bytes
    q = S.weight_bytes(7, "blk.0.ffn_gate.weight", (256, 704), S.Q8_0)
    assert q.numel() == int(g("row_bytes_ffn_gate_q8_0"))


def test_row_major_orientation_matches_stride_example():
    # ne = {4, 3}: 3 rows of 4 floats; element (i0=2, i1=1) is row 1, column 2 -> byte 24 = 6.0
    m = np.arange(12, dtype=np.float32)
    w = OF.decode_weight(m.view(np.uint8), OF.F32, 4)
    assert w.shape == (3, 4)
    assert (1 * 4 + 2) * 4 == int(g("stride_example_byte"))
    assert w[1, 2] == g("stride_example_value")


def test_tiny_model_parameter_count_and_size():
    specs = S.tensor_specs(S.TINY)
    assert len(specs) == int(g("tiny_n_tensors"))
    n = sum(int(np.prod(s)) for _, s in specs)
    assert round(n / 1e6, 2) == g("tiny_model_params_M")
    assert round(n * 4 / MiB, 2) == g("tiny_file_size_MiB")
    hp = S.TINY
    assert hp.n_embd // hp.n_head == int(g("tiny_n_embd_head_k"))
    assert hp.n_head // hp.n_head_kv == int(g("tiny_n_gqa"))
    assert hp.head_dim * hp.n_head_kv == int(g("tiny_n_embd_k_gqa"))


def test_bytes_and_flops_per_token_match_example_13():
    # weights read by one decode step: every weight except the embedding table (one row lookup)
    specs = dict(S.tensor_specs(S.TINY))
    n_read = sum(int(np.prod(s)) for k, s in specs.items() if k != "token_embd.weight")
    assert round(n_read * 4 / 1e6, 1) == g("decode_weight_MB_per_token")
    # matmul FLOPs of a prompt token (no logits): 2 x the layer weights incl. norms, as printed
    n_layers = sum(int(np.prod(s)) for k, s in specs.items() if k.startswith("blk.")) + 256
    assert round(2 * n_layers / 1e6, 2) == g("prompt_MFLOP_per_token")


def test_kv_and_output_buffer_sizes_match_example_10():
    hp = S.TINY
    n_ctx = 4096
    k_f16 = hp.n_layer * OF.type_row_bytes(OF.F16, hp.n_head_kv * hp.head_dim) * n_ctx
    assert round(k_f16 / MiB, 2) == g("kv_f16_K_MiB_4096")
    assert round(2 * k_f16 / MiB, 2) == g("kv_f16_total_MiB_4096")
    k_q8 = hp.n_layer * (hp.n_head_kv * hp.head_dim * n_ctx) // 32 * 34
    assert round(k_q8 / MiB, 2) == g("kv_q8_0_K_MiB_4096")
    row = hp.n_vocab * 4
    assert round(row / MiB, 2) == g("output_buffer_1seq_MiB")
    assert round(4 * row / MiB, 2) == g("output_buffer_4seq_MiB")
    assert round(512 * row / MiB, 2) == g("logits_ubatch_512_MiB")
    assert round(128 * row / MiB, 2) == g("logits_ubatch_128_MiB")
    assert round(32 * row / MiB, 2) == g("logits_ubatch_32_MiB")


def test_context_parameters_and_ubatch_counts():
    assert derive_cparams(4096, 2048, 512, 1) == (int(g("ctx_n_ctx")), int(g("ctx_n_batch")),
                                                  int(g("ctx_n_ubatch")))
    assert derive_cparams(100, 2048, 512, 1) == (256, 256, 256)      # pad to 256, clamp batch
    assert derive_cparams(4097, 8192, 512, 1) == (4352, 4352, 512)
    assert derive_cparams(8320, 8192, 512, 1)[0] == 8448
    assert derive_cparams(512, 64, 512, 1) == (512, 64, 64)          # ubatch <= batch
    assert derive_cparams(512, 64, 512, 0) is None
    assert len(split_simple(2000, 512)) == int(g("prompt_2000_ubatches_at_512"))
    assert len(split_simple(512, 128)) == int(g("batch_512_ubatches_at_128"))
    assert [len(r) for r in split_simple(2000, 512)] == [512, 512, 512, 464]


# ---------------------------------------------------------------- storage formats
def test_q8_0_block_decodes_to_scale_times_quant():
    d = np.float16(0.5)
    q = np.array([i - 16 for i in range(32)], dtype=np.int8)
    q[0], q[31] = -127, 127
    block = np.concatenate([np.frombuffer(d.tobytes(), np.uint8), q.view(np.uint8)])
    assert block.nbytes == 34 and block[:2].tobytes() == b"\x00\x38"       # fp16 0.5 = 0x3800
    w = OF.decode_weight(np.stack([block, block]), OF.Q8_0, 32)
    assert w.shape == (2, 32)
    assert w[0, 0] == -63.5 and w[0, 31] == 63.5 and w[1, 16] == 0.0 and w[1, 17] == 0.5


def test_bf16_decode_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000], dtype=np.uint16)
    v = OF.bf16_to_f64(bits)
    assert list(v[:3]) == [1.0, -2.0, 1.0078125] and v[3] == 0.0 and np.signbit(v[4])


def test_cache_rounding_is_round_to_nearest_even():
    # 1 + 2^-11 lies halfway between fp16 1.0 and 1 + 2^-10: ties go to the even 1.0
    x = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 65504.0, 1e-8])
    r = OF.round_to_type(x, OF.F16)
    assert list(r[:3]) == [1.0, 1 + 2 ** -9, 65504.0]
    assert OF.round_to_type(np.array([1 + 2 ** -30]), OF.F32)[0] == 1.0


# ---------------------------------------------------------------- per-token math
def test_rms_norm_closed_form():
    eps = 1e-6
    x = np.full((1, 8), 3.0)
    y = oracle.rms_norm(x, np.ones(8), eps)
    assert np.allclose(y, 3.0 / math.sqrt(9.0 + eps), rtol=0, atol=1e-15)
    # a gain scales each element; the norm is invariant to scaling x (up to eps)
    gain = np.arange(1, 9, dtype=np.float64)
    x = np.array([[1.0, -2.0, 3.0, -4.0, 5.0, -6.0, 7.0, -8.0]])
    rms = math.sqrt(sum(v * v for v in x[0]) / 8)
    assert np.allclose(oracle.rms_norm(x, gain, 0.0), x / rms * gain, rtol=1e-15)
    assert np.allclose(oracle.rms_norm(1000 * x, gain, 0.0), oracle.rms_norm(x, gain, 0.0))
    assert np.all(oracle.rms_norm(np.zeros((1, 4)), np.ones(4), eps) == 0)


def test_rope_pairs_and_frequencies():
    hd, base = 4, 10000.0
    # position 0 is the identity
    x = np.random.default_rng(0).standard_normal((3, 2, hd))
    assert np.array_equal(oracle.rope(x, np.zeros(3, dtype=int), base), x)
    # pair 0 (elements 0 and 1) turns by pos radians
    e0 = np.zeros((1, 1, hd)); e0[0, 0, 0] = 1.0
    y = oracle.rope(e0, np.array([2]), base)[0, 0]
    assert np.allclose(y, [math.cos(2), math.sin(2), 0, 0], atol=1e-15)
    # pair 1 (elements 2 and 3) turns by pos * base^(-2/hd) = pos / 100 radians
    e2 = np.zeros((1, 1, hd)); e2[0, 0, 3] = 1.0
    y = oracle.rope(e2, np.array([100]), base)[0, 0]
    assert np.allclose(y, [0, 0, -math.sin(1.0), math.cos(1.0)], atol=1e-12)


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(1)
    hd = 32
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))
    y = oracle.rope(q, np.array([77]), 500000.0)
    assert np.allclose(y[..., 0::2] ** 2 + y[..., 1::2] ** 2, q[..., 0::2] ** 2 + q[..., 1::2] ** 2)
    # q(m) . k(n) depends only on m - n
    def dot(m, n):
        return float(np.sum(oracle.rope(q, np.array([m]), 10000.0) * oracle.rope(k, np.array([n]), 10000.0)))
    assert dot(10, 3) == pytest.approx(dot(107, 100), rel=1e-12, abs=1e-12)
    assert dot(5, 5) == pytest.approx(float(np.sum(q * k)), rel=1e-12)


def test_softmax_rows_sum_to_one_and_masked_get_zero():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((5, 9)) * 30
    vis = rng.random((5, 9)) > 0.4
    vis[:, 0] = True
    p = oracle.numerics.softmax_masked(s, vis)
    assert np.all(np.abs(p.sum(-1) - 1) < 1e-12)
    assert np.all(p[~vis] == 0.0)
    one = np.zeros((1, 9), dtype=bool); one[0, 4] = True
    assert oracle.numerics.softmax_masked(s[:1], one)[0, 4] == 1.0


def test_attention_special_cases_and_gqa_mapping():
    rng = np.random.default_rng(3)
    T, H, Hkv, hd, C = 3, 4, 2, 8, 6
    k = rng.standard_normal((C, Hkv, hd))
    v = rng.standard_normal((C, Hkv, hd))
    vis = np.tril(np.ones((T, C), dtype=bool), k=C - T)
    # zero queries: all scores equal -> the plain mean of the visible value rows
    o = oracle.attention(np.zeros((T, H, hd)), k, v, vis, Hkv).reshape(T, H, hd)
    for t in range(T):
        for h in range(H):
            cells = [c for c in range(C) if vis[t, c]]
            assert np.allclose(o[t, h], sum(v[c, h // 2] for c in cells) / len(cells))
    # one visible cell -> exactly that value row; heads 0,1 read KV head 0 and heads 2,3 KV head 1
    one = np.zeros((T, C), dtype=bool); one[:, 2] = True
    o = oracle.attention(rng.standard_normal((T, H, hd)), k, v, one, Hkv).reshape(T, H, hd)
    assert np.allclose(o[:, 0], v[2, 0]) and np.allclose(o[:, 1], v[2, 0])
    assert np.allclose(o[:, 2], v[2, 1]) and np.allclose(o[:, 3], v[2, 1])
    # a large score on one cell selects it (scale 1/sqrt(hd) applied: a 1e3 gap still dominates)
    q = np.zeros((1, H, hd)); q[0, :, 0] = 1.0
    kk = np.zeros((C, Hkv, hd)); kk[4, :, 0] = 1e3
    o = oracle.attention(q, kk, v, np.ones((1, C), dtype=bool), Hkv).reshape(1, H, hd)
    assert np.allclose(o[0, 0], v[4, 0])
    # the scale is 1/sqrt(hd): two cells with key gap delta get weights in ratio exp(delta/sqrt(hd))
    kk = np.zeros((2, Hkv, hd)); kk[0, :, 0] = 2.0
    vv = np.zeros((2, Hkv, hd)); vv[0, :, 0] = 1.0
    o = oracle.attention(q, kk, vv, np.ones((1, 2), dtype=bool), Hkv).reshape(1, H, hd)
    w0 = math.exp(2.0 / math.sqrt(hd)) / (math.exp(2.0 / math.sqrt(hd)) + 1.0)
    assert o[0, 0, 0] == pytest.approx(w0, rel=1e-14)


def test_silu_and_swiglu_values():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.silu(np.array([1.0]))[0] == pytest.approx(0.7310585786300049, rel=1e-15)
    assert oracle.silu(np.array([-1.0]))[0] == pytest.approx(-0.2689414213699951, rel=1e-15)
    assert oracle.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    # the gate is the first operand: silu(gate) * up
    assert oracle.swiglu(np.array([0.0]), np.array([5.0]))[0] == 0.0
    assert oracle.swiglu(np.array([1.0]), np.array([2.0]))[0] == pytest.approx(2 * 0.7310585786300049)


def test_linear_orientation():
    # weight {K=3, M=2}: two rows of three values; y[m] = sum_k w[m][k] x[k]
    w = np.array([[1.0, 2.0, 3.0], [0.0, -1.0, 4.0]])
    x = np.array([[1.0, 1.0, 2.0]])
    assert oracle.linear(x, w).tolist() == [[9.0, 7.0]]
