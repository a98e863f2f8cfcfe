"""Pins of the oracle's Q8_0 cache quantiser (oracle.formats.quantize_q8_0) and of a Q8_0 KV cache
in the oracle context.

What fixes them: the block layout and sizes the pages print ([P2] Example 2: 32 values in 34
bytes, scale first; Memory Math: a q8_0 cache of the tiny model is 1.06 MiB for K), hand-worked
values of a symmetric absmax block, the half-step error bound of rounding to a grid, the
idempotence of quantising values that already lie on the grid, and cached decoding matching the
no-cache forward with the same cache type."""
import numpy as np
import pytest

import oracle
import synthetic as S
from oracle import formats as OF
from oracle.context import forward_no_cache
from synthetic.configs import HParams
from tests.helpers import oracle_weights


def qd(raw):
    """(d as float64, q as int array) of Q8_0 blocks."""
    b = raw.reshape(-1, 34)
    d = np.ascontiguousarray(b[:, :2]).view(np.float16)[:, 0].astype(np.float64)
    return d, np.ascontiguousarray(b[:, 2:]).view(np.int8).astype(np.int64)


def test_block_layout_and_printed_sizes():
    x = np.random.default_rng(1).normal(size=(3, 256))
    raw = OF.quantize_q8_0(x)
    assert raw.shape == (3, 272) and raw.dtype == np.uint8         # ffn_gate row: nb[1] = 272
    # the whole ffn_gate {256, 704} of the tiny model: nb[2] = bytes = 191488
    assert OF.quantize_q8_0(np.zeros((704, 256))).nbytes == 191488
    assert OF.type_row_bytes(OF.Q8_0, 256) * 704 == 191488
    # tiny model: 4 layers x 64 values x 4096 cells -> "K (q8_0): 1.06 MiB"
    per_layer = OF.quantize_q8_0(np.zeros((4096, 64))).nbytes
    assert per_layer == 4096 * 64 // 32 * 34
    assert round(4 * per_layer / 2 ** 20, 2) == 1.06
    # the scale comes first, fp16 little-endian: 1.0 is 0x3C00
    raw = OF.quantize_q8_0(np.array([127.0] + [0.0] * 31))
    assert raw[:2].tolist() == [0x00, 0x3C] and raw[2] == 127


def test_hand_worked_block():
    # values k/2 for k = -16..15: amax 8, d = 8/127, q = round(x * 127 / 8)
    x = np.arange(-16, 16) / 2.0
    d, q = qd(OF.quantize_q8_0(x))
    assert d[0] == np.float16(8.0 / 127.0)
    want = {-8.0: -127, 0.5: 8, 1.5: 24, 3.0: 48, 7.5: 119, -0.5: -8, 0.0: 0}
    for v, qq in want.items():
        assert q[0][list(x).index(v)] == qq, v


def test_halves_round_away_from_zero():
    # amax 127 gives d = 1 exactly, so q = round(x): 2.5 -> 3, -2.5 -> -3, 0.5 -> 1
    x = np.array([127.0, 2.5, -2.5, 0.5, -0.5, 1.4999999] + [0.0] * 26)
    _, q = qd(OF.quantize_q8_0(x))
    assert q[0][:6].tolist() == [127, 3, -3, 1, -1, 1]


def test_zero_block_and_amax_maps_to_127():
    d, q = qd(OF.quantize_q8_0(np.zeros(32)))
    assert d[0] == 0.0 and not q.any()
    x = np.random.default_rng(2).normal(size=(50, 32))
    d, q = qd(OF.quantize_q8_0(x))
    i = np.argmax(np.abs(x), axis=1)
    assert np.array_equal(q[np.arange(50), i], np.where(x[np.arange(50), i] > 0, 127, -127))


def test_error_within_half_a_step():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(400, 128)) * rng.uniform(0.01, 100, size=(400, 1))
    back = OF.round_to_type(x, OF.Q8_0)
    amax = np.abs(x.reshape(400, 4, 32)).max(axis=2)
    step = np.repeat(amax / 127.0, 32, axis=1)
    # half a step of the float32 grid, plus q times the fp16 rounding of d (|q| <= 127)
    bound = step / 2 * (1 + 1e-6) + 127 * step * 2.0 ** -11
    assert np.all(np.abs(back - x) <= bound)
    assert np.max(np.abs(back - x) / step) > 0.45          # the bound is nearly reached


def test_values_on_the_grid_are_fixed_points():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(300, 64))
    once = OF.round_to_type(x, OF.Q8_0)
    raw1, raw2 = OF.quantize_q8_0(x), OF.quantize_q8_0(once)
    assert np.array_equal(raw1, raw2)
    assert np.array_equal(OF.round_to_type(once, OF.Q8_0), once)


MICRO32 = HParams(n_layer=2, n_embd=64, n_head=4, n_head_kv=1, head_dim=32, n_ff=96, n_vocab=97,
                  rope_freq_base=10000.0, rms_eps=1e-6)


@pytest.fixture(scope="module")
def micro32():
    return oracle_weights(MICRO32, 23, {"embd": S.F32, "linear": S.F32})


def test_q8_0_cache_decode_equals_no_cache_forward(micro32):
    toks = S.prompt_tokens(33, 12, MICRO32.n_vocab).numpy()
    full = forward_no_cache(micro32, MICRO32, toks, oracle.Q8_0, oracle.Q8_0)
    ctx = oracle.OracleContext(MICRO32, micro32, n_ctx=256, type_k=oracle.Q8_0, type_v=oracle.Q8_0,
                               n_ubatch=5)
    assert ctx.decode(toks[:7], logits=[1] * 7) == 0
    got = [ctx.get_logits_ith(i) for i in range(7)]
    for t in toks[7:]:
        assert ctx.decode([t]) == 0
        got.append(ctx.get_logits_ith(-1))
    scale = np.max(np.abs(full), axis=1, keepdims=True)
    assert np.max(np.abs(np.array(got) - full) / scale) < 1e-9
    # and the Q8_0 cache changes the logits by about its quantisation step, not more
    f16 = forward_no_cache(micro32, MICRO32, toks, oracle.F16, oracle.F16)
    dev = np.max(np.abs(full - f16) / scale)
    assert 1e-5 < dev < 2e-2, dev
