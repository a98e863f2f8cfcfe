"""GPU parity of the device sampler chain (llm_sample_ith) against the oracle's chain, through the
C ABI.

Rows: the tiny model's own logits rows, and chosen rows written over an output row with the
debug hook (ties at the top-k threshold, a flat row, NaN and -inf entries, 4096 candidates).
The bar: the same token as the oracle on the same float32 row. The device works in float32 and
the oracle in float64, so a case is compared only where no decision lies within 2e-5 of a
boundary (the pick's cumulative weight against u, top-p's cumulative probability against p,
min-p's log ratio against ln min_p: float32 sums of up to 4096 terms stay well inside that);
such near-ties are skipped, counted, and still must pick a candidate of the chain."""
import math

import numpy as np
import pytest

import synthetic as S
from oracle.sampling import SamplerParams, chain_candidates, pick_margin, sample
from tests import gpu_common as G

pytestmark = pytest.mark.gpu
EDGE = 2e-5

PARAMS = [
    SamplerParams(top_k=40, temperature=0.0),
    SamplerParams(top_k=1, temperature=1.0),
    SamplerParams(top_k=40, temperature=1.0),
    SamplerParams(top_k=40, top_p=0.9, temperature=0.8),
    SamplerParams(top_k=100, top_p=0.95, min_p=0.05, temperature=0.7),
    SamplerParams(top_k=4096, temperature=1.5),
    SamplerParams(top_k=4096, top_p=0.5, temperature=1.0),
    SamplerParams(top_k=64, min_p=0.1, temperature=1.0, repeat_penalty=1.3,
                  penalty_tokens=[5, 17, 17, 99, 151935, 0]),
]
US = [0.0, 0.13, 0.5, 0.77, 0.999]


def near_edge(l: np.ndarray, p: SamplerParams, u: float) -> bool:
    """True if a decision of the chain lies within EDGE of its boundary for this row and u."""
    from oracle.sampling import apply_penalty, top_k_order
    lp = apply_penalty(l, p.penalty_tokens, p.repeat_penalty)
    cand = top_k_order(lp, p.top_k)
    lv = lp[cand]
    if p.top_p < 1.0:
        e = np.exp(lv - lv[0])
        if np.min(np.abs(np.cumsum(e) / e.sum() - p.top_p)) < EDGE:
            return True
    if p.min_p > 0.0 and np.min(np.abs(lv[1:] - lv[0] - math.log(p.min_p)), initial=1.0) < EDGE:
        return True
    return pick_margin(l, p, u) < EDGE


def device_pick(ctx, i: int, p: SamplerParams, u: float) -> int:
    return ctx.sample_ith(i, top_k=p.top_k, top_p=p.top_p, min_p=p.min_p, temperature=p.temperature,
                          repeat_penalty=p.repeat_penalty, penalty_tokens=p.penalty_tokens, u=u)


@pytest.fixture(scope="module")
def ctx():
    key = "tiny_f32_1seq"
    c = G.library_ctx(key)
    toks = G.prompts(key)[0][:24]
    assert c.decode(toks, logits=[1] * len(toks)) == 0, c.last_error()
    yield c
    c.free()


def test_sampler_matches_oracle_on_model_rows(ctx):
    compared = skipped = 0
    for i in (0, 7, 23):
        row = ctx.get_logits_ith(i).astype(np.float64)
        for p in PARAMS:
            for u in US:
                want = sample(row, p, u)
                got = device_pick(ctx, i, p, u)
                assert got >= 0, ctx.last_error()
                cand, _ = chain_candidates(row, p)
                assert got in cand.tolist(), (i, p, u, got)
                if near_edge(row, p, u):
                    skipped += 1
                    continue
                assert got == want, (i, p, u, got, want)
                compared += 1
    assert compared >= 0.8 * (compared + skipped), (compared, skipped)


def test_greedy_equals_decode_argmax(ctx):
    for i in range(24):
        assert ctx.sample_ith(i, top_k=40, temperature=0.0) == ctx.get_argmax_ith(i)


def set_row(ctx, i, row):
    assert ctx.debug_set_logits(i, row) == 0, ctx.last_error()
    assert np.array_equal(ctx.get_logits_ith(i), row.astype(np.float32), equal_nan=True)


def test_ties_at_the_top_k_threshold_take_the_lowest_ids(ctx):
    V = ctx.n_vocab
    rng = np.random.default_rng(11)
    row = np.full(V, -5.0, dtype=np.float32)
    hi = rng.choice(V, 30, replace=False)
    row[hi] = rng.normal(size=30).astype(np.float32) + 10.0
    ties = np.sort(rng.choice(np.setdiff1d(np.arange(V), hi), 3000, replace=False))
    row[ties] = 2.0
    set_row(ctx, 3, row)
    for k in (30, 31, 45, 1000, 3030, 4096):
        p = SamplerParams(top_k=k, temperature=1e6)          # near-uniform over the candidates
        cand, _ = chain_candidates(row.astype(np.float64), p)
        for u in (0.0, 0.4999, 0.9999):
            want = sample(row.astype(np.float64), p, u)
            got = device_pick(ctx, 3, p, u)
            assert got in cand.tolist(), (k, u, got)
            if not near_edge(row.astype(np.float64), p, u):
                assert got == want, (k, u, got, want)
    # the last tie admitted at k = 45 is the 15th lowest id among the ties
    p = SamplerParams(top_k=45, temperature=1e6)
    cand, _ = chain_candidates(row.astype(np.float64), p)
    assert sorted(cand[30:].tolist()) == ties[:15].tolist()


def test_flat_row_and_leader_ties(ctx):
    V = ctx.n_vocab
    row = np.zeros(V, dtype=np.float32)
    set_row(ctx, 4, row)
    assert ctx.sample_ith(4, top_k=40, temperature=0.0) == 0
    # uniform over ids 0..49: u picks id floor(u * 50)
    for u in (0.01, 0.33, 0.61, 0.97):
        assert ctx.sample_ith(4, top_k=50, temperature=1.0, u=u) == int(u * 50)
    row[[9000, 77, 150000]] = 3.0
    set_row(ctx, 4, row)
    assert ctx.sample_ith(4, top_k=40, temperature=0.0) == 77
    assert ctx.sample_ith(4, top_k=3, temperature=1.0, u=0.5) == 9000
    assert ctx.sample_ith(4, top_k=3, temperature=1.0, u=0.9) == 150000


def test_nan_and_minus_inf_are_never_picked(ctx):
    V = ctx.n_vocab
    rng = np.random.default_rng(12)
    row = rng.normal(size=V).astype(np.float32)
    row[rng.choice(V, 5000, replace=False)] = np.nan
    row[rng.choice(V, 5000, replace=False)] = -np.inf
    set_row(ctx, 5, row)
    finite = np.isfinite(row)
    for p in PARAMS:
        for u in US:
            got = device_pick(ctx, 5, p, u)
            assert 0 <= got < V and finite[got], (p, u, got)
            r64 = np.where(np.isnan(row), -np.inf, row).astype(np.float64)
            if not near_edge(r64, p, u):
                assert got == sample(r64, p, u), (p, u)


def test_penalty_flips_the_greedy_pick(ctx):
    V = ctx.n_vocab
    row = np.full(V, -1.0, dtype=np.float32)
    row[10], row[20], row[30] = 4.0, 3.0, -0.5
    set_row(ctx, 6, row)
    assert ctx.sample_ith(6, top_k=8, temperature=0.0) == 10
    assert ctx.sample_ith(6, top_k=8, temperature=0.0, repeat_penalty=2.0, penalty_tokens=[10, 10]) == 20
    # 4 / 3 stays above 3 / 3
    assert ctx.sample_ith(6, top_k=3, temperature=0.0, repeat_penalty=3.0, penalty_tokens=[10, 20]) == 10
    # a negative logit moves away from zero: -0.5 * 3 = -1.5 falls below the -1 entries, so with
    # top-k 3 the third candidate is the lowest id among the -1 entries
    p = SamplerParams(top_k=3, temperature=0.0, repeat_penalty=3.0, penalty_tokens=[30])
    cand, _ = chain_candidates(row.astype(np.float64), p)
    assert cand.tolist() == [10, 20, 0]
    p = SamplerParams(top_k=3, temperature=1.0, repeat_penalty=3.0, penalty_tokens=[30, 10, 20])
    for u in US:
        assert device_pick(ctx, 6, p, u) in chain_candidates(row.astype(np.float64), p)[0].tolist()


def test_invalid_arguments_return_minus_one(ctx):
    assert ctx.sample_ith(0, top_k=0) == -1
    assert ctx.sample_ith(0, top_k=4097) == -1
    assert ctx.sample_ith(0, top_p=0.0) == -1
    assert ctx.sample_ith(0, min_p=1.0) == -1
    assert ctx.sample_ith(0, u=1.0) == -1
    assert ctx.sample_ith(0, repeat_penalty=0.0) == -1
    assert ctx.sample_ith(999) == -1
    assert ctx.sample_ith(0, top_k=40, temperature=0.0) >= 0     # the context is still usable
