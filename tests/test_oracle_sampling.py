"""Pins of the oracle's sampler chain against closed forms and frequencies (no oracle code
retyped): greedy = argmax with the lowest id on ties; stratified draws reproduce softmax
probabilities; hand-made distributions for top-k / top-p / min-p; the penalty's sign rule; the
chain's order (cut-offs before temperature)."""
import math

import numpy as np
import pytest

from oracle.sampling import SamplerParams, apply_penalty, chain_candidates, sample


def test_greedy_is_argmax_with_lowest_id_on_ties():
    l = np.array([0.1, 3.0, -2.0, 3.0, 1.0])
    for u in (0.0, 0.3, 0.99):
        assert sample(l, SamplerParams(top_k=5, temperature=0.0), u) == 1
        assert sample(l, SamplerParams(top_k=1, temperature=1.0), u) == 1


def test_stratified_draws_reproduce_softmax():
    rng = np.random.default_rng(3)
    l = rng.normal(size=12)
    p = np.exp(l - l.max()); p /= p.sum()
    N = 20000
    counts = np.zeros(12)
    for i in range(N):
        counts[sample(l, SamplerParams(top_k=12, temperature=1.0), (i + 0.5) / N)] += 1
    assert np.max(np.abs(counts / N - p)) <= 1.0 / N + 1e-12


def test_temperature_scales_log_odds():
    l = np.array([1.0, 0.0])
    N = 20000
    for t in (0.5, 2.0):
        c0 = sum(sample(l, SamplerParams(top_k=2, temperature=t), (i + 0.5) / N) == 0 for i in range(N))
        p0 = 1.0 / (1.0 + math.exp(-1.0 / t))
        assert abs(c0 / N - p0) <= 1.0 / N + 1e-12


def test_top_p_min_p_on_a_known_distribution():
    probs = np.array([0.05, 0.5, 0.15, 0.3])          # order by probability: 1, 3, 2, 0
    l = np.log(probs)
    for p, want in ((0.45, [1]), (0.75, [1, 3]), (0.85, [1, 3, 2]), (0.96, [1, 3, 2, 0])):
        cand, _ = chain_candidates(l, SamplerParams(top_k=4, top_p=p))
        assert cand.tolist() == want, (p, cand)
    cand, _ = chain_candidates(l, SamplerParams(top_k=4, min_p=0.25))      # keep p >= 0.125
    assert cand.tolist() == [1, 3, 2]
    cand, _ = chain_candidates(l, SamplerParams(top_k=2, min_p=0.0))
    assert cand.tolist() == [1, 3]


def test_cut_offs_use_untempered_probabilities():
    # softmax at t = 1: [0.6, 0.4]; top-p 0.7 keeps both. Were the temperature applied first
    # (t = 0.25: [0.835, 0.165]), only one would stay.
    l = np.log(np.array([0.6, 0.4]))
    cand, _ = chain_candidates(l, SamplerParams(top_k=2, top_p=0.7, temperature=0.25))
    assert cand.tolist() == [0, 1]
    assert sample(l, SamplerParams(top_k=2, top_p=0.7, temperature=0.25), 0.99) == 1


def test_repeat_penalty_sign_rule_and_distinct_tokens():
    l = np.array([2.0, -1.0, 0.5, 0.0])
    out = apply_penalty(l, [0, 1, 1, 3], 2.0)
    assert out.tolist() == [1.0, -2.0, 0.5, 0.0]
    # a penalised leader loses the greedy pick
    assert sample(np.array([1.0, 0.9]), SamplerParams(top_k=2, temperature=0.0, repeat_penalty=1.5,
                                                      penalty_tokens=[0]), 0.5) == 1


@pytest.mark.parametrize("u", [0.0, 0.25, 0.5, 0.999999])
def test_pick_lies_in_the_candidate_set(u):
    rng = np.random.default_rng(7)
    l = rng.normal(size=500) * 3
    p = SamplerParams(top_k=40, top_p=0.9, min_p=0.02, temperature=0.8, repeat_penalty=1.2,
                      penalty_tokens=list(range(0, 500, 7)))
    cand, _ = chain_candidates(l, p)
    assert sample(l, p, u) in cand.tolist()
