"""The sampler chain over one logits row ([P1] "llama.cpp AI LLM Engine - Як це працює", the
sampler-chain list after Крок 14 and the paragraph on llama_sampler_chain_init / _add: penalties,
then the cut-offs top-k, top-p, min-p, then temperature, then one token is picked: greedily or
at random by softmax probability).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py). Plain float64 numpy, one step after another.

readings (the pages name the steps, not their formulas):
  - repeat penalty r over a set of earlier tokens (each token once): a logit l > 0 becomes l / r,
    otherwise l * r (the probability of a repeated token goes down for r > 1);
  - top-k: the k largest logits stay; ties at the k-th value are broken by the lower token id;
  - the candidates are then ordered by logit descending, token id ascending;
  - top-p: with probabilities softmax(l) over the remaining candidates, keep the shortest prefix
    of that order whose cumulative probability reaches p (at least one token);
  - min-p: keep the candidates with probability >= min_p * the largest, i.e. l - l_max >= ln(min_p);
  - temperature t > 0 divides the remaining logits; the pick draws u in [0, 1) (an input: the
    random number is the caller's) and returns the first candidate of the order whose cumulative
    probability exp((l - l_max) / t) / Z exceeds u; t <= 0 picks the first candidate (greedy).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Sequence

import numpy as np


@dataclass
class SamplerParams:
    top_k: int = 40
    top_p: float = 1.0
    min_p: float = 0.0
    temperature: float = 1.0
    repeat_penalty: float = 1.0
    penalty_tokens: Sequence[int] = field(default_factory=list)


def apply_penalty(logits: np.ndarray, tokens: Sequence[int], r: float) -> np.ndarray:
    """Repeat penalty: each distinct token of `tokens` once; l > 0 -> l / r, else l * r."""
    out = np.asarray(logits, dtype=np.float64).copy()
    if r == 1.0:
        return out
    for t in sorted(set(int(x) for x in tokens)):
        if 0 <= t < len(out):
            out[t] = out[t] / r if out[t] > 0 else out[t] * r
    return out


def top_k_order(logits: np.ndarray, k: int) -> np.ndarray:
    """Token ids of the k largest logits, ordered by logit descending then id ascending."""
    ids = np.arange(len(logits))
    order = np.lexsort((ids, -logits))          # primary: -logit ascending; secondary: id
    return order[:max(1, min(k, len(logits)))]


def chain_candidates(logits: np.ndarray, p: SamplerParams):
    """The candidates left after penalties, top-k, top-p and min-p, in the chain's order, with
    their (penalised) logits."""
    l = apply_penalty(logits, p.penalty_tokens, p.repeat_penalty)
    cand = top_k_order(l, p.top_k)
    lv = l[cand]
    if p.top_p < 1.0:
        e = np.exp(lv - lv[0])
        prob = e / e.sum()
        cum = np.cumsum(prob)
        n = int(np.searchsorted(cum, p.top_p) + 1)       # first prefix reaching p
        cand, lv = cand[:min(n, len(cand))], lv[:min(n, len(lv))]
    if p.min_p > 0.0:
        keep = (lv - lv[0]) >= math.log(p.min_p)
        keep[0] = True
        cand, lv = cand[keep], lv[keep]
    return cand, lv


def sample(logits: np.ndarray, p: SamplerParams, u: float) -> int:
    """The token the chain picks for the uniform draw u in [0, 1)."""
    cand, lv = chain_candidates(logits, p)
    if p.temperature <= 0.0:
        return int(cand[0])
    w = np.exp((lv - lv[0]) / p.temperature)
    cum = np.cumsum(w)
    j = int(np.searchsorted(cum, u * cum[-1], side="right"))
    return int(cand[min(j, len(cand) - 1)])


def pick_margin(logits: np.ndarray, p: SamplerParams, u: float) -> float:
    """How far u * Z is from the nearest cumulative boundary, relative to Z (for tests that
    compare a float32 implementation: below ~1e-5 both neighbouring tokens are correct)."""
    cand, lv = chain_candidates(logits, p)
    if p.temperature <= 0.0 or len(cand) == 1:
        return 1.0
    w = np.exp((lv - lv[0]) / p.temperature)
    cum = np.cumsum(w) / w.sum()
    return float(np.min(np.abs(cum[:-1] - u))) if len(cum) > 1 else 1.0
