"""Test glue: turning synthetic storage tensors into oracle weights, small model shapes."""
from __future__ import annotations

import functools

import numpy as np
import torch

import synthetic as S
from synthetic.configs import HParams


def to_numpy_raw(t: torch.Tensor) -> np.ndarray:
    """Storage tensor -> numpy array of the same bytes (bf16 as uint16)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_weights(hp: HParams, seed: int, types: dict, cache: bool = True, skip=()):
    import oracle
    w = oracle.OracleWeights(cache=cache)
    for name, wt, shape, t in S.model_weights(hp, seed, types):
        if name in skip:
            continue
        w.add(name, wt, shape[0], to_numpy_raw(t))
    return w


@functools.lru_cache(maxsize=4)
def tiny_weights(seed: int, types_key: tuple = (("embd", 0), ("linear", 0))):
    return oracle_weights(S.TINY, seed, dict(types_key))


# a small model with the tiny model's structure (GQA 4, adjacent-pair RoPE), fast in float64
MICRO = HParams(n_layer=2, n_embd=64, n_head=4, n_head_kv=1, head_dim=16, n_ff=96, n_vocab=97,
                rope_freq_base=10000.0, rms_eps=1e-6)
