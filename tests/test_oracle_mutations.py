"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each one."""
import numpy as np
import pytest

import oracle
from oracle import numerics as N
from tests import test_oracle_model as TM
from tests import test_oracle_pins as TP


def _neox_rope(x, pos, base):
    hd = x.shape[-1]
    i = np.arange(hd // 2, dtype=np.float64)
    ang = pos.astype(np.float64)[:, None] * np.power(base, -2.0 * i / hd)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., : hd // 2], x[..., hd // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def _rope_wrong_sign(x, pos, base):
    return N.rope(x, -pos, base)


def _attn_wrong_scale(q, k, v, vis, hkv):
    return N.attention(q * np.sqrt(q.shape[-1]) / q.shape[-1] * 2, k, v, vis, hkv)


def _attn_wrong_group(q, k, v, vis, hkv):
    T, H, hd = q.shape
    out = np.zeros((T, H, hd))
    for h in range(H):
        g = h % hkv                                   # interleaved instead of consecutive groups
        s = q[:, h, :] @ k[:, g, :].T / np.sqrt(hd)
        out[:, h, :] = N.softmax_masked(s, vis) @ v[:, g, :]
    return out.reshape(T, H * hd)


def _rms_no_mean(x, g, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * g


def _swiglu_swapped(gate, up):
    return N.silu(up) * gate


MUTATIONS = [
    ("rope", _neox_rope, TP.test_rope_pairs_and_frequencies),
    ("rope", _rope_wrong_sign, TP.test_rope_pairs_and_frequencies),
    ("attention", _attn_wrong_scale, TP.test_attention_special_cases_and_gqa_mapping),
    ("attention", _attn_wrong_group, TP.test_attention_special_cases_and_gqa_mapping),
    ("rms_norm", _rms_no_mean, TP.test_rms_norm_closed_form),
    ("swiglu", _swiglu_swapped, TP.test_silu_and_swiglu_values),
]


@pytest.mark.parametrize("target,bad,pin", MUTATIONS, ids=[m[1].__name__ for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, target, bad, pin):
    monkeypatch.setattr(oracle, target, bad)
    with pytest.raises(AssertionError):
        pin()


def test_causality_mistake_caught_by_analytic_model(monkeypatch):
    orig = oracle.memory.Cells.mask

    def no_causal(self, pos, seq_ids, n_kv):
        return orig(self, [10 ** 9] * len(pos), seq_ids, n_kv)
    monkeypatch.setattr(oracle.memory.Cells, "mask", no_causal)
    with pytest.raises(AssertionError):
        TM.test_analytic_uniform_attention_is_mean_of_visible_values()


def test_sequence_mistake_caught_by_analytic_model(monkeypatch):
    orig = oracle.memory.Cells.mask

    def all_seqs(self, pos, seq_ids, n_kv):
        return orig(self, pos, [[0, 1, 2, 3]] * len(pos), n_kv)
    monkeypatch.setattr(oracle.memory.Cells, "mask", all_seqs)
    with pytest.raises(AssertionError):
        TM.test_analytic_uniform_attention_is_mean_of_visible_values()


def test_stale_cache_mistake_caught_by_no_cache_invariant(monkeypatch):
    # forgetting to include the ubatch's own K/V (attend before append)
    orig = oracle.memory.Cells.mask

    def strict(self, pos, seq_ids, n_kv):
        m = orig(self, pos, seq_ids, n_kv)
        for t, p in enumerate(pos):
            for c in range(n_kv):
                if self.pos[c] == p:
                    m[t, c] = False
        m[:, 0] = True
        return m
    monkeypatch.setattr(oracle.memory.Cells, "mask", strict)
    with pytest.raises(AssertionError):
        TM.test_analytic_uniform_attention_is_mean_of_visible_values()
