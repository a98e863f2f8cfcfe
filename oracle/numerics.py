"""The per-token math of one transformer layer, in float64, one plain definition per op.

[P2] Example 4 lists the ops of one decode step of layer 0: GET_ROWS (embedding), RMS_NORM then
MUL by attn_norm.weight, MUL_MAT by attn_q / attn_k / attn_v, RESHAPE to heads, ROPE with the
token positions, SET_ROWS of K and V into the layer's cache, FLASH_ATTN_EXT over the cache, MUL_MAT
by attn_output, ADD of the residual, then ffn_norm, ffn_gate / ffn_up, SWIGLU, ffn_down and the
second ADD. [P1] Крок 13б gives the same layer scheme in words (scores = Q x K^T, causal mask,
softmax, weighted sum of V, output projection, residual). [P2] Example 11 spells the unfused
attention as MUL_MAT(K, Q) -> SOFT_MAX with the mask -> MUL_MAT with V, which is the
formulation written out below.
"""
from __future__ import annotations

import numpy as np


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """MUL_MAT: for a weight {K, M} (M rows of length K) and inputs {K, N}, y[n][m] = sum_k w[m][k] x[n][k].

    [P2] Example 4, the paragraph on ggml's MUL_MAT convention. x is [N, K], w is [M, K]."""
    return x @ w.T


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMS_NORM then MUL by the gain: y = x / sqrt(mean(x^2) + eps) * g, over the last axis.

    reading: the pages name the op only ([P2] Example 4: "rescales the vector to a standard size,
    followed by a learned scale"); this is the standard RMSNorm with eps inside the square root."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos: np.ndarray, freq_base: float) -> np.ndarray:
    """ROPE, rope type 0 ("normal", the Llama layout, [P2] Example 8): x is [T, n_heads, hd].

    reading: the pairs rotated are adjacent elements (2i, 2i+1) of each head; pair i turns by the
    angle pos * freq_base^(-2i/hd) (freq_scale 1, [P2] Example 9), i.e.
        y[2i]   = x[2i] cos(a) - x[2i+1] sin(a)
        y[2i+1] = x[2i] sin(a) + x[2i+1] cos(a).
    """
    hd = x.shape[-1]
    i = np.arange(hd // 2, dtype=np.float64)
    theta = np.power(float(freq_base), -2.0 * i / hd)                     # [hd/2]
    ang = pos.astype(np.float64)[:, None] * theta[None, :]                # [T, hd/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def softmax_masked(scores: np.ndarray, visible: np.ndarray) -> np.ndarray:
    """SOFT_MAX with the mask over the last axis: masked entries are -inf and get weight exactly 0.

    The row maximum is subtracted first. A row with no visible entry is all zeros (reading: the
    decode path never builds one, since a token always sees its own cell)."""
    s = np.where(visible, scores, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(visible, np.exp(s - m), 0.0)
    z = np.sum(e, axis=-1, keepdims=True)
    return np.divide(e, z, out=np.zeros_like(e), where=z > 0)


def attention(q: np.ndarray, k_cells: np.ndarray, v_cells: np.ndarray, visible: np.ndarray,
              n_head_kv: int) -> np.ndarray:
    """Grouped-query attention of the ubatch's queries over the cache cells.

    q: [T, H, hd]; k_cells, v_cells: [C, Hkv, hd] (the cache rows, already rounded to the cache
    type); visible: bool [T, C] (the KQ mask, True = may attend). Returns [T, H * hd].
    reading: scale 1/sqrt(hd); query head h reads KV head h // (H / Hkv) ([P2] Example 8: n_gqa =
    n_head / n_head_kv query heads share one KV head)."""
    T, H, hd = q.shape
    G = H // n_head_kv
    out = np.zeros((T, H, hd), dtype=np.float64)
    for h in range(H):
        g = h // G
        scores = (q[:, h, :] @ k_cells[:, g, :].T) / np.sqrt(hd)          # [T, C]
        p = softmax_masked(scores, visible)
        out[:, h, :] = p @ v_cells[:, g, :]
    return out.reshape(T, H * hd)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SWIGLU(ffn_gate, ffn_up) = silu(gate) * up ([P2] Example 4; the gate is the first operand)."""
    return silu(gate) * up
