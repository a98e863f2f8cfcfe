"""Storage formats -> float64, and the KV-cache rounding.

[P2] Example 2: a tensor has ne (elements per dimension, innermost first) and nb (byte strides);
a row of a {K, M} weight is K contiguous values. A Q8_0 block holds 32 values in 34 bytes: a
2-byte fp16 scale d followed by 32 int8 quants q; the value is d * q, and a row is a whole number
of blocks. [P2] Example 4: the cache stores K/V rows in F16 by default ("cache_k_l0 (f16)").
"""
from __future__ import annotations

import numpy as np

F32, F16, BF16, Q8_0 = 0, 1, 2, 8
QK8_0 = 32
Q8_0_BYTES = 34


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64. A bf16 is the top half of a float32: exact."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def q8_0_to_f64(raw: np.ndarray, ne0: int) -> np.ndarray:
    """Q8_0 rows (uint8 [rows, ne0/32*34]) -> float64 [rows, ne0], value = d * q per block."""
    rows = raw.shape[0]
    blocks = raw.reshape(rows, ne0 // QK8_0, Q8_0_BYTES)
    d = np.ascontiguousarray(blocks[:, :, 0:2]).view(np.float16)[:, :, 0].astype(np.float64)
    q = np.ascontiguousarray(blocks[:, :, 2:]).view(np.int8).astype(np.float64)
    return (d[:, :, None] * q).reshape(rows, ne0)


def decode_weight(raw: np.ndarray, wtype: int, ne0: int) -> np.ndarray:
    """Raw storage of a 2-D weight (rows of ne0 values) -> float64 [rows, ne0]."""
    if wtype == F32:
        return raw.view(np.float32).reshape(-1, ne0).astype(np.float64)
    if wtype == F16:
        return raw.view(np.float16).reshape(-1, ne0).astype(np.float64)
    if wtype == BF16:
        return bf16_to_f64(raw.view(np.uint16).reshape(-1, ne0))
    if wtype == Q8_0:
        return q8_0_to_f64(raw.view(np.uint8).reshape(-1, ne0 // QK8_0 * Q8_0_BYTES), ne0)
    raise ValueError(f"unknown weight type {wtype}")


def round_to_type(x: np.ndarray, t: int) -> np.ndarray:
    """Value a cache row holds after a write of x in type t (round to nearest even), as float64."""
    if t == F32:
        return x.astype(np.float32).astype(np.float64)
    if t == F16:
        return x.astype(np.float16).astype(np.float64)
    raise ValueError(f"unsupported cache type {t}")


def type_row_bytes(t: int, ne0: int) -> int:
    """Bytes of one row of ne0 values ([P2] Example 2: nb[1] = ne0 / block_size * type_size)."""
    if t == Q8_0:
        assert ne0 % QK8_0 == 0
        return ne0 // QK8_0 * Q8_0_BYTES
    return ne0 * {F32: 4, F16: 2, BF16: 2}[t]
