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


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """Rows of values (last axis a whole number of 32-value blocks) -> Q8_0 rows (uint8,
    [..., ne0/32*34]), the byte layout of [P2] Example 2: per block the fp16 scale d (2 bytes,
    little-endian) then 32 int8 quants q.

    The pages give the block layout and the way back (value = d * q), not the quantiser. Reading
    taken: a symmetric absmax scale, so that the block's largest magnitude maps to +-127. The row a
    cache write receives is float32, and the integer decisions are taken in float32:
      amax = max |x| (float32), d = amax / 127 (float32 division), id = 1 / d (float32; 0 if d = 0),
      q = x * id (float32 product) rounded to the nearest integer, halves away from zero,
      stored d = d rounded to fp16 (nearest even).
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    assert x32.shape[-1] % QK8_0 == 0
    lead = x32.shape[:-1]
    b = x32.reshape(-1, x32.shape[-1] // QK8_0, QK8_0)
    amax = np.max(np.abs(b), axis=2)                                   # float32, exact
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    y = (b * inv[:, :, None]).astype(np.float32).astype(np.float64)   # the float32 product, exactly
    q = (np.sign(y) * np.floor(np.abs(y) + 0.5)).astype(np.int8)       # halves away from zero
    out = np.empty(b.shape[:2] + (Q8_0_BYTES,), dtype=np.uint8)
    out[:, :, 0:2] = d.astype(np.float16).view(np.uint8).reshape(b.shape[0], b.shape[1], 2)
    out[:, :, 2:] = q.view(np.uint8)
    return out.reshape(lead + (x32.shape[-1] // QK8_0 * Q8_0_BYTES,))


def round_to_type(x: np.ndarray, t: int) -> np.ndarray:
    """Value a cache row holds after a write of x in type t, as float64: F32/F16 round to nearest
    even; Q8_0 quantises each 32-value block (quantize_q8_0) and reads back d * q."""
    if t == F32:
        return x.astype(np.float32).astype(np.float64)
    if t == F16:
        return x.astype(np.float16).astype(np.float64)
    if t == Q8_0:
        x = np.asarray(x)
        ne0 = x.shape[-1]
        raw = quantize_q8_0(x).reshape(-1, ne0 // QK8_0 * Q8_0_BYTES)
        return q8_0_to_f64(raw, ne0).reshape(x.shape)
    raise ValueError(f"unsupported cache type {t}")


def type_row_bytes(t: int, ne0: int) -> int:
    """Bytes of one row of ne0 values ([P2] Example 2: nb[1] = ne0 / block_size * type_size)."""
    if t == Q8_0:
        assert ne0 % QK8_0 == 0
        return ne0 // QK8_0 * Q8_0_BYTES
    return ne0 * {F32: 4, F16: 2, BF16: 2}[t]
