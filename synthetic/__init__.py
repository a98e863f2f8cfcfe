"""Seeded synthetic inputs: model weights in their storage formats and prompt token ids.

This module is the only code shared by the CPU oracle side and the CUDA side. It contains no
arithmetic of the decode method itself: it draws random numbers from a counter-based integer hash
and packs them into the storage formats the llama weight files use (F32, BF16, F16 and Q8_0
blocks of 32 int8 values plus one fp16 scale). Every step is plain integer arithmetic followed by
one IEEE float multiply and one library cast, so the same seed gives the same bytes on a CPU and
on a GPU.

Distributions (the workloads' recipe):
  * linear weights and embeddings: approximately N(0, sigma^2), sigma = 0.02, drawn as an
    Irwin-Hall sum of four 16-bit uniforms, centred and scaled to unit variance;
  * norm gains: exactly 1.0;
  * Q8_0 blocks: q uniform over the integers [-127, 127], scale d = fp16(|N(0, 2e-4^2)|);
  * prompt tokens: uniform over [0, n_vocab).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from .configs import HParams, Workload, TINY, LLAMA8B, WORKLOADS, tensor_specs  # noqa: F401

M32 = 0xFFFFFFFF
_MIX = 0x45D9F3B            # multiplier of a public-domain 32-bit integer mixing function
_CHUNK = 1 << 24            # elements generated per chunk (bounds temporary memory)

# storage types, numbered like the C-ABI's llm_type
F32, F16, BF16, Q8_0 = 0, 1, 2, 8
TYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16", Q8_0: "q8_0"}
QK8_0 = 32                  # values per Q8_0 block
Q8_0_BLOCK_BYTES = 34       # 2-byte fp16 scale + 32 int8


def hash32(x: torch.Tensor) -> torch.Tensor:
    """Mix int64 tensor values in [0, 2^32) into pseudo-random values in [0, 2^32).

    Every product stays below 2^59, so no int64 overflow happens on any device."""
    x = x ^ (x >> 16)
    x = (x * _MIX) & M32
    x = x ^ (x >> 16)
    x = (x * _MIX) & M32
    x = x ^ (x >> 16)
    return x


def name_key(seed: int, name: str) -> int:
    """32-bit key for (seed, tensor name): FNV-1a over the name's bytes, mixed with the seed."""
    h = 0x811C9DC5
    for b in name.encode():
        h = ((h ^ b) * 0x01000193) & M32
    h ^= (seed * 0x9E3779B1) & M32
    return int(hash32(torch.tensor([h], dtype=torch.int64))[0])


def _draw(key: int, start: int, n: int, lane: int, device) -> torch.Tensor:
    """n hash values for counters start..start+n-1 of stream `lane` of `key` (int64 in [0, 2^32))."""
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    lo = idx & M32
    hi = idx >> 32
    k = hash32(torch.tensor([(key ^ (lane * 0x27D4EB2F)) & M32], dtype=torch.int64, device=device))
    return hash32(lo ^ hash32((hi + k) & M32))


def normal_f32(key: int, n: int, sigma: float, device="cpu", start: int = 0) -> torch.Tensor:
    """Approximately N(0, sigma^2) float32 values (Irwin-Hall sum of four 16-bit uniforms)."""
    a = _draw(key, start, n, 0, device)
    b = _draw(key, start, n, 1, device)
    s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16)     # integer in [0, 4*65535]
    centred = (s - 2 * 65535).to(torch.float32)                   # exact in float32 (< 2^18)
    # each 16-bit uniform has variance 65535^2/12 (to 1e-5); the sum of four has 65535^2/3
    scale = float(torch.tensor(sigma * math.sqrt(3.0) / 65535.0, dtype=torch.float32))
    return centred * scale


def uniform_int(key: int, n: int, lo: int, hi: int, device="cpu", start: int = 0, lane: int = 2):
    """Integers uniform over [lo, hi] (modulo draw; the bias is below 1e-7)."""
    a = _draw(key, start, n, lane, device)
    return lo + (a % (hi - lo + 1))


def weight_bytes(seed: int, name: str, shape: tuple, wtype: int, device="cpu",
                 sigma: float = 0.02, q8_scale_sigma: float = 2e-4) -> torch.Tensor:
    """One weight tensor in its storage format.

    shape is ggml order (ne0 = row length, ne1 = rows). Returns:
      F32  -> float32 tensor [ne1, ne0]      F16 -> float16 [ne1, ne0]
      BF16 -> bfloat16 tensor [ne1, ne0]     Q8_0 -> uint8 [ne1, ne0/32*34] of whole blocks
    Norm gains (names ending in '_norm.weight') are exactly 1.0.
    """
    ne0 = int(shape[0])
    ne1 = int(shape[1]) if len(shape) > 1 else 1
    n = ne0 * ne1
    key = name_key(seed, name)
    if name.endswith("_norm.weight"):
        assert wtype == F32, "norm gains are stored as F32"
        return torch.ones((ne1, ne0), dtype=torch.float32, device=device)
    if wtype in (F32, F16, BF16):
        dt = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[wtype]
        out = torch.empty(n, dtype=dt, device=device)
        for s in range(0, n, _CHUNK):
            m = min(_CHUNK, n - s)
            out[s:s + m] = normal_f32(key, m, sigma, device, start=s).to(dt)
        return out.view(ne1, ne0)
    if wtype == Q8_0:
        assert ne0 % QK8_0 == 0, "a Q8_0 row is made of whole 32-value blocks"
        nb = n // QK8_0
        out = torch.empty((nb, Q8_0_BLOCK_BYTES), dtype=torch.uint8, device=device)
        bchunk = _CHUNK // QK8_0
        for s in range(0, nb, bchunk):
            m = min(bchunk, nb - s)
            d = normal_f32(key ^ 0x5A5A5A5A, m, q8_scale_sigma, device, start=s).abs().to(torch.float16)
            q = uniform_int(key, m * QK8_0, -127, 127, device, start=s * QK8_0).to(torch.int8)
            out[s:s + m, 0:2] = d.view(torch.uint8).view(m, 2)
            out[s:s + m, 2:] = q.view(torch.uint8).view(m, QK8_0)
        return out.view(ne1, (ne0 // QK8_0) * Q8_0_BLOCK_BYTES)
    raise ValueError(f"unsupported weight type {wtype}")


def weight_rows(seed: int, name: str, shape: tuple, wtype: int, rows, device="cpu",
                sigma: float = 0.02, q8_scale_sigma: float = 2e-4) -> torch.Tensor:
    """Rows `rows` (indices into ne1) of the tensor weight_bytes would make, without making the
    rest: the same counters, so the bytes equal weight_bytes(...)[rows]."""
    ne0 = int(shape[0])
    key = name_key(seed, name)
    out = []
    for r in (int(x) for x in rows):
        if wtype in (F32, F16, BF16):
            dt = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[wtype]
            out.append(normal_f32(key, ne0, sigma, device, start=r * ne0).to(dt))
        elif wtype == Q8_0:
            nb, b0 = ne0 // QK8_0, r * (ne0 // QK8_0)
            blk = torch.empty((nb, Q8_0_BLOCK_BYTES), dtype=torch.uint8, device=device)
            d = normal_f32(key ^ 0x5A5A5A5A, nb, q8_scale_sigma, device, start=b0).abs().to(torch.float16)
            q = uniform_int(key, nb * QK8_0, -127, 127, device, start=b0 * QK8_0).to(torch.int8)
            blk[:, 0:2] = d.view(torch.uint8).view(nb, 2)
            blk[:, 2:] = q.view(torch.uint8).view(nb, QK8_0)
            out.append(blk.view(-1))
        else:
            raise ValueError(f"unsupported weight type {wtype}")
    return torch.stack(out)


def prompt_tokens(seed: int, n: int, n_vocab: int, device="cpu") -> torch.Tensor:
    """n token ids uniform over [0, n_vocab) (int32)."""
    key = name_key(seed, "prompt")
    return uniform_int(key, n, 0, n_vocab - 1, device, lane=3).to(torch.int32)


def model_weights(hp: HParams, seed: int, types: dict, device="cpu"):
    """Yield (name, wtype, shape, storage tensor) for every tensor of a llama model."""
    for name, shape in tensor_specs(hp):
        wt = types_for(name, types)
        yield name, wt, shape, weight_bytes(seed, name, shape, wt, device)


def types_for(name: str, types: dict) -> int:
    """Storage type of a tensor under a workload's type map {'norm','embd','linear','output'}."""
    if name.endswith("_norm.weight"):
        return types.get("norm", F32)
    if name == "token_embd.weight":
        return types["embd"]
    if name == "output.weight":
        return types.get("output", types["linear"])
    return types["linear"]
