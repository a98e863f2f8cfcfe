// Device helpers shared by the TMA-staged decode kernels: mbarrier waits bounded by the global
// timer, bulk global->shared copies with an L2 policy, 16-byte weight vectors unpacked to float,
// and the packed (value, lowest index) key of the greedy pick.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "kernels.h"

namespace llm {
namespace dev {

constexpr uint64_t kWaitNs = 2000000000ull;   // every wait gives up after 2 s

// (a0, a1) += (w0 * x0, w1 * x1) as one paired float32 FMA (fma.rn.f32x2): each lane does two
// independent fused multiply-adds per instruction, each rounded as fmaf.
__device__ __forceinline__ void fma2(float& a0, float& a1, float w0, float w1, float x0, float x1) {
    asm("{\n\t.reg .b64 acc, w, x;\n\tmov.b64 acc, {%0, %1};\n\tmov.b64 w, {%2, %3};\n\t"
        "mov.b64 x, {%4, %5};\n\tfma.rn.f32x2 acc, w, x, acc;\n\tmov.b64 {%0, %1}, acc;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// (a0, a1) -= (b, b) as one paired instruction.
__device__ __forceinline__ void sub2(float& a0, float& a1, float b) {
    asm("{\n\t.reg .b64 v, s;\n\tmov.b64 v, {%0, %1};\n\tmov.b64 s, {%2, %2};\n\t"
        "sub.rn.f32x2 v, v, s;\n\tmov.b64 {%0, %1}, v;\n\t}"
        : "+f"(a0), "+f"(a1) : "f"(b));
}

// 8 int8 quants -> floats (see unpack_q8_raw).
__device__ __forceinline__ void unpack_q8x8_raw(const uint2 v, float* w) {
    const uint32_t u[2] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int b = 0; b < 4; b += 2) {
            float f0 = __int_as_float((int)__byte_perm(u[i], 0x4B000000u, 0x7540u + b));
            float f1 = __int_as_float((int)__byte_perm(u[i], 0x4B000000u, 0x7540u + b + 1));
            sub2(f0, f1, 8388736.0f);
            w[4 * i + b] = f0;
            w[4 * i + b + 1] = f1;
        }
    }
}

// 16 int8 quants -> their values as floats without an int-to-float conversion: each byte, biased
// by 128, becomes the low mantissa byte of 2^23 (exponent byte 0x4B), and 2^23 + 128 is
// subtracted exactly.
__device__ __forceinline__ void unpack_q8_raw(const uint4 v, float* w) {
    const uint32_t u[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int b = 0; b < 4; b += 2) {
            float f0 = __int_as_float((int)__byte_perm(u[i], 0x4B000000u, 0x7540u + b));
            float f1 = __int_as_float((int)__byte_perm(u[i], 0x4B000000u, 0x7540u + b + 1));
            sub2(f0, f1, 8388736.0f);
            w[4 * i + b] = f0;
            w[4 * i + b + 1] = f1;
        }
    }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try(bar, parity))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes),
        "r"(smem_u32(bar)), "l"(policy) : "memory");
}
template <int WT> struct Vec;
template <> struct Vec<W_F32>  { static constexpr int N = 4;  static constexpr int ES = 4; };
template <> struct Vec<W_F16>  { static constexpr int N = 8;  static constexpr int ES = 2; };
template <> struct Vec<W_BF16> { static constexpr int N = 8;  static constexpr int ES = 2; };
template <> struct Vec<W_Q8_0> { static constexpr int N = 16; static constexpr int ES = 1; };

template <int WT>
__device__ __forceinline__ void unpack16(const uint4 v, float d, float* w) {
    if constexpr (WT == W_F32) {
        w[0] = __uint_as_float(v.x); w[1] = __uint_as_float(v.y);
        w[2] = __uint_as_float(v.z); w[3] = __uint_as_float(v.w);
    } else if constexpr (WT == W_BF16) {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[2 * i] = __uint_as_float(u[i] << 16);
            w[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    } else if constexpr (WT == W_F16) {
        const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) { const float2 f = __half22float2(h[i]); w[2 * i] = f.x; w[2 * i + 1] = f.y; }
    } else {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int b = 0; b < 4; ++b) w[4 * i + b] = d * (float)(int8_t)((u[i] >> (8 * b)) & 0xffu);
    }
}

__device__ __forceinline__ unsigned long long pack_argmax(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

// One element of a weight matrix as float (F32 / F16 / BF16 / Q8_0 quants times their block scale).
__device__ __forceinline__ float load_elem(const DevMat& m, int64_t row, int64_t col) {
    const int64_t i = row * m.cols + col;
    switch (m.type) {
        case W_F32: return static_cast<const float*>(m.data)[i];
        case W_F16: return __half2float(static_cast<const __half*>(m.data)[i]);
        case W_BF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(m.data)[i]);
        default: {
            const float d = __half2float(m.scales[row * (m.cols / 32) + col / 32]);
            return d * (float)static_cast<const int8_t*>(m.data)[i];
        }
    }
}

// RoPE rotation of frequency theta at position pos as (cos, sin): the angle pos * theta in double,
// reduced to [-pi, pi] in double, then the float sine and cosine.
__device__ __forceinline__ float2 rope_cos_sin(int32_t pos, double theta) {
    const double ang = (double)pos * theta;
    const double r = ang - rint(ang * 0.15915494309189535) * 6.283185307179586;
    float s, c;
    sincosf((float)r, &s, &c);
    return make_float2(c, s);
}

}  // namespace dev
}  // namespace llm
