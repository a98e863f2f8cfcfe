// Device pieces shared by the attention kernels: Q8_0 cache scales, the output store (float32, or
// bf16 hi + lo terms for the tensor-core GEMM that follows) and the merge of split-K partial
// states.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace llm {
namespace attn {

// ---- warp-level tensor-core pieces (mma.sync m16n8k16, f16 inputs, f32 accumulators)
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// x = hi + lo with hi, lo f16 (lo the rounding error of hi)
__device__ __forceinline__ void split_h2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_h2(x0 - hf.x, x1 - hf.y);
}
// d += a b (A 16x16 row-major fragment, B 16x8 column fragment)
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// A Q8_0 cache scale (fp16), read through L2: it may have been written by the previous kernel.
__device__ __forceinline__ float ld_scale(const __half* p) {
    return __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short*>(p))));
}

// The fp16 scales of KV head kvh in a Q8_0 layer cache (quants first, then the scales).
__device__ __forceinline__ const __half* q8_scales(const void* layer, const AttnArgs& a, int kvh) {
    return reinterpret_cast<const __half*>(static_cast<const uint8_t*>(layer) +
                                           kv_q8_scale_offset(a.Hkv, a.n_ctx, a.hd)) +
           (int64_t)kvh * a.n_ctx * (a.hd / 32);
}

__device__ __forceinline__ void store_out(const AttnArgs& a, int64_t oi, float v) {
    if (a.out_b && a.out_f16) {
        static_cast<__half*>(a.out_b)[oi] = __float2half_rn(v);
    } else if (a.out_b) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        static_cast<__nv_bfloat16*>(a.out_b)[oi] = hi;
        if (a.out_b_lo)
            static_cast<__nv_bfloat16*>(a.out_b_lo)[oi] = __float2bfloat16_rn(v - __bfloat162float(hi));
    } else {
        a.out[oi] = v;
    }
}

// Merge the partials of work items [w0, w1) of one tile and KV head into the output rows.
template <int HD, int G>
__device__ void merge_tile(const AttnArgs& a, int kvh, int s0, int nq, int w0, int w1,
                           float* scratch, size_t scratch_floats) {
    const int R = nq * G, NW = w1 - w0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((size_t)R * NW + NW <= scratch_floats) {
        float* wgt = scratch;                                  // [R][NW]
        int* roff = reinterpret_cast<int*>(scratch + (size_t)R * NW);
        __syncthreads();
        for (int w = threadIdx.x; w < NW; w += blockDim.x) roff[w] = a.wi_desc[w0 + w].w;
        __syncthreads();
        for (int r = warp; r < R; r += blockDim.x / 32) {
            float M = -INFINITY;
            for (int w = lane; w < NW; w += 32) {
                const float mw = a.part_m[(int64_t)(roff[w] + r) * a.Hkv + kvh];
                wgt[r * NW + w] = mw;
                M = fmaxf(M, mw);
            }
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float L = 0.f;
            for (int w = lane; w < NW; w += 32) {
                const float mw = wgt[r * NW + w];
                const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - M);
                L += f * a.part_l[(int64_t)(roff[w] + r) * a.Hkv + kvh];
                wgt[r * NW + w] = f;
            }
            for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            const float inv = L > 0.f ? 1.f / L : 0.f;
            for (int w = lane; w < NW; w += 32) wgt[r * NW + w] *= inv;
        }
        __syncthreads();
        // each thread owns outputs idx = threadIdx.x + j * blockDim.x; the partial rows of eight
        // work items are loaded for all of them before any is used
        constexpr int kOut = 4;
        for (int base_idx = 0; base_idx < R * HD; base_idx += kOut * (int)blockDim.x) {
            float O[kOut];
            int rr[kOut], dd[kOut];
            bool live[kOut];
#pragma unroll
            for (int j = 0; j < kOut; ++j) {
                const int idx = base_idx + j * blockDim.x + threadIdx.x;
                live[j] = idx < R * HD;
                rr[j] = live[j] ? idx / HD : 0;
                dd[j] = live[j] ? idx % HD : 0;
                O[j] = 0.f;
            }
            for (int w0b = 0; w0b < NW; w0b += 8) {
                float pv[8][kOut];
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int j = 0; j < kOut; ++j)
                        pv[u][j] = (w0b + u < NW && live[j])
                            ? a.part_o[((int64_t)(roff[w0b + u] + rr[j]) * a.Hkv + kvh) * HD + dd[j]]
                            : 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int j = 0; j < kOut; ++j)
                        if (w0b + u < NW) O[j] = fmaf(wgt[rr[j] * NW + w0b + u], pv[u][j], O[j]);
            }
#pragma unroll
            for (int j = 0; j < kOut; ++j) {
                if (!live[j]) continue;
                const int t = a.perm[s0 + rr[j] / G];
                store_out(a, (int64_t)t * a.ldo + (kvh * G + rr[j] % G) * HD + dd[j], O[j]);
            }
        }
        return;
    }
    for (int idx = threadIdx.x; idx < R * HD; idx += blockDim.x) {
        const int r = idx / HD, d = idx % HD;
        float M = -INFINITY;
        for (int w = w0; w < w1; ++w)
            M = fmaxf(M, a.part_m[(int64_t)(a.wi_desc[w].w + r) * a.Hkv + kvh]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int w = w0; w < w1; ++w) {
                const int64_t row = (int64_t)(a.wi_desc[w].w + r) * a.Hkv + kvh;
                const float mw = a.part_m[row];
                if (mw == -INFINITY) continue;
                const float f = exp2f(mw - M);
                L += f * a.part_l[row];
                O += f * a.part_o[row * HD + d];
            }
        }
        const int t = a.perm[s0 + r / G];
        store_out(a, (int64_t)t * a.ldo + (kvh * G + r % G) * HD + d, L > 0.f ? O / L : 0.f);
    }
}

}  // namespace attn
}  // namespace llm
