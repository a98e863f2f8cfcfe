// Grouped-query attention over the KV cache ([P2] "llama.cpp Architecture", Example 4:
// FLASH_ATTN_EXT of the query heads over the cached keys and values; Example 11: the unfused
// meaning MUL_MAT(K, Q) -> SOFT_MAX with the mask -> MUL_MAT with V).
//
// Work decomposition (built on the host): the ubatch's tokens are grouped by the list of cells
// they may read (one list per distinct sequence set), cut into query tiles of up to TQ tokens,
// and each tile's list is cut into work items (split-K over the cache). A block handles one work
// item for one KV head: the TQ x G query rows of that head group share every K/V row it stages
// in shared memory (16-byte loads of the gathered cells), so each cached row is read once per
// tile rather than once per query head. The softmax is online (running max and sum per row,
// base-2 exponent with log2(e)/sqrt(hd) folded into Q); a cell is visible to a row iff
// cell.pos <= token.pos. Each block writes its partial (o, m, l); the last block of a
// (tile, KV head) to finish (a self-resetting ticket) merges the partials and writes the output.
//
// These CUDA-core tiles serve F32 caches; F16 and Q8_0 caches take the tensor-core tiles
// (attn_mma.cu), and tiles of one token the cluster decode kernels (attn_decode.cu).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <climits>
#include <cmath>

#include "attn_common.cuh"
#include "kernels.h"

namespace llm {

namespace {

using namespace attn;

constexpr int kAttnWarps = 4;
constexpr int kBC = 32;                  // cells per shared-memory tile (one per lane)

template <int HD, int TQ, int G>
struct AttnSmem {
    static constexpr int R = TQ * G;
    static constexpr int RW = (R + kAttnWarps - 1) / kAttnWarps;
    static constexpr size_t q_floats = (size_t)R * HD;
    static constexpr size_t k_floats = (size_t)kBC * (HD + 1);
    static constexpr size_t v_floats = (size_t)kBC * HD;
    static constexpr size_t p_floats = (size_t)kAttnWarps * RW * kBC;
    static constexpr size_t bytes = (q_floats + k_floats + v_floats + p_floats) * sizeof(float) +
                                    (size_t)(2 * kBC + R + 8) * sizeof(int);
    // the merge reuses the q/k/v area
    static constexpr size_t merge_floats = q_floats + k_floats + v_floats;
};

template <int HD, int TQ, int G>
__global__ void __launch_bounds__(kAttnWarps * 32)
attn_kernel(AttnArgs a, float scale_log2) {
    using SM = AttnSmem<HD, TQ, G>;
    constexpr int R = SM::R, RW = SM::RW, DPL = HD / 32;
    extern __shared__ float smem[];
    float* qs = smem;                              // [R][HD]
    float* ks = qs + SM::q_floats;                 // [kBC][HD + 1]
    float* vs = ks + SM::k_floats;                 // [kBC][HD]
    float* ps = vs + SM::v_floats;                 // [warps][RW][kBC]
    int* cpos = reinterpret_cast<int*>(ps + SM::p_floats);   // [kBC]
    int* ccell = cpos + kBC;                       // [kBC] cell of each tile row (-1: none)
    int* rpos = ccell + kBC;                       // [R]
    int* flag = rpos + R;

    const int wi = blockIdx.x, kvh = blockIdx.y;
    // the plan (uploaded before the step's first kernel) can be read before the previous kernel
    // ends; Q and the cache rows it writes only after griddepcontrol.wait
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    const int n_work = a.hdr[0];
    const int4 wd = a.wi_desc[wi];                 // tile, first cell, end cell, partial row
    if (wi >= n_work) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int4 td0 = a.tile_desc[2 * wd.x];        // list, first token, tokens, first item
    const int4 td1 = a.tile_desc[2 * wd.x + 1];    // end item, list start, list length, -
    const int nq = td0.z, s0 = td0.y, c0 = wd.y, c1 = wd.z, base = td1.y;
    const float* K = static_cast<const float*>(a.kc) + (int64_t)kvh * a.n_ctx * HD;
    const float* V = static_cast<const float*>(a.vc) + (int64_t)kvh * a.n_ctx * HD;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    for (int idx = threadIdx.x; idx < R * HD; idx += blockDim.x) {
        const int r = idx / HD, d = idx % HD;
        const int j = r / G, g = r % G;
        float v = 0.f;
        if (j < nq) {
            const int t = a.perm[s0 + j];
            v = a.q[(int64_t)t * a.ldq + (kvh * G + g) * HD + d] * scale_log2;
        }
        qs[idx] = v;
    }
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int j = r / G;
        rpos[r] = j < nq ? a.tok_pos[a.perm[s0 + j]] : -1;
    }

    float m[RW], l[RW], o[RW][DPL];
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[i][e] = 0.f;
    }

    constexpr int EPV = 4;                               // floats per 16-byte vector
    constexpr int VPR = HD / EPV;                        // vectors per cached row
    for (int cb = c0; cb < c1; cb += kBC) {
        __syncthreads();
        if (threadIdx.x < kBC) {
            const int c = threadIdx.x;
            int cell = -1, cp = INT_MAX;
            if (cb + c < c1) {
                cell = a.list_cells[base + cb + c];
                cp = a.list_pos[base + cb + c];
                if (cell < 0 || cell >= a.n_ctx) cell = -1;
            }
            ccell[c] = cell;
            cpos[c] = cp;
        }
        __syncthreads();
#pragma unroll 4
        for (int v = threadIdx.x; v < kBC * VPR; v += blockDim.x) {
            const int c = v / VPR, j = v % VPR;
            const int cell = ccell[c];
            uint4 kq = make_uint4(0u, 0u, 0u, 0u), vq = kq;
            if (cell >= 0) {
                kq = __ldg(reinterpret_cast<const uint4*>(K + (int64_t)cell * HD) + j);
                vq = __ldg(reinterpret_cast<const uint4*>(V + (int64_t)cell * HD) + j);
            }
            const float* ke = reinterpret_cast<const float*>(&kq);
            const float* ve = reinterpret_cast<const float*>(&vq);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                ks[c * (HD + 1) + j * EPV + e] = ke[e];
                vs[c * HD + j * EPV + e] = ve[e];
            }
        }
        __syncthreads();

        const int mypos = cpos[lane];
        float* pw = ps + (size_t)warp * RW * kBC;
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const int r = warp * RW + i;
            float s = -INFINITY;
            if (r < R && mypos <= rpos[r]) {
                const float* qr = qs + r * HD;
                const float* kr = ks + lane * (HD + 1);
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll 8
                for (int d = 0; d < HD; d += 4) {
                    acc0 = fmaf(qr[d], kr[d], acc0);
                    acc1 = fmaf(qr[d + 1], kr[d + 1], acc1);
                    acc2 = fmaf(qr[d + 2], kr[d + 2], acc2);
                    acc3 = fmaf(qr[d + 3], kr[d + 3], acc3);
                }
                s = (acc0 + acc1) + (acc2 + acc3);
            }
            float mx = s;
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[i], mx);
            float p = 0.f, corr = 1.f;
            if (m_new != -INFINITY) {
                corr = exp2f(m[i] - m_new);
                p = exp2f(s - m_new);
            }
            float ssum = p;
            for (int off = 16; off > 0; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
            l[i] = l[i] * corr + ssum;
            m[i] = m_new;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[i][e] *= corr;
            pw[i * kBC + lane] = p;
        }
        __syncwarp();
#pragma unroll 4
        for (int c = 0; c < kBC; ++c) {
            float vv[DPL];
#pragma unroll
            for (int e = 0; e < DPL; ++e) vv[e] = vs[c * HD + lane + 32 * e];
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                const float p = pw[i * kBC + c];
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[i][e] = fmaf(p, vv[e], o[i][e]);
            }
        }
    }

    const int w0 = td0.w, w1 = td1.x;
    const int row0 = wd.w;
    if (w1 - w0 == 1) {                            // a single work item: normalise directly
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const int r = warp * RW + i;
            if (r >= nq * G) continue;
            const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
            const int t = a.perm[s0 + r / G];
#pragma unroll
            for (int e = 0; e < DPL; ++e)
                store_out(a, (int64_t)t * a.ldo + (kvh * G + r % G) * HD + lane + 32 * e, o[i][e] * inv);
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        const int r = warp * RW + i;
        if (r >= nq * G) continue;
        const int64_t row = (int64_t)(row0 + r) * a.Hkv + kvh;
        if (lane == 0) {
            a.part_m[row] = m[i];
            a.part_l[row] = l[i];
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) a.part_o[row * HD + lane + 32 * e] = o[i][e];
    }
    // the last block of this (tile, KV head) merges the partials
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        int* ticket = a.tickets + wd.x * a.Hkv + kvh;
        const int done = atomicAdd(ticket, 1) + 1;
        const bool last = done == w1 - w0;
        if (last) *ticket = 0;                     // ready for the next launch
        *flag = last ? 1 : 0;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    merge_tile<HD, G>(a, kvh, s0, nq, w0, w1, qs, SM::merge_floats);
}

template <int HD, int TQ, int G>
bool launch_tq(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    const size_t smem = AttnSmem<HD, TQ, G>::bytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_work, a.Hkv);
    cfg.blockDim = dim3(kAttnWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    if (a.kv_type != W_F32) return false;          // F16 and Q8_0 caches take the tensor-core tiles
    auto k = attn_kernel<HD, TQ, G>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
}

template <int HD, int G>
bool launch_hd_g(const AttnArgs& a, cudaStream_t st) {
    // tiles of one token: the cluster decode kernels; of several: the tensor-core tiles (F16, Q8_0)
    // or the CUDA-core tiles (F32)
    if (a.max_nq <= 1) return attention_decode_ok(a) && launch_attention_decode(a, st);
    if (a.tile_q == attention_tc_tile_q()) return attention_tc_ok(a) && launch_attention_tc(a, st);
    if (attention_mma_ok(a)) return launch_attention_mma(a, st);
    if (a.k_scale) return false;                   // the quant copies are for the tensor-core tiles
    return launch_tq<HD, kAttnTileQ, G>(a, st);
}

}  // namespace

bool launch_attention(const AttnArgs& a, cudaStream_t st) {
    if (a.n_work <= 0) return true;
    const int G = a.H / a.Hkv;
    if (G != 4) return false;
    switch (a.hd) {
        case 32: return launch_hd_g<32, 4>(a, st);
        case 64: return launch_hd_g<64, 4>(a, st);
        case 128: return launch_hd_g<128, 4>(a, st);
    }
    return false;
}

}  // namespace llm
