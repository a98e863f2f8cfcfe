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

template <typename KT> __device__ __forceinline__ float kv_to_f(KT v);
template <> __device__ __forceinline__ float kv_to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float kv_to_f<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float kv_to_f<int8_t>(int8_t v) { return (float)v; }

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

template <int HD, int TQ, int G, typename KT>
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
    const KT* K = static_cast<const KT*>(a.kc) + (int64_t)kvh * a.n_ctx * HD;
    const KT* V = static_cast<const KT*>(a.vc) + (int64_t)kvh * a.n_ctx * HD;
    constexpr bool Q8 = sizeof(KT) == 1;           // Q8_0: int8 quants and fp16 scales per 32 values
    const __half* KS = Q8 ? q8_scales(a.kc, a, kvh) : nullptr;
    const __half* VS = Q8 ? q8_scales(a.vc, a, kvh) : nullptr;
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

    constexpr int EPV = 16 / (int)sizeof(KT);          // elements per 16-byte vector
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
            float dk = 1.f, dv = 1.f;
            if (cell >= 0) {
                kq = __ldg(reinterpret_cast<const uint4*>(K + (int64_t)cell * HD) + j);
                vq = __ldg(reinterpret_cast<const uint4*>(V + (int64_t)cell * HD) + j);
                if constexpr (Q8) {                  // 16 quants: half of one 32-value block
                    dk = ld_scale(KS + (int64_t)cell * (HD / 32) + j / 2);
                    dv = ld_scale(VS + (int64_t)cell * (HD / 32) + j / 2);
                }
            }
            const KT* ke = reinterpret_cast<const KT*>(&kq);
            const KT* ve = reinterpret_cast<const KT*>(&vq);
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                if constexpr (Q8) {
                    ks[c * (HD + 1) + j * EPV + e] = dk * kv_to_f<KT>(ke[e]);
                    vs[c * HD + j * EPV + e] = dv * kv_to_f<KT>(ve[e]);
                } else {
                    ks[c * (HD + 1) + j * EPV + e] = kv_to_f<KT>(ke[e]);
                    vs[c * HD + j * EPV + e] = kv_to_f<KT>(ve[e]);
                }
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

// Decode-step attention (every query tile holds one token). The K/V rows of cells written by
// earlier steps cannot change while the previous kernel (this step's Q/K/V projection) runs, so
// the block stages them (cp.async, padded rows) before griddepcontrol.wait; only Q and the cells
// written by this step are read after it. Grid (KV head, work item): the active blocks come first.
// Warp g handles query head g of the group: scores with one cell per lane, softmax, then V with
// each lane owning HD/32 output dimensions.
template <int HD, int G, typename KT>
__global__ void __launch_bounds__(128)
attn_step_kernel(AttnArgs a, float scale_log2) {
    constexpr int CH = 64;                                  // cells staged per pass
    constexpr int RB = HD * (int)sizeof(KT);                // bytes of a cached row
    constexpr int RS = RB + 16;                             // padded row stride
    constexpr int VPR = RB / 16;                            // 16-byte chunks per row
    constexpr int DPL = HD / 32;
    static_assert(G == 4, "one warp per query head of the group");
    extern __shared__ __align__(16) uint8_t sm[];
    uint8_t* kb = sm;                                       // [CH][RS]
    uint8_t* vb = kb + CH * RS;                             // [CH][RS]
    float* qs = reinterpret_cast<float*>(vb + CH * RS);     // [G][HD]
    int* ccell = reinterpret_cast<int*>(qs + G * HD);       // [CH]
    int* cvis = ccell + CH;                                 // [CH] visible
    int* cfresh = cvis + CH;                                // [CH] written by this step
    int* flag = cfresh + CH;

    const int kvh = blockIdx.x, wi = blockIdx.y;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    const int n_work = a.hdr[0];
    const int4 wd = a.wi_desc[wi];
    if (wi >= n_work) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int4 td0 = a.tile_desc[2 * wd.x];
    const int4 td1 = a.tile_desc[2 * wd.x + 1];
    const int s0 = td0.y, base = td1.y, c0 = wd.y, c1 = wd.z;
    const int t = a.perm[s0];
    const int tpos = a.tok_pos[t];
    const uint8_t* K = static_cast<const uint8_t*>(a.kc) + (int64_t)kvh * a.n_ctx * RB;
    const uint8_t* V = static_cast<const uint8_t*>(a.vc) + (int64_t)kvh * a.n_ctx * RB;

    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.f;
    bool waited = false;
    for (int cb = c0; cb < c1; cb += CH) {
        if (threadIdx.x < CH) {
            const int ci = cb + threadIdx.x;
            int cell = -1, vis = 0, fresh = 0;
            if (ci < c1) {
                const int cc = a.list_cells[base + ci];
                if (cc >= 0 && cc < a.n_ctx) {
                    cell = cc;
                    vis = a.list_pos[base + ci] <= tpos;
                    for (int j = 0; j < a.n_tok; ++j) fresh |= a.slot[j] == cc;
                }
            }
            ccell[threadIdx.x] = cell;
            cvis[threadIdx.x] = vis && cell >= 0;
            cfresh[threadIdx.x] = fresh;
        }
        __syncthreads();
        // rows of earlier steps: staged now, possibly before the previous kernel has ended
        for (int v = threadIdx.x; v < CH * VPR; v += blockDim.x) {
            const int c = v / VPR, j = v % VPR;
            if (!cvis[c] || cfresh[c]) continue;
            const size_t src = (size_t)ccell[c] * RB + j * 16;
            const uint32_t dk = (uint32_t)__cvta_generic_to_shared(kb + c * RS + j * 16);
            const uint32_t dv = (uint32_t)__cvta_generic_to_shared(vb + c * RS + j * 16);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dk), "l"(K + src) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dv), "l"(V + src) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (!waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
            for (int i = threadIdx.x; i < G * HD; i += blockDim.x)
                qs[i] = a.q[(int64_t)t * a.ldq + (kvh * G + i / HD) * HD + i % HD] * scale_log2;
        }
        // rows written by this step's projection kernel: only now
        for (int v = threadIdx.x; v < CH * VPR; v += blockDim.x) {
            const int c = v / VPR, j = v % VPR;
            if (!cvis[c] || !cfresh[c]) continue;
            const size_t src = (size_t)ccell[c] * RB + j * 16;
            *reinterpret_cast<uint4*>(kb + c * RS + j * 16) = *reinterpret_cast<const uint4*>(K + src);
            *reinterpret_cast<uint4*>(vb + c * RS + j * 16) = *reinterpret_cast<const uint4*>(V + src);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();

        // scores of query head `warp`: lanes own cells lane and lane + 32
        const float* q = qs + warp * HD;
        float s[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int c = lane + 32 * h2;
            s[h2] = -INFINITY;
            if (cvis[c]) {
                const uint8_t* kr = kb + c * RS;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int j = 0; j < VPR; ++j) {
                    const uint4 kv = *reinterpret_cast<const uint4*>(kr + j * 16);
                    const KT* ke = reinterpret_cast<const KT*>(&kv);
                    constexpr int EPV = 16 / (int)sizeof(KT);
#pragma unroll
                    for (int e = 0; e < EPV; e += 2) {
                        a0 = fmaf(q[j * EPV + e], kv_to_f<KT>(ke[e]), a0);
                        a1 = fmaf(q[j * EPV + e + 1], kv_to_f<KT>(ke[e + 1]), a1);
                    }
                }
                s[h2] = a0 + a1;
            }
        }
        float mx = fmaxf(s[0], s[1]);
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        float p[2] = {0.f, 0.f}, corr = 1.f;
        if (m_new != -INFINITY) {
            corr = exp2f(m - m_new);
            p[0] = exp2f(s[0] - m_new);
            p[1] = exp2f(s[1] - m_new);
        }
        float ps = p[0] + p[1];
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = l * corr + ps;
        m = m_new;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] *= corr;
#pragma unroll 4
        for (int c = 0; c < CH; ++c) {
            const float pc = __shfl_sync(0xffffffffu, p[c >> 5], c & 31);
            if (pc == 0.f) continue;
            const KT* vr = reinterpret_cast<const KT*>(vb + c * RS) + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(pc, kv_to_f<KT>(vr[e]), o[e]);
        }
        __syncthreads();
    }
    if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");

    const int w0 = td0.w, w1 = td1.x;
    const int g = warp;
    if (w1 - w0 == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            store_out(a, (int64_t)t * a.ldo + (kvh * G + g) * HD + lane * DPL + e, o[e] * inv);
        return;
    }
    const int64_t row = (int64_t)(wd.w + g) * a.Hkv + kvh;
    if (lane == 0) {
        a.part_m[row] = m;
        a.part_l[row] = l;
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) a.part_o[row * HD + lane * DPL + e] = o[e];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        int* ticket = a.tickets + wd.x * a.Hkv + kvh;
        const int done = atomicAdd(ticket, 1) + 1;
        const bool last = done == w1 - w0;
        if (last) *ticket = 0;
        *flag = last ? 1 : 0;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    merge_tile<HD, G>(a, kvh, s0, 1, w0, w1, reinterpret_cast<float*>(sm), (size_t)(2 * CH * RS) / 4);
}

template <int HD, int G>
bool launch_step(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.Hkv, a.n_work);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    if (a.kv_type == W_F32) {
        constexpr size_t smem = 2 * 64 * (HD * 4 + 16) + G * HD * 4 + 4 * 64 * 4 + 16;
        auto k = attn_step_kernel<HD, G, float>;
        cfg.dynamicSmemBytes = smem;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
    }
    constexpr size_t smem = 2 * 64 * (HD * 2 + 16) + G * HD * 4 + 4 * 64 * 4 + 16;
    auto k = attn_step_kernel<HD, G, __half>;
    cfg.dynamicSmemBytes = smem;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
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
    if (a.kv_type == W_F32) {
        auto k = attn_kernel<HD, TQ, G, float>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
    }
    if (a.kv_type == W_Q8_0) {
        auto k = attn_kernel<HD, TQ, G, int8_t>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
    }
    auto k = attn_kernel<HD, TQ, G, __half>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
}

template <int HD, int G>
bool launch_hd_g(const AttnArgs& a, cudaStream_t st) {
    if (a.max_nq <= 1) {
        if (a.slot && attention_decode_ok(a)) return launch_attention_decode(a, st);
        return a.slot && a.kv_type != W_Q8_0 ? launch_step<HD, G>(a, st) : launch_tq<HD, 1, G>(a, st);
    }
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
