// Decode-step attention with a thread-block cluster per (query token, KV head) ([P2] "llama.cpp
// Architecture", Example 4 FLASH_ATTN_EXT; Example 11 for the unfused meaning).
//
// Every query tile of a decode ubatch holds one token. The kCL blocks of a cluster split the
// token's cell list into equal slices; each block runs the online softmax of the 4 query heads of
// its KV head over its slice (warp g = query head g, one cell per lane per 32 cells, hd/32 output
// dimensions per lane), leaves its partial state (m, l, o) in its own shared memory, and after a
// cluster barrier every block merges a kCL-th of the output dimensions by reading all partial
// states through distributed shared memory (mapa + ld.shared::cluster). A second cluster barrier
// keeps each block's shared memory alive until its peers have read it. No global round trip
// (fence, ticket, partial rows in L2) is on the merge path.
//
// A Q8_0 cache (int8 quants per row, one fp16 scale per 32 values in a separate array) is staged
// as int8 rows plus float scales; a score sums each 32-value block's products, then scales the
// block sum, and a value row's scale is folded into the probability of its cell.
//
// The K/V rows of cells written by earlier steps cannot change while the previous kernel (this
// step's Q/K/V projection) runs, so the first pass stages them with cp.async before
// griddepcontrol.wait; Q and this step's own cells are read after it.
//
// Control flow is uniform per cluster: all blocks of a cluster share the tile (blockIdx.z), the
// only early exit is the tile check, taken by the whole cluster before any cluster barrier.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "attn_common.cuh"
#include "kernels.h"

namespace llm {

namespace {

using namespace attn;

constexpr int kCL = 16;                  // blocks per cluster (non-portable size, opted in)
constexpr int kCH = 64;                  // cells per pass (two per lane)
constexpr int kGQ = 4;                   // query heads per KV head: one warp each

template <typename KT> __device__ __forceinline__ float kvf(KT v);
template <> __device__ __forceinline__ float kvf<float>(float v) { return v; }
template <> __device__ __forceinline__ float kvf<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float kvf<int8_t>(int8_t v) { return (float)v; }

__device__ __forceinline__ uint32_t sm32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A float in block `rank`'s shared memory at the address of `local` in this block's.
__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(sm32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// KT = int8_t: a Q8_0 cache (int8 quants per row, one fp16 scale per 32 values kept apart)
template <int HD, typename KT>
struct DecSmem {
    static constexpr bool Q8 = sizeof(KT) == 1;
    static constexpr int NB = HD / 32;                    // Q8_0 blocks per row
    static constexpr int RB = HD * (int)sizeof(KT);       // bytes of a cached row
    static constexpr int RS = RB + 16;                    // padded stride
    static constexpr size_t bytes = 2 * (size_t)kCH * RS + (size_t)kGQ * HD * 4 /* q */ +
                                    (size_t)kGQ * (HD + 2) * 4 /* partial */ + 3 * kCH * 4 +
                                    (Q8 ? 2 * (size_t)kCH * NB * 4 : 0) /* scales */ + 16;
};


}  // namespace

template <int HD, typename KT>
__global__ void __launch_bounds__(kGQ * 32)
attn_decode_kernel(AttnArgs a, float scale_log2) {
    using SM = DecSmem<HD, KT>;
    constexpr int RB = SM::RB, RS = SM::RS, VPR = RB / 16, DPL = HD / 32, NB = SM::NB;
    constexpr bool Q8 = SM::Q8;
    extern __shared__ __align__(16) uint8_t sm[];
    uint8_t* kb = sm;                                          // [kCH][RS]
    uint8_t* vb = kb + kCH * RS;                               // [kCH][RS]
    float* qs = reinterpret_cast<float*>(vb + kCH * RS);       // [kGQ][HD]
    float* pst = qs + kGQ * HD;                                // partial: m[kGQ], l[kGQ], o[kGQ][HD]
    int* ccell = reinterpret_cast<int*>(pst + kGQ * (HD + 2)); // [kCH]
    int* cvis = ccell + kCH;                                   // [kCH]
    int* cfresh = cvis + kCH;                                  // [kCH]
    float* ksc = reinterpret_cast<float*>(cfresh + kCH);       // Q8_0: [kCH][NB] K scales
    float* vsc = ksc + kCH * NB;                               //        [kCH][NB] V scales

    const uint32_t rank = cluster_rank();
    const int kvh = blockIdx.y, tile = blockIdx.z;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    // the plan was uploaded before the step's first kernel: readable before griddepcontrol.wait
    if (tile >= a.hdr[1]) return;                               // whole cluster (same tile)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int4 td0 = a.tile_desc[2 * tile];
    const int4 td1 = a.tile_desc[2 * tile + 1];
    const int base = td1.y, len = td1.z;
    const int t = a.perm[td0.y];
    const int tpos = a.tok_pos[t];
    const int chunk = (len + kCL - 1) / kCL;
    const int c0 = min(len, (int)rank * chunk), c1 = min(len, c0 + chunk);
    const uint8_t* K = static_cast<const uint8_t*>(a.kc) + (int64_t)kvh * a.n_ctx * RB;
    const uint8_t* V = static_cast<const uint8_t*>(a.vc) + (int64_t)kvh * a.n_ctx * RB;
    const __half* KS = q8_scales(a.kc, a, kvh);
    const __half* VS = q8_scales(a.vc, a, kvh);
    auto load_scales = [&](int c, int cell) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            ksc[c * NB + b] = ld_scale(KS + (int64_t)cell * NB + b);
            vsc[c * NB + b] = ld_scale(VS + (int64_t)cell * NB + b);
        }
    };

    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.f;
    bool waited = false;
    // at least one (possibly empty) pass, so the first wait always happens inside the loop
    for (int cb = c0; cb < c1 || (cb == c0 && !waited); cb += kCH) {
        if (threadIdx.x < kCH) {
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
            if constexpr (Q8) {
                if (vis && cell >= 0 && !fresh) load_scales(threadIdx.x, cell);
            }
        }
        __syncthreads();
        // rows of earlier steps: staged now, possibly before the previous kernel has ended
        for (int v = threadIdx.x; v < kCH * VPR; v += blockDim.x) {
            const int c = v / VPR, j = v % VPR;
            if (!cvis[c] || cfresh[c]) continue;
            const size_t src = (size_t)ccell[c] * RB + j * 16;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm32(kb + c * RS + j * 16)), "l"(K + src) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm32(vb + c * RS + j * 16)), "l"(V + src) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (!waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
            for (int i = threadIdx.x; i < kGQ * HD; i += blockDim.x)
                qs[i] = a.q[(int64_t)t * a.ldq + (kvh * kGQ + i / HD) * HD + i % HD] * scale_log2;
        }
        // rows written by this step's projection kernel: only now
        if constexpr (Q8) {
            if (threadIdx.x < kCH && cvis[threadIdx.x] && cfresh[threadIdx.x])
                load_scales(threadIdx.x, ccell[threadIdx.x]);
        }
        for (int v = threadIdx.x; v < kCH * VPR; v += blockDim.x) {
            const int c = v / VPR, j = v % VPR;
            if (!cvis[c] || !cfresh[c]) continue;
            const size_t src = (size_t)ccell[c] * RB + j * 16;
            *reinterpret_cast<uint4*>(kb + c * RS + j * 16) = __ldcg(reinterpret_cast<const uint4*>(K + src));
            *reinterpret_cast<uint4*>(vb + c * RS + j * 16) = __ldcg(reinterpret_cast<const uint4*>(V + src));
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
            if (Q8 && cvis[c]) {
                const uint8_t* kr = kb + c * RS;
                float acc = 0.f;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    float p0 = 0.f, p1 = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int j = 2 * b + jj;
                        const uint4 kv = *reinterpret_cast<const uint4*>(kr + j * 16);
                        const int8_t* ke = reinterpret_cast<const int8_t*>(&kv);
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            p0 = fmaf(q[j * 16 + e], (float)ke[e], p0);
                            p1 = fmaf(q[j * 16 + e + 1], (float)ke[e + 1], p1);
                        }
                    }
                    acc = fmaf(ksc[c * NB + b], p0 + p1, acc);
                }
                s[h2] = acc;
            } else if (cvis[c]) {
                const uint8_t* kr = kb + c * RS;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int j = 0; j < VPR; ++j) {
                    const uint4 kv = *reinterpret_cast<const uint4*>(kr + j * 16);
                    const KT* ke = reinterpret_cast<const KT*>(&kv);
                    constexpr int EPV = 16 / (int)sizeof(KT);
#pragma unroll
                    for (int e = 0; e < EPV; e += 2) {
                        a0 = fmaf(q[j * EPV + e], kvf<KT>(ke[e]), a0);
                        a1 = fmaf(q[j * EPV + e + 1], kvf<KT>(ke[e + 1]), a1);
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
        for (int c = 0; c < kCH; ++c) {
            const float pc = __shfl_sync(0xffffffffu, p[c >> 5], c & 31);
            if (pc == 0.f) continue;
            const KT* vr = reinterpret_cast<const KT*>(vb + c * RS) + lane * DPL;
            const float pd = Q8 ? pc * vsc[c * NB + lane * DPL / 32] : pc;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(pd, kvf<KT>(vr[e]), o[e]);
        }
        __syncthreads();
    }

    // this block's partial state of its 4 query heads, then the cluster-wide merge
    float* pm = pst;
    float* pl = pst + kGQ;
    float* po = pst + 2 * kGQ;
    if (lane == 0) { pm[warp] = m; pl[warp] = l; }
#pragma unroll
    for (int e = 0; e < DPL; ++e) po[warp * HD + lane * DPL + e] = o[e];
    cluster_sync_all();
    constexpr int OPB = kGQ * HD / kCL;                        // outputs merged per block
    for (int i = threadIdx.x; i < OPB; i += blockDim.x) {
        const int idx = (int)rank * OPB + i;
        const int g = idx / HD, dd = idx % HD;
        float M = -INFINITY;
#pragma unroll
        for (uint32_t r = 0; r < kCL; ++r) M = fmaxf(M, ld_peer(pm + g, r));
        float L = 0.f, O = 0.f;
#pragma unroll
        for (uint32_t r = 0; r < kCL; ++r) {
            const float mr = ld_peer(pm + g, r);
            const float f = (M == -INFINITY || mr == -INFINITY) ? 0.f : exp2f(mr - M);
            L = fmaf(f, ld_peer(pl + g, r), L);
            O = fmaf(f, ld_peer(po + g * HD + dd, r), O);
        }
        store_out(a, (int64_t)t * a.ldo + (kvh * kGQ + g) * HD + dd, L > 0.f ? O / L : 0.f);
    }
    cluster_sync_all();                                         // peers are done reading
}

template <int HD, typename KT>
bool launch_dec(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    constexpr size_t smem = DecSmem<HD, KT>::bytes;
    auto k = attn_decode_kernel<HD, KT>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return false;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCL, a.Hkv, a.n_tok);
    cfg.blockDim = dim3(kGQ * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr_l[2];
    attr_l[0].id = cudaLaunchAttributeClusterDimension;
    attr_l[0].val.clusterDim.x = kCL;
    attr_l[0].val.clusterDim.y = 1;
    attr_l[0].val.clusterDim.z = 1;
    attr_l[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr_l[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr_l;
    cfg.numAttrs = a.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
}

bool attention_decode_ok(const AttnArgs& a) {
    return a.H == kGQ * a.Hkv && (a.hd == 32 || a.hd == 64 || a.hd == 128) && a.n_tok >= 1 &&
           a.n_tok <= 65535 && a.slot != nullptr;
}

bool launch_attention_decode(const AttnArgs& a, cudaStream_t st) {
    if (a.kv_type == W_Q8_0) {
        switch (a.hd) {
            case 32: return launch_dec<32, int8_t>(a, st);
            case 64: return launch_dec<64, int8_t>(a, st);
            case 128: return launch_dec<128, int8_t>(a, st);
        }
        return false;
    }
    const bool f32 = a.kv_type == W_F32;
    switch (a.hd) {
        case 32: return f32 ? launch_dec<32, float>(a, st) : launch_dec<32, __half>(a, st);
        case 64: return f32 ? launch_dec<64, float>(a, st) : launch_dec<64, __half>(a, st);
        case 128: return f32 ? launch_dec<128, float>(a, st) : launch_dec<128, __half>(a, st);
    }
    return false;
}

}  // namespace llm
