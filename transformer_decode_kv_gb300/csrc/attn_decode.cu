// Decode-step attention with a thread-block cluster per (query token, KV head) ([P2] "llama.cpp
// Architecture", Example 4 FLASH_ATTN_EXT; Example 11 for the unfused meaning).
//
// Every query tile of a decode ubatch holds one token. The kCL blocks of a cluster split the
// token's cell list into equal slices and walk them in passes of 64 cells; each block runs the
// online softmax of the 4 query heads of its KV head over its slice, leaves its partial state
// (m, l, o) in its own shared memory, and after a cluster barrier every block merges a kCL-th of
// the output dimensions by reading all partial states through distributed shared memory (mapa +
// ld.shared::cluster). A second cluster barrier keeps each block's shared memory alive until its
// peers have read it. No global round trip (fence, ticket, partial rows in L2) is on the merge
// path. F16 and Q8_0 caches run the contractions on tensor cores (attn_decode_mma_kernel); F32
// caches on CUDA cores (attn_decode_kernel).
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
constexpr int kCH = 64;                  // cells per pass
constexpr int kGQ = 4;                   // query heads per KV head: one warp each per group
constexpr int kGroups = 2;               // warp groups, each taking half of every pass
constexpr int kCG = kCH / kGroups;       // cells per group and pass: one per lane
constexpr int kThreads = kGQ * 32 * kGroups;

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

// The F32-cache kernel's shared memory: two stages of one pass (K rows, V rows, then per cell:
// cell, visible, fresh), Q, and the block and group partial states.
template <int HD>
struct DecSmem {
    static constexpr int RB = HD * 4;                     // bytes of a cached row
    static constexpr int RS = RB + 16;                    // padded stride
    static constexpr size_t rows = 2 * (size_t)kCH * RS;
    static constexpr size_t stage = rows + 3 * kCH * 4;
    static constexpr size_t bytes = 2 * stage + (size_t)kGQ * HD * 4 /* q */ +
                                    2 * (size_t)kGQ * (HD + 2) * 4 /* block and group partials */ + 16;
};

struct Stage {
    uint8_t* kb;
    uint8_t* vb;
    int* ccell;
    int* cvis;
    int* cfresh;
};

}  // namespace

// F32 caches, on CUDA cores. Two warp groups: group g takes cells [32 g, 32 g + 32) of every
// pass of 64 (one cell per lane for the scores), warp g * 4 + h holds query head h of the KV
// head's group. Passes are double buffered: the rows of pass i + 1 are in flight while pass i is
// computed.
template <int HD>
__global__ void __launch_bounds__(kThreads)
attn_decode_kernel(AttnArgs a, float scale_log2) {
    using SM = DecSmem<HD>;
    constexpr int RB = SM::RB, RS = SM::RS, VPR = RB / 16, DPL = HD / 32;
    extern __shared__ __align__(16) uint8_t sm[];
    auto stage_of = [&](int s) {
        uint8_t* b = sm + (size_t)s * SM::stage;
        Stage S;
        S.kb = b;
        S.vb = b + kCH * RS;
        S.ccell = reinterpret_cast<int*>(b + SM::rows);
        S.cvis = S.ccell + kCH;
        S.cfresh = S.cvis + kCH;
        return S;
    };
    float* qs = reinterpret_cast<float*>(sm + 2 * SM::stage);          // [kGQ][HD]
    float* pst = qs + kGQ * HD;                                         // block partial (peers read it)
    float* gst = pst + kGQ * (HD + 2);                                  // group 1's partial

    const uint32_t rank = cluster_rank();
    const int kvh = blockIdx.y, tile = blockIdx.z;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    // the plan was uploaded before the step's first kernel: readable before griddepcontrol.wait
    if (tile >= a.hdr[1]) return;                               // whole cluster (same tile)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = warp / kGQ, hq = warp % kGQ;
    const int4 td0 = a.tile_desc[2 * tile];
    const int4 td1 = a.tile_desc[2 * tile + 1];
    const int base = td1.y, len = td1.z;
    const int t = a.perm[td0.y];
    const int tpos = a.tok_pos[t];
    const int chunk = (len + kCL - 1) / kCL;
    const int c0 = min(len, (int)rank * chunk), c1 = min(len, c0 + chunk);
    const int npass = c1 > c0 ? (c1 - c0 + kCH - 1) / kCH : 1;  // at least one: the wait is in it
    const uint8_t* K = static_cast<const uint8_t*>(a.kc) + (int64_t)kvh * a.n_ctx * RB;
    const uint8_t* V = static_cast<const uint8_t*>(a.vc) + (int64_t)kvh * a.n_ctx * RB;
    // The list entry (cell, position) of the next pass to set up is fetched into registers one
    // pass ahead, so setting up a stage waits on no global load.
    int pf_cell = -1, pf_pos = 0;
    auto fetch = [&](int i) {
        if (threadIdx.x < kCH) {
            const int ci = c0 + i * kCH + threadIdx.x;
            pf_cell = -1;
            pf_pos = 0;
            if (ci < c1) {
                pf_cell = a.list_cells[base + ci];
                pf_pos = a.list_pos[base + ci];
            }
        }
    };
    auto setup = [&](const Stage& S) {
        if (threadIdx.x < kCH) {
            int cell = -1, vis = 0, fresh = 0;
            if (pf_cell >= 0 && pf_cell < a.n_ctx) {
                cell = pf_cell;
                vis = pf_pos <= tpos;
                for (int j = 0; j < a.n_tok; ++j) fresh |= a.slot[j] == cell;
            }
            S.ccell[threadIdx.x] = cell;
            S.cvis[threadIdx.x] = vis && cell >= 0;
            S.cfresh[threadIdx.x] = fresh;
        }
    };
    auto issue = [&](const Stage& S, bool pre_wait) {
        for (int v = threadIdx.x; v < kCH * VPR; v += kThreads) {
            const int c = v / VPR, j = v % VPR;
            if (!S.cvis[c] || (pre_wait && S.cfresh[c])) continue;
            const size_t src = (size_t)S.ccell[c] * RB + j * 16;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm32(S.kb + c * RS + j * 16)), "l"(K + src) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm32(S.vb + c * RS + j * 16)), "l"(V + src) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    // pass 0: rows of earlier steps staged now, possibly before the previous kernel has ended
    {
        const Stage S0 = stage_of(0);
        fetch(0);
        setup(S0);
        __syncthreads();
        issue(S0, true);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (npass > 1) fetch(1);
        for (int i = threadIdx.x; i < kGQ * HD; i += kThreads)
            qs[i] = a.q[(int64_t)t * a.ldq + (kvh * kGQ + i / HD) * HD + i % HD] * scale_log2;
        // rows written by this step's projection kernel: only now
        for (int v = threadIdx.x; v < kCH * VPR; v += kThreads) {
            const int c = v / VPR, j = v % VPR;
            if (!S0.cvis[c] || !S0.cfresh[c]) continue;
            const size_t src = (size_t)S0.ccell[c] * RB + j * 16;
            *reinterpret_cast<uint4*>(S0.kb + c * RS + j * 16) = __ldcg(reinterpret_cast<const uint4*>(K + src));
            *reinterpret_cast<uint4*>(S0.vb + c * RS + j * 16) = __ldcg(reinterpret_cast<const uint4*>(V + src));
        }
    }

    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.f;
    const float* q = qs + hq * HD;
    for (int i = 0; i < npass; ++i) {
        const Stage S = stage_of(i & 1);
        if (i + 1 < npass) {
            // the other stage was last read by pass i - 1, which ended at the barrier below
            const Stage N = stage_of((i + 1) & 1);
            setup(N);
            if (i + 2 < npass) fetch(i + 2);
            __syncthreads();
            issue(N, false);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();

        // score of this lane's cell for query head hq
        const int c = grp * kCG + lane;
        float s = -INFINITY;
        if (S.cvis[c]) {
            const uint8_t* kr = S.kb + c * RS;
            {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int j = 0; j < VPR; ++j) {
                    const float4 kv = *reinterpret_cast<const float4*>(kr + j * 16);
                    const float4 qv = *reinterpret_cast<const float4*>(q + j * 4);   // broadcast
                    a0 = fmaf(qv.x, kv.x, a0);
                    a1 = fmaf(qv.y, kv.y, a1);
                    a0 = fmaf(qv.z, kv.z, a0);
                    a1 = fmaf(qv.w, kv.w, a1);
                }
                s = a0 + a1;
            }
        }
        float mx = s;
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        float p = 0.f, corr = 1.f;
        if (m_new != -INFINITY) {
            corr = exp2f(m - m_new);
            p = exp2f(s - m_new);
        }
        float ps = p;
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = l * corr + ps;
        m = m_new;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] *= corr;
#pragma unroll 4
        for (int k = 0; k < kCG; ++k) {
            const float pc = __shfl_sync(0xffffffffu, p, k);
            if (pc == 0.f) continue;
            const int c2 = grp * kCG + k;
            const float* vr = reinterpret_cast<const float*>(S.vb + c2 * RS) + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[e] = fmaf(pc, vr[e], o[e]);
        }
        __syncthreads();                                        // stage S free for pass i + 2
    }

    // the two groups' states merge into this block's partial, then the cluster-wide merge
    float* pm = pst;
    float* pl = pst + kGQ;
    float* po = pst + 2 * kGQ;
    if (grp == 1) {
        if (lane == 0) { gst[hq] = m; gst[kGQ + hq] = l; }
#pragma unroll
        for (int e = 0; e < DPL; ++e) gst[2 * kGQ + hq * HD + lane * DPL + e] = o[e];
    }
    __syncthreads();
    if (grp == 0) {
        const float m1 = gst[hq], l1 = gst[kGQ + hq];
        const float M = fmaxf(m, m1);
        const float f0 = m == -INFINITY ? 0.f : exp2f(m - M);
        const float f1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
        if (lane == 0) { pm[hq] = M; pl[hq] = l * f0 + l1 * f1; }
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            po[hq * HD + lane * DPL + e] = o[e] * f0 + gst[2 * kGQ + hq * HD + lane * DPL + e] * f1;
    }
    cluster_sync_all();
    constexpr int OPB = kGQ * HD / kCL;                        // outputs merged per block
    for (int i = threadIdx.x; i < OPB; i += kThreads) {
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

// ---- F16 caches: the same decomposition with the contractions on tensor cores ----------------
//
// S^T = K Q^T and O^T += V^T P^T as mma.sync m16n8k16 (f16 inputs, f32 accumulators), the 16 rows
// of an A fragment being 16 cells (scores) or 16 output dimensions (values) and the 8 columns of
// a B fragment the query heads (4 of the group, 4 zero columns). Q and P enter as two f16 terms
// (hi + lo of the float32), so every product is float32-accurate to about 2^-22, as in the
// prefill kernel. A block of MW warps walks its slice in passes of 16 MW cells; warp w takes cells
// 16w .. 16w+15 of every pass and keeps its own online-softmax state; the warps' states merge in
// shared memory, then across the cluster.
//
// Each pass is a chain of dependent steps per warp (MMAs, shuffles of the softmax, the P^T
// exchange); at 8192 cells over 16-block clusters the kernel is latency-bound (9% issue-active,
// DRAM at 16% of peak, stalls spread over fixed-latency waits, L1/shared loads and barriers). The
// K Q^T chain runs in four independent accumulators. Blocks stay at 4 warps (MW) and two stages:
// 8-warp blocks and four stages measured slower at that length (a block above ~113 KB of shared
// memory takes an SM alone and leaves no room for the next GEMV's blocks that start early under
// programmatic dependent launch), three stages within 1%.
constexpr int kMC = 16;                  // cells per warp and pass (one m16 fragment)

// KT = int8_t: a Q8_0 cache. Its int8 rows and fp16 scales are staged as they are, the rows
// expanded to exact f16 values in a shared tile per pass, and the block scales enter outside the
// MMAs: a score sums each 32-dimension block's fragment times the cell's K scale; the P^T fragment
// is multiplied by the cells' V scales for each 32-dimension output block.
//
// NS stages: NS - 1 passes are in flight while one is computed (two are used).
template <int HD, typename KT, int NS, int MW>
struct MmaDecSmem {
    static constexpr int CH = kMC * MW;                  // cells per pass
    static constexpr bool Q8 = sizeof(KT) == 1;
    static constexpr int NB = HD / 32;
    static constexpr int RS = HD + 8;                     // halves per padded f16 row
    static constexpr int RB = HD * (int)sizeof(KT);       // bytes of a cached row
    static constexpr int RSS = Q8 ? RB + 16 : RS * 2;     // bytes per staged row
    static constexpr size_t rows = 2 * (size_t)CH * RSS;
    static constexpr size_t stage = rows + 3 * CH * 4 + (Q8 ? 2 * (size_t)CH * NB * 2 : 0);
    static_assert(stage % 16 == 0, "stages stay 16-byte aligned");
    static constexpr size_t tile = Q8 ? 2 * (size_t)CH * RS * 2 : 0;   // expanded K and V
    // the warp states and the block partial reuse the stages once the passes are done
    static constexpr size_t states = (size_t)MW * kGQ * (HD + 2) * 4 + (size_t)kGQ * (HD + 2) * 4;
    static_assert(states <= 2 * stage, "states fit in the stage area");
    static constexpr size_t bytes = NS * stage + tile + (size_t)kGQ * HD * 4 /* q */ +
                                    (size_t)MW * kMC * 8 * 4 /* P^T per warp */ + 16;
};

// two int8 (low bytes of v, selected by sel) -> an exact half2: the biased byte as the low
// mantissa bits of 1024, minus 1024 + 128
__device__ __forceinline__ uint32_t q8x2_to_h2(uint32_t biased, uint32_t sel) {
    const uint32_t h = __byte_perm(biased, 0x64646464u, sel);
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2half2(__ushort_as_half(0x6480u)));
    return *reinterpret_cast<const uint32_t*>(&v);
}

// CL blocks per cluster: 16 for a few tokens; fewer (down to 1, no peers) when many tokens already
// fill the GPU, so each block walks a longer slice and pays the fixed costs less often.
// NCL clusters per (token, KV head): with 2 (long lists) the list is cut into 2 CL slices and
// twice as many blocks stream it (two per SM); each cluster merges its slices through
// distributed shared memory as before, then block r of the one cluster and block r of the other
// meet through global partial rows: each writes its (max, sum, outputs) and takes a ticket, and
// the second to arrive combines both and stores the output (no block waits for another).
template <int HD, typename KT, int CL, int NS, int MW, int NCL>
__global__ void __launch_bounds__(MW * 32)
attn_decode_mma_kernel(AttnArgs a, float scale_log2) {
    using SM = MmaDecSmem<HD, KT, NS, MW>;
    constexpr int CH = SM::CH, MT = MW * 32;
    constexpr bool Q8 = SM::Q8;
    constexpr int RS = SM::RS, RB = SM::RB, RSS = SM::RSS, VPR = RB / 16, NK = HD / 16, NB = SM::NB;
    extern __shared__ __align__(16) uint8_t sm[];
    struct St { uint8_t* kraw; uint8_t* vraw; int* ccell; int* cvis; int* cfresh; __half* ksc; __half* vsc; };
    auto stage_of = [&](int s) {
        uint8_t* b = sm + (size_t)s * SM::stage;
        St S;
        S.kraw = b;
        S.vraw = b + CH * RSS;
        S.ccell = reinterpret_cast<int*>(b + SM::rows);
        S.cvis = S.ccell + CH;
        S.cfresh = S.cvis + CH;
        S.ksc = reinterpret_cast<__half*>(S.cfresh + CH);
        S.vsc = S.ksc + CH * NB;
        return S;
    };
    __half* tk = reinterpret_cast<__half*>(sm + NS * SM::stage);      // Q8_0: expanded K tile
    __half* tv = tk + CH * RS;                                         //        and V tile
    float* qs = reinterpret_cast<float*>(sm + NS * SM::stage + SM::tile);  // [kGQ][HD]
    float* pT = qs + kGQ * HD;                                          // [warp][16 cells][8]
    float* ws = reinterpret_cast<float*>(sm);                           // after the passes: [warp][kGQ][HD + 2]
    float* pst = ws + MW * kGQ * (HD + 2);                             // block partial (peers read it)

    const uint32_t rank = cluster_rank();
    const int kvh = blockIdx.y, tile = blockIdx.z;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    if (tile >= a.hdr[1]) return;                               // whole cluster (same tile)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, cq = lane & 3;                     // fragment row group, column pair
    const int4 td0 = a.tile_desc[2 * tile];
    const int4 td1 = a.tile_desc[2 * tile + 1];
    const int base = td1.y, len = td1.z;
    const int t = a.perm[td0.y];
    const int tpos = a.tok_pos[t];
    const int clq = NCL > 1 ? (int)(blockIdx.x / CL) : 0;        // which of the NCL clusters
    const int chunk = (len + CL * NCL - 1) / (CL * NCL);
    const int c0 = min(len, (clq * CL + (int)rank) * chunk), c1 = min(len, c0 + chunk);
    const int npass = c1 > c0 ? (c1 - c0 + CH - 1) / CH : 1;
    const uint8_t* K = static_cast<const uint8_t*>(a.kc) + (int64_t)kvh * a.n_ctx * RB;
    const uint8_t* V = static_cast<const uint8_t*>(a.vc) + (int64_t)kvh * a.n_ctx * RB;
    const __half* KS = q8_scales(a.kc, a, kvh);
    const __half* VS = q8_scales(a.vc, a, kvh);

    // list entries of a pass, loaded one pass before its stage is set up
    int pf_cell = -1, pf_pos = 0;
    auto fetch = [&](int i) {
        if (threadIdx.x < CH) {
            const int ci = c0 + i * CH + threadIdx.x;
            pf_cell = -1;
            pf_pos = 0;
            if (ci < c1) {
                pf_cell = a.list_cells[base + ci];
                pf_pos = a.list_pos[base + ci];
            }
        }
    };
    auto setup = [&](const St& S) {
        if (threadIdx.x < CH) {
            int cell = -1, vis = 0, fresh = 0;
            if (pf_cell >= 0 && pf_cell < a.n_ctx) {
                cell = pf_cell;
                vis = pf_pos <= tpos;
                for (int j = 0; j < a.n_tok; ++j) fresh |= a.slot[j] == cell;
            }
            S.ccell[threadIdx.x] = cell;
            S.cvis[threadIdx.x] = vis && cell >= 0;
            S.cfresh[threadIdx.x] = fresh;
        }
    };
    // the stage's rows (and Q8_0 scales) as one cp.async group; before the wait on the previous
    // kernel the rows of this step's cells are left out (loaded after it). Q8_0: hidden cells get
    // zero scales (their int8 rows stay stale but finite).
    auto issue = [&](const St& S, bool pre_wait) {
        if constexpr (Q8) {
            const int c = threadIdx.x % CH;
            const bool isv = threadIdx.x >= CH;                 // MT == 2 CH
            __half* dst = (isv ? S.vsc : S.ksc) + c * NB;
            if (!S.cvis[c]) {
#pragma unroll
                for (int b = 0; b < NB; ++b) dst[b] = __ushort_as_half(0);
            } else if (!(pre_wait && S.cfresh[c])) {
                const __half* src = (isv ? VS : KS) + (int64_t)S.ccell[c] * NB;
                if constexpr (NB >= 2) {
                    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(sm32(dst)), "l"(src),
                                 "n"(NB * 2) : "memory");
                } else {
                    dst[0] = __ushort_as_half(__ldcg(reinterpret_cast<const unsigned short*>(src)));
                }
            }
        }
        for (int v = threadIdx.x; v < CH * VPR; v += MT) {
            const int c = v / VPR, j = v % VPR;
            if (!S.cvis[c]) {
                // the MMA multiplies every row of the tile: a hidden cell's V row must be finite
                if constexpr (!Q8) *reinterpret_cast<uint4*>(S.vraw + c * RSS + j * 16) = make_uint4(0u, 0u, 0u, 0u);
                continue;
            }
            if (pre_wait && S.cfresh[c]) continue;
            const size_t src = (size_t)S.ccell[c] * RB + j * 16;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm32(S.kraw + c * RSS + j * 16)), "l"(K + src) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm32(S.vraw + c * RSS + j * 16)), "l"(V + src) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    {
        const St S0 = stage_of(0);
        fetch(0);
        setup(S0);
        __syncthreads();
        issue(S0, true);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int i = threadIdx.x; i < kGQ * HD; i += MT)
            qs[i] = a.q[(int64_t)t * a.ldq + (kvh * kGQ + i / HD) * HD + i % HD] * scale_log2;
        if (npass > 1) fetch(1);
        for (int v = threadIdx.x; v < CH * VPR; v += MT) {
            const int c = v / VPR, j = v % VPR;
            if (!S0.cvis[c] || !S0.cfresh[c]) continue;
            const size_t src = (size_t)S0.ccell[c] * RB + j * 16;
            *reinterpret_cast<uint4*>(S0.kraw + c * RSS + j * 16) = __ldcg(reinterpret_cast<const uint4*>(K + src));
            *reinterpret_cast<uint4*>(S0.vraw + c * RSS + j * 16) = __ldcg(reinterpret_cast<const uint4*>(V + src));
        }
        if constexpr (Q8) {
            if (threadIdx.x < CH && S0.cvis[threadIdx.x] && S0.cfresh[threadIdx.x]) {
                const int cell = S0.ccell[threadIdx.x];
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    S0.ksc[threadIdx.x * NB + b] = __float2half_rn(ld_scale(KS + (int64_t)cell * NB + b));
                    S0.vsc[threadIdx.x * NB + b] = __float2half_rn(ld_scale(VS + (int64_t)cell * NB + b));
                }
            }
        }
    }
    // passes 1 .. NS - 2 (empty groups past the last pass): NS - 1 groups committed
    for (int j = 1; j < NS - 1; ++j) {
        if (j < npass) {
            const St N = stage_of(j);
            setup(N);
            if (j + 1 < npass) fetch(j + 1);
            __syncthreads();
            issue(N, false);
        } else {
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
    }
    __syncthreads();                                            // qs
    // B fragments of Q^T (column n = query head g, rows = dims): two f16 terms per k-step
    uint32_t qh[NK][2], ql[NK][2];
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
        const float* qr = qs + (g < kGQ ? g : 0) * HD + kk * 16 + 2 * cq;
        const float z = g < kGQ ? 1.f : 0.f;
        split_h2(z * qr[0], z * qr[1], qh[kk][0], ql[kk][0]);
        split_h2(z * qr[8], z * qr[9], qh[kk][1], ql[kk][1]);
    }

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[NK][4];
#pragma unroll
    for (int nt = 0; nt < NK; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
    float* pw = pT + warp * kMC * 8;
    const int cw = warp * kMC;                                  // this warp's cells in a pass
    for (int i = 0; i < npass; ++i) {
        const St S = stage_of(i % NS);
        const int nx = i + NS - 1;                              // the pass issued now
        if (nx < npass) {
            const St N = stage_of(nx % NS);
            setup(N);
            if (nx + 1 < npass) fetch(nx + 1);
            __syncthreads();
            issue(N, false);
        } else {
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        asm volatile("cp.async.wait_group %0;" ::"n"(NS - 1) : "memory");   // pass i has landed
        __syncthreads();
        const __half* kb;
        const __half* vb;
        if constexpr (Q8) {
            // this warp's 16 int8 rows -> exact f16 rows of the tiles (only this warp's MMAs read
            // them, and its previous pass's MMAs are done)
            for (int idx = lane; idx < kMC * (HD / 4); idx += 32) {
                const int cc = cw + idx / (HD / 4), w4 = idx % (HD / 4);
                const uint32_t kq = *reinterpret_cast<const uint32_t*>(S.kraw + cc * RSS + w4 * 4) ^ 0x80808080u;
                const uint32_t vq = *reinterpret_cast<const uint32_t*>(S.vraw + cc * RSS + w4 * 4) ^ 0x80808080u;
                *reinterpret_cast<uint2*>(tk + cc * RS + w4 * 4) = make_uint2(q8x2_to_h2(kq, 0x7170u), q8x2_to_h2(kq, 0x7372u));
                *reinterpret_cast<uint2*>(tv + cc * RS + w4 * 4) = make_uint2(q8x2_to_h2(vq, 0x7170u), q8x2_to_h2(vq, 0x7372u));
            }
            __syncwarp();
            kb = tk;
            vb = tv;
        } else {
            kb = reinterpret_cast<const __half*>(S.kraw);
            vb = reinterpret_cast<const __half*>(S.vraw);
        }

        // S^T [16 cells][8 heads] = K Q^T (Q8_0: per 32-dimension block, times the cells' K scales)
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int mi = lane >> 3, r = lane & 7;
            const __half* kr = kb + (cw + r + (mi & 1) * 8) * RS + (mi >> 1) * 8;
            if constexpr (Q8) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    float sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 2 * b; kk < 2 * b + 2; ++kk) {
                        uint32_t af[4];
                        ldsm_x4(sm32(kr + kk * 16), af[0], af[1], af[2], af[3]);
                        mma16816(sb, af, qh[kk][0], qh[kk][1]);
                        mma16816(sb, af, ql[kk][0], ql[kk][1]);
                    }
                    const float d0 = __half2float(S.ksc[(cw + g) * NB + b]);
                    const float d1 = __half2float(S.ksc[(cw + g + 8) * NB + b]);
                    s[0] = fmaf(d0, sb[0], s[0]); s[1] = fmaf(d0, sb[1], s[1]);
                    s[2] = fmaf(d1, sb[2], s[2]); s[3] = fmaf(d1, sb[3], s[3]);
                }
            } else {
                float acc[4][4] = {};
#pragma unroll
                for (int kk = 0; kk < NK; ++kk) {
                    uint32_t af[4];
                    ldsm_x4(sm32(kr + kk * 16), af[0], af[1], af[2], af[3]);
                    mma16816(acc[kk & 1], af, qh[kk][0], qh[kk][1]);
                    mma16816(acc[2 + (kk & 1)], af, ql[kk][0], ql[kk][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) s[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
            }
        }
        // this thread: cells cw+g (s[0], s[1]) and cw+g+8 (s[2], s[3]), heads 2cq and 2cq+1
        const bool live = cq < kGQ / 2;
        const bool v0 = live && S.cvis[cw + g], v1 = live && S.cvis[cw + g + 8];
        float sv[4] = {v0 ? s[0] : -INFINITY, v0 ? s[1] : -INFINITY, v1 ? s[2] : -INFINITY, v1 ? s[3] : -INFINITY};
        float p[4], corr[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(sv[j], sv[j + 2]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[j], mx);
            corr[j] = m_new == -INFINITY ? 1.f : exp2f(m[j] - m_new);
            p[j] = sv[j] == -INFINITY ? 0.f : exp2f(sv[j] - m_new);
            p[j + 2] = sv[j + 2] == -INFINITY ? 0.f : exp2f(sv[j + 2] - m_new);
            float ps = p[j] + p[j + 2];
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l[j] = l[j] * corr[j] + ps;
            m[j] = m_new;
        }
#pragma unroll
        for (int nt = 0; nt < NK; ++nt) {
            o[nt][0] *= corr[0]; o[nt][1] *= corr[1];
            o[nt][2] *= corr[0]; o[nt][3] *= corr[1];
        }
        // P^T [16 cells][8 heads] through shared memory into B fragments (head g, 4 cells)
        pw[g * 8 + 2 * cq] = p[0];
        pw[g * 8 + 2 * cq + 1] = p[1];
        pw[(g + 8) * 8 + 2 * cq] = p[2];
        pw[(g + 8) * 8 + 2 * cq + 1] = p[3];
        __syncwarp();
        const float pq[4] = {pw[(2 * cq) * 8 + g], pw[(2 * cq + 1) * 8 + g], pw[(2 * cq + 8) * 8 + g],
                             pw[(2 * cq + 9) * 8 + g]};
        // O^T [16 dims][8 heads] += V^T P^T per 16-dimension tile (Q8_0: P^T times the cells' V
        // scales of each 32-dimension block)
        {
            const int mi = lane >> 3, r = lane & 7;
            const __half* vr = vb + (cw + r + (mi >> 1) * 8) * RS + (mi & 1) * 8;
            uint32_t bh0, bl0, bh1, bl1;
            if constexpr (!Q8) {
                split_h2(pq[0], pq[1], bh0, bl0);
                split_h2(pq[2], pq[3], bh1, bl1);
            }
#pragma unroll
            for (int nt = 0; nt < NK; ++nt) {
                if constexpr (Q8) {
                    if ((nt & 1) == 0) {
                        const int b = nt / 2;
                        const __half* vs = S.vsc + (cw + 2 * cq) * NB + b;
                        split_h2(pq[0] * __half2float(vs[0]), pq[1] * __half2float(vs[NB]), bh0, bl0);
                        split_h2(pq[2] * __half2float(vs[8 * NB]), pq[3] * __half2float(vs[9 * NB]), bh1, bl1);
                    }
                }
                uint32_t af[4];
                ldsm_x4_t(sm32(vr + nt * 16), af[0], af[1], af[2], af[3]);
                mma16816(o[nt], af, bh0, bh1);
                mma16816(o[nt], af, bl0, bl1);
            }
        }
        __syncwarp();                                           // pw is rewritten next pass
        __syncthreads();                                        // stage S free for pass i + NS
    }

    // the warps' states -> this block's partial -> the cluster-wide merge
    float* my = ws + warp * kGQ * (HD + 2);
    if (cq < kGQ / 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float* hs = my + (2 * cq + j) * (HD + 2);
            if (g == 0) { hs[0] = m[j]; hs[1] = l[j]; }
#pragma unroll
            for (int nt = 0; nt < NK; ++nt) {
                hs[2 + nt * 16 + g] = o[nt][j];
                hs[2 + nt * 16 + g + 8] = o[nt][j + 2];
            }
        }
    }
    __syncthreads();
    float* pm = pst;
    float* pl = pst + kGQ;
    float* po = pst + 2 * kGQ;
    for (int idx = threadIdx.x; idx < kGQ * HD; idx += MT) {
        const int h = idx / HD, dd = idx % HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < MW; ++w) M = fmaxf(M, ws[(w * kGQ + h) * (HD + 2)]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < MW; ++w) {
            const float* hs = ws + (w * kGQ + h) * (HD + 2);
            const float f = (M == -INFINITY || hs[0] == -INFINITY) ? 0.f : exp2f(hs[0] - M);
            L = fmaf(f, hs[1], L);
            O = fmaf(f, hs[2 + dd], O);
        }
        if (dd == 0) { pm[h] = M; pl[h] = L; }
        po[h * HD + dd] = O;
    }
    cluster_sync_all();
    constexpr int OPB = kGQ * HD / CL;
    // the cluster's (max, sum, unnormalised output) of output oi = rank * OPB + idx
    auto merge = [&](int idx, float& M, float& L, float& O) {
        const int oi = (int)rank * OPB + idx;
        const int h = oi / HD, dd = oi % HD;
        M = -INFINITY;
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) M = fmaxf(M, ld_peer(pm + h, r));
        L = 0.f;
        O = 0.f;
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) {
            const float mr = ld_peer(pm + h, r);
            const float f = (M == -INFINITY || mr == -INFINITY) ? 0.f : exp2f(mr - M);
            L = fmaf(f, ld_peer(pl + h, r), L);
            O = fmaf(f, ld_peer(po + h * HD + dd, r), O);
        }
    };
    if constexpr (NCL == 1) {
        for (int idx = threadIdx.x; idx < OPB; idx += MT) {
            float M, L, O;
            merge(idx, M, L, O);
            const int oi = (int)rank * OPB + idx;
            store_out(a, (int64_t)t * a.ldo + (kvh * kGQ + oi / HD) * HD + oi % HD, L > 0.f ? O / L : 0.f);
        }
    } else {
        // this cluster's share of block `rank`'s outputs (all of one head) goes to global partial
        // rows [tile][cluster][head][KV head]; the ticket [tile][KV head][rank] counts the blocks
        // with this rank that are done, and the last of the NCL combines the shares and stores
        static_assert(OPB <= MT && HD % OPB == 0, "one output per thread, one head per block");
        __shared__ int last_s;
        const int h = (int)rank * OPB / HD, dd = (int)rank * OPB % HD + (int)threadIdx.x;
        float M = -INFINITY, L = 0.f, O = 0.f;
        if (threadIdx.x < OPB) {
            merge(threadIdx.x, M, L, O);
            const int64_t row = ((int64_t)(tile * NCL + clq) * kGQ + h) * a.Hkv + kvh;
            if (threadIdx.x == 0) { a.part_m[row] = M; a.part_l[row] = L; }
            a.part_o[row * HD + dd] = O;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            int* tkt = a.tickets + ((int64_t)tile * a.Hkv + kvh) * CL + rank;
            const int done = atomicAdd(tkt, 1) + 1;
            last_s = done == NCL;
            if (done == NCL) *tkt = 0;                 // zero again for the next launch
        }
        __syncthreads();
        if (last_s && threadIdx.x < OPB) {
            __threadfence();
            float Mx = M;
            for (int q = 0; q < NCL; ++q) {
                if (q == clq) continue;
                Mx = fmaxf(Mx, __ldcg(a.part_m + ((int64_t)(tile * NCL + q) * kGQ + h) * a.Hkv + kvh));
            }
            float Lt = 0.f, Ot = 0.f;
            for (int q = 0; q < NCL; ++q) {
                const int64_t row = ((int64_t)(tile * NCL + q) * kGQ + h) * a.Hkv + kvh;
                const float mq = q == clq ? M : __ldcg(a.part_m + row);
                const float lq = q == clq ? L : __ldcg(a.part_l + row);
                const float oq = q == clq ? O : __ldcg(a.part_o + row * HD + dd);
                const float f = (Mx == -INFINITY || mq == -INFINITY) ? 0.f : exp2f(mq - Mx);
                Lt = fmaf(f, lq, Lt);
                Ot = fmaf(f, oq, Ot);
            }
            store_out(a, (int64_t)t * a.ldo + (kvh * kGQ + h) * HD + dd, Lt > 0.f ? Ot / Lt : 0.f);
        }
    }
    cluster_sync_all();
}

template <int HD, typename KT, int CL, int NS, int MW, int NCL = 1>
bool launch_dec_mma_cl(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    constexpr size_t smem = MmaDecSmem<HD, KT, NS, MW>::bytes;
    auto k = attn_decode_mma_kernel<HD, KT, CL, NS, MW, NCL>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return false;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * NCL, a.Hkv, a.n_tok);
    cfg.blockDim = dim3(MW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr_l[2];
    attr_l[0].id = cudaLaunchAttributeClusterDimension;
    attr_l[0].val.clusterDim.x = CL;
    attr_l[0].val.clusterDim.y = 1;
    attr_l[0].val.clusterDim.z = 1;
    attr_l[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr_l[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr_l;
    cfg.numAttrs = a.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
}

int sm_count() {
    static int n_sm = 0;
    if (n_sm == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (n_sm <= 0) n_sm = 148;
    }
    return n_sm;
}

// The cluster size: 16 unless 16 blocks per (token, KV head) would exceed two blocks per SM.
int dec_cluster(int n_tok, int Hkv) {
    const int64_t units = (int64_t)Hkv * n_tok, n_sm = sm_count();
    return 16 * units <= 2 * n_sm ? 16 : 4 * units <= 2 * n_sm ? 4 : 1;
}

// Two clusters per (token, KV head) when the lists are long (the caller's plan decides; its
// choice is part of a captured step's key) and 2 x 16 blocks per unit still fit two per SM.
bool dec_two_clusters(const AttnArgs& a) {
    const int64_t units = (int64_t)a.Hkv * a.n_tok;
    return a.long_lists && 2 * 16 * units <= 2 * (int64_t)sm_count();
}

template <int HD, typename KT>
bool launch_dec_mma(const AttnArgs& a, cudaStream_t st) {
    switch (dec_cluster(a.n_tok, a.Hkv)) {
        case 16:
            if (dec_two_clusters(a)) return launch_dec_mma_cl<HD, KT, 16, 2, 4, 2>(a, st);
            return launch_dec_mma_cl<HD, KT, 16, 2, 4>(a, st);
        case 4: return launch_dec_mma_cl<HD, KT, 4, 2, 4>(a, st);
    }
    return launch_dec_mma_cl<HD, KT, 1, 2, 4>(a, st);
}

template <int HD>
bool launch_dec(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    constexpr size_t smem = DecSmem<HD>::bytes;
    auto k = attn_decode_kernel<HD>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return false;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCL, a.Hkv, a.n_tok);
    cfg.blockDim = dim3(kThreads);
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
    if (a.kv_type == W_Q8_0) {                                 // tensor cores
        switch (a.hd) {
            case 32: return launch_dec_mma<32, int8_t>(a, st);
            case 64: return launch_dec_mma<64, int8_t>(a, st);
            case 128: return launch_dec_mma<128, int8_t>(a, st);
        }
        return false;
    }
    if (a.kv_type == W_F16) {                                  // tensor cores
        switch (a.hd) {
            case 32: return launch_dec_mma<32, __half>(a, st);
            case 64: return launch_dec_mma<64, __half>(a, st);
            case 128: return launch_dec_mma<128, __half>(a, st);
        }
        return false;
    }
    switch (a.hd) {                                            // F32: CUDA cores
        case 32: return launch_dec<32>(a, st);
        case 64: return launch_dec<64>(a, st);
        case 128: return launch_dec<128>(a, st);
    }
    return false;
}

}  // namespace llm
