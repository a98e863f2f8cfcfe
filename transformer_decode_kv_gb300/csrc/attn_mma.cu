// Prefill attention on tensor cores ([P2] "llama.cpp Architecture", Example 4 FLASH_ATTN_EXT;
// Example 11 for the unfused meaning: scores Q K^T with the KQ mask, softmax, times V).
//
// The same work decomposition as the CUDA-core kernel (kernels_attention.cu): a block takes one
// work item (a query tile of up to 16 tokens of one cell list, and a slice of that list) for one
// KV head. The tile's 16 tokens x 4 query heads of the group are 64 rows; warp w owns rows
// 16w .. 16w+15 (row r: token r / 4, head r % 4). Per 64-cell tile of the slice the block gathers
// the cells' K and V rows (F16, cp.async through L2, double-buffered) and each warp runs
//   S = Q K^T       mma.m16n8k16 f16 x f16 -> f32 (Q as two f16 terms: hi + lo of the float32)
//   mask, online softmax in base 2 (log2 e / sqrt(hd) folded into Q)
//   O += P V        P as two f16 terms, V f16
// so every product is float32-accurate to about 2^-22 and accumulates in float32. A cell is
// visible to a row iff cell.pos <= token.pos (the list already holds only the sequence's cells).
// ONE: Q and P as one f16 term each (half the MMAs), for a forward pass whose matrix products
// already take f16 activations (the attention output is rounded to f16 for them anyway).
// Partial states (o, m, l) and the ticket merge are shared with the CUDA-core kernel.
//
// A Q8_0 cache ([P2] Example 2 blocks: value d * q per 32 values) comes as f16 copies of its
// int8 quants (exact) plus the cache's fp16 scales, gathered with the rows. K: each 32-dim block's
// Q . q products accumulate apart and join S times that block's d of the cell. V: the scale
// varies along the contracted cells, so each 32-dim block of the output takes P times the cells'
// d of that block, split into two f16 terms as P is. The values d * q are never rounded.
//
// mma.sync is enough here: a 512-token ubatch of the 8B shape has 2.1 GFLOP of attention per
// layer, 1% of its matrix work, and this kernel moves it off the CUDA cores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "attn_common.cuh"
#include "kernels.h"

namespace llm {

namespace {

using namespace attn;

constexpr int kWarps = 4;
constexpr int kTC = 64;                    // cells per tile
constexpr int kG = 4;                      // query heads per KV head
constexpr int kTQ = 16;                    // tokens per query tile
constexpr int kRows = kTQ * kG;            // 64 rows: one m16 fragment row block per warp


template <int HD, bool Q8>
struct MmaSmem {
    static constexpr int RS = HD + 8;                       // padded row (halves): no bank conflicts
    static constexpr int NB = HD / 32;                      // Q8_0 blocks per row
    static constexpr size_t tile_bytes = (size_t)kTC * RS * 2;
    static constexpr size_t q_bytes = (size_t)kRows * RS * 2;      // one f16 term of the Q tile
    static constexpr size_t base_bytes = 4 * tile_bytes + 2 * q_bytes + 4 * kTC * 4 + 8 * 4 + 2 * kRows * 4 + 16;
    static constexpr size_t sc_off = (base_bytes + 15) / 16 * 16;
    static constexpr size_t sc_tile = (size_t)kTC * NB;    // halves: one tile's K (or V) scales
    static constexpr size_t bytes = Q8 ? sc_off + 4 * sc_tile * 2 : base_bytes;
};

// Issue the gathers of one tile into buffer (ks, vs): cell indices from shared memory (ccell,
// -1 = none), zeros for missing cells. Q8: also the cells' scales (KS, VS) into (kd, vd).
template <int HD, bool Q8>
__device__ __forceinline__ void gather_tile(const __half* K, const __half* V, const int* ccell,
                                            __half* ks, __half* vs, const __half* KS = nullptr,
                                            const __half* VS = nullptr, __half* kd = nullptr,
                                            __half* vd = nullptr) {
    constexpr int RS = MmaSmem<HD, Q8>::RS, VPR = HD / 8, NB = HD / 32;
    if constexpr (Q8) {
        if (threadIdx.x < 2 * kTC) {
            const int c = threadIdx.x % kTC;
            const bool isv = threadIdx.x >= kTC;
            const int cell = ccell[c];
            __half* dst = (isv ? vd : kd) + c * NB;
            if (cell >= 0) {
                const __half* src = (isv ? VS : KS) + (int64_t)cell * NB;
                if constexpr (NB >= 2) {
                    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_addr(dst)), "l"(src),
                                 "n"(NB * 2) : "memory");
                } else {
                    *dst = *src;
                }
            } else {
#pragma unroll
                for (int b = 0; b < NB; ++b) dst[b] = __float2half(0.f);
            }
        }
    }
    for (int v = threadIdx.x; v < kTC * VPR; v += kWarps * 32) {
        const int c = v / VPR, j = v % VPR;
        const int cell = ccell[c];
        __half* dk = ks + c * RS + j * 8;
        __half* dv = vs + c * RS + j * 8;
        if (cell >= 0) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dk)),
                         "l"(K + (int64_t)cell * HD + j * 8) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dv)),
                         "l"(V + (int64_t)cell * HD + j * 8) : "memory");
        } else {
            *reinterpret_cast<uint4*>(dk) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(dv) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Cell index and position of list entry cb + threadIdx.x (threads 0 .. kTC-1; -1 / INT_MAX past
// the slice's end).
__device__ __forceinline__ void load_index(const AttnArgs& a, int base, int cb, int c1, int& cell, int& pos) {
    cell = -1;
    pos = INT_MAX;
    const int ci = cb + (int)threadIdx.x;
    if (threadIdx.x < kTC && ci < c1) {
        const int cc = a.list_cells[base + ci];
        if (cc >= 0 && cc < a.n_ctx) { cell = cc; pos = a.list_pos[base + ci]; }
    }
}
// Store a tile's indices (threads 0 .. kTC-1) and each warp's minimum position.
__device__ __forceinline__ void store_index(int cell, int pos, int* ccell, int* cpos, int* cmin) {
    if (threadIdx.x < kTC) {
        ccell[threadIdx.x] = cell;
        cpos[threadIdx.x] = pos;
        int mn = pos;
        for (int off = 16; off > 0; off >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        if ((threadIdx.x & 31) == 0) cmin[threadIdx.x >> 5] = mn;
    }
}

}  // namespace

template <int HD, bool Q8, bool ONE>
__global__ void __launch_bounds__(kWarps * 32, 2) attn_mma_kernel(AttnArgs a, float scale_log2) {
    using SM = MmaSmem<HD, Q8>;
    constexpr int RS = SM::RS, KC = HD / 16, NC = HD / 8, NB = SM::NB;
    extern __shared__ __align__(16) uint8_t smem[];
    __half* kbuf[2] = {reinterpret_cast<__half*>(smem), reinterpret_cast<__half*>(smem + SM::tile_bytes)};
    __half* vbuf[2] = {reinterpret_cast<__half*>(smem + 2 * SM::tile_bytes),
                       reinterpret_cast<__half*>(smem + 3 * SM::tile_bytes)};
    __half* qhs = reinterpret_cast<__half*>(smem + 4 * SM::tile_bytes);  // Q tile, hi term
    __half* qls = reinterpret_cast<__half*>(smem + 4 * SM::tile_bytes + SM::q_bytes);   // lo term
    int* cposb = reinterpret_cast<int*>(smem + 4 * SM::tile_bytes + 2 * SM::q_bytes);   // [2][kTC]
    int* ccellb = cposb + 2 * kTC;                                        // [2][kTC]
    int* cminb = ccellb + 2 * kTC;                                        // [2][2] per warp
    int* rmax = cminb + 4;                                                // largest row position
    int* rpos = cminb + 8;                                                // [kRows]
    int* rtok = rpos + kRows;                                             // [kRows] token row of q
    int* flag = rtok + kRows;
    // Q8: [2 buffers][K, V][kTC][NB] scales
    __half* scb = reinterpret_cast<__half*>(smem + SM::sc_off);

    const int wi = blockIdx.x, kvh = blockIdx.y;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    const int n_work = a.hdr[0];
    const int4 wd = a.wi_desc[wi];
    if (wi >= n_work) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int4 td0 = a.tile_desc[2 * wd.x];
    const int4 td1 = a.tile_desc[2 * wd.x + 1];
    const int nq = td0.z, s0 = td0.y, c0 = wd.y, c1 = wd.z, base = td1.y;
    const __half* K = static_cast<const __half*>(a.kc) + (int64_t)kvh * a.n_ctx * HD;
    const __half* V = static_cast<const __half*>(a.vc) + (int64_t)kvh * a.n_ctx * HD;
    const __half* KS = Q8 ? static_cast<const __half*>(a.k_scale) + (int64_t)kvh * a.n_ctx * NB : nullptr;
    const __half* VS = Q8 ? static_cast<const __half*>(a.v_scale) + (int64_t)kvh * a.n_ctx * NB : nullptr;
    auto ksc = [&](int b) { return scb + (2 * b) * SM::sc_tile; };       // buffer b's K scales
    auto vsc = [&](int b) { return scb + (2 * b + 1) * SM::sc_tile; };
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // tile 0: indices, then its gathers; tile 1's indices are loaded while tile 0 is used
    int ncell, npos;
    load_index(a, base, c0, c1, ncell, npos);
    store_index(ncell, npos, ccellb, cposb, cminb);
    for (int r = threadIdx.x; r < kRows; r += kWarps * 32) {
        const int j = r / kG;
        const int t = j < nq ? a.perm[s0 + j] : -1;
        rtok[r] = t;
        rpos[r] = t >= 0 ? a.tok_pos[t] : -1;
    }
    __syncthreads();
    gather_tile<HD, Q8>(K, V, ccellb, kbuf[0], vbuf[0], KS, VS, ksc(0), vsc(0));
    load_index(a, base, c0 + kTC, c1, ncell, npos);
    if (threadIdx.x < 32) {
        int mx = -1;
        for (int r = threadIdx.x; r < kRows; r += 32) mx = max(mx, rpos[r]);
        for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (threadIdx.x == 0) *rmax = mx;
    }

    // the Q tile as two f16 terms (hi + lo of the float32, log2 e / sqrt(hd) folded in); the
    // loads of a batch are all issued before any is used
    constexpr int QV = kRows * HD / 2 / (kWarps * 32);      // float2 per thread
#pragma unroll
    for (int b = 0; b < QV; b += 8) {
        float2 x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int v = threadIdx.x + (b + i) * kWarps * 32;
            const int r = v / (HD / 2), col = (v % (HD / 2)) * 2;
            const int t = rtok[r];
            x[i] = t >= 0 ? *reinterpret_cast<const float2*>(a.q + (int64_t)t * a.ldq + (kvh * kG + r % kG) * HD + col)
                          : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int v = threadIdx.x + (b + i) * kWarps * 32;
            const int r = v / (HD / 2), col = (v % (HD / 2)) * 2;
            uint32_t hi, lo;
            split_h2(x[i].x * scale_log2, x[i].y * scale_log2, hi, lo);
            *reinterpret_cast<uint32_t*>(qhs + r * RS + col) = hi;
            if (!ONE) *reinterpret_cast<uint32_t*>(qls + r * RS + col) = lo;
        }
    }
    const int r0 = warp * 16 + g, r1 = r0 + 8;
    // A-fragment addresses of this warp's rows: (rows 0-7 | 8-15) x (k 0-7 | 8-15)
    const int qrow = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int qcol = (lane >> 4) << 3;

    float o[NC][4];
#pragma unroll
    for (int n = 0; n < NC; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    int buf = 0;
    for (int cb = c0; cb < c1; cb += kTC, buf ^= 1) {
        // the next tile's gathers go out before this tile is used (its indices were loaded during
        // the previous tile); the indices of the one after are loaded now
        const bool more = cb + kTC < c1;
        __syncthreads();           // the other buffer's last readers are done
        if (more) {
            store_index(ncell, npos, ccellb + (buf ^ 1) * kTC, cposb + (buf ^ 1) * kTC, cminb + (buf ^ 1) * 2);
            __syncthreads();
            gather_tile<HD, Q8>(K, V, ccellb + (buf ^ 1) * kTC, kbuf[buf ^ 1], vbuf[buf ^ 1], KS, VS,
                                ksc(buf ^ 1), vsc(buf ^ 1));
            load_index(a, base, cb + 2 * kTC, c1, ncell, npos);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const __half* ks = kbuf[buf];
        const __half* vs = vbuf[buf];
        const int* cpos = cposb + buf * kTC;
        // a tile no row of this block may see (causal prefill) is skipped
        if (min(cminb[buf * 2], cminb[buf * 2 + 1]) > *rmax) continue;

        // S = Q K^T over the tile's 64 cells: 8 fragments of 8 cells
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        auto qk = [&](float (&acc)[8][4], int kc) {
            uint32_t qh[4], ql[4];
            ldsm_x4(smem_addr(qhs + qrow * RS + kc * 16 + qcol), qh[0], qh[1], qh[2], qh[3]);
            if (!ONE) ldsm_x4(smem_addr(qls + qrow * RS + kc * 16 + qcol), ql[0], ql[1], ql[2], ql[3]);
            // K fragments of the 64 cells first, then the hi-term MMAs, then the lo-term ones,
            // so no two consecutive MMAs share an accumulator
            uint32_t kb[4][4];
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) {
                // matrices: (cells 16 n2 + 0..7, dims 16 kc + 0..7), (same cells, +8 dims),
                //           (cells 16 n2 + 8..15, dims 16 kc), (cells +8, dims +8)
                const int cell = 16 * n2 + (lane & 7) + ((lane >> 4) << 3);
                const int dim = 16 * kc + (((lane >> 3) & 1) << 3);
                ldsm_x4(smem_addr(ks + cell * RS + dim), kb[n2][0], kb[n2][1], kb[n2][2], kb[n2][3]);
            }
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) {
                mma16816(acc[2 * n2], qh, kb[n2][0], kb[n2][1]);
                mma16816(acc[2 * n2 + 1], qh, kb[n2][2], kb[n2][3]);
            }
            if (!ONE) {
#pragma unroll
                for (int n2 = 0; n2 < 4; ++n2) {
                    mma16816(acc[2 * n2], ql, kb[n2][0], kb[n2][1]);
                    mma16816(acc[2 * n2 + 1], ql, kb[n2][2], kb[n2][3]);
                }
            }
        };
        if constexpr (Q8) {
            // per 32-dim block: the quants' products, then times the block's d of each cell
            const __half* kd = ksc(buf);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float t[8][4];
#pragma unroll
                for (int n = 0; n < 8; ++n) t[n][0] = t[n][1] = t[n][2] = t[n][3] = 0.f;
                qk(t, 2 * b);
                qk(t, 2 * b + 1);
#pragma unroll
                for (int n = 0; n < 8; ++n) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float dk = __half2float(kd[(8 * n + 2 * t4 + e) * NB + b]);
                        s[n][e] = fmaf(t[n][e], dk, s[n][e]);
                        s[n][2 + e] = fmaf(t[n][2 + e], dk, s[n][2 + e]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int kc = 0; kc < KC; ++kc) qk(s, kc);
        }
        // mask and online softmax (rows r0, r1; this thread's columns 2 t4, 2 t4 + 1 of each
        // fragment; the row's other columns live in the same quad)
        const int p0 = rpos[r0], p1 = rpos[r1];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int cp = cpos[8 * n + 2 * t4 + e];
                if (cp > p0) s[n][e] = -INFINITY;
                if (cp > p1) s[n][2 + e] = -INFINITY;
                mx0 = fmaxf(mx0, s[n][e]);
                mx1 = fmaxf(mx1, s[n][2 + e]);
            }
        }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float cr0 = mn0 == -INFINITY ? 1.f : exp2f(m[0] - mn0);
        const float cr1 = mn1 == -INFINITY ? 1.f : exp2f(m[1] - mn1);
        m[0] = mn0;
        m[1] = mn1;
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                s[n][e] = mn0 == -INFINITY ? 0.f : exp2f(s[n][e] - mn0);
                s[n][2 + e] = mn1 == -INFINITY ? 0.f : exp2f(s[n][2 + e] - mn1);
                ls0 += s[n][e];
                ls1 += s[n][2 + e];
            }
        }
        l[0] = l[0] * cr0 + ls0;
        l[1] = l[1] * cr1 + ls1;
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            o[n][0] *= cr0; o[n][1] *= cr0;
            o[n][2] *= cr1; o[n][3] *= cr1;
        }
        // O += P V: P's accumulator layout is the A layout of the next MMA (16 cells per step)
        if constexpr (Q8) {
            // this thread's cells of step kk: 16 kk + 2 t4 + {0, 1} (A registers 0, 1) and
            // 16 kk + 8 + 2 t4 + {0, 1} (registers 2, 3)
            const __half* vd = vsc(buf);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int ca = 16 * kk + 2 * t4;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float d0 = __half2float(vd[ca * NB + b]), d1 = __half2float(vd[(ca + 1) * NB + b]);
                    const float d2 = __half2float(vd[(ca + 8) * NB + b]), d3 = __half2float(vd[(ca + 9) * NB + b]);
                    uint32_t ph[4], pl[4];
                    split_h2(s[2 * kk][0] * d0, s[2 * kk][1] * d1, ph[0], pl[0]);
                    split_h2(s[2 * kk][2] * d0, s[2 * kk][3] * d1, ph[1], pl[1]);
                    split_h2(s[2 * kk + 1][0] * d2, s[2 * kk + 1][1] * d3, ph[2], pl[2]);
                    split_h2(s[2 * kk + 1][2] * d2, s[2 * kk + 1][3] * d3, ph[3], pl[3]);
                    uint32_t vb[2][4];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int n2 = 2 * b + i;                 // 16-dim groups of block b
                        const int cell = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
                        const int dim = 16 * n2 + ((lane >> 4) << 3);
                        ldsm_x4_t(smem_addr(vs + cell * RS + dim), vb[i][0], vb[i][1], vb[i][2], vb[i][3]);
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        mma16816(o[2 * (2 * b + i)], ph, vb[i][0], vb[i][1]);
                        mma16816(o[2 * (2 * b + i) + 1], ph, vb[i][2], vb[i][3]);
                    }
                    if (!ONE) {
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            mma16816(o[2 * (2 * b + i)], pl, vb[i][0], vb[i][1]);
                            mma16816(o[2 * (2 * b + i) + 1], pl, vb[i][2], vb[i][3]);
                        }
                    }
                }
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t ph[4], pl[4];
                split_h2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
                split_h2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
                split_h2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
                split_h2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
                constexpr int GS = NC / 2 < 4 ? NC / 2 : 4;          // dimension blocks per group
#pragma unroll
                for (int h4 = 0; h4 < NC / 2; h4 += GS) {
                    uint32_t vb[GS][4];
#pragma unroll
                    for (int i = 0; i < GS; ++i) {
                        // matrices (transposed): (cells 16 kk + 0..7, dims 16 n2 + 0..7), (cells +8,
                        // same dims), (cells 16 kk, dims +8), (cells +8, dims +8)
                        const int n2 = h4 + i;
                        const int cell = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
                        const int dim = 16 * n2 + ((lane >> 4) << 3);
                        ldsm_x4_t(smem_addr(vs + cell * RS + dim), vb[i][0], vb[i][1], vb[i][2], vb[i][3]);
                    }
#pragma unroll
                    for (int i = 0; i < GS; ++i) {
                        mma16816(o[2 * (h4 + i)], ph, vb[i][0], vb[i][1]);
                        mma16816(o[2 * (h4 + i) + 1], ph, vb[i][2], vb[i][3]);
                    }
                    if (!ONE) {
#pragma unroll
                        for (int i = 0; i < GS; ++i) {
                            mma16816(o[2 * (h4 + i)], pl, vb[i][0], vb[i][1]);
                            mma16816(o[2 * (h4 + i) + 1], pl, vb[i][2], vb[i][3]);
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
    }

    const int w0 = td0.w, w1 = td1.x;
    const int rows[2] = {r0, r1};
    if (w1 - w0 == 1) {                            // a single work item: normalise directly
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = rows[h];
            if (r / kG >= nq) continue;
            const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
            const int64_t ob = (int64_t)a.perm[s0 + r / kG] * a.ldo + (kvh * kG + r % kG) * HD;
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                store_out(a, ob + 8 * n + 2 * t4, o[n][2 * h] * inv);
                store_out(a, ob + 8 * n + 2 * t4 + 1, o[n][2 * h + 1] * inv);
            }
        }
        return;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = rows[h];
        if (r / kG >= nq) continue;
        const int64_t row = (int64_t)(wd.w + r) * a.Hkv + kvh;
        if (t4 == 0) {
            a.part_m[row] = m[h];
            a.part_l[row] = l[h];
        }
#pragma unroll
        for (int n = 0; n < NC; ++n)
            *reinterpret_cast<float2*>(a.part_o + row * HD + 8 * n + 2 * t4) = make_float2(o[n][2 * h], o[n][2 * h + 1]);
    }
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
    merge_tile<HD, kG>(a, kvh, s0, nq, w0, w1, reinterpret_cast<float*>(smem), 4 * SM::tile_bytes / 4);
}

template <int HD, bool Q8, bool ONE>
bool launch_attention_mma_hd1(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    constexpr size_t smem = MmaSmem<HD, Q8>::bytes;
    auto k = attn_mma_kernel<HD, Q8, ONE>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return false;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_work, a.Hkv);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr_l[1];
    attr_l[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr_l[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr_l;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, a, scale_log2) == cudaSuccess;
}

// one f16 term for Q and P when the output goes to f16 GEMM operands (a single f16 output)
template <int HD, bool Q8>
bool launch_attention_mma_hd(const AttnArgs& a, cudaStream_t st) {
    return a.out_b && a.out_f16 ? launch_attention_mma_hd1<HD, Q8, true>(a, st)
                                : launch_attention_mma_hd1<HD, Q8, false>(a, st);
}

bool attention_mma_ok(const AttnArgs& a) {
    const bool kv = a.kv_type == W_F16 || (a.kv_type == W_Q8_0 && a.k_scale && a.v_scale);
    return kv && a.H == kG * a.Hkv && (a.hd == 32 || a.hd == 64 || a.hd == 128);
}

bool launch_attention_mma(const AttnArgs& a, cudaStream_t st) {
    if (a.kv_type == W_Q8_0) {
        switch (a.hd) {
            case 32: return launch_attention_mma_hd<32, true>(a, st);
            case 64: return launch_attention_mma_hd<64, true>(a, st);
            case 128: return launch_attention_mma_hd<128, true>(a, st);
        }
        return false;
    }
    switch (a.hd) {
        case 32: return launch_attention_mma_hd<32, false>(a, st);
        case 64: return launch_attention_mma_hd<64, false>(a, st);
        case 128: return launch_attention_mma_hd<128, false>(a, st);
    }
    return false;
}

}  // namespace llm
