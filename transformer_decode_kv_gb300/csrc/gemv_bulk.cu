// Decode GEMV with TMA bulk staging (sm_103a): y = x W^T for T <= 8 tokens, HBM-bound.
//
// ([P2] "llama.cpp Architecture", Example 4: MUL_MAT of a {K, M} weight by the ubatch's
// activations; RMS_NORM + MUL before the projections; ROPE + SET_ROWS after Q/K/V; ADD for the
// residual; SWIGLU; the output matrix and the greedy pick of [P1] Крок 14.)
//
// Each block owns a contiguous range of weight rows (an even split of the matrix across the
// grid, so every block streams the same number of bytes) and streams it from HBM into a ring of
// shared-memory stages with cp.async.bulk (one elected producer thread, mbarrier completion,
// evict-first L2 policy). Eight consumer warps read the stages in 512-byte slices (16 bytes per
// lane), multiply with the activations held in shared memory (float32, normalised in the
// prologue when the op starts with RMSNorm) and add their per-row partial sums into shared
// accumulators. Every weight byte is read once per call. The epilogue applies the op that
// follows the projection: store, residual add, SwiGLU (gate and up rows of one feature in the
// same block), RoPE of Q/K with the K/V rows written to their cache cells, or logits with a
// greedy pick folded into a packed atomicMax (value, lowest index).
//
// The weight stream does not depend on the previous kernel, so the producer starts it before
// griddepcontrol.wait (programmatic dependent launch); the consumers wait before touching
// activations. Every mbarrier wait is bounded (2 s) and reported in the error word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "dev_common.cuh"
#include "gemv_bulk.h"

namespace llm {

namespace {

using namespace dev;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr uint32_t kStageBytes = 16384;     // stage size of the general mapping
constexpr uint32_t kMaxStageBytes = 32768;
constexpr uint32_t kSlice = 512;                  // bytes per warp pass (16 per lane)
// Column-stationary Q8_0 rows use 8-byte lane chunks (256-byte slices): 8 quants per lane keep the
// activations of a 14336-wide row (7 slices per warp) in registers, and a chunk stays inside one
// 32-value block.
template <int WT> struct ColsGeom {
    static constexpr int CH = WT == W_Q8_0 ? 8 : 16;      // bytes per lane and slice
    static constexpr int SL = 32 * CH;                      // slice bytes
};
constexpr uint32_t kColsStage = 24576;            // column-stationary stage: whole rows up to 24 KB

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

struct Range { int64_t row0, nrows; int local0; };

// Column-stationary one-token variants with at most 32 weights per lane fit three blocks per SM
// without spilling: two of this kernel and one of the next, which programmatic dependent launch
// starts early to prefetch its weights.
template <int WT, int TM, int EPI, bool NORM, int SPW>
__global__ void __launch_bounds__(kThreads, TM == 1 && SPW > 0 && SPW * ColsGeom<WT>::CH / Vec<WT>::ES <= 32 ? 3
                                            : TM <= 2 ? 2 : 1)
gemv_bulk_kernel(const GemvArgs a) {
    constexpr bool COLS = SPW > 0;
    constexpr int VN = Vec<WT>::N, ES = Vec<WT>::ES;
    constexpr bool Q8 = WT == W_Q8_0;
    extern __shared__ __align__(128) uint8_t smem[];
    const int kStages = a.n_stages;
    const uint32_t SB = COLS ? (uint32_t)a.stage_bytes : kStageBytes;    // bytes per stage
    uint8_t* stages = smem;
    uint8_t* sstages = stages + kStages * SB;                               // Q8 scales
    float* xs = reinterpret_cast<float*>(sstages + (Q8 ? kStages * (SB / 16) : 0));
    const int64_t K = a.K;
    float* acc = xs + (COLS ? 0 : (size_t)TM * K);
    float* red = acc + (size_t)a.rows_cap * TM;                            // [8][TM] + inv[TM]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + (kConsumerWarps + 1) * TM + 2);
    full = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(full) + 7) & ~(uintptr_t)7);
    uint64_t* empty = full + kMaxStages;
    int* abort_flag = reinterpret_cast<int*>(empty + kMaxStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this block's units: an even split of the unit count (rows; features for SwiGLU), in
    // granules of 2 rows for Q/K/V so each RoPE pair stays in one block
    const int gran = EPI == GEPI_QKV ? 2 : 1;
    const int64_t units = (EPI == GEPI_SWIGLU ? a.F : a.M) / gran;
    const int64_t u0 = units * blockIdx.x / gridDim.x * gran;
    const int64_t u1 = units * (blockIdx.x + 1) / gridDim.x * gran;
    const int nloc = (int)(u1 - u0);
    Range rg[2];
    int nrg = 1;
    rg[0] = {a.row0 + u0, u1 - u0, 0};
    if (EPI == GEPI_SWIGLU) { rg[1] = {a.row0 + a.F + u0, u1 - u0, nloc}; nrg = 2; }
    const int64_t row_bytes = K * ES;
    // pieces: each range's bytes in kStageBytes chunks
    int64_t npieces = 0;
    int64_t rg_pieces[2] = {0, 0};
    for (int r = 0; r < nrg; ++r) {
        rg_pieces[r] = (rg[r].nrows * row_bytes + kStageBytes - 1) / kStageBytes;
        npieces += rg_pieces[r];
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the next kernel may start now: its weight stream does not depend on this one, and its
        // consumers wait (griddepcontrol.wait) for this grid to complete
        asm volatile("griddepcontrol.launch_dependents;");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---- producer: the weight stream does not depend on earlier kernels
        if (lane == 0) {
            uint64_t policy;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
            int64_t p = 0, issued = 0;
            for (int r = 0; r < nrg && !*(volatile int*)abort_flag; ++r) {
                const uint8_t* base = static_cast<const uint8_t*>(a.W) + rg[r].row0 * row_bytes;
                const int64_t total = rg[r].nrows * row_bytes;
                for (int64_t off = 0; off < total; off += SB, ++p) {
                    const int s = (int)(p % kStages);
                    const uint32_t ph = (uint32_t)(p / kStages) & 1u;
                    if (p >= kStages && !mbar_wait(&empty[s], ph ^ 1u)) {
                        atomicOr(a.err, ERR_TIMEOUT);
                        *(volatile int*)abort_flag = 1;
                        break;
                    }
                    const uint32_t nb = (uint32_t)(total - off < (int64_t)SB ? total - off : (int64_t)SB);
                    mbar_expect_tx(&full[s], nb + (Q8 ? nb / 16 : 0));
                    bulk_g2s(stages + (size_t)s * SB, base + off, nb, &full[s], policy);
                    if (Q8) {
                        const uint8_t* sb = reinterpret_cast<const uint8_t*>(a.S) +
                                            (rg[r].row0 * row_bytes + off) / 16;
                        bulk_g2s(sstages + (size_t)s * (SB / 16), sb, nb / 16, &full[s], policy);
                    }
                    issued = p + 1;
                }
            }
            // every copy issued has landed before the block may exit
            for (int64_t q = (issued > kStages ? issued - kStages : 0); q < issued; ++q)
                mbar_wait(&full[q % kStages], (uint32_t)(q / kStages) & 1u);
        }
        return;
    }

    // ---- consumers: activations depend on the previous kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int ctid = threadIdx.x;                 // 0 .. 255
    float* inv = red + kConsumerWarps * TM;
    // column-stationary mapping: each warp loads only its own columns of the (single) activation
    // row into registers; the RMS is reduced across the warps
    constexpr int kSpw = SPW > 0 ? SPW : 1;
    constexpr int CH = ColsGeom<WT>::CH, SL = ColsGeom<WT>::SL;
    constexpr int VC = COLS ? CH / ES : VN;               // values per lane chunk
    float xr[kSpw][VC];
    if constexpr (COLS) {
        const int src = a.x_rows ? a.x_rows[0] : 0;
        const float* xg = a.x + (int64_t)src * a.ldx;
        float ss = 0.f;
#pragma unroll
        for (int k2 = 0; k2 < kSpw; ++k2) {
            const int col = (warp * kSpw + k2) * (SL / ES) + lane * VC;
#pragma unroll
            for (int e = 0; e < VC; e += 4) {
                const float4 v = *reinterpret_cast<const float4*>(xg + col + e);
                xr[k2][e] = v.x; xr[k2][e + 1] = v.y; xr[k2][e + 2] = v.z; xr[k2][e + 3] = v.w;
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
        }
        if (NORM) {
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) red[warp] = ss;
            consumer_sync();
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) s += red[w];
            const float sc = 1.0f / sqrtf(s / (float)K + a.eps);
#pragma unroll
            for (int k2 = 0; k2 < kSpw; ++k2) {
                const int col = (warp * kSpw + k2) * (SL / ES) + lane * VC;
#pragma unroll
                for (int e = 0; e < VC; e += 4) {
                    const float4 g = *reinterpret_cast<const float4*>(a.g + col + e);
                    xr[k2][e] *= sc * g.x; xr[k2][e + 1] *= sc * g.y;
                    xr[k2][e + 2] *= sc * g.z; xr[k2][e + 3] *= sc * g.w;
                }
            }
        }
    } else {
    // one pass: every thread loads its share of each activation row (all loads in flight at
        // once), the RMS of each row is reduced across the consumers, and the scaled values go from
        // registers to shared memory
        constexpr int kXPerThread = 16;               // float4 per thread and row: K <= 16384
        for (int t = 0; t < TM; ++t) {
            const int src = (t < a.T) ? (a.x_rows ? a.x_rows[t] : t) : -1;
            float4 xv[kXPerThread];
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < kXPerThread; ++i) {
                const int64_t k = ((int64_t)i * kConsumerWarps * 32 + ctid) * 4;
                xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (src >= 0 && k < K) xv[i] = *reinterpret_cast<const float4*>(a.x + (int64_t)src * a.ldx + k);
                ss += xv[i].x * xv[i].x + xv[i].y * xv[i].y + xv[i].z * xv[i].z + xv[i].w * xv[i].w;
            }
            float sc = 1.f;
            if (NORM) {
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (lane == 0) red[warp * TM + t] = ss;
                consumer_sync();
                if (ctid == 0) {
                    float s = 0.f;
                    for (int w = 0; w < kConsumerWarps; ++w) s += red[w * TM + t];
                    inv[t] = 1.0f / sqrtf(s / (float)K + a.eps);
                }
                consumer_sync();
                sc = src >= 0 ? inv[t] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kXPerThread; ++i) {
                const int64_t k = ((int64_t)i * kConsumerWarps * 32 + ctid) * 4;
                if (k >= K) break;
                float4 v = xv[i];
                if (NORM) {
                    const float4 g = *reinterpret_cast<const float4*>(a.g + k);
                    v.x *= sc * g.x; v.y *= sc * g.y; v.z *= sc * g.z; v.w *= sc * g.w;
                }
                *reinterpret_cast<float4*>(xs + t * K + k) = v;
            }
        }
    }
    for (int i = ctid; i < a.rows_cap * TM; i += kConsumerWarps * 32) acc[i] = 0.f;
    consumer_sync();

    if constexpr (COLS) {
        // ---- column-stationary mapping: stages hold whole rows; warp w always reads the same
        // SPW slices of every row, so its activations sit in registers for the whole kernel.
        constexpr int spw = SPW;                               // slices per warp per row
        constexpr int kMaxSpw = SPW;
        bool ok = true;
        int64_t p = 0;
        const int rps = (int)(SB / row_bytes);                 // rows per stage
        for (int r = 0; r < nrg && ok; ++r) {
            const int64_t nrows = rg[r].nrows;
            for (int64_t row0 = 0; row0 < nrows; row0 += rps, ++p) {
                const int s = (int)(p % kStages);
                if (!mbar_wait(&full[s], (uint32_t)(p / kStages) & 1u) || *(volatile int*)abort_flag) {
                    atomicOr(a.err, ERR_TIMEOUT);
                    *(volatile int*)abort_flag = 1;
                    ok = false;
                    break;
                }
                const int nr = (int)(nrows - row0 < rps ? nrows - row0 : rps);
                const uint8_t* st0 = stages + (size_t)s * SB + (warp * spw) * SL + lane * CH;
                const __half* ssc = reinterpret_cast<const __half*>(sstages + (size_t)s * (SB / 16));
                // all rows of the stage at once (one token in this mapping): two independent
                // accumulators per row, the row reductions interleaved, then lane i adds row i's
                // sum to the shared total. A stage holds kColsStage bytes of whole rows.
                constexpr int RPS = (int)(kColsStage / (SPW * kConsumerWarps * SL)) > 0
                                        ? (int)(kColsStage / (SPW * kConsumerWarps * SL)) : 1;
                static_assert(TM == 1, "column-stationary mapping serves one token");
                float pa[RPS], pb[RPS];
#pragma unroll
                for (int i = 0; i < RPS; ++i) {
                    pa[i] = 0.f;
                    pb[i] = 0.f;
                    if (i < nr) {
#pragma unroll
                        for (int k2 = 0; k2 < kMaxSpw; ++k2) {
                            if constexpr (Q8) {
                                // a lane's 8 quants share one block scale: sum, then scale once
                                const uint2 wv = *reinterpret_cast<const uint2*>(st0 + (size_t)i * row_bytes + k2 * SL);
                                const float d = __half2float(
                                    ssc[((size_t)i * row_bytes + (warp * spw + k2) * SL + lane * CH) / 32]);
                                float w[8];
                                unpack_q8x8_raw(wv, w);
                                float la = 0.f, lb = 0.f;
#pragma unroll
                                for (int e = 0; e < 8; e += 2)
                                    fma2(la, lb, w[e], w[e + 1], xr[k2][e], xr[k2][e + 1]);
                                pa[i] = fmaf(d, la, pa[i]);
                                pb[i] = fmaf(d, lb, pb[i]);
                            } else {
                                const uint4 wv = *reinterpret_cast<const uint4*>(st0 + (size_t)i * row_bytes + k2 * SL);
                                float w[VN];
                                unpack16<WT>(wv, 0.f, w);
#pragma unroll
                                for (int e = 0; e < VN; e += 2)
                                    fma2(pa[i], pb[i], w[e], w[e + 1], xr[k2][e], xr[k2][e + 1]);
                            }
                        }
                    }
                    pa[i] += pb[i];
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int i = 0; i < RPS; ++i) pa[i] += __shfl_xor_sync(0xffffffffu, pa[i], o);
#pragma unroll
                for (int i = 0; i < RPS; ++i)
                    if (lane == i && i < nr) atomicAdd(&acc[rg[r].local0 + (int)(row0 + i)], pa[i]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
        }
    } else {
    // ---- main loop over the pieces. Warp w reads slices [w*SPW, (w+1)*SPW) of each piece; rows
    // hold a whole number of slices, so a warp's position advances row by row without division.
    constexpr int kSlicesPerWarp = kStageBytes / kSlice / kConsumerWarps;
    const uint32_t rbytes = (uint32_t)row_bytes;
    bool ok = true;
    int64_t p = 0;
    for (int r = 0; r < nrg && ok; ++r) {
        const uint32_t total = (uint32_t)(rg[r].nrows * row_bytes);
        // position of this warp's first slice in the range: row and byte within the row
        uint32_t wrow = (uint32_t)(warp * kSlicesPerWarp * kSlice) / rbytes;
        uint32_t wrem = (uint32_t)(warp * kSlicesPerWarp * kSlice) - wrow * rbytes;
        const uint32_t step_rows = kStageBytes / rbytes, step_rem = kStageBytes - step_rows * rbytes;
        for (uint32_t off = 0; off < total; off += kStageBytes, ++p) {
            const int s = (int)(p % kStages);
            if (!mbar_wait(&full[s], (uint32_t)(p / kStages) & 1u) || *(volatile int*)abort_flag) {
                atomicOr(a.err, ERR_TIMEOUT);
                *(volatile int*)abort_flag = 1;
                ok = false;
                break;
            }
            const uint32_t nb = total - off < kStageBytes ? total - off : kStageBytes;
            const int nslices = (int)(nb / kSlice);
            const uint8_t* sw = stages + s * kStageBytes + (warp * kSlicesPerWarp) * kSlice + lane * 16;
            const __half* ssc = reinterpret_cast<const __half*>(sstages + s * (kStageBytes / 16));
            float part[TM];
#pragma unroll
            for (int t = 0; t < TM; ++t) part[t] = 0.f;
            uint32_t row = wrow, rem = wrem;
#pragma unroll
            for (int j = 0; j < kSlicesPerWarp; ++j) {
                if (warp * kSlicesPerWarp + j >= nslices) break;
                if (rem == rbytes) {              // crossed into the next row: flush the last one
#pragma unroll
                    for (int t = 0; t < TM; ++t) {
                        float v = part[t];
                        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                        if (lane == 0) atomicAdd(&acc[(rg[r].local0 + (int)row) * TM + t], v);
                        part[t] = 0.f;
                    }
                    ++row;
                    rem = 0;
                }
                const uint4 wv = *reinterpret_cast<const uint4*>(sw + j * kSlice);
                float d = 0.f;
                if (Q8) d = __half2float(ssc[((warp * kSlicesPerWarp + j) * kSlice + lane * 16) / 32]);
                float w[VN];
                if constexpr (Q8) unpack_q8_raw(wv, w);
                else unpack16<WT>(wv, 0.f, w);
                const uint32_t col = rem / ES + lane * VN;
#pragma unroll
                for (int t = 0; t < TM; ++t) {
                    const float* xp = xs + t * K + col;
                    float ls = 0.f;
#pragma unroll
                    for (int e2 = 0; e2 < VN; e2 += 4) {
                        const float4 xv = *reinterpret_cast<const float4*>(xp + e2);
                        ls = fmaf(w[e2], xv.x, ls);
                        ls = fmaf(w[e2 + 1], xv.y, ls);
                        ls = fmaf(w[e2 + 2], xv.z, ls);
                        ls = fmaf(w[e2 + 3], xv.w, ls);
                    }
                    // Q8_0: a lane's 16 quants share one block scale
                    part[t] = Q8 ? fmaf(d, ls, part[t]) : part[t] + ls;
                }
                rem += kSlice;
            }
            if (warp * kSlicesPerWarp < nslices) {
#pragma unroll
                for (int t = 0; t < TM; ++t) {
                    float v = part[t];
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0) atomicAdd(&acc[(rg[r].local0 + (int)row) * TM + t], v);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            // advance this warp's position by one stage
            wrem += step_rem;
            wrow += step_rows;
            while (wrem >= rbytes) { wrem -= rbytes; ++wrow; }
        }
    }
    }
    consumer_sync();
    if (*(volatile int*)abort_flag) return;

    // ---- epilogue
    const int T = a.T;
    if (EPI == GEPI_STORE || EPI == GEPI_ADD) {
        for (int i = ctid; i < nloc * T; i += kConsumerWarps * 32) {
            const int t = i / nloc, rl = i % nloc;
            float* dst = a.y + (int64_t)t * a.ldy + u0 + rl;
            const float v = acc[rl * TM + t];
            *dst = EPI == GEPI_ADD ? *dst + v : v;
        }
    } else if (EPI == GEPI_SWIGLU) {
        for (int i = ctid; i < nloc * T; i += kConsumerWarps * 32) {
            const int t = i / nloc, rl = i % nloc;
            const float g = acc[rl * TM + t], u = acc[(nloc + rl) * TM + t];
            a.y[(int64_t)t * a.ldy + u0 + rl] = g / (1.0f + expf(-g)) * u;
        }
    } else if (EPI == GEPI_LOGITS) {
        for (int t = 0; t < T; ++t) {
            unsigned long long best = 0;
            for (int rl = ctid; rl < nloc; rl += kConsumerWarps * 32) {
                const float v = acc[rl * TM + t];
                a.y[(int64_t)t * a.ldy + u0 + rl] = v;
                if (v == v) {
                    const unsigned long long pk = pack_argmax(v, (int)(u0 + rl));
                    best = pk > best ? pk : best;
                }
            }
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
                best = ob > best ? ob : best;
            }
            if (lane == 0 && best) atomicMax(a.amax + t, best);
        }
    } else {  // GEPI_QKV: RoPE on Q and K rows, K/V rows to their cache cells, Q to y
        const int hd = a.hd, half = hd / 2;
        const int npairs = nloc / 2;
        for (int i = ctid; i < npairs * T; i += kConsumerWarps * 32) {
            const int t = i / npairs, pl = i % npairs;
            const int64_t r = u0 + 2 * pl;                 // even row of the Q|K|V matrix
            const int head = (int)(r / hd), dd = (int)(r % hd);
            float y0 = acc[(2 * pl) * TM + t], y1 = acc[(2 * pl + 1) * TM + t];
            if (head < a.H + a.Hkv) {
                const float2 e = a.cs[(int64_t)t * half + dd / 2];
                const float r0 = y0 * e.x - y1 * e.y, r1 = y0 * e.y + y1 * e.x;
                y0 = r0; y1 = r1;
            }
            if (head < a.H) {
                float* dst = a.y + (int64_t)t * a.ldy + r;
                dst[0] = y0; dst[1] = y1;
                continue;
            }
            const int32_t cell = a.slot ? a.slot[t] : t;
            if (cell < 0 || cell >= a.n_ctx) { atomicOr(a.err, ERR_SLOT_RANGE); continue; }
            const bool is_k = head < a.H + a.Hkv;
            const int g = is_k ? head - a.H : head - a.H - a.Hkv;
            const int64_t ci = ((int64_t)g * a.n_ctx + cell) * hd + dd;
            void* cache = is_k ? a.kc : a.vc;
            if (a.kv_type == W_F32) {
                static_cast<float*>(cache)[ci] = y0;
                static_cast<float*>(cache)[ci + 1] = y1;
            } else {
                static_cast<__half2*>(cache)[ci / 2] = __floats2half2_rn(y0, y1);
            }
        }
    }
}

template <int WT, int TM, int EPI, bool NORM, int SPW>
bool launch_one(const GemvArgs& a, int grid, size_t smem, cudaStream_t st, bool pdl) {
    auto k = gemv_bulk_kernel<WT, TM, EPI, NORM, SPW>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, a) == cudaSuccess;
}

// column-stationary variants (one token): slices per warp per row
template <int WT, int EPI, bool NORM>
bool launch_cols(const GemvArgs& a, int spw, int grid, size_t smem, cudaStream_t st, bool pdl) {
    switch (spw) {
        case 1: return launch_one<WT, 1, EPI, NORM, 1>(a, grid, smem, st, pdl);
        case 2: return launch_one<WT, 1, EPI, NORM, 2>(a, grid, smem, st, pdl);
        case 4: return launch_one<WT, 1, EPI, NORM, 4>(a, grid, smem, st, pdl);
        case 7: return launch_one<WT, 1, EPI, NORM, 7>(a, grid, smem, st, pdl);
    }
    return false;
}

template <int WT, int EPI, bool NORM>
bool launch_tm(const GemvArgs& a, int spw, int grid, size_t smem, cudaStream_t st, bool pdl) {
    if (spw > 0) return launch_cols<WT, EPI, NORM>(a, spw, grid, smem, st, pdl);
    switch (gemv_bulk_tm(a.T)) {
        case 1: return launch_one<WT, 1, EPI, NORM, 0>(a, grid, smem, st, pdl);
        case 2: return launch_one<WT, 2, EPI, NORM, 0>(a, grid, smem, st, pdl);
        case 4: return launch_one<WT, 4, EPI, NORM, 0>(a, grid, smem, st, pdl);
        default: return launch_one<WT, 8, EPI, NORM, 0>(a, grid, smem, st, pdl);
    }
}

template <int EPI, bool NORM>
bool launch_wt(int wt, const GemvArgs& a, int spw, int grid, size_t smem, cudaStream_t st, bool pdl) {
    switch (wt) {
        case W_F32: return launch_tm<W_F32, EPI, NORM>(a, spw, grid, smem, st, pdl);
        case W_F16: return launch_tm<W_F16, EPI, NORM>(a, spw, grid, smem, st, pdl);
        case W_BF16: return launch_tm<W_BF16, EPI, NORM>(a, spw, grid, smem, st, pdl);
        case W_Q8_0: return launch_tm<W_Q8_0, EPI, NORM>(a, spw, grid, smem, st, pdl);
    }
    return false;
}

int64_t wrow_bytes(int wt, int64_t K) {
    return wt == W_F32 ? K * 4 : wt == W_Q8_0 ? K : K * 2;
}

}  // namespace

int gemv_bulk_tm(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }

// Grid and shared memory of a launch; 0 if the bulk path does not apply.
static int plan_grid(int wt, const GemvArgs& a, int epi, int n_sm, size_t* smem, int* rows_cap,
                     int* n_stages, int* stage_bytes) {
    if (a.T < 1 || a.T > 8) return 0;
    const int64_t rb = wrow_bytes(wt, a.K);
    if (rb % kSlice != 0 || a.K % 4 != 0 || a.K > 16384) return 0;
    if (wt == W_Q8_0 && a.K % 512 != 0) return 0;
    const int tm = gemv_bulk_tm(a.T);
    const int gran = epi == GEPI_QKV ? 2 : 1;
    const int64_t units = (epi == GEPI_SWIGLU ? a.F : a.M) / gran;
    if (units <= 0) return 0;
    // column-stationary mapping: whole rows per stage, each warp owns a fixed eighth of a row
    const int64_t cols_slice = wt == W_Q8_0 ? 256 : kSlice;      // ColsGeom<WT>::SL
    const int64_t spr = rb / cols_slice;
    const int vn = wt == W_F32 ? 4 : 8;                           // values per lane chunk
    const int64_t spw = spr % kConsumerWarps == 0 ? spr / kConsumerWarps : 0;
    const bool cols = tm == 1 && (spw == 1 || spw == 2 || spw == 4 || spw == 7) && spw * vn <= 64 &&
                      rb <= kMaxStageBytes;
    (void)vn;
    const uint32_t sbytes = cols ? (uint32_t)(rb * std::max<int64_t>(1, kColsStage / rb) <= kMaxStageBytes
                                              ? rb * std::max<int64_t>(1, kColsStage / rb) : rb)
                                 : kStageBytes;
    *stage_bytes = cols ? (int)sbytes : 0;
    const size_t per_stage = sbytes + (wt == W_Q8_0 ? sbytes / 16 : 0);
    const size_t fixed = (cols ? 0 : (size_t)tm * a.K * 4) + ((kConsumerWarps + 1) * tm + 2) * 4 + 8 +
                         2 * kMaxStages * 8 + 16;
    for (int per_sm = tm <= 2 ? 2 : 1; per_sm >= 1; --per_sm) {
        const int64_t grid = std::min<int64_t>(units, (int64_t)n_sm * per_sm);
        const int64_t cap = (units + grid - 1) / grid * gran * (epi == GEPI_SWIGLU ? 2 : 1);
        // two blocks per SM leave room for a third: the next kernel's block, started early by
        // programmatic dependent launch, prefetches its weights while these finish. Rows longer
        // than 16 KB (one row per stage, 7 slices per warp) need ~92 registers, so no third
        // block fits beside two of these anyway: they take 108 KB for a third stage instead.
        const size_t budget = per_sm == 2 ? (cols && rb > 16384 ? 108u : 74u) * 1024u : 224u * 1024u;
        const size_t base = fixed + (size_t)cap * tm * 4;
        const int min_stages = cols && per_stage > 20000 ? 2 : 3;
        if (base + min_stages * per_stage > budget) continue;
        const int ns = (int)std::min<size_t>(std::min<size_t>(kMaxStages, cols ? 4 : kMaxStages),
                                             (budget - base) / per_stage);
        *n_stages = ns;
        *smem = base + (size_t)ns * per_stage;
        *rows_cap = (int)cap;
        return (int)grid;
    }
    return 0;
}

bool gemv_bulk_ok(int wt, const GemvArgs& a, int epi, int n_sm) {
    size_t s; int c, ns, sb;
    return plan_grid(wt, a, epi, n_sm, &s, &c, &ns, &sb) > 0;
}

bool launch_gemv_bulk(int wt, GemvArgs a, int epi, bool norm, int n_sm, cudaStream_t st, bool pdl) {
    size_t smem = 0;
    int cap = 0, ns = 0, sb = 0;
    const int grid = plan_grid(wt, a, epi, n_sm, &smem, &cap, &ns, &sb);
    if (grid <= 0) return false;
    a.rows_cap = cap;
    a.n_stages = ns;
    a.stage_bytes = sb;
    const int spw = sb > 0 ? (int)(wrow_bytes(wt, a.K) / (wt == W_Q8_0 ? 256 : kSlice) / kConsumerWarps) : 0;
    // the (epilogue, norm) pairs the decode path uses
    switch (epi) {
        case GEPI_STORE: if (!norm) return launch_wt<GEPI_STORE, false>(wt, a, spw, grid, smem, st, pdl); break;
        case GEPI_ADD: if (!norm) return launch_wt<GEPI_ADD, false>(wt, a, spw, grid, smem, st, pdl); break;
        case GEPI_SWIGLU: if (norm) return launch_wt<GEPI_SWIGLU, true>(wt, a, spw, grid, smem, st, pdl); break;
        case GEPI_QKV: if (norm) return launch_wt<GEPI_QKV, true>(wt, a, spw, grid, smem, st, pdl); break;
        case GEPI_LOGITS: if (norm) return launch_wt<GEPI_LOGITS, true>(wt, a, spw, grid, smem, st, pdl); break;
    }
    return false;
}

}  // namespace llm
