// The sampler chain on the device ([P1] "llama.cpp AI LLM Engine - Як це працює", the sampler
// chain after Крок 14: repeat penalty, top-k, top-p, min-p, temperature, then one token picked
// greedily or at random; a backend sampler picks on the device so the logits need not be copied
// to the host).
//
// One block of 1024 threads over one logits row (V floats):
//   1. the row into a scratch row, the repeat penalty applied to each distinct listed token
//      (l > 0 -> l / r, else l * r);
//   2. the k-th largest value by a 3-pass radix select (11, 11, 10 bits) over an order-preserving
//      integer key (histograms aggregated per warp, the digit found by a block scan);
//      candidates = every value above it, plus the lowest token ids among those equal to it
//      (when more are equal than needed, a block scan over contiguous chunks ranks them);
//   3. a bitonic sort of the candidates by (value descending, token id ascending);
//   4. over the sorted list, with block scans: top-p on the untempered probabilities (the
//      shortest prefix reaching p), min-p (l - l_max >= ln min_p), then temperature and the pick:
//      the first candidate whose cumulative weight exp((l - l_max) / t) exceeds u times the
//      total, u being the caller's uniform draw in [0, 1); t <= 0 picks the first candidate.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace llm {

namespace {

constexpr int kThreadsS = 1024;
constexpr int kWarpsS = kThreadsS / 32;
constexpr int kMaxK = 4096;
constexpr int kPer = kMaxK / kThreadsS;                  // sorted candidates per thread
constexpr int kBins = 2048;

__device__ __forceinline__ uint32_t fkey(float v) {
    if (v != v) return 0u;                                  // NaN sorts below everything
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Calls f(v, x, ok) for every value x = row[v] of the scratch row (16-byte aligned, V % 4 == 0),
// 16 values per thread and step loaded as four float4 before any is used, so each thread keeps
// four loads in flight. Every thread makes the same number of calls (ok = false past the end):
// f may use warp-wide intrinsics.
template <typename F>
__device__ __forceinline__ void for_each_value(const float* row, int V, F&& f) {
    constexpr int kU = 4;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int V4 = V / 4;
    for (int i0 = 0; i0 < V4; i0 += kThreadsS * kU) {
        float4 x[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = i0 + u * kThreadsS + (int)threadIdx.x;
            x[u] = i < V4 ? r4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = i0 + u * kThreadsS + (int)threadIdx.x;
            const bool ok = i < V4;
            f(4 * i, x[u].x, ok);
            f(4 * i + 1, x[u].y, ok);
            f(4 * i + 2, x[u].z, ok);
            f(4 * i + 3, x[u].w, ok);
        }
    }
}

// Inclusive sum over the block's threads (every thread calls it; wsum holds 32 words).
template <typename T>
__device__ T block_scan(T v, T* wsum, T* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const T n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        T w = wsum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const T n = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += n;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += wsum[warp - 1];
    if (total) *total = wsum[kWarpsS - 1];
    __syncthreads();                                        // wsum free for the next scan
    return v;
}

__global__ void __launch_bounds__(kThreadsS) sample_kernel(SampleArgs a) {
    __shared__ uint32_t hist[kBins];
    __shared__ unsigned long long cand[kMaxK];              // (~key << 32) | token id
    __shared__ uint32_t wsum_u[32];
    __shared__ float wsum_f[32];
    __shared__ uint32_t s_prefix, s_remaining, n_cand, s_first;
    const int tid = threadIdx.x, lane = tid & 31;
    const int V = a.V;
    float* row = a.scratch;

    // 1. penalised copy of the row (padded with -inf to a multiple of 4 values; the padding is
    // never a candidate because k <= V); eight independent loads per thread in flight
    const int Vp = (V + 3) & ~3;
    for (int v0 = 0; v0 < Vp; v0 += 8 * kThreadsS) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int v = v0 + u * kThreadsS + tid;
            x[u] = v < V ? a.logits[v] : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int v = v0 + u * kThreadsS + tid;
            if (v < Vp) row[v] = x[u];
        }
    }
    __syncthreads();
    if (a.penalty != 1.0f) {
        // the listed tokens in shared memory (the candidate buffer is free until step 2)
        int* pen = reinterpret_cast<int*>(cand);
        const int np = min(a.n_pen, 2 * kMaxK);
        for (int j = tid; j < np; j += kThreadsS) pen[j] = a.pen_tok[j];
        __syncthreads();
        for (int j = tid; j < np; j += kThreadsS) {
            const int t = pen[j];
            bool first = t >= 0 && t < V;
            for (int i = 0; i < j && first; ++i) first = pen[i] != t;
            if (first) row[t] = row[t] > 0.f ? row[t] / a.penalty : row[t] * a.penalty;
        }
        __syncthreads();
    }
    if (tid == 0) { s_prefix = 0u; s_remaining = (uint32_t)min(a.top_k, V); n_cand = 0u; }
    __syncthreads();

    // 2. radix select of the k-th largest key: digits of 11, 11 and 10 bits from the top
    uint32_t mask = 0u;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
        const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
        for (int i = tid; i < kBins; i += kThreadsS) hist[i] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        for_each_value(row, Vp, [&](int v, float x, bool ok) {
            uint32_t bin = 0xFFFFFFFFu;
            if (ok && v < V) {
                const uint32_t key = fkey(x);
                if ((key & mask) == prefix) bin = (key >> shift) & dmask;
            }
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (bin != 0xFFFFFFFFu && lane == __ffs(same) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(same));
        });
        __syncthreads();
        // thread i holds bins 2047 - 2i and 2046 - 2i (descending): the digit where the count
        // from the top reaches the remaining rank
        const uint32_t rem = s_remaining;
        const int b_hi = kBins - 1 - 2 * tid, b_lo = b_hi - 1;
        const uint32_t c = hist[b_hi] + hist[b_lo];
        const uint32_t incl = block_scan<uint32_t>(c, wsum_u, nullptr);
        const uint32_t excl = incl - c;
        if (excl < rem && incl >= rem) {
            const bool in_hi = excl + hist[b_hi] >= rem;
            const uint32_t d = (uint32_t)(in_hi ? b_hi : b_lo);
            s_prefix = prefix | (d << shift);
            s_remaining = rem - (in_hi ? excl : excl + hist[b_hi]);
        }
        mask |= dmask << shift;
        __syncthreads();
    }
    const uint32_t thr = s_prefix, need_eq = s_remaining;  // take need_eq of the keys == thr
    const uint32_t n_eq = hist[thr & 0x3FFu];                // keys equal to thr (last histogram)

    // candidates above the threshold (and all the equal ones when exactly enough are equal)
    const bool take_all_eq = n_eq == need_eq;
    for_each_value(row, Vp, [&](int v, float x, bool ok) {
        uint32_t key = 0u;
        bool take = false;
        if (ok && v < V) {
            key = fkey(x);
            take = key > thr || (take_all_eq && key == thr);
        }
        const unsigned ball = __ballot_sync(0xffffffffu, take);
        if (ball) {
            uint32_t base = 0u;
            if (lane == 0) base = atomicAdd(&n_cand, (uint32_t)__popc(ball));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (take) {
                const uint32_t j = base + __popc(ball & ((1u << lane) - 1u));
                if (j < (uint32_t)kMaxK) cand[j] = ((unsigned long long)(~key) << 32) | (uint32_t)v;
            }
        }
    });
    if (!take_all_eq) {
        // more keys equal the threshold than needed: the lowest token ids, ranked by a block
        // scan of per-thread counts over contiguous chunks
        __syncthreads();
        const int chunk = (V + kThreadsS - 1) / kThreadsS;
        const int v0 = tid * chunk, v1 = min(V, v0 + chunk);
        uint32_t cnt = 0u;
        for (int v = v0; v < v1; ++v) cnt += fkey(row[v]) == thr;
        uint32_t rank = block_scan<uint32_t>(cnt, wsum_u, nullptr) - cnt;
        for (int v = v0; v < v1 && rank < need_eq; ++v) {
            if (fkey(row[v]) != thr) continue;
            const uint32_t j = atomicAdd(&n_cand, 1u);
            if (j < (uint32_t)kMaxK) cand[j] = ((unsigned long long)(~thr) << 32) | (uint32_t)v;
            ++rank;
        }
    }
    __syncthreads();

    // 3. bitonic sort, ascending on (~key, id) = value descending, id ascending
    const uint32_t n = min(n_cand, (uint32_t)kMaxK);
    uint32_t P = 1u;
    while (P < n) P <<= 1;
    for (uint32_t i = n + tid; i < P; i += kThreadsS) cand[i] = ~0ull;
    __syncthreads();
    for (uint32_t size = 2; size <= P; size <<= 1) {
        for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (uint32_t i = tid; i < P; i += kThreadsS) {
                const uint32_t jx = i ^ stride;
                if (jx > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long x = cand[i], y = cand[jx];
                    if ((x > y) == up) { cand[i] = y; cand[jx] = x; }
                }
            }
            __syncthreads();
        }
    }
    if (n == 0u) {
        if (tid == 0) { *a.out = -1; *a.err = ERR_ROW_RANGE; }
        return;
    }

    // 4. cut-offs, temperature and the pick over the sorted list; thread t holds candidates
    // kPer t .. kPer t + kPer - 1
    const float l0 = row[(uint32_t)cand[0]];
    float lv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const uint32_t i = (uint32_t)(tid * kPer + j);
        lv[j] = i < n ? row[(uint32_t)cand[i]] : -INFINITY;
    }
    uint32_t m = n;
    auto first_index = [&](bool hit, uint32_t i) {          // block-wide smallest i with hit
        if (tid == 0) s_first = 0xFFFFFFFFu;
        __syncthreads();
        if (hit) atomicMin(&s_first, i);
        __syncthreads();
        const uint32_t f = s_first;
        __syncthreads();
        return f;
    };
    if (a.top_p < 1.0f) {
        float e[kPer], loc = 0.f;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            e[j] = (uint32_t)(tid * kPer + j) < m ? expf(lv[j] - l0) : 0.f;
            loc += e[j];
        }
        float z = 0.f;
        float c = block_scan<float>(loc, wsum_f, &z) - loc;
        uint32_t hit = 0xFFFFFFFFu;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            c += e[j];
            const uint32_t i = (uint32_t)(tid * kPer + j);
            if (i < m && hit == 0xFFFFFFFFu && c / z >= a.top_p) hit = i;
        }
        const uint32_t f = first_index(hit != 0xFFFFFFFFu, hit);
        if (f != 0xFFFFFFFFu) m = f + 1;
    }
    if (a.min_p > 0.0f) {
        const float lm = logf(a.min_p);
        uint32_t miss = 0xFFFFFFFFu;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const uint32_t i = (uint32_t)(tid * kPer + j);
            if (i >= 1 && i < m && miss == 0xFFFFFFFFu && !(lv[j] - l0 >= lm)) miss = i;
        }
        const uint32_t f = first_index(miss != 0xFFFFFFFFu, miss);
        if (f != 0xFFFFFFFFu) m = f;
    }
    int token = (int)(uint32_t)cand[0];
    if (a.temperature > 0.0f) {
        float w[kPer], loc = 0.f;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            w[j] = (uint32_t)(tid * kPer + j) < m ? expf((lv[j] - l0) / a.temperature) : 0.f;
            loc += w[j];
        }
        float z = 0.f;
        float c = block_scan<float>(loc, wsum_f, &z) - loc;
        const float target = a.u * z;
        uint32_t hit = 0xFFFFFFFFu;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            c += w[j];
            const uint32_t i = (uint32_t)(tid * kPer + j);
            if (i < m && hit == 0xFFFFFFFFu && c > target) hit = i;
        }
        const uint32_t f = first_index(hit != 0xFFFFFFFFu, hit);
        token = (int)(uint32_t)cand[f != 0xFFFFFFFFu ? f : m - 1];
    }
    if (tid == 0) { *a.out = token; *a.err = 0u; }
}

}  // namespace

int sample_max_k() { return kMaxK; }

bool launch_sample(const SampleArgs& a, cudaStream_t st) {
    if (a.V <= 0 || a.top_k < 1 || a.top_k > kMaxK) return false;
    sample_kernel<<<1, kThreadsS, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace llm
