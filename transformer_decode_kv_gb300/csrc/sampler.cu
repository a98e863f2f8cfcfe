// The sampler chain on the device ([P1] "llama.cpp AI LLM Engine - Як це працює", the sampler
// chain after Крок 14: repeat penalty, top-k, top-p, min-p, temperature, then one token picked
// greedily or at random; a backend sampler picks on the device so the logits need not be copied
// to the host).
//
// One block over one logits row (V floats):
//   1. the row into a scratch row, the repeat penalty applied to each distinct listed token
//      (l > 0 -> l / r, else l * r);
//   2. the k-th largest value by a 4-pass radix select (8-bit digits) over an order-preserving
//      integer key; candidates = every value above it, plus the lowest token ids among those equal
//      to it (a block-wide prefix count over contiguous chunks keeps that deterministic);
//   3. a bitonic sort of the candidates by (value descending, token id ascending);
//   4. one thread walks the sorted list: top-p on the untempered probabilities (the shortest
//      prefix reaching p), min-p (l - l_max >= ln min_p), then temperature and the pick: the first
//      candidate whose cumulative weight exp((l - l_max) / t) exceeds u times the total, u being
//      the caller's uniform draw in [0, 1); t <= 0 picks the first candidate.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace llm {

namespace {

constexpr int kThreadsS = 1024;
constexpr int kMaxK = 4096;

__device__ __forceinline__ uint32_t fkey(float v) {
    if (v != v) return 0u;                                  // NaN sorts below everything
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kThreadsS) sample_kernel(SampleArgs a) {
    __shared__ uint32_t hist[256];
    __shared__ unsigned long long cand[kMaxK];              // (~key << 32) | token id
    __shared__ uint32_t chunk_eq[kThreadsS];
    __shared__ uint32_t s_prefix, s_mask, s_remaining, n_cand;
    const int tid = threadIdx.x;
    const int V = a.V;
    float* row = a.scratch;

    // 1. penalised copy of the row
    for (int v = tid; v < V; v += kThreadsS) row[v] = a.logits[v];
    __syncthreads();
    if (a.penalty != 1.0f) {
        for (int j = tid; j < a.n_pen; j += kThreadsS) {
            const int t = a.pen_tok[j];
            bool first = t >= 0 && t < V;
            for (int i = 0; i < j && first; ++i) first = a.pen_tok[i] != t;
            if (first) row[t] = row[t] > 0.f ? row[t] / a.penalty : row[t] * a.penalty;
        }
    }
    __syncthreads();

    // 2. radix select of the k-th largest key
    const uint32_t k = (uint32_t)min(a.top_k, V);
    if (tid == 0) { s_prefix = 0u; s_mask = 0u; s_remaining = k; n_cand = 0u; }
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreadsS) hist[i] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        for (int v = tid; v < V; v += kThreadsS) {
            const uint32_t key = fkey(row[v]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t rem = s_remaining, acc = 0u;
            int d = 255;
            for (; d > 0; --d) {
                if (acc + hist[d] >= rem) break;
                acc += hist[d];
            }
            s_prefix = prefix | ((uint32_t)d << shift);
            s_mask = mask | (0xFFu << shift);
            s_remaining = rem - acc;
        }
        __syncthreads();
    }
    const uint32_t thr = s_prefix, need_eq = s_remaining;    // take need_eq of the keys == thr

    // candidates above the threshold
    for (int v = tid; v < V; v += kThreadsS) {
        const uint32_t key = fkey(row[v]);
        if (key > thr) {
            const uint32_t j = atomicAdd(&n_cand, 1u);
            if (j < (uint32_t)kMaxK) cand[j] = ((unsigned long long)(~key) << 32) | (uint32_t)v;
        }
    }
    // ties at the threshold: the lowest token ids, by a prefix count over contiguous chunks
    const int chunk = (V + kThreadsS - 1) / kThreadsS;
    const int v0 = tid * chunk, v1 = min(V, v0 + chunk);
    uint32_t cnt = 0u;
    for (int v = v0; v < v1; ++v) cnt += fkey(row[v]) == thr;
    chunk_eq[tid] = cnt;
    __syncthreads();
    if (tid == 0) {
        uint32_t run = 0u;
        for (int i = 0; i < kThreadsS; ++i) { const uint32_t c = chunk_eq[i]; chunk_eq[i] = run; run += c; }
    }
    __syncthreads();
    uint32_t rank = chunk_eq[tid];
    for (int v = v0; v < v1 && rank < need_eq; ++v) {
        if (fkey(row[v]) != thr) continue;
        const uint32_t j = atomicAdd(&n_cand, 1u);
        if (j < (uint32_t)kMaxK) cand[j] = ((unsigned long long)(~thr) << 32) | (uint32_t)v;
        ++rank;
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

    // 4. cut-offs, temperature and the pick, in the sorted order
    if (tid == 0) {
        if (n == 0u) { atomicOr(a.err, ERR_ROW_RANGE); *a.out = -1; return; }
        const float l0 = row[(uint32_t)cand[0]];
        uint32_t m = n;
        if (a.top_p < 1.0f) {
            float z = 0.f;
            for (uint32_t i = 0; i < m; ++i) z += expf(row[(uint32_t)cand[i]] - l0);
            float c = 0.f;
            uint32_t keep = m;
            for (uint32_t i = 0; i < m; ++i) {
                c += expf(row[(uint32_t)cand[i]] - l0);
                if (c / z >= a.top_p) { keep = i + 1; break; }
            }
            m = keep;
        }
        if (a.min_p > 0.0f) {
            const float lm = logf(a.min_p);
            uint32_t keep = 1;
            while (keep < m && row[(uint32_t)cand[keep]] - l0 >= lm) ++keep;
            m = keep;
        }
        int token = (int)(uint32_t)cand[0];
        if (a.temperature > 0.0f) {
            float z = 0.f;
            for (uint32_t i = 0; i < m; ++i) z += expf((row[(uint32_t)cand[i]] - l0) / a.temperature);
            const float target = a.u * z;
            float c = 0.f;
            token = (int)(uint32_t)cand[m - 1];
            for (uint32_t i = 0; i < m; ++i) {
                c += expf((row[(uint32_t)cand[i]] - l0) / a.temperature);
                if (c > target) { token = (int)(uint32_t)cand[i]; break; }
            }
        }
        *a.out = token;
    }
}

}  // namespace

int sample_max_k() { return kMaxK; }

bool launch_sample(const SampleArgs& a, cudaStream_t st) {
    if (a.V <= 0 || a.top_k < 1 || a.top_k > kMaxK) return false;
    sample_kernel<<<1, kThreadsS, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace llm
