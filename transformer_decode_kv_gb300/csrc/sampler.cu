// The sampler chain on the device ([P1] "llama.cpp AI LLM Engine - Як це працює", the sampler
// chain after Крок 14: repeat penalty, top-k, top-p, min-p, temperature, then one token picked
// greedily or at random; a backend sampler picks on the device so the logits need not be copied
// to the host).
//
// One cooperative launch of G blocks; block b owns the contiguous slice [b V / G, (b + 1) V / G)
// of the logits row and keeps it in shared memory:
//   1. the slice with the repeat penalty applied to each distinct listed token of it
//      (l > 0 -> l / r, else l * r);
//   2. the k-th largest value by a 3-pass radix select (11, 11, 10 bits) over an order-preserving
//      integer key: per pass every block adds its slice's histogram to a global one, a grid
//      barrier, then every block finds the digit in it (a block scan); candidates = every value
//      above the k-th, plus the lowest token ids among those equal to it (blocks rank their ties
//      by slice order after one more barrier);
//   3. block 0 sorts the candidates by (value descending, token id ascending) (bitonic);
//   4. block 0, with block scans over the sorted list: top-p on the untempered probabilities (the
//      shortest prefix reaching p), min-p (l - l_max >= ln min_p), then temperature and the pick:
//      the first candidate whose cumulative weight exp((l - l_max) / t) exceeds u times the total,
//      u being the caller's uniform draw in [0, 1); t <= 0 picks the first candidate.
// The grid barriers spin on a generation counter with a bounded wait: past the limit the kernel
// sets the status word and returns, so a stalled grid ends with an error instead of hanging.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace llm {

namespace {

constexpr int kThreadsS = 512;
constexpr int kWarpsS = kThreadsS / 32;
constexpr int kMaxK = 4096;
constexpr int kPer = kMaxK / kThreadsS;                  // sorted candidates per thread (block 0)
constexpr int kBins = 2048;
constexpr int kSliceMax = 4096;                          // values per block
constexpr int kMaxBlocks = 128;
constexpr uint32_t kSpinLimit = 1u << 22;                // x 64 ns sleeps: about a quarter second

// Global state of one sampler: grid barrier, the three histograms, candidates and tie counts.
// The barrier is generation-based and leaves its count at 0, so only the histograms and the
// candidate counter need zeroing, done inside the launch before the first barrier.
struct SampleCtl {
    uint32_t bar_count, bar_gen, n_cand, status;
    uint32_t hist[3][kBins];
    uint32_t ties[kMaxBlocks];
    unsigned long long cand[kMaxK];
};

__device__ __forceinline__ uint32_t fkey(float v) {
    if (v != v) return 0u;                                  // NaN sorts below everything
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
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
        T w = lane < kWarpsS ? wsum[lane] : T(0);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const T n = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += n;
        }
        if (lane < kWarpsS) wsum[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += wsum[warp - 1];
    if (total) *total = wsum[kWarpsS - 1];
    __syncthreads();                                        // wsum free for the next scan
    return v;
}

// Grid-wide barrier over the co-resident blocks of a cooperative launch. false after a timeout
// (the status word is then set, and every block leaves).
__device__ bool grid_sync(SampleCtl* ctl, uint32_t nblocks, int* s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint32_t gen = *(volatile uint32_t*)&ctl->bar_gen;
        __threadfence();
        if (atomicAdd(&ctl->bar_count, 1u) + 1u == nblocks) {
            ctl->bar_count = 0u;
            __threadfence();
            atomicAdd(&ctl->bar_gen, 1u);
        } else {
            uint32_t n = 0;
            while (*(volatile uint32_t*)&ctl->bar_gen == gen) {
                if (++n > kSpinLimit || *(volatile uint32_t*)&ctl->status != 0u) { ok = 0; break; }
                __nanosleep(64);
            }
            if (!ok) atomicOr(&ctl->status, ERR_TIMEOUT);
        }
        __threadfence();
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

struct SampleParams {
    SampleArgs a;
    SampleCtl* ctl;
};

__global__ void __launch_bounds__(kThreadsS) sample_kernel(SampleParams prm) {
    const SampleArgs& a = prm.a;
    SampleCtl* ctl = prm.ctl;
    __shared__ union {
        struct { float vals[kSliceMax]; uint32_t hist[kBins]; } s;   // steps 1-2, every block
        unsigned long long cand[kMaxK];                                // steps 3-4, block 0
    } sm;
    __shared__ uint32_t wsum_u[32];
    __shared__ float wsum_f[32];
    __shared__ uint32_t s_prefix, s_remaining, s_first;
    __shared__ int s_ok;
    const int tid = threadIdx.x, lane = tid & 31;
    const int V = a.V;
    const uint32_t G = gridDim.x;
    const int b0 = (int)((int64_t)V * blockIdx.x / G), b1 = (int)((int64_t)V * (blockIdx.x + 1) / G);
    const int nv = b1 - b0;

    // zero the global histograms and counter (ordered before their use by the first barrier)
    for (int i = blockIdx.x * kThreadsS + tid; i < 3 * kBins; i += G * kThreadsS) (&ctl->hist[0][0])[i] = 0u;
    if (blockIdx.x == 0 && tid == 0) ctl->n_cand = 0u;

    // 1. the penalised slice
    for (int i = tid; i < nv; i += kThreadsS) sm.s.vals[i] = a.logits[b0 + i];
    __syncthreads();
    if (a.penalty != 1.0f) {
        for (int j = tid; j < a.n_pen; j += kThreadsS) {
            const int t = a.pen_tok[j];
            if (t < b0 || t >= b1) continue;
            bool first = true;
            for (int i = 0; i < j && first; ++i) first = a.pen_tok[i] != t;
            if (first) {
                const float l = sm.s.vals[t - b0];
                sm.s.vals[t - b0] = l > 0.f ? l / a.penalty : l * a.penalty;
            }
        }
    }
    if (tid == 0) { s_prefix = 0u; s_remaining = (uint32_t)min(a.top_k, V); }
    if (!grid_sync(ctl, G, &s_ok)) return;

    // 2. radix select of the k-th largest key: digits of 11, 11 and 10 bits from the top
    uint32_t mask = 0u;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
        const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
        for (int i = tid; i < kBins; i += kThreadsS) sm.s.hist[i] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        for (int i0 = 0; i0 < nv; i0 += kThreadsS) {       // same trip count in every lane
            const int i = i0 + tid;
            uint32_t bin = 0xFFFFFFFFu;
            if (i < nv) {
                const uint32_t key = fkey(sm.s.vals[i]);
                if ((key & mask) == prefix) bin = (key >> shift) & dmask;
            }
            if (__any_sync(0xffffffffu, bin != 0xFFFFFFFFu)) {
                const unsigned same = __match_any_sync(0xffffffffu, bin);
                if (bin != 0xFFFFFFFFu && lane == __ffs(same) - 1)
                    atomicAdd(&sm.s.hist[bin], (uint32_t)__popc(same));
            }
        }
        __syncthreads();
        for (int i = tid; i < kBins; i += kThreadsS)
            if (sm.s.hist[i]) atomicAdd(&ctl->hist[pass][i], sm.s.hist[i]);
        if (!grid_sync(ctl, G, &s_ok)) return;
        // every block: the digit where the count from the top reaches the remaining rank (thread
        // i holds the 4 bins 2047 - 4i .. 2044 - 4i, descending)
        const uint32_t rem = s_remaining;
        uint32_t hb[4], c = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hb[j] = __ldcg(&ctl->hist[pass][kBins - 1 - 4 * tid - j]);
            c += hb[j];
        }
        const uint32_t incl = block_scan<uint32_t>(c, wsum_u, nullptr);
        uint32_t acc = incl - c;
        if (acc < rem && incl >= rem) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (acc + hb[j] >= rem) {
                    s_prefix = prefix | ((uint32_t)(kBins - 1 - 4 * tid - j) << shift);
                    s_remaining = rem - acc;
                    break;
                }
                acc += hb[j];
            }
        }
        mask |= dmask << shift;
        __syncthreads();
    }
    const uint32_t thr = s_prefix, need_eq = s_remaining;  // take need_eq of the keys == thr
    const uint32_t n_eq = __ldcg(&ctl->hist[2][thr & 0x3FFu]);   // keys equal to thr, grid-wide
    const bool take_all_eq = n_eq == need_eq;

    // candidates: keys above the threshold (and the equal ones when exactly enough are equal)
    for (int i0 = 0; i0 < nv; i0 += kThreadsS) {
        const int i = i0 + tid;
        uint32_t key = 0u;
        bool take = false;
        if (i < nv) {
            key = fkey(sm.s.vals[i]);
            take = key > thr || (take_all_eq && key == thr);
        }
        const unsigned ball = __ballot_sync(0xffffffffu, take);
        if (ball) {
            uint32_t base = 0u;
            if (lane == 0) base = atomicAdd(&ctl->n_cand, (uint32_t)__popc(ball));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (take) {
                const uint32_t j = base + __popc(ball & ((1u << lane) - 1u));
                if (j < (uint32_t)kMaxK) ctl->cand[j] = ((unsigned long long)(~key) << 32) | (uint32_t)(b0 + i);
            }
        }
    }
    if (!take_all_eq) {
        // more keys equal the threshold than needed: the lowest token ids, ranked by the slices'
        // tie counts (a barrier), then by position within the slice (block scans in order)
        uint32_t my_eq = 0u;
        for (int i = tid; i < nv; i += kThreadsS) my_eq += fkey(sm.s.vals[i]) == thr;
        uint32_t blk_eq = 0u;
        block_scan<uint32_t>(my_eq, wsum_u, &blk_eq);
        if (tid == 0) ctl->ties[blockIdx.x] = blk_eq;
        if (!grid_sync(ctl, G, &s_ok)) return;
        uint32_t before = 0u;                                           // ties of lower slices
        for (uint32_t q = 0; q < blockIdx.x; ++q) before += __ldcg(&ctl->ties[q]);
        for (int i0 = 0; i0 < nv && before < need_eq; i0 += kThreadsS) {   // uniform condition
            const int i = i0 + tid;
            const uint32_t e = i < nv && fkey(sm.s.vals[i]) == thr;
            uint32_t tot = 0u;
            const uint32_t r = block_scan<uint32_t>(e, wsum_u, &tot) - e + before;
            if (e && r < need_eq) {
                const uint32_t j = atomicAdd(&ctl->n_cand, 1u);
                if (j < (uint32_t)kMaxK) ctl->cand[j] = ((unsigned long long)(~thr) << 32) | (uint32_t)(b0 + i);
            }
            before += tot;
        }
    }
    if (!grid_sync(ctl, G, &s_ok)) return;
    if (blockIdx.x != 0) return;

    // 3. bitonic sort in block 0, ascending on (~key, id) = value descending, id ascending
    const uint32_t n = min(__ldcg(&ctl->n_cand), (uint32_t)kMaxK);
    uint32_t P = 1u;
    while (P < n) P <<= 1;
    for (uint32_t i = tid; i < P; i += kThreadsS) sm.cand[i] = i < n ? __ldcg(&ctl->cand[i]) : ~0ull;
    __syncthreads();
    for (uint32_t size = 2; size <= P; size <<= 1) {
        for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (uint32_t i = tid; i < P; i += kThreadsS) {
                const uint32_t jx = i ^ stride;
                if (jx > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long x = sm.cand[i], y = sm.cand[jx];
                    if ((x > y) == up) { sm.cand[i] = y; sm.cand[jx] = x; }
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
    // kPer t .. kPer t + kPer - 1, their values recovered from the keys (bit for bit)
    auto val = [&](uint32_t i) {
        const uint32_t key = ~(uint32_t)(sm.cand[i] >> 32);
        return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
    };
    const float l0 = val(0);
    float lv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const uint32_t i = (uint32_t)(tid * kPer + j);
        lv[j] = i < n ? val(i) : -INFINITY;
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
    int token = (int)(uint32_t)sm.cand[0];
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
        token = (int)(uint32_t)sm.cand[f != 0xFFFFFFFFu ? f : m - 1];
    }
    if (tid == 0) { *a.out = token; *a.err = 0u; }
}

}  // namespace

int sample_max_k() { return kMaxK; }

size_t sample_state_bytes() { return sizeof(SampleCtl); }

bool launch_sample(const SampleArgs& a, void* state, int n_sm, cudaStream_t st) {
    if (a.V <= 0 || a.top_k < 1 || a.top_k > kMaxK || !state) return false;
    const int need = (a.V + kSliceMax - 1) / kSliceMax;              // blocks so a slice fits
    const int G = std::max(need, std::min(64, n_sm));
    if (G > kMaxBlocks || G > n_sm) return false;
    SampleParams p{a, static_cast<SampleCtl*>(state)};
    void* args[] = {&p};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(sample_kernel), dim3(G), dim3(kThreadsS),
                                       args, 0, st) == cudaSuccess;
}

}  // namespace llm
