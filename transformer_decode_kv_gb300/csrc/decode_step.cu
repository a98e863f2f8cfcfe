// One decode step of one token as a single persistent kernel (sm_103a): embedding, every layer's
// RMSNorm -> Q/K/V -> RoPE -> K/V append -> attention -> output projection + residual -> RMSNorm
// -> gate/up -> SwiGLU -> down + residual, then the final norm, the output matrix and the greedy
// pick ([P2] "llama.cpp Architecture", Example 4, the op chain of one decode step; [P1] Крок 13б
// for the layer scheme and Крок 14 for the greedy pick).
//
// Why one kernel: a one-token step reads every weight byte once and does almost no arithmetic, so
// its speed is the HBM stream. Separate kernels stall that stream at each of the ~160 op
// boundaries (ramp-down, launch, ramp-up). Here the stream never depends on activations: each
// block's producer warp walks the block's rows of every matrix of every layer in op order and
// copies them (cp.async.bulk, evict-first) into a ring of shared-memory stages, running ahead of
// the consumers by the ring's depth, across op and layer boundaries and through the attention.
// Only the eight consumer warps wait for data dependencies: a grid-wide phase counter per op
// (every block adds one when its share of the op is written; a block starts an op when all
// blocks have finished the op it reads). The launch is cooperative, so all blocks are resident
// and every wait ends; each wait is also bounded (2 s), after which the block sets the error word
// and a global abort flag that makes every other block stop waiting, and the producer waits for
// its own copies in flight before the block exits.
//
// Work split: each GEMV's rows (gate/up features for SwiGLU, row pairs for Q/K/V so a RoPE pair
// stays in one block) are split evenly over the grid. Consumers use the column-stationary
// mapping: warp w always reads the same 512-byte slices of every row, so its activations sit in
// registers for the whole op (normalised in the prologue when the op starts with RMSNorm), and
// per-row sums meet in shared memory. Attention work items (KV head, slice of the sequence's
// cell list) are spread over the blocks; the block that finishes a head's last item merges the
// partial softmax states (a self-resetting ticket). All activations written during the step are
// read through L2 (ld.global.cg / cp.async.cg), never from a possibly stale L1 line.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "decode_step.h"
#include "dev_common.cuh"

namespace llm {

namespace {

using namespace dev;

constexpr int kCW = 8;                        // consumer warps
constexpr int kThreads = (kCW + 1) * 32;      // + one producer warp
constexpr int kCT = kCW * 32;                 // consumer threads
constexpr uint32_t kSlice = 512;              // bytes of a row one warp reads per pass
constexpr int kMaxStages = 6;
constexpr uint32_t kStage = 28672;            // ring slot: whole rows, or half of a longer row
constexpr int kRpsD = (int)(kStage / 8192);               // rows of 4096 2-byte weights per slot
constexpr int kPartsF = (int)((28672 + kStage - 1) / kStage);  // slots per row of 14336
constexpr int kCH = 32;                       // cells staged per attention pass (one lane each)
constexpr int kG = 4;                         // query heads per KV head
constexpr size_t kSmemBudget = 112 * 1024;    // two blocks per SM

enum : int { OP_QKV = 0, OP_WO = 1, OP_GU = 2, OP_DOWN = 3, OP_LM = 4 };

__device__ __forceinline__ void csync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory");
}
__device__ __forceinline__ int vload(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void stamp(const StepArgs& a, int k, int end) {
    if (a.trace) a.trace[((size_t)blockIdx.x * a.n_trace + k) * 2 + end] = global_ns();
}
__device__ __forceinline__ void set_abort(const StepArgs& a) {
    atomicOr(a.err, ERR_TIMEOUT);
    *reinterpret_cast<volatile int32_t*>(a.abort_flag) = 1;
}

// Wait for an mbarrier phase. The fast path is one try_wait; the global abort flag is read only
// once a wait has lasted 20 us (another block gave up), and a wait of 2 s gives up and sets it.
__device__ bool step_wait(const StepArgs& a, uint64_t* bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        const uint64_t t = global_ns() - t0;
        if (t > 20000 && (it & 15) == 0 && vload(a.abort_flag)) return false;
        if (t > kWaitNs) { set_abort(a); return false; }
    }
}

// Rows of one GEMV that this block owns: 1 range, or 2 for SwiGLU (gate rows, then up rows).
struct OpRows {
    const uint8_t* W;
    int64_t row_bytes;
    int64_t row0[2], nrows[2];
    int nr;
    int64_t u0;          // first unit (row, row pair or feature)
    int nloc;            // rows of the first range
};

__device__ __forceinline__ OpRows op_rows(const StepArgs& a, int layer, int op) {
    const int64_t es = 2;                     // BF16 / F16 weights
    OpRows r{};
    int64_t units, gran = 1, K;
    const StepLayer* L = layer >= 0 ? a.layers + layer : nullptr;
    switch (op) {
        case OP_QKV: r.W = static_cast<const uint8_t*>(L->qkv); K = a.d;
                     units = (int64_t)(a.H + 2 * a.Hkv) * a.hd / 2; gran = 2; break;
        case OP_WO: r.W = static_cast<const uint8_t*>(L->wo); K = (int64_t)a.H * a.hd; units = a.d; break;
        case OP_GU: r.W = static_cast<const uint8_t*>(L->gu); K = a.d; units = a.F; break;
        case OP_DOWN: r.W = static_cast<const uint8_t*>(L->down); K = a.F; units = a.d; break;
        default: r.W = static_cast<const uint8_t*>(a.out); K = a.d; units = a.V; break;
    }
    r.row_bytes = K * es;
    const int64_t u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
    r.u0 = u0;
    r.row0[0] = u0 * gran;
    r.nrows[0] = (u1 - u0) * gran;
    r.nloc = (int)r.nrows[0];
    r.nr = 1;
    if (op == OP_GU) { r.row0[1] = a.F + u0; r.nrows[1] = u1 - u0; r.nr = 2; }
    return r;
}

// Walks the weight chunks this block streams in one step: every op (4 per layer, then the output
// matrix), each of its row ranges, in chunks of one ring slot: as many whole rows as fit, or one
// half of a row longer than a slot.
struct ChunkCursor {
    int k = 0, g = 0, n_ops = 0, parts = 1, pi = 0;
    int64_t i = 0, rps = 0;
    OpRows r{};
    bool done = false;

    __device__ void start(const StepArgs& a) {
        n_ops = a.n_layer * 4 + (a.do_logits ? 1 : 0);
        k = -1;
        next_op(a);
    }
    __device__ void next_op(const StepArgs& a) {
        for (++k; k < n_ops; ++k) {
            const int layer = k < a.n_layer * 4 ? k / 4 : -1;
            r = op_rows(a, layer, layer >= 0 ? k % 4 : OP_LM);
            parts = r.row_bytes <= (int64_t)kStage ? 1 : 2;
            rps = parts == 1 ? kStage / r.row_bytes : 1;
            for (g = 0; g < r.nr && r.nrows[g] == 0; ++g) {}
            i = 0;
            pi = 0;
            if (g < r.nr) return;
        }
        done = true;
    }
    __device__ void next(const StepArgs& a) {
        if (++pi < parts) return;
        pi = 0;
        i += rps;
        if (i < r.nrows[g]) return;
        i = 0;
        for (++g; g < r.nr && r.nrows[g] == 0; ++g) {}
        if (g >= r.nr) next_op(a);
    }
    __device__ const uint8_t* src() const {
        return r.W + (r.row0[g] + i) * r.row_bytes + pi * (r.row_bytes / parts);
    }
    __device__ uint32_t bytes() const {
        if (parts > 1) return (uint32_t)(r.row_bytes / parts);
        return (uint32_t)((r.nrows[g] - i < rps ? r.nrows[g] - i : rps) * r.row_bytes);
    }
};

// ---- producer: every weight row this block owns, in op order, into the stage ring. It also
// keeps up to kPrefetchBytes ahead of its copies requested into L2 (cp.async.bulk.prefetch,
// marked evict-last until the copy, which reads them evict-first), so the HBM stream goes on
// while the ring is full and the consumers wait at a phase boundary. The distance is bounded:
// the grid's prefetched bytes (304 blocks x 128 KB = 39 MB) must stay well inside L2 or they
// evict each other before use (measured: 64-128 KB per block best, 192 KB already worse).
constexpr uint32_t kPrefetchBytes = 128 * 1024;

__device__ void produce(const StepArgs& a, uint8_t* ring, uint64_t* full, uint64_t* empty) {
    uint64_t policy, keep;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    const int NS = a.n_stages;
    const uint32_t SB = kStage;
    ChunkCursor ld, pf;
    ld.start(a);
    pf.start(a);
    uint32_t p = 0;                        // chunks copied
    uint64_t ld_bytes = 0, pf_bytes = 0;   // bytes copied / prefetched
    int op_seen = -1;
    while (!ld.done) {
        for (; !pf.done && pf_bytes < ld_bytes + kPrefetchBytes; pf.next(a)) {
            asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(pf.src()),
                         "r"(pf.bytes()), "l"(keep) : "memory");
            pf_bytes += pf.bytes();
        }
        const int s = (int)(p % NS);
        if (p >= (uint32_t)NS && !step_wait(a, &empty[s], ((p / NS) & 1u) ^ 1u)) break;
        const uint32_t nb = ld.bytes();
        mbar_expect_tx(&full[s], nb);
        bulk_g2s(ring + (size_t)s * SB, ld.src(), nb, &full[s], policy);
        if (ld.k != op_seen) {
            if (op_seen >= 0) stamp(a, 2 + 5 * a.n_layer + op_seen, 1);
            op_seen = ld.k;
            stamp(a, 2 + 5 * a.n_layer + op_seen, 0);
        }
        ++p;
        ld_bytes += nb;
        ld.next(a);
    }
    if (op_seen >= 0) stamp(a, 2 + 5 * a.n_layer + op_seen, 1);
    // the block may exit only after every copy it issued has landed
    const uint32_t q0 = p > (uint32_t)NS ? p - NS : 0;
    for (uint32_t j = q0; j < p; ++j) mbar_wait(&full[j % NS], (j / NS) & 1u);
}

// ---- grid-wide phase counters (consumer thread 0 signals / waits; csync spreads the result)
__device__ __forceinline__ void signal_phase(const StepArgs& a, int ctr) {
    csync();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(a.counters + ctr, 1u);
    }
}
__device__ bool wait_phase(const StepArgs& a, int ctr, int* flag) {
    if (threadIdx.x == 0) {
        const uint32_t target = (a.gen + 1u) * gridDim.x;
        bool ok = true;
        uint64_t t0 = 0;
        for (uint32_t it = 0; (int32_t)(ld_acquire(a.counters + ctr) - target) < 0; ++it) {
            if ((it & 15) == 15 && vload(a.abort_flag)) { ok = false; break; }
            const uint64_t t = global_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > kWaitNs) { set_abort(a); ok = false; break; }
        }
        __threadfence();
        *flag = ok ? 1 : 0;
    }
    csync();
    return *reinterpret_cast<volatile int*>(flag) != 0;
}

template <int WT> __device__ __forceinline__ void unpack8(const uint4 v, float* w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (WT == W_BF16) {
            w[2 * i] = __uint_as_float(u[i] << 16);
            w[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        } else {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
            w[2 * i] = f.x;
            w[2 * i + 1] = f.y;
        }
    }
}

struct Smem {
    uint8_t* ring;
    uint64_t* full;
    uint64_t* empty;
    float* acc;          // [rows_cap]
    float* red;          // [kCW]
    int* flag;
    uint8_t* kb;         // [kCH][hd * kv size + 16]
    uint8_t* vb;
    float* qs;           // [kG][hd]
    int* ccell;          // [kCH]
};

// One GEMV of this block's rows: x (columns owned by the warp) in registers, rows from the ring.
// OP: the op; SPW: 512-byte slices per warp and row (row bytes / 512 / 8); RPS: rows per slot;
// PARTS: slots per row (2: half rows, each read by the four warps owning its columns).
template <int WT, int SPW, int RPS, int PARTS, int OP>
__device__ bool gemv_op(const StepArgs& a, const Smem& sm, int layer, uint32_t& p) {
    constexpr int VN = 8;                                 // 16 bytes of 2-byte weights
    const OpRows r = op_rows(a, layer, OP);
    const StepLayer* L = layer >= 0 ? a.layers + layer : nullptr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, ctid = threadIdx.x;
    const int NS = a.n_stages;
    const uint32_t SB = kStage;
    const int64_t K = r.row_bytes / 2;
    const float* xsrc = OP == OP_WO ? a.o : OP == OP_DOWN ? a.u : a.x;
    const float* gain = OP == OP_QKV ? L->attn_norm : OP == OP_GU ? L->ffn_norm : OP == OP_LM ? a.out_norm : nullptr;

    float xr[SPW][VN];
    float ss = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < SPW; ++k2) {
        const int col = (warp * SPW + k2) * (int)(kSlice / 2) + lane * VN;
#pragma unroll
        for (int e = 0; e < VN; e += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(xsrc + col + e));
            xr[k2][e] = v.x; xr[k2][e + 1] = v.y; xr[k2][e + 2] = v.z; xr[k2][e + 3] = v.w;
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
    }
    if (gain) {
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) sm.red[warp] = ss;
    }
    for (int i = ctid; i < a.rows_cap; i += kCT) sm.acc[i] = 0.f;
    csync();
    if (gain) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kCW; ++w) s += sm.red[w];
        const float sc = 1.0f / sqrtf(s / (float)K + a.eps);
#pragma unroll
        for (int k2 = 0; k2 < SPW; ++k2) {
            const int col = (warp * SPW + k2) * (int)(kSlice / 2) + lane * VN;
#pragma unroll
            for (int e = 0; e < VN; e += 4) {
                const float4 g = *reinterpret_cast<const float4*>(gain + col + e);
                xr[k2][e] *= sc * g.x; xr[k2][e + 1] *= sc * g.y;
                xr[k2][e + 2] *= sc * g.z; xr[k2][e + 3] *= sc * g.w;
            }
        }
    }

    constexpr int WPP = kCW / PARTS;                      // warps per part of a row
    for (int g = 0; g < r.nr; ++g) {
        const int local0 = g == 0 ? 0 : r.nloc;
        for (int64_t i0 = 0; i0 < r.nrows[g]; i0 += RPS) {
            const int n = (int)(r.nrows[g] - i0 < RPS ? r.nrows[g] - i0 : RPS);
#pragma unroll
            for (int pi = 0; pi < PARTS; ++pi, ++p) {
                const int s = (int)(p % NS);
                if (!step_wait(a, &sm.full[s], (p / NS) & 1u)) return false;
                if (warp / WPP == pi) {
                    const uint8_t* st0 = sm.ring + (size_t)s * SB + ((warp % WPP) * SPW) * kSlice + lane * 16;
                    const int64_t rstride = PARTS == 1 ? r.row_bytes : 0;
                    // all rows of the slot at once: independent accumulators (two per row), the
                    // reductions interleaved, then lane i adds row i's sum to the shared total
                    float pa[RPS], pb[RPS];
#pragma unroll
                    for (int i = 0; i < RPS; ++i) {
                        pa[i] = 0.f;
                        pb[i] = 0.f;
                        if (i < n) {
#pragma unroll
                            for (int k2 = 0; k2 < SPW; ++k2) {
                                const uint4 wv = *reinterpret_cast<const uint4*>(st0 + (size_t)i * rstride + k2 * kSlice);
                                float w[VN];
                                unpack8<WT>(wv, w);
#pragma unroll
                                for (int e = 0; e < VN; e += 2) {
                                    pa[i] = fmaf(w[e], xr[k2][e], pa[i]);
                                    pb[i] = fmaf(w[e + 1], xr[k2][e + 1], pb[i]);
                                }
                            }
                        }
                        pa[i] += pb[i];
                    }
                    if constexpr (RPS == 4) {
                        // transposed butterfly: 6 shuffles sum 4 rows over the warp; lanes
                        // 8r .. 8r+7 end with row r's total
                        const bool hi16 = (lane & 16) != 0, hi8 = (lane & 8) != 0;
                        const float s0 = hi16 ? pa[0] : pa[2], s1 = hi16 ? pa[1] : pa[3];
                        const float k0 = hi16 ? pa[2] : pa[0], k1 = hi16 ? pa[3] : pa[1];
                        const float a0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 16);
                        const float a1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 16);
                        float v = (hi8 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, hi8 ? a0 : a1, 8);
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        const int row = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
                        if ((lane & 7) == 0 && row < n) atomicAdd(&sm.acc[local0 + (int)i0 + row], v);
                    } else {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                            for (int i = 0; i < RPS; ++i) pa[i] += __shfl_xor_sync(0xffffffffu, pa[i], o);
#pragma unroll
                        for (int i = 0; i < RPS; ++i)
                            if (lane == i && i < n) atomicAdd(&sm.acc[local0 + (int)i0 + i], pa[i]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[s]);
            }
        }
    }
    csync();

    // ---- epilogue of the op
    const int nloc = r.nloc;
    if (OP == OP_WO || OP == OP_DOWN) {
        for (int i = ctid; i < nloc; i += kCT) {
            float* dst = a.x + r.u0 + i;
            *dst = __ldcg(dst) + sm.acc[i];
        }
    } else if (OP == OP_GU) {
        for (int i = ctid; i < nloc; i += kCT) {
            const float gt = sm.acc[i], up = sm.acc[nloc + i];
            a.u[r.u0 + i] = gt / (1.0f + expf(-gt)) * up;
        }
    } else if (OP == OP_LM) {
        unsigned long long best = 0;
        for (int i = ctid; i < nloc; i += kCT) {
            const float v = sm.acc[i];
            a.logits[r.u0 + i] = v;
            if (v == v) {
                const unsigned long long pk = pack_argmax(v, (int)(r.u0 + i));
                best = pk > best ? pk : best;
            }
        }
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
            best = ob > best ? ob : best;
        }
        if (lane == 0 && best) atomicMax(a.amax, best);
    } else {  // OP_QKV: RoPE on Q and K rows, K/V rows to their cache cell, Q to a.q
        const int hd = a.hd;
        const int64_t row0 = r.row0[0];
        const int32_t cell = a.slot[0];
        for (int pl = ctid; pl < nloc / 2; pl += kCT) {
            const int64_t row = row0 + 2 * pl;
            const int head = (int)(row / hd), dd = (int)(row % hd);
            float y0 = sm.acc[2 * pl], y1 = sm.acc[2 * pl + 1];
            if (head < a.H + a.Hkv) {
                const float2 e = __ldcg(a.cs + dd / 2);
                const float r0 = y0 * e.x - y1 * e.y, r1 = y0 * e.y + y1 * e.x;
                y0 = r0; y1 = r1;
            }
            if (head < a.H) {
                a.q[row] = y0;
                a.q[row + 1] = y1;
                continue;
            }
            if (cell < 0 || cell >= a.n_ctx) { atomicOr(a.err, ERR_SLOT_RANGE); continue; }
            const bool is_k = head < a.H + a.Hkv;
            const int g = is_k ? head - a.H : head - a.H - a.Hkv;
            const int64_t ci = ((int64_t)g * a.n_ctx + cell) * hd + dd;
            void* cache = is_k ? L->kc : L->vc;
            if (a.kv_type == W_F32) {
                static_cast<float*>(cache)[ci] = y0;
                static_cast<float*>(cache)[ci + 1] = y1;
            } else {
                static_cast<__half2*>(cache)[ci / 2] = __floats2half2_rn(y0, y1);
            }
        }
    }
    return true;
}

template <typename KT> __device__ __forceinline__ float kvf(KT v);
template <> __device__ __forceinline__ float kvf<float>(float v) { return v; }
template <> __device__ __forceinline__ float kvf<__half>(__half v) { return __half2float(v); }

// Attention of the token's query heads over its visible cells (split-K work items over the
// sequence's cell list; [P2] Example 4 FLASH_ATTN_EXT, Example 11 for the unfused meaning).
// Work item it = (item wi, KV head) goes to block it mod grid. Cells are staged kCH at a time
// (cp.async through L2); warps 0..3 hold query heads 0..3 of the KV head (one cell per lane for the
// scores, hd/32 output dimensions per lane for V). The rows of cells written by earlier steps
// cannot change during this step, so a block stages its first pass before the Q/K/V phase ends
// (attn_prestage); only the current token's cell and Q are read after it.
template <int HD, typename KT>
struct AttnGeo {
    static constexpr int RB = HD * (int)sizeof(KT), RS = RB + 16, VPR = RB / 16, DPL = HD / 32;
};

// Cells of pass [cb, cb + kCH) of item (wi, kvh): ccell[i] = cache cell or -1 (outside the item
// or not visible); returns through smem. Issues the cp.async copies of every cell that is not the
// current token's own (fresh = false) or only of that one (fresh = true).
template <int HD, typename KT>
__device__ void attn_stage(const StepArgs& a, const Smem& sm, int layer, int wi, int kvh, int cb,
                           bool fresh, bool set_cells) {
    using Gm = AttnGeo<HD, KT>;
    const StepLayer* L = a.layers + layer;
    const int ctid = threadIdx.x;
    if (set_cells) {
        if (ctid < kCH) {
            const int4 wd = a.wi_desc[wi];
            const int base = a.tile_desc[2 * wd.x + 1].y;
            const int ci = cb + ctid;
            int cell = -1;
            if (ci < wd.z) {
                const int cc = a.list_cells[base + ci];
                if (cc >= 0 && cc < a.n_ctx && a.list_pos[base + ci] <= a.pos[0]) cell = cc;
            }
            sm.ccell[ctid] = cell;
        }
        csync();
    }
    const int cur = a.slot[0];
    const uint8_t* K = static_cast<const uint8_t*>(L->kc) + (int64_t)kvh * a.n_ctx * Gm::RB;
    const uint8_t* V = static_cast<const uint8_t*>(L->vc) + (int64_t)kvh * a.n_ctx * Gm::RB;
    for (int v = ctid; v < kCH * Gm::VPR; v += kCT) {
        const int cidx = v / Gm::VPR, j = v % Gm::VPR;
        const int cell = sm.ccell[cidx];
        if (cell < 0 || (cell == cur) != fresh) continue;
        const size_t src = (size_t)cell * Gm::RB + j * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sm.kb + cidx * Gm::RS + j * 16)),
                     "l"(K + src) : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sm.vb + cidx * Gm::RS + j * 16)),
                     "l"(V + src) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Before the Q/K/V phase completes: the first pass of this block's first item.
template <int HD, typename KT>
__device__ void attn_prestage(const StepArgs& a, const Smem& sm, int layer) {
    const int n_work = a.hdr[0];
    const int it = blockIdx.x;
    if (it >= n_work * a.Hkv) return;
    const int wi = it / a.Hkv, kvh = it % a.Hkv;
    attn_stage<HD, KT>(a, sm, layer, wi, kvh, a.wi_desc[wi].y, false, true);
}

template <int HD, typename KT>
__device__ bool attention(const StepArgs& a, const Smem& sm, int layer) {
    using Gm = AttnGeo<HD, KT>;
    constexpr int RS = Gm::RS, VPR = Gm::VPR, DPL = Gm::DPL;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, ctid = threadIdx.x;
    const int n_work = a.hdr[0];
    const int Hkv = a.Hkv;
    bool first = true;
    for (int it = blockIdx.x; it < n_work * Hkv; it += gridDim.x, first = false) {
        const int wi = it / Hkv, kvh = it % Hkv;
        const int4 wd = a.wi_desc[wi];
        const int c0 = wd.y, c1 = wd.z;
        for (int i = ctid; i < kG * HD; i += kCT)
            sm.qs[i] = __ldcg(a.q + (kvh * kG + i / HD) * HD + i % HD) * scale_log2;
        float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] = 0.f;
        for (int cb = c0; cb < c1; cb += kCH) {
            const bool pre = first && cb == c0;          // old cells already in flight
            if (!pre) attn_stage<HD, KT>(a, sm, layer, wi, kvh, cb, false, true);
            attn_stage<HD, KT>(a, sm, layer, wi, kvh, cb, true, false);
            asm volatile("cp.async.wait_all;" ::: "memory");
            csync();
            if (warp < kG) {
                // scores: kCH cells, 32 / kCH lanes per cell each taking a share of the dimensions
                constexpr int LPC = 32 / kCH;
                const int cidx = lane % kCH, part = lane / kCH;
                const float* q = sm.qs + warp * HD;
                const bool valid = sm.ccell[cidx] >= 0;
                float sp = 0.f;
                if (valid) {
                    const uint8_t* kr = sm.kb + cidx * RS;
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int jj = 0; jj < VPR / LPC; ++jj) {
                        const int j = part * (VPR / LPC) + jj;
                        const uint4 kv = *reinterpret_cast<const uint4*>(kr + j * 16);
                        const KT* ke = reinterpret_cast<const KT*>(&kv);
                        constexpr int EPV = 16 / (int)sizeof(KT);
#pragma unroll
                        for (int e = 0; e < EPV; e += 2) {
                            a0 = fmaf(q[j * EPV + e], kvf<KT>(ke[e]), a0);
                            a1 = fmaf(q[j * EPV + e + 1], kvf<KT>(ke[e + 1]), a1);
                        }
                    }
                    sp = a0 + a1;
                }
#pragma unroll
                for (int off = kCH; off < 32; off <<= 1) sp += __shfl_xor_sync(0xffffffffu, sp, off);
                const float s = valid ? sp : -INFINITY;
                float mx = s;
                for (int off = kCH / 2; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_new = fmaxf(m, mx);
                float pr = 0.f, corr = 1.f;
                if (m_new != -INFINITY) {
                    corr = exp2f(m - m_new);
                    pr = exp2f(s - m_new);
                }
                float ps = pr;
                for (int off = kCH / 2; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                l = l * corr + ps;
                m = m_new;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[e] *= corr;
#pragma unroll 4
                for (int cc = 0; cc < kCH; ++cc) {
                    const float pc = __shfl_sync(0xffffffffu, pr, cc);
                    if (pc == 0.f) continue;
                    const KT* vr = reinterpret_cast<const KT*>(sm.vb + cc * RS) + lane * DPL;
#pragma unroll
                    for (int e = 0; e < DPL; ++e) o[e] = fmaf(pc, kvf<KT>(vr[e]), o[e]);
                }
            }
            csync();
        }
        if (n_work == 1) {
            if (warp < kG) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) a.o[(kvh * kG + warp) * HD + lane * DPL + e] = o[e] * inv;
            }
            continue;
        }
        if (warp < kG) {
            const int64_t row = ((int64_t)wi * Hkv + kvh) * kG + warp;
            if (lane == 0) { a.part_m[row] = m; a.part_l[row] = l; }
#pragma unroll
            for (int e = 0; e < DPL; ++e) a.part_o[row * HD + lane * DPL + e] = o[e];
        }
        __threadfence();
        csync();
        if (ctid == 0) {
            const int done = atomicAdd(a.tickets + kvh, 1) + 1;
            const bool last = done == n_work;
            if (last) a.tickets[kvh] = 0;
            *sm.flag = last ? 1 : 0;
        }
        csync();
        if (!*reinterpret_cast<volatile int*>(sm.flag)) continue;
        __threadfence();
        // merge the items' partial states: per query head the weights 2^(m_w - M) / L into
        // shared memory, then every thread sums two output dimensions over the items
        float* wgt = reinterpret_cast<float*>(sm.kb);          // [kG][n_work], staging is free now
        if (warp < kG) {
            float M = -INFINITY;
            for (int w = lane; w < n_work; w += 32)
                M = fmaxf(M, __ldcg(a.part_m + ((int64_t)w * Hkv + kvh) * kG + warp));
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            float Ls = 0.f;
            for (int w = lane; w < n_work; w += 32) {
                const int64_t row = ((int64_t)w * Hkv + kvh) * kG + warp;
                const float mw = __ldcg(a.part_m + row);
                const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - M);
                Ls += f * __ldcg(a.part_l + row);
                wgt[warp * n_work + w] = f;
            }
            for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
            __syncwarp();
            for (int w = lane; w < n_work; w += 32) wgt[warp * n_work + w] *= inv;
        }
        csync();
        for (int idx = ctid; idx < kG * HD; idx += kCT) {
            const int g = idx / HD, dd = idx % HD;
            float acc0 = 0.f, acc1 = 0.f;
            int w = 0;
            for (; w + 1 < n_work; w += 2) {
                const float p0 = __ldcg(a.part_o + (((int64_t)w * Hkv + kvh) * kG + g) * HD + dd);
                const float p1 = __ldcg(a.part_o + (((int64_t)(w + 1) * Hkv + kvh) * kG + g) * HD + dd);
                acc0 = fmaf(wgt[g * n_work + w], p0, acc0);
                acc1 = fmaf(wgt[g * n_work + w + 1], p1, acc1);
            }
            if (w < n_work) acc0 = fmaf(wgt[g * n_work + w], __ldcg(a.part_o + (((int64_t)w * Hkv + kvh) * kG + g) * HD + dd), acc0);
            a.o[(kvh * kG + g) * HD + dd] = acc0 + acc1;
        }
        csync();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    return true;
}

// Counter index of phase `ph` (0 QKV, 1 attention, 2 WO, 3 gate/up, 4 down) of layer l; 0 = embed.
__device__ __forceinline__ int ctr(int l, int ph) { return 1 + 5 * l + ph; }

template <int WT, int HD, typename KT, int SPW_D, int SPW_F, int RPS_D, int PARTS_F>
__global__ void __launch_bounds__(kThreads, 2) decode_step_kernel(const StepArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int NS = a.n_stages;
    const uint32_t SB = kStage;
    Smem sm;
    sm.ring = smem;
    uint8_t* q = smem + (size_t)NS * SB;
    sm.kb = q; q += kCH * (HD * sizeof(KT) + 16);
    sm.vb = q; q += kCH * (HD * sizeof(KT) + 16);
    sm.qs = reinterpret_cast<float*>(q); q += kG * HD * 4;
    sm.acc = reinterpret_cast<float*>(q); q += ((size_t)a.rows_cap * 4 + 15) / 16 * 16;
    sm.red = reinterpret_cast<float*>(q); q += 64;
    sm.ccell = reinterpret_cast<int*>(q); q += kCH * 4;
    sm.flag = reinterpret_cast<int*>(q); q += 16;
    sm.full = reinterpret_cast<uint64_t*>(q); q += kMaxStages * 8;
    sm.empty = reinterpret_cast<uint64_t*>(q);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kCW) {
        if (lane == 0) produce(a, sm.ring, sm.full, sm.empty);
        return;
    }

    // ---- embedding row of the token, RoPE table of its position, greedy-pick reset
    {
        if (threadIdx.x == 0) stamp(a, 0, 0);
        const int32_t id = a.tok[0];
        const bool ok = id >= 0 && id < a.embd.rows;
        const int64_t j0 = (int64_t)a.d * blockIdx.x / gridDim.x, j1 = (int64_t)a.d * (blockIdx.x + 1) / gridDim.x;
        for (int64_t j = j0 + threadIdx.x; j < j1; j += kCT) a.x[j] = ok ? load_elem(a.embd, id, j) : 0.f;
        if (blockIdx.x == 0) {
            for (int i = threadIdx.x; i < a.hd / 2; i += kCT) a.cs[i] = rope_cos_sin(a.pos[0], a.theta[i]);
            if (threadIdx.x == 0) {
                if (a.do_logits) *a.amax = 0ull;
                if (!ok) atomicOr(a.err, ERR_TOKEN_RANGE);
            }
        }
        if (threadIdx.x == 0) stamp(a, 0, 1);
        signal_phase(a, 0);
    }
    uint32_t p = 0;
    const bool t0 = threadIdx.x == 0;
    for (int l = 0; l < a.n_layer; ++l) {
        if (!wait_phase(a, l == 0 ? 0 : ctr(l - 1, 4), sm.flag)) return;
        if (t0) stamp(a, ctr(l, 0), 0);
        if (!gemv_op<WT, SPW_D, RPS_D, 1, OP_QKV>(a, sm, l, p)) return;
        if (t0) stamp(a, ctr(l, 0), 1);
        signal_phase(a, ctr(l, 0));
        attn_prestage<HD, KT>(a, sm, l);
        if (!wait_phase(a, ctr(l, 0), sm.flag)) {
            asm volatile("cp.async.wait_all;" ::: "memory");
            return;
        }
        if (t0) stamp(a, ctr(l, 1), 0);
        attention<HD, KT>(a, sm, l);
        if (t0) stamp(a, ctr(l, 1), 1);
        signal_phase(a, ctr(l, 1));
        if (!wait_phase(a, ctr(l, 1), sm.flag)) return;
        if (t0) stamp(a, ctr(l, 2), 0);
        if (!gemv_op<WT, SPW_D, RPS_D, 1, OP_WO>(a, sm, l, p)) return;
        if (t0) stamp(a, ctr(l, 2), 1);
        signal_phase(a, ctr(l, 2));
        if (!wait_phase(a, ctr(l, 2), sm.flag)) return;
        if (t0) stamp(a, ctr(l, 3), 0);
        if (!gemv_op<WT, SPW_D, RPS_D, 1, OP_GU>(a, sm, l, p)) return;
        if (t0) stamp(a, ctr(l, 3), 1);
        signal_phase(a, ctr(l, 3));
        if (!wait_phase(a, ctr(l, 3), sm.flag)) return;
        if (t0) stamp(a, ctr(l, 4), 0);
        if (!gemv_op<WT, SPW_F, 1, PARTS_F, OP_DOWN>(a, sm, l, p)) return;
        if (t0) stamp(a, ctr(l, 4), 1);
        signal_phase(a, ctr(l, 4));
    }
    if (a.do_logits) {
        if (!wait_phase(a, ctr(a.n_layer - 1, 4), sm.flag)) return;
        if (t0) stamp(a, 1 + 5 * a.n_layer, 0);
        gemv_op<WT, SPW_D, RPS_D, 1, OP_LM>(a, sm, -1, p);
        if (t0) stamp(a, 1 + 5 * a.n_layer, 1);
    }
}

// slices per warp of a row of n 2-byte elements, 0 if the column-stationary mapping does not fit
int spw_of(int64_t n) {
    const int64_t slices = n * 2 / kSlice;
    if (n * 2 % kSlice != 0 || slices % kCW != 0) return 0;
    const int64_t s = slices / kCW;
    return s == 2 || s == 7 ? (int)s : 0;
}

struct Plan {
    size_t smem = 0;
    int stages = 0, stage_bytes = 0, rows_cap = 0, grid = 0;
};

size_t fixed_smem(int hd, int kv_es, int rows_cap) {
    return 2 * (size_t)kCH * (hd * kv_es + 16) + (size_t)kG * hd * 4 + ((size_t)rows_cap * 4 + 15) / 16 * 16 + 64 +
           kCH * 4 + 16 + 2 * kMaxStages * 8;
}

bool make_plan(int32_t d, int32_t H, int32_t Hkv, int32_t hd, int32_t F, int32_t V, int32_t kv_type,
               int n_sm, Plan* pl) {
    pl->grid = 2 * n_sm;
    auto cap = [&](int64_t units, int64_t gran) { return (int)((units + pl->grid - 1) / pl->grid * gran); };
    pl->rows_cap = std::max({cap((int64_t)(H + 2 * Hkv) * hd / 2, 2), cap(d, 1), 2 * cap(F, 1), cap(V, 1)});
    pl->stage_bytes = (int)kStage;
    const size_t fixed = fixed_smem(hd, kv_type == W_F32 ? 4 : 2, pl->rows_cap);
    if (fixed + 2 * (size_t)pl->stage_bytes > kSmemBudget) return false;
    pl->stages = (int)std::min<size_t>(kMaxStages, (kSmemBudget - fixed) / pl->stage_bytes);
    pl->smem = fixed + (size_t)pl->stages * pl->stage_bytes;
    return true;
}

template <int WT, int HD, typename KT>
const void* kernel_for(int spw_d, int spw_f) {
    // d = 4096, n_ff = 14336 (2-byte weights): a slot holds kRpsD rows of length d and a row of
    // length n_ff in kPartsF slots
    if (spw_d == 2 && spw_f == 7) return (const void*)decode_step_kernel<WT, HD, KT, 2, 7, kRpsD, kPartsF>;
    return nullptr;
}

const void* pick_kernel(int32_t wt, int32_t hd, int32_t kv_type, int spw_d, int spw_f) {
    if (wt == W_BF16) {
        if (hd == 128) return kv_type == W_F32 ? kernel_for<W_BF16, 128, float>(spw_d, spw_f)
                                              : kernel_for<W_BF16, 128, __half>(spw_d, spw_f);
        if (hd == 64) return kv_type == W_F32 ? kernel_for<W_BF16, 64, float>(spw_d, spw_f)
                                             : kernel_for<W_BF16, 64, __half>(spw_d, spw_f);
    } else if (wt == W_F16) {
        if (hd == 128) return kv_type == W_F32 ? kernel_for<W_F16, 128, float>(spw_d, spw_f)
                                              : kernel_for<W_F16, 128, __half>(spw_d, spw_f);
        if (hd == 64) return kv_type == W_F32 ? kernel_for<W_F16, 64, float>(spw_d, spw_f)
                                             : kernel_for<W_F16, 64, __half>(spw_d, spw_f);
    }
    return nullptr;
}

}  // namespace

bool decode_step_ok(int32_t wt, int32_t d, int32_t H, int32_t Hkv, int32_t hd, int32_t F, int32_t V,
                    int32_t kv_type, int n_sm) {
    if ((wt != W_BF16 && wt != W_F16) || H != kG * Hkv || (int64_t)H * hd != d || V <= 0) return false;
    if (kv_type != W_F32 && kv_type != W_F16) return false;
    const void* k = pick_kernel(wt, hd, kv_type, spw_of(d), spw_of(F));
    if (!k) return false;
    // the instantiated slot geometry: two rows of length d per slot, rows of length n_ff in halves
    if (kStage / ((uint32_t)d * 2) != (uint32_t)kRpsD || ((uint32_t)F * 2 + kStage - 1) / kStage != (uint32_t)kPartsF ||
        kPartsF > 2 || (F * 2 / kPartsF) % 16 != 0)
        return false;
    Plan pl;
    if (!make_plan(d, H, Hkv, hd, F, V, kv_type, n_sm, &pl)) return false;
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return false;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) != cudaSuccess)
        return false;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, pl.smem) != cudaSuccess)
        return false;
    return per_sm >= 2;
}

int32_t decode_step_cells() { return kCH; }

bool launch_decode_step(int32_t wt, StepArgs a, int n_sm, cudaStream_t st) {
    const void* k = pick_kernel(wt, a.hd, a.kv_type, spw_of(a.d), spw_of(a.F));
    Plan pl;
    if (!k || !make_plan(a.d, a.H, a.Hkv, a.hd, a.F, a.V, a.kv_type, n_sm, &pl)) return false;
    a.n_stages = pl.stages;
    a.stage_bytes = pl.stage_bytes;
    a.rows_cap = pl.rows_cap;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) != cudaSuccess)
        return false;
    void* args[] = {&a};
    return cudaLaunchCooperativeKernel(k, dim3(pl.grid), dim3(kThreads), args, pl.smem, st) == cudaSuccess;
}

}  // namespace llm
