// Tensor-core GEMM for prefill ubatches on sm_103a: tcgen05.mma (BF16 x BF16 -> F32 in TMEM),
// operands staged in shared memory by TMA (cp.async.bulk.tensor, 128-byte swizzle), an mbarrier
// ring of pipeline stages, and fused epilogues read back with tcgen05.ld.
//
// Y[t][m] (op)= sum_k W[m][k] X[t][k] ([P2] "llama.cpp Architecture", Example 4: MUL_MAT of a
// {K, M} weight by the ubatch's activations; ADD for the residual; SWIGLU(ffn_gate, ffn_up)).
//
// The MMA's A operand is a 128-row tile of the weight matrix and its B operand a BN-token tile
// of the activations, both K-major; the accumulator D[128 weight rows][BN tokens] lives in
// TMEM with one weight row per lane, so the epilogue's warp-wide stores write 32 consecutive
// output features of one token (coalesced). SwiGLU: the A tile holds 64 gate rows then the 64
// matching up rows; warps 2-3 pass their up values to warps 0-1 through shared memory.
//
// Roles (128 threads): thread 0 issues TMA loads, thread 32 issues MMAs, all four warps run the
// epilogue. Every mbarrier wait is bounded by a wall-clock limit; a timeout sets ERR_TIMEOUT in
// the error word, skips the remaining work, drains the copies it issued and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>

#include "gemm_tc.h"
#include "kernels.h"

namespace llm {

namespace {

constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBK = 64;           // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr uint64_t kWaitNs = 2000000000ull;    // 2 s bound on any wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete; false after the time limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try(bar, parity))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Request a tile of the map into L2 (no shared memory, no completion): the weight tiles a few
// k-steps ahead, so the copies that follow hit L2 instead of waiting on HBM.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile with the 128-byte swizzle: 8-row groups of
// 128-byte rows, 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);      // start address
    d |= (uint64_t)1 << 16;                         // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset
    d |= (uint64_t)1 << 46;                         // descriptor version
    d |= (uint64_t)2 << 61;                         // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with BF16 A/B, F32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}
// the same with f16 A and B (kind::f16 takes one type for both operands)
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// warp-wide TMEM loads (the warp is reconverged first: every lane must take part)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// silu(g) * u with the fast exponential and divide (a few ulp; the result is then rounded to f16)
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// TMA tile store / reduce-add of a shared-memory box into the map's tensor (bulk-group completion)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// SPLIT: the activations come as two bf16 terms (hi + lo, about 16 significant bits); both are
// multiplied into the same accumulator, so the product keeps float32-like activation precision.
template <int BN, bool SPLIT = false>
struct TcCfg {
    static constexpr uint32_t kA = kBM * kBK * 2;          // 16 KB
    static constexpr uint32_t kB = BN * kBK * 2;
    static constexpr uint32_t kStageB = SPLIT ? 2 * kB : kB;
    static constexpr int kStages = (int)((196608u) / (kA + kStageB));
    static constexpr size_t kSmem = 1024 + (size_t)kStages * (kA + kStageB) + 256;
};

template <int BN, int EPI, bool SPLIT>
__global__ void __launch_bounds__(128, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmB2, int K, int M, int T, int F,
               void* __restrict__ Y, void* __restrict__ Y2, int ldy, uint32_t* __restrict__ err) {
    using C = TcCfg<BN, SPLIT>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::kA;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * C::kStageB);
    uint64_t* empty = full + S;
    uint64_t* accf = empty + S;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = K / kBK;
    // token tiles run fastest, so the blocks that share a weight tile run together and read it
    // from HBM once (the rest hit L2)
    const int row0 = blockIdx.y * (EPI == GEMM_EPI_SWIGLU ? 64 : kBM);
    const int t0 = blockIdx.x * BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
        if (SPLIT)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB2)) : "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"((uint32_t)BN));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (threadIdx.x == 0) {
        // ---- TMA producer
        int issued = 0;
        constexpr int kAhead = 8;                  // weight tiles requested into L2 ahead
        for (int kb = 0; kb < nk && kb < kAhead; ++kb) {
            tma_prefetch_2d(&tmA, kb * kBK, row0);
            if (EPI == GEMM_EPI_SWIGLU) tma_prefetch_2d(&tmA, kb * kBK, F + row0);
        }
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S;
            if (kb + kAhead < nk) {
                tma_prefetch_2d(&tmA, (kb + kAhead) * kBK, row0);
                if (EPI == GEMM_EPI_SWIGLU) tma_prefetch_2d(&tmA, (kb + kAhead) * kBK, F + row0);
            }
            const uint32_t ph = (uint32_t)(kb / S) & 1u;
            if (kb >= S && !mbar_wait(&empty[s], ph ^ 1u)) { atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; break; }
            if (*(volatile int*)abort_flag) break;
            mbar_expect_tx(&full[s], C::kA + C::kStageB);
            if (EPI == GEMM_EPI_SWIGLU) {
                tma_load_2d(sA + s * C::kA, &tmA, &full[s], kb * kBK, row0);
                tma_load_2d(sA + s * C::kA + C::kA / 2, &tmA, &full[s], kb * kBK, F + row0);
            } else {
                tma_load_2d(sA + s * C::kA, &tmA, &full[s], kb * kBK, row0);
            }
            tma_load_2d(sB + s * C::kStageB, &tmB, &full[s], kb * kBK, t0);
            if (SPLIT) tma_load_2d(sB + s * C::kStageB + C::kB, &tmB2, &full[s], kb * kBK, t0);
            issued = kb + 1;
        }
        // drain: every copy this thread issued has landed before the block can exit
        for (int kb = (issued > S ? issued - S : 0); kb < issued; ++kb)
            mbar_wait(&full[kb % S], (uint32_t)(kb / S) & 1u);
    } else if (threadIdx.x == 32) {
        // ---- MMA issuer
        constexpr uint32_t idesc = idesc_bf16(kBM, BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S;
            const uint32_t ph = (uint32_t)(kb / S) & 1u;
            if (!mbar_wait(&full[s], ph)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = sdesc_sw128(smem_u32(sA + s * C::kA));
            const uint64_t bd = sdesc_sw128(smem_u32(sB + s * C::kStageB));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                umma_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
            if (SPLIT) {
                const uint64_t bd2 = sdesc_sw128(smem_u32(sB + s * C::kStageB + C::kB));
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    umma_bf16(tmem, ad + (uint64_t)(kk * 2), bd2 + (uint64_t)(kk * 2), idesc, 1u);
            }
            umma_commit(&empty[s]);
        }
        if (!ok) { atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; }
        umma_commit(accf);
    }
    __syncwarp();

    // ---- epilogue: TMEM -> registers -> global
    const bool have = mbar_wait(accf, 0);
    tc_fence_after();
    if (!have) atomicOr(err, ERR_TIMEOUT);
    const bool live = have && !*(volatile int*)abort_flag;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (EPI != GEMM_EPI_SWIGLU) {
        const int m = row0 + warp * 32 + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + (uint32_t)c0, v);
            if (!live || m >= M) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = t0 + c0 + j;
                if (t >= T) break;
                float* dst = static_cast<float*>(Y) + (int64_t)t * ldy + m;
                if (EPI == GEMM_EPI_ADD) *dst += v[j];
                else *dst = v[j];
            }
        }
    } else {
        // warps 2-3 (up rows) hand their values to warps 0-1 (gate rows) through shared memory;
        // the pipeline stages are free once the accumulator is complete
        float* xu = reinterpret_cast<float*>(smem);          // [64 rows][16 columns]
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + (uint32_t)c0, v);
            if (warp >= 2) {
#pragma unroll
                for (int j = 0; j < 16; ++j) xu[((warp - 2) * 32 + lane) * 17 + j] = v[j];
            }
            __syncthreads();
            if (warp < 2 && live) {
                const int jrow = row0 + warp * 32 + lane;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = t0 + c0 + j;
                    if (t >= T) break;
                    const float g = v[j];
                    const float u = xu[(warp * 32 + lane) * 17 + j];
                    const float o = g / (1.0f + expf(-g)) * u;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(o);
                    static_cast<__nv_bfloat16*>(Y)[(int64_t)t * ldy + jrow] = hi;
                    if (Y2)      // low term of the split output (the next GEMM's second operand)
                        static_cast<__nv_bfloat16*>(Y2)[(int64_t)t * ldy + jrow] =
                            __float2bfloat16_rn(o - __bfloat162float(hi));
                }
            }
            __syncthreads();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)BN));
}

// Token-major GEMM: the MMA's A operand is a 128-token tile of the activations (two bf16 terms,
// hi and lo) and its B operand 256 weight rows (N = 256; for SwiGLU 128 gate rows followed by the
// 128 matching up rows), so one 64 KB stage feeds twice the MMA work of a 48 KB stage of the
// weight-major kernel. The accumulator D[128 tokens][256] has one token per TMEM lane: each thread
// owns its token's 256 outputs. SwiGLU writes silu(g) * u of 128 consecutive features as bf16
// hi and lo terms; store / residual add write float32, through vector atomic adds when the K
// range is split over blockIdx.z (the output then starts zeroed for a store). With a second weight
// map (tmWlo) the weights are two bf16 terms too (a Q8_0 weight d*q as hi + lo): the K loop runs
// over both weight terms, each against both activation terms.
//
// A2 = false: one f16 activation term and f16 weights (a BF16 weight converted exactly, or a
// Q8_0 weight as two f16 terms that hold d*q exactly): one MMA per k-step and weight term, and
// SwiGLU writes a single f16 output.
constexpr int kTnRows = 128;                     // tokens per tile (MMA M)
constexpr int kTnN = 256;                        // 128 gate + 128 up rows (MMA N)
constexpr uint32_t kTnA = kTnRows * kBK * 2;     // 16 KB per activation term
constexpr uint32_t kTnB = kTnN * kBK * 2;        // 32 KB
template <bool A2>
struct TnCfg {
    static constexpr uint32_t kStage = (A2 ? 2 : 1) * kTnA + kTnB;    // 64 KB or 48 KB
    static constexpr int kStages = (int)(196608u / kStage);             // 3 or 4
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + 256;
};

// Epilogue of the token-major GEMM: thread (warp, lane) drains TMEM lane 32 warp + lane, the
// accumulator row of token t, and writes its outputs: SwiGLU silu(gate_j) * up_j of the 128
// features from f0 (gate in columns j, up in 128 + j) as f16 (one term) or bf16 hi + lo, or the
// 256 store / residual-add columns from f0 as float32 (vector atomic adds when K is split).
template <int EPI, bool A2>
__device__ __forceinline__ void tn_epilogue(uint32_t tmem, int warp, int t, int T, int M, int f0, bool live,
                                            bool atomic, void* __restrict__ Y, void* __restrict__ Y2,
                                            int ldy) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (EPI == GEMM_EPI_SWIGLU && !A2) {
#pragma unroll 1
        for (int j0 = 0; j0 < kTnN / 2; j0 += 16) {
            float g[16], u[16];
            tmem_ld16(tmem + lane_base + (uint32_t)j0, g);
            tmem_ld16(tmem + lane_base + (uint32_t)(kTnN / 2 + j0), u);
            if (!live || t >= T) continue;
            uint32_t h[8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const float o0 = g[j] / (1.0f + expf(-g[j])) * u[j];
                const float o1 = g[j + 1] / (1.0f + expf(-g[j + 1])) * u[j + 1];
                const __half2 hv = __floats2half2_rn(o0, o1);
                h[j / 2] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            uint4* dh = reinterpret_cast<uint4*>(static_cast<__half*>(Y) + (int64_t)t * ldy + f0 + j0);
            dh[0] = make_uint4(h[0], h[1], h[2], h[3]);
            dh[1] = make_uint4(h[4], h[5], h[6], h[7]);
        }
    } else if (EPI == GEMM_EPI_SWIGLU) {
        __nv_bfloat16* Yb = static_cast<__nv_bfloat16*>(Y);
        __nv_bfloat16* Yb2 = static_cast<__nv_bfloat16*>(Y2);
#pragma unroll 1
        for (int j0 = 0; j0 < kTnN / 2; j0 += 16) {
            float g[16], u[16];
            tmem_ld16(tmem + lane_base + (uint32_t)j0, g);
            tmem_ld16(tmem + lane_base + (uint32_t)(kTnN / 2 + j0), u);
            if (!live || t >= T) continue;
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const float o0 = g[j] / (1.0f + expf(-g[j])) * u[j];
                const float o1 = g[j + 1] / (1.0f + expf(-g[j + 1])) * u[j + 1];
                const __nv_bfloat162 h = __floats2bfloat162_rn(o0, o1);
                const float2 hf = __bfloat1622float2(h);
                const __nv_bfloat162 l2 = __floats2bfloat162_rn(o0 - hf.x, o1 - hf.y);
                hi[j / 2] = *reinterpret_cast<const uint32_t*>(&h);
                lo[j / 2] = *reinterpret_cast<const uint32_t*>(&l2);
            }
            uint4* dh = reinterpret_cast<uint4*>(Yb + (int64_t)t * ldy + f0 + j0);
            dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
            if (Yb2) {
                uint4* dl = reinterpret_cast<uint4*>(Yb2 + (int64_t)t * ldy + f0 + j0);
                dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
            }
        }
    } else {
        float* Yf = static_cast<float*>(Y);
#pragma unroll 1
        for (int j0 = 0; j0 < kTnN; j0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + (uint32_t)j0, v);
            if (!live || t >= T || f0 + j0 >= M) continue;
            float4* dst = reinterpret_cast<float4*>(Yf + (int64_t)t * ldy + f0 + j0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 w4 = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                if (atomic) {
                    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + q),
                                 "f"(w4.x), "f"(w4.y), "f"(w4.z), "f"(w4.w) : "memory");
                } else {
                    if (EPI == GEMM_EPI_ADD) {
                        const float4 o = dst[q];
                        w4.x += o.x; w4.y += o.y; w4.z += o.z; w4.w += o.w;
                    }
                    dst[q] = w4;
                }
            }
        }
    }
}

// Epilogue through shared memory and TMA stores (f16 operands): warp w stages the accumulator rows
// of its 32 tokens in 128-byte-swizzled boxes of 32 rows (store / add: 8 boxes of 32 float32
// columns, 32 KB per warp; SwiGLU: 2 boxes of 64 f16 features, 8 KB per warp) in the pipeline's
// shared memory, which the MMAs no longer read, and lane 0 writes them with bulk tensor copies:
// a store, or an element-wise reduce-add in L2 for the residual add and for K splits (the partial
// sums of several CTAs then add without atomics). Rows past T are written as zeros (a store) or
// add nothing; a warp whose rows all lie past T writes nothing. The Q/K/V epilogue stores a Q
// tile like a store after the rotation and writes K and V tiles straight to their cache rows.
// half: -1 for all of the tile's columns (warp w of four), or 0 / 1 for the first or second half
// of them (two groups of four warps; warp w reads TMEM lanes of w % 4 and stages its boxes in its
// own shared-memory slice).
template <int EPI>
__device__ __forceinline__ void tn_epilogue_tma(uint32_t tmem, int warp, int lane, int trow0, int T, int f0,
                                                bool live, bool reduce, const CUtensorMap* ymap, uint8_t* smem,
                                                const TnQkv& qe, uint32_t* err, int half = -1) {
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int t = trow0 + lane;
    const bool row_ok = t < T;
    const uint32_t sw = (uint32_t)(lane & 7);
    // column blocks [cb0, cb1) of 32 (non-SwiGLU) or gate column offsets [j0a, j0b) (SwiGLU)
    const int cb0 = half < 0 ? 0 : half * (kTnN / 64), cb1 = half < 0 ? kTnN / 32 : cb0 + kTnN / 64;
    const int j0a = half < 0 ? 0 : half * (kTnN / 4), j0b = half < 0 ? kTnN / 2 : j0a + kTnN / 4;
    uint8_t* wbuf = smem + (size_t)warp * (EPI == GEMM_EPI_SWIGLU ? 8192 : (half < 0 ? 32768 : 16384)) -
                    (EPI == GEMM_EPI_SWIGLU ? 0 : (size_t)cb0 * 4096);
    bool boxes = true;                               // whether this tile goes out through the boxes
    if (EPI == GEMM_EPI_SWIGLU) {
#pragma unroll 1
        for (int j0 = j0a; j0 < j0b; j0 += 32) {
            float g[32], u[32];
            tmem_ld32(tmem + lane_base + (uint32_t)j0, g);
            tmem_ld32(tmem + lane_base + (uint32_t)(kTnN / 2 + j0), u);
            uint32_t h[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const __half2 hv = __floats2half2_rn(row_ok ? silu_mul_fast(g[j], u[j]) : 0.0f,
                                                     row_ok ? silu_mul_fast(g[j + 1], u[j + 1]) : 0.0f);
                h[j / 2] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            uint8_t* row = wbuf + (j0 / 64) * 4096 + lane * 128;
            const uint32_t c0 = (uint32_t)((j0 % 64) / 8);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                st_shared_v4(row + (((c0 + c) ^ sw) << 4), h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
        }
    } else {
        // Q/K/V: which part the tile holds, and this token's cache cell for a K or V tile
        const int qcols = qe.H * qe.hd, kcols = qe.Hkv * qe.hd;
        const bool rot = EPI == GEMM_EPI_QKV && f0 < qcols + kcols;
        const bool kv = EPI == GEMM_EPI_QKV && f0 >= qcols;
        int32_t cell = 0;
        if (kv) {
            cell = row_ok ? qe.slot[t] : 0;
            const bool ok = cell >= 0 && cell < qe.n_ctx;
            if (row_ok && !ok && live) atomicOr(err, ERR_SLOT_RANGE);
            boxes = false;
            live = live && row_ok && ok;
        }
#pragma unroll 1
        for (int b = cb0; b < cb1; ++b) {
            float v[32];
            tmem_ld32(tmem + lane_base + (uint32_t)(32 * b), v);
            const int col = f0 + 32 * b;
            if (rot && row_ok) {
                // adjacent pairs (2i, 2i + 1) of a head turn by the token's angle for pair i
                const int e0 = col % qe.hd;
                const float4* cs4 = reinterpret_cast<const float4*>(qe.cs + (int64_t)t * (qe.hd / 2) + e0 / 2);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 e = cs4[q];            // (cos, sin) of pairs 2q and 2q + 1
                    const float x0 = v[4 * q], x1 = v[4 * q + 1], x2 = v[4 * q + 2], x3 = v[4 * q + 3];
                    v[4 * q] = x0 * e.x - x1 * e.y;
                    v[4 * q + 1] = x0 * e.y + x1 * e.x;
                    v[4 * q + 2] = x2 * e.z - x3 * e.w;
                    v[4 * q + 3] = x2 * e.w + x3 * e.z;
                }
            }
            if (kv) {
                if (live) {
                    const bool isk = col < qcols + kcols;
                    const int kcol = col - (isk ? qcols : qcols + kcols);
                    const int g = kcol / qe.hd, e0 = kcol % qe.hd;
                    __half* dst = static_cast<__half*>(isk ? qe.kc : qe.vc) + ((int64_t)g * qe.n_ctx + cell) * qe.hd + e0;
                    uint32_t h[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const __half2 hv = __floats2half2_rn(v[j], v[j + 1]);
                        h[j / 2] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                    for (int c = 0; c < 4; ++c) d4[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                }
                continue;
            }
            uint8_t* row = wbuf + b * 4096 + lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float* q = v + 4 * c;
                st_shared_v4(row + (((uint32_t)c ^ sw) << 4), row_ok ? __float_as_uint(q[0]) : 0u,
                             row_ok ? __float_as_uint(q[1]) : 0u, row_ok ? __float_as_uint(q[2]) : 0u,
                             row_ok ? __float_as_uint(q[3]) : 0u);
            }
        }
    }
    if (!boxes) return;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0 && live && trow0 < T) {
        constexpr int bw = EPI == GEMM_EPI_SWIGLU ? 64 : 32;
        const int bb0 = EPI == GEMM_EPI_SWIGLU ? j0a / 64 : cb0;
        const int bb1 = EPI == GEMM_EPI_SWIGLU ? (j0b + 63) / 64 : cb1;
#pragma unroll 1
        for (int b = bb0; b < bb1; ++b) {
            if (reduce) tma_reduce_add_2d(ymap, wbuf + b * 4096, f0 + b * bw, trow0);
            else tma_store_2d(ymap, wbuf + b * 4096, f0 + b * bw, trow0);
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    __syncwarp();
}

template <int EPI, bool A2>
__global__ void __launch_bounds__(128, 1)
gemm_tn_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXlo,
               const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWlo,
               const __grid_constant__ CUtensorMap tmY, int use_ymap, const TnQkv qe,
               int planes, int K, int T, int M, int F,
               void* __restrict__ Y, void* __restrict__ Y2, int ldy, uint32_t* __restrict__ err) {
    using C = TnCfg<A2>;
    constexpr int S = C::kStages;
    constexpr uint32_t kTnStage = C::kStage;
    constexpr uint32_t kBOff = (A2 ? 2 : 1) * kTnA;              // weights after the activation terms
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kTnStage);
    uint64_t* empty = full + S;
    uint64_t* accf = empty + S;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk_all = K / kBK;
    const int per = (nk_all + gridDim.z - 1) / gridDim.z;
    const int kb0 = min(nk_all, (int)blockIdx.z * per), nkp = min(nk_all, kb0 + per) - kb0;
    const int nk = nkp * planes;                     // k-steps: this split's K range per weight term
    const int t0 = blockIdx.x * kTnRows;             // token tiles run fastest (weight reuse in L2)
    // SwiGLU: first gate/up feature of the tile; otherwise the first of its 256 weight rows
    const int f0 = blockIdx.y * (EPI == GEMM_EPI_SWIGLU ? kTnN / 2 : kTnN);
    const int w2 = EPI == GEMM_EPI_SWIGLU ? F + f0 : f0 + kTnN / 2;   // second 128-row box

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
        if (A2) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmXlo)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
        if (planes > 1)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmWlo)) : "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"((uint32_t)kTnN));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (threadIdx.x == 0) {
        // ---- TMA producer: per stage the two activation terms and the gate and up rows
        // the weights of the first stages go out before the grid dependency wait (they do not
        // depend on the kernel before), the activations after it
        const int pre = min(nk, S);
        for (int kb = 0; kb < pre; ++kb) {
            uint8_t* st = smem + (size_t)kb * kTnStage;
            const int kx = (kb0 + kb % nkp) * kBK;
            const CUtensorMap* wm = kb < nkp ? &tmW : &tmWlo;
            mbar_expect_tx(&full[kb], kTnStage);
            tma_load_2d(st + kBOff, wm, &full[kb], kx, f0);
            tma_load_2d(st + kBOff + kTnB / 2, wm, &full[kb], kx, w2);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S;
            const uint32_t ph = (uint32_t)(kb / S) & 1u;
            if (kb >= S && !mbar_wait(&empty[s], ph ^ 1u)) { atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; break; }
            if (*(volatile int*)abort_flag) break;
            uint8_t* st = smem + (size_t)s * kTnStage;
            const int kx = (kb0 + kb % nkp) * kBK;
            const CUtensorMap* wm = kb < nkp ? &tmW : &tmWlo;
            if (kb >= S) {
                mbar_expect_tx(&full[s], kTnStage);
                tma_load_2d(st + kBOff, wm, &full[s], kx, f0);
                tma_load_2d(st + kBOff + kTnB / 2, wm, &full[s], kx, w2);
            }
            tma_load_2d(st, &tmX, &full[s], kx, t0);
            if (A2) tma_load_2d(st + kTnA, &tmXlo, &full[s], kx, t0);
            issued = kb + 1;
        }
        if (issued < pre) issued = pre;
        for (int kb = (issued > S ? issued - S : 0); kb < issued; ++kb)
            mbar_wait(&full[kb % S], (uint32_t)(kb / S) & 1u);
    } else if (threadIdx.x == 32) {
        // ---- MMA issuer: D += X_hi W^T + X_lo W^T (A2), or D += X W^T
        constexpr uint32_t idesc = A2 ? idesc_bf16(kTnRows, kTnN) : idesc_f16(kTnRows, kTnN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S;
            const uint32_t ph = (uint32_t)(kb / S) & 1u;
            if (!mbar_wait(&full[s], ph)) { ok = false; break; }
            tc_fence_after();
            const uint8_t* st = smem + (size_t)s * kTnStage;
            const uint64_t ah = sdesc_sw128(smem_u32(st));
            const uint64_t bd = sdesc_sw128(smem_u32(st + kBOff));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                umma_bf16(tmem, ah + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0 ? 1u : 0u);
            if (A2) {
                const uint64_t al = sdesc_sw128(smem_u32(st + kTnA));
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    umma_bf16(tmem, al + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, 1u);
            }
            umma_commit(&empty[s]);
        }
        if (!ok) { atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; }
        umma_commit(accf);
    }
    __syncwarp();

    // ---- epilogue: thread = token; gate columns j and up columns 128 + j of its TMEM lane
    const bool have = mbar_wait(accf, 0);
    tc_fence_after();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    if (!have) atomicOr(err, ERR_TIMEOUT);
    const bool live = have && !*(volatile int*)abort_flag && nk > 0;
    if (!A2 && use_ymap)
        tn_epilogue_tma<EPI>(tmem, warp, lane, t0 + warp * 32, T, f0, live,
                             EPI == GEMM_EPI_ADD || gridDim.z > 1, &tmY, smem, qe, err);
    else if (EPI != GEMM_EPI_QKV)
        tn_epilogue<EPI, A2>(tmem, warp, t0 + warp * 32 + lane, T, M, f0, live, gridDim.z > 1, Y, Y2, ldy);
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)kTnN));
}

// Two-CTA token-major GEMM (tcgen05.mma.cta_group::2), f16 operands: a cluster of two CTAs
// computes a 256-token x 256-row tile. The MMA's A operand is the 256 tokens, 128 in each CTA's
// shared memory, and its B operand the 256 weight rows (for SwiGLU 128 gate + 128 up rows), 128 in
// each CTA; the leader CTA (cluster rank 0) issues every MMA and each CTA's TMEM receives the
// accumulator rows of its own 128 tokens, all 256 columns, so the epilogue is the one-CTA
// kernel's. A stage holds 32 KB per CTA against 48 KB for the same MMA work per SM in the one-CTA
// tile, so six stages fit and each SM pulls two thirds of the bytes through its L2 port.
// Both CTAs' copies of a stage complete on the leader's full barrier (the leader arms it for both
// halves); the leader's commits arrive on the empty and accumulator barriers of both CTAs.
constexpr uint32_t kTn2Half = 128 * kBK * 2;           // 16 KB: 128 rows x 64 f16
constexpr uint32_t kTn2Stage = 2 * kTn2Half;           // this CTA's A half + B half
constexpr int kTn2Stages = 7;
constexpr size_t kTn2Smem = 1024 + (size_t)kTn2Stages * kTn2Stage + 256;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// every thread of both CTAs arrives; shared-memory writes before it are visible after it
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// TMA tile into this CTA's shared memory whose completion is counted on an mbarrier of either CTA
// of the pair (bar: a shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void umma_f16_pair(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// arrive (once) on the mbarrier at this shared offset in both CTAs when the MMAs issued so far end
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)), "h"((uint16_t)3)
        : "memory");
}

// 256 threads: thread 0 issues TMA loads, thread 32 (leader) the MMAs; all eight warps run the
// epilogue, warps 0-3 and 4-7 each half of the tile's columns.
// TRACE: each CTA writes global-timer stamps (ns) to trace[8 * block + i]: 0 start, 1 set-up done,
// 2 first stage ready (leader's MMA thread), 3 last MMA issued, 4 accumulator ready, 5 epilogue
// done, 6 end, 7 the SM id.
template <int EPI, bool TRACE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
gemm_tn2_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmWlo, const __grid_constant__ CUtensorMap tmY, int use_ymap,
                const TnQkv qe, int planes, int K, int T, int M, int F,
                void* __restrict__ Y, int ldy, uint32_t* __restrict__ err, uint64_t* __restrict__ trace) {
    uint64_t* tr = nullptr;
    if (TRACE) {
        tr = trace + 8 * (size_t)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
        if (threadIdx.x == 0) {
            tr[0] = global_ns();
            uint32_t sm;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
            tr[7] = sm;
        }
    }
    constexpr int S = kTn2Stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kTn2Stage);
    uint64_t* empty = full + S;
    uint64_t* accf = empty + S;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk_all = K / kBK;
    const int per = (nk_all + gridDim.z - 1) / gridDim.z;
    const int kb0 = min(nk_all, (int)blockIdx.z * per), nkp = min(nk_all, kb0 + per) - kb0;
    const int nk = nkp * planes;
    const int tm = (int)(blockIdx.x >> 1) * 2 * kTnRows + (int)rank * kTnRows;   // this CTA's tokens
    const int f0 = blockIdx.y * (EPI == GEMM_EPI_SWIGLU ? kTnN / 2 : kTnN);
    // this CTA's 128 weight rows: the gate (rank 0) or up (rank 1) rows of the features from f0,
    // or rows f0 + 128 rank
    const int wrow = EPI == GEMM_EPI_SWIGLU ? (rank ? F + f0 : f0) : f0 + (int)rank * (kTnN / 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
        if (planes > 1)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmWlo)) : "memory");
    }
    if (warp == 0) {
        // the pair allocates the same TMEM columns in both SMs (issued by one warp of each CTA)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"((uint32_t)kTnN));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    tc_fence_before();
    cluster_sync_all();                 // barriers of both CTAs initialised, TMEM address written
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (TRACE && threadIdx.x == 0) tr[1] = global_ns();

    if (threadIdx.x == 0) {
        // ---- TMA producer (both CTAs): this CTA's 128 tokens and 128 weight rows per stage. The
        // weights of the first stages do not depend on the kernel before (launched with
        // programmatic dependent launch, this one may start while that one ends): they are
        // requested before the grid dependency wait, the activations after it.
        const int pre = min(nk, S);
        for (int kb = 0; kb < pre; ++kb) {
            const uint32_t fb = cluster_addr(smem_u32(&full[kb]), 0);
            if (rank == 0) mbar_expect_tx(&full[kb], 2 * kTn2Stage);
            tma_load_2d_pair(smem + (size_t)kb * kTn2Stage + kTn2Half, kb < nkp ? &tmW : &tmWlo, fb,
                             (kb0 + kb % nkp) * kBK, wrow);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S;
            const uint32_t ph = (uint32_t)(kb / S) & 1u;
            if (kb >= S && !mbar_wait(&empty[s], ph ^ 1u)) { atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; break; }
            if (*(volatile int*)abort_flag) break;
            uint8_t* st = smem + (size_t)s * kTn2Stage;
            const uint32_t fb = cluster_addr(smem_u32(&full[s]), 0);
            const int kx = (kb0 + kb % nkp) * kBK;
            if (kb >= S) {
                if (rank == 0) mbar_expect_tx(&full[s], 2 * kTn2Stage);
                tma_load_2d_pair(st + kTn2Half, kb < nkp ? &tmW : &tmWlo, fb, kx, wrow);
            }
            tma_load_2d_pair(st, &tmX, fb, kx, tm);
            issued = kb + 1;
        }
        if (issued < pre) issued = pre;                // the early weight copies are in flight too
        // drain: the copies issued have landed before the CTA can exit (the leader's full barrier
        // counts both CTAs' bytes; the peer sees its last stage consumed)
        if (rank == 0) {
            for (int kb = (issued > S ? issued - S : 0); kb < issued; ++kb)
                mbar_wait(&full[kb % S], (uint32_t)(kb / S) & 1u);
        } else if (issued > 0) {
            mbar_wait(&empty[(issued - 1) % S], (uint32_t)((issued - 1) / S) & 1u);
        }
    } else if (threadIdx.x == 32 && rank == 0) {
        // ---- MMA issuer (leader): D[256 tokens][256] += X W^T, one MMA per 16-wide k-step
        constexpr uint32_t idesc = idesc_f16(2 * kTnRows, kTnN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S;
            const uint32_t ph = (uint32_t)(kb / S) & 1u;
            if (!mbar_wait(&full[s], ph)) { ok = false; break; }
            tc_fence_after();
            if (TRACE && kb == 0) tr[2] = global_ns();
            const uint8_t* st = smem + (size_t)s * kTn2Stage;
            const uint64_t ad = sdesc_sw128(smem_u32(st));
            const uint64_t bd = sdesc_sw128(smem_u32(st + kTn2Half));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
                umma_f16_pair(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0 ? 1u : 0u);
            umma_commit_pair(&empty[s]);
        }
        if (!ok) { atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; }
        umma_commit_pair(accf);
        if (TRACE) tr[3] = global_ns();
    }
    __syncwarp();

    const bool have = mbar_wait(accf, 0);
    tc_fence_after();
    if (TRACE && threadIdx.x == 0) tr[4] = global_ns();
    // the output may be read or written by the kernel before until it has ended; the kernel after
    // may be scheduled now (it waits for this one's end before touching its data)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    if (!have) atomicOr(err, ERR_TIMEOUT);
    const bool live = have && !*(volatile int*)abort_flag && nk > 0;
    // the epilogue on both groups of four warps, each group half of the columns
    if (use_ymap)
        tn_epilogue_tma<EPI>(tmem, warp, lane, tm + (warp & 3) * 32, T, f0, live,
                             EPI == GEMM_EPI_ADD || gridDim.z > 1, &tmY, smem, qe, err, warp >> 2);
    else if (EPI != GEMM_EPI_QKV && warp < 4)
        tn_epilogue<EPI, false>(tmem, warp, tm + warp * 32 + lane, T, M, f0, live, gridDim.z > 1, Y, nullptr, ldy);
    if (TRACE) {
        __syncthreads();
        if (threadIdx.x == 0) tr[5] = global_ns();
    }
    tc_fence_before();
    cluster_sync_all();                 // both CTAs done with the pair's TMEM and shared memory
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)kTnN));
    if (TRACE && threadIdx.x == 0) tr[6] = global_ns();
}

// ---- Q8_0 weights dequantised inside the two-CTA kernel
//
// The weight operand is read from HBM as stored (int8 quants, one fp16 scale per 32 values: 34
// bytes per 32 weights) instead of as precomputed f16 terms (4 bytes per weight). The product is
// computed transposed, D[weight row][token] = (hi + lo) X^T: the weight terms are the MMA's A
// operand, held in tensor memory, and the token tile is B in shared memory. Per k-step of 64
// values a producer thread copies this CTA's 128 x 64 quant tile and the rows' block scales into a
// raw ring (64-byte swizzle), and sixteen converter warps (four threads per weight row, 16 quants
// each) turn it into the two f16 terms hi = rn(d q) and lo = rn(d q - hi) (hi + lo = d q exactly)
// and store them into a ring of tensor-memory stages with tcgen05.st. Compared with terms in
// shared memory this keeps the converters' stores off shared memory, whose bandwidth the MMA's
// operand reads (the token tile is read by both CTAs of the pair, once per term) already fill.
// ([P2] "llama.cpp Architecture", Example 4 MUL_MAT over a q8_0 weight; the block format of the
// GGUF quant types.)
// Warps 0-3: token-tile producer (thread 0), MMA issuer (thread 32, leader CTA), quant-tile
// producer (thread 64); in the peer CTA threads 32 and 96 forward its converters' completion to
// the leader (alternate k-steps). Warps 4-19: converters. Warps 0-15 then run the epilogue (warp w
// holds the 32 weight rows of the tensor-memory lanes it may access, w % 4). SwiGLU: a CTA's 128
// weight rows are the gate rows of 64 features and then their up rows, so a product's two factors
// are in the same CTA.
constexpr uint32_t kQ8Tok = kTn2Half;                     // 128 tokens x 64 f16: 16 KB
constexpr int kQ8TokStages = 6;
constexpr uint32_t kQ8Quants = 128 * kBK;                // 128 rows x 64 quants: 8 KB
constexpr uint32_t kQ8Raw = kQ8Quants + 128 * 4;          // + the rows' two block scales each
constexpr int kQ8RawStages = 6;
constexpr int kQ8AStages = 4;                             // tensor-memory stages of 64 columns (hi, lo)
constexpr uint32_t kQ8ACol0 = kTnN;                       // the accumulator takes columns [0, 256)
constexpr int kQ8ConvWarps = 16;
constexpr int kQ8Threads = 128 + 32 * kQ8ConvWarps;
constexpr size_t kQ8Smem = 1024 + (size_t)kQ8TokStages * kQ8Tok + (size_t)kQ8RawStages * kQ8Raw + 512;
static_assert(kQ8Smem <= 232448, "the Q8_0 rings fit one CTA's shared memory");
static_assert(kQ8ACol0 + 64 * kQ8AStages <= 512, "accumulator and weight stages fit tensor memory");

__device__ __forceinline__ bool mbar_try_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// the same bounded wait, acquiring at cluster scope (arrivals that release from the peer CTA)
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    if (mbar_try_cluster(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_cluster(bar, parity))
        if (global_ns() - t0 > kWaitNs) return false;
    return true;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// four int8 quants (one 32-bit word) times the block scale d as f16 terms: (hi01, hi23, lo01, lo23)
__device__ __forceinline__ void q8x4_terms(uint32_t w, __half2 d, uint32_t& h01, uint32_t& h23, uint32_t& l01,
                                           uint32_t& l23) {
    const uint32_t u = w ^ 0x80808080u;                  // q + 128 as unsigned bytes
    const uint32_t b01 = __byte_perm(u, 0x64646464u, 0x4140u), b23 = __byte_perm(u, 0x64646464u, 0x4342u);
    const __half2 off = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));   // 1152
    // 1024 + (q + 128) - 1152 = q, exact in f16
    const __half2 q01 = __hsub2(*reinterpret_cast<const __half2*>(&b01), off);
    const __half2 q23 = __hsub2(*reinterpret_cast<const __half2*>(&b23), off);
    const __half2 x01 = __hmul2(q01, d), x23 = __hmul2(q23, d);
    const __half2 y01 = __hfma2(q01, d, __hneg2(x01)), y23 = __hfma2(q23, d, __hneg2(x23));
    h01 = *reinterpret_cast<const uint32_t*>(&x01);
    h23 = *reinterpret_cast<const uint32_t*>(&x23);
    l01 = *reinterpret_cast<const uint32_t*>(&y01);
    l23 = *reinterpret_cast<const uint32_t*>(&y23);
}

// A from tensor memory, B from shared memory, D in tensor memory (the pair's MMA)
__device__ __forceinline__ void umma_ts_pair(uint32_t dtmem, uint32_t atmem, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(dtmem),
        "r"(atmem), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// The transposed epilogue, on four groups of four warps (warps 0-15: the converters are idle by
// then): warp w holds D rows 32 (w % 4) .. + 31 of this CTA (weight rows, one per lane, the
// tensor-memory lanes it may read), and group g = w / 4 takes the 32-token chunks g and g + 4 of the
// pair's 256 tokens (tensor-memory columns). With an output map the values go through shared-memory
// boxes of 32 tokens x 128 bytes (128-byte swizzle, written transposed: one lane per column) and
// bulk tensor stores, or element-wise reduce-adds in L2 for the residual add and K splits;
// without one, direct stores.
template <int EPI>
__device__ __forceinline__ void q8t_epilogue(uint32_t tmem, int warp, int lane, int tok0, int T, int mrow0,
                                             bool live, bool split, const CUtensorMap* ymap, void* Y, int ldy,
                                             const TnQkv& qe, uint8_t* stage, uint32_t* err) {
    const int q = warp & 3, grp = warp >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int m = mrow0 + q * 32 + lane;                    // this lane's weight row (not SwiGLU)
    const int qcols = qe.H * qe.hd, kcols = qe.Hkv * qe.hd;
    const bool rot = EPI == GEMM_EPI_QKV && mrow0 < qcols + kcols;
    const bool isq = EPI == GEMM_EPI_QKV && mrow0 < qcols;
    const bool isk = EPI == GEMM_EPI_QKV && !isq && mrow0 < qcols + kcols;
    const bool boxes = ymap != nullptr && (EPI != GEMM_EPI_QKV || isq);
    const bool reduce = EPI == GEMM_EPI_ADD || split;
    // boxes: warp w's two 4 KB buffers (f32 outputs); SwiGLU: per group an exchange area for the
    // handed-over values and two 4 KB f16 boxes (one per chunk, shared by the group's warps)
    uint8_t* wbuf = stage + warp * 8192;
    float* exf = reinterpret_cast<float*>(stage + grp * 17408);
    uint8_t* hbuf = stage + grp * 17408 + 9216;             // 1024-aligned, after the exchange area
    static_assert(2 * 64 * 17 * 4 <= 9216, "exchange area");
    const uint32_t bar_id = 1u + (uint32_t)grp;
    const bool leader = q == 0 && lane == 0;                // issues the group's SwiGLU box stores
#pragma unroll 1
    for (int it = 0, b = grp; b < kTnN / 32; ++it, b += 4) {
        float v[32];
        tmem_ld32(tmem + lane_base + (uint32_t)(32 * b), v);
        const int t0 = tok0 + 32 * b;
        if (EPI == GEMM_EPI_SWIGLU) {
            // warps 0, 1 hold the gate rows of the CTA's 64 features, warps 2, 3 their up rows; the
            // gate warps take tokens 0-15 of the chunk and the up warps tokens 16-31, each handing
            // the other half of its values over through shared memory (ex [2][64 features][17])
            const int f = (q & 1) * 32 + lane;                       // feature within the CTA's 64
            const bool gate = q < 2;
            float* mine = exf + (gate ? 0 : 64 * 17);                // what this warp hands over
            float* theirs = exf + (gate ? 64 * 17 : 0);
            if (it >= 2 && leader && boxes) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
#pragma unroll
            for (int j = 0; j < 16; ++j) mine[f * 17 + j] = v[gate ? 16 + j : j];
            asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
            uint8_t* box = hbuf + (it & 1) * 4096;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int jj = gate ? j : 16 + j;                    // token within the chunk
                const float g = gate ? v[j] : theirs[f * 17 + j];
                const float u = gate ? theirs[f * 17 + j] : v[16 + j];
                const __half h = __float2half_rn(silu_mul_fast(g, u));
                if (boxes) {
                    *reinterpret_cast<__half*>(box + jj * 128 + ((((uint32_t)f >> 3) ^ (uint32_t)(jj & 7)) << 4) +
                                               (f & 7) * 2) = h;
                } else if (live && t0 + jj < T) {
                    static_cast<__half*>(Y)[(int64_t)(t0 + jj) * ldy + mrow0 + f] = h;
                }
            }
            if (boxes) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
            if (boxes && leader && live && t0 < T) {
                tma_store_2d(ymap, box, mrow0, t0);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            continue;
        }
        if (EPI == GEMM_EPI_QKV && rot) {
            // adjacent pairs (2i, 2i + 1) of a head turn by the token's angle for pair i; the pair's
            // two values are in neighbouring lanes
            const int e = m % qe.hd;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int t = min(t0 + j, T - 1);
                const float2 cs = qe.cs[(int64_t)t * (qe.hd / 2) + e / 2];
                const float o = __shfl_xor_sync(0xffffffffu, v[j], 1);
                v[j] = (e & 1) ? fmaf(o, cs.y, v[j] * cs.x) : fmaf(-o, cs.y, v[j] * cs.x);
            }
        }
        if (EPI == GEMM_EPI_QKV && !isq) {
            if (!live) continue;
            const int e = m % qe.hd;
            const int kvh = (m - qcols - (isk ? 0 : kcols)) / qe.hd;
            __half* cache = static_cast<__half*>(isk ? qe.kc : qe.vc);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int t = t0 + j;
                if (t >= T) continue;
                const int32_t cell = qe.slot[t];
                if (cell < 0 || cell >= qe.n_ctx) {
                    if (e == 0) atomicOr(err, ERR_SLOT_RANGE);
                    continue;
                }
                cache[((int64_t)kvh * qe.n_ctx + cell) * qe.hd + e] = __float2half_rn(v[j]);
            }
            continue;
        }
        if (boxes) {
            uint8_t* box = wbuf + (it & 1) * 4096;
            if (it >= 2 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                *reinterpret_cast<float*>(box + j * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(j & 7)) << 4) +
                                          (lane & 3) * 4) = v[j];
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0 && live && t0 < T) {
                if (reduce) tma_reduce_add_2d(ymap, box, mrow0 + q * 32, t0);
                else tma_store_2d(ymap, box, mrow0 + q * 32, t0);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            continue;
        }
        if (!live) continue;
        float* y = static_cast<float*>(Y);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int t = t0 + j;
            if (t >= T) continue;
            float* dst = y + (int64_t)t * ldy + m;
            if (reduce) atomicAdd(dst, v[j]);
            else *dst = v[j];
        }
    }
    // the boxes have been read before the shared memory is given up
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

// TRACE: per CTA 8 values in trace: 0 start (global timer, ns), SM cycles the first converter
// thread spent 1 waiting for quant tiles, 2 waiting for free weight stages, 3 converting; SM cycles
// the MMA thread (leader) spent 4 waiting for token tiles, 5 waiting for converted terms; 6 the
// accumulator ready, 7 the end (global timer, ns).
template <int EPI, bool TRACE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kQ8Threads, 1)
gemm_tn2q8_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmQ,
                  const uint32_t* __restrict__ kscales, int wrows, const __grid_constant__ CUtensorMap tmY,
                  int use_ymap, const TnQkv qe, int K, int T, int M, int F, void* __restrict__ Y, int ldy,
                  uint32_t* __restrict__ err, uint64_t* __restrict__ trace) {
    constexpr int ST = kQ8TokStages, R = kQ8RawStages, SA = kQ8AStages;
    uint64_t* tr = TRACE ? trace + 8 * (size_t)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z))
                         : nullptr;
    if (TRACE && threadIdx.x == 0) tr[0] = global_ns();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* raw = smem + ST * kQ8Tok;
    uint64_t* tfull = reinterpret_cast<uint64_t*>(raw + R * kQ8Raw);   // token tiles (leader: both CTAs)
    uint64_t* tempty = tfull + ST;                                       // token stage read (both CTAs)
    uint64_t* afull = tempty + ST;                                       // weight terms (leader: its 16
                                                                         // warps + the peer's forward)
    uint64_t* aempty = afull + SA;                                       // weight stage read (both CTAs)
    uint64_t* cfull = aempty + SA;                                       // peer: its 16 warps' terms
    uint64_t* rfull = cfull + SA;                                        // quant tile landed (local)
    uint64_t* rempty = rfull + R;                                        // quant tile converted (local)
    uint64_t* accf = rempty + R;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk_all = K / kBK;
    const int per = (nk_all + gridDim.z - 1) / gridDim.z;
    const int kb0 = min(nk_all, (int)blockIdx.z * per), nk = min(nk_all, kb0 + per) - kb0;
    const int tok0 = (int)(blockIdx.x >> 1) * 2 * kTnRows;               // the pair's first token
    const int tm = tok0 + (int)rank * kTnRows;                           // this CTA's B rows
    // this CTA's 128 weight rows: SwiGLU gate rows of features [fg, fg + 64) then their up rows;
    // otherwise rows [mrow0, mrow0 + 128)
    const int fg = blockIdx.y * (kTnN / 2) + (int)rank * 64;
    const int mrow0 = EPI == GEMM_EPI_SWIGLU ? fg : blockIdx.y * kTnN + (int)rank * kTnRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], 1);
        }
        for (int a = 0; a < SA; ++a) {
            mbar_init(&afull[a], kQ8ConvWarps + 1);
            mbar_init(&aempty[a], 1);
            mbar_init(&cfull[a], kQ8ConvWarps);
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(&rfull[r], 1);
            mbar_init(&rempty[r], kQ8ConvWarps);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
    }
    if (warp == 0) {
        // the accumulator (256 columns) and the weight stages (4 x 64 columns), in both SMs
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(512u));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (threadIdx.x == 64) {
        // ---- quant-tile producer: the quants of k-step kb by tensor copy, the rows' scales of
        // that k-step (contiguous in the per-k-step scale layout) by bulk copies, into raw slot
        // kb % R once the converters are done with it. Not written by the kernel before: no grid
        // dependency wait.
        int rissued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int r = kb % R;
            if (kb >= R && !mbar_wait(&rempty[r], ((uint32_t)(kb / R) & 1u) ^ 1u)) {
                atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; break;
            }
            if (*(volatile int*)abort_flag) break;
            uint8_t* dst = raw + (size_t)r * kQ8Raw;
            const int kx = (kb0 + kb) * kBK;
            const uint32_t* ks = kscales + (int64_t)(kb0 + kb) * wrows;
            mbar_expect_tx(&rfull[r], kQ8Raw);
            if (EPI == GEMM_EPI_SWIGLU) {
                tma_load_2d(dst, &tmQ, &rfull[r], kx, fg);
                tma_load_2d(dst + 64 * kBK, &tmQ, &rfull[r], kx, F + fg);
            } else {
                tma_load_2d(dst, &tmQ, &rfull[r], kx, mrow0);
            }
            const int nseg = EPI == GEMM_EPI_SWIGLU ? 2 : 1;
            for (int g = 0; g < nseg; ++g) {
                const int row = EPI == GEMM_EPI_SWIGLU ? (g ? F + fg : fg) : mrow0;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_u32(dst + kQ8Quants + g * (128 / nseg) * 4)),
                    "l"(ks + row), "r"((uint32_t)(128 / nseg) * 4u), "r"(smem_u32(&rfull[r]))
                    : "memory");
            }
            rissued = kb + 1;
        }
        for (int kb = (rissued > R ? rissued - R : 0); kb < rissued; ++kb)
            mbar_wait(&rfull[kb % R], (uint32_t)(kb / R) & 1u);
    } else if (threadIdx.x == 0) {
        // ---- token-tile producer (both CTAs: this CTA's 128 tokens, half of the pair's B)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % ST;
            if (kb >= ST && !mbar_wait(&tempty[s], ((uint32_t)(kb / ST) & 1u) ^ 1u)) {
                atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; break;
            }
            if (*(volatile int*)abort_flag) break;
            if (rank == 0) mbar_expect_tx(&tfull[s], 2 * kQ8Tok);
            tma_load_2d_pair(smem + (size_t)s * kQ8Tok, &tmX, cluster_addr(smem_u32(&tfull[s]), 0), (kb0 + kb) * kBK,
                             tm);
            issued = kb + 1;
        }
        if (rank == 0) {
            for (int kb = (issued > ST ? issued - ST : 0); kb < issued; ++kb)
                mbar_wait(&tfull[kb % ST], (uint32_t)(kb / ST) & 1u);
        } else if (issued > 0) {
            mbar_wait(&tempty[(issued - 1) % ST], (uint32_t)((issued - 1) / ST) & 1u);
        }
    } else if (rank == 1 && (threadIdx.x == 96 || threadIdx.x == 32)) {
        // ---- forwarders (peer CTA, even and odd k-steps): once the peer's 16 converter warps have
        // stored a stage, one arrival on the leader's barrier. An arrival that releases at cluster
        // scope stalls its thread for a long time; here it holds up no converter, and two
        // forwarders take alternate k-steps.
        const uint32_t afull0 = cluster_addr(smem_u32(&afull[0]), 0);
        for (int kb = threadIdx.x == 96 ? 0 : 1; kb < nk; kb += 2) {
            const int a = kb % SA;
            if (!mbar_wait(&cfull[a], (uint32_t)(kb / SA) & 1u)) {
                atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; break;
            }
            mbar_arrive_cluster(afull0 + (uint32_t)(a * 8));
        }
    } else if (threadIdx.x == 32 && rank == 0) {
        // ---- MMA issuer (leader): D[256 weight rows][256 tokens] += (hi + lo) X^T
        constexpr uint32_t idesc = idesc_f16(2 * kTnRows, kTnN);
        bool ok = true;
        long long wa = 0, wb = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % ST, a = kb % SA;
            const long long c0 = TRACE ? clock64() : 0;
            if (!mbar_wait(&tfull[s], (uint32_t)(kb / ST) & 1u)) { ok = false; break; }
            const long long c1 = TRACE ? clock64() : 0;
            if (!mbar_wait_cluster(&afull[a], (uint32_t)(kb / SA) & 1u)) { ok = false; break; }
            if (TRACE) { wa += c1 - c0; wb += clock64() - c1; }
            tc_fence_after();
            const uint64_t bd = sdesc_sw128(smem_u32(smem + (size_t)s * kQ8Tok));
            const uint32_t ahi = tmem + kQ8ACol0 + 64u * (uint32_t)a, alo = ahi + 32u;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                umma_ts_pair(tmem, ahi + 8u * kk, bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0 ? 1u : 0u);
                umma_ts_pair(tmem, alo + 8u * kk, bd + (uint64_t)(kk * 2), idesc, 1u);
            }
            umma_commit_pair(&tempty[s]);
            umma_commit_pair(&aempty[a]);
        }
        if (!ok) { atomicOr(err, ERR_TIMEOUT); *(volatile int*)abort_flag = 1; }
        umma_commit_pair(accf);
        if (TRACE) { tr[4] = (uint64_t)wa; tr[5] = (uint64_t)wb; }
    } else if (warp >= 4) {
        // ---- converters: warp w holds tensor-memory lanes 32 (w % 4) .. + 31 (weight rows) and
        // quant chunk part = (w - 4) / 4 (values 16 part .. 16 part + 15 of the k-step), which is
        // the MMA's k-slice `part` (8 columns of each term's 32)
        const int q = warp & 3, part = (warp - 4) >> 2;
        const int cr = q * 32 + lane;                             // weight row of this CTA's tile
        const uint32_t rs = (uint32_t)((cr >> 1) & 3);
        const uint32_t roff = (uint32_t)cr * kBK + (((uint32_t)part ^ rs) << 4);            // 64-byte swizzle
        const uint32_t soff = kQ8Quants + (uint32_t)cr * 4 + (uint32_t)(part >> 1) * 2;    // its block scale
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + kQ8ACol0 + 8u * (uint32_t)part;
        long long w_raw = 0, w_empty = 0, t_conv = 0;
        bool ok = true;
        for (int kb = 0; kb < nk && ok; ++kb) {
            const int r = kb % R, a = kb % SA;
            const long long t0 = TRACE ? clock64() : 0;
            ok = mbar_wait(&rfull[r], (uint32_t)(kb / R) & 1u);
            if (!ok) break;
            const uint8_t* slot = raw + (size_t)r * kQ8Raw;
            const uint4 v = *reinterpret_cast<const uint4*>(slot + roff);
            const __half2 d = __half2half2(__ushort_as_half(*reinterpret_cast<const unsigned short*>(slot + soff)));
            const long long t1 = TRACE ? clock64() : 0;
            if (kb >= SA) ok = mbar_wait(&aempty[a], ((uint32_t)(kb / SA) & 1u) ^ 1u);
            const long long t2 = TRACE ? clock64() : 0;
            if (TRACE) { w_raw += t1 - t0; w_empty += t2 - t1; }
            if (!ok) break;
            uint32_t h[8], l[8];
            q8x4_terms(v.x, d, h[0], h[1], l[0], l[1]);
            q8x4_terms(v.y, d, h[2], h[3], l[2], l[3]);
            q8x4_terms(v.z, d, h[4], h[5], l[4], l[5]);
            q8x4_terms(v.w, d, h[6], h[7], l[6], l[7]);
            tc_fence_after();                                  // after the wait for the stage to be free
            tmem_st8(tl + 64u * (uint32_t)a, h);
            tmem_st8(tl + 64u * (uint32_t)a + 32u, l);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_local(&rempty[r]);
                mbar_arrive_local(rank == 0 ? &afull[a] : &cfull[a]);   // the leader's own MMA barrier
            }
            if (TRACE) t_conv += clock64() - t2;
        }
        if (!ok) {
            atomicOr(err, ERR_TIMEOUT);
            *(volatile int*)abort_flag = 1;
        }
        if (TRACE && warp == 4 && lane == 0) { tr[1] = (uint64_t)w_raw; tr[2] = (uint64_t)w_empty; tr[3] = (uint64_t)t_conv; }
    }
    __syncwarp();

    if (warp < 16) {
        const bool have = mbar_wait(accf, 0);
        tc_fence_after();
        if (TRACE && threadIdx.x == 0) tr[6] = global_ns();
        // the outputs may be read or written by the kernel before until it has ended
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
        if (!have) atomicOr(err, ERR_TIMEOUT);
        const bool live = have && !*(volatile int*)abort_flag && nk > 0;
        q8t_epilogue<EPI>(tmem, warp, lane, tok0, T, mrow0, live, gridDim.z > 1, use_ymap ? &tmY : nullptr, Y, ldy,
                          qe, smem, err);
    }
    tc_fence_before();
    cluster_sync_all();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u));
    if (TRACE && threadIdx.x == 0) tr[7] = global_ns();
}

__global__ void q8_scales_by_kstep_kernel(const uint32_t* __restrict__ s, int64_t rows, int64_t nk,
                                          uint32_t* __restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;      // [row][kb] order of the source
    if (i >= rows * nk) return;
    const int64_t row = i / nk, kb = i % nk;
    out[kb * rows + row] = s[i];                      // the row's scales 2 kb and 2 kb + 1 as one word
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <int BN, int EPI, bool SPLIT>
bool launch_tc(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, int K, int M,
               int T, int F, void* Y, void* Y2, int ldy, uint32_t* err, cudaStream_t st) {
    using C = TcCfg<BN, SPLIT>;
    auto k = gemm_tc_kernel<BN, EPI, SPLIT>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
            return false;
        attr = true;
    }
    const int rows_per_tile = EPI == GEMM_EPI_SWIGLU ? 64 : kBM;
    const int mtiles = (EPI == GEMM_EPI_SWIGLU ? F : M) / rows_per_tile;
    dim3 grid((T + BN - 1) / BN, mtiles);
    k<<<grid, 128, C::kSmem, st>>>(a, b, b2, K, M, T, F, Y, Y2, ldy, err);
    return cudaGetLastError() == cudaSuccess;
}

template <int EPI>
bool launch_epi(const CUtensorMap& wmap, const CUtensorMap& xmap, const CUtensorMap* xmap_lo,
                int K, int M, int T, int F, void* Y, void* Y2, int ldy, uint32_t* err,
                cudaStream_t st) {
    if (xmap_lo)
        return launch_tc<128, EPI, true>(wmap, xmap, *xmap_lo, K, M, T, F, Y, Y2, ldy, err, st);
    if (tc_token_tile(T) == 256)
        return launch_tc<256, EPI, false>(wmap, xmap, xmap, K, M, T, F, Y, Y2, ldy, err, st);
    return launch_tc<128, EPI, false>(wmap, xmap, xmap, K, M, T, F, Y, Y2, ldy, err, st);
}

}  // namespace

bool tc_make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows, bool f16) {
    auto fn = encode_fn();
    if (!fn) return false;
    if (cols % kBK != 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

void q8_scales_by_kstep(const __half* s, int64_t rows, int64_t K, uint32_t* out, cudaStream_t st) {
    const int64_t n = rows * (K / kBK);
    if (n <= 0) return;
    q8_scales_by_kstep_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(reinterpret_cast<const uint32_t*>(s), rows,
                                                                           K / kBK, out);
}

bool tc_make_map_q8(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    if (cols % kBK != 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int tc_token_tile(int T) { return T > 128 ? 256 : 128; }

bool tc_swiglu_tn_ok(int64_t K, int64_t F) { return K % kBK == 0 && K >= kBK && F % (kTnN / 2) == 0 && F > 0; }
bool tc_tn_ok(int64_t M, int64_t K) { return K % kBK == 0 && K >= kBK && M % kTnN == 0 && M > 0; }

// The two-CTA kernel serves f16 operands when the ubatch fills more than one 128-token tile.
// ymap (f16 operands only): the output's tensor map for the TMA-store epilogue (float32 boxes of
// 32 columns x 32 rows, or f16 boxes of 64 x 32 for SwiGLU, 128-byte swizzle), else direct stores.
template <int EPI, bool TRACE = false>
bool launch_tn2(const CUtensorMap& xmap, const CUtensorMap& wmap, const CUtensorMap* wmap_lo, int K, int T,
                int M, int F, void* Y, int ldy, int splits, uint32_t* err, cudaStream_t st,
                const CUtensorMap* ymap, const TnQkv& qe, uint64_t* trace = nullptr, bool pdl = false) {
    auto k = gemm_tn2_kernel<EPI, TRACE>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTn2Smem) != cudaSuccess)
            return false;
        attr = true;
    }
    const int ntile = EPI == GEMM_EPI_SWIGLU ? F / (kTnN / 2) : M / kTnN;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ((T + 2 * kTnRows - 1) / (2 * kTnRows)), ntile, splits);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = kTn2Smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, xmap, wmap, wmap_lo ? *wmap_lo : wmap, ymap ? *ymap : xmap, ymap ? 1 : 0, qe,
                              wmap_lo ? 2 : 1, K, T, M, F, Y, ldy, err, trace) == cudaSuccess;
}

// The Q8_0 pair kernel serves any token count (a ubatch of at most 128 tokens leaves the peer's
// token rows empty: its tile reads past the ubatch and those outputs are not written). ymap: the
// output's tensor map (tc_make_out_map) for the bulk-store epilogue, else direct stores.
template <int EPI, bool TRACE = false>
bool launch_tn2q8(const CUtensorMap& xmap, const CUtensorMap& qmap, const uint32_t* kscales, int K, int T, int M,
                  int F, void* Y, int ldy, int splits, uint32_t* err, cudaStream_t st, const CUtensorMap* ymap,
                  const TnQkv& qe, bool pdl, uint64_t* trace = nullptr) {
    auto k = gemm_tn2q8_kernel<EPI, TRACE>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQ8Smem) != cudaSuccess)
            return false;
        attr = true;
    }
    const int ntile = EPI == GEMM_EPI_SWIGLU ? F / (kTnN / 2) : M / kTnN;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ((T + 2 * kTnRows - 1) / (2 * kTnRows)), ntile, splits);
    cfg.blockDim = dim3(kQ8Threads);
    cfg.dynamicSmemBytes = kQ8Smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    const int wrows = EPI == GEMM_EPI_SWIGLU ? 2 * F : M;
    return cudaLaunchKernelEx(&cfg, k, xmap, qmap, kscales, wrows, ymap ? *ymap : xmap, ymap ? 1 : 0, qe, K, T, M, F,
                              Y, ldy, err, trace) == cudaSuccess;
}

template <int EPI, bool A2>
bool launch_tn(const CUtensorMap& xmap, const CUtensorMap* xmap_lo, const CUtensorMap& wmap,
               const CUtensorMap* wmap_lo, int K, int T, int M, int F, void* Y, void* Y2, int ldy,
               int splits, uint32_t* err, cudaStream_t st, bool one_cta, const CUtensorMap* ymap,
               const TnQkv& qe = TnQkv{}, bool pdl = false) {
    if (A2) ymap = nullptr;
    if (!A2 && T > kTnRows && !one_cta)
        return launch_tn2<EPI>(xmap, wmap, wmap_lo, K, T, M, F, Y, ldy, splits, err, st, ymap, qe, nullptr, pdl);
    using C = TnCfg<A2>;
    auto k = gemm_tn_kernel<EPI, A2>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
            return false;
        attr = true;
    }
    const int ntile = EPI == GEMM_EPI_SWIGLU ? F / (kTnN / 2) : M / kTnN;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((T + kTnRows - 1) / kTnRows, ntile, splits);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, xmap, xmap_lo ? *xmap_lo : xmap, wmap, wmap_lo ? *wmap_lo : wmap,
                              ymap ? *ymap : xmap, ymap ? 1 : 0, qe, wmap_lo ? 2 : 1, K, T, M, F, Y, Y2, ldy,
                              err) == cudaSuccess;
}

bool launch_gemm_swiglu_tn(const CUtensorMap& xmap, const CUtensorMap* xmap_lo, const CUtensorMap& wmap,
                           int K, int T, int F, void* Y, void* Y2, int ldy, uint32_t* err, cudaStream_t st,
                           const CUtensorMap* wmap_lo, bool one_cta, const CUtensorMap* ymap, bool pdl,
                           const uint32_t* q8_scales) {
    if (T <= 0) return true;
    if (q8_scales) {
        if (xmap_lo || wmap_lo) return false;
        return launch_tn2q8<GEMM_EPI_SWIGLU>(xmap, wmap, q8_scales, K, T, 0, F, Y, ldy, 1, err, st, ymap, TnQkv{}, pdl);
    }
    if (xmap_lo)
        return launch_tn<GEMM_EPI_SWIGLU, true>(xmap, xmap_lo, wmap, wmap_lo, K, T, 0, F, Y, Y2, ldy, 1, err, st,
                                                one_cta, nullptr, TnQkv{}, pdl);
    return launch_tn<GEMM_EPI_SWIGLU, false>(xmap, nullptr, wmap, wmap_lo, K, T, 0, F, Y, nullptr, ldy, 1, err, st,
                                             one_cta, ymap, TnQkv{}, pdl);
}

int tc_tn_splits(int64_t M, int64_t K, int T, int n_sm) {
    const int64_t tiles = (T + kTnRows - 1) / kTnRows * (M / kTnN);
    int s = (int)std::max<int64_t>(1, n_sm / std::max<int64_t>(1, tiles));
    s = std::min(s, 16);                           // a single token tile needs many to fill the SMs
    while (s > 1 && K / kBK / s < 8) --s;          // at least 8 k-steps per split
    return s;
}

bool launch_gemm_tn(const CUtensorMap& xmap, const CUtensorMap* xmap_lo, const CUtensorMap& wmap, int epi,
                    int K, int M, int T, float* Y, int ldy, int splits, uint32_t* err, cudaStream_t st,
                    const CUtensorMap* wmap_lo, bool one_cta, const CUtensorMap* ymap, const TnQkv* qkv, bool pdl,
                    const uint32_t* q8_scales) {
    if (T <= 0) return true;
    if (q8_scales) {
        if (xmap_lo || wmap_lo) return false;
        switch (epi) {
            case GEMM_EPI_QKV:
                if (!qkv || splits != 1 || !tc_tn_qkv_ok(qkv->H, qkv->Hkv, qkv->hd)) return false;
                return launch_tn2q8<GEMM_EPI_QKV>(xmap, wmap, q8_scales, K, T, M, 0, Y, ldy, 1, err, st, ymap, *qkv,
                                                  pdl);
            case GEMM_EPI_STORE:
                return launch_tn2q8<GEMM_EPI_STORE>(xmap, wmap, q8_scales, K, T, M, 0, Y, ldy, splits, err, st, ymap,
                                                    TnQkv{}, pdl);
            case GEMM_EPI_ADD:
                return launch_tn2q8<GEMM_EPI_ADD>(xmap, wmap, q8_scales, K, T, M, 0, Y, ldy, splits, err, st, ymap,
                                                  TnQkv{}, pdl);
        }
        return false;
    }
    if (epi == GEMM_EPI_QKV) {
        if (xmap_lo || !ymap || !qkv || splits != 1 || !tc_tn_qkv_ok(qkv->H, qkv->Hkv, qkv->hd)) return false;
        return launch_tn<GEMM_EPI_QKV, false>(xmap, nullptr, wmap, wmap_lo, K, T, M, 0, Y, nullptr, ldy, 1, err, st,
                                              one_cta, ymap, *qkv, pdl);
    }
    if (epi == GEMM_EPI_STORE)
        return xmap_lo ? launch_tn<GEMM_EPI_STORE, true>(xmap, xmap_lo, wmap, wmap_lo, K, T, M, 0, Y, nullptr, ldy,
                                                         splits, err, st, one_cta, nullptr, TnQkv{}, pdl)
                       : launch_tn<GEMM_EPI_STORE, false>(xmap, nullptr, wmap, wmap_lo, K, T, M, 0, Y, nullptr, ldy,
                                                          splits, err, st, one_cta, ymap, TnQkv{}, pdl);
    if (epi == GEMM_EPI_ADD)
        return xmap_lo ? launch_tn<GEMM_EPI_ADD, true>(xmap, xmap_lo, wmap, wmap_lo, K, T, M, 0, Y, nullptr, ldy,
                                                       splits, err, st, one_cta, nullptr, TnQkv{}, pdl)
                       : launch_tn<GEMM_EPI_ADD, false>(xmap, nullptr, wmap, wmap_lo, K, T, M, 0, Y, nullptr, ldy,
                                                        splits, err, st, one_cta, ymap, TnQkv{}, pdl);
    return false;
}

bool launch_gemm_tn2_traced(const CUtensorMap& xmap, const CUtensorMap& wmap, int epi, int K, int M, int T,
                            int F, void* Y, int ldy, int splits, uint32_t* err, cudaStream_t st,
                            const CUtensorMap* ymap, uint64_t* trace) {
    if (T <= kTnRows) return false;
    switch (epi) {
        case GEMM_EPI_STORE:
            return launch_tn2<GEMM_EPI_STORE, true>(xmap, wmap, nullptr, K, T, M, F, Y, ldy, splits, err, st, ymap,
                                                    TnQkv{}, trace);
        case GEMM_EPI_ADD:
            return launch_tn2<GEMM_EPI_ADD, true>(xmap, wmap, nullptr, K, T, M, F, Y, ldy, splits, err, st, ymap,
                                                  TnQkv{}, trace);
        case GEMM_EPI_SWIGLU:
            return launch_tn2<GEMM_EPI_SWIGLU, true>(xmap, wmap, nullptr, K, T, M, F, Y, ldy, 1, err, st, ymap,
                                                     TnQkv{}, trace);
    }
    return false;
}

bool launch_gemm_tn2q8_traced(const CUtensorMap& xmap, const CUtensorMap& qmap, const uint32_t* scales, int epi,
                              int K, int M, int T, int F, void* Y, int ldy, int splits, uint32_t* err,
                              cudaStream_t st, const CUtensorMap* ymap, uint64_t* trace) {
    switch (epi) {
        case GEMM_EPI_STORE:
            return launch_tn2q8<GEMM_EPI_STORE, true>(xmap, qmap, scales, K, T, M, F, Y, ldy, splits, err, st, ymap,
                                                      TnQkv{}, false, trace);
        case GEMM_EPI_ADD:
            return launch_tn2q8<GEMM_EPI_ADD, true>(xmap, qmap, scales, K, T, M, F, Y, ldy, splits, err, st, ymap,
                                                    TnQkv{}, false, trace);
        case GEMM_EPI_SWIGLU:
            return launch_tn2q8<GEMM_EPI_SWIGLU, true>(xmap, qmap, scales, K, T, M, F, Y, ldy, 1, err, st, ymap,
                                                       TnQkv{}, false, trace);
    }
    return false;
}

bool tc_tn_qkv_ok(int H, int Hkv, int hd) {
    return hd > 0 && kTnN % hd == 0 && hd % 32 == 0 && (H * hd) % kTnN == 0 && (Hkv * hd) % kTnN == 0;
}

bool tc_make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, bool f16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int64_t es = f16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (cols * es) % 16 != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(cols * es)};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), 32u};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int tc_tn2_blocks(int epi, int M, int T, int F, int splits) {
    const int ntile = epi == GEMM_EPI_SWIGLU ? F / (kTnN / 2) : M / kTnN;
    return 2 * ((T + 2 * kTnRows - 1) / (2 * kTnRows)) * ntile * splits;
}

bool tc_shape_ok(int64_t M, int64_t K, int epi, int64_t F) {
    if (K % kBK != 0 || K < kBK) return false;
    if (epi == GEMM_EPI_SWIGLU) return F % 64 == 0 && F > 0;
    return M % kBM == 0 && M > 0;
}

bool launch_gemm_tc(const CUtensorMap& wmap, const CUtensorMap& xmap, int epi, int K, int M,
                    int T, int F, void* Y, int ldy, uint32_t* err, cudaStream_t st,
                    const CUtensorMap* xmap_lo, void* Y2) {
    if (T <= 0) return true;
    switch (epi) {
        case GEMM_EPI_STORE:
            return launch_epi<GEMM_EPI_STORE>(wmap, xmap, xmap_lo, K, M, T, F, Y, Y2, ldy, err, st);
        case GEMM_EPI_ADD:
            return launch_epi<GEMM_EPI_ADD>(wmap, xmap, xmap_lo, K, M, T, F, Y, Y2, ldy, err, st);
        case GEMM_EPI_SWIGLU:
            return launch_epi<GEMM_EPI_SWIGLU>(wmap, xmap, xmap_lo, K, M, T, F, Y, Y2, ldy, err, st);
    }
    return false;
}

}  // namespace llm
