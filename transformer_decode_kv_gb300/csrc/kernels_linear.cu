// Linear layers y = x W^T (ggml MUL_MAT with a {K, M} weight, [P2] "llama.cpp Architecture",
// Example 4) for the weight types of the device store.
//
// Decode (few tokens): a streaming GEMV. Each warp owns RPW weight rows and walks them with
// 16-byte vector loads (4 f32, 8 f16/bf16 or 16 int8 values per lane), so every weight byte is
// read from HBM exactly once per call whatever the token count; the activations of up to TM
// tokens sit in shared memory, K-chunked. Q8_0 rows are dequantised in registers (d * q).
// Prefill (many tokens): a 64x64-tiled FP32 SIMT GEMM that converts weights to f32 in shared
// memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "kernels.h"

namespace llm {

namespace {

constexpr int kGemvWarps = 8;
constexpr int kGemvSmemFloats = 16384;     // 64 KB of activations per block

template <int WT> struct WVec;
template <> struct WVec<W_F32>  { static constexpr int N = 4; };
template <> struct WVec<W_F16>  { static constexpr int N = 8; };
template <> struct WVec<W_BF16> { static constexpr int N = 8; };
template <> struct WVec<W_Q8_0> { static constexpr int N = 16; };

// Load N consecutive weights of row `row` starting at column k (k multiple of N) as floats.
template <int WT>
__device__ __forceinline__ void load_wvec(const void* __restrict__ W, const __half* __restrict__ S,
                                          int64_t K, int64_t row, int64_t k, float* w) {
    if constexpr (WT == W_F32) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(W) + row * K + k));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (WT == W_F16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __half*>(W) + row * K + k));
        const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) { const float2 f = __half22float2(h[i]); w[2 * i] = f.x; w[2 * i + 1] = f.y; }
    } else if constexpr (WT == W_BF16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(W) + row * K + k));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[2 * i] = __uint_as_float(u[i] << 16);
            w[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    } else {
        const int4 v = __ldg(reinterpret_cast<const int4*>(static_cast<const int8_t*>(W) + row * K + k));
        const float d = __half2float(S[row * (K / 32) + k / 32]);
        const int32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int b = 0; b < 4; ++b) w[4 * i + b] = d * (float)(int8_t)((u[i] >> (8 * b)) & 0xff);
        }
    }
}

// SWIGLU: the warp's RPW outputs j use gate rows j and up rows F + j (2 * RPW weight rows).
template <int WT, int TM, int RPW, bool SWIGLU>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_kernel(const void* __restrict__ W, const __half* __restrict__ S, int64_t row0, int64_t M,
            int64_t K, int64_t F, const float* __restrict__ x, int ldx, int T,
            float* __restrict__ y, int ldy, int epi, int kc_max) {
    constexpr int VN = WVec<WT>::N;
    constexpr int NR = SWIGLU ? 2 * RPW : RPW;
    extern __shared__ float xs[];                       // [TM][kc_max]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = ((int64_t)blockIdx.x * kGemvWarps + warp) * RPW;
    int64_t wrow[NR];
    bool live[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const int64_t m = m0 + (r % RPW);
        live[r] = m < M;
        wrow[r] = row0 + (SWIGLU && r >= RPW ? F + m : m);
    }
    float acc[NR][TM];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[r][t] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += kc_max) {
        const int kc = (int)((K - k0) < (int64_t)kc_max ? (K - k0) : (int64_t)kc_max);
        __syncthreads();
        for (int t = 0; t < TM; ++t) {
            for (int j = threadIdx.x * 4; j < kc; j += blockDim.x * 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t < T) v = *reinterpret_cast<const float4*>(x + (int64_t)t * ldx + k0 + j);
                *reinterpret_cast<float4*>(xs + t * kc_max + j) = v;
            }
        }
        __syncthreads();
#pragma unroll 2
        for (int j = lane * VN; j < kc; j += 32 * VN) {
            float w[NR][VN];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (live[r]) load_wvec<WT>(W, S, K, wrow[r], k0 + j, w[r]);
                else {
#pragma unroll
                    for (int e = 0; e < VN; ++e) w[r][e] = 0.f;
                }
            }
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                float xv[VN];
#pragma unroll
                for (int e = 0; e < VN; e += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(xs + t * kc_max + j + e);
                    xv[e] = v.x; xv[e + 1] = v.y; xv[e + 2] = v.z; xv[e + 3] = v.w;
                }
#pragma unroll
                for (int r = 0; r < NR; ++r)
#pragma unroll
                    for (int e = 0; e < VN; ++e) acc[r][t] = fmaf(w[r][e], xv[e], acc[r][t]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int t = 0; t < TM; ++t)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], o);
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int64_t m = m0 + r;
            if (m >= M) continue;
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                if (t >= T) continue;
                float v;
                if constexpr (SWIGLU) {
                    const float g = acc[r][t], u = acc[RPW + r][t];
                    v = g / (1.0f + expf(-g)) * u;
                } else {
                    v = acc[r][t];
                }
                float* dst = y + (int64_t)t * ldy + m;
                *dst = (epi == EPI_ADD) ? *dst + v : v;
            }
        }
    }
}

// ---- tiled SIMT GEMM: y[t][m] (op)= sum_k x[t][k] W[row0 + m][k] -------------------------------
constexpr int BT = 64, BM = 64, BK = 16;

template <int WT>
__device__ __forceinline__ float load_w1(const void* __restrict__ W, const __half* __restrict__ S,
                                         int64_t K, int64_t row, int64_t k) {
    if constexpr (WT == W_F32) return static_cast<const float*>(W)[row * K + k];
    else if constexpr (WT == W_F16) return __half2float(static_cast<const __half*>(W)[row * K + k]);
    else if constexpr (WT == W_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(W)[row * K + k]);
    else return __half2float(S[row * (K / 32) + k / 32]) * (float)static_cast<const int8_t*>(W)[row * K + k];
}

template <int WT>
__global__ void __launch_bounds__(256)
gemm_kernel(const void* __restrict__ W, const __half* __restrict__ S, int64_t row0, int64_t M,
            int64_t K, const float* __restrict__ x, int ldx, int T, float* __restrict__ y, int ldy,
            int epi) {
    __shared__ float As[BK][BT + 4];
    __shared__ float Bs[BK][BM + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;          // 16 x 16 threads, 4 x 4 outputs each
    const int64_t t0 = (int64_t)blockIdx.y * BT, m0 = (int64_t)blockIdx.x * BM;
    float acc[4][4] = {};
    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        // 64 x 16 activations and 64 x 16 weights, 4 each per thread
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + i * 256;
            const int r = e / BK, c = e % BK;
            const int64_t t = t0 + r, m = m0 + r;
            As[c][r] = (t < T) ? x[t * ldx + k0 + c] : 0.f;
            Bs[c][r] = (m < M) ? load_w1<WT>(W, S, K, row0 + m, k0 + c) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < BK; ++c) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[c][ty * 4 + i]; b[i] = Bs[c][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t m = m0 + tx * 4 + j;
            if (m >= M) continue;
            float* dst = y + t * ldy + m;
            *dst = (epi == EPI_ADD) ? *dst + acc[i][j] : acc[i][j];
        }
    }
}

template <int WT, bool SWIGLU>
void gemv_dispatch(const DevMat& W, int64_t row0, int64_t M, int64_t F, const float* x, int ldx,
                   int T, float* y, int ldy, int epi, cudaStream_t st) {
    int tm = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
    int kc = kGemvSmemFloats / tm;
    kc = std::max<int>(512, kc / 512 * 512);
    if (kc > W.cols) kc = (int)W.cols;
    const size_t smem = (size_t)tm * kc * sizeof(float);
    constexpr int RPW = 2;
    const unsigned grid = (unsigned)((M + kGemvWarps * RPW - 1) / (kGemvWarps * RPW));
#define LLM_GEMV_CASE(TMV)                                                                       \
    case TMV: {                                                                                  \
        auto k = gemv_kernel<WT, TMV, RPW, SWIGLU>;                                              \
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);        \
        k<<<grid, kGemvWarps * 32, smem, st>>>(W.data, W.scales, row0, M, W.cols, F, x, ldx, T,  \
                                               y, ldy, epi, kc);                                 \
    } break;
    switch (tm) {
        LLM_GEMV_CASE(1)
        LLM_GEMV_CASE(2)
        LLM_GEMV_CASE(4)
        LLM_GEMV_CASE(8)
    }
#undef LLM_GEMV_CASE
}

template <int WT>
void gemm_dispatch(const DevMat& W, int64_t row0, int64_t M, const float* x, int ldx, int T,
                   float* y, int ldy, int epi, cudaStream_t st) {
    dim3 grid((unsigned)((M + BM - 1) / BM), (unsigned)((T + BT - 1) / BT));
    gemm_kernel<WT><<<grid, 256, 0, st>>>(W.data, W.scales, row0, M, W.cols, x, ldx, T, y, ldy, epi);
}

}  // namespace

int32_t gemv_max_tokens() { return 8; }

void launch_linear(const DevMat& W, int64_t row0, int64_t M, const float* x, int32_t ldx,
                   int32_t T, float* y, int32_t ldy, Epi epi, cudaStream_t st) {
    if (T <= 0 || M <= 0) return;
    if (T <= gemv_max_tokens()) {
        switch (W.type) {
            case W_F32: gemv_dispatch<W_F32, false>(W, row0, M, 0, x, ldx, T, y, ldy, epi, st); break;
            case W_F16: gemv_dispatch<W_F16, false>(W, row0, M, 0, x, ldx, T, y, ldy, epi, st); break;
            case W_BF16: gemv_dispatch<W_BF16, false>(W, row0, M, 0, x, ldx, T, y, ldy, epi, st); break;
            case W_Q8_0: gemv_dispatch<W_Q8_0, false>(W, row0, M, 0, x, ldx, T, y, ldy, epi, st); break;
        }
        return;
    }
    switch (W.type) {
        case W_F32: gemm_dispatch<W_F32>(W, row0, M, x, ldx, T, y, ldy, epi, st); break;
        case W_F16: gemm_dispatch<W_F16>(W, row0, M, x, ldx, T, y, ldy, epi, st); break;
        case W_BF16: gemm_dispatch<W_BF16>(W, row0, M, x, ldx, T, y, ldy, epi, st); break;
        case W_Q8_0: gemm_dispatch<W_Q8_0>(W, row0, M, x, ldx, T, y, ldy, epi, st); break;
    }
}

void launch_linear_swiglu(const DevMat& W, int32_t F, const float* x, int32_t ldx, int32_t T,
                          float* u, int32_t ldu, float* tmp, cudaStream_t st) {
    if (T <= 0) return;
    if (T <= gemv_max_tokens()) {
        switch (W.type) {
            case W_F32: gemv_dispatch<W_F32, true>(W, 0, F, F, x, ldx, T, u, ldu, EPI_STORE, st); break;
            case W_F16: gemv_dispatch<W_F16, true>(W, 0, F, F, x, ldx, T, u, ldu, EPI_STORE, st); break;
            case W_BF16: gemv_dispatch<W_BF16, true>(W, 0, F, F, x, ldx, T, u, ldu, EPI_STORE, st); break;
            case W_Q8_0: gemv_dispatch<W_Q8_0, true>(W, 0, F, F, x, ldx, T, u, ldu, EPI_STORE, st); break;
        }
        return;
    }
    launch_linear(W, 0, 2 * (int64_t)F, x, ldx, T, tmp, 2 * F, EPI_STORE, st);
    launch_swiglu(tmp, T, F, u, st);
}

}  // namespace llm
