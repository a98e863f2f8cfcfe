// Small kernels of the decode path: embedding gather with the RoPE table, RMSNorm, RoPE + K/V append,
// SwiGLU, greedy argmax and the Q8_0 block split.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <climits>

#include "dev_common.cuh"
#include "kernels.h"

namespace llm {

namespace {

using dev::load_elem;
using dev::rope_cos_sin;

__device__ __forceinline__ float block_sum(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    const int nw = (blockDim.x + 31) >> 5;
    v = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
    if (w == 0)
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
    __syncthreads();
    v = red[0];
    __syncthreads();
    return v;
}

__device__ __forceinline__ void store_out(float* y, int64_t i, float v) { y[i] = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* y, int64_t i, float v) {
    y[i] = __float2bfloat16_rn(v);
}
__device__ __forceinline__ void store_out(__half* y, int64_t i, float v) { y[i] = __float2half_rn(v); }

template <typename OT>
__global__ void rmsnorm_kernel(const float* __restrict__ x, const int32_t* __restrict__ rows,
                               int d, const float* __restrict__ g, float eps,
                               OT* __restrict__ y, __nv_bfloat16* __restrict__ ylo) {
    __shared__ float red[32];
    const int r = blockIdx.x;
    const int src = rows ? rows[r] : r;
    const float* xr = x + (int64_t)src * d;
    float ss = 0.f;
    for (int j = threadIdx.x; j < d; j += blockDim.x) ss += xr[j] * xr[j];
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    for (int j = threadIdx.x; j < d; j += blockDim.x) {
        const float v = xr[j] * inv * g[j];
        store_out(y, (int64_t)r * d + j, v);
        if (ylo) {
            const float hi = __bfloat162float(__float2bfloat16_rn(v));
            ylo[(int64_t)r * d + j] = __float2bfloat16_rn(v - hi);
        }
    }
}

// The same for rows of d = 1024 * NV values and an f16 output: 256 threads, each holding NV float4
// of the row in registers, so the row is read once.
template <int NV>
__global__ void __launch_bounds__(256) rmsnorm_f16_vec_kernel(const float* __restrict__ x,
                                                             const int32_t* __restrict__ rows, int d,
                                                             const float* __restrict__ g, float eps,
                                                             __half* __restrict__ y) {
    __shared__ float red[32];
    // launched with programmatic dependent launch: x comes from the kernel before
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    const int r = blockIdx.x;
    const int src = rows ? rows[r] : r;
    const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)src * d);
    float4 v[NV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        v[i] = xr[i * 256 + threadIdx.x];
        ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    uint2* yr = reinterpret_cast<uint2*>(y + (int64_t)r * d);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const float4 gg = g4[i * 256 + threadIdx.x];
        const __half2 a = __floats2half2_rn(v[i].x * inv * gg.x, v[i].y * inv * gg.y);
        const __half2 b = __floats2half2_rn(v[i].z * inv * gg.z, v[i].w * inv * gg.w);
        yr[i * 256 + threadIdx.x] = make_uint2(*reinterpret_cast<const uint32_t*>(&a),
                                               *reinterpret_cast<const uint32_t*>(&b));
    }
}

template <typename KT>
__device__ __forceinline__ KT to_kv(float v);
template <>
__device__ __forceinline__ float to_kv<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half to_kv<__half>(float v) { return __float2half_rn(v); }

template <typename KT>
__global__ void rope_kv_append_kernel(float* __restrict__ qkv, int H, int Hkv, int hd,
                                      const float2* __restrict__ cs,
                                      const int32_t* __restrict__ slot, KT* __restrict__ kc,
                                      KT* __restrict__ vc, int n_ctx, uint32_t* err) {
    const int t = blockIdx.x;
    const int half = hd / 2;
    const int width = (H + 2 * Hkv) * hd;
    float* row = qkv + (int64_t)t * width;
    const int32_t c = slot ? slot[t] : t;
    const bool ok = c >= 0 && c < n_ctx;
    if (!ok && threadIdx.x == 0) atomicOr(err, ERR_SLOT_RANGE);
    const float2* cst = cs + (int64_t)t * half;
    const int npairs = (H + Hkv) * half;
    for (int j = threadIdx.x; j < npairs; j += blockDim.x) {
        const int head = j / half, i = j % half;
        float2* p = reinterpret_cast<float2*>(row + head * hd + 2 * i);
        const float2 xv = *p;
        const float2 e = cst[i];
        const float y0 = xv.x * e.x - xv.y * e.y;
        const float y1 = xv.x * e.y + xv.y * e.x;
        if (head < H) {
            *p = make_float2(y0, y1);
        } else if (ok) {
            KT* dst = kc + ((int64_t)(head - H) * n_ctx + c) * hd + 2 * i;
            dst[0] = to_kv<KT>(y0);
            dst[1] = to_kv<KT>(y1);
        }
    }
    if (!ok) return;
    const float2* v = reinterpret_cast<const float2*>(row + (H + Hkv) * hd);
    for (int j = threadIdx.x; j < Hkv * hd / 2; j += blockDim.x) {
        const int g = (2 * j) / hd, d = (2 * j) % hd;
        const float2 vv = v[j];
        KT* dst = vc + ((int64_t)g * n_ctx + c) * hd + d;
        dst[0] = to_kv<KT>(vv.x);
        dst[1] = to_kv<KT>(vv.y);
    }
}

// One warp per 32-value block; blockIdx.y = token, blockIdx.z = 0 for K, 1 for V.
__global__ void kv_quant_q8_kernel(const float* __restrict__ sk, const float* __restrict__ sv, int ld,
                                   int Hkv, int hd, const int32_t* __restrict__ slot,
                                   int8_t* __restrict__ kc, int8_t* __restrict__ vc, int n_ctx,
                                   uint32_t* err) {
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    const int nb = hd / 32;
    const int blk = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.y;
    const bool is_v = blockIdx.z != 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (blk >= Hkv * nb) return;                                  // whole warp
    const int g = blk / nb, b = blk % nb;
    const int32_t cell = slot[t];
    if (cell < 0 || cell >= n_ctx) {
        if (lane == 0 && b == 0 && g == 0 && !is_v) atomicOr(err, ERR_SLOT_RANGE);
        return;
    }
    const float x = (is_v ? sv : sk)[((int64_t)g * ld + t) * hd + b * 32 + lane];
    float amax = fabsf(x);
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = d != 0.0f ? __frcp_rn(d) : 0.0f;
    const float qf = roundf(__fmul_rn(x, id));                    // halves away from zero
    int8_t* q = is_v ? vc : kc;
    q[((int64_t)g * n_ctx + cell) * hd + b * 32 + lane] = (int8_t)(int)qf;
    if (lane == 0) {
        __half* s = reinterpret_cast<__half*>(q + kv_q8_scale_offset(Hkv, n_ctx, hd));
        s[((int64_t)g * n_ctx + cell) * nb + b] = __float2half_rn(d);
    }
}

// One thread per 8 values of a cell row: an 8-byte load of quants, one 16-byte store of f16.
__global__ void kv_q8_to_f16_kernel(const int8_t* __restrict__ kc, const int8_t* __restrict__ vc,
                                    __half* __restrict__ out, int Hkv, int n_ctx, int hd,
                                    const int32_t* __restrict__ n_kv) {
    const int upr = hd / 8;
    const int64_t n = (int64_t)Hkv * n_ctx * upr;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int64_t row = i / upr;                                  // g * n_ctx + cell
    if ((int)(row % n_ctx) >= __ldg(n_kv)) return;
    const int j = (int)(i % upr);
    const bool is_v = blockIdx.y != 0;
    const int8_t* q = is_v ? vc : kc;
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + row * hd + j * 8));
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t src = k < 2 ? raw.x : raw.y;
        const int sh = (k & 1) * 16;
        const float a = (float)(int8_t)((src >> sh) & 0xffu), b = (float)(int8_t)((src >> (sh + 8)) & 0xffu);
        const __half2 h = __floats2half2_rn(a, b);
        w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    __half* o = out + (is_v ? (int64_t)Hkv * n_ctx * hd : 0) + row * hd + j * 8;
    *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename U>
__global__ void kv_gather_kernel(const U* __restrict__ src, U* __restrict__ dst,
                                 const int32_t* __restrict__ order, int n, int n_src, int upr) {
    const int g = blockIdx.y;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)n * upr) return;
    const int r = (int)(i / upr), u = (int)(i % upr);
    const int o = order[r];
    dst[((int64_t)g * n + r) * upr + u] = o >= 0 ? src[((int64_t)g * n_src + o) * upr + u] : U{};
}

__global__ void bf16_to_f16_kernel(const __nv_bfloat16* __restrict__ x, int64_t n, __half* __restrict__ y) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = __float2half_rn(__bfloat162float(x[i]));
}

__global__ void swiglu_kernel(const float* __restrict__ gu, int64_t T, int F,
                              float* __restrict__ u) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= T * F) return;
    const int64_t t = idx / F, j = idx % F;
    const float g = gu[t * 2 * F + j];
    const float up = gu[t * 2 * F + F + j];
    u[idx] = g / (1.0f + expf(-g)) * up;
}

__device__ __forceinline__ unsigned long long pack_max(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

__global__ void embed_rope_kernel(DevMat E, const int32_t* __restrict__ tok,
                                  const int32_t* __restrict__ pos, int half,
                                  const double* __restrict__ theta, float* __restrict__ x,
                                  float2* __restrict__ cs, unsigned long long* __restrict__ amax,
                                  int n_amax, uint32_t* err) {
    const int t = blockIdx.x;
    const int32_t id = tok[t];
    const bool ok = id >= 0 && id < E.rows;
    if (!ok && threadIdx.x == 0) atomicOr(err, ERR_TOKEN_RANGE);
    for (int64_t j = threadIdx.x; j < E.cols; j += blockDim.x)
        x[(int64_t)t * E.cols + j] = ok ? load_elem(E, id, j) : 0.f;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        cs[(int64_t)t * half + i] = rope_cos_sin(pos[t], theta[i]);
    }
    if (t == 0)
        for (int i = threadIdx.x; i < n_amax; i += blockDim.x) amax[i] = 0ull;
}

__global__ void argmax_kernel(const float* __restrict__ logits, int V,
                              unsigned long long* __restrict__ out) {
    __shared__ float sv[32];
    __shared__ int si[32];
    const float* row = logits + (int64_t)blockIdx.x * V;
    float best = -INFINITY;
    int bi = INT_MAX;
    for (int j = threadIdx.x; j < V; j += blockDim.x) {
        const float v = row[j];
        if (v > best || (v == best && j < bi)) { best = v; bi = j; }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { sv[w] = best; si[w] = bi; }
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        best = l < nw ? sv[l] : -INFINITY;
        bi = l < nw ? si[l] : INT_MAX;
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
        }
        if (l == 0) out[blockIdx.x] = bi == INT_MAX ? 0ull : pack_max(best, bi);
    }
}

__global__ void q8_0_unpack_kernel(const uint8_t* __restrict__ blocks, int64_t nblocks,
                                   int64_t bpr, int8_t* __restrict__ q, __half* __restrict__ d) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblocks) return;
    const uint8_t* src = blocks + b * 34;
    const uint16_t bits = (uint16_t)src[0] | ((uint16_t)src[1] << 8);
    d[b] = __ushort_as_half(bits);
    const int64_t row = b / bpr, kb = b % bpr;
    int8_t* dst = q + row * bpr * 32 + kb * 32;
#pragma unroll
    for (int i = 0; i < 32; ++i) dst[i] = (int8_t)src[2 + i];
}

}  // namespace

void launch_rmsnorm(const float* x, const int32_t* rows, int32_t R, int32_t d, const float* g,
                    float eps, float* y, cudaStream_t st) {
    if (R <= 0) return;
    rmsnorm_kernel<float><<<R, d >= 1024 ? 512 : 256, 0, st>>>(x, rows, d, g, eps, y, nullptr);
}

void launch_rmsnorm_bf16(const float* x, const int32_t* rows, int32_t R, int32_t d,
                         const float* g, float eps, void* yb, void* yb_lo, cudaStream_t st) {
    if (R <= 0) return;
    rmsnorm_kernel<__nv_bfloat16><<<R, d >= 1024 ? 512 : 256, 0, st>>>(
        x, rows, d, g, eps, static_cast<__nv_bfloat16*>(yb), static_cast<__nv_bfloat16*>(yb_lo));
}

void launch_rope_kv_append(float* qkv, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                           const float2* cs, const int32_t* slot, void* kc, void* vc,
                           int32_t n_ctx, int32_t kv_type, uint32_t* err, cudaStream_t st) {
    if (T <= 0) return;
    if (kv_type == W_F32)
        rope_kv_append_kernel<float><<<T, 256, 0, st>>>(qkv, H, Hkv, hd, cs, slot, (float*)kc,
                                                       (float*)vc, n_ctx, err);
    else
        rope_kv_append_kernel<__half><<<T, 256, 0, st>>>(qkv, H, Hkv, hd, cs, slot, (__half*)kc,
                                                        (__half*)vc, n_ctx, err);
}

void launch_kv_quant_q8(const float* sk, const float* sv, int32_t ld, int32_t T, int32_t Hkv,
                        int32_t hd, const int32_t* slot, void* kc, void* vc, int32_t n_ctx,
                        uint32_t* err, cudaStream_t st, bool pdl) {
    if (T <= 0) return;
    constexpr int kWarps = 8;
    const int nblk = Hkv * (hd / 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((nblk + kWarps - 1) / kWarps), (unsigned)T, 2);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, kv_quant_q8_kernel, sk, sv, (int)ld, (int)Hkv, (int)hd, slot,
                       static_cast<int8_t*>(kc), static_cast<int8_t*>(vc), (int)n_ctx, err);
}

void launch_kv_q8_to_f16(const void* kc, const void* vc, void* out, int32_t Hkv, int32_t n_ctx,
                         int32_t hd, const int32_t* n_kv, cudaStream_t st) {
    const int64_t n = (int64_t)Hkv * n_ctx * (hd / 8);
    if (n <= 0) return;
    const dim3 grid((unsigned)((n + 255) / 256), 2);
    kv_q8_to_f16_kernel<<<grid, 256, 0, st>>>(static_cast<const int8_t*>(kc), static_cast<const int8_t*>(vc),
                                              static_cast<__half*>(out), (int)Hkv, (int)n_ctx, (int)hd, n_kv);
}

void launch_kv_gather(const void* src, void* dst, const int32_t* order, int32_t n, int32_t n_head,
                      int32_t n_src, int32_t row_bytes, cudaStream_t st) {
    if (n <= 0) return;
    if (row_bytes % 16 == 0) {
        const int upr = row_bytes / 16;
        const dim3 grid((unsigned)(((int64_t)n * upr + 255) / 256), (unsigned)n_head);
        kv_gather_kernel<uint4><<<grid, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                      order, n, n_src, upr);
    } else {
        const int upr = row_bytes / 2;
        const dim3 grid((unsigned)(((int64_t)n * upr + 255) / 256), (unsigned)n_head);
        kv_gather_kernel<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(src),
                                                         static_cast<uint16_t*>(dst), order, n, n_src, upr);
    }
}

void launch_rmsnorm_f16(const float* x, const int32_t* rows, int32_t R, int32_t d, const float* g,
                        float eps, void* yh, cudaStream_t st, bool pdl) {
    if (R <= 0) return;
    __half* y = static_cast<__half*>(yh);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(R);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (d) {
        case 1024: cudaLaunchKernelEx(&cfg, rmsnorm_f16_vec_kernel<1>, x, rows, d, g, eps, y); return;
        case 2048: cudaLaunchKernelEx(&cfg, rmsnorm_f16_vec_kernel<2>, x, rows, d, g, eps, y); return;
        case 4096: cudaLaunchKernelEx(&cfg, rmsnorm_f16_vec_kernel<4>, x, rows, d, g, eps, y); return;
        case 8192: cudaLaunchKernelEx(&cfg, rmsnorm_f16_vec_kernel<8>, x, rows, d, g, eps, y); return;
    }
    rmsnorm_kernel<__half><<<R, d >= 1024 ? 512 : 256, 0, st>>>(x, rows, d, g, eps, y, nullptr);
}

void launch_bf16_to_f16(const void* x, int64_t n, void* y, cudaStream_t st) {
    if (n <= 0) return;
    bf16_to_f16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), n,
                                                                     static_cast<__half*>(y));
}

void launch_swiglu(const float* gu, int32_t T, int32_t F, float* u, cudaStream_t st) {
    const int64_t n = (int64_t)T * F;
    if (n <= 0) return;
    swiglu_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(gu, T, F, u);
}

void launch_argmax(const float* logits, int32_t R, int32_t V, unsigned long long* amax,
                   cudaStream_t st) {
    if (R <= 0) return;
    argmax_kernel<<<R, 1024, 0, st>>>(logits, V, amax);
}

void launch_embed_rope(const DevMat& E, const int32_t* tok, const int32_t* pos, int32_t T,
                       int32_t hd, const double* theta, float* x, float2* cs,
                       unsigned long long* amax, int32_t n_amax, uint32_t* err, cudaStream_t st) {
    if (T <= 0) return;
    embed_rope_kernel<<<T, 256, 0, st>>>(E, tok, pos, hd / 2, theta, x, cs, amax, n_amax, err);
}

void launch_q8_0_unpack(const uint8_t* blocks, int64_t rows, int64_t cols, int8_t* q, __half* d,
                        cudaStream_t st) {
    const int64_t nb = rows * (cols / 32);
    if (nb <= 0) return;
    q8_0_unpack_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, st>>>(blocks, nb, cols / 32, q, d);
}

}  // namespace llm
