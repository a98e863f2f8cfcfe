// Grouped-query attention over the KV cache ([P2] "llama.cpp Architecture", Example 4:
// FLASH_ATTN_EXT of the 8 query heads over the cached keys and values; Example 11: the unfused
// meaning MUL_MAT(K, Q) -> SOFT_MAX with the mask -> MUL_MAT with V).
//
// Work decomposition (built on the host): the ubatch's tokens are grouped by the list of cells
// they may read (one list per distinct sequence set), cut into query tiles of up to TQ tokens,
// and each tile's list is cut into work items (split-K over the cache). A block handles one work
// item for one KV head: the TQ x G query rows of that head group share every K/V row it stages
// in shared memory, so each cached row is read once per tile rather than once per query head.
// The softmax is online (running max and sum per row, base-2 exponent with log2(e)/sqrt(hd)
// folded into Q); a cell is visible to a row iff cell.pos <= token.pos. Partial (o, m, l) per
// work item are merged by the combine kernel.
#include <cuda_fp16.h>

#include <cfloat>
#include <climits>
#include <cmath>

#include "kernels.h"

namespace llm {

namespace {

constexpr int kAttnWarps = 4;
constexpr int kBC = 32;                  // cells per shared-memory tile (one per lane)

template <typename KT> __device__ __forceinline__ float kv_to_f(KT v);
template <> __device__ __forceinline__ float kv_to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float kv_to_f<__half>(__half v) { return __half2float(v); }

template <int HD, int TQ, int G>
struct AttnSmem {
    static constexpr int R = TQ * G;
    static constexpr int RW = (R + kAttnWarps - 1) / kAttnWarps;
    static constexpr size_t q_floats = (size_t)R * HD;
    static constexpr size_t k_floats = (size_t)kBC * (HD + 1);
    static constexpr size_t v_floats = (size_t)kBC * HD;
    static constexpr size_t p_floats = (size_t)kAttnWarps * RW * kBC;
    static constexpr size_t bytes = (q_floats + k_floats + v_floats + p_floats) * sizeof(float) +
                                    (size_t)(kBC + R) * sizeof(int);
};

template <int HD, int TQ, int G, typename KT>
__global__ void __launch_bounds__(kAttnWarps * 32)
attn_partial_kernel(AttnArgs a, float scale_log2) {
    using SM = AttnSmem<HD, TQ, G>;
    constexpr int R = SM::R, RW = SM::RW, DPL = HD / 32;
    extern __shared__ float smem[];
    float* qs = smem;                              // [R][HD]
    float* ks = qs + SM::q_floats;                 // [kBC][HD + 1]
    float* vs = ks + SM::k_floats;                 // [kBC][HD]
    float* ps = vs + SM::v_floats;                 // [warps][RW][kBC]
    int* cpos = reinterpret_cast<int*>(ps + SM::p_floats);   // [kBC]
    int* rpos = cpos + kBC;                        // [R]

    const int wi = blockIdx.x, kvh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = a.wi_tile[wi];
    const int list = a.tile_list[tile];
    const int nq = a.tile_nq[tile];
    const int s0 = a.tile_start[tile];
    const int c0 = a.wi_c0[wi], c1 = a.wi_c1[wi];
    const int base = a.list_off[list];
    const KT* K = static_cast<const KT*>(a.kc) + (int64_t)kvh * a.n_ctx * HD;
    const KT* V = static_cast<const KT*>(a.vc) + (int64_t)kvh * a.n_ctx * HD;

    for (int idx = threadIdx.x; idx < R * HD; idx += blockDim.x) {
        const int r = idx / HD, d = idx % HD;
        const int j = r / G, g = r % G;
        float v = 0.f;
        if (j < nq) {
            const int t = a.perm[s0 + j];
            v = a.q[(int64_t)t * a.ldq + (kvh * G + g) * HD + d] * scale_log2;
        }
        qs[idx] = v;
    }
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int j = r / G;
        rpos[r] = j < nq ? a.tok_pos[a.perm[s0 + j]] : -1;
    }

    float m[RW], l[RW], o[RW][DPL];
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[i][e] = 0.f;
    }

    for (int cb = c0; cb < c1; cb += kBC) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kBC * HD; idx += blockDim.x) {
            const int c = idx / HD, d = idx % HD;
            float kv = 0.f, vv = 0.f;
            if (cb + c < c1) {
                const int64_t cell = a.list_cells[base + cb + c];
                kv = kv_to_f<KT>(K[cell * HD + d]);
                vv = kv_to_f<KT>(V[cell * HD + d]);
            }
            ks[c * (HD + 1) + d] = kv;
            vs[c * HD + d] = vv;
        }
        for (int c = threadIdx.x; c < kBC; c += blockDim.x)
            cpos[c] = (cb + c < c1) ? a.list_pos[base + cb + c] : INT_MAX;
        __syncthreads();

        const int mypos = cpos[lane];
        float* pw = ps + (size_t)warp * RW * kBC;
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const int r = warp * RW + i;
            float s = -INFINITY;
            if (r < R && mypos <= rpos[r]) {
                const float* qr = qs + r * HD;
                const float* kr = ks + lane * (HD + 1);
                float acc = 0.f;
#pragma unroll 8
                for (int d = 0; d < HD; ++d) acc = fmaf(qr[d], kr[d], acc);
                s = acc;
            }
            float mx = s;
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[i], mx);
            float p = 0.f, corr = 1.f;
            if (m_new != -INFINITY) {
                corr = exp2f(m[i] - m_new);
                p = exp2f(s - m_new);
            }
            float ssum = p;
            for (int off = 16; off > 0; off >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
            l[i] = l[i] * corr + ssum;
            m[i] = m_new;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[i][e] *= corr;
            pw[i * kBC + lane] = p;
        }
        __syncwarp();
#pragma unroll 4
        for (int c = 0; c < kBC; ++c) {
            float vv[DPL];
#pragma unroll
            for (int e = 0; e < DPL; ++e) vv[e] = vs[c * HD + lane + 32 * e];
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                const float p = pw[i * kBC + c];
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[i][e] = fmaf(p, vv[e], o[i][e]);
            }
        }
    }

    const int row0 = a.wi_row_off[wi];
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        const int r = warp * RW + i;
        if (r >= nq * G) continue;
        const int64_t row = (int64_t)(row0 + r) * a.Hkv + kvh;
        if (lane == 0) {
            a.part_m[row] = m[i];
            a.part_l[row] = l[i];
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) a.part_o[row * HD + lane + 32 * e] = o[i][e];
    }
}

template <int HD, int G>
__global__ void attn_combine_kernel(AttnArgs a) {
    const int tile = blockIdx.x, kvh = blockIdx.y;
    const int w0 = a.tile_wi_off[tile], w1 = a.tile_wi_off[tile + 1];
    const int nq = a.tile_nq[tile], s0 = a.tile_start[tile];
    for (int idx = threadIdx.x; idx < nq * G * HD; idx += blockDim.x) {
        const int r = idx / HD, d = idx % HD;
        float M = -INFINITY;
        for (int w = w0; w < w1; ++w)
            M = fmaxf(M, a.part_m[(int64_t)(a.wi_row_off[w] + r) * a.Hkv + kvh]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int w = w0; w < w1; ++w) {
                const int64_t row = (int64_t)(a.wi_row_off[w] + r) * a.Hkv + kvh;
                const float mw = a.part_m[row];
                if (mw == -INFINITY) continue;
                const float f = exp2f(mw - M);
                L += f * a.part_l[row];
                O += f * a.part_o[row * HD + d];
            }
        }
        const int t = a.perm[s0 + r / G];
        const int h = kvh * G + r % G;
        a.out[(int64_t)t * a.ldo + h * HD + d] = L > 0.f ? O / L : 0.f;
    }
}

template <int HD, int TQ, int G>
bool launch_partial(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    const size_t smem = AttnSmem<HD, TQ, G>::bytes;
    dim3 grid(a.n_work, a.Hkv);
    if (a.kv_type == W_F32) {
        auto k = attn_partial_kernel<HD, TQ, G, float>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k<<<grid, kAttnWarps * 32, smem, st>>>(a, scale_log2);
    } else {
        auto k = attn_partial_kernel<HD, TQ, G, __half>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        k<<<grid, kAttnWarps * 32, smem, st>>>(a, scale_log2);
    }
    attn_combine_kernel<HD, G><<<dim3(a.n_tiles, a.Hkv), 128, 0, st>>>(a);
    return true;
}

template <int HD, int G>
bool launch_hd_g(const AttnArgs& a, cudaStream_t st) {
    if (a.max_nq <= 1) return launch_partial<HD, 1, G>(a, st);
    return launch_partial<HD, kAttnTileQ, G>(a, st);
}

}  // namespace

bool launch_attention(const AttnArgs& a, cudaStream_t st) {
    if (a.n_work <= 0) return true;
    const int G = a.H / a.Hkv;
    if (G != 4) return false;
    switch (a.hd) {
        case 32: return launch_hd_g<32, 4>(a, st);
        case 64: return launch_hd_g<64, 4>(a, st);
        case 128: return launch_hd_g<128, 4>(a, st);
    }
    return false;
}

}  // namespace llm
