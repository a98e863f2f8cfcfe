// Tensor-core (tcgen05 + TMA + TMEM) BF16 GEMM for prefill ubatches. See gemm_tc.cu.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace llm {

enum GemmEpi : int32_t {
    GEMM_EPI_STORE = 0,    // Y[t][m] = acc (float32)
    GEMM_EPI_ADD = 1,      // Y[t][m] += acc (float32, the residual add)
    GEMM_EPI_SWIGLU = 2,   // Y[t][j] = silu(gate_j) * up_j (bf16); W rows [0,F) gate, [F,2F) up
    GEMM_EPI_QKV = 3,      // the fused Q/K/V projection's outputs: RoPE, K/V rows to the cache (TnQkv)
};

// The Q/K/V epilogue of the token-major GEMM with f16 operands ([P2] "llama.cpp Architecture",
// Example 4: ROPE of Q and K, SET_ROWS of K and V into the layer's cache): columns [0, H hd) are
// Q, stored rotated (float32) into Y; [H hd, (H + Hkv) hd) are K and the rest V, rotated (K) and
// rounded to f16 into their cache rows. Needs 256 % hd == 0 and H hd, Hkv hd multiples of 256.
struct TnQkv {
    const float2* cs = nullptr;      // [T][hd / 2] cos, sin of each token's angle per pair
    const int32_t* slot = nullptr;   // [T] cache cell of each token (checked against n_ctx)
    void* kc = nullptr;              // f16 [Hkv][n_ctx][hd]
    void* vc = nullptr;
    int n_ctx = 0, H = 0, Hkv = 0, hd = 0;
};

// TMA map of a row-major bf16 (or, with f16, float16) matrix [rows][cols] (cols % 64 == 0, base
// 16-byte aligned), loaded in boxes of 64 columns x box_rows rows with the 128-byte swizzle.
bool tc_make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows,
                 bool f16 = false);

// Token tile the launcher uses for T tokens (the activation map's box height must match).
int tc_token_tile(int T);

// Whether the tensor-core path supports a weight of M rows (or F gate/up rows) by K columns.
bool tc_shape_ok(int64_t M, int64_t K, int epi, int64_t F);

// Y (op)= X W^T for T tokens: wmap over W [rows][K] (box 128 rows, or 64 for SWIGLU), xmap over
// X [>= T rows][K] bf16 (box rows = tc_token_tile(T)). With xmap_lo (box rows 128) the activations
// are X = hi + lo, two bf16 terms both multiplied into the accumulator; SWIGLU then also writes
// the low term of its bf16 output to Y2. Returns false on a launch failure.
bool launch_gemm_tc(const CUtensorMap& wmap, const CUtensorMap& xmap, int epi, int K, int M,
                    int T, int F, void* Y, int ldy, uint32_t* err, cudaStream_t st,
                    const CUtensorMap* xmap_lo = nullptr, void* Y2 = nullptr);

// Gate/up + SwiGLU with the token tile as the MMA's A operand (128 tokens, two bf16 terms: xmap and
// xmap_lo, box 128 rows) and 128 gate + 128 up rows as B (wmap over the [2F][K] gate|up matrix,
// box 128 rows): Y, Y2 [>= T][ldy] bf16 hi and lo terms of silu(gate) * up. F % 128 == 0.
// Without xmap_lo, activations and weights are f16 (one term each; maps made with f16) and Y
// receives a single f16 output.
bool tc_swiglu_tn_ok(int64_t K, int64_t F);
// With wmap_lo the weights are two bf16 terms as well (hi in wmap, lo in wmap_lo; a Q8_0 weight
// d*q split so that hi + lo holds it to 16 bits): four products per k-step instead of two.
// With f16 operands and more than 128 tokens the two-CTA kernel (tcgen05 cta_group::2, 256-token
// tiles) runs unless one_cta is set.
bool launch_gemm_swiglu_tn(const CUtensorMap& xmap, const CUtensorMap* xmap_lo, const CUtensorMap& wmap,
                           int K, int T, int F, void* Y, void* Y2, int ldy, uint32_t* err, cudaStream_t st,
                           const CUtensorMap* wmap_lo = nullptr, bool one_cta = false,
                           const CUtensorMap* ymap = nullptr, bool pdl = false, const uint32_t* q8_scales = nullptr);

// Store / residual add with the token tile as A (two bf16 terms) and 256 weight rows as B (wmap
// over W [M][K], box 128 rows): Y [>= T][ldy] float32 (op)= X W^T. M % 256 == 0. splits > 1
// splits K over blockIdx.z with vector atomic adds (or, with ymap, bulk reduce-adds) into Y (a
// store then needs Y zeroed first).
// Without xmap_lo: f16 activations and weights, one term each.
bool tc_tn_ok(int64_t M, int64_t K);
int tc_tn_splits(int64_t M, int64_t K, int T, int n_sm);
bool launch_gemm_tn(const CUtensorMap& xmap, const CUtensorMap* xmap_lo, const CUtensorMap& wmap, int epi,
                    int K, int M, int T, float* Y, int ldy, int splits, uint32_t* err, cudaStream_t st,
                    const CUtensorMap* wmap_lo = nullptr, bool one_cta = false,
                    const CUtensorMap* ymap = nullptr, const TnQkv* qkv = nullptr, bool pdl = false,
                    const uint32_t* q8_scales = nullptr);
// pdl: launched with programmatic dependent launch (the kernel requests its first weight tiles
// before it waits for the kernel before it to end).
// q8_scales: the weight is Q8_0, wmap its quants (tc_make_map_q8) and q8_scales its fp16 block
// scales in the per-k-step layout of q8_scales_by_kstep; the two-CTA kernel dequantises each
// k-step into exact f16 terms in shared memory (f16 activations, no wmap_lo; any token count).
// The quant map of a Q8_0 weight [rows][cols] int8: boxes of 64 quants x box_rows rows (128; 64 for
// the gate|up matrix of the SwiGLU epilogue), 64-byte swizzle.
bool tc_make_map_q8(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows);
// The fp16 block scales of a Q8_0 weight, s [rows][K / 32], in the layout the Q8_0 GEMM copies per
// k-step: out[kb][row] = the row's two scales of values 64 kb .. 64 kb + 63 (low half first), so
// the scales of 128 consecutive rows of one k-step are 512 contiguous bytes. K % 64 == 0; rows a
// multiple of 4.
void q8_scales_by_kstep(const __half* s, int64_t rows, int64_t K, uint32_t* out, cudaStream_t st);
// Whether the Q/K/V epilogue serves these head counts (f16 operands, ymap given, one K split).
bool tc_tn_qkv_ok(int H, int Hkv, int hd);

// Tensor map of a kernel's output [rows][cols] (float32, or f16 with f16) for the TMA-store
// epilogue of the token-major GEMM with f16 operands: boxes of 128 bytes x 32 rows, 128-byte
// swizzle. Pass it as ymap: the epilogue then stages each warp's rows in shared memory and
// writes them with bulk tensor stores (the residual add and K splits as reduce-adds).
bool tc_make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, bool f16);

// The two-CTA kernel with a timeline: 8 global-timer stamps per CTA in trace (see gemm_tc.cu), for
// tc_tn2_blocks(...) CTAs. Returns false for T <= 128 or a launch failure.
bool launch_gemm_tn2_traced(const CUtensorMap& xmap, const CUtensorMap& wmap, int epi, int K, int M, int T,
                            int F, void* Y, int ldy, int splits, uint32_t* err, cudaStream_t st,
                            const CUtensorMap* ymap, uint64_t* trace);
int tc_tn2_blocks(int epi, int M, int T, int F, int splits);
// The Q8_0 two-CTA kernel with per-CTA wait and conversion counters (8 values per CTA in trace,
// see gemm_tc.cu), for tc_tn2_blocks(...) CTAs.
bool launch_gemm_tn2q8_traced(const CUtensorMap& xmap, const CUtensorMap& qmap, const uint32_t* scales, int epi,
                              int K, int M, int T, int F, void* Y, int ldy, int splits, uint32_t* err,
                              cudaStream_t st, const CUtensorMap* ymap, uint64_t* trace);

}  // namespace llm
