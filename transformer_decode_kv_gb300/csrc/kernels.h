// Launchers of the decode path's CUDA kernels (sm_103a). All pointers are device pointers; every
// launcher enqueues on `st` and returns immediately.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>

namespace llm {

enum WType : int32_t { W_F32 = 0, W_F16 = 1, W_BF16 = 2, W_Q8_0 = 8 };

// A weight matrix in the device store: `rows` rows of `cols` values, row-major. Q8_0 is kept as
// int8 quants [rows][cols] plus fp16 scales [rows][cols / 32] (the same bytes as the file's
// 34-byte blocks, split so each part can be read with aligned vector loads).
struct DevMat {
    int32_t type = -1;
    int64_t rows = 0, cols = 0;
    void* data = nullptr;
    __half* scales = nullptr;
};

// Device error word bits, set by kernels' own bounds checks.
enum : uint32_t { ERR_SLOT_RANGE = 1u, ERR_TOKEN_RANGE = 2u, ERR_ROW_RANGE = 4u, ERR_TIMEOUT = 8u };

// ---- elementwise / small kernels (kernels_misc.cu) --------------------------------------------
// y[r] = x[rows ? rows[r] : r] / sqrt(mean(x^2) + eps) * g, r < R, width d (RMS_NORM + MUL).
void launch_rmsnorm(const float* x, const int32_t* rows, int32_t R, int32_t d, const float* g,
                    float eps, float* y, cudaStream_t st);
// The same with a bf16 output (the A/B operand of a tensor-core GEMM).
// yb_lo (optional) receives the low bf16 term: y = yb + yb_lo to about 16 bits.
void launch_rmsnorm_bf16(const float* x, const int32_t* rows, int32_t R, int32_t d,
                         const float* g, float eps, void* yb, void* yb_lo, cudaStream_t st);
// RoPE (adjacent pairs) on the q and k parts of qkv [T][(H + 2 Hkv) hd] (q in place), then K and
// V rows written to their cache cells slot[t] ([P2] Example 4, ROPE + SET_ROWS). Cache layout:
// [Hkv][n_ctx][hd], element type kv_type (F32 or F16). A slot outside [0, n_ctx) skips the write
// and sets ERR_SLOT_RANGE.
void launch_rope_kv_append(float* qkv, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                           const float2* cs, const int32_t* slot, void* kc, void* vc,
                           int32_t n_ctx, int32_t kv_type, uint32_t* err, cudaStream_t st);
// With slot == nullptr token t's rows go to cell t (a float32 staging area of n_ctx rows per
// head, from which launch_kv_quant_q8 fills a Q8_0 cache).
// Q8_0 cache rows from float32 staging rows sk / sv [Hkv][ld][hd] (token t at row t of each
// head): per 32-value block d = max|x| / 127, q = x * (1 / d) rounded half away from zero, all in
// float32, d stored as fp16 ([P2] Example 2 block: fp16 scale and 32 int8 quants, value d * q).
// The Q8_0 cache of one layer: int8 quants [Hkv][n_ctx][hd], then fp16 scales
// [Hkv][n_ctx][hd / 32] (kv_q8_scale_offset bytes after the quants). A slot outside [0, n_ctx)
// skips the write and sets ERR_SLOT_RANGE. With pdl the kernel may start while the previous one
// runs and waits for it before reading the staging rows.
void launch_kv_quant_q8(const float* sk, const float* sv, int32_t ld, int32_t T, int32_t Hkv,
                        int32_t hd, const int32_t* slot, void* kc, void* vc, int32_t n_ctx,
                        uint32_t* err, cudaStream_t st, bool pdl);
__host__ __device__ inline size_t kv_q8_scale_offset(int32_t Hkv, int32_t n_ctx, int32_t hd) {
    return (size_t)Hkv * (size_t)n_ctx * (size_t)hd;
}
// The int8 quants of every cell below *n_kv (a device word) of one layer's Q8_0 K and V caches as
// f16 (exact) into out = [2][Hkv][n_ctx][hd] (K then V, the F16 cache layout): the tensor-core
// prefill tiles read a Q8_0 cache through this copy and apply the fp16 scales of the cache
// themselves. Cells at or above *n_kv are not written.
void launch_kv_q8_to_f16(const void* kc, const void* vc, void* out, int32_t Hkv, int32_t n_ctx,
                         int32_t hd, const int32_t* n_kv, cudaStream_t st);
// dst[g][i] = src[g][order[i]] for g < n_head (grid y), i < n (zero where order[i] < 0): rows of
// row_bytes (a multiple of 2), src rows strided by n_src rows per head, dst rows packed n per
// head. Used by the defrag to gather one cache region in the new cell order.
void launch_kv_gather(const void* src, void* dst, const int32_t* order, int32_t n, int32_t n_head,
                      int32_t n_src, int32_t row_bytes, cudaStream_t st);
// The same with a single f16 output (the prefill GEMMs' f16 operand); pdl: launched with
// programmatic dependent launch after the kernel that writes x (d of 1024 to 8192).
void launch_rmsnorm_f16(const float* x, const int32_t* rows, int32_t R, int32_t d, const float* g,
                        float eps, void* yh, cudaStream_t st, bool pdl = false);
// y[i] = f16(x[i]) for n bf16 values: exact for |x| in the f16 normal range [2^-14, 65504].
void launch_bf16_to_f16(const void* x, int64_t n, void* y, cudaStream_t st);
// u[t][j] = silu(g[t][j]) * up[t][j] with gu = [T][2F] (gate then up) -> u [T][F].
void launch_swiglu(const float* gu, int32_t T, int32_t F, float* u, cudaStream_t st);
// amax[r] = the largest logit of row r packed with its index (value in the high word in an
// order-preserving encoding, 0xFFFFFFFF - index in the low word: the lowest index wins ties).
void launch_argmax(const float* logits, int32_t R, int32_t V, unsigned long long* amax,
                   cudaStream_t st);
// Decode a packed argmax (-1 if none).
inline int32_t unpack_argmax(unsigned long long p) {
    return p == 0 ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(p & 0xFFFFFFFFull));
}
// Per token: x[t] = embedding row tok[t]; cs[t][i] = (cos, sin) of pos[t] * theta[i] with
// theta[i] = base^(-2i/hd) (a double table), the angle reduced in double before a float
// sincos; amax[0..n_amax) reset to 0.
void launch_embed_rope(const DevMat& E, const int32_t* tok, const int32_t* pos, int32_t T,
                       int32_t hd, const double* theta, float* x, float2* cs,
                       unsigned long long* amax, int32_t n_amax, uint32_t* err, cudaStream_t st);
// Split Q8_0 blocks (34 bytes: fp16 d, 32 int8 q) into quants [rows][cols] and scales.
void launch_q8_0_unpack(const uint8_t* blocks, int64_t rows, int64_t cols, int8_t* q,
                        __half* d, cudaStream_t st);

// ---- linear layers (kernels_linear.cu) --------------------------------------------------------
enum Epi : int32_t { EPI_STORE = 0, EPI_ADD = 1 };
// y[t][m] (op)= sum_k W[row0 + m][k] x[t][k], m < M, t < T ([P2] Example 4, MUL_MAT; ADD for the
// residual). x row stride ldx, y row stride ldy.
void launch_linear(const DevMat& W, int64_t row0, int64_t M, const float* x, int32_t ldx,
                   int32_t T, float* y, int32_t ldy, Epi epi, cudaStream_t st);
// u[t][j] = silu(sum_k G[j][k] x[t][k]) * sum_k U[j][k] x[t][k] for the gate rows [0, F) and up
// rows [F, 2F) of W ([P2] Example 4, ffn_gate, ffn_up, SWIGLU). tmp: [T][2F] scratch used when
// the batched path computes the two projections before the product.
void launch_linear_swiglu(const DevMat& W, int32_t F, const float* x, int32_t ldx, int32_t T,
                          float* u, int32_t ldu, float* tmp, cudaStream_t st);
// Largest T the GEMV path serves; larger T go through the tiled GEMM.
int32_t gemv_max_tokens();

// ---- attention (kernels_attention.cu) ---------------------------------------------------------
constexpr int kAttnTileQ = 16;           // query tokens per attention tile
// Shapes the attention kernels are built for.
inline bool attention_supported(int hd, int n_gqa) {
    return n_gqa == 4 && (hd == 32 || hd == 64 || hd == 128);
}
struct AttnArgs {
    const float* q;          // qkv buffer; q of token t, head h at q[t * ldq + h * hd]
    int32_t ldq;
    const void* kc;          // this layer's K cache [Hkv][n_ctx][hd]
    const void* vc;
    // Q8_0 caches, query tiles of several tokens: kc / vc are f16 copies of the quants and these
    // the cache's fp16 scales [Hkv][n_ctx][hd / 32] (null otherwise)
    const void* k_scale = nullptr;
    const void* v_scale = nullptr;
    int32_t n_ctx, kv_type, H, Hkv, hd;
    const int32_t* tok_pos;  // [T]
    const int32_t* list_cells; const int32_t* list_pos;   // concatenated cell lists
    const int32_t* perm;     // [T] tokens grouped by list
    const int4* tile_desc;   // per tile, 2 x int4: {list, first token, tokens, first item},
                             //                     {end item, list start, list length, 0}
    const int4* wi_desc;     // per work item: {tile, first cell, end cell, first partial row}
    int32_t* tickets;        // [tiles][Hkv] zero between launches (blocks done per tile); holds
                             // kDecTicketsPerHead times as many
    float* part_o;           // [rows][Hkv][hd] unnormalised partial outputs
    float* part_m;           // [rows][Hkv] running max (log2 domain)
    float* part_l;           // [rows][Hkv] running sum
    float* out;              // [T][H * hd]
    void* out_b;             // if set: bf16 output [T][H * hd] instead of out
    void* out_b_lo;          // with out_b: the low bf16 term of the output
    bool out_f16;            // with out_b: a single f16 output instead of bf16 terms
    int32_t ldo;
    const int32_t* hdr;      // device: [0] work items of this ubatch
    int32_t n_work, max_nq;  // grid size (an upper bound of the device count), tile shape
    bool pdl;                // programmatic dependent launch after the previous kernel
    const int32_t* slot;     // decode steps: the cells this ubatch writes (n_tok of them)
    int32_t n_tok;
    int32_t tile_q = kAttnTileQ;   // query tokens per tile of the plan (attention_tc_tile_q() for
                                   // the tcgen05 tiles)
    uint32_t* err = nullptr;       // error word (ERR_TIMEOUT from a bounded wait that ran out)
    // tcgen05 tiles, F16 caches: TMA maps of the whole K and V caches as [layers x Hkv x n_ctx]
    // rows of hd f16 (null: gather every row), and this layer's first row
    const CUtensorMap* kmap = nullptr;
    const CUtensorMap* vmap = nullptr;
    int32_t kv_row0 = 0;
    // decode steps: the ubatch's longest cell list reaches kDecLongList cells (the decode kernel
    // may then split each (token, KV head) over two clusters; tickets then holds
    // [tiles][Hkv][kDecTicketsPerHead])
    bool long_lists = false;
};
constexpr int kDecTicketsPerHead = 16;
constexpr int kDecLongList = 2048;
// Grouped-query attention of every token over the cells of its list with cell.pos <= token.pos:
// split-K partial softmax per work item, then a combine per tile ([P2] Example 4 FLASH_ATTN_EXT;
// Example 11 for the unfused meaning). Scale 1/sqrt(hd).
bool launch_attention(const AttnArgs& a, cudaStream_t st);
// The tcgen05 prefill tiles (attn_tc.cu): F16 cache, head_dim 128, 4 query heads per KV head, a
// single f16 output (forward passes whose matrix products take f16 activations), plans of
// attention_tc_tile_q() tokens per tile.
int attention_tc_tile_q();
bool attention_tc_ok(const AttnArgs& a);
bool launch_attention_tc(const AttnArgs& a, cudaStream_t st);

// ---- the sampler chain on one logits row (sampler.cu)
struct SampleArgs {
    const float* logits = nullptr;   // [V] the row
    int32_t V = 0;
    const int32_t* pen_tok = nullptr;  // device: tokens of the repeat penalty
    int32_t n_pen = 0;
    float penalty = 1.f;
    int32_t top_k = 1;               // 1 .. sample_max_k()
    float top_p = 1.f, min_p = 0.f, temperature = 0.f, u = 0.f;
    int32_t* out = nullptr;          // the picked token (device)
    uint32_t* err = nullptr;         // written 0 on success, ERR_ROW_RANGE without a candidate
};
int sample_max_k();
// Device state one sampler call uses (barrier, histograms, candidates): sample_state_bytes()
// bytes, zeroed once at allocation and again after a call that did not finish (err not written).
size_t sample_state_bytes();
// One cooperative launch over up to 64 blocks (more for rows above 64 x 4096 values); false if
// the row is too long for the SM count or the launch failed.
bool launch_sample(const SampleArgs& a, void* state, int n_sm, cudaStream_t st);
// The prefill tiles (16 tokens x 4 query heads) on tensor cores (attn_mma.cu): F16 KV, or a Q8_0
// cache through its f16 quant copy and scales (k_scale / v_scale), 4 query heads per KV head,
// head_dim 32, 64 or 128. launch_attention uses it when it applies.
bool attention_mma_ok(const AttnArgs& a);
bool launch_attention_mma(const AttnArgs& a, cudaStream_t st);
// Decode steps (one token per query tile) with a 16-block cluster per (token, KV head) merging
// the split-K partial states through distributed shared memory (attn_decode.cu).
bool attention_decode_ok(const AttnArgs& a);
bool launch_attention_decode(const AttnArgs& a, cudaStream_t st);

}  // namespace llm
