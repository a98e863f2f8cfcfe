/*
 * llm.h - C ABI of a single-GPU (sm_103a) decode library for Llama-architecture GQA transformers
 * with a KV cache: llama_decode's processing of a batch, split into ubatches, through token
 * embedding, per-layer RMSNorm / Q,K,V projections / RoPE / K,V append into the cache /
 * grouped-query attention over the cache / output projection / SwiGLU FFN, then the final norm,
 * logits for the flagged positions and a greedy pick.
 *
 * Sources (page title, section):
 *   [P1] "llama.cpp AI LLM Engine - Як це працює": Крок 10 (llama_batch, batch_allocr::init),
 *        Крок 11 (llama_decode and its return values), Крок 12 (init_batch: split and slot search),
 *        Крок 13а-13в (process_ubatch: apply, graph, set_inputs, compute), Крок 14
 *        (llama_get_logits_ith), KV-cache section (seq_pos_max, K/V appended before attention).
 *   [P2] "llama.cpp Architecture": Example 2 (ggml shapes {ne0 = row length, ne1 = rows}, Q8_0
 *        blocks), Example 4 (tensor names and shapes of one decode step), Example 8-10 (hparams,
 *        context parameters, n_ctx padded to 256, KV sizes).
 *   [P4] "デコードループ：バッチ処理、KVキャッシュ、メモリ管理": バッチパイプライン, KVキャッシュの詳細
 *        (cells, slot_info), エラーリカバリとステートロールバック (apply/rollback, return codes).
 *
 * Conventions for every call:
 *   - Pointers named "host" are CPU memory; "device" pointers are CUDA device memory of the GPU the
 *     context was created on. Where either is accepted this is stated.
 *   - The library never keeps a pointer the caller passed in after the call returns, except the
 *     CUDA stream given to llm_ctx_init.
 *   - Errors are reported by return value and never abort the process. llm_last_error() gives a
 *     one-line description of the most recent failure of a context.
 *   - A context is not thread-safe: calls on one context must not overlap.
 */
#ifndef LLM_H
#define LLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage types of weights and cache rows ([P2] Example 2). Q8_0: blocks of 32 values stored as
 * a 2-byte little-endian fp16 scale d followed by 32 int8 quants q (34 bytes); value = d * q; a
 * row holds a whole number of blocks. BF16: the top 16 bits of an IEEE float32. */
typedef enum {
    LLM_TYPE_F32  = 0,
    LLM_TYPE_F16  = 1,
    LLM_TYPE_BF16 = 2,
    LLM_TYPE_Q8_0 = 8
} llm_type;

/* Model hyper-parameters ([P2] Example 8, print_info). head_dim * n_head is the width of the Q
 * projection; n_head must be a multiple of n_head_kv (n_gqa = n_head / n_head_kv query heads
 * share one KV head: query head h reads KV head h / n_gqa). rope_type 0 is the "normal" layout
 * (adjacent element pairs); it is the only one supported. */
typedef struct llm_hparams {
    int32_t n_layer;
    int32_t n_embd;
    int32_t n_head;
    int32_t n_head_kv;
    int32_t head_dim;
    int32_t n_ff;
    int32_t n_vocab;
    float   rope_freq_base;
    float   rms_eps;
    int32_t rope_type;
} llm_hparams;

/* Context flags. */
enum {
    /* Book-keeping only: batches are sanitised, split, given KV slots and committed, but no device
     * memory is allocated and no kernel runs; llm_get_logits_ith returns NULL. Lets the host
     * control plane be tested on a machine without a GPU. */
    LLM_CTX_HOST_ONLY = 1u << 0,
    /* Run one-token ubatches as the single persistent decode-step kernel instead of the per-op
     * kernel sequence (replayed as a CUDA graph). Both compute the same ops in float32 over the
     * stored weights; the persistent kernel serves 2-byte weights of the 8B layer shape only.
     * Off by default: on a GB300 the per-op sequence is as fast or faster (3.43 vs 3.47 ms per
     * 8B BF16 step). */
    LLM_CTX_FUSED_STEP = 1u << 1,
    /* A cache not shared by all sequences (kv_unified = false; [P1] Крок 9-10: n_ctx is divided
     * among the sequences, n_ctx_seq = n_ctx / n_seq_max cells each; [P2] Example 9): sequence s
     * writes only cells [s n_ctx_seq, (s + 1) n_ctx_seq), each token must belong to exactly one
     * sequence (else the batch is invalid, -1), and batches are split with split_equal ([P1]
     * Крок 12, [P4] llama_ubatch n_seq_tokens / n_seqs): each ubatch takes the sequences with
     * unused tokens in ascending, consecutive ids (at most n_ubatch of them) and the same number
     * min(n_ubatch / n_seqs, fewest unused tokens among them) of next tokens from each. Output
     * rows stay in batch order. */
    LLM_CTX_KV_SPLIT = 1u << 2,
};

/* Context parameters ([P1] Крок 9-10 context constructor; [P2] Example 9; [P4] コンテキストの構築).
 * n_ctx is rounded up to a multiple of 256; n_batch becomes min(n_ctx, n_batch) and n_ubatch
 * min(n_batch, n_ubatch). type_k / type_v: both LLM_TYPE_F32, both LLM_TYPE_F16, or both
 * LLM_TYPE_Q8_0 ([P2] Memory Math: a q8_0 cache of 34 bytes per 32 values; [P4] type_k/type_v; each
 * written row is quantised per 32-value block with d = max|x| / 127 and q = round(x / d), the
 * decisions taken in float32; the fused persistent decode step takes F32/F16 only). stream: a cudaStream_t
 * the library launches all its work on (NULL = the library creates its own non-blocking stream).
 * The KV cache is unified: one set of n_ctx cells shared by all n_seq_max sequences. */
typedef struct llm_cparams {
    uint32_t n_ctx;
    uint32_t n_seq_max;      /* 1 .. 256 */
    uint32_t n_batch;
    uint32_t n_ubatch;
    int32_t  type_k;
    int32_t  type_v;
    void    *stream;
    uint32_t flags;
} llm_cparams;

/* A batch ([P1] Крок 10, llama_batch). Arrays have n_tokens entries and are host memory owned by
 * the caller; llm_decode copies what it needs before returning. Fields may be NULL:
 *   pos NULL      -> each sequence continues from llm_seq_pos_max(s) + 1, in batch order;
 *   seq_id NULL   -> every token belongs to sequence 0 (n_seq_id is then ignored);
 *   n_seq_id NULL -> one sequence id per token (seq_id[i][0]);
 *   logits NULL   -> logits only for the last token.
 * logits[i] != 0 requests the logits row of token i. */
typedef struct llm_batch {
    int32_t               n_tokens;
    const int32_t        *token;
    const int32_t        *pos;
    const int32_t        *n_seq_id;
    const int32_t *const *seq_id;
    const int8_t         *logits;
} llm_batch;

typedef struct llm_ctx llm_ctx;

/* Defaults: n_ctx 4096, n_seq_max 1, n_batch 2048, n_ubatch 512, F16 K and V, own stream. */
llm_cparams llm_cparams_default(void);

/* Create a context: validates hp and cp, allocates the device weight store, the KV cache
 * ([P1] KV-cache section: per layer one K and one V buffer for all n_ctx cells), every scratch
 * buffer a ubatch of n_ubatch tokens needs and the output buffers, so llm_decode allocates
 * nothing in the common case. Returns NULL on invalid parameters or failed allocation
 * (llm_last_error(NULL) then describes the failure). */
llm_ctx *llm_ctx_init(const llm_hparams *hp, const llm_cparams *cp);

/* Release every resource of the context (waits for its stream first). NULL is a no-op. */
void llm_ctx_free(llm_ctx *ctx);

/* Copy one named tensor into the device weight store ([P2] Example 4 names and shapes):
 *   token_embd.weight {n_embd, n_vocab}, output_norm.weight {n_embd},
 *   output.weight {n_embd, n_vocab} (optional: absent = tied to token_embd),
 *   blk.N.attn_norm.weight {n_embd}, blk.N.attn_q.weight {n_embd, n_head*head_dim},
 *   blk.N.attn_k.weight / attn_v.weight {n_embd, n_head_kv*head_dim},
 *   blk.N.attn_output.weight {n_head*head_dim, n_embd}, blk.N.ffn_norm.weight {n_embd},
 *   blk.N.ffn_gate.weight / ffn_up.weight {n_embd, n_ff}, blk.N.ffn_down.weight {n_ff, n_embd}.
 * ne[0] is the row length and ne[1] the number of rows (1 for vectors), ggml order. data holds
 * the rows in storage type `type`, nbytes long; it may be host or device memory (any pointer
 * CUDA's unified addressing resolves). Norm gains must be F32; linear weights F32, F16, BF16 or
 * Q8_0 (Q8_0 needs ne[0] % 32 == 0); the three of attn_q/k/v of one layer must share a type,
 * and so must ffn_gate/ffn_up. Returns 0 on success, -1 for an unknown name, a wrong shape, an
 * unsupported type, a size mismatch or a second load of the same name, -2 on a CUDA failure.
 * The call synchronises the device before reading data, so data written by earlier work on any
 * stream is complete. */
int llm_load_weights(llm_ctx *ctx, const char *name, int32_t type, const int64_t ne[2],
                     const void *data, size_t nbytes);

/* 0 if every required tensor is loaded, else -1 (llm_last_error names the first missing one). */
int llm_weights_ready(llm_ctx *ctx);

/* Decode a batch ([P1] Крок 11-13; [P4] process_ubatch). Steps: sanitise and fill defaults; split
 * into ubatches of at most n_ubatch tokens in batch order; find KV cells for every ubatch before
 * committing any (each ubatch takes the lowest-index empty cells, ascending); then per ubatch:
 * commit its cells, run the forward pass on the device (K/V of the ubatch are written to the cache
 * before the attention reads it) and append the flagged tokens' logits rows in batch order.
 * Returns:
 *    0  success
 *    1  no KV slot for the batch: nothing was changed
 *    2  aborted by the abort callback (checked before each ubatch's compute); the current ubatch
 *       is rolled back, earlier ubatches stay in the cache
 *   -1  invalid batch (no tokens, more than n_batch tokens, a token id outside [0, n_vocab), a
 *       sequence id outside [0, n_seq_max), positions of a sequence that are not consecutive or
 *       do not continue from llm_seq_pos_max + 1), or weights not ready
 *   -2  internal / allocation failure
 *   -3  the device computation failed (a CUDA error or a kernel's own bounds check); the current
 *       ubatch is rolled back: seq_rm(s, pos_min(s), -1) for each of its sequences
 * After a non-zero return no logits are readable. The call returns when the device work has
 * finished. */
int32_t llm_decode(llm_ctx *ctx, llm_batch batch);

/* Logits row of the last llm_decode ([P1] Крок 14): i >= 0 is a token index of that batch, i < 0
 * counts from the last output row (-1 = last). Returns a host pointer to n_vocab floats owned by
 * the context and valid until the next llm_decode or llm_ctx_free; NULL if i names a token whose
 * logits were not requested, is out of range, or the context is host-only. The first call after a
 * decode copies the output rows from the device. */
float *llm_get_logits_ith(llm_ctx *ctx, int32_t i);

/* Greedy pick of the same row, computed on the device (the largest logit; the lowest index among
 * equal maxima). -1 where llm_get_logits_ith would return NULL. Does not copy logits rows. */
int32_t llm_get_argmax_ith(llm_ctx *ctx, int32_t i);

/* Number of output rows of the last successful llm_decode. */
int32_t llm_n_outputs(llm_ctx *ctx);

/* Remove sequence seq from the cells holding positions p0 <= pos < p1 ([P4] llama_memory_i::seq_rm,
 * エラーリカバリ); p0 < 0 means 0, p1 < 0 means no upper bound, seq < 0 means every sequence.
 * Cells left with no sequence become empty and are reused by later batches. Returns 1. */
int llm_seq_rm(llm_ctx *ctx, int32_t seq, int32_t p0, int32_t p1);

/* Memory update ([P4] KVキャッシュの詳細: memory_update(optimize=true) defragments the cache by
 * moving cells to close the gaps; the figure "After Defrag" shows the result). With optimize != 0
 * the used cells are packed from cell 0, ordered by sequence (a shared cell: its lowest sequence
 * id), then position; every layer's K/V rows move with their cells (device copies, stream
 * synchronised), so later decodes give the same results up to float summation order.
 * llm_decode runs the same defrag once, and searches again, when a batch finds no free cells.
 * Returns 1 if cells moved, 0 if nothing to do (or optimize == 0), -1 on a device error. */
int llm_memory_update(llm_ctx *ctx, int optimize);

/* Largest / smallest position held for a sequence, -1 if it holds none ([P1] KV-cache section). */
int32_t llm_seq_pos_max(llm_ctx *ctx, int32_t seq);
int32_t llm_seq_pos_min(llm_ctx *ctx, int32_t seq);

/* Abort callback ([P1] Крок 11, return value 2): called before each ubatch's computation; a
 * non-zero return aborts the decode with 2. NULL removes it. */
void llm_set_abort_callback(llm_ctx *ctx, int (*cb)(void *user), void *user);

/* Effective context sizes after rounding / clamping. */
uint32_t llm_n_ctx(llm_ctx *ctx);
/* Cells one sequence can use: n_ctx, or n_ctx / n_seq_max with LLM_CTX_KV_SPLIT ([P2] Example 9
 * n_ctx_seq). */
uint32_t llm_n_ctx_seq(llm_ctx *ctx);
uint32_t llm_n_batch(llm_ctx *ctx);
uint32_t llm_n_ubatch(llm_ctx *ctx);

/* Number of cells holding a position. */
int32_t llm_kv_used_cells(llm_ctx *ctx);

/* One-line description of the last failure of ctx (or of the last failed llm_ctx_init when ctx is
 * NULL). The string is owned by the library. */
const char *llm_last_error(llm_ctx *ctx);

/* Timing counters ([P2] Example 11-12, llama_perf_context_print): decode calls, tokens, ubatches,
 * CUDA-graph replays, and host milliseconds spent inside llm_decode. */
typedef struct llm_perf_data {
    int64_t n_decode_calls;
    int64_t n_tokens;
    int64_t n_ubatches;
    int64_t n_graph_replays;
    double  t_decode_ms;
    int64_t n_fused_steps;   /* one-token ubatches run as the single persistent kernel */
    int64_t n_defrags;       /* cache defrags that moved cells (llm_memory_update or a retry) */
    int64_t weight_device_bytes;  /* device memory holding the weights as stored plus the operand
                                     copies made for the prefill matrix products (a BF16 weight's
                                     f16 copy; Q8_0 weights get none) */
} llm_perf_data;
void llm_perf(llm_ctx *ctx, llm_perf_data *out);

/* ---- sampler chain on the device ([P1] sampler chain after Крок 14: penalties, then the
 * cut-offs top-k, top-p and min-p, then temperature, then one token is picked; a backend sampler
 * picks on the device, so the logits row is not copied to the host).
 * Steps, in order, over logits row i of the last llm_decode (i as in llm_get_logits_ith):
 *   repeat penalty: each distinct token of penalty_tokens once, l > 0 -> l / repeat_penalty,
 *     otherwise l * repeat_penalty (1 = off);
 *   top-k: the top_k largest logits (1 .. 4096; ties at the k-th value: the lower token ids),
 *     ordered by logit descending then token id ascending;
 *   top-p: the shortest prefix of that order whose softmax probability (over the candidates,
 *     before temperature) reaches top_p (1 = off);
 *   min-p: the candidates with l - l_max >= ln(min_p) (0 = off);
 *   pick: temperature <= 0 takes the first candidate (greedy); otherwise the first candidate
 *     whose cumulative weight exp((l - l_max) / temperature) exceeds u times the total.
 * u in [0, 1) is the caller's uniform random draw (the library draws no random numbers).
 * penalty_tokens: host array of n_penalty_tokens (<= 4096) token ids, may be NULL if 0.
 * Returns the token, or -1 for an invalid argument, a row without logits or a device error.
 * Synchronises the context's stream. */
typedef struct llm_sampler_params {
    int32_t top_k;
    float   top_p;
    float   min_p;
    float   temperature;
    float   repeat_penalty;
    const int32_t *penalty_tokens;
    int32_t n_penalty_tokens;
} llm_sampler_params;
int32_t llm_sample_ith(llm_ctx *ctx, int32_t i, const llm_sampler_params *params, float u);

/* ---- test and debugging hooks ---------------------------------------------------------------
 * They expose intermediate state so tests can compare it with an independent implementation
 * (the eval-callback idea of [P2] Example 4). */

/* KV cell index of every token of the last llm_decode (slot_info, [P4] KVキャッシュの詳細), in batch
 * order. Writes min(cap, n) values to out (host) and returns n. */
int32_t llm_debug_last_slots(llm_ctx *ctx, int32_t *out, int32_t cap);

/* Attention visibility of ubatch `ub` of the last llm_decode as the library computed it, expanded
 * to a dense [n_tokens][n_kv] row-major byte matrix (1 = token may attend to the cell) on the host.
 * n_kv is the highest used cell + 1 after that ubatch's commit. Returns n_tokens * n_kv (0 if ub
 * is out of range); writes at most cap bytes. *n_kv_out receives n_kv. */
int64_t llm_debug_ubatch_mask(llm_ctx *ctx, int32_t ub, uint8_t *out, int64_t cap,
                              int32_t *n_kv_out);

/* Keep copies of per-layer intermediates of the last ubatch (enable != 0) on the device. */
int llm_debug_capture(llm_ctx *ctx, int enable);

/* Copy a captured intermediate of the last ubatch to host memory as float32, row-major
 * [n_tokens][width]. name: "embd" (layer ignored), "l_out" (residual stream after layer `layer`),
 * "attn_out" (attention output of layer `layer`, before the output projection), "kq_in" (the Q
 * rows after RoPE of layer `layer`), "k_in" / "v_in" (Q8_0 caches only: the float32 K rows after
 * RoPE and the V rows, [n_tokens][n_head_kv * head_dim], that layer `layer` quantised into the
 * cache), "result_norm" (final-normed output rows; present only when the
 * output matrix ran unfused, not in the one-token GEMV that normalises in its prologue). Returns the number
 * of floats available (0 if none), writes at most cap. */
int64_t llm_debug_get_tensor(llm_ctx *ctx, const char *name, int32_t layer, float *out,
                             int64_t cap);

/* Copy layer `layer`'s K cache (which = 0) or V cache (which = 1) to host memory as stored: type_k
 * / type_v elements laid out [n_head_kv][n_ctx][head_dim] (cell c of KV head g at (g * n_ctx + c)
 * * head_dim). A Q8_0 cache holds the int8 quants in that layout, followed by the fp16 scales
 * [n_head_kv][n_ctx][head_dim / 32] (one per 32-value block; value = scale * quant). which = 2 / 3
 * (Q8_0 caches only; layer ignored beyond its range check): the f16 copy of the K / V quants, same
 * layout, that the last attention over query tiles of several tokens read (the last layer of the
 * last such ubatch), valid for the cells below that ubatch's n_kv. out may be NULL to query the size.
 * Returns the slab's size in bytes (copies at most cap_bytes, after the context's stream has
 * finished), 0 for a bad layer/which or a host-only context. */
int64_t llm_debug_kv_raw(llm_ctx *ctx, int32_t layer, int32_t which, void *out, int64_t cap_bytes);

/* Per-kernel-class device timing. enable != 0 resets the counters and brackets every later launch
 * with CUDA events on the context's stream (small overhead); 0 stops. */
int llm_debug_kernel_timing(llm_ctx *ctx, int enable);

/* Counters of kernel class i (0 <= i < the returned count): its name (NUL-terminated, at most
 * name_cap bytes), launches, summed device milliseconds, and the summed algorithmic bytes moved
 * and FLOPs of those launches (the minimum a launch must read and write, and its arithmetic).
 * Any output pointer may be NULL. Returns the number of classes. */
int32_t llm_debug_kernel_stats(llm_ctx *ctx, int32_t i, char *name, int32_t name_cap,
                               int64_t *launches, double *ms, double *bytes, double *flops);

/* One launch of the tensor-core (tcgen05) GEMM on device buffers, synchronous: W bf16 row-major
 * [rows][K], X bf16 row-major [T][K], K % 64 == 0. epi 0: Y[t][m] = sum_k W[m][k] X[t][k] as
 * float32 (rows = M, M % 128 == 0); epi 1: the same added into Y; epi 2: Y[t][j] (bf16) =
 * silu(gate_j) * up_j with gate rows [0, F) and up rows [F, 2F) of W (F % 64 == 0). ldy is Y's
 * row stride in elements. Returns 0, -1 for an unsupported shape, -3 if the launch failed or the
 * kernel reported an error (its waits are time-bounded). */
int llm_debug_gemm_bf16(int32_t epi, const void *W, int64_t M, int64_t K, const void *X, int32_t T,
                        void *Y, int32_t ldy, int32_t F);

/* One launch of the token-major tensor-core GEMM the prefill ubatches use, on device buffers,
 * synchronous ([P2] "llama.cpp Architecture", Example 4: MUL_MAT of a {K, M} weight by the
 * ubatch's activations, ADD, SWIGLU). W f16 row-major [rows][K] (W_lo optional: a second f16 term
 * of the same weights, both multiplied into the sums, as a Q8_0 weight's d*q is held), X f16
 * row-major [T][K], K % 64 == 0. epi 0: Y[t][m] = sum_k W[m][k] X[t][k] as float32 (rows = M,
 * M % 256 == 0; with splits > 1 the K range is split over `splits` CTAs whose partial sums are
 * added atomically, so Y must start zeroed); epi 1: the same added into Y; epi 2: Y[t][j] (f16,
 * ldy in f16 elements) = silu(gate_j) * up_j with gate rows [0, F) and up rows [F, 2F) of W
 * (F % 128 == 0, splits 1). one_cta != 0 keeps the one-CTA kernel for T > 128 (the two-CTA
 * cta_group::2 kernel otherwise). Returns 0, -1 for an unsupported shape, -3 if the launch
 * failed or the kernel reported an error. */
int llm_debug_gemm_tn_f16(int32_t epi, const void *W, const void *W_lo, int64_t M, int64_t K,
                          const void *X, int32_t T, float *Y, int32_t ldy, int32_t F, int32_t splits,
                          int32_t one_cta);

/* llm_debug_gemm_tn_f16 over a Q8_0 weight held as the library stores it ([P2] "llama.cpp
 * Architecture", Example 2 block: an fp16 scale d and 32 int8 quants q, value d * q): Wq int8
 * row-major [rows][K], Ws fp16 scales [rows][K / 32] (device memory, 16-byte aligned), X f16
 * [T][K]. The two-CTA kernel dequantises each 64-wide k-step into the exact f16 terms of d * q in
 * shared memory; any T >= 1. epi and the remaining arguments as for llm_debug_gemm_tn_f16.
 * Returns 0, -1 for an unsupported shape, -3 on a failure. */
int llm_debug_gemm_tn_q8(int32_t epi, const void *Wq, const void *Ws, int64_t M, int64_t K, const void *X,
                         int32_t T, float *Y, int32_t ldy, int32_t F, int32_t splits);

/* llm_debug_gemm_tn_q8 with per-CTA counters: 8 uint64 values per CTA in trace (start and end
 * global-timer stamps in ns at 0 and 7, the accumulator-ready stamp at 6; SM cycles the first
 * converter thread waited for quant tiles (1), for free stages (2) and spent converting (3); SM
 * cycles the MMA thread of the pair's leader waited for activation tiles (4) and for converted
 * terms (5)), CTAs in launch order. Returns the number of values written (cap must hold them), -1
 * for an unsupported shape or a short buffer, -3 on a failure. */
int64_t llm_debug_gemm_tn_q8_trace(int32_t epi, const void *Wq, const void *Ws, int64_t M, int64_t K,
                                   const void *X, int32_t T, float *Y, int32_t ldy, int32_t F,
                                   int32_t splits, uint64_t *trace, int64_t cap);

/* The two-CTA token-major GEMM of llm_debug_gemm_tn_f16 (T > 128, one weight term) with a
 * timeline: per CTA 8 uint64 values in trace, global-timer stamps in ns (start, set-up done, first
 * stage ready, last MMA issued, accumulator ready, epilogue done, end) and the SM id, CTAs in
 * launch order (x fastest, then y, then z). Returns the number of values written (cap must hold
 * them), -1 for an unsupported shape or a short buffer, -3 on a failure. */
int64_t llm_debug_gemm_tn_f16_trace(int32_t epi, const void *W, int64_t M, int64_t K, const void *X,
                                    int32_t T, float *Y, int32_t ldy, int32_t F, int32_t splits,
                                    uint64_t *trace, int64_t cap);

/* The same GEMM as llm_debug_gemm_bf16, for callers that cannot allocate device memory (for
 * example engines that reserve all GPU memory up front for their own pools, or code that must
 * not trigger the device-wide synchronisation cudaFree performs). The pages have no counterpart:
 * this is an interface of this library only. The call allocates nothing: its scratch (the
 * kernel's error word) is a fixed 256-byte array inside the library that every GPU which loads
 * the library holds until the process exits. The first call on a device looks that array's
 * device address up (cudaGetSymbolAddress) with the device current; make that first call before
 * starting any stream capture. The address is kept for the life of the process: a device reset
 * (cudaDeviceReset, or anything else that destroys the device's primary context) unloads the
 * array, so do not call this entry point on a device after resetting it. Every call shares the
 * array, so calls whose GPU work overlaps (from several host threads or streams) race on it; each
 * call clears the error word before its launch. Arguments, limits and results are those of
 * llm_debug_gemm_bf16: -1 for an unsupported shape, -3 if the launch failed or the kernel
 * reported an error. Synchronous (legacy default stream). */
int llm_gemm_bf16_noalloc(int32_t epi, const void *W, int64_t M, int64_t K, const void *X,
                          int32_t T, void *Y, int32_t ldy, int32_t F);

/* Test hook of llm_gemm_bf16_noalloc: write `value` into its error word on the current device
 * (synchronous), as a previous call that failed would leave it, so a test can check that the
 * next call starts from a cleared word. Returns 0, or -3 if the copy failed. */
int llm_debug_noalloc_scratch_poke(uint32_t value);

/* Timeline of the persistent one-token kernel. enable != 0 makes later one-token steps record, per
 * block, global-timer stamps (ns) at the start and end of each consumer phase and at the first
 * and last weight copy the block's producer issues for each matrix; 0 stops. */
int llm_debug_step_trace_enable(llm_ctx *ctx, int enable);
/* Copy the last recorded step's stamps to out as [n_blocks][n_slots][2] (start, end) uint64
 * values: slot 0 the embedding phase, 1 + 5 l + op the phases of layer l (op 0 Q/K/V, 1 attention,
 * 2 output projection, 3 gate/up, 4 down), 1 + 5 n_layer the output matrix, then
 * 2 + 5 n_layer + j the producer's matrix j (4 per layer, then the output matrix). Returns the
 * number of values (0 if nothing was recorded); writes at most cap. */
int64_t llm_debug_step_trace(llm_ctx *ctx, uint64_t *out, int64_t cap, int32_t *n_blocks,
                             int32_t *n_slots);

/* Overwrite logits row i of the last llm_decode (i as in llm_get_logits_ith) with n_vocab floats
 * from the host array row (for tests of llm_sample_ith on chosen rows: ties, NaN, flat rows).
 * llm_get_argmax_ith keeps the argmax that llm_decode computed. Returns 0, or -1 for a row without logits or a failed copy. Synchronises the stream. */
int llm_debug_set_logits(llm_ctx *ctx, int32_t i, const float *row);

/* Fault injection: kind 1 makes ubatch `ub` of the next llm_decode hand the K/V append kernel a
 * cell index past the cache; the kernel's bounds check skips the write and reports the error
 * word, so llm_decode returns -3 and rolls that ubatch back. kind 0 clears it. */
int llm_debug_inject_fault(llm_ctx *ctx, int32_t kind, int32_t ub);

#ifdef __cplusplus
}
#endif

#endif /* LLM_H */
