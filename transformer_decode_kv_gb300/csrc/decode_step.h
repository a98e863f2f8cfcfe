// One-token decode step as a single persistent kernel. See decode_step.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace llm {

// Device pointers of one layer (a table of these lives in device memory).
struct StepLayer {
    const void* qkv = nullptr;        // fused Q|K|V rows [(H + 2 Hkv) hd][d]
    const void* wo = nullptr;         // output projection [d][H hd]
    const void* gu = nullptr;         // gate rows [0, F) then up rows [F, 2F), [2F][d]
    const void* down = nullptr;       // [d][F]
    const float* attn_norm = nullptr;
    const float* ffn_norm = nullptr;
    void* kc = nullptr;               // this layer's K cache [Hkv][n_ctx][hd]
    void* vc = nullptr;
};

struct StepArgs {
    const StepLayer* layers = nullptr;
    int32_t n_layer = 0, d = 0, H = 0, Hkv = 0, hd = 0, F = 0, V = 0;
    float eps = 0.f;
    DevMat embd;                      // token embedding table [V][d]
    const double* theta = nullptr;    // RoPE frequencies theta_i, i < hd/2
    const void* out = nullptr;        // output matrix [V][d], same type as the layers' weights
    const float* out_norm = nullptr;
    int32_t do_logits = 0;            // the token's logits were requested
    // activations (device scratch)
    float* x = nullptr;               // residual stream [d]
    float* q = nullptr;               // query rows after RoPE [H hd]
    float* o = nullptr;               // attention output [H hd]
    float* u = nullptr;               // SwiGLU output [F]
    float2* cs = nullptr;             // RoPE (cos, sin) of the token's position [hd/2]
    float* logits = nullptr;          // [V]
    unsigned long long* amax = nullptr;   // packed greedy pick of the token
    // this step's inputs (device upload buffer): token, position, cache cell, and the
    // attention work items over the sequence's cell list (same layout as AttnArgs)
    const int32_t* tok = nullptr;
    const int32_t* pos = nullptr;
    const int32_t* slot = nullptr;
    const int32_t* hdr = nullptr;     // [0] work items
    const int4* tile_desc = nullptr;
    const int4* wi_desc = nullptr;
    const int32_t* list_cells = nullptr;
    const int32_t* list_pos = nullptr;
    float* part_o = nullptr;          // [items * Hkv * G][hd] partial outputs
    float* part_m = nullptr;
    float* part_l = nullptr;
    int32_t* tickets = nullptr;       // [Hkv], zero between launches
    int32_t n_ctx = 0, kv_type = 0;
    // grid-wide phase counters [1 + 5 n_layer]: every launch adds gridDim.x to each one, so a
    // phase of launch number `gen` is complete at (gen + 1) * gridDim.x (modulo 2^32)
    uint32_t* counters = nullptr;
    uint32_t gen = 0;
    int32_t* abort_flag = nullptr;    // set by the first block that gives up a wait
    uint32_t* err = nullptr;
    int32_t n_stages = 0, stage_bytes = 0, rows_cap = 0;   // set by the launcher
    // optional timeline (global timer, ns) per block: consumer phase k starts at
    // trace[(b * n_trace + k) * 2] and ends at [.. + 1]; k = 0 embed, 1 + 5 l + op (0 Q/K/V,
    // 1 attention, 2 output projection, 3 gate/up, 4 down), 1 + 5 L the output matrix; then the
    // producer: op j (4 per layer, then the output matrix) first copy issued / last copy issued at
    // k = 2 + 5 L + j
    uint64_t* trace = nullptr;
    int32_t n_trace = 0;
};

// Whether the persistent kernel serves this model on this GPU: BF16 or F16 weights everywhere,
// d = H * hd, d and F multiples of 4096 elements per 8 warps' passes (see decode_step.cu),
// head_dim 64 or 128, 4 query heads per KV head, and two blocks per SM resident.
bool decode_step_ok(int32_t wt, int32_t d, int32_t H, int32_t Hkv, int32_t hd, int32_t F,
                    int32_t V, int32_t kv_type, int n_sm);
// Cells one attention pass of the kernel stages (the work-item length it is planned for).
int32_t decode_step_cells();
// Cooperative launch of one decode step (grid: two blocks per SM).
bool launch_decode_step(int32_t wt, StepArgs a, int n_sm, cudaStream_t st);

}  // namespace llm
