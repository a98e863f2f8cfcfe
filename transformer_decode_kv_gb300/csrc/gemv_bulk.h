// Decode GEMV with TMA bulk staging and fused prologue/epilogues. See gemv_bulk.cu.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kernels.h"

namespace llm {

enum GemvEpi : int32_t {
    GEPI_STORE = 0,    // y[t][m] = acc
    GEPI_ADD = 1,      // y[t][m] += acc (residual)
    GEPI_SWIGLU = 2,   // y[t][j] = silu(acc_gate) * acc_up; W rows [row0, row0+F) gate, +F up
    GEPI_QKV = 3,      // RoPE on Q/K rows, Q -> y, K/V -> cache cells slot[t] (cell t if slot is null)
    GEPI_LOGITS = 4,   // y[t][m] = acc and amax[t] = max packed (value, lowest index)
};

struct GemvArgs {
    const void* W = nullptr;       // weight rows (quants for Q8_0)
    const __half* S = nullptr;     // Q8_0 scales [rows][K/32]
    int64_t row0 = 0, M = 0, K = 0, F = 0;
    const float* x = nullptr;      // activations, row t at x[x_rows ? x_rows[t] : t][*]
    int32_t ldx = 0, T = 0;
    const int32_t* x_rows = nullptr;
    const float* g = nullptr;      // RMSNorm gain (when the op starts with the norm)
    float eps = 0.f;
    float* y = nullptr;
    int32_t ldy = 0;
    // GEPI_QKV
    int32_t H = 0, Hkv = 0, hd = 0, n_ctx = 0, kv_type = 0;
    const float2* cs = nullptr;
    const int32_t* slot = nullptr;
    void* kc = nullptr;
    void* vc = nullptr;
    // GEPI_LOGITS
    unsigned long long* amax = nullptr;
    uint32_t* err = nullptr;
    int32_t rows_cap = 0;          // set by the launcher
    int32_t n_stages = 0;          // set by the launcher
    int32_t stage_bytes = 0;       // set by the launcher (0: general slice mapping)
};

int gemv_bulk_tm(int T);
// Whether the bulk path serves this weight type / shape / token count.
bool gemv_bulk_ok(int wt, const GemvArgs& a, int epi, int n_sm);
// Launch (norm: RMSNorm of the activation rows with gain a.g first). pdl: programmatic dependent
// launch (the kernel starts streaming weights before the previous kernel ends).
bool launch_gemv_bulk(int wt, GemvArgs a, int epi, bool norm, int n_sm, cudaStream_t st, bool pdl);

}  // namespace llm
