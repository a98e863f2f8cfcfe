// The C ABI of include/llm.h: context, device weight store, KV cache, the decode loop and the
// per-ubatch launch sequence.
//
// Decode follows [P1] "llama.cpp AI LLM Engine - Як це працює", Крок 11-14 and [P4] "デコードループ"
// (process_ubatch, エラーリカバリ): sanitise -> split -> slots for every ubatch before any commit ->
// per ubatch: commit (apply), abort check, inputs upload (set_inputs), the device forward pass,
// error check with rollback -> output rows in batch order.
#include "../../include/llm.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "decode_step.h"
#include "gemm_tc.h"
#include "gemv_bulk.h"
#include "host_plan.h"
#include "kernels.h"

using namespace llm;

namespace {

thread_local std::string g_init_error;

size_t type_size(int32_t t) { return t == LLM_TYPE_F32 ? 4 : 2; }

int64_t row_bytes(int32_t t, int64_t cols) {
    switch (t) {
        case LLM_TYPE_F32: return cols * 4;
        case LLM_TYPE_F16:
        case LLM_TYPE_BF16: return cols * 2;
        case LLM_TYPE_Q8_0: return cols / 32 * 34;
    }
    return -1;
}

enum LayerBit : uint32_t {
    B_ATTN_NORM = 1, B_Q = 2, B_K = 4, B_V = 8, B_O = 16, B_FFN_NORM = 32, B_GATE = 64, B_UP = 128,
    B_DOWN = 256, B_ALL = 511
};

struct Layer {
    DevMat qkv, wo, gu, down;
    float* attn_norm = nullptr;
    float* ffn_norm = nullptr;
    uint32_t loaded = 0;
    // TMA maps of the BF16 weights for the tensor-core prefill GEMM
    CUtensorMap mq, mo, mgu, md;
    CUtensorMap mgu128;      // gate|up with 128-row boxes (token-major SwiGLU GEMM)
    bool gu_tn = false;
    // f16 prefill operands: a BF16 layer's weights converted to f16 (mq, mo, mgu128, md over the
    // copies); a Q8_0 layer's quants as stored (the same maps, int8 tiles dequantised by the GEMM)
    bool f16_ready = false, q8_tc = false;
    // Q8_0: the block scales in the per-k-step layout the prefill GEMM copies
    uint32_t *qkv_ks = nullptr, *wo_ks = nullptr, *gu_ks = nullptr, *down_ks = nullptr;
};

// Kernel classes timed by llm_debug_kernel_timing.
enum KClass : int32_t {
    KC_EMBED, KC_ROPE_TABLE, KC_RMSNORM, KC_LINEAR_GEMV, KC_LINEAR_GEMM, KC_ROPE_KV, KC_ATTENTION,
    KC_LM_HEAD, KC_ARGMAX, KC_LINEAR_TC, KC_DECODE_STEP, KC_COUNT
};
const char* const kKClassNames[KC_COUNT] = {"embed", "rope_table", "rmsnorm", "linear_gemv",
                                            "linear_gemm", "rope_kv_append", "attention",
                                            "lm_head", "argmax", "linear_tcgen05", "decode_step"};
struct KStat { int64_t launches = 0; double ms = 0, bytes = 0, flops = 0; };
struct KPending { int32_t cls; cudaEvent_t a, b; double bytes, flops; };

// A captured decode step: the forward pass of one ubatch shape, replayed with new inputs.
struct StepGraph {
    cudaGraphExec_t exec = nullptr;
    std::vector<KPending> timing;   // event pairs recorded inside the graph (timing graphs)
    std::vector<cudaEvent_t> events;
};

// Fixed layout (int32 offsets) of the per-ubatch upload buffer, so captured graphs can keep
// pointers into it: a header, the per-token / per-tile / per-work-item arrays at capacity, then
// the cell lists.
struct InLayout {
    size_t hdr, tok, pos, slot, out_rows, perm, tile_desc, wi_desc, fixed_end, list_cells, list_pos,
        total;
    size_t lcap = 0;
};

// Record of one ubatch for the debug hooks.
struct UbDebug {
    int32_t n_kv = 0;
    std::vector<int32_t> pos, tok_list, list_off, list_cells, list_pos;
};

}  // namespace

struct llm_ctx {
    llm_hparams hp{};
    int32_t n_ctx = 0, n_seq_max = 1, n_batch = 0, n_ubatch = 0, type_k = 1, type_v = 1;
    bool host_only = false;
    int device = 0, n_sm = 148;
    cudaStream_t st = nullptr;
    bool own_stream = false;
    std::string err;

    // weights
    std::vector<Layer> layers;
    DevMat embd, out;
    float* out_norm = nullptr;
    bool embd_loaded = false, out_loaded = false, out_norm_loaded = false, ready = false;
    std::vector<void*> allocs;

    // KV cache: K and V each [n_layer][Hkv][n_ctx][hd] (Q8_0: per layer the quants, then the scales)
    void* kv_k = nullptr;
    void* kv_v = nullptr;
    float* kv_stage = nullptr;                 // Q8_0: this ubatch's K and V rows, [2][Hkv][n_ubatch][hd]
    uint16_t* kv_f16 = nullptr;                // Q8_0: one layer's cache as f16 values, [2][Hkv][n_ctx][hd]
    uint8_t* kv_scratch = nullptr;             // defrag: one cache region's moved rows
    int32_t* d_order = nullptr;                // defrag: old cell of each new cell
    KvCells cells;

    // scratch for one ubatch
    float *x = nullptr, *h = nullptr, *qkv = nullptr, *attn = nullptr, *u = nullptr, *tmp = nullptr;
    float *hout = nullptr;
    float2* rope_cs = nullptr;
    double* d_theta = nullptr;                 // RoPE frequencies base^(-2i/hd), i < hd/2
    // bf16 activations feeding the tensor-core GEMM, and their TMA maps (token box 128 / 256)
    void *hb = nullptr, *attnb = nullptr, *ub = nullptr, *hob = nullptr;
    void *hb_lo = nullptr, *attnb_lo = nullptr, *ub_lo = nullptr, *hob_lo = nullptr;
    CUtensorMap m_hb[2], m_attnb[2], m_ub[2], m_hob[2], m_lm;
    CUtensorMap m_hb_lo, m_attnb_lo, m_ub_lo, m_hob_lo;        // low terms (token box 128)
    bool tc_ok = false;                        // tensor-core prefill GEMMs for the layers
    bool tc_f16 = false;                       // ... with f16 operands (one term each, token-major)
    CUtensorMap m_hh, m_ah, m_uh;              // f16 views of hb, attnb, ub (token box 128)
    CUtensorMap m_y_qkv, m_y_x, m_y_ub;        // outputs of the f16 token-major GEMMs (TMA-store epilogue)
    CUtensorMap m_kc, m_vc;                    // F16 K and V caches as [layers x Hkv x n_ctx][hd] rows
    bool kv_maps = false;
    bool tc_lm = false;                        // ... and for the output matrix
    float *part_o = nullptr, *part_m = nullptr, *part_l = nullptr;
    int32_t* tickets = nullptr;
    int32_t max_rows = 0;
    int32_t* d_in = nullptr;
    int32_t* h_in = nullptr;
    size_t in_cap = 0;
    InLayout io{};
    int32_t max_work = 0;
    uint32_t* d_err = nullptr;
    uint32_t* h_err = nullptr;

    // outputs of the last decode
    float* d_logits = nullptr;
    unsigned long long* d_amax = nullptr;
    int32_t out_cap = 0;
    std::vector<float> h_logits;
    std::vector<unsigned long long> h_amax;
    bool h_logits_valid = false, h_argmax_valid = false;
    std::vector<int32_t> output_ids;
    std::vector<int32_t> rows_by_rank;         // output row of the r-th output token in batch order
    int32_t n_stream = 1;                      // LLM_CTX_KV_SPLIT: one stream per sequence
    int32_t n_outputs = 0;

    // control, debug
    int (*abort_cb)(void*) = nullptr;
    void* abort_ud = nullptr;
    std::vector<int32_t> last_slots;
    bool debug = false;
    std::vector<UbDebug> dbg_ub;
    float *dbg_embd = nullptr, *dbg_lout = nullptr, *dbg_attn = nullptr, *dbg_q = nullptr;
    bool dbg_rnorm_valid = false;   // the final-normed rows exist only on the unfused output path
    float* dbg_rnorm = nullptr;
    float *dbg_kin = nullptr, *dbg_vin = nullptr;   // Q8_0 cache: the float32 K/V rows it was given
    int32_t dbg_T = 0, dbg_O = 0;
    int32_t fault_kind = 0, fault_ub = -1;
    llm_perf_data perf{};
    bool ktime = false;
    std::vector<cudaEvent_t> ev_pool;
    size_t ev_used = 0;
    std::vector<KPending> kpend;
    std::vector<KPending>* kcap = nullptr;     // set while capturing a timing graph
    std::vector<cudaEvent_t>* kcap_events = nullptr;
    KStat kstat[KC_COUNT];
    double att_bytes_now = 0, att_flops_now = 0;

    // decode-step graphs, per (tokens, outputs, output row, tile shape, timing, long lists) key
    bool use_graphs = true, use_pdl = true, use_bulk = true;
    // one-token ubatches as one persistent kernel (decode_step.cu)
    bool use_step = false, step_ok = false;
    bool dec_long = false;                     // this decode ubatch's longest list >= kDecLongList
    StepLayer* d_step_layers = nullptr;
    uint32_t* d_counters = nullptr;     // its grid-wide phase counters [1 + 5 n_layer]
    int32_t* d_abort = nullptr;
    uint32_t step_gen = 0;              // launches since the counters were last zeroed
    bool step_trace = false;
    uint8_t* d_sample_state = nullptr;  // sampler barrier, histograms and candidates
    int32_t* d_sample_tok = nullptr;    // [kMaxPenalty] penalty tokens, the picked token, status
    int32_t* h_sample_tok = nullptr;    // pinned: the same layout
    uint64_t* d_trace = nullptr;        // timeline of the last traced step
    int32_t trace_blocks = 0, trace_slots = 0;
    bool trace_valid = false;
    double step_weight_bytes = 0;
    std::map<uint64_t, StepGraph> graphs;

    SanBatch batch;
    AttnPlan plan;

    int32_t qkv_width() const { return (hp.n_head + 2 * hp.n_head_kv) * hp.head_dim; }
    int32_t q_width() const { return hp.n_head * hp.head_dim; }
    size_t kv_layer_elems() const { return (size_t)hp.n_head_kv * n_ctx * hp.head_dim; }
    bool kv_q8() const { return type_k == LLM_TYPE_Q8_0; }
    // bytes of one layer's K (or V) cache: Q8_0 keeps int8 quants, then one fp16 scale per 32 values
    size_t kv_layer_bytes() const {
        return kv_q8() ? kv_layer_elems() / 32 * 34 : kv_layer_elems() * type_size(type_k);
    }
    double kv_value_bytes() const { return kv_q8() ? 34.0 / 32.0 : (double)type_size(type_k); }
};

namespace {

bool cuda_ok(llm_ctx* c, cudaError_t e, const char* what) {
    if (e == cudaSuccess) return true;
    c->err = std::string(what) + ": " + cudaGetErrorString(e);
    return false;
}

template <typename T>
bool dalloc(llm_ctx* c, T** p, size_t n) {
    *p = nullptr;
    if (n == 0) n = 1;
    void* q = nullptr;
    if (!cuda_ok(c, cudaMalloc(&q, n * sizeof(T)), "cudaMalloc")) return false;
    c->allocs.push_back(q);
    *p = static_cast<T*>(q);
    return true;
}

void dfree(llm_ctx* c, void* p) {
    if (!p) return;
    cudaFree(p);
    c->allocs.erase(std::remove(c->allocs.begin(), c->allocs.end(), p), c->allocs.end());
}

bool alloc_mat(llm_ctx* c, DevMat& m, int32_t type, int64_t rows, int64_t cols) {
    m.type = type;
    m.rows = rows;
    m.cols = cols;
    if (type == LLM_TYPE_Q8_0) {
        int8_t* q = nullptr;
        if (!dalloc(c, &q, (size_t)(rows * cols))) return false;
        if (!dalloc(c, &m.scales, (size_t)(rows * cols / 32))) return false;
        m.data = q;
        c->perf.weight_device_bytes += rows * cols + rows * cols / 32 * 2;
        return true;
    }
    uint8_t* p = nullptr;
    if (!dalloc(c, &p, (size_t)(rows * cols) * type_size(type))) return false;
    m.data = p;
    c->perf.weight_device_bytes += rows * cols * (int64_t)type_size(type);
    return true;
}

// Copy rows (storage format `type`) into rows [row0, row0 + rows) of m.
bool fill_rows(llm_ctx* c, DevMat& m, int64_t row0, int64_t rows, const void* data, size_t nbytes) {
    if (m.type == LLM_TYPE_Q8_0) {
        uint8_t* tmpb = nullptr;
        if (!cuda_ok(c, cudaMalloc(&tmpb, nbytes), "cudaMalloc")) return false;
        bool ok = cuda_ok(c, cudaMemcpyAsync(tmpb, data, nbytes, cudaMemcpyDefault, c->st), "copy");
        if (ok) {
            launch_q8_0_unpack(tmpb, rows, m.cols,
                               static_cast<int8_t*>(m.data) + row0 * m.cols,
                               m.scales + row0 * (m.cols / 32), c->st);
            ok = cuda_ok(c, cudaGetLastError(), "q8_0 unpack") &&
                 cuda_ok(c, cudaStreamSynchronize(c->st), "sync");
        }
        cudaFree(tmpb);
        return ok;
    }
    uint8_t* dst = static_cast<uint8_t*>(m.data) + (size_t)row0 * m.cols * type_size(m.type);
    return cuda_ok(c, cudaMemcpyAsync(dst, data, nbytes, cudaMemcpyDefault, c->st), "copy") &&
           cuda_ok(c, cudaStreamSynchronize(c->st), "sync");
}

void drop_graphs(llm_ctx* c) {
    for (auto& kv : c->graphs) {
        if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
        for (cudaEvent_t e : kv.second.events) cudaEventDestroy(e);
    }
    c->graphs.clear();
}

InLayout make_layout(size_t U, size_t W, size_t L) {
    InLayout o{};
    size_t at = 0;
    auto take = [&](size_t n) { size_t r = at; at += (n + 31) / 32 * 32; return r; };
    o.hdr = take(8);
    o.tok = take(U); o.pos = take(U); o.slot = take(U); o.out_rows = take(U); o.perm = take(U);
    o.tile_desc = take(8 * U);
    o.wi_desc = take(4 * W);
    o.fixed_end = at;
    o.list_cells = take(L); o.list_pos = take(L);
    o.total = at;
    o.lcap = L;
    return o;
}

// Make room for `list_len` list entries in the upload buffer (reallocation drops the graphs,
// whose kernels hold pointers into it).
bool ensure_inputs(llm_ctx* c, size_t list_len) {
    if (c->d_in && list_len <= c->io.lcap) return true;
    const size_t L = std::max(list_len, c->io.lcap * 2);
    const InLayout io = make_layout((size_t)c->n_ubatch, (size_t)c->max_work, L);
    drop_graphs(c);
    if (c->h_in) cudaFreeHost(c->h_in);
    dfree(c, c->d_in);
    c->h_in = nullptr;
    c->d_in = nullptr;
    c->io = InLayout{};
    if (!cuda_ok(c, cudaMallocHost(&c->h_in, io.total * sizeof(int32_t)), "cudaMallocHost")) return false;
    if (!dalloc(c, &c->d_in, io.total)) return false;
    std::memset(c->h_in, 0, io.total * sizeof(int32_t));
    c->io = io;
    return true;
}

bool ensure_outputs(llm_ctx* c, int32_t n) {
    if (n <= c->out_cap) return true;
    drop_graphs(c);
    dfree(c, c->d_logits);
    dfree(c, c->d_amax);
    c->d_logits = nullptr;
    c->d_amax = nullptr;
    c->out_cap = 0;
    if (!dalloc(c, &c->d_logits, (size_t)n * c->hp.n_vocab)) return false;
    if (!dalloc(c, &c->d_amax, (size_t)n)) return false;
    c->out_cap = n;
    return true;
}

void rollback(llm_ctx* c, int32_t i0, int32_t T) {
    // [P4] エラーリカバリ: per sequence the smallest position of the ubatch, then seq_rm(s, pos_min, -1)
    std::vector<int32_t> pmin(c->n_seq_max, INT32_MAX);
    const SanBatch& b = c->batch;
    for (int32_t i = i0; i < i0 + T; ++i)
        for (int32_t s = 0; s < c->n_seq_max; ++s)
            if (b.seqs[i].test(s)) pmin[s] = std::min(pmin[s], b.pos[i]);
    for (int32_t s = 0; s < c->n_seq_max; ++s)
        if (pmin[s] != INT32_MAX) c->cells.seq_rm(s, pmin[s], -1);
}

// ---- kernel timing --------------------------------------------------------------------------
int kt_begin(llm_ctx* c) {
    if (!c->ktime) return -1;
    if (c->kcap) {                                   // capturing a timing graph
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess) return -1;
        if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return -1; }
        c->kcap_events->push_back(a);
        c->kcap_events->push_back(b);
        cudaEventRecordWithFlags(a, c->st, cudaEventRecordExternal);
        c->kcap->push_back({-1, a, b, 0, 0});
        return (int)c->kcap->size() - 1;
    }
    while (c->ev_pool.size() < c->ev_used + 2) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return -1;
        c->ev_pool.push_back(e);
    }
    const int i = (int)c->ev_used;
    c->ev_used += 2;
    cudaEventRecord(c->ev_pool[i], c->st);
    return i;
}

// bytes < 0 marks the attention, whose bytes depend on the step's context (taken at collection)
void kt_end(llm_ctx* c, int i, int32_t cls, double bytes, double flops) {
    if (i < 0) return;
    if (c->kcap) {
        KPending& p = (*c->kcap)[i];
        cudaEventRecordWithFlags(p.b, c->st, cudaEventRecordExternal);
        p.cls = cls;
        p.bytes = bytes;
        p.flops = flops;
        return;
    }
    cudaEventRecord(c->ev_pool[i + 1], c->st);
    c->kpend.push_back({cls, c->ev_pool[i], c->ev_pool[i + 1], bytes, flops});
}

void kt_fold(llm_ctx* c, const std::vector<KPending>& v) {
    for (const KPending& p : v) {
        float ms = 0.f;
        if (p.cls < 0 || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) continue;
        KStat& s = c->kstat[p.cls];
        s.launches += 1;
        s.ms += ms;
        s.bytes += p.bytes < 0 ? c->att_bytes_now : p.bytes;
        s.flops += p.bytes < 0 ? c->att_flops_now : p.flops;
    }
}

// After the stream is synchronised: fold the pending event pairs into the counters.
void kt_collect(llm_ctx* c, const StepGraph* g) {
    if (g) kt_fold(c, g->timing);
    kt_fold(c, c->kpend);
    c->kpend.clear();
    c->ev_used = 0;
}

double wbytes(const DevMat& W, int64_t rows) { return (double)rows * (double)row_bytes(W.type, W.cols); }

void put(int32_t* base, size_t off, const std::vector<int32_t>& v) {
    if (!v.empty()) std::memcpy(base + off, v.data(), v.size() * sizeof(int32_t));
}

// Algorithmic bytes / FLOPs of the attention of the current plan (for the kernel counters).
void attention_work(llm_ctx* c, const int32_t* pos) {
    const AttnPlan& p = c->plan;
    const llm_hparams& hp = c->hp;
    // multi-token tiles over a Q8_0 cache read the f16 copy of its quants and its scales
    const double kv_es = c->kv_q8() && p.max_nq > 1 ? 2.0 + 2.0 / 32.0 : c->kv_value_bytes();
    double by = 0, fl = 0;
    for (int32_t t = 0; t < p.n_tiles(); ++t) {
        const int32_t l = p.tile_list[t];
        by += (double)(p.list_off[l + 1] - p.list_off[l]) * 2.0 * hp.n_head_kv * hp.head_dim * kv_es;
    }
    const int32_t T = (int32_t)p.tok_list.size();
    by += (double)T * hp.n_head * hp.head_dim * 8.0;
    for (int32_t t = 0; t < T; ++t) {
        const int32_t l = p.tok_list[t];
        int64_t vis = 0;
        for (int32_t k = p.list_off[l]; k < p.list_off[l + 1]; ++k) vis += p.list_pos[k] <= pos[t];
        fl += 4.0 * (double)vis * hp.n_head * hp.head_dim;
    }
    c->att_bytes_now = by;
    c->att_flops_now = fl;
}

// Attention work items a decode-shaped ubatch of T tokens may use (the captured grid size).
int32_t attn_cap(llm_ctx* c, int32_t T) {
    return std::min(c->max_work, std::max(T, 4 * c->n_sm / c->hp.n_head_kv));
}

// Which decode-GEMV variant serves each op of a T-token ubatch.
struct OpPaths { bool qkv, wo, gu, down, lm; };

OpPaths op_paths(llm_ctx* c, int32_t T, int32_t O) {
    OpPaths o{false, false, false, false, false};
    if (!c->use_bulk) return o;
    const llm_hparams& h = c->hp;
    const Layer& L = c->layers[0];
    GemvArgs a;
    // the output matrix sees only the O flagged rows: the GEMV serves it after a prefill too
    a.T = std::max(O, 1); a.K = h.n_embd; a.M = h.n_vocab;
    o.lm = O > 0 && O <= gemv_max_tokens() && gemv_bulk_ok(c->out.type, a, GEPI_LOGITS, c->n_sm);
    if (T > gemv_max_tokens()) return o;
    a.T = T;
    a.K = h.n_embd; a.M = c->qkv_width(); o.qkv = gemv_bulk_ok(L.qkv.type, a, GEPI_QKV, c->n_sm);
    a.K = c->q_width(); a.M = h.n_embd; o.wo = gemv_bulk_ok(L.wo.type, a, GEPI_ADD, c->n_sm);
    a.K = h.n_embd; a.F = h.n_ff; o.gu = gemv_bulk_ok(L.gu.type, a, GEPI_SWIGLU, c->n_sm);
    a.K = h.n_ff; a.M = h.n_embd; o.down = gemv_bulk_ok(L.down.type, a, GEPI_ADD, c->n_sm);
    // every layer must share the types of layer 0 for the choice to hold
    for (int32_t il = 1; il < h.n_layer; ++il) {
        const Layer& M = c->layers[il];
        if (M.qkv.type != L.qkv.type || M.wo.type != L.wo.type || M.gu.type != L.gu.type ||
            M.down.type != L.down.type)
            return OpPaths{false, false, false, false, false};
    }
    return o;
}

// Enqueue the forward pass of one ubatch ([P2] Example 4 op chain; [P1] Крок 13б layer scheme).
// Everything that varies between ubatches of the same shape (tokens, positions, cells, lists,
// the attention split) is read from the upload buffer, so the sequence can be captured once and
// replayed.
bool forward_ubatch(llm_ctx* c, int32_t T, int32_t O, int32_t out_row0, int32_t max_nq) {
    const llm_hparams& hp = c->hp;
    cudaStream_t st = c->st;
    const InLayout& io = c->io;
    const int32_t d = hp.n_embd, H = hp.n_head, Hkv = hp.n_head_kv, hd = hp.head_dim, F = hp.n_ff;
    const int32_t* din = c->d_in;
    const int32_t *tok = din + io.tok, *pos = din + io.pos, *slot = din + io.slot;
    const double kv_es = c->kv_value_bytes();
    const bool q8 = c->kv_q8();
    const int32_t U = c->n_ubatch;
    float* stage_k = c->kv_stage;
    float* stage_v = q8 ? c->kv_stage + (size_t)Hkv * U * hd : nullptr;
    const bool gemv = T <= gemv_max_tokens();
    const int32_t lin_cls = gemv ? KC_LINEAR_GEMV : (c->tc_ok ? KC_LINEAR_TC : KC_LINEAR_GEMM);
    const double Td = T, Od = O;
    const int qw = c->q_width(), qkvw = c->qkv_width();
    const OpPaths bulk = op_paths(c, T, O);
    const bool pdl = c->use_pdl;
    unsigned long long* amax = c->d_amax + out_row0;

    int k;
    k = kt_begin(c);
    launch_embed_rope(c->embd, tok, pos, T, hd, c->d_theta, c->x, c->rope_cs, amax, O, c->d_err, st);
    kt_end(c, k, KC_EMBED, Td * d * 8.0 + Td * hd * 4.0, 0);
    if (c->debug) cudaMemcpyAsync(c->dbg_embd, c->x, sizeof(float) * T * d, cudaMemcpyDeviceToDevice, st);

    AttnArgs a{};
    a.ldq = qkvw;
    a.q = c->qkv;
    a.n_ctx = c->n_ctx;
    a.kv_type = c->type_k;
    a.H = H; a.Hkv = Hkv; a.hd = hd;
    a.tok_pos = pos;
    a.list_cells = din + io.list_cells; a.list_pos = din + io.list_pos;
    a.perm = din + io.perm;
    a.tile_desc = reinterpret_cast<const int4*>(din + io.tile_desc);
    a.wi_desc = reinterpret_cast<const int4*>(din + io.wi_desc);
    a.tickets = c->tickets;
    a.part_o = c->part_o; a.part_m = c->part_m; a.part_l = c->part_l;
    a.out = c->attn;
    a.ldo = qw;
    a.hdr = din + io.hdr;
    a.n_work = gemv ? attn_cap(c, T) : c->plan.n_work();  // grid bound (the device count decides)
    a.max_nq = max_nq;
    a.tile_q = max_nq > 1 ? max_nq : kAttnTileQ;
    a.err = c->d_err;
    // prefill with f16 GEMM operands chains its kernels with programmatic dependent launch too
    const bool pdl_pre = c->use_pdl && !gemv && c->tc_ok && c->tc_f16 && !c->ktime;
    a.pdl = (c->use_pdl && gemv) || pdl_pre;
    a.slot = slot;                                   // tiles of one token use the cluster decode kernel
    a.n_tok = T;
    a.long_lists = gemv && c->dec_long;

    GemvArgs g{};
    g.T = T;
    g.eps = hp.rms_eps;
    g.err = c->d_err;

    const double norm_bytes = Td * d * 8.0 + d * 4.0;
    // tensor-core prefill GEMMs: f16 operands (one term each), or activations as split bf16 (hi +
    // lo) operands; box 128 tokens
    const bool tc = !gemv && c->tc_ok;
    const bool f16 = tc && c->tc_f16;
    const int bi = 0;
    if (tc) { a.out_b = c->attnb; a.out_b_lo = f16 ? nullptr : c->attnb_lo; a.out_f16 = f16; }
    // store / residual add: the token-major GEMM when the weight rows come in 256-row tiles
    // (split-K with atomic adds when the tiles alone leave SMs idle), else the weight-major one
    auto tc_gemm = [&](const CUtensorMap& wm, const CUtensorMap& xm, int epi, int K, int M, void* Y,
                       int ldy, const uint32_t* q8s) {
        const CUtensorMap* xlo = f16 ? nullptr
                               : &xm == &c->m_hb[bi] ? &c->m_hb_lo
                               : &xm == &c->m_attnb[bi] ? &c->m_attnb_lo : &c->m_ub_lo;
        if (epi != GEMM_EPI_SWIGLU && tc_tn_ok(M, K)) {
            const int splits = tc_tn_splits(M, K, T, c->n_sm);
            if (splits > 1 && epi == GEMM_EPI_STORE &&
                !cuda_ok(c, cudaMemsetAsync(Y, 0, sizeof(float) * (size_t)T * ldy, st), "memset"))
                return false;
            const CUtensorMap* ym = !f16 ? nullptr : Y == c->qkv ? &c->m_y_qkv : Y == c->x ? &c->m_y_x : nullptr;
            if (!launch_gemm_tn(xm, xlo, wm, epi, K, M, T, static_cast<float*>(Y), ldy, splits, c->d_err, st,
                                nullptr, false, ym, nullptr, pdl_pre && !(splits > 1 && epi == GEMM_EPI_STORE),
                                q8s)) {
                c->err = "tensor-core GEMM launch failed";
                return false;
            }
            return true;
        }
        const CUtensorMap* lo = &xm == &c->m_hb[bi] ? &c->m_hb_lo
                              : &xm == &c->m_attnb[bi] ? &c->m_attnb_lo : &c->m_ub_lo;
        void* y2 = epi == GEMM_EPI_SWIGLU ? c->ub_lo : nullptr;
        if (!launch_gemm_tc(wm, xm, epi, K, M, T, F, Y, ldy, c->d_err, st, lo, y2)) {
            c->err = "tensor-core GEMM launch failed";
            return false;
        }
        return true;
    };
    auto bulk_fail = [&]() { c->err = "decode GEMV launch failed"; return false; };
    for (int32_t il = 0; il < hp.n_layer; ++il) {
        Layer& L = c->layers[il];
        void* kc = static_cast<uint8_t*>(c->kv_k) + (size_t)il * c->kv_layer_bytes();
        void* vc = static_cast<uint8_t*>(c->kv_v) + (size_t)il * c->kv_layer_bytes();
        // ---- attention norm, Q/K/V, RoPE, K/V append
        if (bulk.qkv) {
            k = kt_begin(c);
            g.W = L.qkv.data; g.S = L.qkv.scales; g.row0 = 0; g.M = qkvw; g.K = d;
            g.x = c->x; g.ldx = d; g.x_rows = nullptr; g.g = L.attn_norm;
            g.y = c->qkv; g.ldy = qkvw;
            g.H = H; g.Hkv = Hkv; g.hd = hd; g.n_ctx = c->n_ctx; g.kv_type = c->type_k;
            g.cs = c->rope_cs; g.slot = slot; g.kc = kc; g.vc = vc;
            if (q8) {                               // float32 rows to the staging area, cell = token
                g.kv_type = W_F32; g.n_ctx = U; g.slot = nullptr; g.kc = stage_k; g.vc = stage_v;
            }
            if (!launch_gemv_bulk(L.qkv.type, g, GEPI_QKV, true, c->n_sm, st, pdl)) return bulk_fail();
            kt_end(c, k, lin_cls, wbytes(L.qkv, qkvw) + Td * (d * 4.0 + qw * 4.0 + 2.0 * Hkv * hd * (q8 ? 4.0 : kv_es)),
                   2.0 * Td * qkvw * d);
            if (q8) {
                k = kt_begin(c);
                launch_kv_quant_q8(stage_k, stage_v, U, T, Hkv, hd, slot, kc, vc, c->n_ctx, c->d_err, st, pdl);
                kt_end(c, k, KC_ROPE_KV, Td * 2.0 * Hkv * hd * (4.0 + kv_es), 0);
            }
        } else {
            k = kt_begin(c);
            if (f16) launch_rmsnorm_f16(c->x, nullptr, T, d, L.attn_norm, hp.rms_eps, c->hb, st, pdl_pre && il > 0);
            else if (tc) launch_rmsnorm_bf16(c->x, nullptr, T, d, L.attn_norm, hp.rms_eps, c->hb, c->hb_lo, st);
            else launch_rmsnorm(c->x, nullptr, T, d, L.attn_norm, hp.rms_eps, c->h, st);
            kt_end(c, k, KC_RMSNORM, norm_bytes, 0);
            // F16 cache, f16 GEMM operands: RoPE and the K/V append run in the GEMM's epilogue
            const bool fused_qkv = f16 && !q8 && c->type_k == LLM_TYPE_F16 && c->type_v == LLM_TYPE_F16 &&
                                   tc_tn_qkv_ok(H, Hkv, hd) && tc_tn_ok(qkvw, d);
            k = kt_begin(c);
            if (fused_qkv) {
                TnQkv qe;
                qe.cs = c->rope_cs; qe.slot = slot; qe.kc = kc; qe.vc = vc;
                qe.n_ctx = c->n_ctx; qe.H = H; qe.Hkv = Hkv; qe.hd = hd;
                if (!launch_gemm_tn(c->m_hh, nullptr, L.mq, GEMM_EPI_QKV, d, qkvw, T, c->qkv, qkvw, 1, c->d_err, st,
                                    nullptr, false, &c->m_y_qkv, &qe, pdl_pre, L.q8_tc ? L.qkv_ks : nullptr)) {
                    c->err = "tensor-core GEMM launch failed";
                    return false;
                }
            } else if (tc) {
                if (!tc_gemm(L.mq, f16 ? c->m_hh : c->m_hb[bi], GEMM_EPI_STORE, d, qkvw, c->qkv, qkvw,
                             L.q8_tc ? L.qkv_ks : nullptr))
                    return false;
            }
            else launch_linear(L.qkv, 0, qkvw, c->h, d, T, c->qkv, qkvw, EPI_STORE, st);
            kt_end(c, k, lin_cls, wbytes(L.qkv, qkvw) + Td * (d + qkvw) * 4.0, 2.0 * Td * qkvw * d);
            if (!fused_qkv) {
                k = kt_begin(c);
                if (q8) {
                    launch_rope_kv_append(c->qkv, T, H, Hkv, hd, c->rope_cs, nullptr, stage_k, stage_v, U,
                                          W_F32, c->d_err, st);
                    launch_kv_quant_q8(stage_k, stage_v, U, T, Hkv, hd, slot, kc, vc, c->n_ctx, c->d_err, st, false);
                } else {
                    launch_rope_kv_append(c->qkv, T, H, Hkv, hd, c->rope_cs, slot, kc, vc, c->n_ctx,
                                          c->type_k, c->d_err, st);
                }
                kt_end(c, k, KC_ROPE_KV, Td * ((double)qkvw * 4.0 + qw * 4.0 + 2.0 * Hkv * hd * kv_es), 0);
            }
        }
        if (c->debug && q8) {                       // staging [Hkv][U][hd] -> [T][Hkv * hd]
            const size_t kw = (size_t)Hkv * hd;
            for (int32_t g2 = 0; g2 < Hkv; ++g2) {
                cudaMemcpy2DAsync(c->dbg_kin + (size_t)il * T * kw + (size_t)g2 * hd, sizeof(float) * kw,
                                  stage_k + (size_t)g2 * U * hd, sizeof(float) * hd, sizeof(float) * hd, T,
                                  cudaMemcpyDeviceToDevice, st);
                cudaMemcpy2DAsync(c->dbg_vin + (size_t)il * T * kw + (size_t)g2 * hd, sizeof(float) * kw,
                                  stage_v + (size_t)g2 * U * hd, sizeof(float) * hd, sizeof(float) * hd, T,
                                  cudaMemcpyDeviceToDevice, st);
            }
        }
        // ---- attention over the cache
        a.kc = kc;
        a.vc = vc;
        a.kmap = c->kv_maps ? &c->m_kc : nullptr;
        a.vmap = c->kv_maps ? &c->m_vc : nullptr;
        a.kv_row0 = il * Hkv * c->n_ctx;
        a.k_scale = a.v_scale = nullptr;
        if (q8 && max_nq > 1) {
            // query tiles of several tokens run on tensor cores over f16 copies of the quants of
            // the cells in use and the cache's own scales; one-token tiles read the blocks directly
            const double nkv = c->cells.n_kv();
            k = kt_begin(c);
            launch_kv_q8_to_f16(kc, vc, c->kv_f16, Hkv, c->n_ctx, hd, din + io.hdr + 2, st);
            kt_end(c, k, KC_ROPE_KV, nkv * 2.0 * Hkv * hd * 3.0, 0);
            a.kc = c->kv_f16;
            a.vc = c->kv_f16 + (size_t)Hkv * c->n_ctx * hd;
            a.k_scale = static_cast<const uint8_t*>(kc) + kv_q8_scale_offset(Hkv, c->n_ctx, hd);
            a.v_scale = static_cast<const uint8_t*>(vc) + kv_q8_scale_offset(Hkv, c->n_ctx, hd);
        }
        k = kt_begin(c);
        if (!launch_attention(a, st)) { c->err = "attention shape not supported"; return false; }
        kt_end(c, k, KC_ATTENTION, -1.0, 0);
        if (c->debug) {
            cudaMemcpy2DAsync(c->dbg_q + (size_t)il * T * qw, sizeof(float) * qw, c->qkv,
                              sizeof(float) * qkvw, sizeof(float) * qw, T, cudaMemcpyDeviceToDevice, st);
            if (!tc)
                cudaMemcpyAsync(c->dbg_attn + (size_t)il * T * qw, c->attn, sizeof(float) * T * qw,
                                cudaMemcpyDeviceToDevice, st);
        }
        // ---- output projection + residual
        k = kt_begin(c);
        if (bulk.wo) {
            g.W = L.wo.data; g.S = L.wo.scales; g.row0 = 0; g.M = d; g.K = qw;
            g.x = c->attn; g.ldx = qw; g.x_rows = nullptr; g.g = nullptr; g.y = c->x; g.ldy = d;
            if (!launch_gemv_bulk(L.wo.type, g, GEPI_ADD, false, c->n_sm, st, pdl)) return bulk_fail();
        } else if (tc) {
            if (!tc_gemm(L.mo, f16 ? c->m_ah : c->m_attnb[bi], GEMM_EPI_ADD, qw, d, c->x, d,
                         L.q8_tc ? L.wo_ks : nullptr))
                return false;
        } else {
            launch_linear(L.wo, 0, d, c->attn, qw, T, c->x, d, EPI_ADD, st);
        }
        kt_end(c, k, lin_cls, wbytes(L.wo, d) + Td * (qw + 2.0 * d) * 4.0, 2.0 * Td * d * qw);
        // ---- FFN norm, gate/up, SwiGLU
        if (bulk.gu) {
            k = kt_begin(c);
            g.W = L.gu.data; g.S = L.gu.scales; g.row0 = 0; g.F = F; g.K = d;
            g.x = c->x; g.ldx = d; g.x_rows = nullptr; g.g = L.ffn_norm; g.y = c->u; g.ldy = F;
            if (!launch_gemv_bulk(L.gu.type, g, GEPI_SWIGLU, true, c->n_sm, st, pdl)) return bulk_fail();
            kt_end(c, k, lin_cls, wbytes(L.gu, 2 * (int64_t)F) + Td * (d + F) * 4.0, 4.0 * Td * F * d);
        } else {
            k = kt_begin(c);
            if (f16) launch_rmsnorm_f16(c->x, nullptr, T, d, L.ffn_norm, hp.rms_eps, c->hb, st, pdl_pre);
            else if (tc) launch_rmsnorm_bf16(c->x, nullptr, T, d, L.ffn_norm, hp.rms_eps, c->hb, c->hb_lo, st);
            else launch_rmsnorm(c->x, nullptr, T, d, L.ffn_norm, hp.rms_eps, c->h, st);
            kt_end(c, k, KC_RMSNORM, norm_bytes, 0);
            k = kt_begin(c);
            if (tc && L.gu_tn) {
                if (!launch_gemm_swiglu_tn(f16 ? c->m_hh : c->m_hb[bi], f16 ? nullptr : &c->m_hb_lo, L.mgu128, d, T,
                                           F, c->ub, f16 ? nullptr : c->ub_lo, F, c->d_err, st,
                                           nullptr, false, f16 ? &c->m_y_ub : nullptr, pdl_pre,
                                           L.q8_tc ? L.gu_ks : nullptr)) {
                    c->err = "tensor-core GEMM launch failed";
                    return false;
                }
            } else if (tc) { if (!tc_gemm(L.mgu, c->m_hb[bi], GEMM_EPI_SWIGLU, d, 0, c->ub, F, nullptr)) return false; }
            else launch_linear_swiglu(L.gu, F, c->h, d, T, c->u, F, c->tmp, st);
            kt_end(c, k, lin_cls, wbytes(L.gu, 2 * (int64_t)F) + Td * (d + F) * 4.0, 4.0 * Td * F * d);
        }
        // ---- down projection + residual
        k = kt_begin(c);
        if (bulk.down) {
            g.W = L.down.data; g.S = L.down.scales; g.row0 = 0; g.M = d; g.K = F;
            g.x = c->u; g.ldx = F; g.x_rows = nullptr; g.g = nullptr; g.y = c->x; g.ldy = d;
            if (!launch_gemv_bulk(L.down.type, g, GEPI_ADD, false, c->n_sm, st, pdl)) return bulk_fail();
        } else if (tc) {
            if (!tc_gemm(L.md, f16 ? c->m_uh : c->m_ub[bi], GEMM_EPI_ADD, F, d, c->x, d,
                         L.q8_tc ? L.down_ks : nullptr))
                return false;
        } else {
            launch_linear(L.down, 0, d, c->u, F, T, c->x, d, EPI_ADD, st);
        }
        kt_end(c, k, lin_cls, wbytes(L.down, d) + Td * (F + 2.0 * d) * 4.0, 2.0 * Td * d * F);
        if (c->debug)
            cudaMemcpyAsync(c->dbg_lout + (size_t)il * T * d, c->x, sizeof(float) * T * d,
                            cudaMemcpyDeviceToDevice, st);
    }
    if (O > 0) {
        // keep only the requested rows, final norm, output matrix, greedy pick ([P1] Крок 13б)
        float* lg = c->d_logits + (size_t)out_row0 * hp.n_vocab;
        const int32_t* orows = din + io.out_rows;
        const double lm_bytes = wbytes(c->out, hp.n_vocab) + Od * (d + (double)hp.n_vocab) * 4.0;
        c->dbg_rnorm_valid = false;
        if (bulk.lm) {
            k = kt_begin(c);
            g.T = O;
            g.W = c->out.data; g.S = c->out.scales; g.row0 = 0; g.M = hp.n_vocab; g.K = d;
            g.x = c->x; g.ldx = d; g.x_rows = orows; g.g = c->out_norm; g.y = lg; g.ldy = hp.n_vocab;
            g.amax = amax;
            if (!launch_gemv_bulk(c->out.type, g, GEPI_LOGITS, true, c->n_sm, st, pdl)) return bulk_fail();
            kt_end(c, k, KC_LM_HEAD, lm_bytes, 2.0 * Od * hp.n_vocab * d);
        } else {
            const bool tc_out = tc && c->tc_lm && O > gemv_max_tokens();
            k = kt_begin(c);
            if (tc_out) launch_rmsnorm_bf16(c->x, orows, O, d, c->out_norm, hp.rms_eps, c->hob, c->hob_lo, st);
            launch_rmsnorm(c->x, orows, O, d, c->out_norm, hp.rms_eps, c->hout, st);
            kt_end(c, k, KC_RMSNORM, Od * d * 8.0 + d * 4.0, 0);
            if (c->debug) {
                cudaMemcpyAsync(c->dbg_rnorm, c->hout, sizeof(float) * O * d, cudaMemcpyDeviceToDevice, st);
                c->dbg_rnorm_valid = true;
            }
            k = kt_begin(c);
            if (tc_out) {
                if (!launch_gemm_tc(c->m_lm, c->m_hob[0], GEMM_EPI_STORE, d, hp.n_vocab, O, F, lg,
                                    hp.n_vocab, c->d_err, st, &c->m_hob_lo)) {
                    c->err = "tensor-core GEMM launch failed";
                    return false;
                }
            } else {
                launch_linear(c->out, 0, hp.n_vocab, c->hout, d, O, lg, hp.n_vocab, EPI_STORE, st);
            }
            kt_end(c, k, KC_LM_HEAD, lm_bytes, 2.0 * Od * hp.n_vocab * d);
            k = kt_begin(c);
            launch_argmax(lg, O, hp.n_vocab, amax, st);
            kt_end(c, k, KC_ARGMAX, Od * hp.n_vocab * 4.0, 0);
        }
    }
    c->dbg_T = T;
    c->dbg_O = O;
    return cuda_ok(c, cudaGetLastError(), "kernel launch");
}

bool parse_layer_name(const char* name, int32_t* il, std::string* part) {
    if (std::strncmp(name, "blk.", 4) != 0) return false;
    const char* p = name + 4;
    char* end = nullptr;
    const long v = std::strtol(p, &end, 10);
    if (end == p || *end != '.' || v < 0 || v > 100000) return false;
    std::string rest(end + 1);
    const std::string suffix = ".weight";
    if (rest.size() <= suffix.size() || rest.compare(rest.size() - suffix.size(), suffix.size(), suffix) != 0)
        return false;
    *il = (int32_t)v;
    *part = rest.substr(0, rest.size() - suffix.size());
    return true;
}

}  // namespace

// =============================================================================================
extern "C" {

llm_cparams llm_cparams_default(void) {
    llm_cparams p{};
    p.n_ctx = 4096;
    p.n_seq_max = 1;
    p.n_batch = 2048;
    p.n_ubatch = 512;
    p.type_k = LLM_TYPE_F16;
    p.type_v = LLM_TYPE_F16;
    p.stream = nullptr;
    p.flags = 0;
    return p;
}

llm_ctx* llm_ctx_init(const llm_hparams* hp, const llm_cparams* cp) {
    g_init_error.clear();
    auto fail = [](const std::string& m) -> llm_ctx* { g_init_error = m; return nullptr; };
    if (!hp || !cp) return fail("NULL parameters");
    const llm_hparams& h = *hp;
    if (h.n_layer <= 0 || h.n_embd <= 0 || h.n_head <= 0 || h.n_head_kv <= 0 || h.head_dim <= 0 ||
        h.n_ff <= 0 || h.n_vocab <= 0)
        return fail("hyper-parameters must be positive");
    if (h.n_head % h.n_head_kv != 0) return fail("n_head must be a multiple of n_head_kv");
    if (h.rope_type != 0) return fail("only rope type 0 (normal) is supported");
    if (h.n_embd % 32 != 0 || h.n_ff % 32 != 0) return fail("n_embd and n_ff must be multiples of 32");
    if (!attention_supported(h.head_dim, h.n_head / h.n_head_kv))
        return fail("attention kernels support head_dim 32/64/128 with n_head/n_head_kv = 4");
    if (!(h.rms_eps >= 0.f) || !(h.rope_freq_base > 0.f)) return fail("bad rms_eps / rope_freq_base");
    if (cp->n_ctx == 0 || cp->n_batch == 0 || cp->n_ubatch == 0) return fail("zero context size");
    if (cp->n_seq_max < 1 || cp->n_seq_max > (uint32_t)kMaxSeq) return fail("n_seq_max out of range");
    if ((cp->type_k != LLM_TYPE_F32 && cp->type_k != LLM_TYPE_F16 && cp->type_k != LLM_TYPE_Q8_0) ||
        cp->type_v != cp->type_k)
        return fail("type_k/type_v must both be F32, both F16 or both Q8_0");
    if (cp->n_ctx > (1u << 24)) return fail("n_ctx too large");

    auto* c = new llm_ctx();
    c->hp = h;
    c->n_ctx = (int32_t)((cp->n_ctx + 255) / 256 * 256);          // GGML_PAD(n_ctx, 256)
    c->n_batch = (int32_t)std::min<uint32_t>(cp->n_batch, (uint32_t)c->n_ctx);
    c->n_ubatch = (int32_t)std::min<uint32_t>(cp->n_ubatch, (uint32_t)c->n_batch);
    c->n_seq_max = (int32_t)cp->n_seq_max;
    c->type_k = cp->type_k;
    c->type_v = cp->type_v;
    c->host_only = (cp->flags & LLM_CTX_HOST_ONLY) != 0;
    c->use_step = (cp->flags & LLM_CTX_FUSED_STEP) != 0;
    c->n_stream = (cp->flags & LLM_CTX_KV_SPLIT) ? c->n_seq_max : 1;
    c->cells = KvCells(c->n_ctx, c->n_seq_max, c->n_stream);
    c->layers.resize(h.n_layer);
    if (c->host_only) return c;

    auto die = [&](const std::string& m) -> llm_ctx* {
        g_init_error = m.empty() ? c->err : m;
        llm_ctx_free(c);
        return nullptr;
    };
    if (!cuda_ok(c, cudaGetDevice(&c->device), "cudaGetDevice")) return die("");
    cudaDeviceGetAttribute(&c->n_sm, cudaDevAttrMultiProcessorCount, c->device);
    if (cp->stream) {
        c->st = static_cast<cudaStream_t>(cp->stream);
    } else {
        if (!cuda_ok(c, cudaStreamCreateWithFlags(&c->st, cudaStreamNonBlocking), "stream")) return die("");
        c->own_stream = true;
    }
    const int64_t U = c->n_ubatch, d = h.n_embd;
    const int G = h.n_head / h.n_head_kv;
    const size_t kv_bytes = (size_t)h.n_layer * c->kv_layer_bytes();
    bool ok = dalloc(c, reinterpret_cast<uint8_t**>(&c->kv_k), kv_bytes) &&
              dalloc(c, reinterpret_cast<uint8_t**>(&c->kv_v), kv_bytes) &&
              (!c->kv_q8() || dalloc(c, &c->kv_stage, 2 * (size_t)h.n_head_kv * U * h.head_dim)) &&
              (!c->kv_q8() || dalloc(c, &c->kv_f16, 2 * (size_t)h.n_head_kv * c->n_ctx * h.head_dim)) &&
              dalloc(c, &c->x, U * d) && dalloc(c, &c->h, U * d) &&
              dalloc(c, &c->qkv, U * c->qkv_width()) && dalloc(c, &c->attn, U * c->q_width()) &&
              dalloc(c, &c->u, U * h.n_ff) && dalloc(c, &c->tmp, U * 2 * (int64_t)h.n_ff) &&
              dalloc(c, &c->hout, U * d) && dalloc(c, &c->rope_cs, U * (h.head_dim / 2)) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->hb), U * d) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->attnb), U * c->q_width()) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->ub), U * (int64_t)h.n_ff) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->hob), U * d) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->hb_lo), U * d) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->attnb_lo), U * c->q_width()) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->ub_lo), U * (int64_t)h.n_ff) &&
              dalloc(c, reinterpret_cast<uint16_t**>(&c->hob_lo), U * d) &&
              dalloc(c, &c->d_err, 1) &&
              dalloc(c, &c->d_counters, 1 + 5 * (size_t)h.n_layer) && dalloc(c, &c->d_abort, 1) &&
              cuda_ok(c, cudaMemset(c->d_counters, 0, sizeof(uint32_t) * (1 + 5 * (size_t)h.n_layer)), "memset") &&
              cuda_ok(c, cudaMemset(c->d_abort, 0, sizeof(int32_t)), "memset") &&
              cuda_ok(c, cudaMallocHost(&c->h_err, sizeof(uint32_t)), "cudaMallocHost");
    if (!ok) return die("");
    {
        std::vector<double> th(h.head_dim / 2);
        for (int i = 0; i < h.head_dim / 2; ++i)
            th[i] = std::pow((double)h.rope_freq_base, -2.0 * i / (double)h.head_dim);
        ok = dalloc(c, &c->d_theta, th.size()) &&
             cuda_ok(c, cudaMemcpy(c->d_theta, th.data(), th.size() * sizeof(double),
                                   cudaMemcpyHostToDevice), "copy");
        if (!ok) return die("");
    }
    c->max_rows = (int32_t)std::max<int64_t>(2 * U * G, 8192);
    ok = dalloc(c, &c->tickets, (size_t)U * h.n_head_kv * kDecTicketsPerHead) &&
         cuda_ok(c, cudaMemset(c->tickets, 0, sizeof(int32_t) * U * h.n_head_kv * kDecTicketsPerHead), "memset") &&
         dalloc(c, &c->part_o, (size_t)c->max_rows * h.n_head_kv * h.head_dim) &&
         dalloc(c, &c->part_m, (size_t)c->max_rows * h.n_head_kv) &&
         dalloc(c, &c->part_l, (size_t)c->max_rows * h.n_head_kv) &&
         ensure_outputs(c, std::max<int32_t>(c->n_seq_max, (int32_t)std::min<int64_t>(U, 64))) &&
         (c->max_work = std::max<int32_t>((int32_t)U, c->max_rows / G), true) &&
         ensure_inputs(c, 2 * (size_t)c->n_ctx);
    if (!ok) return die("");
    // KV cells start zeroed so an unwritten cell never holds NaN bit patterns
    ok = cuda_ok(c, cudaMemsetAsync(c->kv_k, 0, kv_bytes, c->st), "memset") &&
         cuda_ok(c, cudaMemsetAsync(c->kv_v, 0, kv_bytes, c->st), "memset") &&
         cuda_ok(c, cudaStreamSynchronize(c->st), "sync");
    if (!ok) return die("");
    // bulk tensor copies of consecutive cells for the tcgen05 prefill attention (F16, hd 128)
    if (c->type_k == LLM_TYPE_F16 && c->type_v == LLM_TYPE_F16 && h.head_dim == 128) {
        const int64_t rows = (int64_t)h.n_layer * h.n_head_kv * c->n_ctx;
        c->kv_maps = rows < INT32_MAX && tc_make_map(&c->m_kc, c->kv_k, rows, h.head_dim, 128, true) &&
                     tc_make_map(&c->m_vc, c->kv_v, rows, h.head_dim, 128, true);
    }
    return c;
}

void llm_ctx_free(llm_ctx* c) {
    if (!c) return;
    if (c->st) cudaStreamSynchronize(c->st);
    drop_graphs(c);
    for (void* p : c->allocs) cudaFree(p);
    c->allocs.clear();
    if (c->h_in) cudaFreeHost(c->h_in);
    if (c->h_err) cudaFreeHost(c->h_err);
    for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
    if (c->own_stream && c->st) cudaStreamDestroy(c->st);
    delete c;
}

int llm_load_weights(llm_ctx* c, const char* name, int32_t type, const int64_t ne[2],
                     const void* data, size_t nbytes) {
    if (!c || !name || !ne) return -1;
    const llm_hparams& h = c->hp;
    auto bad = [&](const std::string& m) { c->err = std::string(name) + ": " + m; return -1; };
    if (type != LLM_TYPE_F32 && type != LLM_TYPE_F16 && type != LLM_TYPE_BF16 && type != LLM_TYPE_Q8_0)
        return bad("unsupported type");
    const int64_t cols = ne[0], rows = ne[1] <= 0 ? 1 : ne[1];
    if (cols <= 0) return bad("bad shape");
    if (type == LLM_TYPE_Q8_0 && cols % 32 != 0) return bad("Q8_0 rows must hold whole 32-value blocks");
    if ((int64_t)nbytes != rows * row_bytes(type, cols)) return bad("byte size does not match shape and type");
    if (!data) return bad("NULL data");
    const int64_t d = h.n_embd, qd = (int64_t)h.n_head * h.head_dim, kvd = (int64_t)h.n_head_kv * h.head_dim;
    const std::string n(name);
    // data may have been produced by work on another stream of this device: wait for it
    if (!c->host_only && !cuda_ok(c, cudaDeviceSynchronize(), "device synchronize")) return -2;
    auto want_shape = [&](int64_t c0, int64_t r0) { return cols == c0 && rows == r0; };

    if (n == "token_embd.weight" || n == "output.weight") {
        if (!want_shape(d, h.n_vocab)) return bad("shape must be {n_embd, n_vocab}");
        bool& flag = n == "token_embd.weight" ? c->embd_loaded : c->out_loaded;
        DevMat& m = n == "token_embd.weight" ? c->embd : c->out;
        if (flag) return bad("loaded twice");
        if (c->host_only) { flag = true; return 0; }
        if (!alloc_mat(c, m, type, rows, cols) || !fill_rows(c, m, 0, rows, data, nbytes)) return -2;
        flag = true;
        return 0;
    }
    if (n == "output_norm.weight") {
        if (type != LLM_TYPE_F32 || !want_shape(d, 1)) return bad("norm gains must be F32 {n_embd}");
        if (c->out_norm_loaded) return bad("loaded twice");
        if (!c->host_only) {
            if (!dalloc(c, &c->out_norm, d)) return -2;
            if (!cuda_ok(c, cudaMemcpy(c->out_norm, data, nbytes, cudaMemcpyDefault), "copy")) return -2;
        }
        c->out_norm_loaded = true;
        return 0;
    }
    int32_t il = -1;
    std::string part;
    if (!parse_layer_name(name, &il, &part) || il >= h.n_layer) return bad("unknown tensor name");
    Layer& L = c->layers[il];
    struct Spec { const char* part; uint32_t bit; int64_t c, r; };
    const Spec specs[] = {
        {"attn_norm", B_ATTN_NORM, d, 1}, {"attn_q", B_Q, d, qd}, {"attn_k", B_K, d, kvd},
        {"attn_v", B_V, d, kvd}, {"attn_output", B_O, qd, d}, {"ffn_norm", B_FFN_NORM, d, 1},
        {"ffn_gate", B_GATE, d, h.n_ff}, {"ffn_up", B_UP, d, h.n_ff}, {"ffn_down", B_DOWN, h.n_ff, d}};
    const Spec* sp = nullptr;
    for (const Spec& s : specs) if (part == s.part) sp = &s;
    if (!sp) return bad("unknown tensor name");
    if (!want_shape(sp->c, sp->r)) return bad("wrong shape");
    if (L.loaded & sp->bit) return bad("loaded twice");
    if (sp->bit == B_ATTN_NORM || sp->bit == B_FFN_NORM) {
        if (type != LLM_TYPE_F32) return bad("norm gains must be F32");
        if (!c->host_only) {
            float*& g = sp->bit == B_ATTN_NORM ? L.attn_norm : L.ffn_norm;
            if (!dalloc(c, &g, d)) return -2;
            if (!cuda_ok(c, cudaMemcpy(g, data, nbytes, cudaMemcpyDefault), "copy")) return -2;
        }
        L.loaded |= sp->bit;
        L.q8_tc = L.f16_ready = false;      // the f16 operands, if any, are stale
        return 0;
    }
    // fused stores: Q, K, V rows stacked in one matrix; gate rows then up rows in another
    DevMat* m = nullptr;
    int64_t row0 = 0, total_rows = 0;
    uint32_t group = 0;
    switch (sp->bit) {
        case B_Q: m = &L.qkv; row0 = 0; total_rows = qd + 2 * kvd; group = B_Q | B_K | B_V; break;
        case B_K: m = &L.qkv; row0 = qd; total_rows = qd + 2 * kvd; group = B_Q | B_K | B_V; break;
        case B_V: m = &L.qkv; row0 = qd + kvd; total_rows = qd + 2 * kvd; group = B_Q | B_K | B_V; break;
        case B_O: m = &L.wo; row0 = 0; total_rows = d; group = B_O; break;
        case B_GATE: m = &L.gu; row0 = 0; total_rows = 2 * (int64_t)h.n_ff; group = B_GATE | B_UP; break;
        case B_UP: m = &L.gu; row0 = h.n_ff; total_rows = 2 * (int64_t)h.n_ff; group = B_GATE | B_UP; break;
        default: m = &L.down; row0 = 0; total_rows = d; group = B_DOWN; break;
    }
    if (L.loaded & group) {
        if (m->type != type) return bad("all tensors of a fused group must share a type");
    } else if (!c->host_only) {
        if (!alloc_mat(c, *m, type, total_rows, cols)) return -2;
    } else {
        m->type = type;
    }
    if (!c->host_only && !fill_rows(c, *m, row0, rows, data, nbytes)) return -2;
    L.loaded |= sp->bit;
    L.q8_tc = L.f16_ready = false;
    return 0;
}

// The persistent one-token kernel serves the model when every linear weight (and the output
// matrix) has one 2-byte type and the shapes fit its mapping; its per-layer table is uploaded here.
static void setup_step(llm_ctx* c) {
    c->step_ok = false;
    if (!c->use_step || c->host_only) return;
    const llm_hparams& h = c->hp;
    const int32_t wt = c->layers.empty() ? -1 : c->layers[0].qkv.type;
    bool same = c->out.type == wt;
    for (const Layer& L : c->layers)
        same = same && L.qkv.type == wt && L.wo.type == wt && L.gu.type == wt && L.down.type == wt;
    if (!same || !decode_step_ok(wt, h.n_embd, h.n_head, h.n_head_kv, h.head_dim, h.n_ff, h.n_vocab,
                                 c->type_k, c->n_sm)) {
        cudaGetLastError();
        return;
    }
    std::vector<StepLayer> t(h.n_layer);
    double wb = wbytes(c->out, h.n_vocab);
    for (int32_t il = 0; il < h.n_layer; ++il) {
        const Layer& L = c->layers[il];
        t[il].qkv = L.qkv.data; t[il].wo = L.wo.data; t[il].gu = L.gu.data; t[il].down = L.down.data;
        t[il].attn_norm = L.attn_norm; t[il].ffn_norm = L.ffn_norm;
        t[il].kc = static_cast<uint8_t*>(c->kv_k) + (size_t)il * c->kv_layer_bytes();
        t[il].vc = static_cast<uint8_t*>(c->kv_v) + (size_t)il * c->kv_layer_bytes();
        wb += wbytes(L.qkv, c->qkv_width()) + wbytes(L.wo, h.n_embd) + wbytes(L.gu, 2 * (int64_t)h.n_ff) +
              wbytes(L.down, h.n_embd);
    }
    if (!c->d_step_layers && !dalloc(c, &c->d_step_layers, t.size())) return;
    if (!cuda_ok(c, cudaMemcpy(c->d_step_layers, t.data(), t.size() * sizeof(StepLayer),
                               cudaMemcpyHostToDevice), "copy"))
        return;
    c->step_weight_bytes = wb;
    c->step_ok = true;
}

// After a failed step the phase counters, the abort flag and the attention tickets are reset.
static bool reset_step_state(llm_ctx* c) {
    c->step_gen = 0;
    return cuda_ok(c, cudaMemsetAsync(c->d_counters, 0, sizeof(uint32_t) * (1 + 5 * (size_t)c->hp.n_layer), c->st), "memset") &&
           cuda_ok(c, cudaMemsetAsync(c->d_abort, 0, sizeof(int32_t), c->st), "memset") &&
           cuda_ok(c, cudaMemsetAsync(c->tickets, 0, sizeof(int32_t) * c->n_ubatch * c->hp.n_head_kv * kDecTicketsPerHead,
                                      c->st), "memset");
}

// One token through the whole model in one cooperative launch (inputs already uploaded).
static bool run_step(llm_ctx* c, int32_t O, int32_t out_row0) {
    const llm_hparams& hp = c->hp;
    const InLayout& io = c->io;
    const int32_t* din = c->d_in;
    StepArgs a;
    a.layers = c->d_step_layers;
    a.n_layer = hp.n_layer; a.d = hp.n_embd; a.H = hp.n_head; a.Hkv = hp.n_head_kv; a.hd = hp.head_dim;
    a.F = hp.n_ff; a.V = hp.n_vocab; a.eps = hp.rms_eps;
    a.embd = c->embd; a.theta = c->d_theta; a.out = c->out.data; a.out_norm = c->out_norm;
    a.do_logits = O > 0 ? 1 : 0;
    a.x = c->x; a.q = c->qkv; a.o = c->attn; a.u = c->u; a.cs = c->rope_cs;
    a.logits = c->d_logits + (size_t)out_row0 * hp.n_vocab;
    a.amax = c->d_amax + out_row0;
    a.tok = din + io.tok; a.pos = din + io.pos; a.slot = din + io.slot; a.hdr = din + io.hdr;
    a.tile_desc = reinterpret_cast<const int4*>(din + io.tile_desc);
    a.wi_desc = reinterpret_cast<const int4*>(din + io.wi_desc);
    a.list_cells = din + io.list_cells; a.list_pos = din + io.list_pos;
    a.part_o = c->part_o; a.part_m = c->part_m; a.part_l = c->part_l; a.tickets = c->tickets;
    a.n_ctx = c->n_ctx; a.kv_type = c->type_k;
    a.counters = c->d_counters; a.gen = c->step_gen; a.abort_flag = c->d_abort; a.err = c->d_err;
    if (c->step_trace) {
        const int32_t slots = 3 + 9 * hp.n_layer, blocks = 2 * c->n_sm;
        if (!c->d_trace) {
            if (!dalloc(c, &c->d_trace, (size_t)blocks * slots * 2)) return false;
            cudaMemsetAsync(c->d_trace, 0, sizeof(uint64_t) * blocks * slots * 2, c->st);
        }
        a.trace = c->d_trace;
        a.n_trace = slots;
        c->trace_blocks = blocks;
        c->trace_slots = slots;
        c->trace_valid = true;
    }
    const int k = kt_begin(c);
    if (!launch_decode_step(c->layers[0].qkv.type, a, c->n_sm, c->st)) {
        c->err = "decode step launch failed";
        return false;
    }
    kt_end(c, k, KC_DECODE_STEP, c->step_weight_bytes + c->att_bytes_now, 0);
    c->step_gen += 1;
    c->perf.n_fused_steps += 1;
    return true;
}

int llm_weights_ready(llm_ctx* c) {
    if (!c) return -1;
    if (!c->embd_loaded) { c->err = "missing token_embd.weight"; return -1; }
    if (!c->out_norm_loaded) { c->err = "missing output_norm.weight"; return -1; }
    for (int32_t il = 0; il < c->hp.n_layer; ++il) {
        if (c->layers[il].loaded != B_ALL) {
            c->err = "missing weights of layer " + std::to_string(il);
            return -1;
        }
    }
    if (!c->out_loaded) c->out = c->embd;   // tied output
    c->ready = true;
    drop_graphs(c);
    c->tc_ok = c->tc_f16 = false;
    if (c->host_only) return 0;
    // tensor-core prefill: every linear weight BF16 with supported shapes
    const llm_hparams& h = c->hp;
    const int64_t d = h.n_embd, qw = c->q_width(), qkvw = c->qkv_width(), F = h.n_ff;
    const int64_t U = c->n_ubatch;
    bool ok = tc_shape_ok(qkvw, d, GEMM_EPI_STORE, 0) && tc_shape_ok(d, qw, GEMM_EPI_ADD, 0) &&
              tc_shape_ok(0, d, GEMM_EPI_SWIGLU, F) && tc_shape_ok(d, F, GEMM_EPI_ADD, 0);
    // Prefill GEMMs on the token-major kernel with f16 operands when every layer's shapes allow it
    // and prefill ubatches can occur: a BF16 weight converted to f16 (exact in the f16 normal
    // range; 2 bytes per weight of extra device memory), made here once; a Q8_0 weight as stored,
    // dequantised by the GEMM into two f16 terms that hold d * q exactly (no extra memory).
    // Otherwise BF16 layers use the bf16 operands (activations as two terms) on the kernels their
    // shapes allow.
    const bool tn_shapes = U > gemv_max_tokens() && tc_tn_ok(qkvw, d) && tc_tn_ok(d, qw) &&
                           tc_swiglu_tn_ok(d, F) && tc_tn_ok(d, F);
    auto f16_copy = [&](const DevMat& W, int64_t rows, int64_t cols, CUtensorMap* map) {
        uint16_t* y = nullptr;
        if (!dalloc(c, &y, (size_t)(rows * cols))) return false;
        c->perf.weight_device_bytes += rows * cols * 2;
        launch_bf16_to_f16(W.data, rows * cols, y, c->st);
        return tc_make_map(map, y, rows, cols, 128, true);
    };
    // a Q8_0 weight: the quants' tensor map, and its scales in the per-k-step layout (1/32 of a
    // byte per weight more)
    auto q8_ks = [&](const DevMat& W, int64_t rows, int64_t cols, CUtensorMap* map, uint32_t** ks, int box_rows) {
        if (!dalloc(c, ks, (size_t)(rows * (cols / 64)))) return false;
        c->perf.weight_device_bytes += rows * (cols / 64) * 4;
        q8_scales_by_kstep(W.scales, rows, cols, *ks, c->st);
        return tc_make_map_q8(map, W.data, rows, cols, box_rows);
    };
    bool f16 = tn_shapes;
    for (int32_t il = 0; ok && il < h.n_layer; ++il) {
        Layer& L = c->layers[il];
        const bool bf16 = L.qkv.type == LLM_TYPE_BF16 && L.wo.type == LLM_TYPE_BF16 &&
                          L.gu.type == LLM_TYPE_BF16 && L.down.type == LLM_TYPE_BF16;
        const bool q8 = L.qkv.type == LLM_TYPE_Q8_0 && L.wo.type == LLM_TYPE_Q8_0 &&
                        L.gu.type == LLM_TYPE_Q8_0 && L.down.type == LLM_TYPE_Q8_0;
        if (bf16 && tn_shapes) {
            L.f16_ready = L.f16_ready || (f16_copy(L.qkv, qkvw, d, &L.mq) && f16_copy(L.wo, d, qw, &L.mo) &&
                                          f16_copy(L.gu, 2 * F, d, &L.mgu128) && f16_copy(L.down, d, F, &L.md));
            ok = L.f16_ready;
            L.gu_tn = ok;
        } else if (bf16) {
            f16 = false;
            ok = tc_make_map(&L.mq, L.qkv.data, qkvw, d, 128) &&
                 tc_make_map(&L.mo, L.wo.data, d, qw, 128) &&
                 tc_make_map(&L.mgu, L.gu.data, 2 * F, d, 64) &&
                 tc_make_map(&L.md, L.down.data, d, F, 128);
            L.gu_tn = ok && tc_swiglu_tn_ok(d, F) && tc_make_map(&L.mgu128, L.gu.data, 2 * F, d, 128);
        } else if (q8 && tn_shapes) {
            L.q8_tc = L.q8_tc || (q8_ks(L.qkv, qkvw, d, &L.mq, &L.qkv_ks, 128) &&
                                  q8_ks(L.wo, d, qw, &L.mo, &L.wo_ks, 128) &&
                                  q8_ks(L.gu, 2 * F, d, &L.mgu128, &L.gu_ks, 64) &&
                                  q8_ks(L.down, d, F, &L.md, &L.down_ks, 128));
            ok = L.q8_tc;
            L.gu_tn = ok;
        } else {
            ok = false;
        }
    }
    if (ok && !cuda_ok(c, cudaStreamSynchronize(c->st), "f16 weights")) return -1;
    ok = ok && (!f16 || (tc_make_map(&c->m_hh, c->hb, U, d, 128, true) &&
                         tc_make_map(&c->m_ah, c->attnb, U, qw, 128, true) &&
                         tc_make_map(&c->m_uh, c->ub, U, F, 128, true) &&
                         tc_make_out_map(&c->m_y_qkv, c->qkv, U, qkvw, false) &&
                         tc_make_out_map(&c->m_y_x, c->x, U, d, false) &&
                         tc_make_out_map(&c->m_y_ub, c->ub, U, F, true)));
    const int boxes[2] = {128, 256};
    for (int i = 0; ok && i < 2; ++i)
        ok = tc_make_map(&c->m_hb[i], c->hb, U, d, boxes[i]) &&
             tc_make_map(&c->m_attnb[i], c->attnb, U, qw, boxes[i]) &&
             tc_make_map(&c->m_ub[i], c->ub, U, F, boxes[i]) &&
             tc_make_map(&c->m_hob[i], c->hob, U, d, boxes[i]);
    ok = ok && tc_make_map(&c->m_hb_lo, c->hb_lo, U, d, 128) &&
         tc_make_map(&c->m_attnb_lo, c->attnb_lo, U, qw, 128) &&
         tc_make_map(&c->m_ub_lo, c->ub_lo, U, F, 128) &&
         tc_make_map(&c->m_hob_lo, c->hob_lo, U, d, 128);
    const bool lm_ok = c->out.type == LLM_TYPE_BF16 && tc_shape_ok(h.n_vocab, d, GEMM_EPI_STORE, 0) &&
                       tc_make_map(&c->m_lm, c->out.data, h.n_vocab, d, 128);
    c->tc_ok = ok;
    c->tc_f16 = ok && f16;
    c->tc_lm = ok && lm_ok;
    setup_step(c);
    return 0;
}

static int defrag(llm_ctx* c);

int32_t llm_decode(llm_ctx* c, llm_batch bt) {
    if (!c) return -2;
    const auto t0 = std::chrono::steady_clock::now();
    struct Timer {
        llm_ctx* c;
        std::chrono::steady_clock::time_point t0;
        ~Timer() {
            c->perf.t_decode_ms += std::chrono::duration<double, std::milli>(
                                       std::chrono::steady_clock::now() - t0).count();
        }
    } timer{c, t0};
    c->n_outputs = 0;
    c->output_ids.clear();
    c->rows_by_rank.clear();
    c->h_logits_valid = c->h_argmax_valid = false;
    if (!c->host_only && !c->ready && llm_weights_ready(c) != 0) return -1;
    if (!c->host_only) cudaSetDevice(c->device);
    SanBatch& b = c->batch;
    std::string why;
    if (!sanitize_batch(bt.n_tokens, bt.token, bt.pos, bt.n_seq_id, bt.seq_id, bt.logits,
                        c->hp.n_vocab, c->n_seq_max, c->n_batch, c->cells, b, &why)) {
        c->err = "invalid batch: " + why;
        return -1;
    }
    // the ubatches ([P1] Крок 12): split_simple over a unified cache, split_equal over a split
    // one; a split reorders the batch into ubatch order (orig maps back to batch indices)
    std::vector<int32_t> ub_off, orig;
    if (c->n_stream == 1) {
        for (int32_t i0 = 0; i0 < b.n; i0 += c->n_ubatch) ub_off.push_back(i0);
        ub_off.push_back(b.n);
        orig.resize(b.n);
        for (int32_t i = 0; i < b.n; ++i) orig[i] = i;
    } else {
        for (int32_t i = 0; i < b.n; ++i)
            if (b.seqs[i].count() != 1) {
                c->err = "invalid batch: a token of a split cache must belong to one sequence";
                return -1;
            }
        split_equal(b.first_seq, c->n_ubatch, orig, ub_off);
        SanBatch pb = b;
        for (int32_t j = 0; j < b.n; ++j) {
            const int32_t i = orig[j];
            pb.token[j] = b.token[i]; pb.pos[j] = b.pos[i]; pb.seqs[j] = b.seqs[i];
            pb.first_seq[j] = b.first_seq[i]; pb.output[j] = b.output[i];
        }
        b = std::move(pb);
    }
    // all slots before any commit: the tokens take the next lowest empty cells (of their stream)
    std::vector<int32_t> slots;
    auto find_slots = [&]() {
        if (c->n_stream == 1) return c->cells.find_free(b.n, slots);
        slots.assign(b.n, -1);
        std::vector<std::vector<int32_t>> of(c->n_stream);
        for (int32_t j = 0; j < b.n; ++j) of[b.first_seq[j]].push_back(j);
        std::vector<int32_t> got;
        for (int32_t s = 0; s < c->n_stream; ++s) {
            if (of[s].empty()) continue;
            if (!c->cells.find_free((int32_t)of[s].size(), got, s)) return false;
            for (size_t k = 0; k < got.size(); ++k) slots[of[s][k]] = got[k];
        }
        return true;
    };
    if (!find_slots()) {
        // one defrag, then one more search ([P4] KVキャッシュの詳細: FAILED_PREPARE -> defrag)
        const int moved = defrag(c);
        if (moved < 0) return -2;
        if (moved == 0 || !find_slots()) {
            c->err = "no KV slot for the batch";
            return 1;
        }
    }
    if (!c->host_only && !ensure_outputs(c, b.n_outputs)) return -2;
    c->last_slots = slots;
    c->dbg_ub.clear();
    c->perf.n_decode_calls += 1;
    const int32_t G = c->hp.n_head / c->hp.n_head_kv;
    int32_t n_out = 0;
    for (int32_t ub = 0; ub + 1 < (int32_t)ub_off.size(); ++ub) {
        const int32_t i0 = ub_off[ub], T = ub_off[ub + 1] - ub_off[ub];
        std::vector<int32_t> us(slots.begin() + i0, slots.begin() + i0 + T);
        c->cells.apply(us, b.pos.data() + i0, b.seqs.data() + i0, T);       // mctx->apply()
        if (c->abort_cb && c->abort_cb(c->abort_ud)) {
            rollback(c, i0, T);
            c->err = "aborted";
            return 2;
        }
        const bool small = T <= gemv_max_tokens();
        const int32_t cap = small ? attn_cap(c, T) : c->max_work;
        // the one-token kernel stages one pass of decode_step_cells() cells per work item
        const bool fused = T == 1 && c->step_ok && !c->debug;
        // prefill tiles: a work item per (tile, KV head) unless that leaves SMs idle; splitting a
        // tile's list costs a merge (measured at 512 tokens: 48 us per layer unsplit, 101 us in
        // 256-cell items, 126 us in 128-cell items)
        // prefill ubatches of a forward pass with f16 GEMM operands over an F16 cache take the
        // tcgen05 attention tiles, whose plan has 32 tokens per tile
        const bool tc_attn = !small && c->tc_ok && c->tc_f16 && c->type_k == LLM_TYPE_F16 &&
                             c->type_v == LLM_TYPE_F16 && c->hp.head_dim == 128 && G == 4;
        const int32_t tile_q = tc_attn ? attention_tc_tile_q() : kAttnTileQ;
        build_attn_plan(c->cells, b, i0, T, tile_q, c->hp.n_head_kv, G, (small ? 4 : 1) * c->n_sm,
                        c->max_rows, cap, c->plan, fused ? decode_step_cells() : small ? 64 : tc_attn ? 128 : 32);
        if (c->debug) {
            UbDebug u;
            u.n_kv = c->cells.n_kv();
            u.pos.assign(b.pos.begin() + i0, b.pos.begin() + i0 + T);
            u.tok_list = c->plan.tok_list;
            u.list_off = c->plan.list_off;
            u.list_cells = c->plan.list_cells;
            u.list_pos = c->plan.list_pos;
            c->dbg_ub.push_back(std::move(u));
        }
        std::vector<int32_t> out_rows;
        for (int32_t t = 0; t < T; ++t)
            if (b.output[i0 + t]) out_rows.push_back(t);
        const int32_t O = (int32_t)out_rows.size();
        c->perf.n_ubatches += 1;
        c->perf.n_tokens += T;
        if (c->host_only) { n_out += O; continue; }

        const AttnPlan& p = c->plan;
        if (!ensure_inputs(c, p.list_cells.size())) { rollback(c, i0, T); return -2; }
        const InLayout& io = c->io;
        int32_t* hi = c->h_in;
        hi[io.hdr + 0] = p.n_work();
        hi[io.hdr + 1] = p.n_tiles();
        hi[io.hdr + 2] = c->cells.n_kv();
        std::memcpy(hi + io.tok, b.token.data() + i0, T * sizeof(int32_t));
        std::memcpy(hi + io.pos, b.pos.data() + i0, T * sizeof(int32_t));
        std::memcpy(hi + io.slot, us.data(), T * sizeof(int32_t));
        if (c->fault_kind == 1 && c->fault_ub == ub) hi[io.slot] = c->n_ctx + 7;
        put(hi, io.out_rows, out_rows);
        put(hi, io.perm, p.perm);
        for (int32_t t = 0; t < p.n_tiles(); ++t) {
            int32_t* d8 = hi + io.tile_desc + 8 * t;
            const int32_t l = p.tile_list[t];
            d8[0] = l; d8[1] = p.tile_start[t]; d8[2] = p.tile_nq[t]; d8[3] = p.tile_wi_off[t];
            d8[4] = p.tile_wi_off[t + 1]; d8[5] = p.list_off[l];
            d8[6] = p.list_off[l + 1] - p.list_off[l]; d8[7] = 0;
        }
        for (int32_t w = 0; w < p.n_work(); ++w) {
            int32_t* d4 = hi + io.wi_desc + 4 * w;
            d4[0] = p.wi_tile[w]; d4[1] = p.wi_c0[w]; d4[2] = p.wi_c1[w]; d4[3] = p.wi_row_off[w];
        }
        put(hi, io.list_cells, p.list_cells); put(hi, io.list_pos, p.list_pos);
        const size_t nl = p.list_cells.size();
        bool ok = cuda_ok(c, cudaMemcpyAsync(c->d_in, hi, io.fixed_end * sizeof(int32_t),
                                             cudaMemcpyHostToDevice, c->st), "inputs upload") &&
                  (nl == 0 || (cuda_ok(c, cudaMemcpyAsync(c->d_in + io.list_cells, hi + io.list_cells,
                                                          nl * sizeof(int32_t), cudaMemcpyHostToDevice,
                                                          c->st), "inputs upload") &&
                               cuda_ok(c, cudaMemcpyAsync(c->d_in + io.list_pos, hi + io.list_pos,
                                                          nl * sizeof(int32_t), cudaMemcpyHostToDevice,
                                                          c->st), "inputs upload"))) &&
                  cuda_ok(c, cudaMemsetAsync(c->d_err, 0, sizeof(uint32_t), c->st), "memset");
        if (c->ktime) attention_work(c, b.pos.data() + i0);
        const int32_t max_nq = p.max_nq <= 1 ? 1 : tile_q;
        int32_t max_len = 0;
        for (size_t l = 0; l + 1 < p.list_off.size(); ++l) max_len = std::max(max_len, p.list_off[l + 1] - p.list_off[l]);
        c->dec_long = max_len >= kDecLongList;
        const StepGraph* sg = nullptr;
        const bool one_kernel = ok && T == 1 && c->step_ok && !c->debug;
        if (one_kernel) ok = run_step(c, O, n_out);
        // decode ubatches (one token per attention tile: the cluster kernels, whose grid follows T)
        // replay a captured graph per key; prefill ubatches size their attention grids from the
        // host plan and launch directly
        if (ok && !one_kernel && (small || max_nq <= 1) && c->use_graphs && !c->debug) {
            const uint64_t key = (uint64_t)T | ((uint64_t)O << 10) | ((uint64_t)n_out << 20) |
                                 ((uint64_t)(max_nq > 1) << 52) | ((uint64_t)c->ktime << 53) |
                                 ((uint64_t)c->dec_long << 54);
            auto it = c->graphs.find(key);
            if (it == c->graphs.end()) {
                StepGraph ng;
                if (c->ktime) { c->kcap = &ng.timing; c->kcap_events = &ng.events; }
                cudaGraph_t graph = nullptr;
                bool cap_ok = cudaStreamBeginCapture(c->st, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
                const bool fwd_ok = cap_ok && forward_ubatch(c, T, O, n_out, max_nq);
                if (cap_ok) cap_ok = cudaStreamEndCapture(c->st, &graph) == cudaSuccess && fwd_ok;
                c->kcap = nullptr;
                c->kcap_events = nullptr;
                if (cap_ok) cap_ok = cudaGraphInstantiate(&ng.exec, graph, 0) == cudaSuccess;
                if (graph) cudaGraphDestroy(graph);
                cudaGetLastError();
                if (cap_ok) {
                    it = c->graphs.emplace(key, std::move(ng)).first;
                } else {
                    // capture is an optimisation: fall back to direct launches from now on
                    for (cudaEvent_t e : ng.events) cudaEventDestroy(e);
                    c->use_graphs = false;
                }
            }
            if (it != c->graphs.end()) {
                sg = &it->second;
                ok = cuda_ok(c, cudaGraphLaunch(sg->exec, c->st), "graph launch");
                c->perf.n_graph_replays += 1;
            }
        }
        if (ok && !sg && !one_kernel) ok = forward_ubatch(c, T, O, n_out, max_nq);
        ok = ok && cuda_ok(c, cudaMemcpyAsync(c->h_err, c->d_err, sizeof(uint32_t),
                                              cudaMemcpyDeviceToHost, c->st), "error word") &&
             cuda_ok(c, cudaStreamSynchronize(c->st), "device computation");
        kt_collect(c, sg);
        if (ok && *c->h_err != 0) {
            c->err = "device check failed (error word " + std::to_string(*c->h_err) + ")";
            ok = false;
        }
        if (!ok) {
            rollback(c, i0, T);
            c->fault_kind = 0;
            if (one_kernel) reset_step_state(c);
            return -3;
        }
        n_out += O;
    }
    c->fault_kind = 0;
    c->n_outputs = n_out;
    c->output_ids.assign(b.n, -1);
    int32_t k = 0;
    for (int32_t j = 0; j < b.n; ++j)                 // rows were written in ubatch order
        if (b.output[j]) c->output_ids[orig[j]] = k++;
    c->rows_by_rank.clear();
    for (int32_t i = 0; i < b.n; ++i)
        if (c->output_ids[i] >= 0) c->rows_by_rank.push_back(c->output_ids[i]);
    return 0;
}

static int32_t resolve_row(llm_ctx* c, int32_t i) {
    if (i < 0) {                                        // counted back from the last output
        const int32_t j = c->n_outputs + i;
        return j >= 0 && j < (int32_t)c->rows_by_rank.size() ? c->rows_by_rank[j] : -1;
    }
    if (i >= (int32_t)c->output_ids.size()) return -1;
    return c->output_ids[i];
}

float* llm_get_logits_ith(llm_ctx* c, int32_t i) {
    if (!c || c->host_only) return nullptr;
    const int32_t j = resolve_row(c, i);
    if (j < 0) return nullptr;
    if (!c->h_logits_valid) {
        c->h_logits.resize((size_t)c->n_outputs * c->hp.n_vocab);
        if (!cuda_ok(c, cudaMemcpyAsync(c->h_logits.data(), c->d_logits,
                                        c->h_logits.size() * sizeof(float), cudaMemcpyDeviceToHost,
                                        c->st), "logits copy") ||
            !cuda_ok(c, cudaStreamSynchronize(c->st), "sync"))
            return nullptr;
        c->h_logits_valid = true;
    }
    return c->h_logits.data() + (size_t)j * c->hp.n_vocab;
}

int32_t llm_get_argmax_ith(llm_ctx* c, int32_t i) {
    if (!c || c->host_only) return -1;
    const int32_t j = resolve_row(c, i);
    if (j < 0) return -1;
    if (!c->h_argmax_valid) {
        c->h_amax.resize(c->n_outputs);
        if (!cuda_ok(c, cudaMemcpyAsync(c->h_amax.data(), c->d_amax,
                                        c->n_outputs * sizeof(unsigned long long),
                                        cudaMemcpyDeviceToHost, c->st), "argmax copy") ||
            !cuda_ok(c, cudaStreamSynchronize(c->st), "sync"))
            return -1;
        c->h_argmax_valid = true;
    }
    return unpack_argmax(c->h_amax[j]);
}

int32_t llm_n_outputs(llm_ctx* c) { return c ? c->n_outputs : 0; }

// Defrag: move the used cells' K/V rows (every layer) to their new cells, then rewrite the cell
// metadata. Each cache region (per layer K and V; Q8_0: quants and scales) is gathered into a
// scratch region in the new cell order (empty cells zeroed), then copied back whole.
static int defrag(llm_ctx* c) {
    std::vector<int32_t> order;
    if (!c->cells.defrag_order(order)) return 0;
    if (!c->host_only) {
        const int32_t n = c->n_ctx, Hkv = c->hp.n_head_kv, hd = c->hp.head_dim;
        if (!c->kv_scratch && !dalloc(c, &c->kv_scratch, c->kv_layer_bytes())) return -1;
        if (!c->d_order && !dalloc(c, &c->d_order, (size_t)c->n_ctx)) return -1;
        if (!cuda_ok(c, cudaMemcpyAsync(c->d_order, order.data(), sizeof(int32_t) * n, cudaMemcpyHostToDevice,
                                        c->st), "copy"))
            return -1;
        struct Region { size_t off; int32_t rb; };
        std::vector<Region> regions;
        if (c->kv_q8()) {
            regions.push_back({0, hd});
            regions.push_back({kv_q8_scale_offset(Hkv, c->n_ctx, hd), hd / 32 * 2});
        } else {
            regions.push_back({0, hd * (int32_t)type_size(c->type_k)});
        }
        for (int32_t il = 0; il < c->hp.n_layer; ++il) {
            for (void* base : {c->kv_k, c->kv_v}) {
                uint8_t* layer = static_cast<uint8_t*>(base) + (size_t)il * c->kv_layer_bytes();
                for (const Region& r : regions) {
                    launch_kv_gather(layer + r.off, c->kv_scratch, c->d_order, n, Hkv, c->n_ctx, r.rb, c->st);
                    if (!cuda_ok(c, cudaMemcpyAsync(layer + r.off, c->kv_scratch, (size_t)Hkv * n * r.rb,
                                                    cudaMemcpyDeviceToDevice, c->st), "copy"))
                        return -1;
                }
            }
        }
        if (!cuda_ok(c, cudaGetLastError(), "defrag launch") || !cuda_ok(c, cudaStreamSynchronize(c->st), "defrag"))
            return -1;
    }
    c->cells.move(order);
    c->perf.n_defrags += 1;
    return 1;
}

int llm_memory_update(llm_ctx* c, int optimize) {
    if (!c) return -1;
    if (!optimize) return 0;
    if (!c->host_only) cudaSetDevice(c->device);
    return defrag(c);
}

int llm_seq_rm(llm_ctx* c, int32_t seq, int32_t p0, int32_t p1) {
    if (!c) return 0;
    if (seq >= c->n_seq_max) return 1;
    c->cells.seq_rm(seq, p0, p1);
    return 1;
}

int32_t llm_seq_pos_max(llm_ctx* c, int32_t s) { return c ? c->cells.seq_pos_max(s) : -1; }
int32_t llm_seq_pos_min(llm_ctx* c, int32_t s) { return c ? c->cells.seq_pos_min(s) : -1; }

void llm_set_abort_callback(llm_ctx* c, int (*cb)(void*), void* ud) {
    if (!c) return;
    c->abort_cb = cb;
    c->abort_ud = ud;
}

uint32_t llm_n_ctx(llm_ctx* c) { return c ? (uint32_t)c->n_ctx : 0; }
uint32_t llm_n_batch(llm_ctx* c) { return c ? (uint32_t)c->n_batch : 0; }
uint32_t llm_n_ubatch(llm_ctx* c) { return c ? (uint32_t)c->n_ubatch : 0; }
int32_t llm_kv_used_cells(llm_ctx* c) { return c ? c->cells.used() : 0; }
uint32_t llm_n_ctx_seq(llm_ctx* c) { return c ? (uint32_t)(c->n_ctx / c->n_stream) : 0; }

const char* llm_last_error(llm_ctx* c) { return c ? c->err.c_str() : g_init_error.c_str(); }

void llm_perf(llm_ctx* c, llm_perf_data* out) {
    if (c && out) *out = c->perf;
}

int32_t llm_debug_last_slots(llm_ctx* c, int32_t* out, int32_t cap) {
    if (!c) return 0;
    const int32_t n = (int32_t)c->last_slots.size();
    if (out) std::memcpy(out, c->last_slots.data(), sizeof(int32_t) * std::max(0, std::min(n, cap)));
    return n;
}

int64_t llm_debug_ubatch_mask(llm_ctx* c, int32_t ub, uint8_t* out, int64_t cap, int32_t* n_kv_out) {
    if (!c || ub < 0 || ub >= (int32_t)c->dbg_ub.size()) return 0;
    const UbDebug& u = c->dbg_ub[ub];
    const int64_t T = (int64_t)u.pos.size(), nkv = u.n_kv, n = T * nkv;
    if (n_kv_out) *n_kv_out = (int32_t)nkv;
    if (!out) return n;
    std::vector<uint8_t> m((size_t)n, 0);
    for (int64_t t = 0; t < T; ++t) {
        const int32_t l = u.tok_list[t];
        for (int32_t k = u.list_off[l]; k < u.list_off[l + 1]; ++k)
            if (u.list_pos[k] <= u.pos[t] && u.list_cells[k] < nkv) m[t * nkv + u.list_cells[k]] = 1;
    }
    std::memcpy(out, m.data(), (size_t)std::min(n, cap));
    return n;
}

int llm_debug_capture(llm_ctx* c, int enable) {
    if (!c) return -1;
    c->debug = enable != 0;
    if (!c->debug || c->host_only || c->dbg_lout) return 0;
    const int64_t U = c->n_ubatch, d = c->hp.n_embd, L = c->hp.n_layer, qw = c->q_width();
    const bool ok = dalloc(c, &c->dbg_embd, U * d) && dalloc(c, &c->dbg_lout, L * U * d) &&
                    dalloc(c, &c->dbg_attn, L * U * qw) && dalloc(c, &c->dbg_q, L * U * qw) &&
                    dalloc(c, &c->dbg_rnorm, U * d) &&
                    (!c->kv_q8() || (dalloc(c, &c->dbg_kin, L * U * c->hp.n_head_kv * c->hp.head_dim) &&
                                     dalloc(c, &c->dbg_vin, L * U * c->hp.n_head_kv * c->hp.head_dim)));
    return ok ? 0 : -2;
}

int64_t llm_debug_get_tensor(llm_ctx* c, const char* name, int32_t layer, float* out, int64_t cap) {
    if (!c || !name || c->host_only || !c->dbg_lout) return 0;
    const std::string n(name);
    const int64_t T = c->dbg_T, d = c->hp.n_embd, qw = c->q_width();
    const float* src = nullptr;
    int64_t cnt = 0;
    if (n == "embd") { src = c->dbg_embd; cnt = T * d; }
    else if (n == "result_norm" && c->dbg_rnorm_valid) { src = c->dbg_rnorm; cnt = (int64_t)c->dbg_O * d; }
    else if (layer >= 0 && layer < c->hp.n_layer) {
        if (n == "l_out") { src = c->dbg_lout + layer * T * d; cnt = T * d; }
        else if (n == "attn_out") { src = c->dbg_attn + layer * T * qw; cnt = T * qw; }
        else if (n == "kq_in") { src = c->dbg_q + layer * T * qw; cnt = T * qw; }
        else if ((n == "k_in" || n == "v_in") && c->dbg_kin) {
            const int64_t kw = (int64_t)c->hp.n_head_kv * c->hp.head_dim;
            src = (n == "k_in" ? c->dbg_kin : c->dbg_vin) + layer * T * kw;
            cnt = T * kw;
        }
    }
    if (!src) return 0;
    if (out && cap > 0) {
        cudaStreamSynchronize(c->st);
        cudaMemcpy(out, src, sizeof(float) * std::min(cnt, cap), cudaMemcpyDeviceToHost);
    }
    return cnt;
}

int64_t llm_debug_kv_raw(llm_ctx* c, int32_t layer, int32_t which, void* out, int64_t cap_bytes) {
    if (!c || c->host_only || layer < 0 || layer >= c->hp.n_layer || which < 0 || which > 3) return 0;
    if (which >= 2 && !c->kv_f16) return 0;
    const int64_t n = which >= 2 ? (int64_t)c->hp.n_head_kv * c->n_ctx * c->hp.head_dim * 2
                                 : (int64_t)c->kv_layer_bytes();
    if (out && cap_bytes > 0) {
        const uint8_t* src = which >= 2 ? reinterpret_cast<const uint8_t*>(c->kv_f16) + (size_t)(which - 2) * n
                           : static_cast<const uint8_t*>(which == 0 ? c->kv_k : c->kv_v) + (size_t)layer * n;
        cudaStreamSynchronize(c->st);
        cudaMemcpy(out, src, (size_t)std::min(n, cap_bytes), cudaMemcpyDeviceToHost);
    }
    return n;
}

int llm_debug_kernel_timing(llm_ctx* c, int enable) {
    if (!c) return -1;
    c->ktime = enable != 0 && !c->host_only;
    if (c->ktime)
        for (KStat& s : c->kstat) s = KStat();
    return 0;
}

int32_t llm_debug_kernel_stats(llm_ctx* c, int32_t i, char* name, int32_t name_cap,
                               int64_t* launches, double* ms, double* bytes, double* flops) {
    if (!c) return 0;
    if (i >= 0 && i < KC_COUNT) {
        if (name && name_cap > 0) {
            std::strncpy(name, kKClassNames[i], (size_t)name_cap - 1);
            name[name_cap - 1] = 0;
        }
        if (launches) *launches = c->kstat[i].launches;
        if (ms) *ms = c->kstat[i].ms;
        if (bytes) *bytes = c->kstat[i].bytes;
        if (flops) *flops = c->kstat[i].flops;
    }
    return KC_COUNT;
}

int llm_debug_gemm_bf16(int32_t epi, const void* W, int64_t M, int64_t K, const void* X, int32_t T,
                        void* Y, int32_t ldy, int32_t F) {
    if (!W || !X || !Y || T <= 0 || epi < 0 || epi > 2) return -1;
    if (!tc_shape_ok(M, K, epi, F)) return -1;
    const int64_t wrows = epi == GEMM_EPI_SWIGLU ? 2 * (int64_t)F : M;
    CUtensorMap wm, xm;
    if (!tc_make_map(&wm, W, wrows, K, epi == GEMM_EPI_SWIGLU ? 64 : 128) ||
        !tc_make_map(&xm, X, T, K, tc_token_tile(T)))
        return -1;
    uint32_t* err = nullptr;
    if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return -3;
    cudaMemset(err, 0, sizeof(uint32_t));
    bool ok = launch_gemm_tc(wm, xm, epi, (int)K, (int)M, T, F, Y, ldy, err, 0);
    uint32_t h = 0;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess &&
         cudaMemcpy(&h, err, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(err);
    return ok && h == 0 ? 0 : -3;
}

int llm_debug_gemm_tn_f16(int32_t epi, const void* W, const void* W_lo, int64_t M, int64_t K, const void* X,
                          int32_t T, float* Y, int32_t ldy, int32_t F, int32_t splits, int32_t one_cta) {
    if (!W || !X || !Y || T <= 0 || epi < 0 || epi > 2 || splits < 1) return -1;
    const bool swiglu = epi == GEMM_EPI_SWIGLU;
    if (swiglu ? !tc_swiglu_tn_ok(K, F) : !tc_tn_ok(M, K)) return -1;
    if (swiglu && splits != 1) return -1;
    const int64_t wrows = swiglu ? 2 * (int64_t)F : M;
    CUtensorMap wm, wl, xm;
    if (!tc_make_map(&wm, W, wrows, K, 128, true) || !tc_make_map(&xm, X, T, K, 128, true) ||
        (W_lo && !tc_make_map(&wl, W_lo, wrows, K, 128, true)))
        return -1;
    uint32_t* err = nullptr;
    if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return -3;
    cudaMemset(err, 0, sizeof(uint32_t));
    // the output through the TMA-store epilogue when its rows are whole 16-byte multiples
    CUtensorMap ym;
    const bool use_y = tc_make_out_map(&ym, Y, T, ldy, swiglu);
    bool ok = swiglu ? launch_gemm_swiglu_tn(xm, nullptr, wm, (int)K, T, F, Y, nullptr, ldy, err, 0,
                                             W_lo ? &wl : nullptr, one_cta != 0, use_y ? &ym : nullptr)
                     : launch_gemm_tn(xm, nullptr, wm, epi, (int)K, (int)M, T, Y, ldy, splits, err, 0,
                                      W_lo ? &wl : nullptr, one_cta != 0, use_y ? &ym : nullptr);
    uint32_t h = 0;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess &&
         cudaMemcpy(&h, err, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(err);
    return ok && h == 0 ? 0 : -3;
}

int llm_debug_gemm_tn_q8(int32_t epi, const void* Wq, const void* Ws, int64_t M, int64_t K, const void* X,
                         int32_t T, float* Y, int32_t ldy, int32_t F, int32_t splits) {
    if (!Wq || !Ws || !X || !Y || T <= 0 || epi < 0 || epi > 2 || splits < 1) return -1;
    if ((reinterpret_cast<uintptr_t>(Ws) & 15) != 0) return -1;
    const bool swiglu = epi == GEMM_EPI_SWIGLU;
    if (swiglu ? (!tc_swiglu_tn_ok(K, F) || splits != 1) : !tc_tn_ok(M, K)) return -1;
    const int64_t wrows = swiglu ? 2 * (int64_t)F : M;
    CUtensorMap qm, xm, ym;
    if (!tc_make_map_q8(&qm, Wq, wrows, K, swiglu ? 64 : 128) || !tc_make_map(&xm, X, T, K, 128, true)) return -1;
    const bool use_y = tc_make_out_map(&ym, Y, T, ldy, swiglu);
    uint32_t* err = nullptr;
    if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return -3;
    cudaMemset(err, 0, sizeof(uint32_t));
    uint32_t* ks = nullptr;
    if (cudaMalloc(&ks, sizeof(uint32_t) * (size_t)(wrows * (K / 64))) != cudaSuccess) { cudaFree(err); return -3; }
    q8_scales_by_kstep(static_cast<const __half*>(Ws), wrows, K, ks, 0);
    bool ok = swiglu ? launch_gemm_swiglu_tn(xm, nullptr, qm, (int)K, T, F, Y, nullptr, ldy, err, 0, nullptr, false,
                                             use_y ? &ym : nullptr, false, ks)
                     : launch_gemm_tn(xm, nullptr, qm, epi, (int)K, (int)M, T, Y, ldy, splits, err, 0, nullptr, false,
                                      use_y ? &ym : nullptr, nullptr, false, ks);
    uint32_t h = 0;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess &&
         cudaMemcpy(&h, err, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(ks);
    cudaFree(err);
    return ok && h == 0 ? 0 : -3;
}

int64_t llm_debug_gemm_tn_q8_trace(int32_t epi, const void* Wq, const void* Ws, int64_t M, int64_t K,
                                   const void* X, int32_t T, float* Y, int32_t ldy, int32_t F, int32_t splits,
                                   uint64_t* trace, int64_t cap) {
    if (!Wq || !Ws || !X || !Y || T <= 0 || epi < 0 || epi > 2 || splits < 1) return -1;
    if ((reinterpret_cast<uintptr_t>(Ws) & 15) != 0) return -1;
    const bool swiglu = epi == GEMM_EPI_SWIGLU;
    if (swiglu ? (!tc_swiglu_tn_ok(K, F) || splits != 1) : !tc_tn_ok(M, K)) return -1;
    const int64_t n = 8 * (int64_t)tc_tn2_blocks(epi, (int)M, T, F, splits);
    if (!trace || cap < n) return -1;
    const int64_t wrows = swiglu ? 2 * (int64_t)F : M;
    CUtensorMap qm, xm, ym;
    if (!tc_make_map_q8(&qm, Wq, wrows, K, swiglu ? 64 : 128) || !tc_make_map(&xm, X, T, K, 128, true)) return -1;
    const bool use_y = tc_make_out_map(&ym, Y, T, ldy, swiglu);
    uint32_t* err = nullptr;
    uint64_t* dtr = nullptr;
    if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return -3;
    if (cudaMalloc(&dtr, sizeof(uint64_t) * n) != cudaSuccess) { cudaFree(err); return -3; }
    cudaMemset(err, 0, sizeof(uint32_t));
    cudaMemset(dtr, 0, sizeof(uint64_t) * n);
    uint32_t* ks = nullptr;
    if (cudaMalloc(&ks, sizeof(uint32_t) * (size_t)(wrows * (K / 64))) != cudaSuccess) {
        cudaFree(dtr); cudaFree(err); return -3;
    }
    q8_scales_by_kstep(static_cast<const __half*>(Ws), wrows, K, ks, 0);
    bool ok = launch_gemm_tn2q8_traced(xm, qm, ks, epi, (int)K, (int)M, T, F, Y, ldy, splits, err, 0,
                                       use_y ? &ym : nullptr, dtr);
    uint32_t h = 0;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess &&
         cudaMemcpy(&h, err, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess &&
         cudaMemcpy(trace, dtr, sizeof(uint64_t) * n, cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(ks);
    cudaFree(dtr);
    cudaFree(err);
    return ok && h == 0 ? n : -3;
}

int64_t llm_debug_gemm_tn_f16_trace(int32_t epi, const void* W, int64_t M, int64_t K, const void* X, int32_t T,
                                    float* Y, int32_t ldy, int32_t F, int32_t splits, uint64_t* trace,
                                    int64_t cap) {
    if (!W || !X || !Y || T <= 128 || epi < 0 || epi > 2 || splits < 1) return -1;
    const bool swiglu = epi == GEMM_EPI_SWIGLU;
    if (swiglu ? (!tc_swiglu_tn_ok(K, F) || splits != 1) : !tc_tn_ok(M, K)) return -1;
    const int64_t n = 8 * (int64_t)tc_tn2_blocks(epi, (int)M, T, F, splits);
    if (!trace || cap < n) return -1;
    const int64_t wrows = swiglu ? 2 * (int64_t)F : M;
    CUtensorMap wm, xm, ym;
    if (!tc_make_map(&wm, W, wrows, K, 128, true) || !tc_make_map(&xm, X, T, K, 128, true)) return -1;
    const bool use_y = tc_make_out_map(&ym, Y, T, ldy, swiglu);
    uint32_t* err = nullptr;
    uint64_t* dtr = nullptr;
    if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return -3;
    if (cudaMalloc(&dtr, sizeof(uint64_t) * n) != cudaSuccess) { cudaFree(err); return -3; }
    cudaMemset(err, 0, sizeof(uint32_t));
    bool ok = launch_gemm_tn2_traced(xm, wm, epi, (int)K, (int)M, T, F, Y, ldy, splits, err, 0,
                                     use_y ? &ym : nullptr, dtr);
    uint32_t h = 0;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess &&
         cudaMemcpy(&h, err, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess &&
         cudaMemcpy(trace, dtr, sizeof(uint64_t) * n, cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(err);
    cudaFree(dtr);
    return ok && h == 0 ? n : -3;
}

int32_t llm_sample_ith(llm_ctx* c, int32_t i, const llm_sampler_params* p, float u) {
    constexpr int32_t kMaxPenalty = 4096;
    if (!c || !p || c->host_only) return -1;
    if (p->top_k < 1 || p->top_k > sample_max_k() || !(p->top_p > 0.f && p->top_p <= 1.f) ||
        !(p->min_p >= 0.f && p->min_p < 1.f) || !(u >= 0.f && u < 1.f) ||
        p->n_penalty_tokens < 0 || p->n_penalty_tokens > kMaxPenalty ||
        (p->n_penalty_tokens > 0 && !p->penalty_tokens) || !(p->repeat_penalty > 0.f)) {
        c->err = "invalid sampler parameters";
        return -1;
    }
    const int32_t j = resolve_row(c, i);
    if (j < 0) { c->err = "no logits for this output"; return -1; }
    if (!c->d_sample_state &&
        !(dalloc(c, &c->d_sample_state, sample_state_bytes()) &&
          cuda_ok(c, cudaMemset(c->d_sample_state, 0, sample_state_bytes()), "memset") &&
          dalloc(c, &c->d_sample_tok, (size_t)kMaxPenalty + 2) &&
          cuda_ok(c, cudaMallocHost(&c->h_sample_tok, sizeof(int32_t) * (kMaxPenalty + 2)), "cudaMallocHost")))
        return -1;
    SampleArgs a;
    a.logits = c->d_logits + (size_t)j * c->hp.n_vocab;
    a.V = c->hp.n_vocab;
    a.pen_tok = c->d_sample_tok;
    a.n_pen = p->n_penalty_tokens;
    a.penalty = p->repeat_penalty;
    a.top_k = p->top_k; a.top_p = p->top_p; a.min_p = p->min_p; a.temperature = p->temperature; a.u = u;
    a.out = c->d_sample_tok + kMaxPenalty;              // then the status word
    a.err = reinterpret_cast<uint32_t*>(c->d_sample_tok + kMaxPenalty + 1);
    if (a.n_pen > 0) std::memcpy(c->h_sample_tok, p->penalty_tokens, sizeof(int32_t) * a.n_pen);
    const bool ok =
        (a.n_pen == 0 || cuda_ok(c, cudaMemcpyAsync(c->d_sample_tok, c->h_sample_tok, sizeof(int32_t) * a.n_pen,
                                                    cudaMemcpyHostToDevice, c->st), "copy")) &&
        cuda_ok(c, cudaMemsetAsync(a.out, 0xFF, 2 * sizeof(int32_t), c->st), "memset") &&
        (launch_sample(a, c->d_sample_state, c->n_sm, c->st) || (c->err = "sampler launch failed", false)) &&
        cuda_ok(c, cudaMemcpyAsync(c->h_sample_tok + kMaxPenalty, a.out, 2 * sizeof(int32_t),
                                   cudaMemcpyDeviceToHost, c->st), "copy") &&
        cuda_ok(c, cudaStreamSynchronize(c->st), "sampler");
    if (!ok) return -1;
    const uint32_t st = static_cast<uint32_t>(c->h_sample_tok[kMaxPenalty + 1]);
    if (st == 0xFFFFFFFFu) {                            // a barrier gave up: reset the state
        cudaMemsetAsync(c->d_sample_state, 0, sample_state_bytes(), c->st);
        cudaStreamSynchronize(c->st);
        c->err = "sampler did not finish";
        return -1;
    }
    if (st != 0) { c->err = "sampler found no candidate"; return -1; }
    return c->h_sample_tok[kMaxPenalty];
}

int llm_debug_set_logits(llm_ctx* c, int32_t i, const float* row) {
    if (!c || !row || c->host_only) return -1;
    const int32_t j = resolve_row(c, i);
    if (j < 0) return -1;
    c->h_logits_valid = false;
    return cuda_ok(c, cudaMemcpyAsync(c->d_logits + (size_t)j * c->hp.n_vocab, row, sizeof(float) * c->hp.n_vocab,
                                      cudaMemcpyHostToDevice, c->st), "copy") &&
                   cuda_ok(c, cudaStreamSynchronize(c->st), "copy")
               ? 0 : -1;
}

int llm_debug_step_trace_enable(llm_ctx* c, int enable) {
    if (!c) return -1;
    c->step_trace = enable != 0 && !c->host_only;
    return 0;
}

int64_t llm_debug_step_trace(llm_ctx* c, uint64_t* out, int64_t cap, int32_t* n_blocks, int32_t* n_slots) {
    if (!c || !c->trace_valid || !c->d_trace) return 0;
    const int64_t n = (int64_t)c->trace_blocks * c->trace_slots * 2;
    if (n_blocks) *n_blocks = c->trace_blocks;
    if (n_slots) *n_slots = c->trace_slots;
    if (out && cap > 0) {
        cudaStreamSynchronize(c->st);
        cudaMemcpy(out, c->d_trace, sizeof(uint64_t) * (size_t)std::min(n, cap), cudaMemcpyDeviceToHost);
    }
    return n;
}

int llm_debug_inject_fault(llm_ctx* c, int32_t kind, int32_t ub) {
    if (!c) return -1;
    c->fault_kind = kind;
    c->fault_ub = ub;
    return 0;
}

}  // extern "C"
