// Prefill attention on the fifth-generation tensor cores (tcgen05, accumulators in TMEM), for query
// tiles of several tokens over an F16 cache with head_dim 128 and 4 query heads per KV head
// ([P2] "llama.cpp Architecture", Example 4 FLASH_ATTN_EXT; Example 11 for the unfused meaning:
// scores Q K^T with the KQ mask, softmax, times V; scale 1/sqrt(hd)).
//
// A CTA takes one work item of the plan (a query tile of up to 32 tokens of one cell list and a
// range of that list) for one KV head. Its 128 MMA rows are the tile's 32 tokens x the 4 query
// heads of the KV head (row r: token r / 4, head r % 4). Per step of 128 cells of the list:
//   S = Q K^T        tcgen05.mma M 128 x N 128 x K 128 into one of two TMEM score buffers
//   softmax          a thread per row reads its 128 scores (tcgen05.ld), masks cells with
//                    position > the token's, and writes P = 2^(s - m) as f16 to shared memory
//   O += P V         tcgen05.mma M 128 x N 128 (head dims) x K 128 (cells) into TMEM, V read as
//                    stored (cells x dims: a B operand in MN-major layout)
// Q and P are one f16 term each and accumulation is float32: the precision of a forward pass
// whose matrix products take f16 activations. Scores are in the log2 domain (log2 e / sqrt(hd)
// folded into Q; the powers of two by the hardware ex2 approximation). The running maximum is raised lazily: O and the row sum are rescaled only when
// a row's maximum grows by more than 8 (P stays below 2^8 otherwise), and the final division
// uses the same maximum for both, so the result does not depend on when rescaling happened.
//
// Roles (224 threads): warp 0 brings the K and V rows of each step with the cells' positions into
// 128-byte-swizzled tiles (bulk tensor copies when the step's cells are consecutive, else a gather
// by cell index, cp.async 16 bytes per copy), warps 1 and 3-6 write the Q tile, warp 2 allocates
// TMEM and one of its threads issues the MMAs, warps 3-6 run the softmax and the epilogue (warp w
// reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31; TMEM loads and stores are warp-wide, so every
// one runs with the whole warp converged, whatever its rows need). Cells past the last one any row
// may see are not visited (the plan ends each work item at the last entry a row may see). Every
// wait is bounded by a wall-clock limit; a timeout sets ERR_TIMEOUT and the CTA drains what it
// issued and frees TMEM.
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "attn_common.cuh"
#include "kernels.h"

namespace llm {

namespace {

using namespace attn;

constexpr int kHD = 128;
constexpr int kG = 4;
constexpr int kTok = 32;                         // tokens per query tile
constexpr int kRows = kTok * kG;                 // 128 MMA rows
constexpr int kCells = 128;                      // cells per step
constexpr int kThreads = 224;
constexpr int kQThreads = 160;                   // warps 1 and 3-6 write the Q tile
constexpr uint32_t kBlk = 128 * 64 * 2;          // [128 rows][64 f16], 128-byte swizzle: 16 KB
constexpr uint32_t kTileB = 2 * kBlk;            // [128 rows][128 f16]: 32 KB
constexpr uint64_t kWaitNs = 2000000000ull;

struct TcSmem {
    // offsets from the 1024-aligned base
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k0 = q + kTileB;
    static constexpr uint32_t v0 = k0 + 2 * kTileB;
    static constexpr uint32_t p = v0 + 2 * kTileB;
    static constexpr uint32_t cpos = p + kTileB;                 // int [2][kCells]
    static constexpr uint32_t rpos = cpos + 2 * kCells * 4;      // int [kRows], then [kTok] tokens
    static constexpr uint32_t misc = rpos + (kRows + kTok) * 4;  // ints: flag, abort, tmem
    static constexpr uint32_t bars = misc + 64;                  // mbarriers
    static constexpr uint32_t bytes = bars + 16 * 8;
    static constexpr size_t alloc = 1024 + (size_t)bytes;
};

__device__ __forceinline__ uint64_t gns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(n));
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t par) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(par)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t par) {
    if (mb_try(b, par)) return true;
    const uint64_t t0 = gns();
    while (!mb_try(b, par))
        if (gns() - t0 > kWaitNs) return false;
    return true;
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// K-major tile of 128 rows with the 128-byte swizzle: 8-row groups 1024 bytes apart
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// MN-major tile (rows = the contracted dimension, 64-element column blocks kBlk bytes apart) with
// the 128-byte swizzle: leading offset = the column-block stride, stride offset = the 8-row
// group stride
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(kBlk >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// kind::f16, f16 A and B, f32 D; transpose_b: B in MN-major layout
__host__ __device__ constexpr uint32_t idesc(int m, int n, bool transpose_b) {
    return (1u << 4) | ((transpose_b ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint64_t* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(b))
                 : "memory");
}
// warp-wide TMEM load of 32 columns (the warp is reconverged first: every lane must take part)
__device__ __forceinline__ void ld32(uint32_t taddr, float* v) {
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
// warp-wide TMEM load of 64 columns; the caller waits (tcgen05.wait::ld) before using v
__device__ __forceinline__ void ld64_nowait(uint32_t taddr, uint32_t* r) {
    __syncwarp();
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,"
        "%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
}

__device__ __forceinline__ void st32(uint32_t taddr, const float* v) {
    __syncwarp();
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}
// 2^x by the hardware approximation (PTX ex2.approx.ftz: a few ulp of float32; -inf gives 0),
// for P, which is rounded to f16 (11 significant bits) right after
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// byte offset of 16-byte chunk `ch` (0..15) of row `r` in a [128 rows][128 f16] tile made of two
// 128-byte-swizzled [128][64] blocks
__device__ __forceinline__ uint32_t swz(int r, int ch) {
    return (uint32_t)((ch >> 3) * kBlk + r * 128 + ((((uint32_t)ch & 7u) ^ ((uint32_t)r & 7u)) << 4));
}

// use_tma: tmK / tmV map this context's K and V caches as [layers x heads x cells][128] f16 rows
// (boxes of 64 dims x 128 rows, 128-byte swizzle): a step whose cells are consecutive comes in four
// bulk tensor copies; other steps are gathered row by row.
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnArgs a, float scale_log2,
                                                              const __grid_constant__ CUtensorMap tmK,
                                                              const __grid_constant__ CUtensorMap tmV, int use_tma) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    int* cposb = reinterpret_cast<int*>(sm + TcSmem::cpos);
    int* rpos = reinterpret_cast<int*>(sm + TcSmem::rpos);
    int* misc = reinterpret_cast<int*>(sm + TcSmem::misc);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + TcSmem::bars);
    uint64_t* kv_full = bars;          // [2] count 1: lane 0 of the gathering warp (+ bulk copy bytes)
    uint64_t* kv_empty = bars + 2;     // [2] count 1: MMA commit after O += P V
    uint64_t* s_full = bars + 4;       // [2] count 1: MMA commit after S = Q K^T
    uint64_t* s_free = bars + 6;       // [2] count 128: the softmax threads read S
    uint64_t* p_full = bars + 8;       // count 128: P written (and O rescaled)
    uint64_t* o_done = bars + 9;       // count 1: O += P V of a step ended
    uint64_t* q_full = bars + 10;      // count kQThreads: the Q tile written
    int* flag = misc + 2;
    int* abort_f = misc + 3;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 4);

    const int wi = blockIdx.x, kvh = blockIdx.y;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    if (wi >= a.hdr[0]) return;                      // past this ubatch's work items
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int4 wd = a.wi_desc[wi];
    const int4 td0 = a.tile_desc[2 * wd.x];
    const int4 td1 = a.tile_desc[2 * wd.x + 1];
    const int nq = td0.z, s0 = td0.y, c0 = wd.y, c1 = wd.z, base = td1.y;
    const int w0 = td0.w, w1 = td1.x;
    const __half* K = static_cast<const __half*>(a.kc) + (int64_t)kvh * a.n_ctx * kHD;
    const __half* V = static_cast<const __half*>(a.vc) + (int64_t)kvh * a.n_ctx * kHD;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (threadIdx.x == 0) {
        mb_init(&kv_full[0], 1); mb_init(&kv_full[1], 1);
        mb_init(q_full, kQThreads);
        mb_init(&kv_empty[0], 1); mb_init(&kv_empty[1], 1);
        mb_init(&s_full[0], 1); mb_init(&s_full[1], 1);
        mb_init(&s_free[0], kRows); mb_init(&s_free[1], kRows);
        mb_init(p_full, kRows);
        mb_init(o_done, 1);
        *abort_f = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(512u));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    int* rtok = rpos + kRows;            // [kTok] token index of each tile row group
    if (threadIdx.x < kTok) {
        const int t = threadIdx.x < nq ? a.perm[s0 + threadIdx.x] : -1;
        rtok[threadIdx.x] = t;
        const int p = t >= 0 ? a.tok_pos[t] : INT_MIN;
#pragma unroll
        for (int h = 0; h < kG; ++h) rpos[threadIdx.x * kG + h] = p;
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_slot;
    const int cend = c1;                  // the plan leaves out entries no row of the tile may see
    const int nt = (cend - c0 + kCells - 1) / kCells;     // steps of 128 cells
    const uint32_t sbuf[2] = {tmem, tmem + 128};
    const uint32_t obuf = tmem + 256;

    // the Q tile: f16 of q times log2(e) / sqrt(hd), 128-byte-swizzled [128 rows][128 dims],
    // written by warps 1 and 3-6 while warp 0 fetches the first keys and values
    const int qt = warp == 1 ? lane : warp >= 3 ? 32 + 32 * (warp - 3) + lane : -1;
    if (qt >= 0) {
#pragma unroll 4
    for (int v = qt; v < kRows * 16; v += kQThreads) {
        const int r = v >> 4, ch = v & 15;
        const int t = rtok[r / kG];
        uint32_t h[4] = {0u, 0u, 0u, 0u};
        if (t >= 0) {
            const float* qp = a.q + (int64_t)t * a.ldq + (kvh * kG + r % kG) * kHD + ch * 8;
            const float4 x0 = *reinterpret_cast<const float4*>(qp);
            const float4 x1 = *reinterpret_cast<const float4*>(qp + 4);
            h[0] = pack_h2(x0.x * scale_log2, x0.y * scale_log2);
            h[1] = pack_h2(x0.z * scale_log2, x0.w * scale_log2);
            h[2] = pack_h2(x1.x * scale_log2, x1.y * scale_log2);
            h[3] = pack_h2(x1.z * scale_log2, x1.w * scale_log2);
        }
        *reinterpret_cast<uint4*>(sm + TcSmem::q + swz(r, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
        proxy_fence();
        mb_arrive(q_full);
    }

    if (warp == 0) {
        // ---- keys and values: every step of 128 list entries into stage j % 2 (after the
        // step that used it two steps earlier has been multiplied into O), with the cells'
        // positions for the mask. Consecutive cells: four bulk tensor copies (K and V, 64 dims
        // each) counted on the stage's barrier; otherwise rows gathered by cell index.
        const int64_t row0 = (int64_t)a.kv_row0 + (int64_t)kvh * a.n_ctx;
        for (int j = 0; j < nt; ++j) {
            const int s = j & 1;
            if (j >= 2 && !mb_wait(&kv_empty[s], (uint32_t)((j >> 1) - 1) & 1u)) {
                if (a.err) atomicOr(a.err, ERR_TIMEOUT);
                *(volatile int*)abort_f = 1;
            }
            if (__any_sync(0xffffffffu, *(volatile int*)abort_f != 0)) break;
            uint8_t* kt = sm + TcSmem::k0 + s * kTileB;
            uint8_t* vt = sm + TcSmem::v0 + s * kTileB;
            int* cpos = cposb + s * kCells;
            const int n = min(kCells, cend - (c0 + j * kCells));      // list entries of the step
            int cell[kCells / 32];
            bool valid = true;
#pragma unroll
            for (int u = 0; u < kCells / 32; ++u) {
                const int i = lane + 32 * u;
                int cc = -1, pos = INT_MAX;
                if (i < n) {
                    cc = a.list_cells[base + c0 + j * kCells + i];
                    pos = a.list_pos[base + c0 + j * kCells + i];
                    if (cc < 0 || cc >= a.n_ctx) { valid = false; pos = INT_MAX; }
                }
                cell[u] = cc;
                cpos[i] = pos;
            }
            const int first = __shfl_sync(0xffffffffu, cell[0], 0);
            int lastv = cell[0];
#pragma unroll
            for (int u = 1; u < kCells / 32; ++u)
                if (u == (n - 1) / 32) lastv = cell[u];
            const int last = __shfl_sync(0xffffffffu, lastv, (n - 1) & 31);
            // a list is ascending: its entries are consecutive cells iff last - first = n - 1
            const bool contig = use_tma && __all_sync(0xffffffffu, valid) && last - first == n - 1;
            if (contig) {
                __syncwarp();
                if (lane == 0) {
                    const uint32_t fb = smem_addr(&kv_full[s]);
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(4 * kBlk)
                                 : "memory");
                    const int y = (int)(row0 + first);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        asm volatile(
                            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                            " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(kt + h * kBlk)),
                            "l"(reinterpret_cast<uint64_t>(&tmK)), "r"(fb), "r"(64 * h), "r"(y)
                            : "memory");
                        asm volatile(
                            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                            " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(vt + h * kBlk)),
                            "l"(reinterpret_cast<uint64_t>(&tmV)), "r"(fb), "r"(64 * h), "r"(y)
                            : "memory");
                    }
                }
            } else {
#pragma unroll 1
                for (int u = 0; u < kCells / 32; ++u) {
                    const int i = lane + 32 * u;
                    const bool ok = cpos[i] != INT_MAX;
#pragma unroll
                    for (int ch = 0; ch < 16; ++ch) {
                        const uint32_t o = swz(i, ch);
                        if (ok) {
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(kt + o)),
                                         "l"(K + (int64_t)cell[u] * kHD + ch * 8) : "memory");
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(vt + o)),
                                         "l"(V + (int64_t)cell[u] * kHD + ch * 8) : "memory");
                        } else {
                            *reinterpret_cast<uint4*>(kt + o) = make_uint4(0u, 0u, 0u, 0u);
                            *reinterpret_cast<uint4*>(vt + o) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                proxy_fence();
                __syncwarp();
                if (lane == 0) mb_arrive(&kv_full[s]);
            }
        }
        // the bulk copies issued have landed before the CTA can leave
        __syncwarp();
        if (lane == 0)
            for (int j = nt > 2 ? nt - 2 : 0; j < nt; ++j) mb_wait(&kv_full[j & 1], (uint32_t)(j >> 1) & 1u);
    } else if (warp == 2) {
        if (lane == 0) {
            // ---- MMA issuer
            constexpr uint32_t ids = idesc(kRows, kCells, false);
            constexpr uint32_t ido = idesc(kRows, kHD, true);
            const uint32_t qa = smem_addr(sm + TcSmem::q);
            const uint32_t pa = smem_addr(sm + TcSmem::p);
            bool ok = true;
            auto pv = [&](int i) {
                if (!mb_wait(p_full, (uint32_t)i & 1u)) { ok = false; return; }
                tc_after();
                const uint32_t va = smem_addr(sm + TcSmem::v0 + (i & 1) * kTileB);
#pragma unroll
                for (int kk = 0; kk < kCells / 16; ++kk)
                    mma(obuf, desc_k(pa + (kk >> 2) * kBlk) + (uint64_t)(2 * (kk & 3)),
                        desc_mn(va + kk * 2048), ido, (i > 0 || kk > 0) ? 1u : 0u);
                commit(o_done);
                commit(&kv_empty[i & 1]);
            };
            ok = nt == 0 || mb_wait(q_full, 0);
            int j = 0;
            for (; j < nt && ok; ++j) {
                const int s = j & 1;
                if (!mb_wait(&kv_full[s], (uint32_t)(j >> 1) & 1u)) { ok = false; break; }
                if (j >= 2 && !mb_wait(&s_free[s], (uint32_t)((j >> 1) - 1) & 1u)) { ok = false; break; }
                tc_after();
                const uint32_t ka = smem_addr(sm + TcSmem::k0 + s * kTileB);
#pragma unroll
                for (int kk = 0; kk < kHD / 16; ++kk)
                    mma(sbuf[s], desc_k(qa + (kk >> 2) * kBlk) + (uint64_t)(2 * (kk & 3)),
                        desc_k(ka + (kk >> 2) * kBlk) + (uint64_t)(2 * (kk & 3)), ids, kk > 0 ? 1u : 0u);
                commit(&s_full[s]);
                if (j >= 1) pv(j - 1);
            }
            if (ok && nt > 0) pv(nt - 1);
            if (!ok) {
                if (a.err) atomicOr(a.err, ERR_TIMEOUT);
                *(volatile int*)abort_f = 1;
            }
        }
        __syncwarp();
    }

    // ---- softmax and epilogue (warps 3-6): thread = row
    float m = -INFINITY, l = 0.f;
    const bool sw = warp >= 3;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    bool live = true;
    if (sw) {
        const int rp = rpos[r];
        uint8_t* prow = sm + TcSmem::p;
        for (int j = 0; j < nt; ++j) {
            const int s = j & 1;
            // the step's scores, and the cells' positions the gathering warps stored
            bool ok = mb_wait(&s_full[s], (uint32_t)(j >> 1) & 1u) && mb_wait(&kv_full[s], (uint32_t)(j >> 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) { live = false; break; }
            tc_after();
            const int4* cpos4 = reinterpret_cast<const int4*>(cposb + s * kCells);
            // the row's 128 scores: two 64-column loads, one wait
            uint32_t v[kCells];
            ld64_nowait(sbuf[s] + lane_base, v);
            ld64_nowait(sbuf[s] + lane_base + 64, v + 64);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            tc_before();
            mb_arrive(&s_free[s]);
            // masked cells (position > the token's) become -inf; the largest visible score
            float mx = -INFINITY;
#pragma unroll
            for (int c4 = 0; c4 < kCells / 4; ++c4) {
                const int4 cp = cpos4[c4];
                if (cp.x > rp) v[4 * c4] = __float_as_uint(-INFINITY);
                if (cp.y > rp) v[4 * c4 + 1] = __float_as_uint(-INFINITY);
                if (cp.z > rp) v[4 * c4 + 2] = __float_as_uint(-INFINITY);
                if (cp.w > rp) v[4 * c4 + 3] = __float_as_uint(-INFINITY);
                mx = fmaxf(mx, fmaxf(fmaxf(__uint_as_float(v[4 * c4]), __uint_as_float(v[4 * c4 + 1])),
                                     fmaxf(__uint_as_float(v[4 * c4 + 2]), __uint_as_float(v[4 * c4 + 3]))));
            }
            const float mn = fmaxf(m, mx);
            float mu = m;
            bool rescale = false;
            if (mn != -INFINITY && (m == -INFINITY || mn > m + 8.f)) {
                rescale = m != -INFINITY && l > 0.f;
                mu = mn;
            }
            // P = 2^(s - mu), packed f16 in place of the scores (a masked cell gives 0)
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kCells; c += 2) {
                const float p0 = mu == -INFINITY ? 0.f : ex2(__uint_as_float(v[c]) - mu);
                const float p1 = mu == -INFINITY ? 0.f : ex2(__uint_as_float(v[c + 1]) - mu);
                sum += p0 + p1;
                v[c / 2] = pack_h2(p0, p1);
            }
            const float f = rescale ? ex2(m - mu) : 1.f;
            l = l * f + sum;
            m = mu;
            // O += P V of the previous step has ended: P's buffer is free and O is stable
            ok = j == 0 || mb_wait(o_done, (uint32_t)(j - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) { live = false; break; }
            tc_after();
#pragma unroll
            for (int ch = 0; ch < kCells / 8; ++ch)
                *reinterpret_cast<uint4*>(prow + swz(r, ch)) = make_uint4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
            // TMEM loads and stores are warp-wide: the whole warp rescales when any of its rows
            // needs it (f = 1 for the others)
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int q = 0; q < kHD / 32; ++q) {
                    float o[32];
                    ld32(obuf + lane_base + 32 * q, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= f;
                    st32(obuf + lane_base + 32 * q, o);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            proxy_fence();
            tc_before();
            mb_arrive(p_full);
        }
        if (live && nt > 0 && !__all_sync(0xffffffffu, mb_wait(o_done, (uint32_t)(nt - 1) & 1u))) live = false;
        tc_after();
        if (!live && a.err) atomicOr(a.err, ERR_TIMEOUT);
    }
    live = live && !*(volatile int*)abort_f;

    const int j = r / kG;
    if (w1 - w0 == 1) {
        // a single work item: normalise and store the tile's rows (f16)
        if (sw) {
#pragma unroll 1
            for (int q = 0; q < kHD / 32; ++q) {
                float o[32];
                if (nt > 0) ld32(obuf + lane_base + 32 * q, o);
                if (!live || j >= nq) continue;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                __half* dst = static_cast<__half*>(a.out_b) + (int64_t)a.perm[s0 + j] * a.ldo +
                              (kvh * kG + r % kG) * kHD + 32 * q;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 h = make_uint4(pack_h2(nt > 0 ? o[8 * c] * inv : 0.f, nt > 0 ? o[8 * c + 1] * inv : 0.f),
                                               pack_h2(nt > 0 ? o[8 * c + 2] * inv : 0.f, nt > 0 ? o[8 * c + 3] * inv : 0.f),
                                               pack_h2(nt > 0 ? o[8 * c + 4] * inv : 0.f, nt > 0 ? o[8 * c + 5] * inv : 0.f),
                                               pack_h2(nt > 0 ? o[8 * c + 6] * inv : 0.f, nt > 0 ? o[8 * c + 7] * inv : 0.f));
                    reinterpret_cast<uint4*>(dst)[c] = h;
                }
            }
        }
    } else {
        // several work items share the tile: this one's partial state (o, m, l), then the last
        // to finish merges them
        if (sw) {
            // TMEM loads are warp-wide: every thread of the warp loads, the rows of the tile store
            const bool mine = j < nq;
            const int64_t row = (int64_t)(wd.w + r) * a.Hkv + kvh;
            if (mine) {
                a.part_m[row] = live ? m : -INFINITY;
                a.part_l[row] = live ? l : 0.f;
            }
#pragma unroll 1
            for (int q = 0; q < kHD / 32; ++q) {
                float o[32];
                if (nt > 0) ld32(obuf + lane_base + 32 * q, o);
                else
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;
                if (!mine) continue;
                float4* dst = reinterpret_cast<float4*>(a.part_o + row * kHD + 32 * q);
#pragma unroll
                for (int c = 0; c < 8; ++c) dst[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            }
        }
    }
    tc_before();
    __syncthreads();
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u));
    if (w1 - w0 == 1) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        int* ticket = a.tickets + wd.x * a.Hkv + kvh;
        const int done = atomicAdd(ticket, 1) + 1;
        const bool last = done == w1 - w0;
        if (last) *ticket = 0;
        *flag = last ? 1 : 0;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    merge_tile<kHD, kG>(a, kvh, s0, nq, w0, w1, reinterpret_cast<float*>(sm + TcSmem::k0), 4 * kTileB / 4);
}

}  // namespace

int attention_tc_tile_q() { return kTok; }

bool attention_tc_ok(const AttnArgs& a) {
    return a.kv_type == W_F16 && !a.k_scale && a.hd == kHD && a.H == kG * a.Hkv && a.out_b && a.out_f16;
}

bool launch_attention_tc(const AttnArgs& a, cudaStream_t st) {
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)kHD));
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcSmem::alloc) !=
            cudaSuccess)
            return false;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_work, a.Hkv);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = TcSmem::alloc;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = a.pdl ? 1 : 0;
    const bool tma = a.kmap && a.vmap;
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel, a, scale_log2, tma ? *a.kmap : CUtensorMap{},
                              tma ? *a.vmap : CUtensorMap{}, tma ? 1 : 0) == cudaSuccess;
}

}  // namespace llm
