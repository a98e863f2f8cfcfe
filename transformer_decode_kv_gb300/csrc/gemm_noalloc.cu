// A variant of the tensor-core GEMM entry point that allocates no device memory.
//
// Who needs it: callers that cannot allocate device memory. Serving engines often reserve all of
// a GPU's memory at start-up for weights and KV cache and hand out only their own pools, so a
// cudaMalloc from a library call either fails or eats into memory that was promised elsewhere;
// and cudaFree synchronises the whole device, which stalls every other stream of a process that
// is running latency-critical work. llm_debug_gemm_bf16 allocates (and frees) its scratch on each
// call; llm_gemm_bf16_noalloc keeps that scratch in a fixed array compiled into the library.
//
// The scratch is the kernel's error word (the tcgen05 GEMM reports a timed-out wait there). It
// lives in g_gemm_noalloc_scratch below, a file-scope __device__ array that every GPU which loads
// the library holds until the process exits. Host code cannot use the array's name as a device
// address, so the first call on each device looks its address up with cudaGetSymbolAddress while
// that device is current and keeps it for later calls.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/llm.h"
#include "gemm_tc.h"

namespace {

// Maximum scratch: 64 words (256 bytes); word 0 is the error word of the running call.
constexpr int kNoAllocScratchWords = 64;
static __device__ __align__(256) uint32_t g_gemm_noalloc_scratch[kNoAllocScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
uint32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
uint32_t* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_ptr[dev] = static_cast<uint32_t*>(p);
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int llm_gemm_bf16_noalloc(int32_t epi, const void* W, int64_t M, int64_t K,
                                     const void* X, int32_t T, void* Y, int32_t ldy, int32_t F) {
    using namespace llm;
    if (!W || !X || !Y || T <= 0 || epi < 0 || epi > 2) return -1;
    if (!tc_shape_ok(M, K, epi, F)) return -1;
    // the error word is the only scratch this call needs; it always fits in the fixed array
    static_assert(kNoAllocScratchWords >= 1, "scratch must hold the error word");
    const int64_t wrows = epi == GEMM_EPI_SWIGLU ? 2 * (int64_t)F : M;
    CUtensorMap wm, xm;
    if (!tc_make_map(&wm, W, wrows, K, epi == GEMM_EPI_SWIGLU ? 64 : 128) ||
        !tc_make_map(&xm, X, T, K, tc_token_tile(T)))
        return -1;
    uint32_t* err = scratch_on_current_device();
    if (!err) return -3;
    // the array keeps the previous call's contents: the error word must start at zero
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), 0) != cudaSuccess) return -3;
    bool ok = launch_gemm_tc(wm, xm, epi, (int)K, (int)M, T, F, Y, ldy, err, 0);
    uint32_t h = 0;
    ok = ok && cudaStreamSynchronize(0) == cudaSuccess &&
         cudaMemcpy(&h, err, sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess;
    return ok && h == 0 ? 0 : -3;
}

extern "C" int llm_debug_noalloc_scratch_poke(uint32_t value) {
    uint32_t* err = scratch_on_current_device();
    if (!err) return -3;
    return cudaMemcpy(err, &value, sizeof(uint32_t), cudaMemcpyHostToDevice) == cudaSuccess ? 0 : -3;
}
