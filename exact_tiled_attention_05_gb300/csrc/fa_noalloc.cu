// fa_noalloc.cu -- a backward pass for callers that cannot allocate device
// memory.
//
// fa_bwd needs a scratch workspace (two fp32 row statistics) that the caller
// allocates.  Some callers cannot do that: code
// that runs where cudaMalloc is unavailable or forbidden (inside a custom
// allocator's own callbacks, a fixed-footprint embedded service that must not
// grow its memory after start-up, or a plug-in whose host framework owns every
// allocation).  fa_bwd_noalloc gives them the same computation with the scratch
// held in one fixed-size array in this library's device memory.
//
// That array lives in every GPU that loads this part of the library and stays
// there until the process exits.  All calls on a device share it: it keeps the
// contents of the previous call (the prep stage rewrites it on every call), and
// two calls whose work overlaps on the GPU (different streams, or different
// host threads without ordering) race on it and give wrong results.
#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.cuh"

namespace {

// 64 MiB and 256 bytes: fa_bwd_workspace_size (8 bytes per row, rows padded to
// whole 128-row tiles, and 256 bytes of work counters) must fit, i.e. up to 2^23
// rows; larger sizes return FA_ERR_WORKSPACE.
constexpr size_t kNoAllocScratchBytes = (size_t(64) << 20) + 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device.  The host-side
// name g_noalloc_scratch is only a stand-in, so the address is looked up once
// per device with that device current.
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return FA_ERR_CUDA;
    if (dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (!p) {
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
                return FA_ERR_CUDA;
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return FA_OK;
}

}  // namespace

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal, void* stream) {
    // The checks run in fa_bwd's order (pointers, shape, workspace, alignment),
    // so a call gets the error fa_bwd would give with a large enough workspace;
    // the fixed scratch stands in for that workspace.  Nothing touches the
    // device before all of them pass.
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    int rc = fa::check_shape(B, H, N, d, scale, causal);
    if (rc != FA_OK) return rc;
    if (fa_bwd_workspace_size(B, H, N, d) > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return FA_ERR_MISALIGNED;
    void* scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != FA_OK) return rc;
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, scratch,
                  kNoAllocScratchBytes, stream);
}
