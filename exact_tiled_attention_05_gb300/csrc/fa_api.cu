// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// validation, TMA tensor-map encoding, workspace layout, launches and the
// device status word.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.cuh"

namespace fa {
namespace {

// Written by kernels that give up on a bounded wait; read and cleared by
// fa_sync_status.  One copy per device that loads the library.
__device__ int g_status;

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

struct DeviceState {
    std::atomic<int> checked{0};  // 0 unknown, 1 supported, -1 unsupported
    std::atomic<int*> status{nullptr};
    std::atomic<int> sms{0};
};
DeviceState g_dev[kMaxDevices];

EncodeTiledFn encode_fn() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

int current_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    const int n = g_dev[dev].sms.load(std::memory_order_relaxed);
    return n > 0 ? n : 148;
}

int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

// Largest power of two <= x (x >= 1).
int floor_pow2(int x) {
    int p = 1;
    while (p * 2 <= x) p *= 2;
    return p;
}

// Checks the current device (sm_103) and returns its status-word address.
int device_ready(int** status_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return kErrCuda;
    if (dev >= kMaxDevices) return kErrUnsupported;
    DeviceState& st = g_dev[dev];
    int c = st.checked.load(std::memory_order_acquire);
    if (c == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return kErrCuda;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return kErrCuda;
        st.sms.store(sms, std::memory_order_relaxed);
        c = (major == 10 && minor == 3) ? 1 : -1;
        st.checked.store(c, std::memory_order_release);
    }
    if (c < 0) return kErrUnsupported;
    int* p = st.status.load(std::memory_order_acquire);
    if (!p) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) return kErrCuda;
        p = static_cast<int*>(addr);
        st.status.store(p, std::memory_order_release);
    }
    *status_out = p;
    return kOk;
}

// [BH, N, d] bf16 tensor -> 3-D map (d, N, BH), box 64 x 128 x 1, 128 B swizzle.
int make_map(CUtensorMap* map, const void* ptr, int BH, int N, int d) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return kErrCuda;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(d) * 2 * static_cast<cuuint64_t>(N)};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                     strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? kOk : kErrCuda;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int H, int N, int d, float scale, int causal) {
    if (B < 1 || H < 1 || N < 1) return kErrInvalidArg;
    if (causal != 0 && causal != 1) return kErrInvalidArg;
    if (!std::isfinite(scale) || !(scale > 0.f)) return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    const int64_t total = static_cast<int64_t>(B) * H * N * d;
    if (total >= (int64_t(1) << 31)) return kErrInvalidArg;
    return kOk;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// The backward's scratch: D = rowsum(dO * O) and lse * log2(e), each fp32
// [B*H, rows padded to whole 128-row tiles].
size_t ws_half(int B, int H, int N) {
    return round256(static_cast<size_t>(B) * H * ((N + 127) / 128) * 128 * sizeof(float));
}
size_t ws_bytes(int B, int H, int N) { return 2 * ws_half(B, H, N); }

int map_cuda(cudaError_t e) { return e == cudaSuccess ? kOk : kErrCuda; }

// Fills the pointer part of BwdArgs after validating the workspace.
int bwd_common(BwdArgs& a, int B, int H, int N, int d, float scale, int causal, void* workspace,
               size_t workspace_bytes) {
    int rc = check_shape(B, H, N, d, scale, causal);
    if (rc) return rc;
    if (!workspace) return kErrWorkspace;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return kErrWorkspace;
    if (workspace_bytes < ws_bytes(B, H, N)) return kErrWorkspace;
    a.delta = static_cast<float*>(workspace);
    a.lse2 = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws_half(B, H, N));
    a.BH = B * H;
    a.N = N;
    a.n_kblk = (N + 127) / 128;
    a.causal = causal;
    rc = device_ready(&a.status);
    if (rc) return rc;
    // dK/dV kernel: about 0.9 wave of CTAs per head group, rounded down to a
    // power of two (measured best: 4 heads on the N = 4096 workload); dQ
    // kernel: about two waves, as the forward
    a.group = clampi(floor_pow2(clampi((current_sms() * 9 / 10) / a.n_kblk, 1, 1 << 20)), 1, a.BH);
    a.group_dq = clampi(floor_pow2(clampi((2 * current_sms()) / a.n_kblk, 1, 1 << 20)), 1, a.BH);
    a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;
    return kOk;
}

// Shared by the dK/dV and dQ stages: validates, fills BwdArgs and the four
// bf16 tensor maps.
int bwd_maps(BwdArgs& a, CUtensorMap* maps, const void* q, const void* k, const void* v,
             const float* lse, const void* dout, int B, int H, int N, int d, float scale,
             int causal, void* workspace, size_t workspace_bytes) {
    int rc = bwd_common(a, B, H, N, d, scale, causal, workspace, workspace_bytes);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return kErrMisaligned;
    a.q = q;
    a.k = k;
    a.v = v;
    a.lse = lse;
    a.dout = dout;
    const int BH = B * H;
    if ((rc = make_map(&maps[0], q, BH, N, d)) || (rc = make_map(&maps[1], k, BH, N, d)) ||
        (rc = make_map(&maps[2], v, BH, N, d)) || (rc = make_map(&maps[3], dout, BH, N, d)))
        return rc;
    return kOk;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 200; }

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, void* stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    int rc = check_shape(B, H, N, d, scale, causal);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return FA_ERR_MISALIGNED;
    FwdArgs a{};
    if ((rc = device_ready(&a.status))) return rc;
    const int BH = B * H;
    CUtensorMap tq, tk, tv, to;
    if ((rc = make_map(&tq, q, BH, N, d)) || (rc = make_map(&tk, k, BH, N, d)) ||
        (rc = make_map(&tv, v, BH, N, d)) || (rc = make_map(&to, o, BH, N, d)))
        return rc;
    a.o = o;
    a.lse = lse;
    a.BH = BH;
    a.N = N;
    a.n_qblk = (N + 255) / 256;
    // about two waves of CTAs per head group, rounded down to a power of two
    // (measured: 8 heads at N = 8192, 16 at N = 4096)
    a.group = clampi(floor_pow2(clampi((2 * current_sms()) / a.n_qblk, 1, 1 << 20)), 1, BH);
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    return map_cuda(launch_fwd(d, tq, tk, tv, to, a, static_cast<cudaStream_t>(stream)));
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    return ws_bytes(B, H, N);
}

int fa_bwd_prep(const void* o, const void* dout, const float* lse, int B, int H, int N, int d,
                void* workspace, size_t workspace_bytes, void* stream) {
    if (!o || !dout || !lse) return FA_ERR_INVALID_ARG;
    BwdArgs a{};
    int rc = bwd_common(a, B, H, N, d, 1.f, 0, workspace, workspace_bytes);
    if (rc) return rc;
    if (!aligned16(o) || !aligned16(dout) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return FA_ERR_MISALIGNED;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    return map_cuda(launch_bwd_prep(d, a, static_cast<cudaStream_t>(stream)));
}

int fa_bwd_main(const void* q, const void* k, const void* v, const float* lse, const void* dout,
                void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !lse || !dout || !dk || !dv) return FA_ERR_INVALID_ARG;
    BwdArgs a{};
    CUtensorMap m[4];
    int rc = bwd_maps(a, m, q, k, v, lse, dout, B, H, N, d, scale, causal, workspace,
                      workspace_bytes);
    if (rc) return rc;
    if (!aligned16(dk) || !aligned16(dv)) return FA_ERR_MISALIGNED;
    a.dk = dk;
    a.dv = dv;
    CUtensorMap tdk, tdv;
    if ((rc = make_map(&tdk, dk, B * H, N, d)) || (rc = make_map(&tdv, dv, B * H, N, d))) return rc;
    return map_cuda(
        launch_bwd_dkdv(d, m[0], m[1], m[2], m[3], tdk, tdv, a, static_cast<cudaStream_t>(stream)));
}

int fa_bwd_dq(const void* q, const void* k, const void* v, const float* lse, const void* dout,
              void* dq, int B, int H, int N, int d, float scale, int causal, void* workspace,
              size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !lse || !dout || !dq) return FA_ERR_INVALID_ARG;
    BwdArgs a{};
    CUtensorMap m[4];
    int rc = bwd_maps(a, m, q, k, v, lse, dout, B, H, N, d, scale, causal, workspace,
                      workspace_bytes);
    if (rc) return rc;
    if (!aligned16(dq)) return FA_ERR_MISALIGNED;
    a.dq = dq;
    CUtensorMap tdq;
    if ((rc = make_map(&tdq, dq, B * H, N, d))) return rc;
    return map_cuda(launch_bwd_dq(d, m[0], m[1], m[2], m[3], tdq, a, static_cast<cudaStream_t>(stream)));
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
           int causal, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    int rc = check_shape(B, H, N, d, scale, causal);
    if (rc) return rc;
    if ((rc = fa_bwd_prep(o, dout, lse, B, H, N, d, workspace, workspace_bytes, stream))) return rc;
    if ((rc = fa_bwd_main(q, k, v, lse, dout, dk, dv, B, H, N, d, scale, causal, workspace,
                          workspace_bytes, stream)))
        return rc;
    return fa_bwd_dq(q, k, v, lse, dout, dq, B, H, N, d, scale, causal, workspace, workspace_bytes,
                     stream);
}

int fa_sync_status(void* stream) {
    int* p = nullptr;
    int rc = device_ready(&p);
    if (rc) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    int host = 0;
    if (cudaMemcpy(&host, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (host != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return FA_ERR_CUDA;
        return host;
    }
    return FA_OK;
}

}  // extern "C"
