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

int check_shape(int B, int H, int N, int d, float scale, int causal) {
    if (B < 1 || H < 1 || N < 1) return kErrInvalidArg;
    if (causal != 0 && causal != 1) return kErrInvalidArg;
    if (!std::isfinite(scale) || !(scale > 0.f)) return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    const int64_t total = static_cast<int64_t>(B) * H * N * d;
    if (total >= (int64_t(1) << 31)) return kErrInvalidArg;
    return kOk;
}

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

int ceil_pow2(int x) {
    int p = 1;
    while (p < x && p < (1 << 30)) p <<= 1;
    return p;
}

// Heads in the last group of a causal work order (see grouped_item): at least
// 3 * sms / nblk, so that the group's work spread over the SMs lasts about 1.5
// times its heaviest item (nblk blocks of a head hold ~nblk^2 / 2 tiles).
int last_group(int sms, int nblk, int group, int BH) {
    const int need = (3 * sms + nblk - 1) / nblk;
    return clampi(group > ceil_pow2(need) ? group : ceil_pow2(need), 1, BH);
}

// Largest power of two <= x (x >= 1).
int floor_pow2(int x) {
    int p = 1;
    while (p * 2 <= x) p *= 2;
    return p;
}

// Checks the current device (sm_103) and returns its status-word address.  It
// also makes the device's primary context current on the calling thread: the
// tensor-map encoding is a driver call that needs a current context, and a
// thread that has made no runtime call yet (a worker thread, for example) has
// none.
int device_ready(int** status_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return kErrCuda;
    if (cudaSetDevice(dev) != cudaSuccess) return kErrCuda;
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

// uint8 tensor [z, y, x] -> 3-D map (x, y, z), box 128 x 128 x 1, 128 B swizzle
// (one FP8 tile of 128 rows by 128 bytes).
int make_map_u8(CUtensorMap* map, const void* ptr, int x, int y, int z) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return kErrCuda;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(x), static_cast<cuuint64_t>(y),
                          static_cast<cuuint64_t>(z)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(x),
                             static_cast<cuuint64_t>(x) * static_cast<cuuint64_t>(y)};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides,
                     box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? kOk : kErrCuda;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// The backward's scratch: D = rowsum(dO * O) and lse * log2(e), each fp32
// [B*H, rows padded to whole 128-row tiles].
size_t ws_half(int B, int H, int N) {
    return round256(static_cast<size_t>(B) * H * ((N + 127) / 128) * 128 * sizeof(float));
}
size_t ws_bytes(int B, int H, int N) { return 2 * ws_half(B, H, N) + 256; }  // + work counters

// FP8 workspace: segment offsets (each 256-byte aligned), in the order fa.h lists.
struct Fp8Layout {
    size_t q8, k8, vt8, sq, sk, sv, vfold, vmax, amax, total;
};
Fp8Layout fp8_layout(int B, int H, int N) {
    const size_t BH = static_cast<size_t>(B) * H;
    const size_t T = (static_cast<size_t>(N) + 127) / 128;
    const size_t codes = round256(BH * T * 128 * 128);
    const size_t per_tile = round256(BH * T * sizeof(float));
    Fp8Layout l{};
    size_t o = 0;
    l.q8 = o; o += codes;
    l.k8 = o; o += codes;
    l.vt8 = o; o += codes;
    l.sq = o; o += per_tile;
    l.sk = o; o += per_tile;
    l.sv = o; o += per_tile;
    l.vfold = o; o += per_tile;
    l.vmax = o; o += round256(BH * sizeof(float));
    l.amax = o; o += 256;
    l.total = o;
    return l;
}

int fp8_shape(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1) return kErrInvalidArg;
    if (d != 128) return kErrUnsupported;
    const int64_t rows = static_cast<int64_t>(B) * H * ((static_cast<int64_t>(N) + 127) / 128) * 128;
    if (rows * 128 >= (int64_t(1) << 31)) return kErrInvalidArg;
    // the quantizers launch one CTA row per head on the grid's y dimension
    if (static_cast<int64_t>(B) * H > 65535) return kErrUnsupported;
    return kOk;
}

// Points the workspace members of Fp8Args into the workspace.
int fp8_workspace(Fp8Args& a, int B, int H, int N, const void* ws, size_t bytes) {
    const Fp8Layout l = fp8_layout(B, H, N);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || bytes < l.total) return kErrWorkspace;
    uint8_t* base = static_cast<uint8_t*>(const_cast<void*>(ws));
    a.q8 = base + l.q8;
    a.k8 = base + l.k8;
    a.vt8 = base + l.vt8;
    a.sq = reinterpret_cast<float*>(base + l.sq);
    a.sk = reinterpret_cast<float*>(base + l.sk);
    a.sv = reinterpret_cast<float*>(base + l.sv);
    a.vfold = reinterpret_cast<float*>(base + l.vfold);
    a.vmax = reinterpret_cast<float*>(base + l.vmax);
    a.amax = reinterpret_cast<float*>(base + l.amax);
    a.BH = B * H;
    a.N = N;
    a.n_tiles = (N + 127) / 128;
    return kOk;
}

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
    a.nlse2 = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws_half(B, H, N));
    a.work = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + 2 * ws_half(B, H, N));
    a.BH = B * H;
    a.N = N;
    a.n_kblk = (N + 127) / 128;
    a.causal = causal;
    rc = device_ready(&a.status);
    if (rc) return rc;
    // Causal head groups (see grouped_item).  dK/dV kernel: work items of a
    // group about 0.9 times the SM count, rounded down to a power of two of
    // heads (4 heads on the N = 4096 workload); dQ kernel: about twice the SM
    // count, as the forward.  Sizes from 0.5 to 4 times made no measurable
    // difference on that workload.
    a.group = clampi(floor_pow2(clampi((current_sms() * 9 / 10) / a.n_kblk, 1, 1 << 20)), 1, a.BH);
    a.group_dq = clampi(floor_pow2(clampi((2 * current_sms()) / a.n_kblk, 1, 1 << 20)), 1, a.BH);
    a.group_last = last_group(current_sms(), a.n_kblk, a.group, a.BH);
    a.group_dq_last = last_group(current_sms(), a.n_kblk, a.group_dq, a.BH);
    a.sms = current_sms();
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

// The three backward stages.  Inside fa_bwd (fused = true) prep zeroes the
// dK/dV and dQ work counters and those two kernels skip their memsets; called
// on their own, each stage zeroes its own counter.
int bwd_prep_impl(const void* o, const void* dout, const float* lse, int B, int H, int N, int d,
                  void* workspace, size_t workspace_bytes, void* stream, bool fused) {
    if (!o || !dout || !lse) return kErrInvalidArg;
    BwdArgs a{};
    int rc = bwd_common(a, B, H, N, d, 1.f, 0, workspace, workspace_bytes);
    if (rc) return rc;
    if (!aligned16(o) || !aligned16(dout) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return kErrMisaligned;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.zero_counters = fused ? 1 : 0;
    return map_cuda(launch_bwd_prep(d, a, static_cast<cudaStream_t>(stream)));
}

int bwd_main_impl(const void* q, const void* k, const void* v, const float* lse, const void* dout,
                  void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                  void* workspace, size_t workspace_bytes, void* stream, bool fused) {
    if (!q || !k || !v || !lse || !dout || !dk || !dv) return kErrInvalidArg;
    BwdArgs a{};
    CUtensorMap m[4];
    int rc = bwd_maps(a, m, q, k, v, lse, dout, B, H, N, d, scale, causal, workspace,
                      workspace_bytes);
    if (rc) return rc;
    if (!aligned16(dk) || !aligned16(dv)) return kErrMisaligned;
    a.dk = dk;
    a.dv = dv;
    a.counters_zeroed = fused ? 1 : 0;
    CUtensorMap tdk, tdv;
    if ((rc = make_map(&tdk, dk, B * H, N, d)) || (rc = make_map(&tdv, dv, B * H, N, d))) return rc;
    return map_cuda(
        launch_bwd_dkdv(d, m[0], m[1], m[2], m[3], tdk, tdv, a, static_cast<cudaStream_t>(stream)));
}

int bwd_dq_impl(const void* q, const void* k, const void* v, const float* lse, const void* dout,
                void* dq, int B, int H, int N, int d, float scale, int causal, void* workspace,
                size_t workspace_bytes, void* stream, bool fused) {
    if (!q || !k || !v || !lse || !dout || !dq) return kErrInvalidArg;
    BwdArgs a{};
    CUtensorMap m[4];
    int rc = bwd_maps(a, m, q, k, v, lse, dout, B, H, N, d, scale, causal, workspace,
                      workspace_bytes);
    if (rc) return rc;
    if (!aligned16(dq)) return kErrMisaligned;
    a.dq = dq;
    a.counters_zeroed = fused ? 1 : 0;
    CUtensorMap tdq;
    if ((rc = make_map(&tdq, dq, B * H, N, d))) return rc;
    return map_cuda(launch_bwd_dq(d, m[0], m[1], m[2], m[3], tdq, a, static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 400; }

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

size_t fa_fwd_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    return 256;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, void* stream) {
    return fa_fwd_ws(q, k, v, o, lse, B, H, N, d, scale, causal, nullptr, 0, stream);
}

int fa_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
              int d, float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    int rc = check_shape(B, H, N, d, scale, causal);
    if (rc) return rc;
    if (workspace && (((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) ||
                      workspace_bytes < fa_fwd_workspace_size(B, H, N, d)))
        return FA_ERR_WORKSPACE;
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
    // causal head groups (see grouped_item): work items of a group about twice
    // the SM count, rounded down to a power of two of heads
    // (measured: 8 heads at N = 8192, 16 at N = 4096)
    a.group = clampi(floor_pow2(clampi((2 * current_sms()) / a.n_qblk, 1, 1 << 20)), 1, BH);
    a.group_last = last_group(current_sms(), a.n_qblk, a.group, BH);
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.work = static_cast<unsigned*>(workspace);
    a.sms = current_sms();
    return map_cuda(launch_fwd(d, tq, tk, tv, to, a, static_cast<cudaStream_t>(stream)));
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    return ws_bytes(B, H, N);
}

int fa_bwd_prep(const void* o, const void* dout, const float* lse, int B, int H, int N, int d,
                void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_prep_impl(o, dout, lse, B, H, N, d, workspace, workspace_bytes, stream, false);
}

int fa_bwd_main(const void* q, const void* k, const void* v, const float* lse, const void* dout,
                void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_main_impl(q, k, v, lse, dout, dk, dv, B, H, N, d, scale, causal, workspace,
                         workspace_bytes, stream, false);
}

int fa_bwd_dq(const void* q, const void* k, const void* v, const float* lse, const void* dout,
              void* dq, int B, int H, int N, int d, float scale, int causal, void* workspace,
              size_t workspace_bytes, void* stream) {
    return bwd_dq_impl(q, k, v, lse, dout, dq, B, H, N, d, scale, causal, workspace,
                       workspace_bytes, stream, false);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
           int causal, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    int rc = check_shape(B, H, N, d, scale, causal);
    if (rc) return rc;
    // prep zeroes the two work counters, so the kernels after it need no memsets
    if ((rc = bwd_prep_impl(o, dout, lse, B, H, N, d, workspace, workspace_bytes, stream, true)))
        return rc;
    if ((rc = bwd_main_impl(q, k, v, lse, dout, dk, dv, B, H, N, d, scale, causal, workspace,
                            workspace_bytes, stream, true)))
        return rc;
    return bwd_dq_impl(q, k, v, lse, dout, dq, B, H, N, d, scale, causal, workspace, workspace_bytes,
                       stream, true);
}

size_t fa_fp8_workspace_size(int B, int H, int N, int d) {
    if (fp8_shape(B, H, N, d) != kOk) return 0;
    return fp8_layout(B, H, N).total;
}

int fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    const unsigned int* signs, int flags, void* workspace, size_t workspace_bytes,
                    void* stream) {
    if (!q || !k || !v) return FA_ERR_INVALID_ARG;
    if (flags & ~(FA_FP8_ROTATE | FA_FP8_PER_TENSOR)) return FA_ERR_INVALID_ARG;
    if ((flags & FA_FP8_ROTATE) && !signs) return FA_ERR_INVALID_ARG;
    int rc = fp8_shape(B, H, N, d);
    if (rc) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FA_ERR_MISALIGNED;
    Fp8Args a{};
    if ((rc = fp8_workspace(a, B, H, N, workspace, workspace_bytes))) return rc;
    if ((rc = device_ready(&a.status))) return rc;
    a.q = q;
    a.k = k;
    a.v = v;
    a.rotate = (flags & FA_FP8_ROTATE) ? 1 : 0;
    a.per_tensor = (flags & FA_FP8_PER_TENSOR) ? 1 : 0;
    for (int i = 0; i < 4; ++i) a.signs[i] = a.rotate ? signs[i] : 0u;
    return map_cuda(launch_fp8_quant(a, static_cast<cudaStream_t>(stream)));
}

int fa_fwd_fp8(const void* workspace, size_t workspace_bytes, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, void* stream) {
    if (!o || !lse) return FA_ERR_INVALID_ARG;
    int rc = fp8_shape(B, H, N, d);
    if (rc) return rc;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (!aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_MISALIGNED;
    Fp8Args a{};
    if ((rc = fp8_workspace(a, B, H, N, workspace, workspace_bytes))) return rc;
    if ((rc = device_ready(&a.status))) return rc;
    const int BH = B * H;
    const int npad = a.n_tiles * 128;
    CUtensorMap tq, tk, tvt, to;
    if ((rc = make_map_u8(&tq, a.q8, 128, npad, BH)) || (rc = make_map_u8(&tk, a.k8, 128, npad, BH)) ||
        (rc = make_map_u8(&tvt, a.vt8, npad, 128, BH)) || (rc = make_map(&to, o, BH, N, 128)))
        return rc;
    a.lse = lse;
    a.n_qblk = (N + 255) / 256;
    a.group = clampi(floor_pow2(clampi((2 * current_sms()) / a.n_qblk, 1, 1 << 20)), 1, BH);
    a.causal = causal;
    a.scale_log2 = scale * 1.4426950408889634f;
    return map_cuda(launch_fwd_fp8(tq, tk, tvt, to, a, static_cast<cudaStream_t>(stream)));
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
