// fa_internal.cuh -- parameters and launch entry points shared between the
// host API (fa_api.cu) and the kernel translation units.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Status codes (mirror fa_status in include/fa.h).
enum : int {
    kOk = 0,
    kErrInvalidArg = 1,
    kErrUnsupported = 2,
    kErrMisaligned = 3,
    kErrWorkspace = 4,
    kErrCuda = 5,
    kErrDeviceTimeout = 6,
};

// A kernel that waits longer than this on one barrier gives up.  A test build
// may shorten it.
#ifndef FA_WAIT_TIMEOUT_NS
#define FA_WAIT_TIMEOUT_NS 2000000000ull
#endif
constexpr uint64_t kWaitTimeoutNs = FA_WAIT_TIMEOUT_NS;

// Test builds only (never set by the library build): with FA_FAULT_INJECT=1 the
// load warps never issue their K/V (forward, dQ kernel) or Q/dO (dK/dV kernel) copies, so a
// bounded wait runs out and the kernel must report FA_ERR_DEVICE_TIMEOUT and
// leave cleanly.  No fault, trap or endless wait is involved.
#ifndef FA_FAULT_INJECT
#define FA_FAULT_INJECT 0
#endif

struct FwdArgs {
    void* o;          // bf16 [BH, N, d]
    float* lse;       // fp32 [BH, N]
    int BH;
    int N;
    int n_qblk;       // query blocks (256 rows each) per head
    int group;        // causal item order: heads per group (heavy blocks first within a group)
    int group_last;   // heads in the last group (at least `group`)
    int causal;
    float scale_log2; // scale * log2(e)
    int* status;      // device status word
    unsigned* work;   // work-item counter (zeroed before the launch), or null: a static
                      // schedule (a table in the launch parameters, else round robin)
    int sms;          // multiprocessors of the device (grid of the persistent launch)
};

// Static schedule of the persistent forward when no work counter is given: CTA
// c runs the items items[start[c]] .. items[start[c + 1] - 1] in that order.
// It travels in the launch parameters, so concurrent launches share nothing.
// The host fills it by greedy longest-first list scheduling over the item costs
// in the counter's fetch order, i.e. what the counter does with modelled item
// times.  Cap = 1 is the table-free launch (round robin: item k * grid + c).
constexpr int kFwdSchedMaxCtas = 256;
template <int Cap>
struct FwdSched {
    uint16_t start[kFwdSchedMaxCtas + 1];
    uint16_t items[Cap];
};

// Causal work order of the persistent kernels: heads in groups of `group`
// (a few heads' K/V or Q/dO stay in L2), the last group of `group_last` heads;
// inside a group the heaviest block of every head first, then the next, and so
// on.  The last group is larger so that its work, spread over all SMs, outlasts
// its heaviest items, which then finish with the rest instead of after it.
// Item t -> head bh and block rank (0 = heaviest).
__host__ __device__ __forceinline__ void grouped_item(int t, int nblk, int BH, int group,
                                                      int group_last, int& bh, int& rank) {
    const int n_reg = BH - group_last;  // heads in the regular groups
    const int t_reg = n_reg * nblk;
    int first, gc, r;
    if (t < t_reg) {
        const int grp = t / (group * nblk);
        first = grp * group;
        gc = group < n_reg - first ? group : n_reg - first;
        r = t - grp * group * nblk;
    } else {
        first = n_reg;
        gc = group_last;
        r = t - t_reg;
    }
    rank = r / gc;
    bh = first + r % gc;
}

// Counters of the persistent backward kernels inside BwdArgs::work, 128 bytes apart.
constexpr int kWorkDkdv = 0;
constexpr int kWorkDq = 32;

struct BwdArgs {
    const void* q;    // bf16 [BH, N, d] (plain pointers for the row-wise stages)
    const void* k;
    const void* v;
    const void* o;
    const void* dout;
    const float* lse; // fp32 [BH, N]
    void* dq;
    void* dk;
    void* dv;
    // workspace, fp32 [BH, n_kblk * 128] (rows padded to whole 128-row tiles):
    float* delta;     // D = rowsum(dO * O); 0 in the padding
    float* nlse2;     // -lse * log2(e); -inf in the padding (P = 0 there)
    unsigned* work;   // 256-byte slot of work-item counters: [kWorkDkdv], [kWorkDq] (each
                      // zeroed before its kernel's launch)
    int sms;          // multiprocessors of the device (grid of the persistent kernels)
    int BH;
    int N;
    int n_kblk;       // 128-row key blocks per head (= 128-row query blocks)
    int group;        // causal item order of the dK/dV kernel: heads per group
    int group_last;   //   heads in its last group (at least `group`)
    int group_dq;     // causal item order of the dQ kernel: heads per group
    int group_dq_last;//   heads in its last group
    int causal;
    float scale;
    float scale_log2;
    int* status;
    int zero_counters;   // prep: zero both work counters (inside fa_bwd)
    int counters_zeroed; // dK/dV and dQ kernels: the prep before them zeroed the counters
};

// FP8 forward (d = 128).  The quantizer reads q, k, v and fills the FP8
// workspace; the attention kernel reads the workspace and writes o and lse.
// Rows are padded to npad = n_tiles * 128 (padding rows hold code 0).
struct Fp8Args {
    const void* q;    // bf16 [BH, N, 128]
    const void* k;
    const void* v;
    uint8_t* q8;      // E4M3 [BH, npad, 128], rows rotated when `rotate`
    uint8_t* k8;      // E4M3 [BH, npad, 128]
    uint8_t* vt8;     // E4M3 [BH, 128, npad]: V^T, keys permuted within each tile
    float* sq;        // fp32 [BH, n_tiles]: per-tile scales (value = code * scale)
    float* sk;
    float* sv;
    float* vfold;     // fp32 [BH, n_tiles]: sv / vmax
    float* vmax;      // fp32 [BH]
    float* amax;      // fp32 [3]: per-tensor |x| maxima (per-tensor mode only)
    float* lse;       // fp32 [BH, N]
    uint32_t signs[4];  // bit j set: column j of Q and K is negated before the Hadamard transform
    int BH;
    int N;
    int n_tiles;      // ceil(N / 128)
    int n_qblk;       // query blocks (256 rows each) per head
    int group;        // causal launch order: heads per group
    int causal;
    int rotate;       // 1: random-sign Hadamard rotation of Q and K rows
    int per_tensor;   // 1: one scale per tensor instead of one per tile
    float scale_log2; // scale * log2(e)
    int* status;
};

// Tensor maps for one [BH, N, d] bf16 tensor: box of 64 columns x 128 rows,
// 128-byte swizzle (what the UMMA shared-memory descriptors expect).
struct TensorMaps3 {
    CUtensorMap a, b, c;
};

// Shape and scalar checks shared by the forward and backward entry points:
// B, H, N >= 1, causal 0 or 1, scale finite and > 0 (kErrInvalidArg); d 64 or
// 128 (kErrUnsupported); B*H*N*d < 2^31 (kErrInvalidArg).  Defined in fa_api.cu.
int check_shape(int B, int H, int N, int d, float scale, int causal);

// Raises a kernel's dynamic shared-memory limit (cudaFuncSetAttribute) the
// first time it is launched on a device, not before every launch.  Kernel: the
// __global__ function (one counter per kernel instance and device).
template <auto Kernel>
cudaError_t smem_limit_once(int bytes) {
    static std::atomic<int> set_on[64];  // per device: the limit already set, 0 = none
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && set_on[dev].load(std::memory_order_acquire) >= bytes)
        return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) set_on[dev].store(bytes, std::memory_order_release);
    return e;
}

// Launchers (defined in the kernel translation units).  Return a cudaError_t.
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& args, cudaStream_t stream);
cudaError_t launch_fp8_quant(const Fp8Args& args, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const CUtensorMap& to, const Fp8Args& args, cudaStream_t stream);
cudaError_t launch_bwd_prep(int d, const BwdArgs& args, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const BwdArgs& args, cudaStream_t stream);
cudaError_t launch_bwd_dq(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const BwdArgs& args, cudaStream_t stream);

}  // namespace fa
