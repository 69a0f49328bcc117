// fa_bwd.cu -- backward pass (prep, main, finish) for sm_103a.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

// ---------------------------------------------------------------------------
// prep: D_i = sum_c dO[i,c] * O[i,c] (fp32) and dQ accumulator <- 0.
// One warp per row; each lane reads 16-byte vectors of O and dO.
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const BwdArgs a) {
    const long long rows = static_cast<long long>(a.BH) * a.N;
    const int lane = threadIdx.x & 31;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    constexpr int kVec = HD / 8;  // 16-byte vectors per row (8 bf16 each)
    for (long long r = warp_global; r < rows; r += nwarps) {
        float acc = 0.f;
        const uint4* orow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.o) + r * HD);
        const uint4* drow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.dout) + r * HD);
        for (int v = lane; v < kVec; v += 32) {
            const uint4 ov = __ldg(orow + v);
            const uint4 dv = __ldg(drow + v);
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
            const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(dw[i] << 16), acc);
                acc = fmaf(__uint_as_float(ow[i] & 0xffff0000u), __uint_as_float(dw[i] & 0xffff0000u), acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) a.delta[r] = acc;
        float4* qa = reinterpret_cast<float4*>(a.dq_acc + r * HD);
        for (int v = lane; v < HD / 4; v += 32) qa[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// ---------------------------------------------------------------------------
// finish: dq = bf16(dQ accumulator); the scale is already folded in.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fa_bwd_finish_kernel(const BwdArgs a, long long n8) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const float4 x0 = reinterpret_cast<const float4*>(a.dq_acc)[2 * i];
        const float4 x1 = reinterpret_cast<const float4*>(a.dq_acc)[2 * i + 1];
        uint4 out;
        out.x = pack_bf16x2(x0.x, x0.y);
        out.y = pack_bf16x2(x0.z, x0.w);
        out.z = pack_bf16x2(x1.x, x1.y);
        out.w = pack_bf16x2(x1.z, x1.w);
        reinterpret_cast<uint4*>(a.dq)[i] = out;
    }
}

int grid_for(long long work_items, int per_block, int max_blocks) {
    long long g = (work_items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > max_blocks) g = max_blocks;
    return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_bwd_prep(int d, const BwdArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.BH) * a.N;
    const int grid = grid_for(rows, 8, 152 * 16);
    if (d == 64)
        fa_bwd_prep_kernel<64><<<grid, 256, 0, stream>>>(a);
    else
        fa_bwd_prep_kernel<128><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_finish(int d, const BwdArgs& a, cudaStream_t stream) {
    const long long n8 = static_cast<long long>(a.BH) * a.N * d / 8;
    const int grid = grid_for(n8, 256, 152 * 16);
    fa_bwd_finish_kernel<<<grid, 256, 0, stream>>>(a, n8);
    return cudaGetLastError();
}

cudaError_t launch_bwd_main(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& a,
                            cudaStream_t stream) {
    (void)d; (void)tq; (void)tk; (void)tv; (void)tdo; (void)a; (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace fa
