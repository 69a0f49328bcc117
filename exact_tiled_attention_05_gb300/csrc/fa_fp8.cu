// fa_fp8.cu -- FP8 (E4M3) attention forward for sm_103a: block quantization
// with incoherent processing, then the fused forward on FP8 tensor cores.
//
// "FlashAttention 1–4" §"FlashAttention-3", FP8 with block quantization and
// incoherent processing: one FP8 scale per tile instead of one per tensor, and
// Q and K multiplied by the same random orthogonal matrix M = diag(s) H / sqrt(d)
// (random signs, then a Hadamard transform) before quantizing, which leaves
// Q K^T unchanged while spreading outlier channels over all coordinates.
//
// Stage 1, fa_fp8_quant_kernel (one CTA per (tensor, head, 128-row tile)):
//   Q, K: rows rotated in fp32 (sign flips, seven butterfly stages, * 1/sqrt(d)),
//   V: not rotated; scale = amax / 448 over the tile (or over the whole tensor
//   for the per-tensor baseline the page compares against), codes =
//   e4m3(x / scale).  Q and K codes keep the
//   [BH, N, d] layout; V is written transposed, [BH, d, N], with the keys of
//   each 128-key tile in the order the forward kernel packs P (below).
// Stage 2, fa_fp8_vfold_kernel: per head, vmax = max over tiles of V's scale
//   and fold_t = scale_t / vmax.
// Stage 3, fa_fwd_fp8_kernel: the bf16 forward's structure (two 128-row Q tiles
//   per CTA, four softmax threads per row in one warp, P handed over in two
//   parts, conditional rescaling) with tcgen05.mma kind::f8f6f4: S = Q8 K8^T
//   (four k-steps of 32), s = S * scale_q * scale_k, P = exp2(.) in fp32 for the
//   row sums, P * fold_j * 16 quantized to E4M3 in TMEM, O += P8 V8^T; at the
//   end O * vmax / (16 l).  lse as the bf16 forward.
//
// P's range.  The running max is raised only when a tile's max exceeds it by
// more than tau = 4 (log2 units), so P <= 2^tau; the factor 2^(8 - tau) = 16
// puts the largest P * fold at or below 256 (E4M3 saturates at 448) while
// keeping weights down to 2^-10 of the row max in E4M3's normal range.
//
// P packing.  A TMEM column of an 8-bit A operand holds four consecutive
// K-indices.  A softmax thread holds keys 8i + 2c + {0, 1} (c = lane % 4) of
// its two rows, so it packs keys {8w + 2c, +1} of repetition w and
// {8(w+4) + 2c, +1} of repetition w + 4 into one word, stored at column
// 16h + 4w + c of part h (keys 64h..64h+63).  The K-index order of P is thus a
// fixed permutation of the tile's keys; V^T is written in the same order, and
// sum_k P[., k] V[k, .] does not depend on the order.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kHD = 128;                   // head dimension of the FP8 path
constexpr int kBM = 128, kBN = 128;
constexpr int kTile8 = 128 * 128;          // bytes of a 128 x 128 FP8 tile (one 128-byte box)
constexpr int kOBox = 128 * 64 * 2;        // one bf16 box of O: 128 rows x 64 columns
constexpr int kThreads = 576;              // TMA, MMA + TMEM, 2 tiles x 8 softmax warps
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kSoftmaxPerTile = 256;
constexpr int kStages = 6;                 // K_j, V_j^T ring
constexpr float kRescaleThreshold = 4.0f;  // tau, log2 units
constexpr float kPScale = 16.0f;           // 2^(8 - tau)
constexpr float kE4M3Max = 448.0f;
constexpr uint32_t kSColStride = 128;      // S_t / P_t at TMEM column 128 t
constexpr uint32_t kOCol0 = 256;           // O_t at 256 + 128 t
constexpr uint32_t kTmemCols = 512;

// ---------------------------------------------------------------------------
// FP8 helpers
// ---------------------------------------------------------------------------

// Two floats -> E4M3 pair (round to nearest even, saturating at +-448), `lo` in
// bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// x rounded to E4M3 (as the packing above rounds it) and back to fp32.
__device__ __forceinline__ float e4m3_round(float x) {
    const uint16_t c = static_cast<uint16_t>(e4m3x2(x, 0.f));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    const uint16_t h = static_cast<uint16_t>(h2 & 0xffffu);
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}

// D[tmem] (+)= A[smem] * B[smem]^T, both E4M3.
__device__ __forceinline__ void umma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, both E4M3.
__device__ __forceinline__ void umma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0 at
// bits 7 and 10), fp32 D, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Key order of P's K-indices within a 128-key tile (see the file comment):
// K-index 4c + e, c = 16h + 4w + q, holds key 64h + 32(e >> 1) + 8w + 2q + (e & 1).
__host__ __device__ __forceinline__ int p_key_of_index(int kidx) {
    const int c = kidx >> 2, e = kidx & 3;
    const int h = c >> 4, w = (c >> 2) & 3, q = c & 3;
    return 64 * h + 32 * (e >> 1) + 8 * w + 2 * q + (e & 1);
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32"
        " [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 16x128b, four repetitions: registers 2r, 2r + 1 go to column 4r + lane % 4 of
// rows lane/4 and lane/4 + 8.
__device__ __forceinline__ void tmem_st_16x128b_x4(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// ---------------------------------------------------------------------------
// Stage 1: rotation and block quantization
// ---------------------------------------------------------------------------
// grid (tiles, BH, 3 tensors), 256 threads; warp w takes rows w, w + 8, ..;
// lane l holds columns 4l..4l+3 of a row.  MODE 0 only reduces |x| of the tile
// into amax[tensor] (per-tensor baseline, first pass); MODE 1 quantizes.
template <int MODE>
__global__ void __launch_bounds__(256) fa_fp8_quant_kernel(const __grid_constant__ Fp8Args a) {
    extern __shared__ float tl[];  // [128][129] fp32 tile (row stride 129 against bank conflicts)
    __shared__ float red[8];
    const int tile = static_cast<int>(blockIdx.x);
    const int bh = static_cast<int>(blockIdx.y);
    const int which = static_cast<int>(blockIdx.z);  // 0 Q, 1 K, 2 V
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = a.N, npad = a.n_tiles * 128;
    const bool rot = a.rotate != 0 && which < 2;
    const uint16_t* src = static_cast<const uint16_t*>(which == 0 ? a.q : which == 1 ? a.k : a.v) +
                          static_cast<size_t>(bh) * N * kHD;
    float sgn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int col = 4 * lane + e;
        sgn[e] = ((a.signs[col >> 5] >> (col & 31)) & 1u) ? -1.f : 1.f;
    }
    float amax = 0.f;
    for (int r = warp; r < 128; r += 8) {
        const int row = tile * 128 + r;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (row < N) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(src + static_cast<size_t>(row) * kHD) + lane);
            x[0] = __uint_as_float(w.x << 16);
            x[1] = __uint_as_float(w.x & 0xffff0000u);
            x[2] = __uint_as_float(w.y << 16);
            x[3] = __uint_as_float(w.y & 0xffff0000u);
        }
        if (rot && row < N) {  // (rows past N stay +0; row is the same for the whole warp)
            // sign flips, then y_i = sum_j (-1)^popcount(i & j) x_j by butterflies
            // h = 1, 2 (inside the lane), 4 .. 64 (across lanes), then * 1/sqrt(d)
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] *= sgn[e];
            float t0 = x[0] + x[1], t1 = x[0] - x[1], t2 = x[2] + x[3], t3 = x[2] - x[3];
            x[0] = t0 + t2;
            x[2] = t0 - t2;
            x[1] = t1 + t3;
            x[3] = t1 - t3;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p = __shfl_xor_sync(0xffffffffu, x[e], m);
                    x[e] = (lane & m) ? (p - x[e]) : (x[e] + p);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] *= 0.08838834764831845f;  // 1 / sqrt(128)
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            tl[r * 129 + 4 * lane + e] = x[e];
            amax = fmaxf(amax, fabsf(x[e]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = red[0];
        for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
        red[0] = m;
    }
    __syncthreads();
    const float amax_tile = red[0];
    if (MODE == 0) {
        if (threadIdx.x == 0)
            atomicMax(reinterpret_cast<unsigned int*>(a.amax + which),
                      __float_as_uint(amax_tile));  // non-negative floats order as their bits
        return;
    }
    const float amax_used = a.per_tensor ? a.amax[which] : amax_tile;
    const float scale = amax_used > 0.f ? amax_used / kE4M3Max : 1.f;
    if (threadIdx.x == 0) {
        float* scales = which == 0 ? a.sq : which == 1 ? a.sk : a.sv;
        scales[bh * a.n_tiles + tile] = scale;
    }
    if (which < 2) {
        uint8_t* dst = (which == 0 ? a.q8 : a.k8) + (static_cast<size_t>(bh) * npad + tile * 128) * kHD;
        for (int r = warp; r < 128; r += 8) {
            const float* x = tl + r * 129 + 4 * lane;
            const uint32_t w = e4m3x2(x[0] / scale, x[1] / scale) | (e4m3x2(x[2] / scale, x[3] / scale) << 16);
            reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(r) * kHD)[lane] = w;
        }
    } else {
        // V^T: row = head column, 128 bytes per tile in P's key order
        uint8_t* dst = a.vt8 + static_cast<size_t>(bh) * kHD * npad + tile * 128;
        for (int col = warp; col < kHD; col += 8) {
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = tl[p_key_of_index(4 * lane + e) * 129 + col];
            const uint32_t w = e4m3x2(x[0] / scale, x[1] / scale) | (e4m3x2(x[2] / scale, x[3] / scale) << 16);
            reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(col) * npad)[lane] = w;
        }
    }
}

// Stage 2: per head, vmax = max_t scale_v[t] and fold[t] = scale_v[t] / vmax.
__global__ void __launch_bounds__(32) fa_fp8_vfold_kernel(const __grid_constant__ Fp8Args a) {
    const int bh = static_cast<int>(blockIdx.x);
    const float* sv = a.sv + static_cast<size_t>(bh) * a.n_tiles;
    float m = 0.f;
    for (int t = threadIdx.x; t < a.n_tiles; t += 32) m = fmaxf(m, sv[t]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (threadIdx.x == 0) a.vmax[bh] = m;
    for (int t = threadIdx.x; t < a.n_tiles; t += 32) a.vfold[static_cast<size_t>(bh) * a.n_tiles + t] = sv[t] / m;
}

// ---------------------------------------------------------------------------
// Stage 3: the FP8 forward
// ---------------------------------------------------------------------------
struct alignas(1024) Fp8Smem {
    uint8_t q[2][kTile8];
    uint8_t kv[kStages][kTile8];
    uint8_t o[2][2 * kOBox];  // bf16 O of each tile, two 64-column boxes
    uint64_t q_full;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2][2];
    uint64_t o_done[2];
    uint64_t out_staged[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Fp8Smem) + 1024 <= 232448, "FP8 forward shared memory exceeds 227 KB");

__device__ __forceinline__ void fp8_timeout(const Fp8Args& a, volatile int* abort) {
    *abort = 1;
    atomicExch(a.status, kErrDeviceTimeout);
}

__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tvt, const __grid_constant__ CUtensorMap to,
                  const Fp8Args a) {
    extern __shared__ uint8_t fp8_smem_raw[];
    Fp8Smem& sm = *reinterpret_cast<Fp8Smem*>(
        (reinterpret_cast<uintptr_t>(fp8_smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int* abort = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = a.N;
    const int BH = a.BH;

    // (head, 256-row query block); causal: head groups, heaviest blocks first
    int bh, qb;
    if (a.causal) {
        const int b = static_cast<int>(blockIdx.x);
        const int grp = b / (a.group * a.n_qblk);
        const int first = grp * a.group;
        const int gc = min(a.group, BH - first);
        const int r = b - grp * a.group * a.n_qblk;
        qb = a.n_qblk - 1 - r / gc;
        bh = first + r % gc;
    } else {
        bh = static_cast<int>(blockIdx.x) / a.n_qblk;
        qb = static_cast<int>(blockIdx.x) % a.n_qblk;
    }
    const int n_kv_all = (N + kBN - 1) / kBN;
    int q0[2], nkv[2];
    for (int t = 0; t < 2; ++t) {
        q0[t] = qb * 2 * kBM + t * kBM;
        if (q0[t] >= N)
            nkv[t] = 0;
        else if (a.causal)
            nkv[t] = (min(q0[t] + kBM, N) - 1) / kBN + 1;
        else
            nkv[t] = n_kv_all;
    }
    const int nmax = max(nkv[0], nkv[1]);

    if (threadIdx.x == 0) {
        sm.abort = 0;
        mbar_init(smem_u32(&sm.q_full), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sm.kv_full[s]), 1);
            mbar_init(smem_u32(&sm.kv_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&sm.s_full[t]), 1);
            mbar_init(smem_u32(&sm.p_full[t][0]), kSoftmaxPerTile);
            mbar_init(smem_u32(&sm.p_full[t][1]), kSoftmaxPerTile);
            mbar_init(smem_u32(&sm.o_done[t]), 1);
            mbar_init(smem_u32(&sm.out_staged[t]), kSoftmaxPerTile);
        }
        mbar_init(smem_u32(&sm.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;

    if (warp == 0) {
        // ===================== TMA producer =====================
        if (elect_one()) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tvt);
            const uint32_t qbar = smem_u32(&sm.q_full);
            const int nact = (nkv[0] > 0) + (nkv[1] > 0);
            mbar_arrive_expect_tx(qbar, nact * kTile8);
            for (int t = 0; t < 2; ++t)
                if (nkv[t] > 0) tma_load_3d(smem_u32(sm.q[t]), &tq, qbar, 0, q0[t], bh);
            int issued = 0;
            bool ok = true;
            const int n_loads = FA_FAULT_INJECT ? 0 : 2 * nmax;
            for (int idx = 0; idx < n_loads; ++idx) {
                const int slot = idx % kStages;
                if (!mbar_wait(smem_u32(&sm.kv_empty[slot]), ((idx / kStages) & 1) ^ 1, kWaitTimeoutNs,
                               abort)) {
                    fp8_timeout(a, abort);
                    ok = false;
                    break;
                }
                const uint32_t fbar = smem_u32(&sm.kv_full[slot]);
                mbar_arrive_expect_tx(fbar, kTile8);
                if (idx & 1)  // V_j^T: 128 head rows x 128 keys
                    tma_load_3d(smem_u32(sm.kv[slot]), &tvt, fbar, (idx >> 1) * kBN, 0, bh);
                else
                    tma_load_3d(smem_u32(sm.kv[slot]), &tk, fbar, 0, (idx >> 1) * kBN, bh);
                ++issued;
            }
            for (int slot = 0; slot < kStages && slot < issued; ++slot) {
                const int last = slot + kStages * ((issued - 1 - slot) / kStages);
                mbar_wait_drain(smem_u32(&sm.kv_full[slot]), (last / kStages) & 1, kWaitTimeoutNs);
            }
            mbar_wait_drain(qbar, 0, kWaitTimeoutNs);
            tma_prefetch_desc(&to);
            for (int t = 0; ok && t < 2; ++t) {
                if (nkv[t] == 0) continue;
                if (!(ok = mbar_wait(smem_u32(&sm.out_staged[t]), 0, kWaitTimeoutNs, abort))) {
                    fp8_timeout(a, abort);
                    break;
                }
                for (int b = 0; b < 2; ++b)
                    tma_store_3d(&to, smem_u32(sm.o[t]) + b * kOBox, b * 64, q0[t], bh);
            }
            bulk_commit_group();
            bulk_wait_group0();
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (elect_one()) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);  // S and O: N = 128 = d
            const uint32_t q_addr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
            bool ok = mbar_wait(smem_u32(&sm.q_full), 0, kWaitTimeoutNs, abort);
            auto wait_kv = [&](int idx) -> bool {
                return mbar_wait(smem_u32(&sm.kv_full[idx % kStages]), (idx / kStages) & 1,
                                 kWaitTimeoutNs, abort);
            };
            auto kv_addr = [&](int idx) -> uint32_t { return smem_u32(sm.kv[idx % kStages]); };
            // S_t = Q8_t K8^T: four k-steps of 32 bytes, both K-major
            auto issue_s = [&](int t, uint32_t k_addr) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_ss_f8(tbase + static_cast<uint32_t>(t) * kSColStride,
                               sdesc_sw128(q_addr[t] + kk * 32, 16, 1024),
                               sdesc_sw128(k_addr + kk * 32, 16, 1024), idesc, kk > 0);
            };
            // O_t += P8_t V8: part q of P (TMEM columns 16q..16q+15 of S_t) is
            // k-steps 2q, 2q + 1; V^T K-major (keys in P's order)
            auto issue_pv = [&](int t, uint32_t vt_addr, int part, bool acc) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int kk = part * 2 + i;
                    umma_ts_f8(tbase + kOCol0 + t * kHD, tbase + static_cast<uint32_t>(t) * kSColStride + kk * 8,
                               sdesc_sw128(vt_addr + kk * 32, 16, 1024), idesc,
                               (acc || part > 0 || i > 0) ? 1u : 0u);
                }
            };
            if (ok && nmax > 0 && (ok = wait_kv(0))) {
                tc_fence_after();
                for (int t = 0; t < 2; ++t) {
                    if (nkv[t] == 0) continue;
                    issue_s(t, kv_addr(0));
                    umma_commit(smem_u32(&sm.s_full[t]));
                }
                umma_commit(smem_u32(&sm.kv_empty[0]));
            }
            for (int j = 0; ok && j < nmax; ++j) {
                const int iv = 2 * j + 1, ik = 2 * j + 2;
                if (!(ok = wait_kv(iv))) break;
                tc_fence_after();
                bool k_ready = false;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j < nkv[t]) {
                        for (int part = 0; part < 2 && ok; ++part) {
                            if (!(ok = mbar_wait(smem_u32(&sm.p_full[t][part]), j & 1, kWaitTimeoutNs, abort)))
                                break;
                            tc_fence_after();
                            issue_pv(t, kv_addr(iv), part, j > 0);
                        }
                        if (!ok) break;
                        umma_commit(smem_u32(&sm.o_done[t]));
                    }
                    if (t == 1) umma_commit(smem_u32(&sm.kv_empty[iv % kStages]));
                    if (j + 1 < nkv[t]) {
                        if (!k_ready) {
                            if (!(ok = wait_kv(ik))) break;
                            tc_fence_after();
                            k_ready = true;
                        }
                        // S_t(j+1) overwrites P_t(j) after PV_t(j) was issued (in order)
                        issue_s(t, kv_addr(ik));
                        umma_commit(smem_u32(&sm.s_full[t]));
                    }
                }
                if (ok && k_ready) umma_commit(smem_u32(&sm.kv_empty[ik % kStages]));
            }
            if (!ok) fp8_timeout(a, abort);
            umma_commit(smem_u32(&sm.drain));
            mbar_wait_drain(smem_u32(&sm.drain), 0, kWaitTimeoutNs);
        }
    } else {
        // ===================== softmax / epilogue =====================
        // As the bf16 forward: warp (wq, sub) reads S_t with the 16x256b shape,
        // lane L holds rows rA = 32 wq + 16 sub + L/4 and rB = rA + 8, key columns
        // 8i + 2(L%4) + {0, 1}.
        const int sw = warp - kFirstSoftmaxWarp;
        const int t = sw >> 3;
        const int sub = (sw >> 2) & 1;
        const int wq = warp & 3;
        const int cq = lane & 3;
        const int rA = wq * 32 + sub * 16 + (lane >> 2);
        const int my_q0 = t == 0 ? q0[0] : q0[1];
        const int my_nkv = t == 0 ? nkv[0] : nkv[1];
        const int qA = my_q0 + rA, qB = qA + 8;
        const uint32_t lanes16 = tbase + (static_cast<uint32_t>(wq * 32 + sub * 16) << 16);
        const uint32_t s_addr = lanes16 + static_cast<uint32_t>(t) * kSColStride;
        const uint32_t o_addr = lanes16 + kOCol0 + t * kHD;
        const float* skr = a.sk + static_cast<size_t>(bh) * a.n_tiles;
        const float* fold = a.vfold + static_cast<size_t>(bh) * a.n_tiles;
        // scores in log2 units: raw S (code units) * scale * log2e * scale_q * scale_k
        const float sl2q = a.scale_log2 * (my_nkv > 0 ? a.sq[static_cast<size_t>(bh) * a.n_tiles + my_q0 / kBM] : 0.f);
        float mA = -INFINITY, mB = -INFINITY;
        uint64_t lA = f2_pack(0.f, 0.f), lB = f2_pack(0.f, 0.f);
        float lcA = 0.f, lcB = 0.f;  // rounding correction of the largest weight, as the bf16 forward
        bool ok = true;
        for (int j = 0; j < my_nkv; ++j) {
            const float sl2 = sl2q * __ldg(skr + j);
            const float fj = __ldg(fold + j) * kPScale;  // exact: a power of two
            const uint64_t sl2_pair = f2_pack(sl2, sl2);
            const uint64_t f_pair = f2_pack(fj, fj);
            ok = mbar_wait_warp(smem_u32(&sm.s_full[t]), j & 1, kWaitTimeoutNs, abort);
            if (!ok) break;
            tc_fence_after();
            uint32_t sa[32], sb[32];  // keys 0-63 and 64-127 of the tile
            tmem_ld_16x256b_x8(s_addr, sa);
            tmem_ld_16x256b_x8(s_addr + 64, sb);
            tmem_wait_ld();
            reg_fence(sa);
            reg_fence(sb);
#define SR(c) ((c) < 32 ? sa[(c)] : sb[(c) - 32])
            const int kbase = j * kBN + 2 * cq;
            if ((j * kBN + kBN > N) || (a.causal && j * kBN + kBN - 1 > my_q0)) {
                const int kendA = a.causal ? min(N, qA + 1) : N;
                const int kendB = a.causal ? min(N, qB + 1) : N;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int ka = kbase + 8 * i + c, kb = ka + 64;
                        if (ka >= kendA) sa[4 * i + c] = __float_as_uint(-INFINITY);
                        if (ka >= kendB) sa[4 * i + 2 + c] = __float_as_uint(-INFINITY);
                        if (kb >= kendA) sb[4 * i + c] = __float_as_uint(-INFINITY);
                        if (kb >= kendB) sb[4 * i + 2 + c] = __float_as_uint(-INFINITY);
                    }
                }
            }
            float ma[2], mb[2];
            ma[0] = __uint_as_float(sa[0]);
            ma[1] = __uint_as_float(sa[1]);
            mb[0] = __uint_as_float(sa[2]);
            mb[1] = __uint_as_float(sa[3]);
#pragma unroll
            for (int i = 1; i < 15; i += 2) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    ma[c] = fmax3(ma[c], __uint_as_float(SR(4 * i + c)), __uint_as_float(SR(4 * i + 4 + c)));
                    mb[c] = fmax3(mb[c], __uint_as_float(SR(4 * i + 2 + c)), __uint_as_float(SR(4 * i + 6 + c)));
                }
            }
            float pmA = fmax3(ma[0], ma[1], fmaxf(__uint_as_float(sb[28]), __uint_as_float(sb[29])));
            float pmB = fmax3(mb[0], mb[1], fmaxf(__uint_as_float(sb[30]), __uint_as_float(sb[31])));
            pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 1));
            pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 1));
            pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 2));
            pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 2));
            bool rescale = false;
            float alphaA = 1.f, alphaB = 1.f;
            {
                const float mxA = pmA * sl2, mxB = pmB * sl2;
                if (mA == -INFINITY) {
                    mA = mxA;
                } else if (mxA > mA + kRescaleThreshold) {
                    rescale = true;
                    alphaA = ex2(mA - mxA);
                    lA = f2_mul(lA, f2_pack(alphaA, alphaA));
                    lcA *= alphaA;
                    mA = mxA;
                }
                if (mB == -INFINITY) {
                    mB = mxB;
                } else if (mxB > mB + kRescaleThreshold) {
                    rescale = true;
                    alphaB = ex2(mB - mxB);
                    lB = f2_mul(lB, f2_pack(alphaB, alphaB));
                    lcB *= alphaB;
                    mB = mxB;
                }
            }
            const float negA = (mA == -INFINITY) ? 0.f : -mA;
            const float negB = (mB == -INFINITY) ? 0.f : -mB;
            const uint64_t negA2 = f2_pack(negA, negA), negB2 = f2_pack(negB, negB);
            const bool any_rescale = __any_sync(0xffffffffu, rescale);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                // word w of each row packs repetitions w and w + 4 of this part:
                // keys {8w + 2cq, +1} and {8(w + 4) + 2cq, +1}
                uint32_t pk[8];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        uint32_t pair[2];
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const int e = hh * 32 + 4 * (w + 4 * r) + 2 * x;
                            const uint64_t x2 = f2_fma(f2_pack_u(SR(e), SR(e + 1)), sl2_pair, x == 0 ? negA2 : negB2);
                            const float2 xv = f2_unpack(x2);
                            const uint64_t p2 = f2_pack(ex2(xv.x), ex2(xv.y));
                            if (x == 0)
                                lA = f2_add(lA, p2);
                            else
                                lB = f2_add(lB, p2);
                            const float2 pf = f2_unpack(f2_mul(p2, f_pair));
                            pair[r] = e4m3x2(pf.x, pf.y);
                        }
                        pk[2 * w + x] = pair[0] | (pair[1] << 16);
                    }
                }
                tmem_st_16x128b_x4(s_addr + hh * 16, pk);
                if (hh == 0 && any_rescale) {
                    ok = mbar_wait_warp(smem_u32(&sm.o_done[t]), (j - 1) & 1, kWaitTimeoutNs, abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t aA = f2_pack(alphaA, alphaA), aB = f2_pack(alphaB, alphaB);
#pragma unroll
                    for (int c = 0; c < kHD / 32; ++c) {
                        uint32_t r[16];
                        tmem_ld_16x256b_x4(o_addr + c * 32, r);
                        tmem_wait_ld();
                        reg_fence(r);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float2 v = f2_unpack(f2_mul(f2_pack_u(r[2 * i], r[2 * i + 1]), (i & 1) ? aB : aA));
                            r[2 * i] = __float_as_uint(v.x);
                            r[2 * i + 1] = __float_as_uint(v.y);
                        }
                        tmem_st_16x256b_x4(o_addr + c * 32, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&sm.p_full[t][hh]));
            }
#undef SR
            if (!ok) break;
            {
                // the row's largest weight as P V used it: fold and scale, E4M3, back
                const float pxA = ex2(fmaf(pmA, sl2, negA)), pxB = ex2(fmaf(pmB, sl2, negB));
                lcA += e4m3_round(pxA * fj) / fj - pxA;
                lcB += e4m3_round(pxB * fj) / fj - pxB;
            }
        }
        if (!ok) {
            if (lane == 0) fp8_timeout(a, abort);
        } else if (my_nkv > 0) {
            const float2 la = f2_unpack(lA), lb = f2_unpack(lB);
            float sA = la.x + la.y, sB = lb.x + lb.y;
            sA += __shfl_xor_sync(0xffffffffu, sA, 1);
            sB += __shfl_xor_sync(0xffffffffu, sB, 1);
            sA += __shfl_xor_sync(0xffffffffu, sA, 2);
            sB += __shfl_xor_sync(0xffffffffu, sB, 2);
            ok = mbar_wait_warp(smem_u32(&sm.o_done[t]), (my_nkv - 1) & 1, kWaitTimeoutNs, abort);
            if (ok) {
                tc_fence_after();
                const float vmax = a.vmax[bh] * (1.0f / kPScale);
                const float invA = vmax / (sA + lcA), invB = vmax / (sB + lcB);
                // O rows into the tile's staging buffer: 64-column boxes of 128-byte
                // rows, column 8i + 2cq is chunk i % 8 of box i / 8 at (i % 8) ^ (row % 8)
                const uint32_t obuf = smem_u32(sm.o[t]);
#pragma unroll
                for (int c = 0; c < kHD / 32; ++c) {
                    uint32_t r[16];
                    tmem_ld_16x256b_x4(o_addr + c * 32, r);
                    tmem_wait_ld();
                    reg_fence(r);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t wa = pack_bf16x2(__uint_as_float(r[4 * i]) * invA, __uint_as_float(r[4 * i + 1]) * invA);
                        const uint32_t wb = pack_bf16x2(__uint_as_float(r[4 * i + 2]) * invB, __uint_as_float(r[4 * i + 3]) * invB);
                        const int ii = c * 4 + i;
                        const uint32_t off = static_cast<uint32_t>((ii / 8) * kOBox + (((ii % 8) ^ (rA & 7)) << 4) + 4 * cq);
                        st_shared_b32(obuf + off + static_cast<uint32_t>(rA * 128), wa);
                        st_shared_b32(obuf + off + static_cast<uint32_t>((rA + 8) * 128), wb);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&sm.out_staged[t]));
                if (cq == 0) {
                    if (qA < N) a.lse[static_cast<size_t>(bh) * N + qA] = (mA + __log2f(sA)) * 0.69314718055994531f;
                    if (qB < N) a.lse[static_cast<size_t>(bh) * N + qB] = (mB + __log2f(sB)) * 0.69314718055994531f;
                }
            } else if (lane == 0) {
                fp8_timeout(a, abort);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_fp8_quant(const Fp8Args& a, cudaStream_t stream) {
    const size_t smem = 128 * 129 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(fa_fp8_quant_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fa_fp8_quant_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(a.n_tiles), static_cast<unsigned>(a.BH), 3);
    if (a.per_tensor) {
        if ((e = cudaMemsetAsync(a.amax, 0, 3 * sizeof(float), stream)) != cudaSuccess) return e;
        fa_fp8_quant_kernel<0><<<grid, 256, smem, stream>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    fa_fp8_quant_kernel<1><<<grid, 256, smem, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fa_fp8_vfold_kernel<<<a.BH, 32, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const CUtensorMap& to, const Fp8Args& a, cudaStream_t stream) {
    const size_t smem = sizeof(Fp8Smem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(a.n_qblk) * static_cast<unsigned>(a.BH);
    fa_fwd_fp8_kernel<<<grid, kThreads, smem, stream>>>(tq, tk, tvt, to, a);
    return cudaGetLastError();
}

}  // namespace fa
