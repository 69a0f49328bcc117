// fa_fp8.cu -- FP8 (E4M3) attention forward for sm_103a: block quantization
// with incoherent processing, then the fused forward on FP8 tensor cores.
//
// "FlashAttention 1–4" §"FlashAttention-3", FP8 with block quantization and
// incoherent processing: one FP8 scale per tile instead of one per tensor, and
// Q and K multiplied by the same random orthogonal matrix M = diag(s) H / sqrt(d)
// (random signs, then a Hadamard transform) before quantizing, which leaves
// Q K^T unchanged while spreading outlier channels over all coordinates.
//
// Stage 1, fa_fp8_quant_qk_kernel / fa_fp8_quant_v_kernel (one CTA per
//   (tensor, head, 128-row tile)): Q, K rows rotated in fp32 (sign flips, seven
//   butterfly stages, * 1/sqrt(d)), V not rotated; scale = amax / 448 over the
//   tile (or over the whole tensor for the per-tensor baseline the page
//   compares against), codes = e4m3(x * (448 / amax)).  Q and K codes keep the
//   [BH, N, d] layout; V is written transposed, [BH, d, N], with the keys of
//   each 128-key tile in the order the forward kernel packs P (below).
// Stage 2, fa_fp8_vfold_kernel: per head, vmax = max over tiles of V's scale
//   and fold_t = scale_t / vmax.
// Stage 3, fa_fwd_fp8_kernel: the bf16 forward's structure (two 128-row Q tiles
//   per CTA, four softmax threads per row in one warp, P handed over in two
//   parts, conditional rescaling) with tcgen05.mma kind::f8f6f4: S = Q8 K8^T
//   (four k-steps of 32), s = S * scale_q * scale_k, P * c_j = exp2(s - m +
//   log2 c_j) in fp32 (c_j = 16 fold_j) quantized to E4M3 into shared memory,
//   O += P8 V8^T, row sums l = sum_j (sum P * c_j) / c_j; at the end
//   O * vmax / (16 l).  lse as the bf16 forward.
//
// P's range.  The running max is raised only when a tile's max exceeds it by
// more than tau = 4 (log2 units), so P <= 2^tau; the factor 2^(8 - tau) = 16
// puts the largest P * fold at or below 256 (E4M3 saturates at 448) while
// keeping weights down to 2^-10 of the row max in E4M3's normal range.
//
// Pipeline.  P goes to shared memory (two buffers per Q tile), not over S in
// TMEM, so S(j+1) may overwrite S(j) as soon as the softmax threads hold S(j)
// in registers: the tensor core computes S(j+1) while the softmax of step j
// runs, and P(j) V_j is an SS product.
//
// P layout.  A softmax thread holds keys 8i + 2c + {0, 1} (i < 16, c = lane % 4)
// of its two rows.  For part h (i = 8h .. 8h + 7) it writes, per row, one
// 16-byte chunk: K position 64h + 16c + 2(i - 8h) + e holds key 8i + 2c + e.
// The K order of P is thus a fixed permutation of the tile's keys; V^T is
// written in the same order, and sum_k P[., k] V[k, .] does not depend on it.
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

// Four floats -> four E4M3 codes in one word, a0 in the lowest byte (the two
// conversions write the two halves of the word).
__device__ __forceinline__ uint32_t e4m3x4(float a0, float a1, float a2, float a3) {
    uint32_t r;
    asm("{\n"
        " .reg .b16 lo, hi;\n"
        " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
        " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
        " mov.b32 %0, {lo, hi};\n"
        "}"
        : "=r"(r)
        : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
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

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0 at
// bits 7 and 10), fp32 D, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Key order of P's K positions within a 128-key tile (see the file comment):
// position 64h + 16c + 2i + e holds key 64h + 8i + 2c + e.
__host__ __device__ __forceinline__ int p_key_of_index(int kpos) {
    const int h = kpos >> 6, c = (kpos >> 4) & 3, i = (kpos >> 1) & 7, e = kpos & 1;
    return 64 * h + 8 * i + 2 * c + e;
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

// ---------------------------------------------------------------------------
// Stage 1: rotation and block quantization
// ---------------------------------------------------------------------------
// Both kernels: 256 threads, 8 threads per row, thread g = lane % 8 of a row
// holds its 16 columns 16g .. 16g + 15; a warp covers 4 rows and the CTA 32 per
// pass, four passes cover the 128-row tile.  MODE 0 only reduces |x| of the
// tile into amax[tensor] (per-tensor baseline, first pass); MODE 1 quantizes:
// scale = amax / 448 and code = e4m3(x * (448 / amax)) (scale 1 and factor 1
// for an all-zero tile).

// |x| maximum of the CTA (all threads call; returns the same value to all).
__device__ __forceinline__ float cta_amax(float m, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) r = fmaxf(r, red[w]);
    return r;
}

// Loads 16 bf16 columns of four rows (one per pass) as fp32; rows past N are 0.
__device__ __forceinline__ void load_rows16(const uint16_t* src, int N, int row0, int g, float (&x)[4][16]) {
    uint4 raw[4][2];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int row = row0 + 32 * p;
        const uint4* ptr = reinterpret_cast<const uint4*>(src + static_cast<size_t>(row) * kHD + 16 * g);
        raw[p][0] = row < N ? __ldg(ptr) : make_uint4(0u, 0u, 0u, 0u);
        raw[p][1] = row < N ? __ldg(ptr + 1) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t w[8] = {raw[p][0].x, raw[p][0].y, raw[p][0].z, raw[p][0].w,
                               raw[p][1].x, raw[p][1].y, raw[p][1].z, raw[p][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[p][2 * i] = __uint_as_float(w[i] << 16);
            x[p][2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

// grid (tiles, BH, 2): Q (z = 0) and K (z = 1).
template <int MODE>
__global__ void __launch_bounds__(256, 3) fa_fp8_quant_qk_kernel(const __grid_constant__ Fp8Args a) {
    __shared__ float red[8];
    const int tile = static_cast<int>(blockIdx.x);
    const int bh = static_cast<int>(blockIdx.y);
    const int which = static_cast<int>(blockIdx.z);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane & 7;
    const int N = a.N, npad = a.n_tiles * 128;
    const int row0 = tile * 128 + warp * 4 + (lane >> 3);  // + 32 p
    const uint16_t* src = static_cast<const uint16_t*>(which == 0 ? a.q : a.k) + static_cast<size_t>(bh) * N * kHD;
    float x[4][16];
    load_rows16(src, N, row0, g, x);
    if (a.rotate) {
        // column 16g + e is negated when bit 16(g % 2) + e of word g / 2 is set
        const uint32_t sbits = a.signs[g >> 1] >> (16 * (g & 1));
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            // sign flips, then y_i = sum_j (-1)^popcount(i & j) x_j by butterflies
            // h = 1, 2, 4, 8 (inside the thread) and 16, 32, 64 (across the
            // row's 8 threads), then * 1/sqrt(d).  Every lane runs the shuffles;
            // rows past N are zeroed afterwards.
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if ((sbits >> e) & 1u) x[p][e] = -x[p][e];
#pragma unroll
            for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (i & h) continue;
                    const float u = x[p][i], v = x[p][i + h];
                    x[p][i] = u + v;
                    x[p][i + h] = u - v;
                }
            }
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float o = __shfl_xor_sync(0xffffffffu, x[p][e], m);
                    x[p][e] = (g & m) ? (o - x[p][e]) : (x[p][e] + o);
                }
            }
            const bool live = row0 + 32 * p < N;
#pragma unroll
            for (int e = 0; e < 16; ++e) x[p][e] = live ? x[p][e] * 0.08838834764831845f : 0.f;  // 1 / sqrt(128)
        }
    }
    float m = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(x[p][e]));
    const float amax_tile = cta_amax(m, red);
    if (MODE == 0) {
        if (threadIdx.x == 0)
            atomicMax(reinterpret_cast<unsigned int*>(a.amax + which),
                      __float_as_uint(amax_tile));  // non-negative floats order as their bits
        return;
    }
    const float amax = a.per_tensor ? a.amax[which] : amax_tile;
    const float r = amax > 0.f ? kE4M3Max / amax : 1.f;
    if (threadIdx.x == 0)
        (which == 0 ? a.sq : a.sk)[bh * a.n_tiles + tile] = amax > 0.f ? amax / kE4M3Max : 1.f;
    uint8_t* dst = (which == 0 ? a.q8 : a.k8) + static_cast<size_t>(bh) * npad * kHD;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = e4m3x2(x[p][4 * k] * r, x[p][4 * k + 1] * r) | (e4m3x2(x[p][4 * k + 2] * r, x[p][4 * k + 3] * r) << 16);
        *reinterpret_cast<uint4*>(dst + static_cast<size_t>(row0 + 32 * p) * kHD + 16 * g) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// grid (tiles, BH): V, written transposed ([BH, d, npad]) with each tile's keys
// in P's order; the tile goes through shared memory for the transpose, kept as
// the bf16 values it was read as (33 KB, so several CTAs share an SM).
template <int MODE>
__global__ void __launch_bounds__(256) fa_fp8_quant_v_kernel(const __grid_constant__ Fp8Args a) {
    extern __shared__ uint16_t tl[];  // [128][130] bf16 tile (row stride 65 words against bank conflicts)
    __shared__ float red[8];
    const int tile = static_cast<int>(blockIdx.x);
    const int bh = static_cast<int>(blockIdx.y);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane & 7;
    const int N = a.N, npad = a.n_tiles * 128;
    const int rl0 = warp * 4 + (lane >> 3);  // tile-local row, + 32 p
    const uint16_t* src = static_cast<const uint16_t*>(a.v) + static_cast<size_t>(bh) * N * kHD;
    float x[4][16];
    load_rows16(src, N, tile * 128 + rl0, g, x);
    float m = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            m = fmaxf(m, fabsf(x[p][e]));
            if (MODE == 1) tl[(rl0 + 32 * p) * 130 + 16 * g + e] = static_cast<uint16_t>(__float_as_uint(x[p][e]) >> 16);
        }
    const float amax_tile = cta_amax(m, red);  // (its barrier also orders the tile writes)
    if (MODE == 0) {
        if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(a.amax + 2), __float_as_uint(amax_tile));
        return;
    }
    const float amax = a.per_tensor ? a.amax[2] : amax_tile;
    const float r = amax > 0.f ? kE4M3Max / amax : 1.f;
    if (threadIdx.x == 0) a.sv[bh * a.n_tiles + tile] = amax > 0.f ? amax / kE4M3Max : 1.f;
    // V^T: row = head column, 128 bytes per tile in P's key order
    uint8_t* dst = a.vt8 + static_cast<size_t>(bh) * kHD * npad + tile * 128;
    for (int col = warp; col < kHD; col += 8) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            v[e] = __uint_as_float(static_cast<uint32_t>(tl[p_key_of_index(4 * lane + e) * 130 + col]) << 16) * r;
        reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(col) * npad)[lane] =
            e4m3x2(v[0], v[1]) | (e4m3x2(v[2], v[3]) << 16);
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
// Shared memory: the two Q tiles, two P buffers per Q tile (P(j) goes to
// buffer j % 2; at the end the tile's bf16 O is staged over its two P
// buffers, one 64-column box each) and the K_j / V_j^T ring.
struct alignas(1024) Fp8Smem {
    uint8_t q[2][kTile8];
    uint8_t p[2][2][kTile8];
    uint8_t kv[kStages][kTile8];
    uint64_t q_full;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];        // S_t(j) in TMEM (MMA commit)
    uint64_t s_free[2];        // S_t(j) read into registers (256 softmax threads)
    uint64_t p_full[2][2][2];  // [tile][buffer][part]: P part in shared memory (256 threads)
    uint64_t p_free[2][2];     // [tile][buffer]: the P V reading the buffer completed (MMA commit)
    uint64_t out_staged[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Fp8Smem) + 1024 <= 232448, "FP8 forward shared memory exceeds 227 KB");
static_assert(2 * kTile8 == 2 * kOBox, "O is staged over a tile's two P buffers");

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
            mbar_init(smem_u32(&sm.s_free[t]), kSoftmaxPerTile);
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&sm.p_full[t][b][0]), kSoftmaxPerTile);
                mbar_init(smem_u32(&sm.p_full[t][b][1]), kSoftmaxPerTile);
                mbar_init(smem_u32(&sm.p_free[t][b]), 1);
            }
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
            for (int idx = 0; idx < n_loads; ++idx) {  // K_0, V_0, K_1, V_1, ..
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
                    tma_store_3d(&to, smem_u32(sm.p[t][b]), b * 64, q0[t], bh);
            }
            bulk_commit_group();
            bulk_wait_group0();
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        // Per step j: S_t(j+1) as soon as the softmax has read S_t(j) into
        // registers, then P_t(j) V_j from shared memory as P's parts arrive.
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
            // O_t += P8_t V8: part h of P (K positions 64h..64h+63) is k-steps
            // 2h, 2h + 1; P and V^T K-major, keys in the same order
            auto issue_pv = [&](int t, uint32_t p_addr, uint32_t vt_addr, int part, bool acc) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int kk = part * 2 + i;
                    umma_ss_f8(tbase + kOCol0 + t * kHD, sdesc_sw128(p_addr + kk * 32, 16, 1024),
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
                // S(j+1): overwrites S(j) once the softmax has it in registers
                if (j + 1 < nmax) {
                    if (!(ok = wait_kv(ik))) break;
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j + 1 >= nkv[t]) continue;
                        if (!(ok = mbar_wait(smem_u32(&sm.s_free[t]), j & 1, kWaitTimeoutNs, abort))) break;
                        tc_fence_after();
                        issue_s(t, kv_addr(ik));
                        umma_commit(smem_u32(&sm.s_full[t]));
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&sm.kv_empty[ik % kStages]));
                }
                // P(j) V_j
                if (!(ok = wait_kv(iv))) break;
                tc_fence_after();
                const int b = j & 1;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= nkv[t]) continue;
                    for (int part = 0; part < 2; ++part) {
                        if (!(ok = mbar_wait(smem_u32(&sm.p_full[t][b][part]), (j >> 1) & 1, kWaitTimeoutNs,
                                             abort)))
                            break;
                        tc_fence_after();
                        issue_pv(t, smem_u32(sm.p[t][b]), kv_addr(iv), part, j > 0);
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&sm.p_free[t][b]));
                }
                if (!ok) break;
                umma_commit(smem_u32(&sm.kv_empty[iv % kStages]));
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
        // P part h of rows rA / rB: the 16-byte chunk 4h + cq, 128-byte swizzle
        const uint32_t p_row_A = static_cast<uint32_t>(rA * 128), p_row_B = static_cast<uint32_t>((rA + 8) * 128);
        const uint32_t p_chunk[2] = {static_cast<uint32_t>(((0 + cq) ^ (rA & 7)) << 4),
                                     static_cast<uint32_t>(((4 + cq) ^ (rA & 7)) << 4)};
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
            // c_j = fold_j * 16 goes into the exponent: 2^(x - m + log2 c_j) = P * c_j
            const float cj = __ldg(fold + j) * kPScale;  // exact: a power of two
            const float lg2c = __log2f(cj);
            const float inv_c = __fdividef(1.0f, cj);
            const uint64_t sl2_pair = f2_pack(sl2, sl2);
            const int b = j & 1;
            if (j >= 2) {  // P buffer b was last read by P(j - 2) V (long done by now)
                ok = mbar_wait_warp(smem_u32(&sm.p_free[t][b]), ((j >> 1) - 1) & 1, kWaitTimeoutNs, abort);
                if (!ok) break;
            }
            ok = mbar_wait_warp(smem_u32(&sm.s_full[t]), j & 1, kWaitTimeoutNs, abort);
            if (!ok) break;
            tc_fence_after();
            uint32_t sa[32], sb[32];  // keys 0-63 and 64-127 of the tile
            tmem_ld_16x256b_x8(s_addr, sa);
            tmem_ld_16x256b_x8(s_addr + 64, sb);
            tmem_wait_ld();
            reg_fence(sa);
            reg_fence(sb);
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.s_free[t]));  // the MMA may now write S(j+1)
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
                // without branches (selects and multiplications by 1 where nothing
                // moves): m = -inf, before the first tile, takes the tile's max
                // without a rescale
                const float mxA = pmA * sl2, mxB = pmB * sl2;
                const bool upA = mxA > mA + kRescaleThreshold, upB = mxB > mB + kRescaleThreshold;
                const bool rsA = upA && mA != -INFINITY, rsB = upB && mB != -INFINITY;
                alphaA = rsA ? ex2(mA - mxA) : 1.f;
                alphaB = rsB ? ex2(mB - mxB) : 1.f;
                lA = f2_mul(lA, f2_pack(alphaA, alphaA));
                lB = f2_mul(lB, f2_pack(alphaB, alphaB));
                lcA *= alphaA;
                lcB *= alphaB;
                mA = upA ? mxA : mA;
                mB = upB ? mxB : mB;
                rescale = rsA || rsB;
            }
            const float negA = ((mA == -INFINITY) ? 0.f : -mA) + lg2c;
            const float negB = ((mB == -INFINITY) ? 0.f : -mB) + lg2c;
            const uint64_t negA2 = f2_pack(negA, negA), negB2 = f2_pack(negB, negB);
            uint64_t tA = f2_pack(0.f, 0.f), tB = f2_pack(0.f, 0.f);  // this tile's sum of P * c_j
            const bool any_rescale = __any_sync(0xffffffffu, rescale);
            const uint32_t pbuf = smem_u32(sm.p[t][b]);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                // chunk of row x: repetitions 8hh .. 8hh + 7, an E4M3 pair each
                uint32_t w[2][4];
#pragma unroll
                for (int i2 = 0; i2 < 4; ++i2) {
                    float pv[2][2][2];  // [repetition 2 i2 + ii][row x][pair element]
#pragma unroll
                    for (int ii = 0; ii < 2; ++ii) {
#pragma unroll
                        for (int x = 0; x < 2; ++x) {
                            const int e = hh * 32 + 4 * (2 * i2 + ii) + 2 * x;
                            const uint64_t x2 = f2_fma(f2_pack_u(SR(e), SR(e + 1)), sl2_pair, x == 0 ? negA2 : negB2);
                            const float2 xv = f2_unpack(x2);
                            const float p0 = ex2(xv.x), p1 = ex2(xv.y);
                            if (x == 0)
                                tA = f2_add(tA, f2_pack(p0, p1));
                            else
                                tB = f2_add(tB, f2_pack(p0, p1));
                            pv[ii][x][0] = p0;
                            pv[ii][x][1] = p1;
                        }
                    }
#pragma unroll
                    for (int x = 0; x < 2; ++x)
                        w[x][i2] = e4m3x4(pv[0][x][0], pv[0][x][1], pv[1][x][0], pv[1][x][1]);
                }
                st_shared_v4(pbuf + p_row_A + p_chunk[hh], w[0][0], w[0][1], w[0][2], w[0][3]);
                st_shared_v4(pbuf + p_row_B + p_chunk[hh], w[1][0], w[1][1], w[1][2], w[1][3]);
                if (hh == 0 && any_rescale) {
                    // O holds P V up to step j - 1: wait for that P V, then scale it
                    // before any of step j's P V is issued (it needs P(j) part 0)
                    ok = mbar_wait_warp(smem_u32(&sm.p_free[t][b ^ 1]), ((j - 1) >> 1) & 1, kWaitTimeoutNs, abort);
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
                    tmem_wait_st();
                    tc_fence_before();
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&sm.p_full[t][b][hh]));
            }
#undef SR
            if (!ok) break;
            {
                const uint64_t ic2 = f2_pack(inv_c, inv_c);
                lA = f2_fma(tA, ic2, lA);
                lB = f2_fma(tB, ic2, lB);
                // the row's largest weight as P V used it (E4M3) against fp32
                const float pxA = ex2(fmaf(pmA, sl2, negA)), pxB = ex2(fmaf(pmB, sl2, negB));
                lcA += (e4m3_round(pxA) - pxA) * inv_c;
                lcB += (e4m3_round(pxB) - pxB) * inv_c;
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
            const int jl = my_nkv - 1;
            ok = mbar_wait_warp(smem_u32(&sm.p_free[t][jl & 1]), (jl >> 1) & 1, kWaitTimeoutNs, abort);
            if (ok) {
                tc_fence_after();
                const float vmax = a.vmax[bh] * (1.0f / kPScale);
                const float invA = vmax / (sA + lcA), invB = vmax / (sB + lcB);
                // O rows into the tile's P buffers (free: every P V of the tile is
                // done): 64-column boxes of 128-byte rows, column 8i + 2cq is chunk
                // i % 8 of box i / 8 at (i % 8) ^ (row % 8)
                const uint32_t obuf = smem_u32(sm.p[t][0]);
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
                        st_shared_b32(obuf + off + p_row_A, wa);
                        st_shared_b32(obuf + off + p_row_B, wb);
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
    const size_t smem_v = 128 * 130 * sizeof(uint16_t);
    cudaError_t e = smem_limit_once<fa_fp8_quant_v_kernel<1>>(static_cast<int>(smem_v));
    if (e != cudaSuccess) return e;
    const dim3 grid_qk(static_cast<unsigned>(a.n_tiles), static_cast<unsigned>(a.BH), 2);
    const dim3 grid_v(static_cast<unsigned>(a.n_tiles), static_cast<unsigned>(a.BH), 1);
    if (a.per_tensor) {
        if ((e = cudaMemsetAsync(a.amax, 0, 3 * sizeof(float), stream)) != cudaSuccess) return e;
        fa_fp8_quant_qk_kernel<0><<<grid_qk, 256, 0, stream>>>(a);
        fa_fp8_quant_v_kernel<0><<<grid_v, 256, 0, stream>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    fa_fp8_quant_qk_kernel<1><<<grid_qk, 256, 0, stream>>>(a);
    fa_fp8_quant_v_kernel<1><<<grid_v, 256, smem_v, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fa_fp8_vfold_kernel<<<a.BH, 32, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const CUtensorMap& to, const Fp8Args& a, cudaStream_t stream) {
    const size_t smem = sizeof(Fp8Smem) + 1024;
    cudaError_t e = smem_limit_once<fa_fwd_fp8_kernel>(static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(a.n_qblk) * static_cast<unsigned>(a.BH);
    fa_fwd_fp8_kernel<<<grid, kThreads, smem, stream>>>(tq, tk, tvt, to, a);
    return cudaGetLastError();
}

}  // namespace fa
