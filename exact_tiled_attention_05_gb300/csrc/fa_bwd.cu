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


// ---------------------------------------------------------------------------
// main: one CTA per (head, 128-key tile j), looping over 128-row query tiles i
// (i >= j when causal).  Everything is computed transposed, keys on the MMA
// M dimension, so dK_j and dV_j accumulate in TMEM for the whole loop:
//   S^T  = K_j Q_i^T                 (TMEM, fp32)
//   dP^T = V_j dO_i^T                (TMEM, fp32)
//   P^T  = exp2(S^T * scale*log2e - lse_i * log2e)      (recomputed from lse)
//   dS^T = P^T * (dP^T - D_i)        (D = rowsum(dO * O) from the prep stage)
//   dV_j += P^T dO_i                 (P^T bf16 from TMEM)
//   dK_j += dS^T Q_i                 (dS^T bf16 from shared memory, K-major)
//   dQ_i  = dS K_j                   (same shared buffer read MN-major)
// and dQ_i is added, times scale, into the fp32 accumulator with vector
// atomics ("FlashAttention 1–4" §"FlashAttention-2": one thread block per K/V
// block, dK/dV kept on chip, dQ accumulated with atomic adds).
// Roles: warp 0 TMA + lse/D staging, warp 1 MMA, warp 2 TMEM allocation,
// warps 4-7 / 8-11 compute for query columns 0-63 / 64-127 of each tile.
// ---------------------------------------------------------------------------
constexpr int kBThreads = 384;
constexpr int kBCompute = 256;  // threads of warps 4..11; each arrives on the compute barriers
constexpr int kBBox = 128 * 64 * 2;

template <int HD>
struct BwdCfg {
    static constexpr int kTile = 128 * HD * 2;
    static constexpr int kBoxes = HD / 64;
    static constexpr int kStages = HD == 128 ? 2 : 3;
    static constexpr uint32_t kS = 0;
    static constexpr uint32_t kDP = 128;
    static constexpr uint32_t kDV = 256;
    static constexpr uint32_t kDK = 256 + HD;
    // d = 128 has no room for a separate dQ block: it reuses the dP^T columns,
    // which are free once the compute warps have read dP^T.
    static constexpr bool kDqInDp = HD == 128;
    static constexpr uint32_t kDQ = kDqInDp ? kDP : 256 + 2 * HD;
    static constexpr uint32_t kTmemCols = 512;
};

template <int HD>
struct alignas(1024) BwdSmem {
    uint8_t k[BwdCfg<HD>::kTile];
    uint8_t v[BwdCfg<HD>::kTile];
    uint8_t q[BwdCfg<HD>::kStages][BwdCfg<HD>::kTile];
    uint8_t dout[BwdCfg<HD>::kStages][BwdCfg<HD>::kTile];
    uint8_t ds[128 * 128 * 2];
    float lse2[BwdCfg<HD>::kStages][128];
    float delta[BwdCfg<HD>::kStages][128];
    uint64_t kv_full;
    uint64_t qd_full[BwdCfg<HD>::kStages];
    uint64_t qd_empty[BwdCfg<HD>::kStages];
    uint64_t s_full, dp_full, p_ready, ds_ready, ds_free, dq_full, dq_drained, dq_staged, dkdv_done,
        drain;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(BwdSmem<128>) <= 232448, "backward d=128 shared memory exceeds 227 KB");
static_assert(sizeof(BwdSmem<64>) <= 232448, "backward d=64 shared memory exceeds 227 KB");

__device__ __forceinline__ void bwd_timeout(const BwdArgs& a, volatile int* abort) {
    *abort = 1;
    atomicExch(a.status, kErrDeviceTimeout);
}

template <int HD>
__global__ void __launch_bounds__(kBThreads, 1)
fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdq, const BwdArgs a) {
    using Cfg = BwdCfg<HD>;
    extern __shared__ __align__(1024) uint8_t bsmem_raw[];
    if ((smem_u32(bsmem_raw) & 1023u) != 0u) {  // the swizzled layouts need 1 KB alignment
        if (threadIdx.x == 0) atomicExch(a.status, kErrUnsupported);
        return;
    }
    BwdSmem<HD>& sm = *reinterpret_cast<BwdSmem<HD>*>(bsmem_raw);
    volatile int* abort = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = a.N;
    const int nq = a.n_kblk;  // query tiles == key tiles (both 128 rows)
    int bh, j;
    if (a.causal) {
        // groups of a.group heads; inside a group the key blocks with the most
        // query tiles (small j) launch first.  Keeping few heads in flight keeps
        // their Q, dO and fp32 dQ accumulator resident in L2.
        const int b = static_cast<int>(blockIdx.x);
        const int grp = b / (a.group * a.n_kblk);
        const int first = grp * a.group;
        const int gc = min(a.group, a.BH - first);
        const int r = b - grp * a.group * a.n_kblk;
        j = r / gc;
        bh = first + r % gc;
    } else {
        bh = static_cast<int>(blockIdx.x) / a.n_kblk;
        j = static_cast<int>(blockIdx.x) % a.n_kblk;
    }
    const int i_begin = a.causal ? j : 0;
    const int niter = nq - i_begin;

    if (threadIdx.x == 0) {
        sm.abort = 0;
        mbar_init(smem_u32(&sm.kv_full), 1);
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(smem_u32(&sm.qd_full[s]), 2);
            mbar_init(smem_u32(&sm.qd_empty[s]), 1);  // the dQ reducer frees the stage
        }
        mbar_init(smem_u32(&sm.s_full), 1);
        mbar_init(smem_u32(&sm.dp_full), 1);
        mbar_init(smem_u32(&sm.p_ready), kBCompute);
        mbar_init(smem_u32(&sm.ds_ready), kBCompute);
        mbar_init(smem_u32(&sm.ds_free), 1);
        mbar_init(smem_u32(&sm.dq_full), 1);
        mbar_init(smem_u32(&sm.dq_drained), kBCompute);
        mbar_init(smem_u32(&sm.dq_staged), kBCompute);
        mbar_init(smem_u32(&sm.dkdv_done), 1);
        mbar_init(smem_u32(&sm.drain), 1);
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&sm.tmem_base), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;

    if (warp == 0) {
        // ===================== loads =====================
        const bool leader = lane == 0;
        if (leader) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdo);
            const uint32_t bar = smem_u32(&sm.kv_full);
            mbar_arrive_expect_tx(bar, 2 * Cfg::kTile);
            for (int b = 0; b < Cfg::kBoxes; ++b) {
                tma_load_3d(smem_u32(sm.k + b * kBBox), &tk, bar, b * 64, j * 128, bh);
                tma_load_3d(smem_u32(sm.v + b * kBBox), &tv, bar, b * 64, j * 128, bh);
            }
        }
        const float* lse_row = a.lse + static_cast<size_t>(bh) * N;
        const float* delta_row = a.delta + static_cast<size_t>(bh) * N;
        int issued = 0;
        for (int it = 0; it < niter; ++it) {
            const int s = it % Cfg::kStages;
            const uint32_t ph = (it / Cfg::kStages) & 1;
            int ok = leader ? mbar_wait(smem_u32(&sm.qd_empty[s]), ph ^ 1, kWaitTimeoutNs, abort) : 1;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (!ok) {
                if (leader) bwd_timeout(a, abort);
                break;
            }
            const int i = i_begin + it;
            const uint32_t fbar = smem_u32(&sm.qd_full[s]);
            if (leader && !FA_FAULT_INJECT) {
                mbar_arrive_expect_tx(fbar, 2 * Cfg::kTile);
                for (int b = 0; b < Cfg::kBoxes; ++b) {
                    tma_load_3d(smem_u32(sm.q[s] + b * kBBox), &tq, fbar, b * 64, i * 128, bh);
                    tma_load_3d(smem_u32(sm.dout[s] + b * kBBox), &tdo, fbar, b * 64, i * 128, bh);
                }
            }
            for (int r = lane; r < 128; r += 32) {
                const int qi = i * 128 + r;
                // rows past the end get lse = +inf, i.e. P = 0
                sm.lse2[s][r] = qi < N ? __ldg(lse_row + qi) * 1.4426950408889634f : INFINITY;
                sm.delta[s][r] = qi < N ? __ldg(delta_row + qi) : 0.f;
            }
            __syncwarp();
            if (leader) mbar_arrive(fbar);
            ++issued;
        }
        if (leader) {
            // Let every copy that was issued land before the CTA can exit.
            for (int s = 0; !FA_FAULT_INJECT && s < Cfg::kStages && s < issued; ++s) {
                const int last = s + Cfg::kStages * ((issued - 1 - s) / Cfg::kStages);
                mbar_wait_drain(smem_u32(&sm.qd_full[s]), (last / Cfg::kStages) & 1, kWaitTimeoutNs);
            }
            mbar_wait_drain(smem_u32(&sm.kv_full), 0, kWaitTimeoutNs);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (elect_one()) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);   // S^T, dP^T
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, HD, 0, 1);   // dV, dK
            constexpr uint32_t id_mnmn = idesc_bf16_f32(128, HD, 1, 1);  // dQ
            const uint32_t k_addr = smem_u32(sm.k), v_addr = smem_u32(sm.v);
            const uint32_t ds_addr = smem_u32(sm.ds);
            bool ok = mbar_wait(smem_u32(&sm.kv_full), 0, kWaitTimeoutNs, abort);
            // D[tmem] = A B^T with both operands K-major over the head dimension.
            auto gemm_kk = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kBBox + (kk % 4) * 32;
                    umma_ss(tbase + d_col, sdesc_sw128(a_addr + off, 16, 1024),
                            sdesc_sw128(b_addr + off, 16, 1024), id_kk, kk > 0);
                }
            };
            for (int it = 0; ok && it < niter; ++it) {
                const int s = it % Cfg::kStages;
                const uint32_t ph = (it / Cfg::kStages) & 1;
                const uint32_t q_addr = smem_u32(sm.q[s]), do_addr = smem_u32(sm.dout[s]);
                if (!(ok = mbar_wait(smem_u32(&sm.qd_full[s]), ph, kWaitTimeoutNs, abort))) break;
                tc_fence_after();
                gemm_kk(Cfg::kS, k_addr, q_addr);  // S^T (after dV of the previous tile in issue order)
                umma_commit(smem_u32(&sm.s_full));
                if (Cfg::kDqInDp && it > 0) {
                    if (!(ok = mbar_wait(smem_u32(&sm.dq_drained), (it - 1) & 1, kWaitTimeoutNs, abort)))
                        break;
                    tc_fence_after();
                }
                gemm_kk(Cfg::kDP, v_addr, do_addr);  // dP^T
                umma_commit(smem_u32(&sm.dp_full));
                if (!(ok = mbar_wait(smem_u32(&sm.p_ready), it & 1, kWaitTimeoutNs, abort))) break;
                tc_fence_after();
                // dV += P^T dO : P^T (bf16) from TMEM; query columns 0-63 packed at
                // TMEM columns [0,32), 64-127 at [64,96); dO MN-major.
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t pcol = Cfg::kS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
                    umma_ts(tbase + Cfg::kDV, tbase + pcol,
                            sdesc_sw128(do_addr + kk * 2048, kBBox, 1024), id_kmn,
                            (it > 0 || kk > 0) ? 1u : 0u);
                }
                if (!(ok = mbar_wait(smem_u32(&sm.ds_ready), it & 1, kWaitTimeoutNs, abort))) break;
                tc_fence_after();
                // dK += dS^T Q : dS^T K-major (rows = keys), Q MN-major.
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk / 4) * kBBox + (kk % 4) * 32;
                    umma_ss(tbase + Cfg::kDK, sdesc_sw128(ds_addr + off, 16, 1024),
                            sdesc_sw128(q_addr + kk * 2048, kBBox, 1024), id_kmn,
                            (it > 0 || kk > 0) ? 1u : 0u);
                }
                // dQ = dS K : the same dS buffer read MN-major (queries contiguous), K MN-major.
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    umma_ss(tbase + Cfg::kDQ, sdesc_sw128(ds_addr + kk * 2048, kBBox, 1024),
                            sdesc_sw128(k_addr + kk * 2048, kBBox, 1024), id_mnmn, kk > 0);
                }
                umma_commit(smem_u32(&sm.dq_full));
                umma_commit(smem_u32(&sm.ds_free));
            }
            if (!ok) bwd_timeout(a, abort);
            umma_commit(smem_u32(&sm.dkdv_done));
            umma_commit(smem_u32(&sm.drain));
            mbar_wait_drain(smem_u32(&sm.drain), 0, kWaitTimeoutNs);
        }
    } else if (warp == 3) {
        // ===================== dQ reducer =====================
        // Adds each staged dQ tile into the fp32 accumulator with TMA bulk
        // reduce-add (whole 128-byte lines instead of per-thread atomics), then
        // hands the stage back to the loader once TMA has read it.
        if (elect_one()) {
            constexpr int kBoxes = HD / 32;
            tma_prefetch_desc(&tdq);
            bool ok = true;
            for (int it = 0; ok && it < niter; ++it) {
                const int s = it % Cfg::kStages;
                const int i = i_begin + it;
                if (!(ok = mbar_wait(smem_u32(&sm.dq_staged), it & 1, kWaitTimeoutNs, abort))) break;
#pragma unroll
                for (int b = 0; b < kBoxes; ++b) {
                    const uint32_t box = (b < kBoxes / 2 ? smem_u32(sm.q[s]) : smem_u32(sm.dout[s])) +
                                         (b % (kBoxes / 2)) * 16384;
                    tma_reduce_add_3d(&tdq, box, b * 32, i * 128, bh);
                }
                bulk_commit_group();
                bulk_wait_group_read0();
                mbar_arrive(smem_u32(&sm.qd_empty[s]));
            }
            if (!ok) bwd_timeout(a, abort);
            bulk_wait_group0();  // every reduction has landed before the CTA exits
        }
    } else if (warp >= 4) {
        // ===================== compute =====================
        const int wg = (warp - 4) >> 2;  // query-column half of S^T / dP^T, and column half of dQ/dK/dV
        const int wq = warp & 3;
        const int row = wq * 32 + lane;   // TMEM lane: key row of S^T/dP^T/dK/dV, query row of dQ
        const int kglob = j * 128 + row;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(wq * 32) << 16);
        const float sl2 = a.scale_log2;
        const uint32_t ds_row = smem_u32(sm.ds) + wg * kBBox + row * 128;
        bool ok = true;
        for (int it = 0; it < niter; ++it) {
            const int s = it % Cfg::kStages;
            const uint32_t ph = (it / Cfg::kStages) & 1;
            const int i = i_begin + it;
            ok = mbar_wait_warp(smem_u32(&sm.s_full), it & 1, kWaitTimeoutNs, abort) &&
                 mbar_wait_warp(smem_u32(&sm.qd_full[s]), ph, kWaitTimeoutNs, abort);
            if (!ok) break;
            tc_fence_after();
            float p[64];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + Cfg::kS + wg * 64, r0);
                tmem_ld32(lane_addr + Cfg::kS + wg * 64 + 32, r1);
                tmem_wait_ld();
                reg_fence(r0);
                reg_fence(r1);
                const uint32_t lse_addr = smem_u32(&sm.lse2[s][wg * 64]);
#pragma unroll
                for (int c4 = 0; c4 < 16; ++c4) {
                    const float4 l4 = ld_shared_f4(lse_addr + c4 * 16);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = c4 * 4 + e;
                        const float sv = __uint_as_float(c < 32 ? r0[c] : r1[c - 32]);
                        p[c] = ex2(fmaf(sv, sl2, -lv[e]));
                    }
                }
            }
            const bool row_valid = kglob < N;
            if (!row_valid) {
#pragma unroll
                for (int c = 0; c < 64; ++c) p[c] = 0.f;
            } else if (a.causal && i == j) {
                // diagonal tile: query q sees key k only when q >= k
                const int qbase = wg * 64;
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (qbase + c < row) p[c] = 0.f;
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
                tmem_st32(lane_addr + Cfg::kS + wg * 64, pk);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.p_ready));

            ok = mbar_wait_warp(smem_u32(&sm.dp_full), it & 1, kWaitTimeoutNs, abort);
            if (ok && it > 0)
                ok = mbar_wait_warp(smem_u32(&sm.ds_free), (it - 1) & 1, kWaitTimeoutNs, abort);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_addr = smem_u32(&sm.delta[s][wg * 64]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
                tmem_ld32(lane_addr + Cfg::kDP + wg * 64 + h * 32, r);
                tmem_wait_ld();
                reg_fence(r);
                uint32_t pk[16];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 d4 = ld_shared_f4(d_addr + (h * 32 + c4 * 4) * 4);
                    const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
                    float ds4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = c4 * 4 + e;
                        ds4[e] = p[h * 32 + c] * (__uint_as_float(r[c]) - dv[e]);
                    }
                    pk[c4 * 2] = pack_bf16x2(ds4[0], ds4[1]);
                    pk[c4 * 2 + 1] = pack_bf16x2(ds4[2], ds4[3]);
                }
                // 32 values = four 16-byte chunks of this key row, 128-byte swizzle
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int chunk = h * 4 + m;
                    st_shared_v4(ds_row + ((chunk ^ (row & 7)) << 4), pk[4 * m], pk[4 * m + 1],
                                 pk[4 * m + 2], pk[4 * m + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.ds_ready));

            ok = mbar_wait_warp(smem_u32(&sm.dq_full), it & 1, kWaitTimeoutNs, abort);
            if (!ok) break;
            tc_fence_after();
            {
                constexpr int kHalf = HD / 2;
                uint32_t r[kHalf];
                if constexpr (kHalf == 64) {
                    uint32_t(&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
                    uint32_t(&r1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
                    tmem_ld32(lane_addr + Cfg::kDQ + wg * kHalf, r0);
                    tmem_ld32(lane_addr + Cfg::kDQ + wg * kHalf + 32, r1);
                    tmem_wait_ld();
                    reg_fence(r0);
                    reg_fence(r1);
                } else {
                    uint32_t(&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
                    tmem_ld32(lane_addr + Cfg::kDQ + wg * kHalf, r0);
                    tmem_wait_ld();
                    reg_fence(r0);
                }
                if (Cfg::kDqInDp) {
                    tc_fence_before();
                    mbar_arrive(smem_u32(&sm.dq_drained));
                }
                // Stage scale * dQ in the Q/dO buffers of this iteration (every MMA
                // that read them has completed): 32-column fp32 boxes, 128-byte
                // swizzle, boxes [0, nb/2) in q[s] and [nb/2, nb) in dout[s].
                constexpr int kBoxes = HD / 32;
                const uint64_t sc2 = f2_pack(a.scale, a.scale);
#pragma unroll
                for (int bl = 0; bl < kHalf / 32; ++bl) {
                    const int b = wg * (kHalf / 32) + bl;
                    const uint32_t box = (b < kBoxes / 2 ? smem_u32(sm.q[s]) : smem_u32(sm.dout[s])) +
                                         (b % (kBoxes / 2)) * 16384 + row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int e = bl * 32 + c * 4;
                        const float2 v0 = f2_unpack(f2_mul(f2_pack_u(r[e], r[e + 1]), sc2));
                        const float2 v1 = f2_unpack(f2_mul(f2_pack_u(r[e + 2], r[e + 3]), sc2));
                        st_shared_v4(box + ((c ^ (row & 7)) << 4), __float_as_uint(v0.x),
                                     __float_as_uint(v0.y), __float_as_uint(v1.x), __float_as_uint(v1.y));
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&sm.dq_staged));
            }
        }
        if (!ok) {
            if (lane == 0) bwd_timeout(a, abort);
        } else {
            ok = mbar_wait_warp(smem_u32(&sm.dkdv_done), 0, kWaitTimeoutNs, abort);
            if (ok) {
                tc_fence_after();
                constexpr int kHalf = HD / 2;
                const bool store = kglob < N;
                const size_t off = (static_cast<size_t>(bh) * N + kglob) * HD + wg * kHalf;
                uint8_t* dv_dst = static_cast<uint8_t*>(a.dv) + off * 2;
                uint8_t* dk_dst = static_cast<uint8_t*>(a.dk) + off * 2;
#pragma unroll 1
                for (int c = 0; c < kHalf; c += 32) {
                    uint32_t rv[32], rk[32];
                    tmem_ld32(lane_addr + Cfg::kDV + wg * kHalf + c, rv);
                    tmem_ld32(lane_addr + Cfg::kDK + wg * kHalf + c, rk);
                    tmem_wait_ld();
                    reg_fence(rv);
                    reg_fence(rk);
                    uint32_t pv[16], pkk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        pv[e] = pack_bf16x2(__uint_as_float(rv[2 * e]), __uint_as_float(rv[2 * e + 1]));
                        pkk[e] = pack_bf16x2(a.scale * __uint_as_float(rk[2 * e]),
                                             a.scale * __uint_as_float(rk[2 * e + 1]));
                    }
                    if (store) {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            st_global_v4(dv_dst + c * 2 + v4 * 16, pv[4 * v4], pv[4 * v4 + 1],
                                         pv[4 * v4 + 2], pv[4 * v4 + 3]);
                            st_global_v4(dk_dst + c * 2 + v4 * 16, pkk[4 * v4], pkk[4 * v4 + 1],
                                         pkk[4 * v4 + 2], pkk[4 * v4 + 3]);
                        }
                    }
                }
            } else if (lane == 0) {
                bwd_timeout(a, abort);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tbase, Cfg::kTmemCols);
    }
}

template <int HD>
cudaError_t launch_bwd_main_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a,
                              cudaStream_t stream) {
    const size_t smem = sizeof(BwdSmem<HD>);
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_main_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(a.n_kblk) * static_cast<unsigned>(a.BH);
    fa_bwd_main_kernel<HD><<<grid, kBThreads, smem, stream>>>(tq, tk, tv, tdo, tdq, a);
    return cudaGetLastError();
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
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                            const BwdArgs& a, cudaStream_t stream) {
    if (d == 64) return launch_bwd_main_t<64>(tq, tk, tv, tdo, tdq, a, stream);
    return launch_bwd_main_t<128>(tq, tk, tv, tdo, tdq, a, stream);
}

}  // namespace fa
