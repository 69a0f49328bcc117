// fa_bwd_dq.cu -- dQ kernel of the backward pass for sm_103a.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

// ---------------------------------------------------------------------------
// dQ: one CTA per (head, 128-row query tile i), looping over 128-key tiles j
// (j <= i when causal), with dQ_i accumulated in TMEM for the whole loop:
//   S    = Q_i K_j^T                  (TMEM, fp32)
//   dP   = dO_i V_j^T                 (TMEM, fp32; two buffers)
//   P    = exp2(S * scale*log2e - lse_i * log2e)       (recomputed from lse)
//   dS   = P * (dP - D_i)             (bf16, written over dP's columns)
//   dQ_i += dS K_j                    (dS from TMEM, K_j MN-major)
//   dq_i  = bf16(scale * dQ_i)
// The same formulas as the dK/dV kernel (the softmax Jacobian), with query
// rows on the MMA M dimension: lse_i and D_i are per-row constants, so a
// thread needs no exchange with the other thread of its row.  S and dP are
// recomputed here rather than sending a partial dQ per (i, j) tile out of
// the SM (see the dK/dV kernel).
// MMA issue order per key tile: S(j), dP(j) into buffer j%2, dQ(j-1).  S(j+1)
// only waits for the compute warps to have read S(j), and dP(j+1) for dQ(j-1)
// to have consumed dS(j-1) from the same buffer, so both are ready when the
// compute warps finish tile j.  K_j is read
// until dQ(j), V_j only until dP(j), so K and V have rings of their own, K
// with one more slot.
// Epilogue: the compute warps stage bf16 scale * dQ, 128-byte swizzled, in K
// slot 0 (free once the last dQ has read it) and warp 0 writes the tile with
// TMA stores (per-thread row stores are the slow path, see the dK/dV kernel).
// Roles: warp 0 TMA loads and stores, warp 1 MMA + TMEM allocation, warps 2-5
// / 6-9 compute for key columns 0-63 / 64-127 of each tile.
// ---------------------------------------------------------------------------
constexpr int kQThreads = 320;
constexpr int kQCompute = 256;       // threads of warps 2..9; each arrives on the compute barriers
constexpr int kQBox = 128 * 64 * 2;  // one 64-column box of a 128-row bf16 tile

template <int HD>
struct DqCfg {
    static constexpr int kTile = 128 * HD * 2;
    static constexpr int kBoxes = HD / 64;
    static constexpr int kKSlots = HD == 128 ? 3 : 6;
    static constexpr int kVSlots = HD == 128 ? 2 : 4;
    static constexpr uint32_t kS = 0;
    static constexpr uint32_t kDP = 128;  // dP / dS buffers at columns 128 and 256
    static constexpr uint32_t kDQ = 384;
    static constexpr uint32_t kTmemCols = 512;
};

template <int HD>
struct alignas(1024) DqSmem {
    uint8_t q[DqCfg<HD>::kTile];
    uint8_t dout[DqCfg<HD>::kTile];
    uint8_t k[DqCfg<HD>::kKSlots][DqCfg<HD>::kTile];
    uint8_t v[DqCfg<HD>::kVSlots][DqCfg<HD>::kTile];
    float nlse2[128];  // -lse * log2(e) per query row (-inf past the end)
    float delta[128];  // D per query row
    uint64_t qd_full;  // Q, dO and their lse * log2(e), D landed
    uint64_t k_full[DqCfg<HD>::kKSlots];
    uint64_t k_empty[DqCfg<HD>::kKSlots];  // committed after dQ(j)
    uint64_t v_full[DqCfg<HD>::kVSlots];
    uint64_t v_empty[DqCfg<HD>::kVSlots];  // committed after dP(j)
    uint64_t s_full;
    uint64_t s_free;       // the compute warps have read S
    uint64_t dp_full[2];   // per dP buffer
    uint64_t ds_ready[2];  // per dP buffer: dS written over it
    uint64_t dq_done;
    uint64_t drain;
    uint64_t out_staged;  // every compute thread has staged its dQ row
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(DqSmem<128>) <= 232448, "dQ kernel d=128 shared memory exceeds 227 KB");
static_assert(sizeof(DqSmem<64>) <= 232448, "dQ kernel d=64 shared memory exceeds 227 KB");

__device__ __forceinline__ void dq_timeout(const BwdArgs& a, volatile int* abort) {
    *abort = 1;
    atomicExch(a.status, kErrDeviceTimeout);
}

template <int HD>
__global__ void __launch_bounds__(kQThreads, 1)
fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap tdq, const BwdArgs a) {
    using Cfg = DqCfg<HD>;
    extern __shared__ __align__(1024) uint8_t qsmem_raw[];
    if ((smem_u32(qsmem_raw) & 1023u) != 0u) {  // the swizzled layouts need 1 KB alignment
        if (threadIdx.x == 0) atomicExch(a.status, kErrUnsupported);
        return;
    }
    DqSmem<HD>& sm = *reinterpret_cast<DqSmem<HD>*>(qsmem_raw);
    volatile int* abort = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = a.N;
    const int nq = a.n_kblk;  // query tiles == key tiles (both 128 rows)
    int bh, i;
    if (a.causal) {
        // groups of a.group_dq heads; inside a group the query tiles with the
        // most key tiles (large i) launch first
        const int b = static_cast<int>(blockIdx.x);
        const int grp = b / (a.group_dq * nq);
        const int first = grp * a.group_dq;
        const int gc = min(a.group_dq, a.BH - first);
        const int r = b - grp * a.group_dq * nq;
        i = nq - 1 - r / gc;
        bh = first + r % gc;
    } else {
        bh = static_cast<int>(blockIdx.x) / nq;
        i = static_cast<int>(blockIdx.x) % nq;
    }
    const int q0 = i * 128;
    const int n = a.causal ? i + 1 : nq;  // key tiles

    if (threadIdx.x == 0) {
        sm.abort = 0;
        mbar_init(smem_u32(&sm.qd_full), 1);
        for (int s = 0; s < Cfg::kKSlots; ++s) {
            mbar_init(smem_u32(&sm.k_full[s]), 1);
            mbar_init(smem_u32(&sm.k_empty[s]), 1);
        }
        for (int s = 0; s < Cfg::kVSlots; ++s) {
            mbar_init(smem_u32(&sm.v_full[s]), 1);
            mbar_init(smem_u32(&sm.v_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sm.dp_full[b]), 1);
            mbar_init(smem_u32(&sm.ds_ready[b]), kQCompute);
        }
        mbar_init(smem_u32(&sm.s_full), 1);
        mbar_init(smem_u32(&sm.s_free), kQCompute);
        mbar_init(smem_u32(&sm.dq_done), 1);
        mbar_init(smem_u32(&sm.drain), 1);
        mbar_init(smem_u32(&sm.out_staged), kQCompute);
        fence_mbar_init();
    }
    if (warp == 1) {
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
        const uint32_t qbar = smem_u32(&sm.qd_full);
        if (leader) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdo);
            mbar_arrive_expect_tx(qbar, 2 * Cfg::kTile + 1024);
            for (int b = 0; b < Cfg::kBoxes; ++b) {
                tma_load_3d(smem_u32(sm.q + b * kQBox), &tq, qbar, b * 64, q0, bh);
                tma_load_3d(smem_u32(sm.dout + b * kQBox), &tdo, qbar, b * 64, q0, bh);
            }
            // the tile's -lse * log2(e) and D (rows past the end: -inf and 0,
            // written by the prep stage)
            const size_t stat = static_cast<size_t>(bh) * nq * 128 + q0;
            bulk_load(smem_u32(sm.nlse2), a.nlse2 + stat, 512, qbar);
            bulk_load(smem_u32(sm.delta), a.delta + stat, 512, qbar);
            // K_j then V_j, each into its own ring
            const int n_loads = FA_FAULT_INJECT ? 0 : n;
            bool ok = true;
            int issued_k = 0, issued_v = 0;
            for (int jj = 0; jj < n_loads; ++jj) {
                const int ks = jj % Cfg::kKSlots, vs = jj % Cfg::kVSlots;
                if (!(ok = mbar_wait(smem_u32(&sm.k_empty[ks]), ((jj / Cfg::kKSlots) & 1) ^ 1,
                                     kWaitTimeoutNs, abort)))
                    break;
                const uint32_t kbar = smem_u32(&sm.k_full[ks]);
                mbar_arrive_expect_tx(kbar, Cfg::kTile);
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.k[ks] + b * kQBox), &tk, kbar, b * 64, jj * 128, bh);
                ++issued_k;
                if (!(ok = mbar_wait(smem_u32(&sm.v_empty[vs]), ((jj / Cfg::kVSlots) & 1) ^ 1,
                                     kWaitTimeoutNs, abort)))
                    break;
                const uint32_t vbar = smem_u32(&sm.v_full[vs]);
                mbar_arrive_expect_tx(vbar, Cfg::kTile);
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.v[vs] + b * kQBox), &tv, vbar, b * 64, jj * 128, bh);
                ++issued_v;
            }
            if (!ok) dq_timeout(a, abort);
            // Let every copy that was issued land before the CTA can exit.
            for (int s = 0; s < Cfg::kKSlots && s < issued_k; ++s) {
                const int last = s + Cfg::kKSlots * ((issued_k - 1 - s) / Cfg::kKSlots);
                mbar_wait_drain(smem_u32(&sm.k_full[s]), (last / Cfg::kKSlots) & 1, kWaitTimeoutNs);
            }
            for (int s = 0; s < Cfg::kVSlots && s < issued_v; ++s) {
                const int last = s + Cfg::kVSlots * ((issued_v - 1 - s) / Cfg::kVSlots);
                mbar_wait_drain(smem_u32(&sm.v_full[s]), (last / Cfg::kVSlots) & 1, kWaitTimeoutNs);
            }
            mbar_wait_drain(qbar, 0, kWaitTimeoutNs);
            // the staged dQ tile
            tma_prefetch_desc(&tdq);
            if (ok && mbar_wait(smem_u32(&sm.out_staged), 0, kWaitTimeoutNs, abort)) {
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_store_3d(&tdq, smem_u32(sm.k[0]) + b * kQBox, b * 64, q0, bh);
                bulk_commit_group();
                bulk_wait_group0();  // written out before the CTA leaves
            } else {
                dq_timeout(a, abort);
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (elect_one()) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);  // S, dP
            constexpr uint32_t id_dq = idesc_bf16_f32(128, HD, 0, 1);   // dQ: dS from TMEM, K MN-major
            const uint32_t q_addr = smem_u32(sm.q), do_addr = smem_u32(sm.dout);
            auto wait_k = [&](int j) -> bool {
                return mbar_wait(smem_u32(&sm.k_full[j % Cfg::kKSlots]), (j / Cfg::kKSlots) & 1,
                                 kWaitTimeoutNs, abort);
            };
            auto wait_v = [&](int j) -> bool {
                return mbar_wait(smem_u32(&sm.v_full[j % Cfg::kVSlots]), (j / Cfg::kVSlots) & 1,
                                 kWaitTimeoutNs, abort);
            };
            auto k_addr = [&](int j) -> uint32_t { return smem_u32(sm.k[j % Cfg::kKSlots]); };
            auto v_addr = [&](int j) -> uint32_t { return smem_u32(sm.v[j % Cfg::kVSlots]); };
            // D[tmem] = A B^T with both operands K-major over the head dimension.
            auto gemm_kk = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kQBox + (kk % 4) * 32;
                    umma_ss(tbase + d_col, sdesc_sw128(a_addr + off, 16, 1024),
                            sdesc_sw128(b_addr + off, 16, 1024), id_kk, kk > 0);
                }
            };
            // dQ += dS(j) K_j : dS (bf16) from TMEM, keys 0-63 packed at columns
            // [0,32) of its dP buffer, keys 64-127 at [64,96); K_j MN-major.
            auto issue_dq = [&](int j) -> bool {
                if (!mbar_wait(smem_u32(&sm.ds_ready[j & 1]), (j >> 1) & 1, kWaitTimeoutNs, abort))
                    return false;
                tc_fence_after();
                const uint32_t buf = Cfg::kDP + static_cast<uint32_t>(j & 1) * 128;
                const uint32_t kj = k_addr(j);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t acol = buf + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
                    umma_ts(tbase + Cfg::kDQ, tbase + acol, sdesc_sw128(kj + kk * 2048, kQBox, 1024),
                            id_dq, (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(smem_u32(&sm.k_empty[j % Cfg::kKSlots]));  // K_j read
                return true;
            };
            bool ok = mbar_wait(smem_u32(&sm.qd_full), 0, kWaitTimeoutNs, abort);
            for (int j = 0; ok && j < n; ++j) {
                // S(j): the compute warps have read S(j-1)
                if (j > 0 && !(ok = mbar_wait(smem_u32(&sm.s_free), (j - 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                if (!(ok = wait_k(j))) break;
                tc_fence_after();
                gemm_kk(Cfg::kS, q_addr, k_addr(j));
                umma_commit(smem_u32(&sm.s_full));
                // dP(j) into buffer j%2: dS(j-2) there was consumed by dQ(j-2),
                // issued earlier (the tensor pipe runs one thread's MMAs in order).
                if (!(ok = wait_v(j))) break;
                tc_fence_after();
                gemm_kk(Cfg::kDP + static_cast<uint32_t>(j & 1) * 128, do_addr, v_addr(j));
                umma_commit(smem_u32(&sm.dp_full[j & 1]));
                umma_commit(smem_u32(&sm.v_empty[j % Cfg::kVSlots]));  // V_j read
                if (j > 0 && !(ok = issue_dq(j - 1))) break;
            }
            if (ok && n > 0) ok = issue_dq(n - 1);
            if (!ok) dq_timeout(a, abort);
            umma_commit(smem_u32(&sm.dq_done));
            // Every MMA (and every commit before it) completes before the CTA leaves.
            umma_commit(smem_u32(&sm.drain));
            mbar_wait_drain(smem_u32(&sm.drain), 0, kWaitTimeoutNs);
        }
    } else {
        // ===================== compute =====================
        const int half = (warp - 2) >> 2;  // key columns [64 half, 64 half + 64) of S / dP
        const int wq = warp & 3;           // TMEM lane quarter this warp may access
        const int row = wq * 32 + lane;    // TMEM lane = query row of the tile
        const int qi = q0 + row;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(wq * 32) << 16);
        const float sl2 = a.scale_log2;
        bool ok = mbar_wait_warp(smem_u32(&sm.qd_full), 0, kWaitTimeoutNs, abort);
        const float nlse2 = ok ? sm.nlse2[row] : 0.f;
        const float dval = ok ? sm.delta[row] : 0.f;
        const uint64_t sl2_pair = f2_pack(sl2, sl2), nl_pair = f2_pack(nlse2, nlse2);
        const uint64_t d_pair = f2_pack(dval, dval);
        for (int j = 0; ok && j < n; ++j) {
            const uint32_t dbuf = Cfg::kDP + static_cast<uint32_t>(j & 1) * 128 + half * 64;
            if (!(ok = mbar_wait_warp(smem_u32(&sm.s_full), j & 1, kWaitTimeoutNs, abort))) break;
            tc_fence_after();
            float p[64];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + Cfg::kS + half * 64, r0);
                tmem_ld32(lane_addr + Cfg::kS + half * 64 + 32, r1);
                tmem_wait_ld();
                reg_fence(r0);
                reg_fence(r1);
                tc_fence_before();
                mbar_arrive(smem_u32(&sm.s_free));
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const uint32_t s0 = c < 32 ? r0[c] : r1[c - 32], s1 = c < 32 ? r0[c + 1] : r1[c - 31];
                    const float2 x = f2_unpack(f2_fma(f2_pack_u(s0, s1), sl2_pair, nl_pair));
                    p[c] = ex2(x.x);
                    p[c + 1] = ex2(x.y);
                }
            }
            const int kbase = j * 128 + half * 64;
            if ((j * 128 + 128 > N) || (a.causal && j * 128 + 127 > q0)) {
                const int kend = a.causal ? min(N, qi + 1) : N;
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (kbase + c >= kend) p[c] = 0.f;
            }
            if (!(ok = mbar_wait_warp(smem_u32(&sm.dp_full[j & 1]), (j >> 1) & 1, kWaitTimeoutNs, abort)))
                break;
            tc_fence_after();
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
                tmem_ld32(lane_addr + dbuf + h * 32, r);
                tmem_wait_ld();
                reg_fence(r);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int e = h * 32 + 2 * c;
                    const float2 ds = f2_unpack(f2_mul(f2_pack(p[e], p[e + 1]),
                                                       f2_sub(f2_pack_u(r[2 * c], r[2 * c + 1]), d_pair)));
                    pk[h * 16 + c] = pack_bf16x2(ds.x, ds.y);
                }
            }
            // dS over the first 32 of the 64 dP columns this thread read
            tmem_st32(lane_addr + dbuf, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.ds_ready[j & 1]));
        }
        if (!ok) {
            if (lane == 0) dq_timeout(a, abort);
        } else {
            ok = mbar_wait_warp(smem_u32(&sm.dq_done), 0, kWaitTimeoutNs, abort);
            if (ok) {
                tc_fence_after();
                // this thread's row of columns [half * d/2, (half + 1) * d/2) of dQ into
                // K slot 0: 64-column boxes of 128-byte rows, 16-byte chunk c of row r
                // at position c ^ (r % 8)
                constexpr int kHalf = HD / 2;
                const int col0 = half * kHalf;
                const uint32_t dst = smem_u32(sm.k[0]) + static_cast<uint32_t>((col0 / 64) * kQBox + row * 128);
#pragma unroll 1
                for (int c = 0; c < kHalf; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(lane_addr + Cfg::kDQ + col0 + c, r);
                    tmem_wait_ld();
                    reg_fence(r);
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack_bf16x2(a.scale * __uint_as_float(r[2 * e]),
                                           a.scale * __uint_as_float(r[2 * e + 1]));
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int chunk = ((col0 % 64) + c) / 8 + m;
                        st_shared_v4(dst + static_cast<uint32_t>((chunk ^ (row & 7)) << 4), w[4 * m],
                                     w[4 * m + 1], w[4 * m + 2], w[4 * m + 3]);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&sm.out_staged));
            } else if (lane == 0) {
                dq_timeout(a, abort);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, Cfg::kTmemCols);
    }
}

template <int HD>
cudaError_t launch_bwd_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a,
                            cudaStream_t stream) {
    const size_t smem = sizeof(DqSmem<HD>);
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_dq_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(a.n_kblk) * static_cast<unsigned>(a.BH);
    fa_bwd_dq_kernel<HD><<<grid, kQThreads, smem, stream>>>(tq, tk, tv, tdo, tdq, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const BwdArgs& a, cudaStream_t stream) {
    if (d == 64) return launch_bwd_dq_t<64>(tq, tk, tv, tdo, tdq, a, stream);
    return launch_bwd_dq_t<128>(tq, tk, tv, tdo, tdq, a, stream);
}

}  // namespace fa
