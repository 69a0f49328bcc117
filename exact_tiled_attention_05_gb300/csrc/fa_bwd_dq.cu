// fa_bwd_dq.cu -- dQ kernel of the backward pass for sm_103a.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

// ---------------------------------------------------------------------------
// dQ: work items (head, 128-row query tile i), each looping over 128-key tiles
// j (j <= i when causal), with dQ_i accumulated in TMEM for the whole loop:
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
// compute warps finish tile j.  K_j is read until dQ(j), V_j only until
// dP(j), so K and V have rings of their own, K with one more slot.
// Persistent: one CTA per SM takes items from a counter in the workspace
// (heavy causal items first, a few heads at a time) until none are left.  The
// key-tile rings, TMEM buffers and barrier phases run on across items, so the
// next item's S(0) and dP(0) are issued while the compute warps still write
// out the previous item's dQ.  That epilogue stages bf16 scale * dQ, 128-byte
// swizzled, in the K slot of the item's last key tile (free once its dQ MMA
// has read it); a store warp writes it out with TMA stores and hands the slot
// back to the loader as soon as the copy has read it.  Q and dO have one
// buffer each: the next item's are loaded once the last S and dP of the
// current item have read them.
// Roles: warp 0 TMA loads and work fetch, warp 1 MMA + TMEM allocation, warps
// 2-5 / 6-9 compute for key columns 0-63 / 64-127 of each tile, warp 10 dQ
// stores.
// ---------------------------------------------------------------------------
constexpr int kQThreads = 352;
constexpr int kQCompute = 256;                // threads of warps 2..9; each arrives on the compute barriers
constexpr int kQItemReaders = 2 + kQCompute;  // MMA thread, store thread, compute threads
constexpr int kQStoreWarp = 10;
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
    float nlse2[2][128];  // per item parity: -lse * log2(e) per query row (-inf past the end)
    float delta[2][128];  // per item parity: D per query row
    int item[2];                           // work items published by the loader (-1: none left)
    uint64_t item_full[2], item_empty[2];  // per queue slot: written / read by every role
    uint64_t qd_full[2];   // per item parity: Q, dO and the row statistics landed
    uint64_t q_free;       // the item's last S has read Q
    uint64_t do_free;      // the item's last dP has read dO
    uint64_t k_full[DqCfg<HD>::kKSlots];
    uint64_t k_empty[DqCfg<HD>::kKSlots];  // after dQ(j); an item's last slot after its dQ store
    uint64_t v_full[DqCfg<HD>::kVSlots];
    uint64_t v_empty[DqCfg<HD>::kVSlots];  // committed after dP(j)
    uint64_t s_full;
    uint64_t s_free;       // the compute warps have read S
    uint64_t dp_full[2];   // per dP buffer
    uint64_t ds_ready[2];  // per dP buffer: dS written over it
    uint64_t dq_done;      // the item's dQ is complete in TMEM
    uint64_t drain;
    uint64_t out_staged;  // every compute thread has staged its dQ row
    uint64_t stage_ack;   // the store thread has seen out_staged (keeps its phases in step)
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(DqSmem<128>) <= 232448, "dQ kernel d=128 shared memory exceeds 227 KB");
static_assert(sizeof(DqSmem<64>) <= 232448, "dQ kernel d=64 shared memory exceeds 227 KB");

// Work item t (fetch order) -> (head, query tile).  Causal: head groups as in
// grouped_item; inside a group the query tiles with the most key tiles (large
// i) come first.
__device__ __forceinline__ void dq_item(const BwdArgs& a, int t, int& bh, int& i) {
    const int nq = a.n_kblk;
    if (a.causal) {
        int rank;
        grouped_item(t, nq, a.BH, a.group_dq, a.group_dq_last, bh, rank);
        i = nq - 1 - rank;
    } else {
        bh = t / nq;
        i = t % nq;
    }
}

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
    const int n_items = a.BH * nq;

    if (threadIdx.x == 0) {
        sm.abort = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sm.item_full[s]), 1);
            mbar_init(smem_u32(&sm.item_empty[s]), kQItemReaders);
            mbar_init(smem_u32(&sm.qd_full[s]), 1);
        }
        mbar_init(smem_u32(&sm.q_free), 1);
        mbar_init(smem_u32(&sm.do_free), 1);
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
        mbar_init(smem_u32(&sm.stage_ack), 1);
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
        // Per item: fetch its index and publish it to the other roles; Q and the
        // row statistics once the previous item's last S has read Q, dO once its
        // last dP has read dO; then K_j and V_j, each into its own ring, whose
        // positions run on across items.
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdo);
            bool ok = true;
            int issued_k = 0, issued_v = 0, issued_qd = 0;
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (k >= 2 && !(ok = mbar_wait(smem_u32(&sm.item_empty[slot]), ((k - 2) >> 1) & 1,
                                               kWaitTimeoutNs, abort)))
                    break;
                const unsigned t = atomicAdd(a.work + kWorkDq, 1u);
                const int item = t < static_cast<unsigned>(n_items) ? static_cast<int>(t) : -1;
                sm.item[slot] = item;
                mbar_arrive(smem_u32(&sm.item_full[slot]));
                if (item < 0) break;
                int bh, i;
                dq_item(a, item, bh, i);
                const int n = a.causal ? i + 1 : nq;  // key tiles
                if (k >= 1 && !(ok = mbar_wait(smem_u32(&sm.q_free), (k - 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                const uint32_t qbar = smem_u32(&sm.qd_full[slot]);
                mbar_arrive_expect_tx(qbar, 2 * Cfg::kTile + 1024);
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.q + b * kQBox), &tq, qbar, b * 64, i * 128, bh);
                // the tile's -lse * log2(e) and D (rows past the end: -inf and 0,
                // written by the prep stage)
                const size_t stat = (static_cast<size_t>(bh) * nq + i) * 128;
                bulk_load(smem_u32(sm.nlse2[slot]), a.nlse2 + stat, 512, qbar);
                bulk_load(smem_u32(sm.delta[slot]), a.delta + stat, 512, qbar);
                ++issued_qd;
                if (k >= 1 && !(ok = mbar_wait(smem_u32(&sm.do_free), (k - 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.dout + b * kQBox), &tdo, qbar, b * 64, i * 128, bh);
                const int n_loads = FA_FAULT_INJECT ? 0 : n;
                for (int jj = 0; jj < n_loads; ++jj) {
                    const int ks = issued_k % Cfg::kKSlots, vs = issued_v % Cfg::kVSlots;
                    if (!(ok = mbar_wait(smem_u32(&sm.k_empty[ks]), ((issued_k / Cfg::kKSlots) & 1) ^ 1,
                                         kWaitTimeoutNs, abort)))
                        break;
                    const uint32_t kbar = smem_u32(&sm.k_full[ks]);
                    mbar_arrive_expect_tx(kbar, Cfg::kTile);
                    for (int b = 0; b < Cfg::kBoxes; ++b)
                        tma_load_3d(smem_u32(sm.k[ks] + b * kQBox), &tk, kbar, b * 64, jj * 128, bh);
                    ++issued_k;
                    if (!(ok = mbar_wait(smem_u32(&sm.v_empty[vs]), ((issued_v / Cfg::kVSlots) & 1) ^ 1,
                                         kWaitTimeoutNs, abort)))
                        break;
                    const uint32_t vbar = smem_u32(&sm.v_full[vs]);
                    mbar_arrive_expect_tx(vbar, Cfg::kTile);
                    for (int b = 0; b < Cfg::kBoxes; ++b)
                        tma_load_3d(smem_u32(sm.v[vs] + b * kQBox), &tv, vbar, b * 64, jj * 128, bh);
                    ++issued_v;
                }
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
            for (int s = 0; s < 2 && s < issued_qd; ++s) {
                const int last = s + 2 * ((issued_qd - 1 - s) / 2);
                mbar_wait_drain(smem_u32(&sm.qd_full[s]), (last >> 1) & 1, kWaitTimeoutNs);
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (elect_one()) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);  // S, dP
            constexpr uint32_t id_dq = idesc_bf16_f32(128, HD, 0, 1);   // dQ: dS from TMEM, K MN-major
            const uint32_t q_addr = smem_u32(sm.q), do_addr = smem_u32(sm.dout);
            auto k_addr = [&](int g) -> uint32_t { return smem_u32(sm.k[g % Cfg::kKSlots]); };
            auto v_addr = [&](int g) -> uint32_t { return smem_u32(sm.v[g % Cfg::kVSlots]); };
            // D[tmem] = A B^T with both operands K-major over the head dimension.
            auto gemm_kk = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kQBox + (kk % 4) * 32;
                    umma_ss(tbase + d_col, sdesc_sw128(a_addr + off, 16, 1024),
                            sdesc_sw128(b_addr + off, 16, 1024), id_kk, kk > 0);
                }
            };
            // dQ (+)= dS(g) K_g : dS (bf16) from TMEM, keys 0-63 packed at columns
            // [0,32) of its dP buffer, keys 64-127 at [64,96); K_g MN-major.  K_g's
            // slot is released here unless it is the item's last (the dQ store
            // stages there and releases it).
            auto issue_dq = [&](int g, bool acc, bool free_k) -> bool {
                if (!mbar_wait(smem_u32(&sm.ds_ready[g & 1]), (g >> 1) & 1, kWaitTimeoutNs, abort))
                    return false;
                tc_fence_after();
                const uint32_t buf = Cfg::kDP + static_cast<uint32_t>(g & 1) * 128;
                const uint32_t kg = k_addr(g);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t acol = buf + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
                    umma_ts(tbase + Cfg::kDQ, tbase + acol, sdesc_sw128(kg + kk * 2048, kQBox, 1024),
                            id_dq, (acc || kk > 0) ? 1u : 0u);
                }
                if (free_k) umma_commit(smem_u32(&sm.k_empty[g % Cfg::kKSlots]));  // K_g read
                return true;
            };
            bool ok = true;
            int g = 0;  // running key-tile count of this CTA (ring positions, barrier phases)
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!(ok = mbar_wait(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                const int item = sm.item[slot];
                mbar_arrive(smem_u32(&sm.item_empty[slot]));
                if (item < 0) break;
                int bh, i;
                dq_item(a, item, bh, i);
                const int n = a.causal ? i + 1 : nq;
                if (!(ok = mbar_wait(smem_u32(&sm.qd_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                for (int j = 0; j < n; ++j, ++g) {
                    // S(j) over S of the previous tile (of this or the previous item),
                    // which the compute warps have read
                    if (g > 0 && !(ok = mbar_wait(smem_u32(&sm.s_free), (g - 1) & 1, kWaitTimeoutNs, abort)))
                        break;
                    if (!(ok = mbar_wait(smem_u32(&sm.k_full[g % Cfg::kKSlots]), (g / Cfg::kKSlots) & 1,
                                         kWaitTimeoutNs, abort)))
                        break;
                    tc_fence_after();
                    gemm_kk(Cfg::kS, q_addr, k_addr(g));
                    umma_commit(smem_u32(&sm.s_full));
                    if (j == n - 1) umma_commit(smem_u32(&sm.q_free));  // the item's Q read
                    // dP(j) into buffer g%2: dS(g-2) there was consumed by dQ(g-2),
                    // issued earlier (the tensor pipe runs one thread's MMAs in order).
                    if (!(ok = mbar_wait(smem_u32(&sm.v_full[g % Cfg::kVSlots]), (g / Cfg::kVSlots) & 1,
                                         kWaitTimeoutNs, abort)))
                        break;
                    tc_fence_after();
                    gemm_kk(Cfg::kDP + static_cast<uint32_t>(g & 1) * 128, do_addr, v_addr(g));
                    umma_commit(smem_u32(&sm.dp_full[g & 1]));
                    umma_commit(smem_u32(&sm.v_empty[g % Cfg::kVSlots]));  // V_j read
                    if (j == n - 1) umma_commit(smem_u32(&sm.do_free));     // the item's dO read
                    if (j > 0 && !(ok = issue_dq(g - 1, j > 1, true))) break;
                }
                if (!ok) break;
                // the item's last dQ; the first dQ of the next item, which overwrites
                // the accumulator, waits for ds_ready, i.e. for the compute warps to
                // have read this one out of TMEM
                if (!(ok = issue_dq(g - 1, n > 1, false))) break;
                umma_commit(smem_u32(&sm.dq_done));
            }
            if (!ok) dq_timeout(a, abort);
            // Every MMA (and every commit before it) completes before the CTA leaves.
            umma_commit(smem_u32(&sm.drain));
            mbar_wait_drain(smem_u32(&sm.drain), 0, kWaitTimeoutNs);
        }
    } else if (warp == kQStoreWarp) {
        // ===================== dQ stores =====================
        // Per item: the staged dQ tile (in the K slot of the item's last key tile)
        // goes out with TMA tile stores; the slot goes back to the loader's K ring
        // as soon as the copy has read it.
        if (elect_one()) {
            tma_prefetch_desc(&tdq);
            bool ok = true;
            int g = 0;  // running key-tile count, as in the MMA warp
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!(ok = mbar_wait(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                const int item = sm.item[slot];
                mbar_arrive(smem_u32(&sm.item_empty[slot]));
                if (item < 0) break;
                int bh, i;
                dq_item(a, item, bh, i);
                g += a.causal ? i + 1 : nq;
                const int ks = (g - 1) % Cfg::kKSlots;
                if (!(ok = mbar_wait(smem_u32(&sm.out_staged), k & 1, kWaitTimeoutNs, abort))) break;
                mbar_arrive(smem_u32(&sm.stage_ack));
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_store_3d(&tdq, smem_u32(sm.k[ks]) + b * kQBox, b * 64, i * 128, bh);
                bulk_commit_group();
                bulk_wait_group_read<0>();
                mbar_arrive(smem_u32(&sm.k_empty[ks]));
            }
            if (!ok) dq_timeout(a, abort);
            bulk_wait_group0();  // written out before the CTA leaves
        }
    } else if (warp >= 2) {
        // ===================== compute =====================
        const int half = (warp - 2) >> 2;  // key columns [64 half, 64 half + 64) of S / dP
        const int wq = warp & 3;           // TMEM lane quarter this warp may access
        const int row = wq * 32 + lane;    // TMEM lane = query row of the tile
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(wq * 32) << 16);
        const float sl2 = a.scale_log2;
        const uint64_t sl2_pair = f2_pack(sl2, sl2);
        bool ok = true;
        int g = 0;  // running key-tile count, as in the MMA warp
        for (int k = 0; ok; ++k) {
            const int slot = k & 1;
            if (!(ok = mbar_wait_warp(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                break;
            const int item = sm.item[slot];
            mbar_arrive(smem_u32(&sm.item_empty[slot]));
            if (item < 0) break;
            int bh, i;
            dq_item(a, item, bh, i);
            const int n = a.causal ? i + 1 : nq;
            const int q0 = i * 128;
            const int qi = q0 + row;
            if (!(ok = mbar_wait_warp(smem_u32(&sm.qd_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                break;
            const float nlse2 = sm.nlse2[slot][row];
            const float dval = sm.delta[slot][row];
            const uint64_t nl_pair = f2_pack(nlse2, nlse2);
            const uint64_t d_pair = f2_pack(dval, dval);
            for (int j = 0; j < n; ++j, ++g) {
                const uint32_t dbuf = Cfg::kDP + static_cast<uint32_t>(g & 1) * 128 + half * 64;
                if (!(ok = mbar_wait_warp(smem_u32(&sm.s_full), g & 1, kWaitTimeoutNs, abort))) break;
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
                if (!(ok = mbar_wait_warp(smem_u32(&sm.dp_full[g & 1]), (g >> 1) & 1, kWaitTimeoutNs, abort)))
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
                mbar_arrive(smem_u32(&sm.ds_ready[g & 1]));
            }
            if (!ok) break;
            // The item's dQ: wait for its last MMA, and for the store thread to have
            // taken the previous item's staged tile (so out_staged never runs two
            // phases ahead of it).
            if (!(ok = mbar_wait_warp(smem_u32(&sm.dq_done), k & 1, kWaitTimeoutNs, abort))) break;
            if (k >= 1 && !(ok = mbar_wait_warp(smem_u32(&sm.stage_ack), (k - 1) & 1, kWaitTimeoutNs, abort)))
                break;
            tc_fence_after();
            // this thread's row of columns [half * d/2, (half + 1) * d/2) of dQ into
            // the K slot of the item's last key tile: 64-column boxes of 128-byte
            // rows, 16-byte chunk c of row r at position c ^ (r % 8)
            constexpr int kHalf = HD / 2;
            const int col0 = half * kHalf;
            const uint32_t dst = smem_u32(sm.k[(g - 1) % Cfg::kKSlots]) +
                                 static_cast<uint32_t>((col0 / 64) * kQBox + row * 128);
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
            // the TMEM reads above come before the next item's first dQ MMA, which
            // waits for this thread's next ds_ready arrival
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&sm.out_staged));
        }
        if (!ok && lane == 0) dq_timeout(a, abort);
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
    cudaError_t e = smem_limit_once<fa_bwd_dq_kernel<HD>>(static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // persistent: one CTA per multiprocessor, work items handed out by a counter
    // (zeroed here, or by the prep kernel inside fa_bwd)
    if (!a.counters_zeroed &&
        (e = cudaMemsetAsync(a.work + kWorkDq, 0, sizeof(unsigned), stream)) != cudaSuccess)
        return e;
    const long long items = static_cast<long long>(a.n_kblk) * a.BH;
    const unsigned grid = static_cast<unsigned>(items < a.sms ? items : a.sms);
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
