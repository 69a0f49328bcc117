// fa_fwd.cu -- fused exact-attention forward pass for sm_103a.
//
// One CTA owns 256 query rows of one (batch, head): two 128-row Q tiles that
// share every K/V tile it streams ("FlashAttention 1–4" §"FlashAttention-2":
// a thread block per query block, K/V streamed in the inner loop; two Q tiles
// per CTA as in §"FlashAttention-4").  Roles, by warp:
//   warp 0       TMA producer: Q tiles once, then K_j, V_j into a ring of
//                shared-memory stages guarded by full/empty mbarriers.
//   warp 1       MMA issuer (and TMEM allocation): S_t = Q_t K_j^T and
//                O_t += P_t V_j on the tcgen05 tensor cores, accumulators in
//                tensor memory (TMEM).
//   warps 2-17   softmax (8 warps per Q tile): with the 16x256b TMEM shape a
//                lane holds 32 scores of each of two rows (r and r + 8), and the
//                four lanes of a quad together hold both rows in full, so a row
//                max is a 3-input max chain plus two shuffles.  Each warp applies
//                the causal/tail mask, runs the online-softmax update and writes
//                P (bf16) back into TMEM over S in two parts (keys 0-63, then
//                64-127), each handed to the MMA warp as soon as it is stored.
//                At the end it normalises O into the tile's Q buffer, which the
//                producer warp writes out with TMA, and writes lse.
//
// Online softmax ("07 GPU、资源估算与 FlashAttention" §7.8; "CS336 Lecture 5
// notes" §11.3-§11.4): per row a running max m (log2 units of the scaled
// score), a running sum l and the unnormalised accumulator O in TMEM.  When a
// tile raises m, O and l are rescaled by exp2(m_old - m_new) before that tile's
// P V is accumulated; warps whose rows all kept their max skip the O pass.
// lse = (m + log2 l) * ln 2.
//
// Causal: key tiles entirely in the future of a Q tile are never loaded or
// multiplied; the diagonal tile and a ragged last tile are masked per element.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kBM = 128;        // query rows per Q tile
constexpr int kBN = 128;        // keys per K/V tile
constexpr int kThreads = 576;   // 18 warps: TMA, MMA (+TMEM allocation), 2 tiles x 8 softmax
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kSoftmaxPerTile = 256;  // threads per Q tile: a quad per pair of rows
constexpr int kBoxBytes = 128 * 64 * 2;  // one TMA box: 128 rows x 64 bf16
// Conditional rescaling ("FlashAttention 1–4" §"FlashAttention-4"): the
// reference max m only moves when a tile's max exceeds it by more than 8 (log2
// units, a factor 256), so most tiles skip the O rescale pass.  P = 2^(s - m)
// then lies in [0, 256] and its largest entry is no longer exactly 1.0, so the
// bf16 rounding of P would bias O on rows close to one-hot.  The fix: per tile,
// the difference between the bf16 and the fp32 value of the row's largest
// weight is added to a correction lc, and O is normalised by l + lc (the
// rounding of the dominant weight cancels in the ratio), while lse uses the
// fp32 sum l of the unrounded weights.
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// Software exp2 for a fraction of the elements ("FlashAttention 1–4"
// §"FlashAttention-4"): with kSoftExpEvery = k > 0, every k-th pair of
// exponentials in a row is computed on the FMA pipes instead of the exp unit.
// Off by default: GB300's exp unit sustains about 32 exponentials per clock per
// SM, twice what the tensor cores consume at d = 128, and each softmax step is
// latency-bound, so every tested fraction (1/4, 1/3, 1/2) measured slower.
// Builds may set FA_SOFT_EXP_EVERY.
#ifndef FA_SOFT_EXP_EVERY
#define FA_SOFT_EXP_EVERY 0
#endif
constexpr int kSoftExpEvery = FA_SOFT_EXP_EVERY;

// P is handed to the MMA warp in two parts, keys 0-63 and 64-127 of the tile:
// P V on the first part overlaps the exponentials of the second.
constexpr int kPParts = 2;

// TMEM accesses of 16 lanes: lane L of the warp holds rows L/4 and L/4 + 8 of
// the 16 addressed.  16x256b: per repetition i, registers 4i..4i+3 are columns
// 8i + 2(L%4) + {0, 1} of the first row, then the same of the second.
// 16x128b: per repetition i, registers 2i, 2i+1 are column 4i + L%4 of the
// first and of the second row.
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

__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x8.b32"
        " [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

template <int HD>
struct FwdCfg {
    static constexpr int kTileBytes = kBN * HD * 2;
    static constexpr int kBoxes = HD / 64;
    static constexpr int kStages = HD == 128 ? 4 : 8;
    static constexpr uint32_t kSColStride = 128;  // S_t at TMEM column t * 128
    static constexpr uint32_t kOCol0 = 256;
    static constexpr uint32_t kTmemCols = 512;
};

template <int HD>
struct alignas(1024) FwdSmem {
    uint8_t q[2][FwdCfg<HD>::kTileBytes];
    uint8_t kv[FwdCfg<HD>::kStages][FwdCfg<HD>::kTileBytes];
    uint64_t q_full;
    uint64_t kv_full[FwdCfg<HD>::kStages];
    uint64_t kv_empty[FwdCfg<HD>::kStages];
    uint64_t s_full[2];
    uint64_t p_full[2][kPParts];  // [tile][part of P]
    uint64_t o_done[2];
    uint64_t out_staged[2];  // per tile: every softmax thread has staged its O rows
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(FwdSmem<128>) + 1024 <= 232448, "forward d=128 shared memory exceeds 227 KB");
static_assert(sizeof(FwdSmem<64>) + 1024 <= 232448, "forward d=64 shared memory exceeds 227 KB");

__device__ __forceinline__ void record_timeout(FwdArgs const& a, volatile int* abort) {
    *abort = 1;
    atomicExch(a.status, kErrDeviceTimeout);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
              const FwdArgs args) {
    using Cfg = FwdCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    FwdSmem<HD>& sm = *reinterpret_cast<FwdSmem<HD>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int* abort = &sm.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = args.N;
    const int BH = args.BH;

    // ---- work unit: (head, 256-row query block) ----
    // Causal: heads are taken in groups of args.group; inside a group the
    // heaviest query blocks (the longest key ranges) launch first, so the
    // block scheduler approximates longest-processing-time-first while the
    // K/V of the heads in flight stay in L2.
    int bh, qb;
    if (args.causal) {
        const int b = static_cast<int>(blockIdx.x);
        const int grp = b / (args.group * args.n_qblk);
        const int first = grp * args.group;
        const int gc = min(args.group, BH - first);
        const int r = b - grp * args.group * args.n_qblk;
        qb = args.n_qblk - 1 - r / gc;
        bh = first + r % gc;
    } else {
        bh = static_cast<int>(blockIdx.x) / args.n_qblk;
        qb = static_cast<int>(blockIdx.x) % args.n_qblk;
    }
    const int n_kv_all = (N + kBN - 1) / kBN;
    int q0[2], nkv[2];
    for (int t = 0; t < 2; ++t) {
        q0[t] = qb * 2 * kBM + t * kBM;
        if (q0[t] >= N) {
            nkv[t] = 0;  // tile beyond the sequence: inactive
        } else if (args.causal) {
            const int last_q = min(q0[t] + kBM, N) - 1;
            nkv[t] = last_q / kBN + 1;
        } else {
            nkv[t] = n_kv_all;
        }
    }
    const int nmax = max(nkv[0], nkv[1]);

    if (threadIdx.x == 0) {
        sm.abort = 0;
        mbar_init(smem_u32(&sm.q_full), 1);
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(smem_u32(&sm.kv_full[s]), 1);
            mbar_init(smem_u32(&sm.kv_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&sm.s_full[t]), 1);
            for (int part = 0; part < kPParts; ++part)
                mbar_init(smem_u32(&sm.p_full[t][part]), kSoftmaxPerTile);
            mbar_init(smem_u32(&sm.o_done[t]), 1);
            mbar_init(smem_u32(&sm.out_staged[t]), kSoftmaxPerTile);
        }
        mbar_init(smem_u32(&sm.drain), 1);
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
        // ===================== TMA producer =====================
        if (elect_one()) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            const uint32_t qbar = smem_u32(&sm.q_full);
            const int nact = (nkv[0] > 0) + (nkv[1] > 0);
            mbar_arrive_expect_tx(qbar, nact * Cfg::kTileBytes);
            for (int t = 0; t < 2; ++t) {
                if (nkv[t] == 0) continue;
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.q[t] + b * kBoxBytes), &tq, qbar, b * 64, q0[t], bh);
            }
            int issued = 0;
            bool ok = true;
            const int n_loads = FA_FAULT_INJECT ? 0 : 2 * nmax;
            for (int idx = 0; idx < n_loads; ++idx) {
                const int slot = idx % Cfg::kStages;
                const uint32_t ph = (idx / Cfg::kStages) & 1;
                if (!mbar_wait(smem_u32(&sm.kv_empty[slot]), ph ^ 1, kWaitTimeoutNs, abort)) {
                    record_timeout(args, abort);
                    ok = false;
                    break;
                }
                const uint32_t fbar = smem_u32(&sm.kv_full[slot]);
                mbar_arrive_expect_tx(fbar, Cfg::kTileBytes);
                const CUtensorMap* map = (idx & 1) ? &tv : &tk;
                const int row = (idx >> 1) * kBN;
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.kv[slot] + b * kBoxBytes), map, fbar, b * 64, row, bh);
                ++issued;
            }
            // Let every copy that was issued land before the CTA can exit.
            for (int slot = 0; slot < Cfg::kStages && slot < issued; ++slot) {
                const int last = slot + Cfg::kStages * ((issued - 1 - slot) / Cfg::kStages);
                mbar_wait_drain(smem_u32(&sm.kv_full[slot]), (last / Cfg::kStages) & 1,
                                kWaitTimeoutNs);
            }
            mbar_wait_drain(qbar, 0, kWaitTimeoutNs);
            // O of each tile, staged by the softmax warps over the tile's Q buffer
            tma_prefetch_desc(&to);
            for (int t = 0; ok && t < 2; ++t) {
                if (nkv[t] == 0) continue;
                if (!(ok = mbar_wait(smem_u32(&sm.out_staged[t]), 0, kWaitTimeoutNs, abort))) {
                    record_timeout(args, abort);
                    break;
                }
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_store_3d(&to, smem_u32(sm.q[t]) + b * kBoxBytes, b * 64, q0[t], bh);
            }
            bulk_commit_group();
            bulk_wait_group0();  // written out before the CTA leaves
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (elect_one()) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, HD, 0, 1);
            const uint32_t q_addr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
            bool ok = mbar_wait(smem_u32(&sm.q_full), 0, kWaitTimeoutNs, abort);
            auto wait_kv = [&](int idx) -> bool {
                return mbar_wait(smem_u32(&sm.kv_full[idx % Cfg::kStages]),
                                 (idx / Cfg::kStages) & 1, kWaitTimeoutNs, abort);
            };
            auto kv_addr = [&](int idx) -> uint32_t { return smem_u32(sm.kv[idx % Cfg::kStages]); };
            // S_t = Q_t K^T : K-major A and B, HD/16 k-steps of 16.
            auto issue_s = [&](int t, uint32_t k_addr) {
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;
                    umma_ss(tbase + (static_cast<uint32_t>(t) * Cfg::kSColStride), sdesc_sw128(q_addr[t] + off, 16, 1024),
                            sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0);
                }
            };
            // O_t += P_t V : P (bf16) from TMEM, V MN-major, k-steps of 16 keys;
            // part q of P (keys 64q..64q+63) is k-steps 4q..4q+3.
            auto issue_pv = [&](int t, uint32_t v_addr, int part, bool acc) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kk = part * 4 + i;
                    umma_ts(tbase + Cfg::kOCol0 + t * HD, tbase + (static_cast<uint32_t>(t) * Cfg::kSColStride) + kk * 8,
                            sdesc_sw128(v_addr + kk * 16 * 128, kBoxBytes, 1024), idesc_o,
                            (acc || part > 0 || i > 0) ? 1u : 0u);
                }
            };
            if (ok && nmax > 0) {
                ok = wait_kv(0);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t) {
                        if (nkv[t] == 0) continue;
                        issue_s(t, kv_addr(0));
                        umma_commit(smem_u32(&sm.s_full[t]));
                    }
                    umma_commit(smem_u32(&sm.kv_empty[0]));
                }
            }
            for (int j = 0; ok && j < nmax; ++j) {
                const int iv = 2 * j + 1, ik = 2 * j + 2;
                if (!(ok = wait_kv(iv))) break;
                tc_fence_after();
                bool k_ready = false;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j < nkv[t]) {
                        for (int part = 0; part < kPParts && ok; ++part) {
                            if (!(ok = mbar_wait(smem_u32(&sm.p_full[t][part]), j & 1, kWaitTimeoutNs,
                                                 abort)))
                                break;
                            tc_fence_after();
                            issue_pv(t, kv_addr(iv), part, j > 0);
                        }
                        if (!ok) break;
                        umma_commit(smem_u32(&sm.o_done[t]));
                    }
                    if (t == 1) umma_commit(smem_u32(&sm.kv_empty[iv % Cfg::kStages]));
                    if (j + 1 < nkv[t]) {
                        if (!k_ready) {
                            if (!(ok = wait_kv(ik))) break;
                            tc_fence_after();
                            k_ready = true;
                        }
                        // S_t(j+1) overwrites P_t(j) only after PV_t(j) was issued;
                        // the tensor pipe executes one thread's MMAs in order.
                        issue_s(t, kv_addr(ik));
                        umma_commit(smem_u32(&sm.s_full[t]));
                    }
                }
                if (ok && k_ready) umma_commit(smem_u32(&sm.kv_empty[ik % Cfg::kStages]));
            }
            if (!ok) record_timeout(args, abort);
            // Every MMA (and every commit before it) completes before the CTA leaves.
            umma_commit(smem_u32(&sm.drain));
            mbar_wait_drain(smem_u32(&sm.drain), 0, kWaitTimeoutNs);
        }
    } else {
        // ===================== softmax / epilogue =====================
        // Softmax warps 8t..8t+7 (counted from warp 2) own Q tile t.  Warp
        // (wq, sub), wq = warp % 4 the TMEM lane quarter it may access and sub
        // which 16 of those 32 lanes, reads S_t with the 16x256b shape: lane L
        // holds rows rA = 32 wq + 16 sub + L/4 and rB = rA + 8, key columns
        // 8i + 2(L%4) + {0, 1}, i = 0..15.  The four threads of a row sit in one
        // warp, so row maxima and sums are combined with two shuffles, and every
        // reader of a row's S columns has passed tcgen05.wait::ld before the warp
        // overwrites them with P.
        const int sw = warp - kFirstSoftmaxWarp;
        const int t = sw >> 3;          // Q tile
        const int sub = (sw >> 2) & 1;  // lanes 0-15 or 16-31 of the quarter
        const int wq = warp & 3;        // TMEM lane quarter this warp may access
        const int cq = lane & 3;        // column group within the row's four threads
        const int rA = wq * 32 + sub * 16 + (lane >> 2);
        const int my_q0 = t == 0 ? q0[0] : q0[1];
        const int my_nkv = t == 0 ? nkv[0] : nkv[1];
        const int qA = my_q0 + rA, qB = qA + 8;
        const uint32_t lanes16 = tbase + (static_cast<uint32_t>(wq * 32 + sub * 16) << 16);
        const uint32_t s_addr = lanes16 + static_cast<uint32_t>(t) * Cfg::kSColStride;
        const uint32_t o_addr = lanes16 + Cfg::kOCol0 + t * HD;
        const float sl2 = args.scale_log2;
        // Per row (A, B): running max in log2 units, this thread's share of the
        // fp32 row sum (for lse), and a correction that turns the row sum into the
        // sum of the bf16 weights P V actually used, for the largest weight of each
        // tile only: that weight's rounding is what biases O when one key
        // dominates, the other weights' rounding errors average out.
        float mA = -INFINITY, mB = -INFINITY;
        uint64_t lA = f2_pack(0.f, 0.f), lB = f2_pack(0.f, 0.f);
        float lcA = 0.f, lcB = 0.f;
        const uint64_t sl2_pair = f2_pack(sl2, sl2);
        bool ok = true;
        for (int j = 0; j < my_nkv; ++j) {
            ok = mbar_wait_warp(smem_u32(&sm.s_full[t]), j & 1, kWaitTimeoutNs, abort);
            if (!ok) break;
            tc_fence_after();
            uint32_t sa[32], sb[32];  // keys 0-63 and 64-127 of the tile
            tmem_ld_16x256b_x8(s_addr, sa);
            tmem_ld_16x256b_x8(s_addr + 64, sb);
            tmem_wait_ld();
            reg_fence(sa);
            reg_fence(sb);
            // register e of the part: repetition e/4, row A for e%4 < 2, key 8(e/4) + 2cq + e%2
#define SR(c) ((c) < 32 ? sa[(c)] : sb[(c) - 32])
            const int kbase = j * kBN + 2 * cq;
            const bool edge = (j * kBN + kBN > N) || (args.causal && j * kBN + kBN - 1 > my_q0);
            if (edge) {
                const int kendA = args.causal ? min(N, qA + 1) : N;
                const int kendB = args.causal ? min(N, qB + 1) : N;
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
            // row maxima: 32 values per row in this thread, then across the four
            float ma[2], mb[2];
            ma[0] = __uint_as_float(sa[0]);
            ma[1] = __uint_as_float(sa[1]);
            mb[0] = __uint_as_float(sa[2]);
            mb[1] = __uint_as_float(sa[3]);
#pragma unroll
            for (int i = 1; i < 15; i += 2) {  // repetitions 1..14 in pairs
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    ma[c] = fmax3(ma[c], __uint_as_float(SR(4 * i + c)),
                                  __uint_as_float(SR(4 * i + 4 + c)));
                    mb[c] = fmax3(mb[c], __uint_as_float(SR(4 * i + 2 + c)),
                                  __uint_as_float(SR(4 * i + 6 + c)));
                }
            }
            // repetition 15
            float pmA = fmax3(ma[0], ma[1], fmaxf(__uint_as_float(sb[28]), __uint_as_float(sb[29])));
            float pmB = fmax3(mb[0], mb[1], fmaxf(__uint_as_float(sb[30]), __uint_as_float(sb[31])));
            pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 1));
            pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 1));
            pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 2));
            pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 2));
            // running-max update; O and the sums are rescaled when it rises by more
            // than the threshold (the row's four threads take the same decision)
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
            // P = exp2(s * scale * log2e - m) as packed bf16 pairs, stored over the
            // S columns (16x128b: repetition i of part q is P column 32q + 4i + cq,
            // keys 64q + 8i + 2cq + {0, 1}).  Each part is signalled as soon as it
            // is stored, so the MMA warp starts P V on it while the rest is computed.
            const bool any_rescale = __any_sync(0xffffffffu, rescale);
#pragma unroll
            for (int hh = 0; hh < kPParts; ++hh) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
#pragma unroll
                    for (int x = 0; x < 2; ++x) {  // row A, row B
                        const int e = hh * 32 + 4 * i + 2 * x;
                        const uint64_t x2 = f2_fma(f2_pack_u(SR(e), SR(e + 1)), sl2_pair,
                                                   x == 0 ? negA2 : negB2);
                        float p0, p1;
                        const int pair = 2 * i + x;
                        if (kSoftExpEvery > 0 &&
                            (pair % (kSoftExpEvery > 0 ? kSoftExpEvery : 1)) == kSoftExpEvery - 1) {
                            // this pair on the FMA pipes, the rest on the exp unit
                            const float2 pv = f2_unpack(exp2_fma_pair(x2));
                            p0 = pv.x;
                            p1 = pv.y;
                        } else {
                            const float2 xv = f2_unpack(x2);
                            p0 = ex2(xv.x);
                            p1 = ex2(xv.y);
                        }
                        if (x == 0)
                            lA = f2_add(lA, f2_pack(p0, p1));
                        else
                            lB = f2_add(lB, f2_pack(p0, p1));
                        pk[2 * i + x] = pack_bf16x2(p0, p1);
                    }
                }
                tmem_st_16x128b_x8(s_addr + hh * 32, pk);
                if (hh == 0 && any_rescale) {
                    // O already holds P V of earlier tiles: wait for the latest one,
                    // then rescale it before any of this tile's P V is issued.
                    ok = mbar_wait_warp(smem_u32(&sm.o_done[t]), (j - 1) & 1, kWaitTimeoutNs, abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t aA = f2_pack(alphaA, alphaA), aB = f2_pack(alphaB, alphaB);
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t r[16];
                        tmem_ld_16x256b_x4(o_addr + c * 32, r);
                        tmem_wait_ld();
                        reg_fence(r);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float2 v = f2_unpack(
                                f2_mul(f2_pack_u(r[2 * i], r[2 * i + 1]), (i & 1) ? aB : aA));
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
                // the loop's rounding steps applied to each row's largest score
                const float pxA = ex2(fmaf(pmA, sl2, negA));
                const float pxB = ex2(fmaf(pmB, sl2, negB));
                const uint32_t pb = pack_bf16x2(pxA, pxB);
                lcA += __uint_as_float(pb << 16) - pxA;
                lcB += __uint_as_float(pb & 0xffff0000u) - pxB;
            }
        }
        if (!ok) {
            if (lane == 0) record_timeout(args, abort);
        } else if (my_nkv > 0) {
            // full row sums across the row's four threads
            const float2 la = f2_unpack(lA), lb = f2_unpack(lB);
            float sA = la.x + la.y, sB = lb.x + lb.y;
            sA += __shfl_xor_sync(0xffffffffu, sA, 1);
            sB += __shfl_xor_sync(0xffffffffu, sB, 1);
            sA += __shfl_xor_sync(0xffffffffu, sA, 2);
            sB += __shfl_xor_sync(0xffffffffu, sB, 2);
            ok = mbar_wait_warp(smem_u32(&sm.o_done[t]), (my_nkv - 1) & 1, kWaitTimeoutNs, abort);
            if (ok) {
                tc_fence_after();
                const float invA = 1.f / (sA + lcA), invB = 1.f / (sB + lcB);
                const bool storeA = qA < N, storeB = qB < N;
                // O rows rA and rB into the tile's Q buffer (free: the tile's last
                // S MMA finished before its last P V), as 64-column boxes of
                // 128-byte rows; column 8i + 2cq is 16-byte chunk i % 8 of box i / 8,
                // at position (i % 8) ^ (row % 8), bytes 4cq.. (rB % 8 == rA % 8)
                const uint32_t qbuf = smem_u32(sm.q[t]);
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t r[16];
                    tmem_ld_16x256b_x4(o_addr + c * 32, r);
                    tmem_wait_ld();
                    reg_fence(r);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t wa = pack_bf16x2(__uint_as_float(r[4 * i]) * invA,
                                                        __uint_as_float(r[4 * i + 1]) * invA);
                        const uint32_t wb = pack_bf16x2(__uint_as_float(r[4 * i + 2]) * invB,
                                                        __uint_as_float(r[4 * i + 3]) * invB);
                        const int ii = c * 4 + i;
                        const uint32_t off = static_cast<uint32_t>(
                            (ii / 8) * kBoxBytes + (((ii % 8) ^ (rA & 7)) << 4) + 4 * cq);
                        st_shared_b32(qbuf + off + static_cast<uint32_t>(rA * 128), wa);
                        st_shared_b32(qbuf + off + static_cast<uint32_t>((rA + 8) * 128), wb);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&sm.out_staged[t]));
                if (cq == 0) {
                    if (storeA)
                        args.lse[static_cast<size_t>(bh) * N + qA] =
                            (mA + __log2f(sA)) * 0.69314718055994531f;
                    if (storeB)
                        args.lse[static_cast<size_t>(bh) * N + qB] =
                            (mB + __log2f(sB)) * 0.69314718055994531f;
                }
            } else if (lane == 0) {
                record_timeout(args, abort);
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
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdArgs& args, cudaStream_t stream) {
    const size_t smem = sizeof(FwdSmem<HD>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(args.n_qblk) * static_cast<unsigned>(args.BH);
    fa_fwd_kernel<HD><<<grid, kThreads, smem, stream>>>(tq, tk, tv, to, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& args, cudaStream_t stream) {
    if (d == 64) return launch_fwd_t<64>(tq, tk, tv, to, args, stream);
    return launch_fwd_t<128>(tq, tk, tv, to, args, stream);
}

}  // namespace fa
