// fa_fwd.cu -- fused exact-attention forward pass for sm_103a.
//
// A work item is 256 query rows of one (batch, head): two 128-row Q tiles that
// share every K/V tile streamed for them ("FlashAttention 1–4"
// §"FlashAttention-2": a thread block per query block, K/V streamed in the
// inner loop; two Q tiles per CTA as in §"FlashAttention-4").  With a work
// counter the kernel is persistent: one CTA per SM takes items until none are
// left, and the K/V ring, TMEM buffers and barrier phases run on across items,
// so the next item's Q, K_0 and first S are under way while the softmax warps
// still write out the previous item's O.  Without one, each CTA takes the item
// of its block index.  Roles, by warp:
//   warp 0       TMA producer and work fetch: Q tiles once per item (each
//                buffer once the previous item's last S has read it), K_j, V_j
//                into a ring of shared-memory stages guarded by full/empty
//                mbarriers.
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
//                At the end of an item it normalises O into a staging buffer
//                (one tile at a time) and writes lse.
//   warp 18      O stores: TMA tile stores of the staged tiles.
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
#include <functional>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <tuple>
#include <utility>
#include <vector>

#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

constexpr int kBM = 128;        // query rows per Q tile
constexpr int kBN = 128;        // keys per K/V tile
constexpr int kThreads = 608;   // 19 warps: TMA, MMA (+TMEM allocation), 2 tiles x 8 softmax, stores
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kStoreWarp = 18;
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
    uint8_t o[FwdCfg<HD>::kTileBytes];  // one normalised O tile waiting for its TMA store
    int item[2];                           // work items published by the producer (-1: none left)
    uint64_t item_full[2], item_empty[2];  // per queue slot: written / read by every role
    uint64_t q_full[2];   // per Q tile: landed
    uint64_t q_free[2];   // per Q tile: the item's last S has read it
    uint64_t kv_full[FwdCfg<HD>::kStages];
    uint64_t kv_empty[FwdCfg<HD>::kStages];
    uint64_t s_full[2];
    uint64_t p_full[2][kPParts];  // [tile][part of P]
    uint64_t o_done[2];
    uint64_t out_staged;  // the softmax threads of one tile have staged its O rows
    uint64_t o_free;      // the store thread has read the staged tile out
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(FwdSmem<128>) + 1024 <= 232448, "forward d=128 shared memory exceeds 227 KB");
static_assert(sizeof(FwdSmem<64>) + 1024 <= 232448, "forward d=64 shared memory exceeds 227 KB");

constexpr int kItemReaders = 2 + 2 * kSoftmaxPerTile;  // MMA thread, store thread, softmax threads

__device__ __forceinline__ void record_timeout(FwdArgs const& a, volatile int* abort) {
    *abort = 1;
    atomicExch(a.status, kErrDeviceTimeout);
}

// Work item t (fetch order) -> (head, 256-row query block) and the key tiles
// of its two Q tiles.  Causal: heads in groups of a.group; inside a group the
// heaviest query blocks (the longest key ranges) come first, so taking items
// in order approximates longest-processing-time-first while the K/V of the
// heads in flight stay in L2.  (The host uses it too, to build the static
// schedule.)
struct FwdItem {
    int bh, q0[2], nkv[2], nmax;
};

__host__ __device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int t) {
    FwdItem it;
    int qb;
    if (a.causal) {
        int rank;
        grouped_item(t, a.n_qblk, a.BH, a.group, a.group_last, it.bh, rank);
        qb = a.n_qblk - 1 - rank;
    } else {
        it.bh = t / a.n_qblk;
        qb = t % a.n_qblk;
    }
    const int n_kv_all = (a.N + kBN - 1) / kBN;
    for (int u = 0; u < 2; ++u) {
        it.q0[u] = qb * 2 * kBM + u * kBM;
        if (it.q0[u] >= a.N) {
            it.nkv[u] = 0;  // tile beyond the sequence: inactive
        } else if (a.causal) {
            const int end = it.q0[u] + kBM < a.N ? it.q0[u] + kBM : a.N;
            it.nkv[u] = (end - 1) / kBN + 1;
        } else {
            it.nkv[u] = n_kv_all;
        }
    }
    it.nmax = it.nkv[0] > it.nkv[1] ? it.nkv[0] : it.nkv[1];
    return it;
}

// Next work item of this CTA: from the counter when there is one, else from
// the static schedule in the launch parameters (Cap > 1), else round robin
// (item k * grid + CTA; with one CTA per item that is the CTA's own item).
template <int Cap>
__device__ __forceinline__ int fwd_fetch(const FwdArgs& a, const FwdSched<Cap>& sc, int k,
                                         int n_items) {
    unsigned long long t;
    if (a.work) {
        t = atomicAdd(a.work, 1u);
    } else if (Cap > 1) {
        const int i = sc.start[blockIdx.x] + k;
        t = i < sc.start[blockIdx.x + 1] ? sc.items[i] : static_cast<unsigned long long>(n_items);
    } else {
        t = static_cast<unsigned long long>(k) * gridDim.x + blockIdx.x;
    }
    return t < static_cast<unsigned long long>(n_items) ? static_cast<int>(t) : -1;
}

template <int HD, int Cap>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
              const FwdArgs args, const __grid_constant__ FwdSched<Cap> sched) {
    using Cfg = FwdCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    FwdSmem<HD>& sm = *reinterpret_cast<FwdSmem<HD>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int* abort = &sm.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = args.N;
    const int n_items = args.BH * args.n_qblk;

    if (threadIdx.x == 0) {
        sm.abort = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sm.item_full[s]), 1);
            mbar_init(smem_u32(&sm.item_empty[s]), kItemReaders);
        }
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(smem_u32(&sm.kv_full[s]), 1);
            mbar_init(smem_u32(&sm.kv_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&sm.q_full[t]), 1);
            mbar_init(smem_u32(&sm.q_free[t]), 1);
            mbar_init(smem_u32(&sm.s_full[t]), 1);
            for (int part = 0; part < kPParts; ++part)
                mbar_init(smem_u32(&sm.p_full[t][part]), kSoftmaxPerTile);
            mbar_init(smem_u32(&sm.o_done[t]), 1);
        }
        mbar_init(smem_u32(&sm.out_staged), kSoftmaxPerTile);
        mbar_init(smem_u32(&sm.o_free), 1);
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
        // ===================== TMA producer and work fetch =====================
        // Per item: fetch it and publish it to the other roles; Q_0, K_0, Q_1 (each
        // Q buffer once the previous item's last S on it has completed), then the
        // rest of the item's K_j, V_j into the ring, whose positions run on across
        // items.
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            bool ok = true;
            int issued = 0;        // ring positions loaded
            int nq[2] = {0, 0};    // Q loads per tile
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (k >= 2 && !(ok = mbar_wait(smem_u32(&sm.item_empty[slot]), ((k - 2) >> 1) & 1,
                                               kWaitTimeoutNs, abort)))
                    break;
                const int item = fwd_fetch(args, sched, k, n_items);
                sm.item[slot] = item;
                mbar_arrive(smem_u32(&sm.item_full[slot]));
                if (item < 0) break;
                const FwdItem it = fwd_item(args, item);
                auto load_q = [&](int u) -> bool {
                    if (it.nkv[u] == 0) return true;
                    if (nq[u] > 0 && !mbar_wait(smem_u32(&sm.q_free[u]), (nq[u] - 1) & 1,
                                                kWaitTimeoutNs, abort))
                        return false;
                    const uint32_t qbar = smem_u32(&sm.q_full[u]);
                    mbar_arrive_expect_tx(qbar, Cfg::kTileBytes);
                    for (int b = 0; b < Cfg::kBoxes; ++b)
                        tma_load_3d(smem_u32(sm.q[u] + b * kBoxBytes), &tq, qbar, b * 64, it.q0[u], it.bh);
                    ++nq[u];
                    return true;
                };
                // load idx of the item: K_{idx/2} for even idx, V_{idx/2} for odd
                auto load_kv = [&](int idx) -> bool {
                    const int s = issued % Cfg::kStages;
                    if (!mbar_wait(smem_u32(&sm.kv_empty[s]), ((issued / Cfg::kStages) & 1) ^ 1,
                                   kWaitTimeoutNs, abort))
                        return false;
                    const uint32_t fbar = smem_u32(&sm.kv_full[s]);
                    mbar_arrive_expect_tx(fbar, Cfg::kTileBytes);
                    const CUtensorMap* map = (idx & 1) ? &tv : &tk;
                    for (int b = 0; b < Cfg::kBoxes; ++b)
                        tma_load_3d(smem_u32(sm.kv[s] + b * kBoxBytes), map, fbar, b * 64,
                                    (idx >> 1) * kBN, it.bh);
                    ++issued;
                    return true;
                };
                const int n_loads = FA_FAULT_INJECT ? 0 : 2 * it.nmax;
                if (!(ok = load_q(0))) break;
                if (n_loads > 0 && !(ok = load_kv(0))) break;
                if (!(ok = load_q(1))) break;
                for (int idx = 1; ok && idx < n_loads; ++idx) ok = load_kv(idx);
            }
            if (!ok) record_timeout(args, abort);
            // Let every copy that was issued land before the CTA can exit.
            for (int s = 0; s < Cfg::kStages && s < issued; ++s) {
                const int last = s + Cfg::kStages * ((issued - 1 - s) / Cfg::kStages);
                mbar_wait_drain(smem_u32(&sm.kv_full[s]), (last / Cfg::kStages) & 1, kWaitTimeoutNs);
            }
            for (int u = 0; u < 2; ++u)
                if (nq[u] > 0) mbar_wait_drain(smem_u32(&sm.q_full[u]), (nq[u] - 1) & 1, kWaitTimeoutNs);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (elect_one()) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, HD, 0, 1);
            const uint32_t q_addr[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
            auto wait_kv = [&](int pos) -> bool {
                return mbar_wait(smem_u32(&sm.kv_full[pos % Cfg::kStages]),
                                 (pos / Cfg::kStages) & 1, kWaitTimeoutNs, abort);
            };
            auto kv_addr = [&](int pos) -> uint32_t { return smem_u32(sm.kv[pos % Cfg::kStages]); };
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
            bool ok = true;
            int pos = 0;              // ring position of the item's K_0
            int cnt[2] = {0, 0};      // S_t issued before the item (phases of s_full, p_full, o_done)
            int nq[2] = {0, 0};       // Q_t loads consumed
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!(ok = mbar_wait(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                const int item = sm.item[slot];
                mbar_arrive(smem_u32(&sm.item_empty[slot]));
                if (item < 0) break;
                const FwdItem it = fwd_item(args, item);
                // S_t(0) over P_t of the previous item, whose P V was issued before it
                // (the tensor pipe executes one thread's MMAs in order)
                if (!(ok = wait_kv(pos))) break;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (it.nkv[t] == 0) continue;
                    if (!(ok = mbar_wait(smem_u32(&sm.q_full[t]), nq[t] & 1, kWaitTimeoutNs, abort))) break;
                    ++nq[t];
                    tc_fence_after();
                    issue_s(t, kv_addr(pos));
                    umma_commit(smem_u32(&sm.s_full[t]));
                    if (it.nkv[t] == 1) umma_commit(smem_u32(&sm.q_free[t]));  // the item's last S_t
                }
                if (!ok) break;
                umma_commit(smem_u32(&sm.kv_empty[pos % Cfg::kStages]));
                for (int j = 0; ok && j < it.nmax; ++j) {
                    const int iv = pos + 2 * j + 1, ik = pos + 2 * j + 2;
                    if (!(ok = wait_kv(iv))) break;
                    tc_fence_after();
                    bool k_ready = false;
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j < it.nkv[t]) {
                            for (int part = 0; part < kPParts && ok; ++part) {
                                if (!(ok = mbar_wait(smem_u32(&sm.p_full[t][part]), (cnt[t] + j) & 1,
                                                     kWaitTimeoutNs, abort)))
                                    break;
                                tc_fence_after();
                                issue_pv(t, kv_addr(iv), part, j > 0);
                            }
                            if (!ok) break;
                            umma_commit(smem_u32(&sm.o_done[t]));
                        }
                        if (t == 1) umma_commit(smem_u32(&sm.kv_empty[iv % Cfg::kStages]));
                        if (j + 1 < it.nkv[t]) {
                            if (!k_ready) {
                                if (!(ok = wait_kv(ik))) break;
                                tc_fence_after();
                                k_ready = true;
                            }
                            // S_t(j+1) overwrites P_t(j) only after PV_t(j) was issued.
                            issue_s(t, kv_addr(ik));
                            umma_commit(smem_u32(&sm.s_full[t]));
                            if (j + 2 == it.nkv[t]) umma_commit(smem_u32(&sm.q_free[t]));  // last S_t
                        }
                    }
                    if (ok && k_ready) umma_commit(smem_u32(&sm.kv_empty[ik % Cfg::kStages]));
                }
                pos += 2 * it.nmax;
                cnt[0] += it.nkv[0];
                cnt[1] += it.nkv[1];
            }
            if (!ok) record_timeout(args, abort);
            // Every MMA (and every commit before it) completes before the CTA leaves.
            umma_commit(smem_u32(&sm.drain));
            mbar_wait_drain(smem_u32(&sm.drain), 0, kWaitTimeoutNs);
        }
    } else if (warp == kStoreWarp) {
        // ===================== O stores =====================
        // Per item and active Q tile (tile 0 first): the normalised tile staged in
        // sm.o goes out with TMA tile stores; the buffer is handed back to the
        // softmax warps as soon as the copy has read it.
        if (elect_one()) {
            tma_prefetch_desc(&to);
            bool ok = true;
            int u = 0;  // staged tiles so far
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!(ok = mbar_wait(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                const int item = sm.item[slot];
                mbar_arrive(smem_u32(&sm.item_empty[slot]));
                if (item < 0) break;
                const FwdItem it = fwd_item(args, item);
                for (int t = 0; t < 2 && ok; ++t) {
                    if (it.nkv[t] == 0) continue;
                    if (!(ok = mbar_wait(smem_u32(&sm.out_staged), u & 1, kWaitTimeoutNs, abort))) break;
                    for (int b = 0; b < Cfg::kBoxes; ++b)
                        tma_store_3d(&to, smem_u32(sm.o) + b * kBoxBytes, b * 64, it.q0[t], it.bh);
                    bulk_commit_group();
                    bulk_wait_group_read<0>();
                    mbar_arrive(smem_u32(&sm.o_free));
                    ++u;
                }
            }
            if (!ok) record_timeout(args, abort);
            bulk_wait_group0();  // written out before the CTA leaves
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
        const uint32_t lanes16 = tbase + (static_cast<uint32_t>(wq * 32 + sub * 16) << 16);
        const uint32_t s_addr = lanes16 + static_cast<uint32_t>(t) * Cfg::kSColStride;
        const uint32_t o_addr = lanes16 + Cfg::kOCol0 + t * HD;
        const float sl2 = args.scale_log2;
        const uint64_t sl2_pair = f2_pack(sl2, sl2);
        bool ok = true;
        // The running counts are only needed as barrier phases, kept as bits (few
        // registers stay live across the key loop): bit 0, S_t tiles before the
        // item (s_full, p_full, o_done); bit 1, O tiles staged before the item by
        // both Q tiles (o_free); bit 2, at least one staged; bits 4-5, items taken
        // mod 4 (queue slot and phase).  The item's queue slot is released only at
        // the end of the item, so its details are read from it again there.
        unsigned par = 0;
        while (ok) {
          const int slot = (par >> 4) & 1;
          if (!(ok = mbar_wait_warp(smem_u32(&sm.item_full[slot]), (par >> 5) & 1, kWaitTimeoutNs, abort)))
              break;
          if (sm.item[slot] < 0) break;
          int my_q0, my_nkv;
          {
              const FwdItem it = fwd_item(args, sm.item[slot]);
              my_q0 = t == 0 ? it.q0[0] : it.q0[1];
              my_nkv = t == 0 ? it.nkv[0] : it.nkv[1];
          }
          const int qA = my_q0 + rA, qB = qA + 8;
          // Per row (A, B): running max in log2 units, this thread's share of the
          // fp32 row sum (for lse), and a correction that turns the row sum into the
          // sum of the bf16 weights P V actually used, for the largest weight of each
          // tile only: that weight's rounding is what biases O when one key
          // dominates, the other weights' rounding errors average out.
          float mA = -INFINITY, mB = -INFINITY;
          uint64_t lA = f2_pack(0.f, 0.f), lB = f2_pack(0.f, 0.f);
          float lcA = 0.f, lcB = 0.f;
          for (int j = 0; j < my_nkv; ++j) {
            const unsigned gpar = (par ^ static_cast<unsigned>(j)) & 1u;  // phase of this S_t
            ok = mbar_wait_warp(smem_u32(&sm.s_full[t]), gpar, kWaitTimeoutNs, abort);
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
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int ka = kbase + 8 * i + c2, kb = ka + 64;
                        if (ka >= kendA) sa[4 * i + c2] = __float_as_uint(-INFINITY);
                        if (ka >= kendB) sa[4 * i + 2 + c2] = __float_as_uint(-INFINITY);
                        if (kb >= kendA) sb[4 * i + c2] = __float_as_uint(-INFINITY);
                        if (kb >= kendB) sb[4 * i + 2 + c2] = __float_as_uint(-INFINITY);
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
                for (int c2 = 0; c2 < 2; ++c2) {
                    ma[c2] = fmax3(ma[c2], __uint_as_float(SR(4 * i + c2)),
                                   __uint_as_float(SR(4 * i + 4 + c2)));
                    mb[c2] = fmax3(mb[c2], __uint_as_float(SR(4 * i + 2 + c2)),
                                   __uint_as_float(SR(4 * i + 6 + c2)));
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
                // without branches (selects and multiplications by 1 where nothing
                // moves; fewer instructions than divergent branches): m = -inf,
                // before the first tile, takes the tile's max without a rescale
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
                    // O already holds P V of earlier tiles of this item (a rescale needs
                    // a finite running max, so j > 0): wait for the latest one, then
                    // rescale it before any of this tile's P V is issued.
                    ok = mbar_wait_warp(smem_u32(&sm.o_done[t]), gpar ^ 1u, kWaitTimeoutNs, abort);
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
          if (!ok) break;
          const FwdItem it = fwd_item(args, sm.item[slot]);
          // this tile's staging follows tile 0's when both are active
          const bool after0 = t == 1 && it.nkv[0] > 0;
          const unsigned prev_staged = ((par >> 2) | (after0 ? 1u : 0u)) & 1u;     // an earlier staging exists
          const unsigned prev_par = ((par >> 1) ^ (after0 ? 1u : 0u) ^ 1u) & 1u;  // its o_free phase
          par ^= (static_cast<unsigned>(((it.nkv[0] > 0) + (it.nkv[1] > 0)) & 1) << 1) |
                 (static_cast<unsigned>(my_nkv) & 1u);
          par |= 4u;
          par = (par & 15u) | ((((par >> 4) + 1u) & 3u) << 4);
          if (my_nkv == 0) {  // inactive tile past the end of the sequence
              mbar_arrive(smem_u32(&sm.item_empty[slot]));
              continue;
          }
          // full row sums across the row's four threads
          const float2 la = f2_unpack(lA), lb = f2_unpack(lB);
          float sA = la.x + la.y, sB = lb.x + lb.y;
          sA += __shfl_xor_sync(0xffffffffu, sA, 1);
          sB += __shfl_xor_sync(0xffffffffu, sB, 1);
          sA += __shfl_xor_sync(0xffffffffu, sA, 2);
          sB += __shfl_xor_sync(0xffffffffu, sB, 2);
          // the item's last P V, and the staging buffer back from the previous store
          if (!(ok = mbar_wait_warp(smem_u32(&sm.o_done[t]), (par & 1u) ^ 1u, kWaitTimeoutNs, abort)))
              break;
          if (prev_staged &&
              !(ok = mbar_wait_warp(smem_u32(&sm.o_free), prev_par, kWaitTimeoutNs, abort)))
              break;
          tc_fence_after();
          const float invA = 1.f / (sA + lcA), invB = 1.f / (sB + lcB);
          // O rows rA and rB into the staging buffer as 64-column boxes of 128-byte
          // rows; column 8i + 2cq is 16-byte chunk i % 8 of box i / 8, at position
          // (i % 8) ^ (row % 8), bytes 4cq.. (rB % 8 == rA % 8)
          const uint32_t obuf = smem_u32(sm.o);
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
                  st_shared_b32(obuf + off + static_cast<uint32_t>(rA * 128), wa);
                  st_shared_b32(obuf + off + static_cast<uint32_t>((rA + 8) * 128), wb);
              }
          }
          // the O reads above come before the next item's first P V into O_t, which
          // waits for this thread's next p_full arrival
          tc_fence_before();
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&sm.out_staged));
          if (cq == 0) {
              if (qA < N)
                  args.lse[static_cast<size_t>(it.bh) * N + qA] = (mA + __log2f(sA)) * 0.69314718055994531f;
              if (qB < N)
                  args.lse[static_cast<size_t>(it.bh) * N + qB] = (mB + __log2f(sB)) * 0.69314718055994531f;
          }
          mbar_arrive(smem_u32(&sm.item_empty[slot]));
        }
        if (!ok && lane == 0) record_timeout(args, abort);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, Cfg::kTmemCols);
    }
}

// Static schedules of the forward without a work counter (FwdSched): a small
// table for up to 512 items (1.5 KB of launch parameters), a large one for up
// to 8192 (17 KB); beyond that, round robin.
constexpr int kSchedSmall = 512;
constexpr int kSchedLarge = 8192;

// Greedy longest-first list scheduling of the items, in the counter's fetch
// order, over `grid` CTAs: each item goes to the CTA whose modelled busy time
// is least (lowest index on ties).  Item cost in half key steps (a key step:
// one K/V tile against both Q tiles): FA_SCHED_STEP per step of the longer Q
// tile plus FA_SCHED_FIXED for the Q loads and the O epilogue.
#ifndef FA_SCHED_STEP
#define FA_SCHED_STEP 2
#endif
#ifndef FA_SCHED_FIXED
#define FA_SCHED_FIXED 2
#endif
template <int Cap>
void build_schedule(const FwdArgs& a, int n_items, int grid, FwdSched<Cap>& sc) {
    std::vector<std::vector<uint16_t>> lists(grid);
    using Slot = std::pair<long long, int>;  // (busy time, CTA)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
    for (int c = 0; c < grid; ++c) free_at.push({0, c});
    for (int t = 0; t < n_items; ++t) {
        const FwdItem it = fwd_item(a, t);
        const Slot s = free_at.top();
        free_at.pop();
        lists[s.second].push_back(static_cast<uint16_t>(t));
        free_at.push({s.first + FA_SCHED_STEP * it.nmax + FA_SCHED_FIXED, s.second});
    }
    int pos = 0;
    for (int c = 0; c < grid; ++c) {
        sc.start[c] = static_cast<uint16_t>(pos);
        for (uint16_t t : lists[c]) sc.items[pos++] = t;
    }
    for (int c = grid; c <= kFwdSchedMaxCtas; ++c) sc.start[c] = static_cast<uint16_t>(pos);
}

// Schedules already built, by the arguments that decide them (a launch with the
// same sizes reuses its table).
struct SchedKey {
    int BH, N, n_qblk, group, group_last, causal, grid;
    bool operator<(const SchedKey& o) const {
        return std::tie(BH, N, n_qblk, group, group_last, causal, grid) <
               std::tie(o.BH, o.N, o.n_qblk, o.group, o.group_last, o.causal, o.grid);
    }
};

template <int Cap>
const FwdSched<Cap>* cached_schedule(const FwdArgs& a, int n_items, int grid) {
    static std::mutex mu;
    static std::map<SchedKey, std::unique_ptr<FwdSched<Cap>>> cache;
    const SchedKey key{a.BH, a.N, a.n_qblk, a.group, a.group_last, a.causal, grid};
    std::lock_guard<std::mutex> lock(mu);
    auto f = cache.find(key);
    if (f != cache.end()) return f->second.get();
    if (cache.size() >= 64) cache.clear();  // bounded; a cleared entry is rebuilt on demand
    auto sc = std::make_unique<FwdSched<Cap>>();
    build_schedule(a, n_items, grid, *sc);
    return (cache[key] = std::move(sc)).get();
}

template <int HD, int Cap>
cudaError_t launch_fwd_cap(unsigned grid, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& args,
                           const FwdSched<Cap>& sc, cudaStream_t stream) {
    const size_t smem = sizeof(FwdSmem<HD>) + 1024;
    cudaError_t e = smem_limit_once<fa_fwd_kernel<HD, Cap>>(static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    fa_fwd_kernel<HD, Cap><<<grid, kThreads, smem, stream>>>(tq, tk, tv, to, args, sc);
    return cudaGetLastError();
}

template <int HD>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdArgs& args, cudaStream_t stream) {
    const long long items = static_cast<long long>(args.n_qblk) * args.BH;
    const int sms = args.sms < kFwdSchedMaxCtas ? args.sms : kFwdSchedMaxCtas;
    // persistent either way: one CTA per multiprocessor (fewer for few items)
    const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
    static const FwdSched<1> none{};
    if (args.work) {
        // work items handed out by a counter in the caller's workspace
        cudaError_t e = cudaMemsetAsync(args.work, 0, sizeof(unsigned), stream);
        if (e != cudaSuccess) return e;
        return launch_fwd_cap<HD, 1>(grid, tq, tk, tv, to, args, none, stream);
    }
    const int n = static_cast<int>(items);
    if (items <= kSchedSmall)
        return launch_fwd_cap<HD, kSchedSmall>(grid, tq, tk, tv, to, args,
                                               *cached_schedule<kSchedSmall>(args, n, grid), stream);
    if (items <= kSchedLarge)
        return launch_fwd_cap<HD, kSchedLarge>(grid, tq, tk, tv, to, args,
                                               *cached_schedule<kSchedLarge>(args, n, grid), stream);
    return launch_fwd_cap<HD, 1>(grid, tq, tk, tv, to, args, none, stream);
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& args, cudaStream_t stream) {
    if (d == 64) return launch_fwd_t<64>(tq, tk, tv, to, args, stream);
    return launch_fwd_t<128>(tq, tk, tv, to, args, stream);
}

}  // namespace fa
