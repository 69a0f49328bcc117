// fa_bwd.cu -- backward pass: D = rowsum(dO * O) and the dK / dV kernel, for sm_103a.
#include "fa_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

// ---------------------------------------------------------------------------
// prep: D_i = sum_c dO[i,c] * O[i,c] (fp32) and -lse_i * log2(e) (negated, so
// that the exponent of P is one fused multiply-add), d/8 threads per row (one
// 16-byte vector of O and of dO each), written for every row of whole 128-row
// tiles so that the two kernels after it load a tile's 128 values with one bulk
// copy; padding rows get D = 0 and -lse * log2(e) = -inf.
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const BwdArgs a) {
    // Within fa_bwd the dK/dV and dQ kernels that follow skip the memsets of
    // their work counters: this kernel zeroes them (the stream runs the two
    // kernels after it).
    if (a.zero_counters && blockIdx.x == 0 && threadIdx.x == 0) {
        a.work[kWorkDkdv] = 0u;
        a.work[kWorkDq] = 0u;
    }
    constexpr int kTPR = HD / 8;       // threads per row, one 16-byte vector (8 bf16) each
    constexpr int kRPW = 32 / kTPR;    // rows per warp pass
    constexpr int kUnroll = 4;         // passes whose loads are in flight together
    const int npad = a.n_kblk * 128;
    const long long rows = static_cast<long long>(a.BH) * npad;
    const int lane = threadIdx.x & 31;
    const int sub = lane % kTPR;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long base = warp_global * kRPW * kUnroll; base < rows; base += nwarps * kRPW * kUnroll) {
        uint4 ov[kUnroll], dv[kUnroll];
        float lv[kUnroll];
        long long rp[kUnroll];
        bool real[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            rp[u] = base + u * kRPW + lane / kTPR;
            const long long bh = rp[u] / npad;
            const int i = static_cast<int>(rp[u] - bh * npad);
            real[u] = rp[u] < rows && i < a.N;
            const long long r = bh * a.N + i;
            ov[u] = dv[u] = make_uint4(0u, 0u, 0u, 0u);
            lv[u] = -INFINITY;
            if (real[u]) {
                ov[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.o) + r * HD) + sub);
                dv[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.dout) + r * HD) + sub);
                if (sub == 0) lv[u] = __ldg(a.lse + r) * -1.4426950408889634f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t ow[4] = {ov[u].x, ov[u].y, ov[u].z, ov[u].w};
            const uint32_t dw[4] = {dv[u].x, dv[u].y, dv[u].z, dv[u].w};
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(__uint_as_float(ow[e] << 16), __uint_as_float(dw[e] << 16), acc);
                acc = fmaf(__uint_as_float(ow[e] & 0xffff0000u), __uint_as_float(dw[e] & 0xffff0000u), acc);
            }
#pragma unroll
            for (int off = kTPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (sub == 0 && rp[u] < rows) {
                a.delta[rp[u]] = real[u] ? acc : 0.f;
                a.nlse2[rp[u]] = lv[u];  // -inf for padding rows
            }
        }
    }
}

// ---------------------------------------------------------------------------
// dK / dV: one CTA per (head, 128-key tile j), looping over 128-row query
// tiles i (i >= j when causal).  Everything is computed transposed, keys on
// the MMA M dimension, so dK_j and dV_j accumulate in TMEM for the whole loop
// ("FlashAttention 1–4" §"FlashAttention-2": one thread block per K/V block,
// dK/dV kept on chip):
//   S^T  = K_j Q_i^T                 (TMEM, fp32)
//   dP^T = V_j dO_i^T                (TMEM, fp32)
//   P^T  = exp2(S^T * scale*log2e - lse_i * log2e)      (recomputed from lse)
//   dS^T = P^T * (dP^T - D_i)        (D = rowsum(dO * O) from the prep stage)
//   dV_j += P^T dO_i                 (P^T bf16 from TMEM, over S^T's columns)
//   dK_j += dS^T Q_i                 (dS^T bf16 from TMEM, over dP^T's columns)
// dQ is left to fa_bwd_dq_kernel: adding a 128 x d fp32 partial of dQ per
// (i, j) tile into global memory costs about as many SM cycles as the tile's
// MMAs on GB300 (reductions leave an SM at ~25 B/clk), so dQ is accumulated on
// chip by a kernel that owns the query tile instead.  With dQ gone dS^T is not
// needed in shared memory, and the 32 KB that held it give Q a third slot.
// MMA issue order per query tile: dP^T(i), dV(i), S^T(i+1), dK(i); S^T(i+1)
// only needs P^T(i) consumed by dV(i), so the compute warps find it ready
// when they finish dS^T(i).  Q_i is read until dK(i), dO_i only until dV(i),
// so Q has one more slot than dO.
// Epilogue: the compute warps stage bf16 dV and scale * dK, 128-byte
// swizzled, in the dO and Q slots of the item's last query tile (free once its
// dV and dK are done) and warp 3 writes them out with TMA tile stores
// (per-thread row stores of a 128-row tile measured ~12 B/clk, the CTA's
// slowest phase), handing the slots back to the dO and Q rings once the copies
// have read them.  K and V are released after the item's last S^T and dP^T,
// so the next item's K and V load while its last query tile is processed.
// Roles: warp 0 TMA loads, warp 1 MMA, warp 2 TMEM allocation, warp 3 TMA
// stores, warps 4-7 / 8-11 compute for query columns 0-63 / 64-127 of each tile.
// ---------------------------------------------------------------------------
constexpr int kBThreads = 384;
constexpr int kBCompute = 256;  // threads of warps 4..11; each arrives on the compute barriers
constexpr int kBBox = 128 * 64 * 2;

template <int HD>
struct BwdCfg {
    static constexpr int kTile = 128 * HD * 2;
    static constexpr int kBoxes = HD / 64;
    static constexpr int kQSlots = HD == 128 ? 3 : 4;
    static constexpr int kDoSlots = HD == 128 ? 2 : 3;
    static constexpr uint32_t kS = 0;    // S^T, then P^T (bf16) in columns [0,32) and [64,96)
    static constexpr uint32_t kDP = 128; // dP^T, then dS^T (bf16) the same way
    static constexpr uint32_t kDV = 256;
    static constexpr uint32_t kDK = 256 + HD;
    static constexpr uint32_t kTmemCols = 512;
};

template <int HD>
struct alignas(1024) BwdSmem {
    uint8_t k[BwdCfg<HD>::kTile];
    uint8_t v[BwdCfg<HD>::kTile];
    uint8_t q[BwdCfg<HD>::kQSlots][BwdCfg<HD>::kTile];
    uint8_t dout[BwdCfg<HD>::kDoSlots][BwdCfg<HD>::kTile];
    float nlse2[BwdCfg<HD>::kQSlots][128];   // -lse * log2(e), with the Q slot
    float delta[BwdCfg<HD>::kDoSlots][128];  // with the dO slot
    int item[2];                             // work items published by the loader (-1: none left)
    uint64_t item_full[2], item_empty[2];    // per queue slot: written / read by every role
    uint64_t kv_full;                        // K_j and V_j of the item landed (once per item)
    uint64_t k_free, v_free;                 // the item's last S^T / dP^T has read K / V (per item)
    uint64_t q_full[BwdCfg<HD>::kQSlots];    // Q tile and its lse * log2(e) landed
    uint64_t q_empty[BwdCfg<HD>::kQSlots];   // after dK(i); an item's last slot after its dK store
    uint64_t do_full[BwdCfg<HD>::kDoSlots];  // dO tile and its D landed
    uint64_t do_empty[BwdCfg<HD>::kDoSlots]; // dO tile and its D free: after dV(i) (an item's last
                                             // slot: after its dV store) and after every compute
                                             // thread has read D in its dS phase
    uint64_t p_ready[2];  // P^T for each thread's queries 0-31, then 32-63
    uint64_t s_full, dp_full, ds_ready, dkdv_done, drain;
    uint64_t out_staged;  // every compute thread has staged its dV / dK row (per item)
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(BwdSmem<128>) <= 232448, "backward d=128 shared memory exceeds 227 KB");
static_assert(sizeof(BwdSmem<64>) <= 232448, "backward d=64 shared memory exceeds 227 KB");

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32"
        " [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Work item t (fetch order) -> (head, key block).  Causal: head groups as in
// grouped_item; inside a group the key blocks with the most query tiles (small
// j) come first.  Keeping few heads in flight keeps their Q and dO in L2.
__device__ __forceinline__ void dkdv_item(const BwdArgs& a, int t, int& bh, int& j) {
    if (a.causal) {
        grouped_item(t, a.n_kblk, a.BH, a.group, a.group_last, bh, j);
    } else {
        bh = t / a.n_kblk;
        j = t % a.n_kblk;
    }
}

constexpr int kItemReaders = 2 + kBCompute;  // MMA thread, store thread, compute threads

__device__ __forceinline__ void bwd_timeout(const BwdArgs& a, volatile int* abort) {
    *abort = 1;
    atomicExch(a.status, kErrDeviceTimeout);
}

template <int HD>
__global__ void __launch_bounds__(kBThreads, 1)
fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                   const BwdArgs a) {
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
    const int n_items = a.BH * nq;

    if (threadIdx.x == 0) {
        sm.abort = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sm.item_full[s]), 1);
            mbar_init(smem_u32(&sm.item_empty[s]), kItemReaders);
        }
        mbar_init(smem_u32(&sm.kv_full), 1);
        mbar_init(smem_u32(&sm.k_free), 1);
        mbar_init(smem_u32(&sm.v_free), 1);
        for (int s = 0; s < Cfg::kQSlots; ++s) {
            mbar_init(smem_u32(&sm.q_full[s]), 1);
            mbar_init(smem_u32(&sm.q_empty[s]), 1);
        }
        for (int s = 0; s < Cfg::kDoSlots; ++s) {
            mbar_init(smem_u32(&sm.do_full[s]), 1);
            mbar_init(smem_u32(&sm.do_empty[s]), 1 + kBCompute);
        }
        mbar_init(smem_u32(&sm.s_full), 1);
        mbar_init(smem_u32(&sm.dp_full), 1);
        mbar_init(smem_u32(&sm.p_ready[0]), kBCompute);
        mbar_init(smem_u32(&sm.p_ready[1]), kBCompute);
        mbar_init(smem_u32(&sm.ds_ready), kBCompute);
        mbar_init(smem_u32(&sm.dkdv_done), 1);
        mbar_init(smem_u32(&sm.drain), 1);
        mbar_init(smem_u32(&sm.out_staged), kBCompute);
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
        // Per item: fetch its index and publish it to the other roles; then the
        // first query tile's Q and dO, K_j and V_j (each buffer once the previous
        // item's last S^T / dP^T has read it), and the remaining query tiles.  Q
        // and dO use rings indexed by the CTA's running tile count g, so one
        // item's tiles follow the previous item's.
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdo);
            int issued_q = 0, issued_do = 0, issued_kv = 0;
            bool ok = true;
            auto load_tile = [&](int bh, int i) -> bool {
                const size_t stat = (static_cast<size_t>(bh) * nq + i) * 128;
                const int qs = issued_q % Cfg::kQSlots;
                if (!mbar_wait(smem_u32(&sm.q_empty[qs]), ((issued_q / Cfg::kQSlots) & 1) ^ 1,
                               kWaitTimeoutNs, abort))
                    return false;
                if (FA_FAULT_INJECT) return true;
                const uint32_t qbar = smem_u32(&sm.q_full[qs]);
                mbar_arrive_expect_tx(qbar, Cfg::kTile + 512);
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.q[qs] + b * kBBox), &tq, qbar, b * 64, i * 128, bh);
                bulk_load(smem_u32(sm.nlse2[qs]), a.nlse2 + stat, 512, qbar);
                ++issued_q;
                const int ds = issued_do % Cfg::kDoSlots;
                if (!mbar_wait(smem_u32(&sm.do_empty[ds]), ((issued_do / Cfg::kDoSlots) & 1) ^ 1,
                               kWaitTimeoutNs, abort))
                    return false;
                const uint32_t dbar = smem_u32(&sm.do_full[ds]);
                mbar_arrive_expect_tx(dbar, Cfg::kTile + 512);
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.dout[ds] + b * kBBox), &tdo, dbar, b * 64, i * 128, bh);
                bulk_load(smem_u32(sm.delta[ds]), a.delta + stat, 512, dbar);
                ++issued_do;
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (k >= 2 && !(ok = mbar_wait(smem_u32(&sm.item_empty[slot]), ((k - 2) >> 1) & 1,
                                               kWaitTimeoutNs, abort)))
                    break;
                const unsigned t = atomicAdd(a.work + kWorkDkdv, 1u);
                const int item = t < static_cast<unsigned>(n_items) ? static_cast<int>(t) : -1;
                sm.item[slot] = item;
                mbar_arrive(smem_u32(&sm.item_full[slot]));
                if (item < 0) break;
                int bh, j;
                dkdv_item(a, item, bh, j);
                const int i_begin = a.causal ? j : 0;
                if (!(ok = load_tile(bh, i_begin))) break;
                const uint32_t kvbar = smem_u32(&sm.kv_full);
                if (k >= 1 && !(ok = mbar_wait(smem_u32(&sm.k_free), (k - 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                mbar_arrive_expect_tx(kvbar, 2 * Cfg::kTile);
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.k + b * kBBox), &tk, kvbar, b * 64, j * 128, bh);
                ++issued_kv;
                if (k >= 1 && !(ok = mbar_wait(smem_u32(&sm.v_free), (k - 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_load_3d(smem_u32(sm.v + b * kBBox), &tv, kvbar, b * 64, j * 128, bh);
                for (int i = i_begin + 1; ok && i < nq; ++i) ok = load_tile(bh, i);
            }
            if (!ok) bwd_timeout(a, abort);
            // Let every copy that was issued land before the CTA can exit.
            for (int s = 0; s < Cfg::kQSlots && s < issued_q; ++s) {
                const int last = s + Cfg::kQSlots * ((issued_q - 1 - s) / Cfg::kQSlots);
                mbar_wait_drain(smem_u32(&sm.q_full[s]), (last / Cfg::kQSlots) & 1, kWaitTimeoutNs);
            }
            for (int s = 0; s < Cfg::kDoSlots && s < issued_do; ++s) {
                const int last = s + Cfg::kDoSlots * ((issued_do - 1 - s) / Cfg::kDoSlots);
                mbar_wait_drain(smem_u32(&sm.do_full[s]), (last / Cfg::kDoSlots) & 1, kWaitTimeoutNs);
            }
            if (issued_kv > 0) mbar_wait_drain(smem_u32(&sm.kv_full), (issued_kv - 1) & 1, kWaitTimeoutNs);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (elect_one()) {
            constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T
            constexpr uint32_t id_kmn = idesc_bf16_f32(128, HD, 0, 1);  // dV, dK: A from TMEM
            const uint32_t k_addr = smem_u32(sm.k), v_addr = smem_u32(sm.v);
            // D[tmem] = A B^T with both operands K-major over the head dimension.
            auto gemm_kk = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr) {
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kBBox + (kk % 4) * 32;
                    umma_ss(tbase + d_col, sdesc_sw128(a_addr + off, 16, 1024),
                            sdesc_sw128(b_addr + off, 16, 1024), id_kk, kk > 0);
                }
            };
            // acc += A B with A (bf16, keys x queries) from TMEM columns a_col:
            // query columns 0-63 packed at [0,32), 64-127 at [64,96); B MN-major.
            auto gemm_tmem_a = [&](uint32_t d_col, uint32_t a_col, uint32_t b_addr, bool acc) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t col = a_col + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
                    umma_ts(tbase + d_col, tbase + col, sdesc_sw128(b_addr + kk * 2048, kBBox, 1024),
                            id_kmn, (acc || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            int g = 0;  // running query-tile count of this CTA (ring positions, barrier phases)
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!(ok = mbar_wait(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                const int item = sm.item[slot];
                mbar_arrive(smem_u32(&sm.item_empty[slot]));
                if (item < 0) break;
                int bh, j;
                dkdv_item(a, item, bh, j);
                const int niter = nq - (a.causal ? j : 0);
                // K_j, V_j of this item; the previous item's MMAs have all been issued
                // (one thread's MMAs run in order), so S^T(0) may overwrite its P^T
                if (!(ok = mbar_wait(smem_u32(&sm.kv_full), k & 1, kWaitTimeoutNs, abort))) break;
                // S^T(0); afterwards S^T(i+1) is issued inside iteration i
                if (!(ok = mbar_wait(smem_u32(&sm.q_full[g % Cfg::kQSlots]), (g / Cfg::kQSlots) & 1,
                                     kWaitTimeoutNs, abort)))
                    break;
                tc_fence_after();
                gemm_kk(Cfg::kS, k_addr, smem_u32(sm.q[g % Cfg::kQSlots]));
                umma_commit(smem_u32(&sm.s_full));
                if (niter == 1) umma_commit(smem_u32(&sm.k_free));  // the item's last S^T read K
                for (int it = 0; ok && it < niter; ++it, ++g) {
                    const int qs = g % Cfg::kQSlots, ds = g % Cfg::kDoSlots;
                    const uint32_t q_addr = smem_u32(sm.q[qs]), do_addr = smem_u32(sm.dout[ds]);
                    // dP^T(i) over dS^T(i-1): dK(i-1), which read it, was issued before.
                    if (!(ok = mbar_wait(smem_u32(&sm.do_full[ds]), (g / Cfg::kDoSlots) & 1,
                                         kWaitTimeoutNs, abort)))
                        break;
                    tc_fence_after();
                    gemm_kk(Cfg::kDP, v_addr, do_addr);
                    umma_commit(smem_u32(&sm.dp_full));
                    if (it + 1 == niter) umma_commit(smem_u32(&sm.v_free));  // the item's last dP^T read V
                    // dV += P^T dO in two parts: queries {0-31, 64-95} (k-steps 0, 1, 4, 5),
                    // each thread's first half of P^T, then {32-63, 96-127}.  The first of
                    // an item overwrites dV: the previous item's dV was read out of TMEM
                    // before its stores, and those before this item's K_j could load.
                    for (int part = 0; ok && part < 2; ++part) {
                        if (!(ok = mbar_wait(smem_u32(&sm.p_ready[part]), g & 1, kWaitTimeoutNs, abort)))
                            break;
                        tc_fence_after();
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int kk = (x >> 1) * 4 + part * 2 + (x & 1);
                            const uint32_t col = Cfg::kS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
                            umma_ts(tbase + Cfg::kDV, tbase + col,
                                    sdesc_sw128(do_addr + kk * 2048, kBBox, 1024), id_kmn,
                                    (it > 0 || part > 0 || x > 0) ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    // dO_i read; the item's last dO slot is released by the dV store
                    if (it + 1 < niter) umma_commit(smem_u32(&sm.do_empty[ds]));
                    // S^T(i+1) over P^T(i): dV(i) was issued before it.
                    if (it + 1 < niter) {
                        const int qs1 = (g + 1) % Cfg::kQSlots;
                        if (!(ok = mbar_wait(smem_u32(&sm.q_full[qs1]), ((g + 1) / Cfg::kQSlots) & 1,
                                             kWaitTimeoutNs, abort)))
                            break;
                        tc_fence_after();
                        gemm_kk(Cfg::kS, k_addr, smem_u32(sm.q[qs1]));
                        umma_commit(smem_u32(&sm.s_full));
                        if (it + 2 == niter) umma_commit(smem_u32(&sm.k_free));  // last S^T read K
                    }
                    if (!(ok = mbar_wait(smem_u32(&sm.ds_ready), g & 1, kWaitTimeoutNs, abort))) break;
                    tc_fence_after();
                    gemm_tmem_a(Cfg::kDK, Cfg::kDP, q_addr, it > 0);  // dK += dS^T Q
                    // Q_i read; the item's last Q slot is released by the dK store
                    if (it + 1 < niter) umma_commit(smem_u32(&sm.q_empty[qs]));
                }
                if (ok) umma_commit(smem_u32(&sm.dkdv_done));  // this item's dK, dV complete
            }
            if (!ok) bwd_timeout(a, abort);
            // Every MMA (and every commit before it) completes before the CTA leaves.
            umma_commit(smem_u32(&sm.drain));
            mbar_wait_drain(smem_u32(&sm.drain), 0, kWaitTimeoutNs);
        }
    } else if (warp == 3) {
        // ===================== dK / dV stores =====================
        // Per item: the staged dV (in the dO slot of the item's last query tile) and
        // dK (in its Q slot) go out with TMA tile stores, as two bulk groups; each
        // slot goes back to its ring as soon as its group has been read out of
        // shared memory (dV first: the dO ring has fewer slots).
        if (elect_one()) {
            tma_prefetch_desc(&tdk);
            tma_prefetch_desc(&tdv);
            bool ok = true;
            int g = 0;  // running query-tile count, as in the MMA warp
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!(ok = mbar_wait(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
                    break;
                const int item = sm.item[slot];
                mbar_arrive(smem_u32(&sm.item_empty[slot]));
                if (item < 0) break;
                int bh, j;
                dkdv_item(a, item, bh, j);
                g += nq - (a.causal ? j : 0);
                const int qs = (g - 1) % Cfg::kQSlots, ds = (g - 1) % Cfg::kDoSlots;
                if (!(ok = mbar_wait(smem_u32(&sm.out_staged), k & 1, kWaitTimeoutNs, abort))) break;
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_store_3d(&tdv, smem_u32(sm.dout[ds]) + b * kBBox, b * 64, j * 128, bh);
                bulk_commit_group();
                for (int b = 0; b < Cfg::kBoxes; ++b)
                    tma_store_3d(&tdk, smem_u32(sm.q[qs]) + b * kBBox, b * 64, j * 128, bh);
                bulk_commit_group();
                bulk_wait_group_read<1>();
                mbar_arrive(smem_u32(&sm.do_empty[ds]));
                bulk_wait_group_read<0>();
                mbar_arrive(smem_u32(&sm.q_empty[qs]));
            }
            if (!ok) bwd_timeout(a, abort);
            bulk_wait_group0();  // written out before the CTA leaves
        }
    } else if (warp >= 4) {
        // ===================== compute =====================
        const int wg = (warp - 4) >> 2;  // query-column half of S^T / dP^T, and column half of dK/dV
        const int wq = warp & 3;
        const int row = wq * 32 + lane;   // TMEM lane: key row of S^T/dP^T/dK/dV
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(wq * 32) << 16);
        const float sl2 = a.scale_log2;
        bool ok = true;
        int g = 0;  // running query-tile count of this CTA, as in the MMA warp
        for (int k = 0; ok; ++k) {
          const int slot = k & 1;
          if (!(ok = mbar_wait_warp(smem_u32(&sm.item_full[slot]), (k >> 1) & 1, kWaitTimeoutNs, abort)))
              break;
          const int item = sm.item[slot];
          mbar_arrive(smem_u32(&sm.item_empty[slot]));
          if (item < 0) break;
          int bh, j;
          dkdv_item(a, item, bh, j);
          const int i_begin = a.causal ? j : 0;
          const int niter = nq - i_begin;
          const bool row_valid = j * 128 + row < N;
          for (int it = 0; it < niter; ++it, ++g) {
            const int qs = g % Cfg::kQSlots, ds = g % Cfg::kDoSlots;
            const int i = i_begin + it;
            ok = mbar_wait_warp(smem_u32(&sm.s_full), g & 1, kWaitTimeoutNs, abort) &&
                 mbar_wait_warp(smem_u32(&sm.q_full[qs]), (g / Cfg::kQSlots) & 1, kWaitTimeoutNs,
                                abort);
            if (!ok) break;
            tc_fence_after();
            // P^T in two halves of this thread's 64 query columns; each half is
            // signalled as soon as it is stored so dV starts on it (the second
            // half's exponentials overlap the first half's MMAs).
            float p[64];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32(lane_addr + Cfg::kS + wg * 64, r0);
                tmem_ld32(lane_addr + Cfg::kS + wg * 64 + 32, r1);
                tmem_wait_ld();
                reg_fence(r0);
                reg_fence(r1);
                const uint32_t lse_addr = smem_u32(&sm.nlse2[qs][wg * 64]);
                const uint64_t sl2_pair = f2_pack(sl2, sl2);
                const bool diag = a.causal && i == j;
                // only the diagonal tile and key rows past the end need a mask
                const bool masked = diag || !row_valid;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    if (masked) {
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 l4 = ld_shared_f4(lse_addr + (part * 8 + c4) * 16);
                            const uint64_t nl[2] = {f2_pack(l4.x, l4.y), f2_pack(l4.z, l4.w)};
#pragma unroll
                            for (int e = 0; e < 4; e += 2) {
                                const int c = part * 32 + c4 * 4 + e;
                                const uint32_t s0 = part == 0 ? r0[c] : r1[c - 32], s1 = part == 0 ? r0[c + 1] : r1[c - 31];
                                const float2 x = f2_unpack(f2_fma(f2_pack_u(s0, s1), sl2_pair, nl[e >> 1]));
                                p[c] = ex2(x.x);
                                p[c + 1] = ex2(x.y);
                                // rows past the end, and on the diagonal tile queries before the key
                                if (!row_valid || wg * 64 + c < row) p[c] = 0.f;
                                if (!row_valid || wg * 64 + c + 1 < row) p[c + 1] = 0.f;
                            }
                        }
                    } else {
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 l4 = ld_shared_f4(lse_addr + (part * 8 + c4) * 16);
                            const uint64_t nl[2] = {f2_pack(l4.x, l4.y), f2_pack(l4.z, l4.w)};
#pragma unroll
                            for (int e = 0; e < 4; e += 2) {
                                const int c = part * 32 + c4 * 4 + e;
                                const uint32_t s0 = part == 0 ? r0[c] : r1[c - 32], s1 = part == 0 ? r0[c + 1] : r1[c - 31];
                                const float2 x = f2_unpack(f2_fma(f2_pack_u(s0, s1), sl2_pair, nl[e >> 1]));
                                p[c] = ex2(x.x);
                                p[c + 1] = ex2(x.y);
                            }
                        }
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(p[part * 32 + 2 * c], p[part * 32 + 2 * c + 1]);
                    // P^T over columns this thread read itself
                    tmem_st16(lane_addr + Cfg::kS + wg * 64 + part * 16, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(smem_u32(&sm.p_ready[part]));
                }
            }

            ok = mbar_wait_warp(smem_u32(&sm.dp_full), g & 1, kWaitTimeoutNs, abort) &&
                 mbar_wait_warp(smem_u32(&sm.do_full[ds]), (g / Cfg::kDoSlots) & 1, kWaitTimeoutNs,
                                abort);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_addr = smem_u32(&sm.delta[ds][wg * 64]);
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
                tmem_ld32(lane_addr + Cfg::kDP + wg * 64 + h * 32, r);
                tmem_wait_ld();
                reg_fence(r);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 d4 = ld_shared_f4(d_addr + (h * 32 + c4 * 4) * 4);
                    const uint64_t dd[2] = {f2_pack(d4.x, d4.y), f2_pack(d4.z, d4.w)};
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int c = c4 * 4 + e;
                        const float2 ds = f2_unpack(f2_mul(f2_pack(p[h * 32 + c], p[h * 32 + c + 1]),
                                                           f2_sub(f2_pack_u(r[c], r[c + 1]), dd[e >> 1])));
                        pk[h * 16 + c4 * 2 + (e >> 1)] = pack_bf16x2(ds.x, ds.y);
                    }
                }
            }
            // D of this slot has been read: with the dV MMA's commit (or the dV
            // store, for an item's last tile) this frees the slot for the next dO
            // tile and its D.
            mbar_arrive(smem_u32(&sm.do_empty[ds]));
            // dS^T over the first 32 of the 64 dP^T columns this thread read
            tmem_st32(lane_addr + Cfg::kDP + wg * 64, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.ds_ready));
          }
          if (!ok) break;
          if (!(ok = mbar_wait_warp(smem_u32(&sm.dkdv_done), k & 1, kWaitTimeoutNs, abort))) break;
          tc_fence_after();
          {
                // this thread's row of columns [wg * d/2, (wg + 1) * d/2) of dV (into
                // the dO slot of the item's last query tile) and dK (into its Q slot),
                // free since every MMA of the item is done: 64-column boxes of 128-byte
                // rows, 16-byte chunk c of row r at position c ^ (r % 8)
                constexpr int kHalf = HD / 2;
                const int col0 = wg * kHalf;
                const uint32_t row_off = static_cast<uint32_t>((col0 / 64) * kBBox + row * 128);
                const uint32_t dv_row = smem_u32(sm.dout[(g - 1) % Cfg::kDoSlots]) + row_off;
                const uint32_t dk_row = smem_u32(sm.q[(g - 1) % Cfg::kQSlots]) + row_off;
#pragma unroll 1
                for (int c = 0; c < kHalf; c += 32) {
                    uint32_t rv[32], rk[32];
                    tmem_ld32(lane_addr + Cfg::kDV + col0 + c, rv);
                    tmem_ld32(lane_addr + Cfg::kDK + col0 + c, rk);
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
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int chunk = ((col0 % 64) + c) / 8 + m;
                        const uint32_t sw = static_cast<uint32_t>((chunk ^ (row & 7)) << 4);
                        st_shared_v4(dv_row + sw, pv[4 * m], pv[4 * m + 1], pv[4 * m + 2], pv[4 * m + 3]);
                        st_shared_v4(dk_row + sw, pkk[4 * m], pkk[4 * m + 1], pkk[4 * m + 2], pkk[4 * m + 3]);
                    }
                }
                // the TMEM reads above come before the next item's first dV / dK, which
                // wait for this thread's next p_ready / ds_ready arrivals
                tc_fence_before();
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&sm.out_staged));
          }
        }
        if (!ok && lane == 0) bwd_timeout(a, abort);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tbase, Cfg::kTmemCols);
    }
}

template <int HD>
cudaError_t launch_bwd_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                              const BwdArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(BwdSmem<HD>);
    cudaError_t e = smem_limit_once<fa_bwd_dkdv_kernel<HD>>(static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // persistent: one CTA per multiprocessor, work items handed out by a counter
    // (zeroed here, or by the prep kernel just before inside fa_bwd)
    if (!a.counters_zeroed &&
        (e = cudaMemsetAsync(a.work + kWorkDkdv, 0, sizeof(unsigned), stream)) != cudaSuccess)
        return e;
    const long long items = static_cast<long long>(a.n_kblk) * a.BH;
    const unsigned grid = static_cast<unsigned>(items < a.sms ? items : a.sms);
    fa_bwd_dkdv_kernel<HD><<<grid, kBThreads, smem, stream>>>(tq, tk, tv, tdo, tdk, tdv, a);
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
    const long long rows = static_cast<long long>(a.BH) * a.n_kblk * 128;
    // 8 warps x 4 passes of 32/(d/8) rows per CTA, up to 8 CTAs per SM
    const int grid = grid_for(rows, 8 * (32 / (d / 8)) * 4, 8 * (a.sms > 0 ? a.sms : 1));
    if (d == 64)
        fa_bwd_prep_kernel<64><<<grid, 256, 0, stream>>>(a);
    else
        fa_bwd_prep_kernel<128><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t stream) {
    if (d == 64) return launch_bwd_dkdv_t<64>(tq, tk, tv, tdo, tdk, tdv, a, stream);
    return launch_bwd_dkdv_t<128>(tq, tk, tv, tdo, tdk, tdv, a, stream);
}

}  // namespace fa
