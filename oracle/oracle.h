/*
 * oracle.h -- fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the independent reference that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition; every function materialises the score
 * row S[i,:] and the probability row P[i,:] of one query at a time):
 *
 *   s_j   = scale * sum_c Q[i,c] K[j,c]         for j in J_i
 *   J_i   = {0..N-1}, or {0..i} when causal (a future key gets score -inf)
 *   m     = max_j s_j,  e_j = exp(s_j - m),  l = sum_j e_j,  P[i,j] = e_j / l
 *   O[i,:] = sum_j P[i,j] V[j,:]                lse[i] = m + ln(l)
 *
 * Sources: "GPU 与 TPU：让硬件不再是黑魔法" (CS336 Lecture 5 notes) §11.1 and
 * §11.4 (O and the saved logsumexp L = m + log l); "谁偷走了 5090 的算力和显存"
 * §3.2 (eager attention, future positions set to -inf); "FlashAttention 1–4:
 * How IO-Awareness Reshaped the Attention Kernel" §"Why attention is memory-bound"
 * (S = QK^T/sqrt(d), P = softmax(S), O = PV).
 *
 * The backward formulas are not printed on the pages (they only say that P is
 * rebuilt from the saved statistics and the gradients follow).  They are derived
 * from the definition above with the softmax Jacobian:
 *   dV[j,:] = sum_i P[i,j] dO[i,:]       dP[i,j] = sum_c dO[i,c] V[j,c]
 *   D_i     = sum_c dO[i,c] O[i,c]       dS[i,j] = P[i,j] (dP[i,j] - D_i)
 *   dQ[i,:] = scale sum_j dS[i,j] K[j,:] dK[j,:] = scale sum_i dS[i,j] Q[i,:]
 *
 * Layouts: every tensor is [BH, N, d] row-major (BH = batch * heads), lse is
 * [BH, N].  Inputs are either fp64 or bfloat16 bit patterns (uint16); a bf16
 * value converts to fp64 exactly.  Outputs are always fp64.
 *
 * Return value: 0 on success, -1 on a bad argument, -2 on allocation failure.
 */
#ifndef FA_ORACLE_H
#define FA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F64 = 0, ORACLE_BF16 = 1 };

/* Online softmax on one row of n given scores split into key blocks of `block`
 * scores (block >= 1), carrying the running max m, the running sum l and the
 * unnormalised weighted sum u (length dv) of the n value rows v[n][dv]
 * (v may be NULL when dv == 0).  Follows the recurrence of "07 GPU、资源估算与
 * FlashAttention" §7.8 and "CS336 Lecture 5 notes" §11.3. */
int oracle_online_row(const double* s, const double* v, long n, long dv, long block,
                      double* m_out, double* l_out, double* u_out);

/* Forward pass by the definition, for the heads listed in bh_list (n_bh of them;
 * bh_list == NULL means all BH heads in order).  o is [n_bh, N, d], lse [n_bh, N]
 * (either may be NULL). */
int oracle_fwd(const void* q, const void* k, const void* v, int dtype,
               long BH, long N, long d, double scale, int causal,
               const int64_t* bh_list, long n_bh,
               double* o, double* lse, int nthreads);

/* Forward pass for selected query rows only: rows is [BH][nrows] (row indices
 * per head); o_rows is [BH, nrows, d], lse_rows [BH, nrows]. */
int oracle_fwd_rows(const void* q, const void* k, const void* v, int dtype,
                    long BH, long N, long d, double scale, int causal,
                    const int64_t* rows, long nrows,
                    double* o_rows, double* lse_rows, int nthreads);

/* Forward pass in the tiled order with the online recurrence: query blocks of
 * block_q rows, key/value blocks of block_k rows (the loop nest of "CS336
 * Lecture 5 notes" §11.4).  Used only to show that the blockwise recurrence and
 * the one-shot definition agree. */
int oracle_fwd_blockwise(const void* q, const void* k, const void* v, int dtype,
                         long BH, long N, long d, double scale, int causal,
                         long block_q, long block_k,
                         double* o, double* lse, int nthreads);

/* Backward pass by the derived formulas above, for the heads in bh_list (NULL =
 * all).  The oracle uses its own fp64 P, O and lse.  dq, dk, dv are
 * [n_bh, N, d]; o_out / lse_out (optional) receive the oracle's own forward. */
int oracle_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype,
               long BH, long N, long d, double scale, int causal,
               const int64_t* bh_list, long n_bh,
               double* dq, double* dk, double* dv,
               double* o_out, double* lse_out, int nthreads);

/* Backward for selected rows of every head, by the same formulas as
 * oracle_bwd: dq_rows [BH, nq, d] holds dQ of the query rows qrows [BH][nq];
 * dk_rows, dv_rows [BH, nk, d] hold dK and dV of the key rows krows [BH][nk]
 * (nq or nk may be 0, with NULL arrays).  dQ of row i needs only row i; dK and
 * dV of key row j sum over every query row that sees key j, so the statistics
 * m, l and D = dO . O of those rows (all rows, or rows i >= j when causal) are
 * computed first.  The values equal oracle_bwd's for the same rows. */
int oracle_bwd_rows(const void* q, const void* k, const void* v, const void* dout, int dtype,
                    long BH, long N, long d, double scale, int causal,
                    const int64_t* qrows, long nq, const int64_t* krows, long nk,
                    double* dq_rows, double* dk_rows, double* dv_rows, int nthreads);

/* Number of threads the oracle uses when asked for nthreads <= 0. */
int oracle_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif
