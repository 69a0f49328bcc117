/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V,   lse = per-row logsumexp,
 *
 * as one fused tiled kernel that never writes the N x N score or probability
 * matrix to memory ("GPU 与 TPU：让硬件不再是黑魔法" (CS336 Lecture 5 notes)
 * §11.4; "FlashAttention 1–4: How IO-Awareness Reshaped the Attention Kernel"
 * §"FlashAttention (v1)" and §"FlashAttention-2"), and the backward pass that
 * rebuilds the probabilities from the saved logsumexp (CS336 Lecture 5 notes
 * §11.5 (3): P = exp(S - L)).
 *
 * Common conventions
 *  - Tensors q, k, v, o, dout, dq, dk, dv: bfloat16, contiguous [B, H, N, d]
 *    row-major (d innermost), passed as untyped device pointers, 16-byte aligned.
 *  - lse: fp32 [B, H, N], natural logarithm of the row's sum of
 *    exp(scale * q.k) over the visible keys (L = m + log l).
 *  - d (head dimension) is 64 or 128; N >= 1 (any length, tails are masked);
 *    B, H >= 1; B*H*N*d < 2^31.  scale is finite and > 0 (callers usually
 *    pass 1/sqrt(d)); causal is 0 or 1 (key j visible to query i iff j <= i).
 *  - Every pointer is caller-owned device memory; the library keeps no pointer
 *    after a call returns and allocates no device memory per call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t, 0 = legacy default
 *    stream) and may be issued from several host threads.
 *  - Argument errors are returned before anything is launched.  A failed launch
 *    returns FA_ERR_CUDA.  Every wait inside the kernels is bounded: a kernel
 *    that gives up records FA_ERR_DEVICE_TIMEOUT in a device status word that
 *    fa_sync_status() reports.  Nothing is printed and nothing aborts.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, non-finite scale ... */
    FA_ERR_UNSUPPORTED = 2,   /* head dim not 64/128, or no sm_103 device     */
    FA_ERR_MISALIGNED = 3,    /* a tensor pointer is not 16-byte aligned      */
    FA_ERR_WORKSPACE = 4,     /* backward workspace missing or too small      */
    FA_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed            */
    FA_ERR_DEVICE_TIMEOUT = 6 /* a kernel wait expired (see fa_sync_status)   */
} fa_status;

/* Forward pass.  Writes o (bf16 [B,H,N,d]) and lse (fp32 [B,H,N]).
 * Steps: scores S = scale*Q K^T tile by tile on the tensor cores, online
 * softmax with a running max m and running sum l per row, unnormalised output
 * accumulator rescaled when the max moves, one normalisation O = acc / l at the
 * end, lse = m + ln l ("FlashAttention 1–4" §"FlashAttention (v1)" recurrence;
 * "07 GPU、资源估算与 FlashAttention" §7.8).  Work items are (head, 256-row
 * query block) pairs; one CTA per multiprocessor runs them back to back in a
 * static schedule computed on the host (heaviest causal blocks first, greedy
 * over the CTAs) and passed in the launch parameters, so the call needs no
 * workspace and concurrent calls share nothing.  fa_fwd_ws below gives the
 * same results with a work counter instead.  `stream` is a cudaStream_t. */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, void* stream);

/* fa_fwd with a workspace holding a work counter: one CTA per multiprocessor
 * takes (head, 256-row query block) items from the counter until none are
 * left (dynamic instead of fa_fwd's static schedule).  workspace:
 * caller-owned device memory of at least fa_fwd_workspace_size() bytes,
 * 256-byte aligned, contents on entry irrelevant; two calls that overlap on the
 * GPU must not share one.  NULL behaves as fa_fwd.  A workspace that is too
 * small or misaligned returns FA_ERR_WORKSPACE.  Results are bitwise equal to
 * fa_fwd's. */
int fa_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int N, int d, float scale, int causal, void* workspace,
              size_t workspace_bytes, void* stream);

/* Bytes of device workspace fa_fwd_ws uses: a 256-byte slot for its work
 * counter (the sizes do not change it; 0 for invalid sizes). */
size_t fa_fwd_workspace_size(int B, int H, int N, int d);

/* Bytes of device workspace fa_bwd needs for these sizes: two fp32 row
 * statistics, D = rowsum(dO * O) and -lse * log2(e), each [B*H, N rounded up to
 * a multiple of 128] and rounded up to 256 bytes, then 256 bytes for the work
 * counters of the dK/dV and dQ kernels (d does not change it).
 * The statistics are those of the backward that rebuilds P from the saved
 * logsumexp ("GPU 与 TPU：让硬件不再是黑魔法" (CS336 Lecture 5 notes) §11.5 (3):
 * P = exp(S - L)): -L log2(e) makes the exponent of P one fused multiply-add,
 * and D_i = sum_c dO[i,c] O[i,c] is the per-row term of the softmax Jacobian,
 * dS = P * (dP - D), that the pages leave to the reader.  0 for non-positive
 * sizes. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/* Backward pass.  Inputs q, k, v, o, lse (as written by fa_fwd) and dout
 * (dL/dO); outputs dq, dk, dv (bf16 [B,H,N,d]).  workspace: caller-owned
 * device memory of at least fa_bwd_workspace_size() bytes, 256-byte aligned;
 * its contents on entry do not matter.  Runs fa_bwd_prep, fa_bwd_main and
 * fa_bwd_dq in order on `stream`.
 * The pages state only that P is recomputed from Q, K and the saved L and that
 * the gradients follow; the formulas used are the softmax Jacobian:
 *   dV = P^T dO, dP = dO V^T, D = rowsum(dO * O), dS = P * (dP - D),
 *   dQ = scale * dS K, dK = scale * dS^T Q. */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv,
           int B, int H, int N, int d, float scale, int causal,
           void* workspace, size_t workspace_bytes, void* stream);

/* The three stages of fa_bwd, exposed so a caller can time or overlap them.
 * prep: D = rowsum(dO * O) and -lse * log2(e) into the workspace.
 * main: per key/value tile, recompute S and P = exp(S - lse) and accumulate
 *       dV and dK on chip; writes dk, dv.
 * dq:   per query tile, recompute S, P and dP = dO V^T and accumulate
 *       dQ = scale * dS K on chip; writes dq.
 * main and dq both read D from the workspace (written by prep) and nothing
 * else of each other, so they may run in either order or concurrently on
 * two streams once prep has finished.  Each takes its work items from its own
 * counter in the workspace, so two calls of the same stage must not overlap
 * on one workspace.  Arguments mean the same as for fa_bwd. */
int fa_bwd_prep(const void* o, const void* dout, const float* lse, int B, int H, int N, int d,
                void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_main(const void* q, const void* k, const void* v, const float* lse,
                const void* dout, void* dk, void* dv,
                int B, int H, int N, int d, float scale, int causal,
                void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_dq(const void* q, const void* k, const void* v, const float* lse,
              const void* dout, void* dq,
              int B, int H, int N, int d, float scale, int causal,
              void* workspace, size_t workspace_bytes, void* stream);

/* Backward pass for callers that cannot allocate device memory: code that runs
 * where cudaMalloc is unavailable or not allowed, such as inside a custom
 * allocator's own callbacks, a service that must keep a fixed device-memory
 * footprint after start-up, or a plug-in whose host framework owns every
 * allocation.  (The pages have no counterpart: this is a packaging choice of
 * this library.)  Same arguments, results and errors as fa_bwd, minus the workspace: the
 * scratch (fa_bwd_workspace_size bytes) lives in one fixed array of 64 MiB +
 * 256 bytes of library device memory, so nothing is allocated.  The checks run
 * in fa_bwd's order: null pointers and bad sizes (FA_ERR_INVALID_ARG,
 * FA_ERR_UNSUPPORTED) first, then the scratch limit: sizes whose workspace
 * exceeds it (more than 2^23 rows B*H*N after rounding N up to a multiple of
 * 128) return FA_ERR_WORKSPACE, then alignment (FA_ERR_MISALIGNED); all before
 * any device call.  The first call on a device looks up the array's device address with
 * that device current; make that first call before any stream capture.  Every
 * call on a device shares the array: calls whose work overlaps on the GPU
 * (other streams, unordered host threads) race on it. */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, float scale, int causal, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 forward ("FlashAttention 1–4" §"FlashAttention-3", paragraph "FP8 with
 * block quantization and incoherent processing").  Head dimension 128 only.
 *
 * Two calls: fa_fp8_quantize turns bf16 q, k, v into E4M3 codes with one fp32
 * scale per 128-row tile (value = code * scale, scale = amax / 448 over the
 * tile), optionally after rotating every row of Q and K by the same orthogonal
 * M = diag(s) H / sqrt(128) (s = random signs, H = Sylvester Hadamard matrix),
 * which leaves Q K^T unchanged; fa_fwd_fp8 then runs attention on the codes
 * with FP8 tensor-core products and writes o (bf16) and lse (fp32) with the
 * meanings of fa_fwd.  Inside, the probabilities P are also rounded to E4M3
 * (after multiplying by 16 and by V's per-tile scale over its largest per-tile
 * scale) for the P V product; the row sums and lse use fp32 P.  The running
 * max is raised when a tile's max exceeds it by more than 4 (log2 units), so
 * the largest rounded weight is 256, inside E4M3's range.
 *
 * Workspace (caller-owned device memory, 256-byte aligned, at least
 * fa_fp8_workspace_size bytes).  With BH = B*H, T = ceil(N / 128) and
 * npad = 128 T, it holds these segments in order, each starting on a 256-byte
 * boundary:
 *   q8   uint8 [BH, npad, 128]  E4M3 codes of (rotated) Q; rows >= N are 0
 *   k8   uint8 [BH, npad, 128]  E4M3 codes of (rotated) K
 *   vt8  uint8 [BH, 128, npad]  E4M3 codes of V transposed: byte (b, c, 128 t + i)
 *                               is V row 128 t + key(i), column c, where for
 *                               i = 64 h + 16 x + 2 w + e (h, e < 2, x < 4, w < 8)
 *                               key(i) = 64 h + 8 w + 2 x + e
 *   sq, sk, sv  fp32 [BH, T]    per-tile scales of Q, K, V
 *   vfold fp32 [BH, T]          sv / vmax
 *   vmax  fp32 [BH]             largest sv of the head
 *   amax  fp32 [4]              per-tensor |x| maxima of Q, K, V (FA_FP8_PER_TENSOR)
 * --------------------------------------------------------------------------- */
#define FA_FP8_ROTATE 1     /* rotate Q and K rows by diag(s) H / sqrt(128) */
#define FA_FP8_PER_TENSOR 2 /* one scale per tensor (the pages' baseline) instead of per tile */

/* Bytes of FP8 workspace for these sizes (0 for sizes the FP8 path does not
 * take: d != 128, non-positive sizes, B*H > 65535, or B*H*128*ceil(N/128)*128
 * >= 2^31). */
size_t fa_fp8_workspace_size(int B, int H, int N, int d);

/* Quantize q, k, v (bf16 [B,H,N,128]) into the workspace.  signs: host array
 * of 4 uint32 words, bit j (word j/32, bit j%32) set means s_j = -1; read
 * during the call, may be NULL when FA_FP8_ROTATE is not in flags.  flags: an
 * OR of FA_FP8_ROTATE and FA_FP8_PER_TENSOR.  Errors: FA_ERR_UNSUPPORTED for
 * d != 128 or B*H > 65535, FA_ERR_WORKSPACE for a missing, misaligned or small workspace,
 * FA_ERR_INVALID_ARG for unknown flags or a NULL signs with FA_FP8_ROTATE. */
int fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    const unsigned int* signs, int flags, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Attention on a workspace that fa_fp8_quantize filled for the same B, H, N, d
 * (on the same stream, or ordered before this call).  Writes o (bf16
 * [B,H,N,128]) and lse (fp32 [B,H,N]); scale and causal as for fa_fwd. */
int fa_fwd_fp8(const void* workspace, size_t workspace_bytes, void* o, float* lse,
               int B, int H, int N, int d, float scale, int causal, void* stream);

/* Synchronises `stream`, then returns and clears the device status word of the
 * current device: FA_OK, or FA_ERR_DEVICE_TIMEOUT if any kernel gave up on a
 * wait since the last call, or FA_ERR_CUDA if the synchronisation failed. */
int fa_sync_status(void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */
