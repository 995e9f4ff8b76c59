/*
 * qlinear.h - C ABI of libqlinear.so: weight-only quantized linear layers over
 * MLX-style affine weights (4, 6 or 8 bits, group 64) kept as stored, for GB300
 * (sm_103a).
 *
 * Sources (TensorFold pull requests, cited by page title and section):
 *   [P1696] PR #1696, LFM3 on Intel Iris Xe (later revision), "What it adds":
 *           MLX 4-bit group 64 "as stored"; N-row matvecs that sum each row as the
 *           one-row kernels do; decode fuses w1 + w3 + SwiGLU and the four attention
 *           matvecs; "Prompt GEMM": an fma chain per 64-wide k block, blocks added
 *           in order, so a row's sum does not depend on how the prompt is cut.
 *   [P1514] PR #1514, LFM3-1.7B on Apple Metal, "What changes": MLX 4/6/8-bit
 *           checkpoints; paired FFN projections keep their retained rounding
 *           boundaries.
 *
 * Weight layout (the pages print none; this is the stated reading): W is [n, k],
 * k contiguous.  Row i of `wq` is a little-endian bit stream of k*bits/32 uint32
 * words; value j of the row is the unsigned field at bits [bits*j, bits*j + bits)
 * (for 4 bits: nibble j%8 of word j/8, low nibble first; for 6 bits a field may
 * straddle two words).  `scales` and `biases` are bf16 bit patterns [n, k/64];
 * the dequantized weight is w[i][j] = scales[i][j/64] * q[i][j] + biases[i][j/64].
 *
 * Conventions for every call:
 *   - every pointer is a DEVICE pointer owned by the caller; the library keeps no
 *     reference to it after the call is enqueued;
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); every call is
 *     asynchronous and enqueues its kernels on `stream`; nothing synchronizes
 *     except qlinear_last_error();
 *   - bf16 values are passed as their uint16_t bit patterns; outputs are float32
 *     unless stated otherwise;
 *   - activations x are row-major [rows, k] with row stride `ldx` elements;
 *     outputs are row-major [rows, n] with row stride `ldy` elements;
 *   - `wq` and `x` must be 16-byte aligned and `ldx` a multiple of 8;
 *   - return value: QL_OK (0) or a negative QL_ERR_* code; arguments are checked
 *     on the host before anything is enqueued, so an error return enqueues nothing
 *     (except QL_ERR_LAUNCH, reported after a failed launch);
 *   - results are deterministic: the same inputs give the same bits, and the
 *     summation order of each output is a function of k (and bits) only.
 *
 * Tolerance against the float64 definition (per output):
 *   |y - y64| <= 1e-5 * sum_j |w[i][j] * x[j]| + 1e-6.
 */
#ifndef QLINEAR_H
#define QLINEAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  QL_OK = 0,
  QL_ERR_NULL = -1,     /* a required pointer is NULL */
  QL_ERR_SHAPE = -2,    /* n <= 0, k <= 0, k % 64 != 0, k too large, m < 0, or shapes that must match do not */
  QL_ERR_BITS = -3,     /* bits not in {4, 6, 8}, or the fused weights differ in bits */
  QL_ERR_GROUP = -4,    /* group != 64 */
  QL_ERR_ROWS = -5,     /* rows outside 1..16 */
  QL_ERR_ALIGN = -6,    /* wq/x not 16-byte aligned, ldx % 8 != 0, or a leading dimension too small */
  QL_ERR_ARCH = -7,     /* the current device is not compute capability 10.3 (sm_103) */
  QL_ERR_LAUNCH = -8,   /* the kernel launch failed (cudaGetLastError after launch) */
  QL_ERR_TIMEOUT = -9,  /* a bounded device-side wait gave up (reported by qlinear_last_error) */
  QL_ERR_CUDA = -10,    /* another CUDA runtime error (device query, tensor-map encoding) */
  QL_ERR_NOMEM = -11,   /* the library could not allocate its scratch buffer */
  QL_ERR_TOO_LARGE = -12 /* the problem does not fit the fixed scratch of qlinear_pgemm_noalloc */
};

/* One quantized weight matrix, as stored.  All pointers are device pointers. */
typedef struct ql_weight {
  const uint32_t *wq;     /* [n, k*bits/32] packed codes, 16-byte aligned                     */
  const uint16_t *scales; /* [n, k/64] bf16 bits                                               */
  const uint16_t *biases; /* [n, k/64] bf16 bits                                               */
  int32_t n;              /* output channels (rows of W), >= 1                                  */
  int32_t k;              /* input channels, multiple of 64, <= 65536                           */
  int32_t bits;           /* 4, 6 or 8                                                          */
  int32_t group;          /* must be 64                                                         */
} ql_weight;

/*
 * qlinear_mv - decode matvec, one activation row: y[i] = sum_j w[i][j] x[j].
 * [P1696] "What it adds" (decode keeps qmv).  Exactly qlinear_mv_rows with rows = 1.
 *   x: bf16 [k]; y: float [n].
 */
int qlinear_mv(const ql_weight *w, const uint16_t *x, float *y, void *stream);

/*
 * qlinear_mv_rows - N-row decode matvec for 1..16 stream rows sharing one weight
 * pass: y[r][i] = sum_j w[i][j] x[r][j].
 * [P1696] "What it adds": streams share a decode step through N-row matvecs that
 * sum each row as the one-row kernels do.  Row r of the result is bit-equal to
 * qlinear_mv on x[r] alone, for every rows in 1..16.
 *   x: bf16 [rows, ldx] (ldx >= k); y: float [rows, ldy] (ldy >= n).
 */
int qlinear_mv_rows(const ql_weight *w, const uint16_t *x, int32_t rows, int64_t ldx,
                    float *y, int64_t ldy, void *stream);

/*
 * qffn_swiglu_mv - fused FFN gate/up decode step: h[r][i] = bf16(silu(a) * c) with
 * a = (w1 x[r])[i], c = (w3 x[r])[i], silu(t) = t / (1 + exp(-t)) in float32, rounded
 * to bf16 (nearest even) - the retained rounding boundary before the down projection.
 * [P1696] "What it adds" (decode fuses w1 + w3 + SwiGLU); [P1514] "What changes".
 * One weight pass over w1 and w3.  a and c are bit-equal to qlinear_mv_rows(w1/w3)
 * and h is bit-equal to qswiglu() applied to those.
 *   w1, w3: same n, k, bits; x: bf16 [rows, ldx]; h: bf16 bits [rows, ldh] (ldh >= n).
 */
int qffn_swiglu_mv(const ql_weight *w1, const ql_weight *w3, const uint16_t *x, int32_t rows,
                   int64_t ldx, uint16_t *h, int64_t ldh, void *stream);

/*
 * qattn_proj_mv - the four attention projections (q, k, v, gate) of one activation
 * in ONE launch.  [P1696] "What it adds" (decode fuses the four attention matvecs).
 * Outputs are dense row-major [rows, n_i]; each is bit-equal to qlinear_mv_rows on
 * that weight alone.
 *   wq, wk, wv, wg: same k and bits, any n; x: bf16 [rows, ldx].
 */
int qattn_proj_mv(const ql_weight *wq, const ql_weight *wk, const ql_weight *wv,
                  const ql_weight *wg, const uint16_t *x, int32_t rows, int64_t ldx,
                  float *q, float *k, float *v, float *g, void *stream);

/*
 * qlinear_pgemm - prompt-window GEMM: Y[m][i] = sum_j w[i][j] X[m][j] for m rows.
 * [P1696] "What it adds" > "Prompt GEMM": each output is an fp32 chain over 64-wide
 * k blocks added in order, so a row's result does not depend on how the prompt is
 * cut into windows.  Here: for every block b the tensor cores form the exact-code
 * partial P_b = sum_{j in b} q[i][j] X[m][j] (codes converted exactly to bf16,
 * fp32 accumulation), the chain y = fma(scale_b, P_b, y) runs over b = 0..k/64-1 in
 * order, and the bias term sum_b bias_b * S_b (S_b = sum_{j in b} X[m][j], split
 * exactly into three bf16 parts) is added last.  Every row depends only on its own
 * X row: row m of any window equals row m of the whole prompt, bit for bit.
 *   X: bf16 [m, ldx] (16-byte aligned, ldx % 8 == 0); Y: float [m, ldy] (ldy >= n).
 *   m may be 0: then nothing is checked beyond the weight and nothing is enqueued
 *   (X and Y may be NULL).  Uses a library-owned device scratch buffer of
 *   m * round_up(3*k/64, 64) bf16 values for the split row sums and, when m >= 2048,
 *   two more of n * (k + round_up(3*k/64, 64)) bf16 values into which the codes are
 *   converted once per call (exactly the values the kernel converts for smaller m, so
 *   the result is the same bits either way); such calls alternate between the two, so
 *   that a call's conversion may run on the SMs the previous call's GEMM leaves idle
 *   in its last tiles.  All are allocated with cudaMalloc on first need per device and
 *   grown on demand (growth synchronizes the device); calls on one device must be
 *   ordered on one stream because they share them.  A kernel the caller launches
 *   between two calls with programmatic dependent launch must wait for the kernel
 *   before it (griddepcontrol.wait) before it ends, as the library's own kernels do.
 *   QL_ERR_TOO_LARGE if m * k/64 >= 2^31.
 */
int qlinear_pgemm(const ql_weight *w, const uint16_t *X, int32_t m, int64_t ldx, float *Y,
                  int64_t ldy, void *stream);

/*
 * qlinear_pgemm_multi - qlinear_pgemm for nw weights that read the same X (a layer's
 * q/k/v/gate projections, or its w1 and w3): Y[i] = X w[i]^T for i < nw, each bit-equal to
 * qlinear_pgemm(w[i], X, ...) on its own.  [P1696] "What it adds": decode fuses the four
 * attention matvecs (qattn_proj_mv) and w1 + w3 (qffn_swiglu_mv); this is the prompt-window
 * counterpart.  Every call on X forms the split row sums S_b of X; here they are formed
 * once for all nw weights, then each weight's GEMM (and, from 2048 rows on, its code
 * conversion) runs in turn.
 *   w: nw weight pointers (1 <= nw <= 16), all with the same k; X as for qlinear_pgemm;
 *   Y[i]: float [m, ldy[i]] with ldy[i] >= w[i]->n (4-byte aligned).  The output buffers
 *   must not overlap X or each other.  m may be 0 (nothing enqueued).  Scratch, stream
 *   ordering and errors as qlinear_pgemm; QL_ERR_SHAPE if nw is out of range or the k
 *   differ.
 */
int qlinear_pgemm_multi(const ql_weight *const *w, int32_t nw, const uint16_t *X, int32_t m, int64_t ldx,
                        float *const *Y, const int64_t *ldy, void *stream);

/*
 * qlinear_pgemm_noalloc - qlinear_pgemm for callers that cannot allocate device
 * memory when they call: code whose device memory belongs to another allocator or
 * is held to a fixed budget, and code that must not pay the device-wide
 * synchronization of growing qlinear_pgemm's scratch buffer (which frees and
 * reallocates it).  The source pages have no counterpart; this is a deployment
 * variant of the same computation, bit-equal to qlinear_pgemm on the same inputs.
 *   Arguments, layouts and errors are those of qlinear_pgemm.  The split row sums
 *   live in one file-scope static device array of 1,048,576 bf16 values (2 MiB),
 *   which every GPU that loads the library holds until the process exits.
 *   Limit: m * round_up(3*k/64, 64) <= 1,048,576 (for example m <= 8192 at k = 2048,
 *   m <= 2730 at k = 8192); larger problems return QL_ERR_TOO_LARGE before anything
 *   is enqueued.  The call itself allocates nothing (no cudaMalloc, cudaFree or
 *   allocating library routine).
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and caches it; make that first
 *   call before any stream capture.
 *   Sharing: all calls on a device use the same array, which keeps the last call's
 *   contents.  Nothing in it needs to start at zero (each call writes every value it
 *   reads before reading it), but calls that overlap on the GPU - on different
 *   streams, or from different host threads - race on it and must be ordered.
 */
int qlinear_pgemm_noalloc(const ql_weight *w, const uint16_t *X, int32_t m, int64_t ldx, float *Y,
                          int64_t ldy, void *stream);

/*
 * qlinear_pgemm_swiglu - the prompt GEMM of the FFN's up projection (w3) with the SwiGLU
 * as its epilogue: H[m][i] = bf16(silu(A[m][i]) * c[m][i]), c = X w3^T computed exactly as
 * qlinear_pgemm computes it and A the gate projection's output (qlinear_pgemm with w1).
 * [P1696] "What it adds" (decode fuses w1 + w3 + SwiGLU; the prompt GEMM); [P1514] "What
 * changes" (paired FFN projections keep their retained rounding boundaries: h is bf16).
 * Bit-equal to qswiglu(A, qlinear_pgemm(w3, X)); c is never written to memory.
 *   X: bf16 [m, ldx] (16-byte aligned, ldx % 8 == 0); A: float [m, lda] (lda >= n);
 *   H: bf16 bits [m, ldh] (ldh >= n).  m may be 0 (nothing enqueued).  Scratch and errors
 *   as qlinear_pgemm.
 */
int qlinear_pgemm_swiglu(const ql_weight *w3, const uint16_t *X, int32_t m, int64_t ldx,
                         const float *A, int64_t lda, uint16_t *H, int64_t ldh, void *stream);

/*
 * qlinear_pgemm_resid_norm - the prompt GEMM of w2 or o with the post-add / next-norm
 * step: resid[m][i] <- bf16(resid[m][i] + y[m][i]) in the GEMM's epilogue (y = X w^T as
 * qlinear_pgemm computes it, never written to memory), then out[m][i] =
 * bf16(r'_i / sqrt(mean_i r'_i^2 + eps) * gamma_i) from the stored r' by the norm kernel of
 * qresid_rmsnorm.  [P1514] "What changes" (post-add/next-norm fusion with the retained
 * rounding boundaries); [P1696] "What it adds" (the prompt GEMM).  Both resid and out are
 * bit-equal to qlinear_pgemm followed by qresid_rmsnorm.
 *   X: bf16 [m, ldx]; resid: bf16 bits [m, ldr] (ldr >= n), read and overwritten; gamma:
 *   bf16 [n]; out: bf16 bits [m, ldo] (ldo >= n, must not overlap resid).  m may be 0.
 *   Errors as qlinear_pgemm, plus QL_ERR_SHAPE for eps < 0.
 */
int qlinear_pgemm_resid_norm(const ql_weight *w, const uint16_t *X, int32_t m, int64_t ldx,
                             uint16_t *resid, int64_t ldr, const uint16_t *gamma, float eps,
                             uint16_t *out, int64_t ldo, void *stream);

/*
 * qswiglu - h[r][i] = bf16(silu(a[r][i]) * c[r][i]) (float32 math, nearest-even
 * rounding): the SwiGLU of qffn_swiglu_mv on its own, used as its "fusion off" control.
 *   a, c: float [rows, lda]; h: bf16 bits [rows, ldh]; rows >= 1, n >= 1.
 */
int qswiglu(const float *a, const float *c, int32_t rows, int32_t n, int64_t lda,
            uint16_t *h, int64_t ldh, void *stream);

/*
 * qattn_qknorm_rope_kv - the step after the attention projections for 1..16 decode
 * streams: QK norm, partial RoPE and the KV store.  [P1696] "What it adds" ("QK norm
 * with partial RoPE"; decode fuses RoPE with the KV store; per-stream KV rings).  The
 * pages print no formula; the definitions (the plain ones, every constant an argument):
 *   norm:  xhat_j = x_j / sqrt(mean_j x_j^2 + eps) * w_j over each head_dim-long head,
 *          w = q_norm_w for q heads, k_norm_w for k heads (bf16 [head_dim] each);
 *   RoPE:  rotate-half on the first rot_dim dims of each normed q and k head, at
 *          position pos[r]: theta_i = pos[r] * rope_base^(-2i/rot_dim), i < rot_dim/2,
 *          (a, b) = (x_i, x_{i+rot_dim/2}) -> (a cos - b sin, a sin + b cos);
 *          dims rot_dim..head_dim-1 pass through;
 *   store: q_out[r] = bf16(rotated q); k and v (v unchanged) of stream r, rounded to
 *          bf16, into slot s = pos[r] mod ring_len (the non-negative remainder) of
 *          stream r's rings.
 * Arithmetic: fp32 for the norm and the rotation (fixed-order sums, so results are
 * deterministic); the angle is formed and reduced modulo 2*pi in float64, its cos/sin
 * taken in fp32; one nearest-even rounding to bf16 per output.
 *   q: float [rows, ldq] (n_q_heads*head_dim used); k, v: float [rows, ldk/ldv]
 *   (n_kv_heads*head_dim used) - the outputs of qattn_proj_mv;
 *   pos: int32 [rows] (device); q_out: bf16 bits [rows, ldqo];
 *   k_ring, v_ring: bf16 bits [rows][ring_len][n_kv_heads*head_dim], slot s of stream r
 *   at element offset (r*ring_len + s)*n_kv_heads*head_dim; other slots are untouched.
 *   Requires 1 <= rows <= 16, head_dim a multiple of 32 in 32..256, rot_dim even in
 *   0..head_dim, ring_len >= 1, rope_base > 0, eps >= 0 (else QL_ERR_ROWS/QL_ERR_SHAPE);
 *   float pointers 4-byte and bf16 pointers 2-byte aligned and leading dimensions at
 *   least the used widths (else QL_ERR_ALIGN).
 */
int qattn_qknorm_rope_kv(const float *q, int64_t ldq, const float *k, int64_t ldk, const float *v,
                         int64_t ldv, int32_t rows, int32_t n_q_heads, int32_t n_kv_heads,
                         int32_t head_dim, int32_t rot_dim, float rope_base, float eps,
                         const uint16_t *q_norm_w, const uint16_t *k_norm_w, const int32_t *pos,
                         uint16_t *q_out, int64_t ldqo, uint16_t *k_ring, uint16_t *v_ring,
                         int32_t ring_len, void *stream);

/*
 * qresid_rmsnorm - post-add / next-norm after the w2 or o projection.  [P1514] "What
 * changes" (post-add/next-norm fusion keeping the retained rounding boundaries).  The
 * residual stream is stored in bf16: resid[r][j] <- bf16(resid[r][j] + y[r][j]), and
 * out[r][j] = bf16(r'_j / sqrt(mean_j r'_j^2 + eps) * gamma_j), computed from the
 * stored (rounded) r'.  fp32 arithmetic, fixed-order sums, nearest-even rounding.
 *   y: float [rows, ldy]; resid: bf16 bits [rows, ldr], read and overwritten;
 *   gamma: bf16 bits [n]; out: bf16 bits [rows, ldo] (must not overlap resid).
 *   Requires rows >= 1 (QL_ERR_ROWS), n >= 1 and eps >= 0 (QL_ERR_SHAPE), aligned
 *   pointers and leading dimensions >= n (QL_ERR_ALIGN).
 */
int qresid_rmsnorm(const float *y, int64_t ldy, uint16_t *resid, int64_t ldr, int32_t rows,
                   int32_t n, const uint16_t *gamma, float eps, uint16_t *out, int64_t ldo,
                   void *stream);

/*
 * qlinear_mv_resid_norm - the w2 / o decode matvec with the post-add / next-norm step as
 * its epilogue, in one launch.  [P1514] "What changes" (post-add/next-norm fusion with the
 * retained rounding boundaries); [P1696] "What it adds" (decode matvecs).
 *   y = W x[r] as qlinear_mv_rows computes it (bit-equal), then
 *   resid[r][i] <- bf16(resid[r][i] + y[r][i])      (bit-equal to qresid_rmsnorm's), and
 *   out[r][i] = bf16(r'_i / sqrt(mean_i r'_i^2 + eps) * gamma_i) from the stored r'.
 * The sum of squares runs in a fixed order of its own (per 16-channel tile, then tiles in
 * order), so out is deterministic and row-local but not bit-equal to qresid_rmsnorm's;
 * both are within half a bf16 ulp plus fp32 error of the float64 value.
 *   x: bf16 [rows, ldx]; resid: bf16 bits [rows, ldr], read and overwritten; gamma: bf16
 *   [n]; out: bf16 bits [rows, ldo] (must not overlap resid).  rows 1..16, n <= 65536.
 *   Uses a library-owned per-device scratch (per-tile sums and a counter that every launch
 *   leaves at zero): calls on one device must be ordered on one stream.  The first call on
 *   a device looks up the scratch's device address and caches it; make that first call
 *   before any stream capture.  Errors as
 *   qlinear_mv_rows, plus QL_ERR_NULL for resid/gamma/out and QL_ERR_SHAPE for eps < 0.
 */
int qlinear_mv_resid_norm(const ql_weight *w, const uint16_t *x, int32_t rows, int64_t ldx,
                          uint16_t *resid, int64_t ldr, const uint16_t *gamma, float eps,
                          uint16_t *out, int64_t ldo, void *stream);

/*
 * qlinear_last_error - synchronizes `stream`, then returns and clears the device
 * status word: QL_OK, or QL_ERR_TIMEOUT if a bounded device-side wait gave up in a
 * kernel enqueued since the last call.  Returns QL_ERR_CUDA if synchronization fails.
 */
int qlinear_last_error(void *stream);

/*
 * qlinear_set_wait_budget_ns - bound, in nanoseconds, for every device-side wait of
 * the kernels enqueued after this call (default 2e9).  A wait that exceeds it makes
 * the kernel record QL_ERR_TIMEOUT and return instead of spinning.  Returns the
 * previous value.
 */
uint64_t qlinear_set_wait_budget_ns(uint64_t ns);

/*
 * qlinear_wait_probe - enqueues one CTA that waits on a shared-memory barrier that
 * nothing ever completes, bounded by `budget_ns`; the kernel records QL_ERR_TIMEOUT
 * and returns.  Exercises the timeout path of qlinear_last_error without a fault.
 */
int qlinear_wait_probe(uint64_t budget_ns, void *stream);

/* qlinear_strerror - static description of a QL_* code. */
const char *qlinear_strerror(int code);

/* qlinear_version - (major << 16) | minor of this library. */
int qlinear_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QLINEAR_H */
