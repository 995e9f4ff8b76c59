// pgemm.cuh - host interface of the prompt-window GEMM (tcgen05 / TMEM / TMA).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qlinear.h"

namespace qlk {

// What the GEMM's epilogue does with each output y[m][n] (the product is computed the
// same way in every mode, so every mode is bit-equal to the plain GEMM followed by the
// separate step):
//   kPgStore:  Y[m][n] = y (fp32)
//   kPgSwiglu: H[m][n] = bf16(silu(A[m][n]) * y), A fp32 (the gate projection's output)
//   kPgResid:  H[m][n] = bf16(H[m][n] + y), H the bf16 residual stream, in place
enum { kPgStore = 0, kPgSwiglu = 1, kPgResid = 2 };
struct PgEpilogue {
  int mode;
  const float *a;
  int64_t lda;
  uint16_t *h;
  int64_t ldh;
};

// Enqueue the row-sum pre-pass and the GEMM.  Arguments are already checked.  epi may
// be null (kPgStore into Y).
int pgemm_run(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
              cudaStream_t st, int *status, const PgEpilogue *epi = nullptr);

// The same for nw weights with the same k that read the same X: one row-sum pre-pass,
// then each weight's GEMM (and code conversion) in turn.  Arguments are already checked.
int pgemm_run_multi(const ql_weight *const *w, int nw, const uint16_t *X, int m, int64_t ldx, float *const *Y,
                    const int64_t *ldy, cudaStream_t st, int *status, const PgEpilogue *epi = nullptr);

// The post-add / next-norm kernels (qpost.cu); y == nullptr normalises the residual as
// it stands.
cudaError_t launch_resid_rmsnorm(const float *y, int64_t ldy, uint16_t *resid, int64_t ldr, int rows, int n,
                                 const uint16_t *gamma, float eps, uint16_t *out, int64_t ldo, cudaStream_t st);

// The same, with the split row sums in a fixed static device array (no allocation);
// QL_ERR_TOO_LARGE if m * round_up(3k/64, 64) exceeds pgemm_noalloc_max_elems().
int pgemm_run_noalloc(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
                      cudaStream_t st, int *status);
int64_t pgemm_noalloc_max_elems();

uint64_t wait_budget_ns();

}  // namespace qlk
