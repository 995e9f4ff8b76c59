// pgemm.cuh - host interface of the prompt-window GEMM (tcgen05 / TMEM / TMA).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qlinear.h"

namespace qlk {

// Enqueue the row-sum pre-pass and the GEMM.  Arguments are already checked.
int pgemm_run(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
              cudaStream_t st, int *status);

// The same, with the split row sums in a fixed static device array (no allocation);
// QL_ERR_TOO_LARGE if m * round_up(3k/64, 64) exceeds pgemm_noalloc_max_elems().
int pgemm_run_noalloc(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
                      cudaStream_t st, int *status);
int64_t pgemm_noalloc_max_elems();

uint64_t wait_budget_ns();

}  // namespace qlk
