// pgemm.cuh - host interface of the prompt-window GEMM (tcgen05 / TMEM / TMA).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qlinear.h"

namespace qlk {

// Enqueue the row-sum pre-pass and the GEMM.  Arguments are already checked.
int pgemm_run(const ql_weight *w, const uint16_t *X, int m, int64_t ldx, float *Y, int64_t ldy,
              cudaStream_t st, int *status);

uint64_t wait_budget_ns();

}  // namespace qlk
