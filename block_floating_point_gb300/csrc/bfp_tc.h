// The tensor-memory (tcgen05) path of the dense projection (bfp_linear_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "bfp_internal.h"

namespace bfp {

constexpr int kTcNotApplicable = 1;  // the shape does not fit the path: the caller takes the mma.sync kernel

// y[m x n] (fp32 and/or bf16, row stride ldy) = x[m x k] . W^T on tcgen05, m <= 32. Returns BFP_OK, a BFP_E*
// code, or kTcNotApplicable (k not a multiple of 64, or the activation rows do not fit in shared memory).
int linear_tc_launch(const Geometry &g, const uint8_t *w, const uint16_t *x, int m, int64_t ldx, float *y,
                     uint16_t *y_bf16, int64_t ldy, uint32_t *status, cudaStream_t st);

// Which kernel bfp_linear runs (process-wide): 0 the library's choice, 1 mma.sync only, 2 tcgen05 where it fits.
int linear_path();

}  // namespace bfp
