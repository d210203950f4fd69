// ssd_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) path of libssd for bf16
// inputs.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

// True when the fused tcgen05 ssd_fwd handles this shape and dtype.
bool tc_fwd_supported(const Dims &d, ssd_dtype_t dtype);
// Workspace bytes the fused path needs.
size_t tc_fwd_workspace(const Dims &d);
cudaError_t tc_fwd(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B, const void *C,
                   const float *D, const float *init, void *y, float *fin, void *ws, cudaStream_t s);

// True when the tcgen05 chunk-state / chunk-scan stage kernels handle this shape.
bool tc_stage_supported(const Dims &d, ssd_dtype_t dtype);
cudaError_t tc_chunk_state(const Dims &d, const void *x, const void *dt, const void *B, const float *cum,
                           float *states, cudaStream_t s);
cudaError_t tc_chunk_scan(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const void *B, const void *C,
                          const float *cum, const float *states_in, const float *D, void *y, cudaStream_t s);

}  // namespace ssd
