// ssd_common.cuh -- small device helpers shared by the libssd kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Problem sizes as the kernels see them (validated on the host).
struct Dims {
    int64_t b, L, H, P, N, G, Q, nc;
    int hpg;  // heads per group, H / G
};

using bf16 = __nv_bfloat16;

// Launch timing: when enabled, mark() records the next event on the stream.
// Entry points call timing_begin() once, then mark() after every launch.
void timing_begin(cudaStream_t s);
void timing_mark(cudaStream_t s, const char *kernel_name);

// Kernel launchers (ssd_simt.cu).  Each returns cudaGetLastError() after the
// launch.
template <typename T>
cudaError_t launch_chunk_cumsum(const Dims &d, const T *dt, const float *A, float *cum, cudaStream_t s);
cudaError_t launch_state_passing(const Dims &d, const float *states, const float *cum, const float *init,
                                 float *states_in, float *final_state, cudaStream_t s);
template <typename T>
cudaError_t launch_chunk_state_simt(const Dims &d, const T *x, const T *dt, const T *B, const float *cum,
                                    float *states, cudaStream_t s);
template <typename T, typename TY>
cudaError_t launch_chunk_scan_simt(const Dims &d, const T *x, const T *dt, const T *B, const T *C,
                                   const float *cum, const float *states_in, const float *D, TY *y,
                                   cudaStream_t s);
template <typename T, typename TY>
cudaError_t launch_selective_scan(const Dims &d, const T *x, const T *dt, const float *A, const T *B,
                                  const T *C, const float *D, const float *init, TY *y, float *final_state,
                                  cudaStream_t s);

// Recurrent step (ssd_decode.cu).
template <typename T, typename TY>
cudaError_t launch_decode_step(const Dims &d, const T *x, const T *dt, const float *A, const T *B, const T *C,
                               const float *D, float *state, TY *y, cudaStream_t s);

}  // namespace ssd
