// ssd_tc.cu -- tcgen05 kernels of libssd (bf16 inputs, fp32 accumulation).
#include "ssd_tc.cuh"

namespace ssd {

bool tc_fwd_supported(const Dims &, ssd_dtype_t) { return false; }
size_t tc_fwd_workspace(const Dims &) { return 0; }
cudaError_t tc_fwd(const Dims &, ssd_dtype_t, const void *, const void *, const float *, const void *, const void *,
                   const float *, const float *, void *, float *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
bool tc_stage_supported(const Dims &, ssd_dtype_t) { return false; }
cudaError_t tc_chunk_state(const Dims &, const void *, const void *, const void *, const float *, float *,
                           cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_chunk_scan(const Dims &, ssd_dtype_t, const void *, const void *, const void *, const void *, const float *,
                          const float *, const float *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace ssd
