// ssd_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) path of libssd for bf16
// inputs.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

// True when the fused tcgen05 ssd_fwd handles this shape and dtype.
bool tc_fwd_supported(const Dims &d, ssd_dtype_t dtype);
// Workspace bytes the fused path needs.
size_t tc_fwd_workspace(const Dims &d);
// `status`: the device status word (bit 0 set when a bounded wait gives up).
cudaError_t tc_fwd(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B, const void *C,
                   const float *D, const float *init, void *y, float *fin, void *ws, unsigned *status, cudaStream_t s);

// True when the tcgen05 chunk-state / chunk-scan stage kernels handle this shape.
bool tc_stage_supported(const Dims &d, ssd_dtype_t dtype);
cudaError_t tc_chunk_state(const Dims &d, const void *x, const void *dt, const void *B, const float *cum,
                           float *states, unsigned *status, cudaStream_t s);
// Workspace of the tensor-core chunk-scan stage (chunk packs and their flags).
size_t tc_chunk_scan_workspace(const Dims &d);
// selftest_ns > 0: launch the scan alone with no pack ever published, so its
// bounded wait gives up after that many nanoseconds (failure-path test).
cudaError_t tc_chunk_scan(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const void *B, const void *C,
                          const float *cum, const float *states_in, const float *D, void *y, void *ws,
                          unsigned *status, uint64_t selftest_ns, cudaStream_t s);

// Packed sequences of unequal lengths (ssd_fwd_varlen) in one launch set:
// `d` is the packed batch (b = 1, L = all steps); each sequence is its first
// row t0 in the packed tensors, its steps len (> 0) and its index seq (its
// init / fin state).  At most kVarlenMaxUnits sequences per call.
constexpr int kVarlenMaxUnits = 960;
// Sequences per launch set: a set of several sequences per scan unit adds
// its units (at most one per SM) to the table.
constexpr int kVarlenSetSeqs = 800;
struct VarlenSeq {
    int t0, len, seq;
};
bool tc_varlen_supported(const Dims &d, ssd_dtype_t dtype);
size_t tc_varlen_workspace(const Dims &d, const VarlenSeq *seqs, int n);
cudaError_t tc_fwd_varlen(const Dims &d, const VarlenSeq *seqs, int n, ssd_dtype_t ydtype, const void *x,
                          const void *dt, const float *A, const void *B, const void *C, const float *D,
                          const float *init, void *y, float *fin, void *ws, unsigned *status, cudaStream_t s);
// Estimated device time in microseconds of one launch set over the
// sequences, and of the fused forward of one sequence of `len` steps (the
// choice between them in ssd_fwd_varlen; a model, not a measurement).
double tc_varlen_cost_us(const Dims &d, const VarlenSeq *seqs, int n);
double tc_fwd_cost_us(const Dims &d, int64_t len);

// Quadratic (dual) form for short sequences (ssd_quad.cu).
bool quad_supported(const Dims &d, ssd_dtype_t dtype);
cudaError_t quad_fwd(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B,
                     const void *C, const float *D, const float *init, void *y, float *fin, unsigned *status,
                     cudaStream_t s);

}  // namespace ssd
