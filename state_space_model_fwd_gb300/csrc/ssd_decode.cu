// ssd_decode.cu -- the recurrent (decode) step: one new token per sequence
// advances the state in place and gives that token's output.
//
//   state[b,h] <- exp(dt[b,h] A[h]) state[b,h] + dt[b,h] x[b,h] B[b,g]^T
//   y[b,h]      = state[b,h] C[b,g] + D[h] x[b,h]
//
// This is the recurrence itself, applied to one step: per token and head the
// cost is O(P N) with a state of constant size (the inference mode of the
// da_be19 thread, post 5/6: linear-time inference with a constant state).
// The step is bound by HBM bandwidth: the fp32 state (P N 4 bytes per head)
// is read and written once, everything else is small.  One warp owns kRows
// consecutive state rows (b, h, p .. p + kRows - 1) of one head: it issues
// the loads of all of them before any arithmetic (kRows 16-byte loads in
// flight per lane), shares the head's scalars and its B and C rows between
// them, and sums each row of y with interleaved shuffle reductions.  Lane l
// owns the float4 runs j = l + 32 jj of n, jj < NJ (NJ = 1 for N <= 128, 2 up
// to N = 256: a kernel per case, so the N <= 128 one holds half the state
// registers and fits more warps per SM).
#include "ssd_common.cuh"

namespace ssd {
namespace {

template <typename T>
__device__ __forceinline__ float4 load4(const T *p);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
template <>
__device__ __forceinline__ float4 load4<bf16>(const bf16 *p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
}

constexpr int kRows = 8;  // state rows per warp (P is a multiple of 16)

template <typename T, typename TY, int NJ>
__global__ void __launch_bounds__(256) decode_step_kernel(Dims d, const T *__restrict__ x, const T *__restrict__ dt,
                                                          const float *__restrict__ A, const T *__restrict__ B,
                                                          const T *__restrict__ C, const float *__restrict__ D,
                                                          float *__restrict__ state, TY *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int64_t row0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kRows;  // (b, h, p0)
    if (row0 >= d.b * d.H * d.P) return;  // warp-uniform; P % kRows == 0, so all kRows rows exist
    const int64_t n4 = d.N / 4;
    float4 *s4 = reinterpret_cast<float4 *>(state + row0 * d.N);
    bool has[NJ];
    float4 s[kRows][NJ];
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        has[jj] = lane + 32 * jj < n4;
#pragma unroll
        for (int r = 0; r < kRows; ++r)
            if (has[jj]) s[r][jj] = __ldcs(s4 + r * n4 + lane + 32 * jj);
    }
    const int64_t bh = row0 / d.P, p0 = row0 % d.P, h = bh % d.H, b = bh / d.H;
    const int64_t g = h / d.hpg;
    const float dtv = to_f32(dt[b * d.H + h]);
    const float a = expf(dtv * A[h]);
    const float dd = D ? D[h] : 0.f;
    const T *Bt = B + (b * d.G + g) * d.N;
    const T *Ct = C + (b * d.G + g) * d.N;
    float xv[kRows], acc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        xv[r] = to_f32(x[bh * d.P + p0 + r]);
        acc[r] = 0.f;
    }
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        if (!has[jj]) continue;
        const int64_t j = lane + 32 * jj;
        const float4 bb = load4<T>(Bt + 4 * j), cc = load4<T>(Ct + 4 * j);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float u = dtv * xv[r];
            float4 v = s[r][jj];
            v.x = fmaf(a, v.x, u * bb.x);
            v.y = fmaf(a, v.y, u * bb.y);
            v.z = fmaf(a, v.z, u * bb.z);
            v.w = fmaf(a, v.w, u * bb.w);
            __stcs(s4 + r * n4 + j, v);
            acc[r] = fmaf(cc.x, v.x, fmaf(cc.y, v.y, fmaf(cc.z, v.z, fmaf(cc.w, v.w, acc[r]))));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int r = 0; r < kRows; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    if (lane < kRows) {
        float out = acc[0], xo = xv[0];
#pragma unroll
        for (int r = 1; r < kRows; ++r)
            if (lane == r) {
                out = acc[r];
                xo = xv[r];
            }
        y[bh * d.P + p0 + lane] = from_f32<TY>(out + dd * xo);
    }
}

}  // namespace

template <typename T, typename TY>
cudaError_t launch_decode_step(const Dims &d, const T *x, const T *dt, const float *A, const T *B, const T *C,
                               const float *D, float *state, TY *y, cudaStream_t s) {
    const int64_t rows = d.b * d.H * d.P;
    if (d.P % kRows != 0 || d.N > 256 || d.N % 4 != 0) return cudaErrorInvalidValue;
    constexpr int kWarps = 8;
    const int64_t blocks = (rows / kRows + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    if (d.N <= 128)
        decode_step_kernel<T, TY, 1><<<(unsigned)blocks, kWarps * 32, 0, s>>>(d, x, dt, A, B, C, D, state, y);
    else
        decode_step_kernel<T, TY, 2><<<(unsigned)blocks, kWarps * 32, 0, s>>>(d, x, dt, A, B, C, D, state, y);
    timing_mark(s, "decode_step");
    return cudaGetLastError();
}

template cudaError_t launch_decode_step<float, float>(const Dims &, const float *, const float *, const float *,
                                                      const float *, const float *, const float *, float *, float *,
                                                      cudaStream_t);
template cudaError_t launch_decode_step<bf16, float>(const Dims &, const bf16 *, const bf16 *, const float *,
                                                     const bf16 *, const bf16 *, const float *, float *, float *,
                                                     cudaStream_t);
template cudaError_t launch_decode_step<bf16, bf16>(const Dims &, const bf16 *, const bf16 *, const float *,
                                                    const bf16 *, const bf16 *, const float *, float *, bf16 *,
                                                    cudaStream_t);

}  // namespace ssd
