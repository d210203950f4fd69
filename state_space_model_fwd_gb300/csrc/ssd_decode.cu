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
// is read and written once, everything else is small.  One warp owns one
// state row (b, h, p); its lanes own float4 runs of n, so a warp moves
// N * 4 contiguous bytes each way and sums its row of y with shuffles.
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

template <typename T, typename TY>
__global__ void __launch_bounds__(256) decode_step_kernel(Dims d, const T *__restrict__ x, const T *__restrict__ dt,
                                                          const float *__restrict__ A, const T *__restrict__ B,
                                                          const T *__restrict__ C, const float *__restrict__ D,
                                                          float *__restrict__ state, TY *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // (b, h, p)
    if (row >= d.b * d.H * d.P) return;  // warp-uniform
    const int64_t p = row % d.P, bh = row / d.P, h = bh % d.H, b = bh / d.H;
    const int64_t g = h / d.hpg;
    const float dtv = to_f32(dt[b * d.H + h]);
    const float xv = to_f32(x[bh * d.P + p]);
    const float a = expf(dtv * A[h]);
    const float u = dtv * xv;
    const T *Bt = B + (b * d.G + g) * d.N;
    const T *Ct = C + (b * d.G + g) * d.N;
    float4 *s4 = reinterpret_cast<float4 *>(state + row * d.N);
    float acc = 0.f;
    for (int64_t j = lane; j < d.N / 4; j += 32) {
        float4 s = s4[j];
        const float4 bb = load4<T>(Bt + 4 * j), cc = load4<T>(Ct + 4 * j);
        s.x = fmaf(a, s.x, u * bb.x);
        s.y = fmaf(a, s.y, u * bb.y);
        s.z = fmaf(a, s.z, u * bb.z);
        s.w = fmaf(a, s.w, u * bb.w);
        __stcs(s4 + j, s);
        acc = fmaf(cc.x, s.x, fmaf(cc.y, s.y, fmaf(cc.z, s.z, fmaf(cc.w, s.w, acc))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) y[bh * d.P + p] = from_f32<TY>(acc + (D ? D[h] : 0.f) * xv);
}

}  // namespace

template <typename T, typename TY>
cudaError_t launch_decode_step(const Dims &d, const T *x, const T *dt, const float *A, const T *B, const T *C,
                               const float *D, float *state, TY *y, cudaStream_t s) {
    const int64_t rows = d.b * d.H * d.P;
    constexpr int kWarps = 8;
    const int64_t blocks = (rows + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    decode_step_kernel<T, TY><<<(unsigned)blocks, kWarps * 32, 0, s>>>(d, x, dt, A, B, C, D, state, y);
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
