// ssd_tc.cu -- tcgen05 / TMEM / TMA kernels of libssd (bf16 inputs, fp32
// state and accumulation).
//
// The fused forward runs in two launches over "segments" (runs of
// consecutive chunks of one batch entry and one head block):
//
//   seg_state_kernel  (segments 0 .. nseg-2)
//       S_seg = sum over the segment's tokens t of
//               exp(sum_{k>t, k in segment} dt_k A) dt_t x_t^T B_t
//       one long-K tcgen05 contraction per segment, accumulated in TMEM;
//       writes S_seg and the segment's total log-decay to the workspace.
//
//   chunk_scan_kernel (every segment)
//       folds the earlier segments' states into the state entering the
//       segment, then walks its chunks: per chunk
//         CB   = C B^T                              (tcgen05, shared by heads)
//         M_h  = CB o exp(cum_t - cum_s) dt_s, s<=t (CUDA cores, bf16, smem)
//         Y^T  = X^T M_h^T (intra) + S C^T (inter)  (tcgen05, TMEM)
//         y    = intra + exp(cum_t) inter + D x     (epilogue, straight to HBM)
//         S    = exp(cum_last) S + (w o X)^T B      (TMEM, w_s = exp(cum_last - cum_s) dt_s)
//       so the running state and the Q x Q score matrix never leave the SM.
//
// ("Mamba-2 in NVIDIA cuTile: Faster Forward Kernels", section "Why Mamba-2
// is a useful kernel example": cumulative decay, state entering each chunk,
// outputs, with the intra-chunk interactions kept on-chip; the da_be19
// thread, post 5/6: quadratic inside a chunk, linear across chunks, the
// work dominated by batched matrix multiplications.)
//
// Tiles: a CTA owns HB heads of one group with HB * P = 128, so every
// state-shaped contraction has M = 128 rows (head, p) and TMEM lane r holds
// row r.  Operand tiles are 128-byte swizzled rows of 64 bf16; TMA loads x,
// B and C tiles of Q rows straight into that layout.
#include <cudaTypedefs.h>

#include "ssd_tc.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kTargetCtas = 148;        // about one CTA per SM of a GB300 (152 SMs)
constexpr int kSmemLimit = 226 * 1024;  // dynamic bytes; leaves room for the static mbarriers

struct TcParams {
    const bf16 *dt;
    const float *A, *D, *init;
    void *y;
    float *fin;
    float *seg_state;  // [b, nseg, H, P, N]
    float *seg_tot;    // [b, nseg, H]  total dt*A of each segment
    unsigned *status;  // bit 0: an mbarrier wait gave up
    long long b, L, H, G;
    int hpg, nc, nseg, cps;  // cps: chunks per segment
    int y_f32;
};

template <int P_, int N_, int Q_>
struct Cfg {
    static constexpr int P = P_, N = N_, Q = Q_;
    static constexpr int HB = 128 / P;          // heads per CTA
    static constexpr int M = 128;               // rows (head, p)
    static constexpr int PB = P / 64;           // 64-wide column blocks of one head's x tile
    static constexpr int X_BYTES = M * Q * 2;   // [M/64 blocks][Q rows][64]
    static constexpr int BC_BYTES = N * Q * 2;  // [N/64 blocks][Q rows][64]
    static constexpr int STAGE_BYTES = X_BYTES + 2 * BC_BYTES;
    static constexpr int XW_BYTES = M * Q * 2;
    static constexpr int SBF_BYTES = M * N * 2;       // [N/64 blocks][M rows][64]
    static constexpr int MM_BYTES = HB * Q * Q * 2;   // per head [Q/64 blocks][Q rows][64]
    // scratch: the bf16 state copy and the low half of the scaled x during the
    // state/inter MMAs, then the masked score matrices
    static constexpr int SCR_BYTES = SBF_BYTES + XW_BYTES > MM_BYTES ? SBF_BYTES + XW_BYTES : MM_BYTES;
    static constexpr int SMALL_FLOATS = 4 * HB * Q + 4 * HB;
    static constexpr int SMALL_BYTES = SMALL_FLOATS * 4 + 128;
    static constexpr int smem_scan(int stages) {
        return stages * STAGE_BYTES + XW_BYTES + SCR_BYTES + SMALL_BYTES + 1024;
    }
    static constexpr int STAGES = smem_scan(2) <= kSmemLimit ? 2 : 1;
    // at least 116 KB so that a single CTA (and its 512 TMEM columns) sits on an SM
    static constexpr int SMEM_SCAN = smem_scan(STAGES) > 116 * 1024 ? smem_scan(STAGES) : 116 * 1024;
    static constexpr bool SCAN_FITS = smem_scan(STAGES) <= kSmemLimit;
    // segment-state kernel: two stages of (x, B) plus the scaled x
    static constexpr int SEG_STAGE_BYTES = X_BYTES + BC_BYTES;
    static constexpr int SMEM_SEG_BASE = 2 * SEG_STAGE_BYTES + 2 * XW_BYTES + SMALL_BYTES + 1024;
    // TMEM columns of the scan kernel
    static constexpr int COL_S = 0;
    static constexpr int COL_R3 = N;                 // inter-chunk term, [M][Q]
    static constexpr int COL_R = N + Q;              // intra-chunk term per head, [M][Q] each
    static constexpr int COL_END = N + Q + HB * Q;
    static constexpr bool CB_ALIAS = COL_END + Q > 512;
    static constexpr int COL_CB = CB_ALIAS ? COL_R : COL_END;  // C B^T, [Q][Q]
    static constexpr int TMEM_USED = CB_ALIAS ? COL_END : COL_END + Q;
    static constexpr bool TMEM_FITS = TMEM_USED <= 512;
    static constexpr uint32_t SEG_TMEM = N < 32 ? 32 : N;
};

constexpr uint32_t kWaitPolls = 1u << 20;  // about 0.1 s of polling per wait

__device__ __forceinline__ void flag_timeout(unsigned *status) {
    if (status) atomicOr(status, 1u);
}

// Bookkeeping of asynchronous work in flight, so that a CTA that gives up
// on a wait can still let its own copies and MMAs land (bounded) before it
// frees TMEM and exits.
struct Inflight {
    int issued = 0;   // chunks whose TMA loads were issued
    int waited = 0;   // chunks whose loads were waited for
    bool mma = false; // a commit not yet waited for
    uint32_t mma_phase = 0;
};

template <int STAGES>
__device__ __forceinline__ void drain(Inflight &f, uint64_t *full_bar, uint64_t *mma_bar) {
    for (int k = f.waited; k < f.issued; ++k)
        mbar_wait(&full_bar[k % STAGES], (uint32_t)((k / STAGES) & 1), kWaitPolls);
    if (f.mma) mbar_wait(mma_bar, f.mma_phase, kWaitPolls);
}

// Inclusive scan of dt*A over one chunk for head h, by one warp.  Writes
// cum (log-decay from the chunk start) and returns the chunk total.
template <int Q>
__device__ __forceinline__ float warp_chunk_cumsum(const float *dtv, float a, float *cum) {
    constexpr int QPL = Q / 32;
    const int lane = threadIdx.x & 31;
    float v[QPL];
    float run = 0.f;
#pragma unroll
    for (int i = 0; i < QPL; ++i) {
        run += dtv[lane * QPL + i] * a;
        v[i] = run;
    }
    float tot = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, tot, off);
        if (lane >= off) tot += o;
    }
    const float excl = tot - run;
#pragma unroll
    for (int i = 0; i < QPL; ++i) cum[lane * QPL + i] = v[i] + excl;
    return __shfl_sync(0xffffffffu, tot, 31);
}

// x tile scaled row-wise by w, split into two bf16 tiles whose sum carries
// the product to about 2^-17 relative: hi = bf16(w x), lo = bf16(w x - hi).
// (One bf16 rounding of w x, 2^-9 relative, is visible in the state entries
// that a single recent token dominates.)  Works on whole 16-byte chunks of
// the swizzled layout: a chunk stays in its row, so its scale is its row's.
template <class C>
__device__ __forceinline__ void build_xw(const uint8_t *xs, uint8_t *xw_hi, uint8_t *xw_lo, const float *w) {
    constexpr int CHUNKS = (C::M / 64) * C::Q * 8;
    for (int i = threadIdx.x; i < CHUNKS; i += kThreads) {
        const int blk = i / (C::Q * 8);
        const int s = (i / 8) % C::Q;
        const int h = blk / C::PB;
        const float ws = w[h * C::Q + s];
        uint4 v = *reinterpret_cast<const uint4 *>(xs + (size_t)i * 16);
        uint4 lo;
        uint32_t *u = reinterpret_cast<uint32_t *>(&v);
        uint32_t *l = reinterpret_cast<uint32_t *>(&lo);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 p2 = *reinterpret_cast<__nv_bfloat162 *>(&u[j]);
            const float2 f = __bfloat1622float2(p2);
            const float a = f.x * ws, b2 = f.y * ws;
            const __nv_bfloat162 hi2 = __floats2bfloat162_rn(a, b2);
            const float2 hf = __bfloat1622float2(hi2);
            u[j] = *reinterpret_cast<const uint32_t *>(&hi2);
            l[j] = pack_bf16x2(a - hf.x, b2 - hf.y);
        }
        *reinterpret_cast<uint4 *>(xw_hi + (size_t)i * 16) = v;
        *reinterpret_cast<uint4 *>(xw_lo + (size_t)i * 16) = lo;
    }
}

// Issue the TMA loads of chunk c: x tiles of the CTA's heads, then B (and C).
template <class C>
__device__ __forceinline__ void issue_chunk_loads(uint8_t *stage, uint64_t *bar, const CUtensorMap *mx,
                                                  const CUtensorMap *mb, const CUtensorMap *mc, int h0, int g,
                                                  int c, int b, bool with_c) {
    const uint32_t bytes = C::X_BYTES + C::BC_BYTES * (with_c ? 2 : 1);
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int hh = 0; hh < C::HB; ++hh)
#pragma unroll
        for (int pb = 0; pb < C::PB; ++pb)
            tma_load_4d(stage + (hh * C::PB + pb) * (C::Q * 128), mx, bar, pb * 64, h0 + hh, c * C::Q, b);
    uint8_t *sb = stage + C::X_BYTES;
#pragma unroll
    for (int nb = 0; nb < C::N / 64; ++nb) tma_load_4d(sb + nb * (C::Q * 128), mb, bar, nb * 64, g, c * C::Q, b);
    if (with_c) {
        uint8_t *sc = sb + C::BC_BYTES;
#pragma unroll
        for (int nb = 0; nb < C::N / 64; ++nb)
            tma_load_4d(sc + nb * (C::Q * 128), mc, bar, nb * 64, g, c * C::Q, b);
    }
}

// ===========================================================================
// Segment local states: S_seg for segments 0 .. nseg-2.
// ===========================================================================
template <class C>
__global__ void __launch_bounds__(kThreads, 1)
    seg_state_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mb, TcParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint8_t *xw = stages + 2 * C::SEG_STAGE_BYTES;
    uint8_t *xw_lo = xw + C::XW_BYTES;
    float *small = reinterpret_cast<float *>(xw_lo + C::XW_BYTES);
    float *dtv = small;               // [HB][Q]
    float *cum = dtv + C::HB * C::Q;  // [HB][Q]
    float *w = cum + C::HB * C::Q;    // [HB][Q]
    float *tail = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(small) + C::SMALL_BYTES);  // [HB][cps]
    __shared__ uint64_t full_bar[2], mma_bar;
    __shared__ uint32_t tmem_base_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, hblk = blockIdx.y, b = blockIdx.z;
    const int h0 = hblk * C::HB;
    const int g = (int)(prm.G == 1 ? 0 : h0 / prm.hpg);
    const int c0 = seg * prm.cps;
    const int c1 = min(prm.nc, c0 + prm.cps);
    const int nch = c1 - c0;
    const long long L = prm.L, H = prm.H;

    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, C::SEG_TMEM);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&full_bar[0], 1);
        mbar_init(&full_bar[1], 1);
        mbar_init(&mma_bar, 1);
        fence_mbar_init();
        prefetch_tmap(&mx);
        prefetch_tmap(&mb);
    }
    // per-chunk totals of dt*A for every chunk of the segment, then the
    // suffix sums: tail[h][k] = sum of the totals of chunks after k.
    for (int item = warp; item < C::HB * nch; item += kThreads / 32) {
        const int hh = item / nch, k = item % nch;
        const long long h = h0 + hh;
        float s = 0.f;
        if (h < H)
            for (int q = lane; q < C::Q; q += 32)
                s += __bfloat162float(prm.dt[((long long)b * L + (long long)(c0 + k) * C::Q + q) * H + h]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) tail[hh * prm.cps + k] = h < H ? s * prm.A[h] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid < C::HB) {
        float run = 0.f;
        for (int k = nch - 1; k >= 0; --k) {
            const float t = tail[tid * prm.cps + k];
            tail[tid * prm.cps + k] = run;
            run += t;
        }
        const long long h = h0 + tid;
        if (h < H) prm.seg_tot[((long long)b * prm.nseg + seg) * H + h] = run;
    }
    const uint32_t tmem = tmem_base_sh;
    __shared__ int abort_sh;
    if (tid == 0) abort_sh = 0;
    Inflight fl;  // meaningful in thread 0, which issues all async work
    if (tid == 0) {
        issue_chunk_loads<C>(stages, &full_bar[0], &mx, &mb, nullptr, h0, g, c0, b, false);
        fl.issued = 1;
    }

    for (int it = 0; it < nch; ++it) {
        const int c = c0 + it;
        const int st = it & 1;
        uint8_t *stage = stages + st * C::SEG_STAGE_BYTES;
        // dt of this chunk
        for (int i = tid; i < C::HB * C::Q; i += kThreads) {
            const int hh = i / C::Q, q = i % C::Q;
            const long long h = h0 + hh;
            dtv[i] = h < H ? __bfloat162float(prm.dt[((long long)b * L + (long long)c * C::Q + q) * H + h]) : 0.f;
        }
        __syncthreads();
        if (abort_sh) break;
        if (warp < C::HB) {
            const long long h = h0 + warp;
            const float a = h < H ? prm.A[h] : 0.f;
            float *cw = cum + warp * C::Q;
            const float total = warp_chunk_cumsum<C::Q>(dtv + warp * C::Q, a, cw);
            __syncwarp();
            const float after = tail[warp * prm.cps + it];
            for (int q = lane; q < C::Q; q += 32)
                w[warp * C::Q + q] = expf(after + total - cw[q]) * dtv[warp * C::Q + q];
        }
        // the previous MMA has finished reading xw and the other stage
        // (waited at the end of the last iteration): prefetch the next chunk
        if (tid == 0 && it + 1 < nch) {
            issue_chunk_loads<C>(stages + (st ^ 1) * C::SEG_STAGE_BYTES, &full_bar[st ^ 1], &mx, &mb, nullptr,
                                 h0, g, c + 1, b, false);
            fl.issued = it + 2;
        }
        if (!mbar_wait(&full_bar[st], (it >> 1) & 1, kWaitPolls)) abort_sh = 1;
        else if (tid == 0) fl.waited = it + 1;
        __syncthreads();
        if (abort_sh) break;
        build_xw<C>(stage, xw, xw_lo, w);
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(C::M, C::N, true, true);
            const uint32_t a0 = smem_u32(xw), a1 = smem_u32(xw_lo), b0 = smem_u32(stage + C::X_BYTES);
#pragma unroll
            for (int ks = 0; ks < C::Q / 16; ++ks)
                mma_bf16(tmem, sdesc(a0 + ks * 2048, C::Q * 128, 1024), sdesc(b0 + ks * 2048, C::Q * 128, 1024),
                         idesc, (it | ks) != 0);
#pragma unroll
            for (int ks = 0; ks < C::Q / 16; ++ks)
                mma_bf16(tmem, sdesc(a1 + ks * 2048, C::Q * 128, 1024), sdesc(b0 + ks * 2048, C::Q * 128, 1024),
                         idesc, true);
            mma_commit(&mma_bar);
            fl.mma = true;
        }
        if (!mbar_wait(&mma_bar, fl.mma_phase, kWaitPolls)) abort_sh = 1;
        else if (tid == 0) fl.mma = false;
        fl.mma_phase ^= 1;
        tc_fence_after();
    }
    __syncthreads();
    if (abort_sh) {
        if (tid == 0) {
            flag_timeout(prm.status);
            drain<2>(fl, full_bar, &mma_bar);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, C::SEG_TMEM);
        return;
    }
    // write the segment state: row r = (head, p) of TMEM lane r
    if (warp < 4) {
        const int r = warp * 32 + lane;
        const int hh = r / C::P, p = r % C::P;
        const long long h = h0 + hh;
        float *dst = prm.seg_state + ((((long long)b * prm.nseg + seg) * H + h) * C::P + p) * C::N;
#pragma unroll 1
        for (int n0 = 0; n0 < C::N; n0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + n0, v);
            tmem_ld_wait();
            if (h < H)
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4 *>(dst + n0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, C::SEG_TMEM);
}

// ===========================================================================
// Chunk scan with the state carried in TMEM.
// ===========================================================================
template <class C>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mb,
                      const __grid_constant__ CUtensorMap mc, TcParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint8_t *xw = stages + C::STAGES * C::STAGE_BYTES;
    uint8_t *scr = xw + C::XW_BYTES;  // bf16 state copy + low half of w x, then the masked score matrices
    uint8_t *xw_lo = scr + C::SBF_BYTES;
    float *small = reinterpret_cast<float *>(scr + C::SCR_BYTES);
    float *dtv = small;                 // [HB][Q]
    float *cum = dtv + C::HB * C::Q;    // [HB][Q]
    float *w = cum + C::HB * C::Q;      // [HB][Q]
    float *ecum = w + C::HB * C::Q;     // [HB][Q]
    float *decay = ecum + C::HB * C::Q; // [HB]
    __shared__ uint64_t full_bar[2], mma_bar;
    __shared__ uint32_t tmem_base_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, hblk = blockIdx.y, b = blockIdx.z;
    const int h0 = hblk * C::HB;
    const int g = (int)(prm.G == 1 ? 0 : h0 / prm.hpg);
    const int c0 = seg * prm.cps;
    const int c1 = min(prm.nc, c0 + prm.cps);
    const int nch = c1 - c0;
    const long long L = prm.L, H = prm.H;
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;     // (head, p) row for warps 0-3 / 4-7
    const int rh = row / C::P, rp = row % C::P;
    const long long hrow = h0 + rh;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;

    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&full_bar[0], 1);
        mbar_init(&full_bar[1], 1);
        mbar_init(&mma_bar, 1);
        fence_mbar_init();
        prefetch_tmap(&mx);
        prefetch_tmap(&mb);
        prefetch_tmap(&mc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    __shared__ int abort_sh;
    if (tid == 0) abort_sh = 0;
    Inflight fl;  // meaningful in thread 0, which issues all async work
    if (tid == 0) {
        issue_chunk_loads<C>(stages, &full_bar[0], &mx, &mb, &mc, h0, g, c0, b, true);
        fl.issued = 1;
    }

    // state entering the segment: fold the earlier segments' states
    if (warp < 4) {
        const float *init_row = (prm.init && hrow < H) ? prm.init + (((long long)b * H + hrow) * C::P + rp) * C::N : nullptr;
#pragma unroll 1
        for (int n0 = 0; n0 < C::N; n0 += 16) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = init_row ? init_row[n0 + j] : 0.f;
            if (hrow < H)
                for (int sp = 0; sp < seg; ++sp) {
                    const float e = expf(prm.seg_tot[((long long)b * prm.nseg + sp) * H + hrow]);
                    const float *src =
                        prm.seg_state + ((((long long)b * prm.nseg + sp) * H + hrow) * C::P + rp) * C::N + n0;
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 s4 = *reinterpret_cast<const float4 *>(src + j);
                        v[j] = fmaf(e, v[j], s4.x);
                        v[j + 1] = fmaf(e, v[j + 1], s4.y);
                        v[j + 2] = fmaf(e, v[j + 2], s4.z);
                        v[j + 3] = fmaf(e, v[j + 3], s4.w);
                    }
                }
            tmem_st16(tmem + lane_off + C::COL_S + n0, v);
        }
        tmem_st_wait();
    }
    const float dh_row = (prm.D && hrow < H) ? prm.D[hrow] : 0.f;

    for (int it = 0; it < nch; ++it) {
        const int c = c0 + it;
        const int st = C::STAGES == 2 ? (it & 1) : 0;
        const uint32_t full_parity = C::STAGES == 2 ? ((it >> 1) & 1) : (it & 1);
        uint8_t *stage = stages + st * C::STAGE_BYTES;
        uint8_t *xs = stage;
        uint8_t *bs = stage + C::X_BYTES;
        uint8_t *cs = bs + C::BC_BYTES;
        if (C::STAGES == 2 && tid == 0 && it + 1 < nch) {
            issue_chunk_loads<C>(stages + (st ^ 1) * C::STAGE_BYTES, &full_bar[st ^ 1], &mx, &mb, &mc, h0, g, c + 1,
                                 b, true);
            fl.issued = it + 2;
        }
        for (int i = tid; i < C::HB * C::Q; i += kThreads) {
            const int hh = i / C::Q, q = i % C::Q;
            const long long h = h0 + hh;
            dtv[i] = h < H ? __bfloat162float(prm.dt[((long long)b * L + (long long)c * C::Q + q) * H + h]) : 0.f;
        }
        __syncthreads();
        // (1) cumulative decay of each head
        if (warp < C::HB) {
            const long long h = h0 + warp;
            const float a = h < H ? prm.A[h] : 0.f;
            float *cw = cum + warp * C::Q;
            const float total = warp_chunk_cumsum<C::Q>(dtv + warp * C::Q, a, cw);
            __syncwarp();
            for (int q = lane; q < C::Q; q += 32) {
                w[warp * C::Q + q] = expf(total - cw[q]) * dtv[warp * C::Q + q];
                ecum[warp * C::Q + q] = expf(cw[q]);
            }
            if (lane == 0) decay[warp] = expf(total);
        }
        if (!mbar_wait(&full_bar[st], full_parity, kWaitPolls)) abort_sh = 1;
        else if (tid == 0) fl.waited = it + 1;
        __syncthreads();
        if (abort_sh) break;
        // (2) scaled x for the state update; bf16 copy of the entering state
        //     (operand of S C^T), then S *= exp(chunk total) in place
        build_xw<C>(xs, xw, xw_lo, w);
        if (warp < 4) {
            const float dec = decay[rh];
#pragma unroll 1
            for (int n0 = 0; n0 < C::N; n0 += 16) {
                float v[16];
                tmem_ld16(tmem + lane_off + C::COL_S + n0, v);
                tmem_ld_wait();
                uint8_t *dst = scr + (n0 / 64) * (C::M * 128);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int col = (n0 % 64) + jj * 8;
                    uint4 pk;
                    pk.x = pack_bf16x2(v[jj * 8 + 0], v[jj * 8 + 1]);
                    pk.y = pack_bf16x2(v[jj * 8 + 2], v[jj * 8 + 3]);
                    pk.z = pack_bf16x2(v[jj * 8 + 4], v[jj * 8 + 5]);
                    pk.w = pack_bf16x2(v[jj * 8 + 6], v[jj * 8 + 7]);
                    *reinterpret_cast<uint4 *>(dst + swz128(row, col)) = pk;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] *= dec;
                tmem_st16(tmem + lane_off + C::COL_S + n0, v);
            }
            tmem_st_wait();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // (3) C B^T, the inter-chunk term S C^T, and S += (w o x)^T B
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sx = smem_u32(xs), sb = smem_u32(bs), sc = smem_u32(cs), ss = smem_u32(scr);
            const uint32_t sw = smem_u32(xw);
            const uint32_t id_cb = idesc_bf16(C::Q, C::Q, false, false);
#pragma unroll
            for (int ks = 0; ks < C::N / 16; ++ks) {
                const uint32_t koff = (ks / 4) * (C::Q * 128) + (ks % 4) * 32;
                mma_bf16(tmem + C::COL_CB, sdesc(sc + koff, 16, 1024), sdesc(sb + koff, 16, 1024), id_cb, ks > 0);
            }
            const uint32_t id_inter = idesc_bf16(C::M, C::Q, false, false);
#pragma unroll
            for (int ks = 0; ks < C::N / 16; ++ks) {
                const uint32_t aoff = (ks / 4) * (C::M * 128) + (ks % 4) * 32;
                const uint32_t boff = (ks / 4) * (C::Q * 128) + (ks % 4) * 32;
                mma_bf16(tmem + C::COL_R3, sdesc(ss + aoff, 16, 1024), sdesc(sc + boff, 16, 1024), id_inter, ks > 0);
            }
            const uint32_t id_state = idesc_bf16(C::M, C::N, true, true);
            const uint32_t swl = smem_u32(xw_lo);
#pragma unroll
            for (int ks = 0; ks < C::Q / 16; ++ks)
                mma_bf16(tmem + C::COL_S, sdesc(sw + ks * 2048, C::Q * 128, 1024),
                         sdesc(sb + ks * 2048, C::Q * 128, 1024), id_state, true);
#pragma unroll
            for (int ks = 0; ks < C::Q / 16; ++ks)
                mma_bf16(tmem + C::COL_S, sdesc(swl + ks * 2048, C::Q * 128, 1024),
                         sdesc(sb + ks * 2048, C::Q * 128, 1024), id_state, true);
            (void)sx;
            mma_commit(&mma_bar);
            fl.mma = true;
        }
        if (!mbar_wait(&mma_bar, fl.mma_phase, kWaitPolls)) abort_sh = 1;
        else if (tid == 0) fl.mma = false;
        fl.mma_phase ^= 1;
        tc_fence_after();
        __syncthreads();
        if (abort_sh) break;
        // (4) masked, decayed score matrix of each head, bf16, into scr
        {
            const int half = warp >> 2;  // warps 0-3: first half of the s columns, 4-7: second half
            int t;
            bool active;
            if (C::Q == 64) {
                t = quarter * 16 + lane;  // M = 64 accumulator: 16 rows per lane quarter
                active = lane < 16;
            } else {
                t = quarter * 32 + lane;
                active = true;
            }
#pragma unroll 1
            for (int s0 = half * (C::Q / 2); s0 < (half + 1) * (C::Q / 2); s0 += 16) {
                float cb[16];
                tmem_ld16(tmem + lane_off + C::COL_CB + s0, cb);
                tmem_ld_wait();
                if (active) {
#pragma unroll
                    for (int hh = 0; hh < C::HB; ++hh) {
                        const float ct = cum[hh * C::Q + t];
                        uint8_t *dst = scr + hh * (C::Q * C::Q * 2) + (s0 / 64) * (C::Q * 128);
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            float m[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int s = s0 + jj * 8 + j;
                                m[j] = (s <= t) ? cb[jj * 8 + j] * __expf(ct - cum[hh * C::Q + s]) * dtv[hh * C::Q + s]
                                                : 0.f;
                            }
                            uint4 pk;
                            pk.x = pack_bf16x2(m[0], m[1]);
                            pk.y = pack_bf16x2(m[2], m[3]);
                            pk.z = pack_bf16x2(m[4], m[5]);
                            pk.w = pack_bf16x2(m[6], m[7]);
                            *reinterpret_cast<uint4 *>(dst + swz128(t, (s0 % 64) + jj * 8)) = pk;
                        }
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // (5) intra-chunk term per head: Y_h^T = X^T M_h^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sx = smem_u32(xs), ss = smem_u32(scr);
            const uint32_t id_intra = idesc_bf16(C::M, C::Q, true, false);
#pragma unroll
            for (int hh = 0; hh < C::HB; ++hh)
#pragma unroll
                for (int ks = 0; ks < C::Q / 16; ++ks) {
                    const uint32_t boff = hh * (C::Q * C::Q * 2) + (ks / 4) * (C::Q * 128) + (ks % 4) * 32;
                    mma_bf16(tmem + C::COL_R + hh * C::Q, sdesc(sx + ks * 2048, C::Q * 128, 1024),
                             sdesc(ss + boff, 16, 1024), id_intra, ks > 0);
                }
            mma_commit(&mma_bar);
            fl.mma = true;
        }
        if (!mbar_wait(&mma_bar, fl.mma_phase, kWaitPolls)) abort_sh = 1;
        else if (tid == 0) fl.mma = false;
        fl.mma_phase ^= 1;
        tc_fence_after();
        __syncthreads();
        if (abort_sh) break;
        // (6) epilogue: y = intra + exp(cum) * inter + D x, rows (head, p)
        {
            const int half = warp >> 2;
            const uint8_t *xrow = xs + (rh * C::PB + rp / 64) * (C::Q * 128);
            const int pc = rp % 64;
            const long long ybase = (((long long)b * L + (long long)c * C::Q) * H + hrow) * C::P + rp;
#pragma unroll 1
            for (int t0 = half * (C::Q / 2); t0 < (half + 1) * (C::Q / 2); t0 += 16) {
                float ri[16], re[16];
                tmem_ld16(tmem + lane_off + C::COL_R + rh * C::Q + t0, ri);
                tmem_ld16(tmem + lane_off + C::COL_R3 + t0, re);
                tmem_ld_wait();
                if (hrow < H) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = t0 + j;
                        const float xv = __bfloat162float(*reinterpret_cast<const bf16 *>(xrow + swz128(t, pc)));
                        const float yv = ri[j] + ecum[rh * C::Q + t] * re[j] + dh_row * xv;
                        const long long off = ybase + (long long)t * H * C::P;
                        if (prm.y_f32)
                            reinterpret_cast<float *>(prm.y)[off] = yv;
                        else
                            reinterpret_cast<bf16 *>(prm.y)[off] = __float2bfloat16_rn(yv);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (C::STAGES == 1 && tid == 0 && it + 1 < nch) {
            issue_chunk_loads<C>(stages, &full_bar[0], &mx, &mb, &mc, h0, g, c + 1, b, true);
            fl.issued = it + 2;
        }
    }
    __syncthreads();
    if (abort_sh) {
        if (tid == 0) {
            flag_timeout(prm.status);
            drain<C::STAGES>(fl, full_bar, &mma_bar);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, 512);
        return;
    }
    // final state: the last segment's TMEM state after its last chunk
    if (seg == prm.nseg - 1 && prm.fin && warp < 4) {
        tc_fence_after();
        float *dst = prm.fin + (((long long)b * H + hrow) * C::P + rp) * C::N;
#pragma unroll 1
        for (int n0 = 0; n0 < C::N; n0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_off + C::COL_S + n0, v);
            tmem_ld_wait();
            if (hrow < H)
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4 *>(dst + n0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 4-D bf16 map over [d3][d2][d1][d0] (d0 innermost), box (64, 1, Q, 1),
// 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3, uint32_t Q) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[4] = {d0, d1, d2, d3};
    cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
    cuuint32_t box[4] = {64, 1, Q, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int nseg, cps, nhb;
};

template <class C>
Plan plan_for(const Dims &d) {
    Plan p;
    p.nhb = (int)((d.H + C::HB - 1) / C::HB);
    const long long units = d.b * p.nhb;
    int nseg = (int)(kTargetCtas / units);
    if (nseg < 1) nseg = 1;
    if (nseg > d.nc) nseg = (int)d.nc;
    p.cps = (int)((d.nc + nseg - 1) / nseg);
    p.nseg = (int)((d.nc + p.cps - 1) / p.cps);
    return p;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

template <class C>
size_t workspace_for(const Dims &d) {
    const Plan p = plan_for<C>(d);
    size_t bytes = 256;  // status word
    if (p.nseg > 1)
        bytes += align256(sizeof(float) * d.b * p.nseg * d.H * C::P * C::N) + align256(sizeof(float) * d.b * p.nseg * d.H);
    return bytes;
}

template <class C>
cudaError_t run_fwd(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B,
                    const void *Cm, const float *D, const float *init, void *y, float *fin, void *ws,
                    cudaStream_t s) {
    const Plan p = plan_for<C>(d);
    CUtensorMap mx, mb, mc;
    if (!make_map(&mx, x, d.P, d.H, d.L, d.b, C::Q) || !make_map(&mb, B, d.N, d.G, d.L, d.b, C::Q) ||
        !make_map(&mc, Cm, d.N, d.G, d.L, d.b, C::Q))
        return cudaErrorInvalidValue;
    TcParams prm;
    prm.dt = static_cast<const bf16 *>(dt);
    prm.A = A;
    prm.D = D;
    prm.init = init;
    prm.y = y;
    prm.fin = fin;
    char *w = static_cast<char *>(ws);
    prm.status = reinterpret_cast<unsigned *>(w);
    prm.seg_state = nullptr;
    prm.seg_tot = nullptr;
    if (p.nseg > 1) {
        prm.seg_state = reinterpret_cast<float *>(w + 256);
        prm.seg_tot = reinterpret_cast<float *>(w + 256 + align256(sizeof(float) * d.b * p.nseg * d.H * C::P * C::N));
    }
    prm.b = d.b;
    prm.L = d.L;
    prm.H = d.H;
    prm.G = d.G;
    prm.hpg = d.hpg;
    prm.nc = (int)d.nc;
    prm.nseg = p.nseg;
    prm.cps = p.cps;
    prm.y_f32 = ydtype == SSD_DTYPE_F32 ? 1 : 0;

    // raise each kernel's dynamic shared memory limit to what this call needs
    static int scan_attr = 0, seg_attr = 0;
    const int seg_smem = C::SMEM_SEG_BASE + (int)(C::HB * p.cps * sizeof(float));
    if (scan_attr < C::SMEM_SCAN) {
        cudaError_t e = cudaFuncSetAttribute(chunk_scan_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_SCAN);
        if (e != cudaSuccess) return e;
        scan_attr = C::SMEM_SCAN;
    }
    if (p.nseg > 1 && seg_attr < seg_smem) {
        cudaError_t e = cudaFuncSetAttribute(seg_state_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             seg_smem);
        if (e != cudaSuccess) return e;
        seg_attr = seg_smem;
    }
    if (seg_smem > kSmemLimit) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(prm.status, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    timing_begin(s);
    if (p.nseg > 1) {
        dim3 grid(p.nseg - 1, p.nhb, (unsigned)d.b);
        seg_state_kernel<C><<<grid, kThreads, seg_smem, s>>>(mx, mb, prm);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        timing_mark(s, "seg_state_tc");
    }
    dim3 grid(p.nseg, p.nhb, (unsigned)d.b);
    chunk_scan_kernel<C><<<grid, kThreads, C::SMEM_SCAN, s>>>(mx, mb, mc, prm);
    e = cudaGetLastError();
    timing_mark(s, "chunk_scan_tc");
    return e;
}

// Dispatch over the compiled tile configurations.
template <class F>
bool dispatch(const Dims &d, F &&f) {
    if (d.P == 64 && d.N == 128 && d.Q == 64) return f(Cfg<64, 128, 64>{}), true;
    if (d.P == 64 && d.N == 128 && d.Q == 128) return f(Cfg<64, 128, 128>{}), true;
    if (d.P == 128 && d.N == 256 && d.Q == 64) return f(Cfg<128, 256, 64>{}), true;
    if (d.P == 64 && d.N == 64 && d.Q == 64) return f(Cfg<64, 64, 64>{}), true;
    return false;
}

}  // namespace

bool tc_fwd_supported(const Dims &d, ssd_dtype_t dtype) {
    if (dtype != SSD_DTYPE_BF16) return false;
    if (d.L == 0 || d.b == 0) return false;
    bool ok = false;
    dispatch(d, [&](auto c) {
        using C = decltype(c);
        ok = C::SCAN_FITS && C::TMEM_FITS && (d.G == 1 || d.hpg % C::HB == 0) && d.L < (1ll << 31) &&
             d.H < (1 << 30) && d.b < (1 << 30);
        if (ok) {
            const Plan p = plan_for<C>(d);
            ok = C::SMEM_SEG_BASE + (int)(C::HB * p.cps * sizeof(float)) <= kSmemLimit;
        }
    });
    return ok;
}

size_t tc_fwd_workspace(const Dims &d) {
    size_t bytes = 0;
    dispatch(d, [&](auto c) { bytes = workspace_for<decltype(c)>(d); });
    return bytes;
}

cudaError_t tc_fwd(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B,
                   const void *C, const float *D, const float *init, void *y, float *fin, void *ws,
                   cudaStream_t s) {
    cudaError_t e = cudaErrorNotSupported;
    dispatch(d, [&](auto c) { e = run_fwd<decltype(c)>(d, ydtype, x, dt, A, B, C, D, init, y, fin, ws, s); });
    return e;
}

bool tc_stage_supported(const Dims &, ssd_dtype_t) { return false; }
cudaError_t tc_chunk_state(const Dims &, const void *, const void *, const void *, const float *, float *,
                           cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t tc_chunk_scan(const Dims &, ssd_dtype_t, const void *, const void *, const void *, const void *,
                          const float *, const float *, const float *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace ssd
