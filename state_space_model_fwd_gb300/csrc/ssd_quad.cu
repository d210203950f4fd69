// ssd_quad.cu -- the quadratic (dual) form of the SSD forward pass on tcgen05,
// for short sequences.
//
// Per head, with cum_t the running sum of dt*A over the whole sequence
// (no chunking) and the decay matrix L_ts = exp(cum_t - cum_s) for s <= t:
//   y     = (L o C B^T) (dt o x) + (exp(cum) o C) init^T + D x
//   final = sum_s exp(cum_{L-1} - cum_s) dt_s x_s^T B_s + exp(cum_{L-1}) init
// (the attention-like form that can beat the chunked algorithm on short
// sequences: the da_be19 thread, post 5/6; its equations are those of the
// quadratic dual form of the SSD layer).
//
// One CTA per (128-step output tile i, head block, batch); a head block is
// HB = 128 / P heads of one group, so every state-shaped contraction has
// M = 128 rows.  The CTA walks the s-tiles j <= i:
//   S   = C_i B_j^T                 (tcgen05, M = 128 t, N = 128 s, K = N)
//   M_h = S o L_h o dt_h            (SIMT: per head mask and decay, as bf16
//                                    hi + lo parts, one after the other)
//   Y_h += M_h x_{j,h}              (tcgen05, K = 128 s, per part)
// plus, once, R_h = C_i init_h^T (init split into bf16 hi + lo), and
// y = Y + exp(cum_t) R + D x.  The CTA of the last tile also forms the final
// state: Fin += (w o x_j)^T B_j, the A operand (bf16 hi + lo) in TMEM.
// Each head's masked scores are computed once, both bf16 parts written (the
// lo part into the init tiles' region, free once R is complete), and the
// MMAs of the two parts issued together.  Score blocks that the mask or the
// sequence end zero out wholly are written as zeros without reading S, and
// the MMAs stop at the last K step holding a step before L.  The y and
// final-state tiles leave through shared memory so that the global stores
// are coalesced.
// Everything is single-buffered and phase by phase; every wait is bounded.
#include <cudaTypedefs.h>

#include "ssd_common.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kQT = 128;             // steps per tile
constexpr int kQuadThreads = 512;    // 16 warps: four per TMEM lane quarter
constexpr int kQuadMaxL = 1024;
constexpr uint64_t kQWaitNs = 100000000ull;

// Phase timestamps of CTA (0, 0, 0) (trace builds only; compiled out
// otherwise): %globaltimer at the marked points.
#ifdef SSD_TRACE
__device__ long long g_quad_trace[64];
#define QMARK(k)                                                                                  \
    do {                                                                                          \
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (k) < 64) \
            g_quad_trace[k] = (long long)globaltimer_ns();                                        \
    } while (0)
#else
#define QMARK(k) \
    do {         \
    } while (0)
#endif

template <int P_, int N_>
struct QCfg {
    static constexpr int P = P_, N = N_, HB = 128 / P;
    static constexpr int CT = kQT * N * 2;          // C or B tile: [N/64][128 rows][64] bf16
    static constexpr int XB = kQT * 64 * 2;         // one head's 64-wide x block: [128 s][64]
    static constexpr int XT = HB * (P / 64) * XB;   // x of the head block
    static constexpr int MS = kQT * kQT * 2;        // masked scores of one head: [2][128 t][64 s]
    static constexpr int IT = kQT * N * 2;          // init hi or lo: [N/64][128 rows (head, p)][64]
    static constexpr int OFF_C = 0, OFF_B = CT, OFF_X = 2 * CT, OFF_MS = OFF_X + XT, OFF_IHI = OFF_MS + MS,
                         OFF_ILO = OFF_IHI + IT, OFF_VEC = OFF_ILO + IT;
    static constexpr int VEC = HB * 2 * kQuadMaxL * 4;  // cum, dt per head
    static constexpr int SMEM = OFF_VEC + VEC + 1024;
    // TMEM: S (later the final state's A operand) | Y | R | Fin
    static constexpr uint32_t T_S = 0, T_Y = 128, T_R = 256, T_F = 384;
};

struct QuadParams {
    const bf16 *x, *dt;
    const float *A, *D, *init;
    void *y;
    float *fin;
    unsigned *status;
    long long L, H;
    int hpg, nt;
};

// Phase-tracked bounded wait of thread 0 (it spins on the non-blocking test:
// the other threads wait at the CTA barrier and take no issue slots); the
// outcome reaches every thread.
__device__ __forceinline__ bool spin_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t k = 0;; ++k) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((k & 63) == 63 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t &phase, volatile int *ok) {
    if (threadIdx.x == 0) {
        if (*ok && !spin_wait(bar, phase & 1, kQWaitNs)) *ok = 0;
        ++phase;
    }
    __syncthreads();
    return *ok != 0;
}

template <class Q, typename YT>
__global__ void __launch_bounds__(kQuadThreads, 1)
    quad_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mb,
                const __grid_constant__ CUtensorMap mc, QuadParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *cs = smem + Q::OFF_C, *bs = smem + Q::OFF_B, *xs = smem + Q::OFF_X, *ms = smem + Q::OFF_MS;
    uint8_t *ihi = smem + Q::OFF_IHI, *ilo = smem + Q::OFF_ILO;
    float *cum = reinterpret_cast<float *>(smem + Q::OFF_VEC);      // [HB][kQuadMaxL]
    float *dts = cum + Q::HB * kQuadMaxL;                           // [HB][kQuadMaxL]
    __shared__ uint64_t tma_bar, mma_bar;
    __shared__ uint32_t tmem_sh;
    __shared__ volatile int ok_sh;
    __shared__ float part_sh[Q::HB][kQuadThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = blockIdx.x, hb = blockIdx.y, b = blockIdx.z;
    const int h0 = hb * Q::HB;
    const int g = h0 / prm.hpg;
    const long long L = prm.L, H = prm.H;
    const int t0 = i * kQT;
    const bool do_fin = prm.fin && i == prm.nt - 1;
    const int steps = (do_fin ? prm.nt : i + 1) * kQT;  // steps whose decay this CTA needs
    const int q4 = warp & 3, cq = warp >> 2;            // lane quarter; quarter of the columns
    const int r = q4 * 32 + lane;                        // TMEM lane of this thread
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;

    QMARK(0);
    if (warp == 0) {
        tmem_alloc(&tmem_sh, 512);
        tmem_relinquish();
    }
    QMARK(1);
    if (tid == 0) {
        mbar_init(&tma_bar, 1);
        mbar_init(&mma_bar, 1);
        fence_mbar_init();
        ok_sh = 1;
        // the first loads go out before the decay and init set-up below: C of
        // this output tile, then B and x of the first s-tile
        mbar_arrive_expect_tx(&tma_bar, Q::CT);
        for (int nb = 0; nb < Q::N / 64; ++nb) tma_load_4d(cs + nb * (kQT * 128), &mc, &tma_bar, nb * 64, g, t0, b);
        mbar_arrive_expect_tx(&mma_bar, Q::CT + Q::XT);
        for (int nb = 0; nb < Q::N / 64; ++nb) tma_load_4d(bs + nb * (kQT * 128), &mb, &mma_bar, nb * 64, g, 0, b);
        for (int hh = 0; hh < Q::HB; ++hh)
            for (int pb = 0; pb < Q::P / 64; ++pb)
                tma_load_5d(xs + (hh * (Q::P / 64) + pb) * Q::XB, &mx, &mma_bar, 0, pb, h0 + hh, 0, b);
    }
    // ---- dt and the running sum of dt*A over the steps this CTA needs
    // (steps past L: dt = 0), per head: thread k takes steps 2k, 2k + 1
    for (int hh = 0; hh < Q::HB; ++hh) {
        const long long h = h0 + hh;
        const float a = prm.A[h];
        float v[2], run = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const long long s = 2 * tid + k;
            const float d = (s < L && s < steps) ? __bfloat162float(prm.dt[((long long)b * L + s) * H + h]) : 0.f;
            dts[hh * kQuadMaxL + s] = d;
            run += d * a;
            v[k] = run;
        }
        float tot = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, tot, off);
            if (lane >= off) tot += o;
        }
        if (lane == 31) part_sh[hh][warp] = tot;
        __syncthreads();
        float pre = 0.f;
        for (int w = 0; w < warp; ++w) pre += part_sh[hh][w];
        const float excl = pre + tot - run;
#pragma unroll
        for (int k = 0; k < 2; ++k) cum[hh * kQuadMaxL + 2 * tid + k] = v[k] + excl;
        __syncthreads();
    }
    // ---- the initial states as bf16 hi + lo, K-major: row (head, p), n; the
    // block's rows are consecutive in global memory, so consecutive threads
    // take consecutive 8-float pieces (coalesced loads)
    if (prm.init) {
        const float *src = prm.init + ((long long)b * H + h0) * Q::P * Q::N;
#pragma unroll 1
        for (int idx = tid; idx < 128 * (Q::N / 8); idx += kQuadThreads) {
            const int rr = idx / (Q::N / 8), n8 = (idx % (Q::N / 8)) * 8;
            const float4 a0 = __ldg(reinterpret_cast<const float4 *>(src + (long long)rr * Q::N + n8));
            const float4 a1 = __ldg(reinterpret_cast<const float4 *>(src + (long long)rr * Q::N + n8 + 4));
            const float v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            uint4 hi, lo;
            uint32_t *hp = &hi.x, *lp = &lo.x;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                hp[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
                lp[k] = pack_bf16x2(v[2 * k] - __uint_as_float(hp[k] << 16),
                                    v[2 * k + 1] - __uint_as_float(hp[k] & 0xFFFF0000u));
            }
            const uint32_t off = (uint32_t)(n8 / 64) * (kQT * 128) + swz128((uint32_t)rr, (uint32_t)(n8 % 64));
            *reinterpret_cast<uint4 *>(ihi + off) = hi;
            *reinterpret_cast<uint4 *>(ilo + off) = lo;
        }
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;
    uint32_t tph = 0, mph = 0;  // barrier phases (thread 0)
    const uint64_t dC = sdesc(smem_u32(cs), 16, 1024), dB = sdesc(smem_u32(bs), 16, 1024);
    // the masked scores' hi part goes to ms, the lo part to ms2: the region of
    // the init tiles, whose MMAs (R) completed with the first score MMAs
    uint8_t *ms2 = ihi;
    const uint64_t dBmn = sdesc(smem_u32(bs), kQT * 128, 1024), dM = sdesc(smem_u32(ms), 16, 1024),
                   dM2 = sdesc(smem_u32(ms2), 16, 1024);
    bool ok = true;

    QMARK(2);
    // ---- C of this output tile (loaded above); R_h = C init_h^T
    ok = cta_wait(&tma_bar, tph, &ok_sh);
    QMARK(3);
    if (ok && prm.init && elect_lane0() && warp == 0) {
        tc_fence_after();
        for (int hh = 0; hh < Q::HB; ++hh) {
            const uint64_t dhi = sdesc(smem_u32(ihi + hh * Q::P * 128), 16, 1024);
            const uint64_t dlo = sdesc(smem_u32(ilo + hh * Q::P * 128), 16, 1024);
            const uint32_t id = idesc_bf16(128, Q::P, false, false);
            const uint32_t tr = tmem + Q::T_R + hh * Q::P;
#pragma unroll
            for (int ks = 0; ks < Q::N / 16; ++ks) {
                const uint32_t adv = (ks / 4) * (kQT * 128) + (ks % 4) * 32;
                mma_bf16(tr, desc_add(dC, adv), desc_add(dhi, adv), id, ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < Q::N / 16; ++ks) {
                const uint32_t adv = (ks / 4) * (kQT * 128) + (ks % 4) * 32;
                mma_bf16(tr, desc_add(dC, adv), desc_add(dlo, adv), id, true);
            }
        }
    }

    // ---- the s-tiles j <= i
    for (int j = 0; ok && j <= i; ++j) {
        if (j == 0) {
            // the first s-tile was loaded at the start, on the MMA barrier
            // (its first phase; no MMA has been committed yet)
            if (!(ok = cta_wait(&mma_bar, mph, &ok_sh))) break;
            QMARK(4);
        } else {
            if (tid == 0) {
                mbar_arrive_expect_tx(&tma_bar, Q::CT + Q::XT);
                for (int nb = 0; nb < Q::N / 64; ++nb)
                    tma_load_4d(bs + nb * (kQT * 128), &mb, &tma_bar, nb * 64, g, j * kQT, b);
                for (int hh = 0; hh < Q::HB; ++hh)
                    for (int pb = 0; pb < Q::P / 64; ++pb)
                        tma_load_5d(xs + (hh * (Q::P / 64) + pb) * Q::XB, &mx, &tma_bar, 0, pb, h0 + hh, j * kQT, b);
            }
            if (!(ok = cta_wait(&tma_bar, tph, &ok_sh))) break;
        }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
            for (int ks = 0; ks < Q::N / 16; ++ks) {
                const uint32_t adv = (ks / 4) * (kQT * 128) + (ks % 4) * 32;
                mma_bf16(tmem + Q::T_S, desc_add(dC, adv), desc_add(dB, adv), id, ks > 0);
            }
            mma_commit(&mma_bar);
        }
        if (!(ok = cta_wait(&mma_bar, mph, &ok_sh))) break;
        QMARK(5 + 8 * j);
        tc_fence_after();
        for (int hh = 0; ok && hh < Q::HB; ++hh) {
            // M_h[t, s] = S[t, s] exp(cum_t - cum_s) dt_s for s <= t < L; this
            // thread: row t = t0 + r, columns s = 32 cq .. + 31 of the K-major
            // score tile (64-wide block cq / 2).  M is rounded to bf16 hi + lo
            // (together about 2^-17 relative), computed once: hi into ms, lo
            // into ms2, then the MMAs of both parts into Y.
            const float *ch = cum + hh * kQuadMaxL, *dh = dts + hh * kQuadMaxL;
            const long long t = t0 + r;
            const float ct = ch[t0 + r];
            const int blk = cq >> 1, cb = (cq & 1) * 32;
            uint8_t *mhi = ms + blk * (kQT * 128), *mlo = ms2 + blk * (kQT * 128);
#pragma unroll 1
            for (int c0 = cb; c0 < cb + 32; c0 += 16) {
                uint32_t wh[8], wl[8];
                // (warp-uniform) every step of the group after every row of the
                // warp, or every row at or past L: zeros, no scores read
                const long long s_lo = (long long)j * kQT + blk * 64 + c0;
                const long long t_lo = t0 + 32 * q4, t_hi = t_lo + 31;
                if (s_lo > t_hi || t_lo >= L) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) wh[k] = wl[k] = 0u;
                } else {
                float v[16];
                tmem_ld16(tmem + lane_off + Q::T_S + blk * 64 + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float m2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int sl = blk * 64 + c0 + 2 * k + e;
                        const long long s = (long long)j * kQT + sl;
                        m2[e] = (s <= t && t < L) ? v[2 * k + e] * __expf(ct - ch[s]) * dh[s] : 0.f;
                    }
                    const uint32_t hw = pack_bf16x2(m2[0], m2[1]);
                    wh[k] = hw;
                    wl[k] = pack_bf16x2(m2[0] - __uint_as_float(hw << 16), m2[1] - __uint_as_float(hw & 0xFFFF0000u));
                }
                }
                *reinterpret_cast<uint4 *>(mhi + swz128((uint32_t)r, (uint32_t)c0)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4 *>(mhi + swz128((uint32_t)r, (uint32_t)(c0 + 8))) =
                    make_uint4(wh[4], wh[5], wh[6], wh[7]);
                *reinterpret_cast<uint4 *>(mlo + swz128((uint32_t)r, (uint32_t)c0)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                *reinterpret_cast<uint4 *>(mlo + swz128((uint32_t)r, (uint32_t)(c0 + 8))) =
                    make_uint4(wl[4], wl[5], wl[6], wl[7]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            QMARK(6 + 8 * j + 2 * hh);
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, false, true);
                // K steps whose 16 columns all lie at or past L hold zeros
                const long long left = L - (long long)j * kQT;
                const int nks = left >= kQT ? kQT / 16 : (int)((left + 15) / 16);
                for (int part = 0; part < 2; ++part) {
                    const uint64_t dm = part == 0 ? dM : dM2;
                    for (int pb = 0; pb < Q::P / 64; ++pb) {
                        const uint64_t dx = sdesc(smem_u32(xs + (hh * (Q::P / 64) + pb) * Q::XB), kQT * 128, 1024);
                        const uint32_t ty = tmem + Q::T_Y + hh * Q::P + pb * 64;
                        for (int ks = 0; ks < nks; ++ks) {
                            const uint32_t adv = (ks / 4) * (kQT * 128) + (ks % 4) * 32;
                            if (j == 0 && part == 0)
                                mma_bf16(ty, desc_add(dm, adv), desc_add(dx, ks * 2048), id, ks > 0);
                            else
                                mma_bf16(ty, desc_add(dm, adv), desc_add(dx, ks * 2048), id, true);
                        }
                    }
                }
                mma_commit(&mma_bar);
            }
            // (both score tiles are rewritten for the next head, and S, B and
            // x for the next tile, only once these MMAs have read them)
            if (!(ok = cta_wait(&mma_bar, mph, &ok_sh))) break;
            tc_fence_after();
        }
    }

    QMARK(40);
    // ---- y = Y + exp(cum_t) R + D x for this thread's row and 32 of the
    // HB * P = 128 columns; the tile leaves through shared memory (rows padded
    // by 16 bytes: conflict-free 16-byte writes from the row-per-lane layout)
    // so that the global stores are coalesced: a row of the tile is HB P
    // consecutive outputs of y (the block's heads are adjacent)
    if (ok) {
        const long long t = t0 + r;
        const int col0 = cq * 32;                      // of the HB * P = 128 columns
        const int rh = col0 / Q::P, pc = col0 % Q::P;  // head, first p
        const long long h = h0 + rh;
        const float et = __expf(cum[rh * kQuadMaxL + t0 + r]);
        const float dd = prm.D ? prm.D[h] : 0.f;
        const uint8_t *xrow = xs + (rh * (Q::P / 64) + pc / 64) * Q::XB;  // x of the diagonal tile (j = i)
        float o[32];
#pragma unroll
        for (int c0 = 0; c0 < 32; c0 += 16) {
            float yv[16], rv[16];
            tmem_ld16(tmem + lane_off + Q::T_Y + col0 + c0, yv);
            if (prm.init) tmem_ld16(tmem + lane_off + Q::T_R + col0 + c0, rv);
            tmem_ld_wait();
            const uint32_t xc = (uint32_t)(pc % 64 + c0);  // column in the 64-wide x block
            const uint4 x0 = *reinterpret_cast<const uint4 *>(xrow + swz128((uint32_t)r, xc));
            const uint4 x1 = *reinterpret_cast<const uint4 *>(xrow + swz128((uint32_t)r, xc + 8));
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float xv = __uint_as_float((k & 1) ? (xw[k / 2] & 0xFFFF0000u) : (xw[k / 2] << 16));
                o[c0 + k] = yv[k] + (prm.init ? et * rv[k] : 0.f) + dd * xv;
            }
        }
        constexpr int ROWB = 128 * (int)sizeof(YT) + 16;  // staging row: the tile row + 16 bytes
        constexpr int CPR = 128 * (int)sizeof(YT) / 16;   // 16-byte pieces per row
        uint8_t *stg = ms;                                 // (ms and the init tiles: free once Y is complete)
        YT *ybase = reinterpret_cast<YT *>(prm.y) + ((long long)b * L * H + h0) * Q::P;
        for (int h2 = 0; h2 < 2; ++h2) {
            if ((r >> 6) == h2) {
                uint8_t *dst = stg + (r & 63) * ROWB + col0 * (int)sizeof(YT);
                if constexpr (sizeof(YT) == 4) {
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        *reinterpret_cast<float4 *>(dst + 4 * k) = make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; k += 8)
                        *reinterpret_cast<uint4 *>(dst + 2 * k) =
                            make_uint4(pack_bf16x2(o[k], o[k + 1]), pack_bf16x2(o[k + 2], o[k + 3]),
                                       pack_bf16x2(o[k + 4], o[k + 5]), pack_bf16x2(o[k + 6], o[k + 7]));
                }
            }
            __syncthreads();
            for (int idx = tid; idx < 64 * CPR; idx += kQuadThreads) {
                const int row = idx / CPR, pcs = idx % CPR;
                const long long tt = t0 + 64 * h2 + row;
                if (tt < L)
                    *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(ybase + tt * H * Q::P) + 16 * pcs) =
                        *reinterpret_cast<const uint4 *>(stg + row * ROWB + 16 * pcs);
            }
            __syncthreads();
        }
    }

    QMARK(41);
    // ---- final state: Fin = sum_j (w o x_j)^T B_j + exp(cum_{L-1}) init
    if (ok && do_fin) {
        const int rh = r / Q::P, rp = r % Q::P;  // this thread's row (head, p)
        const float *ch = cum + rh * kQuadMaxL, *dh = dts + rh * kQuadMaxL;
        const float clast = ch[L - 1];
        tc_fence_before();
        __syncthreads();
        // the s-tiles in the order i, 0, 1, .., i - 1: tile i (= nt - 1) is
        // still in shared memory from the output pass
        for (int jj = 0; ok && jj < prm.nt; ++jj) {
            const int j = jj == 0 ? i : jj - 1;
            if (jj > 0 && tid == 0) {
                mbar_arrive_expect_tx(&tma_bar, Q::CT + Q::XT);
                for (int nb = 0; nb < Q::N / 64; ++nb)
                    tma_load_4d(bs + nb * (kQT * 128), &mb, &tma_bar, nb * 64, g, j * kQT, b);
                for (int hh = 0; hh < Q::HB; ++hh)
                    for (int pb = 0; pb < Q::P / 64; ++pb)
                        tma_load_5d(xs + (hh * (Q::P / 64) + pb) * Q::XB, &mx, &tma_bar, 0, pb, h0 + hh, j * kQT, b);
            }
            if (jj > 0 && !(ok = cta_wait(&tma_bar, tph, &ok_sh))) break;
            // A operand (w o x)^T: row (head, p), steps s = 32 cq .. + 31,
            // hi at column s / 2, lo 64 columns further
            const uint8_t *xb = xs + (rh * (Q::P / 64) + rp / 64) * Q::XB;
            const uint32_t pc = (uint32_t)(rp % 64);
            uint32_t hi[16], lo[16];
            if ((long long)j * kQT + cq * 32 >= L) {  // (warp-uniform: steps at or past L)
#pragma unroll
                for (int k = 0; k < 16; ++k) hi[k] = lo[k] = 0u;
                tmem_st16u(tmem + lane_off + Q::T_S + cq * 16, hi);
                tmem_st16u(tmem + lane_off + Q::T_S + 64 + cq * 16, lo);
            } else {
                constexpr int k0 = 0;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float a2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int sl = cq * 32 + 2 * (k0 + k) + e;
                        const long long s = (long long)j * kQT + sl;
                        const float xv =
                            __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short *>(xb + swz128((uint32_t)sl, pc))
                                            << 16);
                        a2[e] = __expf(clast - ch[s]) * dh[s] * xv;
                    }
                    hi[k] = pack_bf16x2(a2[0], a2[1]);
                    lo[k] = pack_bf16x2(a2[0] - __uint_as_float(hi[k] << 16), a2[1] - __uint_as_float(hi[k] & 0xFFFF0000u));
                }
                tmem_st16u(tmem + lane_off + Q::T_S + cq * 16, hi);
                tmem_st16u(tmem + lane_off + Q::T_S + 64 + cq * 16, lo);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, Q::N, false, true);
                const long long left = L - (long long)j * kQT;  // (steps at or past L: zero operand)
                const int nks = left >= kQT ? kQT / 16 : (int)((left + 15) / 16);
                for (int ks = 0; ks < nks; ++ks) {
                    if (jj == 0)
                        mma_bf16_ta(tmem + Q::T_F, tmem + Q::T_S + ks * 8, desc_add(dBmn, ks * 2048), id, ks > 0);
                    else
                        mma_bf16_ta(tmem + Q::T_F, tmem + Q::T_S + ks * 8, desc_add(dBmn, ks * 2048), id, true);
                }
                for (int ks = 0; ks < nks; ++ks)
                    mma_bf16_ta(tmem + Q::T_F, tmem + Q::T_S + 64 + ks * 8, desc_add(dBmn, ks * 2048), id, true);
                mma_commit(&mma_bar);
            }
            if (!(ok = cta_wait(&mma_bar, mph, &ok_sh))) break;
            tc_fence_after();
        }
        if (ok) {
            // the tile [128 rows (head, p)][N] leaves through shared memory
            // (rows padded by 16 bytes), then coalesced: the block's rows of
            // the final state are consecutive in global memory
            constexpr int ROWF = Q::N * 4 + 16;
            uint8_t *stg = smem + Q::OFF_C;  // (C, B and x are free once the last MMAs completed)
#pragma unroll 1
            for (int n0 = cq * (Q::N / 4); n0 < (cq + 1) * (Q::N / 4); n0 += 16) {
                float v[16];
                tmem_ld16(tmem + lane_off + Q::T_F + n0, v);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; k += 4)
                    *reinterpret_cast<float4 *>(stg + r * ROWF + 4 * (n0 + k)) =
                        make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
            }
            __syncthreads();
            const long long base = ((long long)b * H + h0) * Q::P * Q::N;
            for (int idx = tid; idx < 128 * (Q::N / 4); idx += kQuadThreads) {
                const int row = idx / (Q::N / 4), c4 = idx % (Q::N / 4);
                float4 o = *reinterpret_cast<const float4 *>(stg + row * ROWF + 16 * c4);
                if (prm.init) {
                    const float el = __expf(cum[(row / Q::P) * kQuadMaxL + L - 1]);
                    const float4 a4 = __ldg(reinterpret_cast<const float4 *>(prm.init + base) + idx);
                    o.x = fmaf(el, a4.x, o.x);
                    o.y = fmaf(el, a4.y, o.y);
                    o.z = fmaf(el, a4.z, o.z);
                    o.w = fmaf(el, a4.w, o.w);
                }
                reinterpret_cast<float4 *>(prm.fin + base)[idx] = o;
            }
        }
    }
    QMARK(42);
    // ---- leave: let the MMAs land (bounded), free TMEM, record a timeout
    if (tid == 0) {
        mma_commit(&mma_bar);
        mbar_wait(&mma_bar, mph & 1, kQWaitNs / 5);
        if (!ok_sh && prm.status) atomicOr(prm.status, 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    QMARK(43);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// bf16 map of rank n, box `box`, 128-byte swizzle; rows past the tensor read 0.
bool tiled_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
               const cuuint32_t *box) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Q, typename YT>
cudaError_t run_quad(const Dims &d, const void *x, const void *dt, const float *A, const void *B, const void *Cm,
                     const float *D, const float *init, void *y, float *fin, unsigned *status, cudaStream_t s) {
    CUtensorMap mx, mb, mc;
    {
        // x [b][L][H][P] as (64, P/64, H, L, b); box: one 64-wide block of one head, 128 steps
        const cuuint64_t dims[5] = {64, (cuuint64_t)(d.P / 64), (cuuint64_t)d.H, (cuuint64_t)d.L, (cuuint64_t)d.b};
        const cuuint64_t str[4] = {128, (cuuint64_t)d.P * 2, (cuuint64_t)(d.P * d.H * 2), (cuuint64_t)(d.P * d.H * d.L * 2)};
        const cuuint32_t box[5] = {64, 1, 1, kQT, 1};
        if (!tiled_map(&mx, x, 5, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        // B, C [b][L][G][N] as (N, G, L, b); box (64, 1, 128, 1)
        const cuuint64_t dims[4] = {(cuuint64_t)d.N, (cuuint64_t)d.G, (cuuint64_t)d.L, (cuuint64_t)d.b};
        const cuuint64_t str[3] = {(cuuint64_t)d.N * 2, (cuuint64_t)(d.N * d.G * 2), (cuuint64_t)(d.N * d.G * d.L * 2)};
        const cuuint32_t box[4] = {64, 1, kQT, 1};
        if (!tiled_map(&mb, B, 4, dims, str, box) || !tiled_map(&mc, Cm, 4, dims, str, box))
            return cudaErrorInvalidValue;
    }
    QuadParams prm{};
    prm.x = static_cast<const bf16 *>(x);
    prm.dt = static_cast<const bf16 *>(dt);
    prm.A = A;
    prm.D = D;
    prm.init = init;
    prm.y = y;
    prm.fin = fin;
    prm.status = status;
    prm.L = d.L;
    prm.H = d.H;
    prm.hpg = d.hpg;
    prm.nt = (int)((d.L + kQT - 1) / kQT);
    static int attr = 0;
    if (attr < Q::SMEM) {
        const cudaError_t e =
            cudaFuncSetAttribute(quad_kernel<Q, YT>, cudaFuncAttributeMaxDynamicSharedMemorySize, Q::SMEM);
        if (e != cudaSuccess) return e;
        attr = Q::SMEM;
    }
    dim3 grid((unsigned)prm.nt, (unsigned)(d.H / Q::HB), (unsigned)d.b);
    quad_kernel<Q, YT><<<grid, kQuadThreads, Q::SMEM, s>>>(mx, mb, mc, prm);
    timing_mark(s, "quadratic_tc");
    return cudaGetLastError();
}

template <class F>
bool quad_dispatch(const Dims &d, F &&f) {
    if (d.P == 64 && d.N == 128) return f(QCfg<64, 128>{}), true;
    if (d.P == 64 && d.N == 64) return f(QCfg<64, 64>{}), true;
    if (d.P == 128 && d.N == 128) return f(QCfg<128, 128>{}), true;
    if (d.P == 128 && d.N == 64) return f(QCfg<128, 64>{}), true;
    return false;
}

}  // namespace

#ifdef SSD_TRACE
// (trace builds) the phase timestamps of the last quadratic-form launch
extern "C" __attribute__((visibility("default"))) int ssd_quad_trace_read(long long *out, int n) {
    return cudaMemcpyFromSymbol(out, g_quad_trace, sizeof(long long) * (n < 64 ? n : 64)) == cudaSuccess ? 0 : -1;
}
#endif

bool quad_supported(const Dims &d, ssd_dtype_t dtype) {
    if (dtype != SSD_DTYPE_BF16 || d.L < 1 || d.L > kQuadMaxL || d.b < 1 || d.b > 65535) return false;
    bool ok = false;
    quad_dispatch(d, [&](auto q) {
        using Q = decltype(q);
        ok = Q::SMEM <= 227 * 1024 && d.hpg % Q::HB == 0 && d.H / Q::HB <= 65535;
    });
    return ok;
}

cudaError_t quad_fwd(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B,
                     const void *C, const float *D, const float *init, void *y, float *fin, unsigned *status,
                     cudaStream_t s) {
    cudaError_t e = cudaErrorNotSupported;
    quad_dispatch(d, [&](auto q) {
        using Q = decltype(q);
        e = ydtype == SSD_DTYPE_F32 ? run_quad<Q, float>(d, x, dt, A, B, C, D, init, y, fin, status, s)
                                    : run_quad<Q, bf16>(d, x, dt, A, B, C, D, init, y, fin, status, s);
    });
    return e;
}

}  // namespace ssd
