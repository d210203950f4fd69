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
//       The last CTA of each (batch, head block) to finish then passes the
//       states across segments in order, leaving the state entering each
//       segment in the workspace.
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

constexpr int kTargetCtas = 148;        // about one CTA per SM of a GB300 (152 SMs)
constexpr int kSmemLimit = 226 * 1024;  // dynamic bytes; leaves room for the static mbarriers
constexpr uint64_t kWaitNs = 100000000ull;    // a wait gives up after 0.1 s
constexpr uint64_t kDrainNs = 20000000ull;    // the exit drain gives up after 0.02 s

struct TcParams {
    long long *trace;  // optional event trace of CTA (0, 0, 0) (trace builds only)
    const bf16 *x;     // [b, L, H, P] (the epilogue's D x term)
    const bf16 *dt;
    const float *A, *D, *init;
    void *y;
    float *fin;
    float *seg_state;   // [b, nseg, H, P, N]: segment-local states, then (in place) states entering segments
    float *seg_tot;     // [b, H, nseg]  total dt*A of each segment (may be null)
    const float *cum_in;    // [b, H, nc, Q] given in-chunk cumulative decay (null: computed from dt, A)
    const float *entering;  // [b, nseg, H, P, N] state entering each segment (null: init / segment pass)
    unsigned *status;   // bit 0: a wait gave up
    long long b, L, H, G;
    int hpg, nc, nseg, cps;  // cps: chunks per segment
    int nhb;
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
    static constexpr int XW_BYTES = M * Q * 2;  // one of the hi / lo halves of w x
    static constexpr int SBF_BYTES = M * N * 2; // [N/64 blocks][M rows][64]
    static constexpr int MM_BYTES = HB * Q * Q * 2;  // per head [Q/64 blocks][Q rows][64]
    // per-stage vectors, [HB][Q] each: dt, cum, w, exp(cum), u = exp(cum - r),
    // v = exp(r - cum) dt (r: the cumulative decay at mid-chunk); then per
    // head exp(chunk total) and a flag for chunks whose decay range is too
    // wide to factor in fp32
    static constexpr int V_DT = 0, V_CUM = HB * Q, V_W = 2 * HB * Q, V_ECUM = 3 * HB * Q, V_U = 4 * HB * Q,
                         V_V = 5 * HB * Q, V_DECAY = 6 * HB * Q, V_WIDE = 6 * HB * Q + HB;
    static constexpr int VEC_FLOATS = 6 * HB * Q + 32;
    // exp(cum) of two chunks, handed from the score-matrix warps to the epilogue
    static constexpr int EPI_BYTES = ((2 * HB * Q * 4 + 1023) / 1024) * 1024;

    // scan kernel: TMA stages of (x, B, C), a ring of kVecSlots vector sets,
    // 1 or 2 buffers of w x (hi + lo), the bf16 state copy, the score
    // matrices and the epilogue's exp(cum)
    static constexpr int SCAN_STAGE = X_BYTES + 2 * BC_BYTES;
    // (rounded to 1 KB: the swizzled operand tiles after it need 1024-byte alignment)
    static constexpr int VEC_RING = ((4 * VEC_FLOATS * 4 + 1023) / 1024) * 1024;
    static constexpr int scan_smem(int st, int xwb) {
        return st * SCAN_STAGE + VEC_RING + xwb * 2 * XW_BYTES + SBF_BYTES + MM_BYTES + EPI_BYTES + 1024;
    }
    static constexpr int SCAN_ST = scan_smem(2, 2) <= kSmemLimit || scan_smem(2, 1) <= kSmemLimit ? 2 : 1;
    static constexpr int SCAN_XWB = scan_smem(SCAN_ST, 2) <= kSmemLimit ? 2 : 1;
    static constexpr int SMEM_SCAN = scan_smem(SCAN_ST, SCAN_XWB);
    static constexpr bool SCAN_FITS = SMEM_SCAN <= kSmemLimit;

    // segment-state kernel: TMA stages of (x, B), two buffers of w x (hi +
    // lo), a ring of vector sets, then the chunk totals [HB][cps]
    static constexpr int SEG_STAGE = X_BYTES + BC_BYTES;
    static constexpr int seg_smem(int st) { return st * SEG_STAGE + 4 * XW_BYTES + VEC_RING + 1024 + 4096; }
    static constexpr int SEG_ST = seg_smem(4) <= kSmemLimit ? 4 : (seg_smem(3) <= kSmemLimit ? 3 : 2);
    static constexpr int SMEM_SEG_BASE = SEG_ST * SEG_STAGE + 4 * XW_BYTES + VEC_RING + 1024;  // + [HB][cps]

    // TMEM columns of the scan kernel
    static constexpr int COL_S = 0;
    static constexpr int COL_R3 = N;                 // inter-chunk term, two buffers of [M][Q]
    static constexpr int COL_R = N + 2 * Q;          // intra-chunk term per head, [M][Q] each
    static constexpr int COL_CB = N + 2 * Q + HB * Q;  // C B^T, [Q][Q]
    static constexpr int TMEM_USED = COL_CB + Q;
    static constexpr bool TMEM_FITS = TMEM_USED <= 512;
    static constexpr uint32_t SEG_TMEM = N < 32 ? 32 : N;
};

// Event trace (SSD_TRACE builds): clock64() of role events of CTA (0, 0, 0),
// trace[event * 256 + chunk].  Compiled out otherwise.
#ifdef SSD_TRACE
#define TRACE(ev, it)                                                                                  \
    do {                                                                                               \
        if (prm.trace && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (it) < 256)          \
            prm.trace[(ev) * 256 + (it)] = clock64();                                                  \
    } while (0)
#define TRACE_CTA(slot)                                                                                 \
    do {                                                                                                 \
        if (prm.trace) {                                                                                 \
            const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);             \
            if (cta_ < 1024) prm.trace[32 * 256 + 2 * cta_ + (slot)] = (long long)globaltimer_ns();       \
        }                                                                                                \
    } while (0)
#else
#define TRACE_CTA(slot) \
    do {                \
    } while (0)
#define TRACE(ev, it) \
    do {              \
    } while (0)
#endif

// ---------------------------------------------------------------------------
// waiting with a bound
// ---------------------------------------------------------------------------
__device__ __forceinline__ void flag_timeout(unsigned *status) {
    if (status) atomicOr(status, 1u);
}

// Poll `bar` for the phase of `parity`; give up after kWaitNs of wall time
// or as soon as another role has given up (abort flag), so nothing spins
// forever.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        // sleeps in hardware (up to 20 us) until the phase completes
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitNs) break;
    }
    *abort_flag = 1;
    return false;
}

// Warp-group wait: one elected thread polls, the named barrier hands the
// outcome (and the memory ordering of the completed phase) to the group.
__device__ __forceinline__ bool group_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           volatile int *slot, int bar_id, int gtid, int nthreads) {
    if (gtid == 0) *slot = wait_bounded(bar, parity, abort_flag) ? 1 : 0;
    named_bar_sync(bar_id, nthreads);
    return *slot != 0;
}

// Inclusive scan of dt*A over one chunk for one head, by one warp; returns
// the chunk total.
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

// In-chunk cumulative decay of chunk c for head h into cum[Q] (one warp):
// read from the caller's dA_cumsum when given, else the scan of dt*A.
// Returns the chunk total.
template <class C>
__device__ __forceinline__ float chunk_cum(const TcParams &prm, int b, long long h, int c, const float *dtv, float a,
                                           float *cum) {
    if (prm.cum_in) {
        const int lane = threadIdx.x & 31;
        const float *src = prm.cum_in + (((long long)b * prm.H + (h < prm.H ? h : 0)) * prm.nc + c) * C::Q;
        for (int q = lane; q < C::Q; q += 32) cum[q] = h < prm.H ? __ldg(src + q) : 0.f;
        __syncwarp();
        return cum[C::Q - 1];
    }
    const float total = warp_chunk_cumsum<C::Q>(dtv, a, cum);
    __syncwarp();
    return total;
}

// x tile scaled row-wise by w, split into two bf16 tiles whose sum carries
// the product to about 2^-17 relative: hi = bf16(w x), lo = bf16(w x - hi).
// (One bf16 rounding of w x, 2^-9 relative, is visible in the state entries
// that a single recent token dominates.)  Works on whole 16-byte chunks of
// the swizzled layout: a chunk stays in its row, so its scale is its row's.
template <class C, int NT>
__device__ __forceinline__ void build_xw(const uint8_t *xs, uint8_t *xw_hi, uint8_t *xw_lo, const float *w,
                                         int gtid) {
    constexpr int CHUNKS = (C::M / 64) * C::Q * 8;
#pragma unroll 2
    for (int i = gtid; i < CHUNKS; i += NT) {
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

// TMA loads of chunk c: x tiles of the CTA's heads, B, and (optionally) C.
// Returns the bytes the loads deliver.
template <class C>
__device__ __forceinline__ uint32_t chunk_load_bytes(bool with_c) {
    return C::X_BYTES + C::BC_BYTES * (with_c ? 2 : 1);
}

template <class C>
__device__ __forceinline__ void issue_chunk_loads(uint8_t *xs, uint8_t *bs, uint8_t *cs, uint64_t *bar,
                                                  const CUtensorMap *mx, const CUtensorMap *mb,
                                                  const CUtensorMap *mc, int h0, int g, int c, int b) {
#pragma unroll
    for (int hh = 0; hh < C::HB; ++hh)
#pragma unroll
        for (int pb = 0; pb < C::PB; ++pb)
            tma_load_4d(xs + (hh * C::PB + pb) * (C::Q * 128), mx, bar, pb * 64, h0 + hh, c * C::Q, b);
#pragma unroll
    for (int nb = 0; nb < C::N / 64; ++nb) tma_load_4d(bs + nb * (C::Q * 128), mb, bar, nb * 64, g, c * C::Q, b);
    if (cs)
#pragma unroll
        for (int nb = 0; nb < C::N / 64; ++nb)
            tma_load_4d(cs + nb * (C::Q * 128), mc, bar, nb * 64, g, c * C::Q, b);
}

// ===========================================================================
// Segment-local states (segments 0 .. nseg-2):
//   S_seg = sum_t exp(sum_{k>t in segment} dt_k A) dt_t x_t^T B_t
//   warp 0      : TMA loads of the x and B tiles (kSegStages-deep ring)
//   warp 1      : tcgen05.mma S += (w o x)^T B into TMEM
//   warp 2      : dt and the segment weights w (kVecSlots-deep ring)
//   warps 4-11  : w o x as bf16 hi + lo operand tiles (two buffers);
//                 warps 4-7 move the TMEM state to HBM at the end
// ===========================================================================
constexpr int kSegThreads = 384;
constexpr int kVecSlots = 4;

template <class C>
__global__ void __launch_bounds__(kSegThreads, 1)
    seg_state_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mb, TcParams prm) {
    constexpr int ST = C::SEG_ST, NV = kVecSlots;
    constexpr int HQ = C::HB * C::Q;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xw_base = smem + ST * C::SEG_STAGE;
    float *vec_base = reinterpret_cast<float *>(xw_base + 2 * 2 * C::XW_BYTES);
    float *tot_s = vec_base + NV * C::VEC_FLOATS;  // [HB][cps]
    __shared__ uint64_t full_bar[4], empty_bar[4], vfull_bar[NV], vempty_bar[NV], xfull_bar[2], xempty_bar[2];
    __shared__ uint64_t done_bar, drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ volatile int slot[8];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, hblk = blockIdx.y, b = blockIdx.z;
    const int h0 = hblk * C::HB;
    const int g = (int)(prm.G == 1 ? 0 : h0 / prm.hpg);
    const int c0 = seg * prm.cps;
    const int nch = min(prm.nc, c0 + prm.cps) - c0;
    const long long H = prm.H;
    auto stage_x = [&](int s) { return smem + s * C::SEG_STAGE; };
    auto stage_b = [&](int s) { return smem + s * C::SEG_STAGE + C::X_BYTES; };
    auto xw_hi = [&](int i) { return xw_base + i * 2 * C::XW_BYTES; };
    auto xw_lo = [&](int i) { return xw_base + i * 2 * C::XW_BYTES + C::XW_BYTES; };
    auto vec = [&](int v) { return vec_base + v * C::VEC_FLOATS; };

    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, C::SEG_TMEM);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&vfull_bar[i], 1);
            mbar_init(&vempty_bar[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&xfull_bar[i], 1);
            mbar_init(&xempty_bar[i], 1);
        }
        mbar_init(&done_bar, 1);
        mbar_init(&drain_bar, 1);
        fence_mbar_init();
        abort_sh = 0;
        prefetch_tmap(&mx);
        prefetch_tmap(&mb);
    }
    int nload[4] = {};  // TMA loads issued per stage (producer lane 0)
    // chunk totals of dt*A over the segment: groups of 8 threads reduce one
    // (head, chunk) pair each, in a fixed order (bitwise reproducible); the
    // loop bound is the same for every lane of a warp, so the shuffles see
    // a full warp
    {
        const int grp = tid >> 3, gl = tid & 7;
        const int npair = C::HB * nch;
        for (int j0 = (tid >> 5) * 4; j0 < npair; j0 += kSegThreads / 8) {
            const int j = j0 + (grp & 3);
            const bool valid = j < npair;
            const int hh = valid ? j / nch : 0, k = valid ? j % nch : 0;
            const long long h = h0 + hh;
            float sum = 0.f;
            if (valid && h < H && !prm.cum_in)
#pragma unroll 4
                for (int q = gl; q < C::Q; q += 8)
                    sum += __bfloat162float(prm.dt[((long long)b * prm.L + (long long)(c0 + k) * C::Q + q) * H + h]);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            if (valid && gl == 0) {
                float tot = 0.f;
                if (h < H)  // (with a given cumulative decay, A is not an input)
                    tot = prm.cum_in ? prm.cum_in[(((long long)b * H + h) * prm.nc + c0 + k) * C::Q + C::Q - 1]
                                     : sum * prm.A[h];
                tot_s[hh * prm.cps + k] = tot;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // suffix sums: tot_s[h][k] <- sum of the totals of the chunks after k
    if (tid < C::HB) {
        float run = 0.f;
        for (int k = nch - 1; k >= 0; --k) {
            const float t = tot_s[tid * prm.cps + k];
            tot_s[tid * prm.cps + k] = run;
            run += t;
        }
        const long long h = h0 + tid;
        if (h < H && prm.seg_tot) prm.seg_tot[((long long)b * H + h) * prm.nseg + seg] = run;
    }
    __syncthreads();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0)
            for (int it = 0; it < nch; ++it) {
                const int s = it % ST;
                if (it >= ST && !wait_bounded(&empty_bar[s], ((it / ST) & 1) ^ 1, &abort_sh)) break;
                mbar_arrive_expect_tx(&full_bar[s], chunk_load_bytes<C>(false));
                issue_chunk_loads<C>(stage_x(s), stage_b(s), nullptr, &full_bar[s], &mx, &mb, nullptr, h0, g, c0 + it,
                                     b);
                ++nload[s];
            }
    } else if (warp == 2) {
        // ---------------- segment weights ----------------
        constexpr int PER = HQ / 32;
        float dnext[PER];
        auto fetch_dt = [&](int c) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int idx = lane + 32 * i;
                const int hh = idx / C::Q, q = idx % C::Q;
                const long long h = h0 + hh;
                dnext[i] = h < H ? __bfloat162float(__ldg(prm.dt + ((long long)b * prm.L + (long long)c * C::Q + q) * H + h))
                                 : 0.f;
            }
        };
        fetch_dt(c0);
        for (int it = 0; it < nch; ++it) {
            const int v = it % NV;
            if (it >= NV) {
                int ok = lane == 0 ? (wait_bounded(&vempty_bar[v], ((it / NV) & 1) ^ 1, &abort_sh) ? 1 : 0) : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            }
            float *vv = vec(v);
#pragma unroll
            for (int i = 0; i < PER; ++i) vv[C::V_DT + lane + 32 * i] = dnext[i];
            __syncwarp();
            if (it + 1 < nch) fetch_dt(c0 + it + 1);
#pragma unroll
            for (int hh = 0; hh < C::HB; ++hh) {
                const long long h = h0 + hh;
                const float a = (h < H && prm.A) ? prm.A[h] : 0.f;
                float *cum = vv + C::V_CUM + hh * C::Q;
                const float *dtv = vv + C::V_DT + hh * C::Q;
                const float total = chunk_cum<C>(prm, b, h, c0 + it, dtv, a, cum);
                const float after = tot_s[hh * prm.cps + it];
                for (int q = lane; q < C::Q; q += 32)
                    vv[C::V_W + hh * C::Q + q] = __expf(after + total - cum[q]) * dtv[q];
            }
            __syncwarp();
            if (lane == 0) {
                TRACE(14, it);
                mbar_arrive(&vfull_bar[v]);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(C::M, C::N, true, true);
            for (int it = 0; it < nch; ++it) {
                const int s = it % ST, xb = it & 1;
                if (!wait_bounded(&xfull_bar[xb], (it >> 1) & 1, &abort_sh)) break;
                tc_fence_after();
                const uint32_t ah = smem_u32(xw_hi(xb)), al = smem_u32(xw_lo(xb)), b0 = smem_u32(stage_b(s));
#pragma unroll
                for (int ks = 0; ks < C::Q / 16; ++ks)
                    mma_bf16(tmem, sdesc(ah + ks * 2048, C::Q * 128, 1024), sdesc(b0 + ks * 2048, C::Q * 128, 1024),
                             idesc, (it | ks) != 0);
#pragma unroll
                for (int ks = 0; ks < C::Q / 16; ++ks)
                    mma_bf16(tmem, sdesc(al + ks * 2048, C::Q * 128, 1024), sdesc(b0 + ks * 2048, C::Q * 128, 1024),
                             idesc, true);
                mma_commit(&empty_bar[s]);
                mma_commit(&xempty_bar[xb]);
                TRACE(16, it);
            }
            mma_commit(&done_bar);  // completes once every MMA above has
        }
    } else if (warp >= 4) {
        // ---------------- w o x operand builders ----------------
        const int gtid = tid - 128;
        for (int it = 0; it < nch; ++it) {
            const int s = it % ST, v = it % NV, xb = it & 1;
            if (!group_wait(&full_bar[s], (it / ST) & 1, &abort_sh, &slot[0], 1, gtid, 256)) break;
            if (!group_wait(&vfull_bar[v], (it / NV) & 1, &abort_sh, &slot[1], 1, gtid, 256)) break;
            if (it >= 2 && !group_wait(&xempty_bar[xb], ((it >> 1) & 1) ^ 1, &abort_sh, &slot[2], 1, gtid, 256)) break;
            build_xw<C, 256>(stage_x(s), xw_hi(xb), xw_lo(xb), vec(v) + C::V_W, gtid);
            fence_async_smem();
            named_bar_sync(1, 256);
            if (gtid == 0) {
                TRACE(15, it);
                mbar_arrive(&xfull_bar[xb]);
                mbar_arrive(&vempty_bar[v]);
            }
        }
        // segment state: TMEM lane r = row (head, p)
        if (warp < 8) {
            if (group_wait(&done_bar, 0, &abort_sh, &slot[3], 2, gtid, 128)) {
                tc_fence_after();
                const int q4 = warp & 3;
                const int r = q4 * 32 + lane;
                const int hh = r / C::P, p = r % C::P;
                const long long h = h0 + hh;
                float *dst = prm.seg_state + ((((long long)b * prm.nseg + seg) * H + h) * C::P + p) * C::N;
#pragma unroll 1
                for (int n0 = 0; n0 < C::N; n0 += 32) {
                    float v0[16], v1[16];
                    tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + n0, v0);
                    tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + n0 + 16, v1);
                    tmem_ld_wait();
                    if (h < H) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            *reinterpret_cast<float4 *>(dst + n0 + j) = make_float4(v0[j], v0[j + 1], v0[j + 2], v0[j + 3]);
                            *reinterpret_cast<float4 *>(dst + n0 + 16 + j) =
                                make_float4(v1[j], v1[j + 1], v1[j + 2], v1[j + 3]);
                        }
                    }
                }
            }
        }
    }
    // let this CTA's own copies and MMAs land (they normally have) before
    // TMEM is freed and the CTA exits
    if (warp == 0 && lane == 0)
        for (int s = 0; s < ST; ++s)
            if (nload[s] > 0) mbar_wait(&full_bar[s], (uint32_t)((nload[s] - 1) & 1), kDrainNs);
    if (warp == 1 && lane == 0) {
        mma_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, kDrainNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, C::SEG_TMEM);
    if (abort_sh && tid == 0) flag_timeout(prm.status);
}

// ---------------------------------------------------------------------------
// Pass of states across segments, in place: slot s of the segment-state
// array (the local state of segment s) becomes the state entering segment
// s + 1 = exp(T_s) (state entering s) + local_s, T_s the segment's total
// dt*A.  One thread per four consecutive (p, n) of one (b, h); the loads
// of a batch of segments are issued before any of their results is stored.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) segment_pass_kernel(const float *__restrict__ init, float *seg_state,
                                                           const float *__restrict__ seg_tot, long long H, int PN,
                                                           int nseg) {
    const int PN4 = PN / 4;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    const long long h = blockIdx.y, b = blockIdx.z;
    if (e >= PN4) return;
    float4 acc = init ? __ldg(reinterpret_cast<const float4 *>(init + (b * H + h) * PN) + e)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    const int nsp = nseg - 1;
    const float *tot = seg_tot + (b * H + h) * nseg;
    constexpr int KB = 8;
    for (int s0 = 0; s0 < nsp; s0 += KB) {
        float4 v[KB];
        float ex[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k)
            if (s0 + k < nsp) {
                v[k] = __ldcg(reinterpret_cast<const float4 *>(seg_state + (((b * nseg + s0 + k) * H + h) * PN)) + e);
                ex[k] = expf(__ldcg(tot + s0 + k));
            }
#pragma unroll
        for (int k = 0; k < KB; ++k)
            if (s0 + k < nsp) {
                acc.x = fmaf(ex[k], acc.x, v[k].x);
                acc.y = fmaf(ex[k], acc.y, v[k].y);
                acc.z = fmaf(ex[k], acc.z, v[k].z);
                acc.w = fmaf(ex[k], acc.w, v[k].w);
                __stcg(reinterpret_cast<float4 *>(seg_state + (((b * nseg + s0 + k) * H + h) * PN)) + e, acc);
            }
    }
}

// Scores of a chunk whose decay range is too wide to factor in fp32: direct
// exponent per entry (rare; kept out of line so the hot loop stays small).
struct F8 {
    float v[8];
};

__device__ __noinline__ F8 wide_scores(F8 cb, const float *cum, const float *dtv, int t, int s0) {
    const float ct = cum[t];
    F8 m;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int sc = s0 + j;
        m.v[j] = sc <= t ? cb.v[j] * __expf(ct - cum[sc]) * dtv[sc] : 0.f;
    }
    return m;
}

template <typename T>
__device__ __forceinline__ void store_y(T *p, float v);
template <>
__device__ __forceinline__ void store_y<float>(float *p, float v) { __stcs(p, v); }
template <>
__device__ __forceinline__ void store_y<bf16>(bf16 *p, float v) { *p = __float2bfloat16_rn(v); }

// x[t][p] of this thread's (head, p) column for the Q steps of a chunk,
// two bf16 per register (fetched one chunk ahead, while the epilogue waits).
template <class C>
__device__ __forceinline__ void fetch_x_column(const bf16 *xg, long long stride, bool live, uint32_t (&xp)[C::Q / 2]) {
    const unsigned short *x16 = reinterpret_cast<const unsigned short *>(xg);
#pragma unroll
    for (int j = 0; j < C::Q / 2; ++j) {
        const uint32_t lo = live ? __ldg(x16 + (long long)(2 * j) * stride) : 0u;
        const uint32_t hi = live ? __ldg(x16 + (long long)(2 * j + 1) * stride) : 0u;
        xp[j] = lo | (hi << 16);
    }
}

// Epilogue of one chunk for this thread's row: TMEM row of the intra term
// (its head's buffer) and of the inter term, exp(cum) of its head, and the
// x column fetched ahead.
template <class C, typename T>
__device__ __forceinline__ void epilogue_rows(uint32_t tmem_lane, int it, int rh, const float *ecum,
                                              const uint32_t (&xp)[C::Q / 2], T *yp, long long stride, float dh,
                                              bool live) {
#pragma unroll
    for (int t0 = 0; t0 < C::Q; t0 += 16) {
        float ri[16], re[16];
        tmem_ld16(tmem_lane + C::COL_R + rh * C::Q + t0, ri);
        tmem_ld16(tmem_lane + C::COL_R3 + (it & 1) * C::Q + t0, re);
        tmem_ld_wait();
        if (live) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                const float4 e4 = *reinterpret_cast<const float4 *>(ecum + t0 + j);
                const uint32_t w0 = xp[(t0 + j) / 2], w1 = xp[(t0 + j) / 2 + 1];
                const float x0 = __uint_as_float(w0 << 16), x1 = __uint_as_float(w0 & 0xFFFF0000u);
                const float x2 = __uint_as_float(w1 << 16), x3 = __uint_as_float(w1 & 0xFFFF0000u);
                store_y<T>(yp + (long long)(t0 + j) * stride, fmaf(dh, x0, fmaf(e4.x, re[j], ri[j])));
                store_y<T>(yp + (long long)(t0 + j + 1) * stride, fmaf(dh, x1, fmaf(e4.y, re[j + 1], ri[j + 1])));
                store_y<T>(yp + (long long)(t0 + j + 2) * stride, fmaf(dh, x2, fmaf(e4.z, re[j + 2], ri[j + 2])));
                store_y<T>(yp + (long long)(t0 + j + 3) * stride, fmaf(dh, x3, fmaf(e4.w, re[j + 3], ri[j + 3])));
            }
        }
    }
}

// ===========================================================================
// Chunk scan with the state carried in TMEM (every segment).
//   warp 0     : TMA loads of x, B, C; dt (fetched a chunk ahead), cumulative
//                decay, w, exp(cum) and the factors u, v of exp(cum_t - cum_s)
//   warp 1     : tcgen05.mma issue (C B^T; S C^T; S += (w x)^T B; X^T M^T)
//   warps 4-7  : w o x operand tiles; bf16 state copy and S *= exp(total)
//   warps 8-11 : masked, decayed score matrices M_h (bf16) from C B^T
//   warps 12-15: y = intra + exp(cum) inter + D x, straight to HBM
// ===========================================================================
constexpr int kScanThreads = 512;

template <class C, typename YT>
__global__ void __launch_bounds__(kScanThreads, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mb,
                      const __grid_constant__ CUtensorMap mc, TcParams prm) {
    constexpr int ST = C::SCAN_ST;
    constexpr int XWB = C::SCAN_XWB;
    constexpr int HQ = C::HB * C::Q;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int NV = kVecSlots;
    float *vec_base = reinterpret_cast<float *>(smem + ST * C::SCAN_STAGE);
    uint8_t *xw_base = smem + ST * C::SCAN_STAGE + C::VEC_RING;
    uint8_t *sbf = xw_base + XWB * 2 * C::XW_BYTES;
    uint8_t *mm = sbf + C::SBF_BYTES;
    float *epi_vec = reinterpret_cast<float *>(mm + C::MM_BYTES);  // [2][HB][Q]
    __shared__ uint64_t full_bar[2], empty_bar[2], free_r3_bar[2], epi_bar[2], vfull_bar[NV], vempty_bar[NV];
    __shared__ uint64_t cb_bar, mask_bar, wg1_bar, state_bar, y_bar, free_r_bar, drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ volatile int slot[8];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, hblk = blockIdx.y, b = blockIdx.z;
    const int h0 = hblk * C::HB;
    const int g = (int)(prm.G == 1 ? 0 : h0 / prm.hpg);
    const int c0 = seg * prm.cps;
    const int nch = min(prm.nc, c0 + prm.cps) - c0;
    const long long L = prm.L, H = prm.H;
    auto stage_x = [&](int s) { return smem + s * C::SCAN_STAGE; };
    auto stage_b = [&](int s) { return smem + s * C::SCAN_STAGE + C::X_BYTES; };
    auto stage_c = [&](int s) { return smem + s * C::SCAN_STAGE + C::X_BYTES + C::BC_BYTES; };
    auto vec = [&](int v) { return vec_base + v * C::VEC_FLOATS; };
    auto xw_hi = [&](int i) { return xw_base + i * 2 * C::XW_BYTES; };
    auto xw_lo = [&](int i) { return xw_base + i * 2 * C::XW_BYTES + C::XW_BYTES; };

    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
            mbar_init(&free_r3_bar[i], 1);
            mbar_init(&epi_bar[i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&vfull_bar[i], 1);
            mbar_init(&vempty_bar[i], 1);
        }
        mbar_init(&cb_bar, 1);
        mbar_init(&mask_bar, 1);
        mbar_init(&wg1_bar, 1);
        mbar_init(&state_bar, 1);
        mbar_init(&y_bar, 1);
        mbar_init(&free_r_bar, 1);
        mbar_init(&drain_bar, 1);
        fence_mbar_init();
        abort_sh = 0;
        prefetch_tmap(&mx);
        prefetch_tmap(&mb);
        prefetch_tmap(&mc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        TRACE(13, 0);
        TRACE_CTA(0);
    }
    const uint32_t tmem = tmem_base_sh;
    int nload[2] = {0, 0};  // TMA loads issued per stage (producer lane 0)
    const int q4 = warp & 3;                  // TMEM lane quarter of this warp
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0)
            for (int it = 0; it < nch; ++it) {
                const int s = it % ST;
                if (it >= ST && !wait_bounded(&empty_bar[s], ((it / ST) & 1) ^ 1, &abort_sh)) break;
                mbar_arrive_expect_tx(&full_bar[s], chunk_load_bytes<C>(true));
                issue_chunk_loads<C>(stage_x(s), stage_b(s), stage_c(s), &full_bar[s], &mx, &mb, &mc, h0, g, c0 + it,
                                     b);
                ++nload[s];
                TRACE(0, it);
            }
    } else if (warp == 2) {
        // ---------------- per-chunk vectors (run up to NV chunks ahead) ----------------
        constexpr int PER = HQ / 32;
        float dnext[PER];
        auto fetch_dt = [&](int c) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int idx = lane + 32 * i;
                const int hh = idx / C::Q, q = idx % C::Q;
                const long long h = h0 + hh;
                dnext[i] = h < H ? __bfloat162float(__ldg(prm.dt + ((long long)b * L + (long long)c * C::Q + q) * H + h))
                                 : 0.f;
            }
        };
        fetch_dt(c0);
        for (int it = 0; it < nch; ++it) {
            const int v = it % NV;
            if (it >= NV) {
                int ok = lane == 0 ? (wait_bounded(&vempty_bar[v], ((it / NV) & 1) ^ 1, &abort_sh) ? 1 : 0) : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            }
            float *vv = vec(v);
#pragma unroll
            for (int i = 0; i < PER; ++i) vv[C::V_DT + lane + 32 * i] = dnext[i];
            __syncwarp();
            if (it + 1 < nch) fetch_dt(c0 + it + 1);  // in flight while this chunk's vectors are computed
#pragma unroll
            for (int hh = 0; hh < C::HB; ++hh) {
                const long long h = h0 + hh;
                const float a = (h < H && prm.A) ? prm.A[h] : 0.f;
                float *cum = vv + C::V_CUM + hh * C::Q;
                const float *dtv = vv + C::V_DT + hh * C::Q;
                const float total = chunk_cum<C>(prm, b, h, c0 + it, dtv, a, cum);
                const float r = cum[C::Q / 2 - 1];
                // exp(cum_t - cum_s) = u_t v_s / dt_s factors in fp32 only while
                // each half-chunk's decay stays within e^80
                const bool wide = (cum[0] - r) > 80.f || (r - total) > 80.f;
                for (int q = lane; q < C::Q; q += 32) {
                    const float cq = cum[q];
                    vv[C::V_W + hh * C::Q + q] = __expf(total - cq) * dtv[q];
                    vv[C::V_ECUM + hh * C::Q + q] = __expf(cq);
                    vv[C::V_U + hh * C::Q + q] = wide ? 0.f : __expf(cq - r);
                    vv[C::V_V + hh * C::Q + q] = wide ? 0.f : __expf(r - cq) * dtv[q];
                }
                if (lane == 0) {
                    vv[C::V_DECAY + hh] = __expf(total);
                    vv[C::V_WIDE + hh] = wide ? 1.f : 0.f;
                }
            }
            __syncwarp();
            if (lane == 0) {
                TRACE(1, it);
                mbar_arrive(&vfull_bar[v]);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t id_cb = idesc_bf16(C::Q, C::Q, false, false);
            const uint32_t id_inter = idesc_bf16(C::M, C::Q, false, false);
            const uint32_t id_state = idesc_bf16(C::M, C::N, true, true);
            const uint32_t id_intra = idesc_bf16(C::M, C::Q, true, false);
            for (int it = 0; it < nch; ++it) {
                const int s = it % ST;
                const int xb = XWB == 2 ? (it & 1) : 0;
                const uint32_t sx = smem_u32(stage_x(s)), sb = smem_u32(stage_b(s)), sc = smem_u32(stage_c(s));
                // C B^T: needs the chunk's tiles and the previous scores consumed
                if (!wait_bounded(&full_bar[s], (it / ST) & 1, &abort_sh)) break;
                if (it > 0 && !wait_bounded(&mask_bar, (it - 1) & 1, &abort_sh)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < C::N / 16; ++ks) {
                    const uint32_t koff = (ks / 4) * (C::Q * 128) + (ks % 4) * 32;
                    mma_bf16(tmem + C::COL_CB, sdesc(sc + koff, 16, 1024), sdesc(sb + koff, 16, 1024), id_cb, ks > 0);
                }
                mma_commit(&cb_bar);
                TRACE(2, it);
                // S C^T into inter buffer it & 1, and S += (w x)^T B: need the bf16
                // state copy, the scaled state and w x (warps 4-7), and the
                // epilogue two chunks back done with that inter buffer
                if (!wait_bounded(&wg1_bar, it & 1, &abort_sh)) break;
                if (it >= 2 && !wait_bounded(&free_r3_bar[it & 1], ((it >> 1) & 1) ^ 1, &abort_sh)) break;
                tc_fence_after();
                const uint32_t ss = smem_u32(sbf);
#pragma unroll
                for (int ks = 0; ks < C::N / 16; ++ks) {
                    const uint32_t aoff = (ks / 4) * (C::M * 128) + (ks % 4) * 32;
                    const uint32_t boff = (ks / 4) * (C::Q * 128) + (ks % 4) * 32;
                    mma_bf16(tmem + C::COL_R3 + (it & 1) * C::Q, sdesc(ss + aoff, 16, 1024),
                             sdesc(sc + boff, 16, 1024), id_inter, ks > 0);
                }
                const uint32_t swh = smem_u32(xw_hi(xb)), swl = smem_u32(xw_lo(xb));
#pragma unroll
                for (int ks = 0; ks < C::Q / 16; ++ks)
                    mma_bf16(tmem + C::COL_S, sdesc(swh + ks * 2048, C::Q * 128, 1024),
                             sdesc(sb + ks * 2048, C::Q * 128, 1024), id_state, true);
#pragma unroll
                for (int ks = 0; ks < C::Q / 16; ++ks)
                    mma_bf16(tmem + C::COL_S, sdesc(swl + ks * 2048, C::Q * 128, 1024),
                             sdesc(sb + ks * 2048, C::Q * 128, 1024), id_state, true);
                mma_commit(&state_bar);
                TRACE(3, it);
                // X^T M_h^T per head: needs the score matrices (warps 8-11) and
                // the last epilogue done with the intra buffers
                if (!wait_bounded(&mask_bar, it & 1, &abort_sh)) break;
                if (it > 0 && !wait_bounded(&free_r_bar, (it - 1) & 1, &abort_sh)) break;
                tc_fence_after();
                const uint32_t sm = smem_u32(mm);
#pragma unroll
                for (int hh = 0; hh < C::HB; ++hh)
#pragma unroll
                    for (int ks = 0; ks < C::Q / 16; ++ks) {
                        const uint32_t boff = hh * (C::Q * C::Q * 2) + (ks / 4) * (C::Q * 128) + (ks % 4) * 32;
                        mma_bf16(tmem + C::COL_R + hh * C::Q, sdesc(sx + ks * 2048, C::Q * 128, 1024),
                                 sdesc(sm + boff, 16, 1024), id_intra, ks > 0);
                    }
                mma_commit(&y_bar);
                // every read of the stage and of the vector set is done once these MMAs are
                mma_commit(&empty_bar[s]);
                mma_commit(&vempty_bar[it % NV]);
                TRACE(4, it);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- w x operands; state copy and decay ----------------
        const int gtid = tid - 128;
        const int row = q4 * 32 + lane, rh = row / C::P, rp = row % C::P;
        const long long hrow = h0 + rh;
        // state entering the segment
        {
            const float *src = nullptr;
            if (prm.entering)
                src = prm.entering + ((((long long)b * prm.nseg + seg) * H + hrow) * C::P + rp) * C::N;
            else if (seg > 0)
                src = prm.seg_state + ((((long long)b * prm.nseg + (seg - 1)) * H + hrow) * C::P + rp) * C::N;
            else if (prm.init)
                src = prm.init + (((long long)b * H + hrow) * C::P + rp) * C::N;
            if (hrow >= H) src = nullptr;
#pragma unroll 1
            for (int n0 = 0; n0 < C::N; n0 += 32) {
                float v0[16], v1[16];
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    const float4 a = src ? __ldcg(reinterpret_cast<const float4 *>(src + n0 + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 c2 = src ? __ldcg(reinterpret_cast<const float4 *>(src + n0 + 16 + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v0[j] = a.x; v0[j + 1] = a.y; v0[j + 2] = a.z; v0[j + 3] = a.w;
                    v1[j] = c2.x; v1[j + 1] = c2.y; v1[j + 2] = c2.z; v1[j + 3] = c2.w;
                }
                tmem_st16(tmem + lane_off + C::COL_S + n0, v0);
                tmem_st16(tmem + lane_off + C::COL_S + n0 + 16, v1);
            }
            tmem_st_wait();
        }
        if (gtid == 0) TRACE(13, 1);
        for (int it = 0; it < nch; ++it) {
            const int s = it % ST;
            const int xb = XWB == 2 ? (it & 1) : 0;
            if (!group_wait(&full_bar[s], (it / ST) & 1, &abort_sh, &slot[0], 1, gtid, 128)) break;
            if (!group_wait(&vfull_bar[it % NV], (it / NV) & 1, &abort_sh, &slot[7], 1, gtid, 128)) break;
            if (gtid == 0) TRACE(5, it);
            const float *vv = vec(it % NV);
            if (XWB == 1 && it > 0) {
                if (!group_wait(&state_bar, (it - 1) & 1, &abort_sh, &slot[1], 1, gtid, 128)) break;
            }
            build_xw<C, 128>(stage_x(s), xw_hi(xb), xw_lo(xb), vv + C::V_W, gtid);
            if (gtid == 0) TRACE(6, it);
            if (XWB == 2 && it > 0) {
                if (!group_wait(&state_bar, (it - 1) & 1, &abort_sh, &slot[1], 1, gtid, 128)) break;
            }
            if (gtid == 0) TRACE(7, it);
            tc_fence_after();
            const float dec = vv[C::V_DECAY + rh];
#pragma unroll 1
            for (int n0 = 0; n0 < C::N; n0 += 32) {
                float v0[16], v1[16];
                tmem_ld16(tmem + lane_off + C::COL_S + n0, v0);
                tmem_ld16(tmem + lane_off + C::COL_S + n0 + 16, v1);
                tmem_ld_wait();
                uint8_t *dst = sbf + (n0 / 64) * (C::M * 128);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float *v = jj < 2 ? v0 + jj * 8 : v1 + (jj - 2) * 8;
                    uint4 pk;
                    pk.x = pack_bf16x2(v[0], v[1]);
                    pk.y = pack_bf16x2(v[2], v[3]);
                    pk.z = pack_bf16x2(v[4], v[5]);
                    pk.w = pack_bf16x2(v[6], v[7]);
                    *reinterpret_cast<uint4 *>(dst + swz128(row, (n0 % 64) + jj * 8)) = pk;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    v0[j] *= dec;
                    v1[j] *= dec;
                }
                tmem_st16(tmem + lane_off + C::COL_S + n0, v0);
                tmem_st16(tmem + lane_off + C::COL_S + n0 + 16, v1);
            }
            fence_async_smem();
            tmem_st_wait();
            tc_fence_before();
            named_bar_sync(1, 128);
            if (gtid == 0) {
                TRACE(8, it);
                mbar_arrive(&wg1_bar);
            }
        }
        // final state after the segment's last chunk
        if (seg == prm.nseg - 1 && prm.fin) {  // (a uniform test: group_wait handles an abort)
            if (group_wait(&state_bar, (nch - 1) & 1, &abort_sh, &slot[2], 1, gtid, 128)) {
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
        }
    } else if (warp >= 8 && warp < 12) {
        // ---------------- masked, decayed score matrices ----------------
        //   M_h[t, s] = CB[t, s] exp(cum_t - cum_s) dt_s = CB[t, s] u_t v_s   (s <= t)
        // Q = 64: C B^T is an M = 64 accumulator (rows 16 q4 .. 16 q4 + 15 in
        // lanes 0-15); lanes 16-31 take the row of lane - 16 and either the
        // second head (two heads) or the second half of the columns.
        // Q = 128: lane = row, every thread covers all heads and columns.
        const int gtid = tid - 256;
        constexpr bool HALVES = C::Q == 64;
        const int t = HALVES ? q4 * 16 + (lane & 15) : q4 * 32 + lane;
        const int half = HALVES ? (lane >> 4) : 0;
        constexpr int NH = (HALVES && C::HB == 2) ? 1 : C::HB;              // heads per thread
        constexpr int NCOL = (HALVES && C::HB == 1) ? C::Q / 2 : C::Q;       // columns per thread
        for (int it = 0; it < nch; ++it) {
            if (!group_wait(&vfull_bar[it % NV], (it / NV) & 1, &abort_sh, &slot[3], 2, gtid, 128)) break;
            if (!group_wait(&cb_bar, it & 1, &abort_sh, &slot[4], 2, gtid, 128)) break;
            if (gtid == 0) TRACE(9, it);
            tc_fence_after();
            const float *vv = vec(it % NV);
#pragma unroll 1
            for (int cb0 = 0; cb0 < C::Q; cb0 += 32) {
                float cb[32];
                tmem_ld16(tmem + lane_off + C::COL_CB + cb0, *reinterpret_cast<float(*)[16]>(cb));
                tmem_ld16(tmem + lane_off + C::COL_CB + cb0 + 16, *reinterpret_cast<float(*)[16]>(cb + 16));
                tmem_ld_wait();
                if (HALVES) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) cb[j] = __shfl_sync(0xffffffffu, cb[j], lane & 15);
                }
                // (two heads: each half-warp its head; one head: each half-warp
                // its half of the columns)
                const bool mine = !(HALVES && C::HB == 1) || (cb0 / 32) == half;
#pragma unroll
                for (int hi = 0; hi < (mine ? NH : 0); ++hi) {
                    const int hh = (HALVES && C::HB == 2) ? half : hi;
                    const float *vvv = vv + C::V_V + hh * C::Q;
                    const bool wide = vv[C::V_WIDE + hh] != 0.f;
                    const float ut = vv[C::V_U + hh * C::Q + t];
                    uint8_t *dst = mm + hh * (C::Q * C::Q * 2) + (cb0 / 64) * (C::Q * 128);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        float m[8];
                        if (!wide) {
                            const float4 va = *reinterpret_cast<const float4 *>(vvv + cb0 + jj * 8);
                            const float4 vb = *reinterpret_cast<const float4 *>(vvv + cb0 + jj * 8 + 4);
                            const float vs[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int sc = cb0 + jj * 8 + j;
                                const float prod = cb[jj * 8 + j] * ut * vs[j];
                                m[j] = sc <= t ? prod : 0.f;
                            }
                        } else {
                            F8 c8;
#pragma unroll
                            for (int j = 0; j < 8; ++j) c8.v[j] = cb[jj * 8 + j];
                            const F8 r8 = wide_scores(c8, vv + C::V_CUM + hh * C::Q, vv + C::V_DT + hh * C::Q, t,
                                                      cb0 + jj * 8);
#pragma unroll
                            for (int j = 0; j < 8; ++j) m[j] = r8.v[j];
                        }
                        uint4 pk;
                        pk.x = pack_bf16x2(m[0], m[1]);
                        pk.y = pack_bf16x2(m[2], m[3]);
                        pk.z = pack_bf16x2(m[4], m[5]);
                        pk.w = pack_bf16x2(m[6], m[7]);
                        *reinterpret_cast<uint4 *>(dst + swz128(t, (cb0 % 64) + jj * 8)) = pk;
                    }
                }
                __syncwarp();
            }
            (void)NCOL;
            // exp(cum) for the epilogue (the stage may be refilled before it runs)
            for (int i = gtid; i < HQ; i += 128) epi_vec[(it & 1) * HQ + i] = vv[C::V_ECUM + i];
            fence_async_smem();
            tc_fence_before();
            named_bar_sync(2, 128);
            if (gtid == 0) {
                TRACE(10, it);
                mbar_arrive(&mask_bar);
                mbar_arrive(&epi_bar[it & 1]);
            }
        }
    } else if (warp >= 12) {
        // ---------------- epilogue ----------------
        // y = intra + exp(cum) inter + D x for row (head, p), 16 steps t at a
        // time: TMEM loads, x from L2 (the tile was just loaded), stores.
        const int gtid = tid - 384;
        const int row = q4 * 32 + lane, rh = row / C::P, rp = row % C::P;
        const long long hrow = h0 + rh;
        const bool live = hrow < H;
        const float dh = (prm.D && live) ? prm.D[hrow] : 0.f;
        const long long ystride = H * C::P;
        auto row_base = [&](int c) {
            return (((long long)b * L + (long long)c * C::Q) * H + (live ? hrow : 0)) * C::P + rp;
        };
        uint32_t xp[C::Q / 2];
        fetch_x_column<C>(prm.x + row_base(c0), ystride, live, xp);
        for (int it = 0; it < nch; ++it) {
            const int c = c0 + it;
            if (!group_wait(&y_bar, it & 1, &abort_sh, &slot[6], 3, gtid, 128)) break;
            if (!group_wait(&epi_bar[it & 1], (it >> 1) & 1, &abort_sh, &slot[5], 3, gtid, 128)) break;
            if (gtid == 0) TRACE(11, it);
            tc_fence_after();
            const float *ecum = epi_vec + (it & 1) * HQ + rh * C::Q;
            const long long base = row_base(c);
            epilogue_rows<C, YT>(tmem + lane_off, it, rh, ecum, xp, reinterpret_cast<YT *>(prm.y) + base, ystride,
                                 dh, live);
            // TMEM reads are done: let the next chunk's MMAs in, then fetch its x
            tc_fence_before();
            named_bar_sync(3, 128);
            if (gtid == 0) {
                TRACE(12, it);
                mbar_arrive(&free_r_bar);
                mbar_arrive(&free_r3_bar[it & 1]);
            }
            if (it + 1 < nch) fetch_x_column<C>(prm.x + row_base(c + 1), ystride, live, xp);
        }
    }
    // let this CTA's own copies and MMAs land (they normally have) before
    // TMEM is freed and the CTA exits
    if (warp == 0 && lane == 0)
        for (int s = 0; s < ST; ++s)
            if (nload[s] > 0) mbar_wait(&full_bar[s], (uint32_t)((nload[s] - 1) & 1), kDrainNs);
    if (warp == 1 && lane == 0) {
        mma_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, kDrainNs);
    }
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0) flag_timeout(prm.status);
    if (tid == 0) TRACE_CTA(1);
    if (warp == 1) tmem_dealloc(tmem, 512);
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

// Workspace: status word | segment states | segment totals.  The status
// word is cleared on the stream by every call.
template <class C>
size_t header_bytes(const Dims &) {
    return 256;
}

#ifdef SSD_TRACE
constexpr size_t kTraceBytes = (32 * 256 + 2048) * sizeof(long long);
#endif

template <class C>
size_t workspace_for(const Dims &d) {
    const Plan p = plan_for<C>(d);
    size_t bytes = header_bytes<C>(d);
    if (p.nseg > 1)
        bytes += align256(sizeof(float) * d.b * p.nseg * d.H * C::P * C::N) + align256(sizeof(float) * d.b * p.nseg * d.H);
#ifdef SSD_TRACE
    bytes += kTraceBytes;
#endif
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
    prm.x = static_cast<const bf16 *>(x);
    prm.dt = static_cast<const bf16 *>(dt);
    prm.A = A;
    prm.D = D;
    prm.init = init;
    prm.y = y;
    prm.fin = fin;
    char *w = static_cast<char *>(ws);
    const size_t hdr = header_bytes<C>(d);
    prm.status = reinterpret_cast<unsigned *>(w);
    prm.seg_state = nullptr;
    prm.seg_tot = nullptr;
    if (p.nseg > 1) {
        prm.seg_state = reinterpret_cast<float *>(w + hdr);
        prm.seg_tot = reinterpret_cast<float *>(w + hdr + align256(sizeof(float) * d.b * p.nseg * d.H * C::P * C::N));
    }
    prm.nhb = p.nhb;
    prm.cum_in = nullptr;
    prm.entering = nullptr;
    prm.trace = nullptr;
#ifdef SSD_TRACE
    prm.trace = reinterpret_cast<long long *>(w + workspace_for<C>(d) - kTraceBytes);
#endif
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
    auto scan_kernel = prm.y_f32 ? chunk_scan_kernel<C, float> : chunk_scan_kernel<C, bf16>;
    const int seg_smem = C::SMEM_SEG_BASE + (int)(C::HB * p.cps * sizeof(float));
    if (scan_attr < C::SMEM_SCAN) {
        cudaError_t e = cudaFuncSetAttribute(chunk_scan_kernel<C, float>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_SCAN);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chunk_scan_kernel<C, bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    cudaError_t e = cudaMemsetAsync(w, 0, hdr, s);
    if (e != cudaSuccess) return e;
    timing_begin(s);
    if (p.nseg > 1) {
        dim3 grid(p.nseg - 1, p.nhb, (unsigned)d.b);
        seg_state_kernel<C><<<grid, kSegThreads, seg_smem, s>>>(mx, mb, prm);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        timing_mark(s, "seg_state_tc");
        const int pn = (int)(C::P * C::N);
        dim3 pgrid((unsigned)((pn / 4 + 255) / 256), (unsigned)d.H, (unsigned)d.b);
        segment_pass_kernel<<<pgrid, 256, 0, s>>>(init, prm.seg_state, prm.seg_tot, d.H, pn, p.nseg);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        timing_mark(s, "segment_pass");
    }
    dim3 grid(p.nseg, p.nhb, (unsigned)d.b);
    scan_kernel<<<grid, kScanThreads, C::SMEM_SCAN, s>>>(mx, mb, mc, prm);
    e = cudaGetLastError();
    timing_mark(s, "chunk_scan_tc");
    return e;
}

// Dispatch over the compiled tile configurations.
template <class F>
bool dispatch(const Dims &d, F &&f) {
    if (d.P == 64 && d.N == 128 && d.Q == 64) return f(Cfg<64, 128, 64>{}), true;
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
             d.H < (1 << 30) && d.b < 65536;
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

bool tc_stage_supported(const Dims &d, ssd_dtype_t dtype) {
    if (dtype != SSD_DTYPE_BF16 || d.L == 0 || d.b == 0) return false;
    bool ok = false;
    dispatch(d, [&](auto c) {
        using C = decltype(c);
        ok = C::SCAN_FITS && C::TMEM_FITS && (d.G == 1 || d.hpg % C::HB == 0) && d.L < (1ll << 31) &&
             d.H < (1 << 30) && d.b < 65536 && d.nc < 65536 &&
             C::SMEM_SEG_BASE + (int)(C::HB * sizeof(float)) <= kSmemLimit;
    });
    return ok;
}

namespace {

// Parameters of a one-chunk-per-segment launch of the fused kernels, as the
// stage entry points use them.
TcParams stage_params(const Dims &d, const void *dt, const float *cum) {
    TcParams prm{};
    prm.dt = static_cast<const bf16 *>(dt);
    prm.cum_in = cum;
    prm.b = d.b;
    prm.L = d.L;
    prm.H = d.H;
    prm.G = d.G;
    prm.hpg = d.hpg;
    prm.nc = (int)d.nc;
    prm.nseg = (int)d.nc;
    prm.cps = 1;
    prm.y_f32 = 1;
    return prm;
}

template <class C>
cudaError_t run_chunk_state(const Dims &d, const void *x, const void *dt, const void *B, const float *cum,
                            float *states, cudaStream_t s) {
    CUtensorMap mx, mb;
    if (!make_map(&mx, x, d.P, d.H, d.L, d.b, C::Q) || !make_map(&mb, B, d.N, d.G, d.L, d.b, C::Q))
        return cudaErrorInvalidValue;
    TcParams prm = stage_params(d, dt, cum);
    prm.seg_state = states;  // [b, nc, H, P, N]: one segment per chunk
    prm.nhb = (int)((d.H + C::HB - 1) / C::HB);
    const int smem = C::SMEM_SEG_BASE + (int)(C::HB * sizeof(float));
    static int attr = 0;
    if (attr < smem) {
        cudaError_t e = cudaFuncSetAttribute(seg_state_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = smem;
    }
    timing_begin(s);
    dim3 grid((unsigned)d.nc, (unsigned)prm.nhb, (unsigned)d.b);
    seg_state_kernel<C><<<grid, kSegThreads, smem, s>>>(mx, mb, prm);
    const cudaError_t e = cudaGetLastError();
    timing_mark(s, "chunk_state_tc");
    return e;
}

template <class C>
cudaError_t run_chunk_scan(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const void *B,
                           const void *Cm, const float *cum, const float *states_in, const float *D, void *y,
                           cudaStream_t s) {
    CUtensorMap mx, mb, mc;
    if (!make_map(&mx, x, d.P, d.H, d.L, d.b, C::Q) || !make_map(&mb, B, d.N, d.G, d.L, d.b, C::Q) ||
        !make_map(&mc, Cm, d.N, d.G, d.L, d.b, C::Q))
        return cudaErrorInvalidValue;
    TcParams prm = stage_params(d, dt, cum);
    prm.x = static_cast<const bf16 *>(x);
    prm.entering = states_in;  // [b, nc, H, P, N]: the state entering each chunk
    prm.D = D;
    prm.y = y;
    prm.y_f32 = ydtype == SSD_DTYPE_F32 ? 1 : 0;
    prm.nhb = (int)((d.H + C::HB - 1) / C::HB);
    static int attr = 0;
    if (attr < C::SMEM_SCAN) {
        cudaError_t e = cudaFuncSetAttribute(chunk_scan_kernel<C, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_SCAN);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chunk_scan_kernel<C, bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM_SCAN);
        if (e != cudaSuccess) return e;
        attr = C::SMEM_SCAN;
    }
    auto kern = prm.y_f32 ? chunk_scan_kernel<C, float> : chunk_scan_kernel<C, bf16>;
    timing_begin(s);
    dim3 grid((unsigned)d.nc, (unsigned)prm.nhb, (unsigned)d.b);
    kern<<<grid, kScanThreads, C::SMEM_SCAN, s>>>(mx, mb, mc, prm);
    const cudaError_t e = cudaGetLastError();
    timing_mark(s, "chunk_scan_stage_tc");
    return e;
}

}  // namespace

cudaError_t tc_chunk_state(const Dims &d, const void *x, const void *dt, const void *B, const float *cum,
                           float *states, cudaStream_t s) {
    cudaError_t e = cudaErrorNotSupported;
    dispatch(d, [&](auto c) { e = run_chunk_state<decltype(c)>(d, x, dt, B, cum, states, s); });
    return e;
}

cudaError_t tc_chunk_scan(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const void *B,
                          const void *C, const float *cum, const float *states_in, const float *D, void *y,
                          cudaStream_t s) {
    cudaError_t e = cudaErrorNotSupported;
    dispatch(d, [&](auto c) { e = run_chunk_scan<decltype(c)>(d, ydtype, x, dt, B, C, cum, states_in, D, y, s); });
    return e;
}

}  // namespace ssd
