// ssd_tc.cu -- tcgen05 / TMEM / TMA kernels of libssd (bf16 inputs, fp32
// state and accumulation).
//
// Per head, with cum_t the in-chunk cumulative decay (the sum of dt*A over
// the chunk's steps up to t) and T the cum of the chunk's last step, one
// chunk of the forward pass is
//   y_t   = exp(cum_t) C_t S_in + sum_{s<=t} (C_t . B_s) exp(cum_t - cum_s) dt_s x_s + D x_t
//   S_out = exp(T) S_in + sum_s exp(T - cum_s) dt_s x_s B_s^T
// (cumulative decay, the state entering each chunk and the outputs, with
// the intra-chunk interactions kept on-chip: "Mamba-2 in NVIDIA cuTile:
// Faster Forward Kernels", section "Why Mamba-2 is a useful kernel example";
// quadratic inside a chunk and linear across chunks: the da_be19 thread,
// post 5/6).
//
// Every per-head decay is kept out of the score matrix.  With a per-head
// exponent rho the state is held scaled, Ss = exp(rho) S_in, and
//   a_s  = exp(rho - cum_s) dt_s x_s                  A operand (TMEM)
//   R_t  = C_t . Ss + sum_{s<=t} CB[t, s] a_s          one tcgen05 accumulator
//   y_t  = exp(cum_t - rho) R_t + D x_t
//   Ss  <- Ss + sum_s a_s B_s^T  = exp(rho - T) S_out  (rho <- rho - T)
// CB = C B^T masked to s <= t does not depend on the head: it is computed
// once per chunk and group (cb_mask_kernel) and read by every head block
// that shares the group, as the B operand of the intra-chunk contraction.
// rho moves (to a per-chunk reference rc, with a_s and y_t taken relative to
// rc) only when an exponent would leave [-kLambda, kLambda]; Ss is then
// rescaled in TMEM.  A chunk whose own decay range exceeds 2 kLambda takes a
// direct per-entry path for its intra-chunk term.
//
// The fused forward is three launches:
//   cb_mask_kernel     CB of every (chunk, group), bf16 (a warp-level MMA)
//   seg_state_kernel   the local state of each segment (a run of consecutive
//                      chunks, from a zero state) but the last, or of each
//                      half of it, one long-K contraction per CTA, and its
//                      total decay
//   chunk_scan_kernel  every segment: the state entering it (the pass across
//                      the earlier segments' local states), then the scaled
//                      state chain and the outputs
//
// Tiles: a CTA owns HB heads of one group with HB * P = 128, so every
// state-shaped contraction has M = 128 rows (head, p) and TMEM lane r holds
// row r.  x, B, C and CB tiles arrive by TMA in 128-byte swizzled rows of 64
// bf16.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "ssd_tc.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kSmemLimit = 226 * 1024;  // dynamic bytes; leaves room for the static mbarriers
constexpr uint64_t kWaitNs = 100000000ull;    // a wait gives up after 0.1 s
constexpr uint64_t kDrainNs = 20000000ull;    // the exit drain gives up after 0.02 s
constexpr float kLambda = 64.f;               // |exponent| bound of the scaled operands

// A packed batch of sequences of unequal lengths (x, dt, B, C, y as one
// [1, Ltot, ..] tensor).  A sequence: its steps are rows t0 .. t0 + len - 1,
// its chunk packs and flags start at plane cbase (times G), its states are
// init / fin [seq].  A unit of the chunk scan (blockIdx.y) or of the
// segment-state pass (blockIdx.z) adds its chunks c0 .. c0 + nch - 1 of the
// sequence; for the scan, slot = the sequence's first local-state slot and
// nprev = the local states before its segment (0: the first segment); for
// the segment-state pass, slot = the slot it writes.
struct VlUnit {
    int t0, len, cbase, seq;
    int c0, nch, slot, nprev;
};
// A scan unit with seq < 0 runs several whole sequences one after another:
// sequences t0 .. t0 + len - 1 of the table's sequence section, nch chunks
// in all; the state is written out and reset at each boundary.

// The chunk a role of the scan is at, walking its unit's chunks in order:
// its sequence's table entry j and its chunk c within that sequence (the
// entry's fields are read where needed: two registers per role).
struct VlCursor {
    const VlUnit *tab;
    int j, c;
    __device__ __forceinline__ int t0() const { return __ldg(&tab[j].t0); }
    __device__ __forceinline__ int len() const { return __ldg(&tab[j].len); }
    __device__ __forceinline__ int cbase() const { return __ldg(&tab[j].cbase); }
    __device__ __forceinline__ int seq() const { return __ldg(&tab[j].seq); }
    // one chunk on; true when it starts the next sequence
    template <int Q>
    __device__ __forceinline__ bool next() {
        if (++c < (len() + Q - 1) / Q) return false;
        ++j;
        c = 0;
        return true;
    }
};

struct TcParams {
    long long *trace;  // optional event trace of CTA (0, 0, 0) (trace builds only)
    const bf16 *x;     // [b, L, H, P]
    const bf16 *dt;
    const float *A, *D, *init;
    void *y;
    float *fin;
    // segment-local states (each segment from a zero state): [b, nseg, H, P, N],
    // or with seg_cl [b, nseg, H, N/4, P, 4] (four columns of one row per 16
    // bytes, rows innermost: a warp's 32 rows read or write 512 contiguous bytes)
    float *seg_state;
    int seg_cl;
    float *seg_tot;     // [b, H, nseg]  total dt*A of each segment (may be null)
    const float *cum_in;    // [b, H, nc_cum, cum_q] the caller's in-chunk cumulative decay (null: computed)
    int cum_q, nc_cum;      // the caller's chunk length (64 or 128: one or two tiles) and chunk count
    const float *entering;  // [b, nseg, H, P, N] state entering each segment (null: init / seg_state)
    unsigned *status;   // the device status word: bit 0 = a wait gave up (may be null)
    // limit of the wait for a chunk pack's ready flag (the self-test of the
    // failure path shortens it), and whether the producer waits for that
    // flag before it issues any load of the chunk
    unsigned long long flag_wait_ns;
    int flag_first;
    long long b, L, H, G;
    int hpg, nc, nseg, cps;  // cps: chunks per segment
    // the segment-state pass runs on nsub sub-segments of each segment (of
    // ceil(cps / nsub) chunks, the last one shorter); seg_state and seg_tot
    // hold nslot = nseg * nsub slots
    int nsub, nslot;
    int nhb;
    int dt_tma;  // dt has a TMA map (H % 8 == 0): the vector warps take it from a TMA ring
    // [b, nc, G] set to 1 by the C B^T kernel once a matrix is in memory;
    // the chunk scan's TMA producer polls the flag of a chunk before loading
    // its matrix (the C B^T grid is wholly resident or done by then)
    unsigned *cb_ready;
    const uint8_t *pack;  // [b, nc, G] masked C B^T tiles (CBM_BYTES each)
    // launched with a programmatic dependency on the segment-state kernel:
    // the state warps of segments > 0 wait for it before reading the states
    // entering them
    int dep_seg;
    // packed sequences (null: the equal-length batch b): the scan's units
    // at vl[vl_scan0 + blockIdx.y], the segment-state pass's at
    // vl[vl_seg0 + blockIdx.z]
    const VlUnit *vl;
    int vl_scan0, vl_seg0;
};

template <int P_, int N_, int Q_>
struct Cfg {
    static constexpr int P = P_, N = N_, Q = Q_;
    static constexpr int HB = 128 / P;           // heads per CTA
    static constexpr int M = 128;                // rows (head, p)
    static constexpr int PB = P / 64;            // 64-wide column blocks of one head's x tile
    static constexpr int X_BYTES = M * Q * 2;    // [Q steps][M/64 = 2 blocks (head, 64 p)][64], one TMA box
    static constexpr int BC_BYTES = N * Q * 2;   // [N/64 blocks][Q rows][64]
    static constexpr int CBM_BYTES = Q * Q * 2;  // [Q rows t][Q s]
    // chunk pack in a scan stage: [CB (K-major, swizzled) | B tile | C tile],
    // each in the shared-memory image the MMAs read; the C B^T kernel stores
    // CB alone (one bulk copy of CBM_BYTES), B and C come from the inputs
    static constexpr int PACK_BYTES = CBM_BYTES + 2 * BC_BYTES;
    // vector set of one chunk (floats): per head [Q] arrays dt, cum, a-factor,
    // epilogue factor; then per head the state rescale factor (applied twice),
    // the factor of the bf16 state copy, rho after the chunk; then two block flags
    // (some head rescales, some head takes the wide path)
    static constexpr int V_DT = 0, V_CUM = HB * Q, V_AL = 2 * HB * Q, V_EF = 3 * HB * Q;
    static constexpr int V_F = 4 * HB * Q, V_SBF = V_F + HB, V_RHON = V_SBF + HB, V_FLAG = V_RHON + HB;
    static constexpr int VEC_FLOATS = 4 * HB * Q + 32;
    static constexpr int NV = 4;  // vector sets in flight
    static constexpr int DT_BOX = 8 * 4 * Q * 2;  // dt of 8 heads (one 16-byte box row) x 4 chunks, one TMA box
    static constexpr int DT_RING = 2 * DT_BOX;
    static constexpr int VEC_RING = ((NV * VEC_FLOATS * 4 + 1023) / 1024) * 1024;

    // scan kernel: TMA stages of (x, B, C, CB), the vector ring, and the y
    // tile of one chunk ([half][M/64 blocks][Q/2 steps][64], fp32 or bf16)
    // that the TMA stores to HBM
    static constexpr int SCAN_STAGE = X_BYTES + PACK_BYTES;
    // y staging: one [Q/4 steps][32 p] tile per compute warp (fp32, the
    // larger case), the source of the warp's TMA store of its outputs
    static constexpr int YSTAGE = 16 * (Q / 4) * 32 * 4;
    static_assert(YSTAGE >= 16 * 2048, "the scan prologue's per-warp 2 KB transpose area");
    static constexpr int scan_smem(int st) { return st * SCAN_STAGE + VEC_RING + DT_RING + YSTAGE + 1024; }
    static constexpr int SCAN_ST = scan_smem(4) <= kSmemLimit ? 4 : (scan_smem(3) <= kSmemLimit ? 3 : 2);
    static constexpr int SMEM_SCAN = scan_smem(SCAN_ST);
    static constexpr bool SCAN_FITS = SMEM_SCAN <= kSmemLimit;
    // scan TMEM: Ss [N] | bf16 copy of Ss [N/2] x NB | A hi+lo [Q] x NB | R [Q] x NB
    static constexpr int tmem_cols(int nb) { return N + nb * (N / 2 + 2 * Q); }
    static constexpr int NB = tmem_cols(2) <= 512 ? 2 : 1;
    static constexpr int COL_S = 0, COL_SB = N, COL_A = N + NB * N / 2, COL_R = COL_A + NB * Q;
    static constexpr bool TMEM_FITS = tmem_cols(NB) <= 512;
    // state warp groups of the scan: with N = 256 the state pass (a TMEM
    // round trip per 32 columns) is long enough that a second group of four
    // warps, each group half of the columns, shortens the per-chunk loop;
    // at N <= 128 the smaller register budget of the larger CTA costs more
    static constexpr int SG = N >= 256 ? 2 : 1;
    static constexpr int SCAN_THREADS = 768 + 128 * (SG - 1);
    // registers per thread: at launch (the kernel's allocation), and after
    // setmaxnreg for warps 0-3 (producer, MMA, vectors: few live values) and
    // the compute warps; the split adds up to the launch allocation exactly
    static constexpr int REG_LAUNCH = SG == 1 ? 80 : 72;
    static constexpr int REG_LO = SG == 1 ? 48 : 40, REG_HI = SG == 1 ? 88 : 80;
    static_assert(128 * REG_LO + 128 * SG * REG_LAUNCH + 512 * REG_HI == SCAN_THREADS * REG_LAUNCH,
                  "register split of the chunk scan");

    // segment-state kernel: TMA stages of (x, B) and the vector ring
    static constexpr int SEG_STAGE = X_BYTES + BC_BYTES;
    static constexpr int seg_smem(int st) { return st * SEG_STAGE + VEC_RING + HB * DT_RING + 1024; }
    static constexpr int SEG_ST = seg_smem(4) <= kSmemLimit ? 4 : (seg_smem(3) <= kSmemLimit ? 3 : 2);
    static constexpr int SMEM_SEG = seg_smem(SEG_ST);
    static constexpr int SEG_NA = N + 3 * Q <= 512 ? 3 : 2;  // A buffers of the segment-state kernel
    static constexpr int SEG_COLS = N + SEG_NA * Q;           // S [N] | A hi+lo [Q] x SEG_NA
    static constexpr uint32_t SEG_TMEM =
        SEG_COLS <= 64 ? 64 : SEG_COLS <= 128 ? 128 : SEG_COLS <= 256 ? 256 : 512;

    // C B^T kernel: the masked C B^T and one or two stages of C and B tiles
    static constexpr int smem_cb(int nst) { return CBM_BYTES + nst * 2 * BC_BYTES + 1024; }
    static constexpr int SMEM_CB = smem_cb(1);
};

// Event trace (SSD_TRACE builds): clock64() of role events of CTA (0, 0, 0),
// trace[event * 256 + chunk].  Compiled out otherwise.
#ifdef SSD_TRACE
// (kept in shared memory while the kernel runs: a global store before an
// mbarrier arrive would delay the arrive until the store is performed)
#define TRACE_DECL __shared__ long long trace_sh[32 * 16]
#define TRACE(ev, it)                                                                                  \
    do {                                                                                               \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (it) < 16)                         \
            trace_sh[(ev) * 16 + (it)] = clock64();                                                    \
    } while (0)
#define TRACE_INIT()                                                                                   \
    do {                                                                                               \
        for (int i_ = threadIdx.x; i_ < 32 * 16; i_ += blockDim.x) trace_sh[i_] = 0;                   \
    } while (0)
#define TRACE_FLUSH()                                                                                  \
    do {                                                                                               \
        if (prm.trace && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)                         \
            for (int i_ = threadIdx.x; i_ < 32 * 16; i_ += blockDim.x)                                 \
                if (trace_sh[i_]) prm.trace[(i_ / 16) * 256 + i_ % 16] = trace_sh[i_];                 \
    } while (0)
#define TRACE_CTA(slot)                                                                                 \
    do {                                                                                                 \
        if (prm.trace) {                                                                                 \
            const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);             \
            if (cta_ < 1024) prm.trace[32 * 256 + 2 * cta_ + (slot)] = (long long)globaltimer_ns();       \
        }                                                                                                \
    } while (0)
#define TRACE_CTA2(slot)                                                                                \
    do {                                                                                                 \
        if (prm.trace) {                                                                                 \
            const int cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);             \
            if (cta_ < 1024) prm.trace[32 * 256 + 2048 + 2 * cta_ + (slot)] = (long long)globaltimer_ns(); \
        }                                                                                                \
    } while (0)
#else
#define TRACE_DECL
#define TRACE_INIT() \
    do {             \
    } while (0)
#define TRACE_FLUSH() \
    do {              \
    } while (0)
#define TRACE_CTA2(slot) \
    do {                 \
    } while (0)
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

// Poll a flag in global memory (set by another grid) until it is non-zero,
// with the same bound as wait_bounded; then order the acquire before this
// thread's TMA reads.
__device__ __forceinline__ bool wait_flag(const unsigned *flag, volatile int *abort_flag, uint64_t limit_ns) {
    if (ld_acquire_gpu(flag) == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(flag) == 0) {
            if (*abort_flag || globaltimer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                return false;
            }
            __nanosleep(200);
        }
    }
    fence_async_global();
    return true;
}

// Phase parity to wait for at the it-th use of one of n ring slots: the
// fill of round it / n ("full" side) or the release of the previous round
// ("free" side, only for it >= n).
__device__ __forceinline__ uint32_t fill_parity(int it, int n) { return (uint32_t)((it / n) & 1); }
__device__ __forceinline__ uint32_t free_parity(int it, int n) { return (uint32_t)(((it / n) & 1) ^ 1); }

// Per-chunk vectors are computed by one warp with everything in registers:
// lane l holds steps q = QPL l .. QPL l + QPL - 1 of every head of the CTA.

template <class C>
struct ChunkDt {
    static constexpr int QPL = C::Q / 32;
    float d[C::HB][QPL];
};

// dt of chunk c of the sequence whose steps start at row t0 and stop before
// step slen (plain loads; the caller keeps kDtAhead chunks in flight).
template <class C>
__device__ __forceinline__ void fetch_dt(const TcParams &prm, int b, int h0, int c, int t0, long long slen,
                                         ChunkDt<C> &o) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int hh = 0; hh < C::HB; ++hh)
#pragma unroll
        for (int j = 0; j < ChunkDt<C>::QPL; ++j) {
            const long long h = h0 + hh;
            const long long t = (long long)c * C::Q + ChunkDt<C>::QPL * lane + j;
            // (steps past the sequence in a partial last chunk: dt = 0)
            o.d[hh][j] = h < prm.H && t < slen
                             ? __bfloat162float(__ldg(prm.dt + ((long long)b * prm.L + t0 + t) * prm.H + h))
                             : 0.f;
        }
}

// dt of the chunks ahead for a vector warp.  With a TMA map, lane 0 keeps
// two boxes of four chunks each ([4 Q steps][8 heads] bf16) in flight in a
// private ring, so no global load of the warp is outstanding when it arrives
// on a barrier (an arrive waits for the arriving thread's earlier loads), and
// one TMA operation serves four chunks; without a map (H not a multiple of 8)
// each chunk's dt is loaded when needed.
constexpr int kDtGroup = 4;

// (VL: a packed sequence, with its first row t0 in the map and its length)
template <class C, bool VL = false>
struct DtFeed {
    uint8_t *ring;
    uint64_t *bar;  // [2], count 1
    const CUtensorMap *map;
    int b, h0, n;
    int issued;  // boxes issued so far (box i went to slot i % 2)
    // the sequence's first row in the map and its length: steps at or past
    // slen (a partial last chunk, which in a packed batch holds the next
    // sequence's first steps) take dt = 0
    int t0;
    long long slen;
    // first chunk of the box of steps 4 gi .. 4 gi + 3 (chunk_of is linear,
    // increasing or decreasing; chunks past the segment are only read along)
    template <class F>
    __device__ __forceinline__ int box_start(int gi, F chunk_of) const {
        return min(chunk_of(kDtGroup * gi), chunk_of(kDtGroup * gi + kDtGroup - 1));
    }
    template <class F>
    __device__ __forceinline__ void issue(int gi, F chunk_of) {
        const int k = gi & 1;
        mbar_arrive_expect_tx(&bar[k], C::DT_BOX);
        tma_load_3d(ring + k * C::DT_BOX, map, &bar[k], h0 & ~7, (VL ? t0 : 0) + box_start(gi, chunk_of) * C::Q,
                    b);
        ++issued;
    }
    template <class F>
    __device__ __forceinline__ void start(const TcParams &prm, F chunk_of) {
        issued = 0;
        if (prm.dt_tma && (threadIdx.x & 31) == 0)
            for (int gi = 0; gi < 2 && kDtGroup * gi < n; ++gi) issue(gi, chunk_of);
    }
    // dt of step `it` (chunk chunk_of(it)); false when the wait gave up
    template <class F>
    __device__ __forceinline__ bool take(const TcParams &prm, int it, F chunk_of, volatile int *abort_flag,
                                         ChunkDt<C> &o) {
        const int lane = threadIdx.x & 31;
        if (!prm.dt_tma) {
            fetch_dt<C>(prm, b, h0, chunk_of(it), VL ? t0 : 0, VL ? slen : prm.L, o);
            return true;
        }
        const int gi = it / kDtGroup, k = gi & 1;
        if (it % kDtGroup == 0) {
            int ok = lane == 0 ? (wait_bounded(&bar[k], (uint32_t)((gi >> 1) & 1), abort_flag) ? 1 : 0) : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        }
        const int row0 = (chunk_of(it) - box_start(gi, chunk_of)) * C::Q;
        const long long tq = (long long)chunk_of(it) * C::Q + ChunkDt<C>::QPL * lane;  // this lane's first step
        const unsigned short *d16 = reinterpret_cast<const unsigned short *>(ring + k * C::DT_BOX);
#pragma unroll
        for (int hh = 0; hh < C::HB; ++hh)
#pragma unroll
            for (int j = 0; j < ChunkDt<C>::QPL; ++j)
                o.d[hh][j] = h0 + hh < prm.H && (!VL || tq + j < slen)
                                 ? __uint_as_float(
                                       (uint32_t)d16[(row0 + ChunkDt<C>::QPL * lane + j) * 8 + (h0 & 7) + hh] << 16)
                                 : 0.f;
        __syncwarp();
        // the box is used up after its last step: refill its slot two boxes on
        if ((it % kDtGroup == kDtGroup - 1 || it == n - 1) && lane == 0 && kDtGroup * (gi + 2) < n) {
            fence_async_smem();
            issue(gi + 2, chunk_of);
        }
        return true;
    }
    // let outstanding boxes land before the CTA exits (lane 0)
    __device__ __forceinline__ void drain() {
        if ((threadIdx.x & 31) == 0)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int nk = issued > k ? (issued - k + 1) / 2 : 0;  // boxes slot k received
                if (nk > 0) mbar_wait(&bar[k], (uint32_t)((nk - 1) & 1), kDrainNs);
            }
    }
};

// The caller's dA_cumsum for tile c of head h, relative to the tile's start:
// a chunk of cum_q = 128 steps is two tiles, and the second tile's values are
// those of the chunk minus the chunk's value before the tile.
template <class C>
__device__ __forceinline__ const float *tile_cum(const TcParams &prm, int b, long long h, int c, float &base) {
    const int tpc = prm.cum_q / C::Q;  // tiles per caller chunk
    const int cc = c / tpc, off = (c % tpc) * C::Q;
    const float *src = prm.cum_in + (((long long)b * prm.H + h) * prm.nc_cum + cc) * prm.cum_q + off;
    base = off > 0 ? __ldg(src - 1) : 0.f;
    return src;
}

// In-chunk cumulative decay of every head for this lane's steps: the scan of
// dt*A (all heads' shuffle chains interleaved), or the caller's dA_cumsum.
// T[hh] = the chunk total (cum of the last step).
template <class C>
__device__ __forceinline__ void chunk_cums(const TcParams &prm, int b, int h0, int c, const ChunkDt<C> &dt,
                                           const float (&Ah)[C::HB], float (&cum)[C::HB][C::Q / 32],
                                           float (&T)[C::HB]) {
    constexpr int QPL = C::Q / 32;
    const int lane = threadIdx.x & 31;
    if (prm.cum_in) {
#pragma unroll
        for (int hh = 0; hh < C::HB; ++hh) {
            const long long h = h0 + hh;
            float base;
            const float *src = tile_cum<C>(prm, b, h < prm.H ? h : 0, c, base);
#pragma unroll
            for (int j = 0; j < QPL; ++j) cum[hh][j] = h < prm.H ? __ldg(src + QPL * lane + j) - base : 0.f;
            T[hh] = h < prm.H ? __ldg(src + C::Q - 1) - base : 0.f;
        }
        return;
    }
    float run[C::HB], tot[C::HB];
#pragma unroll
    for (int hh = 0; hh < C::HB; ++hh) {
        const float a = Ah[hh];
        run[hh] = 0.f;
#pragma unroll
        for (int j = 0; j < QPL; ++j) {
            run[hh] += dt.d[hh][j] * a;
            cum[hh][j] = run[hh];
        }
        tot[hh] = run[hh];
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
#pragma unroll
        for (int hh = 0; hh < C::HB; ++hh) {
            const float o = __shfl_up_sync(0xffffffffu, tot[hh], off);
            if (lane >= off) tot[hh] += o;
        }
#pragma unroll
    for (int hh = 0; hh < C::HB; ++hh) {
        const float excl = tot[hh] - run[hh];
#pragma unroll
        for (int j = 0; j < QPL; ++j) cum[hh][j] += excl;
        T[hh] = __shfl_sync(0xffffffffu, tot[hh], 31);
    }
}

// In-chunk cumulative decay of one head hh of the block for this lane's
// steps (or the caller's dA_cumsum); T = the chunk total.
template <class C>
__device__ __forceinline__ void head_cums(const TcParams &prm, int b, int h0, int hh, int c, const ChunkDt<C> &dt,
                                          float a, float (&cum)[C::Q / 32], float &T) {
    constexpr int QPL = C::Q / 32;
    const int lane = threadIdx.x & 31;
    const long long h = h0 + hh;
    if (prm.cum_in) {
        float base;
        const float *src = tile_cum<C>(prm, b, h < prm.H ? h : 0, c, base);
#pragma unroll
        for (int j = 0; j < QPL; ++j) cum[j] = h < prm.H ? __ldg(src + QPL * lane + j) - base : 0.f;
        T = h < prm.H ? __ldg(src + C::Q - 1) - base : 0.f;
        return;
    }
    float run = 0.f;
#pragma unroll
    for (int j = 0; j < QPL; ++j) {
        run += dt.d[hh][j] * a;
        cum[j] = run;
    }
    float tot = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, tot, off);
        if (lane >= off) tot += o;
    }
    const float excl = tot - run;
#pragma unroll
    for (int j = 0; j < QPL; ++j) cum[j] += excl;
    T = __shfl_sync(0xffffffffu, tot, 31);
}

// Decay rate A of each head of the block (0 past H), loaded once per CTA.
template <class C>
__device__ __forceinline__ void load_decay(const TcParams &prm, int h0, float (&Ah)[C::HB]) {
#pragma unroll
    for (int hh = 0; hh < C::HB; ++hh) Ah[hh] = (h0 + hh < prm.H && prm.A) ? prm.A[h0 + hh] : 0.f;
}

// Order-preserving integer key of a float (for warp min / max reductions).
__device__ __forceinline__ int fkey(float f) {
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float unkey(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF); }

// Build this thread's part of the A operand of one chunk in TMEM:
//   a_s = f_s x_s for the NS steps s in [NS part, NS part + NS), split into
//   bf16 hi and lo (hi = bf16(a), lo = bf16(a - hi): together about 2^-17
//   relative; a single bf16 rounding of a, 2^-9, shows in state entries that
//   one recent token dominates).  Column j of the hi block holds s = 2j,
//   2j + 1; the lo block follows Q / 2 columns later.
template <class C, int NS>
__device__ __forceinline__ void build_a(const uint8_t *xs, int blk, uint32_t pcol, const float *f, int part,
                                       uint32_t tmem_a) {
    static_assert(NS == 16 || NS == 32, "parts of 16 or 32 steps");
    static_assert(C::M / 64 == 2, "two 64-wide column blocks per step");
    uint32_t hi[NS / 2], lo[NS / 2];
    // the x tile is [step s][block][64] in 128-byte lines (line 2 s + blk),
    // 128-byte swizzled: the 16-byte chunk of column pcol sits at position
    // chunk ^ (line % 8); with line % 8 = 2 (s % 4) + blk, the byte offset of
    // (s, blk, pcol) is 256 s + sw[s % 4]
    const uint8_t *sw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        sw[k] = xs + blk * 128 + (((((pcol >> 3) ^ (uint32_t)(2 * k + blk)) & 7u) << 4) | ((pcol & 7u) << 1));
#pragma unroll
    for (int j = 0; j < NS / 2; ++j) {
        const int s0 = part * NS + 2 * j;
        const uint32_t x0 = *reinterpret_cast<const unsigned short *>(sw[s0 & 3] + s0 * 256);
        const uint32_t x1 = *reinterpret_cast<const unsigned short *>(sw[(s0 + 1) & 3] + (s0 + 1) * 256);
        const float a0 = __uint_as_float(x0 << 16) * f[2 * j];
        const float a1 = __uint_as_float(x1 << 16) * f[2 * j + 1];
        const uint32_t h = pack_bf16x2(a0, a1);
        hi[j] = h;
        lo[j] = pack_bf16x2(a0 - __uint_as_float(h << 16), a1 - __uint_as_float(h & 0xFFFF0000u));
    }
    if constexpr (NS == 32) {
        tmem_st16u(tmem_a + part * 16, hi);
        tmem_st16u(tmem_a + C::Q / 2 + part * 16, lo);
    } else {
        tmem_st8u(tmem_a + part * 8, hi);
        tmem_st8u(tmem_a + C::Q / 2 + part * 8, lo);
    }
}

// This thread's x values of the NS steps from NS part on, read from the
// swizzled x tile (layout as for build_a), two bf16 per word (step 2j in the
// low half).  They serve both the A operand and the D x term of the output.
template <class C, int NS>
__device__ __forceinline__ void load_x_part(const uint8_t *xs, int blk, uint32_t pcol, int part,
                                            uint32_t (&xk)[NS / 2]) {
    static_assert(C::M / 64 == 2, "two 64-wide column blocks per step");
    const uint8_t *sw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        sw[k] = xs + blk * 128 + (((((pcol >> 3) ^ (uint32_t)(2 * k + blk)) & 7u) << 4) | ((pcol & 7u) << 1));
#pragma unroll
    for (int j = 0; j < NS / 2; ++j) {
        const int s0 = part * NS + 2 * j;
        const uint32_t x0 = *reinterpret_cast<const unsigned short *>(sw[s0 & 3] + s0 * 256);
        const uint32_t x1 = *reinterpret_cast<const unsigned short *>(sw[(s0 + 1) & 3] + (s0 + 1) * 256);
        xk[j] = x0 | (x1 << 16);
    }
}

// The A operand part of build_a from x values already in registers, for the
// chunk scan, whose A buffer interleaves the parts per K step: K step k
// (steps 16 k .. 16 k + 15) holds its hi words in columns 16 k .. 16 k + 7
// and its lo words in the next 8, so each warp writes its part with one
// 16-column store (fewer tensor-memory operations on the compute chain).
template <class C, int NS>
__device__ __forceinline__ void build_a_regs(const uint32_t (&xk)[NS / 2], const float *f, int part,
                                             uint32_t tmem_a) {
    uint32_t hi[NS / 2], lo[NS / 2];
#pragma unroll
    for (int j = 0; j < NS / 2; j += 2) {
        const float4 f4 = *reinterpret_cast<const float4 *>(f + 2 * j);
        const float a0 = __uint_as_float(xk[j] << 16) * f4.x;
        const float a1 = __uint_as_float(xk[j] & 0xFFFF0000u) * f4.y;
        const float a2 = __uint_as_float(xk[j + 1] << 16) * f4.z;
        const float a3 = __uint_as_float(xk[j + 1] & 0xFFFF0000u) * f4.w;
        const uint32_t h0 = pack_bf16x2(a0, a1), h1 = pack_bf16x2(a2, a3);
        hi[j] = h0;
        hi[j + 1] = h1;
        lo[j] = pack_bf16x2(a0 - __uint_as_float(h0 << 16), a1 - __uint_as_float(h0 & 0xFFFF0000u));
        lo[j + 1] = pack_bf16x2(a2 - __uint_as_float(h1 << 16), a3 - __uint_as_float(h1 & 0xFFFF0000u));
    }
    static_assert(NS == 16, "one K step per part");
    uint32_t hl[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        hl[j] = hi[j];
        hl[8 + j] = lo[j];
    }
    tmem_st16u(tmem_a + part * 16, hl);  // K step `part`: hi in 8 columns, lo in the next 8
}

// Every lane of the warp waits for the phase (bounded); uniform result.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    const bool ok = wait_bounded(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, ok) != 0;
}

// TMA loads of chunk c: x tiles of the CTA's heads, B, and (optionally) C.
template <class C>
__device__ __forceinline__ void issue_chunk_loads(uint8_t *xs, uint8_t *bs, uint8_t *cs, uint64_t *bar,
                                                  const CUtensorMap *mx, const CUtensorMap *mb,
                                                  const CUtensorMap *mc, int h0, int g, int c, int b, int t0 = 0) {
    const int row = t0 + c * C::Q;
    tma_load_5d(xs, mx, bar, 0, 0, h0, row, b);  // x: [Q][HB][PB][64], 256 contiguous bytes per step
#pragma unroll
    for (int nb = 0; nb < C::N / 64; ++nb) tma_load_4d(bs + nb * (C::Q * 128), mb, bar, nb * 64, g, row, b);
    if (cs)
#pragma unroll
        for (int nb = 0; nb < C::N / 64; ++nb)
            tma_load_4d(cs + nb * (C::Q * 128), mc, bar, nb * 64, g, row, b);
}

// ===========================================================================
// Chunk packs, one per (chunk, group, batch) tile; one CTA per tile, or (where
// the scan leaves SMs free) one CTA on each such SM walking the tiles in chunk
// order with the next tile's loads in flight:
//   CB[t, s] = C_t . B_s for s <= t (0 above the diagonal), bf16, stored
//   K-major and swizzled (the shared-memory image the chunk scan's MMAs read,
//   so that it arrives there with one bulk copy): pack[(b, c, g)].  The
//   64 x 64 x N product runs on the warp-level tensor-core MMA, which needs
//   no TMEM: these CTAs share SMs with segment-state CTAs whose TMEM
//   allocations fill the SM's 512 columns.
// ===========================================================================
// The tiles of the C B^T pass in chunk-major order.  An equal-length batch:
// tile t = (chunk c, batch b, group g), c slowest.  Packed sequences: chunk
// level c holds chunk c of every sequence that long (the units are ordered
// longest first, so these are the first units), vl_off[c] = the chunks
// before level c (vl_off[nlvl] = all of them), then the group.
struct CbWalk {
    int nc, G, nbatch;
    long long ntiles;
    const VlUnit *vl;
    const int *vl_off;
    int nlvl;
};

struct CbTile {
    int row, bq, g;  // first step's row and batch coordinate in the B / C maps, group
    long long plane;  // pack and flag index
};

template <class C, bool VL>
__device__ __forceinline__ CbTile cb_tile(const CbWalk &w, long long t) {
    CbTile o;
    if constexpr (!VL) {
        const long long per_chunk = (long long)w.nbatch * w.G;
        const int c = (int)(t / per_chunk), rem = (int)(t % per_chunk), b = rem / w.G;
        o.g = rem % w.G;
        o.row = c * C::Q;
        o.bq = b;
        o.plane = ((long long)b * w.nc + c) * w.G + o.g;
        return o;
    }
    const int k = (int)(t / w.G);
    o.g = (int)(t % w.G);
    int lo = 0, hi = w.nlvl - 1;  // the last level whose first chunk is at or before k
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(w.vl_off + mid) <= k) lo = mid;
        else hi = mid - 1;
    }
    const int i = k - __ldg(w.vl_off + lo);
    const int t0 = __ldg(&w.vl[i].t0), cbase = __ldg(&w.vl[i].cbase);
    o.row = t0 + lo * C::Q;
    o.bq = 0;
    o.plane = ((long long)cbase + lo) * w.G + o.g;
    return o;
}

// (at most 72 registers: with segments a C B^T CTA shares its SM with two
// segment-state CTAs of 384 threads at 72)
template <class C, bool VL>
__global__ void __maxnreg__(72) cb_mask_kernel(const __grid_constant__ CUtensorMap mb,
                                                      const __grid_constant__ CUtensorMap mc, uint8_t *pack,
                                                      const CbWalk walk, int nst, unsigned *ready, unsigned *status) {
    static_assert(C::Q == 64, "four warps of 16 rows");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *cbs = smem;
    // nst stages of [C tile | B tile]
    auto stage_c = [&](int s) { return smem + C::CBM_BYTES + s * 2 * C::BC_BYTES; };
    auto stage_b = [&](int s) { return smem + C::CBM_BYTES + s * 2 * C::BC_BYTES + C::BC_BYTES; };
    __shared__ uint64_t full_bar[2];
    __shared__ int ok_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // tiles in chunk-major order (every batch and group of a chunk before the
    // next chunk), this CTA's every gridDim.x-th
    const long long ntiles = walk.ntiles;
    if constexpr (!VL) griddep_launch();
    if (tid == 32) {
        for (int s = 0; s < 2; ++s) mbar_init(&full_bar[s], 1);
        fence_mbar_init();
        prefetch_tmap(&mb);
        prefetch_tmap(&mc);
    }
    // packed sequences: launched while the setup kernel writes the unit
    // table and clears the flags; wait for it, then let the next grid go
    if constexpr (VL) {
        griddep_wait();
        griddep_launch();
    }
    __syncthreads();
    int nload[2] = {0, 0};  // loads issued per stage (thread 32)
    auto issue = [&](long long t, int s) {
        const CbTile tl = cb_tile<C, VL>(walk, t);
        mbar_arrive_expect_tx(&full_bar[s], 2 * C::BC_BYTES);
        // one box each ([N/64][Q][64], 128-byte swizzle)
        tma_load_5d(stage_c(s), &mc, &full_bar[s], 0, tl.row, 0, tl.g, tl.bq);
        tma_load_5d(stage_b(s), &mb, &full_bar[s], 0, tl.row, 0, tl.g, tl.bq);
        ++nload[s];
    };
    if (tid == 32)
        for (int k = 0; k < nst; ++k)
            if (blockIdx.x + (long long)k * gridDim.x < ntiles) issue(blockIdx.x + (long long)k * gridDim.x, k);
    int k = 0;
    for (long long t = blockIdx.x; t < ntiles; t += gridDim.x, ++k) {
        const int s = k % nst;
        if (tid == 32) {
            const int ok = mbar_wait(&full_bar[s], (uint32_t)((k / nst) & 1), kWaitNs) ? 1 : 0;
            if (!ok) flag_timeout(status);
            ok_sh = ok;
        }
        __syncthreads();
        if (!ok_sh) break;
        // C B^T on the warp tensor cores (a 64 x 64 x N product per tile, too
        // small to pay for TMEM): warp w owns rows t = 16 w .. 16 w + 15, all
        // 64 columns s as eight 8-wide tiles.  Element (row r, k) of the
        // staged C and B tiles sits at (k / 64) Q 128 + r 128 + 16 ((k % 64) / 8
        // ^ r % 8) + 2 (k % 8).
        float acc[8][4];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[jj][e] = 0.f;
        const uint8_t *cs = stage_c(s), *bs = stage_b(s);
        const int ra = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);  // C row this lane addresses
        const int ka = lane >> 4;                                        // its 8-column half of the k step
        const int rb = (lane & 7) + 8 * (lane >> 4);                     // B row (within two s tiles)
        const int kb = (lane >> 3) & 1;
#pragma unroll 1
        for (int k0 = 0; k0 < C::N; k0 += 16) {
            const int blk = (k0 / 64) * (C::Q * 128), kc = (k0 % 64) / 8;
            uint32_t a[4];
            ldsm_x4(a, cs + blk + ra * 128 + (((kc + ka) ^ (ra & 7)) << 4));
#pragma unroll
            for (int jj = 0; jj < 8; jj += 2) {
                const int r = 8 * jj + rb;
                uint32_t bq[4];
                ldsm_x4(bq, bs + blk + r * 128 + (((kc + kb) ^ (r & 7)) << 4));
                mma_16816_bf16(acc[jj], a, bq[0], bq[1]);
                mma_16816_bf16(acc[jj + 1], a, bq[2], bq[3]);
            }
        }
        // every warp has read the stage: refill it with this CTA's tile nst on
        __syncthreads();
        if (tid == 32 && t + (long long)nst * gridDim.x < ntiles) issue(t + (long long)nst * gridDim.x, s);
        // masked (s <= t) bf16 pairs into the pack image: row t, 16-byte
        // chunk s / 8 at position (s / 8) ^ (t % 8) (the previous tile's
        // store has finished reading it: thread 0 waited for it before the
        // barriers above)
        const int t0 = 16 * warp + (lane >> 2), q = lane & 3;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int s0 = 8 * jj + 2 * q;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int tr = t0 + 8 * h;
                const uint32_t w = pack_bf16x2(s0 <= tr ? acc[jj][2 * h] : 0.f, s0 + 1 <= tr ? acc[jj][2 * h + 1] : 0.f);
                *reinterpret_cast<uint32_t *>(cbs + tr * 128 + ((jj ^ (tr & 7)) << 4) + 4 * q) = w;
            }
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            const long long plane = cb_tile<C, VL>(walk, t).plane;
            bulk_store(pack + plane * C::CBM_BYTES, cbs, C::CBM_BYTES);
            bulk_commit_group();
            bulk_wait_all();
            __threadfence();
            if (ready) st_release_gpu(ready + plane, 1u);
        }
    }
    // (after a wait that gave up) let this CTA's own loads land before it exits
    if (tid == 32)
        for (int s = 0; s < nst; ++s)
            if (nload[s] > 0) mbar_wait(&full_bar[s], (uint32_t)((nload[s] - 1) & 1), kDrainNs);
}

// ===========================================================================
// Segment-local states (segments 0 .. nseg-2, or their nsub sub-segments,
// each from a zero state):
//   S_seg = sum_t exp(sum_{k>t, k in segment} dt_k A) dt_t x_t^T B_t
//   warp 0      : TMA loads of the x and B tiles
//   warp 1      : tcgen05.mma S += A^T B, A read from TMEM
//   warps 2, 3  : dt and the segment weights of one head each (a ring of
//                 vector sets), and the segment's total decay
//   warps 4 ..  : the A operand (weights x x, bf16 hi + lo) into TMEM, two
//                 or three buffers; then the state to HBM
// ===========================================================================
// NBG groups of four operand-builder warps (each group Q / NBG of the steps):
// four groups with the deep ring (one CTA per SM), or two groups with two
// stages and two A buffers in 256 TMEM columns, so that two CTAs share an SM
template <class C, int NBG>
struct SegT {
    static constexpr int THREADS = 128 + 128 * NBG;
    static constexpr int ABW = 4 * NBG;  // operand-builder warps 4 .. 4 + ABW - 1
    static constexpr int NS = C::Q / NBG;
    static constexpr int ST = NBG == 4 ? C::SEG_ST : 2;
    static constexpr int NA = NBG == 4 ? C::SEG_NA : 2;
    static constexpr uint32_t TMEM = NBG == 4 ? C::SEG_TMEM : 256;
    static constexpr int SMEM = C::seg_smem(ST);
    // two CTAs of 384 threads at 72 registers beside a C B^T CTA (128 x 72)
    // fit the 64 K registers of an SM
    static constexpr int MAXREG = NBG == 4 ? 64 : 72;
    static_assert(NBG == 4 || C::N + 2 * C::Q <= 256, "two A buffers and S in 256 columns");
};

// VL: the units are packed sequences' sub-segments (prm.vl)
template <class C, int NBG, bool VL>
__global__ void __launch_bounds__(SegT<C, NBG>::THREADS) __maxnreg__((SegT<C, NBG>::MAXREG))
    seg_state_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mb,
                     const __grid_constant__ CUtensorMap mdt, TcParams prm) {
    using T = SegT<C, NBG>;
    constexpr int ST = T::ST, NV = C::NV;
    constexpr int kSegThreads = T::THREADS, kSegABWarps = T::ABW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *vec_base = reinterpret_cast<float *>(smem + ST * C::SEG_STAGE);
    uint8_t *dt_ring = smem + ST * C::SEG_STAGE + C::VEC_RING;
    __shared__ uint64_t dt_bar[2 * C::HB];  // a dt ring per vector warp
    TRACE_DECL;
    constexpr int NA = T::NA;
    __shared__ uint64_t full_bar[4], empty_bar[4], vfull_bar[NV], vempty_bar[NV], afull_bar[NA], afree_bar[NA];
    __shared__ uint64_t done_bar, drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ volatile int slot[8];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.z, hblk = blockIdx.x, b = blockIdx.y;
    const int h0 = hblk * C::HB;
    const int g = (int)(prm.G == 1 ? 0 : h0 / prm.hpg);
    // sub-segment `seg` of segment seg / nsub, written to slot `seg` of batch
    // entry b; a packed sequence's unit names its chunks and its slot (of
    // batch entry 0)
    const int csub = (prm.cps + prm.nsub - 1) / prm.nsub;
    const int sbeg = (seg / prm.nsub) * prm.cps;
    int c0 = sbeg + (seg % prm.nsub) * csub;
    int nch = min(min(prm.nc, sbeg + prm.cps), c0 + csub) - c0;
    int bq = b, t0 = 0, sslot = seg;
    long long slen = prm.L;
    if constexpr (VL) {
        const VlUnit u = prm.vl[prm.vl_seg0 + seg];
        c0 = u.c0;
        nch = u.nch;
        bq = 0;
        t0 = u.t0;
        slen = u.len;
        sslot = u.slot;
    }
    const long long H = prm.H;
    // the segment's chunks are taken last to first, so the decay of the
    // chunks after each one (its weights' offset) accumulates as they come
    auto chunk_of = [&](int it) { return c0 + nch - 1 - it; };
    auto stage_x = [&](int s) { return smem + s * C::SEG_STAGE; };
    auto stage_b = [&](int s) { return smem + s * C::SEG_STAGE + C::X_BYTES; };
    // the chunk scan after this kernel may be scheduled at once: its first
    // segment needs nothing from here
    griddep_launch();
    if (tid == 0) TRACE_CTA2(0);
    auto vec = [&](int v) { return vec_base + v * C::VEC_FLOATS; };

    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, T::TMEM);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1 + kSegABWarps);  // the MMAs' commit and each operand-builder warp
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&vfull_bar[i], C::HB);  // one vector warp per head
            mbar_init(&vempty_bar[i], kSegABWarps);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(&afull_bar[i], kSegABWarps);
            mbar_init(&afree_bar[i], 1);
        }
        mbar_init(&done_bar, 1);
        mbar_init(&drain_bar, 1);
        for (int i = 0; i < 2 * C::HB; ++i) mbar_init(&dt_bar[i], 1);
        fence_mbar_init();
        abort_sh = 0;
        prefetch_tmap(&mx);
        prefetch_tmap(&mb);
        if (prm.dt_tma) prefetch_tmap(&mdt);
    }
    TRACE_INIT();
    int nload[4] = {};  // TMA loads issued per stage (producer lane 0)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    constexpr uint32_t COL_A = C::N;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0)
            for (int it = 0; it < nch; ++it) {
                const int s = it % ST, c = chunk_of(it);
                if (it >= ST && !wait_bounded(&empty_bar[s], free_parity(it, ST), &abort_sh)) break;
                mbar_arrive_expect_tx(&full_bar[s], C::X_BYTES + C::BC_BYTES);
                issue_chunk_loads<C>(stage_x(s), stage_b(s), nullptr, &full_bar[s], &mx, &mb, nullptr, h0, g, c, bq,
                                     t0);
                ++nload[s];
                TRACE(18, it);
            }
    } else if (warp == 2 || (warp == 3 && C::HB > 1)) {
        // ---------------- segment weights, one warp per head ----------------
        //   w_s = exp(after + T - cum_s) dt_s, after = decay of the later chunks
        constexpr int QPL = C::Q / 32;
        const int hv = warp - 2;
        float after = 0.f;
        DtFeed<C, VL> feed{dt_ring + hv * C::DT_RING, dt_bar + 2 * hv, &mdt, bq, h0, nch, 0, t0, slen};
        feed.start(prm, chunk_of);
        const float a = (h0 + hv < H && prm.A) ? prm.A[h0 + hv] : 0.f;
        // dt of the next chunk is read while this one is processed: the
        // shared-memory reads wait behind the operand builders' traffic
        ChunkDt<C> dt_next;
        bool have = nch > 0 && feed.take(prm, 0, chunk_of, &abort_sh, dt_next);
        for (int it = 0; it < nch; ++it) {
            if (!have) break;
            const int v = it % NV, c = chunk_of(it);
            const ChunkDt<C> dt = dt_next;
            if (it + 1 < nch) have = feed.take(prm, it + 1, chunk_of, &abort_sh, dt_next);
            float cum[QPL], T;
            head_cums<C>(prm, b, h0, hv, c, dt, a, cum, T);
            float w[QPL];
#pragma unroll
            for (int j = 0; j < QPL; ++j) w[j] = __expf(after + T - cum[j]) * dt.d[hv][j];
            after += T;
            if (it >= NV) {
                int ok = lane == 0 ? (wait_bounded(&vempty_bar[v], free_parity(it, NV), &abort_sh) ? 1 : 0) : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            }
            float *vv = vec(v);
#pragma unroll
            for (int j = 0; j < QPL; ++j) vv[C::V_AL + hv * C::Q + QPL * lane + j] = w[j];
            __syncwarp();
            if (lane == 0) {
                if (hv == 0) TRACE(14, it);
                mbar_arrive(&vfull_bar[v]);
            }
        }
        feed.drain();
        // total dt*A of the segment, for the pass across segments
        if (lane == 0 && h0 + hv < H && prm.seg_tot)
            prm.seg_tot[((long long)bq * H + h0 + hv) * prm.nslot + sslot] = after;
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // (the whole warp runs the loop, so its descriptors stay
        // warp-uniform; one elected lane issues)
        const uint32_t idesc = idesc_bf16(C::M, C::N, false, true);
        for (int it = 0; it < nch; ++it) {
            const int s = it % ST, a = it % NA;
            if (!warp_wait(&afull_bar[a], fill_parity(it, NA), &abort_sh)) break;
            if (!warp_wait(&full_bar[s], fill_parity(it, ST), &abort_sh)) break;
            tc_fence_after();
            const uint32_t ta = tmem + COL_A + a * C::Q;
            const uint64_t db = sdesc(smem_u32(stage_b(s)), C::Q * 128, 1024);
            if (elect_one()) {
                if (it == 0) {
#pragma unroll
                    for (int ks = 0; ks < C::Q / 16; ++ks)
                        mma_bf16_ta(tmem, ta + ks * 8, desc_add(db, ks * 2048), idesc, ks != 0);
                } else {
#pragma unroll
                    for (int ks = 0; ks < C::Q / 16; ++ks)
                        mma_bf16_ta(tmem, ta + ks * 8, desc_add(db, ks * 2048), idesc, true);
                }
#pragma unroll
                for (int ks = 0; ks < C::Q / 16; ++ks)
                    mma_bf16_ta(tmem, ta + C::Q / 2 + ks * 8, desc_add(db, ks * 2048), idesc, true);
                mma_commit(&empty_bar[s]);
                mma_commit(&afree_bar[a]);
                TRACE(16, it);
            }
            __syncwarp();
        }
        if (elect_one()) mma_commit(&done_bar);  // completes once every MMA above has
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------- A operand builders: thread = row (head, p), 1 / NBG of the steps ----------------
        constexpr int NAB = kSegThreads - 128;
        const int gtid = tid - 128;
        const int q4 = warp & 3, part = (warp - 4) >> 2;
        const int row = q4 * 32 + lane, rh = row / C::P, rp = row % C::P;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t pcol = (uint32_t)(rp % 64);
        const int blk = rh * C::PB + rp / 64;
        // every warp waits and arrives on its own (no group-wide barrier per chunk)
        for (int it = 0; it < nch; ++it) {
            const int s = it % ST, v = it % NV, a = it % NA;
            if (!warp_wait(&full_bar[s], fill_parity(it, ST), &abort_sh)) break;
            if (gtid == 0) TRACE(19, it);
            if (!warp_wait(&vfull_bar[v], fill_parity(it, NV), &abort_sh)) break;
            if (it >= NA && !warp_wait(&afree_bar[a], free_parity(it, NA), &abort_sh)) break;
            if (gtid == 0) TRACE(17, it);
            tc_fence_after();
            build_a<C, T::NS>(stage_x(s), blk, pcol, vec(v) + C::V_AL + rh * C::Q + part * T::NS, part,
                              tmem + lane_off + COL_A + a * C::Q);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (gtid == 0) TRACE(15, it);
                mbar_arrive(&afull_bar[a]);
                mbar_arrive(&empty_bar[s]);
                mbar_arrive(&vempty_bar[v]);
            }
        }
        // segment state: TMEM lane r = row (head, p); each group of four
        // warps 1 / NBG of the columns
        const long long hrow = h0 + rh;
        if (group_wait(&done_bar, 0, &abort_sh, &slot[3], 1, gtid, NAB)) {
            tc_fence_after();
            const long long blk0 = (((long long)bq * prm.nslot + sslot) * H + hrow) * C::P * C::N;
            // element n of this row: at 4 (n/4) P + n%4 in the column-block
            // layout, at n in the row layout
            float *dst = prm.seg_state + blk0 + (prm.seg_cl ? rp * 4 : rp * C::N);
            const int cstep = prm.seg_cl ? C::P : 1;
#pragma unroll 1
            for (int n0 = part * (C::N / NBG); n0 < (part + 1) * (C::N / NBG); n0 += 16) {
                float v[16];
                tmem_ld16(tmem + lane_off + n0, v);
                tmem_ld_wait();
                if (hrow < H) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        __stcg(reinterpret_cast<float4 *>(dst + (long long)(n0 + j) * cstep),
                               make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]));
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
    TRACE_FLUSH();
    if (warp == 1) tmem_dealloc(tmem, T::TMEM);
    if (abort_sh && tid == 0) flag_timeout(prm.status);
    // complete only after the C B^T grid before this one: a grid that waits
    // for this one then sees those matrices too
    griddep_wait();
    if (tid == 0) TRACE_CTA2(1);
}

// Epilogue fix-up of a chunk whose decay range is too wide to scale (rare;
// kept out of line so the hot path stays small): R holds the inter-chunk
// term only; replace this thread's NS accumulator columns by
//   ef_t R_t + sum_{s<=t} CB[t, s] exp(cum_t - cum_s) dt_s x_s
// computed with direct per-entry decay factors, so the caller stores them
// with a unit factor.
template <class C, int NS>
__device__ __noinline__ void wide_fixup(uint32_t taddr, const float *ef, const uint8_t *xs, int blk, const uint8_t *cbm,
                                        const float *cum, const float *dtv, uint32_t pcol, int t0) {
    const unsigned short *x16 = reinterpret_cast<const unsigned short *>(xs);
    const unsigned short *c16 = reinterpret_cast<const unsigned short *>(cbm);
#pragma unroll 1
    for (int j0 = 0; j0 < NS; j0 += 16) {
        float v[16];
        tmem_ld16(taddr + j0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = t0 + j0 + j;
            const float ct = cum[t];
            float acc = 0.f;
#pragma unroll 1
            for (int s = 0; s <= t; ++s) {
                const float xv = __uint_as_float((uint32_t)x16[swz128((uint32_t)(2 * s + blk), pcol) >> 1] << 16);
                const float cb = __uint_as_float((uint32_t)c16[swz128((uint32_t)t, (uint32_t)s) >> 1] << 16);
                acc = fmaf(cb * __expf(ct - cum[s]) * dtv[s], xv, acc);
            }
            v[j] = fmaf(ef[j0 + j], v[j], acc);
        }
        tmem_st16(taddr + j0, v);
    }
    tmem_st_wait();
}

// ===========================================================================
// Chunk scan with the scaled state carried in TMEM (every segment).
//   warp 0     : TMA loads of x and the chunk pack (C B^T, B, C)
//   warp 1     : tcgen05.mma issue, per chunk  Ss += A B (once the state
//                warps are done with Ss);  R = A CB^T;  R += SB C^T
//   warp 2     : dt, cumulative decay, rho, the A factors and output
//                factors (a ring of vector sets)
//   warps 4-7  : state: Ss rescale when the reference moves, and its bf16
//                copy SB (the A operand of the inter-chunk term); with
//                C::SG = 2 warps 24-27 take the second half of the columns
//   (warps 0-3 give registers back with setmaxnreg, the compute warps take
//   them: C::REG_LO / C::REG_HI per thread)
//   warps 8-23 : compute, a quarter of the steps each: first the state
//                entering the segment into Ss (a quarter of the columns
//                each); then per chunk c the A operand into TMEM from the
//                staged x (kept in registers), and chunk c - 1's output
//                y = factor R + D x, staged per warp in shared memory and
//                written with one TMA store per warp
// ===========================================================================
constexpr int kComputeWarps = 16;  // warps 8..23

// VL: the units are packed sequences (prm.vl); MULTI: each unit runs several
// whole sequences one after another (with VL)
template <class C, typename YT, bool VL, bool MULTI = false>
__global__ void __launch_bounds__(C::SCAN_THREADS, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mdt,
                      const __grid_constant__ CUtensorMap my, const __grid_constant__ CUtensorMap mb,
                      const __grid_constant__ CUtensorMap mc, TcParams prm) {
    constexpr int ST = C::SCAN_ST, NV = C::NV, NB = C::NB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *vec_base = reinterpret_cast<float *>(smem + ST * C::SCAN_STAGE);
    uint8_t *dt_ring = smem + ST * C::SCAN_STAGE + C::VEC_RING;
    uint8_t *ystage = dt_ring + C::DT_RING;
    __shared__ uint64_t dt_bar[2];
    TRACE_DECL;
    // a stage's x tile and chunk pack land on separate barriers: the A
    // builders need only x, the MMAs only the pack
    __shared__ uint64_t full_bar[4], pfull_bar[4], empty_bar[4], vfull_bar[NV], vempty_bar[NV];
    __shared__ uint64_t afull_bar[NB], afree_bar[NB], rfull_bar[NB], rfree_bar[NB], sbfree_bar[NB];
    __shared__ uint64_t rt_bar, sdone_bar, drain_bar, sinit_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ volatile int slot[12];
    __shared__ __align__(16) float ones_sh[32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.z, hblk = blockIdx.x, b = blockIdx.y;
    const int h0 = hblk * C::HB;
    const int g = (int)(prm.G == 1 ? 0 : h0 / prm.hpg);
    // the unit's sequence: batch coordinate bq of the maps, first row t0,
    // length slen, first pack plane pbase (per group), state index sidx; its
    // segment: first local-state slot slot0 of the sequence, the local
    // states before it nprev, whether it follows others (segk > 0) and
    // whether it ends the sequence
    int bq = b, t0 = 0, sidx = b;
    long long slen = prm.L, pbase = (long long)b * prm.nc;
    int c0 = seg * prm.cps, nch = min(prm.nc, c0 + prm.cps) - c0;
    int segk = seg, slot0 = 0, nprev = seg * prm.nsub;
    bool last = seg == prm.nseg - 1;
    // (packed sequences: the table entry the unit's chunk walk starts at, and
    // whether the unit runs several sequences)
    int vj0 = 0;
    constexpr bool multi = MULTI;
    static_assert(VL || !MULTI, "several sequences per unit are packed sequences");
    if constexpr (VL) {
        VlUnit u = prm.vl[prm.vl_scan0 + b];
        vj0 = prm.vl_scan0 + b;
        if constexpr (MULTI) {
            vj0 = u.t0;
            nch = u.nch;
            u = prm.vl[vj0];
            u.c0 = 0;
            u.nprev = 0;
        } else {
            nch = u.nch;
        }
        bq = 0;
        t0 = u.t0;
        slen = u.len;
        sidx = u.seq;
        pbase = u.cbase;
        c0 = u.c0;
        segk = u.nprev > 0 ? 1 : 0;
        slot0 = u.slot;
        nprev = u.nprev;
        last = multi || c0 + nch >= (u.len + C::Q - 1) / C::Q;
    }
    const long long H = prm.H;
    auto stage_x = [&](int s) { return smem + s * C::SCAN_STAGE; };
    auto stage_cb = [&](int s) { return smem + s * C::SCAN_STAGE + C::X_BYTES; };
    auto stage_b = [&](int s) { return smem + s * C::SCAN_STAGE + C::X_BYTES + C::CBM_BYTES; };
    auto stage_c = [&](int s) { return smem + s * C::SCAN_STAGE + C::X_BYTES + C::CBM_BYTES + C::BC_BYTES; };
    auto vec = [&](int v) { return vec_base + v * C::VEC_FLOATS; };

    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&pfull_bar[i], 1);
            mbar_init(&empty_bar[i], 1 + kComputeWarps);  // the MMAs' commit; each compute warp once x is in registers
                                                            // (after its output step on a wide chunk)
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&vfull_bar[i], 1);
            mbar_init(&vempty_bar[i], 1 + kComputeWarps);  // state warps; each compute warp
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&afull_bar[i], kComputeWarps);
            mbar_init(&afree_bar[i], 1);
            mbar_init(&rfull_bar[i], 1);
            mbar_init(&rfree_bar[i], kComputeWarps);
            mbar_init(&sbfree_bar[i], 1);
        }
        mbar_init(&rt_bar, 1);
        mbar_init(&sinit_bar, kComputeWarps);  // the entering state is in Ss
        mbar_init(&sdone_bar, 1);
        mbar_init(&drain_bar, 1);
        for (int i = 0; i < 2; ++i) mbar_init(&dt_bar[i], 1);
        fence_mbar_init();
        abort_sh = 0;
        prefetch_tmap(&mx);
        prefetch_tmap(&mb);
        prefetch_tmap(&mc);
        if (prm.dt_tma) prefetch_tmap(&mdt);
    }
    if (tid < 32) ones_sh[tid] = 1.f;
    TRACE_INIT();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        TRACE(13, 0);
        TRACE_CTA(0);
    }
    const uint32_t tmem = tmem_base_sh;
    int nload[4] = {0, 0, 0, 0}, npack[4] = {0, 0, 0, 0};  // x boxes and packs issued per stage (producer lane 0)
    const int q4 = warp & 3;                  // TMEM lane quarter of this warp
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;

    if (warp < 4) {
        // (the whole warpgroup gives registers back at one program point)
        reg_dec<C::REG_LO>();
        if (warp == 0) {
            // ---------------- TMA producer ----------------
            VlCursor cur{prm.vl, vj0, c0};
            if (lane == 0)
                for (int it = 0; it < nch; ++it) {
                    const int s = it % ST;
                    if (it >= ST && !wait_bounded(&empty_bar[s], free_parity(it, ST), &abort_sh)) break;
                    long long plane = (pbase + c0 + it) * prm.G + g;
                    int row = t0 + (c0 + it) * C::Q;
                    if constexpr (MULTI) {
                        plane = ((long long)cur.cbase() + cur.c) * prm.G + g;
                        row = cur.t0() + cur.c * C::Q;
                        if (it + 1 < nch) cur.next<C::Q>();
                    }
                    // the x box, then the pack (C B^T, B, C)
                    if (prm.flag_first && !wait_flag(prm.cb_ready + plane, &abort_sh, prm.flag_wait_ns)) break;
                    mbar_arrive_expect_tx(&full_bar[s], C::X_BYTES);
                    tma_load_5d(stage_x(s), &mx, &full_bar[s], 0, 0, h0, row, bq);
                    ++nload[s];
                    // once the C B^T kernel has published the tile's masked C B^T:
                    // it, and the tile's B and C from the inputs (no copy of a
                    // stage is issued unless all three are)
                    if (!prm.flag_first && !wait_flag(prm.cb_ready + plane, &abort_sh, prm.flag_wait_ns)) break;
                    mbar_arrive_expect_tx(&pfull_bar[s], C::PACK_BYTES);
                    bulk_load(stage_cb(s), prm.pack + plane * C::CBM_BYTES, C::CBM_BYTES, &pfull_bar[s]);
                    tma_load_5d(stage_b(s), &mb, &pfull_bar[s], 0, row, 0, g, bq);
                    tma_load_5d(stage_c(s), &mc, &pfull_bar[s], 0, row, 0, g, bq);
                    ++npack[s];
                    TRACE(0, it);
                }
        } else if (warp == 2) {
            // ---------------- per-chunk vectors (run up to NV chunks ahead) ----------------
            constexpr int QPL = C::Q / 32;
            float rho[C::HB];
#pragma unroll
            for (int hh = 0; hh < C::HB; ++hh) rho[hh] = 0.f;
            auto chunk_of = [&](int it) { return c0 + it; };
            DtFeed<C, VL> feed{dt_ring, dt_bar, &mdt, bq, h0, nch, 0, t0, slen};
            // (a unit of several sequences takes each chunk's dt with plain
            // loads: its chunks' rows are not evenly spaced)
            if (!multi) feed.start(prm, chunk_of);
            VlCursor cur{prm.vl, vj0, c0};
            float Ah[C::HB];
            load_decay<C>(prm, h0, Ah);
            for (int it = 0; it < nch; ++it) {
                const int v = it % NV;
                ChunkDt<C> dt;
                if constexpr (MULTI) {
                    fetch_dt<C>(prm, 0, h0, cur.c, cur.t0(), cur.len(), dt);
                    if (cur.c == 0)  // a sequence starts: its state from its initial one, rho = 0
#pragma unroll
                        for (int hh = 0; hh < C::HB; ++hh) rho[hh] = 0.f;
                    if (it + 1 < nch) cur.next<C::Q>();
                } else if (!feed.take(prm, it, chunk_of, &abort_sh, dt)) {
                    break;
                }
                float cum[C::HB][QPL], T[C::HB];
                chunk_cums<C>(prm, b, h0, c0 + it, dt, Ah, cum, T);
                // range [lo, hi] of the cumulative decay over the chunk and its start (0)
                int klo[C::HB], khi[C::HB];
#pragma unroll
                for (int hh = 0; hh < C::HB; ++hh) {
                    float lo = 0.f, hi = 0.f;
#pragma unroll
                    for (int j = 0; j < QPL; ++j) {
                        lo = fminf(lo, cum[hh][j]);
                        hi = fmaxf(hi, cum[hh][j]);
                    }
                    klo[hh] = __reduce_min_sync(0xffffffffu, fkey(lo));
                    khi[hh] = __reduce_max_sync(0xffffffffu, fkey(hi));
                }
                bool rescale = false, wide = false;
                float al[C::HB][QPL], ef[C::HB][QPL], f[C::HB], sbf[C::HB], rn[C::HB];
#pragma unroll
                for (int hh = 0; hh < C::HB; ++hh) {
                    const float lo = unkey(klo[hh]), hi = unkey(khi[hh]);
                    // rho stays while every exponent rho - cum_s stays within kLambda;
                    // else it moves to the lowest reference the chunk allows,
                    // hi - kLambda (rho then grows by the decay of each later chunk,
                    // so the lowest start keeps it longest before the next move);
                    // a range wider than 2 kLambda centres the state at the chunk's
                    // end and leaves the intra-chunk term to the direct path.
                    // The rescale exp(rc - rho) may fall below the fp32 range (rho
                    // up to kLambda, rc down to -kLambda) while the rescaled state
                    // does not: the state warps apply it as two factors
                    // f = exp((rc - rho) / 2).  sbf < 0: the bf16 copy is the
                    // rescaled state; else the old state times sbf.
                    float rc = rho[hh];
                    f[hh] = 1.f;
                    sbf[hh] = 1.f;
                    bool hw = false;
                    if (rho[hh] - lo > kLambda || hi - rho[hh] > kLambda) {
                        rescale = true;
                        if (hi - lo <= 2.f * kLambda) {
                            rc = hi - kLambda;
                            f[hh] = __expf(0.5f * (rc - rho[hh]));
                            sbf[hh] = -1.f;
                        } else {
                            // (after a decay of more than 2 kLambda the old state is
                            // below fp32 resolution: f may flush to zero)
                            hw = true;
                            rc = T[hh];
                            f[hh] = __expf(0.5f * (T[hh] - rho[hh]));
                            sbf[hh] = __expf(-rho[hh]);
                        }
                    }
                    wide |= hw;
#pragma unroll
                    for (int j = 0; j < QPL; ++j) {
                        al[hh][j] = __expf(rc - cum[hh][j]) * dt.d[hh][j];
                        ef[hh][j] = __expf(hw ? cum[hh][j] : cum[hh][j] - rc);
                    }
                    rn[hh] = rc - T[hh];
                    rho[hh] = rn[hh];
                }
                if (it >= NV) {
                    int ok = lane == 0 ? (wait_bounded(&vempty_bar[v], free_parity(it, NV), &abort_sh) ? 1 : 0) : 0;
                    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                }
                float *vv = vec(v);
#pragma unroll
                for (int hh = 0; hh < C::HB; ++hh) {
#pragma unroll
                    for (int j = 0; j < QPL; ++j) {
                        const int q = hh * C::Q + QPL * lane + j;
                        vv[C::V_DT + q] = dt.d[hh][j];
                        vv[C::V_CUM + q] = cum[hh][j];
                        vv[C::V_AL + q] = al[hh][j];
                        vv[C::V_EF + q] = ef[hh][j];
                    }
                    if (lane == 0) {
                        vv[C::V_F + hh] = f[hh];
                        vv[C::V_SBF + hh] = sbf[hh];
                        vv[C::V_RHON + hh] = rn[hh];
                    }
                }
                if (lane == 0) {
                    vv[C::V_FLAG] = rescale ? 1.f : 0.f;
                    vv[C::V_FLAG + 1] = wide ? 1.f : 0.f;
                }
                __syncwarp();
                if (lane == 0) {
                    TRACE(1, it);
                    mbar_arrive(&vfull_bar[v]);
                }
            }
            if (!multi) feed.drain();
        } else if (warp == 1) {
            // ---------------- MMA issuer: the whole warp runs the loop (its
            // descriptors stay warp-uniform), one elected lane issues ----------------
            {
                const uint32_t id_intra = idesc_bf16(C::M, C::Q, false, false);
                const uint32_t id_state = idesc_bf16(C::M, C::N, false, true);
                const uint32_t id_inter = idesc_bf16(C::M, C::Q, false, false);
                for (int it = 0; it < nch; ++it) {
                    const int s = it % ST, a = it % NB;
                    // one descriptor per operand tile, advanced by constants (the
                    // single issuing thread must not spend cycles per MMA)
                    const uint64_t dcb = sdesc(smem_u32(stage_cb(s)), 16, 1024);
                    const uint64_t db = sdesc(smem_u32(stage_b(s)), C::Q * 128, 1024);
                    const uint64_t dc = sdesc(smem_u32(stage_c(s)), 16, 1024);
                    const uint32_t ta = tmem + C::COL_A + a * C::Q, tr = tmem + C::COL_R + a * C::Q;
                    const uint32_t tsb = tmem + C::COL_SB + a * (C::N / 2);
                    if (!warp_wait(&pfull_bar[s], fill_parity(it, ST), &abort_sh)) break;
                    TRACE(20, it);
                    if (!warp_wait(&afull_bar[a], fill_parity(it, NB), &abort_sh)) break;
                    TRACE(21, it);
                    // Ss += A^T B first: the state chain (state warps -> these
                    // MMAs -> state warps) is the longest loop of the pipeline, so
                    // it waits for no other MMA; once the state warps have read
                    // (and rescaled) Ss and written SB
                    if (!warp_wait(&rt_bar, (uint32_t)(it & 1), &abort_sh)) break;
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::Q / 16; ++ks)
                        mma_bf16_ta(tmem + C::COL_S, ta + ks * 16, desc_add(db, ks * 2048), id_state, true);
#pragma unroll
                    for (int ks = 0; ks < C::Q / 16; ++ks)
                        mma_bf16_ta(tmem + C::COL_S, ta + ks * 16 + 8, desc_add(db, ks * 2048), id_state, true);
                    mma_commit(&sdone_bar);
                    }
                    __syncwarp();
                    if (it >= NB && !warp_wait(&rfree_bar[a], free_parity(it, NB), &abort_sh)) break;
                    TRACE(22, it);
                    tc_fence_after();
                    const bool wide = vec(it % NV)[C::V_FLAG + 1] != 0.f;  // (the A builders saw this slot filled)
                    if (elect_one()) {
                    // R = A CB^T (hi, then lo)
                    if (!wide) {
#pragma unroll
                        for (int ks = 0; ks < C::Q / 16; ++ks)
                            mma_bf16_ta(tr, ta + ks * 16, desc_add(dcb, ks * 32), id_intra, ks > 0);
#pragma unroll
                        for (int ks = 0; ks < C::Q / 16; ++ks)
                            mma_bf16_ta(tr, ta + ks * 16 + 8, desc_add(dcb, ks * 32), id_intra, true);
                    }
                    mma_commit(&afree_bar[a]);
                    TRACE(2, it);
                    // R += SB C^T
#pragma unroll
                    for (int ks = 0; ks < C::N / 16; ++ks)
                        mma_bf16_ta(tr, tsb + ks * 8, desc_add(dc, (ks / 4) * (C::Q * 128) + (ks % 4) * 32), id_inter,
                                    !wide || ks > 0);
                    mma_commit(&rfull_bar[a]);
                    mma_commit(&sbfree_bar[a]);
                    mma_commit(&empty_bar[s]);
                    }
                    __syncwarp();
                }
            }
        }
    } else if ((warp >= 4 && warp < 8) || warp >= 24) {
        // ---------------- state: rescale and bf16 copy (C::SG groups of four
        // warps, each a 1 / SG share of the columns) ----------------
        constexpr int NT = 128 * C::SG;  // threads of the state groups
        constexpr int NCOL = C::N / C::SG;
        const int half = warp >= 24 ? 1 : 0;
        const int gtid = half ? tid - 768 + 128 : tid - 128;
        const int row = q4 * 32 + lane, rh = row / C::P, rp = row % C::P;
        const long long hrow = h0 + rh;
        // the compute warps write the state entering the segment into Ss
        if (!group_wait(&sinit_bar, 0, &abort_sh, &slot[3], 1, gtid, NT)) {
            // (abort: fall through; every wait below gives up at once)
        }
        tc_fence_after();
        if (gtid == 0) TRACE(13, 1);
        float rho_end = 0.f;
        // the final state S = exp(-rho) Ss of sequence seq_idx (fin [seq, H, P, N])
        auto write_fin = [&](long long seq_idx, float rho_e) {
            tc_fence_after();
            const float sc = __expf(-rho_e);
            float *dst = prm.fin + (((long long)seq_idx * H + hrow) * C::P + rp) * C::N;
            if constexpr (C::SG == 1 && C::DT_RING >= 4 * 2048) {
                // coalesced: each 16-column block goes through this warp's
                // 2 KB of the dt ring (idle once the last chunk's vector
                // set has been taken), the piece index XOR-ed with bits
                // 1-2 of the row, then out eight rows per store (the 32
                // rows of a warp are consecutive p of one head)
                float *scr = reinterpret_cast<float *>(dt_ring) + (warp - 4) * 512;
                float *dst0 = dst - (long long)lane * C::N;  // row of lane 0
                const int pc = lane & 3;
#pragma unroll 1
                for (int n0 = 0; n0 < C::N; n0 += 16) {
                    float v[16];
                    tmem_ld16(tmem + lane_off + C::COL_S + n0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<float4 *>(scr + lane * 16 + 4 * (j ^ ((lane >> 1) & 3))) =
                            make_float4(v[4 * j] * sc, v[4 * j + 1] * sc, v[4 * j + 2] * sc, v[4 * j + 3] * sc);
                    __syncwarp();
                    if (hrow < H)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = (lane >> 2) + 8 * i;
                            *reinterpret_cast<float4 *>(dst0 + (long long)r * C::N + n0 + 4 * pc) =
                                *reinterpret_cast<const float4 *>(scr + r * 16 + 4 * (pc ^ ((r >> 1) & 3)));
                        }
                    __syncwarp();
                }
            } else {
#pragma unroll 1
                for (int n0 = half * NCOL; n0 < (half + 1) * NCOL; n0 += 16) {
                    float v[16];
                    tmem_ld16(tmem + lane_off + C::COL_S + n0, v);
                    tmem_ld_wait();
                    if (hrow < H)
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(dst + n0 + j) =
                                make_float4(v[j] * sc, v[j + 1] * sc, v[j + 2] * sc, v[j + 3] * sc);
                }
            }
        };
        VlCursor cur{prm.vl, vj0, c0};
        int prev_seq = 0;  // (several sequences: the one the previous chunk ended)
        for (int it = 0; it < nch; ++it) {
            const int v = it % NV, sb = it % NB;
            // one thread waits for every phase this chunk needs (the vector
            // set, the previous state MMAs, the SB buffer), then one named
            // barrier hands the outcome to the state warps, which always leave
            // the loop together
            if (gtid == 0)
                slot[0] = (wait_bounded(&vfull_bar[v], fill_parity(it, NV), &abort_sh) &&
                           (it == 0 || wait_bounded(&sdone_bar, (uint32_t)((it - 1) & 1), &abort_sh)) &&
                           (it < NB || wait_bounded(&sbfree_bar[sb], free_parity(it, NB), &abort_sh)))
                              ? 1
                              : 0;
            named_bar_sync(1, NT);
            if (!slot[0]) break;
            if (gtid == 0) TRACE(7, it);
            tc_fence_after();
            if constexpr (MULTI) {
                if (it > 0 && cur.c == 0) {
                    // a sequence ends with the previous chunk (its state MMAs are
                    // done): its final state out, the next one's initial state
                    // (or zero) in, before this chunk's state MMAs are released
                    if (prm.fin) write_fin(prev_seq, rho_end);
                    const float *ini =
                        prm.init ? prm.init + (((long long)cur.seq() * H + hrow) * C::P + rp) * C::N : nullptr;
#pragma unroll 1
                    for (int n0 = half * NCOL; n0 < (half + 1) * NCOL; n0 += 32) {
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            const float4 q = ini && hrow < H ? __ldg(reinterpret_cast<const float4 *>(ini + n0 + j))
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                            v[j] = q.x;
                            v[j + 1] = q.y;
                            v[j + 2] = q.z;
                            v[j + 3] = q.w;
                        }
                        tmem_st32(tmem + lane_off + C::COL_S + n0, v);
                    }
                    tmem_st_wait();
                    // (every state thread has written its rows before any reads them back)
                    named_bar_sync(1, NT);
                }
            }
            const float *vv = vec(v);
            const float f = vv[C::V_F + rh], sbf = vv[C::V_SBF + rh];  // (f applied twice)
            const bool rescale = vv[C::V_FLAG] != 0.f;
            rho_end = vv[C::V_RHON + rh];
#pragma unroll 1
            for (int n0 = half * NCOL; n0 < (half + 1) * NCOL; n0 += 32) {
                float v[32];
                tmem_ld32(tmem + lane_off + C::COL_S + n0, v);
                tmem_ld_wait();
                uint32_t w[16];
                // (sbf and f are uniform per warp: one head per warp)
                if (sbf == 1.f) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                } else if (sbf > 0.f) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j] * sbf, v[2 * j + 1] * sbf);
                }
                if (rescale) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = (v[j] * f) * f;
                    tmem_st32(tmem + lane_off + C::COL_S + n0, v);
                }
                if (sbf < 0.f) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                }
                tmem_st16u(tmem + lane_off + C::COL_SB + sb * (C::N / 2) + n0 / 2, w);
            }
            tmem_st_wait();
            tc_fence_before();
            named_bar_sync(1, NT);
            if (gtid == 0) {
                TRACE(8, it);
                mbar_arrive(&rt_bar);
                mbar_arrive(&vempty_bar[v]);
            }
            if constexpr (MULTI) {
                if (it + 1 < nch) {
                    const int seq_now = cur.seq();
                    if (cur.next<C::Q>()) prev_seq = seq_now;
                }
            }
        }
        // final state after the segment's last chunk
        if (last && prm.fin) {  // (a uniform test: group_wait handles an abort)
            if (group_wait(&sdone_bar, (uint32_t)((nch - 1) & 1), &abort_sh, &slot[9], 1, gtid, NT)) {
                tc_fence_after();
                write_fin(multi ? (long long)cur.seq() : (long long)sidx, rho_end);
            }
        }
    } else if (warp >= 8 && warp < 24) {
        // ---------------- compute warps: thread = row (head, p), a quarter of the Q steps ----------------
        reg_inc<C::REG_HI>();
        // Chunk c: the A operand from the staged x (kept in registers), then
        // the output of chunk c - 1:  y = factor R + D x.
        const int part = (warp - 8) >> 2;
        constexpr int NS = C::Q / 4;
        const int row = q4 * 32 + lane, rh = row / C::P, rp = row % C::P;
        const uint32_t pcol = (uint32_t)(rp % 64);
        const int blk = rh * C::PB + rp / 64;
        const long long hrow = h0 + rh;
        const float dh = (prm.D && hrow < H) ? prm.D[hrow] : 0.f;
        // The state entering the segment (rho = 0: Ss = S_in), this warp's
        // quarter of the columns.  After segment 0 it is the pass across the
        // earlier segments' local states L_j (each from a zero state) and
        // totals T_j:
        //   S_in = e^{T_0 + .. + T_{k-1}} init + sum_j e^{T_{j+1} + .. + T_{k-1}} L_j
        {
            if (prm.dep_seg && segk > 0) griddep_wait();
            // (the 32 rows of a warp are 32 consecutive p of one head)
            const bool live = hrow < H;
            const float *dense = nullptr;  // a state in the row layout [.., P, N]: given, init, or init weighted
            const long long rowoff = (((long long)sidx * H + (live ? hrow : 0)) * C::P + rp) * C::N;
            if (prm.entering)
                dense = prm.entering + ((((long long)b * prm.nseg + seg) * H + (live ? hrow : 0)) * C::P + rp) * C::N;
            else if (prm.init)
                dense = prm.init + rowoff;
            // after segment 0 the local states are in the column-block layout
            // (nprev of them before this segment: its earlier sub-segments)
            const bool pass = !prm.entering && segk > 0;
            const long long sstride = H * C::P * C::N;
            const float *loc =
                pass ? prm.seg_state + (((long long)bq * prm.nslot + slot0) * H + (live ? hrow : 0)) * C::P * C::N +
                           rp * 4
                     : nullptr;
            const float *tot =
                pass ? prm.seg_tot + ((long long)bq * H + (live ? hrow : 0)) * prm.nslot + slot0 : nullptr;
            float ttot = 0.f;  // T_0 + .. + T_{k-1}
            if (pass && live)
                for (int j = 0; j < nprev; ++j) ttot += __ldcg(tot + j);
            const float wd = pass ? __expf(ttot) : 1.f;  // weight of the dense state
            // a row-layout state goes through this warp's 2 KB of the y
            // staging area (no y tile is staged before every compute warp
            // has passed here): 16-byte pieces read eight rows per load,
            // stored with the piece index XOR-ed by bits 1-2 of the row,
            // read back one row per lane, both without bank conflicts
            float *scr = reinterpret_cast<float *>(ystage) + (warp - 8) * 512;
            const float *dense0 = dense ? dense - (long long)lane * C::N : nullptr;  // row of lane 0
            constexpr int NCOL = C::N / 4;  // this warp's columns
#pragma unroll 1
            for (int n0 = part * NCOL; n0 < (part + 1) * NCOL; n0 += 16) {
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.f;
                if (live && dense0) {
                    const int pc = lane & 3;
                    float4 t4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = (lane >> 2) + 8 * i;
                        t4[i] = __ldg(reinterpret_cast<const float4 *>(dense0 + (long long)r * C::N + n0 + 4 * pc));
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = (lane >> 2) + 8 * i;
                        *reinterpret_cast<float4 *>(scr + r * 16 + 4 * (pc ^ ((r >> 1) & 3))) = t4[i];
                    }
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(scr + lane * 16 + 4 * (j ^ ((lane >> 1) & 3)));
                        v[4 * j] = wd * a4.x;
                        v[4 * j + 1] = wd * a4.y;
                        v[4 * j + 2] = wd * a4.z;
                        v[4 * j + 3] = wd * a4.w;
                    }
                    __syncwarp();
                }
                if (live && pass) {
                    // two segments' loads in flight before either is used
                    float pre = 0.f;  // T_0 + .. + T_j
                    for (int k = 0; k < nprev; k += 2) {
                        const bool two = k + 1 < nprev;
                        float4 l0[4], l1[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const long long o = (long long)(n0 / 4 + j) * (C::P * 4);
                            l0[j] = __ldcg(reinterpret_cast<const float4 *>(loc + k * sstride + o));
                            l1[j] = two ? __ldcg(reinterpret_cast<const float4 *>(loc + (k + 1) * sstride + o))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        const float t0 = __ldcg(tot + k), t1 = two ? __ldcg(tot + k + 1) : 0.f;
                        pre += t0;
                        const float w0 = __expf(ttot - pre);
                        pre += t1;
                        const float w1 = two ? __expf(ttot - pre) : 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            v[4 * j] = fmaf(w1, l1[j].x, fmaf(w0, l0[j].x, v[4 * j]));
                            v[4 * j + 1] = fmaf(w1, l1[j].y, fmaf(w0, l0[j].y, v[4 * j + 1]));
                            v[4 * j + 2] = fmaf(w1, l1[j].z, fmaf(w0, l0[j].z, v[4 * j + 2]));
                            v[4 * j + 3] = fmaf(w1, l1[j].w, fmaf(w0, l0[j].w, v[4 * j + 3]));
                        }
                    }
                }
                tmem_st16(tmem + lane_off + C::COL_S + n0, v);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sinit_bar);
        }
        uint32_t xprev[NS / 2];
        bool wide_prev = false;
        VlCursor ocur{prm.vl, vj0, c0};  // (packed sequences: the chunk whose output is next)
        for (int c = 0; c <= nch; ++c) {
            uint32_t xcur[NS / 2];
            bool wide = false;
            if (c < nch) {
                const int s = c % ST, v = c % NV, a = c % NB;
                if (!warp_wait(&full_bar[s], fill_parity(c, ST), &abort_sh)) break;
                if (warp == 8 && lane == 0) TRACE(12, c);
                if (!warp_wait(&vfull_bar[v], fill_parity(c, NV), &abort_sh)) break;
                if (c >= NB && !warp_wait(&afree_bar[a], free_parity(c, NB), &abort_sh)) break;
                if (warp == 8 && lane == 0) TRACE(5, c);
                tc_fence_after();
                const float *vv = vec(v);
                load_x_part<C, NS>(stage_x(s), blk, pcol, part, xcur);
                build_a_regs<C, NS>(xcur, vv + C::V_AL + rh * C::Q + part * NS, part,
                                    tmem + lane_off + C::COL_A + a * C::Q);
                wide = vv[C::V_FLAG + 1] != 0.f;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (warp == 8) TRACE(6, c);
                    mbar_arrive(&afull_bar[a]);
                    if (!wide) mbar_arrive(&empty_bar[s]);  // (a wide chunk's output step still reads the stage)
                }
            }
            if (c > 0) {
                const int cp = c - 1, s = cp % ST, v = cp % NV, r = cp % NB;
                if (!warp_wait(&rfull_bar[r], fill_parity(cp, NB), &abort_sh)) break;
                if (warp == 8 && lane == 0) TRACE(9, cp);
                tc_fence_after();
                const float *vv = vec(v);
                const float *ef = vv + C::V_EF + rh * C::Q + part * NS;
                const uint32_t tr = tmem + lane_off + C::COL_R + r * C::Q + part * NS;
                if (wide_prev) {
                    wide_fixup<C, NS>(tr, ef, stage_x(s), blk, stage_cb(s), vv + C::V_CUM + rh * C::Q,
                                      vv + C::V_DT + rh * C::Q, pcol, part * NS);
                    ef = ones_sh;
                }
                float acc[NS];
                tmem_ld16(tr, *reinterpret_cast<float(*)[16]>(acc));
                tmem_ld_wait();
                // straight to global memory: a warp writes one contiguous
                // run of 32 p per step; a partial last chunk stops at L
                // into the warp's [NS steps][32 p] staging tile (row j: the 32
                // consecutive p of step j), then one TMA store of the tile;
                // the store clips steps past L and heads past H
                YT *yt = reinterpret_cast<YT *>(ystage) + (warp - 8) * (NS * 32);
                if (lane == 0) bulk_wait_read_all();  // the previous chunk's store has read the tile
                __syncwarp();
#pragma unroll
                for (int j = 0; j < NS; j += 4) {
                    const float4 e4 = *reinterpret_cast<const float4 *>(ef + j);
                    const uint32_t w0 = xprev[j / 2], w1 = xprev[j / 2 + 1];
                    yt[(j + 0) * 32 + lane] = from_f32<YT>(fmaf(dh, __uint_as_float(w0 << 16), e4.x * acc[j]));
                    yt[(j + 1) * 32 + lane] = from_f32<YT>(fmaf(dh, __uint_as_float(w0 & 0xFFFF0000u), e4.y * acc[j + 1]));
                    yt[(j + 2) * 32 + lane] = from_f32<YT>(fmaf(dh, __uint_as_float(w1 << 16), e4.z * acc[j + 2]));
                    yt[(j + 3) * 32 + lane] = from_f32<YT>(fmaf(dh, __uint_as_float(w1 & 0xFFFF0000u), e4.w * acc[j + 3]));
                }
                fence_async_smem();
                __syncwarp();
                // step of the tile's first row in its sequence, the sequence's
                // first row and length
                long long trow = (long long)(c0 + cp) * C::Q + part * NS, yt0 = t0, ylen = slen;
                if constexpr (MULTI) {
                    trow = (long long)ocur.c * C::Q + part * NS;
                    yt0 = ocur.t0();
                    ylen = ocur.len();
                    if (cp + 1 < nch) ocur.next<C::Q>();
                }
                if (!VL || trow + NS <= ylen) {
                    if (lane == 0) {
                        tma_store_4d(&my, yt, (q4 * 32) % C::P, (int)(h0 + (q4 * 32) / C::P), (int)(yt0 + trow), bq);
                        bulk_commit_group();
                    }
                } else if constexpr (VL) {
                    // a packed sequence's partial last chunk: its rows stop at
                    // the sequence's end (the next rows belong to the next one)
                    if (h0 + (q4 * 32) / C::P < H) {
                        YT *yg = static_cast<YT *>(prm.y) +
                                 ((yt0 + trow) * H + h0 + (q4 * 32) / C::P) * C::P + (q4 * 32) % C::P + lane;
                        for (int j = 0; j < NS && trow + j < ylen; ++j)
                            yg[(long long)j * H * C::P] = yt[j * 32 + lane];
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (warp == 8) TRACE(10, cp);
                    mbar_arrive(&rfree_bar[r]);
                    mbar_arrive(&vempty_bar[v]);
                    if (wide_prev) mbar_arrive(&empty_bar[s]);
                }
            }
#pragma unroll
            for (int j = 0; j < NS / 2; ++j) xprev[j] = xcur[j];
            wide_prev = wide;
        }
    }
    // the compute warps' y stores complete before the CTA exits
    if (warp >= 8 && warp < 24 && lane == 0) bulk_wait_all();
    // let this CTA's own copies and MMAs land (they normally have) before
    // TMEM is freed and the CTA exits
    if (warp == 0 && lane == 0)
        for (int s = 0; s < ST; ++s) {
            if (nload[s] > 0) mbar_wait(&full_bar[s], (uint32_t)((nload[s] - 1) & 1), kDrainNs);
            if (npack[s] > 0) mbar_wait(&pfull_bar[s], (uint32_t)((npack[s] - 1) & 1), kDrainNs);
        }
    if (warp == 1 && lane == 0) {
        mma_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, kDrainNs);
    }
    tc_fence_before();
    __syncthreads();
    TRACE_FLUSH();
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

// 5-D map of B [b][L][G][N] viewed as (64, L, N/64, G, b), box (64, Q, N/64,
// 1, 1): one box per chunk lands as [N/64 blocks][Q steps][64] in shared memory
// (128-byte swizzle), the layout of N/64 separate (64, Q) boxes.
bool make_bt_map(CUtensorMap *m, const void *base, uint64_t N, uint64_t G, uint64_t L, uint64_t b, uint32_t Q) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[5] = {64, L, N / 64, G, b};
    cuuint64_t strides[4] = {G * N * 2, 128, N * 2, L * G * N * 2};
    cuuint32_t box[5] = {64, Q, (cuuint32_t)(N / 64), 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D map of x [b][L][H][P] viewed as (64, P/64, H, L, b), box (64, P/64, HB,
// Q, 1): one box per chunk holds the CTA's heads with 256 contiguous bytes
// per step ([Q][HB][P/64][64] in shared memory, 128-byte swizzle).
bool make_x_map(CUtensorMap *m, const void *base, uint64_t P, uint64_t H, uint64_t L, uint64_t b, uint32_t HB,
                uint32_t Q) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[5] = {64, P / 64, H, L, b};
    cuuint64_t strides[4] = {128, P * 2, P * H * 2, P * H * L * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)(P / 64), HB, Q, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map of y [b][L][H][P] (fp32 or bf16) as (P, H, L, b), box (32 p, 1
// head, Q/4 steps, 1), no swizzle: a compute warp's [Q/4][32] output tile.
// Stores clip at L and H.
bool make_y_map(CUtensorMap *m, void *base, bool f32, uint64_t P, uint64_t H, uint64_t L, uint64_t b, uint32_t Q) {
    auto enc = get_encode();
    if (!enc) return false;
    const uint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[4] = {P, H, L, b};
    cuuint64_t strides[3] = {P * es, P * H * es, P * H * L * es};
    cuuint32_t box[4] = {32, 1, Q / 4, 1};
    cuuint32_t el[4] = {1, 1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides,
               box, el, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// 3-D map of dt [b][L][H] (bf16), box (8 heads, 4 Q steps, 1); needs the row
// stride H * 2 bytes to be a multiple of 16 (H % 8 == 0).
bool make_dt_map(CUtensorMap *m, const void *base, uint64_t H, uint64_t L, uint64_t b, uint32_t Q) {
    auto enc = get_encode();
    if (!enc || H % 8 != 0) return false;
    cuuint64_t dims[3] = {H, L, b};
    cuuint64_t strides[2] = {H * 2, H * L * 2};
    cuuint32_t box[3] = {8, (cuuint32_t)(kDtGroup * Q), 1};
    cuuint32_t el[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, el,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int nseg, cps, nhb;
    int nsub;  // sub-segments of the segment-state pass (2: its two-CTAs-per-SM form)
};

// SM count of the current device (one chunk-scan CTA fits per SM); the
// GB300's 152 when no device can be queried (a workspace size asked for on
// a host without a GPU).
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 152;
    }
    return n;
}

template <class C>
Plan plan_for(const Dims &d) {
    Plan p;
    p.nhb = (int)((d.H + C::HB - 1) / C::HB);
    const long long units = d.b * p.nhb;
    int nseg = (int)(sm_count() / units);
    if (nseg < 1) nseg = 1;
    if (nseg > d.nc) nseg = (int)d.nc;
    p.cps = (int)((d.nc + nseg - 1) / nseg);
    p.nseg = (int)((d.nc + p.cps - 1) / p.cps);
    // The scans of the later segments wait for the whole segment-state pass:
    // its local states are formed on half segments by the two-group kernel,
    // two CTAs per SM, where S and two A buffers fit 256 TMEM columns and a
    // segment has two chunks or more (its CTAs take every SM, so the first
    // segment's scan starts once they end, which costs less than it saves).
    p.nsub = (p.nseg > 1 && C::N + 2 * C::Q <= 256 && p.cps >= 2) ? 2 : 1;
    return p;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// chunk packs [b, nc, G] of CBM_BYTES (the masked C B^T of each tile)
template <class C>
size_t pack_bytes(const Dims &d) {
    return align256((size_t)C::CBM_BYTES * d.b * d.nc * d.G);
}

// Workspace: chunk-pack ready flags [b, nc, G] | chunk packs | local
// states and totals of the nseg * nsub (sub-)segments.  The flags are
// cleared on the stream by every call.
size_t flag_bytes(const Dims &d) { return align256(sizeof(unsigned) * d.b * d.nc * d.G); }

template <class C>
size_t header_bytes(const Dims &d) {
    return flag_bytes(d);
}

#ifdef SSD_TRACE
constexpr size_t kTraceBytes = (32 * 256 + 4096) * sizeof(long long);
#endif

template <class C>
size_t workspace_for(const Dims &d) {
    const Plan p = plan_for<C>(d);
    size_t bytes = header_bytes<C>(d) + pack_bytes<C>(d);
    if (p.nseg > 1)
        bytes += align256(sizeof(float) * d.b * p.nseg * p.nsub * d.H * C::P * C::N) +
                 align256(sizeof(float) * d.b * p.nseg * p.nsub * d.H);
#ifdef SSD_TRACE
    bytes += kTraceBytes;
#endif
    return bytes;
}

// Launch with (pdl) or without a programmatic dependency on the previous
// work of the stream.  The first launch of an entry point never has one, so
// it waits for everything before it on the stream as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, int threads, int smem, cudaStream_t s, bool pdl,
                     Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <class C>
cudaError_t raise_smem(const void *fn, int bytes, int &done) {
    if (done >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done = bytes;
    return e;
}

// (walk: the packed sequences' tiles; null: the batch's)
template <class C>
cudaError_t launch_cb(const Dims &d, const void *B, const void *Cm, uint8_t *pack, unsigned *ready, unsigned *status,
                      cudaStream_t s, int ncta = 0, int nst_max = 2, const CbWalk *walk = nullptr) {
    // (packed sequences: launched with a programmatic dependency on the setup
    // kernel, which it waits for inside)
    CUtensorMap mb, mc;
    if (!make_bt_map(&mb, B, d.N, d.G, d.L, d.b, C::Q) || !make_bt_map(&mc, Cm, d.N, d.G, d.L, d.b, C::Q))
        return cudaErrorInvalidValue;
    CbWalk w{(int)d.nc, (int)d.G, (int)d.b, (long long)d.nc * d.b * d.G, nullptr, nullptr, 0};
    if (walk) w = *walk;
    // ncta > 0: that many CTAs walk the tiles, two stages deep (one CTA per SM
    // the scan leaves free); otherwise one CTA per tile
    const long long ntiles = w.ntiles;
    const int nst = ncta > 0 && ncta < ntiles ? nst_max : 1;
    const unsigned grid = ncta > 0 && ncta < ntiles ? (unsigned)ncta : (unsigned)ntiles;
    const int smem = C::smem_cb(nst);
    static int attr = 0;
    auto kern = walk ? cb_mask_kernel<C, true> : cb_mask_kernel<C, false>;
    static int attr_vl = 0;
    cudaError_t e =
        raise_smem<C>(reinterpret_cast<const void *>(kern), C::smem_cb(2), walk ? attr_vl : attr);
    if (e != cudaSuccess) return e;
    e = launch_k(kern, dim3(grid), 128, smem, s, walk != nullptr, mb, mc, pack, w, nst, ready, status);
    timing_mark(s, "cb_mask_tc");
    return e;
}

// pdl: the scan may start while the kernel before it on the stream (the
// C B^T kernel, which publishes its packs through ready flags) still runs.
template <class C, bool VL = false, bool MULTI = false>
cudaError_t launch_scan(const Dims &d, TcParams prm, ssd_dtype_t ydtype, const void *x, const void *B, const void *Cm,
                        dim3 grid, const char *name, bool pdl, cudaStream_t s) {
    CUtensorMap mx, mdt = {}, my, mb, mc;
    if (!make_bt_map(&mb, B, d.N, d.G, d.L, d.b, C::Q) || !make_bt_map(&mc, Cm, d.N, d.G, d.L, d.b, C::Q))
        return cudaErrorInvalidValue;
    prm.dt_tma = make_dt_map(&mdt, prm.dt, d.H, d.L, d.b, C::Q) ? 1 : 0;
    const bool f32 = ydtype == SSD_DTYPE_F32;
    if (!make_x_map(&mx, x, d.P, d.H, d.L, d.b, C::HB, C::Q)) return cudaErrorInvalidValue;
    if (!make_y_map(&my, prm.y, f32, d.P, d.H, d.L, d.b, C::Q)) return cudaErrorInvalidValue;
    static int attr_f = 0, attr_b = 0;
    // the warps' register split assumes the kernel's launch allocation: a
    // build that allocates otherwise must not run (an increase that cannot
    // be met would wait forever)
    {
        cudaFuncAttributes fa;
        cudaError_t e = f32 ? cudaFuncGetAttributes(&fa, chunk_scan_kernel<C, float, VL, MULTI>)
                            : cudaFuncGetAttributes(&fa, chunk_scan_kernel<C, bf16, VL, MULTI>);
        if (e != cudaSuccess) return e;
        if ((fa.numRegs + 7) / 8 * 8 != C::REG_LAUNCH) return cudaErrorInvalidConfiguration;
    }
    cudaError_t e;
    if (f32) {
        e = raise_smem<C>(reinterpret_cast<const void *>(chunk_scan_kernel<C, float, VL, MULTI>), C::SMEM_SCAN, attr_f);
        if (e != cudaSuccess) return e;
        e = launch_k(chunk_scan_kernel<C, float, VL, MULTI>, grid, C::SCAN_THREADS, C::SMEM_SCAN, s, pdl, mx, mdt, my, mb, mc, prm);
    } else {
        e = raise_smem<C>(reinterpret_cast<const void *>(chunk_scan_kernel<C, bf16, VL, MULTI>), C::SMEM_SCAN, attr_b);
        if (e != cudaSuccess) return e;
        e = launch_k(chunk_scan_kernel<C, bf16, VL, MULTI>, grid, C::SCAN_THREADS, C::SMEM_SCAN, s, pdl, mx, mdt, my, mb, mc, prm);
    }
    timing_mark(s, name);
    return e;
}

template <class C, int NBG = 4, bool VL = false>
cudaError_t launch_seg_state(const Dims &d, TcParams prm, const void *x, const void *B, dim3 grid,
                             const char *name, bool pdl, cudaStream_t s) {
    CUtensorMap mx, mb, mdt = {};
    if (!make_x_map(&mx, x, d.P, d.H, d.L, d.b, C::HB, C::Q) || !make_map(&mb, B, d.N, d.G, d.L, d.b, C::Q))
        return cudaErrorInvalidValue;
    prm.dt_tma = make_dt_map(&mdt, prm.dt, d.H, d.L, d.b, C::Q) ? 1 : 0;
    const int smem = SegT<C, NBG>::SMEM;
    static int attr = 0;
    cudaError_t e = raise_smem<C>(reinterpret_cast<const void *>(seg_state_kernel<C, NBG, VL>), smem, attr);
    if (e != cudaSuccess) return e;
    e = launch_k(seg_state_kernel<C, NBG, VL>, grid, SegT<C, NBG>::THREADS, smem, s, pdl, mx, mb, mdt, prm);
    timing_mark(s, name);
    return e;
}

TcParams base_params(const Dims &d, const void *dt, unsigned *status) {
    TcParams prm{};
    prm.dt = static_cast<const bf16 *>(dt);
    prm.status = status;
    prm.flag_wait_ns = kWaitNs;
    prm.b = d.b;
    prm.L = d.L;
    prm.H = d.H;
    prm.G = d.G;
    prm.hpg = d.hpg;
    prm.nc = (int)d.nc;
    prm.cum_q = (int)d.Q;
    prm.nc_cum = (int)d.nc;
    return prm;
}

template <class C>
cudaError_t run_fwd(const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B,
                    const void *Cm, const float *D, const float *init, void *y, float *fin, void *ws,
                    unsigned *status, cudaStream_t s) {
    const Plan p = plan_for<C>(d);
    TcParams prm = base_params(d, dt, status);
    prm.x = static_cast<const bf16 *>(x);
    prm.A = A;
    prm.D = D;
    prm.init = init;
    prm.y = y;
    prm.fin = fin;
    char *w = static_cast<char *>(ws);
    const size_t hdr = header_bytes<C>(d);
    prm.cb_ready = reinterpret_cast<unsigned *>(w);
    uint8_t *pack = reinterpret_cast<uint8_t *>(w + hdr);
    prm.pack = pack;
    const size_t seg_off = hdr + pack_bytes<C>(d);
    if (p.nseg > 1) {
        prm.seg_state = reinterpret_cast<float *>(w + seg_off);
        prm.seg_cl = 1;
        prm.seg_tot = reinterpret_cast<float *>(
            w + seg_off + align256(sizeof(float) * d.b * p.nseg * p.nsub * d.H * C::P * C::N));
    }
    prm.nhb = p.nhb;
    prm.nseg = p.nseg;
    prm.cps = p.cps;
    prm.nsub = p.nsub;
    prm.nslot = p.nseg * p.nsub;
#ifdef SSD_TRACE
    prm.trace = reinterpret_cast<long long *>(w + workspace_for<C>(d) - kTraceBytes);
#endif
    cudaError_t e = cudaMemsetAsync(w, 0, hdr, s);
    if (e != cudaSuccess) return e;
    timing_begin(s);
    // with one segment the scan's CTAs leave SMs free: the C B^T tiles are
    // walked by one CTA on each of those, and the scan starts at once
    const long long units = d.b * p.nhb, spare = sm_count() - units;
    // with segments, at most one C B^T CTA per SM (single stage), so that two
    // segment-state CTAs fit beside it on every SM
    e = p.nseg == 1 ? launch_cb<C>(d, B, Cm, pack, prm.cb_ready, prm.status, s, spare >= 8 ? (int)spare : 0)
                    : launch_cb<C>(d, B, Cm, pack, prm.cb_ready, prm.status, s, sm_count(), 1);
    if (e != cudaSuccess) return e;
    if (p.nseg > 1) {
        const dim3 grid(p.nhb, (unsigned)d.b, (unsigned)((p.nseg - 1) * p.nsub));
        if constexpr (C::N + 2 * C::Q <= 256)
            e = p.nsub == 2 ? launch_seg_state<C, 2>(d, prm, x, B, grid, "seg_state_tc", true, s)
                            : launch_seg_state<C>(d, prm, x, B, grid, "seg_state_tc", true, s);
        else
            e = launch_seg_state<C>(d, prm, x, B, grid, "seg_state_tc", true, s);
        if (e != cudaSuccess) return e;
        prm.dep_seg = 1;
    }
    // segments in the slowest grid dimension: the first segment's CTAs, which
    // need nothing from the segment-state kernel, are scheduled first
    return launch_scan<C>(d, prm, ydtype, x, B, Cm, dim3(p.nhb, (unsigned)d.b, p.nseg), "chunk_scan_tc", true, s);
}

// ---------------------------------------------------------------------------
// Packed sequences of unequal lengths in one launch set: the sequences
// longest first, each cut into segments of cps chunks (one segment each when
// their units fill the SMs), a scan unit per (segment, head block) and a
// segment-state unit per sub-segment of every segment but a sequence's last.
// The table reaches the device as a kernel parameter of the setup kernel,
// which also clears the pack flags (it takes the place of the flag memset):
// [0, n) the sequences (the C B^T walk; without segments also the scan's
// units), then the scan units, then the segment-state units.
// ---------------------------------------------------------------------------
constexpr int kVlEntries = kVarlenMaxUnits;
struct VlArgs {
    int n, nlvl, ntotal;  // sequences; chunk levels (the longest sequence's chunks); entries
    VlUnit u[kVlEntries];
};
static_assert(sizeof(VlArgs) <= 31 * 1024, "kernel parameter space");

// vl_off[c] = the chunks of levels below c = sum over sequences of min(nc_i, c).
template <int Q>
__global__ void varlen_setup_kernel(const __grid_constant__ VlArgs a, VlUnit *vl, int *vl_off, unsigned *flags,
                                    long long nflags) {
    // the C B^T grid may launch at once: it waits for this grid's completion
    // before it reads the table or touches a flag
    griddep_launch();
    const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x, nthr = (long long)gridDim.x * blockDim.x;
    for (long long i = tid; i < a.ntotal; i += nthr) vl[i] = a.u[i];
    for (long long c = tid; c <= a.nlvl; c += nthr) {
        long long o = 0;
        for (int i = 0; i < a.n; ++i) o += min((a.u[i].len + Q - 1) / Q, (int)c);
        vl_off[c] = (int)o;
    }
    for (long long i = tid; i < nflags; i += nthr) flags[i] = 0u;
}

// The shape of one launch set.
struct VlPlan {
    int n = 0, nlvl = 0;
    long long nchunks = 0;
    int cps = 0, nsub = 1;  // chunks per segment (the longest sequence's: no segments), sub-segments
    int nscan = 0, nsegu = 0, maxseg = 1;  // units of the scan and of the segment-state pass; most segments
    // several whole sequences per scan unit: the units' chunk target, the
    // most chunks and sequences of one unit (0: one sequence per unit)
    int gchunks = 0, gmaxc = 0, gmaxn = 0;
    bool segmented() const { return nsegu > 0; }
    bool grouped() const { return gchunks > 0; }
    long long entries() const { return n + (segmented() ? (long long)nscan + nsegu : grouped() ? nscan : 0); }
};

// Consecutive sequences (longest first) into units of at most `target`
// chunks (a longer sequence alone); calls f(first, count, chunks) per unit.
template <int Q, class F>
void varlen_groups(const VarlenSeq *seqs, int n, int target, F f) {
    int i0 = 0, cnt = 0, ch = 0;
    for (int i = 0; i < n; ++i) {
        const int nc = (seqs[i].len + Q - 1) / Q;
        if (cnt > 0 && ch + nc > target) {
            f(i0, cnt, ch);
            i0 = i;
            cnt = 0;
            ch = 0;
        }
        ++cnt;
        ch += nc;
    }
    if (cnt > 0) f(i0, cnt, ch);
}

// The cost model of a launch set (microseconds), fitted to GB300 timings of
// the 130M-shaped heads (one sequence of 128 to 8192 steps; sets of 4 to 256
// sequences), within ~12 %:
//   one segment per sequence: kSetUs + max(the longest unit, ceil(units /
//     SMs) x the mean unit), a unit (one scan CTA) taking kUnitUs +
//     kSetChunkUs per 64-step tile;
//   a fused forward: kFwdUs + kFwdChunkUs per tile of a segment + kPrevUs
//     per local state the last segment's prologue combines; a set with
//     segments the same plus kSetUs / 4 (its setup kernel), its tiles those
//     of a segment or, when the units overflow the SMs, 1.15 x the tiles
//     per SM;
//   several sequences per unit: kSetUs + waves x (kUnitUs + kSetChunkUs
//     per tile of the largest unit + kSeqUs per sequence boundary in the
//     unit with the most: the state written out and reset, the state chain
//     stalled meanwhile).
// Tile costs scale by 1.35 for N = 256.
constexpr double kSetUs = 8.0, kUnitUs = 6.5, kSetChunkUs = 1.7, kSeqUs = 3.5;
constexpr double kFwdUs = 17.6, kFwdChunkUs = 2.1, kPrevUs = 0.75;
double n_scale(long long N) { return N > 128 ? 1.35 : 1.0; }

double set_cost_us(const VlPlan &p, long long nhb, long long N) {
    const long long sms = sm_count();
    const double per_sm = (double)p.nchunks * nhb / sms;
    if (p.grouped()) {
        const long long waves = ((long long)p.nscan * nhb + sms - 1) / sms;
        return kSetUs + (double)waves * (kUnitUs + kSetChunkUs * n_scale(N) * p.gmaxc + kSeqUs * (p.gmaxn - 1));
    }
    if (p.segmented())
        return kSetUs / 4 + kFwdUs + kPrevUs * (p.maxseg - 1) * p.nsub +
               kFwdChunkUs * n_scale(N) * std::max((double)p.cps, 1.15 * per_sm);
    const long long waves = ((long long)p.n * nhb + sms - 1) / sms;
    const double tile = kSetChunkUs * n_scale(N);
    const double longest = kUnitUs + tile * p.nlvl, mean = kUnitUs + tile * (double)p.nchunks / p.n;
    return kSetUs + std::max(longest, (double)waves * mean);
}

// Segments of cps chunks when they shorten the set by the model: the fewest
// chunks per segment that keep the scan's units within the SMs when the
// sequences alone leave SMs free, else about 1.25 x the tiles per SM (only
// the sequences longer than that are cut).
template <class C>
VlPlan varlen_plan(const VarlenSeq *seqs, int n, int H) {
    VlPlan base;
    base.n = n;
    for (int i = 0; i < n; ++i) {
        const int nc = (seqs[i].len + C::Q - 1) / C::Q;
        base.nchunks += nc;
        base.nlvl = std::max(base.nlvl, nc);
    }
    const long long nhb = (H + C::HB - 1) / C::HB, sms = sm_count();
    auto units = [&](int cps) {
        long long u = 0;
        for (int i = 0; i < n; ++i) u += ((seqs[i].len + C::Q - 1) / C::Q + cps - 1) / cps;
        return u;
    };
    auto make = [&](int cps) {
        VlPlan p = base;
        p.cps = cps;
        p.nscan = (int)units(cps);
        if (cps < p.nlvl) {
            p.nsub = (cps >= 2 && C::N + 2 * C::Q <= 256) ? 2 : 1;
            p.nsegu = (int)(p.nscan - n) * p.nsub;
            p.maxseg = (p.nlvl + cps - 1) / cps;
        }
        return p;
    };
    VlPlan best = make(base.nlvl);
    int cut;
    if ((long long)n * nhb < sms) {
        int lo = 1, hi = base.nlvl;
        while (lo < hi) {
            const int mid = (lo + hi) / 2;
            if (units(mid) * nhb <= sms) hi = mid;
            else lo = mid + 1;
        }
        cut = lo;
    } else {
        cut = (int)std::ceil(1.25 * (double)base.nchunks * nhb / sms);
    }
    if (cut >= 1 && cut < base.nlvl) {
        const VlPlan q = make(cut);
        if (q.entries() <= kVlEntries && set_cost_us(q, nhb, C::N) < set_cost_us(best, nhb, C::N)) best = q;
    }
    // several short sequences per unit, the units one wave (their CTAs' fixed
    // cost paid once per SM rather than once per sequence)
    if ((long long)n * nhb > sms && n > 1) {
        int target = std::max<int>(base.nlvl, (int)((base.nchunks * nhb + sms - 1) / sms));
        for (;; ++target) {
            VlPlan q = base;
            q.cps = base.nlvl;
            q.gchunks = target;
            varlen_groups<C::Q>(seqs, n, target, [&](int, int cnt, int ch) {
                ++q.nscan;
                q.gmaxc = std::max(q.gmaxc, ch);
                q.gmaxn = std::max(q.gmaxn, cnt);
            });
            if ((long long)q.nscan * nhb <= sms || target >= base.nchunks) {
                if (q.nscan < n && q.entries() <= kVlEntries && set_cost_us(q, nhb, C::N) < set_cost_us(best, nhb, C::N))
                    best = q;
                break;
            }
        }
    }
    return best;
}

// Entries of the set (the sequences in the given order, longest first).
template <class C>
void varlen_entries(const VarlenSeq *seqs, const VlPlan &p, VlArgs &a) {
    a.n = p.n;
    a.nlvl = p.nlvl;
    int k = 0, slot = 0;
    for (int i = 0; i < p.n; ++i) {
        const int nc = (seqs[i].len + C::Q - 1) / C::Q;
        a.u[i] = VlUnit{seqs[i].t0, seqs[i].len, k, seqs[i].seq, 0, nc, 0, 0};
        k += nc;
    }
    a.ntotal = p.n;
    if (p.grouped()) {
        varlen_groups<C::Q>(seqs, p.n, p.gchunks, [&](int i0, int cnt, int ch) {
            a.u[a.ntotal++] = VlUnit{i0, cnt, 0, -1, 0, ch, 0, 0};
        });
        return;
    }
    if (!p.segmented()) return;
    // scan units, the longest first (the block scheduler hands out SMs in
    // unit order): every sequence's full segments, first segments before
    // later ones, then the shorter last segments; a later segment holds its
    // SM while the segment-state pass runs, but a long one started last
    // would end last
    std::vector<int> slot0(p.n);
    for (int i = 0; i < p.n; ++i) {
        slot0[i] = slot;
        slot += ((a.u[i].nch + p.cps - 1) / p.cps - 1) * p.nsub;
    }
    for (int seg = 0; seg < p.maxseg; ++seg)
        for (int i = 0; i < p.n; ++i) {
            const int c0 = seg * p.cps, nc = a.u[i].nch;
            if (c0 >= nc) continue;
            VlUnit u = a.u[i];
            u.c0 = c0;
            u.nch = std::min(nc, c0 + p.cps) - c0;
            u.slot = slot0[i];
            u.nprev = seg * p.nsub;
            a.u[a.ntotal++] = u;
        }
    std::stable_sort(a.u + p.n, a.u + a.ntotal, [](const VlUnit &x, const VlUnit &y) { return x.nch > y.nch; });
    const int csub = (p.cps + p.nsub - 1) / p.nsub;
    for (int i = 0; i < p.n; ++i) {
        const int nseg = (a.u[i].nch + p.cps - 1) / p.cps;
        for (int seg = 0; seg + 1 < nseg; ++seg)
            for (int sub = 0; sub < p.nsub; ++sub) {
                VlUnit u = a.u[i];
                u.c0 = seg * p.cps + sub * csub;
                u.nch = std::min(seg * p.cps + p.cps, u.c0 + csub) - u.c0;
                u.slot = slot0[i] + seg * p.nsub + sub;
                u.nprev = 0;
                a.u[a.ntotal++] = u;
            }
    }
}

struct VlLayout {
    size_t flags, pack, table, off, states, totals, total;
};

template <class C>
VlLayout varlen_layout(const Dims &d, const VlPlan &p) {
    VlLayout l;
    const long long nplanes = p.nchunks * d.G;
    const long long entries = p.entries();
    l.flags = 0;
    l.pack = align256(sizeof(unsigned) * nplanes);
    l.table = l.pack + align256((size_t)C::CBM_BYTES * nplanes);
    l.off = l.table + align256(sizeof(VlUnit) * entries);
    l.states = l.off + align256(sizeof(int) * (p.nlvl + 1));
    l.totals = l.states + (p.segmented() ? align256(sizeof(float) * p.nsegu * d.H * C::P * C::N) : 0);
    l.total = l.totals + (p.segmented() ? align256(sizeof(float) * p.nsegu * d.H) : 0);
    return l;
}

template <class C>
cudaError_t run_fwd_varlen(const Dims &d, const VlPlan &p, const VlArgs &a, ssd_dtype_t ydtype, const void *x,
                           const void *dt, const float *A, const void *B, const void *Cm, const float *D,
                           const float *init, void *y, float *fin, void *ws, unsigned *status, cudaStream_t s) {
    const VlLayout l = varlen_layout<C>(d, p);
    char *w = static_cast<char *>(ws);
    const long long nflags = p.nchunks * d.G;
    TcParams prm = base_params(d, dt, status);
    prm.x = static_cast<const bf16 *>(x);
    prm.A = A;
    prm.D = D;
    prm.init = init;
    prm.y = y;
    prm.fin = fin;
    prm.cb_ready = reinterpret_cast<unsigned *>(w + l.flags);
    prm.pack = reinterpret_cast<uint8_t *>(w + l.pack);
    prm.nhb = (int)((d.H + C::HB - 1) / C::HB);
    prm.nseg = 1;
    prm.cps = (int)d.nc;
    prm.nsub = p.nsub;
    prm.nslot = std::max(1, p.nsegu);
    VlUnit *vl = reinterpret_cast<VlUnit *>(w + l.table);
    int *vl_off = reinterpret_cast<int *>(w + l.off);
    prm.vl = vl;
    prm.vl_scan0 = p.segmented() || p.grouped() ? p.n : 0;
    prm.vl_seg0 = p.n + p.nscan;
    if (p.segmented()) {
        prm.seg_state = reinterpret_cast<float *>(w + l.states);
        prm.seg_cl = 1;
        prm.seg_tot = reinterpret_cast<float *>(w + l.totals);
    }
    const long long work = std::max<long long>(std::max<long long>(nflags, a.nlvl + 1), a.ntotal);
    const unsigned blocks = (unsigned)std::min<long long>((work + 255) / 256, sm_count());
    timing_begin(s);
    varlen_setup_kernel<C::Q><<<blocks, 256, 0, s>>>(a, vl, vl_off, prm.cb_ready, nflags);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    timing_mark(s, "varlen_setup");
    const CbWalk walk{(int)d.nc, (int)d.G, 1, nflags, vl, vl_off, a.nlvl};
    uint8_t *pack = reinterpret_cast<uint8_t *>(w + l.pack);
    if (!p.segmented()) {
        // one segment per sequence: the C B^T tiles are walked by one CTA on
        // each SM the scan leaves free (as for an equal-length batch); units
        // of several sequences take their chunks sequence by sequence, out of
        // the walk's level order, so their tiles are all launched at once
        const long long units = (long long)p.nscan * prm.nhb, spare = sm_count() - units;
        e = launch_cb<C>(d, B, Cm, pack, prm.cb_ready, prm.status, s, spare >= 8 && !p.grouped() ? (int)spare : 0, 2,
                         &walk);
        if (e != cudaSuccess) return e;
        return p.grouped() ? launch_scan<C, true, true>(d, prm, ydtype, x, B, Cm, dim3(prm.nhb, (unsigned)p.nscan, 1),
                                                        "chunk_scan_tc", true, s)
                           : launch_scan<C, true>(d, prm, ydtype, x, B, Cm, dim3(prm.nhb, (unsigned)p.nscan, 1),
                                                  "chunk_scan_tc", true, s);
    }
    // segments: at most one C B^T CTA per SM beside the segment-state CTAs
    e = launch_cb<C>(d, B, Cm, pack, prm.cb_ready, prm.status, s, sm_count(), 1, &walk);
    if (e != cudaSuccess) return e;
    const dim3 sgrid(prm.nhb, 1, (unsigned)p.nsegu);
    if constexpr (C::N + 2 * C::Q <= 256)
        e = p.nsub == 2 ? launch_seg_state<C, 2, true>(d, prm, x, B, sgrid, "seg_state_tc", true, s)
                        : launch_seg_state<C, 4, true>(d, prm, x, B, sgrid, "seg_state_tc", true, s);
    else
        e = launch_seg_state<C, 4, true>(d, prm, x, B, sgrid, "seg_state_tc", true, s);
    if (e != cudaSuccess) return e;
    prm.dep_seg = 1;
    return launch_scan<C, true>(d, prm, ydtype, x, B, Cm, dim3(prm.nhb, (unsigned)p.nscan, 1), "chunk_scan_tc", true,
                                s);
}

// Dispatch over the compiled tile configurations.
template <class F>
bool dispatch(const Dims &d, F &&f) {
    if (d.P == 64 && d.N == 128 && d.Q == 64) return f(Cfg<64, 128, 64>{}), true;
    if (d.P == 128 && d.N == 256 && d.Q == 64) return f(Cfg<128, 256, 64>{}), true;
    if (d.P == 64 && d.N == 64 && d.Q == 64) return f(Cfg<64, 64, 64>{}), true;
    return false;
}

template <class C>
bool shape_ok(const Dims &d) {
    return C::SCAN_FITS && C::TMEM_FITS && (d.G == 1 || d.hpg % C::HB == 0) && d.L < (1ll << 31) &&
           d.H < (1 << 30) && d.b < 65536 && d.nc < 65536 && d.G < 65536 && d.b * d.nc * d.G < (1ll << 31);
}

// The fused forward's output does not depend on the chunk length beyond
// rounding (chunked and unchunked sums agree exactly in exact arithmetic),
// so a 128-step chunk runs as two 64-step tiles: the tile configurations
// hold a 64-step chunk's operands in TMEM and shared memory.
Dims fwd_tiles(const Dims &d) {
    Dims t = d;
    if (d.Q == 128) {
        t.Q = 64;
        t.nc = (d.L + 63) / 64;
    }
    return t;
}

}  // namespace

bool tc_fwd_supported(const Dims &dq, ssd_dtype_t dtype) {
    const Dims d = fwd_tiles(dq);
    if (dtype != SSD_DTYPE_BF16) return false;
    if (d.L == 0 || d.b == 0) return false;
    bool ok = false;
    dispatch(d, [&](auto c) {
        using C = decltype(c);
        ok = shape_ok<C>(d) && C::SMEM_SEG <= kSmemLimit;
    });
    return ok;
}

size_t tc_fwd_workspace(const Dims &dq) {
    const Dims d = fwd_tiles(dq);
    size_t bytes = 0;
    dispatch(d, [&](auto c) { bytes = workspace_for<decltype(c)>(d); });
    return bytes;
}

cudaError_t tc_fwd(const Dims &dq, ssd_dtype_t ydtype, const void *x, const void *dt, const float *A, const void *B,
                   const void *C, const float *D, const float *init, void *y, float *fin, void *ws,
                   unsigned *status, cudaStream_t s) {
    const Dims d = fwd_tiles(dq);
    cudaError_t e = cudaErrorNotSupported;
    dispatch(d, [&](auto c) { e = run_fwd<decltype(c)>(d, ydtype, x, dt, A, B, C, D, init, y, fin, ws, status, s); });
    return e;
}

bool tc_varlen_supported(const Dims &dq, ssd_dtype_t dtype) {
    if (!tc_fwd_supported(dq, dtype)) return false;
    const Dims d = fwd_tiles(dq);
    return d.b == 1 && d.L < (1ll << 30) && (d.L / 64 + kVarlenMaxUnits) * d.G < (1ll << 31);
}

namespace {
// The sequences sorted longest first (the order of a set's units).
std::vector<VarlenSeq> longest_first(const VarlenSeq *seqs, int n) {
    std::vector<VarlenSeq> v(seqs, seqs + n);
    auto longer = [](const VarlenSeq &p, const VarlenSeq &q) { return p.len > q.len; };
    if (!std::is_sorted(v.begin(), v.end(), longer)) std::stable_sort(v.begin(), v.end(), longer);
    return v;
}
}  // namespace

size_t tc_varlen_workspace(const Dims &dq, const VarlenSeq *seqs, int n) {
    const Dims d = fwd_tiles(dq);
    if (n <= 0 || n > kVarlenMaxUnits) return 0;
    const std::vector<VarlenSeq> v = longest_first(seqs, n);
    size_t bytes = 0;
    dispatch(d, [&](auto c) {
        using C = decltype(c);
        bytes = varlen_layout<C>(d, varlen_plan<C>(v.data(), n, (int)d.H)).total;
    });
    return bytes;
}

cudaError_t tc_fwd_varlen(const Dims &dq, const VarlenSeq *seqs, int n, ssd_dtype_t ydtype, const void *x,
                          const void *dt, const float *A, const void *B, const void *C, const float *D,
                          const float *init, void *y, float *fin, void *ws, unsigned *status, cudaStream_t s) {
    const Dims d = fwd_tiles(dq);
    if (n <= 0 || n > kVarlenMaxUnits) return cudaErrorInvalidValue;
    const std::vector<VarlenSeq> v = longest_first(seqs, n);
    thread_local VlArgs a;  // (the launch copies it into its parameters)
    cudaError_t e = cudaErrorNotSupported;
    dispatch(d, [&](auto c) {
        using Cf = decltype(c);
        const VlPlan p = varlen_plan<Cf>(v.data(), n, (int)d.H);
        varlen_entries<Cf>(v.data(), p, a);
        e = run_fwd_varlen<Cf>(d, p, a, ydtype, x, dt, A, B, C, D, init, y, fin, ws, status, s);
    });
    return e;
}

double tc_varlen_cost_us(const Dims &dq, const VarlenSeq *seqs, int n) {
    const Dims d = fwd_tiles(dq);
    if (n == 0) return 0.0;
    const std::vector<VarlenSeq> v = longest_first(seqs, n);
    double us = 0;
    dispatch(d, [&](auto c) {
        using C = decltype(c);
        us = set_cost_us(varlen_plan<C>(v.data(), n, (int)d.H), (d.H + C::HB - 1) / C::HB, C::N);
    });
    return us;
}

double tc_fwd_cost_us(const Dims &dq, int64_t len) {
    Dims d = fwd_tiles(dq);
    d.b = 1;
    d.L = len;
    d.nc = (len + d.Q - 1) / d.Q;
    double us = 0;
    dispatch(d, [&](auto c) {
        const Plan p = plan_for<decltype(c)>(d);
        us = kFwdUs + kFwdChunkUs * n_scale(d.N) * p.cps + kPrevUs * (p.nseg - 1) * p.nsub;
    });
    return us;
}

bool tc_stage_supported(const Dims &dq, ssd_dtype_t dtype) {
    if (dtype != SSD_DTYPE_BF16 || dq.L == 0 || dq.b == 0) return false;
    const Dims d = fwd_tiles(dq);
    bool ok = false;
    dispatch(d, [&](auto c) {
        using C = decltype(c);
        ok = shape_ok<C>(d) && C::SMEM_SEG <= kSmemLimit;
    });
    return ok;
}

namespace {

// A stage call's chunks of dq.Q steps run as segments of dq.Q / 64 tiles of
// 64 steps (d = the tile dimensions).
template <class C>
cudaError_t run_chunk_state(const Dims &dq, const Dims &d, const void *x, const void *dt, const void *B,
                            const float *cum, float *states, unsigned *status, cudaStream_t s) {
    TcParams prm = base_params(d, dt, status);
    prm.cum_in = cum;
    prm.cum_q = (int)dq.Q;
    prm.nc_cum = (int)dq.nc;
    prm.seg_state = states;  // [b, nc, H, P, N]: one segment per chunk
    prm.nseg = (int)dq.nc;
    prm.cps = (int)(dq.Q / C::Q);
    prm.nsub = 1;
    prm.nslot = prm.nseg;
    prm.nhb = (int)((d.H + C::HB - 1) / C::HB);
    timing_begin(s);
    return launch_seg_state<C>(d, prm, x, B, dim3((unsigned)prm.nhb, (unsigned)d.b, (unsigned)dq.nc),
                               "chunk_state_tc", false, s);
}

// The chunk packs of a stage call and their ready flags live in the
// caller's workspace: flags [b, nc, G] | packs.  With `selftest_ns` > 0 the
// C B^T kernel is not launched, so no pack is ever published and the scan's
// wait for its first pack runs out after that many nanoseconds (the test of
// the bounded waits; the producer waits before it issues any load).
template <class C>
size_t scan_stage_workspace(const Dims &d) {
    return flag_bytes(d) + pack_bytes<C>(d);
}

template <class C>
cudaError_t run_chunk_scan(const Dims &dq, const Dims &d, ssd_dtype_t ydtype, const void *x, const void *dt,
                           const void *B, const void *Cm, const float *cum, const float *states_in, const float *D,
                           void *y, void *ws, unsigned *status, uint64_t selftest_ns, cudaStream_t s) {
    TcParams prm = base_params(d, dt, status);
    prm.cum_in = cum;
    prm.cum_q = (int)dq.Q;
    prm.nc_cum = (int)dq.nc;
    prm.entering = states_in;  // [b, nc, H, P, N]: the state entering each chunk
    prm.x = static_cast<const bf16 *>(x);
    prm.D = D;
    prm.y = y;
    prm.nseg = (int)dq.nc;
    prm.cps = (int)(dq.Q / C::Q);
    prm.nsub = 1;
    prm.nslot = prm.nseg;
    prm.nhb = (int)((d.H + C::HB - 1) / C::HB);
    char *w = static_cast<char *>(ws);
    prm.cb_ready = reinterpret_cast<unsigned *>(w);
    uint8_t *pack = reinterpret_cast<uint8_t *>(w + flag_bytes(d));
    prm.pack = pack;
    if (selftest_ns > 0) {
        prm.flag_wait_ns = selftest_ns;
        prm.flag_first = 1;
    }
    cudaError_t e = cudaMemsetAsync(w, 0, flag_bytes(d), s);
    timing_begin(s);
    if (e == cudaSuccess && selftest_ns == 0) e = launch_cb<C>(d, B, Cm, pack, prm.cb_ready, status, s);
    if (e == cudaSuccess)
        e = launch_scan<C>(d, prm, ydtype, x, B, Cm, dim3((unsigned)prm.nhb, (unsigned)d.b, (unsigned)dq.nc),
                           "chunk_scan_stage_tc", selftest_ns == 0, s);
    return e;
}

}  // namespace

cudaError_t tc_chunk_state(const Dims &dq, const void *x, const void *dt, const void *B, const float *cum,
                           float *states, unsigned *status, cudaStream_t s) {
    const Dims d = fwd_tiles(dq);
    cudaError_t e = cudaErrorNotSupported;
    dispatch(d, [&](auto c) { e = run_chunk_state<decltype(c)>(dq, d, x, dt, B, cum, states, status, s); });
    return e;
}

size_t tc_chunk_scan_workspace(const Dims &dq) {
    const Dims d = fwd_tiles(dq);
    size_t bytes = 0;
    dispatch(d, [&](auto c) { bytes = scan_stage_workspace<decltype(c)>(d); });
    return bytes;
}

cudaError_t tc_chunk_scan(const Dims &dq, ssd_dtype_t ydtype, const void *x, const void *dt, const void *B,
                          const void *C, const float *cum, const float *states_in, const float *D, void *y,
                          void *ws, unsigned *status, uint64_t selftest_ns, cudaStream_t s) {
    const Dims d = fwd_tiles(dq);
    cudaError_t e = cudaErrorNotSupported;
    dispatch(d, [&](auto c) {
        e = run_chunk_scan<decltype(c)>(dq, d, ydtype, x, dt, B, C, cum, states_in, D, y, ws, status, selftest_ns,
                                        s);
    });
    return e;
}

}  // namespace ssd
