// ssd_api.cu -- the extern "C" entry points of libssd: argument validation
// on the host, then kernel launches on the caller's stream.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "ssd.h"
#include "ssd_common.cuh"
#include "ssd_tc.cuh"

namespace {

using ssd::bf16;
using ssd::Dims;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_in(int64_t v, int64_t lo, int64_t hi) {
    return v >= lo && v <= hi && (v & (v - 1)) == 0;
}

// Shape checks shared by every entry point.  `need_chunks` adds the chunked
// algorithm's restriction Q in {64, 128}; the last chunk may be partial
// (nc = ceil(L / Q)).
ssd_status_t check_shape(const ssd_shape_t *s, bool need_chunks, Dims *d) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads <= 0 || s->headdim <= 0 || s->dstate <= 0 ||
        s->ngroups <= 0)
        return SSD_ERR_INVALID_ARG;
    if (s->dtype != SSD_DTYPE_F32 && s->dtype != SSD_DTYPE_BF16) return SSD_ERR_INVALID_ARG;
    if (s->ydtype != SSD_DTYPE_F32 && s->ydtype != s->dtype) return SSD_ERR_INVALID_ARG;
    if (s->nheads % s->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (!pow2_in(s->headdim, 16, 128) || !pow2_in(s->dstate, 16, 256)) return SSD_ERR_UNSUPPORTED;
    if (need_chunks) {
        if (s->chunk_size <= 0) return SSD_ERR_INVALID_ARG;
        if (s->chunk_size != 64 && s->chunk_size != 128) return SSD_ERR_UNSUPPORTED;
    }
    // every index is formed in int64; keep each grid dimension in range
    if (s->batch > 65535 || s->nheads > 65535) return SSD_ERR_UNSUPPORTED;
    d->b = s->batch;
    d->L = s->seqlen;
    d->H = s->nheads;
    d->P = s->headdim;
    d->N = s->dstate;
    d->G = s->ngroups;
    d->Q = need_chunks ? s->chunk_size : 64;
    d->nc = need_chunks ? (s->seqlen + s->chunk_size - 1) / s->chunk_size : 0;
    d->hpg = (int)(s->nheads / s->ngroups);
    return SSD_OK;
}

bool ptrs_ok(std::initializer_list<const void *> required, std::initializer_list<const void *> optional) {
    for (const void *p : required)
        if (!p || !aligned16(p)) return false;
    for (const void *p : optional)
        if (p && !aligned16(p)) return false;
    return true;
}

// A failed runtime call also records itself as the thread's "last error";
// clear that record so a later, unrelated call does not report it again.
ssd_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return SSD_OK;
    (void)cudaGetLastError();
    return SSD_ERR_CUDA;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// Library-owned device words and buffers (file-scope __device__ symbols).
// Host code holds only a host-side stand-in for such a symbol; the device
// address comes from cudaGetSymbolAddress with the device current, looked up
// once per (device, context): a context destroyed and created again
// (cudaDeviceReset) maps the module anew at another address.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

CUcontext current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            (void)cudaGetLastError();
            return (PFN_cuCtxGetCurrent_v4000) nullptr;
        }
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    CUcontext ctx = nullptr;
    if (fn && fn(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    return ctx;
}

struct SymbolCache {
    std::mutex m;
    CUcontext ctx[kMaxDevices] = {};
    void *ptr[kMaxDevices] = {};
};

template <typename Sym>
cudaError_t symbol_address(const Sym &sym, SymbolCache &cache, void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(cache.m);
    const CUcontext ctx = current_context();
    if (!cache.ptr[dev] || !ctx || ctx != cache.ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, sym);  // (makes the device's context current if none was)
        if (e != cudaSuccess) return e;
        cache.ptr[dev] = p;
        cache.ctx[dev] = current_context();
    }
    *out = cache.ptr[dev];
    return cudaSuccess;
}

// The device status word every kernel of this library latches failures into
// (bit 0: a bounded wait gave up), and the word ssd_get_device_status
// exchanges it into.
static __device__ unsigned g_device_status;
static __device__ unsigned g_device_status_read;
SymbolCache g_status_cache, g_status_read_cache;

cudaError_t device_status_word(unsigned **out) {
    void *p = nullptr;
    const cudaError_t e = symbol_address(g_device_status, g_status_cache, &p);
    *out = static_cast<unsigned *>(p);
    return e;
}

// Atomically take the status word (so no bit latched by a kernel on another
// stream between a read and a clear is lost).
__global__ void take_status_kernel(unsigned *word, unsigned *out) { *out = atomicExch(word, 0u); }

// Workspace of the unfused (four-launch) path: cumsum [b, H, nc, Q] (nc Q
// >= L: a partial last chunk takes a whole chunk's entries), chunk states,
// states entering chunks.
size_t staged_cum_bytes(const Dims &d) { return align256(sizeof(float) * d.b * d.H * d.nc * d.Q); }
size_t staged_workspace(const Dims &d) {
    return staged_cum_bytes(d) + 2 * align256(sizeof(float) * d.b * d.nc * d.H * d.P * d.N);
}

template <typename T, typename TY>
ssd_status_t fwd_staged(const Dims &d, const void *x, const void *dt, const float *A, const void *B,
                        const void *C, const float *D, const float *init, void *y, float *fin, void *ws,
                        cudaStream_t s) {
    char *w = static_cast<char *>(ws);
    float *cum = reinterpret_cast<float *>(w);
    float *states = reinterpret_cast<float *>(w + staged_cum_bytes(d));
    float *states_in = reinterpret_cast<float *>(w + staged_cum_bytes(d) +
                                                 align256(sizeof(float) * d.b * d.nc * d.H * d.P * d.N));
    const T *xt = static_cast<const T *>(x), *dtt = static_cast<const T *>(dt);
    const T *Bt = static_cast<const T *>(B), *Ct = static_cast<const T *>(C);
    ssd::timing_begin(s);
    cudaError_t e = ssd::launch_chunk_cumsum<T>(d, dtt, A, cum, s);
    ssd::timing_mark(s, "chunk_cumsum");
    if (e == cudaSuccess) e = ssd::launch_chunk_state_simt<T>(d, xt, dtt, Bt, cum, states, s);
    ssd::timing_mark(s, "chunk_state_simt");
    if (e == cudaSuccess) e = ssd::launch_state_passing(d, states, cum, init, states_in, fin, s);
    ssd::timing_mark(s, "state_passing");
    if (e == cudaSuccess)
        e = ssd::launch_chunk_scan_simt<T, TY>(d, xt, dtt, Bt, Ct, cum, states_in, D, static_cast<TY *>(y), s);
    ssd::timing_mark(s, "chunk_scan_simt");
    return from_cuda(e);
}

// L == 0: nothing to compute; the final state is the initial state.
ssd_status_t empty_sequence(const Dims &d, const float *init, float *fin, cudaStream_t s) {
    if (!fin || d.b == 0) return SSD_OK;
    const size_t bytes = sizeof(float) * d.b * d.H * d.P * d.N;
    cudaError_t e = init ? cudaMemcpyAsync(fin, init, bytes, cudaMemcpyDeviceToDevice, s)
                         : cudaMemsetAsync(fin, 0, bytes, s);
    return from_cuda(e);
}

// --- launch timing ---------------------------------------------------------
constexpr int kMaxTimed = 16;
struct LaunchTimer {
    bool on = false;
    bool hold = false;  // inside an entry point made of others: their launches append
    int used = 0;
    cudaEvent_t ev[kMaxTimed + 1] = {};
    const char *name[kMaxTimed] = {};
};
LaunchTimer g_timer;

}  // namespace

namespace ssd {
void timing_begin(cudaStream_t s) {
    if (!g_timer.on || (g_timer.hold && g_timer.used > 0)) return;
    g_timer.used = 0;
    if (cudaEventRecord(g_timer.ev[0], s) == cudaSuccess) g_timer.used = 1;
}
void timing_mark(cudaStream_t s, const char *kernel_name) {
    if (!g_timer.on || g_timer.used == 0 || g_timer.used > kMaxTimed) return;
    if (cudaEventRecord(g_timer.ev[g_timer.used], s) == cudaSuccess) {
        g_timer.name[g_timer.used - 1] = kernel_name;
        ++g_timer.used;
    }
}
}  // namespace ssd

extern "C" {

ssd_status_t ssd_launch_timing_enable(int enable) {
    if (enable && !g_timer.on) {
        for (int i = 0; i <= kMaxTimed; ++i)
            if (cudaEventCreate(&g_timer.ev[i]) != cudaSuccess) return SSD_ERR_CUDA;
        g_timer.on = true;
        g_timer.used = 0;
    } else if (!enable && g_timer.on) {
        for (int i = 0; i <= kMaxTimed; ++i) cudaEventDestroy(g_timer.ev[i]);
        g_timer.on = false;
        g_timer.used = 0;
    }
    return SSD_OK;
}

const char *ssd_launch_timing_name(int i) {
    if (!g_timer.on || i < 0 || i >= g_timer.used - 1) return nullptr;
    return g_timer.name[i];
}

int ssd_launch_timing_read(float *ms, int cap) {
    if (!g_timer.on || g_timer.used < 2) return -1;
    const int n = g_timer.used - 1;
    if (cudaEventSynchronize(g_timer.ev[n]) != cudaSuccess) return -1;
    for (int i = 0; i < n && i < cap; ++i)
        if (cudaEventElapsedTime(&ms[i], g_timer.ev[i], g_timer.ev[i + 1]) != cudaSuccess) return -1;
    return n;
}

const char *ssd_status_string(ssd_status_t st) {
    switch (st) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: null or misaligned pointer, or invalid shape";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: shape outside what the GPU kernels run";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA: a CUDA launch failed";
        case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace missing or too small";
        case SSD_ERR_SCRATCH_LIMIT:
            return "SSD_ERR_SCRATCH_LIMIT: shape needs more scratch than ssd_fwd_noalloc's static buffer holds";
        case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: a bounded wait inside a kernel gave up (outputs incomplete)";
    }
    return "SSD_ERR_UNKNOWN";
}

int ssd_abi_version(void) { return (2 << 16) | 0; }

size_t ssd_fwd_workspace_size(const ssd_shape_t *shape) {
    Dims d;
    if (check_shape(shape, true, &d) != SSD_OK) return 0;
    if (ssd::tc_fwd_supported(d, shape->dtype)) return ssd::tc_fwd_workspace(d);
    return staged_workspace(d);
}

ssd_status_t ssd_fwd(const ssd_shape_t *shape, const void *x, const void *dt, const float *A, const void *B,
                     const void *C, const float *D, const float *init_state, void *y, float *final_state,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, true, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0) return SSD_OK;
    if (d.L == 0) {
        if (!ptrs_ok({A}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
        return empty_sequence(d, init_state, final_state, stream);
    }
    if (!ptrs_ok({x, dt, A, B, C, y}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
    const bool tc = ssd::tc_fwd_supported(d, shape->dtype);
    const size_t need = tc ? ssd::tc_fwd_workspace(d) : staged_workspace(d);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return SSD_ERR_WORKSPACE;
    if (tc) {
        unsigned *status = nullptr;
        const cudaError_t e = device_status_word(&status);
        if (e != cudaSuccess) return from_cuda(e);
        return from_cuda(
            ssd::tc_fwd(d, shape->ydtype, x, dt, A, B, C, D, init_state, y, final_state, workspace, status, stream));
    }
    if (shape->dtype == SSD_DTYPE_F32)
        return fwd_staged<float, float>(d, x, dt, A, B, C, D, init_state, y, final_state, workspace, stream);
    if (shape->ydtype == SSD_DTYPE_F32)
        return fwd_staged<bf16, float>(d, x, dt, A, B, C, D, init_state, y, final_state, workspace, stream);
    return fwd_staged<bf16, bf16>(d, x, dt, A, B, C, D, init_state, y, final_state, workspace, stream);
}

}  // extern "C"

namespace {
// Validates a packed variable-length batch; on success the sub-shape of
// every sequence is `one` with its seqlen replaced.
ssd_status_t check_varlen(const ssd_shape_t *shape, const int64_t *cu, int64_t nseq, ssd_shape_t *one) {
    Dims d;
    ssd_status_t st = check_shape(shape, true, &d);
    if (st != SSD_OK) return st;
    if (shape->batch != 1 || nseq < 0 || (nseq > 0 && !cu)) return SSD_ERR_INVALID_ARG;
    if (nseq > 0 && (cu[0] != 0 || cu[nseq] != shape->seqlen)) return SSD_ERR_INVALID_ARG;
    for (int64_t s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return SSD_ERR_INVALID_ARG;
    *one = *shape;
    return SSD_OK;
}

// How a packed batch runs on the tensor-core path: the `nfwd` longest
// sequences one fused forward each (their segments fill the SMs), the rest
// in launch sets of up to kVarlenMaxUnits sequences (a unit per sequence and
// head block), whichever split the cost model rates fastest.  `order` holds
// the non-empty sequences, longest first.
struct VarlenPlan {
    bool tc = false;
    std::vector<ssd::VarlenSeq> order;
    size_t nfwd = 0;
};

constexpr size_t kMaxSeparate = 8;  // longest sequences considered for a fused forward of their own

VarlenPlan plan_varlen(const ssd_shape_t *shape, const int64_t *cu, int64_t nseq) {
    VarlenPlan p;
    Dims d;
    if (check_shape(shape, true, &d) != SSD_OK || !ssd::tc_varlen_supported(d, shape->dtype)) return p;
    p.tc = true;
    for (int64_t s = 0; s < nseq; ++s)
        if (cu[s + 1] > cu[s]) p.order.push_back({(int)cu[s], (int)(cu[s + 1] - cu[s]), (int)s});
    std::stable_sort(p.order.begin(), p.order.end(),
                     [](const ssd::VarlenSeq &a, const ssd::VarlenSeq &b) { return a.len > b.len; });
    const size_t m = p.order.size();
    auto sets_cost = [&](size_t from) {
        double us = 0;
        for (size_t i = from; i < m; i += ssd::kVarlenSetSeqs)
            us += ssd::tc_varlen_cost_us(d, p.order.data() + i,
                                         (int)std::min<size_t>(ssd::kVarlenSetSeqs, m - i));
        return us;
    };
    double best = sets_cost(0), sep = 0;
    for (size_t k = 1; k <= std::min(m, kMaxSeparate); ++k) {
        sep += ssd::tc_fwd_cost_us(d, p.order[k - 1].len);
        if (sep >= best) break;  // (the separate forwards alone already cost more)
        const double us = sep + sets_cost(k);
        if (us < best) {
            best = us;
            p.nfwd = k;
        }
    }
    return p;
}
// Workspace bytes of a plan: the largest of its fused forwards and sets.
size_t varlen_workspace(const ssd_shape_t *shape, const int64_t *cu, int64_t nseq, const VarlenPlan &p) {
    ssd_shape_t one = *shape;
    size_t need = 0;
    if (p.tc) {
        Dims d;
        (void)check_shape(shape, true, &d);
        for (size_t i = 0; i < p.order.size(); ++i) {
            if (i < p.nfwd) {
                one.seqlen = p.order[i].len;
                need = std::max(need, ssd_fwd_workspace_size(&one));
            } else {
                const int n = (int)std::min<size_t>(ssd::kVarlenSetSeqs, p.order.size() - i);
                need = std::max(need, ssd::tc_varlen_workspace(d, p.order.data() + i, n));
                i += n - 1;
            }
        }
        return need;
    }
    for (int64_t s = 0; s < nseq; ++s) {
        one.seqlen = cu[s + 1] - cu[s];
        if (one.seqlen == 0) continue;
        need = std::max(need, ssd_fwd_workspace_size(&one));
    }
    return need;
}
}  // namespace

extern "C" {

size_t ssd_fwd_varlen_workspace_size(const ssd_shape_t *shape, const int64_t *cu_seqlens, int64_t nseq) {
    ssd_shape_t one;
    if (check_varlen(shape, cu_seqlens, nseq, &one) != SSD_OK) return 0;
    return varlen_workspace(shape, cu_seqlens, nseq, plan_varlen(shape, cu_seqlens, nseq));
}

ssd_status_t ssd_fwd_varlen(const ssd_shape_t *shape, const int64_t *cu_seqlens, int64_t nseq, const void *x,
                            const void *dt, const float *A, const void *B, const void *C, const float *D,
                            const float *init_states, void *y, float *final_states, void *workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
    ssd_shape_t one;
    ssd_status_t st = check_varlen(shape, cu_seqlens, nseq, &one);
    if (st != SSD_OK) return st;
    if (nseq == 0) return SSD_OK;
    if (!ptrs_ok({x, dt, A, B, C, y}, {D, init_states, final_states})) return SSD_ERR_INVALID_ARG;
    const size_t e = shape->dtype == SSD_DTYPE_F32 ? 4 : 2;
    const size_t ye = shape->ydtype == SSD_DTYPE_F32 ? 4 : 2;
    const int64_t H = shape->nheads, P = shape->headdim, N = shape->dstate, G = shape->ngroups;
    // every sequence's pointers are checked before anything is enqueued
    for (int64_t s = 0; s < nseq; ++s) {
        const int64_t t0 = cu_seqlens[s];
        if (cu_seqlens[s + 1] == t0) continue;
        const char *px = static_cast<const char *>(x) + t0 * H * P * e;
        const char *pdt = static_cast<const char *>(dt) + t0 * H * e;
        const char *pb = static_cast<const char *>(B) + t0 * G * N * e;
        const char *py = static_cast<const char *>(y) + t0 * H * P * ye;
        if (!ptrs_ok({px, pdt, pb, py}, {})) return SSD_ERR_INVALID_ARG;
    }
    const VarlenPlan p = plan_varlen(shape, cu_seqlens, nseq);
    if (varlen_workspace(shape, cu_seqlens, nseq, p) > workspace_bytes) return SSD_ERR_WORKSPACE;
    // one sequence's own fused forward
    auto own = [&](int64_t s) {
        const int64_t t0 = cu_seqlens[s];
        one.seqlen = cu_seqlens[s + 1] - t0;
        const float *ini = init_states ? init_states + s * H * P * N : nullptr;
        float *fin = final_states ? final_states + s * H * P * N : nullptr;
        return ssd_fwd(&one, static_cast<const char *>(x) + t0 * H * P * e,
                       static_cast<const char *>(dt) + t0 * H * e, A, static_cast<const char *>(B) + t0 * G * N * e,
                       static_cast<const char *>(C) + t0 * G * N * e, D, ini,
                       static_cast<char *>(y) + t0 * H * P * ye, fin, workspace, workspace_bytes, stream);
    };
    if (!p.tc) {
        for (int64_t s = 0; s < nseq; ++s)
            if ((st = own(s)) != SSD_OK) return st;
        return SSD_OK;
    }
    Dims d;
    (void)check_shape(shape, true, &d);
    // the launch list of this call holds every launch it makes
    ssd::timing_begin(stream);
    g_timer.hold = true;
    struct Release {
        ~Release() { g_timer.hold = false; }
    } release;
    // empty sequences: the final state is the initial one
    for (int64_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] == cu_seqlens[s]) {
            Dims d1 = d;
            d1.b = 1;
            st = empty_sequence(d1, init_states ? init_states + s * H * P * N : nullptr,
                                final_states ? final_states + s * H * P * N : nullptr, stream);
            if (st != SSD_OK) return st;
        }
    for (size_t i = 0; i < p.nfwd; ++i)
        if ((st = own(p.order[i].seq)) != SSD_OK) return st;
    unsigned *status = nullptr;
    if (p.nfwd < p.order.size()) {
        const cudaError_t ce = device_status_word(&status);
        if (ce != cudaSuccess) return from_cuda(ce);
    }
    for (size_t i = p.nfwd; i < p.order.size(); i += ssd::kVarlenSetSeqs) {
        const int n = (int)std::min<size_t>(ssd::kVarlenSetSeqs, p.order.size() - i);
        st = from_cuda(ssd::tc_fwd_varlen(d, p.order.data() + i, n, shape->ydtype, x, dt, A, B, C, D, init_states,
                                          y, final_states, workspace, status, stream));
        if (st != SSD_OK) return st;
    }
    return SSD_OK;
}

ssd_status_t ssd_chunk_cumsum(const ssd_shape_t *shape, const void *dt, const float *A, float *dA_cumsum,
                              cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, true, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0 || d.L == 0) return SSD_OK;
    if (!ptrs_ok({dt, A, dA_cumsum}, {})) return SSD_ERR_INVALID_ARG;
    ssd::timing_begin(stream);
    const cudaError_t e =
        shape->dtype == SSD_DTYPE_F32
            ? ssd::launch_chunk_cumsum<float>(d, static_cast<const float *>(dt), A, dA_cumsum, stream)
            : ssd::launch_chunk_cumsum<bf16>(d, static_cast<const bf16 *>(dt), A, dA_cumsum, stream);
    ssd::timing_mark(stream, "chunk_cumsum");
    return from_cuda(e);
}

ssd_status_t ssd_chunk_state(const ssd_shape_t *shape, const void *x, const void *dt, const void *B,
                             const float *dA_cumsum, float *states, cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, true, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0 || d.L == 0) return SSD_OK;
    if (!ptrs_ok({x, dt, B, dA_cumsum, states}, {})) return SSD_ERR_INVALID_ARG;
    if (ssd::tc_stage_supported(d, shape->dtype)) {
        unsigned *status = nullptr;
        const cudaError_t e = device_status_word(&status);
        if (e != cudaSuccess) return from_cuda(e);
        return from_cuda(ssd::tc_chunk_state(d, x, dt, B, dA_cumsum, states, status, stream));
    }
    if (shape->dtype == SSD_DTYPE_F32)
        return from_cuda(ssd::launch_chunk_state_simt<float>(d, static_cast<const float *>(x),
                                                             static_cast<const float *>(dt),
                                                             static_cast<const float *>(B), dA_cumsum, states,
                                                             stream));
    return from_cuda(ssd::launch_chunk_state_simt<bf16>(d, static_cast<const bf16 *>(x),
                                                        static_cast<const bf16 *>(dt),
                                                        static_cast<const bf16 *>(B), dA_cumsum, states, stream));
}

ssd_status_t ssd_state_passing(const ssd_shape_t *shape, const float *states, const float *dA_cumsum,
                               const float *init_state, float *states_in, float *final_state,
                               cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, true, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0) return SSD_OK;
    if (d.L == 0) {
        if (!ptrs_ok({}, {init_state, final_state})) return SSD_ERR_INVALID_ARG;
        return empty_sequence(d, init_state, final_state, stream);
    }
    if (!ptrs_ok({states, dA_cumsum}, {init_state, states_in, final_state})) return SSD_ERR_INVALID_ARG;
    ssd::timing_begin(stream);
    const cudaError_t e = ssd::launch_state_passing(d, states, dA_cumsum, init_state, states_in, final_state, stream);
    ssd::timing_mark(stream, "state_passing");
    return from_cuda(e);
}

size_t ssd_chunk_scan_workspace_size(const ssd_shape_t *shape) {
    Dims d;
    if (check_shape(shape, true, &d) != SSD_OK) return 0;
    if (ssd::tc_stage_supported(d, shape->dtype)) return ssd::tc_chunk_scan_workspace(d);
    return 0;
}

}  // extern "C"

namespace {
// The chunk-scan stage, or (selftest_ns > 0) its failure-path self-test.
ssd_status_t chunk_scan_call(const ssd_shape_t *shape, const void *x, const void *dt, const void *B, const void *C,
                             const float *dA_cumsum, const float *states_in, const float *D, void *y,
                             void *workspace, size_t workspace_bytes, uint64_t selftest_ns, cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, true, &d);
    if (st != SSD_OK) return st;
    const bool tc = ssd::tc_stage_supported(d, shape->dtype);
    if (selftest_ns > 0 && !tc) return SSD_ERR_UNSUPPORTED;
    if (d.b == 0 || d.L == 0) return SSD_OK;
    if (!ptrs_ok({x, dt, B, C, dA_cumsum, states_in, y}, {D})) return SSD_ERR_INVALID_ARG;
    if (tc) {
        const size_t need = ssd::tc_chunk_scan_workspace(d);
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return SSD_ERR_WORKSPACE;
        unsigned *status = nullptr;
        const cudaError_t e = device_status_word(&status);
        if (e != cudaSuccess) return from_cuda(e);
        return from_cuda(ssd::tc_chunk_scan(d, shape->ydtype, x, dt, B, C, dA_cumsum, states_in, D, y, workspace,
                                            status, selftest_ns, stream));
    }
    if (shape->dtype == SSD_DTYPE_F32)
        return from_cuda(ssd::launch_chunk_scan_simt<float, float>(
            d, static_cast<const float *>(x), static_cast<const float *>(dt), static_cast<const float *>(B),
            static_cast<const float *>(C), dA_cumsum, states_in, D, static_cast<float *>(y), stream));
    const bf16 *xb = static_cast<const bf16 *>(x), *dtb = static_cast<const bf16 *>(dt);
    const bf16 *Bb = static_cast<const bf16 *>(B), *Cb = static_cast<const bf16 *>(C);
    if (shape->ydtype == SSD_DTYPE_F32)
        return from_cuda(ssd::launch_chunk_scan_simt<bf16, float>(d, xb, dtb, Bb, Cb, dA_cumsum, states_in, D,
                                                                  static_cast<float *>(y), stream));
    return from_cuda(ssd::launch_chunk_scan_simt<bf16, bf16>(d, xb, dtb, Bb, Cb, dA_cumsum, states_in, D,
                                                             static_cast<bf16 *>(y), stream));
}
}  // namespace

extern "C" {

ssd_status_t ssd_chunk_scan(const ssd_shape_t *shape, const void *x, const void *dt, const void *B, const void *C,
                            const float *dA_cumsum, const float *states_in, const float *D, void *y,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return chunk_scan_call(shape, x, dt, B, C, dA_cumsum, states_in, D, y, workspace, workspace_bytes, 0, stream);
}

ssd_status_t ssd_selftest_scan_timeout(const ssd_shape_t *shape, const void *x, const void *dt, const void *B,
                                       const void *C, const float *dA_cumsum, const float *states_in,
                                       const float *D, void *y, void *workspace, size_t workspace_bytes,
                                       uint64_t wait_ns, cudaStream_t stream) {
    if (wait_ns < 100000ull) wait_ns = 100000ull;
    if (wait_ns > 1000000000ull) wait_ns = 1000000000ull;
    return chunk_scan_call(shape, x, dt, B, C, dA_cumsum, states_in, D, y, workspace, workspace_bytes, wait_ns,
                           stream);
}

ssd_status_t ssd_get_device_status(cudaStream_t stream) {
    unsigned *word = nullptr, *taken = nullptr;
    cudaError_t e = device_status_word(&word);
    if (e == cudaSuccess) {
        void *p = nullptr;
        e = symbol_address(g_device_status_read, g_status_read_cache, &p);
        taken = static_cast<unsigned *>(p);
    }
    if (e != cudaSuccess) return from_cuda(e);
    take_status_kernel<<<1, 1, 0, stream>>>(word, taken);
    e = cudaGetLastError();
    unsigned v = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&v, taken, sizeof(v), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return from_cuda(e);
    return (v & 1u) ? SSD_ERR_TIMEOUT : SSD_OK;
}

ssd_status_t ssd_fwd_quadratic(const ssd_shape_t *shape, const void *x, const void *dt, const float *A, const void *B,
                               const void *C, const float *D, const float *init_state, void *y, float *final_state,
                               cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, false, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0) return SSD_OK;
    if (d.L == 0) {
        if (!ptrs_ok({A}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
        return empty_sequence(d, init_state, final_state, stream);
    }
    if (!ssd::quad_supported(d, shape->dtype)) return SSD_ERR_UNSUPPORTED;
    if (!ptrs_ok({x, dt, A, B, C, y}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
    unsigned *status = nullptr;
    const cudaError_t e = device_status_word(&status);
    if (e != cudaSuccess) return from_cuda(e);
    ssd::timing_begin(stream);
    return from_cuda(
        ssd::quad_fwd(d, shape->ydtype, x, dt, A, B, C, D, init_state, y, final_state, status, stream));
}

ssd_status_t ssd_decode_step(const ssd_shape_t *shape, const void *x, const void *dt, const float *A, const void *B,
                             const void *C, const float *D, float *state, void *y, cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, false, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0) return SSD_OK;
    if (!ptrs_ok({x, dt, A, B, C, state, y}, {D})) return SSD_ERR_INVALID_ARG;
    ssd::timing_begin(stream);
    if (shape->dtype == SSD_DTYPE_F32)
        return from_cuda(ssd::launch_decode_step<float, float>(
            d, static_cast<const float *>(x), static_cast<const float *>(dt), A, static_cast<const float *>(B),
            static_cast<const float *>(C), D, state, static_cast<float *>(y), stream));
    const bf16 *xb = static_cast<const bf16 *>(x), *dtb = static_cast<const bf16 *>(dt);
    const bf16 *Bb = static_cast<const bf16 *>(B), *Cb = static_cast<const bf16 *>(C);
    if (shape->ydtype == SSD_DTYPE_F32)
        return from_cuda(
            ssd::launch_decode_step<bf16, float>(d, xb, dtb, A, Bb, Cb, D, state, static_cast<float *>(y), stream));
    return from_cuda(
        ssd::launch_decode_step<bf16, bf16>(d, xb, dtb, A, Bb, Cb, D, state, static_cast<bf16 *>(y), stream));
}

ssd_status_t selective_scan_fwd(const ssd_shape_t *shape, const void *x, const void *dt, const float *A,
                                const void *B, const void *C, const float *D, const float *init_state, void *y,
                                float *final_state, cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, false, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0) return SSD_OK;
    if (d.L == 0) {
        if (!ptrs_ok({A}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
        return empty_sequence(d, init_state, final_state, stream);
    }
    if (!ptrs_ok({x, dt, A, B, C, y}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
    if (shape->dtype == SSD_DTYPE_F32)
        return from_cuda(ssd::launch_selective_scan<float, float>(
            d, static_cast<const float *>(x), static_cast<const float *>(dt), A, static_cast<const float *>(B),
            static_cast<const float *>(C), D, init_state, static_cast<float *>(y), final_state, stream));
    const bf16 *xb = static_cast<const bf16 *>(x), *dtb = static_cast<const bf16 *>(dt);
    const bf16 *Bb = static_cast<const bf16 *>(B), *Cb = static_cast<const bf16 *>(C);
    if (shape->ydtype == SSD_DTYPE_F32)
        return from_cuda(ssd::launch_selective_scan<bf16, float>(d, xb, dtb, A, Bb, Cb, D, init_state,
                                                                 static_cast<float *>(y), final_state, stream));
    return from_cuda(ssd::launch_selective_scan<bf16, bf16>(d, xb, dtb, A, Bb, Cb, D, init_state,
                                                            static_cast<bf16 *>(y), final_state, stream));
}

// ---------------------------------------------------------------------------
// ssd_fwd_noalloc: ssd_fwd with scratch from a static device buffer.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

// The scratch every ssd_fwd_noalloc call uses; one copy per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

SymbolCache g_scratch_cache;

// Device address of the static scratch on the current device (host code only
// sees a host-side stand-in for the symbol), looked up once per device and
// context.
cudaError_t noalloc_scratch(void **out) { return symbol_address(g_noalloc_scratch, g_scratch_cache, out); }

}  // namespace

extern "C" ssd_status_t ssd_fwd_noalloc(const ssd_shape_t *shape, const void *x, const void *dt, const float *A,
                                        const void *B, const void *C, const float *D, const float *init_state,
                                        void *y, float *final_state, cudaStream_t stream) {
    Dims d;
    ssd_status_t st = check_shape(shape, true, &d);
    if (st != SSD_OK) return st;
    if (d.b == 0) return SSD_OK;
    if (d.L == 0) {
        if (!ptrs_ok({A}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
        return empty_sequence(d, init_state, final_state, stream);
    }
    if (!ptrs_ok({x, dt, A, B, C, y}, {D, init_state, final_state})) return SSD_ERR_INVALID_ARG;
    const bool tc = ssd::tc_fwd_supported(d, shape->dtype);
    const size_t need = tc ? ssd::tc_fwd_workspace(d) : staged_workspace(d);
    if (need > SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return from_cuda(e);
    // the kernels write every scratch word they later read, except the
    // chunk-pack ready flags, which the fused path clears on the stream
    // before use
    if (tc) {
        unsigned *status = nullptr;
        e = device_status_word(&status);
        if (e != cudaSuccess) return from_cuda(e);
        return from_cuda(
            ssd::tc_fwd(d, shape->ydtype, x, dt, A, B, C, D, init_state, y, final_state, scratch, status, stream));
    }
    if (shape->dtype == SSD_DTYPE_F32)
        return fwd_staged<float, float>(d, x, dt, A, B, C, D, init_state, y, final_state, scratch, stream);
    if (shape->ydtype == SSD_DTYPE_F32)
        return fwd_staged<bf16, float>(d, x, dt, A, B, C, D, init_state, y, final_state, scratch, stream);
    return fwd_staged<bf16, bf16>(d, x, dt, A, B, C, D, init_state, y, final_state, scratch, stream);
}
