"""GB300-native Mamba-2 SSD chunked forward pass -- Python binding of libssd.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libssd.so`` behind the C ABI declared in ``include/ssd.h``.
PyTorch supplies device memory and the current CUDA stream.  There is no CPU
or PyTorch fallback: if the library has not been built, every call raises.

Tensor layouts (contiguous):
    x [b, L, H, P], dt [b, L, H], A [H] fp32, B/C [b, L, G, N], D [H] fp32,
    init_state / final_state [b, H, P, N] fp32, y [b, L, H, P],
    dA_cumsum [b, H, nc, Q] fp32, states / states_in [b, nc, H, P, N] fp32.
x, dt, B, C (and y) share one dtype: torch.float32 or torch.bfloat16.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libssd.so")

SSD_OK = 0
SSD_ERR_TIMEOUT = 6
SSD_DTYPE_F32 = 0
SSD_DTYPE_BF16 = 1

EXPORTED = ("ssd_status_string", "ssd_abi_version", "ssd_fwd_workspace_size", "ssd_fwd",
            "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan",
            "selective_scan_fwd", "ssd_launch_timing_enable", "ssd_launch_timing_read",
            "ssd_launch_timing_name", "ssd_fwd_noalloc", "ssd_chunk_scan_workspace_size",
            "ssd_get_device_status", "ssd_selftest_scan_timeout", "ssd_decode_step",
            "ssd_fwd_varlen_workspace_size", "ssd_fwd_varlen", "ssd_fwd_quadratic")


class ssd_shape_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("dtype", ctypes.c_int), ("ydtype", ctypes.c_int)]


class SSDError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libssd.so and declare its signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libssd.so is not built ({path}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        shp = ctypes.POINTER(ssd_shape_t)
        lib.ssd_status_string.argtypes = [i32]
        lib.ssd_status_string.restype = ctypes.c_char_p
        lib.ssd_abi_version.restype = i32
        lib.ssd_fwd_workspace_size.argtypes = [shp]
        lib.ssd_fwd_workspace_size.restype = sz
        lib.ssd_fwd.argtypes = [shp] + [vp] * 10 + [sz, vp]
        lib.ssd_chunk_cumsum.argtypes = [shp, vp, vp, vp, vp]
        lib.ssd_chunk_state.argtypes = [shp, vp, vp, vp, vp, vp, vp]
        lib.ssd_state_passing.argtypes = [shp, vp, vp, vp, vp, vp, vp]
        lib.ssd_chunk_scan.argtypes = [shp] + [vp] * 9 + [sz, vp]
        lib.ssd_chunk_scan_workspace_size.argtypes = [shp]
        lib.ssd_chunk_scan_workspace_size.restype = sz
        lib.ssd_selftest_scan_timeout.argtypes = [shp] + [vp] * 9 + [sz, ctypes.c_uint64, vp]
        lib.ssd_get_device_status.argtypes = [vp]
        lib.ssd_decode_step.argtypes = [shp] + [vp] * 9
        lib.ssd_fwd_quadratic.argtypes = [shp] + [vp] * 10
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.ssd_fwd_varlen_workspace_size.argtypes = [shp, i64p, ctypes.c_int64]
        lib.ssd_fwd_varlen_workspace_size.restype = sz
        lib.ssd_fwd_varlen.argtypes = [shp, i64p, ctypes.c_int64] + [vp] * 10 + [sz, vp]
        lib.selective_scan_fwd.argtypes = [shp] + [vp] * 9 + [vp]
        lib.ssd_launch_timing_enable.argtypes = [i32]
        lib.ssd_launch_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float), i32]
        lib.ssd_launch_timing_name.argtypes = [i32]
        lib.ssd_launch_timing_name.restype = ctypes.c_char_p
        lib.ssd_fwd_noalloc.argtypes = [shp] + [vp] * 10
        lib.ssd_fwd_noalloc.restype = i32
        for name in ("ssd_fwd", "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan",
                     "selective_scan_fwd", "ssd_launch_timing_enable", "ssd_launch_timing_read",
                     "ssd_fwd_noalloc", "ssd_get_device_status", "ssd_selftest_scan_timeout", "ssd_decode_step",
                     "ssd_fwd_varlen", "ssd_fwd_quadratic"):
            getattr(lib, name).restype = i32
        if path == LIB_PATH:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().ssd_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != SSD_OK:
        raise SSDError(fn, status, status_string(status))


def get_device_status(stream=None) -> int:
    """Wait for the stream, then read and clear the current device's status
    word: SSD_OK, or SSD_ERR_TIMEOUT when a bounded wait inside any of this
    library's kernels gave up since the previous read (the outputs of that
    call are incomplete)."""
    return int(load_library().ssd_get_device_status(_stream(stream)))


def check_device_status(stream=None) -> None:
    """get_device_status(), raising SSDError unless it is SSD_OK."""
    _check("ssd_get_device_status", get_device_status(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSD_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return SSD_DTYPE_BF16
    raise TypeError(f"x must be float32 or bfloat16, got {t.dtype}")


def _need(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def make_shape(x: torch.Tensor, B: torch.Tensor, chunk_size: int, y_dtype=torch.float32) -> ssd_shape_t:
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    yc = SSD_DTYPE_F32 if y_dtype == torch.float32 else _dtype_code(torch.empty(0, dtype=y_dtype))
    return ssd_shape_t(b, L, H, P, N, G, int(chunk_size), _dtype_code(x), yc)


def _check_inputs(x, dt, A, B, C, D, init_state):
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [b, L, H, P] and B, C [b, L, G, N]")
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    _need(x, "x")
    _need(dt, "dt", x.dtype, (b, L, H))
    _need(A, "A", torch.float32, (H,))
    _need(B, "B", x.dtype, (b, L, G, N))
    _need(C, "C", x.dtype, (b, L, G, N))
    _need(D, "D", torch.float32, (H,))
    _need(init_state, "init_state", torch.float32, (b, H, P, N))
    return b, L, H, P, G, N


def ssd_fwd_workspace_size(shape: ssd_shape_t) -> int:
    return int(load_library().ssd_fwd_workspace_size(ctypes.byref(shape)))


def ssd_fwd(x, dt, A, B, C, D=None, init_state=None, chunk_size=64, *, y=None, final_state=None,
            workspace=None, return_final_state=True, y_dtype=torch.float32, stream=None):
    """Fused SSD forward.  Returns ``(y, final_state)`` (final_state None when
    ``return_final_state`` is False and no buffer was given).  ``y_dtype``
    is float32 (default) or the input dtype."""
    lib = load_library()
    b, L, H, P, G, N = _check_inputs(x, dt, A, B, C, D, init_state)
    if y is not None:
        y_dtype = y.dtype
    shape = make_shape(x, B, chunk_size, y_dtype)
    if y is None:
        y = torch.empty(x.shape, device=x.device, dtype=y_dtype)
    _need(y, "y", y_dtype, x.shape)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), device=x.device, dtype=torch.float32)
    _need(final_state, "final_state", torch.float32, (b, H, P, N))
    ws_bytes = int(lib.ssd_fwd_workspace_size(ctypes.byref(shape)))
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 16), device=x.device, dtype=torch.uint8)
    st = lib.ssd_fwd(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                     _ptr(init_state), _ptr(y), _ptr(final_state), _ptr(workspace),
                     workspace.numel(), _stream(stream))
    _check("ssd_fwd", st)
    return y, final_state


def ssd_fwd_noalloc(x, dt, A, B, C, D=None, init_state=None, chunk_size=64, *, y, final_state=None,
                    stream=None):
    """ssd_fwd for callers that cannot allocate device memory: the library
    takes its scratch from a static device buffer (SSD_NOALLOC_SCRATCH_BYTES)
    and this wrapper allocates nothing either -- the caller passes y (and
    final_state, if wanted).  Calls whose GPU work overlaps share that buffer
    and race; serialise them.  Returns ``(y, final_state)``."""
    lib = load_library()
    b, L, H, P, G, N = _check_inputs(x, dt, A, B, C, D, init_state)
    _need(y, "y", None, x.shape)
    _need(final_state, "final_state", torch.float32, (b, H, P, N))
    shape = make_shape(x, B, chunk_size, y.dtype)
    st = lib.ssd_fwd_noalloc(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                             _ptr(init_state), _ptr(y), _ptr(final_state), _stream(stream))
    _check("ssd_fwd_noalloc", st)
    return y, final_state


def ssd_chunk_cumsum(dt, A, chunk_size, *, out=None, stream=None):
    lib = load_library()
    b, L, H = dt.shape
    _need(dt, "dt")
    _need(A, "A", torch.float32, (H,))
    Q = int(chunk_size)
    nc = -(-L // Q) if Q > 0 else 0
    if out is None:
        out = torch.empty((b, H, nc, Q), device=dt.device, dtype=torch.float32)
    _need(out, "dA_cumsum", torch.float32, (b, H, nc, Q))
    # the shape fields that do not concern this stage are set to valid values
    shape = ssd_shape_t(b, L, H, 16, 16, 1, Q, _dtype_code(dt), SSD_DTYPE_F32)
    _check("ssd_chunk_cumsum", lib.ssd_chunk_cumsum(ctypes.byref(shape), _ptr(dt), _ptr(A), _ptr(out),
                                                    _stream(stream)))
    return out


def ssd_chunk_state(x, dt, B, dA_cumsum, *, out=None, stream=None):
    lib = load_library()
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Q = dA_cumsum.shape[-1]
    nc = dA_cumsum.shape[2]
    _need(x, "x")
    _need(dt, "dt", x.dtype, (b, L, H))
    _need(B, "B", x.dtype, (b, L, G, N))
    _need(dA_cumsum, "dA_cumsum", torch.float32, (b, H, nc, Q))
    if out is None:
        out = torch.empty((b, nc, H, P, N), device=x.device, dtype=torch.float32)
    _need(out, "states", torch.float32, (b, nc, H, P, N))
    shape = make_shape(x, B, Q)
    _check("ssd_chunk_state", lib.ssd_chunk_state(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(B),
                                                  _ptr(dA_cumsum), _ptr(out), _stream(stream)))
    return out


def ssd_state_passing(states, dA_cumsum, init_state=None, *, out=None, final_state=None,
                      return_final_state=True, stream=None):
    lib = load_library()
    b, nc, H, P, N = states.shape
    Q = dA_cumsum.shape[-1]
    _need(states, "states", torch.float32)
    _need(dA_cumsum, "dA_cumsum", torch.float32, (b, H, nc, Q))
    _need(init_state, "init_state", torch.float32, (b, H, P, N))
    if out is None:
        out = torch.empty_like(states)
    _need(out, "states_in", torch.float32, states.shape)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), device=states.device, dtype=torch.float32)
    _need(final_state, "final_state", torch.float32, (b, H, P, N))
    shape = ssd_shape_t(b, nc * Q, H, P, N, 1, Q, SSD_DTYPE_F32, SSD_DTYPE_F32)
    _check("ssd_state_passing", lib.ssd_state_passing(ctypes.byref(shape), _ptr(states), _ptr(dA_cumsum),
                                                      _ptr(init_state), _ptr(out), _ptr(final_state),
                                                      _stream(stream)))
    return out, final_state


def ssd_chunk_scan(x, dt, B, C, dA_cumsum, states_in, D=None, *, out=None, y_dtype=torch.float32,
                   workspace=None, stream=None):
    lib = load_library()
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Q = dA_cumsum.shape[-1]
    nc = dA_cumsum.shape[2]
    _need(x, "x")
    _need(dt, "dt", x.dtype, (b, L, H))
    _need(B, "B", x.dtype, (b, L, G, N))
    _need(C, "C", x.dtype, (b, L, G, N))
    _need(dA_cumsum, "dA_cumsum", torch.float32, (b, H, nc, Q))
    _need(states_in, "states_in", torch.float32, (b, nc, H, P, N))
    _need(D, "D", torch.float32, (H,))
    if out is not None:
        y_dtype = out.dtype
    if out is None:
        out = torch.empty(x.shape, device=x.device, dtype=y_dtype)
    _need(out, "y", y_dtype, x.shape)
    shape = make_shape(x, B, Q, y_dtype)
    ws_bytes = int(lib.ssd_chunk_scan_workspace_size(ctypes.byref(shape)))
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, device=x.device, dtype=torch.uint8)
    _check("ssd_chunk_scan", lib.ssd_chunk_scan(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(B), _ptr(C),
                                                _ptr(dA_cumsum), _ptr(states_in), _ptr(D), _ptr(out),
                                                _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                                _stream(stream)))
    return out


def selftest_scan_timeout(x, dt, B, C, dA_cumsum, states_in, D=None, *, out, wait_ns=2_000_000,
                          stream=None) -> int:
    """Failure-path self-test: the chunk-scan stage kernel alone with no
    operand pack ever published, so its bounded wait gives up after
    ``wait_ns``; returns the status of the enqueue (read the device status
    with get_device_status afterwards)."""
    lib = load_library()
    Q = dA_cumsum.shape[-1]
    shape = make_shape(x, B, Q, out.dtype)
    ws_bytes = int(lib.ssd_chunk_scan_workspace_size(ctypes.byref(shape)))
    workspace = torch.empty(max(ws_bytes, 16), device=x.device, dtype=torch.uint8)
    return int(lib.ssd_selftest_scan_timeout(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(B), _ptr(C),
                                             _ptr(dA_cumsum), _ptr(states_in), _ptr(D), _ptr(out),
                                             _ptr(workspace), workspace.numel(), int(wait_ns), _stream(stream)))


def selective_scan_fwd(x, dt, A, B, C, D=None, init_state=None, *, y=None, final_state=None,
                       return_final_state=True, y_dtype=torch.float32, stream=None):
    """The recurrence as a sequential scan on the fp32 ALUs (no chunking)."""
    lib = load_library()
    b, L, H, P, G, N = _check_inputs(x, dt, A, B, C, D, init_state)
    if y is not None:
        y_dtype = y.dtype
    shape = make_shape(x, B, 0, y_dtype)
    if y is None:
        y = torch.empty(x.shape, device=x.device, dtype=y_dtype)
    _need(y, "y", y_dtype, x.shape)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), device=x.device, dtype=torch.float32)
    _need(final_state, "final_state", torch.float32, (b, H, P, N))
    _check("selective_scan_fwd", lib.selective_scan_fwd(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A),
                                                        _ptr(B), _ptr(C), _ptr(D), _ptr(init_state),
                                                        _ptr(y), _ptr(final_state), _stream(stream)))
    return y, final_state


def ssd_fwd_varlen_workspace_size(shape: ssd_shape_t, cu_seqlens) -> int:
    cu = [int(v) for v in (cu_seqlens.tolist() if isinstance(cu_seqlens, torch.Tensor) else cu_seqlens)]
    cu_arr = (ctypes.c_int64 * len(cu))(*cu)
    return int(load_library().ssd_fwd_varlen_workspace_size(ctypes.byref(shape), cu_arr, len(cu) - 1))


def ssd_fwd_varlen(x, dt, A, B, C, D=None, init_states=None, cu_seqlens=None, chunk_size=64, *, y=None,
                   final_states=None, return_final_states=True, y_dtype=torch.float32, workspace=None, stream=None):
    """Packed variable-length batch: x [1, Ltot, H, P] etc. hold nseq
    sequences back to back; ``cu_seqlens`` (a host sequence of nseq + 1
    offsets) marks them.  Returns ``(y, final_states [nseq, H, P, N])``."""
    lib = load_library()
    b, L, H, P, G, N = _check_inputs(x, dt, A, B, C, D, None)
    cu = [int(v) for v in (cu_seqlens.tolist() if isinstance(cu_seqlens, torch.Tensor) else cu_seqlens)]
    nseq = len(cu) - 1
    _need(init_states, "init_states", torch.float32, (nseq, H, P, N))
    if y is not None:
        y_dtype = y.dtype
    shape = make_shape(x, B, chunk_size, y_dtype)
    if y is None:
        y = torch.empty(x.shape, device=x.device, dtype=y_dtype)
    _need(y, "y", y_dtype, x.shape)
    if final_states is None and return_final_states:
        final_states = torch.empty((nseq, H, P, N), device=x.device, dtype=torch.float32)
    _need(final_states, "final_states", torch.float32, (nseq, H, P, N))
    cu_arr = (ctypes.c_int64 * len(cu))(*cu)
    ws_bytes = int(lib.ssd_fwd_varlen_workspace_size(ctypes.byref(shape), cu_arr, nseq))
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 16), device=x.device, dtype=torch.uint8)
    _check("ssd_fwd_varlen", lib.ssd_fwd_varlen(ctypes.byref(shape), cu_arr, nseq, _ptr(x), _ptr(dt), _ptr(A),
                                                _ptr(B), _ptr(C), _ptr(D), _ptr(init_states), _ptr(y),
                                                _ptr(final_states), _ptr(workspace), workspace.numel(),
                                                _stream(stream)))
    return y, final_states


def ssd_fwd_quadratic(x, dt, A, B, C, D=None, init_state=None, *, y=None, final_state=None,
                      return_final_state=True, y_dtype=torch.float32, stream=None):
    """The quadratic (dual) form, y = (L o C B^T)(dt o x) + ..., for short
    sequences (L <= 1024).  Returns ``(y, final_state)``."""
    lib = load_library()
    b, L, H, P, G, N = _check_inputs(x, dt, A, B, C, D, init_state)
    if y is not None:
        y_dtype = y.dtype
    shape = make_shape(x, B, 0, y_dtype)
    if y is None:
        y = torch.empty(x.shape, device=x.device, dtype=y_dtype)
    _need(y, "y", y_dtype, x.shape)
    if final_state is None and return_final_state:
        final_state = torch.empty((b, H, P, N), device=x.device, dtype=torch.float32)
    _need(final_state, "final_state", torch.float32, (b, H, P, N))
    _check("ssd_fwd_quadratic", lib.ssd_fwd_quadratic(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                                      _ptr(C), _ptr(D), _ptr(init_state), _ptr(y),
                                                      _ptr(final_state), _stream(stream)))
    return y, final_state


def ssd_decode_step(x, dt, A, B, C, D=None, *, state, y=None, y_dtype=torch.float32, stream=None):
    """One recurrent step: ``state`` [b, H, P, N] fp32 is advanced in place by
    the token x [b, H, P], dt [b, H], B, C [b, G, N]; returns y [b, H, P]."""
    lib = load_library()
    if x.dim() != 3 or B.dim() != 3:
        raise ValueError("x must be [b, H, P] and B, C [b, G, N]")
    b, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    _need(x, "x")
    _need(dt, "dt", x.dtype, (b, H))
    _need(A, "A", torch.float32, (H,))
    _need(B, "B", x.dtype, (b, G, N))
    _need(C, "C", x.dtype, (b, G, N))
    _need(D, "D", torch.float32, (H,))
    _need(state, "state", torch.float32, (b, H, P, N))
    if y is not None:
        y_dtype = y.dtype
    if y is None:
        y = torch.empty((b, H, P), device=x.device, dtype=y_dtype)
    _need(y, "y", y_dtype, (b, H, P))
    yc = SSD_DTYPE_F32 if y_dtype == torch.float32 else _dtype_code(torch.empty(0, dtype=y_dtype))
    shape = ssd_shape_t(b, 1, H, P, N, G, 0, _dtype_code(x), yc)
    _check("ssd_decode_step", lib.ssd_decode_step(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                                  _ptr(C), _ptr(D), _ptr(state), _ptr(y), _stream(stream)))
    return y


def launch_timing(enable: bool) -> None:
    """Turn per-launch CUDA-event timing inside the library on or off."""
    _check("ssd_launch_timing_enable", load_library().ssd_launch_timing_enable(1 if enable else 0))


def launch_times_ms() -> list:
    """[(kernel name, device ms)] for each kernel launch of the most recent call."""
    lib = load_library()
    buf = (ctypes.c_float * 16)()
    n = lib.ssd_launch_timing_read(buf, 16)
    if n < 0:
        return []
    return [((lib.ssd_launch_timing_name(i) or b"?").decode(), float(buf[i])) for i in range(min(n, 16))]


__all__ = ["ssd_fwd_quadratic", "ssd_fwd_varlen", "ssd_fwd_varlen_workspace_size", "ssd_decode_step", "get_device_status", "check_device_status", "selftest_scan_timeout", "ssd_fwd_noalloc", "launch_timing", "launch_times_ms", "ssd_fwd", "ssd_fwd_workspace_size", "ssd_chunk_cumsum", "ssd_chunk_state",
           "ssd_state_passing", "ssd_chunk_scan", "selective_scan_fwd", "ssd_shape_t", "SSDError",
           "load_library", "status_string", "EXPORTED", "LIB_PATH"]
