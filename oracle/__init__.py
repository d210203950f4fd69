"""fp64 CPU oracle for the Mamba-2 SSD forward pass.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the benchmark's
CPU-baseline / reference leg are the only callers.  The CUDA product path
never imports this package, and this package imports nothing from the product.

The oracle is the plain selective-SSM recurrence (``ssd_oracle.c``), the
definition the chunked SSD algorithm reproduces up to rounding order:

    h_t = exp(dt_t * A) * h_{t-1} + dt_t * x_t B_t^T        (state [P, N])
    y_t = h_t C_t + D * x_t

("Why SSM and linear-RNN FLOPs do not convert into GPU FLOPs", paragraph 1:
the scalar-decay selective-SSM step; "Mamba-2 in NVIDIA cuTile: Faster
Forward Kernels", section "Why Mamba-2 is a useful kernel example": the
forward pass whose three stages -- cumulative decay, state entering each
chunk, outputs -- are exposed below by their definitions.)

Per-stage references are the definitions of each intermediate, not the
chunked algorithm:

* ``chunk_cumsum``: inclusive running sum of dt*A inside each chunk.
* ``chunk_states``: the state the recurrence reaches over one chunk alone,
  starting from zero (each chunk run as its own sequence).
* ``states_entering``: the recurrence's state just before each chunk starts.

All arithmetic is IEEE fp64.  Inputs are promoted from whatever the caller
holds (bf16-rounded values are passed as their exact float64 values).
Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ssd_oracle.c`` into ``oracle/_build/libssd_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def open_library(path: str):
    """Load an oracle shared object built from ``ssd_oracle.c`` (the tests
    also load copies with a deliberately planted mistake)."""
    lib = ctypes.CDLL(path)
    i64 = ctypes.c_int64
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_ssd_recurrence.argtypes = [i64] * 6 + [dp] * 10 + [i64]
    lib.oracle_ssd_recurrence.restype = ctypes.c_int
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def ssd_recurrence(x, dt, A, B, C, D=None, init_state=None, snap_every=None, lib=None):
    """Run the recurrence in fp64.

    Shapes: x [b, L, H, P], dt [b, L, H], A [H], B/C [b, L, G, N], D [H] or
    None, init_state [b, H, P, N] or None.  Returns ``(y, final_state)``, or
    ``(y, final_state, snaps)`` when ``snap_every`` is given, where
    ``snaps[:, k]`` is the state entering step ``k * snap_every``.
    """
    x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
    D, init_state = _f64(D), _f64(init_state)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt.shape == (b, L, H) and A.shape == (H,)
    assert B.shape == (b, L, G, N) and C.shape == (b, L, G, N)
    assert D is None or D.shape == (H,)
    assert init_state is None or init_state.shape == (b, H, P, N)
    y = np.empty((b, L, H, P), dtype=np.float64)
    final = np.empty((b, H, P, N), dtype=np.float64)
    snaps = None
    every = 0
    if snap_every is not None:
        every = int(snap_every)
        nsnap = (L + every - 1) // every
        snaps = np.empty((b, nsnap, H, P, N), dtype=np.float64)
    rc = (lib or _load()).oracle_ssd_recurrence(
        b, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
        _ptr(D), _ptr(init_state), _ptr(y), _ptr(final), _ptr(snaps), every)
    if rc != 0:
        raise ValueError("oracle_ssd_recurrence rejected its arguments")
    if snaps is not None:
        return y, final, snaps
    return y, final


def _pad_steps(a, Lp):
    """a [b, L, ...] padded with zero steps to length Lp along axis 1."""
    if a.shape[1] == Lp:
        return a
    pad = [(0, 0)] * a.ndim
    pad[1] = (0, Lp - a.shape[1])
    return np.pad(a, pad)


def chunk_cumsum(dt, A, chunk_size):
    """Inclusive running sum of dt*A inside each chunk: [b, H, nc, Q],
    nc = ceil(L / Q).

    ("Mamba-2 in NVIDIA cuTile", section "Why Mamba-2 is a useful kernel
    example": the first kernel prepares the cumulative decay values.)
    A partial last chunk (L % Q != 0) holds its missing steps as dt = 0
    steps: the running sum stays at its last value.
    """
    dt = _f64(dt)
    A = _f64(A)
    b, L, H = dt.shape
    Q = int(chunk_size)
    nc = -(-L // Q)
    dA = _pad_steps(dt * A[None, None, :], nc * Q)          # [b, nc*Q, H]
    dA = dA.reshape(b, nc, Q, H)
    return np.cumsum(dA, axis=2).transpose(0, 3, 1, 2).copy()  # [b, H, nc, Q]


def chunk_states(x, dt, A, B, chunk_size):
    """State each chunk produces on its own from a zero start: [b, nc, H, P, N].

    Each chunk is run through the recurrence as an independent sequence, so
    the value is by definition sum_q exp(sum_{k>q} dt_k A) dt_q x_q B_q^T over
    the chunk.  A partial last chunk (L % Q != 0) is run over its own steps
    (as dt = 0 steps, the missing ones neither decay nor feed the state).
    """
    x, dt, B = _f64(x), _f64(dt), _f64(B)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Q = int(chunk_size)
    nc = -(-L // Q)
    x, dt, B = (_pad_steps(a, nc * Q) for a in (x, dt, B))
    zeros_c = np.zeros((b * nc, Q, G, N))
    _, fin = ssd_recurrence(x.reshape(b * nc, Q, H, P), dt.reshape(b * nc, Q, H),
                            A, B.reshape(b * nc, Q, G, N), zeros_c)
    return fin.reshape(b, nc, H, P, N)


def states_entering(x, dt, A, B, C, chunk_size, init_state=None):
    """State entering each chunk (the state after the previous chunk's last
    step; the initial state for chunk 0): [b, nc, H, P, N]; also returns the
    final state.  ("Mamba-2 in NVIDIA cuTile", section "Why Mamba-2 is a
    useful kernel example": the second kernel computes the state entering
    each chunk.)"""
    y, fin, snaps = ssd_recurrence(x, dt, A, B, C, None, init_state,
                                   snap_every=chunk_size)
    return snaps, fin


__all__ = ["build", "ssd_recurrence", "chunk_cumsum", "chunk_states",
           "states_entering", "num_threads", "set_num_threads"]
