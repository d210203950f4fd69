"""Seeded synthetic inputs for the SSD forward workloads.

This module holds no part of the method's arithmetic: it only draws random
tensors.  Both the CUDA path (through the tests and the benchmark) and the
fp64 oracle consume exactly the arrays it returns, so the two sides see the
same bf16-rounded values.

Generator: SplitMix64 used as a counter-based generator (the 64-bit finaliser
of Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014) keyed per (seed, tensor), 53-bit uniforms, Box-Muller normals.

Value distributions (Mamba-2 layer initialisation shapes):
  x ~ N(0, 1)
  dt = softplus(N(0, 0.5) + inv_softplus(u)), u log-uniform in [1e-3, 1e-1],
       u drawn once per head (a dt bias), the noise per (batch, step, head)
  A_h = -exp(U[0, ln 16])
  B, C ~ N(0, 1) / sqrt(N)
  D ~ N(0, 1)
  init_state ~ N(0, 0.1^2)   (only for the workloads that carry one)
bf16 workloads round x, dt, B, C to bf16 (round to nearest even) on the host;
A, D and the initial state stay fp32.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22


@dataclasses.dataclass(frozen=True)
class SSDConfig:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int
    dtype: str          # "f32" or "bf16"
    has_init: bool
    seed: int

    @property
    def nchunks(self) -> int:
        return self.seqlen // self.chunk_size

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def replace(self, **kw) -> "SSDConfig":
        return dataclasses.replace(self, **kw)


# The five SSD forward workloads (plus the Q=128 sweep point of the last).
CONFIGS = {
    "tiny_f32": SSDConfig("tiny_f32", 1, 256, 2, 16, 16, 1, 64, "f32", False, 1000),
    "mamba2_130m": SSDConfig("mamba2_130m", 4, 2048, 24, 64, 128, 1, 64, "bf16", False, 1001),
    "mamba2_2p7b": SSDConfig("mamba2_2p7b", 2, 4096, 80, 64, 128, 1, 64, "bf16", True, 1002),
    "long_16k": SSDConfig("long_16k", 1, 16384, 48, 64, 128, 1, 64, "bf16", False, 1003),
    "wide_head": SSDConfig("wide_head", 2, 8192, 64, 128, 256, 8, 64, "bf16", True, 1004),
    "wide_head_q128": SSDConfig("wide_head_q128", 2, 8192, 64, 128, 256, 8, 128, "bf16", True, 1004),
}


def _mix(z):
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([(seed * 1009 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(k * _GAMMA + _GAMMA)[0]


def _uniform_block(key, start, count):
    """53-bit uniforms in (0, 1] for counters start .. start+count-1."""
    with np.errstate(over="ignore"):
        i = np.arange(start, start + count, dtype=np.uint64)
        z = _mix(key + (i + np.uint64(1)) * _GAMMA)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    key = _key(seed, stream)
    out = np.empty(n, dtype=np.float64)

    def work(s):
        c = min(_BLOCK, n - s)
        out[s:s + c] = _uniform_block(key, s, c)

    with ThreadPoolExecutor(8) as ex:
        list(ex.map(work, range(0, n, _BLOCK)))
    return out


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """Standard normals, element i from counters 2i, 2i+1 (Box-Muller)."""
    key = _key(seed, stream)
    out = np.empty(n, dtype=np.float64)

    def work(s):
        c = min(_BLOCK, n - s)
        u = _uniform_block(key, 2 * s, 2 * c)
        u1, u2 = u[0::2], u[1::2]
        out[s:s + c] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    with ThreadPoolExecutor(8) as ex:
        list(ex.map(work, range(0, n, _BLOCK)))
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _softplus(z):
    return np.logaddexp(0.0, z)


def _inv_softplus(u):
    return u + np.log(-np.expm1(-u))


@dataclasses.dataclass
class SSDInputs:
    """Host arrays of one workload.  x, dt, B, C are float32 arrays (f32
    workloads) or uint16 bf16 bit patterns (bf16 workloads)."""
    cfg: SSDConfig
    x: np.ndarray
    dt: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: np.ndarray
    init_state: np.ndarray | None

    def values(self, name: str) -> np.ndarray:
        """float32 view of the values a tensor holds (bf16 widened exactly)."""
        a = getattr(self, name)
        if a is None:
            return None
        if a.dtype == np.uint16:
            return bf16_bits_to_f32(a)
        return a

    def as_f64(self) -> dict:
        """Exact float64 copies, the oracle's inputs."""
        return {k: (None if self.values(k) is None else self.values(k).astype(np.float64))
                for k in ("x", "dt", "A", "B", "C", "D", "init_state")}

    def to_torch(self, device="cuda", pin_memory=False):
        """torch tensors (bf16 / fp32) on ``device`` ("cpu" with pin_memory
        for host staging buffers)."""
        import torch

        def t(a):
            if a is None:
                return None
            if a.dtype == np.uint16:
                tt = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
            else:
                tt = torch.from_numpy(np.ascontiguousarray(a))
            if device == "cpu":
                return tt.pin_memory() if pin_memory else tt.clone()
            return tt.to(device)

        return {k: t(getattr(self, k)) for k in ("x", "dt", "A", "B", "C", "D", "init_state")}


def make_inputs(cfg: SSDConfig) -> SSDInputs:
    b, L, H, P, N, G = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    s = cfg.seed
    x = normal(s, 1, b * L * H * P).reshape(b, L, H, P)
    u = np.exp(np.log(1e-3) + (np.log(1e-1) - np.log(1e-3)) * uniform(s, 3, H))
    dt = _softplus(0.5 * normal(s, 2, b * L * H).reshape(b, L, H) + _inv_softplus(u)[None, None, :])
    A = -np.exp(np.log(16.0) * uniform(s, 4, H))
    Bm = normal(s, 5, b * L * G * N).reshape(b, L, G, N) / np.sqrt(N)
    Cm = normal(s, 6, b * L * G * N).reshape(b, L, G, N) / np.sqrt(N)
    D = normal(s, 7, H)
    init = (0.1 * normal(s, 8, b * H * P * N).reshape(b, H, P, N)).astype(np.float32) \
        if cfg.has_init else None
    if cfg.dtype == "bf16":
        cv = to_bf16_bits
    else:
        def cv(a):
            return np.ascontiguousarray(a, dtype=np.float32)
    return SSDInputs(cfg, cv(x), cv(dt), A.astype(np.float32), cv(Bm), cv(Cm),
                     D.astype(np.float32), init)
