"""The C ABI on the host: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU
(CPU only: no call here reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

import state_space_model_fwd_gb300 as ssd
from state_space_model_fwd_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")

OK, INVALID, UNSUPPORTED, CUDA_ERR, WORKSPACE, SCRATCH, TIMEOUT = 0, 1, 2, 3, 4, 5, 6


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ssd.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SSD_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    assert set(ssd.EXPORTED) <= set(names), names


def test_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"libssd.so does not export {name}"


def test_status_strings(lib):
    for code in range(7):
        s = ssd.status_string(code)
        assert s.startswith("SSD_"), s
    assert "TIMEOUT" in ssd.status_string(TIMEOUT)
    assert ssd.status_string(99) == "SSD_ERR_UNKNOWN"
    assert lib.ssd_abi_version() >> 16 == 2


def shape(**kw):
    d = dict(batch=2, seqlen=256, nheads=4, headdim=64, dstate=128, ngroups=1, chunk_size=64,
             dtype=1, ydtype=0)
    d.update(kw)
    return ssd.ssd_shape_t(**d)


FAKE = ctypes.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p((1 << 20) + 8)


def fwd(lib, s, ptrs=None, ws=FAKE, ws_bytes=1 << 40):
    p = ptrs or [FAKE] * 9
    return lib.ssd_fwd(ctypes.byref(s), *p, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(nheads=6, ngroups=4), INVALID),        # H % G != 0
    (dict(chunk_size=32), UNSUPPORTED),
    (dict(chunk_size=0), INVALID),
    (dict(headdim=48), UNSUPPORTED),
    (dict(dstate=512), UNSUPPORTED),
    (dict(dtype=7), INVALID),
    (dict(dtype=0, ydtype=1), INVALID),          # bf16 y from fp32 input
    (dict(batch=-1), INVALID),
    (dict(nheads=0), INVALID),
])
def test_shape_validation(lib, kw, code):
    assert fwd(lib, shape(**kw)) == code


def test_null_and_misaligned_pointers(lib):
    s = shape()
    for i in (0, 1, 2, 3, 4, 7):                   # x, dt, A, B, C, y are required
        p = [FAKE] * 9
        p[i] = None
        assert fwd(lib, s, p) == INVALID, i
        p[i] = MISALIGNED
        assert fwd(lib, s, p) == INVALID, i
    p = [FAKE] * 9
    p[6] = MISALIGNED                               # optional init_state, misaligned
    assert fwd(lib, s, p) == INVALID


def test_workspace_checks(lib):
    s = shape()
    need = lib.ssd_fwd_workspace_size(ctypes.byref(s))
    assert need > 0
    assert fwd(lib, s, ws=None) == WORKSPACE
    assert fwd(lib, s, ws_bytes=need - 1) == WORKSPACE
    # a partial last chunk is supported: its workspace covers ceil(L / Q) chunks
    assert lib.ssd_fwd_workspace_size(ctypes.byref(shape(seqlen=250))) == lib.ssd_fwd_workspace_size(
        ctypes.byref(shape(seqlen=256)))
    assert lib.ssd_fwd_workspace_size(ctypes.byref(shape(chunk_size=32))) == 0


def test_empty_batch_is_a_no_op(lib):
    assert fwd(lib, shape(batch=0), [None] * 9, ws=None, ws_bytes=0) == OK


def test_stage_entry_points_validate(lib):
    s = shape(chunk_size=96)
    assert lib.ssd_chunk_cumsum(ctypes.byref(s), FAKE, FAKE, FAKE, None) == UNSUPPORTED
    s = shape()
    assert lib.ssd_chunk_cumsum(ctypes.byref(s), None, FAKE, FAKE, None) == INVALID
    assert lib.ssd_chunk_state(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, None) == INVALID
    assert lib.ssd_state_passing(ctypes.byref(s), None, FAKE, None, FAKE, None, None) == INVALID
    assert lib.ssd_chunk_scan(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 1 << 40,
                              None) == INVALID
    # the tensor-core stage needs its workspace (chunk packs and ready flags)
    s = shape(dtype=1)
    need = lib.ssd_chunk_scan_workspace_size(ctypes.byref(s))
    assert need > 0
    assert lib.ssd_chunk_scan(ctypes.byref(s), *([FAKE] * 8), None, 0, None) == WORKSPACE
    assert lib.ssd_chunk_scan(ctypes.byref(s), *([FAKE] * 8), FAKE, need - 1, None) == WORKSPACE
    # the FFMA stage (fp32 inputs) needs none
    assert lib.ssd_chunk_scan_workspace_size(ctypes.byref(shape(dtype=0))) == 0
    # the failure-path self-test exists only on the tensor-core path
    assert lib.ssd_selftest_scan_timeout(ctypes.byref(shape(dtype=0)), *([FAKE] * 8), FAKE, 1 << 40, 10 ** 6,
                                         None) == UNSUPPORTED
    assert lib.selective_scan_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, None, FAKE, None, None, FAKE, None,
                                  None) == INVALID
    # the sequential scan has no chunk restriction, but still checks groups
    assert lib.selective_scan_fwd(ctypes.byref(shape(nheads=5, ngroups=2)), *([FAKE] * 9), None) == INVALID


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 64, 2, 16)
    with pytest.raises(TypeError):
        ssd.ssd_fwd(x, torch.zeros(1, 64, 2), torch.zeros(2), torch.zeros(1, 64, 1, 16),
                    torch.zeros(1, 64, 1, 16))


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        ssd.load_library(str(tmp_path / "libssd.so"))


def _a256(v):
    return (v + 255) // 256 * 256


@pytest.mark.parametrize("name", ["mamba2_130m", "mamba2_2p7b", "long_16k", "wide_head", "wide_head_q128"])
def test_workspace_layout_of_the_tensor_core_path(lib, name):
    """ssd_fwd's workspace on the bf16 tensor-core path: one ready flag per
    chunk pack, the chunk packs (the masked C B^T of a 64-step tile, bf16),
    and, when the sequence is cut into segments, the segment states (fp32)
    and the segment totals.  With no GPU to query, the segment
    plan assumes the GB300's 152 SMs."""
    import ssd_inputs as si
    import bench
    cfg = si.CONFIGS[name]
    s = ssd.ssd_shape_t(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups,
                        cfg.chunk_size, 1, 1)
    b, L, H, P, N, G = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    nseg, _, nt = bench.tc_plan(cfg, 152)
    nsub = bench.tc_nsub(cfg, 152)
    want = _a256(4 * b * nt * G) + _a256(b * nt * G * 64 * 64 * 2)
    if nseg > 1:
        want += _a256(4 * b * nseg * nsub * H * P * N) + _a256(4 * b * nseg * nsub * H)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(s)) == want


def test_decode_step_validates(lib):
    s = shape(seqlen=1)
    p = [FAKE] * 8
    assert lib.ssd_decode_step(ctypes.byref(shape(nheads=6, ngroups=4)), *p, None) == INVALID
    for i in (0, 1, 2, 3, 4, 6, 7):                  # x, dt, A, B, C, state, y required; D optional
        q = list(p)
        q[i] = None
        assert lib.ssd_decode_step(ctypes.byref(s), *q, None) == INVALID, i
    assert lib.ssd_decode_step(ctypes.byref(shape(batch=0)), *([None] * 8), None) == OK


CBM = 64 * 64 * 2  # one chunk's masked C B^T (64 x 64 bf16)


def varlen_ws(lib, lens, H):
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    arr = (ctypes.c_int64 * len(cu))(*cu)
    return lib.ssd_fwd_varlen_workspace_size(ctypes.byref(shape(batch=1, seqlen=cu[-1], nheads=H)), arr, len(lens))


def test_varlen_plan_cuts_long_sequences_in_a_set(lib):
    """One long sequence among short ones whose units fill the SMs: the set
    cuts the sequences longer than ~1.25 x the tiles per SM into segments
    (here 16384 steps = 256 tiles into 12 segments of 22, the short ones
    whole) rather than running the long one on its own (152 SMs assumed
    without a GPU)."""
    got = varlen_ws(lib, [100] * 200 + [16384], 8)
    # flags | packs of 656 chunks | 201 sequences + 212 scan units + 22
    # segment-state units of 32 bytes | 257 level offsets | 22 local states
    # (8 heads, 64 x 128 fp32) | their totals, each 256-aligned
    assert got == 2816 + 656 * CBM + 14080 + 1280 + 22 * 8 * 64 * 128 * 4 + 768


def test_varlen_plan_splits_off_long_sequences(lib):
    """Too many short sequences to leave table room for segments: the long
    one runs as a fused forward of its own (its segments filling the SMs),
    the short ones as launch sets of up to 800; the workspace is the
    largest of those."""
    own = lib.ssd_fwd_workspace_size(ctypes.byref(shape(batch=1, seqlen=16384, nheads=8)))
    # the first set, 800 one-tile sequences in 37 units of up to 22: flags |
    # packs | 800 sequences + 37 units of 32 bytes | 2 level offsets
    rest = 3328 + 800 * CBM + 26880 + 256
    # all 801 of a first set without segments or groups: 1055 chunks, 801 units, 257 levels
    together = 4352 + 1055 * CBM + 25856 + 1280
    assert varlen_ws(lib, [16] * 900 + [16384], 8) == max(own, rest)
    assert own > max(rest, together)


def test_varlen_plan_groups_short_sequences(lib):
    """64 sequences of 100 / 156 steps with 24 heads (768 one-sequence units,
    five waves): the set packs consecutive sequences (longest first) into
    units of up to 15 chunks, the fewest per unit that keep the units (11 x
    12 head blocks) within one wave; the table holds the 64 sequences and
    the 11 units."""
    got = varlen_ws(lib, [100, 156] * 32, 24)
    # flags | packs of 160 chunks | 64 + 11 entries of 32 bytes | 4 level offsets
    assert got == 768 + 160 * CBM + 2560 + 256


def test_varlen_validates(lib):
    i64 = ctypes.c_int64
    s = shape(batch=1, seqlen=300)
    good = (i64 * 4)(0, 100, 164, 300)
    # three short sequences (at most 3 chunks: segments would not pay) run
    # as one launch set: flags | packs of their 2 + 1 + 3 chunks | 3 units of
    # 32 bytes | 4 chunk-level offsets, each 256-aligned
    assert lib.ssd_fwd_varlen_workspace_size(ctypes.byref(s), good, 3) == 256 + 6 * CBM + 256 + 256
    for bad in ((0, 100, 90, 300), (1, 100, 164, 300), (0, 100, 164, 299)):
        arr = (i64 * 4)(*bad)
        assert lib.ssd_fwd_varlen_workspace_size(ctypes.byref(s), arr, 3) == 0
        assert lib.ssd_fwd_varlen(ctypes.byref(s), arr, 3, *([FAKE] * 10), 1 << 40, None) == INVALID
    assert lib.ssd_fwd_varlen(ctypes.byref(shape(batch=2, seqlen=300)), good, 3, *([FAKE] * 10), 1 << 40,
                              None) == INVALID
    # a sequence start that leaves dt misaligned (H = 4 bf16: 8 bytes a step)
    odd = (i64 * 3)(0, 3, 300)
    assert lib.ssd_fwd_varlen(ctypes.byref(s), odd, 2, *([FAKE] * 10), 1 << 40, None) == INVALID
    assert lib.ssd_fwd_varlen(ctypes.byref(s), good, 3, *([FAKE] * 10), 16, None) == WORKSPACE
