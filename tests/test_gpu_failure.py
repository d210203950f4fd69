"""Failure detection and out-of-bounds writes on the GPU, without a fault.

* The bounded waits: the chunk-scan stage kernel is launched alone with its
  operand packs never published, so every CTA's wait for its first pack runs
  out (a flag that nothing sets); the kernel drains and exits, the device
  status word reads SSD_ERR_TIMEOUT, and the context keeps working.
* Guard regions: every output buffer sits between two guard regions filled
  with a byte pattern, its own bytes filled with NaN; after the call the
  guards are intact (no write past either end) and the output is finite
  (every element written).
"""
import numpy as np
import pytest
import torch

import ssd_inputs as si
import state_space_model_fwd_gb300 as ssd

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side of an output
PATTERN = 0xA5


def guarded(shape, dtype):
    """(raw, view): `view` is a contiguous tensor of `shape` inside `raw`,
    between two GUARD-byte regions of PATTERN, its own bytes set to 0xFF
    (NaN for fp32 and bf16)."""
    es = torch.empty(0, dtype=dtype).element_size()
    nbytes = int(np.prod(shape)) * es
    raw = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    raw[GUARD:GUARD + nbytes].fill_(0xFF)
    view = raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
    assert view.data_ptr() % 16 == 0
    return raw, view


def assert_guards(raw, view, what):
    nbytes = view.numel() * view.element_size()
    head, tail = raw[:GUARD], raw[GUARD + nbytes:]
    assert bool((head == PATTERN).all()), f"{what}: write before the start of the buffer"
    assert bool((tail == PATTERN).all()), f"{what}: write past the end of the buffer"
    assert bool(torch.isfinite(view.float()).all()), f"{what}: elements left unwritten"


def test_bounded_wait_gives_up_and_reports_timeout():
    cfg = si.SSDConfig("timeout", 1, 256, 4, 64, 128, 1, 64, "bf16", True, 601)
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    cum = ssd.ssd_chunk_cumsum(t["dt"], t["A"], 64)
    st = ssd.ssd_chunk_state(t["x"], t["dt"], t["B"], cum)
    sin, _ = ssd.ssd_state_passing(st, cum, t["init_state"])
    assert ssd.get_device_status() == ssd.SSD_OK
    y = torch.zeros(t["x"].shape, device="cuda", dtype=torch.float32)
    # 2 ms: every CTA's wait for its first operand pack runs out
    assert ssd.selftest_scan_timeout(t["x"], t["dt"], t["B"], t["C"], cum, sin, t["D"], out=y,
                                     wait_ns=2_000_000) == ssd.SSD_OK
    assert ssd.get_device_status() == ssd.SSD_ERR_TIMEOUT
    assert ssd.get_device_status() == ssd.SSD_OK          # reading cleared it
    assert torch.count_nonzero(y) == 0                   # nothing was computed
    # the context still works: the same stage, published normally
    y2 = ssd.ssd_chunk_scan(t["x"], t["dt"], t["B"], t["C"], cum, sin, t["D"])
    y3, _ = ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"])
    assert ssd.get_device_status() == ssd.SSD_OK
    rms = float(y3.double().pow(2).mean().sqrt())
    assert float((y2.double() - y3.double()).abs().max()) <= 2e-2 * rms


FULL = ["mamba2_130m", "mamba2_2p7b", "long_16k", "wide_head", "wide_head_q128"]


@pytest.mark.parametrize("name", FULL)
@pytest.mark.parametrize("y_dtype", [torch.bfloat16, torch.float32])
def test_ssd_fwd_writes_stay_inside_outputs(name, y_dtype):
    cfg = si.CONFIGS[name]
    t = si.make_inputs(cfg).to_torch("cuda")
    ry, y = guarded(t["x"].shape, y_dtype)
    rf, fin = guarded((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), torch.float32)
    ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"], cfg.chunk_size,
                y=y, final_state=fin)
    torch.cuda.synchronize()
    assert_guards(ry, y, f"{name} y")
    assert_guards(rf, fin, f"{name} final_state")


STAGE_CASES = [
    si.SSDConfig("guard_tc", 2, 640, 4, 64, 128, 1, 64, "bf16", True, 602),
    si.SSDConfig("guard_tc_wide", 1, 384, 4, 128, 256, 2, 64, "bf16", True, 603),
    si.SSDConfig("guard_simt", 1, 512, 3, 32, 64, 1, 128, "bf16", True, 604),
    si.SSDConfig("guard_f32", 1, 256, 2, 16, 16, 1, 64, "f32", True, 605),
]


@pytest.mark.parametrize("cfg", STAGE_CASES, ids=lambda c: c.name)
def test_stage_writes_stay_inside_outputs(cfg):
    t = si.make_inputs(cfg).to_torch("cuda")
    b, L, H, P, N, Q = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.chunk_size
    nc = L // Q
    rc, cum = guarded((b, H, nc, Q), torch.float32)
    ssd.ssd_chunk_cumsum(t["dt"], t["A"], Q, out=cum)
    rs, st = guarded((b, nc, H, P, N), torch.float32)
    ssd.ssd_chunk_state(t["x"], t["dt"], t["B"], cum, out=st)
    ri, sin = guarded((b, nc, H, P, N), torch.float32)
    rf, fin = guarded((b, H, P, N), torch.float32)
    ssd.ssd_state_passing(st, cum, t["init_state"], out=sin, final_state=fin)
    ry, y = guarded(t["x"].shape, t["x"].dtype)
    ssd.ssd_chunk_scan(t["x"], t["dt"], t["B"], t["C"], cum, sin, t["D"], out=y)
    rq, yq = guarded(t["x"].shape, t["x"].dtype)
    ssd.selective_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"], y=yq,
                           final_state=None, return_final_state=False)
    torch.cuda.synchronize()
    for raw, view, what in ((rc, cum, "dA_cumsum"), (rs, st, "states"), (ri, sin, "states_in"),
                            (rf, fin, "final_state"), (ry, y, "chunk-scan y"), (rq, yq, "sequential-scan y")):
        assert_guards(raw, view, f"{cfg.name} {what}")


# Packed sequences whose last one ends in a partial chunk (its y rows are
# written with plain stores that stop at the sequence's end): one launch set
# with one segment each, one with several sequences per scan unit, one with
# segments, and one with the long sequence as a fused forward of its own.
VARLEN_GUARD = [
    ("one_set", 8, [1, 63, 100, 129, 7, 200] * 8 + [37]),
    ("grouped", 24, [100, 156] * 32 + [37]),
    ("segments", 8, [1000, 700, 300, 37]),
    ("own_forward", 8, [16] * 900 + [16384, 37]),
]


@pytest.mark.parametrize("name,H,lens", VARLEN_GUARD, ids=[c[0] for c in VARLEN_GUARD])
@pytest.mark.parametrize("y_dtype", [torch.bfloat16, torch.float32])
def test_varlen_writes_stay_inside_outputs(name, H, lens, y_dtype):
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    cfg = si.SSDConfig("varlen_guard_" + name, 1, cu[-1], H, 64, 128, 1, 64, "bf16", False, 607)
    t = si.make_inputs(cfg).to_torch("cuda")
    ry, y = guarded(t["x"].shape, y_dtype)
    rf, fins = guarded((len(lens), H, 64, 128), torch.float32)
    ssd.ssd_fwd_varlen(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], None, cu, 64, y=y, final_states=fins)
    torch.cuda.synchronize()
    ssd.check_device_status()
    assert_guards(ry, y, f"{name} y")
    assert_guards(rf, fins, f"{name} final_states")
