"""ssd_fwd_noalloc: the forward pass for callers that cannot allocate device
memory (a host application or inference server that owns the device memory
pool, or a latency-critical path that must not call cudaMalloc after
start-up).  Its scratch is a static device buffer inside libssd; these tests
check that it gives bit for bit the results of ssd_fwd (the same kernels,
deterministic), call after call, and that it refuses shapes whose scratch
would not fit.

This file is collected last on purpose: the static buffer is shared by every
call in the process, so running after all other tests also checks that no
earlier work leaves it in a state that changes a result.
"""
import ctypes

import numpy as np
import pytest
import torch

import ssd_inputs as si
import state_space_model_fwd_gb300 as ssd

SCRATCH_LIMIT_STATUS = 5

# largest first, so that every later call runs on top of what a larger one
# left in the shared buffer
CASES = [
    # the 2048-token Mamba-2 130M-shaped layer (about 20 MB of scratch)
    si.CONFIGS["mamba2_130m"],
    # several segments of one chunk each: the scratch holds segment states
    si.SSDConfig("noalloc_segments", 2, 640, 4, 64, 128, 1, 64, "bf16", True, 501),
    # fp32 inputs: the four-stage path keeps its intermediates in the scratch
    si.SSDConfig("noalloc_f32", 1, 256, 2, 16, 16, 1, 64, "f32", True, 502),
]


def _compare(cfg):
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    y_ref, f_ref = ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                               chunk_size=cfg.chunk_size)
    y = torch.full_like(y_ref, float("nan"))
    f = torch.full_like(f_ref, float("nan"))
    ssd.ssd_fwd_noalloc(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                        chunk_size=cfg.chunk_size, y=y, final_state=f)
    assert ssd.get_device_status() == ssd.SSD_OK
    for got, want, what in ((y, y_ref, "y"), (f, f_ref, "final_state")):
        assert torch.isfinite(got).all(), f"{cfg.name}: {what} not fully written"
        assert torch.equal(got, want), f"{cfg.name} {what}: differs from ssd_fwd"


@pytest.mark.gpu
def test_noalloc_matches_ssd_fwd_on_consecutive_calls():
    # consecutive calls with different shapes share the one static buffer;
    # the smaller cases come back at the end, after the largest, to show
    # nothing carries over
    for cfg in CASES + [CASES[1], CASES[0], CASES[1]]:
        _compare(cfg)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """Host-side refusal, before anything is enqueued (no GPU needed): fp32
    inputs at this length need ~270 MB of intermediates."""
    lib = ssd.load_library()
    shape = ssd.ssd_shape_t(1, 65536, 8, 64, 128, 1, 64, ssd.SSD_DTYPE_F32, ssd.SSD_DTYPE_F32)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(shape)) > (32 << 20)
    fake = ctypes.c_void_p(1 << 20)
    st = lib.ssd_fwd_noalloc(ctypes.byref(shape), fake, fake, fake, fake, fake, None, None, fake, None, None)
    assert st == SCRATCH_LIMIT_STATUS
    assert "static" in ssd.status_string(st)
