"""The recurrent (decode) step on the GPU against the fp64 oracle.

A sequence fed token by token through ssd_decode_step must reproduce the
recurrence over the whole sequence (the oracle), output by output and in its
final state; and a state left by the chunked forward (prefill) must continue
into decode steps as if the sequence had never been split (split/resume,
pin p5 of the oracle).
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
import state_space_model_fwd_gb300 as ssd
from tests.test_gpu_parity import check_bf16_y

pytestmark = pytest.mark.gpu


def rel_err(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.all(np.isfinite(got))
    return float(np.max(np.abs(got - want)) / max(np.sqrt(np.mean(want ** 2)), 1e-30))


CASES = [
    si.SSDConfig("dec_f32", 2, 24, 3, 16, 16, 1, 64, "f32", True, 701),
    si.SSDConfig("dec_bf16_p64_n128", 3, 24, 6, 64, 128, 2, 64, "bf16", True, 702),
    si.SSDConfig("dec_bf16_p128_n256_g8", 2, 16, 16, 128, 256, 8, 64, "bf16", True, 703),
    si.SSDConfig("dec_bf16_p32_n64_noinit", 1, 16, 4, 32, 64, 4, 64, "bf16", False, 704),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("y_dtype", ["f32", "in"])
def test_decode_steps_reproduce_the_recurrence(cfg, y_dtype):
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    f = inp.as_f64()
    b, L, H, P, N = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate
    state = (t["init_state"].clone() if t["init_state"] is not None
             else torch.zeros(b, H, P, N, device="cuda"))
    ydt = torch.float32 if y_dtype == "f32" else t["x"].dtype
    ys = []
    for k in range(L):
        # (clone: a batch-1 slice is a view at an offset the library may
        # rightly refuse as unaligned)
        ys.append(ssd.ssd_decode_step(t["x"][:, k].clone(), t["dt"][:, k].clone(), t["A"],
                                      t["B"][:, k].clone(), t["C"][:, k].clone(), t["D"],
                                      state=state, y_dtype=ydt))
    torch.cuda.synchronize()
    y = torch.stack(ys, 1).double().cpu().numpy()
    y_ref, fin_ref = oracle.ssd_recurrence(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], f["init_state"])
    if ydt == torch.float32:
        assert rel_err(y, y_ref) <= 1e-4
    else:   # bf16 y: the arithmetic within 1e-4 x RMS beyond the output's half ulp
        check_bf16_y(y, y_ref, 1e-4, f"{cfg.name} decode y (bf16)")
    assert rel_err(state.double().cpu().numpy(), fin_ref) <= 1e-4


def test_prefill_then_decode_is_one_sequence():
    """ssd_fwd over the first 256 tokens (tensor-core path), then 8 decode
    steps from its final state, against the oracle over all 264 tokens."""
    cfg = si.SSDConfig("prefill_decode", 2, 264, 4, 64, 128, 1, 64, "bf16", True, 705)
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    L0 = 256
    sl = lambda a: a[:, :L0].contiguous()
    y0, state = ssd.ssd_fwd(sl(t["x"]), sl(t["dt"]), t["A"], sl(t["B"]), sl(t["C"]), t["D"], t["init_state"],
                            chunk_size=64)
    ys = [ssd.ssd_decode_step(t["x"][:, k].clone(), t["dt"][:, k].clone(), t["A"],
                              t["B"][:, k].clone(), t["C"][:, k].clone(), t["D"], state=state)
          for k in range(L0, cfg.seqlen)]
    torch.cuda.synchronize()
    f = inp.as_f64()
    y_ref, fin_ref = oracle.ssd_recurrence(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], f["init_state"])
    assert rel_err(y0.double().cpu().numpy(), y_ref[:, :L0]) <= 1e-2
    assert rel_err(torch.stack(ys, 1).double().cpu().numpy(), y_ref[:, L0:]) <= 1e-2
    assert rel_err(state.double().cpu().numpy(), fin_ref) <= 1e-2


def test_decode_writes_stay_inside_outputs():
    cfg = si.SSDConfig("dec_guard", 4, 1, 8, 64, 128, 2, 64, "bf16", True, 706)
    t = si.make_inputs(cfg).to_torch("cuda")
    G = 4096
    raw = torch.full((4 * 8 * 64 * 2 + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    y = raw[G:G + 4 * 8 * 64 * 2].view(torch.bfloat16).view(4, 8, 64)
    rawS = torch.full((4 * 8 * 64 * 128 * 4 + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    S = rawS[G:-G].view(torch.float32).view(4, 8, 64, 128)
    S.copy_(t["init_state"])
    ssd.ssd_decode_step(t["x"][:, 0].clone(), t["dt"][:, 0].clone(), t["A"], t["B"][:, 0].clone(),
                        t["C"][:, 0].clone(), t["D"], state=S, y=y)
    torch.cuda.synchronize()
    for r in (raw, rawS):
        assert bool((r[:G] == 0xA5).all()) and bool((r[-G:] == 0xA5).all())
