"""The quadratic (dual) form kernel on the GPU against the fp64 oracle.

ssd_fwd_quadratic computes y = (L o C B^T)(dt o x) + (exp(cum) o C) init^T
+ D x without chunks; the recurrence (the oracle) reaches the same result
(pin p1 ties the two forms together on the CPU).
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
    assert got.shape == want.shape
    assert np.all(np.isfinite(got))
    return float(np.max(np.abs(got - want)) / max(np.sqrt(np.mean(want ** 2)), 1e-30))


CASES = [
    si.SSDConfig("quad_1", 2, 1, 4, 64, 128, 1, 64, "bf16", True, 901),
    si.SSDConfig("quad_64", 2, 64, 4, 64, 128, 1, 64, "bf16", True, 902),
    si.SSDConfig("quad_100", 1, 100, 6, 64, 64, 3, 64, "bf16", True, 903),
    si.SSDConfig("quad_128_p128", 2, 128, 4, 128, 128, 2, 64, "bf16", True, 904),
    si.SSDConfig("quad_300", 1, 300, 4, 64, 128, 2, 64, "bf16", False, 905),
    si.SSDConfig("quad_777_p128_n64", 1, 777, 2, 128, 64, 1, 64, "bf16", True, 906),
    si.SSDConfig("quad_1024", 1, 1024, 8, 64, 128, 1, 64, "bf16", True, 907),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_quadratic_form_matches_the_recurrence(cfg):
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    f = inp.as_f64()
    y_ref, fin_ref = oracle.ssd_recurrence(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], f["init_state"])
    y, fin = ssd.ssd_fwd_quadratic(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"])
    y16, fin16 = ssd.ssd_fwd_quadratic(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                                       y_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert rel_err(y.double().cpu().numpy(), y_ref) <= 1e-2
    assert rel_err(fin.double().cpu().numpy(), fin_ref) <= 1e-2
    check_bf16_y(y16.double().cpu().numpy(), y_ref, 1e-2, f"{cfg.name} bf16 y")
    assert torch.equal(fin, fin16)


def test_quadratic_form_without_optional_inputs():
    cfg = CASES[2]
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    f = inp.as_f64()
    y, fin = ssd.ssd_fwd_quadratic(t["x"], t["dt"], t["A"], t["B"], t["C"], None, None, return_final_state=False)
    torch.cuda.synchronize()
    assert fin is None
    y_ref, _ = oracle.ssd_recurrence(f["x"], f["dt"], f["A"], f["B"], f["C"], None, None)
    assert rel_err(y.double().cpu().numpy(), y_ref) <= 1e-2


def test_quadratic_form_agrees_with_chunked_form():
    """Two algorithms, one result: the quadratic kernel and the chunked
    ssd_fwd on the same 512-step inputs."""
    cfg = si.SSDConfig("quad_vs_chunked", 2, 512, 8, 64, 128, 1, 64, "bf16", True, 908)
    t = si.make_inputs(cfg).to_torch("cuda")
    args = (t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"])
    yq, fq = ssd.ssd_fwd_quadratic(*args)
    yc, fc = ssd.ssd_fwd(*args, chunk_size=64)
    torch.cuda.synchronize()
    assert rel_err(yq.double().cpu().numpy(), yc.double().cpu().numpy()) <= 2e-2
    assert rel_err(fq.double().cpu().numpy(), fc.double().cpu().numpy()) <= 2e-2


def test_quadratic_form_refuses_long_or_fp32():
    x = torch.zeros(1, 2048, 2, 64, device="cuda", dtype=torch.bfloat16)
    dt = torch.zeros(1, 2048, 2, device="cuda", dtype=torch.bfloat16)
    B = torch.zeros(1, 2048, 1, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ssd.SSDError):
        ssd.ssd_fwd_quadratic(x, dt, -torch.ones(2, device="cuda"), B, B)
    with pytest.raises(ssd.SSDError):
        ssd.ssd_fwd_quadratic(x[:, :64].float(), dt[:, :64].float(), -torch.ones(2, device="cuda"),
                              B[:, :64].float(), B[:, :64].float())
