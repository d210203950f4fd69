"""Ragged lengths (L % Q != 0) and packed variable-length batches on the GPU,
against the fp64 oracle.

A partial last chunk is processed as if padded with dt = 0 steps (which
neither decay nor feed the state); nothing is written for the padding.  The
oracle needs no padding: it runs the recurrence over the L real steps.
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
import state_space_model_fwd_gb300 as ssd
from tests.test_gpu_parity import check_bf16_y

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


def rel_err(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape
    assert np.all(np.isfinite(got))
    return float(np.max(np.abs(got - want)) / max(np.sqrt(np.mean(want ** 2)), 1e-30))


def to_np(t):
    return t.detach().double().cpu().numpy()


RAGGED = [
    si.SSDConfig("rg_tc_333", 2, 333, 4, 64, 128, 1, 64, "bf16", True, 801),
    si.SSDConfig("rg_tc_q128", 1, 1000, 4, 64, 128, 2, 128, "bf16", True, 802),
    si.SSDConfig("rg_tc_wide", 1, 200, 4, 128, 256, 2, 64, "bf16", True, 803),
    si.SSDConfig("rg_tc_segments", 1, 4133, 8, 64, 128, 1, 64, "bf16", False, 804),
    si.SSDConfig("rg_tc_h6", 1, 97, 6, 64, 64, 3, 64, "bf16", True, 805),
    si.SSDConfig("rg_simt_bf16", 2, 150, 3, 32, 64, 1, 64, "bf16", True, 806),
    si.SSDConfig("rg_f32", 1, 333, 2, 16, 16, 1, 64, "f32", True, 807),
    si.SSDConfig("rg_short", 1, 5, 2, 64, 128, 1, 64, "bf16", True, 808),
    # Q = 128 chunks run as two 64-step tiles: a last chunk of one partial tile
    si.SSDConfig("rg_tc_q128_onetile", 1, 936, 4, 64, 128, 1, 128, "bf16", True, 809),
]


@pytest.mark.parametrize("cfg", RAGGED, ids=lambda c: c.name)
def test_ssd_fwd_ragged(cfg):
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    y, fin = ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                         chunk_size=cfg.chunk_size)
    f = inp.as_f64()
    y_ref, fin_ref = oracle.ssd_recurrence(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], f["init_state"])
    assert rel_err(to_np(y), y_ref) <= TOL[cfg.dtype]
    assert rel_err(to_np(fin), fin_ref) <= TOL[cfg.dtype]


@pytest.mark.parametrize("cfg", [RAGGED[0], RAGGED[1], RAGGED[2], RAGGED[5], RAGGED[6], RAGGED[8]],
                         ids=lambda c: c.name)
def test_stages_ragged(cfg):
    """Each stage entry point with a partial last chunk against the oracle's
    stage definitions (its missing cumsum entries repeat the last value)."""
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    f = inp.as_f64()
    Q = cfg.chunk_size
    tol = TOL[cfg.dtype]
    cum = ssd.ssd_chunk_cumsum(t["dt"], t["A"], Q)
    cum_ref = oracle.chunk_cumsum(f["dt"], f["A"], Q)
    assert cum.shape == cum_ref.shape
    assert np.max(np.abs(to_np(cum) - cum_ref)) / np.max(np.abs(cum_ref)) <= 1e-5
    cum_in = torch.from_numpy(cum_ref.astype(np.float32)).cuda()
    st = ssd.ssd_chunk_state(t["x"], t["dt"], t["B"], cum_in)
    st_ref = oracle.chunk_states(f["x"], f["dt"], f["A"], f["B"], Q)
    assert rel_err(to_np(st), st_ref) <= tol
    sin_ref, fin_ref = oracle.states_entering(f["x"], f["dt"], f["A"], f["B"], f["C"], Q, f["init_state"])
    sin, fin = ssd.ssd_state_passing(torch.from_numpy(st_ref.astype(np.float32)).cuda(), cum_in, t["init_state"])
    assert rel_err(to_np(sin), sin_ref) <= 1e-5
    assert rel_err(to_np(fin), fin_ref) <= 1e-5
    y = ssd.ssd_chunk_scan(t["x"], t["dt"], t["B"], t["C"], cum_in,
                           torch.from_numpy(sin_ref.astype(np.float32)).cuda(), t["D"])
    y_ref, _ = oracle.ssd_recurrence(f["x"], f["dt"], f["A"], f["B"], f["C"], f["D"], f["init_state"])
    assert rel_err(to_np(y), y_ref) <= tol


def test_ragged_writes_stay_inside_y():
    cfg = RAGGED[0]
    t = si.make_inputs(cfg).to_torch("cuda")
    G = 4096
    n = t["x"].numel() * 2
    raw = torch.full((n + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    raw[G:G + n].fill_(0xFF)
    y = raw[G:G + n].view(torch.bfloat16).view(t["x"].shape)
    ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"], 64, y=y)
    torch.cuda.synchronize()
    assert bool((raw[:G] == 0xA5).all()) and bool((raw[G + n:] == 0xA5).all())
    assert bool(torch.isfinite(y.float()).all())


@pytest.mark.parametrize("dtype,chunk", [("bf16", 64), ("bf16", 128), ("f32", 64)])
def test_varlen_packed_batch(dtype, chunk):
    """Six sequences of unequal lengths (one empty) packed along L: every
    sequence against the oracle run on it alone, from its own initial state."""
    lens = [100, 256, 37, 513, 0, 64]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    H, P, N, G = 8, 64, 128, 2
    if dtype == "f32":
        P, N = 32, 64
    cfg = si.SSDConfig("varlen", 1, cu[-1], H, P, N, G, chunk, dtype, False, 809)
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    init = 0.1 * torch.randn(len(lens), H, P, N, device="cuda", generator=torch.Generator("cuda").manual_seed(9))
    y, fins = ssd.ssd_fwd_varlen(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], init, cu, chunk_size=chunk)
    torch.cuda.synchronize()
    f = inp.as_f64()
    ini = init.double().cpu().numpy()
    tol = TOL[dtype]
    for s, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        y_ref, fin_ref = oracle.ssd_recurrence(f["x"][:, a:e], f["dt"][:, a:e], f["A"], f["B"][:, a:e],
                                               f["C"][:, a:e], f["D"], ini[s:s + 1])
        if e > a:
            assert rel_err(to_np(y[:, a:e]), y_ref) <= tol, s
        assert rel_err(to_np(fins[s:s + 1]), fin_ref) <= tol, s


# Packed batches and the launches they take: one launch set with one segment
# per sequence or several short sequences per scan unit (their units fill
# the SMs), a set whose sequences are cut into
# segments (a segment-state pass, then the scan: few sequences, or one long
# among many), or the longest sequence as a fused forward of its own and the
# rest as a set (too many sequences to leave table room for segments).
# (name, H, P, N, G, chunk, lengths, launch list; the lengths keep every
# sequence's dt 16-byte aligned: even starts for H = 4, multiples of 4 for
# H = 6)
ONE_SET = ["varlen_setup", "cb_mask_tc", "chunk_scan_tc"]
SEG_SET = ["varlen_setup", "cb_mask_tc", "seg_state_tc", "chunk_scan_tc"]
OWN_FWD = ["cb_mask_tc", "seg_state_tc", "chunk_scan_tc"]
VARLEN_SETS = [
    ("short_many", 8, 64, 128, 2, 64, [1, 63, 64, 65, 100, 129, 7, 200, 31, 64] * 4, ONE_SET),
    ("short_q128", 8, 64, 128, 2, 128, [300, 1, 128, 129, 77, 256, 40], ONE_SET),
    ("q128_segments", 8, 64, 128, 2, 128, [3000, 1, 1280, 1290, 770, 2560, 400], SEG_SET),
    ("wide_head", 4, 128, 256, 2, 64, [700, 6, 1300, 64, 2, 1900], SEG_SET),
    ("h6_plain_dt", 6, 64, 64, 3, 64, [1000, 36, 2000, 4, 640, 0, 8], SEG_SET),
    ("few_long_halves", 24, 64, 128, 1, 64, [1000, 700, 300, 5], SEG_SET),
    ("long_in_set", 8, 64, 128, 1, 64, [100, 37] * 100 + [16384], SEG_SET),
    ("long_on_its_own", 8, 64, 128, 1, 64, [16] * 900 + [16384], OWN_FWD + ONE_SET * 2),
]


@pytest.mark.parametrize("case", VARLEN_SETS, ids=[c[0] for c in VARLEN_SETS])
@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16], ids=["y_f32", "y_bf16"])
def test_varlen_launch_set(case, ydt):
    """Every sequence of a packed batch against the oracle run on it alone
    (from its own initial state); y starts as NaN, so a row left unwritten
    fails; the launch list shows which path ran.  bf16 y: 1e-2 x RMS beyond
    half a bf16 ulp of each value (the store's rounding)."""
    name, H, P, N, G, chunk, lens, kernels = case
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    cfg = si.SSDConfig("varlen_" + name, 1, cu[-1], H, P, N, G, chunk, "bf16", False, 811)
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    init = 0.1 * torch.randn(len(lens), H, P, N, device="cuda", generator=torch.Generator("cuda").manual_seed(12))
    y = torch.full(t["x"].shape, float("nan"), device="cuda", dtype=ydt)
    fins = torch.full((len(lens), H, P, N), float("nan"), device="cuda")
    ssd.launch_timing(True)
    try:
        ssd.ssd_fwd_varlen(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], init, cu, chunk_size=chunk, y=y,
                           final_states=fins)
        torch.cuda.synchronize()
        names = [n for n, _ in ssd.launch_times_ms()]
    finally:
        ssd.launch_timing(False)
    ssd.check_device_status()
    assert names == kernels, names
    f = inp.as_f64()
    ini = init.double().cpu().numpy()
    tol = TOL["bf16"]
    errs = []
    for s, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        y_ref, fin_ref = oracle.ssd_recurrence(f["x"][:, a:e], f["dt"][:, a:e], f["A"], f["B"][:, a:e],
                                               f["C"][:, a:e], f["D"], ini[s:s + 1])
        if e > a:
            if ydt == torch.bfloat16:
                errs.append(check_bf16_y(to_np(y[:, a:e]), y_ref, tol, f"sequence {s}")[1])
            else:
                errs.append(rel_err(to_np(y[:, a:e]), y_ref))
                assert errs[-1] <= tol, (s, errs[-1])
        assert rel_err(to_np(fins[s:s + 1]), fin_ref) <= tol, s
    print(f"{name} {ydt}: max err / RMS over {len(lens)} sequences {max(errs):.2e}"
          + (" (beyond half a bf16 ulp)" if ydt == torch.bfloat16 else ""))


@pytest.mark.parametrize("mix", ["ragged4", "short64", "long_and_short"])
def test_varlen_bench_mixes(mix):
    """The packed batches the benchmark times (130M-shaped heads, 8192
    tokens, bf16 y, no initial state), every sequence against the oracle."""
    import bench
    lens = bench.VARLEN_MIXES[mix]
    base = si.CONFIGS["mamba2_130m"]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    cfg = base.replace(name="varlen_" + mix, batch=1, seqlen=cu[-1], has_init=False)
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    H, P, N = base.nheads, base.headdim, base.dstate
    y = torch.full(t["x"].shape, float("nan"), device="cuda", dtype=torch.bfloat16)
    fins = torch.full((len(lens), H, P, N), float("nan"), device="cuda")
    ssd.ssd_fwd_varlen(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], None, cu, base.chunk_size, y=y,
                       final_states=fins)
    torch.cuda.synchronize()
    ssd.check_device_status()
    f = inp.as_f64()
    errs = []
    for s, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        y_ref, fin_ref = oracle.ssd_recurrence(f["x"][:, a:e], f["dt"][:, a:e], f["A"], f["B"][:, a:e],
                                               f["C"][:, a:e], f["D"], None)
        errs.append(check_bf16_y(to_np(y[:, a:e]), y_ref, TOL["bf16"], f"sequence {s}")[1])
        assert rel_err(to_np(fins[s:s + 1]), fin_ref) <= TOL["bf16"], s
    print(f"{mix}: max err / RMS over {len(lens)} sequences {max(errs):.2e} (beyond half a bf16 ulp)")


def test_varlen_more_sequences_than_one_set():
    """2000 short sequences of random lengths (some empty): more than one
    launch set holds (800), so they run as three sets one after another,
    each packing several sequences per scan unit; each sequence against the
    oracle from its own initial state."""
    rng = np.random.default_rng(21)
    lens = [int(v) for v in rng.integers(0, 48, 2000)]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    H, P, N, G = 8, 64, 128, 2
    cfg = si.SSDConfig("varlen_many", 1, cu[-1], H, P, N, G, 64, "bf16", False, 813)
    inp = si.make_inputs(cfg)
    t = inp.to_torch("cuda")
    init = 0.1 * torch.randn(len(lens), H, P, N, device="cuda", generator=torch.Generator("cuda").manual_seed(14))
    y = torch.full(t["x"].shape, float("nan"), device="cuda", dtype=torch.float32)
    fins = torch.full((len(lens), H, P, N), float("nan"), device="cuda")
    ssd.launch_timing(True)
    try:
        ssd.ssd_fwd_varlen(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], init, cu, 64, y=y, final_states=fins)
        torch.cuda.synchronize()
        names = [n for n, _ in ssd.launch_times_ms()]
    finally:
        ssd.launch_timing(False)
    ssd.check_device_status()
    assert names == ONE_SET * 3, names
    f = inp.as_f64()
    ini = init.double().cpu().numpy()
    ys, fs = to_np(y), to_np(fins)
    for s, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        y_ref, fin_ref = oracle.ssd_recurrence(f["x"][:, a:e], f["dt"][:, a:e], f["A"], f["B"][:, a:e],
                                               f["C"][:, a:e], f["D"], ini[s:s + 1])
        if e > a:
            assert rel_err(ys[:, a:e], y_ref) <= TOL["bf16"], s
        assert rel_err(fs[s:s + 1], fin_ref) <= TOL["bf16"], s
