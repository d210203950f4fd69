"""Benchmark of the fused SSD forward (ssd_fwd) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one ssd_fwd call (the whole chunked forward: cumulative decay,
chunk states, state passing, chunk outputs) over one batch of the Mamba-2
130M-shaped layer workload: batch 4, L 2048, H 24, P 64, N 128, G 1, Q 64,
bf16 inputs and y, fp32 state and accumulation.  Inputs are seeded synthetic
tensors (ssd_inputs.py), resident in HBM before timing starts; L2 (129 MB,
larger than this workload's 58 MB) is flushed by a 512 MB write between
timed steps, outside the timed events.

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) give every rank
its own independent batch: weak scaling, no data-path collective.
--impl reference times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import ssd_inputs as si  # noqa: E402

WORKLOAD = "mamba2_130m"
FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
Y_BYTES = 2  # y in bf16, the input dtype (fp32 state and accumulation)


# ---------------------------------------------------------------------------
# byte / flop models (algorithmic, per call)
# ---------------------------------------------------------------------------
def elem_bytes(dtype):
    return 4 if dtype == "f32" else 2


def compulsory_bytes(cfg, y_bytes=Y_BYTES):
    """Reads of x, dt, B, C, A, D (+ init) and writes of y and final state."""
    b, L, H, P, N, G = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    e = elem_bytes(cfg.dtype)
    rd = b * L * H * P * e + b * L * H * e + 2 * b * L * G * N * e + 2 * H * 4
    if cfg.has_init:
        rd += b * H * P * N * 4
    wr = b * L * H * P * y_bytes + b * H * P * N * 4
    return rd + wr


def chunked_flops(cfg, q=None):
    """Tensor-core flops of the chunked algorithm with full q x q tiles (q =
    the chunk size unless given): per token H (4PN + 2qP) + G 2qN, plus the
    state pass 2PN H / q."""
    H, P, N, G = cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    Q = cfg.chunk_size if q is None else q
    per_tok = H * (4 * P * N + 2 * Q * P) + G * 2 * Q * N + H * 2 * P * N / Q
    return per_tok * cfg.tokens


# steps per tile of the fused tensor-core forward: a 128-step chunk runs as two
# 64-step tiles, so the work executed is that of 64-step tiles
FWD_TILE = 64


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)

        def find(keys):
            for k in keys:
                for kk, v in pk.items():
                    if kk.lower() == k and isinstance(v, (int, float)):
                        return float(v)
            return None
        hbm = find(["hbm_gbs", "hbm_gb_s", "hbm_bandwidth_gbs"])
        tf = find(["bf16_tflops", "bf16_dense_tflops"])
        tfs = find(["bf16_tflops_sustained"])
        if hbm:
            return {"hbm_gbs": hbm, "bf16_tflops": tf or FALLBACK_BF16_TFLOPS,
                    "bf16_tflops_sustained": tfs, "source": "measured"}
    except (OSError, ValueError):
        pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------
def smi_gpu_id(local_rank):
    """nvidia-smi's id of this rank's GPU: CUDA numbers the visible devices
    from 0, nvidia-smi names the physical ones (index or UUID), so a
    CUDA_VISIBLE_DEVICES list maps one onto the other."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if 0 <= local_rank < len(ids):
        return ids[local_rank]
    return str(local_rank)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# ncu traffic recorded under profiles/ (null when the kernel source changed)
# ---------------------------------------------------------------------------
def code_of(text):
    """The source text without comments, trailing spaces and blank lines: a
    change to comments alone leaves the recorded profiles valid."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_sha():
    """Hash of the code of the CUDA sources, the key of the recorded ncu
    summaries under profiles/."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "state_space_model_fwd_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_sha():
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


# Multi-rank host logic (replicas: every rank its own batch, no data-path
# collective).  Plain functions so that they run under gloo on CPU as well.
def rank_config(cfg, rank):
    """Each rank draws its own batch: the same shapes, a seed offset by rank."""
    return cfg.replace(seed=cfg.seed + 7919 * rank)


def max_over_ranks(x, world, device=None):
    """Largest value over the ranks (the slowest rank's time); x on one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time."""
    return world * tokens_per_rank / (ms * 1e-3)


def run_reference(args):
    """The fp64 CPU oracle timed on this host's cores: each step runs the
    recurrence over a bounded sample of heads of the workload, scaled to
    tokens/s of the whole workload by the fraction of heads sampled."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = si.CONFIGS[args.workload]
    inp = si.make_inputs(cfg)
    f = inp.as_f64()
    nh = max(1, min(cfg.nheads, args.ref_heads))
    g_of = [h * cfg.ngroups // cfg.nheads for h in range(nh)]
    sl = dict(x=f["x"][:, :, :nh], dt=f["dt"][:, :, :nh], A=f["A"][:nh], D=f["D"][:nh],
              init=None if f["init_state"] is None else f["init_state"][:, :nh])
    Bs = f["B"][:, :, g_of]
    Cs = f["C"][:, :, g_of]

    def step():
        oracle.ssd_recurrence(sl["x"], sl["dt"], sl["A"], Bs, Cs, sl["D"], sl["init"])

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times) * cfg.nheads / nh
    value = cfg.tokens / t
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": "ssd_fwd_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg.name, "batch": cfg.batch, "seqlen": cfg.seqlen,
                                        "nheads": cfg.nheads, "headdim": cfg.headdim, "dstate": cfg.dstate,
                                        "ngroups": cfg.ngroups, "chunk_size": cfg.chunk_size},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"fp64 recurrence over {nh} of {cfg.nheads} heads, all batches and steps, "
                                   f"scaled by {cfg.nheads}/{nh}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def oracle_sample_time(cfg, f, budget_s):
    """Seconds the oracle takes over the whole workload, from a sample of
    heads grown (x4) while it fits the budget, scaled by the heads."""
    import oracle
    nh = 1
    while True:
        g_of = [h * cfg.ngroups // cfg.nheads for h in range(nh)]
        t0 = time.perf_counter()
        oracle.ssd_recurrence(f["x"][:, :, :nh], f["dt"][:, :, :nh], f["A"][:nh], f["B"][:, :, g_of],
                              f["C"][:, :, g_of], f["D"][:nh],
                              None if f["init_state"] is None else f["init_state"][:, :nh])
        t_one = time.perf_counter() - t0
        if t_one * 4 > budget_s or nh == cfg.nheads:
            break
        nh = min(cfg.nheads, nh * 4)
    return t_one * cfg.nheads / nh, nh, t_one


def cpu_baseline(cfg, inp, budget_s=12.0):
    """Oracle time on this host for a bounded sample of heads, scaled: on
    every core (OpenMP over batch, head, channel) and on one core."""
    import oracle
    oracle.build()
    f = inp.as_f64()
    cores = oracle.num_threads()
    t_full, nh, t_one = oracle_sample_time(cfg, f, budget_s)
    oracle.set_num_threads(1)
    try:
        t1_full, nh1, t1_one = oracle_sample_time(cfg, f, budget_s / 2)
    finally:
        oracle.set_num_threads(cores)
    return {"value": cfg.tokens / t_full, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 recurrence over {nh} of {cfg.nheads} heads (all batches, all {cfg.seqlen} steps), "
                      f"{t_one:.2f} s, scaled by {cfg.nheads}/{nh}",
            "one_core": {"value": cfg.tokens / t1_full, "unit": "tokens/s", "cores": 1,
                         "sample": f"{nh1} of {cfg.nheads} heads, {t1_one:.2f} s, scaled by {cfg.nheads}/{nh1}"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(si.CONFIGS))
    ap.add_argument("--ref-heads", type=int, default=4)
    ap.add_argument("--no-sweep", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["stages", "sequential", "crossover", "decode", "varlen"],
                    help="run one part of the sweep alone and print its JSON (for profiling that part)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)
    if args.only:
        return run_only(args)

    import torch
    import state_space_model_fwd_gb300 as ssd

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count

    cfg = si.CONFIGS[args.workload]
    cfg_rank = rank_config(cfg, rank)
    inp = si.make_inputs(cfg_rank)
    t = inp.to_torch(dev)
    y = torch.empty(t["x"].shape, device=dev, dtype=torch.bfloat16)
    fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), device=dev, dtype=torch.float32)
    ws = torch.empty(max(16, ssd.ssd_fwd_workspace_size(ssd.make_shape(t["x"], t["B"], cfg.chunk_size,
                                                                       torch.bfloat16))),
                     device=dev, dtype=torch.uint8)
    flush = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"], cfg.chunk_size,
                    y=y, final_state=fin, workspace=ws)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    # per-launch device times (a separate, untimed pass with events between
    # the launches; run first, its steps also settle the device: in a fresh
    # process the first tens of steps run slower)
    ssd.launch_timing(True)
    per_launch = []
    for _ in range(max(10, args.steps // 2)):
        flush.zero_()
        step()
        per_launch.append(ssd.launch_times_ms())
    ssd.launch_timing(False)
    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(smi_gpu_id(local_rank)) as clk:
        barrier()
        wall0 = time.perf_counter()
        for s, e in evs:
            flush.zero_()
            s.record(stream)
            step()
            e.record(stream)
        barrier()
        wall = time.perf_counter() - wall0
    step_ms = [s.elapsed_time(e) for s, e in evs]
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    launches_per_step = len(per_launch[-1])
    kernel_names = [name for name, _ in per_launch[-1]]
    launch_ms = [statistics.mean(p[i][1] for p in per_launch) for i in range(launches_per_step)]
    dom = int(np.argmax(launch_ms))

    peaks = load_peaks()
    cbytes = compulsory_bytes(cfg)
    dom_name = kernel_names[dom] if dom < len(kernel_names) else f"launch{dom}"
    # achieved: the operation's compulsory bytes (reads of x, dt, B, C, A, D,
    # init; writes of y, final state) over the dominant kernel's time; the
    # bytes the kernel itself moves (its own intermediates included) are
    # reported beside it
    achieved = cbytes / (launch_ms[dom] * 1e-3) / 1e9
    dom_bytes = KERNEL_BYTES(cfg, dom_name)
    tokens = cfg.tokens
    value = job_tokens_per_s(tokens, world, ms)

    # end-to-end through the C ABI with host buffers: every step copies its
    # inputs in from pinned host memory, calls ssd_fwd, and reads y and the
    # final state back.  Serial: one stream.  Pipelined: double buffers on
    # three streams, so step i+1's copies in and step i-1's copies out overlap
    # step i's kernels (the copy engines and the SMs work side by side).
    h = inp.to_torch("cpu", pin_memory=True)
    # bytes crossing the link per step: the packed buffers (each tensor at a
    # 256-byte aligned offset, so a few hundred bytes of padding at most)
    h2d = packed({k: v for k, v in h.items() if v is not None})[0].numel()
    d2h = packed({"y": y, "fin": fin})[0].numel()
    e2e_serial_ms = max_over_ranks(e2e_serial(ssd, dev, h, y, fin, ws, cfg, args.steps), world, dev)
    e2e_ms = max_over_ranks(e2e_pipelined(ssd, dev, h, y, fin, ws, cfg, args.steps), world, dev)
    barrier()

    sweep = {}
    if not args.no_sweep and rank == 0:
        with ClockSampler(smi_gpu_id(local_rank)) as clk_sweep:
            sweep = run_sweep(ssd, dev, flush, peaks)
        sweep["clocks"] = clk_sweep.summary()

    if rank == 0:
        clocks = clk.summary()
        traffic = recorded_traffic(dom_name, cfg.name)
        line = {
            "metric": "ssd_fwd_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "batch": cfg.batch, "seqlen": cfg.seqlen, "nheads": cfg.nheads,
                       "headdim": cfg.headdim, "dstate": cfg.dstate, "ngroups": cfg.ngroups,
                       "chunk_size": cfg.chunk_size, "state_dtype": "f32", "y_dtype": "bf16",
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": "flushed between timed steps (512 MB write, outside the step events)"},
            "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps,
            "launches_per_step": launches_per_step,
            "launch_ms": {kernel_names[i] if i < len(kernel_names) else f"launch{i}": round(v, 5)
                          for i, v in enumerate(launch_ms)},
            "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "algorithmic_bytes": cbytes, "kernel_ms": launch_ms[dom],
                         "kernel_bytes": dom_bytes,
                         "kernel_bytes_frac": dom_bytes / (launch_ms[dom] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                         "peak_source": peaks["source"]},
            "op_roofline": {"compulsory_bytes": cbytes, "flops": chunked_flops(cfg, FWD_TILE),
                            "achieved_gbs": cbytes / (ms * 1e-3) / 1e9,
                            "frac_hbm": cbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                            "achieved_tflops": chunked_flops(cfg, FWD_TILE) / (ms * 1e-3) / 1e12},
            "e2e": {"value": job_tokens_per_s(tokens, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "mode": "pipelined (double-buffered, 3 streams)",
                    "serial_ms_per_step": e2e_serial_ms,
                    "serial_value": job_tokens_per_s(tokens, world, e2e_serial_ms)},
            "wall_s_timed_region": wall,
            "sm_count": nsm,
            "sweep": sweep,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(cfg, inp)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def packed(tensors, dev=None, pin=False):
    """One contiguous byte buffer holding `tensors` at 256-byte aligned
    offsets, and views of it with the tensors' dtypes and shapes: a step's
    inputs (or outputs) then cross the host link as one copy."""
    import torch
    offs, total = {}, 0
    for k, v in tensors.items():
        offs[k] = total
        total += -(-(v.numel() * v.element_size()) // 256) * 256
    buf = torch.empty(total, dtype=torch.uint8, device=dev, pin_memory=pin)
    views = {k: buf[o:o + v.numel() * v.element_size()].view(v.dtype).view(v.shape) for (k, v), o in
             zip(tensors.items(), offs.values())}
    return buf, views


def e2e_buffers(dev, h, y, fin, nsets):
    """Pinned host copies of the inputs and outputs, and `nsets` device sets,
    each packed into one buffer per direction."""
    src = {k: v for k, v in h.items() if v is not None}
    h_in, hv = packed(src, pin=True)
    for k, v in src.items():
        hv[k].copy_(v)
    d_in = [packed(src, dev=dev) for _ in range(nsets)]
    d_out = [packed({"y": y, "fin": fin}, dev=dev) for _ in range(nsets)]
    h_out = [packed({"y": y, "fin": fin}, pin=True)[0] for _ in range(nsets)]
    return h_in, d_in, d_out, h_out


def e2e_serial(ssd, dev, h, y, fin, ws, cfg, steps):
    """ms per step of copy in -> ssd_fwd -> copy out on one stream (one
    packed copy each way)."""
    import torch
    h_in, d_in, d_out, h_out = e2e_buffers(dev, h, y, fin, 1)
    (din, d), (dout, o), hout = d_in[0], d_out[0], h_out[0]
    stream = torch.cuda.current_stream(dev)

    def one():
        din.copy_(h_in, non_blocking=True)
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d.get("init_state"), cfg.chunk_size,
                    y=o["y"], final_state=o["fin"], workspace=ws)
        hout.copy_(dout, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps


def e2e_pipelined(ssd, dev, h, y, fin, ws, cfg, steps):
    """ms per step with two buffer sets: inputs of step i copied in on one
    stream while step i-1 computes on a second and step i-2's outputs go out
    on a third.  Every step still copies all its inputs in and its outputs
    out (one packed copy each way); the timed region runs from the first copy
    in to the last copy out."""
    import torch
    s_in, s_c, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    h_in, d_in, d_out, h_out = e2e_buffers(dev, h, y, fin, 2)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            j = i % 2
            (din, d), (dout, o) = d_in[j], d_out[j]
            if i >= 2:
                s_in.wait_event(ev_c[j])    # step i-2 no longer reads input set j
            with torch.cuda.stream(s_in):
                din.copy_(h_in, non_blocking=True)
                ev_in[j].record(s_in)
            s_c.wait_event(ev_in[j])
            if i >= 2:
                s_c.wait_event(ev_out[j])   # step i-2's outputs have been read back
            with torch.cuda.stream(s_c):
                ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d.get("init_state"), cfg.chunk_size,
                            y=o["y"], final_state=o["fin"], workspace=ws)
                ev_c[j].record(s_c)
            s_out.wait_event(ev_c[j])
            with torch.cuda.stream(s_out):
                h_out[j].copy_(dout, non_blocking=True)
                ev_out[j].record(s_out)

    run(3)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    run(steps)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps


def tc_plan(cfg, target_ctas=152):
    """Segment plan of the fused tensor-core path (mirrors the library):
    CTAs own 128/P heads; segments of consecutive 64-step tiles (a 128-step
    chunk is two of them) fill about one CTA per SM (target_ctas = the SM
    count)."""
    hb = 128 // cfg.headdim
    nhb = -(-cfg.nheads // hb)
    units = cfg.batch * nhb
    nc = -(-cfg.seqlen // 64)
    nseg = max(1, min(nc, target_ctas // units))
    cps = -(-nc // nseg)
    nseg = -(-nc // cps)
    return nseg, cps, nc


def tc_nsub(cfg, target_ctas=152):
    """Sub-segments of the segment-state pass (mirrors the library): halves
    wherever there are segments, S and two A buffers fit 256 TMEM columns
    (N + 128 <= 256) and a segment has two tiles or more."""
    nseg, cps, _ = tc_plan(cfg, target_ctas)
    return 2 if nseg > 1 and cfg.dstate + 128 <= 256 and cps >= 2 else 1


def KERNEL_BYTES(cfg, name):
    """Algorithmic bytes one launch of the named kernel must move."""
    b, L, H, P, N, G, Q = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups, cfg.chunk_size
    e = elem_bytes(cfg.dtype)
    nc = L // Q
    x = b * L * H * P * e
    dt = b * L * H * e
    bc = b * L * G * N * e
    st = b * nc * H * P * N * 4
    cum = b * H * L * 4
    y = b * L * H * P * Y_BYTES
    init = b * H * P * N * 4 if cfg.has_init else 0
    fin = b * H * P * N * 4
    nseg, cps, nt = tc_plan(cfg)
    nsub = tc_nsub(cfg)
    one_seg = b * H * P * N * 4  # one segment state of every (batch, head)
    seg_states = (nseg - 1) * nsub * one_seg
    # segment k's entering state combines the k nsub earlier local states
    seg_reads = one_seg * nsub * nseg * (nseg - 1) // 2
    covered = min(nt, (nseg - 1) * cps) / nt  # share of the sequence the segment-state kernel reads
    # chunk packs: the masked C B^T of each 64-step tile (bf16)
    pack = b * nt * G * 64 * 64 * 2
    return {
        "chunk_cumsum": dt + cum,
        "chunk_state_simt": x + dt + bc + cum + st,
        "state_passing": st + cum + init + st + fin,
        "chunk_scan_simt": x + dt + 2 * bc + cum + st + y,
        # fused tensor-core path: chunk packs (read B, C; write the masked
        # C B^T), segment-local states (written once), chunk scan (reads B, C
        # and every pack once per (batch, chunk, group), and the earlier
        # segments' local states and the initial state for the state entering
        # each segment)
        "cb_mask_tc": 2 * bc + pack,
        "seg_state_tc": covered * (x + dt + bc) + seg_states,
        "chunk_scan_tc": x + dt + 2 * bc + pack + seg_reads + nseg * init + y + fin,
    }.get(name, compulsory_bytes(cfg))


def run_sweep(ssd, dev, flush, peaks, steps=10):
    """Device-timed ssd_fwd on the other workloads, plus the sequential scan on
    the 16K-token one (the chunked-versus-sequential comparison)."""
    import torch
    out = {}
    for name in ("mamba2_2p7b", "long_16k", "wide_head", "wide_head_q128"):
        cfg = si.CONFIGS[name]
        inp = si.make_inputs(cfg)
        t = inp.to_torch(dev)
        y = torch.empty(t["x"].shape, device=dev, dtype=torch.bfloat16)
        fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), device=dev, dtype=torch.float32)
        ws = torch.empty(max(16, ssd.ssd_fwd_workspace_size(ssd.make_shape(t["x"], t["B"], cfg.chunk_size,
                                                                           torch.bfloat16))),
                         device=dev, dtype=torch.uint8)

        def run():
            ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"], cfg.chunk_size,
                        y=y, final_state=fin, workspace=ws)

        ms = time_device(run, flush, steps)
        cb = compulsory_bytes(cfg)
        kernels = kernel_times(ssd, run, flush, steps)
        dom = max(kernels, key=kernels.get)
        rec = {"tokens_per_s": cfg.tokens / (ms * 1e-3), "ms": ms,
               "frac_hbm": cb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
               "tflops": chunked_flops(cfg, FWD_TILE) / (ms * 1e-3) / 1e12,
               "tile_steps": FWD_TILE,
               "launch_ms": {k: round(v, 5) for k, v in kernels.items()},
               "dominant_kernel": dom,
               "dominant_kernel_frac_hbm": cb / (kernels[dom] * 1e-3) / 1e9 / peaks["hbm_gbs"],
               "dominant_kernel_traffic": recorded_traffic(dom, name)}
        if name == "long_16k":
            rec.update(sequential_scan(ssd, dev, flush, t, y, fin, cfg))
            rec["chunked_vs_sequential_speedup"] = rec["selective_scan_ms"] / ms
        out[name] = rec
        del t, y, fin, ws
        torch.cuda.empty_cache()
    out["stages"] = stage_sweep(ssd, dev, flush, peaks, steps)
    out["crossover"] = crossover_sweep(ssd, dev, flush, steps)
    out["decode"] = decode_sweep(ssd, dev, flush, peaks, steps)
    out["varlen"] = varlen_sweep(ssd, dev, flush, peaks, steps)
    return out


def sequential_scan(ssd, dev, flush, t, y, fin, cfg, steps=3):
    """selective_scan_fwd on resident inputs, against the measured FFMA peak."""
    def scan():
        ssd.selective_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"],
                               y=y, final_state=fin)
    sms = time_device(scan, flush, steps)
    scan_flops = 5.0 * cfg.tokens * cfg.nheads * cfg.headdim * cfg.dstate
    ffma = ffma_peak_tflops(dev)
    return {"selective_scan_ms": sms,
            "selective_scan_roofline": {
                "bound": "alu", "achieved": scan_flops / (sms * 1e-3) / 1e12, "peak": ffma, "unit": "TFLOP/s",
                "frac": scan_flops / (sms * 1e-3) / 1e12 / ffma,
                "flops": scan_flops, "flops_model": "5 fp32 flops per (token, head, p, n): decay, input, output",
                "peak_source": "measured: cuBLAS SGEMM 8192^3 with TF32 off (FFMA), best of 5"}}


def run_only(args):
    """One part of the sweep on its own (stage entry points on the 2.7B-shaped
    layer, the sequential scan on the 16K-token one, the chunked-vs-quadratic
    crossover, or the decode step), printed as one JSON line; its kernels are
    the only ones launched, which is what a profiler capture of them wants."""
    import torch
    import state_space_model_fwd_gb300 as ssd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES, device=dev, dtype=torch.uint8)
    peaks = load_peaks()
    steps = max(1, args.steps)
    if args.only == "stages":
        out = stage_sweep(ssd, dev, flush, peaks, steps)
    elif args.only == "sequential":
        cfg = si.CONFIGS["long_16k"]
        t = si.make_inputs(cfg).to_torch(dev)
        y = torch.empty(t["x"].shape, device=dev, dtype=torch.bfloat16)
        fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), device=dev, dtype=torch.float32)
        out = {"workload": cfg.name, **sequential_scan(ssd, dev, flush, t, y, fin, cfg, steps)}
    elif args.only == "crossover":
        out = crossover_sweep(ssd, dev, flush, steps)
    elif args.only == "varlen":
        out = varlen_sweep(ssd, dev, flush, peaks, steps)
    else:
        out = decode_sweep(ssd, dev, flush, peaks, steps)
    print(json.dumps({"only": args.only, **out}), flush=True)


def stage_sweep(ssd, dev, flush, peaks, steps):
    """The four stage entry points on the 2.7B-shaped layer, each timed per
    launch: the bandwidth-bound ones (chunk cumsum, state passing) against the
    HBM peak with the bytes each must move."""
    import torch
    cfg = si.CONFIGS["mamba2_2p7b"]
    t = si.make_inputs(cfg).to_torch(dev)
    b, L, H, P, N, Q = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.chunk_size
    nc = -(-L // Q)
    cum = torch.empty(b, H, nc, Q, device=dev)
    st = torch.empty(b, nc, H, P, N, device=dev)
    sin = torch.empty_like(st)
    fin = torch.empty(b, H, P, N, device=dev)
    y = torch.empty(t["x"].shape, device=dev, dtype=torch.bfloat16)
    calls = {
        "chunk_cumsum": lambda: ssd.ssd_chunk_cumsum(t["dt"], t["A"], Q, out=cum),
        "chunk_state": lambda: ssd.ssd_chunk_state(t["x"], t["dt"], t["B"], cum, out=st),
        "state_passing": lambda: ssd.ssd_state_passing(st, cum, t["init_state"], out=sin, final_state=fin),
        "chunk_scan": lambda: ssd.ssd_chunk_scan(t["x"], t["dt"], t["B"], t["C"], cum, sin, t["D"], out=y),
    }
    nbytes = {
        "chunk_cumsum": b * L * H * 2 + b * H * nc * Q * 4,
        "state_passing": 2 * st.numel() * 4 + b * H * nc * 4 + 2 * fin.numel() * 4,
    }
    rec = {"workload": "2.7B-shaped layer (b=2, L=4096, H=80, P=64, N=128, Q=64)"}
    for name, fn in calls.items():
        fn()
        kernels = kernel_times(ssd, fn, flush, steps)
        ms = sum(kernels.values())
        r = {"ms": ms, "launch_ms": {k: round(v, 5) for k, v in kernels.items()}}
        if name in nbytes:
            gbs = nbytes[name] / (ms * 1e-3) / 1e9
            r.update({"bytes": nbytes[name], "achieved_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]})
        rec[name] = r
    del st, sin
    torch.cuda.empty_cache()
    return rec


def crossover_sweep(ssd, dev, flush, steps):
    """Chunked (ssd_fwd) against the quadratic dual form (ssd_fwd_quadratic)
    on the 130M-shaped layer at short lengths: ms of each, per length."""
    import torch
    rows = []
    for L in (64, 128, 256, 512, 1024):
        cfg = si.CONFIGS[WORKLOAD].replace(seqlen=L)
        t = si.make_inputs(cfg).to_torch(dev)
        y = torch.empty(t["x"].shape, device=dev, dtype=torch.bfloat16)
        fin = torch.empty((cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate), device=dev, dtype=torch.float32)
        ws = torch.empty(max(16, ssd.ssd_fwd_workspace_size(ssd.make_shape(t["x"], t["B"], 64, torch.bfloat16))),
                         device=dev, dtype=torch.uint8)
        args = (t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["init_state"])
        chunked = time_graph(lambda: ssd.ssd_fwd(*args, 64, y=y, final_state=fin, workspace=ws), flush, steps)
        quad = time_graph(lambda: ssd.ssd_fwd_quadratic(*args, y=y, final_state=fin), flush, steps)
        rows.append({"seqlen": L, "tokens": cfg.tokens, "chunked_ms": chunked, "quadratic_ms": quad,
                     "faster": "quadratic" if quad < chunked else "chunked"})
    return {"workload": "130M-shaped layer (b=4, H=24, P=64, N=128, G=1), bf16 y",
            "timing": "CUDA graph of one call, replayed after an L2 flush; device events around the replay",
            "rows": rows}


def time_graph(fn, flush, steps):
    """Device time of fn captured in a CUDA graph (no host launch work inside
    the timed region), L2 flushed before every replay."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return time_device(g.replay, flush, steps)


VARLEN_MIXES = {
    # 8192 tokens of the 130M-shaped layer in each, like the b=4, L=2048 batch
    "ragged4": [3001, 1500, 2600, 1091],
    "short64": [100, 156] * 32,
    "long_and_short": [4096] + [128] * 32,
}


def varlen_sweep(ssd, dev, flush, peaks, steps):
    """ssd_fwd_varlen on packed batches of unequal lengths (130M-shaped
    layer, 8192 tokens, ragged last chunks), beside the equal-length batch
    of the same tokens: device time of the whole call (a CUDA graph, so the
    host's per-sequence launches are not in it)."""
    import torch
    base = si.CONFIGS[WORKLOAD]
    H, P, N, G = base.nheads, base.headdim, base.dstate, base.ngroups
    rows = {}
    for name, lens in VARLEN_MIXES.items():
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        cfg = base.replace(name="varlen_" + name, batch=1, seqlen=cu[-1], has_init=False)
        t = si.make_inputs(cfg).to_torch(dev)
        y = torch.empty(t["x"].shape, device=dev, dtype=torch.bfloat16)
        fins = torch.empty((len(lens), H, P, N), device=dev, dtype=torch.float32)
        shape = ssd.make_shape(t["x"], t["B"], base.chunk_size, torch.bfloat16)
        ws = torch.empty(max(16, ssd.ssd_fwd_varlen_workspace_size(shape, cu)), device=dev, dtype=torch.uint8)

        def run():
            ssd.ssd_fwd_varlen(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], None, cu, base.chunk_size,
                               y=y, final_states=fins, workspace=ws)

        ms = time_graph(run, flush, steps)
        # (warm, after an L2 flush; events between the launches, which
        # include the host's time before the first one)
        flush.zero_()
        ssd.launch_timing(True)
        run()
        torch.cuda.synchronize()
        launches = [[n, round(t_ms, 5)] for n, t_ms in ssd.launch_times_ms()]
        ssd.launch_timing(False)
        nbytes = (cu[-1] * H * P * 2 + cu[-1] * H * 2 + 2 * cu[-1] * G * N * 2 + 2 * H * 4
                  + cu[-1] * H * P * 2 + len(lens) * H * P * N * 4)
        rows[name] = {"nseq": len(lens), "tokens": cu[-1], "min_len": min(lens), "max_len": max(lens),
                      "launches": launches, "ms": ms, "tokens_per_s": cu[-1] / (ms * 1e-3), "bytes": nbytes,
                      "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        del t, y, fins, ws
    t = si.make_inputs(base).to_torch(dev)
    y = torch.empty(t["x"].shape, device=dev, dtype=torch.bfloat16)
    fin = torch.empty((base.batch, H, P, N), device=dev, dtype=torch.float32)
    ws = torch.empty(max(16, ssd.ssd_fwd_workspace_size(ssd.make_shape(t["x"], t["B"], base.chunk_size,
                                                                       torch.bfloat16))),
                     device=dev, dtype=torch.uint8)
    eq = time_graph(lambda: ssd.ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], None, base.chunk_size,
                                        y=y, final_state=fin, workspace=ws), flush, steps)
    torch.cuda.empty_cache()
    return {"workload": "130M-shaped layer (H=24, P=64, N=128, G=1), 8192 tokens packed, bf16 y, no initial state",
            "timing": "CUDA graph of one call, replayed after an L2 flush; device events around the replay",
            "equal_batch_ms": eq, "rows": rows}


def decode_sweep(ssd, dev, flush, peaks, steps):
    """One recurrent step of the 2.7B-shaped layer for a batch of 64
    sequences: the state (fp32) read and written once, bound by HBM."""
    import torch
    b, H, P, N, G = 64, 80, 64, 128, 1
    gen = torch.Generator(device=dev).manual_seed(5)
    x = torch.randn(b, H, P, device=dev, generator=gen).to(torch.bfloat16)
    dt = (0.05 * torch.rand(b, H, device=dev, generator=gen)).to(torch.bfloat16)
    A = -torch.rand(H, device=dev, generator=gen) * 4 - 1
    B = (torch.randn(b, G, N, device=dev, generator=gen) / N ** 0.5).to(torch.bfloat16)
    C = (torch.randn(b, G, N, device=dev, generator=gen) / N ** 0.5).to(torch.bfloat16)
    D = torch.randn(H, device=dev, generator=gen)
    state = 0.1 * torch.randn(b, H, P, N, device=dev, generator=gen)
    y = torch.empty(b, H, P, device=dev, dtype=torch.bfloat16)
    ms = time_device(lambda: ssd.ssd_decode_step(x, dt, A, B, C, D, state=state, y=y), flush, steps)
    nbytes = 2 * state.numel() * 4 + x.numel() * 2 + y.numel() * 2 + dt.numel() * 2 + 2 * B.numel() * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"2.7B-shaped layer, one token for {b} sequences (b={b}, H={H}, P={P}, N={N})",
            "ms": ms, "tokens_per_s": b / (ms * 1e-3), "bytes": nbytes, "achieved_gbs": gbs,
            "frac_hbm": gbs / peaks["hbm_gbs"]}


def kernel_times(ssd, fn, flush, steps):
    """Mean device time of each kernel launch of one call (library launch
    timing: events between the launches)."""
    import torch
    ssd.launch_timing(True)
    runs = []
    for _ in range(max(3, steps)):
        flush.zero_()
        fn()
        runs.append(ssd.launch_times_ms())
    ssd.launch_timing(False)
    torch.cuda.synchronize()
    names = [n for n, _ in runs[-1]]
    return {n: statistics.mean(r[i][1] for r in runs) for i, n in enumerate(names)}


def ffma_peak_tflops(dev):
    """FP32 FFMA throughput of this GPU, measured: cuBLAS SGEMM with TF32
    disabled runs on the FFMA pipes; best of 5 timed 8192^3 products."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        n = 8192
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        for _ in range(2):
            torch.matmul(a, b, out=c)
        best = None
        for _ in range(5):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            torch.matmul(a, b, out=c)
            e.record()
            e.synchronize()
            ms = s.elapsed_time(e)
            best = ms if best is None else min(best, ms)
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def time_device(fn, flush, steps):
    import torch
    for _ in range(3):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        e.synchronize()
        ts.append(s.elapsed_time(e))
    return statistics.mean(ts)


if __name__ == "__main__":
    main()
