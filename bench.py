#!/usr/bin/env python
"""Throughput of the uncertainty-tracked linear-attention scan hot path.

One step = one pass of the whole path over one batch of synthetic input,
inputs resident in HBM, through the C-ABI binding.  The default workload is
the long context (B=1, H=16, T=65536, d_k=d_v=128, bf16 inputs, fp32 state):
one kdn_diag_scan_fwd plus the standalone Moebius scan over 4096 sequences x
16384 steps (kdn_mobius_scan).  The same line carries, under "workloads", the
750M-shaped layer (8x16 heads, d=128, T=4096) and the 1.3B-shaped layer
(16x32 heads, d=64, T=4096), each timed the same way with one lambda sequence
per head computed in the scan's own launch (kdn_diag_mobius_scan_fwd).

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own batch
of the same shape on its own GPU (heads are independent: no data-path
collective; weak scaling); the timing is the max over ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
    python bench.py --workload layer750m_bwd   # the backward pass (training);
                                               # also layer1p3b_bwd, longctx_bwd,
                                               # heads32_t1024_bwd, heads16_t4096_bwd
                                               # (one wave each, for ncu)
    python bench.py --workload decode2k        # batched one-token decoding
    python bench.py --workload layer750m_lin   # the non-metaplastic limit; also
                                               # longctx_lin, heads128_t512_lin
    python bench.py --workload layer750m       # or layer1p3b, heads32_t2048_d64:
                                               # one scan workload (--no-extra: no
                                               # other workloads in the line)

Metric: scan tokens/s = B*H*T token-heads per second of the whole step.
Roofline of the dominant kernel (the diagonal scan): FP32 ALU bound,
10 FLOP per state element per token (I update 4, mean update 3, readout 3), peak =
SMs x 128 FP32 lanes x 2 FLOP x max SM clock.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "scan tokens/s (B·H·T per s) and % of binding HBM/FP32 roofline, fwd"
FP32_LANES_PER_SM = 128          # FP32 FMA lanes per SM (GB300)
SM_MAX_MHZ_FALLBACK = 2070.0     # maximum SM clock of GB300
HBM_GBS_FALLBACK = 6800.0
DIAG_FLOP_PER_ELEMENT_TOKEN = 10
MOBIUS_BYTES_PER_STEP = 20
# scan workloads whose numbers the default line carries besides its own
EXTRA_WORKLOADS = ("layer750m", "layer1p3b")
# dram__bytes_read.sum + dram__bytes_write.sum of one scan call (all its
# kernels: tensor-core aggregates, carry, full pass with the lambda walkers)
# per workload, from the ncu captures of the current kernels summarised in
# profiles/ (launches_*.md); workloads without such a capture report null.
DIAG_TRAFFIC_BYTES = {
    # aggregates + carry + full pass, read + write
    "longctx": (766_564_608 + 22_931_712) + (37_774_336 + 0) + (1_114_039_296 + 501_455_872),
    "layer750m": (350_242_304 + 68_923_392) + (100_699_648 + 36_041_728) + (647_612_160 + 244_894_464),
    "layer1p3b": 1_112_063_488 + 520_773_888,
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="longctx")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only --workload (by default the scan workloads' line also "
                         "carries the 750M- and 1.3B-shaped layers)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# ----------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.cmd = ["nvidia-smi", f"--id={gpu_id}", "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", "100"]
        self.proc = None

    def __enter__(self):
        self.first = []
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            # wait for two samples: nvidia-smi's start-up (NVML
            # initialisation) can hold up kernel launches of this process for
            # up to a few hundred ms, which must not fall inside the timed
            # region
            import select
            for _ in range(2):
                ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
                if not ready:
                    break
                line = self.proc.stdout.readline()
                if line.strip():
                    self.first.append(line)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in self.first + out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device_index]
        return str(device_index)


# ----------------------------------------------------------------------------
# distributed plumbing (barrier and max-over-ranks only; no data collective)

class Dist:
    def __init__(self, use_gpu: bool):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if use_gpu else "gloo"
            if use_gpu:
                import torch
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# CPU oracle arm (baseline leg and --impl reference)

def oracle_sample(w, inputs, n_heads: int, t_tokens: int):
    """Runs the fp64 oracle on the first n_heads heads (all rows) over the
    first t_tokens tokens, plus the Moebius scan of those heads' sequences
    (or of the same number of steps of the standalone sequences).
    Returns (seconds, token-heads processed, threads used)."""
    import oracle
    B, H = w.B, w.H
    heads = [(bh // H, bh % H) for bh in range(n_heads)]
    sl = lambda x: x.reshape(B * H, *x.shape[2:])[:n_heads, :t_tokens].unsqueeze(0)
    q, k, v, beta, d = (sl(inputs[n]) for n in ("q", "k", "v", "beta", "d"))
    A = inputs["A"][[h for _, h in heads]]
    # heads of the sample become the H axis of a B=1 batch, each with its own A
    steps = n_heads * t_tokens
    mN = min(w.mobius_N, max(1, steps // w.mobius_T)) if not w.mobius_fused else n_heads
    mT = w.mobius_T if not w.mobius_fused else t_tokens
    ma, mb, mc, md = (inputs[n][:mN, :mT] for n in ("ma", "mb", "mc", "md"))
    lam0 = inputs["lam0"][:mN]
    oracle.load()
    t0 = time.perf_counter()
    oracle.diag_scan(q, k, v, beta, d, A, inputs["I_prior"])
    oracle.mobius_scan(ma, mb, mc, md, lam0)
    dt = time.perf_counter() - t0
    return dt, n_heads * t_tokens, min(oracle.max_threads(), n_heads)


def oracle_single_core(n_heads: int = 4):
    """The oracle on one host core: the first n_heads heads of the 32-head,
    2048-token, d = 64 workload (all their 64x64 state rows, all tokens, their
    Moebius steps)."""
    import oracle
    from bayesian_scan_gb300 import workloads
    w1 = workloads.get("heads32_t2048_d64")
    inputs = workloads.make(w1)
    n = oracle.max_threads()
    oracle.set_threads(1)
    try:
        dt, units, _ = oracle_sample(w1, inputs, n_heads, w1.T)
    finally:
        oracle.set_threads(n)
    return {"workload": w1.name, "value": units / dt, "unit": "tokens/s", "cores": 1,
            "sample": f"{n_heads} heads x {w1.T} tokens, fp64 oracle, {dt:.2f} s"}


def calibrate_oracle(w, inputs, budget_s: float):
    """Pick (n_heads, t_tokens) so one oracle sample takes about budget_s on
    this host: whole sequences of as many heads as fit (a multiple of the
    thread count), or a prefix of the tokens when even one round is too long."""
    import oracle
    threads = oracle.max_threads()
    t_cal = min(w.T, 256)
    dt, _, _ = oracle_sample(w, inputs, 1, t_cal)
    per_token = dt / t_cal                       # one head, one thread
    affordable = budget_s * threads / max(per_token, 1e-12)   # token-heads
    total_heads = w.B * w.H
    if affordable >= threads * w.T:
        n_heads = int(affordable // w.T) // threads * threads
        return max(1, min(total_heads, n_heads)), w.T
    n_heads = min(total_heads, threads)
    return n_heads, max(16, min(w.T, int(affordable // n_heads)))


def run_reference(args, w, dist):
    """The reference arm: the fp64 CPU oracle as it stands, on host cores."""
    from bayesian_scan_gb300 import workloads
    if dist.rank != 0:
        return 0
    inputs = workloads.make(w)
    per_step_budget = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    n_heads, t_tokens = calibrate_oracle(w, inputs, per_step_budget)
    for _ in range(args.warmup):
        oracle_sample(w, inputs, n_heads, t_tokens)
    tot_t, tot_units, cores = 0.0, 0, 1
    for _ in range(args.steps):
        dt, units, cores = oracle_sample(w, inputs, n_heads, t_tokens)
        tot_t += dt
        tot_units += units
    value = tot_units / tot_t
    sample = (f"per step: {n_heads} heads x {t_tokens} tokens of the {w.name} workload "
              f"(all {w.dv}x{w.dk} state rows) + their Moebius steps, fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d_k": w.dk, "d_v": w.dv,
            "inputs": "bf16" if "bfloat16" in str(w.dtype) else "fp32", "state": "fp32",
            "mobius": f"{w.mobius_N}x{w.mobius_T} fp32" + (" (one per head)" if w.mobius_fused else ""),
            "l2": "inputs larger than the 129 MB L2, no flush"}


# ----------------------------------------------------------------------------
# our arm

def scan_numbers(args, w, dist, dev, K):
    """Times K steps of one scan workload on this rank (inputs resident in
    HBM, CUDA events on the launching stream, barrier + synchronize on both
    sides) and returns its numbers.  A step is one kdn_diag_mobius_scan_fwd
    call when the workload's lambda runs per head (the scan and lambda in one
    launch), else one kdn_diag_scan_fwd plus one kdn_mobius_scan of the
    standalone sequences."""
    import torch

    from bayesian_scan_gb300 import kdn, workloads

    # every rank draws its own batch of the same shape (weak scaling)
    w_rank = w if dist.rank == 0 else type(w)(**{**w.__dict__, "seed": w.seed + 7919 * dist.rank})
    host = workloads.make(w_rank)
    names = ("q", "k", "v", "beta", "d", "A")
    mnames = ("ma", "mb", "mc", "md", "lam0")
    x = {n: host[n].to(dev) for n in names + mnames}
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    o_buf = torch.empty(B, H, T, dv, device=dev)
    fs_buf = torch.empty(2, B, H, dv, dk, device=dev)
    lam_buf = torch.empty(w.mobius_N, w.mobius_T, device=dev)
    stream = torch.cuda.current_stream(dev)
    fused = w.mobius_fused

    def diag():
        if fused:
            kdn.diag_mobius_scan_fwd(*(x[n] for n in names + mnames), I_prior=w.I_prior, out=o_buf,
                                     final_state=fs_buf, lambda_out=lam_buf, stream=stream)
        else:
            kdn.diag_scan_fwd(*(x[n] for n in names), I_prior=w.I_prior, out=o_buf,
                              final_state=fs_buf, stream=stream)

    def mobius():
        if not fused:
            kdn.mobius_scan(*(x[n] for n in mnames), out=lam_buf, stream=stream)

    plan = kdn.diag_scan_plan(B, H, T, dk, dv, w.dtype)
    mplan = kdn.mobius_scan_plan(w.mobius_N, w.mobius_T)
    for _ in range(args.warmup):
        diag()
        mobius()
    torch.cuda.synchronize(dev)
    st = kdn.get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error after warm-up: {kdn.status_string(st)}")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for(dist.local_rank))
    dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        start.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            diag()
            ev[i][1].record(stream)
            mobius()
            ev[i][2].record(stream)
        stop.record(stream)
        torch.cuda.synchronize(dev)
    dist.barrier()
    st = kdn.get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {kdn.status_string(st)}")
    total_ms = start.elapsed_time(stop)
    diag_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / K
    mob_ms = sum(b.elapsed_time(c) for _, b, c in ev) / K
    max_ms = dist.max(total_ms)
    tokens = B * H * T

    peaks = measured_peaks()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", SM_MAX_MHZ_FALLBACK))
    alu_peak = nsm * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12    # TFLOP/s
    flop = DIAG_FLOP_PER_ELEMENT_TOKEN * dv * dk * tokens
    achieved = flop / (diag_ms / 1e3) / 1e12
    hbm_peak = float(peaks.get("hbm_gbs", HBM_GBS_FALLBACK))
    mbytes = MOBIUS_BYTES_PER_STEP * w.mobius_N * w.mobius_T
    peak_src = f"{nsm} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {sm_max:.0f} MHz (recipe unit counts and max SM clock)"
    kernel = ("diag_scan_kernel with the per-head lambda walkers (whole kdn_diag_mobius_scan_fwd call)"
              if fused else "diag_scan_kernel (whole kdn_diag_scan_fwd call)")
    res = {
        "value": dist.world * tokens * K / (max_ms / 1e3), "ms_per_step": max_ms / K,
        "roofline": {"kernel": kernel, "bound": "alu", "achieved": achieved, "peak": alu_peak,
                     "unit": "TFLOP/s", "frac": achieved / alu_peak,
                     "traffic": DIAG_TRAFFIC_BYTES.get(w.name), "peak_source": peak_src,
                     "ms_per_call": diag_ms, "token_parts": plan["parts"]},
        "gpu_launches": K * (plan["kernels"] + (0 if fused else mplan["kernels"])),
        "clocks": sampler.summary(),
    }
    if fused:
        # lambda graded inside the scan's launch: the launch's roofline time is
        # max(FLOP / FP32 peak, all its bytes / HBM peak), its bytes the scan's
        # plus lambda's 20 per step
        es = 2 if w.dtype == torch.bfloat16 else 4
        scan_bytes = tokens * ((2 * dk + 2 * dv + 1) * es + 4 * dv) + 2 * B * H * dv * dk * 4
        t_roof = max(flop / (alu_peak * 1e12), (scan_bytes + mbytes) / (hbm_peak * 1e9))
        res["mobius_roofline"] = {
            "fused": True, "bound": "alu (lambda runs inside the scan launch)",
            "lambda_bytes": mbytes, "launch_bytes": scan_bytes + mbytes,
            "roofline_ms": t_roof * 1e3, "frac": t_roof / (diag_ms / 1e3), "ms_per_call": diag_ms,
            "peak_source": ("measured" if "hbm_gbs" in peaks else "fallback") + " HBM; FP32 as roofline"}
    else:
        mob_gbs = mbytes / (mob_ms / 1e3) / 1e9
        res["mobius_roofline"] = {"bound": "hbm", "achieved": mob_gbs, "peak": hbm_peak, "unit": "GB/s",
                                  "frac": mob_gbs / hbm_peak, "ms_per_call": mob_ms,
                                  "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"}
    del x, o_buf, fs_buf, lam_buf
    return res, host


def run_ours(args, w, dist):
    import torch

    from bayesian_scan_gb300 import workloads

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    K = args.steps
    res, host = scan_numbers(args, w, dist, dev, K)
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    line = {
        "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w),
        "roofline": res["roofline"], "mobius_roofline": res["mobius_roofline"],
        "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
    }
    if not args.no_e2e:
        line["e2e"] = measure_e2e(args, w, host, dev, dist)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        n_heads, t_tokens = calibrate_oracle(w, host, 12.0)
        dt, units, cores = oracle_sample(w, host, n_heads, t_tokens)
        line["cpu_baseline"] = {
            "value": units / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_heads} heads x {t_tokens} tokens of the same inputs (all "
                      f"{dv}x{dk} state rows) + their Moebius steps, fp64 oracle, {dt:.1f} s",
            "single_core": oracle_single_core()}
    del host
    # the other layer configurations of the same metric, timed the same way
    # in the same run (a step each: one fused scan + lambda launch)
    extra = [] if args.no_extra else [n for n in EXTRA_WORKLOADS if n != w.name]
    if extra:
        line["workloads"] = {}
        for name in extra:
            we = workloads.get(name)
            torch.cuda.empty_cache()
            r, _ = scan_numbers(args, we, dist, dev, K)
            r["config"] = workload_config(we)
            line["workloads"][name] = r
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_decode(args, w, dist):
    """Batched decoding: each step is one kdn_diag_step over all B x H heads
    (one token each) on a device-resident state larger than L2; `value` is
    token-heads per second, the roofline HBM (16 bytes of state per element
    plus the token's inputs and outputs)."""
    import torch

    from bayesian_scan_gb300 import kdn, workloads
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    w_rank = w if dist.rank == 0 else type(w)(**{**w.__dict__, "seed": w.seed + 7919 * dist.rank})
    host = workloads.make(w_rank, with_mobius=False)
    names = ("q", "k", "v", "beta", "d")
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    # contiguous per-token inputs [B,H,...] for T successive steps
    tok = [{n: host[n][:, :, t].contiguous().to(dev) for n in names} for t in range(T)]
    A = host["A"].to(dev)
    state = torch.stack([torch.zeros(B, H, dv, dk), torch.full((B, H, dv, dk), w.I_prior)]).to(dev)
    out = torch.empty(B, H, dv, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        x = tok[i % T]
        kdn.diag_step(*(x[n] for n in names), A, state, I_prior=w.I_prior, out=out, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    K = args.steps
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for(dist.local_rank))
    dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        start.record(stream)
        for i in range(K):
            step(i)
        stop.record(stream)
        torch.cuda.synchronize(dev)
    dist.barrier()
    st = kdn.get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {kdn.status_string(st)}")
    ms = start.elapsed_time(stop)
    max_ms = dist.max(ms)
    heads = B * H
    value = dist.world * heads * K / (max_ms / 1e3)
    es = 2 if w.dtype == torch.bfloat16 else 4
    step_bytes = heads * dv * dk * 16 + heads * (2 * dk + 2 * dv + 1) * es + heads * dv * 4
    gbs = step_bytes / (ms / K / 1e3) / 1e9
    peaks = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", HBM_GBS_FALLBACK))
    line = {
        "metric": "decode token-heads/s (one kdn_diag_step over B x H heads per step)",
        "value": value, "unit": "token-heads/s", "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": max_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "d_k": dk, "d_v": dv,
                   "inputs": "bf16" if es == 2 else "fp32", "state": "fp32, device resident, "
                   f"{2 * heads * dv * dk * 4 / 1e6:.0f} MB (larger than the 129 MB L2, no flush)"},
        "roofline": {"kernel": "diag_step_kernel", "bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                     "unit": "GB/s", "frac": gbs / hbm_peak, "traffic": None,
                     "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"},
        "gpu_launches": K,
        "clocks": sampler.summary(),
    }
    if not args.no_e2e:
        # each step: the token's inputs from page-locked host memory, the step,
        # the outputs back (the state stays on the device)
        pin = [{n: host[n][:, :, t].contiguous().pin_memory() for n in names} for t in range(T)]
        out_h = torch.empty(B, H, dv).pin_memory()
        xs = {n: torch.empty_like(tok[0][n]) for n in names}

        def e2e_step(i):
            for n in names:
                xs[n].copy_(pin[i % T][n], non_blocking=True)
            kdn.diag_step(*(xs[n] for n in names), A, state, I_prior=w.I_prior, out=out, stream=stream)
            out_h.copy_(out, non_blocking=True)

        e2e_step(0)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(K):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        dt = dist.max(time.perf_counter() - t0)
        line["e2e"] = {"value": dist.world * heads * K / dt, "unit": "token-heads/s", "steps": K,
                       "h2d_bytes_per_step": heads * (2 * dk + 2 * dv + 1) * es,
                       "d2h_bytes_per_step": heads * dv * 4,
                       "path": "page-locked token inputs -> device copies -> kdn.diag_step -> "
                               "page-locked output (state device resident)"}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        import oracle
        n_heads = min(heads, 64)
        sl = lambda x: x.reshape(B * H, *x.shape[2:])[:n_heads].reshape(1, n_heads, *x.shape[2:])
        args_o = [sl(host[n][:, :, :1]) for n in names]
        A_o = host["A"].repeat(B)[:n_heads].contiguous()
        I0 = torch.full((1, n_heads, dv, dk), w.I_prior)
        mu0 = torch.zeros(1, n_heads, dv, dk)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 5.0:
            oracle.diag_scan(*args_o, A_o, w.I_prior, I0, mu0)
            reps += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": reps * n_heads / dt, "unit": "token-heads/s",
                                "cores": oracle.max_threads(), "kind": "oracle",
                                "sample": f"{reps} one-token oracle steps over {n_heads} heads "
                                          f"({dv}x{dk} state rows), fp64, {dt:.1f} s"}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def measure_e2e(args, w, host, dev, dist):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory, runs both scans and reads the results
    back (o, final state, lambda)."""
    import torch

    from bayesian_scan_gb300 import kdn
    names = ("q", "k", "v", "beta", "d", "A")
    mnames = ("ma", "mb", "mc", "md", "lam0")
    pinned = {n: host[n].pin_memory() for n in names + mnames}
    K = max(3, min(args.steps, 20))
    h2d = sum(pinned[n].numel() * pinned[n].element_size() for n in names + mnames)
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    d2h = 4 * (B * H * T * dv + 2 * B * H * dv * dk + w.mobius_N * w.mobius_T)

    # page-locked result buffers, reused by every step (the call writes them)
    out_h = torch.empty(B, H, T, dv, dtype=torch.float32, pin_memory=True)
    fs_h = torch.empty(2, B, H, dv, dk, dtype=torch.float32, pin_memory=True)
    lam_h = torch.empty(w.mobius_N, w.mobius_T, dtype=torch.float32, pin_memory=True)

    def step():
        kdn.diag_scan_fwd(*(pinned[n] for n in names), I_prior=w.I_prior, out=out_h, final_state=fs_h)
        kdn.mobius_scan(*(pinned[n] for n in mnames), out=lam_h)

    step()   # warm-up (allocator, pinned staging)
    dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    torch.cuda.synchronize(dev)
    dt = dist.max(time.perf_counter() - t0)
    dist.barrier()
    return {"value": dist.world * B * H * T * K / dt, "unit": "tokens/s", "steps": K,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "kdn.diag_scan_fwd / kdn.mobius_scan on page-locked host tensors -> "
                    "kdn_diag_scan_fwd_host / kdn_mobius_scan_host (pipelined H2D, kernels, D2H; sync)"}


# backward: per state element and token, the adjoint step and the gradient
# sums (24 FLOP) plus one evaluation of the forward state it needs (6 FLOP);
# the kernel's second evaluation of the forward (checkpoint replay) is not
# counted
BWD_FLOP_PER_ELEMENT_TOKEN = 30


def bwd_inputs(w, dev):
    import torch

    from bayesian_scan_gb300 import workloads
    host = workloads.make(w, with_mobius=False)
    gout, _ = workloads.draw_cotangents(w.B, w.H, w.T, w.dk, w.dv, seed=w.seed + 1)
    host["gout"] = gout
    return host


def oracle_bwd_sample(w, host, n_heads: int, t_tokens: int):
    """The fp64 reverse-mode oracle on the first n_heads heads over the first
    t_tokens tokens.  Returns (seconds, token-heads, threads)."""
    import oracle
    B, H = w.B, w.H
    sl = lambda x: x.reshape(B * H, *x.shape[2:])[:n_heads, :t_tokens].unsqueeze(0)
    q, k, v, beta, d, gout = (sl(host[n]) for n in ("q", "k", "v", "beta", "d", "gout"))
    A = host["A"].repeat(B)[:n_heads].contiguous()
    oracle.load()
    t0 = time.perf_counter()
    oracle.diag_scan_bwd(q, k, v, beta, d, A, host["I_prior"], dout=gout)
    return time.perf_counter() - t0, n_heads * t_tokens, min(oracle.max_threads(), n_heads)


def calibrate_oracle_bwd(w, host, budget_s: float):
    import oracle
    threads = oracle.max_threads()
    dt, _, _ = oracle_bwd_sample(w, host, 1, 64)
    per_token = dt / 64
    n_heads = min(w.B * w.H, threads)
    # every state of a sampled head is kept: bound the sample's memory to ~2 GB
    mem_tokens = int(2e9 / (16 * w.dv * w.dk * n_heads))
    t = int(budget_s / max(per_token, 1e-12))
    return n_heads, max(16, min(w.T, t, mem_tokens))


def run_backward(args, w, dist):
    """Training step of the scan: one kdn_diag_scan_bwd over the workload
    (the gradient flowing into the outputs given, no final-state gradient);
    `value` is token-heads per second, the roofline the FP32 ALUs."""
    import torch

    from bayesian_scan_gb300 import kdn
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    w_rank = w if dist.rank == 0 else type(w)(**{**w.__dict__, "seed": w.seed + 7919 * dist.rank})
    host = bwd_inputs(w_rank, dev)
    names = ("q", "k", "v", "beta", "d", "A")
    x = {n: host[n].to(dev) for n in names + ("gout",)}
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    stream = torch.cuda.current_stream(dev)
    ws = torch.empty(kdn.diag_scan_bwd_workspace(B, H, T, dk, dv), device=dev, dtype=torch.uint8)

    def step():
        return kdn.diag_scan_bwd(*(x[n] for n in names), x["gout"], I_prior=w.I_prior,
                                 grad_init_state=False, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = kdn.get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error after warm-up: {kdn.status_string(st)}")
    K = args.steps
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for(dist.local_rank))
    dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        start.record(stream)
        for _ in range(K):
            step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
    dist.barrier()
    st = kdn.get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {kdn.status_string(st)}")
    ms = start.elapsed_time(stop)
    max_ms = dist.max(ms)
    tokens = B * H * T
    value = dist.world * tokens * K / (max_ms / 1e3)
    peaks = measured_peaks()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", SM_MAX_MHZ_FALLBACK))
    alu_peak = nsm * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    achieved = BWD_FLOP_PER_ELEMENT_TOKEN * dv * dk * tokens / (ms / K / 1e3) / 1e12
    es = 2 if w.dtype == torch.bfloat16 else 4
    line = {
        "metric": "scan backward tokens/s (B·H·T per s) and % of FP32 roofline",
        "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": max_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "T": T, "d_k": dk, "d_v": dv,
                   "inputs": "bf16" if es == 2 else "fp32", "grad_out": "fp32 N(0,1)",
                   "grad_final_state": "none", "l2": "inputs larger than the 129 MB L2, no flush"},
        "roofline": {"kernel": "diag_bwd_kernel (whole kdn_diag_scan_bwd call)", "bound": "alu",
                     "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                     "frac": achieved / alu_peak, "traffic": None,
                     "flop_per_element_token": BWD_FLOP_PER_ELEMENT_TOKEN,
                     "peak_source": f"{nsm} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {sm_max:.0f} MHz"
                                    " (recipe unit counts and max SM clock)"},
        "gpu_launches": 3 * K,
        "clocks": sampler.summary(),
    }
    if not args.no_e2e:
        pin = {n: host[n].pin_memory() for n in names + ("gout",)}
        xs = {n: torch.empty_like(x[n]) for n in names + ("gout",)}
        outs = {"q": (B, H, T, dk), "k": (B, H, T, dk), "v": (B, H, T, dv), "beta": (B, H, T, dv),
                "d": (B, H, T), "A": (H,)}
        res = {n: torch.empty(shp).pin_memory() for n, shp in outs.items()}

        def e2e_step():
            for n in xs:
                xs[n].copy_(pin[n], non_blocking=True)
            g = kdn.diag_scan_bwd(*(xs[n] for n in names), xs["gout"], I_prior=w.I_prior,
                                  grad_init_state=False, workspace=ws, stream=stream)
            for n in res:
                res[n].copy_(g[n], non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(1, min(K, 5))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize(dev)
        dt = dist.max(time.perf_counter() - t0)
        line["e2e"] = {"value": dist.world * tokens * n_e2e / dt, "unit": "tokens/s", "steps": n_e2e,
                       "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values()),
                       "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in res.values()),
                       "path": "page-locked inputs and output gradient -> device copies -> "
                               "kdn.diag_scan_bwd -> page-locked gradients"}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        n_heads, t_tokens = calibrate_oracle_bwd(w, host, 10.0)
        dt, units, reps, cores = 0.0, 0, 0, 1
        while dt < 10.0 and reps < 100:
            d1, u1, cores = oracle_bwd_sample(w, host, n_heads, t_tokens)
            dt, units, reps = dt + d1, units + u1, reps + 1
        line["cpu_baseline"] = {
            "value": units / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x ({n_heads} heads x {t_tokens} tokens) of the same inputs (all "
                      f"{dv}x{dk} state rows), fp64 reverse-mode oracle, {dt:.1f} s"}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# non-metaplastic limit: per state element and token one FMA for the write
# (in the scaled form Ew += (W beta_i v_i) k_j) and one for the readout
LIN_FLOP_PER_ELEMENT_TOKEN = 4


def run_lin(args, w, dist):
    """The non-metaplastic scan (kdn_lin_scan_fwd) over the workload; `value`
    is token-heads per second, the roofline the FP32 ALUs."""
    import torch

    from bayesian_scan_gb300 import kdn, workloads
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    w_rank = w if dist.rank == 0 else type(w)(**{**w.__dict__, "seed": w.seed + 7919 * dist.rank})
    host = workloads.make(w_rank, with_mobius=False)
    names = ("q", "k", "v", "beta", "d", "A")
    x = {n: host[n].to(dev) for n in names}
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    out = torch.empty(B, H, T, dv, device=dev)
    fmu = torch.empty(B, H, dv, dk, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kdn.lin_scan_fwd(*(x[n] for n in names), I_prior=w.I_prior, out=out, final_mu=fmu,
                         stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for(dist.local_rank))
    dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        start.record(stream)
        for _ in range(K):
            step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
    dist.barrier()
    st = kdn.get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {kdn.status_string(st)}")
    ms = start.elapsed_time(stop)
    max_ms = dist.max(ms)
    tokens = B * H * T
    value = dist.world * tokens * K / (max_ms / 1e3)
    peaks = measured_peaks()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", SM_MAX_MHZ_FALLBACK))
    alu_peak = nsm * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    achieved = LIN_FLOP_PER_ELEMENT_TOKEN * dv * dk * tokens / (ms / K / 1e3) / 1e12
    plan = kdn.diag_scan_plan(B, H, T, dk, dv, w.dtype)
    es = 2 if w.dtype == torch.bfloat16 else 4
    tc_path = dk == 128 and dv == 128 and es == 2
    if tc_path:
        # chunked tensor-core kernel: its speed of light is HBM (inputs in,
        # outputs and the final mean out); its FP32 work is small
        step_bytes = tokens * ((2 * dk + 2 * dv + 1) * es + dv * 4) + B * H * dv * dk * 4
        gbs = step_bytes / (ms / K / 1e3) / 1e9
        hbm_peak = float(peaks.get("hbm_gbs", HBM_GBS_FALLBACK))
        roof = {"kernel": "lin_tc_kernel (whole kdn_lin_scan_fwd call)", "bound": "hbm",
                "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                "traffic": None, "bytes_per_step": step_bytes,
                "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
                "fp32_equivalent": {"achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                                    "flop_per_element_token": LIN_FLOP_PER_ELEMENT_TOKEN}}
    else:
        roof = {"kernel": "diag_scan_kernel<..., LIN> (whole kdn_lin_scan_fwd call)",
                "bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": achieved / alu_peak, "traffic": None,
                "flop_per_element_token": LIN_FLOP_PER_ELEMENT_TOKEN,
                "peak_source": f"{nsm} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {sm_max:.0f} MHz"
                               " (recipe unit counts and max SM clock)"}
    line = {
        "metric": "non-metaplastic scan tokens/s (B·H·T per s) and % of binding roofline, fwd",
        "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": K,
        "warmup": args.warmup, "ms_per_step": max_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "T": T, "d_k": dk, "d_v": dv,
                   "inputs": "bf16" if es == 2 else "fp32",
                   "state": "fp32 mu (importance held at I_prior)",
                   "l2": "inputs larger than the 129 MB L2, no flush"},
        "roofline": roof,
        "gpu_launches": K * plan["kernels"],
        "clocks": sampler.summary(),
    }
    if not args.no_e2e:
        pin = {n: host[n].pin_memory() for n in names}
        xs = {n: torch.empty_like(x[n]) for n in names}
        out_h = torch.empty(B, H, T, dv).pin_memory()

        def e2e_step():
            for n in names:
                xs[n].copy_(pin[n], non_blocking=True)
            kdn.lin_scan_fwd(*(xs[n] for n in names), I_prior=w.I_prior, out=out, final_mu=fmu,
                             stream=stream)
            out_h.copy_(out, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(1, min(K, 20))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize(dev)
        dt = dist.max(time.perf_counter() - t0)
        line["e2e"] = {"value": dist.world * tokens * n_e2e / dt, "unit": "tokens/s", "steps": n_e2e,
                       "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values()),
                       "d2h_bytes_per_step": out_h.numel() * 4,
                       "path": "page-locked inputs -> device copies -> kdn.lin_scan_fwd -> "
                               "page-locked output"}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        import oracle
        n_heads = min(B * H, oracle.max_threads())
        sl = lambda t_: t_.reshape(B * H, *t_.shape[2:])[:n_heads].unsqueeze(0)
        args_o = [sl(host[n]) for n in ("q", "k", "v", "beta", "d")]
        A_o = host["A"].repeat(B)[:n_heads].contiguous()
        t_tok = T
        t0 = time.perf_counter()
        oracle.lin_scan(*(a_[:, :, :64] for a_ in args_o), A_o, w.I_prior)
        per_tok = (time.perf_counter() - t0) / 64
        t_tok = max(64, min(T, int(10.0 / max(per_tok, 1e-9))))
        dt, reps = 0.0, 0
        while dt < 10.0 and reps < 100:
            t0 = time.perf_counter()
            oracle.lin_scan(*(a_[:, :, :t_tok] for a_ in args_o), A_o, w.I_prior)
            dt += time.perf_counter() - t0
            reps += 1
        line["cpu_baseline"] = {"value": reps * n_heads * t_tok / dt, "unit": "tokens/s",
                                "cores": n_heads, "kind": "oracle",
                                "sample": f"{reps} x ({n_heads} heads x {t_tok} tokens) of the same "
                                          f"inputs (all {dv}x{dk} state rows), fp64 oracle, {dt:.1f} s"}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_reference_bwd(args, w, dist):
    """Reference arm of the backward workload: the fp64 reverse-mode oracle."""
    if dist.rank != 0:
        return 0
    host = bwd_inputs(w, None)
    per_step = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    n_heads, t_tokens = calibrate_oracle_bwd(w, host, per_step)
    for _ in range(args.warmup):
        oracle_bwd_sample(w, host, n_heads, t_tokens)
    tot_t, tot_units, cores = 0.0, 0, 1
    for _ in range(args.steps):
        dt, units, cores = oracle_bwd_sample(w, host, n_heads, t_tokens)
        tot_t += dt
        tot_units += units
    value = tot_units / tot_t
    sample = (f"per step: {n_heads} heads x {t_tokens} tokens of the {w.name} workload "
              f"(all {w.dv}x{w.dk} state rows), fp64 reverse-mode oracle")
    print(json.dumps({
        "impl": "reference", "metric": "scan backward tokens/s (B·H·T per s) and % of FP32 roofline",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d_k": w.dk, "d_v": w.dv},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def main():
    args = parse_args()
    from bayesian_scan_gb300 import workloads
    w = workloads.get(args.workload)
    dist = Dist(use_gpu=args.impl == "ours")
    try:
        if w.name in workloads.DECODE:
            if args.impl == "reference":
                if dist.rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the "
                                      "oracle on the scan workloads; decode steps are timed by our arm's "
                                      "cpu_baseline"}), flush=True)
                return 0
            return run_decode(args, w, dist)
        if w.name in workloads.LIN:
            if args.impl == "reference":
                if dist.rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the "
                                      "oracle on the metaplastic scan workloads; the non-metaplastic "
                                      "scan's oracle is timed by our arm's cpu_baseline"}), flush=True)
                return 0
            return run_lin(args, w, dist)
        if w.name in workloads.TRAIN:
            if args.impl == "reference":
                return run_reference_bwd(args, w, dist)
            return run_backward(args, w, dist)
        if args.impl == "reference":
            return run_reference(args, w, dist)
        return run_ours(args, w, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
