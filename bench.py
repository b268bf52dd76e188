#!/usr/bin/env python
"""Benchmark: packed tokens/s of varlen conv1d + selective scan, forward + backward.

One step = the whole hot path on one pack batch, through the C ABI:
position indices -> conv1d fwd -> selective scan fwd -> selective scan bwd ->
conv1d bwd (each call includes its fixed-order reductions).  Default workload:
the Mamba-1.4B layer shape (D=4096, N=16, W=4, bf16 I/O, fp32 state), 8 packs
of 4096 tokens with log-normal lengths (median 800), seeded synthetic data.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU ("replicas only": the path has no cross-GPU exchange); value =
tokens of all ranks / the slowest rank's time.  `--impl reference` times the
double-precision CPU oracle (the only reference this method has) on the host
cores, on a bounded channel sample of the same workload.

Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "packed tokens/s for varlen conv1d+selective scan fwd+bwd; % of roofline"

# Algorithmic per-token counts of each stage (bytes moved, FP32-pipe ops with
# FMA = 1, MUFU ops), e = bytes per I/O element, as the path's scope defines
# them: the forward reads u, delta_raw, z and writes out; the backward reads
# u, delta_raw, z, dout and writes du, d delta_raw, dz; the backward's FP32
# count is 13 D N + 24 D (the state recompute, the reverse recurrence, the
# four channel / state sums and the C.h of y).  The roofline fractions use
# these.
def per_token_counts(D, N, e, W=4):
    return {
        "conv_fwd": dict(bytes=2 * e * D + 4, fp32=(W + 3) * D, mufu=2 * D),
        "scan_fwd": dict(bytes=4 * e * D + 2 * e * N + 4, fp32=4 * D * N + 10 * D, mufu=D * N + 4 * D),
        "scan_bwd": dict(bytes=7 * e * D + 2 * e * N + 8 * N + 4, fp32=13 * D * N + 24 * D, mufu=D * N + 6 * D),
        "conv_bwd": dict(bytes=3 * e * D + 4, fp32=(3 * W + 6) * D, mufu=2 * D),
    }


# What this implementation moves on top of those counts, per token: the
# forward also writes its pre-gate output y (e D bytes) and the backward reads
# it for dz instead of recomputing C.h (e D bytes, and D N fewer FP32 ops).
def implementation_extra_bytes(D, e):
    return {"scan_fwd": e * D, "scan_bwd": e * D}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the latest
# ncu capture of a kernel, per token, with the kernel it was taken on; the
# line reports it only for that kernel.
LAST_CAPTURE_TRAFFIC = {
    ("m14b", "scan_bwd"): {"bytes_per_token": (411.232768e6 + 444.166912e6) / 8192,
                           "kernel": "scan_bwd16_kernel",
                           "source": "ncu --set full capture of scan_bwd16_kernel on m14b_small (T=8192), "
                                     "scaled by tokens"},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="m14b")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-comparators", action="store_true",
                   help="skip the no-reset concat bound and the packed-vs-padded comparison")
    p.add_argument("--comparator-steps", type=int, default=10)
    p.add_argument("--comparator-d", type=int, default=4096,
                   help="channels for the packed-vs-padded comparison (the long-tail workload's width)")
    p.add_argument("--no-configs", action="store_true",
                   help="skip timing the other workloads (m130m and m14b_fwd forward, long-tail fwd+bwd)")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target wall time of the CPU-oracle baseline sample")
    p.add_argument("--clock-log", default=None,
                   help="file for the nvidia-smi clock samples of the timed region ({rank} is replaced); "
                        "default: a temporary file")
    return p.parse_args(argv)


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate(tokens_per_rank: int, seconds: float, world: int, device=None) -> tuple[float, float]:
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    t = max_over_ranks(seconds, device)
    return tokens_per_rank * world / t, t


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None):
        self.gpu = gpu_index
        self.path = path
        self.proc = None
        self.fh = None

    def start(self):
        if not self.path:
            return
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        return parse_clocks(open(self.path).read())


def parse_clocks(text: str):
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
            "reasons": sorted(reasons)}


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(w, r, channels, threads=None):
    """Runs the oracle's conv1d fwd -> scan fwd -> scan bwd -> conv1d bwd on a
    column sample of the workload; returns (seconds, threads)."""
    import numpy as np
    import oracle
    idx = np.arange(channels)
    col = lambda a: np.ascontiguousarray(a[:, idx], dtype=np.float64)  # noqa: E731
    cu = w["cu_seqlens"]
    threads = threads or oracle.default_threads()
    x, dr, z, dout = col(r["x"]), col(r["delta_raw"]), col(r["z"]), col(r["dout"])
    B, C = np.asarray(r["B"], np.float64), np.asarray(r["C"], np.float64)
    A, Dk, dtb = r["A"][idx], r["Dskip"][idx], r["dt_bias"][idx]
    cw, cb = r["conv_w"][idx], r["conv_b"][idx]
    t0 = time.perf_counter()
    u = oracle.conv1d_fwd_threaded(x, cw, cb, cu, threads=threads)
    oracle.scan_fwd_threaded(u, dr, A, B, C, Dk, z, dtb, cu, threads=threads)
    g = oracle.scan_bwd_threaded(u, dr, A, B, C, Dk, z, dtb, dout, cu, threads=threads)
    oracle.conv1d_bwd_threaded(x, cw, cb, g["du"], cu, threads=threads)
    return time.perf_counter() - t0, threads


def load_workload(name):
    from selective_ssm_packed_gb300 import workloads
    w = workloads.make(name, backward=True, scan_input=False)
    wl = w["workload"]
    r = workloads.rounded(w, wl.dtype)
    for k in workloads.ACTIVATIONS:
        w.pop(k, None)
    return w, r


def config_of(w, world):
    wl = w["workload"]
    return {"workload": f"{wl.name}: {wl.description}", "T": w["T"], "D": wl.D, "N": wl.N, "W": wl.W,
            "io_dtype": wl.dtype, "num_seqs": len(w["lengths"]), "seed": wl.seed,
            "l2": "no flush: each (T, D) input is larger than the 129 MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ---------------------------------------------------------------- reference arm
def sized_sample(w, r, seconds):
    """Channel count whose oracle run takes about `seconds` (calibrated on 16)."""
    D = w["workload"].D
    ch0 = min(16, D)
    sec0, _ = oracle_sample(w, r, ch0)
    ch = int(ch0 * seconds / max(sec0, 1e-3))
    return max(ch0, min(D, (ch // 16) * 16 or ch0))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w, r = load_workload(args.workload)
    D, T = w["workload"].D, w["T"]
    # each step: a channel sample sized so that all steps together take ~2 minutes
    ch = sized_sample(w, r, 120.0 / max(1, args.steps + args.warmup))
    times, threads = [], 1
    for i in range(args.warmup + args.steps):
        sec, threads = oracle_sample(w, r, ch)
        if i >= args.warmup:
            times.append(sec)
    sec = sum(times) / len(times)
    value = T * (ch / D) / sec
    # ms_per_step is what one timed step took (a channel sample of the step);
    # the whole step's time is extrapolated from it by D / ch
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "ms_per_full_step_extrapolated": sec * 1e3 * D / ch, "sample_channels": ch,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: {ch} of {D} channels over all {T} tokens, conv1d + "
                                       f"selective scan fwd + bwd in double; tokens/s scaled by {D}/{ch}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def probe_alu(n_sm):
    """FP32 / packed-FP32 / MUFU throughput of this GPU (ops/s), or {}."""
    import __graft_entry__
    try:
        lib = ctypes.CDLL(__graft_entry__.PROBE_PATH)
    except OSError:
        return {}
    fn = lib.vssm_probe_alu
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    out = {}
    for kind, name, iters in ((0, "fp32_fma", 20000), (1, "fp32x2_fma", 20000), (2, "mufu_ex2", 5000)):
        v = ctypes.c_double(0.0)
        if fn(kind, n_sm * 8, iters, ctypes.byref(v)) == 0:
            out[name + "_tops"] = v.value / 1e12
    return out


def time_case(torch, vs, binding, device, cu_np, D, N, Wc, steps, seed, dtype=None, backward=True,
              flush=None, fused=False):
    """Seconds per step for the packed layout cu_np, on seeded device-generated
    inputs with the workloads' value distributions (timing only).  A step is
    pos, conv fwd, scan fwd and, with backward, scan bwd and conv bwd.  With
    `flush` (a device tensor larger than the L2), the tensor is overwritten
    before every step, outside the timed events, and the median of the
    per-step times is returned; otherwise steps run back to back.  With
    `fused`, the conv1d and scan forwards run as one call (u computed on chip)."""
    import numpy as np
    tdt = dtype or torch.bfloat16
    T = int(cu_np[-1])
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def rnd(*shape, scale=1.0):
        return (scale * torch.randn(*shape, generator=g, device=device)).to(tdt)

    x, dr, z, dout = rnd(T, D), rnd(T, D, scale=0.5), rnd(T, D), rnd(T, D)
    B, C = rnd(T, N), rnd(T, N)
    A = (-(torch.arange(N, device=device, dtype=torch.float32) + 1.0)).repeat(D, 1).contiguous()
    Dsk = torch.ones(D, device=device)
    dt = torch.exp(torch.empty(D, device=device).uniform_(math.log(1e-3), math.log(1e-1), generator=g))
    dtb = (dt + torch.log(-torch.expm1(-dt))).contiguous()
    bound = 1.0 / math.sqrt(Wc)
    cw = torch.empty(D, Wc, device=device).uniform_(-bound, bound, generator=g)
    cb = torch.empty(D, device=device).uniform_(-bound, bound, generator=g)
    cu = torch.from_numpy(np.ascontiguousarray(cu_np, dtype=np.int32)).to(device)
    pos = torch.empty(T, dtype=torch.int32, device=device)
    u = torch.empty(T, D, dtype=tdt, device=device)
    out = torch.empty_like(u)
    ypre = torch.empty_like(u)  # the forward's pre-gate output, which the backward takes for dz
    states = torch.empty(vs.chunk_states_shape(T, D, N), dtype=torch.float32, device=device)
    grads = {"du": torch.empty_like(u), "ddelta_raw": torch.empty_like(u), "dz": torch.empty_like(u),
             "dA": torch.empty(D, N, device=device), "dB": torch.empty(T, N, device=device),
             "dC": torch.empty(T, N, device=device), "dDskip": torch.empty(D, device=device),
             "d_dt_bias": torch.empty(D, device=device)}
    dx = torch.empty_like(u)
    dw = torch.empty(D, Wc, device=device)
    db = torch.empty(D, device=device)
    ws = {k: torch.empty(n, dtype=torch.uint8, device=device) for k, n in (
        ("cf", binding.conv1d_fwd_workspace_size(T, D, Wc)), ("cb", binding.conv1d_bwd_workspace_size(T, D, Wc)),
        ("sf", binding.scan_fwd_workspace_size(T, D, N)), ("sb", binding.scan_bwd_workspace_size(T, D, N)))}

    def step():
        vs.varlen_position_indices(cu, T, out=pos)
        if fused:
            # the backward needs u, y and the saved states; a forward pass does not
            vs.varlen_conv1d_scan_fwd(x, cw, cb, dr, A, B, C, Dsk, z, dtb, cu, pos, u=u if backward else None,
                                      out=out, chunk_states=states if backward else None, workspace=ws["sf"],
                                      y=ypre if backward else None)
            if not backward:
                return
        else:
            vs.varlen_conv1d_fwd(x, cw, cb, cu, pos, out=u, workspace=ws["cf"])
            if not backward:  # a forward pass: no pre-gate output or saved states needed
                vs.varlen_selective_scan_fwd(u, dr, A, B, C, Dsk, z, dtb, cu, pos, out=out, workspace=ws["sf"])
                return
            vs.varlen_selective_scan_fwd(u, dr, A, B, C, Dsk, z, dtb, cu, pos, out=out, chunk_states=states,
                                         workspace=ws["sf"], y=ypre)
        vs.varlen_selective_scan_bwd(u, dr, A, B, C, Dsk, z, dtb, dout, cu, states, pos, grads=grads,
                                     workspace=ws["sb"], y=ypre)
        vs.varlen_conv1d_bwd(x, cw, cb, grads["du"], cu, pos, dx=dx, dweight=dw, dbias=db, workspace=ws["cb"])

    for _ in range(3):
        step()
    torch.cuda.synchronize(device)
    if flush is not None:
        times = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step()
            b.record()
            torch.cuda.synchronize(device)
            times.append(a.elapsed_time(b) / 1e3)
        sec = statistics.median(times)
    else:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            step()
        b.record()
        torch.cuda.synchronize(device)
        sec = a.elapsed_time(b) / 1e3 / steps
    for k in ("sf", "sb") if backward else ("sf",):
        st = binding.read_status(ws[k])
        if st != 0:
            raise RuntimeError(f"device status {binding.ERR.get(st, st)} in a timing run ({k})")
    return sec


def comparators(args, torch, vs, binding, device, w, step_sec):
    """The no-reset concat bound on the bench workload (cu_seqlens = [0, T],
    same kernels) and the long-tail packs packed vs right-padded into the
    buckets [512 .. 8192] (each sequence its own row), real tokens/s."""
    import numpy as np
    from selective_ssm_packed_gb300 import workloads as wls
    wl = w["workload"]
    T = w["T"]
    res = {}
    csec = time_case(torch, vs, binding, device, np.array([0, T], dtype=np.int32), wl.D, wl.N, wl.W,
                     args.comparator_steps, seed=11)
    res["concat_no_reset"] = {"value": T / csec, "unit": "tokens/s", "ms_per_step": csec * 1e3,
                              "packed_over_concat": csec / step_sec,
                              "config": f"{args.workload} with cu_seqlens = [0, {T}] (one sequence)"}
    lengths = wls.pack_lengths("longtail")
    cu_pk = wls.cu_seqlens_from_lengths(lengths)
    rows = [wls.bucket_of(L) for L in lengths]
    Dc = args.comparator_d
    T_real, T_pad = int(cu_pk[-1]), int(sum(rows))
    psec = time_case(torch, vs, binding, device, cu_pk, Dc, 16, 4, args.comparator_steps, seed=12)
    # the right-padded layout (each sequence its own row of its bucket length)
    # holds ~2.2 M tokens, too many for one call's buffers at D = 4096: its rows
    # run in groups of at most the packed call's token count, and the groups'
    # step times add up to the padded step
    groups, cur, cur_t = [], [], 0
    for L in sorted(rows):
        if cur and cur_t + L > T_real:
            groups.append(cur)
            cur, cur_t = [], 0
        cur.append(L)
        cur_t += L
    if cur:
        groups.append(cur)
    qsec = 0.0
    for gi, grp in enumerate(groups):
        qsec += time_case(torch, vs, binding, device, wls.cu_seqlens_from_lengths(grp), Dc, 16, 4,
                          max(2, args.comparator_steps // 4), seed=13 + gi)
    res["longtail_packed_vs_padded"] = {
        "packed_tokens_per_s": T_real / psec, "padded_real_tokens_per_s": T_real / qsec,
        "packed_ms_per_step": psec * 1e3, "padded_ms_per_step": qsec * 1e3,
        "speedup": qsec / psec, "real_tokens": T_real, "padded_tokens": T_pad,
        "padding_rate": 1.0 - T_real / T_pad, "padded_row_groups": len(groups),
        "config": f"long-tail packs ({len(lengths)} sequences, {T_real} tokens), D={Dc}, N=16, bf16, "
                  f"buckets {list(wls.BUCKETS)}; same kernels, fwd+bwd; padded rows in "
                  f"{len(groups)} groups of at most {T_real} tokens, times summed"}
    # the fused conv1d + scan forward against the two calls, on the bench
    # workload's layout: the forward alone and the whole step
    fz = {}
    for key, bwd in (("forward", False), ("step", True)):
        two = time_case(torch, vs, binding, device, w["cu_seqlens"], wl.D, wl.N, wl.W, args.comparator_steps,
                        seed=15, backward=bwd)
        one = time_case(torch, vs, binding, device, w["cu_seqlens"], wl.D, wl.N, wl.W, args.comparator_steps,
                        seed=15, backward=bwd, fused=True)
        fz[key] = {"two_calls_ms": two * 1e3, "fused_ms": one * 1e3, "speedup": two / one}
    fz["config"] = (f"{args.workload} layout, D={wl.D}, N={wl.N}; conv1d fwd + scan fwd as two calls vs "
                    "varlen_conv1d_scan_fwd (u computed on chip; written out only for the backward)")
    res["fused_conv_scan_fwd"] = fz
    # the packer (host side): arrival-order packing against local greedy on the
    # bench workload's length mix, as the article compares them
    rng = np.random.default_rng(14)
    mix = np.clip(np.exp(rng.normal(np.log(800), 1.0, 20000)), 32, 4096).astype(np.int32)
    pk = {}
    for name, method, window in (("sequential", "sequential", 1), ("local_greedy_w1000", "local_greedy", 1000)):
        t0 = time.perf_counter()
        packs, pad = binding.pack_sequences(mix, 4096, method, window)
        pk[name] = {"packs": len(packs), "padding_rate": pad, "ms": (time.perf_counter() - t0) * 1e3}
    pk["config"] = "20000 lengths LogN(ln 800, 1) clipped [32, 4096], packs of 4096 tokens, host C++"
    res["packing"] = pk
    return res


def path_bound(counts, stages, T, hbm_gbs, fp32_tops, mufu_tops):
    """The path roofline of the given stages: per bound, the time T tokens need
    at the peak, and the slowest of them."""
    tot = {k: sum(counts[s][k] for s in stages) for k in ("bytes", "fp32", "mufu")}
    parts = {"hbm": tot["bytes"] * T / (hbm_gbs * 1e9), "fp32": tot["fp32"] * T / (fp32_tops * 1e12)}
    if mufu_tops:
        parts["mufu"] = tot["mufu"] * T / (mufu_tops * 1e12)
    return parts, max(parts.values())


def other_configs(args, torch, vs, binding, device, longtail_sec, hbm_gbs, fp32_tops, mufu_tops):
    """Tokens/s and path-roofline fraction of the other workloads: the
    Mamba-130M forward (fp32; its tensors fit in the L2, so it is timed both
    with a 512 MiB write between steps and back to back), the Mamba-1.4B
    forward, and the long-tail forward + backward (timed by the comparator)."""
    from selective_ssm_packed_gb300 import workloads as wls
    res = {}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    for name, flushed in (("m130m", True), ("m14b_fwd", False)):
        wl = wls.WORKLOADS[name]
        cu = wls.cu_seqlens_from_lengths(wls.pack_lengths(name))
        T = int(cu[-1])
        tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        e = 4 if wl.dtype == "f32" else 2
        counts = per_token_counts(wl.D, wl.N, e, wl.W)
        parts, t_roof = path_bound(counts, ("conv_fwd", "scan_fwd"), T, hbm_gbs, fp32_tops, mufu_tops)
        entry = {"config": f"{name}: {wl.description}; pos + conv1d fwd + selective scan fwd",
                 "T": T, "path_bound_ms": {k: v * 1e3 for k, v in parts.items()}}
        runs = (("l2_flushed", flush), ("back_to_back", None)) if flushed else (("back_to_back", None),)
        for key, fl in runs:
            sec = time_case(torch, vs, binding, device, cu, wl.D, wl.N, wl.W, 50, seed=wl.seed, dtype=tdt,
                            backward=False, flush=fl)
            entry[key] = {"value": T / sec, "unit": "tokens/s", "ms_per_step": sec * 1e3,
                          "frac_of_path_roofline": t_roof / sec}
        if flushed:
            entry["l2"] = "each (T, D) tensor is 24 MiB and fits in the 129 MB L2: l2_flushed overwrites " \
                          "a 512 MiB buffer before every step (median of 50 steps)"
        res[name] = entry
    if longtail_sec:
        wl = wls.WORKLOADS["longtail"]
        T = int(wls.cu_seqlens_from_lengths(wls.pack_lengths("longtail"))[-1])
        counts = per_token_counts(wl.D, wl.N, 2, wl.W)
        parts, t_roof = path_bound(counts, tuple(counts), T, hbm_gbs, fp32_tops, mufu_tops)
        res["longtail"] = {"config": f"longtail: {wl.description}; the whole step",
                           "T": T, "value": T / longtail_sec, "unit": "tokens/s",
                           "ms_per_step": longtail_sec * 1e3, "frac_of_path_roofline": t_roof / longtail_sec,
                           "path_bound_ms": {k: v * 1e3 for k, v in parts.items()}}
    del flush
    return res


def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__
    import selective_ssm_packed_gb300 as vs
    from selective_ssm_packed_gb300 import binding

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init("nccl")
    if rank == 0 or world == 1:
        __graft_entry__.build()
    barrier(device)
    __graft_entry__.build()

    w, r = load_workload(args.workload)
    wl = w["workload"]
    T, D, N, Wc = w["T"], wl.D, wl.N, wl.W
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    e = 2 if wl.dtype == "bf16" else 4

    def dev(a, dt=tdt):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device).to(dt)

    names_in = ("x", "delta_raw", "z", "B", "C", "dout")
    inp = {k: dev(r[k]) for k in names_in}
    prm = {k: dev(r[k], torch.float32) for k in ("A", "Dskip", "dt_bias", "conv_w", "conv_b")}
    cu = torch.from_numpy(w["cu_seqlens"]).to(device)
    pos = torch.empty(T, dtype=torch.int32, device=device)
    u = torch.empty(T, D, dtype=tdt, device=device)
    out = torch.empty_like(u)
    ypre = torch.empty_like(u)  # the forward's pre-gate output, which the backward takes for dz
    states = torch.empty(vs.chunk_states_shape(T, D, N), dtype=torch.float32, device=device)
    grads = {"du": torch.empty_like(u), "ddelta_raw": torch.empty_like(u), "dz": torch.empty_like(u),
             "dA": torch.empty(D, N, device=device), "dB": torch.empty(T, N, device=device),
             "dC": torch.empty(T, N, device=device), "dDskip": torch.empty(D, device=device),
             "d_dt_bias": torch.empty(D, device=device)}
    dx = torch.empty_like(u)
    dw = torch.empty(D, Wc, device=device)
    db = torch.empty(D, device=device)
    ws = {k: torch.empty(n, dtype=torch.uint8, device=device) for k, n in (
        ("cf", binding.conv1d_fwd_workspace_size(T, D, Wc)), ("cb", binding.conv1d_bwd_workspace_size(T, D, Wc)),
        ("sf", binding.scan_fwd_workspace_size(T, D, N)), ("sb", binding.scan_bwd_workspace_size(T, D, N)))}
    stream = torch.cuda.current_stream(device)
    STAGES = ("pos", "conv_fwd", "scan_fwd", "scan_bwd", "conv_bwd")

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        vs.varlen_position_indices(cu, T, out=pos)
        mark(1)
        vs.varlen_conv1d_fwd(inp["x"], prm["conv_w"], prm["conv_b"], cu, pos, out=u, workspace=ws["cf"])
        mark(2)
        vs.varlen_selective_scan_fwd(u, inp["delta_raw"], prm["A"], inp["B"], inp["C"], prm["Dskip"],
                                     inp["z"], prm["dt_bias"], cu, pos, out=out, chunk_states=states,
                                     workspace=ws["sf"], y=ypre)
        mark(3)
        vs.varlen_selective_scan_bwd(u, inp["delta_raw"], prm["A"], inp["B"], inp["C"], prm["Dskip"],
                                     inp["z"], prm["dt_bias"], inp["dout"], cu, states, pos,
                                     grads=grads, workspace=ws["sb"], y=ypre)
        mark(4)
        vs.varlen_conv1d_bwd(inp["x"], prm["conv_w"], prm["conv_b"], grads["du"], cu, pos,
                             dx=dx, dweight=dw, dbias=db, workspace=ws["cb"])
        mark(5)

    # this library's launches per step: position indices 1; conv fwd 1; scan
    # fwd 1, plus the A-row preparation 1 and 2 to widen B and C for bf16 I/O;
    # scan bwd 1, plus the B/C rows 1, the tile parameters 1 (N = 16), the
    # dB/dC tile sum 1 and 3 fixed-order row sums of 2 launches (dA, dDskip,
    # d_dt_bias); conv bwd 1 plus 2 row sums of 2 (dweight, dbias)
    KERNELS_PER_STEP = (1 + 1 + (1 + 1 + (2 if wl.dtype == "bf16" else 0))
                        + (1 + 1 + (1 if wl.N == 16 else 0) + 1 + 3 * 2) + (1 + 2 * 2))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    for k in ("sf", "sb"):
        st = binding.read_status(ws[k])
        if st != 0:
            raise RuntimeError(f"device status {binding.ERR.get(st, st)} after warm-up ({k})")

    # --- device-resident throughput, per-stage events on the launching stream
    clocks_path = args.clock_log.replace("{rank}", str(rank)) if args.clock_log else \
        os.path.join(tempfile.gettempdir(), f"vssm_clocks_{os.getpid()}_rank{rank}.csv")
    sampler = ClockSampler(local, clocks_path)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    barrier(device)
    torch.cuda.synchronize(device)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # the library's own events around each call's main kernel, on the same
    # stream, so that a kernel's launch duration is timed apart from its call
    binding.debug_set(binding.VSSM_DBG_KERNEL_EVENTS, 1)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(device)
    kernel_ms = {}
    for s in STAGES[1:]:
        tot, n = binding.kernel_time(s)
        kernel_ms[s] = tot / n if n else None
    binding.debug_set(binding.VSSM_DBG_KERNEL_EVENTS, 0)
    clocks = sampler.stop()
    barrier(device)
    sec = t_start.elapsed_time(t_end) / 1e3
    value, sec_max = aggregate(T, sec / args.steps, world, device)
    stage_ms = {s: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)) / args.steps
                for j, s in enumerate(STAGES)}
    for k in ("sf", "sb"):
        st = binding.read_status(ws[k])
        if st != 0:
            raise RuntimeError(f"device status {binding.ERR.get(st, st)} in the timed region ({k})")

    # --- end to end through the public API with host buffers.  Every step copies
    #     its own inputs in from pinned host memory and its results back out;
    #     the copies run on their own streams, double-buffered on the device, so
    #     step k+1's inputs and step k's results move while the GPU computes.
    e2e = None
    if not args.no_e2e:
        host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inp.items()}
        for k in host_in:
            host_in[k].copy_(inp[k])
        cu_host = torch.from_numpy(w["cu_seqlens"]).pin_memory()
        out_like = {"out": out, "dx": dx, "ddelta_raw": grads["ddelta_raw"], "dz": grads["dz"],
                    "dB": grads["dB"], "dC": grads["dC"], "dA": grads["dA"], "dDskip": grads["dDskip"],
                    "d_dt_bias": grads["d_dt_bias"], "dweight": dw, "dbias": db}
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out_like.items()}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + cu_host.numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        # two device sets of inputs and results; scratch (u, states, workspaces) is shared
        sets = []
        for _ in range(2):
            si = {k: torch.empty_like(v) for k, v in inp.items()}
            si["cu"] = torch.empty_like(cu)
            so = {k: torch.empty_like(v) for k, v in out_like.items()}
            sets.append((si, so))
        s_in = torch.cuda.Stream(device)
        s_out = torch.cuda.Stream(device)

        def compute(si, so):
            g = {"du": grads["du"], "ddelta_raw": so["ddelta_raw"], "dz": so["dz"], "dA": so["dA"],
                 "dB": so["dB"], "dC": so["dC"], "dDskip": so["dDskip"], "d_dt_bias": so["d_dt_bias"]}
            c = si["cu"]
            vs.varlen_position_indices(c, T, out=pos)
            vs.varlen_conv1d_fwd(si["x"], prm["conv_w"], prm["conv_b"], c, pos, out=u, workspace=ws["cf"])
            vs.varlen_selective_scan_fwd(u, si["delta_raw"], prm["A"], si["B"], si["C"], prm["Dskip"],
                                         si["z"], prm["dt_bias"], c, pos, out=so["out"], chunk_states=states,
                                         workspace=ws["sf"], y=ypre)
            vs.varlen_selective_scan_bwd(u, si["delta_raw"], prm["A"], si["B"], si["C"], prm["Dskip"],
                                         si["z"], prm["dt_bias"], si["dout"], c, states, pos,
                                         grads=g, workspace=ws["sb"], y=ypre)
            vs.varlen_conv1d_bwd(si["x"], prm["conv_w"], prm["conv_b"], g["du"], c, pos,
                                 dx=so["dx"], dweight=so["dweight"], dbias=so["dbias"], workspace=ws["cb"])

        def run_e2e(n):
            """n steps; returns seconds for all of them (events on the compute stream,
            which waits for the last copies before its end event) and each stream's
            mean busy time per step in ms (from the moment its waits are met)."""
            ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
            copied = [ev() for _ in range(n)]    # inputs of step k on the device
            computed = [ev() for _ in range(n)]  # results of step k ready
            drained = [ev() for _ in range(n)]   # results of step k on the host
            in0, c0, o0 = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s_in.wait_event(a)
            s_out.wait_event(a)
            for k in range(n):
                si, so = sets[k % 2]
                with torch.cuda.stream(s_in):
                    if k >= 2:
                        s_in.wait_event(computed[k - 2])       # set k%2 no longer read by compute
                    in0[k].record(s_in)
                    for name, h in host_in.items():
                        si[name].copy_(h, non_blocking=True)
                    si["cu"].copy_(cu_host, non_blocking=True)
                    copied[k].record(s_in)
                stream.wait_event(copied[k])
                if k >= 2:
                    stream.wait_event(drained[k - 2])          # results of set k%2 copied out
                c0[k].record(stream)
                compute(si, so)
                computed[k].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(computed[k])
                    o0[k].record(s_out)
                    for name, h in host_out.items():
                        h.copy_(so[name], non_blocking=True)
                    drained[k].record(s_out)
            stream.wait_event(drained[n - 1])
            b.record(stream)
            torch.cuda.synchronize(device)
            busy = {name: sum(x.elapsed_time(y) for x, y in zip(s0, s1)) / n
                    for name, s0, s1 in (("h2d", in0, copied), ("compute", c0, computed), ("d2h", o0, drained))}
            return a.elapsed_time(b) / 1e3, busy

        def host_link(n):
            """The host link on its own: n steps' input and result copies, both
            directions at once on the copy streams, with nothing computed.
            Returns seconds per step: the floor under the end-to-end step."""
            si, so = sets[0]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s_in.wait_event(a)
            s_out.wait_event(a)
            for _ in range(n):
                with torch.cuda.stream(s_in):
                    for name, h in host_in.items():
                        si[name].copy_(h, non_blocking=True)
                    si["cu"].copy_(cu_host, non_blocking=True)
                with torch.cuda.stream(s_out):
                    for name, h in host_out.items():
                        h.copy_(so[name], non_blocking=True)
            ein, eout = torch.cuda.Event(), torch.cuda.Event()
            ein.record(s_in)
            eout.record(s_out)
            stream.wait_event(ein)
            stream.wait_event(eout)
            b.record(stream)
            torch.cuda.synchronize(device)
            return a.elapsed_time(b) / 1e3 / n

        run_e2e(2)
        nl = max(4, args.e2e_steps // 2)
        l0 = host_link(nl)  # the link is shared with the host's other work: timed on both sides
        barrier(device)
        esec, busy = run_e2e(args.e2e_steps)
        esec /= args.e2e_steps
        ev, _ = aggregate(T, esec, world, device)
        l1 = host_link(nl)
        lsec = min(l0, l1)
        e2e = {"value": ev, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": esec * 1e3, "steps": args.e2e_steps,
               "stream_busy_ms_per_step": busy,
               "copies": "pinned host buffers; input and result copies on their own streams, "
                         "double-buffered on the device, overlapping the neighbouring steps' compute",
               "host_link": {"ms_per_step": lsec * 1e3,
                             "ms_per_step_before_after": [l0 * 1e3, l1 * 1e3],
                             "GB/s_each_way": {"h2d": h2d / lsec / 1e9, "d2h": d2h / lsec / 1e9},
                             "e2e_frac_of_link_floor": lsec / esec,
                             "what": "the same copies alone, both directions at once, no compute; "
                                     "timed before and after the end-to-end run, the faster taken"}}
        for k in ("sf", "sb"):
            st = binding.read_status(ws[k])
            if st != 0:
                raise RuntimeError(f"device status {binding.ERR.get(st, st)} in the e2e run ({k})")

    # --- comparators: no-reset concat bound, packed vs right-padded (rank 0, one GPU)
    comp = None
    if rank == 0 and world == 1 and not args.no_comparators:
        comp = comparators(args, torch, vs, binding, device, w, sec / args.steps)

    # --- roofline of the dominant kernel, plus every stage for context
    counts = per_token_counts(D, N, e, Wc)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    n_sm = torch.cuda.get_device_properties(device).multi_processor_count
    fp32_peak_tops = n_sm * 128 * sm_max * 1e6 / 1e12         # FP32 pipe, FMA = 1 op
    probes = probe_alu(n_sm) if rank == 0 else {}
    stages = {}
    for s in ("conv_fwd", "scan_fwd", "scan_bwd", "conv_bwd"):
        c, ms = counts[s], stage_ms[s]
        stages[s] = {"ms": ms, "GB/s": c["bytes"] * T / (ms * 1e-3) / 1e9,
                     "fp32_Tops/s": c["fp32"] * T / (ms * 1e-3) / 1e12,
                     "mufu_Tops/s": c["mufu"] * T / (ms * 1e-3) / 1e12,
                     "kernel_ms": kernel_ms.get(s)}
    dom = max(("conv_fwd", "scan_fwd", "scan_bwd", "conv_bwd"), key=lambda s: stage_ms[s])
    c = counts[dom]
    # the dominant call's main kernel, timed by its own events in the timed
    # region (the call's time when those are missing)
    k_ms = kernel_ms.get(dom) or stage_ms[dom]
    t_hbm = c["bytes"] * T / (hbm_peak * 1e9)
    t_alu = c["fp32"] * T / (fp32_peak_tops * 1e12)
    if t_alu >= t_hbm:
        roof = {"kernel": dom, "bound": "alu", "achieved": c["fp32"] * T / (k_ms * 1e-3) / 1e12,
                "peak": fp32_peak_tops, "unit": "Tops/s (fp32 pipe, FMA=1)",
                "peak_source": f"{n_sm} SMs x 128 FP32 lanes x {sm_max:.0f} MHz (max SM clock)"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": c["bytes"] * T / (k_ms * 1e-3) / 1e9,
                "peak": hbm_peak, "unit": "GB/s", "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["launch_ms"] = k_ms
    roof["launch_timing"] = ("CUDA events the library records on the launching stream around the call's main "
                             "kernel, averaged over the timed steps" if kernel_ms.get(dom) else
                             "the call's CUDA-event time (kernel events unavailable)")
    tr = LAST_CAPTURE_TRAFFIC.get((args.workload if args.workload != "m14b_small" else "m14b", dom))
    roof["traffic"] = tr["bytes_per_token"] * T if tr else None
    if tr:
        roof["traffic_source"] = tr["source"]
        roof["traffic_kernel"] = tr["kernel"]
    roof["algorithmic_per_token"] = c
    roof["counts"] = ("algorithmic per-token counts of the path's scope; this implementation also moves "
                      "the pre-gate output y (per token: "
                      + ", ".join(f"{k} +{v} B" for k, v in implementation_extra_bytes(D, e).items()) + ")")
    # whole-step roofline (the metric's definition): slowest of HBM, FP32, MUFU bounds
    mufu_tops = probes.get("mufu_ex2_tops")
    t_parts, t_roof = path_bound(counts, tuple(counts), T, hbm_peak, fp32_peak_tops, mufu_tops)
    step_ms = sec * 1e3 / args.steps
    path_roofline = {"step_bound_ms": {k: v * 1e3 for k, v in t_parts.items()},
                     "roofline_tokens_per_s": T / t_roof, "frac_of_roofline": t_roof / (step_ms * 1e-3),
                     "alu_probe_tops": probes}

    # --- the other workloads (rank 0, one GPU only)
    cfgs = None
    if rank == 0 and world == 1 and not args.no_configs:
        lt = comp["longtail_packed_vs_padded"]["packed_ms_per_step"] / 1e3 \
            if comp and args.comparator_d == 4096 else None
        cfgs = other_configs(args, torch, vs, binding, device, lt, hbm_peak, fp32_peak_tops, mufu_tops)

    # --- CPU oracle baseline (rank 0, one GPU only): all host cores, and one core
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        ch = sized_sample(w, r, args.cpu_seconds)
        csec, threads = oracle_sample(w, r, ch)
        cpu = {"value": T * (ch / D) / csec, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{ch} of {D} channels over all {T} tokens (conv1d + selective scan fwd + bwd, "
                         f"double), {csec:.1f} s; tokens/s scaled by {D}/{ch}"}
        # one core: a sample sized to about 3 s from a 16-channel probe
        c16, _ = oracle_sample(w, r, 16, threads=1)
        ch1 = max(16, min(D, int(16 * 3.0 / max(c16, 1e-3)) // 16 * 16))
        csec1, _ = oracle_sample(w, r, ch1, threads=1)
        cpu["one_core"] = {"value": T * (ch1 / D) / csec1, "unit": "tokens/s", "cores": 1,
                           "sample": f"{ch1} of {D} channels over all {T} tokens, {csec1:.1f} s"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": sec_max * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": config_of(w, world), "roofline": roof, "path_roofline": path_roofline,
                "stages": stages, "cpu_baseline": cpu, "e2e": e2e, "comparators": comp, "configs": cfgs,
                "gpu_launches": KERNELS_PER_STEP * args.steps, "clocks": clocks}
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
