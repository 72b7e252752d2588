#!/usr/bin/env python3
"""Benchmark: one 2:4 sparse FFN training step (prune both weights fresh,
forward, double-pruned backward, masked weight gradients) on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0. The metric is the step's dense-equivalent
throughput (12 * M * d * ffn FLOP per step / step time), reported with its
fraction of the 2:4-sparse bf16 tensor peak; the standalone 1e9-element prune
and the V:2:M (128:2:8) prune of a W_up-shaped weight are reported beside it in
GB/s. Multi-GPU runs are independent replicas (one
step per GPU, no collective on the data path): weak scaling, value = all
ranks' FLOP / the slowest rank's time.

--impl reference times the CPU oracle (oracle/, numpy) on the host cores on a
bounded slice of the same workload; it is a slow reference, not a target.
"""
from __future__ import annotations

import argparse
import ctypes
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SPARSE_RATIO = 2.0  # nominal 2:4-sparse / dense tensor throughput
# DRAM bytes per launch of the dominant kernel, from an ncu capture; used only while
# the kernel's sources are the ones that were captured.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "spmm_kernel_dram_traffic.json")
KERNEL_SOURCES = ("gemm24_kernels.cu", "p24_ptx.cuh", "p24_internal.h")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "semi_structured_sparse_prune24_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic(workload: str) -> tuple[float | None, str | None]:
    """Per-launch DRAM bytes (read + write) of spmm_kernel at this workload and how they
    were obtained, or (None, None) when no capture matches the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, None
    if rec.get("kernel_source_sha256") != kernel_source_hash():
        return None, None
    v = rec.get("per_launch_bytes", {}).get(workload)
    return v, (None if v is None else rec.get("scaling"))
L2_BYTES = 129 * 2 ** 20


def load_peaks() -> tuple[dict, str]:
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, device_index: int):
        ident = str(device_index)
        try:
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={ident}", f"--query-gpu={self.QUERY}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def stop(self, window: tuple | None = None) -> dict | None:
        """window: (start, end) local wall-clock datetimes of the timed region; samples
        outside it are dropped (all are kept if none can be placed inside it)."""
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out, _ = self.p.communicate()
        return parse_clock_samples(out, window)


def parse_clock_samples(text: str, window: tuple | None = None) -> dict | None:
    """Median SM clock, max clock and active throttle reasons from nvidia-smi CSV lines
    of ClockSampler.QUERY. Lines whose timestamp falls outside `window` are left out."""
    import datetime
    rows = []
    for line in text.splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm, mx = float(f[1]), float(f[2])
        except ValueError:
            continue
        ts = None
        if len(f) >= 10:
            try:
                ts = datetime.datetime.strptime(f[9], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None
        rows.append((sm, mx, f[5:9], ts))
    inside = rows
    if window is not None:
        lo, hi = window
        inside = [r for r in rows if r[3] is not None and lo <= r[3] <= hi]
    in_window = bool(inside)
    if not inside:
        inside = rows
    if not inside:
        return None
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = {n for r in inside for n, v in zip(names, r[2]) if v.lower() == "active"}
    return {"sm_mhz": statistics.median(r[0] for r in inside), "sm_max_mhz": max(r[1] for r in inside),
            "samples": len(inside), "samples_in_timed_region": in_window, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ distributed plumbing
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")  # barrier + timing reduction only
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle (CPU) sample
def oracle_sample_step(d: int, m_s: int, f_s: int, w_sigma: float, seed: int = 0) -> float:
    """One oracle step on a slice of the workload: m_s tokens x f_s hidden units
    (full model width d). Returns seconds. Inputs drawn like the workload's."""
    import numpy as np  # noqa: F401

    from oracle import prune24_oracle as O
    from synth24 import normal_bf16

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view("uint16")

    X = bits(normal_bf16((m_s, d), 1.0, seed, 1))
    Wu = bits(normal_bf16((f_s, d), w_sigma, seed, 2))
    Wd = bits(normal_bf16((d, f_s), w_sigma, seed, 3))
    dY = bits(normal_bf16((m_s, d), 1.0, seed, 6))
    bu = np.zeros(f_s, np.float32)
    bd = np.zeros(d, np.float32)
    t0 = time.perf_counter()
    O.ffn_step(X, Wu, bu, Wd, bd, dY)
    return time.perf_counter() - t0


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, seconds_target: float = 15.0) -> dict:
    m_s, f_s = 1024, 1024
    oracle_sample_step(w.d, 64, 64, w.w_sigma)  # import + first-touch warmup
    times = []
    t_start = time.perf_counter()
    while not times or (time.perf_counter() - t_start < seconds_target and len(times) < 20):
        times.append(oracle_sample_step(w.d, m_s, f_s, w.w_sigma))
    t = statistics.median(times)
    flop = 12 * m_s * w.d * f_s
    return {"value": flop / t / 1e12, "unit": "TFLOPS (dense-equivalent)", "cores": cpu_cores(), "kind": "oracle",
            "sample": (f"oracle ffn_step (numpy fp32 GEMMs via BLAS on all visible cores, prune+double-prune "
                       f"included) on a slice of the workload: {m_s} tokens x {f_s} hidden units at d={w.d}; "
                       f"median of {len(times)} runs, {t:.2f} s each")}


# ------------------------------------------------------------------ end to end, per configuration
def config_e2e(P, cw, ci: dict, co: dict, dev, stream, args) -> dict:
    """The configuration's step fed from pinned host buffers through StepPipeline: the
    inputs (X, W_up, W_down, dY) copied in and the results (Y, dX, dW_up, dW_down, db)
    copied out every step, overlapped with neighbouring steps' compute."""
    from semi_structured_sparse_prune24_gb300.pipeline import StepPipeline
    hin = {k: ci[k].cpu().pin_memory() for k in ("X", "W_up", "W_down", "dY")}
    hout = {k: torch.empty(co[k].shape, dtype=co[k].dtype).pin_memory()
            for k in ("Y", "dX", "dW_up", "dW_down", "db_up", "db_down")}
    pipe = StepPipeline(cw.M, cw.d, cw.ffn, act24=cw.act24, b_up=ci["b_up"], b_down=ci["b_down"], device=dev)
    for _ in range(args.warmup):
        pipe.submit(hin, hout)
    pipe.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    pipe.start_after(e0)
    for _ in range(args.steps):
        pipe.submit(hin, hout)
    pipe.finish_on(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if P.p24_query_status() != 0:
        raise RuntimeError("device status word set during the end-to-end steps")
    ems = e0.elapsed_time(e1) / args.steps
    out = {"value": cw.dense_equiv_flop / (ems * 1e-3) / 1e12, "unit": "TFLOPS (dense-equivalent)",
           "ms_per_step": ems, "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin.values()),
           "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout.values())}
    del pipe, hin, hout
    return out


# ------------------------------------------------------------------ hybrid activations
def bench_hybrid(P, dev, stream, seed, args, peaks) -> dict:
    """The hybrid ELL + dense-overflow path on synthetic ReLU activations: z ~ N(0, 1)
    shifted by t = 2.326 (about 1% nonzero), every 50th token by 1.28 (about 10%, so it
    overflows an ELL of width 256). Shape of the 1.3B FFN: H [8192, 8192], d = 2048.
    Times the format (HBM-bound stream of H), hybrid -> dense Y = H . W_down^T and
    dense -> hybrid dH = (dY . W_down) at H's nonzeros (both gather one 4 KB row of
    W_down^T per nonzero, from L2: W_down^T is 32 MB), beside the dense tensor-core
    product of the same H for context, and an L2-resident copy as the gather roofline."""
    from synth24 import normal_bf16
    R, Cc, N, E = 8192, 8192, 2048, 256
    z = normal_bf16((R, Cc), 1.0, seed, 7, dev).float()
    thr = torch.full((R, 1), 2.326, device=dev)
    thr[::50] = 1.28
    H = torch.relu(z - thr).to(torch.bfloat16)
    del z
    Wt = normal_bf16((Cc, N), 0.02, seed, 3, dev)          # W_down^T [ffn, d]
    Wd = Wt.t().contiguous()                                # W_down [d, ffn]
    G = normal_bf16((R, N), 1.0, seed, 6, dev)              # dY
    h = P.hyb_compress(H, E, R // 16)
    Y = P.hyb_spmm(h, Wt)
    S_ell, S_ovf = P.hyb_sddmm(h, G, Wt)
    Yd = torch.empty((R, N), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize(dev)
    if P.p24_query_status() != 0:
        raise RuntimeError("device status word set by the hybrid format")
    nnz = int(h.nnz.sum().item())
    n_ovf = int(h.n_ovf.item())

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / args.steps

    t_c = timed(lambda: P.hyb_compress(H, E, R // 16, out=h))
    t_s = timed(lambda: P.hyb_spmm(h, Wt, Y=Y))
    t_d = timed(lambda: P.hyb_sddmm(h, G, Wt, S_ell=S_ell, S_ovf=S_ovf))
    t_dense = timed(lambda: P.p24_gemm_nt(H, Wd, C_out=Yd))
    # L2-resident copy (16 MB each way) as the reference for the gathers
    a = torch.empty(16 * 2 ** 20, dtype=torch.bfloat16, device=dev)    # 32 MB, twice: L2-resident
    bcopy = torch.empty_like(a)

    def copies():
        for _ in range(20):
            bcopy.copy_(a)
    t_l2 = timed(copies) / 20
    l2_gbs = 2 * a.numel() * 2 / (t_l2 * 1e-3) / 1e9
    if P.p24_query_status() != 0:
        raise RuntimeError("device status word set during the hybrid timings")
    gathered = nnz * N * 2                                   # one row of W_down^T per nonzero
    c_bytes = R * Cc * 2 + R * E * 4 + R * 8 + n_ovf * Cc * 4
    out = {"shape": {"tokens": R, "ffn": Cc, "d": N, "E": E, "cap": R // 16},
           "density": nnz / (R * Cc), "overflow_rows": n_ovf,
           "compress": {"ms": t_c, "value": c_bytes / (t_c * 1e-3) / 1e9, "unit": "GB/s", "bound": "hbm",
                        "frac": c_bytes / (t_c * 1e-3) / 1e9 / peaks["hbm_gbs"],
                        "algorithmic_bytes": c_bytes},
           "hybrid_to_dense": {"ms": t_s, "gathered_GBs": gathered / (t_s * 1e-3) / 1e9,
                               "frac_of_l2_copy": gathered / (t_s * 1e-3) / 1e9 / l2_gbs,
                               "tflops": 2 * nnz * N / (t_s * 1e-3) / 1e12},
           "dense_to_hybrid": {"ms": t_d, "gathered_GBs": gathered / (t_d * 1e-3) / 1e9,
                               "frac_of_l2_copy": gathered / (t_d * 1e-3) / 1e9 / l2_gbs,
                               "tflops": 2 * nnz * N / (t_d * 1e-3) / 1e12},
           "dense_tensor_core_same_product_ms": t_dense,
           "l2_copy_GBs": l2_gbs,
           "note": "gathered bytes = nonzeros x d x 2 (one W_down^T row per nonzero); the L2 figure is a "
                   "32 MB L2-resident copy measured in this run"}
    del H, Wt, Wd, G, h, Y, S_ell, S_ovf, Yd, a, bcopy
    return out


# ------------------------------------------------------------------ our arm
def run_ours(args, world, rank, local):
    import semi_structured_sparse_prune24_gb300 as P
    from synth24 import WORKLOADS, ffn_inputs, normal_bf16

    w = WORKLOADS[args.workload]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    # inputs resident in HBM (seeded per rank)
    seed = rank
    X = normal_bf16((w.M, w.d), w.x_sigma, seed, 1, dev)
    Wu = normal_bf16((w.ffn, w.d), w.w_sigma, seed, 2, dev)
    Wd = normal_bf16((w.d, w.ffn), w.w_sigma, seed, 3, dev)
    dY = normal_bf16((w.M, w.d), w.dy_sigma, seed, 6, dev)
    bu = torch.zeros(w.ffn, dtype=torch.float32, device=dev)
    bd = torch.zeros(w.d, dtype=torch.float32, device=dev)
    out = P.ffn24_step(X, Wu, bu, Wd, bd, dY, act24=w.act24)
    ws = torch.empty(P.ffn24_workspace_size(w.M, w.d, w.ffn, w.act24), dtype=torch.uint8, device=dev)

    def step(events=None):
        P.ffn24_step(X, Wu, bu, Wd, bd, dY, act24=w.act24, out=out, workspace=ws, events=events)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if P.p24_query_status() != 0:
        raise RuntimeError("device status word set after warm-up")

    # per-phase events (raw cudaEvent_t handles), created up front
    nph = P.STEP_PHASES
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nph * args.steps)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize(dev)
    handles = [(ctypes.c_void_p * (2 * nph))(*[evs[i * 2 * nph + j].cuda_event for j in range(2 * nph)])
               for i in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    launches0 = P.p24_launch_count()
    wall0 = datetime.datetime.now()
    t0.record(stream)
    for i in range(args.steps):
        step(handles[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = datetime.datetime.now()
    launches = P.p24_launch_count() - launches0
    barrier(world)
    clk = clocks.stop((wall0, wall1))
    if P.p24_query_status() != 0:
        raise RuntimeError("device status word set during the timed steps")
    ms_step = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)

    phase_ms = [statistics.mean(evs[i * 2 * nph + 2 * p].elapsed_time(evs[i * 2 * nph + 2 * p + 1])
                                for i in range(args.steps)) for p in range(nph)]
    flop = w.dense_equiv_flop
    value = world * flop / (ms_step * 1e-3) / 1e12
    sparse_peak = peaks["bf16_tflops_sustained"] * SPARSE_RATIO
    dense_peak = peaks["bf16_tflops_sustained"]
    gemm_flop = 2 * w.M * w.d * w.ffn  # every one of the six GEMMs
    kernels = {
        "spmm_kernel (tcgen05.mma.sp)": {"phases": [2, 3, 4, 7], "bound": "tensor", "peak": sparse_peak,
                                         "per_launch": gemm_flop, "unit": "TFLOP/s"},
        "dw_kernel (tcgen05.mma, masked)": {"phases": [6, 8], "bound": "tensor", "peak": dense_peak,
                                            "per_launch": gemm_flop, "unit": "TFLOP/s"},
        "double_prune_interior_kernel (fused prune + double prune)": {
            "phases": [0, 1], "bound": "hbm", "peak": peaks["hbm_gbs"],
            "per_launch": int(4.25 * w.d * w.ffn), "unit": "GB/s"},
        # db_up is fused into the dH GEMM's epilogue; phase 5 is the column sums of dY
        "colsum (db_down)": {"phases": [5], "bound": "hbm", "peak": peaks["hbm_gbs"],
                             "per_launch": 2 * w.M * w.d, "unit": "GB/s"},
    }
    breakdown = {}
    for name, k in kernels.items():
        tot = sum(phase_ms[p] for p in k["phases"])
        avg = tot / len(k["phases"])
        scale = 1e12 if k["unit"] == "TFLOP/s" else 1e9
        ach = k["per_launch"] / (avg * 1e-3) / scale
        breakdown[name] = {"ms_per_step": tot, "launches_per_step": len(k["phases"]), "avg_launch_ms": avg,
                           "achieved": ach, "unit": k["unit"], "frac": ach / k["peak"]}
    dominant = max(breakdown, key=lambda n: breakdown[n]["ms_per_step"])
    dk = kernels[dominant]
    roofline = {"kernel": dominant, "bound": dk["bound"], "achieved": breakdown[dominant]["achieved"],
                "peak": dk["peak"], "unit": dk["unit"], "frac": breakdown[dominant]["frac"],
                "traffic": captured_traffic(args.workload)[0] if dominant.startswith("spmm_kernel") else None,
                "traffic_source": captured_traffic(args.workload)[1] if dominant.startswith("spmm_kernel") else None,
                "peak_source": f"{peak_src} bf16_tflops_sustained" +
                               (" x 2 (nominal 2:4 ratio)" if dk["peak"] == sparse_peak else "")
                               if dk["unit"] == "TFLOP/s" else f"{peak_src} hbm_gbs"}

    # ---- the same step with SLOPE's low-rank adapters (rank 64) on both linears
    slope = None
    if not args.no_adapters:
        r = 64
        ad = {"L_up": normal_bf16((w.ffn, r), 0.02, seed, 10, dev), "R_up": normal_bf16((r, w.d), 0.02, seed, 11, dev),
              "L_down": normal_bf16((w.d, r), 0.02, seed, 12, dev),
              "R_down": normal_bf16((r, w.ffn), 0.02, seed, 13, dev)}
        ws_ad = torch.empty(P.ffn24_workspace_size_lowrank(w.M, w.d, w.ffn, w.act24, r), dtype=torch.uint8,
                            device=dev)
        out_ad = P.ffn24_step(X, Wu, bu, Wd, bd, dY, act24=w.act24, workspace=ws_ad, adapters=ad)
        for _ in range(args.warmup):
            P.ffn24_step(X, Wu, bu, Wd, bd, dY, act24=w.act24, out=out_ad, workspace=ws_ad, adapters=ad)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a0.record(stream)
        for _ in range(args.steps):
            P.ffn24_step(X, Wu, bu, Wd, bd, dY, act24=w.act24, out=out_ad, workspace=ws_ad, adapters=ad)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        if P.p24_query_status() != 0:
            raise RuntimeError("device status word set during the adapter steps")
        ad_ms = a0.elapsed_time(a1) / args.steps
        ad_flop = 12 * w.M * r * (w.d + w.ffn)  # T, term, U, dX term, dL, dR of both linears
        slope = {"r": r, "ms_per_step": ad_ms, "value": (flop + ad_flop) / (ad_ms * 1e-3) / 1e12,
                 "unit": "TFLOPS (dense-equivalent, adapter FLOPs included)", "adapter_flop": ad_flop,
                 "overhead_vs_plain_step": ad_ms / ms_step - 1.0}
        del out_ad, ws_ad, ad
        torch.cuda.empty_cache()

    # ---- V:N:M activations (256:2:8, 75% sparse H): the same step with H pruned V:2:M
    #      along ffn and the down forward on the V:2:M GEMM (gathered W_down^T rows)
    vnm = None
    if not args.no_vnm:
        try:
            VV, VM = 256, 8
            ws_v = torch.empty(P.ffn24_workspace_size(w.M, w.d, w.ffn, vnm=(VV, VM)), dtype=torch.uint8, device=dev)
            out_v = P.ffn24_step(X, Wu, bu, Wd, bd, dY, workspace=ws_v, vnm=(VV, VM))
            for _ in range(args.warmup):
                P.ffn24_step(X, Wu, bu, Wd, bd, dY, out=out_v, workspace=ws_v, vnm=(VV, VM))
            evv = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nph * args.steps)]
            for e in evv:
                e.record(stream)
            torch.cuda.synchronize(dev)
            hv = [(ctypes.c_void_p * (2 * nph))(*[evv[i * 2 * nph + j].cuda_event for j in range(2 * nph)])
                  for i in range(args.steps)]
            v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            v0.record(stream)
            for i in range(args.steps):
                P.ffn24_step(X, Wu, bu, Wd, bd, dY, out=out_v, workspace=ws_v, vnm=(VV, VM), events=hv[i])
            v1.record(stream)
            torch.cuda.synchronize(dev)
            if P.p24_query_status() != 0:
                raise RuntimeError("device status word set during the V:N:M steps")
            vms = v0.elapsed_time(v1) / args.steps
            vph = [statistics.mean(evv[i * 2 * nph + 2 * q].elapsed_time(evv[i * 2 * nph + 2 * q + 1])
                                   for i in range(args.steps)) for q in range(nph)]
            down_ms = vph[3]
            kc = 4 * w.ffn // VM                     # condensed reduction length of the down GEMM
            executed = 2 * w.M * w.d * kc             # dense-equivalent FLOP of the condensed product
            vnm = {"V": VV, "M": VM, "ms_per_step": vms, "value": flop / (vms * 1e-3) / 1e12,
                   "unit": "TFLOPS (dense-equivalent of the dense FFN step)",
                   "speedup_vs_2to4_step": ms_step / vms, "phase_ms": dict(zip(P.STEP_PHASE_NAMES, vph)),
                   "down_gemm": {"kernel": "spmm_kernel gathered-B (vnm24_spmm)", "ms": down_ms,
                                 "dense_equiv_tflops": gemm_flop / (down_ms * 1e-3) / 1e12,
                                 "achieved": executed / (down_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                                 "peak": sparse_peak, "frac": executed / (down_ms * 1e-3) / 1e12 / sparse_peak,
                                 "note": "achieved counts the condensed product 2*M*d*(4*ffn/M_group) at the "
                                         "2:4 sparse rate; dense_equiv counts 2*M*d*ffn"}}
            del out_v, ws_v
            # the V:2:M prune of an H-shaped activation, masked in place, on its own
            Hv = torch.relu(normal_bf16((w.M, w.ffn), 1.0, seed, 7, dev))
            ci, hs = P.vnm24_compress(Hv, VV, VM)
            for _ in range(args.warmup):
                P.vnm24_compress(Hv, VV, VM, out=hs, colidx=ci, A_masked=Hv)
            p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            p0.record(stream)
            for _ in range(args.steps):
                P.vnm24_compress(Hv, VV, VM, out=hs, colidx=ci, A_masked=Hv)
            p1.record(stream)
            torch.cuda.synchronize(dev)
            pms = p0.elapsed_time(p1) / args.steps
            per_elt = 2 + 2 + 4 / VM + 0.5 / VM + 4 / (VV * VM)   # read, masked write, values, nibbles, offsets
            gbs = per_elt * Hv.numel() / (pms * 1e-3) / 1e9
            vnm["prune_H"] = {"ms": pms, "value": gbs, "unit": "GB/s", "frac_hbm": gbs / peaks["hbm_gbs"],
                              "algorithmic_bytes_per_elt": per_elt, "shape": [w.M, w.ffn]}
            del Hv, ci, hs
        except Exception as exc:  # a failure here must not cost the bench line
            vnm = {"error": f"{type(exc).__name__}: {exc}"}
        torch.cuda.empty_cache()

    # ---- hybrid ELL + dense-overflow activations: format and its two training products
    #      on the 1.3B FFN shape (8192 tokens x 8192 hidden units, d = 2048)
    hyb = None
    if not args.no_hybrid:
        try:
            hyb = bench_hybrid(P, dev, stream, seed, args, peaks)
        except Exception as exc:  # a failure here must not cost the bench line
            hyb = {"error": f"{type(exc).__name__}: {exc}"}
        torch.cuda.empty_cache()

    # ---- a short step (GPT-2-size FFN), eager against a CUDA-graph replay: the
    #      per-launch host work that a graph removes
    graphs = None
    if not args.no_graphs:
        from semi_structured_sparse_prune24_gb300.graph import StepGraph
        ws_small = WORKLOADS["gpt2"]
        small = ffn_inputs(ws_small, seed=seed, device=dev, bias=True)
        g = StepGraph(small, act24=False)
        n_rep = 50

        def timed(fn):
            for _ in range(5):
                fn()
            t0_, t1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            t0_.record(g.stream)
            for _ in range(n_rep):
                fn()
            t1_.record(g.stream)
            torch.cuda.synchronize(dev)
            return t0_.elapsed_time(t1_) / n_rep

        ws_e = torch.empty(P.ffn24_workspace_size(ws_small.M, ws_small.d, ws_small.ffn), dtype=torch.uint8, device=dev)
        eager_out = P.ffn24_step(small["X"], small["W_up"], small["b_up"], small["W_down"], small["b_down"],
                                 small["dY"], workspace=ws_e, stream=g.stream)
        eager_ms = timed(lambda: P.ffn24_step(small["X"], small["W_up"], small["b_up"], small["W_down"], small["b_down"],
                                              small["dY"], out=eager_out, workspace=ws_e, stream=g.stream))
        graph_ms = timed(g.replay)
        graphs = {"workload": ws_small.name, "eager_ms_per_step": eager_ms, "graph_ms_per_step": graph_ms,
                  "graph_value": ws_small.dense_equiv_flop / (graph_ms * 1e-3) / 1e12,
                  "eager_value": ws_small.dense_equiv_flop / (eager_ms * 1e-3) / 1e12,
                  "unit": "TFLOPS (dense-equivalent)", "note": "back-to-back steps on resident inputs, L2-warm"}
        del g, small, eager_out, ws_e
        torch.cuda.empty_cache()

    # ---- the other configurations, one GPU each (inputs resident, same timing)
    configs = None
    if not args.no_sweep:
        configs = {}

        def time_calls(fn):
            for _ in range(args.warmup):
                fn()
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            c0.record(stream)
            for _ in range(args.steps):
                fn()
            c1.record(stream)
            torch.cuda.synchronize(dev)
            return c0.elapsed_time(c1) / args.steps

        for key in ("gpt2", "1p3b", "7b_act24", "70b_m2048", "70b_m8192", "70b_tail"):
            cw = WORKLOADS[key]
            ci = ffn_inputs(cw, seed=seed, device=dev, bias=False)
            cws = torch.empty(P.ffn24_workspace_size(cw.M, cw.d, cw.ffn, cw.act24), dtype=torch.uint8, device=dev)
            co = P.ffn24_step(ci["X"], ci["W_up"], ci["b_up"], ci["W_down"], ci["b_down"], ci["dY"], act24=cw.act24,
                              workspace=cws)
            cms = time_calls(lambda: P.ffn24_step(ci["X"], ci["W_up"], ci["b_up"], ci["W_down"], ci["b_down"], ci["dY"],
                                                  act24=cw.act24, out=co, workspace=cws))
            cv = cw.dense_equiv_flop / (cms * 1e-3) / 1e12
            configs[cw.name] = {"ms_per_step": cms, "value": cv, "pct_sparse_peak": cv / sparse_peak,
                                "dense_equiv_flop": cw.dense_equiv_flop,
                                "e2e": config_e2e(P, cw, ci, co, dev, stream, args)}
            del ci, cws, co
        # single linears (prune + forward + double-pruned dX + masked dW): the 70B tail
        # shape and the tiny check
        for name, (lm, ln, lk) in (("ffn_70b_tail_linear_M1000_K8200_N28672", (1000, 28672, 8200)),
                                   ("tiny_single_linear_N256_K512_M128", (128, 256, 512))):
            lx = normal_bf16((lm, lk), 1.0, seed, 1, dev)
            lw = normal_bf16((ln, lk), 0.01, seed, 2, dev)
            ldy = normal_bf16((lm, ln), 1.0, seed, 6, dev)
            fwd, bwdT = P.Sparse24.empty(ln, lk, dev), P.Sparse24.empty(lk, ln, dev)
            ly = torch.empty((lm, ln), dtype=torch.bfloat16, device=dev)
            ldx = torch.empty((lm, lk), dtype=torch.bfloat16, device=dev)
            ldw = torch.empty((ln, lk), dtype=torch.bfloat16, device=dev)

            def linear_step():
                P.prune24_compress_both(lw, fwd, bwdT)
                P.spmm24_fwd(lx, fwd, Y=ly)
                P.spmm24_bwd_dx(ldy, bwdT, dX=ldx)
                P.masked_dw_gemm(ldy, lx, fwd, dW=ldw)
            lms = time_calls(linear_step)
            lf = 6 * lm * ln * lk
            lv = lf / (lms * 1e-3) / 1e12
            configs[name] = {"ms_per_step": lms, "value": lv, "pct_sparse_peak": lv / sparse_peak,
                             "dense_equiv_flop": lf}
            del lx, lw, ldy, fwd, bwdT, ly, ldx, ldw
        torch.cuda.empty_cache()

    # ---- standalone prune of 1e9 bf16 ([31250, 32000]), HBM-bound
    prune = None
    if not args.no_prune:
        del ws
        torch.cuda.empty_cache()
        Wp = normal_bf16((31250, 32000), 0.01, seed, 2, dev)
        sp = P.Sparse24.empty(31250, 32000, dev)
        for _ in range(args.warmup):
            P.prune24_compress(Wp, sp)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            P.prune24_compress(Wp, sp)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        pms = e0.elapsed_time(e1) / args.steps
        gbs = 3.125e9 / (pms * 1e-3) / 1e9
        prune = {"value": gbs, "unit": "GB/s", "ms": pms, "frac_hbm": gbs / peaks["hbm_gbs"],
                 "elements": 31250 * 32000, "algorithmic_bytes_per_elt": 3.125,
                 "note": "input 2 GB > L2, no flush needed"}
        del Wp, sp
        torch.cuda.empty_cache()
        # ---- V:2:M prune (128:2:8, 75% sparse) of a W_up-shaped weight [ffn, d]
        try:
            Wv = normal_bf16((w.ffn, w.d), w.w_sigma, seed, 2, dev)
            ci, vs = P.vnm24_compress(Wv, 128, 8)
            for _ in range(args.warmup):
                P.vnm24_compress(Wv, 128, 8, out=vs, colidx=ci)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for _ in range(args.steps):
                P.vnm24_compress(Wv, 128, 8, out=vs, colidx=ci)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            vms = e0.elapsed_time(e1) / args.steps
            # read 2 B; write 2 of every 8 values (0.5 B) and one nibble per 8 (0.0625 B); 4 B per 128 x 8 block
            per_elt = 2 + 0.5 + 0.0625 + 4 / (128 * 8)
            vgbs = per_elt * Wv.numel() / (vms * 1e-3) / 1e9
            prune["vnm_128_2_8"] = {"value": vgbs, "unit": "GB/s", "ms": vms, "frac_hbm": vgbs / peaks["hbm_gbs"],
                                    "shape": [w.ffn, w.d], "algorithmic_bytes_per_elt": per_elt,
                                    "note": f"vnm24_compress, input {Wv.numel() * 2 >> 20} MB" +
                                            (" > L2, no flush needed" if Wv.numel() * 2 > L2_BYTES else
                                             " (fits in L2: L2-warm)")}
            del Wv, ci, vs
        except Exception as exc:  # a failure here must not cost the bench line
            prune["vnm_128_2_8"] = {"error": f"{type(exc).__name__}: {exc}"}
        torch.cuda.empty_cache()
        ws = torch.empty(P.ffn24_workspace_size(w.M, w.d, w.ffn, w.act24), dtype=torch.uint8, device=dev)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hin = {k: v.cpu().pin_memory() for k, v in (("X", X), ("W_up", Wu), ("W_down", Wd), ("dY", dY))}
        hout = {k: torch.empty(out[k].shape, dtype=out[k].dtype).pin_memory()
                for k in ("Y", "dX", "dW_up", "dW_down", "db_up", "db_down")}
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        d2h = sum(t.numel() * t.element_size() for t in hout.values())
        # the package's StepPipeline: two device slots, copies on their own streams,
        # overlapped with the previous / next step's compute
        from semi_structured_sparse_prune24_gb300.pipeline import StepPipeline
        del ws
        torch.cuda.empty_cache()
        pipe = StepPipeline(w.M, w.d, w.ffn, act24=w.act24, b_up=bu, b_down=bd, device=dev)
        for _ in range(args.warmup):
            pipe.submit(hin, hout)
        pipe.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        pipe.start_after(e0)
        for _ in range(args.steps):
            pipe.submit(hin, hout)
        pipe.finish_on(stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        if P.p24_query_status() != 0:
            raise RuntimeError("device status word set during the end-to-end steps")
        ems = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
        # the copies alone, each direction on its own (what the overlap has to hide)
        def copy_ms(fn, s_):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            c0.record(s_)
            with torch.cuda.stream(s_):
                fn()
            c1.record(s_)
            torch.cuda.synchronize(dev)
            return c0.elapsed_time(c1)
        cin = copy_ms(lambda: [pipe.inputs[0][k].copy_(hin[k], non_blocking=True) for k in hin], pipe.s_in)
        cout = copy_ms(lambda: [hout[k].copy_(pipe.outputs[0][k], non_blocking=True) for k in hout], pipe.s_out)
        del pipe
        torch.cuda.empty_cache()
        e2e = {"value": world * flop / (ems * 1e-3) / 1e12, "unit": "TFLOPS (dense-equivalent)", "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "copy_in_ms_alone": cin, "copy_out_ms_alone": cout,
               "copy_in_gbs": h2d / (cin * 1e-3) / 1e9, "copy_out_gbs": d2h / (cout * 1e-3) / 1e9,
               "note": "pinned host X, dY, W_up, W_down copied in and Y, dX, dW_up, dW_down, db copied out every "
                       "step through the package's StepPipeline (copy-in, compute and copy-out streams, two device "
                       "slots: the copies of neighbouring steps overlap the compute)"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": "sparse FFN fwd+bwd dense-equiv TFLOPS, % of 2:4 bf16 TC peak; prune GB/s",
            "value": value, "unit": "TFLOPS (dense-equivalent)", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "pct_sparse_peak": value / world / sparse_peak,
            # composite roofline: four sparse GEMMs at the sparse rate, two dW GEMMs at the dense rate
            "pct_composite_roofline": (4 * gemm_flop / (sparse_peak * 1e12) + 2 * gemm_flop / (dense_peak * 1e12))
            / (ms_step * 1e-3),
            "config": {"workload": w.name, "M": w.M, "d": w.d, "ffn": w.ffn, "reprune_every_step": w.reprune,
                       "act24": w.act24, "global_batch": w.M * world,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": f"inputs larger than L2 ({L2_BYTES // 2 ** 20} MB): X {X.numel() * 2 >> 20} MB, "
                             f"W_up/W_down {Wu.numel() * 2 >> 20} MB each; no flush between steps"},
            "phase_ms": dict(zip(P.STEP_PHASE_NAMES, phase_ms)),
            "kernels": breakdown,
            "roofline": roofline,
            "slope_adapters": slope,
            "vnm_activations": vnm,
            "hybrid_activations": hyb,
            "graphs": graphs,
            "configs": configs,
            "prune": prune,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
            "peaks": {"source": peak_src, **peaks, "sparse_ratio": SPARSE_RATIO},
        }
        print(json.dumps(line))


# ------------------------------------------------------------------ reference arm (CPU oracle)
def run_reference(args, world, rank):
    from synth24 import WORKLOADS
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    m_s, f_s = 512, 512
    for _ in range(args.warmup):
        oracle_sample_step(w.d, m_s, f_s, w.w_sigma)
    times = [oracle_sample_step(w.d, m_s, f_s, w.w_sigma) for _ in range(args.steps)]
    t = statistics.mean(times)
    flop = 12 * m_s * w.d * f_s
    value = flop / t / 1e12
    sample = (f"oracle ffn_step on a slice of the workload: {m_s} tokens x {f_s} hidden units at d={w.d} "
              f"(numpy, BLAS on all visible cores)")
    print(json.dumps({
        "impl": "reference",
        "metric": "sparse FFN fwd+bwd dense-equiv TFLOPS, % of 2:4 bf16 TC peak; prune GB/s",
        "value": value, "unit": "TFLOPS (dense-equivalent)", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 accumulate on bf16 inputs", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "d": w.d, "ffn": w.ffn, "sample_tokens": m_s,
                   "sample_hidden": f_s},
        "cpu_baseline": {"value": value, "unit": "TFLOPS (dense-equivalent)", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS (dense-equivalent)", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="70b_m16384")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prune", action="store_true")
    ap.add_argument("--no-adapters", action="store_true")
    ap.add_argument("--no-graphs", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-vnm", action="store_true")
    ap.add_argument("--no-hybrid", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
