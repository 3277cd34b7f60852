"""Benchmark of the fused tensor-product convolution forward (tp_conv_forward).

One step = one pass of the whole hot path (segment lookup, gather, per-edge
weight/harmonic stream, fused all-path contraction, segmented sum and store)
over the medium workload: N=4096 nodes of a radius graph (r=5, mean degree
32, E=131064 destination-sorted edges), 128x0e+128x1o+128x2e features,
harmonics 0e+1o+2e+3o, fp32, per-edge weights N(0,1)/sqrt(13).

Prints ONE JSON line (rank 0). Inputs are synthetic (seeded), resident in HBM
before the timed region; the per-step input (0.92 GB, dominated by the weight
stream) is larger than the 129 MB L2, so no flush is needed.

  python bench.py [--steps K] [--warmup W] [--workload medium|large|xlarge|tiny]
  python bench.py --impl reference      # the fp64 CPU oracle timed on the host cores
  torchrun --nproc-per-node N bench.py --gpus N   # N independent replicas (weak scaling)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "edges/sec of fused TP-conv forward; achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="medium", choices=["tiny", "medium", "large", "xlarge"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU-oracle sample time")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-backward", action="store_true", help="skip the backward timing (medium only)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no measured peaks file)"


def source_hash() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "equivariant_gnn_tensor_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


def build_inputs(wname: str, seed: int, tpc, torch, device):
    """Synthetic inputs of a workload, resident on `device`."""
    from workloads import WORKLOADS, make_features, make_graph
    wl = WORKLOADS[wname]
    desc = tpc.tp_desc_create(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    rng, src, dst, vec, n = make_graph(wl, seed)
    E = len(src)
    x, w, _ = make_features(rng, wl, n, E, desc.dim_x, desc.weight_numel, desc.n_paths, desc.dim_out,
                            dtype=np.float32)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    d_dst = torch.as_tensor(dst).to(device)
    perm, row_ptr, _ = tpc.tp_csr_build(d_dst, n)
    p = perm.long()
    d_vec = torch.as_tensor(vec.astype(np.float32)).to(device)[p].contiguous()
    sh = tpc.tp_spherical_harmonics(desc, d_vec, normalize=True)
    inputs = dict(
        x=torch.as_tensor(x).to(device).to(tdt).contiguous(),
        w=torch.as_tensor(w).to(device)[p].to(tdt).contiguous(),
        sh=sh,
        src=torch.as_tensor(src).to(device)[p].contiguous(),
        row_ptr=row_ptr,
    )
    torch.cuda.synchronize()
    return wl, desc, inputs, n, E, (x, w, src, dst, vec)


def algorithmic_bytes(desc, n, E, esz):
    """Compulsory bytes of one forward: w, sh, src, one read of x, one write of
    out, row pointers."""
    return (E * desc.weight_numel * esz + E * desc.dim_sh * 4 + E * 4 + n * desc.dim_x * esz
            + n * desc.dim_out * 4 + (n + 1) * 4)


def backward_bytes(desc, n, E):
    """Compulsory bytes of one fp32 backward: w read and dw written, sh read and
    dsh written, src and the source permutation, x and grad_out read, dx
    written, both row-pointer arrays."""
    return (2 * E * desc.weight_numel * 4 + 2 * E * desc.dim_sh * 4 + 2 * E * 4 + 3 * n * desc.dim_x * 4
            + 2 * (n + 1) * 4)


def time_backward(desc, inp, n, E, out, ws, stream, tpc, torch, steps: int = 200):
    """Backward (dx, dw, dsh) of the medium graph, the fwd+bwd configuration's
    second half: CUDA events over `steps` calls; returns the dict reported
    under "backward"."""
    gen = torch.Generator(device=out.device).manual_seed(7)
    go = torch.randn((n, desc.dim_out), device=out.device, generator=gen)
    counts = inp["row_ptr"][1:] - inp["row_ptr"][:-1]
    dst = torch.repeat_interleave(torch.arange(n, device=out.device, dtype=torch.int32), counts.long())
    src_perm, src_row_ptr, _ = tpc.tp_csr_build(inp["src"], n)
    dx = torch.empty((n, desc.dim_x), device=out.device)
    dw = torch.empty((E, desc.weight_numel), device=out.device)
    dsh = torch.empty((E, desc.dim_sh), device=out.device)

    def bwd():
        tpc.tp_conv_backward(desc, go, inp["x"], inp["sh"], inp["w"], inp["src"], dst, inp["row_ptr"], src_perm,
                             src_row_ptr, dx=dx, dw=dw, dsh=dsh, stream=stream)

    for _ in range(3):
        bwd()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        bwd()
    e1.record(stream)
    torch.cuda.synchronize()
    bwd_us = e0.elapsed_time(e1) / steps * 1e3
    if tpc.tp_device_status(reset=True) != 0:
        raise RuntimeError("device status set during the backward timing")
    nbytes = backward_bytes(desc, n, E)
    return {"bwd_us": bwd_us, "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (bwd_us * 1e-6) / 1e9,
            "steps": steps, "kernels": "seg_conv_kernel (dw, dsh by destination; dx by source)"}


def cpu_baseline(wl, host, n, target_s: float):
    """The oracle (plain C, fp64, OpenMP) on a bounded sample of destination
    rows of the same workload; returns (edges/s, cores, description)."""
    from oracle import cref, so3, tp
    x, w, src, dst, vec = host
    plan = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    cores = len(os.sched_getaffinity(0))
    order = np.argsort(dst, kind="stable")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(dst, minlength=n), out=row_ptr[1:])

    def run(rows, reps=1):
        sel = np.concatenate([order[row_ptr[r]:row_ptr[r + 1]] for r in rows]) if len(rows) else np.zeros(0, int)
        lrp = np.zeros(len(rows) + 1, dtype=np.int64)
        np.cumsum([row_ptr[r + 1] - row_ptr[r] for r in rows], out=lrp[1:])
        sh = so3.sh_concat([t.l for t in plan.irr_sh], vec[sel])
        xs = x.astype(np.float64)
        ws = w[sel].astype(np.float64)
        t0 = time.perf_counter()
        for _ in range(reps):
            cref.conv_forward(plan, xs, sh, ws, src[sel], lrp, len(rows), threads=cores)
        return time.perf_counter() - t0, len(sel)

    rows = np.arange(min(n, 32))
    dt, ne = run(rows)                       # warm-up + calibration
    scale = max(1.0, target_s / max(dt, 1e-3))
    k = int(min(n, max(32, len(rows) * scale)))
    rows = np.arange(k)
    dt, ne = run(rows)
    reps = 1
    if k == n and dt < 0.5 * target_s:      # the whole workload is quick: repeat it
        reps = int(min(200, max(1, target_s / max(dt, 1e-3))))
        dt, ne = run(rows, reps)
    what = f"first {k} destination rows" if k < n else f"all {n} destination rows"
    return ne * reps / dt, cores, f"{what} ({ne} edges) x {reps} of the workload, fp64 oracle, {dt:.1f} s"


def bench_reference(args):
    """--impl reference: the fp64 CPU oracle timed on the host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from workloads import WORKLOADS, make_features, make_graph
    from oracle import cref, so3, tp
    wl = WORKLOADS[args.workload]
    plan = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    rng, src, dst, vec, n = make_graph(wl, args.seed)
    E = len(src)
    x, w, _ = make_features(rng, wl, n, E, plan.dim_in, plan.weight_numel, plan.n_paths, plan.dim_out,
                            dtype=np.float32)
    cores = len(os.sched_getaffinity(0))
    order = np.argsort(dst, kind="stable")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(dst, minlength=n), out=row_ptr[1:])
    n_rows = min(n, 64)
    sel = order[:row_ptr[n_rows]]
    sh = so3.sh_concat([t.l for t in plan.irr_sh], vec[sel])
    xs, ws = x.astype(np.float64), w[sel].astype(np.float64)
    lrp = row_ptr[:n_rows + 1]
    steps = args.steps if args.steps is not None else 5
    for _ in range(max(1, args.warmup if args.warmup < 3 else 1)):
        cref.conv_forward(plan, xs, sh, ws, src[sel], lrp, n_rows, threads=cores)
    t0 = time.perf_counter()
    for _ in range(steps):
        cref.conv_forward(plan, xs, sh, ws, src[sel], lrp, n_rows, threads=cores)
    dt = time.perf_counter() - t0
    ne = len(sel)
    val = ne * steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "edges/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: N={n} E={E} {wl.irreps_in} x {wl.irreps_sh}",
                   "sample": f"first {n_rows} destination rows ({ne} edges) per step"},
        "cpu_baseline": {"value": val, "unit": "edges/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n_rows} destination rows ({ne} edges) of {args.workload}, fp64 C oracle"},
        "e2e": {"value": val, "unit": "edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import equivariant_gnn_tensor_gb300 as tpc

    wl, desc, inp, n, E, host = build_inputs(args.workload, args.seed + rank, tpc, torch, device)
    esz = 2 if wl.dtype == "bf16" else 4
    steps = args.steps if args.steps is not None else {"tiny": 20000, "medium": 6000, "large": 600,
                                                       "xlarge": 600}[args.workload]
    warmup = max(3, args.warmup)
    out = torch.empty((n, desc.dim_out), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    fdt = tpc.TP_BF16_IN_F32_OUT if wl.dtype == "bf16" else tpc.TP_F32
    ws_bytes = tpc.tp_conv_forward_workspace_size(desc, fdt, n, E)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device) if ws_bytes else None
    launches_per_step = 2 if ws_bytes else 1   # split kernel + partial merge, or the generic kernel

    def step():
        tpc.tp_conv_forward(desc, inp["x"], inp["sh"], inp["w"], inp["src"], inp["row_ptr"], n, out=out,
                            workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if tpc.tp_device_status(reset=True) != 0:
        raise RuntimeError("device status set during warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world, device)
    kernel_ms = ms_local / steps     # per step: the forward kernel (+ the tiny partial merge)
    value = E * steps * world / (ms / 1e3)

    # end to end through the public call with host buffers (pinned), copies inside the timed region
    pin = {k: v.cpu().pin_memory() for k, v in inp.items()}
    out_h = torch.empty_like(out, device="cpu").pin_memory()
    dev_bufs = {k: torch.empty_like(v) for k, v in inp.items()}
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = out.numel() * out.element_size()

    def e2e_step():
        for k in pin:
            dev_bufs[k].copy_(pin[k], non_blocking=True)
        tpc.tp_conv_forward(desc, dev_bufs["x"], dev_bufs["sh"], dev_bufs["w"], dev_bufs["src"],
                            dev_bufs["row_ptr"], n, out=out, workspace=ws, stream=stream)
        out_h.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    e2e_val = E * args.e2e_steps * world / (e2e_ms / 1e3)
    status = tpc.tp_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    peak, peak_src = measured_peaks()
    abytes = algorithmic_bytes(desc, n, E, esz)
    achieved = abytes / (kernel_ms * 1e-3) / 1e9
    key = f"fwd:{args.workload}"
    line = {
        "metric": METRIC, "value": value, "unit": "edges/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: N={n} E={E} {wl.irreps_in} x {wl.irreps_sh} -> {wl.irreps_out}",
                   "paths": desc.n_paths, "weight_numel": desc.weight_numel,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": f"per-step input {abytes / 1e9:.2f} GB > 129 MB L2 (no flush needed)"},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic(key), "algorithmic_bytes": abytes,
                     "kernel_us": kernel_ms * 1e3, "peak_source": peak_src},
        "e2e": {"value": e2e_val, "unit": "edges/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": steps * launches_per_step,
        "clocks": clocks,
    }
    if args.workload == "medium" and not args.no_backward and wl.dtype == "f32":
        bk = time_backward(desc, inp, n, E, out, ws, stream, tpc, torch)
        bk["frac"] = bk["achieved_gbs"] / peak
        line["backward"] = bk
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample = cpu_baseline(wl, host, n, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "edges/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
