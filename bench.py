"""Benchmark of the fused tensor-product convolution forward (tp_conv_forward).

One step = one pass of the whole hot path (segment lookup, gather, per-edge
weight/harmonic stream, fused all-path contraction, segmented sum and store)
over one workload. The headline line is the largest single-GPU workload, the
very large one: N=262144 nodes of a radius graph (r=5, mean degree 32,
E=8390944 destination-sorted edges), 32x0e+32x1o features, harmonics 0e+1o+2e,
outputs 32x0e+32x1o+32x2e, fp32, per-edge weights N(0,1) (8.29 GB of
compulsory bytes per step). The same JSON line embeds, each timed on its own,
the medium (fp32, 13 paths, mul 128) and large (bf16 x and w, 23 paths,
mul 64) workloads, the tiny workload's per-call latency, and the backward
(dx, dw, dsh) of the medium graph.

Prints ONE JSON line (rank 0). Inputs are synthetic (seeded), resident in HBM
before each timed region; every per-step input is larger than the 129 MB L2,
so no flush is needed.

  python bench.py [--steps K] [--warmup W] [--workload xlarge|large|medium|tiny]
                  [--configs medium,large,tiny | --configs ""]
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
    ap.add_argument("--workload", default="xlarge", choices=["tiny", "medium", "large", "xlarge"])
    ap.add_argument("--configs", default="xlarge_vec,xlarge_mlp,medium,medium_vec,medium_mlp,large,tiny",
                    help="other workloads timed into the same line (comma list; empty for none)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU-oracle sample time")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-backward", action="store_true", help="skip the backward timing (medium graph)")
    ap.add_argument("--backward-steps", type=int, default=100, help="timed calls of the backward")
    ap.add_argument("--no-symc", action="store_true", help="skip the symmetric contraction timing")
    ap.add_argument("--nodes", type=int, default=None,
                    help="node count of the headline workload (same graph recipe; for profiling small cases)")
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


def measured_sm_mhz() -> float:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p)).get("sm_max_mhz", 2070.0))
    return 2070.0


def source_hash(files) -> str:
    """Hash of the kernel sources a traffic figure was taken on (paths relative
    to the repository root)."""
    h = hashlib.sha256()
    for f in sorted(files):
        h.update(f.encode())
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current device code of that kernel (the files listed with it: kernel
    source, shared headers, instantiation file), else None."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(kernel_key)
    if not e or not all(os.path.exists(os.path.join(ROOT, f)) for f in e.get("files", [])):
        return None
    if not e.get("files") or e.get("source_hash") != source_hash(e["files"]):
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


NODES_OVERRIDE = {}  # workload -> node count (--nodes)


def build_inputs(wname: str, seed: int, tpc, torch, device):
    """Synthetic inputs of a workload, resident on `device`. Returns (wl, desc,
    inputs, n, E, host) with host = (x, w, src, dst, vec, grad_out) as drawn
    (grad_out None unless the workload has a backward)."""
    import dataclasses
    from workloads import WORKLOADS, make_features, make_graph
    wl = WORKLOADS[wname]
    if wname in NODES_OVERRIDE:   # the same graph recipe on fewer (or more) nodes, for profiling
        wl = dataclasses.replace(wl, n_nodes=NODES_OVERRIDE[wname])
    desc = tpc.tp_desc_create(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    rng, src, dst, vec, n = make_graph(wl, seed)
    E = len(src)
    x, w, g = make_features(rng, wl, n, E, desc.dim_x, desc.weight_numel, desc.n_paths, desc.dim_out,
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
    inputs["vec"] = d_vec      # destination-sorted edge vectors (tp_conv_forward_vec)
    torch.cuda.synchronize()
    return wl, desc, inputs, n, E, (x, w, src, dst, vec, g)


def backward_inputs(tpc, torch, inp, n, grad_out):
    """What tp_conv_backward needs beyond the forward's inputs: grad_out on the
    device, the sorted destination of every edge and the source CSR of the
    destination-sorted edge list (tp_csr_build of src)."""
    dev = inp["x"].device
    go = torch.as_tensor(grad_out).to(dev).contiguous()
    counts = inp["row_ptr"][1:] - inp["row_ptr"][:-1]
    dst = torch.repeat_interleave(torch.arange(n, device=dev, dtype=torch.int32), counts.long())
    src_perm, src_row_ptr, _ = tpc.tp_csr_build(inp["src"], n)
    return go, dst, src_perm, src_row_ptr


def describe(wl, n, E):
    return f"{wl.name}: N={n} E={E} {wl.irreps_in} x {wl.irreps_sh} -> {wl.irreps_out} ({wl.dtype})"


def algorithmic_bytes(desc, n, E, esz, from_vectors=False, radial=False):
    """Compulsory bytes of one forward: w (none when the radial network computes
    it in the kernel; its parameters instead), sh (or the 12-byte edge vectors
    when the harmonics are evaluated in the kernel), src, one read of x, one
    write of out, row pointers."""
    per_edge_h = 12 if from_vectors else desc.dim_sh * 4
    w_bytes = (16 * 2 + 17 * desc.weight_numel) * 4 if radial else E * desc.weight_numel * esz
    return (w_bytes + E * per_edge_h + E * 4 + n * desc.dim_x * esz + n * desc.dim_out * 4 + (n + 1) * 4)


def backward_bytes(desc, n, E, esz=4):
    """Compulsory bytes of one backward: w read (esz bytes an element) and dw
    written (float32), sh read and dsh written, src and the source
    permutation, x read (esz), grad_out read, dx written, both row-pointer
    arrays."""
    return (E * desc.weight_numel * (esz + 4) + 2 * E * desc.dim_sh * 4 + 2 * E * 4
            + n * desc.dim_x * (esz + 4) + n * desc.dim_out * 4 + 2 * (n + 1) * 4)


def time_backward(tpc, torch, desc, inp, n, E, grad_out, stream, steps: int = 100, bf16: bool = False):
    """Backward (dx, dw, dsh) of the medium graph with its own grad_out, the
    fwd+bwd configuration's second half: CUDA events over `steps` calls;
    returns the dict reported under "backward". With bf16, x and w are the
    same values rounded to bfloat16 (the gradients stay float32)."""
    go, dst, src_perm, src_row_ptr = backward_inputs(tpc, torch, inp, n, grad_out)
    dev = inp["x"].device
    if bf16:
        inp = dict(inp, x=inp["x"].to(torch.bfloat16), w=inp["w"].to(torch.bfloat16))
    dx = torch.empty((n, desc.dim_x), device=dev)
    dw = torch.empty((E, desc.weight_numel), device=dev)
    dsh = torch.empty((E, desc.dim_sh), device=dev)
    nb = tpc.tp_conv_backward_workspace_size(desc, tpc.TP_BF16_IN_F32_OUT if bf16 else tpc.TP_F32, n, E)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None

    def bwd():
        tpc.tp_conv_backward(desc, go, inp["x"], inp["sh"], inp["w"], inp["src"], dst, inp["row_ptr"], src_perm,
                             src_row_ptr, dx=dx, dw=dw, dsh=dsh, workspace=ws, stream=stream)

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
    nbytes = backward_bytes(desc, n, E, 2 if bf16 else 4)
    return {"bwd_us": bwd_us, "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (bwd_us * 1e-6) / 1e9,
            "steps": steps, "launches_per_call": 2,
            "kernels": ("ring_bwd_kernel (one pass by source: dx, dw, dsh) + carry_fixup_kernel (partial dx rows)"
                        if nb else "seg_conv_kernel (dw, dsh by destination; dx by source)")}


_BUILT = {}


class Forward:
    """One workload's inputs on the device and its forward call; with
    `from_vectors` the call is tp_conv_forward_vec (harmonics evaluated in the
    kernel from the 12-byte edge vectors)."""

    def __init__(self, wname, seed, tpc, torch, device, stream, from_vectors=False, radial=False):
        self.tpc, self.torch, self.stream = tpc, torch, stream
        key = (wname, seed)
        if key not in _BUILT:   # one set of device inputs per workload, shared by its variants
            _BUILT.clear()
            torch.cuda.empty_cache()
            _BUILT[key] = build_inputs(wname, seed, tpc, torch, device)
        self.wl, self.desc, inp, self.n, self.E, self.host = _BUILT[key]
        self.inp = dict(inp)
        self.vec = self.inp.pop("vec")
        self.from_vectors = from_vectors or radial
        self.radial = radial
        if radial:   # the weights come from the radial network in the kernel: no weight stream
            from workloads import make_radial_mlp
            self.mlp = [torch.as_tensor(a).to(device) for a in make_radial_mlp(seed, self.wl.wid, 16,
                                                                              self.desc.weight_numel)]
            del self.inp["w"]
        self.esz = 2 if self.wl.dtype == "bf16" else 4
        self.out = torch.empty((self.n, self.desc.dim_out), dtype=torch.float32, device=device)
        fdt = tpc.TP_BF16_IN_F32_OUT if self.wl.dtype == "bf16" else tpc.TP_F32
        ws_bytes = tpc.tp_conv_forward_workspace_size(self.desc, fdt, self.n, self.E)
        self.ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device) if ws_bytes else None
        # the warp-ring kernel + its partial-row merge, or the generic kernel alone
        self.launches_per_step = 2 if ws_bytes else 1
        self.abytes = algorithmic_bytes(self.desc, self.n, self.E, self.esz, self.from_vectors, radial)

    def step(self):
        i = self.inp
        if self.radial:
            self.tpc.tp_conv_forward_mlp(self.desc, i["x"], self.vec, *self.mlp, i["src"], i["row_ptr"], self.n,
                                         out=self.out, workspace=self.ws, stream=self.stream)
        elif self.from_vectors:
            self.tpc.tp_conv_forward_vec(self.desc, i["x"], self.vec, i["w"], i["src"], i["row_ptr"], self.n,
                                         out=self.out, workspace=self.ws, stream=self.stream)
        else:
            self.tpc.tp_conv_forward(self.desc, i["x"], i["sh"], i["w"], i["src"], i["row_ptr"], self.n, out=self.out,
                                     workspace=self.ws, stream=self.stream)

    def timed(self, steps, warmup, local, world=1, device=None):
        """CUDA-event time of `steps` back-to-back steps (ms, max over ranks)
        with nvidia-smi clocks sampled during the timed region."""
        torch = self.torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        if self.tpc.tp_device_status(reset=True) != 0:
            raise RuntimeError("device status set during warm-up")
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(self.stream)
        for _ in range(steps):
            self.step()
        ev1.record(self.stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        clocks = sampler.stop()
        ms_local = ev0.elapsed_time(ev1)
        if self.tpc.tp_device_status(reset=True) != 0:
            raise RuntimeError("device status set during the timed region")
        return max_over_ranks(ms_local, world, device), ms_local, clocks

    def roofline(self, kernel_ms, peak, peak_src, key):
        achieved = self.abytes / (kernel_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profiled_traffic(key), "algorithmic_bytes": self.abytes, "kernel_us": kernel_ms * 1e3,
                "peak_source": peak_src}

    def describe(self):
        extra = (", harmonics and weights (radial network Linear(1,16)-SiLU-Linear(16,P*mul)) from edge vectors"
                 if self.radial else (", harmonics from edge vectors" if self.from_vectors else ""))
        return describe(self.wl, self.n, self.E) + extra

    def fma_roofline(self, kernel_ms, sm_mhz):
        """Radial-network mode is bound by FP32 arithmetic: algorithmic FMAs per
        edge = 16 per weight (the second layer) + 16 (the first) + the
        contraction's distinct(i,k) + min(2la+1, 2lc+1) per path and channel,
        against 152 SMs x 128 FP32 lanes x the maximum SM clock."""
        from oracle import tp
        wl = self.wl
        plan = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
        contr = 0
        for P, C in zip(plan.paths, plan.cg):
            distinct = int(np.count_nonzero(np.any(C != 0, axis=1)))
            contr += (distinct + min(2 * P.la + 1, 2 * P.lc + 1)) * plan.mul
        per_edge = 16 * self.desc.weight_numel + 16 + contr
        fma = per_edge * self.E
        achieved = fma / (kernel_ms * 1e-3) / 1e12
        peak = 152 * 128 * sm_mhz * 1e6 / 1e12
        return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFMA/s", "frac": achieved / peak,
                "traffic": None, "fma_per_edge": per_edge, "kernel_us": kernel_ms * 1e3,
                "peak_source": f"derived: 152 SMs x 128 FP32 lanes x {sm_mhz:.0f} MHz (maximum SM clock)"}

    def e2e(self, steps):
        """The same forward through the public call with the inputs in pinned
        host memory: every step copies all its inputs host->device, makes the
        call and reads out back device->host, all inside the timed region. The
        steps are pipelined as a serving loop would run them: two device input
        sets, the copies on a stream of their own, so step k+1's host->device
        copies overlap step k's kernel and its device->host read (the call
        waits on its inputs' copies; a set is refilled only after the call
        that read it)."""
        torch = self.torch
        pin = {k: v.cpu().pin_memory() for k, v in self.inp.items()}
        out_h = torch.empty_like(self.out, device="cpu").pin_memory()
        sets = [{k: torch.empty_like(v) for k, v in self.inp.items()} for _ in range(2)]
        outs = [torch.empty_like(self.out) for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = self.out.numel() * self.out.element_size()
        compute, copy = self.stream, torch.cuda.Stream(device=self.out.device)
        ready = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]

        def upload(s):
            with torch.cuda.stream(copy):
                copy.wait_event(freed[s])
                for k in pin:
                    sets[s][k].copy_(pin[k], non_blocking=True)
                ready[s].record(copy)

        def call(s):
            compute.wait_event(ready[s])
            b = sets[s]
            self.tpc.tp_conv_forward(self.desc, b["x"], b["sh"], b["w"], b["src"], b["row_ptr"], self.n,
                                     out=outs[s], workspace=self.ws, stream=compute)
            freed[s].record(compute)
            with torch.cuda.stream(compute):
                out_h.copy_(outs[s], non_blocking=True)

        def run(n_steps):
            upload(0)
            for i in range(n_steps):
                if i + 1 < n_steps:
                    upload((i + 1) % 2)
                call(i % 2)

        for e in freed:
            e.record(compute)
        run(2)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(compute)
        copy.wait_event(e0)
        run(steps)
        compute.wait_stream(copy)
        e1.record(compute)
        torch.cuda.synchronize()
        # same inputs, same kernel and launch geometry: bitwise the resident-input result
        if not torch.equal(out_h, self.out.cpu()):
            raise RuntimeError("end-to-end result differs from the resident-input result")
        del pin, sets, outs
        return e0.elapsed_time(e1), h2d, d2h


def symmetric_contraction_bench(tpc, torch, device, stream, peak, peak_src, local, steps: int = 500):
    """The symmetric contraction of the lesson's MACE descriptor (32x0e+32x1o
    -> 32x0e, degrees 1..3) on N=1048576 nodes with 10 elements (x: 512 MiB,
    larger than L2): per step one read of x and the element indices, one
    write of out (the weights stay in L1/L2)."""
    N, n_el = 1048576, 10
    s = tpc.tp_symc_create("32x0e+32x1o", "32x0e", 3)
    g = torch.Generator(device=device).manual_seed(11)
    x = torch.randn((N, s.dim_in), device=device, generator=g)
    w = torch.randn((n_el, s.n_weights, s.mul), device=device, generator=g)
    el = torch.randint(0, n_el, (N,), device=device, dtype=torch.int32, generator=g)
    out = torch.empty((N, s.dim_out), device=device)
    for _ in range(5):
        tpc.tp_symmetric_contraction(s, x, w, el, out=out, stream=stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        tpc.tp_symmetric_contraction(s, x, w, el, out=out, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop()
    if tpc.tp_device_status(reset=True) != 0:
        raise RuntimeError("device status set during the symmetric contraction timing")
    us = e0.elapsed_time(e1) / steps * 1e3
    nbytes = N * (s.dim_in + s.dim_out + 1) * 4 + n_el * s.n_weights * s.mul * 4
    ach = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"symmetric contraction 32x0e+32x1o -> 32x0e, degrees 1..3, N={N}, {n_el} elements (fp32)",
            "value": N / (us * 1e-6), "unit": "nodes/s", "steps": steps, "kernel_us": us,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                         "traffic": None, "algorithmic_bytes": nbytes, "kernel_us": us, "peak_source": peak_src},
            "clocks": clk, "gpu_launches": steps,
            "kernel": "symc_jit (compiled at run time for this descriptor; the table kernel symc_kernel when "
                      "tp_set_tuning(disable_symc_jit=1))"}


def tiny_latency(tpc, torch, device, stream, calls: int = 20000):
    """The tiny workload (512 edges) is launch-bound: per-call device time
    (CUDA events over back-to-back calls) and per-call host time of the public
    Python call (wall clock, including the ctypes marshalling)."""
    f = Forward("tiny", 0, tpc, torch, device, stream)
    for _ in range(100):
        f.step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    t0 = time.perf_counter()
    for _ in range(calls):
        f.step()
    t1 = time.perf_counter()
    e1.record(stream)
    torch.cuda.synchronize()
    gpu_us = e0.elapsed_time(e1) / calls * 1e3
    return {"workload": f.describe(), "calls": calls, "us_per_call_device": gpu_us,
            "us_per_call_host": (t1 - t0) / calls * 1e6, "edges_per_s": f.E / (gpu_us * 1e-6),
            "launches_per_call": f.launches_per_step,
            "note": "launch-bound (0.53 MB of compulsory bytes): reported as latency, not against the roofline"}


def cpu_baseline(wl, host, n, target_s: float):
    """The oracle (plain C, fp64, OpenMP) on a bounded sample of destination
    rows of the same workload; returns (edges/s, cores, description)."""
    from oracle import cref, so3, tp
    x, w, src, dst, vec = host[:5]
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

    # the first destination rows holding at most 2^21 edges (bounded host
    # memory), repeated for about target_s seconds
    k = int(np.searchsorted(row_ptr, 1 << 21, side="right")) - 1
    k = max(1, min(n, k))
    rows = np.arange(k)
    dt, ne = run(rows)                       # warm-up + calibration
    reps = int(min(200, max(1, math.ceil(target_s / max(dt, 1e-3)))))
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
    # per step: the first destination rows holding at most 2^16 edges
    n_rows = max(1, min(n, int(np.searchsorted(row_ptr, 1 << 16, side="right")) - 1))
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
        "config": {"workload": describe(wl, n, E), "sample": f"first {n_rows} destination rows ({ne} edges) per step"},
        "cpu_baseline": {"value": val, "unit": "edges/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n_rows} destination rows ({ne} edges) of {args.workload}, fp64 C oracle"},
        "e2e": {"value": val, "unit": "edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


DEFAULT_STEPS = {"tiny": 20000, "medium": 2000, "large": 300, "xlarge": 500}


def bench_ours(args):
    if args.nodes:
        NODES_OVERRIDE[args.workload] = args.nodes
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import equivariant_gnn_tensor_gb300 as tpc

    stream = torch.cuda.current_stream(device)
    peak, peak_src = measured_peaks()
    warmup = max(3, args.warmup)

    # ---- headline workload -------------------------------------------------------
    f = Forward(args.workload, args.seed + rank, tpc, torch, device, stream)
    steps = args.steps if args.steps is not None else DEFAULT_STEPS[args.workload]
    ms, ms_local, clocks = f.timed(steps, warmup, local, world, device)
    kernel_ms = ms_local / steps
    value = f.E * steps * world / (ms / 1e3)
    e2e_ms, h2d, d2h = f.e2e(args.e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_val = f.E * args.e2e_steps * world / (e2e_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "edges/s", "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if f.wl.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": f.describe(), "paths": f.desc.n_paths, "weight_numel": f.desc.weight_numel,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": f"per-step input {f.abytes / 1e9:.2f} GB > 129 MB L2 (no flush needed)"},
        "hbm_gbs": f.abytes / (kernel_ms * 1e-3) / 1e9,
        "roofline": f.roofline(kernel_ms, peak, peak_src, f"fwd:{args.workload}"),
        "e2e": {"value": e2e_val, "unit": "edges/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": steps * f.launches_per_step,
        "clocks": clocks,
    }
    host, wl_head, head_n = f.host, f.wl, f.n
    del f
    torch.cuda.empty_cache()

    # ---- the other workloads, each timed on its own (single GPU runs only) --------
    if world == 1:
        cfgs = {}
        for name in [c for c in args.configs.split(",") if c and c != args.workload]:
            if name == "tiny":
                cfgs["tiny"] = tiny_latency(tpc, torch, device, stream)
                continue
            base, _, mode = name.partition("_")
            g = Forward(base, args.seed, tpc, torch, device, stream, from_vectors=mode == "vec",
                        radial=mode == "mlp")
            k = DEFAULT_STEPS[base]
            _, ms_c, clk = g.timed(k, warmup, local)
            cfgs[name] = {"workload": g.describe(), "value": g.E * k / (ms_c / 1e3), "unit": "edges/s",
                          "steps": k, "kernel_us": ms_c / k * 1e3,
                          "roofline": g.roofline(ms_c / k, peak, peak_src, f"fwd:{name}"), "clocks": clk,
                          "gpu_launches": k * g.launches_per_step}
            if mode == "mlp":   # arithmetic-bound: the FMA roofline, the byte one beside it
                cfgs[name]["roofline_bytes"] = cfgs[name]["roofline"]
                cfgs[name]["roofline"] = g.fma_roofline(ms_c / k, measured_sm_mhz())
            del g
            torch.cuda.empty_cache()
        line["configs"] = cfgs
        if not args.no_symc:
            line["symmetric_contraction"] = symmetric_contraction_bench(tpc, torch, device, stream, peak, peak_src,
                                                                        local)
        if not args.no_backward:
            # the fwd+bwd workload: the medium graph and features with its own grad_out
            b = Forward("fwdbwd", args.seed, tpc, torch, device, stream)
            bk = time_backward(tpc, torch, b.desc, b.inp, b.n, b.E, b.host[5], stream, steps=args.backward_steps)
            bk["frac"] = bk["achieved_gbs"] / peak
            bk["roofline"] = {"bound": "hbm", "achieved": bk["achieved_gbs"], "peak": peak, "unit": "GB/s",
                              "frac": bk["achieved_gbs"] / peak, "traffic": profiled_traffic("bwd:fwdbwd"),
                              "algorithmic_bytes": bk["algorithmic_bytes"], "kernel_us": bk["bwd_us"],
                              "peak_source": peak_src}
            bk["workload"] = b.describe()
            line["backward"] = bk
            bh = time_backward(tpc, torch, b.desc, b.inp, b.n, b.E, b.host[5], stream, steps=args.backward_steps,
                               bf16=True)
            bh["frac"] = bh["achieved_gbs"] / peak
            bh["workload"] = b.describe() + ", x and w rounded to bf16 (gradients fp32)"
            line["backward_bf16"] = bh
            del b
            torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample = cpu_baseline(wl_head, host, head_n, args.cpu_seconds)
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
