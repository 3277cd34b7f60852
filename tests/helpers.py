"""Shared helpers of the GPU parity tests: seeded problems, device transfer
through PyTorch, the library calls and the error measure.

Tolerances (max |gpu - oracle| / RMS(oracle), per output tensor):
FP32_TOL for float32 inputs and BF16_TOL for bfloat16 x and w, the bounds the
library promises. The current kernels compute in float32 on the same rounded
inputs the oracle consumes, so every test additionally holds them to FP32_TOL.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import so3, tp

FP32_TOL = 1e-5
BF16_TOL = 2e-2
DEV = "cuda"


def make_problem(irr_in, irr_sh, irr_out, n_src, n_dst, E, seed=0, dst=None, src=None, normalize=True):
    plan = tp.Plan(irr_in, irr_sh, irr_out)
    rng = np.random.default_rng(seed)
    if src is None:
        src = rng.integers(0, n_src, E)
    if dst is None:
        dst = rng.integers(0, n_dst, E)
    E = len(src)
    vec = rng.standard_normal((E, 3))
    sh = so3.sh_concat([t.l for t in plan.irr_sh], vec, normalize=normalize) if E else np.zeros((0, plan.dim_sh))
    x = rng.standard_normal((n_src, plan.dim_in))
    w = rng.standard_normal((E, plan.weight_numel))
    return dict(plan=plan, irreps=(irr_in, irr_sh, irr_out), n_src=n_src, n_dst=n_dst, src=np.asarray(src, np.int64),
                dst=np.asarray(dst, np.int64), vec=vec, sh=sh, x=x, w=w)


def dev_tensor(a, dtype=torch.float32):
    return torch.as_tensor(np.ascontiguousarray(a)).to(DEV).to(dtype).contiguous()


def rounded(a, dtype):
    """The values the GPU sees, as float64 numpy (float32 or RNE bfloat16)."""
    t = torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32)).to(dtype)
    return t.float().double().numpy()


def gpu_sorted_inputs(tpc, prob, dtype=torch.float32):
    """Move a problem to the GPU, destination-sort its edges with tp_csr_build
    and gather the per-edge arrays in that order."""
    d_dst = dev_tensor(prob["dst"], torch.int32)
    perm, row_ptr, dst_sorted = tpc.tp_csr_build(d_dst, prob["n_dst"])
    p = perm.long()
    x = dev_tensor(prob["x"], dtype)
    sh = dev_tensor(prob["sh"])[p].contiguous()
    w = dev_tensor(prob["w"], dtype)[p].contiguous()
    src = dev_tensor(prob["src"], torch.int32)[p].contiguous()
    return dict(x=x, sh=sh, w=w, src=src, row_ptr=row_ptr, dst=dst_sorted, perm=perm)


def oracle_forward(prob, dtype=torch.float32):
    pl = prob["plan"]
    return tp.conv_forward(pl, rounded(prob["x"], dtype), rounded(prob["sh"], torch.float32),
                           rounded(prob["w"], dtype), prob["src"], prob["dst"], prob["n_dst"])


def deg_tol(degree: int) -> float:
    """FP32_TOL for a row that sums `degree` edges in one sequential float32
    accumulation: the rounding of such a sum grows like sqrt(terms), so rows
    far above the workloads' degrees (<= 64) get sqrt(degree / 64) more room."""
    return FP32_TOL * max(1.0, (degree / 64.0) ** 0.5)


def err(got, ref):
    if isinstance(got, torch.Tensor):
        got = got.detach().double().cpu().numpy()
    return tp.rms_rel_err(got, ref)


class tuning:
    """Context manager: tp_set_tuning(**fields) inside the block, defaults after."""

    def __init__(self, tpc, **fields):
        self.tpc, self.fields = tpc, fields

    def __enter__(self):
        self.tpc.tp_set_tuning(**self.fields)
        return self

    def __exit__(self, *exc):
        self.tpc.tp_set_tuning()
        return False
