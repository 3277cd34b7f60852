"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times: the medium, large (bf16) and very large workloads are built exactly as
the benchmark builds them, the forward runs with its default workspace (the
warp-ring kernel), and sampled destination rows - random ones, the first, the
last and the one with the most edges - are recomputed one by one by the fp64 C
oracle from the host copies of the same inputs (the bf16 ones after the same
round-to-nearest-even), with harmonics from the oracle's own code."""
import os
import sys

import numpy as np
import pytest
import torch

from helpers import BF16_TOL, FP32_TOL, deg_tol, err
from oracle import cref, so3, tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


def _sample_rows(rng, row_ptr, n, k=48):
    deg = np.diff(row_ptr)
    rows = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    rows.update([0, n - 1, int(np.argmax(deg))])
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["medium", "large", "xlarge"])
def test_fullsize_sampled_rows(tpc, name):
    import bench
    dev = torch.device("cuda:0")
    wl, desc, inp, n, E, host = bench.build_inputs(name, 0, tpc, torch, dev)
    x, w, src, dst, vec, _ = host
    out = tpc.tp_conv_forward(desc, inp["x"], inp["sh"], inp["w"], inp["src"], inp["row_ptr"], n)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0

    plan = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    order = np.argsort(dst, kind="stable")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(dst, minlength=n), out=row_ptr[1:])
    rows = _sample_rows(np.random.default_rng(123), row_ptr, n)
    sel = np.concatenate([order[row_ptr[r]:row_ptr[r + 1]] for r in rows])
    lrp = np.zeros(len(rows) + 1, dtype=np.int64)
    np.cumsum(row_ptr[rows + 1] - row_ptr[rows], out=lrp[1:])
    if wl.dtype == "bf16":   # the values the GPU multiplies
        xs = torch.as_tensor(x).to(torch.bfloat16).double().numpy()
        ws = torch.as_tensor(w[sel]).to(torch.bfloat16).double().numpy()
    else:
        xs, ws = x.astype(np.float64), w[sel].astype(np.float64)
    sh = so3.sh_concat([t.l for t in plan.irr_sh], vec[sel].astype(np.float64))
    ref = cref.conv_forward(plan, xs, sh, ws, src[sel], lrp, len(rows))
    got = out[torch.as_tensor(rows, device=dev)].double().cpu().numpy()
    deg = row_ptr[rows + 1] - row_ptr[rows]
    assert err(got, ref) <= (BF16_TOL if wl.dtype == "bf16" else FP32_TOL)
    for g, r, d in zip(got, ref, deg):   # every row against its own magnitude
        if d:
            # bf16 inputs run on the tensor cores, which round the per-edge
            # matrices to bf16; fp32 inputs keep fp32 math throughout
            assert err(g, r) <= (BF16_TOL if wl.dtype == "bf16" else deg_tol(int(d)))
        else:
            assert not np.any(g)


def test_fullsize_radial_network_sampled_rows(tpc):
    """The very large workload through tp_conv_forward_mlp as bench.py times
    it (harmonics and the radial network Linear(1,16)-SiLU-Linear(16,224) of
    the float32 edge vectors evaluated in the kernel, the benchmark's
    workspace): sampled rows against the fp64 C oracle, with the oracle's
    radial network and harmonics of the same float32 vectors."""
    import bench
    from workloads import make_radial_mlp
    dev = torch.device("cuda:0")
    wl, desc, inp, n, E, host = bench.build_inputs("xlarge", 0, tpc, torch, dev)
    x, _, src, dst, vec, _ = host
    del inp["w"], inp["sh"]
    mlp = make_radial_mlp(0, wl.wid, 16, desc.weight_numel)
    ws = torch.empty(tpc.tp_conv_forward_workspace_size(desc, tpc.TP_F32, n, E), dtype=torch.uint8, device=dev)
    out = tpc.tp_conv_forward_mlp(desc, inp["x"], inp["vec"], *(torch.as_tensor(a).to(dev) for a in mlp),
                                  inp["src"], inp["row_ptr"], n, workspace=ws)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0

    plan = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    order = np.argsort(dst, kind="stable")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(dst, minlength=n), out=row_ptr[1:])
    rows = _sample_rows(np.random.default_rng(321), row_ptr, n)
    sel = np.concatenate([order[row_ptr[r]:row_ptr[r + 1]] for r in rows])
    lrp = np.zeros(len(rows) + 1, dtype=np.int64)
    np.cumsum(row_ptr[rows + 1] - row_ptr[rows], out=lrp[1:])
    v = vec[sel].astype(np.float32).astype(np.float64)
    ws_ref = tp.radial_mlp(v, *mlp)
    sh = so3.sh_concat([t.l for t in plan.irr_sh], v)
    ref = cref.conv_forward(plan, x.astype(np.float64), sh, ws_ref, src[sel], lrp, len(rows))
    got = out[torch.as_tensor(rows, device=dev)].double().cpu().numpy()
    deg = row_ptr[rows + 1] - row_ptr[rows]
    assert err(got, ref) <= FP32_TOL
    for g, r, d in zip(got, ref, deg):
        if d:
            assert err(g, r) <= deg_tol(int(d))
        else:
            assert not np.any(g)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
def test_backward_fwdbwd_fullsize(tpc, bf16):
    """The backward of the fwd+bwd configuration at its full size (the medium
    graph, N=4096, E=131064, 13 paths, mul 128, with its own grad_out), run
    exactly as bench.py times it (float32 x and w, and the same values rounded
    to bfloat16), checked on samples the fp64 C oracle recomputes from the host
    copies: about 50 dx rows (random ones, the first, the last and the source
    with the most edges) through the oracle's own source CSR, and about 2000
    edges of dw and dsh."""
    import bench
    dev = torch.device("cuda:0")
    wl, desc, inp, n, E, host = bench.build_inputs("fwdbwd", 0, tpc, torch, dev)
    x, w, src, dst, vec, g = host
    go, dst_d, sp, srp = bench.backward_inputs(tpc, torch, inp, n, g)
    xd, wd = inp["x"], inp["w"]
    if bf16:
        xd, wd = xd.to(torch.bfloat16), wd.to(torch.bfloat16)
        x = torch.as_tensor(x).to(torch.bfloat16).float().numpy()
        w = torch.as_tensor(w).to(torch.bfloat16).float().numpy()
    dx, dw, dsh = tpc.tp_conv_backward(desc, go, xd, inp["sh"], wd, inp["src"], dst_d, inp["row_ptr"], sp, srp)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0

    plan = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    order = np.argsort(dst, kind="stable")           # the oracle's own destination sort
    src_s, dst_s = src[order], dst[order]
    sh_s = so3.sh_concat([t.l for t in plan.irr_sh], vec[order].astype(np.float32).astype(np.float64))
    x64, w_s, g64 = x.astype(np.float64), w[order].astype(np.float64), g.astype(np.float64)
    rng = np.random.default_rng(321)

    edges = np.unique(np.concatenate([rng.choice(E, 2000, replace=False), [0, E - 1]]))
    rdw, rdsh = cref.conv_backward_edges(plan, x64, sh_s, w_s, g64, src_s, dst_s, edges=edges)
    ed = torch.as_tensor(edges, device=dev)
    assert err(dw[ed], rdw) <= FP32_TOL
    assert err(dsh[ed], rdsh) <= FP32_TOL

    sp_o, srp_o, _ = tp.csr_build(src_s, n)
    outdeg = np.diff(srp_o)
    rows = np.unique(np.concatenate([rng.choice(n, 48, replace=False), [0, n - 1, int(np.argmax(outdeg))]]))
    rdx = cref.conv_backward_dx(plan, sh_s, w_s, g64, dst_s, sp_o, srp_o, n, rows=rows)
    got = dx[torch.as_tensor(rows, device=dev)].double().cpu().numpy()
    assert err(got, rdx) <= FP32_TOL
    for gr, rr, d in zip(got, rdx, outdeg[rows]):
        if d:
            assert err(gr, rr) <= deg_tol(int(d))
        else:
            assert not np.any(gr)
