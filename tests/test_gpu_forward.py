"""GPU parity of tp_conv_forward against the fp64 oracle, element by element,
on seeded problems that span several chunks and warps with ragged tails, every
kernel shape and channel width, and the edge cases of the method (empty graph,
destinations without edges, unreachable output blocks, bipartite graphs,
out-of-range sources), plus run-to-run bitwise determinism."""
import numpy as np
import pytest
import torch

from helpers import (BF16_TOL, FP32_TOL, deg_tol, dev_tensor, err, gpu_sorted_inputs, make_problem, oracle_forward,
                     rounded, tuning)
from oracle import cref, so3, tp
from workloads import WORKLOADS, make_features, make_graph

pytestmark = pytest.mark.gpu


def run(tpc, prob, dtype=torch.float32, workspace="auto"):
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob, dtype)
    out = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"],
                              workspace=workspace)
    torch.cuda.synchronize()
    return out, desc, g


SHAPES = [
    ("32x0e+32x1o", "0e+1o+2e", "32x0e+32x1o+32x2e"),              # tiny / very large workloads
    ("128x0e+128x1o+128x2e", "0e+1o+2e+3o", "128x0e+128x1o+128x2e"),  # medium / fwd+bwd
    ("64x0e+64x1o+64x2e+64x3o", "0e+1o+2e+3o", "64x0e+64x1o+64x2e+64x3o"),  # large
    ("32x0e+32x1o", "0e+1o", "32x0e+32x1o"),                        # the lesson's worked example
    ("16x0+16x1+16x2", "0+1+2", "16x0+16x1+16x2"),                  # SO(3)
    ("8x0e+8x1o", "0e+1o+2e+3o", "8x0e+8x1o+8x2e+8x3o"),            # mul 8: most lanes idle
    ("40x2e+40x0e", "1o+0e+2e", "40x1o+40x2e+40x0e"),               # block order, mul 40
    ("96x1o", "0e+1o+2e", "96x0e+96x1e+96x2e"),                     # single input block, mul 96
    ("24x0e+24x2e", "0e+2e", "24x0e+24x2e+24x3o"),                  # missing degree, unreachable 3o
]


@pytest.mark.parametrize("workspace", ["auto", None], ids=["split", "generic"])
@pytest.mark.parametrize("irr", SHAPES, ids=lambda c: "|".join(c))
def test_forward_matches_oracle(tpc, irr, workspace):
    """With a workspace, shapes that have a compiled path program run the
    edge-balanced kernel (destinations cut across CTAs are merged from
    partials); without one, or for other shapes, the per-destination kernel."""
    prob = make_problem(*irr, n_src=300, n_dst=257, E=5000, seed=1)
    out, _, _ = run(tpc, prob, workspace=workspace)
    ref = oracle_forward(prob)
    assert err(out, ref) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


@pytest.mark.parametrize("workspace", ["auto", None], ids=["split", "generic"])
@pytest.mark.parametrize("irr", SHAPES[:3], ids=lambda c: "|".join(c))
def test_forward_bf16_inputs(tpc, irr, workspace):
    """bf16 inputs on the CUDA-core kernels: fp32 math on the same rounded
    inputs, so the fp32 bound holds too (the tensor-core kernel, which rounds
    the per-edge matrices to bf16, is disabled here; tests/test_gpu_mma.py)."""
    prob = make_problem(*irr, n_src=200, n_dst=190, E=3000, seed=2)
    with tuning(tpc, disable_mma=1):
        out, _, _ = run(tpc, prob, torch.bfloat16, workspace=workspace)
    ref = oracle_forward(prob, torch.bfloat16)
    e = err(out, ref)
    assert e <= BF16_TOL
    assert e <= FP32_TOL


def test_tiny_workload(tpc):
    wl = WORKLOADS["tiny"]
    rng, src, dst, vec, n = make_graph(wl)
    prob = make_problem(wl.irreps_in, wl.irreps_sh, wl.irreps_out, n, n, len(src), src=src, dst=dst)
    pl = prob["plan"]
    x, w, _ = make_features(rng, wl, n, len(src), pl.dim_in, pl.weight_numel, pl.n_paths, pl.dim_out)
    from oracle import so3
    prob.update(x=x, w=w, sh=so3.sh_concat([t.l for t in pl.irr_sh], vec))
    out, _, _ = run(tpc, prob)
    assert err(out, oracle_forward(prob)) <= FP32_TOL


@pytest.mark.parametrize("workspace", ["auto", None], ids=["split", "generic"])
def test_degree_extremes_and_empty_rows(tpc, workspace):
    """One destination with 1000 edges (many chunks, cut across several CTAs
    by the edge-balanced split), many with none, a ragged mix."""
    rng = np.random.default_rng(5)
    n_dst = 700
    dst = np.concatenate([np.full(1000, 3), rng.integers(0, n_dst // 2, 3000) * 2, [n_dst - 1]])
    rng.shuffle(dst)
    prob = make_problem(*SHAPES[1], n_src=50, n_dst=n_dst, E=len(dst), seed=6, dst=dst)
    out, _, _ = run(tpc, prob, workspace=workspace)
    ref = oracle_forward(prob)
    # destination 3 sums 1000 edges: measure every row against its own RMS (the
    # whole-tensor RMS, diluted by empty rows, understates its magnitude)
    on = out.double().cpu().numpy()
    for d, c in zip(*np.unique(dst, return_counts=True)):
        assert err(on[d], ref[d]) <= deg_tol(c), d
    empty = np.setdiff1d(np.arange(n_dst), dst)
    assert len(empty) > 100 and not out[torch.as_tensor(empty)].any()


def test_empty_graph_zeroes_output(tpc):
    prob = make_problem(*SHAPES[0], n_src=10, n_dst=33, E=0, seed=0)
    desc = tpc.tp_desc_create(*prob["irreps"])
    out = torch.full((33, desc.dim_out), 7.0, device="cuda")
    z = torch.zeros(0, device="cuda")
    row_ptr = torch.zeros(34, dtype=torch.int32, device="cuda")
    tpc.tp_conv_forward(desc, torch.zeros((10, desc.dim_x), device="cuda"), z.view(0, desc.dim_sh),
                        torch.zeros((0, desc.weight_numel), device="cuda"), torch.zeros(0, dtype=torch.int32,
                                                                                      device="cuda"),
                        row_ptr, 33, out=out)
    torch.cuda.synchronize()
    assert not out.any()


def test_bipartite_sources(tpc):
    """The gather/scatter example's shape: more sources than destinations."""
    prob = make_problem(*SHAPES[3], n_src=5000, n_dst=40, E=3000, seed=9)
    out, _, _ = run(tpc, prob)
    assert err(out, oracle_forward(prob)) <= FP32_TOL
    prob = make_problem(*SHAPES[3], n_src=3, n_dst=900, E=3000, seed=10)
    out, _, _ = run(tpc, prob)
    assert err(out, oracle_forward(prob)) <= FP32_TOL


@pytest.mark.parametrize("irr,dtype", [(SHAPES[0], torch.float32), (SHAPES[1], torch.float32),
                                       (SHAPES[2], torch.bfloat16), (SHAPES[3], torch.float32)],
                         ids=["tiny", "medium", "large-bf16", "lesson"])
def test_split_kernel_default_geometry(tpc, irr, dtype):
    """The warp-ring kernel in its default launch geometry against the oracle."""
    prob = make_problem(*irr, n_src=400, n_dst=333, E=9000, seed=14)
    with tuning(tpc, disable_mma=1):
        out, _, _ = run(tpc, prob, dtype)
    assert err(out, oracle_forward(prob, dtype)) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


RING_GEOMETRIES = {
    "eps1-S2-w1": dict(ring_stage_bytes=1, ring_stages=2, ring_warps=1),
    "eps30-S3": dict(ring_stage_bytes=1000000, ring_stages=3),
    "S8-w8": dict(ring_stages=8, ring_warps=8, ring_stage_bytes=4096),
    "rounds3": dict(ring_rounds=3),
    "rounds16-eps5": dict(ring_rounds=16, ring_stage_bytes=5000),
    "eps30-pack": dict(ring_stage_bytes=1000000, ring_pack=1),
    "nopack": dict(ring_pack=2),
    "rounds4-S4": dict(ring_rounds=4, ring_stages=4),
}


@pytest.mark.parametrize("geo", list(RING_GEOMETRIES))
@pytest.mark.parametrize("irr,dtype", [(SHAPES[0], torch.float32), (SHAPES[1], torch.float32),
                                       (SHAPES[2], torch.bfloat16)], ids=["cpt1", "cpt4", "cpt2-bf16"])
def test_ring_geometries(tpc, irr, dtype, geo):
    """The warp ring with chunks of 1 to 30 edges, 2 to 8 stages, 1 to 8 warps
    per block, several pieces per warp, packed or scalar FMAs, on a graph with a 1000-edge
    destination (cut across many pieces), empty destinations and a ragged tail."""
    rng = np.random.default_rng(21)
    n_dst = 500
    dst = np.concatenate([np.full(1000, 7), rng.integers(0, n_dst // 2, 5003) * 2, [n_dst - 1]])
    rng.shuffle(dst)
    prob = make_problem(*irr, n_src=300, n_dst=n_dst, E=len(dst), seed=22, dst=dst)
    with tuning(tpc, disable_mma=1, **RING_GEOMETRIES[geo]):
        out, _, _ = run(tpc, prob, dtype)
    ref = oracle_forward(prob, dtype)
    on = out.double().cpu().numpy()
    for d, c in zip(*np.unique(dst, return_counts=True)):
        assert err(on[d], ref[d]) <= deg_tol(c), d
    empty = np.setdiff1d(np.arange(n_dst), dst)
    assert len(empty) > 100 and not out[torch.as_tensor(empty)].any()
    assert tpc.tp_device_status(reset=True) == 0


def test_split_kernel_is_used_for_program_shapes(tpc):
    for irr in SHAPES[:4]:
        desc = tpc.tp_desc_create(*irr)
        assert tpc.tp_conv_forward_workspace_size(desc, tpc.TP_F32, 1000, 100000) > 0, irr
    desc = tpc.tp_desc_create(*SHAPES[4])   # SO(3): no compiled program
    assert tpc.tp_conv_forward_workspace_size(desc, tpc.TP_F32, 1000, 100000) == 0


def test_deterministic(tpc):
    prob = make_problem(*SHAPES[2], n_src=500, n_dst=480, E=16000, seed=11)
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob)
    a = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"])
    b = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_out_of_range_source_is_skipped_and_flagged(tpc):
    prob = make_problem(*SHAPES[0], n_src=64, n_dst=64, E=2000, seed=12)
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob)
    bad = g["src"].clone()
    bad[17] = 64
    bad[1000] = -5
    out = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], bad, g["row_ptr"], 64)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    # the other edges are unaffected: compare with the oracle minus the two bad edges
    keep = np.ones(2000, bool)
    perm = g["perm"].cpu().numpy()
    keep[perm[[17, 1000]]] = False
    sub = dict(prob)
    sub.update(src=prob["src"][keep], dst=prob["dst"][keep], sh=prob["sh"][keep], w=prob["w"][keep])
    assert err(out, oracle_forward(sub)) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


def test_bad_row_pointers_flagged(tpc):
    prob = make_problem(*SHAPES[0], n_src=64, n_dst=64, E=2000, seed=13)
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob)
    rp = g["row_ptr"].clone()
    rp[10] = 5000          # beyond E
    rp[20] = rp[19] - 1    # decreasing
    tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], rp, 64)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_SEGMENT


@pytest.mark.parametrize("mode", ["split", "generic"])
def test_wait_timeout_is_reported_and_writes_stay_in_bounds(tpc, mode):
    """A main-loop wait limit of 1 ns (tp_set_tuning) makes pipeline waits give
    up on real chunks whose copies are still in flight; every copy still lands,
    because the waits after a failure keep the full limit. The call returns,
    TP_DEV_ERR_TIMEOUT is reported, no byte outside `out` changes (guard rows
    around it keep their sentinel) although the split kernel runs several pieces
    per warp, and the next call with default settings is correct again."""
    irr = SHAPES[1]
    plan = tp.Plan(*irr)
    n, E = 4096, 100000
    rng = np.random.default_rng(50)
    dst = np.sort(rng.integers(0, n, E))
    src = rng.integers(0, n, E)
    x = rng.standard_normal((n, plan.dim_in), dtype=np.float32)
    w = rng.standard_normal((E, plan.weight_numel), dtype=np.float32)
    vec = rng.standard_normal((E, 3))
    sh = so3.sh_concat([t.l for t in plan.irr_sh], vec)
    desc = tpc.tp_desc_create(*irr)
    d_x, d_w, d_sh = dev_tensor(x), dev_tensor(w), dev_tensor(sh)
    d_src = dev_tensor(src, torch.int32)
    _, row_ptr, _ = tpc.tp_csr_build(dev_tensor(dst, torch.int32), n)
    guard = 97
    big = torch.full((n + 2 * guard, desc.dim_out), 12345.0, device="cuda")
    out = big[guard:guard + n]
    fields = dict(wait_limit_ns=1, ring_rounds=4) if mode == "split" else dict(wait_limit_ns=1, disable_split=1)
    hit = False
    for _ in range(3):
        with tuning(tpc, **fields):
            tpc.tp_conv_forward(desc, d_x, d_sh, d_w, d_src, row_ptr, n, out=out)
            torch.cuda.synchronize()
        st = tpc.tp_device_status(reset=True)
        assert st & ~tpc.TP_DEV_ERR_TIMEOUT == 0
        assert torch.all(big[:guard] == 12345.0) and torch.all(big[guard + n:] == 12345.0)
        hit = hit or bool(st & tpc.TP_DEV_ERR_TIMEOUT)
        if hit:
            break
    assert hit, "no pipeline wait ran out under a 1 ns limit"
    again = tpc.tp_conv_forward(desc, d_x, d_sh, d_w, d_src, row_ptr, n)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    rows = np.array([0, 1, 2, 777, 2048, n - 1])
    rp = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(np.bincount(dst, minlength=n), out=rp[1:])
    sel = np.concatenate([np.arange(rp[r], rp[r + 1]) for r in rows])
    lrp = np.zeros(len(rows) + 1, dtype=np.int64)
    np.cumsum(rp[rows + 1] - rp[rows], out=lrp[1:])
    sh32 = sh.astype(np.float32).astype(np.float64)
    ref = cref.conv_forward(plan, x.astype(np.float64), sh32[sel], w[sel].astype(np.float64), src[sel], lrp,
                            len(rows))
    assert err(again[torch.as_tensor(rows, device="cuda")], ref) <= FP32_TOL


@pytest.mark.parametrize("normalize", [True, False], ids=["unit", "raw"])
@pytest.mark.parametrize("irr,dtype", [(SHAPES[0], torch.float32), (SHAPES[1], torch.float32),
                                       (SHAPES[2], torch.bfloat16), (SHAPES[3], torch.float32)],
                         ids=["tiny", "medium", "large-bf16", "lesson"])
def test_forward_from_edge_vectors(tpc, irr, dtype, normalize):
    """tp_conv_forward_vec evaluates the harmonics in the kernel: against the
    oracle's own (Legendre-based, fp64) harmonics of the same float32 vectors,
    vectors of random length, several chunks per warp and a ragged tail."""
    prob = make_problem(*irr, n_src=300, n_dst=257, E=5003, seed=60, normalize=normalize)
    pl = prob["plan"]
    v32 = rounded(prob["vec"], torch.float32)
    prob["sh"] = so3.sh_concat([t.l for t in pl.irr_sh], v32, normalize=normalize)
    desc = tpc.tp_desc_create(*irr)
    g = gpu_sorted_inputs(tpc, prob, dtype)
    vec = dev_tensor(prob["vec"])[g["perm"].long()].contiguous()
    out = tpc.tp_conv_forward_vec(desc, g["x"], vec, g["w"], g["src"], g["row_ptr"], prob["n_dst"],
                                  normalize=normalize)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    assert err(out, oracle_forward(prob, dtype)) <= FP32_TOL


def test_forward_from_edge_vectors_needs_a_compiled_kernel(tpc):
    prob = make_problem(*SHAPES[4], n_src=20, n_dst=20, E=100, seed=61)
    desc = tpc.tp_desc_create(*SHAPES[4])
    g = gpu_sorted_inputs(tpc, prob)
    vec = dev_tensor(prob["vec"])
    with pytest.raises(tpc.TPError) as ei:
        tpc.tp_conv_forward_vec(desc, g["x"], vec, g["w"], g["src"], g["row_ptr"], prob["n_dst"])
    assert tpc.STATUS_NAMES[ei.value.status] == "TP_ERR_UNSUPPORTED"


@pytest.mark.parametrize("irr", [SHAPES[0], SHAPES[1], SHAPES[2], SHAPES[3]], ids=["tiny", "medium", "large", "lesson"])
def test_forward_with_radial_network(tpc, irr):
    """tp_conv_forward_mlp computes the weights in the kernel from the edge
    length (Linear(1,16) -> SiLU -> Linear(16, P*mul)) and the harmonics from
    the vectors: against the oracle's radial network and harmonics (fp64) of
    the same float32 inputs."""
    from workloads import make_radial_mlp
    prob = make_problem(*irr, n_src=300, n_dst=257, E=4001, seed=62)
    pl = prob["plan"]
    w1, b1, w2, b2 = make_radial_mlp(62, 0, 16, pl.weight_numel)
    v32 = rounded(prob["vec"], torch.float32)
    prob["w"] = tp.radial_mlp(v32, w1, b1, w2, b2)
    prob["sh"] = so3.sh_concat([t.l for t in pl.irr_sh], v32)
    desc = tpc.tp_desc_create(*irr)
    g = gpu_sorted_inputs(tpc, prob)
    vec = dev_tensor(prob["vec"])[g["perm"].long()].contiguous()
    out = tpc.tp_conv_forward_mlp(desc, g["x"], vec, dev_tensor(w1), dev_tensor(b1), dev_tensor(w2), dev_tensor(b2),
                                  g["src"], g["row_ptr"], prob["n_dst"])
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    ref = tp.conv_forward(pl, rounded(prob["x"], torch.float32), prob["sh"], prob["w"], prob["src"], prob["dst"],
                          prob["n_dst"])
    assert err(out, ref) <= FP32_TOL


RADIAL_GEOMETRIES = {
    "default": {},
    "eps1-S2-w1": dict(ring_stage_bytes=1, ring_stages=2, ring_warps=1),
    "eps3-S4": dict(ring_stage_bytes=1500, ring_stages=4),
    "S8-w8": dict(ring_stages=8, ring_warps=8),
    "rounds5": dict(ring_rounds=5),
    "nopack": dict(ring_pack=2),
}


@pytest.mark.parametrize("geo", list(RADIAL_GEOMETRIES))
@pytest.mark.parametrize("irr", [SHAPES[0], SHAPES[3]], ids=["cpt1", "lesson"])
def test_radial_network_geometries(tpc, irr, geo):
    """The radial-network forward with edge pairs (a chunk's weights formed in
    registers from the block's copy of the second layer) in chunks of 1, 3 and
    8 edges, 2 to 8 stages, 1 to 8 warps, several pieces per warp, and the
    one-edge-at-a-time kernel (nopack), on a graph with a 1000-edge destination
    cut across pieces, destinations of one edge between longer ones (pairs
    split across destinations), empty destinations and a ragged tail: every
    row against the oracle's radial network and harmonics (fp64) of the same
    float32 inputs."""
    from workloads import make_radial_mlp
    rng = np.random.default_rng(77)
    n_dst = 500
    dst = np.concatenate([np.full(1000, 7), rng.integers(0, n_dst // 2, 5003) * 2, [n_dst - 1],
                          np.arange(1, 60, 2)])
    rng.shuffle(dst)
    prob = make_problem(*irr, n_src=300, n_dst=n_dst, E=len(dst), seed=78, dst=dst)
    pl = prob["plan"]
    w1, b1, w2, b2 = make_radial_mlp(78, 0, 16, pl.weight_numel)
    v32 = rounded(prob["vec"], torch.float32)
    prob["w"] = tp.radial_mlp(v32, w1, b1, w2, b2)
    prob["sh"] = so3.sh_concat([t.l for t in pl.irr_sh], v32)
    desc = tpc.tp_desc_create(*irr)
    g = gpu_sorted_inputs(tpc, prob)
    vec = dev_tensor(prob["vec"])[g["perm"].long()].contiguous()
    with tuning(tpc, disable_mma=1, **RADIAL_GEOMETRIES[geo]):
        out = tpc.tp_conv_forward_mlp(desc, g["x"], vec, dev_tensor(w1), dev_tensor(b1), dev_tensor(w2),
                                      dev_tensor(b2), g["src"], g["row_ptr"], n_dst)
        torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    ref = tp.conv_forward(pl, rounded(prob["x"], torch.float32), prob["sh"], prob["w"], prob["src"], prob["dst"],
                          n_dst)
    on = out.double().cpu().numpy()
    for d, c in zip(*np.unique(dst, return_counts=True)):
        assert err(on[d], ref[d]) <= deg_tol(c), d
    empty = np.setdiff1d(np.arange(n_dst), dst)
    assert len(empty) > 100 and not out[torch.as_tensor(empty)].any()


def test_radial_network_out_of_range_source(tpc):
    """An edge whose source is out of range adds nothing and sets
    TP_DEV_ERR_INDEX; the other edges match the oracle without it."""
    from workloads import make_radial_mlp
    prob = make_problem(*SHAPES[0], n_src=64, n_dst=64, E=2000, seed=79)
    pl = prob["plan"]
    w1, b1, w2, b2 = make_radial_mlp(79, 0, 16, pl.weight_numel)
    v32 = rounded(prob["vec"], torch.float32)
    prob["w"] = tp.radial_mlp(v32, w1, b1, w2, b2)
    prob["sh"] = so3.sh_concat([t.l for t in pl.irr_sh], v32)
    desc = tpc.tp_desc_create(*SHAPES[0])
    g = gpu_sorted_inputs(tpc, prob)
    vec = dev_tensor(prob["vec"])[g["perm"].long()].contiguous()
    bad = g["src"].clone()
    bad[17] = 64
    bad[1001] = -5
    out = tpc.tp_conv_forward_mlp(desc, g["x"], vec, dev_tensor(w1), dev_tensor(b1), dev_tensor(w2), dev_tensor(b2),
                                  bad, g["row_ptr"], 64)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    keep = np.ones(2000, bool)
    keep[g["perm"].cpu().numpy()[[17, 1001]]] = False
    ref = tp.conv_forward(pl, rounded(prob["x"], torch.float32), prob["sh"][keep], prob["w"][keep],
                          prob["src"][keep], prob["dst"][keep], 64)
    assert err(out, ref) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


def test_radial_network_alignment(tpc):
    """The radial network's w2 and b2 are read in 16-byte pieces: a w2 or b2
    that is 4- but not 16-byte aligned is refused with TP_ERR_ALIGN before
    anything is launched, and the aligned call succeeds."""
    from workloads import make_radial_mlp
    prob = make_problem(*SHAPES[1], n_src=64, n_dst=64, E=500, seed=80)
    pl = prob["plan"]
    desc = tpc.tp_desc_create(*SHAPES[1])
    g = gpu_sorted_inputs(tpc, prob)
    vec = dev_tensor(prob["vec"])[g["perm"].long()].contiguous()
    w1, b1, w2, b2 = (dev_tensor(a) for a in make_radial_mlp(80, 0, 16, pl.weight_numel))
    w2_off = torch.empty(w2.numel() + 1, device="cuda")[1:].view_as(w2).copy_(w2)
    b2_off = torch.empty(b2.numel() + 1, device="cuda")[1:].copy_(b2)
    for a, b in ((w2_off, b2), (w2, b2_off)):
        with pytest.raises(tpc.TPError) as ei:
            tpc.tp_conv_forward_mlp(desc, g["x"], vec, w1, b1, a, b, g["src"], g["row_ptr"], 64)
        assert tpc.STATUS_NAMES[ei.value.status] == "TP_ERR_ALIGN"
    tpc.tp_conv_forward_mlp(desc, g["x"], vec, w1, b1, w2, b2, g["src"], g["row_ptr"], 64)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
