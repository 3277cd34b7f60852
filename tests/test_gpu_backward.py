"""GPU parity of tp_conv_backward (dx, dw, dsh) against the oracle's exact
gradients, including the 16-node / 64-edge finite-difference graph, and the
source-side CSR the input gradient uses: the one-pass ring kernel by source
(every program shape, one, two and four channels per lane, several ring and
piece geometries, bfloat16 inputs) and the generic two-kernel path."""
import numpy as np
import pytest
import torch

from helpers import deg_tol, FP32_TOL, dev_tensor, err, gpu_sorted_inputs, make_problem, rounded, tuning
from oracle import so3, tp
from workloads import WORKLOADS, make_features, make_graph

pytestmark = pytest.mark.gpu


def run_backward(tpc, prob, g_np, dtype=torch.float32):
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob, dtype)
    sp, srp, _ = tpc.tp_csr_build(g["src"], prob["n_src"])
    go = dev_tensor(g_np)
    dx, dw, dsh = tpc.tp_conv_backward(desc, go, g["x"], g["sh"], g["w"], g["src"], g["dst"], g["row_ptr"], sp, srp)
    torch.cuda.synchronize()
    perm = g["perm"].cpu().numpy()
    return dx, dw, dsh, perm


def oracle_backward(prob, g_np, dtype=torch.float32):
    f32 = torch.float32
    return tp.conv_backward(prob["plan"], rounded(prob["x"], dtype), rounded(prob["sh"], f32),
                            rounded(prob["w"], dtype), prob["src"], prob["dst"], rounded(g_np, f32))


# the ring kernel by source (default) and the generic two-kernel backward
PATHS = {"ring": {}, "generic": {"disable_ring_bwd": 1}}


SHAPES = [
    ("128x0e+128x1o+128x2e", "0e+1o+2e+3o", "128x0e+128x1o+128x2e"),
    ("32x0e+32x1o", "0e+1o+2e", "32x0e+32x1o+32x2e"),
    ("64x0e+64x1o+64x2e+64x3o", "0e+1o+2e+3o", "64x0e+64x1o+64x2e+64x3o"),
    ("40x2e+40x0e", "1o+0e+2e", "40x1o+40x2e+40x0e"),
    ("24x0e+24x2e", "0e+2e", "24x0e+24x2e+24x3o"),
]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("irr", SHAPES, ids=lambda c: "|".join(c))
def test_backward_matches_oracle(tpc, irr, path):
    prob = make_problem(*irr, n_src=211, n_dst=190, E=3000, seed=21)
    g_np = np.random.default_rng(22).standard_normal((190, prob["plan"].dim_out))
    with tuning(tpc, **PATHS[path]):
        dx, dw, dsh, perm = run_backward(tpc, prob, g_np)
    rdx, rdw, rdsh = oracle_backward(prob, g_np)
    assert err(dx, rdx) <= FP32_TOL
    assert err(dw, rdw[perm]) <= FP32_TOL
    assert err(dsh, rdsh[perm]) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


def test_backward_fd_graph(tpc):
    """The 16-node, 64-edge graph with the medium irreps (the oracle's own
    gradients are pinned against central differences on it)."""
    wl = WORKLOADS["fd"]
    rng, src, dst, vec, n = make_graph(wl)
    prob = make_problem(wl.irreps_in, wl.irreps_sh, wl.irreps_out, n, n, len(src), src=src, dst=dst)
    pl = prob["plan"]
    x, w, g = make_features(rng, wl, n, len(src), pl.dim_in, pl.weight_numel, pl.n_paths, pl.dim_out)
    prob.update(x=x, w=w, sh=so3.sh_concat([t.l for t in pl.irr_sh], vec))
    dx, dw, dsh, perm = run_backward(tpc, prob, g)
    rdx, rdw, rdsh = oracle_backward(prob, g)
    assert err(dx, rdx) <= FP32_TOL
    assert err(dw, rdw[perm]) <= FP32_TOL
    assert err(dsh, rdsh[perm]) <= FP32_TOL


@pytest.mark.parametrize("path", sorted(PATHS))
def test_backward_sources_without_edges_and_heavy_rows(tpc, path):
    """A source with 700 edges (cut into pieces of several warps, whose
    partial rows are merged), sources without edges and a heavy destination."""
    rng = np.random.default_rng(30)
    src = np.concatenate([np.full(700, 5), rng.integers(0, 100, 1500) * 3])
    dst = np.concatenate([rng.integers(0, 40, 700), np.full(1500, 2)])
    prob = make_problem(*SHAPES[0], n_src=400, n_dst=40, E=len(src), seed=31, src=src, dst=dst)
    g_np = np.random.default_rng(32).standard_normal((40, prob["plan"].dim_out))
    with tuning(tpc, **PATHS[path]):
        dx, dw, dsh, perm = run_backward(tpc, prob, g_np)
    rdx, rdw, rdsh = oracle_backward(prob, g_np)
    # source 5 sums 700 edges: its float32 rounding is relative to its own
    # magnitude, which the whole-tensor RMS (mostly empty rows) understates;
    # measure each used row against its own RMS instead
    dxn = dx.double().cpu().numpy()
    for s, c in zip(*np.unique(src, return_counts=True)):
        assert err(dxn[s], rdx[s]) <= deg_tol(c), s
    assert err(dw, rdw[perm]) <= FP32_TOL
    assert err(dsh, rdsh[perm]) <= FP32_TOL
    unused = np.setdiff1d(np.arange(400), src)
    assert not dx[torch.as_tensor(unused)].any()


@pytest.mark.parametrize("path", sorted(PATHS))
def test_backward_deterministic(tpc, path):
    prob = make_problem(*SHAPES[0], n_src=300, n_dst=300, E=6000, seed=40)
    g_np = np.random.default_rng(41).standard_normal((300, prob["plan"].dim_out))
    with tuning(tpc, **PATHS[path]):
        a = run_backward(tpc, prob, g_np)
        b = run_backward(tpc, prob, g_np)
    for u, v in zip(a[:3], b[:3]):
        assert torch.equal(u, v)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_backward_out_of_range_source_gives_zero_edge_rows(tpc, path):
    """An edge whose source is out of range (so the source CSR, built from the
    good sources, no longer matches src) is skipped and flagged; its dw and
    dsh rows are still written (as zeros), the other edges are unaffected."""
    prob = make_problem(*SHAPES[1], n_src=64, n_dst=64, E=1500, seed=44)
    g_np = np.random.default_rng(45).standard_normal((64, prob["plan"].dim_out))
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob)
    bad = g["src"].clone()
    bad[100] = 64
    sp, srp, _ = tpc.tp_csr_build(g["src"], prob["n_src"])
    dw = torch.full((1500, desc.weight_numel), 7.0, device="cuda")
    dsh = torch.full((1500, desc.dim_sh), 7.0, device="cuda")
    with tuning(tpc, **PATHS[path]):
        tpc.tp_conv_backward(desc, dev_tensor(g_np), g["x"], g["sh"], g["w"], bad, g["dst"], g["row_ptr"], sp, srp,
                             dw=dw, dsh=dsh)
        torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    assert not dw[100].any() and not dsh[100].any()
    perm = g["perm"].cpu().numpy()
    _, rdw, rdsh = oracle_backward(prob, g_np)
    keep = np.ones(1500, bool)
    keep[100] = False
    assert err(dw[torch.as_tensor(keep, device="cuda")], rdw[perm][keep]) <= FP32_TOL
    assert err(dsh[torch.as_tensor(keep, device="cuda")], rdsh[perm][keep]) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


# every compiled program shape, with one, two and four channels per lane
PROGRAM_SHAPES = [
    ("{m}x0e+{m}x1o", "0e+1o", "{m}x0e+{m}x1o"),
    ("{m}x0e+{m}x1o", "0e+1o+2e", "{m}x0e+{m}x1o+{m}x2e"),
    ("{m}x0e+{m}x1o+{m}x2e", "0e+1o+2e+3o", "{m}x0e+{m}x1o+{m}x2e"),
    ("{m}x0e+{m}x1o+{m}x2e+{m}x3o", "0e+1o+2e+3o", "{m}x0e+{m}x1o+{m}x2e+{m}x3o"),
]


@pytest.mark.parametrize("mul", [32, 64, 128])
@pytest.mark.parametrize("shape", range(4))
def test_ring_backward_program_shapes(tpc, shape, mul):
    irr = tuple(t.format(m=mul) for t in PROGRAM_SHAPES[shape])
    prob = make_problem(*irr, n_src=97, n_dst=83, E=1201, seed=50 + shape)
    g_np = np.random.default_rng(51).standard_normal((83, prob["plan"].dim_out))
    dx, dw, dsh, perm = run_backward(tpc, prob, g_np)
    rdx, rdw, rdsh = oracle_backward(prob, g_np)
    assert err(dx, rdx) <= FP32_TOL
    assert err(dw, rdw[perm]) <= FP32_TOL
    assert err(dsh, rdsh[perm]) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


@pytest.mark.parametrize("geo", [dict(bwd_stages=2), dict(bwd_stages=5, bwd_warps=1), dict(bwd_stage_bytes=1),
                                 dict(bwd_stage_bytes=100000, bwd_warps=3), dict(bwd_warps=2, bwd_stages=8)],
                         ids=lambda g: ",".join(f"{k}={v}" for k, v in g.items()))
def test_ring_backward_geometries(tpc, geo):
    """Ring depth, chunk size (1..10 edges) and warps per block do not change
    the sums (each edge's gradients and each source's row are summed in a
    fixed order), so the results are bitwise equal to the default geometry's;
    the mid-size shape has 10-edge chunks at the largest stage target."""
    for irr in (SHAPES[1], SHAPES[0]):
        prob = make_problem(*irr, n_src=150, n_dst=120, E=2500, seed=60)
        g_np = np.random.default_rng(61).standard_normal((120, prob["plan"].dim_out))
        ref = run_backward(tpc, prob, g_np)
        with tuning(tpc, **geo):
            got = run_backward(tpc, prob, g_np)
        rdx, rdw, rdsh = oracle_backward(prob, g_np)
        assert err(got[0], rdx) <= FP32_TOL
        assert err(got[1], rdw[got[3]]) <= FP32_TOL
        assert err(got[2], rdsh[got[3]]) <= FP32_TOL
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        assert tpc.tp_device_status(reset=True) == 0


@pytest.mark.parametrize("irr", [SHAPES[0], SHAPES[1], SHAPES[2]], ids=lambda c: "|".join(c))
def test_backward_bf16_inputs(tpc, irr):
    """bfloat16 x and w (the forward's bfloat16 inputs), float32 math: the
    oracle takes the same rounded values in float64, so the float32 bound holds."""
    prob = make_problem(*irr, n_src=180, n_dst=170, E=2600, seed=70)
    g_np = np.random.default_rng(71).standard_normal((170, prob["plan"].dim_out))
    dx, dw, dsh, perm = run_backward(tpc, prob, g_np, torch.bfloat16)
    rdx, rdw, rdsh = oracle_backward(prob, g_np, torch.bfloat16)
    assert err(dx, rdx) <= FP32_TOL
    assert err(dw, rdw[perm]) <= FP32_TOL
    assert err(dsh, rdsh[perm]) <= FP32_TOL
    assert tpc.tp_device_status(reset=True) == 0


def test_backward_bf16_needs_a_program(tpc):
    """The generic backward is float32 only: bfloat16 inputs of a descriptor
    without a compiled program are rejected, not converted."""
    prob = make_problem(*SHAPES[3], n_src=20, n_dst=20, E=100, seed=72)
    g_np = np.zeros((20, prob["plan"].dim_out))
    with pytest.raises(tpc.TPError) as ei:
        run_backward(tpc, prob, g_np, torch.bfloat16)
    assert tpc.STATUS_NAMES[ei.value.status] == "TP_ERR_UNSUPPORTED"


def test_ring_backward_out_of_range_destination(tpc):
    """An edge whose destination is out of range is flagged and gets zero dw
    and dsh rows and no dx term; every other result is unaffected."""
    prob = make_problem(*SHAPES[1], n_src=64, n_dst=64, E=1500, seed=74)
    g_np = np.random.default_rng(75).standard_normal((64, prob["plan"].dim_out))
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob)
    bad = g["dst"].clone()
    bad[200] = 64
    sp, srp, _ = tpc.tp_csr_build(g["src"], prob["n_src"])
    dx, dw, dsh = tpc.tp_conv_backward(desc, dev_tensor(g_np), g["x"], g["sh"], g["w"], g["src"], bad,
                                       g["row_ptr"], sp, srp)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    assert not dw[200].any() and not dsh[200].any()
    perm = g["perm"].cpu().numpy()
    keep = np.ones(1500, bool)
    keep[200] = False
    e_orig = perm[200]
    kp = np.setdiff1d(np.arange(1500), [e_orig])
    sub = dict(prob, src=prob["src"][kp], dst=prob["dst"][kp], sh=prob["sh"][kp], w=prob["w"][kp])
    rdx, rdw, rdsh = oracle_backward(sub, g_np)
    assert err(dx, rdx) <= FP32_TOL
    inv = np.empty(1500, np.int64)
    inv[kp] = np.arange(1499)
    assert err(dw[torch.as_tensor(keep, device="cuda")], rdw[inv[perm[keep]]]) <= FP32_TOL
    assert err(dsh[torch.as_tensor(keep, device="cuda")], rdsh[inv[perm[keep]]]) <= FP32_TOL


def test_ring_backward_wait_timeout_is_reported_and_writes_stay_in_bounds(tpc):
    """A main-loop wait limit of 1 ns makes the backward's pipeline waits give
    up on chunks whose copies are still in flight; every copy still lands (the
    waits after a failure keep the full limit), the call returns,
    TP_DEV_ERR_TIMEOUT is reported, nothing outside dx, dw and dsh changes
    (guard rows around each keep their sentinel), and the next call with the
    default settings is correct again. One-edge chunks of the smallest
    program shape (little arithmetic per chunk) let a warp reach chunks still
    in flight."""
    n, E = 4000, 400000
    prob = make_problem(*(t.format(m=32) for t in PROGRAM_SHAPES[0]), n_src=n, n_dst=n, E=E, seed=80)
    g_np = np.random.default_rng(81).standard_normal((n, prob["plan"].dim_out))
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob)
    sp, srp, _ = tpc.tp_csr_build(g["src"], prob["n_src"])
    go = dev_tensor(g_np)
    guard = 53

    def banded(rows, cols):
        big = torch.full((rows + 2 * guard, cols), 12345.0, device="cuda")
        return big, big[guard:guard + rows]

    bx, dx = banded(n, desc.dim_x)
    bw, dw = banded(E, desc.weight_numel)
    bs, dsh = banded(E, desc.dim_sh)
    hit = False
    for _ in range(10):
        with tuning(tpc, wait_limit_ns=1, bwd_stage_bytes=1):
            tpc.tp_conv_backward(desc, go, g["x"], g["sh"], g["w"], g["src"], g["dst"], g["row_ptr"], sp, srp,
                                 dx=dx, dw=dw, dsh=dsh)
            torch.cuda.synchronize()
        st = tpc.tp_device_status(reset=True)
        assert st & ~tpc.TP_DEV_ERR_TIMEOUT == 0
        for big, rows in ((bx, n), (bw, E), (bs, E)):
            assert torch.all(big[:guard] == 12345.0) and torch.all(big[guard + rows:] == 12345.0)
        hit = hit or bool(st & tpc.TP_DEV_ERR_TIMEOUT)
        if hit:
            break
    assert hit, "no pipeline wait ran out under a 1 ns limit"
    dx, dw, dsh, perm = run_backward(tpc, prob, g_np)
    assert tpc.tp_device_status(reset=True) == 0
    rdx, rdw, rdsh = oracle_backward(prob, g_np)
    assert err(dx, rdx) <= FP32_TOL
    assert err(dw, rdw[perm]) <= FP32_TOL
    assert err(dsh, rdsh[perm]) <= FP32_TOL


@pytest.mark.parametrize("path", sorted(PATHS))
def test_backward_empty_graph_zeroes_dx(tpc, path):
    """No edges: dx is all zeros (every source row written), dw and dsh are empty."""
    prob = make_problem(*SHAPES[0], n_src=10, n_dst=7, E=0, seed=1)
    g_np = np.random.default_rng(2).standard_normal((7, prob["plan"].dim_out))
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob)
    sp, srp, _ = tpc.tp_csr_build(g["src"], prob["n_src"])
    dx = torch.full((10, desc.dim_x), 5.0, device="cuda")
    with tuning(tpc, **PATHS[path]):
        _, dw, dsh = tpc.tp_conv_backward(desc, dev_tensor(g_np), g["x"], g["sh"], g["w"], g["src"], g["dst"],
                                          g["row_ptr"], sp, srp, dx=dx)
        torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    assert not dx.any() and dw.numel() == 0 and dsh.numel() == 0
