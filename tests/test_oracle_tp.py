"""Oracle pins for the tensor-product convolution itself: path enumeration
against the page's worked example, brute force vs the vectorised and C
versions, scatter semantics, rotation and inversion equivariance, layout
invariance, exact adjoint identities and finite differences, and the stable
counting sort."""
import json
import math
import os

import numpy as np
import pytest

from oracle import cref
from oracle import irreps as I
from oracle import so3, tp
from workloads import WORKLOADS, make_features, make_graph, subgraph_uniform

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))
RNG = np.random.default_rng(77)


def test_paths_page_example():
    g = GOLD["channelwise_32x0e32x1o_sh_0e1o"]
    plan = tp.Plan(g["irreps_in"], g["irreps_sh"], g["irreps_out"])
    assert plan.n_paths == g["num_paths"]
    assert f"{plan.weight_numel}x0e" == g["weight_irreps"]
    # the descriptor prints one output block per path, grouped by output type
    per_path = sorted((P.lc, -plan.irr_out[P.c].p) for P in plan.paths)
    unsimplified = "+".join(str(I.MulIrrep(plan.mul, l, -q)) for l, q in per_path)
    assert unsimplified == g["path_outputs_unsimplified"]
    instr = tp.enumerate_instructions_lmax(I.parse(g["irreps_in"]), I.parse(g["irreps_sh"]), 1)
    assert len(instr) == len(g["e3nn_lmax1_instructions"])
    for got, want in zip(instr, g["e3nn_lmax1_instructions"]):
        assert (got[0], got[1], got[2]) == (want["in1"], want["in2"], want["out"])
        assert [got[3][0], 1] == want["path_shape"]
    # the e3nn loop keeps a 1e block that the explicit output list drops
    extra = [t for t in instr if (t[3][1], t[3][2]) not in {(0, 1), (1, -1)}]
    assert [(t[3][1], {1: "e", -1: "o"}[t[3][2]]) for t in extra] == [(1, g["dropped_type"][1])]


@pytest.mark.parametrize("name,P,paths", [
    ("tiny", 7, [(0, 0, 0), (0, 1, 1), (0, 2, 2), (1, 0, 1), (1, 1, 0), (1, 1, 2), (1, 2, 1)]),
    ("medium", 13, [(0, 0, 0), (0, 1, 1), (0, 2, 2), (1, 0, 1), (1, 1, 0), (1, 1, 2), (1, 2, 1), (1, 3, 2),
                    (2, 0, 2), (2, 1, 1), (2, 2, 0), (2, 2, 2), (2, 3, 1)]),
    ("large", 23, None),
    ("xlarge", 7, None),
])
def test_paths_per_workload(name, P, paths):
    w = WORKLOADS[name]
    plan = tp.Plan(w.irreps_in, w.irreps_sh, w.irreps_out)
    assert plan.n_paths == P
    if paths is not None:
        assert [(p.la, p.lb, p.lc) for p in plan.paths] == paths
    for p in plan.paths:       # triangle and parity
        assert abs(p.la - p.lb) <= p.lc <= p.la + p.lb
        assert plan.irr_in[p.a].p * plan.irr_sh[p.b].p == plan.irr_out[p.c].p


def test_path_rejections():
    with pytest.raises(ValueError):
        tp.Plan("32x0e", "0e", "16x0e")                     # uvu needs equal multiplicity
    with pytest.raises(ValueError):
        tp.Plan("32x0e", "2x0e", "32x0e")                    # harmonics have multiplicity 1
    with pytest.raises(ValueError):
        tp.Plan("32x0e", "0e", "32x0e+32x0e")                # duplicate output type
    plan = tp.Plan("8x0e+8x1o", "0e+1o", "8x0e+8x1o+8x1e+8x3o")
    # 1e comes from 1o x 1o; 3o is unreachable and stays zero
    assert {(p.la, p.lb, p.lc) for p in plan.paths} == {(0, 0, 0), (0, 1, 1), (1, 0, 1), (1, 1, 0), (1, 1, 1)}


def random_problem(irr_in, irr_sh, irr_out, n_src, n_dst, E, seed=0, unit_sh=True):
    rng = np.random.default_rng(seed)
    plan = tp.Plan(irr_in, irr_sh, irr_out)
    x = rng.standard_normal((n_src, plan.dim_in))
    v = rng.standard_normal((E, 3))
    ls = [t.l for t in plan.irr_sh]
    sh = so3.sh_concat(ls, v, normalize=unit_sh)
    w = rng.standard_normal((E, plan.weight_numel))
    src = rng.integers(0, n_src, E)
    dst = rng.integers(0, n_dst, E)
    return plan, x, v, sh, w, src, dst


def test_brute_force_matches_vectorised():
    plan, x, v, sh, w, src, dst = random_problem("4x0e+4x1o+4x2e", "0e+1o+2e+3o", "4x0e+4x1o+4x2e+4x3o", 6, 5, 30)
    a = tp.conv_forward_brute(plan, x, sh, w, src, dst, 5)
    b = tp.conv_forward(plan, x, sh, w, src, dst, 5)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


def test_c_oracle_matches_numpy():
    plan, x, v, sh, w, src, dst = random_problem("8x0e+8x1o+8x2e", "0e+1o+2e+3o", "8x0e+8x1o+8x2e", 20, 17, 300, seed=3)
    perm, row_ptr, dsts = tp.csr_build(dst, 17)
    ref = tp.conv_forward(plan, x, sh, w, src, dst, 17)
    got = cref.conv_forward(plan, x, sh[perm], w[perm], src[perm], row_ptr, 17)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    rows = np.array([16, 3, 3, 0], dtype=np.int32)
    np.testing.assert_allclose(cref.conv_forward(plan, x, sh[perm], w[perm], src[perm], row_ptr, 17, rows=rows),
                               ref[rows], rtol=1e-12, atol=1e-12)
    g = np.random.default_rng(1).standard_normal((17, plan.dim_out))
    dx, dw, dsh = tp.conv_backward(plan, x, sh, w, src, dst, g)
    dw_c, dsh_c = cref.conv_backward_edges(plan, x, sh, w, g, src, dst)
    np.testing.assert_allclose(dw_c, dw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dsh_c, dsh, rtol=1e-12, atol=1e-12)
    sp, srp, _ = tp.csr_build(src, 20)
    dx_c = cref.conv_backward_dx(plan, sh, w, g, dst, sp, srp, 20)
    np.testing.assert_allclose(dx_c, dx, rtol=1e-12, atol=1e-12)


def test_scatter_semantics_page_example():
    """The gather/scatter example: scalars only, so each path reduces to
    x[src]*w and the op must equal index_add of the gathered rows."""
    g = GOLD["gather_scatter"]
    plan = tp.Plan("3x0e", "0e", "3x0e")
    rng = np.random.default_rng(5)
    x = rng.standard_normal((g["n_nodes"], 3))
    src, dst = np.array(g["senders"]), np.array(g["receivers"])
    sh = np.ones((4, 1))
    w = rng.standard_normal((4, 3))
    out = tp.conv_forward(plan, x, sh, w, src, dst, g["n_dst"])
    ref = np.zeros((g["n_dst"], 3))
    for e in range(4):
        ref[dst[e]] += x[src[e]] * w[e]
    np.testing.assert_array_equal(out, ref)
    assert not out[g["isolated_destination"]].any()
    # bipartite: 5 sources, 4 destinations
    assert out.shape == (4, 3)


def _block_rotate(plan_irreps, D_by_l, vec):
    out = vec.copy()
    for t, o in zip(plan_irreps, I.offsets(plan_irreps)):
        blk = vec[..., o:o + t.dim].reshape(vec.shape[:-1] + (t.ir_dim, t.mul))
        out[..., o:o + t.dim] = np.einsum("ij,...ju->...iu", D_by_l[t.l], blk).reshape(vec.shape[:-1] + (t.dim,))
    return out


@pytest.mark.parametrize("irr", [("4x0e+4x1o", "0e+1o+2e", "4x0e+4x1o+4x2e"),
                                 ("3x0e+3x1o+3x2e+3x3o", "0e+1o+2e+3o", "3x0e+3x1o+3x2e+3x3o"),
                                 ("2x0+2x1+2x2", "0+1+2", "2x0+2x1+2x2")])
def test_rotation_equivariance(irr):
    plan, x, v, sh, w, src, dst = random_problem(*irr, 7, 6, 40, seed=11)
    R = so3.random_rotation(RNG)
    D = {l: so3.wigner_D(l, R) for l in range(4)}
    out = tp.conv_forward(plan, x, sh, w, src, dst, 6)
    sh_rot = so3.sh_concat([t.l for t in plan.irr_sh], v @ R.T)
    np.testing.assert_allclose(sh_rot, _block_rotate(plan.irr_sh, D, sh), atol=1e-12)
    out_rot = tp.conv_forward(plan, _block_rotate(plan.irr_in, D, x), sh_rot, w, src, dst, 6)
    np.testing.assert_allclose(out_rot, _block_rotate(plan.irr_out, D, out), atol=1e-11)


def test_inversion_parity():
    plan, x, v, sh, w, src, dst = random_problem("3x0e+3x1o+3x2e", "0e+1o+2e+3o", "3x0e+3x1o+3x2e", 5, 5, 30, seed=4)
    sign = lambda irr: np.concatenate([np.full(t.dim, float(t.p)) for t in irr])
    out = tp.conv_forward(plan, x, sh, w, src, dst, 5)
    sh_inv = so3.sh_concat([t.l for t in plan.irr_sh], -v)
    np.testing.assert_allclose(sh_inv, sh * sign(plan.irr_sh), atol=1e-13)
    out_inv = tp.conv_forward(plan, x * sign(plan.irr_in), sh_inv, w, src, dst, 5)
    np.testing.assert_allclose(out_inv, out * sign(plan.irr_out), atol=1e-12)


def test_layout_invariance():
    """Computing in mul_ir (convert in, compute, convert out) is the same map."""
    plan, x, v, sh, w, src, dst = random_problem("3x0e+3x1o+3x2e", "0e+1o+2e", "3x0e+3x1o+3x2e", 5, 5, 20, seed=8)
    out = tp.conv_forward(plan, x, sh, w, src, dst, 5)
    x_mi = I.convert_layout(x, plan.irr_in, "ir_mul", "mul_ir")
    # an independent mul_ir evaluation, brute force
    out_mi = np.zeros((5, plan.dim_out))
    mul = plan.mul
    for e in range(len(src)):
        for p, P in enumerate(plan.paths):
            C = plan.cg[p]
            oa, ob, oc = plan.off_in[P.a], plan.off_sh[P.b], plan.off_out[P.c]
            na, nb, nc = 2 * P.la + 1, 2 * P.lb + 1, 2 * P.lc + 1
            xa = x_mi[src[e], oa:oa + na * mul].reshape(mul, na)
            t = np.einsum("ijk,ui,j->uk", C, xa, sh[e, ob:ob + nb]) * w[e, p * mul:(p + 1) * mul, None]
            out_mi[dst[e], oc:oc + nc * mul] += t.ravel()
    np.testing.assert_allclose(I.convert_layout(out_mi, plan.irr_out, "mul_ir", "ir_mul"), out, atol=1e-12)


def test_unreached_output_and_empty_graph():
    plan = tp.Plan("4x0e+4x1o", "0e+1o", "4x0e+4x1o+4x3o")
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, plan.dim_in))
    sh = so3.sh_concat([0, 1], rng.standard_normal((5, 3)))
    w = rng.standard_normal((5, plan.weight_numel))
    out = tp.conv_forward(plan, x, sh, w, rng.integers(0, 3, 5), rng.integers(0, 3, 5), 3)
    assert not out[:, plan.oblock_slice(2)].any()
    empty = tp.conv_forward(plan, x, sh[:0], w[:0], np.zeros(0, int), np.zeros(0, int), 3)
    assert empty.shape == (3, plan.dim_out) and not empty.any()


def test_backward_adjoint_identities():
    """<g, f(dx, sh, w)> = <dx_grad, dx> etc., exact since f is linear in each input."""
    plan, x, v, sh, w, src, dst = random_problem("3x0e+3x1o+3x2e", "0e+1o+2e+3o", "3x0e+3x1o+3x2e", 6, 6, 40, seed=9)
    g = np.random.default_rng(2).standard_normal((6, plan.dim_out))
    dx, dw, dsh = tp.conv_backward(plan, x, sh, w, src, dst, g)
    f = lambda X, S, W: float(np.sum(g * tp.conv_forward(plan, X, S, W, src, dst, 6)))
    rng = np.random.default_rng(3)
    d = rng.standard_normal(x.shape)
    assert abs(f(d, sh, w) - np.sum(dx * d)) < 1e-10 * (1 + abs(np.sum(dx * d)))
    d = rng.standard_normal(w.shape)
    assert abs(f(x, sh, d) - np.sum(dw * d)) < 1e-10 * (1 + abs(np.sum(dw * d)))
    d = rng.standard_normal(sh.shape)
    assert abs(f(x, d, w) - np.sum(dsh * d)) < 1e-10 * (1 + abs(np.sum(dsh * d)))


def test_backward_finite_differences_fd_graph():
    """Central differences on the 16-node, 64-edge graph with the medium irreps."""
    wl = WORKLOADS["fd"]
    rng, src, dst, vec, n = make_graph(wl)
    plan = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    sh = so3.sh_concat([t.l for t in plan.irr_sh], vec)
    x, w, g = make_features(rng, wl, n, len(src), plan.dim_in, plan.weight_numel, plan.n_paths, plan.dim_out)
    dx, dw, dsh = tp.conv_backward(plan, x, sh, w, src, dst, g)
    f = lambda X, S, W: float(np.sum(g * tp.conv_forward(plan, X, S, W, src, dst, n)))
    h = 1e-3
    pick = np.random.default_rng(4)
    for arr, grad, which in ((x, dx, 0), (w, dw, 2), (sh, dsh, 1)):
        for _ in range(6):
            idx = tuple(pick.integers(0, s) for s in arr.shape)
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = [x, sh, w]
            args_m = [x, sh, w]
            args_p[which], args_m[which] = ap, am
            fd = (f(*args_p) - f(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-8 * max(1.0, abs(grad[idx])), (which, idx, fd, grad[idx])


def test_csr_counting_sort():
    rng = np.random.default_rng(6)
    for n, E in ((1, 0), (1, 5), (7, 40), (50, 300)):
        keys = rng.integers(0, n, E)
        perm, rp, ks = tp.csr_build(keys, n)
        perm2, rp2, ks2 = tp.csr_build_loops(keys, n)
        assert np.array_equal(perm, perm2) and np.array_equal(rp, rp2) and np.array_equal(ks, ks2)
        assert rp[0] == 0 and rp[-1] == E and np.all(np.diff(rp) >= 0)
        assert np.all(np.diff(ks) >= 0)
        for d in range(n):   # stability: original order within each key
            assert np.all(np.diff(perm[rp[d]:rp[d + 1]]) > 0)
    with pytest.raises(ValueError):
        tp.csr_build(np.array([0, 3]), 3)


def test_workload_generator_shapes():
    wl = WORKLOADS["tiny"]
    rng, src, dst, vec, n = make_graph(wl)
    assert (n, len(src)) == (32, 512)
    np.testing.assert_allclose(np.linalg.norm(vec, axis=1), 1.0, rtol=1e-14)
    wl = WORKLOADS["medium"]
    rng, src, dst, vec, n = make_graph(wl)
    assert np.all(np.diff(dst) >= 0) and np.all(src != dst)
    assert 120_000 < len(src) < 142_000
    assert np.all(np.linalg.norm(vec, axis=1) < 5.0)


def test_rms_rel_err_hand_computed():
    """The error measure every GPU parity assertion divides by, pinned to
    values worked out by hand: max |got - ref| over the tensor, divided by the
    root mean square of the reference (not of `got`, not a mean error)."""
    # ref = [3, 4]: RMS = sqrt((9 + 16) / 2) = sqrt(12.5); largest difference 1
    assert tp.rms_rel_err(np.array([3.0, 5.0]), np.array([3.0, 4.0])) == pytest.approx(1.0 / math.sqrt(12.5),
                                                                                       rel=1e-15)
    # the maximum, not the mean, of the differences: |[0.5, -2, 0]| -> 2; RMS of ref = 2
    assert tp.rms_rel_err(np.array([2.5, 0.0, 2.0]), np.array([2.0, 2.0, 2.0])) == pytest.approx(1.0, rel=1e-15)
    # the reference's RMS, not got's: swapping the arguments changes the value
    assert tp.rms_rel_err(np.array([3.0, 4.0]), np.array([3.0, 5.0])) == pytest.approx(1.0 / math.sqrt(17.0),
                                                                                       rel=1e-15)
    # 2-D tensors use every element
    ref = np.array([[1.0, -1.0], [1.0, -1.0]])
    assert tp.rms_rel_err(ref + np.array([[0.0, 0.0], [0.0, 0.25]]), ref) == pytest.approx(0.25, rel=1e-15)
    # an all-zero reference: the plain max difference; an empty tensor: 0
    assert tp.rms_rel_err(np.array([0.0, -0.5]), np.zeros(2)) == 0.5
    assert tp.rms_rel_err(np.zeros((0, 4)), np.zeros((0, 4))) == 0.0


def test_silu_identities_and_library():
    """silu(0) = 0; silu(z) - silu(-z) = z (sigmoid(z) + sigmoid(-z) = 1);
    silu(z)/z -> 1 and silu(-z) -> 0 for large z; equal to torch's SiLU in fp64."""
    import torch
    z = np.linspace(-30.0, 30.0, 601)
    s = tp.silu(z)
    assert tp.silu(0.0) == 0.0
    np.testing.assert_allclose(s - tp.silu(-z), z, rtol=0, atol=1e-13)
    assert abs(tp.silu(40.0) / 40.0 - 1.0) < 1e-15 and abs(tp.silu(-40.0)) < 1e-15
    ref = torch.nn.functional.silu(torch.as_tensor(z, dtype=torch.float64)).numpy()
    np.testing.assert_allclose(s, ref, rtol=1e-14, atol=1e-300)


def test_radial_mlp_structure():
    """The network's pieces fixed independently of its formula: with w2 = 0 the
    weights are b2; with w2 the unit matrix e_i (x) e_j, weight j is the hidden
    unit i = silu(w1_i |v| + b1_i), which depends on the vector only through its
    length; and the output is affine in (w2, b2)."""
    rng = np.random.default_rng(5)
    H, numel, E = 16, 12, 9
    vec = rng.standard_normal((E, 3))
    w1, b1 = rng.standard_normal(H), rng.standard_normal(H)
    b2 = rng.standard_normal(numel)
    np.testing.assert_array_equal(tp.radial_mlp(vec, w1, b1, np.zeros((H, numel)), b2), np.broadcast_to(b2, (E, numel)))
    w2 = np.zeros((H, numel))
    w2[3, 7] = 1.0
    out = tp.radial_mlp(vec, w1, b1, w2, np.zeros(numel))
    r = np.linalg.norm(vec, axis=1)
    np.testing.assert_allclose(out[:, 7], tp.silu(w1[3] * r + b1[3]), rtol=1e-15)
    assert not np.any(np.delete(out, 7, axis=1))
    R = so3.random_rotation(rng)   # rotating (or flipping) the vectors changes nothing
    np.testing.assert_allclose(tp.radial_mlp(-vec @ R.T, w1, b1, w2, b2), tp.radial_mlp(vec, w1, b1, w2, b2), rtol=1e-13)
    wa, wb = rng.standard_normal((H, numel)), rng.standard_normal((H, numel))
    ba, bb = rng.standard_normal(numel), rng.standard_normal(numel)
    np.testing.assert_allclose(tp.radial_mlp(vec, w1, b1, wa + wb, ba + bb),
                               tp.radial_mlp(vec, w1, b1, wa, ba) + tp.radial_mlp(vec, w1, b1, wb, bb), rtol=1e-12)


def test_mean_reduction_special_cases():
    """reduce="mean": every edge of a destination carrying the same message
    gives that message; one edge gives the sum; destinations without edges stay
    zero; sum = mean x (number of edges)."""
    plan = tp.Plan("4x0e+4x1o", "0e+1o+2e", "4x0e+4x1o+4x2e")
    rng = np.random.default_rng(9)
    x = rng.standard_normal((3, plan.dim_in))
    vec = rng.standard_normal((1, 3))
    sh1 = so3.sh_concat([0, 1, 2], vec)
    w1 = rng.standard_normal((1, plan.weight_numel))
    # destination 0: five copies of one edge; destination 1: one other edge; 2: none
    src = np.array([2, 2, 2, 2, 2, 0])
    dst = np.array([0, 0, 0, 0, 0, 1])
    sh = np.repeat(sh1, 6, axis=0)
    w = np.repeat(w1, 6, axis=0)
    mean = tp.conv_forward_mean(plan, x, sh, w, src, dst, 3)
    single = tp.conv_forward(plan, x, sh[:1], w[:1], src[:1], np.array([0]), 1)[0]
    np.testing.assert_allclose(mean[0], single, rtol=1e-13)
    np.testing.assert_allclose(mean[1], tp.conv_forward(plan, x, sh, w, src, dst, 3)[1], rtol=0, atol=0)
    assert not np.any(mean[2])
    np.testing.assert_allclose(5 * mean[0], tp.conv_forward(plan, x, sh, w, src, dst, 3)[0], rtol=1e-13)


def test_unsimplified_outputs():
    """Per-path output blocks: their listing for the lesson's example is the
    printed D=32x0e+32x0e+32x1o+32x1o, and adding the blocks of one output type
    gives the simplified output."""
    g = GOLD["channelwise_32x0e32x1o_sh_0e1o"]
    plan = tp.Plan(g["irreps_in"], g["irreps_sh"], g["irreps_out"])
    order = tp.unsimplified_order(plan)
    listing = "+".join(str(I.MulIrrep(plan.mul, plan.paths[p].lc, plan.irr_out[plan.paths[p].c].p)) for p in order)
    assert listing == g["path_outputs_unsimplified"]
    for irr in [("4x0e+4x1o", "0e+1o+2e", "4x0e+4x1o+4x2e"), ("8x0e+8x1o+8x2e", "0e+1o+2e+3o", "8x0e+8x1o+8x2e")]:
        plan = tp.Plan(*irr)
        _, x, _, sh, w, src, dst = random_problem(*irr, n_src=9, n_dst=7, E=40, seed=3)
        un = tp.conv_forward_unsimplified(plan, x, sh, w, src, dst, 7)
        simp = np.zeros((7, plan.dim_out))
        col = 0
        for p in tp.unsimplified_order(plan):
            P = plan.paths[p]
            width = (2 * P.lc + 1) * plan.mul
            simp[:, plan.oblock_slice(P.c)] += un[:, col:col + width]
            col += width
        assert col == un.shape[1]
        np.testing.assert_allclose(simp, tp.conv_forward(plan, x, sh, w, src, dst, 7), atol=1e-12)
