"""Pins of the symmetric-contraction oracle (oracle/symc.py) against what the
pages print and what the mathematics fixes: the lesson's weight irreps and
path counts, equivariance under rotations and inversion, symmetry of every
basis tensor, closed forms of the low degrees, and the vectorised sum against
explicit loops."""
import json
import math
import os

import numpy as np
import pytest

from oracle import irreps as I
from oracle import so3, symc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


def test_lesson_descriptor_counts():
    g = GOLD["symmetric_contraction_32x0e32x1o"]
    plan = symc.SymPlan(g["irreps_in"], g["irreps_out"], g["degrees"])
    assert [plan.num_paths(n) for n in g["degrees"]] == g["num_paths"]
    weights = "+".join(f"{plan.weights_per_degree(n) * plan.mul}x0e" for n in g["degrees"])
    assert weights == g["weight_irreps"]


@pytest.mark.parametrize("irr", [("4x0e+4x1o", "4x0e+4x1o"), ("4x0e+4x1o+4x2e", "4x0e+4x1o+4x2e"),
                                 ("4x0+4x1+4x2", "4x0+4x1")])
def test_basis_symmetric_and_independent(irr):
    plan = symc.SymPlan(*irr, [1, 2, 3])
    for nu, c, B in plan.terms:
        flat = B.reshape(B.shape[0], -1)
        assert np.linalg.matrix_rank(flat) == B.shape[0]
        np.testing.assert_allclose(np.linalg.norm(flat, axis=1), 1.0, rtol=1e-12)
        for t in range(nu - 1):   # symmetric in the nu slots
            np.testing.assert_allclose(np.swapaxes(B, 1 + t, 2 + t), B, atol=1e-12)


def _rotate(plan_irreps, x, R, inversion=False):
    out = np.empty_like(x)
    for t, o in zip(plan_irreps, I.offsets(plan_irreps)):
        D = so3.wigner_D(t.l, R) * (t.p if (inversion and t.p) else 1)
        blk = x[:, o:o + t.dim].reshape(len(x), t.ir_dim, t.mul)
        out[:, o:o + t.dim] = np.einsum("ij,nju->niu", D, blk).reshape(len(x), t.dim)
    return out


@pytest.mark.parametrize("irr", [("4x0e+4x1o", "4x0e+4x1o"), ("4x0e+4x1o+4x2e", "4x0e+4x1o+4x2e")])
def test_equivariance(irr):
    rng = np.random.default_rng(2)
    plan = symc.SymPlan(*irr, [1, 2, 3])
    x = rng.standard_normal((5, plan.dim_in))
    w = rng.standard_normal((3, plan.n_weights, plan.mul))
    el = np.array([0, 2, 1, 1, 0])
    f = symc.symmetric_contraction(plan, x, w, el)
    for _ in range(2):
        R = so3.random_rotation(rng)
        np.testing.assert_allclose(symc.symmetric_contraction(plan, _rotate(plan.irr_in, x, R), w, el),
                                   _rotate(plan.irr_out, f, R), atol=1e-10)
    np.testing.assert_allclose(symc.symmetric_contraction(plan, _rotate(plan.irr_in, x, np.eye(3), True), w, el),
                               _rotate(plan.irr_out, f, np.eye(3), True), atol=1e-10)


def test_closed_forms_scalar_vector():
    """0e+1o -> 0e: degree 1 is the scalar b0, degree 2 spans b0^2 and |v|^2/sqrt(3),
    degree 3 spans b0^3 and b0 |v|^2 (the symmetrised b0 v.v: nine entries of
    1/3, one per ordering of (0, m, m)), per channel."""
    plan = symc.SymPlan("2x0e+2x1o", "2x0e", [1, 2, 3])
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, plan.dim_in))
    b0 = x[:, 0:2]
    v = x[:, 2:8].reshape(4, 3, 2)
    vv = np.sum(v * v, axis=1)
    w = rng.standard_normal((1, plan.n_weights, 2))
    got = symc.symmetric_contraction(plan, x, w, np.zeros(4, int))
    want = (w[0, 0] * b0 + w[0, 1] * b0 ** 2 + w[0, 2] * vv / math.sqrt(3) + w[0, 3] * b0 ** 3
            + w[0, 4] * b0 * vv)
    np.testing.assert_allclose(got, want, rtol=1e-12)


def test_brute_force_matches_vectorised():
    rng = np.random.default_rng(4)
    plan = symc.SymPlan("2x0e+2x1o+2x2e", "2x0e+2x1o", [1, 2, 3])
    x = rng.standard_normal((3, plan.dim_in))
    w = rng.standard_normal((2, plan.n_weights, plan.mul))
    el = np.array([1, 0, 1])
    np.testing.assert_allclose(symc.symmetric_contraction_brute(plan, x, w, el),
                               symc.symmetric_contraction(plan, x, w, el), atol=1e-12)
