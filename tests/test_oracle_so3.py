"""Oracle pins for spherical harmonics, Wigner-D and Clebsch-Gordan tensors.

Each check is tied to something other than the oracle itself: the addition
theorem, closed forms, orthogonality by exact quadrature, scipy's complex
harmonics (a library routine) and sympy's exact Clebsch-Gordan values.
"""
import math

import numpy as np
import pytest
from scipy.special import roots_legendre, sph_harm_y

from oracle import so3

RNG = np.random.default_rng(2024)


def unit(n):
    v = RNG.standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


@pytest.mark.parametrize("l", [0, 1, 2, 3, 4])
def test_sh_addition_theorem(l):
    Y = so3.real_sh(l, unit(200))
    np.testing.assert_allclose((Y ** 2).sum(1), 2 * l + 1, rtol=1e-13)


def test_sh_low_degrees_closed_form():
    v = unit(50)
    x, y, z = v.T
    np.testing.assert_allclose(so3.real_sh(0, v)[:, 0], 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(so3.real_sh(1, v), math.sqrt(3) * np.stack([y, z, x], 1), atol=1e-14)
    Y2 = so3.real_sh(2, v)
    s15 = math.sqrt(15)
    ref2 = np.stack([s15 * x * y, s15 * y * z, math.sqrt(5) / 2 * (3 * z * z - 1), s15 * x * z,
                     s15 / 2 * (x * x - y * y)], 1)
    np.testing.assert_allclose(Y2, ref2, atol=1e-13)


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_sh_against_scipy_complex(l):
    """Real harmonics as the standard combinations of scipy's complex ones
    (which carry the Condon-Shortley sign), times sqrt(4 pi)."""
    v = unit(40)
    theta = np.arccos(np.clip(v[:, 2], -1, 1))
    phi = np.arctan2(v[:, 1], v[:, 0])
    ref = np.zeros((40, 2 * l + 1))
    for m in range(-l, l + 1):
        Yc = sph_harm_y(l, abs(m), theta, phi)
        if m > 0:
            ref[:, m + l] = math.sqrt(2) * (-1) ** m * Yc.real
        elif m < 0:
            ref[:, m + l] = math.sqrt(2) * (-1) ** m * Yc.imag
        else:
            ref[:, m + l] = Yc.real
    np.testing.assert_allclose(so3.real_sh(l, v), ref * math.sqrt(4 * math.pi), atol=1e-12)


def test_sh_orthonormal_by_quadrature():
    """Mean over the sphere of Y_lm Y_l'm' = delta (component normalisation);
    Gauss-Legendre in cos(theta) x uniform phi is exact for these degrees."""
    zs, wz = roots_legendre(12)
    phis = np.arange(24) * (2 * math.pi / 24)
    Z, PH = np.meshgrid(zs, phis, indexing="ij")
    W = np.repeat(wz[:, None], 24, 1) * (2 * math.pi / 24) / (4 * math.pi)
    s = np.sqrt(1 - Z ** 2)
    pts = np.stack([s * np.cos(PH), s * np.sin(PH), Z], -1).reshape(-1, 3)
    Y = so3.sh_concat([0, 1, 2, 3], pts)
    G = (Y * W.reshape(-1, 1)).T @ Y
    np.testing.assert_allclose(G, np.eye(16), atol=1e-13)


def test_sh_raw_polynomial_is_homogeneous():
    v = unit(10)
    for l in range(4):
        a = so3.real_sh(l, 2.5 * v, normalize=False)
        np.testing.assert_allclose(a, 2.5 ** l * so3.real_sh(l, v), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(so3.real_sh(l, 2.5 * v, normalize=True), so3.real_sh(l, v), atol=1e-13)


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_wigner_D_is_a_representation(l):
    R1, R2 = so3.random_rotation(RNG), so3.random_rotation(RNG)
    D1, D2 = so3.wigner_D(l, R1), so3.wigner_D(l, R2)
    np.testing.assert_allclose(D1 @ D1.T, np.eye(2 * l + 1), atol=1e-12)
    np.testing.assert_allclose(so3.wigner_D(l, R1 @ R2), D1 @ D2, atol=1e-12)
    v = unit(30)
    np.testing.assert_allclose(so3.real_sh(l, v @ R1.T), so3.real_sh(l, v) @ D1.T, atol=1e-12)


def test_wigner_D1_is_permuted_rotation():
    R = so3.random_rotation(RNG)
    P = np.array([[0, 1, 0], [0, 0, 1], [1, 0, 0]], dtype=float)   # (x,y,z) -> (y,z,x)
    np.testing.assert_allclose(so3.wigner_D(1, R), P @ R @ P.T, atol=1e-13)


def test_rotation_matrix():
    R = so3.rotation_matrix(np.array([0.2, -0.3, 0.1]))
    np.testing.assert_allclose(R @ R.T, np.eye(3), atol=1e-15)
    assert abs(np.linalg.det(R) - 1) < 1e-14
    np.testing.assert_allclose(so3.rotation_matrix(np.array([0, 0, math.pi / 2])) @ [1, 0, 0], [0, 1, 0], atol=1e-15)


TRIPLES = [(l1, l2, l3) for l1 in range(4) for l2 in range(4) for l3 in range(abs(l1 - l2), min(l1 + l2, 3) + 1)]


@pytest.mark.parametrize("l1,l2,l3", TRIPLES)
def test_cg_equivariant_and_orthonormal(l1, l2, l3):
    C = so3.real_cg(l1, l2, l3)
    n3 = 2 * l3 + 1
    G = np.einsum("ijk,ijq->kq", C, C)
    np.testing.assert_allclose(G, np.eye(n3), atol=1e-13)
    R = so3.random_rotation(RNG)
    D1, D2, D3 = (so3.wigner_D(l, R) for l in (l1, l2, l3))
    lhs = np.einsum("ijk,ia,jb->abk", C, D1, D2)
    rhs = np.einsum("kc,abc->abk", D3, C)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12)
    first = C.ravel()[np.flatnonzero(np.abs(C.ravel()) > 1e-9)[0]]
    assert first > 0


@pytest.mark.parametrize("l1,l2", [(1, 1), (1, 2), (2, 2), (2, 3), (3, 3), (0, 3), (1, 3)])
def test_cg_stacked_over_l3_is_orthogonal(l1, l2):
    """All l3 together form an orthogonal change of basis of l1 x l2."""
    M = np.concatenate([so3.real_cg(l1, l2, l3).reshape((2 * l1 + 1) * (2 * l2 + 1), -1)
                        for l3 in range(abs(l1 - l2), l1 + l2 + 1)], axis=1)
    assert M.shape[0] == M.shape[1]
    np.testing.assert_allclose(M.T @ M, np.eye(M.shape[0]), atol=1e-12)


def test_cg_closed_forms_and_selection():
    for l in range(4):
        np.testing.assert_allclose(so3.real_cg(0, l, l)[0], np.eye(2 * l + 1), atol=1e-14)
        np.testing.assert_allclose(so3.real_cg(l, 0, l)[:, 0, :], np.eye(2 * l + 1), atol=1e-14)
    np.testing.assert_allclose(so3.real_cg(1, 1, 0)[:, :, 0], np.eye(3) / math.sqrt(3), atol=1e-15)
    assert not so3.real_cg(1, 1, 3).any() and not so3.real_cg(0, 1, 2).any()
    # the antisymmetric 1x1->1 coupling is the cross product, (y,z,x) ordering
    C = so3.real_cg(1, 1, 1)
    a, b = RNG.standard_normal(3), RNG.standard_normal(3)
    P = np.array([[0, 1, 0], [0, 0, 1], [1, 0, 0]], dtype=float)
    got = np.einsum("ijk,i,j->k", C, P @ a, P @ b)
    np.testing.assert_allclose(np.abs(got), np.abs(P @ np.cross(a, b)) / math.sqrt(2), atol=1e-14)


def test_cg_nnz_counts():
    want = {(0, 0, 0): 1, (0, 1, 1): 3, (0, 2, 2): 5, (1, 0, 1): 3, (1, 1, 0): 3, (1, 1, 2): 11, (1, 2, 1): 11}
    for t, n in want.items():
        assert int((so3.real_cg(*t) != 0).sum()) == n


@pytest.mark.parametrize("l1,l2,l3", [t for t in TRIPLES if sum(t) % 2 == 0])
def test_cg_projects_product_of_harmonics(l1, l2, l3):
    """sum_ij C[i,j,k] Y1_i(r) Y2_j(r) = c Y3_k(r) with
    |c| = sqrt((2l1+1)(2l2+1)/(2l3+1)) |<l1 0 l2 0|l3 0>| (sympy, exact)."""
    from sympy.physics.wigner import clebsch_gordan
    v = unit(25)
    C = so3.real_cg(l1, l2, l3)
    lhs = np.einsum("ijk,ni,nj->nk", C, so3.real_sh(l1, v), so3.real_sh(l2, v))
    Y3 = so3.real_sh(l3, v)
    c = float(np.sum(lhs * Y3) / np.sum(Y3 * Y3))
    np.testing.assert_allclose(lhs, c * Y3, atol=1e-12)
    cg0 = float(clebsch_gordan(l1, l2, l3, 0, 0, 0))
    np.testing.assert_allclose(abs(c), math.sqrt((2 * l1 + 1) * (2 * l2 + 1) / (2 * l3 + 1)) * abs(cg0), rtol=1e-12)
