"""Rotation-group machinery of the oracle (test infrastructure), all float64.

* Real spherical harmonics from associated Legendre functions ("cuEquivariance
  in PyTorch", Spherical harmonics and a NumPy reference; Lesson 12a,
  section 21.5, which evaluates them with ``normalize=False`` and "component"
  normalisation). Reading taken where the pages are silent: real basis ordered
  m = -l..l, z is the pole, m<0 ~ sin(|m| phi), m>0 ~ cos(m phi), no
  Condon-Shortley sign (so l=1 is sqrt(3)(y, z, x)); component normalisation
  sum_m Y_lm(r)^2 = 2l+1 on the unit sphere. With ``normalize=False`` the raw
  homogeneous polynomial |r|^l Y_lm(r/|r|) is returned.
* Rotation matrices from axis-angle vectors (Rodrigues' formula), as the
  ``exp_map(rotation)`` of the Linear example on the same page.
* Wigner-D matrices of the real basis, obtained from the harmonics themselves:
  D^l(R) is the matrix with Y_l(R r) = D^l(R) Y_l(r), solved by least squares
  over sample directions.
* Real Clebsch-Gordan tensors C^{l1 l2 l3}[i,j,k] (Lesson 12a, section 21.4:
  the ``[ijk]`` factor of the descriptor; section 21.1: known ahead of time and
  mostly zero) as the one-dimensional null space of the equivariance constraint
  sum_ij C[i,j,k] D1[i,a] D2[j,b] = sum_c D3[k,c] C[a,b,c]. Reading taken:
  orthonormal over (i,j) for every k, sign such that the first entry above
  1e-9 in magnitude, in (i,j,k) row-major order, is positive.
"""
from __future__ import annotations

import math
from functools import lru_cache

import numpy as np


def _assoc_legendre(lmax: int, z: np.ndarray) -> dict:
    """P_l^m(z) for 0<=m<=l<=lmax, without the Condon-Shortley sign, by the
    standard three-term recurrences in l."""
    P = {}
    s = np.sqrt(np.clip(1.0 - z * z, 0.0, None))
    for m in range(lmax + 1):
        # P_m^m = (2m-1)!! s^m
        dfact = 1.0
        for k in range(1, 2 * m, 2):
            dfact *= k
        P[(m, m)] = dfact * s ** m
        if m + 1 <= lmax:
            P[(m + 1, m)] = (2 * m + 1) * z * P[(m, m)]
        for l in range(m + 2, lmax + 1):
            P[(l, m)] = ((2 * l - 1) * z * P[(l - 1, m)] - (l + m - 1) * P[(l - 2, m)]) / (l - m)
    return P


def real_sh(l: int, vec: np.ndarray, normalize: bool = True) -> np.ndarray:
    """Component-normalised real spherical harmonics of degree ``l`` for the rows
    of ``vec`` [n, 3]; returns [n, 2l+1] ordered m = -l..l."""
    vec = np.asarray(vec, dtype=np.float64)
    r = np.linalg.norm(vec, axis=1)
    safe = np.where(r > 0, r, 1.0)
    u = vec / safe[:, None]
    x, y, z = u[:, 0], u[:, 1], u[:, 2]
    phi = np.arctan2(y, x)
    P = _assoc_legendre(l, z)
    out = np.empty((vec.shape[0], 2 * l + 1))
    for m in range(-l, l + 1):
        am = abs(m)
        # orthonormal factor times sqrt(4 pi) -> component normalisation
        norm = math.sqrt((2 * l + 1) * math.factorial(l - am) / math.factorial(l + am))
        if m > 0:
            ang = math.sqrt(2.0) * np.cos(am * phi)
        elif m < 0:
            ang = math.sqrt(2.0) * np.sin(am * phi)
        else:
            ang = 1.0
        out[:, m + l] = norm * P[(l, am)] * ang
    if not normalize:
        out = out * (r ** l)[:, None]
    return out


def sh_concat(ls: list[int], vec: np.ndarray, normalize: bool = True) -> np.ndarray:
    """Concatenate real_sh over the degrees ``ls`` (one copy of each)."""
    return np.concatenate([real_sh(l, vec, normalize) for l in ls], axis=1)


def rotation_matrix(axis_angle: np.ndarray) -> np.ndarray:
    """exp of the skew matrix of ``axis_angle`` (Rodrigues)."""
    w = np.asarray(axis_angle, dtype=np.float64)
    th = float(np.linalg.norm(w))
    K = np.array([[0.0, -w[2], w[1]], [w[2], 0.0, -w[0]], [-w[1], w[0], 0.0]])
    if th < 1e-300:
        return np.eye(3)
    K = K / th
    return np.eye(3) + math.sin(th) * K + (1.0 - math.cos(th)) * (K @ K)


def random_rotation(rng: np.random.Generator) -> np.ndarray:
    v = rng.standard_normal(3)
    v = v / np.linalg.norm(v) * rng.uniform(0.3, 3.0)
    return rotation_matrix(v)


_SAMPLE = np.random.default_rng(12345).standard_normal((64, 3))


def wigner_D(l: int, R: np.ndarray) -> np.ndarray:
    """D^l(R) with real_sh(l, R r) = D^l(R) real_sh(l, r), by least squares
    over 64 fixed sample directions (exact up to rounding: the harmonics of
    degree l span an invariant subspace)."""
    pts = _SAMPLE / np.linalg.norm(_SAMPLE, axis=1, keepdims=True)
    Y = real_sh(l, pts)
    Yr = real_sh(l, pts @ R.T)
    Dt, *_ = np.linalg.lstsq(Y, Yr, rcond=None)
    return Dt.T


@lru_cache(maxsize=None)
def _cg_cached(l1: int, l2: int, l3: int) -> np.ndarray:
    n1, n2, n3 = 2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1
    if not (abs(l1 - l2) <= l3 <= l1 + l2):
        return np.zeros((n1, n2, n3))
    rng = np.random.default_rng([l1, l2, l3, 7])
    rows = []
    eye = np.eye(n1 * n2 * n3)
    for _ in range(2):
        R = random_rotation(rng)
        D1, D2, D3 = wigner_D(l1, R), wigner_D(l2, R), wigner_D(l3, R)
        # linear map C -> sum_ij C[i,j,k] D1[i,a] D2[j,b] - sum_c D3[k,c] C[a,b,c]
        cols = []
        for t in range(n1 * n2 * n3):
            C = eye[t].reshape(n1, n2, n3)
            lhs = np.einsum("ijk,ia,jb->abk", C, D1, D2)
            rhs = np.einsum("kc,abc->abk", D3, C)
            cols.append((lhs - rhs).ravel())
        rows.append(np.stack(cols, axis=1))
    A = np.concatenate(rows, axis=0)
    _, s, vt = np.linalg.svd(A)
    if s[-1] > 1e-8 * max(1.0, s[0]) or (len(s) > 1 and s[-2] < 1e-6):
        raise RuntimeError(f"CG null space of ({l1},{l2},{l3}) is not one-dimensional")
    C = vt[-1].reshape(n1, n2, n3)
    # orthonormal over (i,j) for each k: by Schur's lemma every column has the
    # same norm, so scale the whole tensor to total squared norm 2l3+1
    C = C * math.sqrt(n3 / float(np.sum(C * C)))
    C[np.abs(C) < 1e-12] = 0.0
    flat = C.ravel()
    first = flat[np.flatnonzero(np.abs(flat) > 1e-9)[0]]
    if first < 0:
        C = -C
    C.setflags(write=False)
    return C


def real_cg(l1: int, l2: int, l3: int) -> np.ndarray:
    """Real Clebsch-Gordan tensor [2l1+1, 2l2+1, 2l3+1] (zeros if the triangle
    rule fails)."""
    return _cg_cached(int(l1), int(l2), int(l3)).copy()
