"""Symmetric contraction (oracle; test infrastructure), fp64.

What it computes (Lesson 12a: Foundations of cuEquivariance, section 21.4.1,
"A descriptor you have already derived for MACE"; "cuEquivariance in PyTorch",
Other operations and layers: SymmetricContraction is MACE-style, with uniform
multiplicities, a contraction degree, a number of elements and integer element
indices): per node n and channel u, with b[n, i, u] the node's features (i over
the components of every input block) and e = element[n],

    out[n, L, k, u] = sum_{nu=1..nu_max} sum_q a_nu[e, q, u]
                      * sum_{i_1..i_nu} B_{nu,q}[i_1, .., i_nu, k] prod_t b[n, i_t, u]

so degree nu is a polynomial of degree nu in the node's own features, one
weight per basis tensor per channel (the printout "[]·a[u]·b[u]·...·b[u] -> C[u]").

Reading taken where the pages are silent: for each degree nu and output irrep
L, the basis tensors B_{nu,q} span all tensors that are symmetric in
(i_1..i_nu) and equivariant, sum B(D x .. x D) = D_L B for every rotation
(and, for O(3), every inversion); the basis is made canonical by taking the
reduced row echelon form of the spanning set (tensors flattened row-major over
(i_1, .., i_nu, k)) and scaling each tensor to unit Frobenius norm with a
positive leading entry. For 32x0e+32x1o -> 32x0e and nu = 1, 2, 3 this gives
1, 2, 2 tensors per degree with 1, 4, 10 nonzero entries - the weight irreps
32x0e+64x0e+64x0e and the num_paths 1, 4, 10 the lesson prints.
"""
from __future__ import annotations

import itertools
from functools import lru_cache

import numpy as np

from . import irreps as I
from .so3 import random_rotation, wigner_D


def _rep(irr, R, inversion=False):
    """Block-diagonal representation of a list of irreps (mul 1 each)."""
    blocks = []
    for t in irr:
        D = wigner_D(t.l, R)
        if inversion and t.p == -1:
            D = -D
        blocks.append(D)
    n = sum(b.shape[0] for b in blocks)
    out = np.zeros((n, n))
    o = 0
    for b in blocks:
        out[o:o + b.shape[0], o:o + b.shape[0]] = b
        o += b.shape[0]
    return out


def _null_space(A, tol=1e-9):
    _, s, vt = np.linalg.svd(A)
    rank = int(np.sum(s > tol * max(1.0, s[0]))) if s.size else 0
    return vt[rank:]


def _rref_canonical(V, tol=1e-10):
    """Rows spanning a subspace -> the canonical basis: reduced row echelon
    form, each row scaled to unit norm with a positive leading entry."""
    A = V.copy()
    rows, cols = A.shape
    r = 0
    for c in range(cols):
        if r == rows:
            break
        piv = r + int(np.argmax(np.abs(A[r:, c])))
        if abs(A[piv, c]) < tol:
            continue
        A[[r, piv]] = A[[piv, r]]
        A[r] /= A[r, c]
        for q in range(rows):
            if q != r:
                A[q] -= A[q, c] * A[r]
        r += 1
    A = A[:r]
    A[np.abs(A) < 1e-12] = 0.0
    out = []
    for row in A:
        row = row / np.linalg.norm(row)
        lead = row[np.flatnonzero(np.abs(row) > 1e-9)[0]]
        out.append(row if lead > 0 else -row)
    return np.array(out).reshape(len(out), -1) if out else np.zeros((0, cols))


@lru_cache(maxsize=None)
def _basis_cached(in_types: tuple, out_type: tuple, nu: int):
    irr_in = [I.MulIrrep(1, l, p) for l, p in in_types]
    L, pL = out_type
    D = sum(2 * l + 1 for l, _ in in_types)
    K = 2 * L + 1
    n = D ** nu * K
    rng = np.random.default_rng([7, nu, L, D])
    # the symmetric tensors: one column per multiset i_1 <= .. <= i_nu and k,
    # the normalised sum of the unit tensors of its orderings
    cols = []
    for multi in itertools.combinations_with_replacement(range(D), nu):
        orders = set(itertools.permutations(multi))
        for k in range(K):
            c = np.zeros(n)
            for o in orders:
                c[np.ravel_multi_index(o + (k,), (D,) * nu + (K,))] = 1.0
            cols.append(c / np.sqrt(len(orders)))
    S = np.array(cols).T                      # [n, n_sym]
    ops = []
    for _ in range(2):
        R = random_rotation(rng)
        ops.append((_rep(irr_in, R), wigner_D(L, R)))
    if any(p != 0 for _, p in in_types):   # O(3): inversion as well
        ops.append((_rep(irr_in, np.eye(3), inversion=True), pL * np.eye(K)))
    cons = []
    for Din, Dout in ops:
        # T -> T (Din x .. x Din) - Dout T as a linear map on the flattened T
        M = np.eye(1)
        for _ in range(nu):
            M = np.kron(M, Din.T)
        cons.append((np.kron(M, np.eye(K)) - np.kron(np.eye(D ** nu), Dout)) @ S)
    C = _null_space(np.concatenate(cons, axis=0))   # coefficients over the symmetric columns
    V = C @ S.T
    B = _rref_canonical(V)
    B.setflags(write=False)
    return B


def symmetric_basis(irr_in, out_irrep, nu: int) -> np.ndarray:
    """Canonical basis tensors [n_q, D, .., D, 2L+1] (nu copies of D) of the
    symmetric, equivariant degree-nu maps from one channel of irr_in (its types,
    mul ignored) to the output irrep (mul ignored)."""
    in_types = tuple((t.l, t.p) for t in irr_in)
    D = sum(2 * l + 1 for l, _ in in_types)
    B = _basis_cached(in_types, (out_irrep.l, out_irrep.p), nu)
    return B.reshape((B.shape[0],) + (D,) * nu + (2 * out_irrep.l + 1,)).copy()


class SymPlan:
    """Everything the oracle needs about one symmetric contraction."""

    def __init__(self, irreps_in: str, irreps_out: str, degrees):
        self.irr_in = I.parse(irreps_in)
        self.irr_out = I.parse(irreps_out)
        muls = {t.mul for t in self.irr_in} | {t.mul for t in self.irr_out}
        if len(muls) != 1:
            raise ValueError("uniform multiplicity required")
        self.mul = muls.pop()
        self.degrees = list(degrees)
        self.D = sum(t.ir_dim for t in self.irr_in)
        self.dim_in = I.dim(self.irr_in)
        self.dim_out = I.dim(self.irr_out)
        # (nu, output block c, basis tensors [n_q, D..D, 2L+1]) in weight order:
        # for each degree, for each output block
        self.terms = []
        for nu in self.degrees:
            for c, t in enumerate(self.irr_out):
                B = symmetric_basis(self.irr_in, t, nu)
                if B.shape[0]:
                    self.terms.append((nu, c, B))
        self.n_weights = sum(B.shape[0] for _, _, B in self.terms)   # per channel and element

    def num_paths(self, nu: int) -> int:
        return sum(int(np.count_nonzero(B)) for n, _, B in self.terms if n == nu)

    def weights_per_degree(self, nu: int) -> int:
        return sum(B.shape[0] for n, _, B in self.terms if n == nu)

    def components(self, x):
        """x [N, dim_in] in ir_mul -> b [N, D, mul] (component i of every block)."""
        parts = []
        o = 0
        for t in self.irr_in:
            parts.append(x[:, o:o + t.dim].reshape(len(x), t.ir_dim, t.mul))
            o += t.dim
        return np.concatenate(parts, axis=1)


def symmetric_contraction(plan: SymPlan, x, weights, element) -> np.ndarray:
    """out [N, dim_out] (ir_mul). weights [num_elements, n_weights, mul] in the
    order of plan.terms; element [N] integer indices into weights."""
    b = plan.components(np.asarray(x, dtype=np.float64))
    N = b.shape[0]
    wsel = np.asarray(weights, dtype=np.float64)[np.asarray(element, dtype=np.int64)]   # [N, n_weights, mul]
    out = np.zeros((N, plan.dim_out))
    offs = I.offsets(plan.irr_out)
    q0 = 0
    for nu, c, B in plan.terms:
        letters = "abc"[:nu]
        # prod_t b[n, i_t, u] contracted with B[q, i_1..i_nu, k]
        expr = "q" + letters + "k," + ",".join(f"n{l}u" for l in letters) + "->nqku"
        poly = np.einsum(expr, B, *([b] * nu))
        contrib = np.einsum("nqku,nqu->nku", poly, wsel[:, q0:q0 + B.shape[0]])
        t = plan.irr_out[c]
        out[:, offs[c]:offs[c] + t.dim] += contrib.reshape(N, t.dim)
        q0 += B.shape[0]
    return out


def symmetric_contraction_brute(plan: SymPlan, x, weights, element) -> np.ndarray:
    """The same sum written as explicit loops (tiny inputs)."""
    b = plan.components(np.asarray(x, dtype=np.float64))
    N = b.shape[0]
    out = np.zeros((N, plan.dim_out))
    offs = I.offsets(plan.irr_out)
    for n in range(N):
        q0 = 0
        for nu, c, B in plan.terms:
            L2 = B.shape[-1]
            for q in range(B.shape[0]):
                for u in range(plan.mul):
                    a = weights[element[n], q0 + q, u]
                    for idx in itertools.product(range(plan.D), repeat=nu):
                        for k in range(L2):
                            coef = B[(q,) + idx + (k,)]
                            if coef == 0.0:
                                continue
                            p = 1.0
                            for i in idx:
                                p *= b[n, i, u]
                            out[n, offs[c] + k * plan.mul + u] += a * coef * p
            q0 += B.shape[0]
    return out
