"""Channelwise (uvu) tensor-product convolution, fp64 (oracle; test infrastructure).

What it computes (Lesson 12a: Foundations of cuEquivariance, section 21.4, the
descriptor ``[ijk]·a[uv]·b[iu]·c[jv] -> D[kuv]`` with v = 1; "cuEquivariance in
PyTorch", Channelwise product with external per-example weights and
SegmentedPolynomial: gather and scatter)::

    out[d, c, k, u] = sum_{e: dst[e] = d} sum_{p = (a, b, c)} w[e, p, u]
                      * sum_{i, j} C_p[i, j, k] * x[src[e], a, i, u] * sh[e, b, j]

* a runs over the blocks of the node irreps, b over the blocks of the edge
  harmonics, c over the output blocks; C_p is the real Clebsch-Gordan tensor
  of (l_a, l_b, l_c) from ``so3``.
* Paths (section 21.4, the e3nn instruction loop and its filtered counterpart):
  for a in input blocks, for b in harmonic blocks, for l_o from |l_a-l_b| to
  l_a+l_b ascending, keep (l_o, p_a p_b) when that irrep type is one of the
  outputs; uvu needs mul(out) = mul(a). The path order fixes the weight layout
  w[e, p*mul + u] (weights "a[uv]" with v = 1).
* Reading taken: paths that land on the same output irrep type sum into the one
  output block of that type; outputs appear in the order of the output string;
  an output block no path reaches stays zero; destinations without edges are
  zero ("repeated receivers sum, and destinations without incoming edges remain
  zero").
* Features use the ``ir_mul`` layout: block element (i, u) at off + i*mul + u.

Radial network (same page, Trainable message passing): w = radial(|edge vector|)
with radial = Linear(1, H) -> SiLU -> Linear(H, weight_numel) (``radial_mlp``).

Backward (the map is linear in each of x, sh, w, so these are exact)::

    dx[s,a,i,u] = sum_{e: src[e]=s} sum_{p: a_p=a} w[e,p,u] sum_{j,k} C_p[i,j,k] sh[e,b,j] g[dst[e],c,k,u]
    dw[e,p,u]   = sum_{i,j,k} C_p[i,j,k] x[src[e],a,i,u] sh[e,b,j] g[dst[e],c,k,u]
    dsh[e,b,j]  = sum_{p: b_p=b} sum_{i,k,u} C_p[i,j,k] x[src[e],a,i,u] w[e,p,u] g[dst[e],c,k,u]
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import irreps as I
from .so3 import real_cg


@dataclass(frozen=True)
class Path:
    a: int    # input block index
    b: int    # harmonic block index
    c: int    # output block index
    la: int
    lb: int
    lc: int


def _product_types(t1: I.MulIrrep, t2: I.MulIrrep):
    """Irrep types in t1 x t2, l ascending (triangle rule; parity multiplies)."""
    p = t1.p * t2.p if (t1.p != 0 and t2.p != 0) else 0
    return [(lo, p) for lo in range(abs(t1.l - t2.l), t1.l + t2.l + 1)]


def enumerate_paths(irr_in, irr_sh, irr_out) -> list[Path]:
    """Channelwise paths filtered by the requested output types (section 21.4:
    ``32x0e+32x1o`` x ``0e+1o`` -> ``32x0e+32x1o`` gives 4 paths)."""
    out_types = {}
    for c, t in enumerate(irr_out):
        if t.ir() in out_types:
            raise ValueError("duplicate output irrep type")
        out_types[t.ir()] = c
    paths = []
    for a, ta in enumerate(irr_in):
        for b, tb in enumerate(irr_sh):
            for ir in _product_types(ta, tb):
                if ir in out_types:
                    c = out_types[ir]
                    if irr_out[c].mul != ta.mul:
                        raise ValueError("uvu needs equal input/output multiplicity")
                    paths.append(Path(a, b, c, ta.l, tb.l, ir[0]))
    return paths


def enumerate_instructions_lmax(irr_in, irr_sh, lmax: int):
    """The e3nn-style loop of section 21.4: every product irrep with l <= lmax
    becomes its own instruction and its own output block. Returns a list of
    (a, b, out_index, (mul, l, p)) tuples."""
    instr = []
    for a, ta in enumerate(irr_in):
        for b, tb in enumerate(irr_sh):
            for ir in _product_types(ta, tb):
                if ir[0] <= lmax:
                    instr.append((a, b, len(instr), (ta.mul, ir[0], ir[1])))
    return instr


class Plan:
    """Everything the oracle needs about one (irreps_in, irreps_sh, irreps_out)."""

    def __init__(self, irreps_in: str, irreps_sh: str, irreps_out: str):
        self.irr_in = I.parse(irreps_in)
        self.irr_sh = I.parse(irreps_sh)
        self.irr_out = I.parse(irreps_out)
        for t in self.irr_sh:
            if t.mul != 1:
                raise ValueError("harmonic irreps must have multiplicity 1")
        muls = {t.mul for t in self.irr_in} | {t.mul for t in self.irr_out}
        if len(muls) != 1:
            raise ValueError("uniform multiplicity required")
        self.mul = muls.pop()
        self.paths = enumerate_paths(self.irr_in, self.irr_sh, self.irr_out)
        self.off_in = I.offsets(self.irr_in)
        self.off_sh = I.offsets(self.irr_sh)
        self.off_out = I.offsets(self.irr_out)
        self.dim_in = I.dim(self.irr_in)
        self.dim_sh = I.dim(self.irr_sh)
        self.dim_out = I.dim(self.irr_out)
        self.n_paths = len(self.paths)
        self.weight_numel = self.n_paths * self.mul
        self.cg = [real_cg(p.la, p.lb, p.lc) for p in self.paths]

    # views into ir_mul blocks -------------------------------------------------
    def xblock(self, x: np.ndarray, a: int) -> np.ndarray:
        t = self.irr_in[a]
        o = self.off_in[a]
        return x[..., o:o + t.dim].reshape(x.shape[:-1] + (t.ir_dim, t.mul))

    def shblock(self, sh: np.ndarray, b: int) -> np.ndarray:
        t = self.irr_sh[b]
        o = self.off_sh[b]
        return sh[..., o:o + t.ir_dim]

    def oblock_slice(self, c: int) -> slice:
        return slice(self.off_out[c], self.off_out[c] + self.irr_out[c].dim)


def conv_forward_brute(plan: Plan, x, sh, w, src, dst, n_dst: int) -> np.ndarray:
    """Explicit loops over edges, paths and (i, j, k); a separate scatter.
    For tiny graphs only."""
    mul = plan.mul
    out = np.zeros((n_dst, plan.dim_out))
    for e in range(len(src)):
        s, d = int(src[e]), int(dst[e])
        msg = np.zeros(plan.dim_out)
        for p, P in enumerate(plan.paths):
            C = plan.cg[p]
            wp = w[e, p * mul:(p + 1) * mul]
            oa, ob, oc = plan.off_in[P.a], plan.off_sh[P.b], plan.off_out[P.c]
            for i in range(2 * P.la + 1):
                for j in range(2 * P.lb + 1):
                    for k in range(2 * P.lc + 1):
                        cijk = C[i, j, k]
                        if cijk == 0.0:
                            continue
                        xs = x[s, oa + i * mul:oa + (i + 1) * mul]
                        msg[oc + k * mul:oc + (k + 1) * mul] += wp * cijk * xs * sh[e, ob + j]
        out[d] += msg
    return out


def edge_messages(plan: Plan, x, sh, w, src) -> np.ndarray:
    """Per-edge messages m[e] (before the scatter), vectorised over edges."""
    E = len(src)
    mul = plan.mul
    xs = x[src]
    m = np.zeros((E, plan.dim_out))
    for p, P in enumerate(plan.paths):
        xa = plan.xblock(xs, P.a)                       # [E, 2la+1, mul]
        shb = plan.shblock(sh, P.b)                     # [E, 2lb+1]
        t = np.einsum("ijk,eiu,ej->eku", plan.cg[p], xa, shb)
        t *= w[:, None, p * mul:(p + 1) * mul]
        sl = plan.oblock_slice(P.c)
        m[:, sl] += t.reshape(E, (2 * P.lc + 1) * mul)
    return m


def conv_forward(plan: Plan, x, sh, w, src, dst, n_dst: int) -> np.ndarray:
    """Gather, contract every path, sum-scatter to ``dst`` (np.add.at)."""
    out = np.zeros((n_dst, plan.dim_out))
    np.add.at(out, np.asarray(dst, dtype=np.int64), edge_messages(plan, x, sh, w, src))
    return out


def unsimplified_order(plan: Plan) -> list[int]:
    """Path indices in the order of the per-path ("unsimplified") output blocks:
    grouped by output irrep type in the order of the output list, paths of one
    type in path order (Lesson 12a, section 21.4: the descriptor of
    32x0e+32x1o x 0e+1o prints D=32x0e+32x0e+32x1o+32x1o)."""
    return [p for c in range(len(plan.irr_out)) for p, P in enumerate(plan.paths) if P.c == c]


def conv_forward_unsimplified(plan: Plan, x, sh, w, src, dst, n_dst: int) -> np.ndarray:
    """Gather, contract, sum-scatter with one output block of mul*(2 l_c + 1)
    per path (in ``unsimplified_order``) instead of one per output type."""
    E = len(src)
    mul = plan.mul
    xs = x[src]
    blocks = []
    for p in unsimplified_order(plan):
        P = plan.paths[p]
        t = np.einsum("ijk,eiu,ej->eku", plan.cg[p], plan.xblock(xs, P.a), plan.shblock(sh, P.b))
        t *= w[:, None, p * mul:(p + 1) * mul]
        blocks.append(t.reshape(E, (2 * P.lc + 1) * mul))
    m = np.concatenate(blocks, axis=1) if blocks else np.zeros((E, 0))
    out = np.zeros((n_dst, m.shape[1]))
    np.add.at(out, np.asarray(dst, dtype=np.int64), m)
    return out


def conv_forward_mean(plan: Plan, x, sh, w, src, dst, n_dst: int) -> np.ndarray:
    """reduce="mean" ("cuEquivariance in PyTorch", Other operations and layers:
    the convolution layer's mean reduction): the sum of a destination's
    messages divided by its number of incoming edges; destinations without
    edges stay zero."""
    out = conv_forward(plan, x, sh, w, src, dst, n_dst)
    deg = np.bincount(np.asarray(dst, dtype=np.int64), minlength=n_dst)
    return out / np.maximum(deg, 1)[:, None]


def conv_backward(plan: Plan, x, sh, w, src, dst, g):
    """Exact gradients (dx, dw, dsh) of <g, conv_forward(x, sh, w)>."""
    E = len(src)
    mul = plan.mul
    xs = x[src]
    gd = g[dst]
    dxs = np.zeros_like(xs)
    dw = np.zeros_like(w)
    dsh = np.zeros_like(sh)
    for p, P in enumerate(plan.paths):
        C = plan.cg[p]
        xa = plan.xblock(xs, P.a)                                  # [E, ia, u]
        shb = plan.shblock(sh, P.b)                                # [E, jb]
        gc = gd[:, plan.oblock_slice(P.c)].reshape(E, 2 * P.lc + 1, mul)  # [E, k, u]
        wp = w[:, p * mul:(p + 1) * mul]                           # [E, u]
        dw[:, p * mul:(p + 1) * mul] += np.einsum("ijk,eiu,ej,eku->eu", C, xa, shb, gc)
        o = plan.off_sh[P.b]
        dsh[:, o:o + 2 * P.lb + 1] += np.einsum("ijk,eiu,eu,eku->ej", C, xa, wp, gc)
        oa = plan.off_in[P.a]
        da = np.einsum("ijk,ej,eu,eku->eiu", C, shb, wp, gc)
        dxs[:, oa:oa + (2 * P.la + 1) * mul] += da.reshape(E, (2 * P.la + 1) * mul)
    dx = np.zeros_like(x)
    np.add.at(dx, np.asarray(src, dtype=np.int64), dxs)
    return dx, dw, dsh


def silu(z):
    """SiLU (sigmoid-weighted linear unit) z * sigmoid(z) with sigmoid(z) =
    1 / (1 + exp(-z)), evaluated as exp(-|z|) / (1 + exp(-|z|)) for z < 0 so
    that no exponential overflows."""
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(-np.abs(z))
    return np.where(z >= 0, z / (1.0 + e), z * e / (1.0 + e))


def radial_mlp(vec, w1, b1, w2, b2):
    """Per-edge weights from the edge length by the radial network of
    "cuEquivariance in PyTorch", Trainable message passing: Linear(1, H) ->
    SiLU -> Linear(H, weight_numel) applied to |edge_vector|.
    vec [E, 3]; w1, b1 [H]; w2 [H, weight_numel]; b2 [weight_numel] -> [E, weight_numel]."""
    r = np.linalg.norm(np.asarray(vec, dtype=np.float64), axis=1)
    h = silu(r[:, None] * np.asarray(w1, np.float64)[None, :] + np.asarray(b1, np.float64)[None, :])
    return h @ np.asarray(w2, np.float64) + np.asarray(b2, np.float64)[None, :]


def csr_build(keys, n: int):
    """Stable counting sort of ``keys`` in [0, n): returns (perm, row_ptr,
    keys_sorted) with perm[k] = original position of the k-th sorted item,
    equal keys keeping their original order, row_ptr[0] = 0, row_ptr[n] = E."""
    keys = np.asarray(keys, dtype=np.int64)
    if keys.size and (keys.min() < 0 or keys.max() >= n):
        raise ValueError("key out of range")
    counts = np.bincount(keys, minlength=n)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    perm = np.argsort(keys, kind="stable")
    return perm.astype(np.int32), row_ptr.astype(np.int32), keys[perm].astype(np.int32)


def csr_build_loops(keys, n: int):
    """The same counting sort written as explicit loops (tiny inputs): count,
    exclusive scan, then place items in input order."""
    keys = [int(k) for k in keys]
    count = [0] * n
    for k in keys:
        count[k] += 1
    row_ptr = [0] * (n + 1)
    for d in range(n):
        row_ptr[d + 1] = row_ptr[d] + count[d]
    cursor = row_ptr[:n]
    cursor = list(cursor)
    perm = [0] * len(keys)
    for e, k in enumerate(keys):
        perm[cursor[k]] = e
        cursor[k] += 1
    return (np.array(perm, dtype=np.int32), np.array(row_ptr, dtype=np.int32),
            np.array([keys[p] for p in perm], dtype=np.int32))


def rms_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / sqrt(mean(ref^2)) over one output tensor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    if rms == 0.0:
        return float(np.max(np.abs(got - ref)))
    return float(np.max(np.abs(got - ref)) / rms)
