"""Seeded synthetic workloads for the fused tensor-product convolution.

This module only draws random numbers and builds graphs. It holds none of the
tensor-product arithmetic (no irreps parsing, no spherical harmonics, no
Clebsch-Gordan coefficients): every size that depends on the method (feature
widths, number of weights per edge) is passed in by the caller. Both the CUDA
path's tests/benchmark and the fp64 oracle consume the arrays made here.

Workloads (sizes follow the benchmark table of the equivariant graph
convolution this library implements):

* ``tiny``      N=32, E=512, src/dst uniform (unsorted), unit edge vectors.
* ``medium``    N=4096 radius graph (r=5, mean degree ~32, E~131k), cell-ordered
                nodes, dst-sorted.
* ``large``     N=65536, in-degree ~ Poisson(32) (E~2.1M), src uniform,
                unit edge vectors, dst-sorted; x and w later rounded to bf16.
* ``xlarge``    N=262144 radius graph (r=5, E~8.4M), cell-ordered, dst-sorted.
* ``fd``        16 nodes, 64 uniform random edges (finite-difference checks).

Random draws use ``numpy.random.default_rng([seed, workload_id])`` in the fixed
order graph -> edge vectors -> x -> w -> grad_out (w in blocks of 65536 rows,
each block from a generator seeded by the next draw of the stream).
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "radius_graph", "make_graph", "make_features", "make_radial_mlp"]


@dataclass(frozen=True)
class Workload:
    name: str
    wid: int                 # id mixed into the seed
    irreps_in: str
    irreps_sh: str
    irreps_out: str
    n_nodes: int
    graph: str               # "uniform" | "radius" | "poisson"
    n_edges: int = 0         # for "uniform"
    radius: float = 5.0      # for "radius"
    mean_degree: float = 32.0
    dtype: str = "f32"       # "f32" or "bf16" (x and w rounded to bf16)
    w_scale: str = "one"     # "one": N(0,1); "inv_sqrt_paths": N(0,1)/sqrt(P)
    backward: bool = False
    notes: dict = field(default_factory=dict)

    def box_side(self) -> float:
        """Side of the periodic cube whose density gives ``mean_degree``
        neighbours inside a ball of ``radius``."""
        return (self.n_nodes * (4.0 / 3.0) * math.pi * self.radius ** 3 / self.mean_degree) ** (1.0 / 3.0)


WORKLOADS = {
    "tiny": Workload("tiny", 0, "32x0e+32x1o", "0e+1o+2e", "32x0e+32x1o+32x2e",
                     32, "uniform", n_edges=512),
    "medium": Workload("medium", 1, "128x0e+128x1o+128x2e", "0e+1o+2e+3o",
                       "128x0e+128x1o+128x2e", 4096, "radius", w_scale="inv_sqrt_paths"),
    "large": Workload("large", 2, "64x0e+64x1o+64x2e+64x3o", "0e+1o+2e+3o",
                      "64x0e+64x1o+64x2e+64x3o", 65536, "poisson", dtype="bf16",
                      w_scale="inv_sqrt_paths"),
    "xlarge": Workload("xlarge", 3, "32x0e+32x1o", "0e+1o+2e", "32x0e+32x1o+32x2e",
                       262144, "radius"),
    "fwdbwd": Workload("fwdbwd", 4, "128x0e+128x1o+128x2e", "0e+1o+2e+3o",
                       "128x0e+128x1o+128x2e", 4096, "radius", w_scale="inv_sqrt_paths",
                       backward=True),
    "fd": Workload("fd", 5, "128x0e+128x1o+128x2e", "0e+1o+2e+3o",
                   "128x0e+128x1o+128x2e", 16, "uniform", n_edges=64, backward=True),
}
# the fwd+bwd workload reuses the medium graph and features: same seed stream
_SEED_ALIAS = {"fwdbwd": 1}


def _rng(w: Workload, seed: int) -> np.random.Generator:
    return np.random.default_rng([seed, _SEED_ALIAS.get(w.name, w.wid)])


def _unit_vectors(rng: np.random.Generator, n: int) -> np.ndarray:
    v = rng.standard_normal((n, 3))
    nrm = np.linalg.norm(v, axis=1, keepdims=True)
    nrm[nrm == 0] = 1.0
    return v / nrm


def radius_graph(pos: np.ndarray, box: float, r: float):
    """All ordered pairs (j -> i), i != j, with minimum-image distance < r in a
    periodic cube of side ``box``. Returns (src, dst, vec) with vec = pos[src] -
    pos[dst] (minimum image), sorted by (dst, src). Uses a cell list; needs at
    least 3 cells per side so the 27 neighbour cells are distinct."""
    n = pos.shape[0]
    nc = int(math.floor(box / r))
    if nc < 3:
        raise ValueError("box too small for a 27-cell neighbour search")
    cell = np.minimum((pos / (box / nc)).astype(np.int64), nc - 1)
    cid = (cell[:, 0] * nc + cell[:, 1]) * nc + cell[:, 2]
    order = np.argsort(cid, kind="stable")
    if not np.array_equal(order, np.arange(n)):
        raise ValueError("radius_graph expects nodes already in cell order")
    counts = np.bincount(cid, minlength=nc ** 3)
    start = np.concatenate([[0], np.cumsum(counts)[:-1]])
    r2 = r * r
    srcs, dsts = [], []
    for ox in (-1, 0, 1):
        for oy in (-1, 0, 1):
            for oz in (-1, 0, 1):
                nb = (((cell[:, 0] + ox) % nc) * nc + (cell[:, 1] + oy) % nc) * nc + (cell[:, 2] + oz) % nc
                cnt = counts[nb]
                tot = int(cnt.sum())
                if tot == 0:
                    continue
                ii = np.repeat(np.arange(n, dtype=np.int64), cnt)
                first = np.repeat(np.cumsum(cnt) - cnt, cnt)
                jj = start[nb][ii] + (np.arange(tot, dtype=np.int64) - first)
                d = pos[jj] - pos[ii]
                d -= box * np.round(d / box)
                keep = (np.einsum("ij,ij->i", d, d) < r2) & (ii != jj)
                srcs.append(jj[keep])
                dsts.append(ii[keep])
    src = np.concatenate(srcs)
    dst = np.concatenate(dsts)
    o = np.lexsort((src, dst))
    src, dst = src[o], dst[o]
    vec = pos[src] - pos[dst]
    vec -= box * np.round(vec / box)
    return src.astype(np.int32), dst.astype(np.int32), vec


def make_graph(w: Workload, seed: int = 0):
    """Draw the graph of workload ``w``. Returns (rng, src, dst, edge_vec, n_nodes);
    ``rng`` continues the same stream for the features."""
    rng = _rng(w, seed)
    n = w.n_nodes
    if w.graph == "uniform":
        src = rng.integers(0, n, size=w.n_edges).astype(np.int32)
        dst = rng.integers(0, n, size=w.n_edges).astype(np.int32)
        vec = _unit_vectors(rng, w.n_edges)
    elif w.graph == "poisson":
        deg = rng.poisson(w.mean_degree, size=n)
        dst = np.repeat(np.arange(n, dtype=np.int32), deg)
        src = rng.integers(0, n, size=dst.shape[0]).astype(np.int32)
        vec = _unit_vectors(rng, dst.shape[0])
    elif w.graph == "radius":
        box = w.box_side()
        pos = rng.uniform(0.0, box, size=(n, 3))
        nc = int(math.floor(box / w.radius))
        cell = np.minimum((pos / (box / nc)).astype(np.int64), nc - 1)
        cid = (cell[:, 0] * nc + cell[:, 1]) * nc + cell[:, 2]
        pos = pos[np.argsort(cid, kind="stable")]          # relabel in cell order
        src, dst, vec = radius_graph(pos, box, w.radius)
    else:
        raise ValueError(w.graph)
    return rng, src, dst, vec, n


def _normal_rows(rng: np.random.Generator, rows: int, cols: int, dtype, chunk: int = 65536) -> np.ndarray:
    """[rows, cols] N(0,1) draws. Blocks of ``chunk`` rows each come from their
    own generator, seeded by one draw from ``rng`` per block, and are filled on
    several threads (the full-size weight streams hold up to 3e9 values)."""
    from concurrent.futures import ThreadPoolExecutor
    n_blocks = (rows + chunk - 1) // chunk
    seeds = rng.integers(0, 2 ** 63, size=n_blocks)
    out = np.empty((rows, cols), dtype=dtype)

    def fill(i):
        lo, hi = i * chunk, min(rows, (i + 1) * chunk)
        np.random.default_rng(int(seeds[i])).standard_normal((hi - lo, cols), dtype=dtype, out=out[lo:hi])

    if n_blocks:
        with ThreadPoolExecutor(max(1, min(16, n_blocks, os.cpu_count() or 1))) as ex:
            list(ex.map(fill, range(n_blocks)))
    return out


def make_features(rng: np.random.Generator, w: Workload, n_nodes: int, n_edges: int,
                  dim_x: int, weight_numel: int, n_paths: int, dim_out: int, dtype=np.float64):
    """Draw x [N, dim_x], w [E, weight_numel] and (for backward workloads)
    grad_out [N, dim_out], continuing ``rng`` (w in blocks of rows, see
    ``_normal_rows``). ``dtype`` float64 (default) or float32; the full-size
    workloads use float32 draws so the weight stream (up to 1.9e9 values)
    fits in host memory."""
    x = rng.standard_normal((n_nodes, dim_x), dtype=dtype)
    wt = _normal_rows(rng, n_edges, weight_numel, dtype)
    if w.w_scale == "inv_sqrt_paths":
        wt *= dtype(1.0 / math.sqrt(n_paths))
    g = rng.standard_normal((n_nodes, dim_out), dtype=dtype) if w.backward else None
    return x, wt, g


def make_radial_mlp(seed: int, wid: int, hidden: int, weight_numel: int, dtype=np.float32):
    """Parameters of a radial network Linear(1, hidden) -> SiLU ->
    Linear(hidden, weight_numel): w1, b1 ~ N(0, 1) [hidden]; w2 ~ N(0, 1/hidden)
    [hidden, weight_numel] (hidden-major); b2 ~ N(0, 0.01) [weight_numel]. Drawn
    from a stream of their own, default_rng([seed, wid, 7])."""
    rng = np.random.default_rng([seed, wid, 7])
    w1 = rng.standard_normal(hidden).astype(dtype)
    b1 = rng.standard_normal(hidden).astype(dtype)
    w2 = (rng.standard_normal((hidden, weight_numel)) / math.sqrt(hidden)).astype(dtype)
    b2 = (0.1 * rng.standard_normal(weight_numel)).astype(dtype)
    return w1, b1, w2, b2


def subgraph_uniform(seed: int, n_nodes: int, n_edges: int, wid: int = 99):
    """A small uniform random graph with unit edge vectors (unsorted dst)."""
    rng = np.random.default_rng([seed, wid])
    src = rng.integers(0, n_nodes, size=n_edges).astype(np.int32)
    dst = rng.integers(0, n_nodes, size=n_edges).astype(np.int32)
    vec = _unit_vectors(rng, n_edges)
    return rng, src, dst, vec
