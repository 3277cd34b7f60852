"""ctypes front end of the plain-C fp64 oracle (oracle/tpconv_ref.c).

Test infrastructure only. ``build()`` compiles the C file with gcc and OpenMP
into ``oracle/_build/``; the functions below take numpy arrays and a
``tp.Plan`` and return float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .tp import Plan

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tpconv_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libtpconv_ref.so")
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB_PATH)
        _lib.ref_num_threads.restype = ctypes.c_int
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads() -> int:
    return int(_load().ref_num_threads())


def _tables(plan: Plan):
    pi = np.array([[P.la, P.lb, P.lc, plan.off_in[P.a], plan.off_sh[P.b], plan.off_out[P.c]]
                   for P in plan.paths], dtype=np.int32).reshape(-1)
    flat = [np.ascontiguousarray(C, dtype=np.float64).ravel() for C in plan.cg]
    cg_off = np.zeros(len(flat), dtype=np.int64)
    if flat:
        cg_off[1:] = np.cumsum([f.size for f in flat])[:-1]
    cg = np.concatenate(flat) if flat else np.zeros(1)
    return pi, cg, cg_off


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def conv_forward(plan: Plan, x, sh, w, src, row_ptr, n_dst: int, rows=None, threads: int = 0):
    """out rows for dst-sorted edges (``row_ptr`` over the edge order). With
    ``rows`` given, only those destination rows are computed (in that order)."""
    lib = _load()
    pi, cg, cg_off = _tables(plan)
    x, sh, w = _f64(x), _f64(sh), _f64(w)
    src = _i32(src)
    rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
    rows_a = None if rows is None else _i32(rows)
    n_list = n_dst if rows is None else len(rows_a)
    out = np.zeros((n_list, plan.dim_out))
    lib.ref_conv_forward(ctypes.c_int(plan.n_paths), _p(pi), _p(cg), _p(cg_off), ctypes.c_int(plan.mul),
                         ctypes.c_int(plan.dim_in), ctypes.c_int(plan.dim_sh), ctypes.c_int(plan.dim_out),
                         ctypes.c_int(plan.weight_numel), _p(x), _p(sh), _p(w), _p(src), _p(rp),
                         ctypes.c_int(n_dst), _p(rows_a), ctypes.c_int(n_list), _p(out), ctypes.c_int(threads))
    return out


def conv_backward_edges(plan: Plan, x, sh, w, g, src, dst, edges=None, threads: int = 0):
    """(dw, dsh) for the listed edges (all when None)."""
    lib = _load()
    pi, cg, cg_off = _tables(plan)
    x, sh, w, g = _f64(x), _f64(sh), _f64(w), _f64(g)
    src, dst = _i32(src), _i32(dst)
    ed = None if edges is None else np.ascontiguousarray(edges, dtype=np.int64)
    n_list = len(src) if edges is None else len(ed)
    dw = np.zeros((n_list, plan.weight_numel))
    dsh = np.zeros((n_list, plan.dim_sh))
    lib.ref_conv_backward_edges(ctypes.c_int(plan.n_paths), _p(pi), _p(cg), _p(cg_off), ctypes.c_int(plan.mul),
                                ctypes.c_int(plan.dim_in), ctypes.c_int(plan.dim_sh), ctypes.c_int(plan.dim_out),
                                ctypes.c_int(plan.weight_numel), _p(x), _p(sh), _p(w), _p(g), _p(src), _p(dst),
                                _p(ed), ctypes.c_int64(n_list), _p(dw), _p(dsh), ctypes.c_int(threads))
    return dw, dsh


def conv_backward_dx(plan: Plan, sh, w, g, dst, src_perm, src_row_ptr, n_src: int, rows=None, threads: int = 0):
    """dx rows; the edges of source s are src_perm[src_row_ptr[s]:src_row_ptr[s+1]]."""
    lib = _load()
    pi, cg, cg_off = _tables(plan)
    sh, w, g = _f64(sh), _f64(w), _f64(g)
    dst, sp = _i32(dst), _i32(src_perm)
    srp = np.ascontiguousarray(src_row_ptr, dtype=np.int64)
    rows_a = None if rows is None else _i32(rows)
    n_list = n_src if rows is None else len(rows_a)
    dx = np.zeros((n_list, plan.dim_in))
    lib.ref_conv_backward_dx(ctypes.c_int(plan.n_paths), _p(pi), _p(cg), _p(cg_off), ctypes.c_int(plan.mul),
                             ctypes.c_int(plan.dim_in), ctypes.c_int(plan.dim_sh), ctypes.c_int(plan.dim_out),
                             ctypes.c_int(plan.weight_numel), _p(sh), _p(w), _p(g), _p(dst), _p(sp), _p(srp),
                             _p(rows_a), ctypes.c_int(n_list), _p(dx), ctypes.c_int(threads))
    return dx
