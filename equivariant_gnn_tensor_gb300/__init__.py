"""Python binding of libtpconv.so, the sm_103a fused equivariant
tensor-product convolution (see include/tpconv.h for the C contract).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels. PyTorch supplies device memory and the current CUDA
stream. Importing this package raises if the library has not been built;
there is no CPU fallback.

Entry points (same names as the C ABI)::

    desc = tp_desc_create("128x0e+128x1o+128x2e", "0e+1o+2e+3o", "128x0e+128x1o+128x2e")
    sh = tp_spherical_harmonics(desc, vec)                 # [E, dim_sh]
    perm, row_ptr, dst_sorted = tp_csr_build(dst, n_dst)   # stable, dst-sorted CSR
    out = tp_conv_forward(desc, x, sh, w, src, row_ptr, n_dst)
    dx, dw, dsh = tp_conv_backward(desc, grad_out, x, sh, w, src, dst_sorted, row_ptr,
                                   src_perm, src_row_ptr)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtpconv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
                      " (or python equivariant_gnn_tensor_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

TP_OK = 0
STATUS_NAMES = {0: "TP_OK", 1: "TP_ERR_PARSE", 2: "TP_ERR_UNSUPPORTED", 4: "TP_ERR_INDEX",
                5: "TP_ERR_ALIGN", 6: "TP_ERR_CUDA", 7: "TP_ERR_ARG", 8: "TP_ERR_TIMEOUT", 9: "TP_ERR_CAPACITY"}
TP_F32, TP_BF16_IN_F32_OUT = 0, 1
TP_IR_MUL, TP_MUL_IR = 0, 1
TP_DEV_ERR_INDEX, TP_DEV_ERR_TIMEOUT, TP_DEV_ERR_SEGMENT = 1, 2, 4
TP_REDUCE_SUM, TP_REDUCE_MEAN = 0, 1
EXPORTS = ["tp_desc_create", "tp_desc_create_unsimplified", "tp_desc_query", "tp_desc_path", "tp_desc_cg", "tp_desc_destroy",
           "tp_spherical_harmonics", "tp_csr_workspace_size", "tp_csr_build", "tp_csr_build_noalloc",
           "tp_csr_build_noalloc_max_edges", "tp_conv_forward_workspace_size", "tp_conv_forward",
           "tp_conv_forward_vec", "tp_conv_forward_mlp", "tp_conv_forward_ex_workspace_size", "tp_conv_forward_ex",
           "tp_transpose_layout", "tp_symc_create", "tp_symc_query", "tp_symc_term", "tp_symc_destroy",
           "tp_symmetric_contraction", "tp_symc_kernel_source",
           "tp_conv_backward", "tp_conv_backward_workspace_size", "tp_set_tuning", "tp_get_tuning", "tp_device_status", "tp_status_string",
           "tp_abi_version"]


class TPError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib.tp_status_string(status).decode()
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({msg})")


class _Info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_paths", "mul", "dim_x", "dim_sh", "dim_out", "weight_numel", "n_in", "n_sh", "n_out",
        "lmax_in", "lmax_sh", "lmax_out", "cg_nnz", "layout")]


class _Tuning(ctypes.Structure):
    _fields_ = [("ring_stage_bytes", ctypes.c_int32), ("ring_stages", ctypes.c_int32), ("ring_warps", ctypes.c_int32),
                ("ring_rounds", ctypes.c_int32), ("ring_pack", ctypes.c_int32), ("disable_split", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("disable_mma", ctypes.c_int32), ("mma_stages", ctypes.c_int32),
                ("bwd_stage_bytes", ctypes.c_int32), ("bwd_stages", ctypes.c_int32), ("bwd_warps", ctypes.c_int32),
                ("disable_ring_bwd", ctypes.c_int32), ("disable_symc_jit", ctypes.c_int32)]


class _Mlp(ctypes.Structure):
    _fields_ = [("w1", ctypes.c_void_p), ("b1", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("b2", ctypes.c_void_p),
                ("hidden", ctypes.c_int32)]


class _FwdArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("x", ctypes.c_void_p), ("sh", ctypes.c_void_p), ("vec", ctypes.c_void_p),
                ("normalize", ctypes.c_int32), ("mlp", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("src", ctypes.c_void_p), ("row_ptr", ctypes.c_void_p), ("index_bits", ctypes.c_int32),
                ("reduce", ctypes.c_int32), ("N_src", ctypes.c_int32), ("N_dst", ctypes.c_int32),
                ("E", ctypes.c_int64), ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


class _SymcInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("mul", "dim_in", "dim_out", "max_degree", "n_weights", "n_terms")] + \
        [("num_paths", ctypes.c_int32 * 3), ("weights_per_degree", ctypes.c_int32 * 3)]


class _Path(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("a", "b", "c", "la", "lb", "lc")]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_sigs = {
    "tp_desc_create": [ctypes.c_char_p, ctypes.c_char_p, ctypes.c_char_p, ctypes.c_int, ctypes.POINTER(_vp)],
    "tp_desc_create_unsimplified": [ctypes.c_char_p, ctypes.c_char_p, ctypes.c_char_p, ctypes.c_int,
                                    ctypes.POINTER(_vp)],
    "tp_desc_query": [_vp, ctypes.POINTER(_Info)],
    "tp_desc_path": [_vp, _i32, ctypes.POINTER(_Path)],
    "tp_desc_cg": [_vp, _i32, _vp, _i64],
    "tp_spherical_harmonics": [_vp, _vp, _i64, _i32, _vp, _vp],
    "tp_csr_workspace_size": [_i64, _i32, ctypes.POINTER(_sz)],
    "tp_csr_build": [_vp, _i64, _i32, _vp, _vp, _vp, _vp, _sz, _vp],
    "tp_csr_build_noalloc": [_vp, _i64, _i32, _vp, _vp, _vp, _vp],
    "tp_conv_forward_workspace_size": [_vp, ctypes.c_int, _i32, _i64, ctypes.POINTER(_sz)],
    "tp_conv_forward": [_vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp, _sz, _vp],
    "tp_conv_forward_vec": [_vp, ctypes.c_int, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp, _sz, _vp],
    "tp_conv_forward_mlp": [_vp, ctypes.c_int, _vp, _vp, _i32, ctypes.POINTER(_Mlp), _vp, _vp, _i32, _i32, _i64, _vp,
                            _vp, _sz, _vp],
    "tp_conv_forward_ex_workspace_size": [_vp, ctypes.POINTER(_FwdArgs), ctypes.POINTER(_sz)],
    "tp_conv_forward_ex": [_vp, ctypes.POINTER(_FwdArgs), _vp],
    "tp_transpose_layout": [_vp, _i32, ctypes.c_int, _vp, _vp, _i64, _i32, _vp],
    "tp_symc_create": [ctypes.c_char_p, ctypes.c_char_p, _i32, ctypes.POINTER(_vp)],
    "tp_symc_query": [_vp, ctypes.POINTER(_SymcInfo)],
    "tp_symc_term": [_vp, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32), ctypes.POINTER(_i32), _vp, _i64],
    "tp_symmetric_contraction": [_vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp],
    "tp_symc_kernel_source": [_vp, _vp, _i64, ctypes.POINTER(_i64)],
    "tp_conv_backward_workspace_size": [_vp, ctypes.c_int, _i32, _i64, ctypes.POINTER(_sz)],
    "tp_conv_backward": [_vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i64, _vp, _vp,
                         _vp, _vp, _sz, _vp],
    "tp_device_status": [ctypes.POINTER(_i32), _i32, _vp],
    "tp_set_tuning": [ctypes.POINTER(_Tuning)],
    "tp_get_tuning": [ctypes.POINTER(_Tuning)],
}
for _n, _a in _sigs.items():
    getattr(_lib, _n).argtypes = _a
    getattr(_lib, _n).restype = ctypes.c_int
_lib.tp_desc_destroy.argtypes = [_vp]
_lib.tp_desc_destroy.restype = None
_lib.tp_symc_destroy.argtypes = [_vp]
_lib.tp_symc_destroy.restype = None
_lib.tp_status_string.argtypes = [ctypes.c_int]
_lib.tp_status_string.restype = ctypes.c_char_p
_lib.tp_csr_build_noalloc_max_edges.argtypes = []
_lib.tp_csr_build_noalloc_max_edges.restype = ctypes.c_int64
_lib.tp_abi_version.argtypes = []
_lib.tp_abi_version.restype = ctypes.c_int32


def _check(status: int, what: str):
    if status != TP_OK:
        raise TPError(status, what)


class Descriptor:
    """Owns a tp_desc (host memory); fields mirror tp_desc_info."""

    def __init__(self, handle: int, irreps):
        self._h = _vp(handle)
        self.irreps_in, self.irreps_sh, self.irreps_out = irreps
        info = _Info()
        _check(_lib.tp_desc_query(self._h, ctypes.byref(info)), "tp_desc_query")
        for f, _ in _Info._fields_:
            setattr(self, f, int(getattr(info, f)))

    @property
    def handle(self):
        return self._h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.tp_desc_destroy(h)
            self._h = _vp(0)

    def __repr__(self):
        return (f"Descriptor({self.irreps_in!r} x {self.irreps_sh!r} -> {self.irreps_out!r}, "
                f"paths={self.n_paths}, weight_numel={self.weight_numel})")


class SymcDescriptor:
    """Owns a tp_symc (host memory); fields mirror tp_symc_info."""

    def __init__(self, handle: int, irreps_in: str, irreps_out: str):
        self._h = _vp(handle)
        self.irreps_in, self.irreps_out = irreps_in, irreps_out
        info = _SymcInfo()
        _check(_lib.tp_symc_query(self._h, ctypes.byref(info)), "tp_symc_query")
        for f in ("mul", "dim_in", "dim_out", "max_degree", "n_weights", "n_terms"):
            setattr(self, f, int(getattr(info, f)))
        self.num_paths = list(info.num_paths)[:self.max_degree]
        self.weights_per_degree = list(info.weights_per_degree)[:self.max_degree]

    @property
    def handle(self):
        return self._h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.tp_symc_destroy(h)
            self._h = _vp(0)


def tp_symc_create(irreps_in: str, irreps_out: str, max_degree: int) -> SymcDescriptor:
    h = _vp()
    _check(_lib.tp_symc_create(irreps_in.encode(), irreps_out.encode(), max_degree, ctypes.byref(h)), "tp_symc_create")
    return SymcDescriptor(h.value, irreps_in, irreps_out)


def tp_symc_query(symc: SymcDescriptor) -> dict:
    return {f: getattr(symc, f) for f in ("mul", "dim_in", "dim_out", "max_degree", "n_weights", "n_terms",
                                          "num_paths", "weights_per_degree")}


def tp_symc_term(symc: SymcDescriptor, t: int, D: int, out_dim: int = None):
    """(nu, output block, basis [n_q, D, .., D, 2L+1] float64) of term t; D is
    the number of input components per channel."""
    nu, c, nq = _i32(), _i32(), _i32()
    _check(_lib.tp_symc_term(symc.handle, t, ctypes.byref(nu), ctypes.byref(c), ctypes.byref(nq), None, 0),
           "tp_symc_term")
    return int(nu.value), int(c.value), int(nq.value)


def tp_symc_basis(symc: SymcDescriptor, t: int, D: int, K: int) -> np.ndarray:
    nu, c, nq = tp_symc_term(symc, t, D)
    arr = np.zeros((nq,) + (D,) * nu + (K,), dtype=np.float64)
    _check(_lib.tp_symc_term(symc.handle, t, ctypes.byref(_i32()), ctypes.byref(_i32()), ctypes.byref(_i32()),
                             arr.ctypes.data_as(_vp), arr.size), "tp_symc_term")
    return arr


def tp_symc_kernel_source(symc: SymcDescriptor) -> str:
    """The CUDA source of the kernel specialised for this descriptor."""
    n = _i64()
    _check(_lib.tp_symc_kernel_source(symc.handle, None, 0, ctypes.byref(n)), "tp_symc_kernel_source")
    buf = ctypes.create_string_buffer(n.value + 1)
    _check(_lib.tp_symc_kernel_source(symc.handle, buf, n.value + 1, ctypes.byref(n)), "tp_symc_kernel_source")
    return buf.value.decode()


def tp_symc_destroy(symc: SymcDescriptor):
    symc.__del__()


def tp_abi_version() -> int:
    return int(_lib.tp_abi_version())


def tp_status_string(status: int) -> str:
    return _lib.tp_status_string(status).decode()


def tp_desc_create(irreps_in: str, irreps_sh: str, irreps_out: str, layout: str = "ir_mul") -> Descriptor:
    lay = {"ir_mul": TP_IR_MUL, "mul_ir": TP_MUL_IR}[layout]
    h = _vp()
    _check(_lib.tp_desc_create(irreps_in.encode(), irreps_sh.encode(), irreps_out.encode(), lay, ctypes.byref(h)),
           "tp_desc_create")
    return Descriptor(h.value, (irreps_in, irreps_sh, irreps_out))


def tp_desc_create_unsimplified(irreps_in: str, irreps_sh: str, irreps_out: str) -> Descriptor:
    """Descriptor with one output block per path (grouped by output type)."""
    h = _vp()
    _check(_lib.tp_desc_create_unsimplified(irreps_in.encode(), irreps_sh.encode(), irreps_out.encode(), TP_IR_MUL,
                                            ctypes.byref(h)), "tp_desc_create_unsimplified")
    return Descriptor(h.value, (irreps_in, irreps_sh, irreps_out))


def tp_desc_query(desc: Descriptor) -> dict:
    return {f: getattr(desc, f) for f, _ in _Info._fields_}


def tp_desc_path(desc: Descriptor, p: int) -> tuple:
    info = _Path()
    _check(_lib.tp_desc_path(desc.handle, p, ctypes.byref(info)), "tp_desc_path")
    return (info.a, info.b, info.c, info.la, info.lb, info.lc)


def tp_desc_cg(desc: Descriptor, p: int) -> np.ndarray:
    a, b, c, la, lb, lc = tp_desc_path(desc, p)
    out = np.zeros((2 * la + 1, 2 * lb + 1, 2 * lc + 1), dtype=np.float64)
    _check(_lib.tp_desc_cg(desc.handle, p, out.ctypes.data_as(_vp), out.size), "tp_desc_cg")
    return out


# --- tensors -----------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t):
    return _vp(t.data_ptr()) if t is not None and t.numel() > 0 else _vp(0)


def _dev_ptr(t, name, dtype=None, ndim=None):
    """Device address of a checked tensor as an int (None for no tensor or
    an empty one); the ctypes signatures take it as void*."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream):
    s = stream if stream is not None else _torch().cuda.current_stream()
    return s.cuda_stream


def tp_spherical_harmonics(desc: Descriptor, vec, normalize: bool = True, out=None, stream=None):
    """Real harmonics of the desc's harmonic irreps for vec [E, 3] float32."""
    torch = _torch()
    E = vec.shape[0]
    if out is None:
        out = torch.empty((E, desc.dim_sh), dtype=torch.float32, device=vec.device)
    _check(_lib.tp_spherical_harmonics(desc.handle, _dev_ptr(vec, "vec", torch.float32, 2), E, int(bool(normalize)),
                                       _dev_ptr(out, "sh", torch.float32, 2), _stream(stream)),
           "tp_spherical_harmonics")
    return out


def tp_csr_workspace_size(E: int, N: int) -> int:
    n = _sz()
    _check(_lib.tp_csr_workspace_size(E, N, ctypes.byref(n)), "tp_csr_workspace_size")
    return int(n.value)


def tp_csr_build(keys, N: int, perm=None, row_ptr=None, keys_sorted=None, workspace=None, stream=None):
    """Stable counting sort of int32 keys in [0, N) -> (perm, row_ptr, keys_sorted)."""
    torch = _torch()
    E = keys.shape[0]
    dev = keys.device
    if perm is None:
        perm = torch.empty(E, dtype=torch.int32, device=dev)
    if row_ptr is None:
        row_ptr = torch.empty(N + 1, dtype=torch.int32, device=dev)
    if keys_sorted is None:
        keys_sorted = torch.empty(E, dtype=torch.int32, device=dev)
    ws_bytes = tp_csr_workspace_size(E, N)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _check(_lib.tp_csr_build(_dev_ptr(keys, "keys", torch.int32, 1), E, N, _dev_ptr(perm, "perm", torch.int32, 1),
                             _dev_ptr(row_ptr, "row_ptr", torch.int32, 1),
                             _dev_ptr(keys_sorted, "keys_sorted", torch.int32, 1),
                             _dev_ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)),
           "tp_csr_build")
    return perm, row_ptr, keys_sorted


def tp_csr_build_noalloc_max_edges() -> int:
    return int(_lib.tp_csr_build_noalloc_max_edges())


def tp_csr_build_noalloc(keys, N: int, perm, row_ptr, keys_sorted=None, stream=None):
    """tp_csr_build without any device allocation, for callers that cannot
    allocate device memory themselves (a plugin's enqueue callback handed only
    its tensors, a program whose memory belongs to another allocator): the
    caller passes every output buffer and the library uses its own fixed
    scratch array (E <= tp_csr_build_noalloc_max_edges()). Calls that overlap
    on the GPU share that array and race."""
    torch = _torch()
    E = keys.shape[0]
    _check(_lib.tp_csr_build_noalloc(_dev_ptr(keys, "keys", torch.int32, 1), E, N,
                                     _dev_ptr(perm, "perm", torch.int32, 1),
                                     _dev_ptr(row_ptr, "row_ptr", torch.int32, 1),
                                     _dev_ptr(keys_sorted, "keys_sorted", torch.int32, 1), _stream(stream)),
           "tp_csr_build_noalloc")
    return perm, row_ptr, keys_sorted


def _fwd_dtype(x, w):
    torch = _torch()
    if x.dtype != w.dtype:
        raise TypeError("x and w must have the same dtype")
    dtype = {torch.float32: TP_F32, torch.bfloat16: TP_BF16_IN_F32_OUT}.get(x.dtype)
    if dtype is None:
        raise TypeError(f"unsupported dtype {x.dtype}")
    return dtype


def tp_conv_forward_workspace_size(desc: Descriptor, dtype: int, n_dst: int, E: int) -> int:
    n = _sz()
    _check(_lib.tp_conv_forward_workspace_size(desc.handle, dtype, n_dst, E, ctypes.byref(n)),
           "tp_conv_forward_workspace_size")
    return int(n.value)


def tp_conv_forward(desc: Descriptor, x, sh, w, src, row_ptr, n_dst: int, out=None, workspace="auto", stream=None):
    """out[n_dst, dim_out] float32 for destination-sorted edges. x and w are both
    float32 (TP_F32) or both bfloat16 (TP_BF16_IN_F32_OUT). `workspace`: a
    uint8 CUDA tensor of tp_conv_forward_workspace_size bytes, "auto" to
    allocate one here, or None for the generic (workspace-free) kernel."""
    torch = _torch()
    dtype = _fwd_dtype(x, w)
    E = src.shape[0]
    if out is None:
        out = torch.empty((n_dst, desc.dim_out), dtype=torch.float32, device=x.device)
    if isinstance(workspace, str):
        nb = tp_conv_forward_workspace_size(desc, dtype, n_dst, E)
        workspace = torch.empty(nb, dtype=torch.uint8, device=x.device) if nb else None
    ws_ptr = _dev_ptr(workspace, "workspace", torch.uint8)
    ws_n = workspace.numel() if workspace is not None else 0
    _check(_lib.tp_conv_forward(desc.handle, dtype, _dev_ptr(x, "x", None, 2), _dev_ptr(sh, "sh", torch.float32, 2),
                                _dev_ptr(w, "w", None, 2), _dev_ptr(src, "src", torch.int32, 1),
                                _dev_ptr(row_ptr, "row_ptr", torch.int32, 1), x.shape[0], n_dst, E,
                                _dev_ptr(out, "out", torch.float32, 2), ws_ptr, ws_n, _stream(stream)),
           "tp_conv_forward")
    return out


def tp_conv_forward_vec(desc: Descriptor, x, vec, w, src, row_ptr, n_dst: int, normalize: bool = True, out=None,
                        workspace="auto", stream=None):
    """tp_conv_forward with the harmonics evaluated in the kernel from edge
    vectors vec [E, 3] float32 (destination-sorted edge order)."""
    torch = _torch()
    dtype = _fwd_dtype(x, w)
    E = src.shape[0]
    if out is None:
        out = torch.empty((n_dst, desc.dim_out), dtype=torch.float32, device=x.device)
    if isinstance(workspace, str):
        nb = tp_conv_forward_workspace_size(desc, dtype, n_dst, E)
        workspace = torch.empty(nb, dtype=torch.uint8, device=x.device) if nb else None
    ws_ptr = _dev_ptr(workspace, "workspace", torch.uint8)
    ws_n = workspace.numel() if workspace is not None else 0
    _check(_lib.tp_conv_forward_vec(desc.handle, dtype, _dev_ptr(x, "x", None, 2),
                                    _dev_ptr(vec, "vec", torch.float32, 2), int(bool(normalize)),
                                    _dev_ptr(w, "w", None, 2), _dev_ptr(src, "src", torch.int32, 1),
                                    _dev_ptr(row_ptr, "row_ptr", torch.int32, 1), x.shape[0], n_dst, E,
                                    _dev_ptr(out, "out", torch.float32, 2), ws_ptr, ws_n, _stream(stream)),
           "tp_conv_forward_vec")
    return out


def tp_conv_forward_mlp(desc: Descriptor, x, vec, w1, b1, w2, b2, src, row_ptr, n_dst: int, normalize: bool = True,
                        out=None, workspace="auto", stream=None):
    """tp_conv_forward_vec with the weights computed in the kernel by the radial
    network silu(|v| w1 + b1) @ w2 + b2 (w1, b1 [16]; w2 [16, weight_numel];
    b2 [weight_numel]; float32)."""
    torch = _torch()
    E = src.shape[0]
    if out is None:
        out = torch.empty((n_dst, desc.dim_out), dtype=torch.float32, device=x.device)
    if isinstance(workspace, str):
        nb = tp_conv_forward_workspace_size(desc, TP_F32, n_dst, E)
        workspace = torch.empty(nb, dtype=torch.uint8, device=x.device) if nb else None
    ws_ptr = _dev_ptr(workspace, "workspace", torch.uint8)
    ws_n = workspace.numel() if workspace is not None else 0
    f = torch.float32
    mlp = _Mlp(_dev_ptr(w1, "w1", f, 1), _dev_ptr(b1, "b1", f, 1), _dev_ptr(w2, "w2", f, 2),
               _dev_ptr(b2, "b2", f, 1), int(w1.shape[0]))
    _check(_lib.tp_conv_forward_mlp(desc.handle, TP_F32 if x.dtype == f else TP_BF16_IN_F32_OUT,
                                    _dev_ptr(x, "x", None, 2), _dev_ptr(vec, "vec", f, 2), int(bool(normalize)),
                                    ctypes.byref(mlp), _dev_ptr(src, "src", torch.int32, 1),
                                    _dev_ptr(row_ptr, "row_ptr", torch.int32, 1), x.shape[0], n_dst, E,
                                    _dev_ptr(out, "out", f, 2), ws_ptr, ws_n, _stream(stream)),
           "tp_conv_forward_mlp")
    return out


def tp_conv_forward_ex(desc: Descriptor, x, src, row_ptr, n_dst: int, w=None, sh=None, vec=None, normalize=True,
                       mlp=None, reduce: str = "sum", out=None, workspace=None, stream=None):
    """The forward with int32 or int64 indices (src, row_ptr dtype), the
    descriptor's layout for x and out (mul_ir converted on the device), and
    reduce "sum" or "mean". Harmonics as rows `sh` or from edge vectors `vec`;
    mlp = (w1, b1, w2, b2) computes the weights from the edge length (needs vec)."""
    torch = _torch()
    E = src.shape[0]
    if src.dtype != row_ptr.dtype or src.dtype not in (torch.int32, torch.int64):
        raise TypeError("src and row_ptr must both be int32 or both int64")
    f = torch.float32
    dtype = TP_F32 if x.dtype == f else TP_BF16_IN_F32_OUT
    if out is None:
        out = torch.empty((n_dst, desc.dim_out), dtype=f, device=x.device)
    keep = []
    mlp_p = None
    if mlp is not None:
        w1, b1, w2, b2 = mlp
        m = _Mlp(_dev_ptr(w1, "w1", f, 1), _dev_ptr(b1, "b1", f, 1), _dev_ptr(w2, "w2", f, 2),
                 _dev_ptr(b2, "b2", f, 1), int(w1.shape[0]))
        keep.append(m)
        mlp_p = ctypes.addressof(m)
    a = _FwdArgs(dtype, _dev_ptr(x, "x", None, 2), _dev_ptr(sh, "sh", f, 2),
                 _dev_ptr(vec, "vec", f, 2), int(bool(normalize)), mlp_p, _dev_ptr(w, "w", None, 2),
                 _dev_ptr(src, "src", None, 1), _dev_ptr(row_ptr, "row_ptr", None, 1),
                 64 if src.dtype == torch.int64 else 32, {"sum": TP_REDUCE_SUM, "mean": TP_REDUCE_MEAN}[reduce],
                 x.shape[0], n_dst, E, _dev_ptr(out, "out", f, 2), None, 0)
    n = _sz()
    _check(_lib.tp_conv_forward_ex_workspace_size(desc.handle, ctypes.byref(a), ctypes.byref(n)),
           "tp_conv_forward_ex_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(int(n.value), 1), dtype=torch.uint8, device=x.device)
    a.workspace = _dev_ptr(workspace, "workspace", torch.uint8)
    a.workspace_bytes = workspace.numel()
    _check(_lib.tp_conv_forward_ex(desc.handle, ctypes.byref(a), _stream(stream)), "tp_conv_forward_ex")
    return out


def tp_transpose_layout(desc: Descriptor, which: str, source: str, src, dst=None, stream=None):
    """Blockwise mul_ir <-> ir_mul conversion of rows of the desc's input
    (which="in") or output (which="out") irreps; `source` is src's layout."""
    torch = _torch()
    if dst is None:
        dst = torch.empty_like(src)
    lay = {"ir_mul": TP_IR_MUL, "mul_ir": TP_MUL_IR}[source]
    _check(_lib.tp_transpose_layout(desc.handle, {"in": 0, "out": 1}[which], lay, _dev_ptr(src, "src", None, 2),
                                    _dev_ptr(dst, "dst", None, 2), src.shape[0], src.element_size(), _stream(stream)),
           "tp_transpose_layout")
    return dst


def tp_conv_backward_workspace_size(desc: Descriptor, dtype: int, n_src: int, E: int) -> int:
    n = _sz()
    _check(_lib.tp_conv_backward_workspace_size(desc.handle, dtype, n_src, E, ctypes.byref(n)),
           "tp_conv_backward_workspace_size")
    return int(n.value)


def tp_conv_backward(desc: Descriptor, grad_out, x, sh, w, src, dst, row_ptr, src_perm, src_row_ptr,
                     dx=None, dw=None, dsh=None, workspace="auto", stream=None):
    """(dx, dw, dsh) float32 for destination-sorted edges; (src_perm,
    src_row_ptr) is tp_csr_build(src, n_src) in that edge order. x and w are
    both float32 or both bfloat16 (float32 math); grad_out and sh float32.
    `workspace`: a uint8 CUDA tensor of tp_conv_backward_workspace_size bytes,
    "auto" to allocate one here, or None."""
    torch = _torch()
    dtype = _fwd_dtype(x, w)
    E = src.shape[0]
    n_src, n_dst = x.shape[0], grad_out.shape[0]
    if dx is None:
        dx = torch.empty((n_src, desc.dim_x), dtype=torch.float32, device=x.device)
    if dw is None:
        dw = torch.empty((E, desc.weight_numel), dtype=torch.float32, device=x.device)
    if dsh is None:
        dsh = torch.empty((E, desc.dim_sh), dtype=torch.float32, device=x.device)
    if isinstance(workspace, str):
        nb = tp_conv_backward_workspace_size(desc, dtype, n_src, E)
        workspace = torch.empty(nb, dtype=torch.uint8, device=x.device) if nb else None
    ws_ptr = _dev_ptr(workspace, "workspace", torch.uint8)
    ws_n = workspace.numel() if workspace is not None else 0
    f = torch.float32
    _check(_lib.tp_conv_backward(desc.handle, dtype, _dev_ptr(grad_out, "grad_out", f, 2), _dev_ptr(x, "x", None, 2),
                                 _dev_ptr(sh, "sh", f, 2), _dev_ptr(w, "w", None, 2),
                                 _dev_ptr(src, "src", torch.int32, 1), _dev_ptr(dst, "dst", torch.int32, 1),
                                 _dev_ptr(row_ptr, "row_ptr", torch.int32, 1),
                                 _dev_ptr(src_perm, "src_perm", torch.int32, 1),
                                 _dev_ptr(src_row_ptr, "src_row_ptr", torch.int32, 1), n_src, n_dst, E,
                                 _dev_ptr(dx, "dx", f, 2), _dev_ptr(dw, "dw", f, 2), _dev_ptr(dsh, "dsh", f, 2),
                                 ws_ptr, ws_n, _stream(stream)),
           "tp_conv_backward")
    return dx, dw, dsh


TUNING_FIELDS = [f for f, _ in _Tuning._fields_]


def tp_set_tuning(**fields):
    """Process-wide launch tuning / test hooks (see tp_tuning in the header);
    fields not given keep the library default. With no arguments every
    default is restored."""
    bad = set(fields) - set(TUNING_FIELDS)
    if bad:
        raise TypeError(f"unknown tuning fields {sorted(bad)}")
    if not fields:
        _check(_lib.tp_set_tuning(None), "tp_set_tuning")
        return
    t = _Tuning(**{k: int(v) for k, v in fields.items()})
    _check(_lib.tp_set_tuning(ctypes.byref(t)), "tp_set_tuning")


def tp_get_tuning() -> dict:
    t = _Tuning()
    _check(_lib.tp_get_tuning(ctypes.byref(t)), "tp_get_tuning")
    return {f: int(getattr(t, f)) for f in TUNING_FIELDS}


def tp_symmetric_contraction(symc: SymcDescriptor, x, weights, element, out=None, stream=None):
    """out [N, dim_out] float32 of the symmetric contraction of x [N, dim_in]
    with weights [num_elements, n_weights, mul] selected by element [N] int32."""
    torch = _torch()
    N = x.shape[0]
    if out is None:
        out = torch.empty((N, symc.dim_out), dtype=torch.float32, device=x.device)
    f = torch.float32
    _check(_lib.tp_symmetric_contraction(symc.handle, _dev_ptr(x, "x", f, 2), _dev_ptr(weights, "weights", f, 3),
                                         _dev_ptr(element, "element", torch.int32, 1), N, weights.shape[0],
                                         _dev_ptr(out, "out", f, 2), _stream(stream)),
           "tp_symmetric_contraction")
    return out


def tp_device_status(reset: bool = True, stream=None) -> int:
    """Device status bits (TP_DEV_ERR_*); synchronises the stream."""
    v = _i32()
    _check(_lib.tp_device_status(ctypes.byref(v), int(bool(reset)), _stream(stream)), "tp_device_status")
    return int(v.value)


__all__ = ["Descriptor", "TPError", "LIB_PATH", "EXPORTS"] + EXPORTS
