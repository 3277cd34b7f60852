"""Host-side checks of the C-ABI library (no GPU needed): every symbol the
header declares is exported, the descriptor builder (Racah-formula
Clebsch-Gordan tensors, path table) agrees with the independent oracle, and
argument errors come back as status codes without touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import tp
from workloads import WORKLOADS

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tpconv.h")


def header_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"TPCONV_API\s+(?:const\s+)?\w+\s*\*?\s*(tp_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(tpc):
    names = header_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(tpc._lib, n), n
    assert set(names) == set(tpc.EXPORTS)
    assert tpc.tp_abi_version() == 1
    assert tpc.tp_status_string(4) == "index out of range"


CONFIGS = [(w.irreps_in, w.irreps_sh, w.irreps_out) for w in WORKLOADS.values()] + [
    ("32x0e+32x1o", "0e+1o", "32x0e+32x1o"),
    ("16x0+16x1+16x2", "0+1+2+3", "16x0+16x1+16x2+16x3"),
    ("8x2e+8x0e", "1o+0e", "8x1o+8x2e+8x3o"),
    ("24x1o", "0e+1o+2e", "24x0e+24x1e+24x2e"),
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "|".join(c))
def test_descriptor_matches_oracle(tpc, cfg):
    d = tpc.tp_desc_create(*cfg)
    pl = tp.Plan(*cfg)
    assert (d.n_paths, d.mul, d.dim_x, d.dim_sh, d.dim_out, d.weight_numel) == \
        (pl.n_paths, pl.mul, pl.dim_in, pl.dim_sh, pl.dim_out, pl.weight_numel)
    nnz = 0
    for p in range(d.n_paths):
        P = pl.paths[p]
        assert tpc.tp_desc_path(d, p) == (P.a, P.b, P.c, P.la, P.lb, P.lc)
        C = tpc.tp_desc_cg(d, p)
        np.testing.assert_allclose(C, pl.cg[p], atol=1e-13)
        nnz += int((pl.cg[p] != 0).sum())
    assert d.cg_nnz == nnz


@pytest.mark.parametrize("cfg,status", [
    (("32x0e+32x1q", "0e", "32x0e"), "TP_ERR_PARSE"),
    (("32x0e+", "0e", "32x0e"), "TP_ERR_PARSE"),
    (("32x0e", "0", "32x0e"), "TP_ERR_PARSE"),             # O3 vs SO3 mismatch
    (("32x4e", "0e", "32x4e"), "TP_ERR_UNSUPPORTED"),      # l > 3
    (("32x0e", "2x0e", "32x0e"), "TP_ERR_UNSUPPORTED"),    # harmonic multiplicity
    (("32x0e", "0e", "16x0e"), "TP_ERR_UNSUPPORTED"),      # uvu multiplicity
    (("12x0e", "0e", "12x0e"), "TP_ERR_UNSUPPORTED"),      # mul % 8
    (("256x0e", "0e", "256x0e"), "TP_ERR_UNSUPPORTED"),    # mul > 128
    (("32x0e", "1o", "32x0e"), "TP_ERR_UNSUPPORTED"),      # no path
    (("32x0e+32x0o", "0e", "32x0e+32x0o"), "TP_ERR_UNSUPPORTED"),  # two input blocks of one degree
    (("24x1o", "0e+1o", "24x1o+24x1e"), "TP_ERR_UNSUPPORTED"),     # two output blocks of one degree
])
def test_descriptor_errors(tpc, cfg, status):
    with pytest.raises(tpc.TPError) as ei:
        tpc.tp_desc_create(*cfg)
    assert tpc.STATUS_NAMES[ei.value.status] == status
    assert tpc.tp_desc_create("32x0e", "0e", "32x0e", layout="mul_ir").layout == tpc.TP_MUL_IR


def test_argument_errors_need_no_gpu(tpc):
    """Validation happens before any CUDA call: bogus pointers are never touched."""
    lib = tpc._lib
    d = tpc.tp_desc_create("32x0e+32x1o", "0e+1o+2e", "32x0e+32x1o+32x2e")
    vp = ctypes.c_void_p
    good, odd = vp(0x10000), vp(0x10004)
    # null out / row_ptr
    assert lib.tp_conv_forward(d.handle, 0, good, good, good, good, vp(0), 4, 4, 10, good, vp(0), 0, vp(0)) == 7
    # misaligned x
    assert lib.tp_conv_forward(d.handle, 0, odd, good, good, good, good, 4, 4, 10, good, vp(0), 0, vp(0)) == 5
    # negative sizes, bad dtype, E >= 2^31
    assert lib.tp_conv_forward(d.handle, 0, good, good, good, good, good, -1, 4, 10, good, vp(0), 0, vp(0)) == 7
    assert lib.tp_conv_forward(d.handle, 5, good, good, good, good, good, 4, 4, 10, good, vp(0), 0, vp(0)) == 7
    assert lib.tp_conv_forward(d.handle, 0, good, good, good, good, good, 4, 4, 1 << 31, good, vp(0), 0, vp(0)) == 7
    # edges but no source nodes
    assert lib.tp_conv_forward(d.handle, 0, good, good, good, good, good, 0, 4, 10, good, vp(0), 0, vp(0)) == 4
    # no destinations: nothing to do
    assert lib.tp_conv_forward(d.handle, 0, vp(0), vp(0), vp(0), vp(0), vp(0), 0, 0, 0, vp(0), vp(0), 0, vp(0)) == 0
    n = ctypes.c_size_t()
    assert lib.tp_csr_workspace_size(1000, 50, ctypes.byref(n)) == 0 and n.value >= 3 * 4000
    assert lib.tp_csr_workspace_size(-1, 50, ctypes.byref(n)) == 7
    # workspace too small / misaligned
    assert lib.tp_csr_build(good, 1000, 50, good, good, vp(0), good, 16, vp(0)) == 7
    assert lib.tp_csr_build(good, 1000, 50, good, good, vp(0), vp(0x10010), n.value, vp(0)) == 5
    assert lib.tp_csr_build(good, 10, 0, good, good, vp(0), good, n.value, vp(0)) == 4


def test_radial_network_argument_errors_need_no_gpu(tpc):
    """The radial network's checks come before any CUDA call too, so bogus
    addresses are never touched: w2 and b2 must be 16-byte aligned and w1, b1
    4-byte aligned; only float32 inputs and 16 hidden units; no null pointer."""
    lib = tpc._lib
    d = tpc.tp_desc_create("32x0e+32x1o", "0e+1o+2e", "32x0e+32x1o+32x2e")
    vp = ctypes.c_void_p
    good = vp(0x10000)

    def call(w1=0x20000, b1=0x20040, w2=0x30000, b2=0x40000, hidden=16, dtype=0):
        m = tpc._Mlp(w1, b1, w2, b2, hidden)
        st = lib.tp_conv_forward_mlp(d.handle, dtype, good, good, 1, ctypes.byref(m), good, good, 4, 4, 10, good,
                                     vp(0), 0, vp(0))
        return tpc.STATUS_NAMES[st]

    assert call(w2=0x30004) == "TP_ERR_ALIGN"
    assert call(b2=0x40008) == "TP_ERR_ALIGN"
    assert call(w1=0x20002) == "TP_ERR_ALIGN"
    assert call(hidden=8) == "TP_ERR_UNSUPPORTED"
    assert call(dtype=tpc.TP_BF16_IN_F32_OUT) == "TP_ERR_UNSUPPORTED"
    assert call(w2=0) == "TP_ERR_ARG"


def test_tuning_hooks_validate_and_reset(tpc):
    """tp_set_tuning stores in-range settings, rejects out-of-range ones with
    TP_ERR_ARG (leaving the previous settings), and NULL restores defaults."""
    assert tpc.tp_get_tuning() == {f: 0 for f in tpc.TUNING_FIELDS}
    tpc.tp_set_tuning(ring_stages=3, ring_rounds=4, wait_limit_ns=5)
    got = tpc.tp_get_tuning()
    assert (got["ring_stages"], got["ring_rounds"], got["wait_limit_ns"], got["ring_warps"]) == (3, 4, 5, 0)
    for bad in (dict(ring_stages=1), dict(ring_stages=9), dict(ring_warps=9), dict(ring_rounds=17),
                dict(ring_pack=3), dict(disable_split=2), dict(wait_limit_ns=-1), dict(ring_stage_bytes=-4),
                dict(disable_mma=2), dict(mma_stages=2), dict(mma_stages=9), dict(bwd_stage_bytes=-1),
                dict(bwd_stages=1), dict(bwd_stages=9), dict(bwd_warps=9), dict(disable_ring_bwd=2), dict(disable_symc_jit=2)):
        with pytest.raises(tpc.TPError) as ei:
            tpc.tp_set_tuning(**bad)
        assert tpc.STATUS_NAMES[ei.value.status] == "TP_ERR_ARG"
    assert tpc.tp_get_tuning()["ring_rounds"] == 4
    tpc.tp_set_tuning()
    assert tpc.tp_get_tuning() == {f: 0 for f in tpc.TUNING_FIELDS}


SYMC_CASES = [("32x0e+32x1o", "32x0e", 3), ("32x0e+32x1o+32x2e", "32x0e+32x1o", 3), ("32x0+32x1", "32x0+32x1", 2),
              ("32x1o", "32x0e+32x1o+32x2e", 3)]


@pytest.mark.parametrize("case", SYMC_CASES, ids=lambda c: "|".join(map(str, c)))
def test_symmetric_contraction_basis_matches_oracle(tpc, case):
    """The library builds its basis from symmetrised Clebsch-Gordan coupling
    trees; the oracle as a null space of the equivariance and symmetry
    constraints. Both reduce to the same canonical form."""
    from oracle import symc
    irr_in, irr_out, deg = case
    s = tpc.tp_symc_create(irr_in, irr_out, deg)
    plan = symc.SymPlan(irr_in, irr_out, range(1, deg + 1))
    assert s.n_terms == len(plan.terms) and s.n_weights == plan.n_weights
    assert s.num_paths == [plan.num_paths(n) for n in range(1, deg + 1)]
    assert (s.dim_in, s.dim_out) == (plan.dim_in, plan.dim_out)
    for t, (nu, c, B) in enumerate(plan.terms):
        assert tpc.tp_symc_term(s, t, plan.D)[:2] == (nu, c)
        got = tpc.tp_symc_basis(s, t, plan.D, B.shape[-1])
        np.testing.assert_allclose(got, B, atol=1e-12)


def test_symmetric_contraction_lesson_counts(tpc):
    import json
    g = json.load(open(os.path.join(os.path.dirname(HEADER), "..", "tests", "golden",
                                    "pages_worked_examples.json")))["symmetric_contraction_32x0e32x1o"]
    s = tpc.tp_symc_create(g["irreps_in"], g["irreps_out"], max(g["degrees"]))
    assert s.num_paths == g["num_paths"]
    assert "+".join(f"{n * s.mul}x0e" for n in s.weights_per_degree) == g["weight_irreps"]
