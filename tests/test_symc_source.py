"""The kernel tp_symmetric_contraction specialises for each descriptor: its
generated source compiles with NVRTC for sm_103a (no GPU needed), and it holds
one fused multiply-add per distinct monomial of each (row, weight) group,
which is the oracle's basis with index orderings merged."""
import ctypes
import ctypes.util

import numpy as np
import pytest

from oracle import symc

CASES = [("32x0e+32x1o", "32x0e", 3), ("32x0e+32x1o+32x2e", "32x0e+32x1o", 3), ("64x0+64x1", "64x0+64x1", 2),
         ("32x1o", "32x0e+32x1o+32x2e", 3), ("96x0e+96x1o", "96x0e+96x1o", 1)]


def nvrtc():
    for name in ("libnvrtc.so.13", "libnvrtc.so", ctypes.util.find_library("nvrtc")):
        if not name:
            continue
        try:
            return ctypes.CDLL(name)
        except OSError:
            pass
    pytest.skip("NVRTC is not installed")


@pytest.mark.parametrize("case", CASES, ids=lambda c: "|".join(map(str, c)))
def test_generated_kernel_compiles_for_sm103a(tpc, case):
    lib = nvrtc()
    s = tpc.tp_symc_create(*case)
    src = tpc.tp_symc_kernel_source(s).encode()
    prog = ctypes.c_void_p()
    assert lib.nvrtcCreateProgram(ctypes.byref(prog), src, b"symc_jit.cu", 0, None, None) == 0
    opts = (ctypes.c_char_p * 3)(b"--gpu-architecture=sm_103a", b"--std=c++17", b"-default-device")
    rc = lib.nvrtcCompileProgram(prog, 3, opts)
    n = ctypes.c_size_t()
    lib.nvrtcGetProgramLogSize(prog, ctypes.byref(n))
    log = ctypes.create_string_buffer(n.value + 1)
    lib.nvrtcGetProgramLog(prog, log)
    size = ctypes.c_size_t()
    ok = rc == 0 and lib.nvrtcGetCUBINSize(prog, ctypes.byref(size)) == 0 and size.value > 0
    lib.nvrtcDestroyProgram(ctypes.byref(prog))
    assert ok, log.value.decode()


def test_generated_terms_match_the_basis(tpc):
    """Count the FMAs of each (row, weight) group in the source against the
    oracle's basis: the number of distinct sorted index tuples with a nonzero
    summed coefficient."""
    import re
    irr_in, irr_out, deg = CASES[1]
    s = tpc.tp_symc_create(irr_in, irr_out, deg)
    src = tpc.tp_symc_kernel_source(s)
    plan = symc.SymPlan(irr_in, irr_out, range(1, deg + 1))
    expect = 0
    for (nu, c, B) in plan.terms:
        for q in range(B.shape[0]):
            merged = {}
            for idx in zip(*np.nonzero(np.abs(B[q]) > 1e-12)):
                key = (tuple(sorted(idx[:nu])), idx[nu])
                merged[key] = merged.get(key, 0.0) + B[q][idx]
            expect += sum(1 for v in merged.values() if abs(v) > 1e-9)
    got = len(re.findall(r"= 0x[0-9a-fp.+-]+f \* |= fmaf\(-?0x|= -0x[0-9a-fp.+-]+f \* |const float u\d+ = -?0x", src))
    assert got == expect
