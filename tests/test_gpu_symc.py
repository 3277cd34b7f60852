"""GPU parity of tp_symmetric_contraction against the oracle (oracle/symc.py):
several irreps, degrees 1..3, several elements per batch, ragged node counts,
and an element index out of range; both the kernel compiled for each
descriptor (the default) and the table kernel."""
import numpy as np
import pytest
import torch

from helpers import FP32_TOL, dev_tensor, err, tuning
from oracle import symc

pytestmark = pytest.mark.gpu

CASES = [("32x0e+32x1o", "32x0e", 3), ("32x0e+32x1o+32x2e", "32x0e+32x1o", 3), ("64x0+64x1", "64x0+64x1", 2),
         ("32x1o", "32x0e+32x1o+32x2e", 3), ("96x0e+96x1o", "96x0e+96x1o", 1)]


PATHS = {"specialised": {}, "table": {"disable_symc_jit": 1}}


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("case", CASES, ids=lambda c: "|".join(map(str, c)))
@pytest.mark.parametrize("N", [1, 37, 3001])
def test_symmetric_contraction_matches_oracle(tpc, case, N, path):
    irr_in, irr_out, deg = case
    plan = symc.SymPlan(irr_in, irr_out, range(1, deg + 1))
    s = tpc.tp_symc_create(irr_in, irr_out, deg)
    rng = np.random.default_rng(N + deg)
    x = rng.standard_normal((N, plan.dim_in)).astype(np.float32)
    n_el = 5
    w = rng.standard_normal((n_el, plan.n_weights, plan.mul)).astype(np.float32)
    el = rng.integers(0, n_el, N).astype(np.int32)
    with tuning(tpc, **PATHS[path]):
        out = tpc.tp_symmetric_contraction(s, dev_tensor(x), dev_tensor(w), dev_tensor(el, torch.int32))
        torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    ref = symc.symmetric_contraction(plan, x.astype(np.float64), w.astype(np.float64), el)
    assert err(out, ref) <= FP32_TOL


def test_specialised_kernel_runs(tpc):
    """The default call runs the kernel compiled for the descriptor: its sums
    are in another order than the table kernel's, so on a degree-3 case the two
    results are close but not bitwise equal."""
    case = CASES[1]
    s = tpc.tp_symc_create(*case)
    plan = symc.SymPlan(case[0], case[1], range(1, case[2] + 1))
    rng = np.random.default_rng(9)
    x = dev_tensor(rng.standard_normal((4000, plan.dim_in)))
    w = dev_tensor(rng.standard_normal((3, plan.n_weights, plan.mul)))
    el = dev_tensor(rng.integers(0, 3, 4000), torch.int32)
    a = tpc.tp_symmetric_contraction(s, x, w, el)
    with tuning(tpc, disable_symc_jit=1):
        b = tpc.tp_symmetric_contraction(s, x, w, el)
    torch.cuda.synchronize()
    assert not torch.equal(a, b)
    assert torch.allclose(a, b, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("path", sorted(PATHS))
def test_symmetric_contraction_bad_element(tpc, path):
    plan = symc.SymPlan("32x0e+32x1o", "32x0e", [1, 2, 3])
    s = tpc.tp_symc_create("32x0e+32x1o", "32x0e", 3)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((50, plan.dim_in)).astype(np.float32)
    w = rng.standard_normal((2, plan.n_weights, plan.mul)).astype(np.float32)
    el = rng.integers(0, 2, 50).astype(np.int32)
    el[7] = 2
    with tuning(tpc, **PATHS[path]):
        out = tpc.tp_symmetric_contraction(s, dev_tensor(x), dev_tensor(w), dev_tensor(el, torch.int32))
        torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    assert not out[7].any()
    keep = np.arange(50) != 7
    ref = symc.symmetric_contraction(plan, x[keep].astype(np.float64), w.astype(np.float64), el[keep])
    assert err(out[torch.as_tensor(keep, device="cuda")], ref) <= FP32_TOL


def test_symmetric_contraction_no_nodes(tpc):
    s = tpc.tp_symc_create("32x0e+32x1o", "32x0e", 3)
    x = torch.zeros((0, s.dim_in), device="cuda")
    w = torch.zeros((2, s.n_weights, s.mul), device="cuda")
    el = torch.zeros((0,), dtype=torch.int32, device="cuda")
    out = tpc.tp_symmetric_contraction(s, x, w, el)
    torch.cuda.synchronize()
    assert out.shape == (0, s.dim_out)
    assert tpc.tp_device_status(reset=True) == 0
