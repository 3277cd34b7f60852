"""GPU parity: the CSR builder (bit-exact against the oracle's stable
counting sort) and the spherical-harmonics kernel (against the oracle's
Legendre-based harmonics)."""
import numpy as np
import pytest
import torch

from helpers import dev_tensor
from oracle import so3, tp

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E,N,kind", [
    (0, 5, "uniform"), (1, 1, "uniform"), (100, 1, "uniform"), (5000, 37, "uniform"),
    (2047, 3000, "uniform"), (2049, 3000, "uniform"), (70001, 70000, "uniform"),
    (300000, 262144, "uniform"), (50000, 257, "skewed"), (40000, 1 << 16, "sorted"),
    (33000, 1 << 12, "reversed"),
])
def test_csr_bit_exact(tpc, E, N, kind):
    rng = np.random.default_rng(E + N)
    if kind == "uniform":
        keys = rng.integers(0, N, E)
    elif kind == "skewed":   # one heavy key plus a tail
        keys = np.where(rng.random(E) < 0.5, 7, rng.integers(0, N, E))
    elif kind == "sorted":
        keys = np.sort(rng.integers(0, N, E))
    else:
        keys = np.sort(rng.integers(0, N, E))[::-1].copy()
    perm, row_ptr, ks = tpc.tp_csr_build(dev_tensor(keys, torch.int32), N)
    rp, rr, rk = tp.csr_build(keys, N)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(row_ptr.cpu().numpy(), rr)
    assert np.array_equal(ks.cpu().numpy(), rk)
    assert tpc.tp_device_status(reset=True) == 0


def test_csr_out_of_range_keys_set_status(tpc):
    keys = np.array([0, 3, 9, 1, -2, 2], dtype=np.int32)   # 9 and -2 outside [0, 4)
    perm, row_ptr, ks = tpc.tp_csr_build(dev_tensor(keys, torch.int32), 4)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    # outputs stay inside their arrays; perm is still a permutation
    assert sorted(perm.cpu().numpy().tolist()) == list(range(6))
    assert tpc.tp_device_status(reset=True) == 0


@pytest.mark.parametrize("ls", [[0, 1, 2], [0, 1, 2, 3], [2, 0, 3], [1]])
@pytest.mark.parametrize("normalize", [True, False])
def test_spherical_harmonics(tpc, ls, normalize):
    par = lambda l: "e" if l % 2 == 0 else "o"
    irr = "+".join(f"{l}{par(l)}" for l in ls)
    # any descriptor with these harmonics will do: l0 x l0 always reaches 0e
    desc = tpc.tp_desc_create(f"8x{ls[0]}{par(ls[0])}", irr, "8x0e")
    rng = np.random.default_rng(3)
    vec = rng.standard_normal((5000, 3)) * rng.uniform(0.2, 3.0, (5000, 1))
    vec[0] = [0.0, 0.0, 2.0]
    vec[1] = [1e-3, -2e-3, 0.0]
    got = tpc.tp_spherical_harmonics(desc, dev_tensor(vec), normalize=normalize).cpu().double().numpy()
    v32 = vec.astype(np.float32).astype(np.float64)
    ref = so3.sh_concat(ls, v32, normalize=normalize)
    scale = np.maximum(1.0, np.abs(ref))
    assert np.max(np.abs(got - ref) / scale) < 2e-5
