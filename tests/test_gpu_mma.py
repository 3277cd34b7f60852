"""GPU parity of the tensor-core forward (tcgen05), which tp_conv_forward uses
for bfloat16 inputs of the 64x0e+64x1o+64x2e+64x3o shape with harmonics
0e+1o+2e+3o (23 paths): the per-edge matrices M (fp32 from the harmonics) enter
the MMA as a pair of bfloat16 matrices hi + lo (about 16 bits of M), every
product and sum is fp32. Checked against
the fp64 oracle at the bf16 tolerance, and - with the tensor-core kernel
disabled - the same calls on the fp32 CUDA-core kernel at the fp32 tolerance,
across edge counts with ragged tails, a 1000-edge destination cut across many
pieces, empty destinations, more sources than destinations, every stage count,
out-of-range sources, bitwise determinism and a pipeline wait that gives up."""
import numpy as np
import pytest
import torch

from helpers import BF16_TOL, FP32_TOL, deg_tol, dev_tensor, err, gpu_sorted_inputs, make_problem, oracle_forward, tuning

pytestmark = pytest.mark.gpu

IRR = ("64x0e+64x1o+64x2e+64x3o", "0e+1o+2e+3o", "64x0e+64x1o+64x2e+64x3o")
# measured max |gpu - oracle| / RMS of this kernel: about 1e-5 on dense
# problems, up to 4e-5 on rows of a few edges (the hi + lo split of M keeps
# about 16 bits); held to this bound, 100x inside BF16_TOL
MMA_TOL = 2e-4


def run(tpc, prob, workspace="auto"):
    desc = tpc.tp_desc_create(*prob["irreps"])
    g = gpu_sorted_inputs(tpc, prob, torch.bfloat16)
    out = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"],
                              workspace=workspace)
    torch.cuda.synchronize()
    return out, desc, g


def row_errors(out, ref):
    """max |gpu - oracle| / RMS of each row that has edges, against that row's own RMS."""
    on = out.double().cpu().numpy()
    rows = np.flatnonzero(np.any(ref != 0, axis=1))
    return np.array([err(on[r], ref[r]) for r in rows])


@pytest.mark.parametrize("E", [1, 2, 3, 255, 256, 257, 5003, 40000])
def test_mma_matches_oracle(tpc, E):
    prob = make_problem(*IRR, n_src=300, n_dst=257, E=E, seed=70 + E)
    ref = oracle_forward(prob, torch.bfloat16)
    out, _, _ = run(tpc, prob)
    assert tpc.tp_device_status(reset=True) == 0
    re = row_errors(out, ref)
    whole = err(out, ref)
    print(f"E={E}: whole-tensor {whole:.3e}, per-row max {re.max():.3e} median {np.median(re):.3e}")
    assert re.max() <= MMA_TOL
    if E >= 5000:   # every destination has edges: the whole-tensor measure applies as well
        assert whole <= MMA_TOL
    assert whole <= BF16_TOL
    with tuning(tpc, disable_mma=1):   # the fp32 CUDA-core kernel on the same inputs
        out32, _, _ = run(tpc, prob)
    assert row_errors(out32, ref).max() <= FP32_TOL
    if E >= 5000:
        assert err(out32, ref) <= FP32_TOL
    if E >= 256:   # the tensor-core kernel ran: its bf16 M makes the sums differ in the last bits
        assert not torch.equal(out, out32)


@pytest.mark.parametrize("stages", [3, 4, 6, 8])
def test_mma_stage_counts_and_heavy_rows(tpc, stages):
    """A 1000-edge destination (cut across many pieces), empty destinations,
    more sources than destinations, a ragged tail, 3..8 shared-memory stages
    (8 stages leave room for one CTA per SM instead of two)."""
    rng = np.random.default_rng(80)
    n_dst = 600
    dst = np.concatenate([np.full(1000, 7), rng.integers(0, n_dst // 2, 20003) * 2, [n_dst - 1]])
    rng.shuffle(dst)
    prob = make_problem(*IRR, n_src=900, n_dst=n_dst, E=len(dst), seed=81, dst=dst)
    ref = oracle_forward(prob, torch.bfloat16)
    with tuning(tpc, mma_stages=stages):
        out, _, _ = run(tpc, prob)
    assert tpc.tp_device_status(reset=True) == 0
    assert err(out, ref) <= MMA_TOL
    on = out.double().cpu().numpy()
    for d, c in zip(*np.unique(dst, return_counts=True)):
        assert err(on[d], ref[d]) <= MMA_TOL * max(1.0, (c / 64.0) ** 0.5), d
    empty = np.setdiff1d(np.arange(n_dst), dst)
    assert len(empty) > 100 and not out[torch.as_tensor(empty)].any()


def test_mma_deterministic(tpc):
    prob = make_problem(*IRR, n_src=500, n_dst=480, E=30000, seed=90)
    desc = tpc.tp_desc_create(*IRR)
    g = gpu_sorted_inputs(tpc, prob, torch.bfloat16)
    a = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"])
    b = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_mma_out_of_range_source(tpc):
    prob = make_problem(*IRR, n_src=64, n_dst=64, E=3000, seed=91)
    desc = tpc.tp_desc_create(*IRR)
    g = gpu_sorted_inputs(tpc, prob, torch.bfloat16)
    bad = g["src"].clone()
    bad[17] = 64
    bad[2000] = -5
    out = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], bad, g["row_ptr"], 64)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    keep = np.ones(3000, bool)
    perm = g["perm"].cpu().numpy()
    keep[perm[[17, 2000]]] = False
    sub = dict(prob)
    sub.update(src=prob["src"][keep], dst=prob["dst"][keep], sh=prob["sh"][keep], w=prob["w"][keep])
    assert err(out, oracle_forward(sub, torch.bfloat16)) <= MMA_TOL
    assert tpc.tp_device_status(reset=True) == 0


def test_mma_wait_timeout(tpc):
    """A 1 ns main-loop wait limit: waits give up, TP_DEV_ERR_TIMEOUT is
    reported, every copy and MMA in flight still completes before the CTA
    exits, nothing outside `out` is written, and the next call is correct."""
    prob = make_problem(*IRR, n_src=4000, n_dst=4000, E=60000, seed=92)
    desc = tpc.tp_desc_create(*IRR)
    g = gpu_sorted_inputs(tpc, prob, torch.bfloat16)
    n = prob["n_dst"]
    guard = 61
    big = torch.full((n + 2 * guard, desc.dim_out), 12345.0, device="cuda")
    out = big[guard:guard + n]
    hit = False
    for _ in range(3):
        with tuning(tpc, wait_limit_ns=1):
            tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], n, out=out)
            torch.cuda.synchronize()
        st = tpc.tp_device_status(reset=True)
        assert st & ~tpc.TP_DEV_ERR_TIMEOUT == 0
        assert torch.all(big[:guard] == 12345.0) and torch.all(big[guard + n:] == 12345.0)
        hit = hit or bool(st & tpc.TP_DEV_ERR_TIMEOUT)
        if hit:
            break
    assert hit
    again = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], n)
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    assert err(again, oracle_forward(prob, torch.bfloat16)) <= MMA_TOL
