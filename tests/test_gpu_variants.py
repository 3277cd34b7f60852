"""GPU parity of the forward's variants (tp_conv_forward_ex, tp_transpose_layout):
reduce="mean", int64 indices, the mul_ir row layout, and their combinations
with edge vectors and the radial network, against the oracle; the blockwise
layout conversion bit-exact against the oracle's."""
import numpy as np
import pytest
import torch

from helpers import FP32_TOL, dev_tensor, err, gpu_sorted_inputs, make_problem, oracle_forward, rounded
from oracle import irreps as I
from oracle import so3, tp

pytestmark = pytest.mark.gpu

SHAPES = [
    ("32x0e+32x1o", "0e+1o+2e", "32x0e+32x1o+32x2e"),
    ("128x0e+128x1o+128x2e", "0e+1o+2e+3o", "128x0e+128x1o+128x2e"),
    ("64x0e+64x1o+64x2e+64x3o", "0e+1o+2e+3o", "64x0e+64x1o+64x2e+64x3o"),
    ("16x0+16x1+16x2", "0+1+2", "16x0+16x1+16x2"),      # no compiled program: the generic kernel
]
IDS = ["tiny", "medium", "large", "so3"]


def _mean_ref(prob, dtype=torch.float32):
    ref = oracle_forward(prob, dtype)
    deg = np.bincount(prob["dst"], minlength=prob["n_dst"])
    return ref / np.maximum(deg, 1)[:, None], deg


@pytest.mark.parametrize("irr", SHAPES, ids=IDS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_reduce_mean(tpc, irr, dtype):
    """Even destinations only (odd ones stay empty) plus one with 60 extra edges."""
    rng = np.random.default_rng(70)
    dst = np.concatenate([np.full(60, 6), rng.integers(0, 257 // 2 + 1, 4940) * 2])
    prob = make_problem(*irr, n_src=300, n_dst=257, E=len(dst), seed=71, dst=dst)
    desc = tpc.tp_desc_create(*irr)
    g = gpu_sorted_inputs(tpc, prob, dtype)
    out = tpc.tp_conv_forward_ex(desc, g["x"], g["src"], g["row_ptr"], prob["n_dst"], w=g["w"], sh=g["sh"],
                                 reduce="mean")
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    ref, deg = _mean_ref(prob, dtype)
    assert np.sum(deg == 0) > 0 and np.max(deg) > 30
    # bf16 on the large shape runs the tensor-core kernel (about 16 bits of M)
    tol = 2e-4 if (dtype == torch.bfloat16 and irr == SHAPES[2]) else FP32_TOL
    assert err(out, ref) <= tol


@pytest.mark.parametrize("irr", SHAPES, ids=IDS)
def test_int64_indices_match_int32(tpc, irr):
    prob = make_problem(*irr, n_src=211, n_dst=190, E=3001, seed=72)
    desc = tpc.tp_desc_create(*irr)
    g = gpu_sorted_inputs(tpc, prob)
    o32 = tpc.tp_conv_forward_ex(desc, g["x"], g["src"], g["row_ptr"], prob["n_dst"], w=g["w"], sh=g["sh"])
    o64 = tpc.tp_conv_forward_ex(desc, g["x"], g["src"].long(), g["row_ptr"].long(), prob["n_dst"], w=g["w"],
                                 sh=g["sh"])
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    assert torch.equal(o32, o64)
    assert err(o64, oracle_forward(prob)) <= FP32_TOL


def test_int64_index_outside_int32_is_flagged(tpc):
    prob = make_problem(*SHAPES[0], n_src=64, n_dst=64, E=1000, seed=73)
    desc = tpc.tp_desc_create(*SHAPES[0])
    g = gpu_sorted_inputs(tpc, prob)
    src = g["src"].long()
    src[10] = (1 << 40) + 3   # does not fit int32: must not alias a valid row
    out = tpc.tp_conv_forward_ex(desc, g["x"], src, g["row_ptr"].long(), 64, w=g["w"], sh=g["sh"])
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) & tpc.TP_DEV_ERR_INDEX
    keep = np.ones(1000, bool)
    keep[g["perm"].cpu().numpy()[10]] = False
    sub = dict(prob)
    sub.update(src=prob["src"][keep], dst=prob["dst"][keep], sh=prob["sh"][keep], w=prob["w"][keep])
    assert err(out, oracle_forward(sub)) <= FP32_TOL


@pytest.mark.parametrize("which", ["in", "out"])
@pytest.mark.parametrize("irr", SHAPES + [("8x2e+8x0e", "1o+0e", "8x1o+8x2e+8x3o")], ids=IDS + ["order"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_transpose_layout_bit_exact(tpc, irr, which, dtype):
    desc = tpc.tp_desc_create(*irr)
    plan = tp.Plan(*irr)
    irreps = plan.irr_in if which == "in" else plan.irr_out
    dim = plan.dim_in if which == "in" else plan.dim_out
    rows = 777
    a = np.random.default_rng(74).standard_normal((rows, dim))
    a = rounded(a, dtype)
    t = dev_tensor(a, dtype)
    mi = tpc.tp_transpose_layout(desc, which, "ir_mul", t)
    torch.cuda.synchronize()
    want = I.convert_layout(a, irreps, "ir_mul", "mul_ir")
    assert np.array_equal(mi.double().cpu().numpy(), want)
    back = tpc.tp_transpose_layout(desc, which, "mul_ir", mi)
    torch.cuda.synchronize()
    assert torch.equal(back, t)


@pytest.mark.parametrize("irr", SHAPES, ids=IDS)
def test_mul_ir_descriptor(tpc, irr):
    """x given and out returned in mul_ir (a descriptor created with layout
    mul_ir): the oracle's ir_mul result converted blockwise."""
    prob = make_problem(*irr, n_src=300, n_dst=257, E=5000, seed=75)
    plan = prob["plan"]
    desc = tpc.tp_desc_create(*irr, layout="mul_ir")
    g = gpu_sorted_inputs(tpc, prob)
    x_mi = dev_tensor(I.convert_layout(rounded(prob["x"], torch.float32), plan.irr_in, "ir_mul", "mul_ir"))
    out = tpc.tp_conv_forward_ex(desc, x_mi, g["src"], g["row_ptr"], prob["n_dst"], w=g["w"], sh=g["sh"])
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    ref = I.convert_layout(oracle_forward(prob), plan.irr_out, "ir_mul", "mul_ir")
    assert err(out, ref) <= FP32_TOL
    with pytest.raises(tpc.TPError):   # the plain entry point takes ir_mul rows only
        tpc.tp_conv_forward(desc, x_mi, g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"])


def test_all_variants_together(tpc):
    """mul_ir rows, int64 indices, mean reduction, harmonics from edge vectors
    and weights from the radial network, in one call."""
    from workloads import make_radial_mlp
    irr = SHAPES[1]
    prob = make_problem(*irr, n_src=300, n_dst=257, E=4000, seed=76)
    plan = prob["plan"]
    w1, b1, w2, b2 = make_radial_mlp(76, 0, 16, plan.weight_numel)
    v32 = rounded(prob["vec"], torch.float32)
    prob["w"] = tp.radial_mlp(v32, w1, b1, w2, b2)
    prob["sh"] = so3.sh_concat([t.l for t in plan.irr_sh], v32)
    desc = tpc.tp_desc_create(*irr, layout="mul_ir")
    g = gpu_sorted_inputs(tpc, prob)
    vec = dev_tensor(prob["vec"])[g["perm"].long()].contiguous()
    x_mi = dev_tensor(I.convert_layout(rounded(prob["x"], torch.float32), plan.irr_in, "ir_mul", "mul_ir"))
    out = tpc.tp_conv_forward_ex(desc, x_mi, g["src"].long(), g["row_ptr"].long(), prob["n_dst"], vec=vec,
                                 mlp=tuple(dev_tensor(a) for a in (w1, b1, w2, b2)), reduce="mean")
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    ref = tp.conv_forward_mean(plan, rounded(prob["x"], torch.float32), prob["sh"], prob["w"], prob["src"],
                               prob["dst"], prob["n_dst"])
    assert err(out, I.convert_layout(ref, plan.irr_out, "ir_mul", "mul_ir")) <= FP32_TOL


@pytest.mark.parametrize("irr", [("32x0e+32x1o", "0e+1o", "32x0e+32x1o")] + SHAPES, ids=["lesson"] + IDS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_unsimplified_outputs(tpc, irr, dtype):
    """One output block per path (tp_desc_create_unsimplified) against the
    oracle's per-path blocks, with empty destinations and int32 / int64 indices."""
    rng = np.random.default_rng(77)
    dst = rng.integers(0, 120, 2500) * 2
    prob = make_problem(*irr, n_src=200, n_dst=241, E=len(dst), seed=78, dst=dst)
    plan = prob["plan"]
    desc = tpc.tp_desc_create_unsimplified(*irr)
    order = tp.unsimplified_order(plan)
    assert desc.n_out == plan.n_paths and desc.dim_out == sum(plan.mul * (2 * plan.paths[p].lc + 1) for p in order)
    for pos, p in enumerate(order):
        assert tpc.tp_desc_path(desc, p)[2] == pos
    g = gpu_sorted_inputs(tpc, prob, dtype)
    out = tpc.tp_conv_forward(desc, g["x"], g["sh"], g["w"], g["src"], g["row_ptr"], prob["n_dst"])
    out64 = tpc.tp_conv_forward_ex(desc, g["x"], g["src"].long(), g["row_ptr"].long(), prob["n_dst"], w=g["w"],
                                   sh=g["sh"])
    torch.cuda.synchronize()
    assert tpc.tp_device_status(reset=True) == 0
    ref = tp.conv_forward_unsimplified(plan, rounded(prob["x"], dtype), rounded(prob["sh"], torch.float32),
                                       rounded(prob["w"], dtype), prob["src"], prob["dst"], prob["n_dst"])
    assert err(out, ref) <= FP32_TOL
    assert torch.equal(out, out64)
    with pytest.raises(tpc.TPError):   # the backward has no per-path outputs
        sp, srp, _ = tpc.tp_csr_build(g["src"], prob["n_src"])
        tpc.tp_conv_backward(desc, out, g["x"].float(), g["sh"], g["w"].float(), g["src"], g["dst"], g["row_ptr"],
                             sp, srp)
