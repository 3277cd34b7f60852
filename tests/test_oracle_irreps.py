"""Oracle pins: irreps parsing and block layouts against the values the pages
print (tests/golden/pages_worked_examples.json)."""
import json
import os

import numpy as np
import pytest

from oracle import irreps as I

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


@pytest.mark.parametrize("case", GOLD["irreps_dims"], ids=lambda c: c["irreps"])
def test_dims_printed_on_pages(case):
    irr = I.parse(case["irreps"], case.get("group"))
    assert I.dim(irr) == case["dim"]


def test_parse_details():
    irr = I.parse(" 32x0e +32x1o+ 2e ")
    assert [(t.mul, t.l, t.p) for t in irr] == [(32, 0, 1), (32, 1, -1), (1, 2, 1)]
    assert I.to_string(irr) == "32x0e+32x1o+1x2e"
    assert [t.p for t in I.parse("0+1+2")] == [0, 0, 0]
    with pytest.raises(ValueError):
        I.parse("32x0e+32x1")          # mixed O3 / SO3
    with pytest.raises(ValueError):
        I.parse("32x0q")
    with pytest.raises(ValueError):
        I.parse("32x0e", group="SO3")
    assert I.offsets(I.parse("32x0e+32x1o+32x2e")) == [0, 32, 128]


def test_layout_worked_example():
    g = GOLD["layout_arange6_2x1o"]
    irr = I.parse("2x1o")
    x = np.arange(6.0)
    assert list(I.block_shape(irr[0], "mul_ir")) == g["mul_ir_shape"]
    assert list(I.block_shape(irr[0], "ir_mul")) == g["ir_mul_shape"]
    assert x.reshape(I.block_shape(irr[0], "mul_ir")).tolist() == g["mul_ir"]
    x_ir = I.convert_layout(x, irr, "mul_ir", "ir_mul")
    assert x_ir.reshape(I.block_shape(irr[0], "ir_mul")).tolist() == g["ir_mul"]


def test_layout_round_trip_is_blockwise():
    irr = I.parse("3x0e+2x1o+4x2e")
    x = np.random.default_rng(0).standard_normal((5, I.dim(irr)))
    y = I.convert_layout(x, irr, "mul_ir", "ir_mul")
    assert np.array_equal(I.convert_layout(y, irr, "ir_mul", "mul_ir"), x)
    # blockwise, not a transpose of the whole flattened row
    assert not np.array_equal(y, x.reshape(5, -1))
    # scalars (l=0) are unchanged by the conversion
    assert np.array_equal(y[:, :3], x[:, :3])
    # 2x1o block: (mul, 3) -> (3, mul)
    assert np.array_equal(y[:, 3:9].reshape(5, 3, 2), np.swapaxes(x[:, 3:9].reshape(5, 2, 3), 1, 2))
