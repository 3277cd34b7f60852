"""Irreps strings, dimensions and block layouts (oracle; test infrastructure).

Follows Lesson 12a: Foundations of cuEquivariance, section 21.2 ("Irreps, with
the group written down": terms ``[mul x] l [e|o]``, O(3) parity letters, SO(3)
without them, dim = sum mul*(2l+1)) and section 21.3 ("Data layouts": a block
of multiplicity m and irrep dimension 2l+1 is stored either as (m, 2l+1),
``mul_ir``, or as (2l+1, m), ``ir_mul``; conversion is per block, as the
"cuEquivariance in PyTorch" page, Layouts and weights, also stresses).
"""
from __future__ import annotations

import re
from dataclasses import dataclass

import numpy as np

_TERM = re.compile(r"^(?:(\d+)\s*x\s*)?(\d+)\s*([eo]?)$")


@dataclass(frozen=True)
class MulIrrep:
    mul: int
    l: int
    p: int  # +1 even, -1 odd, 0 for SO(3) (no parity)

    @property
    def ir_dim(self) -> int:
        return 2 * self.l + 1

    @property
    def dim(self) -> int:
        return self.mul * self.ir_dim

    def ir(self):
        return (self.l, self.p)

    def __str__(self):
        par = {1: "e", -1: "o", 0: ""}[self.p]
        return f"{self.mul}x{self.l}{par}"


def parse(s: str, group: str | None = None) -> list[MulIrrep]:
    """Parse ``"32x0e + 32x1o"``. Whitespace is ignored, terms are separated by
    ``+``, the multiplicity defaults to 1. ``group`` is "O3", "SO3" or None
    (decided from the string: parity letters on every term -> O3, on none ->
    SO3)."""
    body = s.replace(" ", "").replace("\t", "")
    if body == "":
        return []
    out = []
    kinds = set()
    for term in body.split("+"):
        m = _TERM.match(term)
        if m is None:
            raise ValueError(f"cannot parse irreps term {term!r} in {s!r}")
        mul = int(m.group(1)) if m.group(1) is not None else 1
        l = int(m.group(2))
        par = m.group(3)
        kinds.add(bool(par))
        p = {"e": 1, "o": -1, "": 0}[par]
        out.append(MulIrrep(mul, l, p))
    if len(kinds) > 1:
        raise ValueError(f"mixed O3/SO3 terms in {s!r}")
    is_o3 = kinds == {True}
    if group is not None:
        if group == "O3" and not is_o3:
            raise ValueError(f"O3 irreps need parity letters: {s!r}")
        if group == "SO3" and is_o3:
            raise ValueError(f"SO3 irreps take no parity letters: {s!r}")
    return out


def dim(irreps: list[MulIrrep]) -> int:
    return sum(t.dim for t in irreps)


def offsets(irreps: list[MulIrrep]) -> list[int]:
    off, acc = [], 0
    for t in irreps:
        off.append(acc)
        acc += t.dim
    return off


def to_string(irreps: list[MulIrrep]) -> str:
    return "+".join(str(t) for t in irreps)


def block_shape(t: MulIrrep, layout: str) -> tuple[int, int]:
    """Shape of one block in the given layout (section 21.3)."""
    if layout == "mul_ir":
        return (t.mul, t.ir_dim)
    if layout == "ir_mul":
        return (t.ir_dim, t.mul)
    raise ValueError(layout)


def convert_layout(x: np.ndarray, irreps: list[MulIrrep], source: str, target: str) -> np.ndarray:
    """Blockwise transpose between ``mul_ir`` and ``ir_mul`` over the last axis."""
    if source == target:
        return x.copy()
    out = np.empty_like(x)
    for t, o in zip(irreps, offsets(irreps)):
        blk = x[..., o:o + t.dim].reshape(x.shape[:-1] + block_shape(t, source))
        out[..., o:o + t.dim] = np.swapaxes(blk, -1, -2).reshape(x.shape[:-1] + (t.dim,))
    return out
