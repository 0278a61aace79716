"""Partition of one selective-scan problem over ranks (one GPU per rank).

Every (batch, channel) row of the selective scan (page "PaddleNLP Kernel
算子库：CUDA 与 Triton 双实现的高性能 NLP GPU 算子实战指南", section 4.1) is an
independent recurrence, so the problem shards over batch x dim with no
exchange at all. The plan flattens the rows as r = b * dim + d, cuts the range
into `world` contiguous parts of nearly equal size, and moves each cut to a
group boundary (a multiple of dim / groups) whenever one lies within a
tolerance of the ideal cut, so that a rank needs only the B/C of the groups it
owns. Each part is returned as rectangular blocks (b0, b1, d0, d1), each
either whole groups or the channels of a single group, so a block is itself a
well-formed problem: its channels, A/D/delta_bias rows and B/C groups are
plain slices, and a kernel run on the block maps its channels to groups as
the whole problem does.

This module holds the host-side plan and the slicing of operands; the
arithmetic on each block is the library's (or, in the tests, the oracle's).
"""
from __future__ import annotations

from typing import List, NamedTuple


class Block(NamedTuple):
    b0: int
    b1: int
    d0: int
    d1: int

    @property
    def rows(self) -> int:
        return (self.b1 - self.b0) * (self.d1 - self.d0)


def _cuts(total: int, world: int, unit: int, tol: float) -> List[int]:
    """world + 1 nondecreasing cut points over [0, total]; interior cuts sit on
    a multiple of `unit` when one lies within tol * total / world of the ideal
    cut, else on the ideal cut itself."""
    cuts = [0]
    share = total / world
    for k in range(1, world):
        ideal = k * share
        snapped = round(ideal / unit) * unit
        c = snapped if abs(snapped - ideal) <= tol * share else int(round(ideal))
        cuts.append(min(max(c, cuts[-1]), total))
    cuts.append(total)
    return cuts


def _blocks(r0: int, r1: int, dim: int, dpg: int) -> List[Block]:
    """Rows [r0, r1) of the flattened (batch, dim) range as blocks that are
    whole groups or lie inside one group."""
    out: List[Block] = []
    r = r0
    while r < r1:
        b, d = divmod(r, dim)
        if d == 0 and r1 - r >= dim:  # whole batch rows
            nb = (r1 - r) // dim
            out.append(Block(b, b + nb, 0, dim))
            r += nb * dim
            continue
        end = min(r1, (b + 1) * dim)          # stay within this batch row
        d_end = end - b * dim
        if d % dpg == 0 and d_end - d >= dpg:  # whole groups
            d_end = d + (d_end - d) // dpg * dpg
        else:                                  # inside one group
            d_end = min(d_end, (d // dpg + 1) * dpg)
        out.append(Block(b, b + 1, d, d_end))
        r = b * dim + d_end
    return out


def plan(batch: int, dim: int, groups: int, world: int, tol: float = 0.25) -> List[List[Block]]:
    """Blocks of each rank: a list of `world` lists. Every (b, d) row is in
    exactly one block of exactly one rank; a rank's blocks are contiguous in
    the flattened row order. groups = 1 for fixed or one-group B/C."""
    if world < 1 or batch < 0 or dim < 0 or groups < 1 or (dim and dim % groups):
        raise ValueError("need world >= 1, batch, dim >= 0 and dim divisible by groups")
    total = batch * dim
    dpg = dim // groups if dim else 1
    cuts = _cuts(total, world, dpg, tol)
    return [_blocks(cuts[k], cuts[k + 1], dim, dpg) for k in range(world)]


def block_operands(x: dict, blk: Block, groups: int) -> dict:
    """The operands of one block, as slices (views) of the whole problem's:
    u, delta, z (batch, dim, seqlen); A (dim, dstate); D, delta_bias (dim,);
    B, C fixed (dim, dstate) or variable (batch, groups, dstate, seqlen), the
    latter cut to the block's groups. Returns a dict with the same keys and
    'groups' (the block's group count)."""
    dim = x["u"].shape[1]
    dpg = dim // groups
    g0, g1 = blk.d0 // dpg, (blk.d1 - 1) // dpg + 1
    out = {}
    for k in ("u", "delta", "z"):
        t = x.get(k)
        out[k] = None if t is None else t[blk.b0:blk.b1, blk.d0:blk.d1]
    out["A"] = x["A"][blk.d0:blk.d1]
    for k in ("D", "delta_bias"):
        t = x.get(k)
        out[k] = None if t is None else t[blk.d0:blk.d1]
    for k in ("B", "C"):
        t = x[k]
        if t.dim() == 2:                       # fixed (dim, dstate)
            out[k] = t[blk.d0:blk.d1]
        else:                                  # (batch, groups, dstate, seqlen)
            out[k] = t[blk.b0:blk.b1, g0:g1]
    out["groups"] = g1 - g0
    return out
