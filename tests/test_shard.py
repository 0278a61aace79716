"""The multi-GPU partition of one problem (batch x dim over ranks), on CPU.

Every (batch, channel) row is an independent recurrence, so splitting the
rows over ranks needs no exchange. These tests pin the plan (each row in
exactly one block of exactly one rank; blocks are whole groups or inside one
group; cuts on group boundaries whenever the rows allow it, so a rank holds
only its own groups' B/C; balanced shares) and run the fp64 oracle shard by
shard on gloo ranks (world size 2 and 3): the shards, put back together, equal
the whole-problem oracle bit for bit. Not measured on GPUs: every run of this
pool has one GPU.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from state_space_model_03_gb300 import shard, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")


def _check_plan(batch, dim, groups, world):
    parts = shard.plan(batch, dim, groups, world)
    assert len(parts) == world
    dpg = dim // groups
    seen = np.zeros((batch, dim), dtype=np.int64)
    prev_end = 0
    for blocks in parts:
        for blk in blocks:
            assert 0 <= blk.b0 < blk.b1 <= batch and 0 <= blk.d0 < blk.d1 <= dim
            whole = blk.d0 % dpg == 0 and blk.d1 % dpg == 0
            inside = blk.d0 // dpg == (blk.d1 - 1) // dpg
            assert whole or inside
            if blk.b1 - blk.b0 > 1:
                assert (blk.d0, blk.d1) == (0, dim)
            start = blk.b0 * dim + blk.d0
            assert start == prev_end  # contiguous in the flattened row order
            prev_end = (blk.b1 - 1) * dim + blk.d1
            seen[blk.b0:blk.b1, blk.d0:blk.d1] += 1
    assert prev_end == batch * dim
    assert (seen == 1).all()
    return parts


@pytest.mark.parametrize("batch,dim,groups,world", [
    (8, 1536, 1, 1), (8, 1536, 1, 2), (8, 1536, 1, 8), (4, 4096, 4, 2), (4, 4096, 4, 8), (4, 4096, 4, 16),
    (2, 5120, 1, 8), (1, 2048, 1, 8), (3, 24, 3, 2), (3, 24, 3, 5), (1, 7, 7, 3), (2, 10, 5, 7),
    (5, 96, 8, 3), (1, 1, 1, 4), (0, 16, 2, 2), (6, 40, 4, 4),
])
def test_plan_covers_every_row_once(batch, dim, groups, world):
    _check_plan(batch, dim, groups, world)


@pytest.mark.parametrize("batch,dim,groups,world", [(4, 4096, 4, 2), (4, 4096, 4, 8), (4, 4096, 4, 16),
                                                    (8, 1536, 1, 8), (3, 24, 3, 3), (2, 64, 4, 8)])
def test_group_aligned_when_the_units_divide(batch, dim, groups, world):
    """batch * groups a multiple of world: every cut is a group boundary, so no
    (batch, group) B/C slab is needed by two ranks, and the shares are equal."""
    parts = _check_plan(batch, dim, groups, world)
    dpg = dim // groups
    owners = {}
    for r, blocks in enumerate(parts):
        assert sum(b.rows for b in blocks) == batch * dim // world
        for blk in blocks:
            assert blk.d0 % dpg == 0 and blk.d1 % dpg == 0
            for b in range(blk.b0, blk.b1):
                for g in range(blk.d0 // dpg, blk.d1 // dpg):
                    assert owners.setdefault((b, g), r) == r


def test_balance_within_a_group_when_units_are_few():
    """Fewer (batch, group) slabs than ranks: cuts fall inside groups and the
    shares stay within one row of equal."""
    parts = _check_plan(2, 5120, 1, 8)
    rows = [sum(b.rows for b in blocks) for blocks in parts]
    assert max(rows) - min(rows) <= 1


def test_block_operands_are_views_with_the_blocks_groups():
    w = workloads.Workload("sh_g", 2, 24, 16, 4, groups=3, bc_4d=True, dtype="bf16", seed=5)
    x = workloads.make_inputs(w)
    blk = shard.Block(1, 2, 8, 12)  # inside group 1 (8 channels per group)
    o = shard.block_operands(x, blk, 3)
    assert o["groups"] == 1 and tuple(o["B"].shape) == (1, 1, 4, 16)
    assert o["u"].data_ptr() == x["u"][1, 8].data_ptr()
    assert torch.equal(o["B"][0, 0], x["B"][1, 1])
    whole = shard.Block(0, 1, 8, 24)
    o = shard.block_operands(x, whole, 3)
    assert o["groups"] == 2 and torch.equal(o["C"][0], x["C"][0, 1:3])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = {
    "grouped": workloads.Workload("sh_grouped", 3, 24, 40, 4, groups=3, bc_4d=True, dtype="bf16",
                                  return_last_state=True, seed=21),
    "fixed": workloads.Workload("sh_fixed", 2, 10, 33, 3, bc="fixed", dtype="fp32", has_z=False,
                                bc_std=0.25, return_last_state=True, seed=22),
}


def _rank_worker(rank, world, port, case, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    from state_space_model_03_gb300 import shard as sh, workloads as wl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = CASES[case]
        x = wl.make_inputs(w)
        if x["B"].dim() == 3:
            x["B"], x["C"] = x["B"].unsqueeze(1), x["C"].unsqueeze(1)
        groups = 1 if w.bc == "fixed" else x["B"].shape[1]
        mine = []
        for blk in sh.plan(w.batch, w.dim, groups, world)[rank]:
            o = sh.block_operands(x, blk, groups)
            out, last = oracle.selective_scan_ref(**{k: o[k] for k in NAMES}, delta_softplus=w.delta_softplus,
                                                  return_last_state=True)
            mine.append((tuple(blk), out, last))
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            out = np.full((w.batch, w.dim, w.seqlen), np.nan)
            last = np.full((w.batch, w.dim, w.dstate), np.nan)
            count = np.zeros((w.batch, w.dim), dtype=np.int64)
            for part in gathered:
                for (b0, b1, d0, d1), o_, l_ in part:
                    out[b0:b1, d0:d1] = o_
                    last[b0:b1, d0:d1] = l_
                    count[b0:b1, d0:d1] += 1
            ref_out, ref_last = oracle.selective_scan_ref(**{k: x[k] for k in NAMES},
                                                          delta_softplus=w.delta_softplus, return_last_state=True)
            q.put((bool((count == 1).all()), bool(np.array_equal(out, ref_out)),
                   bool(np.array_equal(last, ref_last))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("world", [2, 3])
def test_sharded_oracle_equals_the_whole_problem_gloo(case, world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_worker, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    once, out_eq, last_eq = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert once and out_eq and last_eq
