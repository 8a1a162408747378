"""Data-parallel exchange of the delayed-scaling state across two CPU ranks
(gloo). With the amax MAX reduction before each update, every rank's state
equals that of one process that saw all ranks' rows (the oracle state machine,
updated from the amax of the union), bit for bit, NaN and Inf included."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp8_delayed_scaling_row_gb300 import dp
from oracle import fp8 as ofp8
from oracle.delayed_scaling import ScalingState

FMTS = [ofp8.E4M3, ofp8.E4M3, ofp8.E4M3, ofp8.E4M3]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rows(rank, step):
    """Rank-local values per tensor slot (one slot has a NaN on one rank at step 6, one an Inf at step 5)."""
    rng = np.random.default_rng(1000 * step + rank)
    vals = [rng.standard_normal(64).astype(np.float32) * (rank + 1) * (i + 1) for i in range(4)]
    if step == 6 and rank == 1:
        vals[2][7] = np.nan
    if step == 5 and rank == 0:
        vals[1][3] = -np.inf
    return vals


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    st = ScalingState(4, 3)
    for step in range(8):
        cur = torch.tensor([ofp8.amax(v) for v in _rows(rank, step)], dtype=torch.float32)
        dp.allreduce_amax_(cur)
        for i in range(4):
            st.record(i, cur[i].item() if not np.isnan(cur[i].item()) else np.float32(np.nan))
        st.update(FMTS)
    g = torch.full((5,), float(rank + 1))
    dp.allreduce_grads_([g, None])
    out.put((rank, st.scale.copy(), st.scale_inv.copy(), st.amax_history.copy(), g.numpy().copy()))
    dist.destroy_process_group()


def test_two_ranks_keep_the_state_of_one_process_over_all_rows():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ref = ScalingState(4, 3)
    for step in range(8):
        union = [np.concatenate([a, b]) for a, b in zip(_rows(0, step), _rows(1, step))]
        for i in range(4):
            ref.record(i, ofp8.amax(union[i]))
        ref.update(FMTS)
    for rank, scale, scale_inv, hist, g in res:
        assert np.array_equal(scale.view(np.uint32), ref.scale.view(np.uint32)), rank
        assert np.array_equal(scale_inv.view(np.uint32), ref.scale_inv.view(np.uint32)), rank
        assert np.array_equal(hist.view(np.uint32), ref.amax_history.view(np.uint32)), rank
        assert np.all(g == 3.0)  # 1 + 2
    assert np.isnan(ref.amax_history).any() and np.isinf(ref.amax_history).any()  # both reached the window


def test_single_process_is_a_no_op():
    t = torch.tensor([1.0, float("nan"), 3.0])
    before = t.clone()
    dp.allreduce_amax_(t)
    assert torch.equal(t.view(torch.int32), before.view(torch.int32))
    with pytest.raises(TypeError):
        dp.allreduce_amax_(torch.zeros(3, dtype=torch.float64))
