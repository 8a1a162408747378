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


# ---- the LayerNormMLP step itself, rows split over two ranks
MLP_M, MLP_D, MLP_F, MLP_STEPS = 48, 32, 64, 4


def _mlp_inputs(step):
    from fp8_delayed_scaling_row_gb300 import synth
    x = synth.activations(2 * MLP_M, MLP_D, dist="outliers", step=step)
    dy = synth.grad(2 * MLP_M, MLP_D, step=step)
    return x, dy


def _mlp_step(x, dy, p, fs, bs, rec, exchange):
    """One oracle LayerNormMLP forward + backward with the states' updates after
    `exchange` (the data-parallel hook) has combined the recorded amaxes."""
    from oracle import modules as omod
    _, ctx, _ = omod.ln_mlp_fwd(x, p["gamma"], p["beta"], p["w1"], p["b1"], p["w2"], p["b2"], fs, rec, update=False)
    g = omod.ln_mlp_bwd(dy, ctx, bs, rec, update=False)
    exchange(fs, bs, g)
    fs.update([rec.fwd_fmt()] * 4)
    bs.update([rec.bwd_fmt()] * 2)
    return g


def _mlp_worker(rank, world, port, out):
    from fp8_delayed_scaling_row_gb300 import synth
    from oracle.delayed_scaling import Recipe
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rec = Recipe("hybrid", 3)
    p = synth.mlp_params(MLP_D, MLP_F, bias_std=0.02)
    fs, bs = ScalingState(4, 3), ScalingState(2, 3)

    def exchange(fs, bs, g):
        for st in (fs, bs):
            cur = torch.from_numpy(st.amax_cur.copy())
            dp.allreduce_amax_(cur)
            st.amax_cur[:] = cur.numpy()
        ts = [torch.from_numpy(np.ascontiguousarray(g[k], dtype=np.float64)) for k in ("dw1", "dw2", "dgamma", "dbeta")]
        dp.allreduce_grads_(ts)
        for k, t in zip(("dw1", "dw2", "dgamma", "dbeta"), ts):
            g[k] = t.numpy()

    grads = []
    for step in range(MLP_STEPS):
        x, dy = _mlp_inputs(step)
        rows = slice(rank * MLP_M, (rank + 1) * MLP_M)
        g = _mlp_step(x[rows], dy[rows], p, fs, bs, rec, exchange)
        grads.append({k: g[k] for k in ("dw1", "dw2", "dgamma", "dbeta")})
    out.put((rank, fs.copy(), bs.copy(), grads))
    dist.destroy_process_group()


def test_two_ranks_of_a_layernorm_mlp_keep_one_process_state():
    """Each rank runs the oracle LayerNormMLP on half of the rows. Every amax of
    the step is a maximum over rows, so with the MAX exchange each rank's forward
    and backward states equal, bit for bit, those of one process over all rows;
    the summed weight and LayerNorm gradients equal that process's gradients up
    to the bf16 rounding of each half (1e-2 relative Frobenius, the parity bound)."""
    from fp8_delayed_scaling_row_gb300 import synth
    from oracle.delayed_scaling import Recipe
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_mlp_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    rec = Recipe("hybrid", 3)
    p = synth.mlp_params(MLP_D, MLP_F, bias_std=0.02)
    fs, bs = ScalingState(4, 3), ScalingState(2, 3)
    ref = []
    for step in range(MLP_STEPS):
        x, dy = _mlp_inputs(step)
        g = _mlp_step(x, dy, p, fs, bs, rec, lambda *a: None)
        ref.append(g)
    assert (fs.scale != 1).all() and (bs.scale != 1).all()  # the scales moved
    for rank, rfs, rbs, grads in res:
        for a, b in ((rfs, fs), (rbs, bs)):
            for name in ("scale", "scale_inv", "amax_history"):
                assert np.array_equal(getattr(a, name).view(np.uint32), getattr(b, name).view(np.uint32)), (rank, name)
        for step in range(MLP_STEPS):
            for k in ("dw1", "dw2", "dgamma", "dbeta"):
                got, want = grads[step][k], np.asarray(ref[step][k], np.float64)
                assert np.linalg.norm(got - want) <= 1e-2 * np.linalg.norm(want), (rank, step, k)
