"""The data-parallel exchange of dp.py on the library's own device state (GPU).

Two gloo ranks share the one GPU as two processes. Each runs the library's
LayerNormMLP forward and backward on its half of the tokens, with the state
updates deferred. Between a module call and its update, the rank copies its
device amax_cur to the host, reduces it with dp.allreduce_amax_ (MAX over the
ranks), and copies it back. The gradients are summed the same way with
dp.allreduce_grads_. Only host copies cross the ranks, and neither process's
kernels wait on the other's.

Every amax of the step is a maximum over rows, so after the exchange each rank's
forward and backward states must equal, bit for bit, those of one process that
runs all tokens with the updates inside the module calls (the backward's update
rides in the LayerNorm backward launch). The summed weight and LayerNorm
gradients must equal that process's gradients within the 1e-2 relative
Frobenius parity bound, since each half is rounded to bf16 before the sum.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp8_delayed_scaling_row_gb300 import dp, synth
from helpers import bf16_dev

pytestmark = pytest.mark.gpu

M, D, F, HIST, STEPS, SEED = 1024, 256, 768, 4, 4, 23
GRADS = ("dw1", "dw2", "db1", "db2", "dgamma", "dbeta")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _exchange(meta):
    cur = meta.amax_cur.cpu()
    dp.allreduce_amax_(cur)
    meta.amax_cur.copy_(cur)


def _run(rank, world, deferred):
    """The steps of one process over rows [rank M / world, (rank + 1) M / world)."""
    from fp8_delayed_scaling_row_gb300 import lnfp8 as L
    torch.cuda.set_device(0)
    rec = L.Recipe("hybrid", HIST)
    p = synth.mlp_params(D, F, seed=SEED, bias_std=0.02)
    dev = {k: bf16_dev(v) for k, v in p.items()}
    fm, bm = L.ScalingMeta(4, HIST), L.ScalingMeta(2, HIST)
    r0, r1 = rank * M // world, (rank + 1) * M // world
    ctx, grads = L.mlp_ctx(r1 - r0, D, F), L.mlp_grads(r1 - r0, D, F)
    states, sums = [], []
    for step in range(STEPS):
        x = bf16_dev(synth.activations(M, D, dist="outliers", seed=SEED, step=step)[r0:r1])
        dy = bf16_dev(synth.grad(M, D, seed=SEED, step=step)[r0:r1])
        L.ln_mlp_fwd(x, dev["gamma"], dev["beta"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], fm, rec, ctx=ctx,
                     defer_update=deferred)
        if deferred:
            _exchange(fm)
            L.amax_history_update(fm, rec, [rec.fwd_dtype] * 4, scale_inv_before=ctx.sinv_saved)
        g = L.ln_mlp_bwd(dy, x, dev["gamma"], ctx, bm, rec, grads=grads, defer_update=deferred)
        if deferred:
            _exchange(bm)
            L.amax_history_update(bm, rec, [rec.bwd_dtype] * 2)
        L.sync_status()
        s = {k: getattr(g, k).float().cpu() for k in GRADS}
        dp.allreduce_grads_(list(s.values()))
        sums.append({k: v.numpy().astype(np.float64) for k, v in s.items()})
        states.append({f"{d}_{k}": getattr(m, k).cpu().numpy().copy() for d, m in (("fwd", fm), ("bwd", bm))
                       for k in ("scale", "scale_inv", "amax_history")})
    return states, sums


def _rank_worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out.put((rank, _run(rank, world, True)))
    except Exception as e:  # reported to the parent, which fails the test with it
        out.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_on_the_library_state_keep_one_process_state():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=600) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, r in res:
        assert not isinstance(r, str), f"rank {rank}: {r}"
    want_states, want_sums = _run(0, 1, False)
    assert (want_states[-1]["fwd_scale"] != 1).all() and (want_states[-1]["bwd_scale"] != 1).all()
    for rank, (states, sums) in res:
        for step in range(STEPS):
            for k, want in want_states[step].items():
                assert np.array_equal(states[step][k].view(np.uint32), want.view(np.uint32)), (rank, step, k)
            for k in GRADS:
                got, want = sums[step][k], want_sums[step][k]
                assert np.linalg.norm(got - want) <= 1e-2 * np.linalg.norm(want), (rank, step, k)
