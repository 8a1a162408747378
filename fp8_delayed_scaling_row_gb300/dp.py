"""Data-parallel exchange of the delayed-scaling state (host plumbing over
torch.distributed; no arithmetic of the method here).

The path shards over tokens: each rank casts and multiplies its own rows. Two
things cross ranks in a data-parallel step:

* the running amaxes, reduced with MAX before the state update, so that every
  rank derives the same scales (a rank that saw a larger value than the others
  must not cast with a scale the others do not use);
* the weight, bias and LayerNorm gradients, reduced with SUM (the usual
  data-parallel gradient reduction).

The amax reduction runs on the fp32 bit patterns viewed as int32: for the
non-negative magnitudes the library records (|x|, NaN > Inf > finite) that
order is the numeric one, so the result equals the amax of the union of the
ranks' rows bit for bit, NaN included. Use it with ``defer_update=True`` on the
module calls, then ``amax_history_update``:

    y, ctx = lnfp8.ln_mlp_fwd(..., meta_fwd, recipe, defer_update=True)
    dp.allreduce_amax_(meta_fwd.amax_cur)
    lnfp8.amax_history_update(meta_fwd, recipe, dtypes, scale_inv_before=ctx.sinv_saved)
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def _active(group) -> bool:
    return dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1


def allreduce_amax_(amax_cur: torch.Tensor, group=None) -> torch.Tensor:
    """In place: amax_cur <- max over ranks (fp32 magnitude bit order). A no-op on one rank."""
    if amax_cur.dtype != torch.float32:
        raise TypeError("amax_cur must be float32")
    if _active(group):
        bits = amax_cur.view(torch.int32)
        dist.all_reduce(bits, op=dist.ReduceOp.MAX, group=group)
    return amax_cur


def allreduce_grads_(tensors, group=None) -> None:
    """In place: every tensor <- sum over ranks (data-parallel gradient reduction)."""
    if not _active(group):
        return
    for t in tensors:
        if t is not None:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
