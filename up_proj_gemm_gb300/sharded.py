"""Head-sharded (column-parallel) query up-projection over a process group.

Each rank owns a contiguous block of heads: rows [h0 * D, h1 * D) of W (and
of the bias), D = Dn + Dr. The partitioning follows from what the method
computes:
  * forward: q's heads are independent. The rotate-half pair (i, i + Dr/2)
    and every 32-channel MXFP8 block lie inside one head, so a rank's q
    slice [T, h1 - h0, D] needs only its own rows of W. No exchange.
  * backward (TransformerEngine PR "Add a backwards linear function to be
    used with the fused mla q up-proj", sequence diagram: the RoPE backward,
    then the linear backward): dW and db of a rank's heads need only that
    rank's dq slice, so they stay local; dx = sum over heads of
    dq_pre[:, head] W[head, :] is a sum over ranks of each rank's partial dx:
    one sum all-reduce of [T, K].
The collective is torch.distributed (NCCL on GPUs), issued on the caller's
stream after the local dgrad, with the result landing in the local dx.

Every local step runs in the library's kernels (``fwd``, ``bwd_dgrad``,
``bwd_wgrad``); this module only slices and hands over tensors. ``ops`` may
replace those three calls (the host-side logic is tested that way on CPU
ranks); by default they are the CUDA entry points.
"""
from __future__ import annotations

from dataclasses import dataclass

__all__ = ["HeadShard", "head_shard", "shard_weight", "sharded_fwd", "sharded_bwd"]


@dataclass(frozen=True)
class HeadShard:
    """Rank ``rank`` of ``world`` owns heads [h0, h1) of H."""

    rank: int
    world: int
    H: int
    h0: int
    h1: int

    @property
    def heads(self) -> int:
        return self.h1 - self.h0


def head_shard(H: int, rank: int, world: int) -> HeadShard:
    """Contiguous, balanced head blocks: the first H % world ranks take one
    head more. Every rank gets at least one head (world <= H)."""
    if not (0 < world <= H) or not (0 <= rank < world):
        raise ValueError(f"cannot split {H} heads over {world} ranks (rank {rank})")
    base, extra = divmod(H, world)
    h0 = rank * base + min(rank, extra)
    return HeadShard(rank, world, H, h0, h0 + base + (1 if rank < extra else 0))


def _rows(sh: HeadShard, D: int) -> slice:
    return slice(sh.h0 * D, sh.h1 * D)


def shard_weight(W, bias, sh: HeadShard, D: int):
    """This rank's rows of W [H * D, K] and of the bias [H * D] (views)."""
    r = _rows(sh, D)
    return W[r], (None if bias is None else bias[r])


def _default_ops():
    from . import bwd_dgrad, bwd_wgrad, fwd
    return {"fwd": fwd, "bwd_dgrad": bwd_dgrad, "bwd_wgrad": bwd_wgrad}


def sharded_fwd(x, W_local, cos, sin, sh: HeadShard, Dn, Dr, bias_local=None, pos=None, ops=None, **kw):
    """This rank's q slice [T, heads, D] (bf16, or MXFP8 codes and scales with
    out_mode "mxfp8"): the forward on the rank's own rows of W. No exchange."""
    ops = ops or _default_ops()
    return ops["fwd"](x, W_local, cos, sin, sh.heads, Dn, Dr, bias=bias_local, pos=pos, **kw)


def sharded_bwd(dq_local, x, W_local, cos, sin, sh: HeadShard, Dn, Dr, pos=None, want_db=False, group=None,
                ops=None, all_reduce=None):
    """Backward of one rank: dx (summed over the ranks), and this rank's dW
    rows and db entries. dq_local: the rank's slice [T, heads, D] of dq.
    ``all_reduce(tensor, group)`` defaults to torch.distributed.all_reduce
    (sum, in place); with world == 1 nothing is exchanged."""
    import torch
    ops = ops or _default_ops()
    T = x.shape[0]
    # dgrad hands the rotated rope channels to wgrad (one RoPE backward per rank)
    rope = torch.empty((T, sh.heads, Dr), dtype=torch.bfloat16, device=dq_local.device)
    dx = ops["bwd_dgrad"](dq_local, W_local, cos, sin, sh.heads, Dn, Dr, pos=pos, dq_pre_rope=rope)
    dW, db = ops["bwd_wgrad"](dq_local, x, cos, sin, sh.heads, Dn, Dr, pos=pos, db=want_db, dq_pre_rope=rope)
    if sh.world > 1:
        if all_reduce is None:
            import torch.distributed as dist

            def all_reduce(t, g):
                dist.all_reduce(t, op=dist.ReduceOp.SUM, group=g)
        all_reduce(dx, group)
    return dx, dW, db
