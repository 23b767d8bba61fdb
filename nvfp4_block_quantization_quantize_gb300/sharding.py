"""Row sharding of one tensor's quantization across ranks (host logic).

Blocks never span rows (1x16) or 16-row bands (16x16, columnwise), so a
tensor splits into contiguous row shards that are quantized independently:
each rank passes its shard's first global row as ``row_offset`` (so stochastic
rounding draws the unsharded tensor's counters) and, for a per-tensor global
scale, the tensor amax -- the one exchange the path has: an all-reduce MAX of
one fp32 value (exact and order-free).  Per-row and no global scale need no
exchange at all.  A rank's columnwise output is a column slice
[:, r0/2 : r1/2] of the whole tensor's.
"""
from __future__ import annotations

import torch


def shard_rows(M: int, world: int, rank: int, align: int = 16) -> tuple[int, int]:
    """[r0, r1) of rank's shard: `align`-row units split as evenly as possible."""
    if M % align:
        raise ValueError(f"M={M} is not a multiple of the shard alignment {align}")
    units = M // align
    base, extra = divmod(units, world)
    u0 = rank * base + min(rank, extra)
    u1 = u0 + base + (1 if rank < extra else 0)
    return u0 * align, u1 * align


def global_amax(local_amax: torch.Tensor, group=None) -> torch.Tensor:
    """All-reduce MAX of the shards' amaxes (one fp32 per rank)."""
    import torch.distributed as dist
    out = local_amax.clone()
    dist.all_reduce(out, op=dist.ReduceOp.MAX, group=group)
    return out


def sharded_quantize(x_shard: torch.Tensor, row_offset: int, *, gamax_mode: str = "none",
                     group=None, quantize_fn=None, amax_fn=None, **kw) -> dict:
    """Quantize this rank's row shard as part of the whole tensor.

    ``gamax_mode`` "tensor" computes the shard amax, exchanges the maximum and
    quantizes with it given; "none" and "row" need no exchange.  By default the
    shard is quantized by the CUDA library; ``quantize_fn`` / ``amax_fn`` take
    the same arguments as nvfp4_quantize / nvfp4_amax.
    """
    if quantize_fn is None or amax_fn is None:
        from . import nvfp4_amax, nvfp4_quantize
        quantize_fn = quantize_fn or nvfp4_quantize
        amax_fn = amax_fn or nvfp4_amax
    if gamax_mode == "tensor":
        # the amax of what is quantized: x + residual under error feedback
        A = global_amax(amax_fn(x_shard, residual=kw.get("residual")).reshape(1).float(), group)
        out = quantize_fn(x_shard, row_offset=row_offset, gamax_mode="tensor_given", gamax=A, **kw)
        out["gamax"] = A
        return out
    return quantize_fn(x_shard, row_offset=row_offset, gamax_mode=gamax_mode, **kw)
