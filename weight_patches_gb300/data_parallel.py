"""Data-parallel use of the LoRA linear: tokens sharded over ranks.

The forward is token-local, so ranks that each hold a contiguous block of token rows need no
exchange on the data path.  The closed-form backward (Unsloth fast_lora walkthrough,
sections 2 and 4) splits the same way for dX, but dA_g = s_g (dY_g B_g)^T X and
dB_g = s_g dY_g^T (X A_g^T) are sums over token rows, so the per-shard results are added by
one all-reduce of the fp32 dA/dB across the group.  ``torch.distributed`` carries it (NCCL on
GPUs); every other step runs in the CUDA library.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence, Tuple

import torch
import torch.distributed as dist


def shard_rows(T: int, rank: int, world: int) -> Tuple[int, int]:
    """[start, end) of the token rows rank ``rank`` of ``world`` holds: contiguous blocks whose
    sizes differ by at most one, covering [0, T) exactly once in rank order."""
    if world < 1 or not 0 <= rank < world or T < 0:
        raise ValueError("need 0 <= rank < world and T >= 0")
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, group=None, device=None) -> float:
    """The largest value over the ranks of the group (the whole job's time is the slowest
    rank's); the value itself when torch.distributed is not initialised."""
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def lora_linear_bwd_dp(X_local: torch.Tensor, W, dY_local: torch.Tensor, adapters: Sequence,
                       request_scale: float = 1.0, group=None,
                       local_bwd: Optional[Callable] = None, **kw):
    """Backward of one LoRA linear over the token shard this rank holds: (dX_local, dA, dB) with
    dX for the local rows and dA, dB summed over every rank of ``group``.  ``local_bwd`` computes
    the shard's (dX, [dA_g], [dB_g]) and defaults to the library's ``lora_linear_bwd``; extra
    keyword arguments go to it."""
    if local_bwd is None:
        from . import lora_linear_bwd as local_bwd
    dX, dA, dB = local_bwd(X_local, W, dY_local, adapters, request_scale, **kw)
    if dist.is_available() and dist.is_initialized():
        # one flat fp32 buffer: a single all-reduce for every dA_g and dB_g
        flat = torch.cat([t.reshape(-1) for t in list(dA) + list(dB)])
        dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
        out, off = [], 0
        for t in list(dA) + list(dB):
            n = t.numel()
            out.append(flat[off:off + n].view_as(t))
            off += n
        dA, dB = out[:len(dA)], out[len(dA):]
    return dX, list(dA), list(dB)
