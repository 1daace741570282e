"""Host-side helpers for running verification on several GPUs as replicas.

Requests are independent: every packed row depends only on its own logits and
on its owner request's parameters, so a batch splits by request into
contiguous blocks, one per rank, with each block's cu_rows rebased to start at
zero.  Verification then needs no exchange at all.  The only cross-rank step
is the prefix-acceptance counters (acc[j] = #{a_b > j}, ver[j] = #{k_b > j},
hist[a]), which are sums over requests: one int64 sum all-reduce of
2*k_max + 1 values gives the job-wide counters at read time.

Definitions: xLLM docs "自适应投机推理" §"自适应 draft 步长（MTP）"
(per-position prefix acceptance from accepted and verified counts), and the
independence of requests in the ragged packed layout of §"启动示例".
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def request_shard(cu_rows: np.ndarray, world: int, rank: int) -> Tuple[int, int, int, int]:
    """Contiguous block of requests [b_lo, b_hi) for `rank` of `world`, with
    packed rows [r_lo, r_hi): boundaries are placed so every rank gets about
    R / world rows (requests are never split).  Pure host arithmetic."""
    cu = np.asarray(cu_rows, dtype=np.int64)
    B = cu.size - 1
    if world < 1 or not (0 <= rank < world):
        raise ValueError("rank must lie in [0, world)")
    R = int(cu[B])

    def boundary(q: int) -> int:
        # first request whose start reaches q * R / world (rows)
        if q <= 0:
            return 0
        if q >= world:
            return B
        target = (q * R + world - 1) // world
        return int(np.searchsorted(cu[:B], target, side="left"))

    b_lo, b_hi = boundary(rank), boundary(rank + 1)
    b_hi = max(b_hi, b_lo)
    return b_lo, b_hi, int(cu[b_lo]), int(cu[b_hi])


def rebase(cu_rows: np.ndarray, b_lo: int, b_hi: int) -> np.ndarray:
    """cu_rows of the requests [b_lo, b_hi), starting at zero."""
    cu = np.asarray(cu_rows, dtype=np.int64)
    return (cu[b_lo:b_hi + 1] - cu[b_lo]).astype(np.int32)


def reduce_prefix_stats(acc, ver, hist=None, group=None):
    """Sum the prefix-acceptance counters of all ranks in place (torch int64
    tensors on the rank's device; gloo for CPU tensors, NCCL for CUDA).  A
    no-op outside an initialised process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return acc, ver, hist
    for t in (acc, ver, hist):
        if t is not None:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return acc, ver, hist


def prefix_acceptance(acc, ver) -> np.ndarray:
    """acc[j] / ver[j] (0 where no request had a j-th draft)."""
    a = np.asarray(acc, dtype=np.float64)
    v = np.asarray(ver, dtype=np.float64)
    out = np.zeros_like(a)
    np.divide(a, v, out=out, where=v > 0)
    return out


def max_over_ranks(x: float, device=None, group=None) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def sum_over_ranks(x: float, device=None, group=None) -> float:
    """The sum of every rank's x (units processed by the whole job)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def init_from_env(backend: Optional[str] = None):
    """(world, rank, local_rank) from the torchrun environment; initialises the
    process group when world > 1 (NCCL with CUDA, else gloo)."""
    import os
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        be = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        dist.init_process_group(be)
    return world, rank, local
