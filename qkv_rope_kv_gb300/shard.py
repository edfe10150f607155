"""Head sharding of the QKV stage across GPUs (host-side arithmetic, no kernels).

The stage has no exchange step: every output row depends only on its own
weight row, x (replicated) and, for RoPE, its position inside its head.  So the
stage shards by kv-head groups with no collective: rank r of W owns kv heads
[r*nkv/W, (r+1)*nkv/W), the q heads that attend to them, the matching rows of
the concatenated wq|wk|wv matrix and bias, and columns [k0*hd, k1*hd) of every
layer's K and V regions.  A rank runs the ordinary single-GPU plan on its
slice (n_head/W q heads, n_head_kv/W kv heads).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class HeadShard:
    rank: int
    world: int
    n_head: int          # local q heads
    n_head_kv: int       # local kv heads
    q_rows: tuple        # [start, stop) in the global q section
    kv_rows: tuple       # [start, stop) in the global k section (same for v)
    concat_rows: tuple   # three [start, stop) ranges of the global concat matrix: q, k, v

    @property
    def kv_cols(self) -> tuple:
        """Columns of the global K/V regions this rank stores."""
        return self.kv_rows


def head_shard(n_head: int, n_head_kv: int, head_dim: int, world: int, rank: int) -> HeadShard:
    if n_head % n_head_kv:
        raise ValueError("n_head must be a multiple of n_head_kv")
    if n_head_kv % world:
        raise ValueError("n_head_kv (%d) must be a multiple of the world size (%d)" % (n_head_kv, world))
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    group = n_head // n_head_kv
    kv_local = n_head_kv // world
    k0, k1 = rank * kv_local, (rank + 1) * kv_local
    q0, q1 = k0 * group, k1 * group
    nqt, nkt = n_head * head_dim, n_head_kv * head_dim
    q_rows = (q0 * head_dim, q1 * head_dim)
    kv_rows = (k0 * head_dim, k1 * head_dim)
    concat = (q_rows, (nqt + kv_rows[0], nqt + kv_rows[1]), (nqt + nkt + kv_rows[0], nqt + nkt + kv_rows[1]))
    return HeadShard(rank, world, q1 - q0, kv_local, q_rows, kv_rows, concat)


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over the default process group (gloo on CPU, nccl on a GPU)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
