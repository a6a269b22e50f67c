"""Sequence-parallel (context-parallel) decode: each rank holds a contiguous shard of the
KV sequence, computes split partials of its shard, and the partials of all ranks are
merged with the same LSE weights as the splits of one device.

"AI Infra: math and infra optimisation in large models", section 2.6 "Sequence
Parallelism": when the context does not fit one device, the KV sequence is sharded
over devices; thanks to the LSE form, each device only needs to hand over its partial
output and one LSE scalar per row, and the merge is exact.  Only that exchange is done
here (an all-gather of the partials); every arithmetic step runs in libfd's kernels.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist

from . import _binding as fd


def gather_partials(lse_part: torch.Tensor, o_part: torch.Tensor,
                    group: Optional[dist.ProcessGroup] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """All-gather per-rank partials along the split axis, rank-major.

    lse_part [B, Hq, S] and o_part [B, Hq, S, d] (the same S on every rank).  Returns
    [B, Hq, world * S] and [B, Hq, world * S, d]; splits of rank r occupy
    [r * S, (r + 1) * S).  The merge is order-independent, so any rank order is exact;
    rank-major keeps the sequence order for readers of the partials.
    """
    world = dist.get_world_size(group)
    lse_part = lse_part.contiguous()
    o_part = o_part.contiguous()
    lse_list = [torch.empty_like(lse_part) for _ in range(world)]
    o_list = [torch.empty_like(o_part) for _ in range(world)]
    dist.all_gather(lse_list, lse_part, group=group)
    dist.all_gather(o_list, o_part, group=group)
    return torch.cat(lse_list, dim=2), torch.cat(o_list, dim=2)


def shard_num_splits(B: int, Hq: int, Hkv: int, d: int, shard_capacity: int,
                     num_splits: int, group: Optional[dist.ProcessGroup] = None) -> int:
    """The split count every rank uses for its shard.  num_splits > 0 is taken as is;
    0 resolves the library's count for this rank's shard capacity and takes the largest
    over the ranks (the gather needs the same count everywhere; a shard with more splits
    than its heuristic count is still exact)."""
    if num_splits > 0:
        return num_splits
    S = fd.resolve_num_splits(B, Hq, Hkv, d, shard_capacity, 0)
    if dist.get_world_size(group) > 1:
        backend = dist.get_backend(group)
        dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
        t = torch.tensor([S], dtype=torch.int64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        S = int(t.item())
    return S


def sp_decode_attention(q: torch.Tensor, k_shard: torch.Tensor, v_shard: torch.Tensor,
                        seq_lens_shard: torch.Tensor, num_splits: int = 0,
                        group: Optional[dist.ProcessGroup] = None, block_table=None,
                        page_size: int = 0, out_dtype=torch.float32):
    """Decode one step over a KV sequence sharded across the ranks of `group`.

    Each rank passes the same q [B, Hq, d] and its own shard of the cache (its token
    count in `seq_lens_shard`; a rank whose shard is empty for a row passes 0 there,
    which yields LSE = -inf, weight 0).  num_splits is per shard (0: see
    shard_num_splits).  Returns (out, lse_out), identical on every rank.
    """
    B, Hq, d = q.shape
    Hkv = k_shard.shape[1]
    cap = k_shard.shape[2] if block_table is None else block_table.shape[1] * page_size
    S = shard_num_splits(B, Hq, Hkv, d, cap, num_splits, group)
    ws = torch.zeros(fd.workspace_size(B, Hq, Hkv, d, S), dtype=torch.uint8, device=q.device)
    S = fd.decode_partial(q, k_shard, v_shard, seq_lens_shard, ws, block_table, page_size, S)
    lse_part, o_part = fd.workspace_partials(ws, B, Hq, d, S)
    lse_all, o_all = gather_partials(lse_part, o_part, group)
    return fd.merge_partials(lse_all, o_all, out_dtype=out_dtype)
