"""Decode-context-parallel verify attention: every sequence's KV is split
across the ranks of a process group, each rank attends over its own shard,
and the shard results are exchanged and merged by log-sum-exp.

The pages name a decode-context-parallel degree for the verify kernel
(sglang PR 34517 digest, "Key code excerpts": ``get_num_kv_heads(attn_tp_size,
attn_dcp_size)``) and merge split-KV segments by log-sum-exp (sglang PR 36330
digest, "Implementation breakdown" item 1, the "reduce segments" kernel).
Here the merge runs across ranks:

1. ``verify_attn_partial`` (C-ABI, GPU) on this rank's shard: fp32 o,
   normalised over the shard's visible keys, and its natural-log lse;
2. an all-gather of (o, lse) over the group (NCCL on CUDA tensors; a gloo
   group stages them through host memory);
3. ``verify_attn_merge_partials`` (C-ABI, GPU): out = sum_i exp(lse_i - LSE)
   o_i, in rank order, so every rank computes the same bf16 output.

A shard is a contiguous range of key positions [o_b, o_b + S_b) of sequence
b reached through its own block table, with kv_extent_b = (the sequence's
total keys) - o_b giving its causal position (see ``verify_attn_partial``).
The exchange moves 4 * total_q * Hq * (256 + 1) bytes per rank.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import torch
import torch.distributed as dist

from . import merge_partials, verify_attn_partial

MAX_RANKS = 16  # shards verify_attn_merge_partials combines in one launch


def gather_shard_results(o: torch.Tensor, lse: torch.Tensor,
                         group=None) -> List[Tuple[torch.Tensor, torch.Tensor]]:
    """All-gathers this rank's shard result (o [total_q, Hq, D] fp32, lse
    [total_q, Hq] fp32) over ``group``. Returns the (o, lse) of every rank in
    rank order, on ``o``'s device. A gloo group gets host copies of CUDA
    tensors (the copy synchronises the current stream)."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    if world == 1:
        return [(o, lse)]
    if world > MAX_RANKS:
        raise ValueError(f"at most {MAX_RANKS} ranks per merge (group has {world})")
    staged = o.is_cuda and dist.get_backend(group) == "gloo"
    so = (o.cpu() if staged else o).contiguous()
    sl = (lse.cpu() if staged else lse).contiguous()
    os_ = [torch.empty_like(so) for _ in range(world)]
    ls_ = [torch.empty_like(sl) for _ in range(world)]
    dist.all_gather(os_, so, group=group)
    dist.all_gather(ls_, sl, group=group)
    if staged:
        os_ = [x.to(o.device) for x in os_]
        ls_ = [x.to(o.device) for x in ls_]
    return list(zip(os_, ls_))


def dcp_verify_attn(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, kv_extent,
                    max_seqlen_q: int, max_seqlen_k: int, softmax_scale: float,
                    k_descale=None, v_descale=None, out: Optional[torch.Tensor] = None,
                    group=None, workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                    stream=None) -> torch.Tensor:
    """Verify attention with every sequence's keys sharded over ``group``.

    Every rank passes the same q, cu_seqlens_q and max_seqlen_q, and its own
    shard: k_cache / v_cache / block_table / seqused_k (the shard's keys) and
    kv_extent [B] int32 (total keys of the sequence minus the shard's first
    key position; None on a rank whose shards end every sequence).
    max_seqlen_k bounds the shard's lengths. Returns out [total_q, Hq, 256]
    bf16, the same on every rank."""
    o, lse = verify_attn_partial(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                                 max_seqlen_q, max_seqlen_k, softmax_scale, k_descale, v_descale,
                                 kv_extent=kv_extent, workspace=workspace, num_splits=num_splits,
                                 stream=stream)
    parts = gather_shard_results(o, lse, group)
    return merge_partials(parts, out=out, stream=stream)
