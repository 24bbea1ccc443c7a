"""Attention with the keys and values sharded over ranks (context parallel).

Each rank holds all queries and one shard of the keys and values.  It attends
to its shard with the prefill (or decode) kernel, the ranks exchange their
(o, lse) once, and ``attn_merge`` combines them with the two-block softmax
merge of the CS149 Lecture 9 notes, concept 9 -- the only exchange step
key-sharded attention needs.  Non-causal: a causal mask over sharded keys
would leave query rows with no visible key in some shards, which the prefill
kernel does not take.

The exchange is a ``torch.distributed`` all-gather (NCCL between GPUs); the
merge runs in the CUDA library.
"""
import torch
import torch.distributed as dist

from . import binding


def gather_partials(o_local, lse_local, group=None):
    """All-gather every rank's (o, lse) for the same queries.  Returns
    (o_parts [S, ...], lse_parts [S, ...]) stacked in rank order."""
    world = dist.get_world_size(group)
    o_parts = [torch.empty_like(o_local) for _ in range(world)]
    lse_parts = [torch.empty_like(lse_local) for _ in range(world)]
    dist.all_gather(o_parts, o_local.contiguous(), group=group)
    dist.all_gather(lse_parts, lse_local.contiguous(), group=group)
    return torch.stack(o_parts), torch.stack(lse_parts)


def attention_kv_sharded(q, k_shard, v_shard, scale=None, group=None):
    """softmax(scale q K^T) V over the keys of every rank's shard.

    q [B, H, Nq, d] (the same on every rank), k_shard / v_shard
    [B, H, Nk_r, d] (this rank's keys, any split).  Returns (o, lse) over all
    keys, on every rank."""
    if q.shape[2] == 1:
        o, lse = binding.attn_fwd_decode(q, k_shard, v_shard, scale=scale)
    else:
        o, lse = binding.attn_fwd(q, k_shard, v_shard, causal=False, scale=scale)
    o_parts, lse_parts = gather_partials(o, lse, group)
    return binding.attn_merge(o_parts, lse_parts)
