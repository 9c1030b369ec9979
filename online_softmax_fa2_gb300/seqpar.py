"""Attention over keys sharded across devices (sequence parallelism), through the library.

Each rank holds every query row and one contiguous shard of the keys and values.  It computes
the state (m, l, u) of every row over its own shard (attn_fwd_partial), the ranks exchange
these states (one all-gather of B*H*Nq*(2 + dv) floats per rank), and every rank merges them
(attn_merge_states_rows) into the output and log-sum-exp of attention over the whole key axis.
The shards must cover each sequence's keys exactly once ("How Does FlashAttention Preserve
Global Softmax Across Tiles?", sections 3 and 4: the states of disjoint key sets merge to the
state of their union; a key counted twice would be weighted twice).

The exchange is plain torch.distributed; every step that computes runs in the library's
kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def gather_states(part: torch.Tensor, group=None) -> torch.Tensor:
    """All ranks' states stacked along a new leading axis: [R, *part.shape] (rank order).  The
    state s of row r then sits at r * row_stride + s * split_stride floats with
    row_stride = part.shape[-1] and split_stride = part.numel()."""
    world = dist.get_world_size(group)
    flat = part.contiguous().view(-1)
    out = torch.empty(world * flat.numel(), dtype=part.dtype, device=part.device)
    dist.all_gather_into_tensor(out, flat, group=group)  # concatenated in rank order
    return out.view((world,) + tuple(part.shape))


def sequence_parallel_attn(q, k_shard, v_shard, key_offset, nk_total, group=None, kv_lens=None,
                           bias=None, causal=False, scale=None, stream=None):
    """o [B, Nq, H, dv] and lse [B, H, Nq] of attention over all ranks' key shards (this rank's
    is keys [key_offset, key_offset + k_shard.shape[1]) of nk_total).  Every rank passes the same
    q, kv_lens, causal and scale; bias (if any) covers this rank's keys only."""
    import online_softmax_fa2_gb300 as ofa

    B, Nq, H, _ = q.shape
    dv = v_shard.shape[3]
    s = torch.cuda.current_stream(q.device) if stream is None else stream
    # the partial kernel, the collective and the merge run in that order on one stream
    with torch.cuda.stream(s):
        part = ofa.attn_fwd_partial(q, k_shard, v_shard, key_offset, nk_total, kv_lens=kv_lens, bias=bias,
                                    causal=causal, scale=scale, stream=s)
        allp = gather_states(part, group)
        world = allp.shape[0]
        return ofa.attn_merge_states_rows(allp, B, H, Nq, dv, world, row_stride=2 + dv,
                                          split_stride=part.numel(), dtype=q.dtype, stream=s)
