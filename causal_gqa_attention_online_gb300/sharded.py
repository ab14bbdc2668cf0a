"""Decode over one long context whose key axis is sharded across GPUs.

"Attention execution mapping" (LuisaCompute), section 5: splitting the key
axis needs a legal merge of the (max, sum, acc) state.  Here every rank holds
a contiguous shard of each sequence's keys, computes the attention of the
query rows over its shard with the library's kernels (a partial O normalised
by its own sum, and its LSE), the ranks exchange those partials with one
all-gather, and every rank merges them with the library's LSE combine kernel:

    L = log sum_r exp(lse_r),   O = sum_r exp(lse_r - L) O_r.

A shard without a legal key of a row contributes lse = -inf and is ignored.
Scope: decode (one query row per sequence), bottom-right causal, no window:
then the legal keys of a shard are exactly its first clamp(Kb - k_lo, 0,
shard_len) keys, so each rank runs the ordinary padded-layout kernel with
those per-sequence lengths.  The exchange is the only collective; its
backend is the process group's (NCCL across GPUs; with gloo the partials go
through host memory).  This module only marshals arguments: every step of
the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import torch

from . import binding


def shard_key_lengths(seqlens_k: torch.Tensor, key_offset: int, shard_len: int) -> torch.Tensor:
    """Keys of each sequence that fall in the shard [key_offset, key_offset +
    shard_len): clamp(Kb - key_offset, 0, shard_len), int32 on the host."""
    if seqlens_k.device.type != "cpu" or seqlens_k.dtype != torch.int32:
        raise ValueError("seqlens_k must be an int32 CPU tensor")
    if key_offset < 0 or shard_len < 0:
        raise ValueError("key_offset and shard_len must be non-negative")
    return (seqlens_k.to(torch.int64) - key_offset).clamp(0, shard_len).to(torch.int32)


def gather_partials(o_part: torch.Tensor, lse_part: torch.Tensor, group=None):
    """All-gather the ranks' partials into [world, *o_part.shape] and
    [world, *lse_part.shape] (rank order).  With the gloo backend, device
    tensors are staged through host memory."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    via_host = dist.get_backend(group) == "gloo" and o_part.is_cuda
    src_o = o_part.cpu() if via_host else o_part.contiguous()
    src_l = lse_part.cpu() if via_host else lse_part.contiguous()
    out_o = torch.empty((world,) + tuple(src_o.shape), dtype=src_o.dtype, device=src_o.device)
    out_l = torch.empty((world,) + tuple(src_l.shape), dtype=src_l.dtype, device=src_l.device)
    dist.all_gather(list(out_o.unbind(0)), src_o, group=group)
    dist.all_gather(list(out_l.unbind(0)), src_l, group=group)
    if via_host:
        out_o = out_o.to(o_part.device, non_blocking=False)
        out_l = out_l.to(lse_part.device, non_blocking=False)
    return out_o, out_l


def attn_decode_sharded_keys(q, k_shard, v_shard, seqlens_k, key_offset, *, group=None,
                             scale=None, stream=None):
    """Decode attention of q [B, 1, Hq, D] over keys sharded across the ranks
    of ``group``: this rank holds keys [key_offset, key_offset + Ks) of every
    sequence in k_shard [B, Ks, Hkv, D] / v_shard [B, Ks, Hkv, Dv];
    ``seqlens_k`` (int32, host) holds the full key counts.  Returns the merged
    (o [B, 1, Hq, Dv], lse [B, 1, Hq]) on every rank."""
    B, Qn, Hq, _ = q.shape
    if Qn != 1:
        raise ValueError("the sharded decode takes one query row per sequence")
    Ks = k_shard.shape[1]
    Dv = v_shard.shape[3]
    local = shard_key_lengths(seqlens_k, key_offset, Ks).to(q.device)
    o_part, lse_part = binding.attn_fwd(q, k_shard, v_shard, seqlens_k=local, scale=scale,
                                        stream=stream)
    if stream is not None:  # the collective follows torch's current stream
        torch.cuda.current_stream(q.device).wait_stream(stream)
    o_all, lse_all = gather_partials(o_part.view(B * Hq, Dv), lse_part.view(B * Hq), group)
    o, lse = binding.attn_lse_combine_parts(o_all, lse_all, stream=stream)
    return o.view(B, 1, Hq, Dv), lse.view(B, 1, Hq)
