"""Decode context parallelism across processes: the exchange step.

Under decode context parallelism ("ブロック表", 設計動機: the DCP interleave of a
request's positions over ranks), rank k of W holds its share of every
request's keys and decodes over them with ``bkv_paged_decode_cp``, which
leaves a normalised output and a natural-log sum of exponentials per query
row.  The ranks then exchange those states and merge them exactly with
``bkv_merge_attn_states``.  That exchange is the one step of the path that
needs a collective: this module does it as two all-gathers over a
``torch.distributed`` process group (NCCL for device tensors) followed by
the merge kernel.  Everything else on the path is per rank.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import bkv


def gather_states(out: torch.Tensor, lse: torch.Tensor, group=None):
    """All-gather this rank's decode state.

    ``out`` is (num_reqs, q_len, H_q, D) and ``lse`` (num_reqs, q_len, H_q)
    fp32; returns ``(outs, lses)`` of shape (W, ...) with rank k's state at
    index k, the layout ``bkv_merge_attn_states`` takes."""
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    if tuple(lse.shape) != tuple(out.shape[:-1]):
        raise ValueError("lse must have out's shape without its last dimension")
    world = dist.get_world_size(group)
    out_c, lse_c = out.contiguous(), lse.contiguous()
    outs = [torch.empty_like(out_c) for _ in range(world)]
    lses = [torch.empty_like(lse_c) for _ in range(world)]
    dist.all_gather(outs, out_c, group=group)
    dist.all_gather(lses, lse_c, group=group)
    return torch.stack(outs), torch.stack(lses)


def merge_across_ranks(out: torch.Tensor, lse: torch.Tensor, merged_out: torch.Tensor,
                       merged_lse: torch.Tensor | None = None, group=None, stream=None) -> torch.Tensor:
    """Gather every rank's (out, lse) and merge them into ``merged_out`` (and ``merged_lse``) on this
    rank with the library's merge kernel: the attention over all ranks' keys."""
    outs, lses = gather_states(out, lse, group)
    bkv.bkv_merge_attn_states(outs, lses, merged_out, merged_lse, stream=stream)
    return merged_out
