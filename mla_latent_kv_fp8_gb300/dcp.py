"""Decode context parallelism (DCP) across GPUs: the exchange around the decode.

"Kimi K3 on AMD Instinct MI355X" post, section 1 "Cache", DCP paragraph: the
latent history of every request is cut into shards, one per GPU of the group,
so each GPU stores a fraction of the positions; the queries are exchanged so
that every GPU attends with all of them to its own shard, and the partial
answers, each carrying its log-sum-exp, are merged with softmax weights.

Here a group of W ranks (torch.distributed, NCCL on GPUs) holds contiguous,
page-aligned shards of every history (``shard_plan``): rank r the r-th shard,
the last rank the tail, where the T draft positions of a multi-token verify
sit.  One step (``dcp_decode``):

  1. all-gather the queries along the head dim: each rank brings its own heads
     (tensor parallelism splits heads), every rank ends with all H heads;
  2. decode all H heads over the local shard (``mla_decode_paged`` on this
     rank's own paged cache): a partial answer (bf16 out, fp32 lse) per row.  A
     shard before the last holds only positions every draft query sees, so for
     T > 1 it is decoded as T = 1 with T*H rows; the last shard keeps the causal
     rule;
  3. all-gather the partial answers: [W, B, T, H, 512] and [W, B, T, H], in
     rank (= shard) order;
  4. merge them by their normalisers (``mla_merge_partials``) and keep this
     rank's heads.

Steps 2 and 4 run in the library's CUDA kernels; this module only moves
tensors between ranks and reshapes them.  The local decode and the merge are
parameters, so that the exchange and its bookkeeping can be exercised on CPU
ranks (gloo) with precomputed partial answers.
"""
from __future__ import annotations

from typing import Callable

import torch
import torch.distributed as dist


def shard_plan(lens, block_table, n_shards: int, T: int = 1):
    """Contiguous, page-aligned shards of every history: shards 0..n-2 hold
    ceil(L / (64 n)) pages each, the last shard the rest (with the T draft
    positions at its end).  Returns, per shard, (block table int32 [B, width],
    lengths int32 [B]) on the CPU, the table holding that shard's pages of the
    global ``block_table`` in order."""
    B = len(lens)
    sh_pages = [-(-int(n) // (n_shards * 64)) for n in lens]
    tails = [int(n) - (n_shards - 1) * 64 * sp for n, sp in zip(lens, sh_pages)]
    if min(tails) < T:
        raise ValueError("a history too short for this many shards")
    bt = block_table.cpu()

    def table(offsets, widths):
        t = torch.zeros((B, max(max(widths), 1)), dtype=torch.int32)
        for b in range(B):
            t[b, :widths[b]] = bt[b, offsets[b]:offsets[b] + widths[b]]
        return t

    plan = [(table([s * sp for sp in sh_pages], sh_pages),
             torch.tensor([64 * sp for sp in sh_pages], dtype=torch.int32)) for s in range(n_shards - 1)]
    plan.append((table([(n_shards - 1) * sp for sp in sh_pages], [-(-n // 64) for n in tails]),
                 torch.tensor(tails, dtype=torch.int32)))
    return plan


def gather_queries(q_local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather bf16 queries [B, T, H_local, 576] along the head dim: every rank
    returns [B, T, W * H_local, 576], rank r's heads at [r * H_local, ...)."""
    W = dist.get_world_size(group)
    parts = [torch.empty_like(q_local) for _ in range(W)]
    dist.all_gather(parts, q_local.contiguous(), group=group)
    return torch.cat(parts, dim=2).contiguous()


def gather_partials(out_s: torch.Tensor, lse_s: torch.Tensor, group=None):
    """All-gather every rank's partial answer over its shard: returns
    ([W, B, T, H, 512], [W, B, T, H]) stacked in rank order (the merge input)."""
    W = dist.get_world_size(group)
    outs = [torch.empty_like(out_s) for _ in range(W)]
    lses = [torch.empty_like(lse_s) for _ in range(W)]
    dist.all_gather(outs, out_s.contiguous(), group=group)
    dist.all_gather(lses, lse_s.contiguous(), group=group)
    return torch.stack(outs).contiguous(), torch.stack(lses).contiguous()


def local_shard_decode(cache, kv_scale, block_table, seq_lens, sm_scale, *, last_shard: bool, n_splits: int = 0,
                       stream=None) -> Callable:
    """The library's decode over this rank's shard, as the ``local_decode`` of
    ``dcp_decode``: q [B, T, H, 576] -> (out bf16 [B, T, H, 512], lse fp32 [B, T, H]).
    A shard before the last is decoded as T = 1 with T*H rows."""
    from . import _lib

    def run(q):
        B, T, H, _ = q.shape
        qq = q if (last_shard or T == 1) else q.reshape(B, 1, T * H, q.shape[-1])
        out = torch.empty((*qq.shape[:3], 512), dtype=torch.bfloat16, device=q.device)
        lse = torch.empty(qq.shape[:3], dtype=torch.float32, device=q.device)
        _lib.mla_decode_paged(qq, cache, kv_scale, block_table, seq_lens, n_splits, sm_scale, out, lse, stream)
        return out.reshape(B, T, H, 512), lse.reshape(B, T, H)

    return run


def library_merge(stream=None) -> Callable:
    """mla_merge_partials over the shard dim, as the ``merge`` of ``dcp_decode``."""
    from . import merge_partials

    def run(po, pl):
        return merge_partials(po, pl, stream=stream)

    return run


def dcp_decode(q_local: torch.Tensor, local_decode: Callable, merge: Callable, group=None, *,
               keep_local_heads: bool = True):
    """One DCP decode step (module docstring): gather the queries, decode the
    local shard, gather the partial answers, merge.  Returns (out, lse) for this
    rank's heads (or for all heads with keep_local_heads=False) and the gathered
    partials (for inspection)."""
    r = dist.get_rank(group)
    Hl = q_local.shape[2]
    q_all = gather_queries(q_local, group)
    out_s, lse_s = local_decode(q_all)
    po, pl = gather_partials(out_s, lse_s, group)
    out, lse = merge(po, pl)
    if keep_local_heads:
        out, lse = out[:, :, r * Hl:(r + 1) * Hl], lse[:, :, r * Hl:(r + 1) * Hl]
    return out, lse, (po, pl)
