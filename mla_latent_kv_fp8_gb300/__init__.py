"""GB300-native (sm_103a) MLA decode over a paged FP8 latent-KV cache.

The product is the C ABI library ``libmla_decode.so`` (include/mla_decode.h):
split-KV decode kernels on tcgen05 tensor cores and CUDA cores, the
log-sum-exp merge kernels and the FP8 latent-append kernel.  This package holds its sources (``csrc/``), the
in-tree build, the ctypes binding and the seeded synthetic input generators.
"""
from __future__ import annotations

import torch

from . import synth  # noqa: F401  (input generation only)


def _binding():
    from . import _lib
    return _lib


def decode(case, n_splits: int = 0, stream=None, out=None, lse=None):
    """Run mla_decode_paged on a synth.DecodeCase that lives on the GPU.

    Allocates ``out`` (bf16 [B,T,H,512]) and ``lse`` (fp32 [B,T,H]) with torch
    unless given; every step of the attention runs in the library's kernels."""
    b = _binding()
    B, T, H = case.q.shape[:3]
    if out is None:
        out = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device=case.q.device)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=case.q.device)
    b.mla_decode_paged(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                       n_splits, case.sm_scale, out, lse, stream)
    return out, lse


def merge_partials(partial_out, partial_lse, stream=None, out=None, lse=None):
    """Run mla_merge_partials over the leading (shard) dim of ``partial_out``
    (bf16 or fp32 [S, ..., 512]) and ``partial_lse`` (fp32 [S, ...])."""
    b = _binding()
    S = partial_out.shape[0]
    if out is None:
        out = torch.empty(partial_out.shape[1:], dtype=torch.bfloat16, device=partial_out.device)
    if lse is None:
        lse = torch.empty(partial_lse.shape[1:], dtype=torch.float32, device=partial_out.device)
    b.mla_merge_partials(partial_out, partial_lse, S, out, lse, stream)
    return out, lse
