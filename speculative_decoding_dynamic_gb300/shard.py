"""Stage 1 and greedy verification over a vocabulary split across processes.

When the LM head is split by vocabulary rows over several GPUs, each rank
holds a slice of every logit row. Each rank runs eagle_shard_partials on its
slice, the partials (k keys and two floats per row) are all-gathered, and
every rank runs eagle_shard_merge on the gathered partials; eagle_expand_topk
and eagle_verify_argmax continue from the merged results. Every step runs in
libeagle's kernels; this module only computes slice bounds and moves buffers
(torch.distributed: NCCL for CUDA tensors, gloo for host tensors).
"""
from __future__ import annotations

import torch

KEYS_PER_ROW = 16  # width of a partial's key list (the library's largest top-k)


def slice_bounds(vocab: int, n_shards: int, esize: int) -> list[tuple[int, int]]:
    """(offset, size) of each rank's slice: contiguous, every offset on a
    16-byte boundary (a multiple of 16 / esize entries), the last slice takes
    the rest."""
    if n_shards < 1 or vocab < n_shards:
        raise ValueError("need 1 <= n_shards <= vocab")
    unit = 16 // esize
    per = -(-vocab // n_shards)
    per = -(-per // unit) * unit
    out = []
    for r in range(n_shards):
        lo = min(vocab, r * per)
        hi = min(vocab, lo + per) if r < n_shards - 1 else vocab
        out.append((lo, hi - lo))
    if any(n <= 0 for _, n in out):
        raise ValueError("too many slices for this vocabulary")
    return out


def all_gather_partials(part_max_sum: torch.Tensor, part_keys: torch.Tensor, group=None):
    """The exchange: every rank's ([rows, 2] fp32, [rows, 16] 64-bit keys)
    partials to every rank, stacked in rank order as ([S, rows, 2], [S, rows, 16])."""
    import torch.distributed as dist
    S = dist.get_world_size(group)
    keys = part_keys.view(torch.int64)
    ms_all = torch.empty((S,) + tuple(part_max_sum.shape), dtype=part_max_sum.dtype, device=part_max_sum.device)
    keys_all = torch.empty((S,) + tuple(keys.shape), dtype=keys.dtype, device=keys.device)
    dist.all_gather(list(ms_all.unbind(0)), part_max_sum.contiguous(), group=group)
    dist.all_gather(list(keys_all.unbind(0)), keys.contiguous(), group=group)
    return ms_all, keys_all


def sharded_stage1(E, cfg, ws, logits_slice: torch.Tensor, vocab_offset: int, group=None, stream=None):
    """Partials of this rank's slice, the exchange, and the merge.

    logits_slice: [rows, shard_vocab] CUDA tensor of this rank's slice.
    Returns (row_lse [rows], topk_ids [rows, k], topk_logits [rows, k], row_argmax [rows])."""
    import torch.distributed as dist
    rows, sv = logits_slice.shape
    dev = logits_slice.device
    ms = torch.empty(rows, 2, dtype=torch.float32, device=dev)
    keys = torch.empty(rows, KEYS_PER_ROW, dtype=torch.int64, device=dev)
    E.eagle_shard_partials(cfg, ws, rows, sv, vocab_offset, logits_slice, ms, keys, stream)
    ms_all, keys_all = all_gather_partials(ms, keys, group)
    S = dist.get_world_size(group)
    k = cfg.top_k
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    ids = torch.empty(rows, k, dtype=torch.int32, device=dev)
    vals = torch.empty(rows, k, dtype=torch.float32, device=dev)
    arg = torch.empty(rows, dtype=torch.int32, device=dev)
    E.eagle_shard_merge(cfg, ws, S, rows, ms_all, keys_all, lse, ids, vals, arg, stream)
    return lse, ids, vals, arg
