"""Context-parallel split of the indexer over GPUs (host side).

Each GPU holds a contiguous slice of every request's tokens, scores and
selects inside it (pmqa_logits_topk_range), the slices' top-k lists of
(position, logit) are all-gathered, and every GPU merges them
(pmqa_topk_merge) into the rows' top-k: each of a row's k largest logits lies
in its own slice's top-k, so the union's top-k is the row's top-k. The pages
name decode context parallelism (DCP) among the configurations of the
sparse-MLA decode path (page "[Bug][ROCm]: ROCM_AITER_MLA can select an aiter
MLA decode kernel that silently returns uncorrelated output", chat-gpts.plus
summary, closing notes); the split itself is this library's design.

The same split serves the sparse MLA decode that consumes the top-k: each GPU
attends only to the listed positions inside its slice
(pmqa_sparse_mla_decode_range), the slices' outputs and log-sum-exps are
all-gathered, and every GPU merges them by their LSE (pmqa_sparse_mla_merge);
the pages name the LSE output as what decode context parallelism uses.

The functions here only compute slice bounds, restrict a block table to a
slice's pages and move the candidate lists and partial outputs between
processes; every step of the computation runs in the library's kernels.
"""

from __future__ import annotations

import numpy as np

from . import pmqa


def slice_bounds(context_lens, world: int, rank: int):
    """Tokens [begin_i, end_i) of request i held by `rank` of `world`: equal
    contiguous slices, begin_i = floor(rank * ctx_i / world)."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    begin = (rank * ctx) // world
    end = ((rank + 1) * ctx) // world
    return begin.astype(np.int32), end.astype(np.int32)


def slice_table(block_tables, begin, end, block_size: int) -> np.ndarray:
    """A copy of block_tables [bs, W] keeping only the entries of pages that
    hold tokens of [begin_i, end_i); every other entry is -1, as on a GPU that
    stores only its slice of the cache."""
    bt = np.asarray(block_tables)
    out = np.full_like(bt, -1)
    for i in range(bt.shape[0]):
        b, e = int(begin[i]), int(end[i])
        if e > b:
            p0, p1 = b // block_size, (e - 1) // block_size + 1
            out[i, p0:p1] = bt[i, p0:p1]
    return out


def gather_lists(idx, vals, group=None):
    """All-gather of every rank's [rows, k] candidate lists into
    [world, rows, k] tensors, in rank order (torch.distributed: NCCL between
    GPUs, gloo on the host)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    out_i = [torch.empty_like(idx) for _ in range(world)]
    out_v = [torch.empty_like(vals) for _ in range(world)]
    dist.all_gather(out_i, idx.contiguous(), group=group)
    dist.all_gather(out_v, vals.contiguous(), group=group)
    return torch.stack(out_i), torch.stack(out_v)


def cp_topk(q, kv_cache, weights, context_lens, block_tables, max_model_len: int, k: int,
            token_begin, token_end, *, group=None, ws=None, stream=None):
    """One context-parallel step on this rank: the slice's top-k, the
    all-gather of every rank's lists, the merge. Returns (idx, vals) [rows, k]
    of the whole rows, the same on every rank."""
    idx, vals = pmqa.pmqa_logits_topk_range(q, kv_cache, weights, context_lens, block_tables,
                                            max_model_len, k, token_begin, token_end,
                                            want_vals=True, ws=ws, stream=stream)
    all_i, all_v = gather_lists(idx, vals, group)
    return pmqa.pmqa_topk_merge(all_i, all_v, k, want_vals=True, stream=stream)


def gather_parts(out, lse, group=None):
    """All-gather of every rank's partial decode: out [rows, heads, 512] (bf16,
    moved as its 16-bit patterns) and lse [rows, heads] into [world, ...]
    tensors in rank order."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    bits = out.contiguous().view(torch.int16)
    out_b = [torch.empty_like(bits) for _ in range(world)]
    out_l = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(out_b, bits, group=group)
    dist.all_gather(out_l, lse.contiguous(), group=group)
    return torch.stack(out_b).view(torch.bfloat16), torch.stack(out_l)


def cp_mla_decode(q, kv_cache, indices, block_tables, next_n: int, q_scale: float,
                  kv_scale: float, sm_scale: float, token_begin, token_end, *, group=None,
                  ws=None, stream=None):
    """One context-parallel decode step on this rank: the slice's partial
    decode, the all-gather of every rank's (out, lse), the merge. Returns
    (out, lse) of the whole rows, the same on every rank."""
    out, lse = pmqa.pmqa_sparse_mla_decode_range(q, kv_cache, indices, block_tables, next_n,
                                                 q_scale, kv_scale, sm_scale, token_begin,
                                                 token_end, ws=ws, stream=stream)
    outs, lses = gather_parts(out, lse, group)
    return pmqa.pmqa_sparse_mla_merge(outs, lses, stream=stream)
