"""Seeded synthetic problems for the sparse MLA decode that consumes the
indexer's top-k positions.

Layouts (the pages give the data types and head counts, not the widths; the
widths are the MLA layout of a 512-wide compressed KV plus a 64-wide rotary
key):

* q            uint8 [bs, next_n, heads, 576]  fp8 e4m3fn bit patterns
* kv           uint8 [num_blocks, block_size, 576]: one latent row per slot,
               fp8 e4m3fn; its first 512 values are also the value vector
* q_scale, kv_scale, sm_scale  Python floats (per-tensor fp8 scales and the
               softmax scale)
* indices      int32 [bs * next_n, topk]: positions in the row's request, -1
               for an empty entry
* context_lens int32 [bs]; block_tables int32 [bs, max_blocks_per_seq]

Value recipe: q and the latent rows are standard normal draws rounded to
e4m3fn (the indexer's recipe); q_scale 0.5, kv_scale 2.0 and sm_scale
576^-0.5, so a score is about a standard normal draw. A row lists
min(topk, valid_len) distinct positions of its causal window, drawn uniformly
and in random order (what the indexer's top-k returns on random logits), then
-1. Listed slots hold their own draws; the other slots of a request repeat a
block of 4096 drawn rows; slots that no request owns are poisoned with fp8
NaN bytes so an unmasked read shows up. Every draw comes from numpy's PCG64 seeded with
``seed``; the module holds none of the decode's arithmetic.
"""

from __future__ import annotations

import dataclasses

import numpy as np

from .inputs import FP8_NAN, to_e4m3fn_bytes

MLA_DIM = 576
MLA_VDIM = 512


@dataclasses.dataclass
class MlaProblem:
    q: np.ndarray
    kv: np.ndarray
    indices: np.ndarray
    context_lens: np.ndarray
    block_tables: np.ndarray
    q_scale: float
    kv_scale: float
    sm_scale: float
    bs: int
    next_n: int
    heads: int
    block_size: int
    name: str = "custom"

    @property
    def rows(self) -> int:
        return self.bs * self.next_n

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])

    @property
    def num_blocks(self) -> int:
        return int(self.kv.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def listed(self) -> int:
        """Listed (non -1) entries over all rows."""
        return int((self.indices >= 0).sum())


def valid_len(ctx: int, next_n: int, j: int) -> int:
    return max(0, min(ctx - next_n + j + 1, ctx))


def make_mla_problem(bs: int, next_n: int, heads: int, block_size: int, context_lens,
                     topk: int = 2048, *, seed: int = 0, q_scale: float = 0.5,
                     kv_scale: float = 2.0, sm_scale: float = MLA_DIM ** -0.5,
                     holes: float = 0.0, repeats: float = 0.0, extra_blocks: int = 2,
                     width: int | None = None, name: str = "custom",
                     rng: np.random.Generator | None = None) -> MlaProblem:
    """Draw one problem. ``holes``: fraction of listed entries replaced by -1
    anywhere in the row; ``repeats``: fraction replaced by a copy of another
    listed position of the same row. The pool holds ceil(ctx_i / P) +
    extra_blocks pages per request, owned in a random disjoint order."""
    rng = np.random.default_rng(seed) if rng is None else rng
    ctx = np.asarray(context_lens, dtype=np.int64).reshape(bs)
    P = block_size
    nblk = (ctx + P - 1) // P
    if width is None:
        width = int(max(1, nblk.max() if bs else 1))
    per = nblk + extra_blocks
    num_blocks = max(int(per.sum()), 1)
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((bs, width), -1, dtype=np.int32)
    off = 0
    for i in range(bs):
        tables[i, : nblk[i]] = perm[off: off + nblk[i]]
        off += int(per[i])
    q = to_e4m3fn_bytes(rng.standard_normal((bs, next_n, heads, MLA_DIM), dtype=np.float32))
    idx = np.full((bs * next_n, topk), -1, dtype=np.int32)
    for i in range(bs):
        for j in range(next_n):
            vl = valid_len(int(ctx[i]), next_n, j)
            n = min(topk, vl)
            if n == 0:
                continue
            row = rng.choice(vl, size=n, replace=False).astype(np.int32)
            if repeats > 0 and n > 1:
                rep = rng.random(n) < repeats
                row[rep] = row[rng.integers(0, n, size=int(rep.sum()))]
            if holes > 0:
                row[rng.random(n) < holes] = -1
            idx[i * next_n + j, :n] = row
    # Slots a row lists get their own draws; the other slots a request owns
    # repeat a block of drawn rows (no call reads them, but the pool keeps its
    # full size and spread); slots no request owns are poisoned.
    slots = num_blocks * P
    owner = np.full(slots, -1, dtype=np.int64)
    for i in range(bs):
        pages = tables[i, : nblk[i]].astype(np.int64)
        owner[(pages[:, None] * P + np.arange(P)[None, :]).reshape(-1)[: ctx[i]]] = i
    fill = to_e4m3fn_bytes(rng.standard_normal((min(slots, 4096), MLA_DIM), dtype=np.float32))
    kv = np.resize(fill, (slots, MLA_DIM))
    kv[owner < 0] = FP8_NAN
    listed = np.zeros(slots, dtype=bool)
    for r in range(bs * next_n):
        t = idx[r][idx[r] >= 0].astype(np.int64)
        pages = tables[r // next_n, t // P].astype(np.int64)
        listed[pages * P + t % P] = True
    sl = np.flatnonzero(listed)
    kv[sl] = to_e4m3fn_bytes(rng.standard_normal((sl.size, MLA_DIM), dtype=np.float32))
    return MlaProblem(q=q, kv=kv.reshape(num_blocks, P, MLA_DIM), indices=idx,
                      context_lens=ctx.astype(np.int32), block_tables=tables,
                      q_scale=float(q_scale), kv_scale=float(kv_scale),
                      sm_scale=float(sm_scale), bs=bs, next_n=next_n, heads=heads,
                      block_size=P, name=name)


# Workloads of the sparse MLA decode, 16 query heads, top-2048 positions:
# the pages' reproduction shape (one request of 8192 tokens, 4 query rows);
# the speculative-verify batch of the indexer (32 requests x 4 rows, contexts
# 16K-64K, pages of one token); a long-context batch on pages of 64 tokens.
MLA_CONFIGS = {
    "M0": dict(desc="bs1 nn4 H16 P1 ctx8192 top2048"),
    "M1": dict(desc="bs32 nn4 H16 P1 ctx~U[16384,65536] top2048"),
    "M2": dict(desc="bs8 nn2 H16 P64 ctx=131072+U[0,71679] top2048"),
}


def mla_config(name: str, seed: int = 0) -> MlaProblem:
    rng = np.random.default_rng(seed)
    if name == "M0":
        return make_mla_problem(1, 4, 16, 1, [8192], rng=rng, name=name)
    if name == "M1":
        ctx = rng.integers(16384, 65536, size=32, endpoint=True)
        return make_mla_problem(32, 4, 16, 1, ctx, rng=rng, name=name)
    if name == "M2":
        ctx = 131072 + rng.integers(0, 71679, size=8, endpoint=True)
        return make_mla_problem(8, 2, 16, 64, ctx, rng=rng, name=name)
    raise KeyError(name)
