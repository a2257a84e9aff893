"""Seeded synthetic problems for the FP8 paged MQA-logits indexer.

Layouts follow the problem statement on the page "[Bug] aiter ops triton
attention pa" (stepcodex.com), section "Minimal reproduction":

* q            uint8 [bs, next_n, heads, 128]   fp8 e4m3fn bit patterns
* kv           uint8 [num_blocks, block_size, 132]: per token 128 fp8 e4m3fn
               bytes, then the 4 little-endian bytes of an fp32 scale
* weights      float32 [bs*next_n, heads]
* context_lens int32 [bs]
* block_tables int32 [bs, max_blocks_per_seq]

Value recipe (the same for every workload): q and K are standard normal draws
rounded to e4m3fn, scales are U[0.01, 0.1] fp32, weights are standard normal
fp32. Every draw comes from numpy's PCG64 seeded with ``seed``. Pool slots,
page tails and table entries that no request may read are poisoned (fp8 NaN
bytes, NaN scale, table entry -1) so that an unmasked read shows up.

The fp32 -> e4m3fn rounding of the draws is torch's cast (round to nearest
even); values are clamped to +-448 first, which standard normal draws never
reach.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

HEAD_DIM = 128
ROW_BYTES = HEAD_DIM + 4
FP8_NAN = 0x7F
F32_NAN_LE = np.array([0x00, 0x00, 0xC0, 0x7F], dtype=np.uint8)


@dataclasses.dataclass
class Problem:
    q: np.ndarray
    kv: np.ndarray
    weights: np.ndarray
    context_lens: np.ndarray
    block_tables: np.ndarray
    bs: int
    next_n: int
    heads: int
    block_size: int
    max_model_len: int
    k: int = 2048
    name: str = "custom"

    @property
    def head_dim(self) -> int:
        return HEAD_DIM

    @property
    def num_blocks(self) -> int:
        return int(self.kv.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def rows(self) -> int:
        return self.bs * self.next_n

    @property
    def total_ctx(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())


def to_e4m3fn_bytes(x: np.ndarray) -> np.ndarray:
    """Round float32 values to fp8 e4m3fn and return the bit patterns."""
    t = torch.from_numpy(np.clip(x, -448.0, 448.0).astype(np.float32, copy=False))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pack_kv(k_bytes: np.ndarray, scales: np.ndarray, block_size: int) -> np.ndarray:
    """Pack [slots,128] fp8 bytes and [slots] fp32 scales into [blocks, P, 132]."""
    slots = k_bytes.shape[0]
    assert slots % block_size == 0
    kv = np.empty((slots, ROW_BYTES), dtype=np.uint8)
    kv[:, :HEAD_DIM] = k_bytes
    kv[:, HEAD_DIM:] = scales.astype("<f4").view(np.uint8).reshape(slots, 4)
    return kv.reshape(slots // block_size, block_size, ROW_BYTES)


def make_problem(
    bs: int,
    next_n: int,
    heads: int,
    block_size: int,
    context_lens,
    max_model_len: int,
    *,
    seed: int = 0,
    table: str = "perm",
    extra_blocks: int = 0,
    width: int | None = None,
    k: int = 2048,
    scale_range=(0.01, 0.1),
    poison: bool = True,
    name: str = "custom",
    rng: np.random.Generator | None = None,
) -> Problem:
    """Draw one problem.

    table = "identity": request i owns the next ceil(ctx_i/P) blocks in order.
    table = "perm":     the pool holds sum(ceil(ctx_i/P) + extra_blocks) blocks
                        and each request owns a disjoint random set of them.
    table = "perm_full": bs == 1; the pool holds ``width`` blocks and the table
                        row is a random permutation of the whole pool.
    extra_blocks is per request for "perm" and a pool total for "identity".
    """
    rng = np.random.default_rng(seed) if rng is None else rng
    ctx = np.asarray(context_lens, dtype=np.int64).reshape(bs)
    P = block_size
    nblk = (ctx + P - 1) // P
    if width is None:
        width = max(1, -(-max_model_len // P))
    tables = np.full((bs, width), -1, dtype=np.int32)
    if table == "identity":
        num_blocks = int(nblk.sum()) + extra_blocks
        off = 0
        for i in range(bs):
            n = int(nblk[i])
            tables[i, :n] = np.arange(off, off + n, dtype=np.int32)
            off += n
        if bs == 1:
            tables[0, :] = np.arange(width, dtype=np.int32) % max(num_blocks, 1)
    elif table == "perm":
        per = nblk + extra_blocks
        num_blocks = int(per.sum())
        perm = rng.permutation(num_blocks).astype(np.int32)
        off = 0
        for i in range(bs):
            n = int(nblk[i])
            tables[i, :n] = perm[off:off + n]
            off += int(per[i])
    elif table == "perm_full":
        assert bs == 1
        num_blocks = width
        tables[0, :] = rng.permutation(num_blocks).astype(np.int32)
    else:
        raise ValueError(table)
    num_blocks = max(num_blocks, 1)

    q = to_e4m3fn_bytes(rng.standard_normal((bs, next_n, heads, HEAD_DIM), dtype=np.float32))
    slots = num_blocks * P
    k_bytes = to_e4m3fn_bytes(rng.standard_normal((slots, HEAD_DIM), dtype=np.float32))
    lo, hi = scale_range
    scales = rng.uniform(lo, hi, size=slots).astype(np.float32)
    weights = rng.standard_normal((bs * next_n, heads), dtype=np.float32)
    kv = pack_kv(k_bytes, scales, P)

    if poison:
        used = np.zeros(slots, dtype=bool)
        for i in range(bs):
            c = int(ctx[i])
            if c == 0:
                continue
            blocks = tables[i, : int(nblk[i])].astype(np.int64)
            tok = (blocks[:, None] * P + np.arange(P)[None, :]).reshape(-1)[:c]
            used[tok] = True
        flat = kv.reshape(slots, ROW_BYTES)
        flat[~used, :HEAD_DIM] = FP8_NAN
        flat[~used, HEAD_DIM:] = F32_NAN_LE

    return Problem(
        q=q, kv=kv, weights=weights, context_lens=ctx.astype(np.int32),
        block_tables=tables, bs=bs, next_n=next_n, heads=heads, block_size=P,
        max_model_len=max_model_len, k=k, name=name,
    )


# The five workloads, in order: single request at ctx 3000 with an identity
# table; single request at ctx 8192 on a shuffled pool; batch decode; speculative
# verify with four draft rows; long-context paged decode with a partial last page.
CONFIGS = {
    "C0": dict(desc="bs1 nn1 H32 P1 ctx3000 identity-table mml4096"),
    "C1": dict(desc="bs1 nn1 H64 P1 ctx8192 shuffled-8208-slot-pool mml16384"),
    "C2": dict(desc="bs64 nn1 H64 P1 ctx~U[4096,32768] shuffled-pool mml32768"),
    "C3": dict(desc="bs32 nn4 H64 P1 ctx~U[16384,65536] shuffled-pool mml65536"),
    "C4": dict(desc="bs8 nn2 H64 P64 ctx=131072+U[0,71679] shuffled-pages mml202752"),
}


def config_problem(name: str, seed: int = 0) -> Problem:
    rng = np.random.default_rng(seed)
    if name == "C0":
        return make_problem(1, 1, 32, 1, [3000], 4096, table="identity",
                            extra_blocks=16, width=3016, rng=rng, name=name)
    if name == "C1":
        return make_problem(1, 1, 64, 1, [8192], 16384, table="perm_full",
                            width=8208, rng=rng, name=name)
    if name == "C2":
        ctx = rng.integers(4096, 32768, size=64, endpoint=True)
        return _pool_problem(64, 1, 1, ctx, 32768, 1024, rng, name)
    if name == "C3":
        ctx = rng.integers(16384, 65536, size=32, endpoint=True)
        return _pool_problem(32, 4, 1, ctx, 65536, 1024, rng, name)
    if name == "C4":
        ctx = 131072 + rng.integers(0, 71679, size=8, endpoint=True)
        return make_problem(8, 2, 64, 64, ctx, 202752, table="perm",
                            extra_blocks=4, rng=rng, name=name)
    raise KeyError(name)


def _pool_problem(bs, next_n, P, ctx, mml, spare_slots, rng, name):
    """Block size 1 on a shared pool of sum(ctx)+spare slots, disjoint shuffled."""
    total = int(np.asarray(ctx, dtype=np.int64).sum())
    # Spread the spare slots over the requests so the pool is sum(ctx)+spare.
    extra = np.zeros(bs, dtype=np.int64)
    extra[: spare_slots % bs] = 1
    extra += spare_slots // bs
    prob = _perm_with_extra(bs, next_n, 64, P, ctx, mml, extra, rng, name)
    assert prob.num_blocks == total + spare_slots
    return prob


def _perm_with_extra(bs, next_n, heads, P, ctx, mml, extra, rng, name):
    ctx = np.asarray(ctx, dtype=np.int64)
    nblk = (ctx + P - 1) // P
    per = nblk + extra
    num_blocks = int(per.sum())
    width = -(-mml // P)
    tables = np.full((bs, width), -1, dtype=np.int32)
    perm = rng.permutation(num_blocks).astype(np.int32)
    off = 0
    for i in range(bs):
        tables[i, : nblk[i]] = perm[off: off + nblk[i]]
        off += int(per[i])
    q = to_e4m3fn_bytes(rng.standard_normal((bs, next_n, heads, HEAD_DIM), dtype=np.float32))
    slots = num_blocks * P
    k_bytes = to_e4m3fn_bytes(rng.standard_normal((slots, HEAD_DIM), dtype=np.float32))
    scales = rng.uniform(0.01, 0.1, size=slots).astype(np.float32)
    weights = rng.standard_normal((bs * next_n, heads), dtype=np.float32)
    kv = pack_kv(k_bytes, scales, P)
    used = np.zeros(slots, dtype=bool)
    for i in range(bs):
        used[tables[i, : nblk[i]].astype(np.int64)] = True
    flat = kv.reshape(slots, ROW_BYTES)
    flat[~used, :HEAD_DIM] = FP8_NAN
    flat[~used, HEAD_DIM:] = F32_NAN_LE
    return Problem(q=q, kv=kv, weights=weights, context_lens=ctx.astype(np.int32),
                   block_tables=tables, bs=bs, next_n=next_n, heads=heads,
                   block_size=P, max_model_len=mml, k=2048, name=name)


def random_logits(rows: int, width: int, *, seed: int = 0, ties: bool = False) -> np.ndarray:
    """Random fp32 rows [rows, width] to exercise a stand-alone top-k.

    Every entry is finite, including those a top-k must ignore. With ``ties``
    the values come from a set of 64 so that many entries compare equal.
    """
    rng = np.random.default_rng(seed)
    if ties:
        return rng.integers(-32, 32, size=(rows, width)).astype(np.float32) * 0.25
    return rng.standard_normal((rows, width), dtype=np.float32)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [
    "HEAD_DIM", "ROW_BYTES", "Problem", "make_problem", "config_problem", "CONFIGS",
    "pack_kv", "to_e4m3fn_bytes", "random_logits", "ceil_div",
]


# ---------------------------------------------------------------- prefill


@dataclasses.dataclass
class PrefillProblem:
    """Non-paged (prefill) indexer problem.

    * q        uint8 [m, heads, 128]  fp8 e4m3fn bit patterns
    * k        uint8 [n, 128]         fp8 e4m3fn bit patterns
    * k_scale  float32 [n]
    * weights  float32 [m, heads]
    * ks, ke   int32 [m]: query row r reads keys ks[r] <= t < ke[r]
    """
    q: np.ndarray
    k: np.ndarray
    k_scale: np.ndarray
    weights: np.ndarray
    ks: np.ndarray
    ke: np.ndarray
    heads: int
    name: str = "custom"

    @property
    def m(self) -> int:
        return int(self.q.shape[0])

    @property
    def n(self) -> int:
        return int(self.k.shape[0])

    @property
    def pairs(self) -> int:
        """(query row, key) pairs inside the rows' ranges."""
        lo = np.clip(self.ks.astype(np.int64), 0, self.n)
        hi = np.clip(self.ke.astype(np.int64), 0, self.n)
        return int(np.maximum(hi - lo, 0).sum())


def prefill_ranges(m: int, n: int, kind: str, rng: np.random.Generator, segments: int = 4):
    """Key ranges [ks, ke) of m query rows over n keys.

    causal:  the query rows are the last m positions of one sequence of n
             tokens; row r reads keys 0 .. n - m + r.
    packed:  ``segments`` sequences packed back to back (query and key position
             p are the same token, so m == n); row r reads from its sequence's
             start up to itself.
    random:  independent ranges, some empty, some reaching outside [0, n).
    full:    every row reads every key.
    """
    if kind == "causal":
        ke = n - m + np.arange(m, dtype=np.int64) + 1
        ks = np.zeros(m, dtype=np.int64)
        ke = np.clip(ke, 0, None)
    elif kind == "packed":
        assert m == n
        cuts = np.sort(rng.choice(np.arange(1, n), size=min(segments - 1, max(n - 1, 0)),
                                  replace=False)) if n > 1 else np.zeros(0, dtype=np.int64)
        starts = np.concatenate([[0], cuts]).astype(np.int64)
        seg = np.searchsorted(starts, np.arange(n), side="right") - 1
        ks = starts[seg]
        ke = np.arange(n, dtype=np.int64) + 1
    elif kind == "random":
        a = rng.integers(-8, n + 8, size=m)
        b = rng.integers(-8, n + 8, size=m)
        ks, ke = np.minimum(a, b), np.maximum(a, b)
        empty = rng.random(m) < 0.1
        ke[empty] = ks[empty]
    elif kind == "full":
        ks = np.zeros(m, dtype=np.int64)
        ke = np.full(m, n, dtype=np.int64)
    else:
        raise ValueError(kind)
    return ks.astype(np.int32), ke.astype(np.int32)


def make_prefill(m: int, n: int, heads: int, *, ranges: str = "causal", seed: int = 0,
                 poison: bool = True, scale_range=(0.01, 0.1), name: str = "custom",
                 rng: np.random.Generator | None = None) -> PrefillProblem:
    """Draw one prefill problem with the decode recipe's value distributions.

    Keys that no row's range covers are poisoned (fp8 NaN bytes, NaN scale)."""
    rng = np.random.default_rng(seed) if rng is None else rng
    q = to_e4m3fn_bytes(rng.standard_normal((m, heads, HEAD_DIM), dtype=np.float32))
    k = to_e4m3fn_bytes(rng.standard_normal((n, HEAD_DIM), dtype=np.float32))
    lo, hi = scale_range
    k_scale = rng.uniform(lo, hi, size=n).astype(np.float32)
    weights = rng.standard_normal((m, heads), dtype=np.float32)
    ks, ke = prefill_ranges(m, n, ranges, rng)
    if poison and n > 0:
        cover = np.zeros(n + 1, dtype=np.int64)
        a = np.clip(ks.astype(np.int64), 0, n)
        b = np.clip(ke.astype(np.int64), 0, n)
        keep = b > a
        np.add.at(cover, a[keep], 1)
        np.add.at(cover, b[keep], -1)
        unused = np.cumsum(cover)[:n] == 0
        k[unused] = FP8_NAN
        k_scale[unused] = np.float32("nan")
    return PrefillProblem(q=q, k=k, k_scale=k_scale, weights=weights, ks=ks, ke=ke,
                          heads=heads, name=name)


# Prefill workloads: the query rows are the last M positions of an N-token
# sequence (causal ranges), heads 32, head dimension 128.
PREFILL_CONFIGS = {
    "PF0": dict(desc="prefill M512 N1024 H32 causal", m=512, n=1024, heads=32),
    "PF1": dict(desc="prefill M4096 N8192 H32 causal", m=4096, n=8192, heads=32),
}


def prefill_config(name: str, seed: int = 0) -> PrefillProblem:
    c = PREFILL_CONFIGS[name]
    return make_prefill(c["m"], c["n"], c["heads"], ranges="causal", seed=seed, name=name)
