"""Host side of the context-parallel split (CPU, no GPU): slice bounds, the
block table restricted to a slice, and the all-gather of the slices'
candidate lists over a two-rank gloo group, checked on oracle logits: the
top-k of the gathered union equals each row's top-k."""

import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import oracle
from sparse_attention_indexer_pmqa_gb300.context_parallel import (gather_lists, slice_bounds,
                                                                 slice_table)
from synth import make_problem
from tests.parity import valid_len


def test_slices_partition_every_context():
    ctx = np.array([0, 1, 2, 3, 127, 128, 129, 4097, 202751], dtype=np.int32)
    for world in (1, 2, 3, 4, 8):
        cover = np.zeros((len(ctx), int(ctx.max()) + 1), dtype=np.int32)
        prev_end = np.zeros(len(ctx), dtype=np.int64)
        for rank in range(world):
            b, e = slice_bounds(ctx, world, rank)
            assert np.all(b == prev_end) and np.all(e >= b)
            prev_end = e.astype(np.int64)
            for i in range(len(ctx)):
                cover[i, b[i]:e[i]] += 1
        assert np.array_equal(prev_end, ctx)
        for i, c in enumerate(ctx):
            assert np.all(cover[i, :c] == 1)


def test_slice_table_keeps_only_the_slice_pages():
    bt = np.arange(2 * 10, dtype=np.int32).reshape(2, 10) + 100
    b = np.array([5, 0], dtype=np.int32)
    e = np.array([17, 0], dtype=np.int32)
    t = slice_table(bt, b, e, 4)  # tokens 5..16 -> pages 1..4
    assert np.array_equal(t[0], [-1, 101, 102, 103, 104, -1, -1, -1, -1, -1])
    assert np.all(t[1] == -1)


def _topk_window(row64, lo, hi, k):
    """Positions of the k largest of row64[lo:hi] (value desc, position asc)."""
    pos = np.arange(lo, hi)
    order = np.lexsort((pos, -row64[lo:hi]))
    sel = pos[order[:k]]
    return sel, row64[sel]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    prob = make_problem(3, 2, 16, 16, [900, 40, 2500], 2560, seed=4, table="perm")
    _, r64, _ = oracle.logits(prob, want64=True)
    k = 300
    b, e = slice_bounds(prob.context_lens, world, rank)
    idx = np.full((prob.rows, k), -1, dtype=np.int32)
    val = np.full((prob.rows, k), -np.inf, dtype=np.float32)
    for r in range(prob.rows):
        i, j = divmod(r, prob.next_n)
        hi = max(int(b[i]), min(valid_len(int(prob.context_lens[i]), prob.next_n, j), int(e[i])))
        s, v = _topk_window(r64[r], int(b[i]), hi, k)
        idx[r, :len(s)], val[r, :len(s)] = s, v
    all_i, all_v = gather_lists(torch.from_numpy(idx), torch.from_numpy(val))
    out[rank] = (all_i.numpy(), all_v.numpy(), idx, val)
    torch.distributed.destroy_process_group()


def test_gather_over_gloo_and_the_union_top_k():
    world = 2
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    prob = make_problem(3, 2, 16, 16, [900, 40, 2500], 2560, seed=4, table="perm")
    _, r64, _ = oracle.logits(prob, want64=True)
    k = 300
    for rank in range(world):
        all_i, all_v, _, _ = res[rank]
        for src in range(world):  # rank order, the same on every rank
            assert np.array_equal(all_i[src], res[src][2])
            assert np.array_equal(all_v[src], res[src][3])
    all_i, all_v = res[0][0], res[0][1]
    for r in range(prob.rows):
        i, j = divmod(r, prob.next_n)
        n = valid_len(int(prob.context_lens[i]), prob.next_n, j)
        want, _ = _topk_window(r64[r], 0, n, k)
        cand = all_i[:, r, :].reshape(-1)
        cand = cand[cand >= 0]
        got, _ = _topk_window(np.where(np.isin(np.arange(r64.shape[1]), cand), r64[r], -np.inf),
                              0, n, min(k, n))
        assert np.array_equal(np.sort(got), np.sort(want))


def _mla_rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    from synth.mla import MlaProblem, make_mla_problem

    prob = make_mla_problem(2, 3, 16, 1, [1200, 700], topk=512, seed=5)
    b, e = slice_bounds(prob.context_lens, world, rank)
    filt = prob.indices.copy()
    for r in range(prob.rows):
        i = r // prob.next_n
        filt[r][(filt[r] < b[i]) | (filt[r] >= e[i])] = -1
    o, l, _ = oracle.sparse_mla(MlaProblem(**{**prob.__dict__, "indices": filt}))
    go = [torch.empty(o.shape, dtype=torch.float64) for _ in range(world)]
    gl = [torch.empty(l.shape, dtype=torch.float64) for _ in range(world)]
    torch.distributed.all_gather(go, torch.from_numpy(o))
    torch.distributed.all_gather(gl, torch.from_numpy(l))
    out[rank] = (torch.stack(go).numpy(), torch.stack(gl).numpy())
    torch.distributed.destroy_process_group()


def test_lse_merge_of_slice_decodes_over_gloo():
    """The decode split by context: each rank's oracle decode over the listed
    positions of its slice, gathered over a two-rank gloo group, merged by the
    slices' log-sum-exps (w_g = exp(lse_g - max), out = sum w_g out_g / sum w_g,
    lse = max + ln sum w_g), equals the oracle's whole decode."""
    from synth.mla import make_mla_problem

    world = 2
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_mla_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    outs, lses = res[0]
    assert np.array_equal(outs, res[1][0]) and np.array_equal(lses, res[1][1])
    M = lses.max(axis=0)
    w = np.where(np.isneginf(lses), 0.0, np.exp(lses - np.where(np.isneginf(M), 0.0, M)))
    L = w.sum(axis=0)
    merged = (w[..., None] * outs).sum(axis=0) / np.where(L > 0, L, 1.0)[..., None]
    lse = np.where(L > 0, M + np.log(np.where(L > 0, L, 1.0)), -np.inf)
    prob = make_mla_problem(2, 3, 16, 1, [1200, 700], topk=512, seed=5)
    ref, lref, _ = oracle.sparse_mla(prob)
    np.testing.assert_allclose(merged, ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lref, rtol=1e-12)
