"""Context-parallel split of the indexer, run on one GPU.

Each of G slices of every request's tokens is scored and selected by
pmqa_logits_topk_range against a block table that holds only the pages of that
slice (every other entry -1), as a GPU that keeps only its slice's cache would
have; pmqa_topk_merge then combines the G lists. The merged top-k must equal
the oracle's top-k of the whole row (up to swaps within the tolerance of the
k-th value), and each slice's list the oracle's top-k of that slice.
"""

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_pmqa_gb300.context_parallel import slice_bounds, slice_table
from synth import make_problem
from tests.parity import check_topk_rows

pytestmark = pytest.mark.gpu

CASES = [
    # bs, next_n, heads, block_size, context lengths, max_model_len
    (3, 1, 64, 1, [3000, 5000, 129], 5120),
    (2, 4, 64, 1, [4100, 700], 5120),
    (3, 2, 64, 64, [5000, 2100, 130], 5120),
    (2, 3, 32, 16, [2600, 45], 2816),
    (4, 1, 128, 3, [1, 0, 2500, 777], 2560),
]


def dev(prob, bt=None):
    return dict(q=torch.from_numpy(prob.q).cuda().view(torch.float8_e4m3fn),
                kv=torch.from_numpy(prob.kv).cuda(), w=torch.from_numpy(prob.weights).cuda(),
                ctx=torch.from_numpy(prob.context_lens).cuda(),
                bt=torch.from_numpy(prob.block_tables if bt is None else bt).cuda())


@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("k", [100, 2048])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"bs{c[0]}nn{c[1]}H{c[2]}P{c[3]}")
def test_slices_then_merge_give_the_rows_top_k(cuda_lib, case, G, k):
    bs, nn, H, P, ctx, mml = case
    prob = make_problem(bs, nn, H, P, ctx, mml, seed=sum(ctx) + G, table="perm", extra_blocks=2)
    _, r64, tol = oracle.logits(prob, want64=True, want_tol=True)
    ws = cuda_lib.workspace(bs, nn, mml, k, cuda_lib.PMQA_OP_LOGITS_TOPK)
    lists_i, lists_v = [], []
    for rank in range(G):
        begin, end = slice_bounds(prob.context_lens, G, rank)
        d = dev(prob, slice_table(prob.block_tables, begin, end, P))
        b_t = torch.from_numpy(begin).cuda()
        e_t = torch.from_numpy(end).cuda()
        idx, vals = cuda_lib.pmqa_logits_topk_range(d["q"], d["kv"], d["w"], d["ctx"], d["bt"],
                                                    mml, k, b_t, e_t, want_vals=True, ws=ws)
        torch.cuda.synchronize()
        # no entry outside the slice was read (they are -1 in this table)
        assert cuda_lib.pmqa_read_device_status(ws) == 0
        gi, gv = idx.cpu().numpy(), vals.cpu().numpy()
        check_topk_rows(gi, r64, tol, prob.context_lens, nn, k, vals=gv, begin=begin, end=end)
        lists_i.append(idx)
        lists_v.append(vals)
    mi, mv = cuda_lib.pmqa_topk_merge(torch.stack(lists_i), torch.stack(lists_v), k,
                                      want_vals=True)
    torch.cuda.synchronize()
    check_topk_rows(mi.cpu().numpy(), r64, tol, prob.context_lens, nn, k, vals=mv.cpu().numpy())


def test_whole_range_equals_the_fused_call(cuda_lib):
    prob = make_problem(3, 2, 64, 16, [3000, 40, 2049], 3072, seed=8, table="perm", extra_blocks=2)
    d = dev(prob)
    k = 2048
    i_f, v_f = cuda_lib.pmqa_logits_topk(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], 3072, k,
                                         want_vals=True)
    begin = torch.zeros(3, dtype=torch.int32, device="cuda")
    end = d["ctx"].clone()
    i_r, v_r = cuda_lib.pmqa_logits_topk_range(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], 3072, k,
                                               begin, end, want_vals=True)
    torch.cuda.synchronize()
    i_f, v_f, i_r, v_r = (t.cpu().numpy() for t in (i_f, v_f, i_r, v_r))
    for r in range(prob.rows):
        o_f, o_r = np.argsort(i_f[r]), np.argsort(i_r[r])
        assert np.array_equal(i_f[r][o_f], i_r[r][o_r])
        assert np.array_equal(v_f[r][o_f], v_r[r][o_r])


def test_empty_and_clamped_slices(cuda_lib):
    """Slices that are empty, reversed or reach outside [0, ctx) clamp to it."""
    prob = make_problem(4, 2, 64, 1, [500, 300, 800, 64], 1024, seed=12, table="perm")
    _, r64, tol = oracle.logits(prob, want64=True, want_tol=True)
    d = dev(prob)
    begin = np.array([100, 300, -50, 40], dtype=np.int32)
    end = np.array([100, 200, 5000, 64], dtype=np.int32)
    idx, vals = cuda_lib.pmqa_logits_topk_range(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], 1024,
                                                64, torch.from_numpy(begin).cuda(),
                                                torch.from_numpy(end).cuda(), want_vals=True)
    torch.cuda.synchronize()
    idx, vals = idx.cpu().numpy(), vals.cpu().numpy()
    assert np.all(idx[0:4] == -1) and np.all(np.isneginf(vals[0:4]))  # empty and reversed
    check_topk_rows(idx, r64, tol, prob.context_lens, 2, 64, vals=vals,
                    begin=np.clip(begin, 0, prob.context_lens),
                    end=np.maximum(np.clip(begin, 0, prob.context_lens),
                                   np.clip(end, 0, prob.context_lens)))


@pytest.mark.parametrize("ties", [False, True])
def test_merge_of_given_lists(cuda_lib, ties):
    """The merge alone, on lists with empty slots and (optionally) many equal
    values: the chosen values equal the largest ones of the union."""
    rng = np.random.default_rng(3 + ties)
    lists, rows, k_in, k = 3, 5, 700, 512
    vals = (rng.integers(-8, 8, size=(lists, rows, k_in)) * 0.5 if ties
            else rng.standard_normal((lists, rows, k_in))).astype(np.float32)
    idx = np.arange(lists * rows * k_in, dtype=np.int32).reshape(lists, rows, k_in)
    idx[:, 2, 100:] = -1  # row 2: 300 valid candidates < k
    idx[:, 4, :] = -1     # row 4: none
    mi, mv = torch.from_numpy(idx).cuda(), torch.from_numpy(vals).cuda()
    oi, ov = cuda_lib.pmqa_topk_merge(mi, mv, k, want_vals=True)
    torch.cuda.synchronize()
    oi, ov = oi.cpu().numpy(), ov.cpu().numpy()
    for r in range(rows):
        valid = idx[:, r, :] >= 0
        pool = vals[:, r, :][valid]
        ke = min(k, pool.size)
        assert np.all(oi[r, ke:] == -1) and np.all(np.isneginf(ov[r, ke:]))
        sel = oi[r, :ke]
        assert len(np.unique(sel)) == ke
        flat = {int(p): float(v) for p, v in zip(idx[:, r, :][valid], pool)}
        got = np.sort([flat[int(p)] for p in sel])[::-1]
        assert np.array_equal(got, np.sort(pool)[::-1][:ke])
        assert np.array_equal(np.sort(ov[r, :ke])[::-1], got)
