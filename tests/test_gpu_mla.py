"""Sparse MLA decode on the GPU against the oracle, element by element, with
the tolerance of tests.parity.check_mla (derived from the kernel's
arithmetic; a_abs, d_abs and s_abs are the oracle's sum p |v|, sum p |v - out|
and largest score magnitude)."""

import numpy as np
import pytest
import torch

import oracle
from synth.inputs import to_e4m3fn_bytes
from synth.mla import MLA_DIM, MlaProblem, make_mla_problem, mla_config
from tests.parity import check_mla

pytestmark = pytest.mark.gpu


def run(lib, prob, *, ws=None):
    dev = "cuda"
    q = torch.from_numpy(prob.q.reshape(prob.rows, prob.heads, MLA_DIM)).to(dev)
    kv = torch.from_numpy(prob.kv).to(dev)
    idx = torch.from_numpy(prob.indices).to(dev)
    bt = torch.from_numpy(prob.block_tables).to(dev)
    if ws is None:
        ws = lib.mla_workspace(prob.rows)
    out, lse = lib.pmqa_sparse_mla_decode(q, kv, idx, bt, prob.next_n, prob.q_scale,
                                          prob.kv_scale, prob.sm_scale, want_lse=True, ws=ws)
    torch.cuda.synchronize()
    status = lib.pmqa_read_device_status(ws)
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), status


def check(out, lse, prob, rows=None):
    ref, lref, tol = oracle.sparse_mla(prob, rows=rows, want_tol=True)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    return check_mla(out, lse, ref, lref, tol)


@pytest.mark.parametrize("bs,nn,P,ctx,topk,kw", [
    (1, 1, 1, [300], 2048, {}),                               # one row, ragged last tile
    (2, 3, 1, [900, 3000], 512, dict(holes=0.1)),             # holes anywhere
    (2, 4, 1, [5000, 2049], 2048, dict(repeats=0.05)),        # repeated positions
    (3, 2, 64, [7000, 129, 4097], 1000, {}),                  # pages of 64, topk % 128 != 0
    (4, 1, 1, [0, 3, 1, 2500], 256, {}),                      # empty and tiny rows
    (2, 2, 48, [5000, 777], 1024, {}),                        # pages of 48: position / P divides
    (1, 3, 3, [2000], 512, dict(holes=0.05)),                 # pages of 3
])
def test_parity_small(cuda_lib, bs, nn, P, ctx, topk, kw):
    prob = make_mla_problem(bs, nn, 16, P, ctx, topk=topk, seed=sum(ctx) + topk, **kw)
    out, lse, status = run(cuda_lib, prob)
    assert status == 0
    check(out, lse, prob)


@pytest.mark.parametrize("scale", [4.0, 16.0])
def test_peaked_scores_move_the_running_maximum(cuda_lib, scale):
    """sm_scale 4x and 16x the default: scores spread over tens of units, so
    the reference maximum moves inside a row and O is rescaled in TMEM."""
    prob = make_mla_problem(4, 2, 16, 1, [6000, 3000, 9000, 2048], seed=int(scale),
                            sm_scale=scale * MLA_DIM ** -0.5)
    out, lse, status = run(cuda_lib, prob)
    assert status == 0
    check(out, lse, prob)


def test_increasing_scores_rescale_every_tile(cuda_lib):
    """Listed positions ordered so each tile's scores exceed the last by more
    than the rescale slack: O is rescaled at every tile of the row."""
    prob = make_mla_problem(1, 1, 16, 1, [2048], seed=11, sm_scale=8 * MLA_DIM ** -0.5)
    ref, _, _ = oracle.sparse_mla(prob)
    # order the row's positions by their head-0 score, lowest first
    qd = oracle.e4m3fn_table()[prob.q.reshape(16, MLA_DIM)[0].astype(np.int64)]
    kd = oracle.e4m3fn_table()[prob.kv[prob.block_tables[0, prob.indices[0]], 0].astype(np.int64)]
    prob.indices[0] = prob.indices[0][np.argsort(kd @ qd)]
    out, lse, status = run(cuda_lib, prob)
    assert status == 0
    check(out, lse, prob)


def test_zero_query_is_the_mean(cuda_lib):
    prob = make_mla_problem(2, 2, 16, 1, [3000, 700], seed=3)
    prob.q[:] = 0
    out, lse, status = run(cuda_lib, prob)
    assert status == 0
    check(out, lse, prob)
    n = (prob.indices >= 0).sum(axis=1)
    np.testing.assert_allclose(lse, np.log(n)[:, None].repeat(16, axis=1), rtol=0, atol=1e-5)


def test_one_dominant_position(cuda_lib):
    """One listed position scores 448 * 448 above the rest: its value row
    comes out (to bf16 rounding)."""
    prob = make_mla_problem(1, 1, 16, 1, [4000], topk=2048, seed=5)
    q = np.zeros((16, MLA_DIM), dtype=np.uint8)
    q[:, 0] = to_e4m3fn_bytes(np.array([448.0], dtype=np.float32))[0]
    prob.q[:] = q.reshape(prob.q.shape)
    slots = prob.block_tables[0, prob.indices[0]]
    prob.kv[slots, 0, 0] = 0
    prob.kv[slots[1500], 0, 0] = to_e4m3fn_bytes(np.array([448.0], dtype=np.float32))[0]
    prob.sm_scale = 1.0
    out, lse, status = run(cuda_lib, prob)
    assert status == 0
    check(out, lse, prob)


def test_rows_split_over_ctas(cuda_lib):
    """More rows than SMs (the tiles split evenly over the CTAs, rows cut at
    arbitrary tile boundaries, parts combined by the second kernel), a few
    rows (each row over the same number of CTAs), and rows held whole by one
    CTA each (no combine)."""
    for bs, nn, seed in ((60, 3, 1), (1, 4, 2), (37, 3, 3)):
        ctx = np.random.default_rng(seed).integers(2100, 9000, size=bs)
        prob = make_mla_problem(bs, nn, 16, 1, ctx, seed=seed)
        out, lse, status = run(cuda_lib, prob)
        assert status == 0
        check(out, lse, prob)


def test_workspace_is_reusable(cuda_lib):
    """The workspace carries nothing from one call to the next: three calls on
    one workspace agree bit for bit."""
    prob = make_mla_problem(9, 4, 16, 1, [4000] * 9, seed=8)
    ws = cuda_lib.mla_workspace(prob.rows)
    first = run(cuda_lib, prob, ws=ws)
    for _ in range(2):
        again = run(cuda_lib, prob, ws=ws)
        assert np.array_equal(again[0], first[0]) and np.array_equal(again[1], first[1])


def test_positions_outside_the_table_are_skipped_and_flagged(cuda_lib):
    prob = make_mla_problem(1, 2, 16, 1, [1000], topk=256, seed=4)
    bad = prob.indices.copy()
    bad[0, 7] = prob.max_blocks_per_seq + 5      # past the table
    prob_bad = MlaProblem(**{**prob.__dict__, "indices": bad})
    out, lse, status = run(cuda_lib, prob_bad)
    assert status & cuda_lib.PMQA_DEV_BAD_CONTEXT
    skipped = MlaProblem(**{**prob.__dict__, "indices": bad.copy()})
    skipped.indices[0, 7] = -1
    check(out, lse, skipped)


@pytest.mark.parametrize("name", ["M0", "M1", "M2"])
def test_workloads_sampled_rows(cuda_lib, name):
    """The full workloads in the benchmark's launch; the oracle checks a sample
    of rows (all rows of M0)."""
    prob = mla_config(name)
    out, lse, status = run(cuda_lib, prob)
    assert status == 0
    rng = np.random.default_rng(0)
    rows = None if prob.rows <= 8 else np.sort(rng.choice(prob.rows, 8, replace=False))
    _, cos_diff = check(out, lse, prob, rows=rows)
    assert cos_diff < 1e-4


def test_decode_over_the_indexers_top_k(cuda_lib):
    """The two steps of a decode chained: the fused indexer call selects each
    row's top-2048 positions, the decode attends to exactly those (a latent
    cache of the same requests and pages)."""
    from synth import make_problem

    ctx = [3000, 5000, 2500, 9000]
    ip = make_problem(4, 2, 64, 1, ctx, 9216, seed=6, table="perm", extra_blocks=2, k=2048)
    dq = torch.from_numpy(ip.q).cuda().view(torch.float8_e4m3fn)
    idx = cuda_lib.pmqa_logits_topk(dq, torch.from_numpy(ip.kv).cuda(),
                                    torch.from_numpy(ip.weights).cuda(),
                                    torch.from_numpy(ip.context_lens).cuda(),
                                    torch.from_numpy(ip.block_tables).cuda(), ip.max_model_len,
                                    ip.k)
    prob = make_mla_problem(4, 2, 16, 1, ctx, topk=2048, seed=7)
    prob.indices = idx.cpu().numpy()
    out, lse, status = run(cuda_lib, prob)
    assert status == 0
    check(out, lse, prob)


@pytest.mark.parametrize("slices,P", [(2, 1), (4, 1), (3, 16)])
def test_context_parallel_decode(cuda_lib, slices, P):
    """The decode split by context: each slice attends to its listed positions
    only, against a block table that maps only its pages (checked against the
    oracle with the listing restricted to the slice), and the LSE merge of the
    slices against the oracle's whole decode."""
    from sparse_attention_indexer_pmqa_gb300.context_parallel import slice_bounds, slice_table

    prob = make_mla_problem(3, 4, 16, P, [5000, 300, 9000], topk=2048, seed=12 + slices,
                            holes=0.05)
    dev = "cuda"
    q = torch.from_numpy(prob.q.reshape(prob.rows, prob.heads, MLA_DIM)).to(dev)
    kv = torch.from_numpy(prob.kv).to(dev)
    idx = torch.from_numpy(prob.indices).to(dev)
    outs, lses = [], []
    for rank in range(slices):
        b, e = slice_bounds(prob.context_lens, slices, rank)
        bt = torch.from_numpy(slice_table(prob.block_tables, b, e, P)).to(dev)
        ws = cuda_lib.mla_workspace(prob.rows)
        out, lse = cuda_lib.pmqa_sparse_mla_decode_range(
            q, kv, idx, bt, prob.next_n, prob.q_scale, prob.kv_scale, prob.sm_scale,
            torch.from_numpy(b).to(dev), torch.from_numpy(e).to(dev), ws=ws)
        torch.cuda.synchronize()
        assert cuda_lib.pmqa_read_device_status(ws) == 0  # no page outside the slice was read
        filt = prob.indices.copy()
        for r in range(prob.rows):
            i = r // prob.next_n
            outside = (filt[r] < b[i]) | (filt[r] >= e[i])
            filt[r][outside] = -1
        part = MlaProblem(**{**prob.__dict__, "indices": filt})
        check(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
              part)
        outs.append(out)
        lses.append(lse)
    mo, ml = cuda_lib.pmqa_sparse_mla_merge(torch.stack(outs), torch.stack(lses))
    torch.cuda.synchronize()
    ref, lref, tol = oracle.sparse_mla(prob, want_tol=True)
    check_mla(mo.float().cpu().numpy(), ml.cpu().numpy(), ref, lref, tol, parts=slices)
