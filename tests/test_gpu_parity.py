"""GPU parity: libpmqa (through its C ABI) against the CPU oracle.

Logits: -inf pattern bit-exact, finite entries within 1e-3 (1 + sum_h |w_h||x_h|).
Top-k: index sets equal up to swaps inside the tolerance of the k-th value.
Sizes span several 128-token tiles with ragged tails; the five workloads run at
their full sizes in the launch configuration the benchmark times.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import config_problem, make_problem
from synth.inputs import random_logits
from tests.parity import check_logits, check_topk_exact, check_topk_rows

pytestmark = pytest.mark.gpu


def dev(prob):
    return dict(
        q=torch.from_numpy(prob.q).cuda().view(torch.float8_e4m3fn),
        kv=torch.from_numpy(prob.kv).cuda(),
        w=torch.from_numpy(prob.weights).cuda(),
        ctx=torch.from_numpy(prob.context_lens).cuda(),
        bt=torch.from_numpy(prob.block_tables).cuda(),
    )


def gpu_logits(L, prob, d=None, ws=None):
    d = d or dev(prob)
    out = L.pmqa_logits(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], prob.max_model_len, ws=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def gpu_fused(L, prob, k, d=None, ws=None, logits=None):
    d = d or dev(prob)
    idx, vals = L.pmqa_logits_topk(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], prob.max_model_len,
                                   k, want_vals=True, ws=ws, logits=logits)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), vals.cpu().numpy()


def oracle_all(prob):
    out, o64, tol = oracle.logits(prob, want64=True, want_tol=True)
    return out, o64, tol


SMALL = [
    # bs, next_n, heads, block_size, context lengths, max_model_len, table
    (1, 1, 32, 1, [300], 512, "identity"),
    (3, 1, 64, 1, [1, 127, 129], 256, "perm"),
    (2, 1, 16, 1, [200, 0], 256, "perm"),
    (4, 2, 64, 1, [1, 2, 255, 513], 640, "perm"),
    (2, 3, 32, 16, [33, 400], 512, "perm"),
    (3, 4, 64, 1, [3, 4, 700], 768, "perm"),
    (2, 4, 128, 64, [130, 1000], 1024, "perm"),
    (2, 2, 128, 1, [640, 129], 640, "perm"),
    (5, 1, 128, 64, [64, 65, 127, 1, 300], 320, "perm"),
    (2, 4, 16, 1, [77, 5], 128, "perm"),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"bs{c[0]}nn{c[1]}H{c[2]}P{c[3]}")
def test_logits_small(cuda_lib, case):
    bs, nn, H, P, ctx, mml, table = case
    prob = make_problem(bs, nn, H, P, ctx, mml, seed=sum(ctx) + H, table=table, extra_blocks=2)
    ref, _, tol = oracle_all(prob)
    check_logits(gpu_logits(cuda_lib, prob), ref, tol)


@pytest.mark.parametrize("k", [1, 7, 100, 2048])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"bs{c[0]}nn{c[1]}H{c[2]}P{c[3]}")
def test_fused_topk_small(cuda_lib, case, k):
    bs, nn, H, P, ctx, mml, table = case
    prob = make_problem(bs, nn, H, P, ctx, mml, seed=sum(ctx) + H + 1, table=table, extra_blocks=2)
    ref, r64, tol = oracle_all(prob)
    logits = torch.empty((bs * nn, mml), dtype=torch.float32, device="cuda")
    idx, vals = gpu_fused(cuda_lib, prob, k, logits=logits)
    check_topk_rows(idx, r64, tol, prob.context_lens, nn, k, vals=vals)
    check_logits(logits.cpu().numpy(), ref, tol)


# Shapes the prior art on the pages mishandled or rejected: block sizes other
# than 1 and 64 (256 with a partial last page; sizes that are not powers of two;
# sizes that are not multiples of 4, which move as 16-byte windows rather than
# page runs), three draft rows, and heads 32 and 128 with them.
BLOCKS = [
    # bs, next_n, heads, block_size, context lengths, max_model_len
    (2, 1, 64, 256, [300, 1000], 1024),
    (1, 3, 32, 256, [2100], 2304),
    (2, 3, 32, 3, [100, 250], 256),
    (2, 2, 64, 6, [77, 300], 384),
    (3, 3, 128, 12, [50, 129, 260], 384),
    (2, 3, 64, 32, [513, 97], 640),
    (2, 2, 16, 5, [128, 333], 384),
]


@pytest.mark.parametrize("case", BLOCKS, ids=lambda c: f"bs{c[0]}nn{c[1]}H{c[2]}P{c[3]}")
def test_block_sizes_and_draft_rows(cuda_lib, case):
    bs, nn, H, P, ctx, mml = case
    prob = make_problem(bs, nn, H, P, ctx, mml, seed=sum(ctx) + 7 * P, table="perm", extra_blocks=3)
    ref, r64, tol = oracle_all(prob)
    check_logits(gpu_logits(cuda_lib, prob), ref, tol)
    for k in (7, 2048):
        logits = torch.empty((bs * nn, mml), dtype=torch.float32, device="cuda")
        idx, vals = gpu_fused(cuda_lib, prob, k, logits=logits)
        check_topk_rows(idx, r64, tol, prob.context_lens, nn, k, vals=vals)
        check_logits(logits.cpu().numpy(), ref, tol)


# A pool past 2 GB: byte offsets of rows no longer fit in 31 bits, which
# selects the gather with 64-bit offsets (windows) and exercises the page runs'
# 64-bit addressing. The small problem's blocks are moved past 2 GB + 1 MB of
# zero blocks; the oracle runs on the small problem (the same logical cache).
@pytest.mark.parametrize("P,nn", [(1, 2), (3, 1), (64, 4)])
def test_pool_past_2_gb(cuda_lib, P, nn):
    import dataclasses

    prob = make_problem(2, nn, 64, P, [700, 300], 1024, seed=11 + P, table="perm",
                        extra_blocks=3)
    ref, r64, tol = oracle_all(prob)
    shift = -(-(2**31 + 2**20) // (P * 132))
    kv = np.zeros((shift + prob.num_blocks, P, 132), dtype=np.uint8)
    kv[shift:] = prob.kv
    bt = np.where(prob.block_tables >= 0, prob.block_tables + shift, -1).astype(np.int32)
    big = dataclasses.replace(prob, kv=kv, block_tables=bt)
    assert big.num_blocks * P * 132 > 2**31
    d = dev(big)
    check_logits(gpu_logits(cuda_lib, big, d=d), ref, tol)
    idx, vals = gpu_fused(cuda_lib, big, 2048, d=d)
    check_topk_rows(idx, r64, tol, prob.context_lens, nn, 2048, vals=vals)


# The scale's sign: relu(s * x) = |s| * relu(-x) for s < 0, which the kernel
# applies per token by flipping the sign of the row's signed sum. Mixed signs
# put both kinds of token in every warp; an all-negative range makes every
# token of every tile flip. Block sizes 1 (row windows) and 64 (page runs),
# one and four draft rows.
SIGNED = [
    # bs, next_n, heads, block_size, context lengths, max_model_len, scale range
    (3, 1, 64, 1, [300, 129, 1000], 1024, (-0.1, 0.1)),
    (2, 4, 64, 1, [700, 260], 768, (-0.1, 0.1)),
    (2, 1, 32, 64, [1000, 130], 1024, (-0.1, 0.1)),
    (2, 4, 64, 64, [513, 1000], 1024, (-0.1, 0.1)),
    (2, 1, 64, 1, [640, 300], 640, (-0.1, -0.01)),
    (2, 4, 64, 64, [513, 1000], 1024, (-0.1, -0.01)),
    (2, 2, 128, 1, [400, 129], 512, (-0.1, -0.01)),
]


@pytest.mark.parametrize("case", SIGNED, ids=lambda c: f"nn{c[1]}H{c[2]}P{c[3]}s{c[6][1]:+g}")
def test_negative_and_mixed_scales(cuda_lib, case):
    bs, nn, H, P, ctx, mml, sr = case
    prob = make_problem(bs, nn, H, P, ctx, mml, seed=sum(ctx) + nn + P, table="perm",
                        extra_blocks=2, scale_range=sr)
    ref, r64, tol = oracle_all(prob)
    if sr[1] < 0:  # every scale negative: the scores come from the q.k < 0 terms alone
        assert np.any(ref[np.isfinite(ref)] != 0)
    check_logits(gpu_logits(cuda_lib, prob), ref, tol)
    for k in (7, 2048):
        logits = torch.empty((bs * nn, mml), dtype=torch.float32, device="cuda")
        idx, vals = gpu_fused(cuda_lib, prob, k, logits=logits)
        check_topk_rows(idx, r64, tol, prob.context_lens, nn, k, vals=vals)
        check_logits(logits.cpu().numpy(), ref, tol)


@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("k", [1, 5, 300, 2048])
def test_standalone_topk_exact(cuda_lib, k, ties):
    ctx, nn, mml = [0, 1, 7, 129, 3000, 5000], 2, 5120
    vals = random_logits(len(ctx) * nn, mml, seed=k, ties=ties)
    t = torch.from_numpy(vals).cuda()
    c = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    idx, got = cuda_lib.pmqa_topk(t, c, nn, k, want_vals=True)
    idx, got = idx.cpu().numpy(), got.cpu().numpy()
    check_topk_exact(idx, vals, ctx, nn, k)
    ke_rows = [min(k, max(0, min(cx - nn + j + 1, cx))) for cx in ctx for j in range(nn)]
    for r, ke in enumerate(ke_rows):
        assert np.array_equal(got[r, :ke], vals[r, idx[r, :ke]])
    # the oracle's own selection agrees on the chosen values
    ref = oracle.topk(vals.astype(np.float64), ctx, nn, k)
    for r, ke in enumerate(ke_rows):
        assert np.array_equal(np.sort(vals[r, ref[r, :ke]]), np.sort(vals[r, idx[r, :ke]]))


def test_standalone_topk_of_oracle_logits(cuda_lib):
    prob = make_problem(4, 2, 32, 1, [5000, 2049, 2048, 17], 6144, seed=3)
    out, _, _ = oracle_all(prob)
    t = torch.from_numpy(out).cuda()
    c = torch.from_numpy(prob.context_lens).cuda()
    idx = cuda_lib.pmqa_topk(t, c, 2, 2048).cpu().numpy()
    check_topk_exact(idx, out, prob.context_lens, 2, 2048)


# ------------------------------------------------------------- invariants


def test_permutation_invariance_bit_exact(cuda_lib):
    prob = make_problem(3, 2, 64, 1, [900, 130, 2000], 2048, seed=21, table="identity",
                        extra_blocks=5)
    a = gpu_logits(cuda_lib, prob)
    perm = np.random.default_rng(5).permutation(prob.num_blocks)
    kv2 = np.empty_like(prob.kv)
    kv2[perm] = prob.kv
    prob.kv = kv2
    prob.block_tables = np.where(prob.block_tables >= 0,
                                 perm[np.maximum(prob.block_tables, 0)], -1).astype(np.int32)
    b = gpu_logits(cuda_lib, prob)
    assert np.array_equal(a, b)


def test_context_2048_to_2049_bit_exact(cuda_lib):
    prob = make_problem(1, 1, 32, 1, [2049], 4096, seed=42, table="identity", extra_blocks=16)
    a = gpu_logits(cuda_lib, prob)
    prob.context_lens[:] = 2048
    b = gpu_logits(cuda_lib, prob)
    assert np.array_equal(a[0, :2048], b[0, :2048])
    assert np.isneginf(b[0, 2048]) and np.isfinite(a[0, 2048])
    idx, _ = gpu_fused(cuda_lib, prob, 2048)
    assert np.array_equal(np.sort(idx[0]), np.arange(2048))
    prob.context_lens[:] = 2049
    ref, r64, tol = oracle_all(prob)
    idx, vals = gpu_fused(cuda_lib, prob, 2048)
    check_topk_rows(idx, r64, tol, [2049], 1, 2048, vals=vals)


def test_workspace_is_reusable(cuda_lib):
    """Calls leave the workspace clean: repeated and reshaped calls agree."""
    prob = make_problem(4, 2, 64, 1, [3000, 5000, 100, 2500], 5120, seed=8)
    d = dev(prob)
    ws = cuda_lib.workspace(4, 2, 5120, 512, cuda_lib.PMQA_OP_LOGITS_TOPK)
    i1, v1 = gpu_fused(cuda_lib, prob, 512, d=d, ws=ws)
    i2, v2 = gpu_fused(cuda_lib, prob, 512, d=d, ws=ws)
    assert np.array_equal(np.sort(i1, axis=1), np.sort(i2, axis=1))
    prob.context_lens[:] = [2999, 17, 100, 2400]  # within each request's table
    d = dev(prob)
    i3, v3 = gpu_fused(cuda_lib, prob, 512, d=d, ws=ws)
    _, r64, tol = oracle_all(prob)
    check_topk_rows(i3, r64, tol, prob.context_lens, 2, 512, vals=v3)
    assert cuda_lib.pmqa_read_device_status(ws) == 0


def test_stages_match_the_fused_call(cuda_lib):
    """SCORE then SELECT (two calls) selects what the fused call selects."""
    prob = make_problem(3, 2, 64, 16, [3000, 1500, 2049], 4096, seed=12, table="perm")
    d = dev(prob)
    k = 1024
    ws = cuda_lib.workspace(3, 2, 4096, k, cuda_lib.PMQA_OP_LOGITS_TOPK)
    i_f, v_f = gpu_fused(cuda_lib, prob, k, d=d, ws=ws)
    idx = torch.empty((6, k), dtype=torch.int32, device="cuda")
    vals = torch.empty((6, k), dtype=torch.float32, device="cuda")
    args = (d["q"], d["kv"], d["w"], d["ctx"], d["bt"], prob.max_model_len, k)
    cuda_lib.pmqa_logits_topk_stages(*args, cuda_lib.PMQA_STAGE_SCORE, idx=idx, vals=vals, ws=ws)
    cuda_lib.pmqa_logits_topk_stages(*args, cuda_lib.PMQA_STAGE_SELECT, idx=idx, vals=vals, ws=ws)
    torch.cuda.synchronize()
    i_s, v_s = idx.cpu().numpy(), vals.cpu().numpy()
    for r in range(6):  # same set, same values (order within a row may differ)
        o_f, o_s = np.argsort(i_f[r]), np.argsort(i_s[r])
        assert np.array_equal(i_f[r][o_f], i_s[r][o_s])
        assert np.array_equal(v_f[r][o_f], v_s[r][o_s])
    _, r64, tol = oracle_all(prob)
    check_topk_rows(i_s, r64, tol, prob.context_lens, 2, k, vals=v_s)
    assert cuda_lib.pmqa_read_device_status(ws) == 0


def test_bad_table_entry_sets_status_without_fault(cuda_lib):
    prob = make_problem(2, 1, 64, 1, [300, 200], 512, seed=9)
    prob.block_tables[1, 10] = prob.num_blocks + 7
    d = dev(prob)
    ws = cuda_lib.workspace(2, 1, 512, 0, cuda_lib.PMQA_OP_LOGITS)
    out = cuda_lib.pmqa_logits(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], 512, ws=ws)
    st = cuda_lib.pmqa_read_device_status(ws)
    assert st & cuda_lib.PMQA_DEV_BAD_BLOCK_ID
    assert cuda_lib.pmqa_read_device_status(ws) == 0  # cleared by the read
    o = out.cpu().numpy()
    prob.block_tables[1, 10] = prob.block_tables[1, 11]
    ref, _, tol = oracle_all(prob)
    assert np.array_equal(o[0], gpu_logits(cuda_lib, prob)[0])
    assert o[1, 10] == 0.0  # the bad token reads as zeros


def test_context_longer_than_max_model_len_is_flagged(cuda_lib):
    prob = make_problem(1, 1, 32, 1, [100], 128, seed=10)
    d = dev(prob)
    d["ctx"][0] = 200
    ws = cuda_lib.workspace(1, 1, 128, 0, cuda_lib.PMQA_OP_LOGITS)
    cuda_lib.pmqa_logits(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], 128, ws=ws)
    assert cuda_lib.pmqa_read_device_status(ws) & cuda_lib.PMQA_DEV_BAD_CONTEXT


@pytest.mark.parametrize("k", [100, 2048, 3000])
def test_fused_topk_with_every_logit_equal(cuda_lib, k):
    """Zero weights make every admitted logit exactly 0: the whole row sits in
    one key bin, more candidates than the selection keeps in shared memory,
    and any k_eff of them are a correct answer."""
    prob = make_problem(3, 2, 64, 16, [5000, 2100, 130], 5120, seed=5, table="perm",
                        extra_blocks=2)
    prob.weights[:] = 0.0
    ref, r64, tol = oracle_all(prob)
    for ws in (None, cuda_lib.workspace(3, 2, 5120, k, cuda_lib.PMQA_OP_LOGITS_TOPK)):
        idx, vals = gpu_fused(cuda_lib, prob, k, ws=ws)
        check_topk_rows(idx, r64, tol, prob.context_lens, prob.next_n, k, vals=vals)
        assert np.all(vals[idx >= 0] == 0.0)
        if ws is not None:
            assert cuda_lib.pmqa_read_device_status(ws) == 0


def test_context_beyond_the_block_table_is_clamped_in_the_fused_call(cuda_lib):
    """A context longer than block_size * max_blocks_per_seq (but within
    max_model_len): the KV pass and the selection clamp it to the table's reach
    alike, so no selected position lies past it, and the status says so."""
    P, W, mml = 16, 20, 512
    prob = make_problem(2, 2, 64, P, [P * W, 300], mml, seed=31, table="perm", extra_blocks=2,
                        width=W)
    ref, r64, tol = oracle_all(prob)
    d = dev(prob)
    d["ctx"][0] = 400  # the table reaches 320 tokens
    for k in (7, 2048):
        ws = cuda_lib.workspace(prob.bs, prob.next_n, mml, k, cuda_lib.PMQA_OP_LOGITS_TOPK)
        logits = torch.empty((prob.rows, mml), dtype=torch.float32, device="cuda")
        idx, vals = gpu_fused(cuda_lib, prob, k, d=d, ws=ws, logits=logits)
        assert cuda_lib.pmqa_read_device_status(ws) == cuda_lib.PMQA_DEV_BAD_CONTEXT
        assert idx.max() < P * W
        check_topk_rows(idx, r64, tol, prob.context_lens, prob.next_n, k, vals=vals)
        check_logits(logits.cpu().numpy(), ref, tol)


# ------------------------------------------------------------- full workloads


@pytest.fixture(scope="module", params=["C0", "C1", "C2", "C3", "C4"])
def workload(request):
    prob = config_problem(request.param)
    ref, r64, tol = oracle_all(prob)
    return prob, ref, r64, tol


def test_workload_logits(cuda_lib, workload):
    prob, ref, _, tol = workload
    check_logits(gpu_logits(cuda_lib, prob), ref, tol)


def test_workload_fused_topk(cuda_lib, workload):
    prob, _, r64, tol = workload
    idx, vals = gpu_fused(cuda_lib, prob, prob.k)
    check_topk_rows(idx, r64, tol, prob.context_lens, prob.next_n, prob.k, vals=vals)


def test_workload_standalone_topk(cuda_lib, workload):
    prob, ref, _, _ = workload
    t = torch.from_numpy(ref).cuda()
    c = torch.from_numpy(prob.context_lens).cuda()
    idx = cuda_lib.pmqa_topk(t, c, prob.next_n, prob.k).cpu().numpy()
    check_topk_exact(idx, ref, prob.context_lens, prob.next_n, prob.k)


@pytest.mark.parametrize("nn,H", [(1, 64), (2, 32), (4, 64), (3, 128)])
def test_many_short_requests(cuda_lib, nn, H):
    """Each CTA walks many requests, several shorter than the copy pipeline."""
    rng = np.random.default_rng(nn * H)
    ctx = rng.integers(0, 400, size=300)
    ctx[::7] = rng.integers(1, 4, size=len(ctx[::7]))
    prob = make_problem(300, nn, H, 1, ctx, 512, seed=nn + H, table="perm")
    ref, r64, tol = oracle_all(prob)
    d = dev(prob)
    ws = cuda_lib.workspace(300, nn, 512, 64, cuda_lib.PMQA_OP_LOGITS_TOPK)
    check_logits(gpu_logits(cuda_lib, prob, d=d, ws=ws), ref, tol)
    idx, vals = gpu_fused(cuda_lib, prob, 64, d=d, ws=ws)
    check_topk_rows(idx, r64, tol, prob.context_lens, nn, 64, vals=vals)
    assert cuda_lib.pmqa_read_device_status(ws) == 0


# Row lengths that pick each selection kernel: up to 32768 positions (one CTA
# per row, logits in shared memory), up to 65536 (one CTA per row, the logits
# in two halves through shared memory), above (several CTAs per row, here up
# to 64 and 74 of them).
@pytest.mark.parametrize("mml", [32768, 40000, 65536, 70000, 262144, 300000])
@pytest.mark.parametrize("ties", [False, True])
def test_standalone_topk_each_selection_kernel(cuda_lib, mml, ties):
    ctx, nn, k = [mml, mml - 1, 33000, 2049, 1], 1, 2048
    vals = random_logits(len(ctx) * nn, mml, seed=mml + ties, ties=ties)
    t = torch.from_numpy(vals).cuda()
    c = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    idx, got = cuda_lib.pmqa_topk(t, c, nn, k, want_vals=True)
    idx, got = idx.cpu().numpy(), got.cpu().numpy()
    check_topk_exact(idx, vals, ctx, nn, k)
    for r, cx in enumerate(ctx):
        ke = min(k, cx)
        assert np.array_equal(got[r, :ke], vals[r, idx[r, :ke]])


def test_fused_topk_with_rows_read_in_place(cuda_lib):
    """max_model_len between 32768 and 65536: the fused call's selection reads
    each row in place."""
    prob = make_problem(3, 2, 64, 16, [33000, 40000, 100], 40000, seed=21, table="perm",
                        extra_blocks=2)
    ref, r64, tol = oracle_all(prob)
    logits = torch.empty((prob.rows, prob.max_model_len), dtype=torch.float32, device="cuda")
    idx, vals = gpu_fused(cuda_lib, prob, 2048, logits=logits)
    check_logits(logits.cpu().numpy(), ref, tol)
    check_topk_rows(idx, r64, tol, prob.context_lens, prob.next_n, 2048, vals=vals)


@pytest.mark.parametrize("mml", [4096, 40000, 70000, 300000])
def test_fused_call_replays_from_a_cuda_graph(cuda_lib, mml):
    """The fused call (KV pass + programmatic-dependent selection) captured in a
    CUDA graph and replayed gives what the direct call gives, with the same
    workspace state afterwards (every call leaves it zeroed)."""
    ctx = [mml - 5, mml // 2, 3000]
    prob = make_problem(3, 2, 64, 16, ctx, mml, seed=mml, table="perm", extra_blocks=2)
    d = dev(prob)
    k = 2048
    ws = cuda_lib.workspace(prob.bs, prob.next_n, mml, k, cuda_lib.PMQA_OP_LOGITS_TOPK)
    idx_direct, vals_direct = cuda_lib.pmqa_logits_topk(d["q"], d["kv"], d["w"], d["ctx"], d["bt"],
                                                        mml, k, want_vals=True, ws=ws)
    torch.cuda.synchronize()
    idx = torch.empty_like(idx_direct)
    vals = torch.empty_like(vals_direct)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        # one call on the capture stream first, so that any lazy setup is done
        cuda_lib.pmqa_logits_topk(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], mml, k, idx=idx,
                                  vals=vals, ws=ws, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            cuda_lib.pmqa_logits_topk(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], mml, k,
                                      idx=idx, vals=vals, ws=ws, stream=stream)
    for _ in range(2):
        idx.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        a, b = idx.cpu().numpy(), idx_direct.cpu().numpy()
        # same selected sets per row (order within a row is unspecified)
        assert np.array_equal(np.sort(a, axis=1), np.sort(b, axis=1))
        assert np.array_equal(np.sort(vals.cpu().numpy(), axis=1),
                              np.sort(vals_direct.cpu().numpy(), axis=1))
    assert cuda_lib.pmqa_read_device_status(ws) == 0
