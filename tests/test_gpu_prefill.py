"""GPU parity of the prefill (non-paged) logits: libpmqa through its C ABI
against the CPU oracle.

-inf pattern bit-exact; finite entries within 1e-3 (1 + sum_h |w_h||x_h|).
Small cases span several 128-key tiles and super-groups with ragged tails;
the prefill workload runs at its full size (4096 query rows, 8192 keys,
heads 32, causal ranges) in the launch configuration the benchmark times,
checked on sampled rows.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import make_prefill, prefill_config
from tests.parity import check_logits

pytestmark = pytest.mark.gpu


def dev(p):
    return dict(
        q=torch.from_numpy(p.q).cuda().view(torch.float8_e4m3fn),
        k=torch.from_numpy(p.k).cuda().view(torch.float8_e4m3fn),
        s=torch.from_numpy(p.k_scale).cuda(),
        w=torch.from_numpy(p.weights).cuda(),
        ks=torch.from_numpy(p.ks).cuda(),
        ke=torch.from_numpy(p.ke).cuda(),
    )


def gpu_mqa(L, p, d=None, ws=None, out=None):
    d = d or dev(p)
    res = L.pmqa_mqa_logits(d["q"], d["k"], d["s"], d["w"], d["ks"], d["ke"], ws=ws, out=out)
    torch.cuda.synchronize()
    return res.cpu().numpy()


SMALL = [
    # m, n, heads, ranges
    (1, 1, 32, "full"),
    (5, 130, 32, "causal"),
    (16, 128, 32, "full"),
    (37, 1000, 32, "causal"),
    (100, 100, 32, "packed"),
    (64, 700, 64, "random"),
    (9, 300, 128, "causal"),
    (70, 513, 16, "random"),
    (33, 257, 16, "causal"),
    (300, 300, 64, "packed"),
    (17, 2049, 128, "full"),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"m{c[0]}n{c[1]}H{c[2]}{c[3]}")
def test_prefill_small(cuda_lib, case):
    m, n, H, ranges = case
    p = make_prefill(m, n, H, ranges=ranges, seed=m * 7 + n + H)
    ref, _, tol = oracle.mqa_logits(p, want_tol=True)
    ws = cuda_lib.workspace(p.m, 1, p.n, 0, cuda_lib.PMQA_OP_MQA_LOGITS)
    check_logits(gpu_mqa(cuda_lib, p, ws=ws), ref, tol)
    assert cuda_lib.pmqa_read_device_status(ws) == 0


def test_prefill_negative_and_mixed_scales(cuda_lib):
    p = make_prefill(48, 600, 32, ranges="full", seed=3, poison=False)
    rng = np.random.default_rng(4)
    p.k_scale *= np.where(rng.random(600) < 0.5, -1.0, 1.0).astype(np.float32)
    p.k_scale[256:384] = -np.abs(p.k_scale[256:384])  # one tile all negative
    ref, _, tol = oracle.mqa_logits(p, want_tol=True)
    check_logits(gpu_mqa(cuda_lib, p), ref, tol)


def test_prefill_empty_rows_and_out_of_range_bounds(cuda_lib):
    p = make_prefill(40, 400, 64, ranges="full", seed=8, poison=False)
    p.ks[:] = 0
    p.ke[:] = 0
    p.ks[5], p.ke[5] = -50, 20      # clamps to [0, 20)
    p.ks[17], p.ke[17] = 390, 900   # clamps to [390, 400)
    p.ks[30], p.ke[30] = 200, 100   # empty
    ref, _, tol = oracle.mqa_logits(p, want_tol=True)
    got = gpu_mqa(cuda_lib, p)
    check_logits(got, ref, tol)
    assert np.isneginf(got[0]).all() and np.isfinite(got[17, 390:]).all()


def test_prefill_all_rows_empty_writes_only_neg_inf(cuda_lib):
    p = make_prefill(20, 300, 32, ranges="full", seed=2, poison=False)
    p.ke[:] = p.ks[:]
    out = torch.zeros((20, 300), dtype=torch.float32, device="cuda")
    got = gpu_mqa(cuda_lib, p, out=out)
    assert np.isneginf(got).all()


def test_prefill_repeat_calls_are_identical(cuda_lib):
    p = make_prefill(96, 1111, 32, ranges="causal", seed=12)
    d = dev(p)
    a = gpu_mqa(cuda_lib, p, d=d)
    b = gpu_mqa(cuda_lib, p, d=d)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def _rows_problem(p, rows):
    """The same problem restricted to the given query rows (rows are independent)."""
    sub = make_prefill(1, 1, p.heads, ranges="full", seed=0, poison=False)
    sub.q = p.q[rows].copy()
    sub.weights = p.weights[rows].copy()
    sub.ks = p.ks[rows].copy()
    sub.ke = p.ke[rows].copy()
    sub.k = p.k
    sub.k_scale = p.k_scale
    return sub


@pytest.mark.slow
def test_prefill_full_size_sampled_rows(cuda_lib):
    p = prefill_config("PF1")
    d = dev(p)
    ws = cuda_lib.workspace(p.m, 1, p.n, 0, cuda_lib.PMQA_OP_MQA_LOGITS)
    got = gpu_mqa(cuda_lib, p, d=d, ws=ws)
    assert cuda_lib.pmqa_read_device_status(ws) == 0
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 15, 16, p.m - 1],
                                     rng.choice(p.m, size=27, replace=False)]))
    ref, _, tol = oracle.mqa_logits(_rows_problem(p, rows), want_tol=True)
    check_logits(got[rows], ref, tol)
    # every row: exactly its causal range is finite
    fin = np.isfinite(got)
    assert np.array_equal(fin.sum(axis=1), p.ke.astype(np.int64))
    assert all(fin[r, : p.ke[r]].all() for r in (0, p.m // 2, p.m - 1))


@pytest.mark.parametrize("m,n,H,ranges", [
    (2048, 8192, 64, "causal"),
    (1024, 4096, 128, "causal"),
    (6144, 6144, 32, "packed"),
])
def test_prefill_larger_shapes_sampled_rows(cuda_lib, m, n, H, ranges):
    p = make_prefill(m, n, H, ranges=ranges, seed=m + H)
    d = dev(p)
    ws = cuda_lib.workspace(p.m, 1, p.n, 0, cuda_lib.PMQA_OP_MQA_LOGITS)
    got = gpu_mqa(cuda_lib, p, d=d, ws=ws)
    assert cuda_lib.pmqa_read_device_status(ws) == 0
    rng = np.random.default_rng(m)
    rows = np.unique(np.concatenate([[0, 1, m // 2, m - 1], rng.choice(m, size=20, replace=False)]))
    ref, _, tol = oracle.mqa_logits(_rows_problem(p, rows), want_tol=True)
    check_logits(got[rows], ref, tol)
    # every row's finite entries are exactly its clamped key range
    lo = np.clip(p.ks.astype(np.int64), 0, n)
    hi = np.clip(p.ke.astype(np.int64), 0, n)
    assert np.array_equal(np.isfinite(got).sum(axis=1), np.maximum(hi - lo, 0))


@pytest.mark.parametrize("H", [32, 128])
def test_prefill_replays_from_a_cuda_graph(cuda_lib, H):
    """Both prefill launches (the prep kernel and the main kernel, its
    programmatic dependent) captured in a CUDA graph on a side stream: every
    replay rewrites the whole output bit-identically to the direct call."""
    p = make_prefill(200, 1500, H, ranges="causal", seed=H)
    ref, _, tol = oracle.mqa_logits(p, want_tol=True)
    d = dev(p)
    ws = cuda_lib.workspace(p.m, 1, p.n, 0, cuda_lib.PMQA_OP_MQA_LOGITS)
    direct = gpu_mqa(cuda_lib, p, d=d, ws=ws)
    args = (d["q"], d["k"], d["s"], d["w"], d["ks"], d["ke"])
    out = torch.empty((p.m, p.n), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        # one call on the capture stream first, so that any lazy setup is done
        cuda_lib.pmqa_mqa_logits(*args, out=out, ws=ws, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            cuda_lib.pmqa_mqa_logits(*args, out=out, ws=ws, stream=stream)
    for _ in range(2):
        out.fill_(7.0)
        graph.replay()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), direct.view(np.uint32))
    check_logits(got, ref, tol)
    assert cuda_lib.pmqa_read_device_status(ws) == 0
