"""pmqa_logits_topk_noalloc: the fused call for callers that cannot allocate
device memory (for example a plugin whose host program owns the device-memory
pool, or a loop that must not call cudaMalloc). It uses a fixed 32 MiB scratch
array inside the library instead of a caller workspace.

Kept in the last-collected file so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_indexer_pmqa_gb300 import build, pmqa
from synth import make_problem
from tests.parity import check_topk_rows


def test_noalloc_rejects_problems_beyond_its_scratch():
    build.build()
    lib = pmqa.load()
    # 64 rows x 65536 positions needs a 32 MiB+ candidate area: refused up front
    p = pmqa.Problem(q=0x10000, kv_cache=0x20000, weights=0x30000, context_lens=0x40000,
                     block_tables=0x50000, bs=64, next_n=1, heads=64, head_dim=128,
                     block_size=1, max_blocks_per_seq=65536, max_model_len=65536,
                     num_blocks=1 << 20)
    assert lib.pmqa_logits_topk_noalloc(ctypes.byref(p), 2048, ctypes.c_void_p(0x60000), None,
                                        None, None) == pmqa.PMQA_ERR_WORKSPACE
    assert lib.pmqa_logits_topk_noalloc(None, 16, ctypes.c_void_p(0x60000), None, None,
                                        None) == pmqa.PMQA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point(cuda_lib):
    prob = make_problem(6, 2, 64, 1, [3000, 5000, 129, 2049, 1, 4100], 5120, seed=77,
                        table="perm", extra_blocks=3, k=2048)
    d = dict(q=torch.from_numpy(prob.q).cuda().view(torch.float8_e4m3fn),
             kv=torch.from_numpy(prob.kv).cuda(), w=torch.from_numpy(prob.weights).cuda(),
             ctx=torch.from_numpy(prob.context_lens).cuda(),
             bt=torch.from_numpy(prob.block_tables).cuda())
    rows, k, mml = prob.rows, prob.k, prob.max_model_len
    ref_idx, ref_vals = cuda_lib.pmqa_logits_topk(d["q"], d["kv"], d["w"], d["ctx"], d["bt"],
                                                  mml, k, want_vals=True)
    torch.cuda.synchronize()
    ref_idx, ref_vals = ref_idx.cpu().numpy(), ref_vals.cpu().numpy()
    _, r64, tol = oracle.logits(prob, want64=True, want_tol=True)
    check_topk_rows(ref_idx, r64, tol, prob.context_lens, prob.next_n, k, vals=ref_vals)
    for _call in range(2):  # two calls in a row share the scratch array
        idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
        vals = torch.full((rows, k), 7.0, dtype=torch.float32, device="cuda")
        logits = torch.full((rows, mml), 7.0, dtype=torch.float32, device="cuda")
        cuda_lib.pmqa_logits_topk_noalloc(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], mml, k,
                                          idx=idx, vals=vals, logits=logits)
        torch.cuda.synchronize()
        got_i, got_v = idx.cpu().numpy(), vals.cpu().numpy()
        check_topk_rows(got_i, r64, tol, prob.context_lens, prob.next_n, k, vals=got_v)
        for r in range(rows):
            # same positions as the workspace entry point, values within tolerance
            assert np.array_equal(np.sort(got_i[r]), np.sort(ref_idx[r]))
            order_a, order_b = np.argsort(got_i[r]), np.argsort(ref_idx[r])
            va, vb = got_v[r][order_a], ref_vals[r][order_b]
            fin = np.isfinite(vb)
            assert np.array_equal(np.isfinite(va), fin)
            pos = np.sort(ref_idx[r])[fin]
            assert np.all(np.abs(va[fin].astype(np.float64) - vb[fin]) <= tol[r, pos])
        lg = logits.cpu().numpy()
        assert np.array_equal(np.isneginf(lg), np.isneginf(r64))


@pytest.mark.gpu
def test_noalloc_clamps_a_context_beyond_the_table_over_stale_scratch(cuda_lib):
    """The scratch keeps the previous call's compact logits. A following call
    whose context runs past block_size * max_blocks_per_seq must select only
    from positions its KV pass scored, never from what an earlier call left."""
    P, W, mml, k = 16, 20, 512, 2048
    big = make_problem(2, 2, 64, P, [mml, mml], mml, seed=41, table="perm", extra_blocks=2)
    big.weights *= 100.0  # large leftovers past position P * W
    db = {n: torch.from_numpy(a).cuda() for n, a in
          (("kv", big.kv), ("w", big.weights), ("ctx", big.context_lens), ("bt", big.block_tables))}
    qb = torch.from_numpy(big.q).cuda().view(torch.float8_e4m3fn)
    idx = torch.empty((big.rows, k), dtype=torch.int32, device="cuda")
    cuda_lib.pmqa_logits_topk_noalloc(qb, db["kv"], db["w"], db["ctx"], db["bt"], mml, k, idx=idx)
    prob = make_problem(2, 2, 64, P, [P * W, 300], mml, seed=42, table="perm", extra_blocks=2,
                        width=W)
    _, r64, tol = oracle.logits(prob, want64=True, want_tol=True)
    d = {n: torch.from_numpy(a).cuda() for n, a in
         (("kv", prob.kv), ("w", prob.weights), ("ctx", prob.context_lens),
          ("bt", prob.block_tables))}
    q = torch.from_numpy(prob.q).cuda().view(torch.float8_e4m3fn)
    d["ctx"][0] = 400  # the table reaches 320 tokens
    vals = torch.empty((prob.rows, k), dtype=torch.float32, device="cuda")
    cuda_lib.pmqa_logits_topk_noalloc(q, d["kv"], d["w"], d["ctx"], d["bt"], mml, k, idx=idx,
                                      vals=vals)
    torch.cuda.synchronize()
    got_i, got_v = idx.cpu().numpy(), vals.cpu().numpy()
    assert got_i.max() < P * W
    check_topk_rows(got_i, r64, tol, prob.context_lens, prob.next_n, k, vals=got_v)
