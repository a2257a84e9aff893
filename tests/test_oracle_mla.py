"""The sparse MLA decode oracle against what the mathematics fixes (CPU).

Pins: a two-token example worked by hand, the uniform-weight and one-hot
closed forms, torch's scaled dot-product attention on dense listings (a
library routine, run in float64 on the dequantised tensors), and the
invariances of the definition (listing order, page size, holes, repeats).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from synth.inputs import to_e4m3fn_bytes
from synth.mla import MLA_DIM, MLA_VDIM, MlaProblem, make_mla_problem

E4M3 = None


def dequant(codes, scale):
    global E4M3
    if E4M3 is None:
        E4M3 = oracle.e4m3fn_table()
    return E4M3[codes.astype(np.int64)] * scale


def one_request(kv_rows, q_rows, listing, *, q_scale=1.0, kv_scale=1.0, sm_scale=1.0, P=1):
    """A problem of one request whose logical tokens are kv_rows (codes
    [n, 576]) on pages of P tokens (identity table), one query row with
    q_rows (codes [heads, 576]) and the given listing."""
    n = kv_rows.shape[0]
    nblk = -(-n // P)
    kv = np.zeros((nblk * P, MLA_DIM), dtype=np.uint8)
    kv[:n] = kv_rows
    return MlaProblem(q=q_rows[None, None].copy(), kv=kv.reshape(nblk, P, MLA_DIM),
                      indices=np.asarray(listing, dtype=np.int32)[None, :],
                      context_lens=np.array([n], dtype=np.int32),
                      block_tables=np.arange(nblk, dtype=np.int32)[None, :],
                      q_scale=q_scale, kv_scale=kv_scale, sm_scale=sm_scale, bs=1, next_n=1,
                      heads=q_rows.shape[0], block_size=P)


def code(x):
    return int(to_e4m3fn_bytes(np.array([x], dtype=np.float32))[0])


def test_two_token_example_worked_by_hand():
    """q = e_0; k_A = (2, 1, 0, ...), k_B = (0, -1, 0, ...); sm_scale = ln(3)/2.
    Scores ln 3 and 0, weights 3/4 and 1/4, out = 3/4 (2, 1) + 1/4 (0, -1)
    = (1.5, 0.5), lse = ln(3 + 1)."""
    q = np.zeros((1, MLA_DIM), dtype=np.uint8)
    q[0, 0] = code(1.0)
    kv = np.zeros((2, MLA_DIM), dtype=np.uint8)
    kv[0, 0], kv[0, 1] = code(2.0), code(1.0)
    kv[1, 1] = code(-1.0)
    p = one_request(kv, q, [0, 1], sm_scale=math.log(3.0) / 2)
    out, lse, _ = oracle.sparse_mla(p)
    want = np.zeros(MLA_VDIM)
    want[:2] = [1.5, 0.5]
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-15)
    assert lse[0, 0] == pytest.approx(math.log(4.0), abs=1e-15)


def test_zero_query_gives_the_mean_of_the_listed_values():
    """q = 0: every score is 0, so out is the plain mean of the listed value
    rows (a repeated position counted twice) and lse = ln(listed count)."""
    rng = np.random.default_rng(3)
    n = 300
    kv = to_e4m3fn_bytes(rng.standard_normal((n, MLA_DIM), dtype=np.float32))
    q = np.zeros((4, MLA_DIM), dtype=np.uint8)
    listing = np.concatenate([rng.choice(n, 200, replace=False), [5, 5, -1, 7]])
    p = one_request(kv, q, listing, kv_scale=0.75, q_scale=3.0)
    out, lse, _ = oracle.sparse_mla(p)
    sel = listing[listing >= 0]
    want = dequant(kv[sel, :MLA_VDIM], 0.75).mean(axis=0)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], want, rtol=1e-13, atol=1e-15)
        assert lse[0, h] == pytest.approx(math.log(sel.size), abs=1e-13)


def test_one_dominant_score_selects_its_value_row():
    """A score 448 * 448 above the others: out is that token's value row to
    double precision (exp(-200704) underflows to 0) and lse is its score."""
    rng = np.random.default_rng(4)
    n = 64
    kv = to_e4m3fn_bytes(rng.standard_normal((n, MLA_DIM), dtype=np.float32))
    kv[:, 0] = code(0.0)
    kv[17, 0] = code(448.0)
    q = np.zeros((2, MLA_DIM), dtype=np.uint8)
    q[:, 0] = code(448.0)
    p = one_request(kv, q, np.arange(n))
    out, lse, _ = oracle.sparse_mla(p)
    for h in range(2):
        np.testing.assert_array_equal(out[0, h], dequant(kv[17, :MLA_VDIM], 1.0))
        assert lse[0, h] == 448.0 * 448.0


def sdpa(q, k, v, scale):
    """torch's scaled dot-product attention, float64 on the CPU: q [H, D],
    k [n, D], v [n, Dv] -> [H, Dv]."""
    H = q.shape[0]
    qt = torch.from_numpy(q)[None, :, None, :]
    kt = torch.from_numpy(k)[None, None].expand(1, H, -1, -1)
    vt = torch.from_numpy(v)[None, None].expand(1, H, -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("seed,n,sm", [(0, 37, 576 ** -0.5), (1, 700, 576 ** -0.5),
                                       (2, 129, 0.2)])
def test_dense_listing_matches_scaled_dot_product_attention(seed, n, sm):
    """Listing every token once is dense attention over the request: torch's
    routine on q_scale * q, kv_scale * k (576 wide) and the first 512 columns
    as values gives the same output."""
    rng = np.random.default_rng(seed)
    kv = to_e4m3fn_bytes(rng.standard_normal((n, MLA_DIM), dtype=np.float32))
    q = to_e4m3fn_bytes(rng.standard_normal((16, MLA_DIM), dtype=np.float32))
    listing = rng.permutation(n)
    p = one_request(kv, q, listing, q_scale=0.5, kv_scale=2.0, sm_scale=sm)
    out, _, _ = oracle.sparse_mla(p)
    k = dequant(kv, 2.0)
    want = sdpa(dequant(q, 0.5), k, k[:, :MLA_VDIM], sm)
    np.testing.assert_allclose(out[0], want, rtol=1e-10, atol=1e-12)


def test_repeated_listing_matches_attention_over_the_repeated_keys():
    """A position listed twice weighs twice: the same as dense attention over
    a key set that holds that token twice."""
    rng = np.random.default_rng(5)
    n = 50
    kv = to_e4m3fn_bytes(rng.standard_normal((n, MLA_DIM), dtype=np.float32))
    q = to_e4m3fn_bytes(rng.standard_normal((16, MLA_DIM), dtype=np.float32))
    listing = np.concatenate([np.arange(n), [3, 3, 10]])
    p = one_request(kv, q, listing, sm_scale=0.1)
    out, _, _ = oracle.sparse_mla(p)
    k = dequant(kv[listing], 1.0)
    np.testing.assert_allclose(out[0], sdpa(dequant(q, 1.0), k, k[:, :MLA_VDIM], 0.1),
                               rtol=1e-10, atol=1e-12)


def test_listing_order_page_size_and_holes_do_not_matter():
    """The same logical cache on pages of 1 and of 64 tokens (permuted pages),
    the listing shuffled and with -1 holes: identical results."""
    base = make_mla_problem(2, 3, 16, 1, [900, 2100], topk=512, seed=9, holes=0.1)
    out0, lse0, _ = oracle.sparse_mla(base)
    # repack onto pages of 64 under a random page permutation
    P = 64
    rng = np.random.default_rng(10)
    nb = [-(-c // P) for c in base.context_lens]
    perm = rng.permutation(sum(nb)).astype(np.int32)
    kv = np.full((sum(nb) * P, MLA_DIM), 0x7F, dtype=np.uint8)
    bt = np.full((2, max(nb)), -1, dtype=np.int32)
    off = 0
    for i, c in enumerate(base.context_lens):
        bt[i, : nb[i]] = perm[off: off + nb[i]]
        off += nb[i]
        for t in range(int(c)):
            kv[bt[i, t // P] * P + t % P] = base.kv[base.block_tables[i, t], 0]
    idx = base.indices.copy()
    for r in range(idx.shape[0]):
        idx[r] = rng.permutation(idx[r])
    paged = MlaProblem(q=base.q, kv=kv.reshape(-1, P, MLA_DIM), indices=idx,
                       context_lens=base.context_lens, block_tables=bt,
                       q_scale=base.q_scale, kv_scale=base.kv_scale, sm_scale=base.sm_scale,
                       bs=2, next_n=3, heads=16, block_size=P)
    out1, lse1, _ = oracle.sparse_mla(paged)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13)


def test_empty_rows_and_row_subsets():
    p = make_mla_problem(2, 2, 16, 1, [3, 0], topk=16, seed=2)
    assert (p.indices[2:] == -1).all()
    out, lse, _ = oracle.sparse_mla(p)
    assert (out[2:] == 0).all() and np.isneginf(lse[2:]).all()
    assert np.isfinite(lse[:2]).all()
    sub, lsub, _ = oracle.sparse_mla(p, rows=[1, 0])
    np.testing.assert_array_equal(sub, out[[1, 0]])
    np.testing.assert_array_equal(lsub, lse[[1, 0]])


def test_tolerance_aggregates_bound_what_they_should():
    """a_abs >= |out| (triangle inequality), d_abs >= 0, and s_abs bounds
    every score's magnitude, so lse <= max score + ln(count) <= s_abs + ln(count)."""
    p = make_mla_problem(1, 2, 16, 1, [1500], topk=1024, seed=7)
    out, lse, tol = oracle.sparse_mla(p, want_tol=True)
    assert (tol["a_abs"] >= np.abs(out) - 1e-12).all()
    assert (tol["d_abs"] >= 0).all()
    n = (p.indices >= 0).sum(axis=1)[:, None]
    assert (lse <= tol["s_abs"] + np.log(n) + 1e-9).all()


def test_position_outside_the_table_is_rejected():
    p = make_mla_problem(1, 1, 16, 1, [100], topk=8, seed=1)
    p.indices[0, 3] = p.max_blocks_per_seq  # past every table entry
    with pytest.raises(ValueError):
        oracle.sparse_mla(p)
