"""Pins for the prefill (non-paged) oracle.

The prefill definition is the decode one with the paging removed and one key
range per query row, so its strongest pin is the decode oracle (pinned in
test_oracle.py) on the same numbers laid out as one-token pages. The other
pins are closed forms, library GEMM special cases and invariants.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import make_prefill, pack_kv, Problem

pytestmark = pytest.mark.filterwarnings("ignore")


def torch_decode(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.float().double().numpy()


def as_decode_problem(p) -> Problem:
    """Query row r as request r (next_n 1, context min(ke_r, n)) over one-token
    pages that hold key t in block t: the decode problem with the same logits
    wherever ks_r <= 0."""
    m, n, H = p.m, p.n, p.heads
    ctx = np.clip(p.ke.astype(np.int64), 0, n).astype(np.int32)
    kv = pack_kv(p.k, p.k_scale, 1)
    bt = np.tile(np.arange(max(n, 1), dtype=np.int32), (m, 1))
    return Problem(q=p.q.reshape(m, 1, H, 128), kv=kv, weights=p.weights, context_lens=ctx,
                   block_tables=bt, bs=m, next_n=1, heads=H, block_size=1, max_model_len=n)


@pytest.mark.parametrize("H", [1, 4, 32])
def test_equals_decode_oracle_on_one_token_pages(H):
    p = make_prefill(24, 300, H, ranges="causal", seed=H, poison=False)
    out, o64, tol = oracle.mqa_logits(p, want64=True, want_tol=True)
    d = as_decode_problem(p)
    rout, r64, rtol = oracle.logits(d, want64=True, want_tol=True)
    assert np.array_equal(out, rout)
    assert np.array_equal(o64, r64)
    assert np.array_equal(tol, rtol)


def test_range_start_masks_and_keeps_the_rest():
    """Raising ks only turns entries below it to -inf; the rest are unchanged."""
    p = make_prefill(16, 200, 8, ranges="full", seed=7, poison=False)
    base, _, _ = oracle.mqa_logits(p)
    rng = np.random.default_rng(1)
    p.ks = rng.integers(0, 200, size=16).astype(np.int32)
    p.ke = np.maximum(p.ke, p.ks)
    got, _, _ = oracle.mqa_logits(p)
    for r in range(16):
        a, b = int(p.ks[r]), int(p.ke[r])
        assert np.all(np.isneginf(got[r, :a])) and np.all(np.isneginf(got[r, b:]))
        assert np.array_equal(got[r, a:b], base[r, a:b])


def test_ranges_outside_the_keys_clamp_and_empty_rows():
    p = make_prefill(6, 50, 2, ranges="full", seed=2, poison=False)
    base, _, _ = oracle.mqa_logits(p)
    p.ks = np.array([-5, 10, 30, 49, 60, -100], dtype=np.int32)
    p.ke = np.array([5, 10, 80, 50, 70, -50], dtype=np.int32)
    got, _, _ = oracle.mqa_logits(p)
    fin = np.isfinite(got)
    assert fin[0, :5].all() and not fin[0, 5:].any()
    assert not fin[1].any() and not fin[4].any() and not fin[5].any()
    assert fin[2, 30:].all() and not fin[2, :30].any()
    assert fin[3, 49] and fin[3].sum() == 1
    assert np.array_equal(got[fin], base[fin])


def test_all_ones_closed_form():
    """q = k = 1.0: x_h = 128 s_n, logit = 128 s_n sum_h w_h for s_n > 0, 0 for s_n <= 0."""
    H, m, n = 4, 3, 20
    p = make_prefill(m, n, H, ranges="full", seed=0, poison=False)
    p.q[:] = 0x38
    p.k[:] = 0x38
    p.weights[:] = np.array([0.5, 0.25, -1.0, 2.0], dtype=np.float32)
    p.k_scale[:] = np.linspace(-0.5, 0.5, n).astype(np.float32)
    _, o64, tol = oracle.mqa_logits(p, want64=True, want_tol=True)
    s = p.k_scale.astype(np.float64)
    expect = np.where(s > 0, 128.0 * s * 1.75, 0.0)
    for r in range(m):
        assert np.array_equal(o64[r], expect)
        np.testing.assert_allclose(tol[r], 1e-3 * (1 + 128 * np.abs(s) * 3.75), rtol=1e-15)


@pytest.mark.parametrize("d0", [0, 77, 127])
def test_one_hot_query_reads_one_key_column(d0):
    p = make_prefill(2, 64, 1, ranges="full", seed=d0, poison=False)
    p.q[:] = 0
    p.q[:, 0, d0] = 0x38
    p.weights[:] = 1.0
    out, o64, _ = oracle.mqa_logits(p, want64=True)
    expect = np.maximum(torch_decode(p.k[:, d0]) * p.k_scale.astype(np.float64), 0.0)
    assert np.array_equal(o64[0], expect) and np.array_equal(o64[1], expect)
    assert np.array_equal(out[0], expect.astype(np.float32))


def test_nonnegative_inputs_reduce_to_library_gemm():
    """q, k >= 0 and s > 0 keep every x >= 0, so the relu drops out and
    logits = s_n * ((w Q) K^T)[m, n], a library matrix product."""
    m, n, H = 12, 90, 8
    p = make_prefill(m, n, H, ranges="full", seed=11, poison=False)
    p.q &= 0x7F
    p.k &= 0x7F
    p.q[p.q == 0x7F] = 0x7E
    p.k[p.k == 0x7F] = 0x7E
    _, o64, _ = oracle.mqa_logits(p, want64=True)
    qd = torch_decode(p.q)                      # [m, H, 128]
    kd = torch_decode(p.k)                      # [n, 128]
    wq = np.einsum("mh,mhd->md", p.weights.astype(np.float64), qd)
    expect = (wq @ kd.T) * p.k_scale.astype(np.float64)[None, :]
    np.testing.assert_allclose(o64, expect, rtol=1e-12, atol=1e-12)


def test_packed_segments_match_per_segment_problems():
    """Packed sequences: each segment's rows equal the same rows computed on
    that segment's keys alone (shifted by its start)."""
    p = make_prefill(120, 120, 4, ranges="packed", seed=5, poison=False)
    out, _, _ = oracle.mqa_logits(p)
    starts = np.unique(p.ks)
    bounds = list(starts) + [120]
    for a, b in zip(bounds[:-1], bounds[1:]):
        sub = make_prefill(b - a, b - a, 4, ranges="full", seed=0, poison=False)
        sub.q = p.q[a:b].copy()
        sub.k = p.k[a:b].copy()
        sub.k_scale = p.k_scale[a:b].copy()
        sub.weights = p.weights[a:b].copy()
        sub.ks = np.zeros(b - a, dtype=np.int32)
        sub.ke = np.arange(1, b - a + 1, dtype=np.int32)
        so, _, _ = oracle.mqa_logits(sub)
        assert np.array_equal(out[a:b, a:b], so)
        assert np.all(np.isneginf(out[a:b, :a])) and np.all(np.isneginf(out[a:b, b:]))


def test_poisoned_keys_are_never_read():
    p = make_prefill(40, 256, 4, ranges="random", seed=9)
    out, _, _ = oracle.mqa_logits(p)
    assert not np.isnan(out).any()
    assert np.isfinite(out).sum() == p.pairs


def test_causal_generator_ranges():
    p = make_prefill(5, 12, 1, ranges="causal", seed=0)
    assert list(p.ks) == [0] * 5 and list(p.ke) == [8, 9, 10, 11, 12]
