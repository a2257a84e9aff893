"""The acceptance rules of tests/parity.py, checked on planted results (CPU).

A top-k answer may differ from the oracle's set only at positions whose oracle
logit lies within that position's own tolerance of the k-th value; logits must
keep the -inf pattern exactly and every finite entry within its tolerance.
"""

import numpy as np
import pytest

from tests.parity import check_logits, check_topk_rows


def _row(n=64, seed=0):
    rng = np.random.default_rng(seed)
    vals = rng.permutation(n).astype(np.float64)  # distinct: 0 .. n-1
    return vals[None, :], np.full((1, n), 0.25)


def _oracle_pick(row, k):
    return np.argsort(-row[0], kind="stable")[:k].astype(np.int32)


def test_exact_set_passes_and_padding_is_checked():
    r64, tol = _row()
    k = 10
    idx = _oracle_pick(r64, k)[None, :]
    assert check_topk_rows(idx, r64, tol, [64], 1, k) == 0
    # ctx 8 < k: every valid position, then -1
    short = np.concatenate([_oracle_pick(r64[:, :8], 8), np.full(4, -1, np.int32)])[None, :]
    assert check_topk_rows(short, r64, tol, [8], 1, 12) == 0
    bad = short.copy()
    bad[0, -1] = 3
    with pytest.raises(AssertionError, match="past k_eff"):
        check_topk_rows(bad, r64, tol, [8], 1, 12)


def test_swap_within_the_tolerance_of_the_kth_value_passes():
    r64, tol = _row()
    k = 10
    idx = _oracle_pick(r64, k)
    kth_pos = idx[-1]
    below = int(np.flatnonzero(r64[0] == r64[0, kth_pos] - 1)[0])
    # both the k-th and the next value lie 0.5 apart after this change, within 0.6
    r64b = r64.copy()
    r64b[0, below] = r64[0, kth_pos] - 0.5
    tolb = np.full_like(tol, 0.6)
    swapped = idx.copy()
    swapped[-1] = below
    assert check_topk_rows(swapped[None, :], r64b, tolb, [64], 1, k) == 1


def test_swap_beyond_the_tolerance_fails():
    r64, tol = _row()
    k = 10
    idx = _oracle_pick(r64, k)
    below = int(np.flatnonzero(r64[0] == r64[0, idx[-1]] - 1)[0])  # 1.0 below, tol 0.25
    swapped = idx.copy()
    swapped[-1] = below
    with pytest.raises(AssertionError, match="tolerance"):
        check_topk_rows(swapped[None, :], r64, tol, [64], 1, k)


def test_swap_within_twice_but_not_once_the_tolerance_fails():
    r64, tol = _row()
    k = 10
    idx = _oracle_pick(r64, k)
    below = int(np.flatnonzero(r64[0] == r64[0, idx[-1]] - 1)[0])
    tol2 = np.full_like(tol, 0.6)  # gap 1.0: inside 2 x 0.6, outside 0.6
    swapped = idx.copy()
    swapped[-1] = below
    with pytest.raises(AssertionError, match="tolerance"):
        check_topk_rows(swapped[None, :], r64, tol2, [64], 1, k)


def test_repeated_or_out_of_window_positions_fail():
    r64, tol = _row()
    k = 4
    idx = _oracle_pick(r64, k)
    rep = idx.copy()
    rep[1] = rep[0]
    with pytest.raises(AssertionError, match="repeated"):
        check_topk_rows(rep[None, :], r64, tol, [64], 1, k)
    out = idx.copy()
    out[0] = 64
    with pytest.raises(AssertionError, match="outside"):
        check_topk_rows(out[None, :], r64, tol, [64], 1, k)


def test_logit_rules():
    ref = np.array([[1.0, 2.0, -np.inf]], dtype=np.float32)
    tol = np.array([[0.1, 0.1, 0.1]])
    assert check_logits(ref.copy(), ref, tol) == 0.0
    off = ref.copy()
    off[0, 1] += 0.05
    assert check_logits(off, ref, tol) == pytest.approx(0.5, rel=1e-5)
    bad = ref.copy()
    bad[0, 0] += 0.2
    with pytest.raises(AssertionError, match="tolerance"):
        check_logits(bad, ref, tol)
    mask = ref.copy()
    mask[0, 2] = 0.0
    with pytest.raises(AssertionError, match="-inf pattern"):
        check_logits(mask, ref, tol)
