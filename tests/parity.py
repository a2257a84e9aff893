"""Comparison rules between the CUDA path and the oracle.

Logits: the -inf pattern must match exactly; every finite entry must satisfy
|gpu - oracle| <= 1e-3 * (1 + sum_h |w_h| |x_h|) (the oracle's tolerance array).
Top-k: per row the selected set has exactly min(k, valid_len) distinct positions
inside the window and -1 after; it equals the oracle's set except for positions
whose oracle logit lies within that position's own tolerance of the oracle's
k-th value: a position chosen in place of an oracle pick sits at most tol below
the k-th value, and an oracle pick left out sits at most tol above it.
"""

from __future__ import annotations

import numpy as np


def valid_len(ctx: int, nn: int, j: int) -> int:
    return max(0, min(ctx - nn + j + 1, ctx))


def check_logits(gpu: np.ndarray, ref: np.ndarray, tol: np.ndarray) -> float:
    """Returns the largest |error| / tolerance over finite entries."""
    assert gpu.shape == ref.shape
    ninf_g, ninf_r = np.isneginf(gpu), np.isneginf(ref)
    bad = np.argwhere(ninf_g != ninf_r)
    assert bad.size == 0, f"-inf pattern differs at {bad[:5].tolist()} (of {len(bad)})"
    fin = ~ninf_r
    assert np.all(np.isfinite(gpu[fin])), "non-finite logits where the oracle is finite"
    if not fin.any():
        return 0.0
    err = np.abs(gpu[fin].astype(np.float64) - ref[fin].astype(np.float64))
    ratio = err / tol[fin]
    worst = float(ratio.max())
    assert worst <= 1.0, f"logit error {worst:.3g} x tolerance (max abs {err.max():.3g})"
    return worst


def check_topk_rows(idx: np.ndarray, ref64: np.ndarray, tol: np.ndarray, ctx, nn: int, k: int,
                    vals: np.ndarray | None = None, begin=None, end=None) -> int:
    """Check GPU top-k against oracle values; returns the number of tie swaps.
    With begin/end (per request) the rows choose only among the admitted
    positions inside [begin_i, end_i)."""
    ctx = np.asarray(ctx)
    swaps = 0
    for r in range(idx.shape[0]):
        i, j = divmod(r, nn)
        n = valid_len(int(ctx[i]), nn, j)
        lo = 0
        if begin is not None:
            lo = min(max(int(begin[i]), 0), int(ctx[i]))
            n = max(lo, min(n, max(lo, min(int(end[i]), int(ctx[i])))))
        ke = min(k, n - lo)
        sel = idx[r, :ke]
        assert np.all(idx[r, ke:] == -1), f"row {r}: slots past k_eff not -1"
        assert np.all((sel >= lo) & (sel < n)), f"row {r}: position outside the window"
        assert len(np.unique(sel)) == ke, f"row {r}: repeated positions"
        if ke == 0:
            continue
        row = np.full(n, -np.inf)
        row[lo:n] = ref64[r, lo:n]
        order = np.lexsort((np.arange(n), -row))
        ref_set = order[:ke]
        kth = row[ref_set[-1]]
        g, o = set(sel.tolist()), set(ref_set.tolist())
        extra, missing = g - o, o - g
        for p in extra:
            assert row[p] >= kth - float(tol[r, p]), \
                f"row {r}: chose {p} ({row[p]}) more than its tolerance below the k-th {kth}"
        for p in missing:
            assert row[p] <= kth + float(tol[r, p]), \
                f"row {r}: missed {p} ({row[p]}) more than its tolerance above the k-th {kth}"
        swaps += len(extra)
        if vals is not None:
            assert np.all(np.isneginf(vals[r, ke:])), f"row {r}: padding values not -inf"
            err = np.abs(vals[r, :ke].astype(np.float64) - row[sel])
            assert np.all(err <= tol[r, sel]), f"row {r}: returned values off by {err.max()}"
    return swaps


def check_topk_exact(idx: np.ndarray, vals32: np.ndarray, ctx, nn: int, k: int) -> None:
    """Top-k of given fp32 rows: the chosen values equal the oracle's as a multiset."""
    ctx = np.asarray(ctx)
    for r in range(idx.shape[0]):
        i, j = divmod(r, nn)
        n = valid_len(int(ctx[i]), nn, j)
        ke = min(k, n)
        sel = idx[r, :ke]
        assert np.all(idx[r, ke:] == -1)
        assert np.all((sel >= 0) & (sel < n))
        assert len(np.unique(sel)) == ke
        want = np.sort(vals32[r, :n])[::-1][:ke]
        got = np.sort(vals32[r, sel])[::-1]
        assert np.array_equal(got, want), f"row {r}: selected values differ from the top-{ke}"


def check_mla(out, lse, ref, lref, tol, parts: int = 1):
    """Sparse MLA decode outputs against the oracle's. Tolerance per output
    entry, from the kernel's arithmetic: scores within e_s = 2^-9 * s_abs of
    exact (fp8 products summed on the tensor cores) move an output by at most
    e_s * d_abs; the softmax weights enter the second product as two fp8 terms
    (relative error 2^-8), at most 2^-7 * a_abs with margin; the bf16 output
    rounds by 2^-9 relative, 2^-8 |out| with margin. lse within e_s + 1e-4;
    rows with no listed position exactly 0 and -inf. A merge of `parts` > 1
    partial decodes (each rounded to bf16 before the merge) adds 2^-8 * a_abs.
    Returns (worst error as a
    fraction of its bound, cos_diff = 1 - 2 <x, y> / (|x|^2 + |y|^2), the
    agreement measure the pages quote for MLA decode)."""
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    e_s = 2.0 ** -9 * tol["s_abs"]
    bound = e_s[..., None] * tol["d_abs"] + 2.0 ** -7 * tol["a_abs"] + 2.0 ** -8 * np.abs(ref) + 1e-6
    if parts > 1:
        bound = bound + 2.0 ** -8 * tol["a_abs"]
    err = np.abs(out - ref)
    bad = err > bound
    assert not bad.any(), (
        f"{int(bad.sum())} outputs beyond tolerance; worst excess "
        f"{float((err - bound).max()):.3g} at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    empty = np.isneginf(lref)
    assert np.array_equal(np.isneginf(lse), empty), "-inf pattern of lse"
    assert (out[empty] == 0).all()
    fin = ~empty
    lerr = np.abs(lse[fin] - lref[fin])
    assert (lerr <= e_s[fin] + 1e-4).all(), f"lse error {lerr.max():.3g}"
    den = (out * out).sum() + (ref * ref).sum()
    cos_diff = 1.0 - 2.0 * (out * ref).sum() / den if den > 0 else 0.0
    return float((err / bound).max()), float(cos_diff)
