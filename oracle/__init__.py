"""CPU oracle for the FP8 MQA-logits indexer (paged decode and non-paged
prefill), its per-row top-k, and the sparse MLA decode that consumes the
top-k positions.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The product library never
loads it and it never loads the product library.

The arithmetic lives in ``pmqa_oracle.c`` (plain C, double precision); this
module only compiles it with gcc and marshals numpy arrays to it. Each function
there cites the passage of the pages it follows.

Parity pins: every function here is pinned by tests under ``tests/`` marked
``not gpu`` (fp8 code points and a full comparison with torch's e4m3fn decode,
one-hot and sign-flip closed forms, library GEMV special cases, invariants,
brute-force top-k; for the MLA decode a worked two-token example, the
uniform-weight and one-hot closed forms and torch's scaled dot-product
attention on a dense listing); none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pmqa_oracle.c")
_LIB = os.path.join(_HERE, "libpmqa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA) and return the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        lib.pmqa_ref_e4m3fn_table.argtypes = [P]
        lib.pmqa_ref_e4m3fn_table.restype = None
        lib.pmqa_ref_logits.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int64, P, P, P, ctypes.c_int]
        lib.pmqa_ref_logits.restype = ctypes.c_int
        lib.pmqa_ref_topk.argtypes = [P, ctypes.c_int64, P, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, P, ctypes.c_int]
        lib.pmqa_ref_topk.restype = ctypes.c_int
        lib.pmqa_ref_mqa_logits.argtypes = [P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int]
        lib.pmqa_ref_mqa_logits.restype = ctypes.c_int
        D, I = ctypes.c_double, ctypes.c_int
        lib.pmqa_ref_sparse_mla.argtypes = [P, D, P, D, P, P, P, I, I, I, I, I, ctypes.c_int64,
                                            D, P, P, P, P, P, I]
        lib.pmqa_ref_sparse_mla.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def e4m3fn_table() -> np.ndarray:
    out = np.empty(256, dtype=np.float64)
    _load().pmqa_ref_e4m3fn_table(_ptr(out))
    return out


def logits(prob, *, want64: bool = False, want_tol: bool = False, nthreads: int | None = None):
    """Return (logits fp32, logits fp64 or None, tolerance fp64 or None).

    ``prob`` carries numpy arrays q, kv, weights, context_lens, block_tables and
    the sizes bs, next_n, heads, block_size, max_model_len.
    """
    lib = _load()
    q = np.ascontiguousarray(prob.q, dtype=np.uint8)
    kv = np.ascontiguousarray(prob.kv, dtype=np.uint8)
    w = np.ascontiguousarray(prob.weights, dtype=np.float32)
    ctx = np.ascontiguousarray(prob.context_lens, dtype=np.int32)
    bt = np.ascontiguousarray(prob.block_tables, dtype=np.int32)
    rows, mml = prob.bs * prob.next_n, prob.max_model_len
    out = np.empty((rows, mml), dtype=np.float32)
    out64 = np.empty((rows, mml), dtype=np.float64) if want64 else None
    tol = np.empty((rows, mml), dtype=np.float64) if want_tol else None
    P = prob.block_size
    num_blocks = kv.shape[0]
    assert kv.shape[1:] == (P, 132)
    rc = lib.pmqa_ref_logits(_ptr(q), _ptr(kv), _ptr(w), _ptr(ctx), _ptr(bt), prob.bs,
                             prob.next_n, prob.heads, q.shape[-1], P, num_blocks, bt.shape[1],
                             mml, _ptr(out), _ptr(out64), _ptr(tol),
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle pmqa_ref_logits failed with %d" % rc)
    return out, out64, tol


def mqa_logits(prob, *, want64: bool = False, want_tol: bool = False,
               nthreads: int | None = None):
    """Prefill (non-paged) logits: (fp32 [m, n], fp64 or None, tolerance or None).

    ``prob`` carries numpy arrays q [m, heads, 128], k [n, 128], k_scale [n],
    weights [m, heads], ks [m] and ke [m].
    """
    lib = _load()
    q = np.ascontiguousarray(prob.q, dtype=np.uint8)
    k = np.ascontiguousarray(prob.k, dtype=np.uint8)
    sc = np.ascontiguousarray(prob.k_scale, dtype=np.float32)
    w = np.ascontiguousarray(prob.weights, dtype=np.float32)
    ks = np.ascontiguousarray(prob.ks, dtype=np.int32)
    ke = np.ascontiguousarray(prob.ke, dtype=np.int32)
    m, heads = q.shape[0], q.shape[1]
    n = k.shape[0]
    assert k.shape[1] == q.shape[2] and sc.shape == (n,) and w.shape == (m, heads)
    assert ks.shape == (m,) and ke.shape == (m,)
    out = np.empty((m, n), dtype=np.float32)
    out64 = np.empty((m, n), dtype=np.float64) if want64 else None
    tol = np.empty((m, n), dtype=np.float64) if want_tol else None
    rc = lib.pmqa_ref_mqa_logits(_ptr(q), _ptr(k), _ptr(sc), _ptr(w), _ptr(ks), _ptr(ke), m, n,
                                 heads, q.shape[2], _ptr(out), _ptr(out64), _ptr(tol),
                                 nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle pmqa_ref_mqa_logits failed with %d" % rc)
    return out, out64, tol


def topk(vals: np.ndarray, context_lens, next_n: int, k: int, *, nthreads: int | None = None):
    """Row top-k over the causal window: int32 [rows, k], -1 past min(k, valid)."""
    lib = _load()
    v = np.ascontiguousarray(vals, dtype=np.float64)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    rows, width = v.shape
    assert rows == ctx.shape[0] * next_n
    idx = np.empty((rows, k), dtype=np.int32)
    rc = lib.pmqa_ref_topk(_ptr(v), width, _ptr(ctx), ctx.shape[0], next_n, k, _ptr(idx),
                           nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle pmqa_ref_topk failed with %d" % rc)
    return idx


def valid_len(context_len: int, next_n: int, j: int) -> int:
    """Entries of draft row j that the causal window admits."""
    return max(0, min(context_len - next_n + j + 1, context_len))


def sparse_mla(prob, *, rows=None, want_tol: bool = False, nthreads: int | None = None):
    """Sparse MLA decode of ``prob`` (a synth.mla.MlaProblem, or any object
    with its fields): (out [R, heads, 512] fp64, lse [R, heads] fp64, tol)
    where tol is None or a dict of the per-entry aggregates a_abs, d_abs
    [R, heads, 512] and s_abs [R, heads]. ``rows`` restricts the call to those
    query rows (in that order)."""
    lib = _load()
    nn = prob.next_n
    all_rows = np.arange(prob.bs * nn) if rows is None else np.asarray(rows, dtype=np.int64)
    q = np.ascontiguousarray(prob.q.reshape(prob.bs * nn, prob.heads, -1)[all_rows],
                             dtype=np.uint8)
    idx = np.ascontiguousarray(prob.indices[all_rows], dtype=np.int32)
    req = np.ascontiguousarray(all_rows // nn, dtype=np.int32)
    kv = np.ascontiguousarray(prob.kv, dtype=np.uint8)
    bt = np.ascontiguousarray(prob.block_tables, dtype=np.int32)
    R, H = q.shape[0], q.shape[1]
    assert q.shape[2] == 576 and kv.shape[2] == 576
    out = np.empty((R, H, 512), dtype=np.float64)
    lse = np.empty((R, H), dtype=np.float64)
    a_abs = np.empty_like(out) if want_tol else None
    d_abs = np.empty_like(out) if want_tol else None
    s_abs = np.empty_like(lse) if want_tol else None
    rc = lib.pmqa_ref_sparse_mla(_ptr(q), prob.q_scale, _ptr(kv), prob.kv_scale, _ptr(idx),
                                 _ptr(req), _ptr(bt), R, H, idx.shape[1], kv.shape[1],
                                 bt.shape[1], kv.shape[0], prob.sm_scale, _ptr(out), _ptr(lse),
                                 _ptr(a_abs), _ptr(d_abs), _ptr(s_abs),
                                 nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle pmqa_ref_sparse_mla failed with %d" % rc)
    tol = dict(a_abs=a_abs, d_abs=d_abs, s_abs=s_abs) if want_tol else None
    return out, lse, tol
