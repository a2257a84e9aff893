"""ctypes binding of libpmqa (include/pmqa.h). Argument marshalling only.

Functions carry the C names. Tensors are torch CUDA tensors; torch supplies
device memory and the current stream, every step of the computation runs in
the library's kernels. There is no CPU path: if the library is missing,
``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

PMQA_OK = 0
PMQA_ERR_INVALID_ARG = -1
PMQA_ERR_UNSUPPORTED = -2
PMQA_ERR_WORKSPACE = -3
PMQA_ERR_CUDA = -4
PMQA_ERR_DEVICE = -5

PMQA_DEV_BAD_BLOCK_ID = 0x1
PMQA_DEV_BAD_CONTEXT = 0x2
PMQA_DEV_TIMEOUT = 0x4
PMQA_DEV_OVERFLOW = 0x8
PMQA_DEV_INTERNAL = 0x10

PMQA_OP_LOGITS = 0
PMQA_OP_TOPK = 1
PMQA_OP_LOGITS_TOPK = 2
PMQA_OP_MQA_LOGITS = 3

PMQA_STAGE_SCORE = 1
PMQA_STAGE_SELECT = 2

EXPORTED = (
    "pmqa_workspace_bytes", "pmqa_workspace_init", "pmqa_logits", "pmqa_topk",
    "pmqa_logits_topk", "pmqa_logits_topk_stages", "pmqa_logits_topk_noalloc",
    "pmqa_logits_topk_range",
    "pmqa_mqa_logits", "pmqa_topk_merge", "pmqa_sparse_mla_workspace_bytes",
    "pmqa_sparse_mla_decode", "pmqa_sparse_mla_decode_range", "pmqa_sparse_mla_merge",
    "pmqa_gather_probe", "pmqa_read_device_status", "pmqa_status_string", "pmqa_version",
)


class PmqaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {code} ({status_string(code)})")


class Problem(ctypes.Structure):
    """Mirror of struct pmqa_problem."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("kv_cache", ctypes.c_void_p),
        ("weights", ctypes.c_void_p),
        ("context_lens", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p),
        ("bs", ctypes.c_int32),
        ("next_n", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("max_model_len", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
    ]


class MqaProblem(ctypes.Structure):
    """Mirror of struct pmqa_mqa_problem."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("weights", ctypes.c_void_p),
        ("ks", ctypes.c_void_p),
        ("ke", ctypes.c_void_p),
        ("m", ctypes.c_int32),
        ("n", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
    ]


class MlaProblem(ctypes.Structure):
    """Mirror of struct pmqa_mla_problem."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("kv_cache", ctypes.c_void_p),
        ("indices", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p),
        ("q_scale", ctypes.c_float),
        ("kv_scale", ctypes.c_float),
        ("sm_scale", ctypes.c_float),
        ("bs", ctypes.c_int32),
        ("next_n", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libpmqa.so (built by build.build()); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise FileNotFoundError(
            f"{path} is missing: build it with sparse_attention_indexer_pmqa_gb300.build.build()")
    lib = ctypes.CDLL(path)
    V, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    PP = ctypes.POINTER(Problem)
    PM = ctypes.POINTER(MqaProblem)
    PL = ctypes.POINTER(MlaProblem)
    sig = {
        "pmqa_workspace_bytes": ([I32, I32, I32, I32, ctypes.c_int], SZ),
        "pmqa_workspace_init": ([V, SZ, V], ctypes.c_int),
        "pmqa_logits": ([PP, V, V, SZ, V], ctypes.c_int),
        "pmqa_topk": ([V, V, I32, I32, I32, I32, V, V, V, SZ, V], ctypes.c_int),
        "pmqa_logits_topk": ([PP, I32, V, V, V, V, SZ, V], ctypes.c_int),
        "pmqa_logits_topk_stages": ([PP, I32, V, V, V, V, SZ, V, I32], ctypes.c_int),
        "pmqa_logits_topk_noalloc": ([PP, I32, V, V, V, V], ctypes.c_int),
        "pmqa_logits_topk_range": ([PP, V, V, I32, V, V, V, SZ, V], ctypes.c_int),
        "pmqa_mqa_logits": ([PM, V, V, SZ, V], ctypes.c_int),
        "pmqa_topk_merge": ([V, V, I32, I32, I32, I32, V, V, V], ctypes.c_int),
        "pmqa_sparse_mla_workspace_bytes": ([I32], SZ),
        "pmqa_sparse_mla_decode": ([PL, V, V, V, SZ, V], ctypes.c_int),
        "pmqa_sparse_mla_decode_range": ([PL, V, V, V, V, V, SZ, V], ctypes.c_int),
        "pmqa_sparse_mla_merge": ([V, V, I32, I32, I32, V, V, V], ctypes.c_int),
        "pmqa_gather_probe": ([V, ctypes.c_uint64, V, I64, I32, I32, V, V], ctypes.c_int),
        "pmqa_read_device_status": ([V, V], ctypes.c_int),
        "pmqa_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "pmqa_version": ([], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    del I64
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().pmqa_status_string(code).decode()


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(code: int, what: str) -> None:
    if code != PMQA_OK:
        raise PmqaError(code, what)


def make_problem(q, kv_cache, weights, context_lens, block_tables, max_model_len: int) -> Problem:
    """Fill a pmqa_problem from tensors shaped as in the C header."""
    bs, next_n, heads, head_dim = q.shape
    num_blocks, block_size = kv_cache.shape[0], kv_cache.shape[1]
    assert kv_cache.shape[-1] == head_dim + 4, "kv rows hold head_dim fp8 bytes + fp32 scale"
    for t in (q, kv_cache, weights, context_lens, block_tables):
        assert t.is_cuda and t.is_contiguous()
    return Problem(
        q=q.data_ptr(), kv_cache=kv_cache.data_ptr(), weights=weights.data_ptr(),
        context_lens=context_lens.data_ptr(), block_tables=block_tables.data_ptr(),
        bs=bs, next_n=next_n, heads=heads, head_dim=head_dim, block_size=block_size,
        max_blocks_per_seq=block_tables.shape[1], max_model_len=max_model_len,
        num_blocks=num_blocks)


def pmqa_workspace_bytes(bs: int, next_n: int, max_model_len: int, k: int, op: int) -> int:
    return int(load().pmqa_workspace_bytes(bs, next_n, max_model_len, k, op))


def workspace(bs: int, next_n: int, max_model_len: int, k: int, op: int, device=None, stream=None):
    """A zero-initialised workspace tensor for the given operation."""
    import torch

    n = pmqa_workspace_bytes(bs, next_n, max_model_len, k, op)
    if n == 0:
        raise PmqaError(PMQA_ERR_INVALID_ARG, "pmqa_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    pmqa_workspace_init(ws, stream=stream)
    return ws


def pmqa_workspace_init(ws, stream=None) -> None:
    _check(load().pmqa_workspace_init(_ptr(ws), ws.numel(), _stream(stream)),
           "pmqa_workspace_init")


def pmqa_logits(q, kv_cache, weights, context_lens, block_tables, max_model_len: int, *,
                out=None, ws=None, stream=None):
    """fp32 logits [bs*next_n, max_model_len]."""
    import torch

    p = make_problem(q, kv_cache, weights, context_lens, block_tables, max_model_len)
    rows = p.bs * p.next_n
    if out is None:
        out = torch.empty((rows, max_model_len), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(p.bs, p.next_n, max_model_len, 0, PMQA_OP_LOGITS, q.device, stream)
    _check(load().pmqa_logits(ctypes.byref(p), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "pmqa_logits")
    return out


def pmqa_topk(logits, context_lens, next_n: int, k: int, *, idx=None, vals=None,
              want_vals: bool = False, ws=None, stream=None):
    """int32 positions [rows, k] (and fp32 values) of each row's top-k."""
    import torch

    rows, mml = logits.shape
    bs = context_lens.shape[0]
    assert rows == bs * next_n
    if idx is None:
        idx = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    if vals is None and want_vals:
        vals = torch.empty((rows, k), dtype=torch.float32, device=logits.device)
    if ws is None:
        ws = workspace(bs, next_n, mml, k, PMQA_OP_TOPK, logits.device, stream)
    _check(load().pmqa_topk(_ptr(logits), _ptr(context_lens), bs, next_n, mml, k, _ptr(idx),
                            _ptr(vals), _ptr(ws), ws.numel(), _stream(stream)), "pmqa_topk")
    return (idx, vals) if want_vals or vals is not None else idx


def pmqa_logits_topk(q, kv_cache, weights, context_lens, block_tables, max_model_len: int,
                     k: int, *, idx=None, vals=None, logits=None, want_vals: bool = False,
                     ws=None, stream=None):
    """Fused logits + top-k; returns idx, or (idx, vals) when values are asked for."""
    import torch

    p = make_problem(q, kv_cache, weights, context_lens, block_tables, max_model_len)
    rows = p.bs * p.next_n
    if idx is None:
        idx = torch.empty((rows, k), dtype=torch.int32, device=q.device)
    if vals is None and want_vals:
        vals = torch.empty((rows, k), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(p.bs, p.next_n, max_model_len, k, PMQA_OP_LOGITS_TOPK, q.device, stream)
    _check(load().pmqa_logits_topk(ctypes.byref(p), k, _ptr(idx), _ptr(vals), _ptr(logits),
                                   _ptr(ws), ws.numel(), _stream(stream)), "pmqa_logits_topk")
    return (idx, vals) if want_vals or vals is not None else idx


def pmqa_logits_topk_stages(q, kv_cache, weights, context_lens, block_tables, max_model_len: int,
                            k: int, stages: int, *, idx, ws, vals=None, logits=None,
                            stream=None):
    """One or both launches of the fused call (PMQA_STAGE_SCORE, then
    PMQA_STAGE_SELECT with the same arguments and workspace)."""
    p = make_problem(q, kv_cache, weights, context_lens, block_tables, max_model_len)
    _check(load().pmqa_logits_topk_stages(ctypes.byref(p), k, _ptr(idx), _ptr(vals), _ptr(logits),
                                          _ptr(ws), ws.numel(), _stream(stream), stages),
           "pmqa_logits_topk_stages")
    return idx


def pmqa_logits_topk_noalloc(q, kv_cache, weights, context_lens, block_tables,
                             max_model_len: int, k: int, *, idx, vals=None, logits=None,
                             stream=None):
    """Fused logits + top-k with the library's built-in device scratch; the
    caller passes every output buffer, nothing is allocated."""
    p = make_problem(q, kv_cache, weights, context_lens, block_tables, max_model_len)
    _check(load().pmqa_logits_topk_noalloc(ctypes.byref(p), k, _ptr(idx), _ptr(vals), _ptr(logits),
                                           _stream(stream)), "pmqa_logits_topk_noalloc")
    return idx


def pmqa_logits_topk_range(q, kv_cache, weights, context_lens, block_tables, max_model_len: int,
                           k: int, token_begin, token_end, *, idx=None, vals=None,
                           want_vals: bool = False, ws=None, stream=None):
    """The fused call on the slice [token_begin[i], token_end[i]) of each
    request's tokens; positions in idx are the requests' own (global) ones."""
    import torch

    p = make_problem(q, kv_cache, weights, context_lens, block_tables, max_model_len)
    rows = p.bs * p.next_n
    for t in (token_begin, token_end):
        assert t.is_cuda and t.is_contiguous() and t.dtype == torch.int32 and t.numel() == p.bs
    if idx is None:
        idx = torch.empty((rows, k), dtype=torch.int32, device=q.device)
    if vals is None and want_vals:
        vals = torch.empty((rows, k), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(p.bs, p.next_n, max_model_len, k, PMQA_OP_LOGITS_TOPK, q.device, stream)
    _check(load().pmqa_logits_topk_range(ctypes.byref(p), _ptr(token_begin), _ptr(token_end), k,
                                         _ptr(idx), _ptr(vals), _ptr(ws), ws.numel(),
                                         _stream(stream)), "pmqa_logits_topk_range")
    return (idx, vals) if want_vals or vals is not None else idx


def make_mqa_problem(q, k, k_scale, weights, ks, ke) -> MqaProblem:
    """Fill a pmqa_mqa_problem from tensors shaped as in the C header."""
    m, heads, head_dim = q.shape
    n = k.shape[0]
    assert k.shape[1] == head_dim and k_scale.shape[0] == n
    for t in (q, k, k_scale, weights, ks, ke):
        assert t.is_cuda and t.is_contiguous()
    return MqaProblem(q=q.data_ptr(), k=k.data_ptr(), k_scale=k_scale.data_ptr(),
                      weights=weights.data_ptr(), ks=ks.data_ptr(), ke=ke.data_ptr(),
                      m=m, n=n, heads=heads, head_dim=head_dim)


def pmqa_mqa_logits(q, k, k_scale, weights, ks, ke, *, out=None, ws=None, stream=None):
    """Prefill logits fp32 [m, n] over the rows' key ranges [ks, ke)."""
    import torch

    p = make_mqa_problem(q, k, k_scale, weights, ks, ke)
    if out is None:
        out = torch.empty((p.m, p.n), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(p.m, 1, p.n, 0, PMQA_OP_MQA_LOGITS, q.device, stream)
    _check(load().pmqa_mqa_logits(ctypes.byref(p), _ptr(out), _ptr(ws), ws.numel(),
                                  _stream(stream)), "pmqa_mqa_logits")
    return out


def pmqa_topk_merge(idx, vals, k: int, *, out_idx=None, out_vals=None, want_vals: bool = False,
                    stream=None):
    """Top-k per row of the union of candidate lists idx/vals [lists, rows, k_in]
    (-1 marks an empty slot); returns out_idx [rows, k] (and out_vals)."""
    import torch

    lists, rows, k_in = idx.shape
    assert vals.shape == idx.shape and idx.is_contiguous() and vals.is_contiguous()
    if out_idx is None:
        out_idx = torch.empty((rows, k), dtype=torch.int32, device=idx.device)
    if out_vals is None and want_vals:
        out_vals = torch.empty((rows, k), dtype=torch.float32, device=idx.device)
    _check(load().pmqa_topk_merge(_ptr(idx), _ptr(vals), lists, rows, k_in, k, _ptr(out_idx),
                                  _ptr(out_vals), _stream(stream)), "pmqa_topk_merge")
    return (out_idx, out_vals) if want_vals or out_vals is not None else out_idx


def make_mla_problem(q, kv_cache, indices, block_tables, next_n: int, q_scale: float,
                     kv_scale: float, sm_scale: float) -> MlaProblem:
    """Fill a pmqa_mla_problem from tensors shaped as in the C header (q may
    also be given as [bs, next_n, heads, 576])."""
    bs = block_tables.shape[0]
    heads, head_dim = q.shape[-2], q.shape[-1]
    rows = q.numel() // (heads * head_dim)
    assert rows == bs * next_n and indices.shape[0] == rows
    num_blocks, block_size = kv_cache.shape[0], kv_cache.shape[1]
    assert kv_cache.shape[-1] == head_dim
    for t in (q, kv_cache, indices, block_tables):
        assert t.is_cuda and t.is_contiguous()
    return MlaProblem(q=q.data_ptr(), kv_cache=kv_cache.data_ptr(), indices=indices.data_ptr(),
                      block_tables=block_tables.data_ptr(), q_scale=q_scale, kv_scale=kv_scale,
                      sm_scale=sm_scale, bs=bs, next_n=next_n, heads=heads, head_dim=head_dim,
                      v_head_dim=512, topk=indices.shape[1], block_size=block_size,
                      max_blocks_per_seq=block_tables.shape[1], num_blocks=num_blocks)


def pmqa_sparse_mla_workspace_bytes(rows: int) -> int:
    return int(load().pmqa_sparse_mla_workspace_bytes(rows))


def mla_workspace(rows: int, device=None, stream=None):
    """A zero-initialised workspace for pmqa_sparse_mla_decode."""
    import torch

    n = pmqa_sparse_mla_workspace_bytes(rows)
    if n == 0:
        raise PmqaError(PMQA_ERR_INVALID_ARG, "pmqa_sparse_mla_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    pmqa_workspace_init(ws, stream=stream)
    return ws


def pmqa_sparse_mla_decode(q, kv_cache, indices, block_tables, next_n: int, q_scale: float,
                           kv_scale: float, sm_scale: float, *, out=None, lse=None,
                           want_lse: bool = False, ws=None, stream=None):
    """Sparse MLA decode over the listed positions: bf16 out [rows, heads, 512]
    (and fp32 lse [rows, heads] when asked for or given)."""
    import torch

    p = make_mla_problem(q, kv_cache, indices, block_tables, next_n, q_scale, kv_scale, sm_scale)
    rows = p.bs * p.next_n
    if out is None:
        out = torch.empty((rows, p.heads, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((rows, p.heads), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = mla_workspace(rows, q.device, stream)
    _check(load().pmqa_sparse_mla_decode(ctypes.byref(p), _ptr(out), _ptr(lse), _ptr(ws),
                                         ws.numel(), _stream(stream)), "pmqa_sparse_mla_decode")
    return (out, lse) if want_lse or lse is not None else out


def pmqa_sparse_mla_decode_range(q, kv_cache, indices, block_tables, next_n: int, q_scale: float,
                                 kv_scale: float, sm_scale: float, token_begin, token_end, *,
                                 out=None, lse=None, ws=None, stream=None):
    """The decode over each request's slice [token_begin[i], token_end[i]) of
    its tokens: (bf16 out [rows, heads, 512], fp32 lse [rows, heads])."""
    import torch

    p = make_mla_problem(q, kv_cache, indices, block_tables, next_n, q_scale, kv_scale, sm_scale)
    rows = p.bs * p.next_n
    for t in (token_begin, token_end):
        assert t.is_cuda and t.is_contiguous() and t.dtype == torch.int32 and t.numel() == p.bs
    if out is None:
        out = torch.empty((rows, p.heads, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((rows, p.heads), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = mla_workspace(rows, q.device, stream)
    _check(load().pmqa_sparse_mla_decode_range(ctypes.byref(p), _ptr(token_begin), _ptr(token_end),
                                               _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                               _stream(stream)), "pmqa_sparse_mla_decode_range")
    return out, lse


def pmqa_sparse_mla_merge(outs, lses, *, out=None, lse=None, stream=None):
    """LSE-weighted merge of partial decodes outs [parts, rows, heads, 512]
    (bf16) with lses [parts, rows, heads]; returns (out, lse)."""
    import torch

    parts, rows, heads, vdim = outs.shape
    assert lses.shape == (parts, rows, heads) and vdim == 512
    assert outs.is_contiguous() and lses.is_contiguous() and outs.dtype == torch.bfloat16
    if out is None:
        out = torch.empty((rows, heads, vdim), dtype=torch.bfloat16, device=outs.device)
    if lse is None:
        lse = torch.empty((rows, heads), dtype=torch.float32, device=outs.device)
    _check(load().pmqa_sparse_mla_merge(_ptr(outs), _ptr(lses), parts, rows, heads, _ptr(out),
                                        _ptr(lse), _stream(stream)), "pmqa_sparse_mla_merge")
    return out, lse


def pmqa_gather_probe(pool, rows, row_pitch, method, *, out=None, stream=None):
    """Read the pool's rows `rows` (int32) as 16-byte aligned windows by one
    of three issue methods (a timing aid; include/pmqa.h). Returns `out`
    (uint32 [2] viewed as int32: status bits, XOR of what was read), which
    accumulates over calls when passed in."""
    import torch

    assert rows.dtype == torch.int32 and rows.is_contiguous() and pool.is_contiguous()
    if out is None:
        out = torch.zeros(2, dtype=torch.int32, device=pool.device)
    _check(load().pmqa_gather_probe(_ptr(pool), pool.numel() * pool.element_size(), _ptr(rows),
                                    rows.numel(), row_pitch, method, _ptr(out), _stream(stream)),
           "pmqa_gather_probe")
    return out


def pmqa_read_device_status(ws, stream=None) -> int:
    rc = load().pmqa_read_device_status(_ptr(ws), _stream(stream))
    if rc < 0:
        raise PmqaError(rc, "pmqa_read_device_status")
    return rc


def pmqa_version() -> int:
    return int(load().pmqa_version())
