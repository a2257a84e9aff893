"""Host-only checks of the C ABI: the library loads without a GPU, exports every
function include/pmqa.h declares, and rejects bad arguments before touching
the device."""

import ctypes
import os
import re

import pytest

from sparse_attention_indexer_pmqa_gb300 import build, pmqa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pmqa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pmqa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pmqa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(pmqa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert pmqa.pmqa_version() == 300
    assert pmqa.status_string(0) == "ok"
    assert pmqa.status_string(-3) == "workspace too small"
    assert pmqa.status_string(12345) == "unknown status"


def test_workspace_sizes(lib):
    assert pmqa.pmqa_workspace_bytes(4, 2, 1000, 2048, pmqa.PMQA_OP_LOGITS) == 256
    rows, mml = 8, 1000
    counters = 256 + 3 * 256  # status word, then three 256-aligned per-row counter arrays
    hist = rows * 2048 * 4  # per-row key histograms
    ties = -(-rows * mml * 8 // 256) * 256  # tie lists of (position, key)
    topk = pmqa.pmqa_workspace_bytes(4, 2, mml, 2048, pmqa.PMQA_OP_TOPK)
    assert topk == counters + hist + ties
    fused = pmqa.pmqa_workspace_bytes(4, 2, mml, 2048, pmqa.PMQA_OP_LOGITS_TOPK)
    assert fused == topk + rows * mml * 4  # plus the compact logits
    assert pmqa.pmqa_workspace_bytes(-1, 1, 10, 1, 0) == 0
    assert pmqa.pmqa_workspace_bytes(1, 1, 10, 1, 7) == 0


def _problem(**kw):
    # fake, suitably aligned device addresses: argument checks run before any CUDA call
    base = dict(q=0x10000, kv_cache=0x20000, weights=0x30000, context_lens=0x40000,
                block_tables=0x50000, bs=2, next_n=1, heads=64, head_dim=128, block_size=1,
                max_blocks_per_seq=64, max_model_len=64, num_blocks=128)
    base.update(kw)
    return pmqa.Problem(**base)


WS = ctypes.c_void_p(0x100000)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(heads=48), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(next_n=5), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(next_n=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(bs=-1), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(block_size=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(max_model_len=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(num_blocks=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(q=None), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(q=0x10004), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(weights=0x30008), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(kv_cache=0x20002), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(kv_cache=0x20004), pmqa.PMQA_ERR_INVALID_ARG),
])
def test_problem_validation(lib, kw, code):
    p = _problem(**kw)
    assert lib.pmqa_logits(ctypes.byref(p), ctypes.c_void_p(0x60000), WS, 1 << 20, None) == code
    assert lib.pmqa_logits_topk(ctypes.byref(p), 16, ctypes.c_void_p(0x70000), None, None, WS,
                                1 << 20, None) == code


def test_stage_flags(lib):
    p = _problem()
    need = pmqa.pmqa_workspace_bytes(2, 1, 64, 16, pmqa.PMQA_OP_LOGITS_TOPK)
    I = ctypes.c_void_p(0x70000)
    for bad in (0, 4, -1):
        assert lib.pmqa_logits_topk_stages(ctypes.byref(p), 16, I, None, None, WS, need, None,
                                           bad) == pmqa.PMQA_ERR_INVALID_ARG
    # the usual argument checks run for every stage choice
    assert lib.pmqa_logits_topk_stages(ctypes.byref(p), 16, None, None, None, WS, need, None,
                                       pmqa.PMQA_STAGE_SELECT) == pmqa.PMQA_ERR_INVALID_ARG
    assert lib.pmqa_logits_topk_stages(ctypes.byref(p), 16, I, None, None, WS, need - 1, None,
                                       pmqa.PMQA_STAGE_SCORE) == pmqa.PMQA_ERR_WORKSPACE


def test_null_problem_and_outputs(lib):
    assert lib.pmqa_logits(None, ctypes.c_void_p(0x60000), WS, 1 << 20, None) == -1
    p = _problem()
    assert lib.pmqa_logits(ctypes.byref(p), None, WS, 1 << 20, None) == -1
    assert lib.pmqa_logits_topk(ctypes.byref(p), 16, None, None, None, WS, 1 << 20, None) == -1
    assert lib.pmqa_logits_topk(ctypes.byref(p), 0, ctypes.c_void_p(0x70000), None, None, WS,
                                1 << 20, None) == -1


def test_workspace_checks(lib):
    p = _problem()
    out = ctypes.c_void_p(0x60000)
    assert lib.pmqa_logits(ctypes.byref(p), out, WS, 255, None) == pmqa.PMQA_ERR_WORKSPACE
    assert lib.pmqa_logits(ctypes.byref(p), out, ctypes.c_void_p(0x100010), 1 << 20, None) == -1
    need = pmqa.pmqa_workspace_bytes(2, 1, 64, 16, pmqa.PMQA_OP_LOGITS_TOPK)
    assert lib.pmqa_logits_topk(ctypes.byref(p), 16, ctypes.c_void_p(0x70000), None, None, WS,
                                need - 1, None) == pmqa.PMQA_ERR_WORKSPACE


def test_topk_validation(lib):
    L = ctypes.c_void_p(0x10000)
    C = ctypes.c_void_p(0x20000)
    I = ctypes.c_void_p(0x30000)
    need = pmqa.pmqa_workspace_bytes(2, 1, 64, 8, pmqa.PMQA_OP_TOPK)
    assert lib.pmqa_topk(L, C, 2, 1, 64, 0, I, None, WS, need, None) == -1
    assert lib.pmqa_topk(L, C, 2, 0, 64, 8, I, None, WS, need, None) == -1
    assert lib.pmqa_topk(L, C, 2, 1, 64, 8, I, None, WS, need - 1, None) == -3
    assert lib.pmqa_topk(None, C, 2, 1, 64, 8, I, None, WS, need, None) == -1
    assert lib.pmqa_topk(L, C, 2, 1, 64, 8, ctypes.c_void_p(0x30002), None, WS, need, None) == -1
    big = pmqa.pmqa_workspace_bytes(70000, 1, 64, 8, pmqa.PMQA_OP_TOPK)
    assert lib.pmqa_topk(L, C, 70000, 1, 64, 8, I, None, WS, big, None) == -2


def test_empty_batch_is_a_no_op(lib):
    p = _problem(bs=0, q=None)
    assert lib.pmqa_logits(ctypes.byref(p), ctypes.c_void_p(0x60000), WS, 1 << 20, None) == 0
    assert lib.pmqa_topk(None, None, 0, 1, 64, 8, None, None, WS, 1 << 20, None) == 0


def test_workspace_init_checks(lib):
    assert lib.pmqa_workspace_init(None, 1024, None) == -1
    assert lib.pmqa_workspace_init(ctypes.c_void_p(0x100004), 1024, None) == -1
    assert lib.pmqa_read_device_status(None, None) == -1


def _mqa(**kw):
    base = dict(q=0x10000, k=0x20000, k_scale=0x30000, weights=0x40000, ks=0x50000,
                ke=0x58000, m=8, n=256, heads=32, head_dim=128)
    base.update(kw)
    return pmqa.MqaProblem(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(heads=48), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(m=1 << 27, heads=16), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(n=(1 << 31) - 100), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(m=-1), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(n=-1), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(heads=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(q=None), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(ke=None), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(q=0x10008), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(k=0x20004), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(weights=0x40004), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(k_scale=0x30002), pmqa.PMQA_ERR_INVALID_ARG),
])
def test_mqa_problem_validation(lib, kw, code):
    p = _mqa(**kw)
    assert lib.pmqa_mqa_logits(ctypes.byref(p), ctypes.c_void_p(0x60000), WS, 1 << 20, None) == code


def test_mqa_workspace_and_empty_shapes(lib):
    assert pmqa.pmqa_workspace_bytes(0, 0, 0, 0, pmqa.PMQA_OP_MQA_LOGITS) == 256
    assert pmqa.pmqa_workspace_bytes(8, 1, 256, 0, pmqa.PMQA_OP_MQA_LOGITS) == 512
    assert pmqa.pmqa_workspace_bytes(129, 1, 9, 0, pmqa.PMQA_OP_MQA_LOGITS) == 256 + 512
    assert pmqa.pmqa_workspace_bytes(-1, 1, 9, 0, pmqa.PMQA_OP_MQA_LOGITS) == 0
    p = _mqa()
    out = ctypes.c_void_p(0x60000)
    need = pmqa.pmqa_workspace_bytes(8, 1, 256, 0, pmqa.PMQA_OP_MQA_LOGITS)
    assert lib.pmqa_mqa_logits(None, out, WS, need, None) == -1
    assert lib.pmqa_mqa_logits(ctypes.byref(p), None, WS, need, None) == -1
    assert lib.pmqa_mqa_logits(ctypes.byref(p), out, WS, need - 1, None) == pmqa.PMQA_ERR_WORKSPACE
    assert lib.pmqa_mqa_logits(ctypes.byref(p), out, ctypes.c_void_p(0x100010), need, None) == -1
    # nothing to compute: no pointer is needed and nothing is launched
    assert lib.pmqa_mqa_logits(ctypes.byref(_mqa(m=0, q=None)), None, WS, 256, None) == 0
    assert lib.pmqa_mqa_logits(ctypes.byref(_mqa(n=0, k=None)), None, WS, need, None) == 0


def _mla(**kw):
    base = dict(q=0x10000, kv_cache=0x20000, indices=0x30000, block_tables=0x40000,
                q_scale=0.5, kv_scale=2.0, sm_scale=0.04, bs=2, next_n=2, heads=16, head_dim=576,
                v_head_dim=512, topk=2048, block_size=1, max_blocks_per_seq=64, num_blocks=128)
    base.update(kw)
    return pmqa.MlaProblem(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(heads=32), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(head_dim=512), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(v_head_dim=576), pmqa.PMQA_ERR_UNSUPPORTED),
    (dict(bs=-1), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(next_n=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(topk=-1), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(block_size=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(max_blocks_per_seq=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(num_blocks=0), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(q_scale=float("nan")), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(sm_scale=float("inf")), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(q=None), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(indices=None), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(q=0x10008), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(kv_cache=0x20004), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(indices=0x30002), pmqa.PMQA_ERR_INVALID_ARG),
    (dict(block_tables=0x40001), pmqa.PMQA_ERR_INVALID_ARG),
])
def test_mla_problem_validation(lib, kw, code):
    need = pmqa.pmqa_sparse_mla_workspace_bytes(4)
    p = _mla(**kw)
    assert lib.pmqa_sparse_mla_decode(ctypes.byref(p), ctypes.c_void_p(0x60000), None, WS, need,
                                      None) == code


def test_mla_workspace_outputs_and_empty_batch(lib):
    need = pmqa.pmqa_sparse_mla_workspace_bytes(4)
    # status word, the parts' (m, l), the parts' outputs: two parts per CTA, at most 256 CTAs
    assert need == 256 + 2 * 256 * 16 * 2 * 4 + 2 * 256 * 16 * 512 * 4
    assert pmqa.pmqa_sparse_mla_workspace_bytes(-1) == 0
    p = _mla()
    out = ctypes.c_void_p(0x60000)
    assert lib.pmqa_sparse_mla_decode(None, out, None, WS, need, None) == -1
    assert lib.pmqa_sparse_mla_decode(ctypes.byref(p), None, None, WS, need, None) == -1
    assert lib.pmqa_sparse_mla_decode(ctypes.byref(p), ctypes.c_void_p(0x60002), None, WS, need,
                                      None) == -1
    assert lib.pmqa_sparse_mla_decode(ctypes.byref(p), out, ctypes.c_void_p(0x70002), WS, need,
                                      None) == -1
    assert lib.pmqa_sparse_mla_decode(ctypes.byref(p), out, None, WS, need - 1,
                                      None) == pmqa.PMQA_ERR_WORKSPACE
    assert lib.pmqa_sparse_mla_decode(ctypes.byref(p), out, None, ctypes.c_void_p(0x100010), need,
                                      None) == -1
    # no rows: nothing is read or launched
    empty = _mla(bs=0, q=None, kv_cache=None, indices=None, block_tables=None)
    assert lib.pmqa_sparse_mla_decode(ctypes.byref(empty), None, None, WS, need, None) == 0


def test_mla_range_and_merge_validation(lib):
    need = pmqa.pmqa_sparse_mla_workspace_bytes(4)
    p = _mla()
    out = ctypes.c_void_p(0x60000)
    B, E = ctypes.c_void_p(0x80000), ctypes.c_void_p(0x81000)
    assert lib.pmqa_sparse_mla_decode_range(ctypes.byref(p), None, E, out, None, WS, need,
                                            None) == -1
    assert lib.pmqa_sparse_mla_decode_range(ctypes.byref(p), B, None, out, None, WS, need,
                                            None) == -1
    assert lib.pmqa_sparse_mla_decode_range(ctypes.byref(p), ctypes.c_void_p(0x80002), E, out,
                                            None, WS, need, None) == -1
    assert lib.pmqa_sparse_mla_decode_range(ctypes.byref(_mla(heads=8)), B, E, out, None, WS,
                                            need, None) == pmqa.PMQA_ERR_UNSUPPORTED
    O, L = ctypes.c_void_p(0x90000), ctypes.c_void_p(0xA0000)
    assert lib.pmqa_sparse_mla_merge(O, L, 0, 4, 16, out, None, None) == -1
    assert lib.pmqa_sparse_mla_merge(O, L, 2, -1, 16, out, None, None) == -1
    assert lib.pmqa_sparse_mla_merge(O, L, 2, 4, 32, out, None, None) == pmqa.PMQA_ERR_UNSUPPORTED
    assert lib.pmqa_sparse_mla_merge(None, L, 2, 4, 16, out, None, None) == -1
    assert lib.pmqa_sparse_mla_merge(O, L, 2, 4, 16, None, None, None) == -1
    assert lib.pmqa_sparse_mla_merge(O, ctypes.c_void_p(0xA0002), 2, 4, 16, out, None, None) == -1
    assert lib.pmqa_sparse_mla_merge(None, None, 2, 0, 16, None, None, None) == 0


def test_gather_probe_validation(lib):
    pool, rows, out = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000), ctypes.c_void_p(0x300000)
    f = lib.pmqa_gather_probe
    assert f(pool, 1 << 20, rows, -1, 132, 0, out, None) == -1
    assert f(pool, 1 << 20, rows, 10, 132, 3, out, None) == -1
    assert f(pool, 1 << 20, rows, 10, 132, -1, out, None) == -1
    assert f(pool, 1 << 20, rows, 10, 128, 0, out, None) == pmqa.PMQA_ERR_UNSUPPORTED
    assert f(None, 1 << 20, rows, 10, 576, 1, out, None) == -1
    assert f(pool, 1 << 20, None, 10, 576, 1, out, None) == -1
    assert f(pool, 1 << 20, rows, 10, 576, 2, None, None) == -1
    assert f(ctypes.c_void_p(0x100008), 1 << 20, rows, 10, 132, 0, out, None) == -1
    assert f(pool, 1 << 20, ctypes.c_void_p(0x200002), 10, 132, 0, out, None) == -1
    assert f(pool, 1 << 20, rows, 10, 132, 0, ctypes.c_void_p(0x300002), None) == -1
    assert f(None, 0, None, 0, 132, 2, None, None) == 0  # nothing to read: no launch
