"""Pins for the CPU oracle against what the pages and the mathematics fix.

None of these retypes the oracle's formula: each checks a closed form, a
special case that reduces to a library routine, an invariant, or brute force.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import make_problem, pack_kv
from synth.inputs import to_e4m3fn_bytes

pytestmark = pytest.mark.filterwarnings("ignore")


def torch_decode(b: np.ndarray) -> np.ndarray:
    """Library decode of e4m3fn bit patterns (torch), as float64."""
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.float().double().numpy()


def le_scales(kv: np.ndarray) -> np.ndarray:
    flat = kv.reshape(-1, 132)
    return np.frombuffer(np.ascontiguousarray(flat[:, 128:]).tobytes(), dtype="<f4").astype(np.float64)


# ---------------------------------------------------------------- fp8 decode


def test_e4m3fn_code_points():
    tab = oracle.e4m3fn_table()
    assert tab[0x38] == 1.0
    assert tab[0x7E] == 448.0
    assert tab[0x08] == 2.0 ** -6
    assert tab[0x01] == 2.0 ** -9
    assert tab[0x77] == 240.0
    assert tab[0xB8] == -1.0
    assert tab[0x00] == 0.0 and tab[0x80] == 0.0 and np.signbit(tab[0x80])
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])
    assert np.nanmax(tab) == 448.0 and np.nanmin(tab) == -448.0


def test_e4m3fn_table_matches_torch_everywhere():
    tab = oracle.e4m3fn_table()
    ref = torch_decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan)
    assert np.array_equal(tab[~nan], ref[~nan])
    assert np.array_equal(np.signbit(tab[~nan]), np.signbit(ref[~nan]))


# ---------------------------------------------------------------- logits


def single_head(ctx=37, P=1, seed=1, mml=64, **kw):
    return make_problem(1, 1, 1, P, [ctx], mml, seed=seed, **kw)


@pytest.mark.parametrize("d0", [0, 5, 64, 127])
def test_one_hot_query_reads_one_byte_and_the_le_scale(d0):
    """q = e_d0 (fp8 1.0), H=1, w=1: logit_t = relu(fp8(k_t[d0]) * scale_t)."""
    p = single_head(ctx=40, seed=d0)
    p.q[:] = 0
    p.q[0, 0, 0, d0] = 0x38
    p.weights[:] = 1.0
    out, out64, _ = oracle.logits(p, want64=True)
    phys = p.block_tables[0, :40]
    k = torch_decode(p.kv.reshape(-1, 132)[phys, d0])
    s = le_scales(p.kv)[phys]
    expect = np.maximum(k * s, 0.0)
    assert np.array_equal(out64[0, :40], expect)
    assert np.array_equal(out[0, :40], expect.astype(np.float32))
    assert np.all(np.isneginf(out[0, 40:]))


def test_relu_sign_flip_reduces_to_library_gemv():
    """relu(x) - relu(-x) = x and relu(x) + relu(-x) = |x| (H=1, w=1)."""
    p = single_head(ctx=50, seed=3)
    p.weights[:] = 1.0
    neg = make_problem(1, 1, 1, 1, [50], 64, seed=3)
    neg.weights[:] = 1.0
    neg.q[:] = p.q ^ 0x80  # flip the fp8 sign bit: q -> -q
    _, a, _ = oracle.logits(p, want64=True)
    _, b, _ = oracle.logits(neg, want64=True)
    phys = p.block_tables[0, :50]
    kd = torch_decode(p.kv.reshape(-1, 132)[phys, :128])
    qd = torch_decode(p.q[0, 0, 0])
    x = (kd @ qd) * le_scales(p.kv)[phys]  # library GEMV, exact in double
    np.testing.assert_allclose(a[0, :50] - b[0, :50], x, rtol=1e-14, atol=0)
    np.testing.assert_allclose(a[0, :50] + b[0, :50], np.abs(x), rtol=1e-14, atol=0)


def test_positive_inputs_reduce_to_gemv_and_tolerance_closed_form():
    p = single_head(ctx=33, seed=4)
    p.q &= 0x7F
    p.kv[..., :128] &= 0x7F  # every fp8 entry >= 0
    p.kv.reshape(-1, 132)[:, :128][p.kv.reshape(-1, 132)[:, :128] == 0x7F] = 0x7E
    p.weights[:] = 1.0
    _, o64, tol = oracle.logits(p, want64=True, want_tol=True)
    phys = p.block_tables[0, :33]
    x = (torch_decode(p.kv.reshape(-1, 132)[phys, :128]) @ torch_decode(p.q[0, 0, 0])) \
        * le_scales(p.kv)[phys]
    np.testing.assert_allclose(o64[0, :33], x, rtol=1e-15)
    np.testing.assert_allclose(tol[0, :33], 1e-3 * (1 + np.abs(x)), rtol=1e-14)
    assert np.all(tol[0, 33:] == 0)


def test_tolerance_uses_weight_magnitudes():
    """tol = 1e-3 (1 + |w| |x|) for one head with a negative weight."""
    p = single_head(ctx=25, seed=40)
    p.weights[:] = -2.0
    _, _, tol = oracle.logits(p, want_tol=True)
    phys = p.block_tables[0, :25]
    x = (torch_decode(p.kv.reshape(-1, 132)[phys, :128]) @ torch_decode(p.q[0, 0, 0])) \
        * le_scales(p.kv)[phys]
    np.testing.assert_allclose(tol[0, :25], 1e-3 * (1 + 2 * np.abs(x)), rtol=1e-14)


def test_head_sum_and_weight_rows():
    """Rows use weights[i*next_n+j]; heads add with their weights."""
    bs, nn, H, ctx = 2, 2, 3, [21, 30]
    p = make_problem(bs, nn, H, 1, ctx, 48, seed=5)
    # head 1 repeats head 0, so logit = (w0 + w1) relu(x0) + w2 relu(x2)
    p.q[:, :, 1] = p.q[:, :, 0]
    _, full, _ = oracle.logits(p, want64=True)
    for i in range(bs):
        for j in range(nn):
            r = i * nn + j
            parts = []
            for h in (0, 2):
                one = make_problem(1, 1, 1, 1, [ctx[i]], 48, seed=5)
                one.kv = p.kv
                one.block_tables = p.block_tables[i:i + 1].copy()
                one.q = np.ascontiguousarray(p.q[i:i + 1, j:j + 1, h:h + 1])
                one.weights = np.ones((1, 1), np.float32)
                one.context_lens = np.array([ctx[i]], np.int32)
                _, o, _ = oracle.logits(one, want64=True)
                parts.append(o[0])
            w = p.weights[r].astype(np.float64)
            n = oracle.valid_len(ctx[i], nn, j)
            expect = (w[0] + w[1]) * parts[0][:n] + w[2] * parts[1][:n]
            np.testing.assert_allclose(full[r, :n], expect, rtol=1e-13, atol=1e-300)


@pytest.mark.parametrize("nn", [1, 2, 4])
def test_mask_is_exact(nn):
    ctx = [0, 1, 2, 3, 5, 130, 257]
    p = make_problem(len(ctx), nn, 4, 1, ctx, 300, seed=6)
    out, _, _ = oracle.logits(p)
    for i, c in enumerate(ctx):
        for j in range(nn):
            row = out[i * nn + j]
            t = np.arange(300)
            valid = (t < c) & (t <= c - nn + j)
            assert np.all(np.isfinite(row[valid]))
            assert np.all(np.isneginf(row[~valid]))


def test_nonnegative_weights_give_nonnegative_logits():
    p = make_problem(3, 2, 8, 1, [100, 64, 7], 128, seed=7)
    p.weights = np.abs(p.weights)
    out, _, _ = oracle.logits(p)
    fin = np.isfinite(out)
    assert fin.sum() > 0 and np.all(out[fin] >= 0)


def test_linear_in_weights():
    p = make_problem(2, 1, 8, 1, [90, 45], 96, seed=8)
    rng = np.random.default_rng(0)
    w1 = rng.integers(-8, 8, size=p.weights.shape).astype(np.float32) / 4
    w2 = rng.integers(-8, 8, size=p.weights.shape).astype(np.float32) / 4
    outs = []
    for w in (w1, w2, w1 + w2):  # all exact in fp32
        p.weights = w
        outs.append(oracle.logits(p, want64=True)[1])
    fin = np.isfinite(outs[2])
    np.testing.assert_allclose(outs[2][fin], outs[0][fin] + outs[1][fin], rtol=1e-12, atol=1e-12)


def test_doubling_scales_doubles_logits_bit_exactly():
    p = make_problem(2, 2, 16, 1, [77, 130], 160, seed=9)
    a, _, _ = oracle.logits(p)
    flat = p.kv.reshape(-1, 132)
    s = np.frombuffer(np.ascontiguousarray(flat[:, 128:]).tobytes(), dtype="<f4").copy()
    flat[:, 128:] = (s * np.float32(2)).astype("<f4").view(np.uint8).reshape(-1, 4)
    b, _, _ = oracle.logits(p)
    fin = np.isfinite(a)
    assert np.array_equal(np.isfinite(b), fin)
    assert np.array_equal(b[fin], a[fin] * np.float32(2))


@pytest.mark.parametrize("P", [1, 16])
def test_physical_permutation_invariance(P):
    p = make_problem(3, 2, 8, P, [100, 33, 64], 128, seed=10, table="identity", extra_blocks=3)
    a, _, _ = oracle.logits(p)
    rng = np.random.default_rng(1)
    perm = rng.permutation(p.num_blocks)  # block b moves to slot perm[b]
    kv2 = np.empty_like(p.kv)
    kv2[perm] = p.kv
    bt2 = np.where(p.block_tables >= 0, perm[np.maximum(p.block_tables, 0)], -1).astype(np.int32)
    p.kv, p.block_tables = kv2, bt2
    b, _, _ = oracle.logits(p)
    assert np.array_equal(a, b)


def test_paged_layout_equals_single_token_blocks():
    """The same logical tokens stored in 64-token pages or in 1-token blocks."""
    ctx = [200, 64, 1, 129]
    p1 = make_problem(4, 2, 8, 1, ctx, 256, seed=11, table="perm")
    P = 64
    rows = []
    tables = np.full((4, 4), -1, np.int32)
    nxt = 0
    for i, c in enumerate(ctx):
        npg = -(-c // P)
        tok = p1.kv.reshape(-1, 132)[p1.block_tables[i, :c]]
        pad = np.full((npg * P - c, 132), 0x7F, np.uint8)  # poisoned page tail
        rows.append(np.concatenate([tok, pad]))
        tables[i, :npg] = np.arange(nxt, nxt + npg)
        nxt += npg
    flat = np.concatenate(rows)
    order = np.random.default_rng(2).permutation(nxt)
    pages = flat.reshape(nxt, P, 132)
    kv = np.empty_like(pages)
    kv[order] = pages
    p64 = make_problem(4, 2, 8, P, ctx, 256, seed=11)
    p64.q, p64.weights = p1.q, p1.weights
    p64.kv = kv
    p64.block_tables = np.where(tables >= 0, order[np.maximum(tables, 0)], -1).astype(np.int32)
    a, _, _ = oracle.logits(p1)
    b, _, _ = oracle.logits(p64)
    assert np.array_equal(a, b)


def test_causal_rows_are_shifted_copies():
    nn, ctx = 3, [50, 9]
    p = make_problem(2, nn, 8, 1, ctx, 64, seed=12)
    p.q[:, :] = p.q[:, nn - 1:nn]
    p.weights[:] = np.repeat(p.weights[nn - 1::nn], nn, axis=0)
    out, _, _ = oracle.logits(p)
    for i, c in enumerate(ctx):
        last = out[i * nn + nn - 1]
        for j in range(nn):
            n = c - nn + j + 1
            assert np.array_equal(out[i * nn + j, :n], last[:n])
            assert np.all(np.isneginf(out[i * nn + j, n:]))


def test_context_2048_to_2049_boundary():
    p = make_problem(1, 1, 32, 1, [2049], 4096, seed=13, table="identity", extra_blocks=16)
    a, a64, _ = oracle.logits(p, want64=True)
    p.context_lens[:] = 2048
    b, b64, _ = oracle.logits(p, want64=True)
    assert np.array_equal(a[0, :2048], b[0, :2048])
    assert np.isneginf(b[0, 2048]) and np.isfinite(a[0, 2048])
    ib = oracle.topk(b64, [2048], 1, 2048)
    assert np.array_equal(np.sort(ib[0]), np.arange(2048))
    ia = oracle.topk(a64, [2049], 1, 2048)
    assert np.all(ia[0] >= 0) and len(set(ia[0].tolist())) == 2048


def test_poisoned_slots_are_never_read():
    p = make_problem(4, 1, 8, 1, [10, 20, 30, 40], 64, seed=14, table="perm", extra_blocks=5)
    out, _, _ = oracle.logits(p)
    t = np.arange(64)
    for i, c in enumerate([10, 20, 30, 40]):
        assert np.all(np.isfinite(out[i, t < c]))


def test_bad_table_entry_is_an_error():
    p = make_problem(1, 1, 4, 1, [10], 16, seed=15)
    p.block_tables[0, 3] = p.num_blocks
    with pytest.raises(ValueError):
        oracle.logits(p)


# ---------------------------------------------------------------- top-k


def brute_topk(row: np.ndarray, n: int, k: int) -> list:
    """Repeatedly take the largest remaining value, lowest index first."""
    taken = np.zeros(n, bool)
    out = []
    for _ in range(min(k, n)):
        best = -1
        for t in range(n):
            if not taken[t] and (best < 0 or row[t] > row[best]):
                best = t
        taken[best] = True
        out.append(best)
    return out + [-1] * (k - len(out))


@pytest.mark.parametrize("ties", [False, True])
def test_topk_matches_brute_force(ties):
    rng = np.random.default_rng(3)
    ctx, nn, k = [1, 7, 40, 64], 2, 12
    width = 70
    vals = (rng.integers(-3, 3, (8, width)).astype(np.float64) if ties
            else rng.standard_normal((8, width)))
    vals[:, 60:] = 1e9  # outside every window: must be ignored
    idx = oracle.topk(vals, ctx, nn, k)
    for i, c in enumerate(ctx):
        for j in range(nn):
            r = i * nn + j
            n = max(0, min(c - nn + j + 1, c))
            assert idx[r].tolist() == brute_topk(vals[r], n, k)


def test_topk_against_library_sort():
    rng = np.random.default_rng(4)
    vals = rng.standard_normal((3, 5000))
    idx = oracle.topk(vals, [5000, 4000, 100], 1, 2048)
    for r, n in enumerate([5000, 4000, 100]):
        order = np.lexsort((np.arange(n), -vals[r, :n]))[:2048]
        got = idx[r][idx[r] >= 0]
        assert np.array_equal(got, order)
        assert np.all(idx[r][len(got):] == -1)


# ---------------------------------------------------------------- generator


def test_generator_layout_and_poison():
    p = make_problem(3, 1, 4, 16, [17, 32, 1], 64, seed=16, table="perm", extra_blocks=2)
    assert p.kv.shape == (2 + 2 + 1 + 6, 16, 132)
    used = set()
    for i, c in enumerate([17, 32, 1]):
        for t in range(c):
            used.add(int(p.block_tables[i, t // 16]) * 16 + t % 16)
    flat = p.kv.reshape(-1, 132)
    for s in range(flat.shape[0]):
        poisoned = np.all(flat[s, :128] == 0x7F)
        assert poisoned == (s not in used)
    kb = to_e4m3fn_bytes(np.array([1.0, -2.0, 1000.0], np.float32))
    assert kb.tolist() == [0x38, 0xC0, 0x7E]
    kv = pack_kv(np.zeros((2, 128), np.uint8), np.array([1.0, 0.5], np.float32), 1)
    assert kv[0, 0, 128:].tolist() == [0, 0, 0x80, 0x3F]
