"""The oracle against values the pages print (fixtures under tests/golden/,
each citing its page and section)."""

import os

import numpy as np
import pytest

import oracle
from synth import make_problem
from synth.inputs import ROW_BYTES

pytestmark = pytest.mark.filterwarnings("ignore")

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append([int(x) for x in line.split()])
    return out


@pytest.mark.parametrize("ctx,P,last", rows("last_page_tokens.txt"))
def test_last_page_holds_the_stated_token_count(ctx, P, last):
    """Exactly `last` tokens of the request's last page reach the logits; the
    page's other slots (poisoned) are never read."""
    p = make_problem(1, 1, 4, P, [ctx], ctx + 2 * P, seed=ctx, table="perm", extra_blocks=1)
    out, _, _ = oracle.logits(p)
    nblk = -(-ctx // P)
    first = (nblk - 1) * P
    assert np.isfinite(out[0, first:first + P]).sum() == last
    assert not np.isnan(out).any()


@pytest.mark.parametrize("ctx,max_blocks,row_bytes,k", rows("repro_shapes.txt"))
def test_reproduction_shapes(ctx, max_blocks, row_bytes, k):
    """The driver's shapes: a KV row of 128 + 4 bytes, an identity table over
    ctx + 16 blocks, k = min(2048, ctx) selected positions."""
    assert ROW_BYTES == row_bytes
    p = make_problem(1, 1, 32, 1, [ctx], ctx + 64, seed=1, table="identity", extra_blocks=16,
                     width=max_blocks)
    assert p.kv.shape[1:] == (1, row_bytes) and p.block_tables.shape == (1, max_blocks)
    assert np.array_equal(p.block_tables[0, :ctx], np.arange(ctx))
    _, o64, _ = oracle.logits(p, want64=True)
    idx = oracle.topk(o64, p.context_lens, 1, 2048)
    assert (idx[0] >= 0).sum() == k
