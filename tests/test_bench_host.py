"""Host-side pieces of bench.py: multi-rank aggregation over a gloo process
group (world size 2, CPU), algorithmic byte counts, and the JSON contract of
the reference arm on a tiny bounded run."""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import make_problem  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mx = bench.max_over_ranks(1.5 + rank, dist)          # per-rank step times
    sm = bench.sum_over_ranks(1000.0 * (rank + 1), dist)  # per-rank tokens
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_rank_aggregation_gloo_world2():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == (2.5, 3000.0)  # max of step times, sum of tokens, on every rank


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(3.25, None) == 3.25
    assert bench.sum_over_ranks(7.0, None) == 7.0


def test_algorithmic_bytes_counts():
    prob = make_problem(2, 2, 16, 4, [10, 3], 16, seed=1)
    ab = bench.algorithmic_bytes(prob, 8)
    assert ab["kv"] == 132 * 13
    assert ab["block_table"] == 4 * (3 + 1)          # ceil(10/4) + ceil(3/4)
    assert ab["weights"] == 4 * 4 * 16
    assert ab["topk_out"] == 4 * 4 * 8
    assert ab["total"] == sum(v for k, v in ab.items() if k != "total")
    # admitted positions per row: ctx - next_n + j + 1 clamped to [0, ctx]
    assert bench.valid_positions(prob) == (9 + 10) + (2 + 3)
    sb = bench.score_kernel_bytes(prob)
    assert sb["compact_logits"] == 4 * 24
    assert sb["total"] == sb["kv"] + sb["block_table"] + sb["q"] + sb["weights"] + \
        sb["context_lens"] + sb["compact_logits"]


def test_reference_arm_json_line():
    """--impl reference times the oracle on bounded samples and prints one
    JSON line with the fields the driver reads."""
    pytest.importorskip("numpy")
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "C0", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_default_run_times_every_config_and_the_prefill():
    """With no flags the line carries every config and the prefill beside the
    headline; --headline-only (used by the profiling commands) times the
    headline alone unless --prefill asks for the prefill too."""
    a = bench.parse_args([])
    assert a.all and a.workload == bench.DEFAULT_WORKLOAD and a.steps >= 1 and a.warmup >= 3
    a = bench.parse_args(["--headline-only"])
    assert not a.all and not a.prefill
    a = bench.parse_args(["--headline-only", "--prefill"])
    assert not a.all and a.prefill
    from synth import CONFIGS

    assert set(CONFIGS) >= {"C0", "C1", "C2", "C3", "C4"}


def test_kv_roofline_counts_the_kv_stream_only():
    prob = make_problem(2, 2, 16, 4, [10, 3], 16, seed=1)
    kr = bench.kv_roofline(prob, score_ms=1e-3, step_ms=2e-3, peak=1000.0)
    assert kr["kv_bytes"] == 132 * 13
    assert kr["achieved"] == pytest.approx(132 * 13 / 1e-6 / 1e9)
    assert kr["frac"] == pytest.approx(kr["achieved"] / 1000.0)
    assert kr["fused_frac"] == pytest.approx(kr["frac"] / 2)
    other = kr["other_bytes"]
    assert "kv" not in other and other["compact_logits"] == 4 * 24
    assert other["total"] == sum(v for k, v in other.items() if k != "total")


def test_cpu_description_and_cpu_ranges():
    d = bench.cpu_description()
    assert d["cpu_model"] and d["logical_cpus"] >= 1 and d["affinity"]
    assert bench._ranges([0, 1, 2, 5, 7, 8]) == "0-2,5,7-8"
    assert bench._ranges([3]) == "3"


def test_gather_probe_row_lists():
    """The rows `bench.py --gather-ceiling` hands the probe are the rows the
    kernels read: every token through the block table (pages of 4, a partial
    last page), and every listed position of every query row (holes
    skipped)."""
    from synth.mla import make_mla_problem

    prob = make_problem(2, 1, 16, 4, [10, 3], 16, seed=2, table="perm")
    rows = bench.kv_rows(prob)
    want = [prob.block_tables[i, t // 4] * 4 + t % 4 for i, c in enumerate([10, 3])
            for t in range(c)]
    assert rows.dtype == np.int32 and rows.tolist() == want
    mp_ = make_mla_problem(2, 2, 16, 1, [300, 40], topk=64, seed=3, holes=0.2)
    rows = bench.mla_rows(mp_)
    want = [mp_.block_tables[r // 2, pos] for r in range(4) for pos in mp_.indices[r] if pos >= 0]
    assert rows.tolist() == want
