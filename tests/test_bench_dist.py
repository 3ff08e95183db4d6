"""bench.py's multi-rank path on CPU: world_size 2 over gloo (no GPU).

The decode and writer units shard across ranks with no data-path collective; the only
collectives are the timing barrier and the max over ranks, which these tests exercise,
together with the whole-job rate and the per-rank input shards.
"""

import json
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
from quantized_kv_cache_06_gb300.workloads import make_workload  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    bench.init_dist(w, lr, "gloo")
    bench.barrier(w)
    # rank 0 is slower on the first value, rank 1 on the second
    vals = bench.max_over_ranks([1.0 + r, 5.0 - r, 3.0], w)
    rate = bench.weak_scaling_rate(w, 100.0, vals[0])
    bench.barrier(w)
    torch.distributed.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "vals": vals, "rate": rate}, f)


def test_max_over_ranks_and_rate_two_gloo_ranks(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        with open(tmp_path / f"rank{r}.json") as f:
            d = json.load(f)
        assert d["rank"] == r and d["world"] == 2
        assert d["vals"] == [2.0, 5.0, 3.0]  # every rank sees the slowest rank's times
        assert d["rate"] == pytest.approx(2 * 100.0 / 2.0)  # both ranks' units over the max time


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.weak_scaling_rate(1, 10.0, 2.0) == 5.0
    bench.init_dist(1, 0, "gloo")
    bench.barrier(1)
    assert not torch.distributed.is_initialized()


def test_rank_shards_are_independent_batches_of_one_shape():
    a, b = make_workload(2), make_workload(2, shard=1)
    assert a.k_raw.shape == b.k_raw.shape and np.array_equal(a.seq_lens, b.seq_lens)
    assert not np.array_equal(a.k_raw, b.k_raw)
    assert not np.array_equal(a.block_table, b.block_table)
    c = make_workload(2, shard=1)
    assert np.array_equal(b.k_raw, c.k_raw)  # reproducible per shard


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        batch, steps, warmup, gpus, workload, sub = None, 1, 0, 2, 4, 0

    bench.run_reference(Args())
    assert capsys.readouterr().out == ""


def test_next_rows_cpu_baselines_cover_each_row():
    # the oracle timed beside each next row, on the tiny workload: every row present, in the
    # unit of its GPU figure, positive, and labelled as the oracle
    base = bench.next_rows_cpu_baselines(make_workload(1))
    assert set(base) == {"tq_dequant_rows", "tq_paged_prefill", "qjl_residual_keys", "int8q_prefill", "recipe_modes"}
    entries = [base["tq_dequant_rows"], base["tq_paged_prefill"], base["int8q_prefill"],
               *base["qjl_residual_keys"].values()]
    for rec in ("turboquant25", "turboquant35"):
        entries += list(base["recipe_modes"][rec].values())
    for e in entries:
        assert e["kind"] == "oracle" and e["unit"] == "GB/s" and e["value"] > 0 and e["cores"] >= 1
