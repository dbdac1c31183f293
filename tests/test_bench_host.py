"""bench.py's host-side multi-rank logic on the CPU: the max over ranks of
the timed interval (world_size 2, gloo, two spawned processes), the
whole-job throughput arithmetic, and the reference arm (the CPU oracle),
which rank 0 alone runs under torchrun while the other ranks exit without
work.  No GPU is touched."""
import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
torch = pytest.importorskip("torch")
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        out.put((rank, bench.max_over_ranks(values[rank], world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    values = [3.25, 7.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 7.5, 1: 7.5}


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5


def test_whole_job_throughput_counts_every_rank():
    # 99 MB per step, 1000 steps in 22 ms on each of 4 replicas
    one = bench.whole_job_gbps(1, 99_090_444, 1000, 22.0)
    assert one == pytest.approx(99_090_444 * 1000 / 0.022 / 1e9)
    assert bench.whole_job_gbps(4, 99_090_444, 1000, 22.0) == pytest.approx(4 * one)


class _Args:
    steps = 1
    warmup = 0


def test_reference_arm_rank0_only():
    assert bench.run_reference(_Args(), 1, 2) is None      # other ranks exit without work
    line = bench.run_reference(_Args(), 0, 2)
    json.dumps(line)
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_cpu_baseline_rows_cover_every_timed_row():
    """The CPU leg the bench runs beside the other rows: one entry per GEMV row
    (the A16-Q8, W4A4 and W4A8 lanes included) plus the dequant, each with a
    positive rate."""
    rows = bench.cpu_baseline_rows(rows_per_matrix=4)
    names = [r["row"] for r in rows]
    assert bench.A16Q8_ROW in names and "a6 dequant NVFP4 -> f32" in names
    assert "f1 W4A4 GEMV, integer-exact contract" in names
    assert "f2 Q4_K x Q8 (W4A8) GEMV, integer sub-block sums" in names
    assert len(names) == len(bench.ORACLE_ROWS) + 4
    assert all(r["GBps"] > 0 and r["seconds"] >= 0 for r in rows)


def test_tokens_equivalent_rate():
    # 22.1 us per step, 32 layers: 1 / (32 * 22.1e-6) = 1414.03 tokens/s per replica
    assert bench.tokens_equivalent(0.0221, 1) == pytest.approx(1414.03, abs=0.01)
    assert bench.tokens_equivalent(0.0221, 8) == pytest.approx(8 * 1414.03, abs=0.1)


def test_oracle_all_cores_split_matches_one_call():
    """The all-cores CPU baseline runs the oracle's own rows on several host
    threads; the values equal one single-threaded call."""
    import numpy as np
    import oracle
    import synth
    import bench
    layer = synth.make_layer("nvfp4", 96, 512, config=5, matrix=0, row_scale=True)
    T = oracle.Tensor("nvfp4", 96, 512, layer["w"], layer["scales"], scale2=layer["scale2"])
    _, xf = synth.draw_x(1, 512, config=5, matrix=1)
    rows = np.arange(96)
    parts = bench.oracle_rows_all_cores(oracle, T, xf, rows, 4)
    y = np.concatenate([p[0] for p in parts], axis=1)
    assert np.array_equal(y, oracle.gemv(T, xf, rows=rows)[0])
