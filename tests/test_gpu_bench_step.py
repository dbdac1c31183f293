"""The bench's timed step exactly as bench.py launches it, every output row
against the CPU oracle: q4_gemv_grouped(gate, up) (2 x 14336x4096 NVFP4,
shared bf16 x, batch 1) then q4_gemv(down) (4096x14336), chained by
programmatic dependent launch, captured by the bench's own graph planner and
replayed over rotating weight copies.  Here the copies hold different
weights, so an output that came from the wrong copy, or a launch that read
a stale x, fails.  Tolerance: |y_gpu - y_ref| <= 1e-5 * sum|w||x| + 1e-6.
"""
import numpy as np
import pytest

import oracle
import synth

from _helpers import oracle_gemv_all_rows, within_tolerance

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")
bench = pytest.importorskip("bench")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def step_setup():
    from bit_block_quantized_gb300 import build
    build.build()
    hosts, dev, xs, ys, set_bytes, copies, _ = bench.build_workload(torch, q4, synth, copies=2, distinct=True)
    auxes = bench.mlp_auxes(q4, dev)
    assert auxes[0][0].scale2 != auxes[1][0].scale2              # the copies really differ
    refs = []
    for host in hosts:
        per = []
        for name, N, K, layer, xbits in host:
            t = oracle.Tensor("nvfp4", N, K, layer["w"], layer["scales"], scale2=layer["scale2"])
            per.append(oracle_gemv_all_rows(t, oracle.bf16_bits_to_f32(xbits)))
        refs.append(per)
    yield dev, xs, ys, auxes, refs, copies
    del dev
    torch.cuda.empty_cache()


def check_outputs(ys, ref):
    for (name, _, _), y, (r, bound) in zip(bench.SET, ys, ref):
        ok, worst = within_tolerance(y.cpu().numpy(), r, bound)
        assert ok, f"{name}: worst error / tolerance = {worst}"


@pytest.mark.parametrize("steps", [2, 3, 20])
def test_bench_step_graph_matches_oracle_every_row(step_setup, steps):
    dev, xs, ys, auxes, refs, copies = step_setup
    stream = torch.cuda.Stream()
    gate_up, down, step = bench.mlp_step_fns(q4, dev, auxes, xs, ys)
    with torch.cuda.stream(stream):
        gate_up(0, stream)
        assert q4.q4_last_gemv_path() == "gemv_tma_group"
        down(0, stream)
        assert q4.q4_last_gemv_path() == "gemv_tma"
        torch.cuda.synchronize()
        plan = bench.timed_graphs(torch, step, stream, steps, copies)
        assert sum(n for _, n in plan) >= 1
        for y in ys:
            y.fill_(float("nan"))
        bench.replay(plan)
        torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    check_outputs(ys, refs[(steps - 1) % copies])     # the last step ran on copy (steps - 1) % copies


def test_bench_timed_graph_plan_runs_exact_step_count(step_setup):
    """Above the per-graph cap, the planner replays whole rotations and one
    remainder graph; the step count and the last copy still match."""
    dev, xs, ys, auxes, refs, copies = step_setup
    stream = torch.cuda.Stream()
    _, _, step = bench.mlp_step_fns(q4, dev, auxes, xs, ys)
    seen = []
    plan = bench.timed_graphs(torch, lambda c, s: seen.append(c) or step(c, s), stream, 9, copies, cap=4)
    assert [n for _, n in plan] == [2, 1] and seen == [0, 1, 0, 1, 0]      # chunk 4 (x2), remainder 1
    with torch.cuda.stream(stream):
        for y in ys:
            y.fill_(float("nan"))
        bench.replay(plan)
        torch.cuda.synchronize()
    check_outputs(ys, refs[0])
