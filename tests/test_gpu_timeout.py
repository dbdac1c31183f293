"""The bounded waits' failure path on the GPU, with no fault and no hang: the
wait limit is shortened (q4_set_wait_limit) so that waits run out on a
healthy kernel; the kernel must record Q4_ETIMEOUT, stop its roles, wait for
its own copies and MMAs in flight, free tensor memory and return; the
context stays usable and the next call with the default limit is correct.

  * the batch-1 NVFP4 GEMV on the FP4 tensor cores (role waits);
  * the batch-1 Q4_0 GEMV on the TMA-fed block-format kernel (role waits);
  * the GEMV chain's grid barrier, whose sync words the caller re-zeroes
    after a timeout, as its header requires."""
import numpy as np
import pytest

import oracle
import synth

from _helpers import aux_for, oracle_gemv_all_rows, to_device, to_oracle, within_tolerance, x_device

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()
    yield
    q4.q4_set_wait_limit(0)


@pytest.fixture(autouse=True)
def default_limit_after():
    yield
    assert q4.q4_set_wait_limit(0) == q4.Q4_OK
    q4.q4_last_error()


def test_fp4tc_role_wait_times_out_then_recovers():
    N, K = 14336, 4096
    layer = synth.make_layer("nvfp4", N, K, config=130, matrix=0, row_scale=True)
    d = to_device(layer)
    xb, xf = synth.draw_x(1, K, config=130, matrix=1)
    x = x_device(xb)
    y = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    aux = aux_for(layer, d, x_dtype=torch.bfloat16)
    aux.flags = q4.Q4_FLAG_FP4_SLICES
    assert q4.q4_last_error() == q4.Q4_OK
    assert q4.q4_set_wait_limit(1) == q4.Q4_OK          # one SM clock: role waits give up at once
    q4.q4_gemv("nvfp4", d["w"], d["scales"], aux, x, y, 1, N, K)
    assert q4.q4_last_gemv_path() == "gemv_fp4tc"
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_ETIMEOUT
    assert q4.q4_last_error() == q4.Q4_OK                 # reading clears it
    assert q4.q4_set_wait_limit(0) == q4.Q4_OK
    y.fill_(float("nan"))
    q4.q4_gemv("nvfp4", d["w"], d["scales"], aux, x, y, 1, N, K)
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    ref, bound = oracle_gemv_all_rows(to_oracle(layer), xf)
    ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
    assert ok, worst


def test_blk_tc_role_wait_times_out_then_recovers():
    # 4096 x 11008: six 2048-k stages per CTA through a three-stage ring, so
    # the producer waits for freed slots and the decode warps for full ones
    N, K = 4096, 11008
    layer = synth.make_layer("q40", N, K, config=132, matrix=0)
    d = to_device(layer)
    xb, xf = synth.draw_x(1, K, config=132, matrix=1, dtype="f32")
    x = x_device(xb)
    y = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    aux = aux_for(layer, d, x_dtype=torch.float32)
    assert q4.q4_last_error() == q4.Q4_OK
    assert q4.q4_set_wait_limit(1) == q4.Q4_OK
    q4.q4_gemv("q40", d["w"], d["scales"], aux, x, y, 1, N, K)
    assert q4.q4_last_gemv_path() == "gemv_blk_tc_q40"
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_ETIMEOUT
    assert q4.q4_set_wait_limit(0) == q4.Q4_OK
    y.fill_(float("nan"))
    q4.q4_gemv("q40", d["w"], d["scales"], aux, x, y, 1, N, K)
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    ref, bound = oracle_gemv_all_rows(to_oracle(layer), xf)
    ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
    assert ok, worst


def test_chain_grid_barrier_times_out_then_recovers_after_rezeroing():
    layers = [synth.make_layer("nvfp4", N, 4096, config=131, matrix=i) for i, N in enumerate((2048, 1024))]
    ds = [to_device(L) for L in layers]
    xb, xf = synth.draw_x(1, 4096, config=131, matrix=5)
    x = x_device(xb)
    ys = [torch.zeros((1, L["N"]), device="cuda") for L in layers]
    groups = [[("nvfp4", d["w"], d["scales"], aux_for(L, d, x_dtype=torch.bfloat16), x, y, L["N"], 4096)]
              for L, d, y in zip(layers, ds, ys)]
    # A barrier no arrival can complete: the count starts far above the grid size, so no CTA
    # is the last to arrive and every CTA's bounded spin runs out (with a one-clock limit it
    # would otherwise race the arrivals: CTAs with equal work can all arrive before any checks).
    sync = torch.tensor([1 << 30, 0], dtype=torch.int32, device="cuda")
    assert q4.q4_set_wait_limit(1) == q4.Q4_OK
    q4.q4_gemv_chain(groups, 1, sync=sync)
    assert q4.q4_last_gemv_path() == "gemv_tma_chain"
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_ETIMEOUT
    assert q4.q4_set_wait_limit(0) == q4.Q4_OK
    sync.zero_()                                          # the caller's duty after a timeout
    for y in ys:
        y.fill_(float("nan"))
    q4.q4_gemv_chain(groups, 1, sync=sync)
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    assert sync.cpu().tolist()[0] == 0
    for L, y in zip(layers, ys):
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst
