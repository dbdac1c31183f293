"""Small-batch decode-GEMM on the tcgen05 tensor cores (M >= 9, bf16 x),
through the C ABI, against the CPU oracle.

NVFP4 is checked against the oracle's exact f64 GEMV.  Q4_K is checked against
the oracle with every weight rounded once to bf16, the precision of the staged
tile.  Both use |y_gpu - y_ref| <= 1e-5 * sum|w||x| + 1e-6.

The shapes cover:
  * K split 1, 2, 4 and 8 ways over a thread-block cluster;
  * ragged weight tiles (N not a multiple of 128);
  * batch padding and several 128-row batch chunks (M = 9 .. 200);
  * the full 14336 x 4096 layer at M = 16, 64 and 128, every row.
"""
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


def gpu_gemm(layer, d, xdev, M):
    N, K = layer["N"], layer["K"]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    aux = aux_for(layer, d, x_dtype=torch.bfloat16)
    rc = q4.q4_gemv(layer["fmt"], d["w"], d["scales"], aux, xdev, y, M, N, K)
    assert rc == q4.Q4_OK
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    return y


def reference(layer, xf, rows=None):
    t = to_oracle(layer)
    if layer["fmt"] == "q4k":
        return oracle.gemm_bf16_weights(t, xf, rows=rows)
    if rows is None:
        return oracle_gemv_all_rows(t, xf)
    return oracle.gemv(t, xf, rows=rows)


def check(layer, M, config, rows=None, d=None):
    d = d or to_device(layer)
    xbits, xf = synth.draw_x(M, layer["K"], config=config, matrix=7)
    y = gpu_gemm(layer, d, x_device(xbits), M).cpu().numpy()
    ref, bound = reference(layer, xf, rows)
    if rows is not None:
        y = y[:, rows]
    ok, worst = within_tolerance(y, ref, bound)
    assert ok, f"worst error / tolerance = {worst}"
    return worst


# K = 256, 512, 1024 and 4096 give 1, 2, 4 and 8 cluster ranks over K for
# these few-tile shapes; N = 300 / 257 / 130 end in a ragged tile.
SHAPES = [(300, 256), (300, 512), (257, 1024), (130, 4096)]


@pytest.mark.parametrize("fmt", ["nvfp4", "q4k"])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [9, 16, 33, 64, 100, 128, 200])
def test_gemm_tc_matches_oracle(fmt, N, K, M):
    layer = synth.make_layer(fmt, N, K, config=40, matrix=M % 7, row_scale=True)
    check(layer, M, config=40 + M)


@pytest.mark.parametrize("fmt", ["nvfp4", "q4k"])
def test_gemm_tc_single_row_and_single_tile(fmt):
    for N in (1, 127, 128):
        check(synth.make_layer(fmt, N, 1024, config=41, matrix=N), 20, config=41)


@pytest.mark.parametrize("fmt", ["nvfp4", "q4k"])
def test_gemm_tc_deterministic(fmt):
    """Partial tiles are summed in cluster-rank order: repeated calls agree bit for bit."""
    layer = synth.make_layer(fmt, 257, 4096, config=42, matrix=0)
    d = to_device(layer)
    xbits, _ = synth.draw_x(64, 4096, config=42, matrix=7)
    x = x_device(xbits)
    y0 = gpu_gemm(layer, d, x, 64)
    for _ in range(3):
        assert torch.equal(gpu_gemm(layer, d, x, 64), y0)


def test_gemm_tc_kernel_is_the_one_that_runs():
    """The M >= 9 bf16 NVFP4 / Q4_K call launches the tcgen05 kernel; M <= 8
    and f32 x do not."""
    for fmt in ("nvfp4", "q4k"):
        layer = synth.make_layer(fmt, 256, 1024, config=43, matrix=0)
        d = to_device(layer)
        xbits, _ = synth.draw_x(16, 1024, config=43, matrix=7)
        gpu_gemm(layer, d, x_device(xbits), 16)
        assert q4.q4_last_gemv_path() == "gemm_tc"
        gpu_gemm(layer, d, x_device(xbits[:8]), 8)
        assert q4.q4_last_gemv_path() != "gemm_tc"


def test_gemm_nvfp4_k_not_multiple_of_256_uses_the_gemv_path():
    """K % 256 != 0 is outside the tensor-core kernel's tiling; the same call
    still answers through the GEMV kernels."""
    check(synth.make_layer("nvfp4", 70, 4128, config=44, matrix=0), 12, config=44)
    assert q4.q4_last_gemv_path() == "gemv_general"


def test_gemm_q4k_bf16_staging_error_is_small():
    """Information, not parity: the bf16-rounded Q4_K weights stay within a
    bf16 half-ulp of the exact f32 weights, and the GEMM against the exact
    oracle is off by about that much."""
    layer = synth.make_layer("q4k", 256, 1024, config=45, matrix=0)
    t = to_oracle(layer)
    W = oracle.dequant(t).astype(np.float64)
    Wb = oracle.bf16_bits_to_f32(oracle.round_bf16(W.astype(np.float32))).astype(np.float64)
    assert np.all(np.abs(Wb - W) <= np.abs(W) * 2.0 ** -8)
    xbits, xf = synth.draw_x(16, 1024, config=45, matrix=7)
    y = gpu_gemm(layer, to_device(layer), x_device(xbits), 16).cpu().numpy()
    exact, bound = oracle.gemv(t, xf)
    assert np.all(np.abs(y - exact) <= 2.0 ** -8 * bound + 1e-6)


FULL = [("nvfp4", 16), ("nvfp4", 64), ("nvfp4", 128), ("q4k", 16), ("q4k", 64), ("q4k", 128)]


@pytest.mark.parametrize("fmt,M", FULL)
def test_gemm_tc_full_size_every_row(fmt, M):
    """The small-batch workload: M x 14336 x 4096, weights drawn like the
    1024 x 4096 NVFP4 case (N(0, 0.02)), x ~ N(0, 1) bf16; every row."""
    N, K = 14336, 4096
    layer = synth.make_layer(fmt, N, K, config=4, matrix=0)
    check(layer, M, config=4)
