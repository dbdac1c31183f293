"""The batch-1 NVFP4 GEMV on the native block-scaled FP4 tensor cores
(tcgen05.mma.kind::mxf4nvf4), through the C ABI, against the CPU oracle:
|y_gpu - y_ref| <= 1e-5 * sum|w||x| + 1e-6.

x enters the MMA as exact 2-bit FP4 slices of its 16-value blocks; blocks
the slices cannot hold go to the CUDA cores.  These cases aim at that
split: subnormal elements, an element far below its block's top, a block
far below the range's top, non-positive and zero x, one block holding a
huge value among tiny ones, uneven K ranges across a cluster's ranks, and
ragged 128-row tiles; plus the ordinary shapes, the grouped launch and the
full 4096 x 14336 MLP set, every row.  The path is opt-in
(Q4_FLAG_FP4_SLICES)."""
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


def slices_aux(layer, d):
    aux = aux_for(layer, d, x_dtype=torch.bfloat16)
    aux.flags = q4.Q4_FLAG_FP4_SLICES
    return aux


def run(layer, xbits):
    d = to_device(layer)
    N, K = layer["N"], layer["K"]
    y = torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_gemv("nvfp4", d["w"], d["scales"], slices_aux(layer, d), x_device(xbits), y, 1, N, K)
    torch.cuda.synchronize()
    assert q4.q4_last_gemv_path() == "gemv_fp4tc"
    assert q4.q4_last_error() == q4.Q4_OK
    return y.cpu().numpy()


def check(layer, xbits):
    xbits = np.ascontiguousarray(np.asarray(xbits, np.uint16).reshape(1, -1))
    y = run(layer, xbits)
    ref, bound = oracle.gemv(to_oracle(layer), oracle.bf16_bits_to_f32(xbits))
    ok, worst = within_tolerance(y, ref, bound)
    assert ok, f"worst error / tolerance = {worst}"
    return worst


def with_exponent(bits, e):
    """bf16 patterns with the biased exponent replaced by e (sign, fraction kept)."""
    return ((bits & 0x807F) | (e << 7)).astype(np.uint16)


@pytest.mark.parametrize("N,K", [(300, 4096), (129, 2304), (4096, 11008)])
def test_residual_blocks(N, K):
    layer = synth.make_layer("nvfp4", N, K, config=120, matrix=0, row_scale=True)
    xb, _ = synth.draw_x(1, K, config=120, matrix=1)
    x = xb[0].copy()
    x[16:32] = x[16:32] & 0x807F                      # subnormal block (exponent 0)
    x[40] = with_exponent(x[40:41], 127 - 30)[0]      # one element 2^30 below its block's top
    x[64:80] = with_exponent(x[64:80], 127 - 40)      # a block 2^40 below the range's top
    x[300] = 0x8001                                   # a lone negative subnormal
    x[K - 16:] = with_exponent(x[K - 16:], 127 - 24)  # the last block, at the 2^24 edge
    check(layer, x)


def test_huge_and_tiny_in_one_block():
    layer = synth.make_layer("nvfp4", 256, 4096, config=121, matrix=0)
    xb, _ = synth.draw_x(1, 4096, config=121, matrix=1)
    x = with_exponent(xb[0], 127 - 33)                # everything ~2^-33 ...
    x[7] = 0x7149                                     # ... but one value near 1e30
    x[5000 % 4096] = 0xE1A0                           # and one near -3.7e20
    check(layer, x)


@pytest.mark.parametrize("kind", ["zeros", "negative", "one", "powers"])
def test_special_activations(kind):
    N, K = 200, 1024
    layer = synth.make_layer("nvfp4", N, K, config=122, matrix=0, outliers=True)
    xb, _ = synth.draw_x(1, K, config=122, matrix=1)
    if kind == "zeros":
        x = np.zeros(K, np.uint16)
        assert not run(layer, x.reshape(1, K)).any()
    elif kind == "negative":
        x = xb[0] | 0x8000
    elif kind == "one":
        x = np.full(K, 0x3F80, np.uint16)             # all ones: the row sums
    else:
        x = (np.arange(K) % 64 + 64).astype(np.uint16) << 7     # 2^-63 .. 2^0: 32 binades per block set
    if kind != "zeros":
        check(layer, x)


def test_uneven_k_ranges_and_ragged_tiles():
    """K = 43 slots of 256 split over 8 ranks of 6 slots (the last one 1),
    N = 77 rows in one ragged tile; and 3 ragged tiles with a 9-slot K."""
    for N, K, cfg in ((77, 11008, 123), (300, 2304, 124)):
        layer = synth.make_layer("nvfp4", N, K, config=cfg, matrix=0, row_scale=True)
        xb, _ = synth.draw_x(1, K, config=cfg, matrix=1)
        check(layer, xb[0])


def test_repeated_calls_agree_bit_for_bit():
    layer = synth.make_layer("nvfp4", 1029, 14336, config=125, matrix=0)
    xb, _ = synth.draw_x(1, 14336, config=125, matrix=1)
    y0 = run(layer, xb)
    for _ in range(3):
        assert np.array_equal(run(layer, xb).view(np.uint32), y0.view(np.uint32))


@pytest.mark.parametrize("N,K", [(45, 4096), (16, 256), (7, 11008), (1, 2048), (300, 6144), (263, 14336),
                                 (33, 2304), (4099, 4096)])
def test_ordinary_shapes(N, K):
    layer = synth.make_layer("nvfp4", N, K, config=126, matrix=0, row_scale=True)
    xb, _ = synth.draw_x(1, K, config=126, matrix=1)
    check(layer, xb[0])


def test_grouped_members_share_x_and_default_path_is_unchanged():
    K = 4096
    layers = [synth.make_layer("nvfp4", N, K, config=127, matrix=i, row_scale=True) for i, N in enumerate((300, 17))]
    xb, xf = synth.draw_x(1, K, config=127, matrix=9)
    x = x_device(xb)
    devs = [to_device(L) for L in layers]
    ys = [torch.full((1, L["N"]), float("nan"), device="cuda") for L in layers]
    descs = [("nvfp4", d["w"], d["scales"], slices_aux(L, d), x, y, L["N"], K) for L, d, y in zip(layers, devs, ys)]
    q4.q4_gemv_grouped(descs, 1)
    assert q4.q4_last_gemv_path() == "gemv_fp4tc_group"
    torch.cuda.synchronize()
    for L, y in zip(layers, ys):
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst
    # without the flag the same call takes the TMA-fed kernel
    descs = [("nvfp4", d["w"], d["scales"], aux_for(L, d, x_dtype=torch.bfloat16), x, y, L["N"], K)
             for L, d, y in zip(layers, devs, ys)]
    q4.q4_gemv_grouped(descs, 1)
    assert q4.q4_last_gemv_path() == "gemv_tma_group"


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_mlp_set_every_row(N, K):
    layer = synth.make_layer("nvfp4", N, K, config=5, matrix=0, row_scale=True)
    xb, xf = synth.draw_x(1, K, config=5, matrix=5)
    y = run(layer, xb)
    ref, bound = oracle_gemv_all_rows(to_oracle(layer), xf)
    ok, worst = within_tolerance(y, ref, bound)
    assert ok, worst
