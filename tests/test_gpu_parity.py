"""CUDA path vs the CPU oracle, through the C ABI.

Dequant and repack: bit-exact.  GEMV: |y_gpu - y_ref| <= 1e-5 * sum|w||x| + 1e-6
against the oracle's f64 accumulation of the pinned weights.  Shapes span
several tiles with ragged tails; the full-size workloads are checked on
every row.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import packing

from _helpers import aux_for, oracle_gemv_all_rows, to_device, to_oracle, within_tolerance, x_device

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu

ROW_FORMATS = ["nvfp4", "mxfp4", "q4k", "q40"]
ALL_GEMV = ROW_FORMATS + ["gptq", "awq"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def tma_fits(K, M):
    """The TMA-fed kernel's shared-memory rule: the staged x (2 bytes per k
    and batch column, K rounded up to 2048-k stages) and the fixed areas
    leave room for at least 3 ring stages of 18 KB in 112 KB."""
    mt = 1 if M == 1 else 2 if M == 2 else 4
    nst = -(-K // 2048)
    fixed = 1024 + 144 + 2 * 8 * 16 * mt * 4 + 8 * nst * 2 * 8 * mt * 4 * 8
    return (112 * 1024 - fixed) // 18432 >= 3


def shape_for(fmt, small=True):
    """(N, K) spanning several CTA tiles with ragged tails."""
    return {"nvfp4": (37, 4128), "mxfp4": (41, 2080), "q4k": (29, 1536), "q40": (33, 2080),
            "gptq": (264, 1152), "awq": (264, 1152), "nvfp4_splithalf": (19, 528),
            "logical": (72, 384)}[fmt]


def gpu_dequant(layer, out_dtype=torch.float32):
    d = to_device(layer)
    N, K = layer["N"], layer["K"]
    out = torch.empty((N, K), dtype=out_dtype, device="cuda")
    aux = aux_for(layer, d, out_dtype=out_dtype)
    q4.q4_dequant(layer["fmt"], d["w"], d["scales"], aux, out, N, K)
    torch.cuda.synchronize()
    return out


def gpu_gemv(layer, xdev, M):
    d = to_device(layer)
    N, K = layer["N"], layer["K"]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    aux = aux_for(layer, d, x_dtype=xdev.dtype)
    q4.q4_gemv(layer["fmt"], d["w"], d["scales"], aux, xdev, y, M, N, K)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def bits_equal(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


# ----------------------------------------------------------------- dequant

@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "q4k", "q40", "gptq", "awq", "nvfp4_splithalf",
                                 "logical"])
def test_dequant_bit_exact(fmt):
    N, K = shape_for(fmt)
    layer = synth.make_layer(fmt, N, K, config=20, matrix=1, outliers=True)
    ref = oracle.dequant(to_oracle(layer))
    got = gpu_dequant(layer).cpu().numpy()
    assert bits_equal(got, ref)
    got16 = gpu_dequant(layer, torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got16, oracle.round_bf16(ref))


def test_dequant_gptq_act_order_bit_exact():
    layer = synth.make_layer("gptq", 64, 512, config=20, matrix=2, act_order=True)
    assert bits_equal(gpu_dequant(layer).cpu().numpy(), oracle.dequant(to_oracle(layer)))


def test_nvfp4_every_finite_e4m3_scale_and_code():
    """All 254 finite E4M3FN bytes x all 16 E2M1 codes, bit-for-bit
    (the exhaustive sweep of Muser book, Chapter 7, section 7.2)."""
    scales = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], np.uint8)
    N = scales.size
    row = np.frombuffer(bytes.fromhex("1032547698badcfe"), np.uint8)
    for scale2 in (0.25, 1.0, 3.0e-5):
        layer = {"fmt": "nvfp4", "N": N, "K": 16, "w": np.tile(row, (N, 1)), "scales": scales[:, None].copy(),
                 "zeros": None, "g_idx": None, "group": 128, "scale2": scale2}
        assert bits_equal(gpu_dequant(layer).cpu().numpy(), oracle.dequant(to_oracle(layer)))


def test_mxfp4_every_e8m0_scale():
    scales = np.arange(255, dtype=np.uint8)
    row = np.tile(np.frombuffer(bytes.fromhex("1032547698badcfe"), np.uint8), 2)
    layer = {"fmt": "mxfp4", "N": 255, "K": 32, "w": np.tile(row, (255, 1)), "scales": scales[:, None].copy(),
             "zeros": None, "g_idx": None, "group": 128, "scale2": 1.0}
    got = gpu_dequant(layer).cpu().numpy()
    ref = oracle.dequant(to_oracle(layer))
    assert bits_equal(got, ref)            # includes the +-inf overflow rows (b >= 253)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "q4k", "q40", "nvfp4_splithalf"])
def test_dequant_random_bytes(fmt):
    """Uniform random payload bytes (every code), random valid scales and
    block headers, bit-for-bit."""
    N, K = 23, 512
    rng = np.random.default_rng(11)
    layer = {"fmt": fmt, "N": N, "K": K, "zeros": None, "g_idx": None, "group": 128, "scale2": 0.0371}
    if fmt in ("nvfp4", "mxfp4", "nvfp4_splithalf"):
        layer["w"] = synth.random_bytes((N, K // 2), 1)
        nsc = K // 16 if fmt != "mxfp4" else K // 32
        excl = (0x7F, 0xFF) if fmt != "mxfp4" else (0xFF, 0xFE, 0xFD)
        layer["scales"] = synth.random_bytes((N, nsc), 2, exclude=excl)
    elif fmt == "q4k":
        b = synth.random_bytes((N, K // 256, 144), 3)
        h = rng.uniform(-2, 2, (N, K // 256, 2)).astype(np.float16).view(np.uint8).reshape(N, K // 256, 4)
        b[:, :, :4] = h
        layer["w"], layer["scales"] = b, None
    else:
        b = synth.random_bytes((N, K // 32, 18), 4)
        b[:, :, :2] = rng.uniform(-2, 2, (N, K // 32)).astype(np.float16).view(np.uint8).reshape(N, K // 32, 2)
        layer["w"], layer["scales"] = b, None
    assert bits_equal(gpu_dequant(layer).cpu().numpy(), oracle.dequant(to_oracle(layer)))


# -------------------------------------------------------------------- GEMV

def check_gemv(layer, M, config=20, xdtype="bf16", rows=None):
    K = layer["K"]
    xbits, xf = synth.draw_x(M, K, config=config, matrix=5, dtype=xdtype)
    y = gpu_gemv(layer, x_device(xbits), M)
    if rows is None:
        ref, bound = oracle_gemv_all_rows(to_oracle(layer), xf)
    else:
        ref, bound = oracle.gemv(to_oracle(layer), xf, rows=rows)
        y = y[:, rows]
    ok, worst = within_tolerance(y, ref, bound)
    assert ok, f"worst error / tolerance = {worst}"
    return worst


# Shapes whose rows are whole 16-byte multiples take the bulk-copy pipeline.
PIPELINE_SHAPES = {"nvfp4": (37, 4096), "mxfp4": (41, 2048), "q4k": (29, 1536), "q40": (33, 2048),
                   "gptq": (264, 1152), "awq": (264, 1152)}


@pytest.mark.parametrize("fmt", ALL_GEMV)
@pytest.mark.parametrize("pipeline", [False, True])
def test_gemv_batch1(fmt, pipeline):
    N, K = PIPELINE_SHAPES[fmt] if pipeline else shape_for(fmt)
    layer = synth.make_layer(fmt, N, K, config=21, matrix=1, outliers=True)
    check_gemv(layer, 1)
    check_gemv(layer, 1, xdtype="f32")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_gemv_nvfp4_tensor_core_path(M):
    """NVFP4 with K % 128 == 0 and bf16 x runs the mma.sync decode-dot kernel:
    ragged 16-row tiles, uneven K split over the warps, batch 1..8."""
    for N, K in ((45, 4096), (16, 128), (7, 1152), (263, 14336)):
        check_gemv(synth.make_layer("nvfp4", N, K, config=30, matrix=M, row_scale=True), M, config=30 + M)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_gemv_mxfp4_tensor_core_path(M):
    """MXFP4 with bf16 x on the tensor cores (E8M0 scale folded into the f16
    A fragment): batch 1..4 with K % 256 == 0 on the TMA-fed kernel (scales
    read by the lanes one stage ahead; 4096 x 11008 has 344-byte scale rows
    that no tensor map could read), otherwise the register-fed kernel."""
    for N, K in ((41, 2048), (263, 11008), (16, 128), (1, 256)):
        check_gemv(synth.make_layer("mxfp4", N, K, config=33, matrix=M, outliers=True), M, config=33 + M)
        assert q4.q4_last_gemv_path() == ("gemv_tma" if M <= 4 and K % 256 == 0 and tma_fits(K, M) else "gemv_mma")


def test_gemv_mxfp4_scales_outside_the_exact_f16_range():
    """E8M0 scales whose E2M1 multiples are not all f16 numbers (2^-40, 2^20;
    2^-23 and 2^13 are the edges that still are) send those warps' tiles
    (register-fed kernel) or stages (TMA-fed kernel, batch 1 and 4) to f32;
    the result stays within tolerance."""
    layer = synth.make_layer("mxfp4", 40, 4096, config=34, matrix=0)
    s = layer["scales"].copy()
    s[3, 5] = 127 - 40
    s[17, :] = 127 + 20
    s[30, 100] = 127 - 23
    s[31, 7] = 127 + 13
    layer = dict(layer, scales=s)
    for M in (1, 4, 8):
        check_gemv(layer, M, config=34)
        assert q4.q4_last_gemv_path() == ("gemv_tma" if M <= 4 else "gemv_mma")


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_q4k_tensor_core_path(M, xdtype):
    """Q4_K with f32 x at batch 2..8 runs the register-fed mma.sync kernel
    with one fresh accumulator per 32-k sub-block (step and offset applied on
    the CUDA cores), x staged as hi + lo f16 parts; ragged 16-row tiles and
    uneven K splits.  At batch 5..8 with K = 11008 the staged x would not fit
    in shared memory, so the batch runs as two launches of at most 4 rows.
    Batch 1, and bf16 x at any batch up to 8 (two rows per launch), take the
    TMA-fed kernel (gemv_blk_tc)."""
    for N, K in ((29, 1536), (263, 4096), (16, 256), (40, 11008)):
        check_gemv(synth.make_layer("q4k", N, K, config=35, matrix=M, outliers=True), M, config=35 + M,
                   xdtype=xdtype)
        assert q4.q4_last_gemv_path() == ("gemv_blk_tc_q4k" if M == 1 or xdtype == "bf16" else "gemv_mma_q4k")


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_q40_tensor_core_path(M, xdtype):
    """Q4_0 on the same kernels: A = q - 8, d applied per 32-k block; the code
    words of even blocks are assembled across a 4-byte boundary."""
    for N, K in ((33, 2048), (263, 11008), (16, 256)):
        check_gemv(synth.make_layer("q40", N, K, config=37, matrix=M, outliers=True), M, config=37 + M,
                   xdtype=xdtype)
        assert q4.q4_last_gemv_path() == ("gemv_blk_tc_q40" if M == 1 or xdtype == "bf16" else "gemv_mma_q40")


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_gptq_tensor_core_path(M, xdtype):
    """GPTQ (group 128, no act-order) on the tensor cores: one word of 8 codes
    per lane feeds two MMAs; s * (D - z * S) per group."""
    for N, K in ((264, 1152), (520, 4096), (16, 128), (40, 11008)):
        check_gemv(synth.make_layer("gptq", N, K, config=38, matrix=M, outliers=True), M, config=38 + M,
                   xdtype=xdtype)
        assert q4.q4_last_gemv_path() == "gemv_mma_gptq"


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 3, 4, 8, 11])
def test_gemv_awq_tensor_core_path(M, xdtype):
    """AWQ (group 128, N % 128 == 0) on the TMA-fed tensor-core kernel: the
    weights are the MMA's B operand, (q - z) * 2^b formed exactly in f16, the
    K range split over up to 8 cluster ranks (uneven: 9 and 86 groups), batch
    1..8 per launch and 11 as two launches."""
    for N, K in ((128, 1152), (384, 4096), (11008, 128), (768, 11008)):
        check_gemv(synth.make_layer("awq", N, K, config=39, matrix=M, outliers=True), M, config=39 + M,
                   xdtype=xdtype)
        assert q4.q4_last_gemv_path() == "gemv_awq_tc"
    # N % 128 != 0 stays on the CUDA-core kernel
    check_gemv(synth.make_layer("awq", 264, 1152, config=39, matrix=M), M, config=39, xdtype=xdtype)
    assert q4.q4_last_gemv_path() != "gemv_awq_tc"


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 3, 4, 5, 8, 11])
def test_gemv_gptq_tma_tensor_core_path(M, xdtype):
    """GPTQ (group 128, N % 128 == 0) on the TMA-fed tensor-core kernel: the
    weights are the MMA's A operand (byte t of a word holds k = 2t, 2t+1;
    q - z and 16 (q - z) formed exactly in f16, odd-k x staged divided by
    16), x hi and lo terms share the n8 columns (two B tiles at batch 5..8),
    the K range split over up to 8 cluster ranks, batch 11 as two launches."""
    for N, K in ((128, 1152), (384, 4096), (11008, 128), (768, 11008)):
        check_gemv(synth.make_layer("gptq", N, K, config=42, matrix=M, outliers=True), M, config=42 + M,
                   xdtype=xdtype)
        assert q4.q4_last_gemv_path() == "gemv_gptq_tc"
    # N % 128 != 0 stays on the register-fed kernel
    check_gemv(synth.make_layer("gptq", 264, 1152, config=42, matrix=M), M, config=42, xdtype=xdtype)
    assert q4.q4_last_gemv_path() != "gemv_gptq_tc"


def test_gemv_gptq_tma_tensor_core_edge_values():
    """x over 1e30 .. 1e-10, an all-zero x (exactly 0), every code and every
    stored zero (0..15, i.e. zero points 1..16) in use, and act-order (g_idx)
    tensors staying on the general kernel."""
    N, K = 256, 2048
    layer = synth.make_layer("gptq", N, K, config=43, matrix=0)
    for M in (1, 3):
        xf = np.random.default_rng(M).normal(0, 1e-10, (M, K)).astype(np.float32)
        xf[:, 7] = 1e30
        xf[:, 1501] = -3e20
        y = gpu_gemv(layer, x_device(xf), M)
        assert q4.q4_last_gemv_path() == "gemv_gptq_tc"
        ref, bound = oracle.gemv(to_oracle(layer), xf)
        ok, worst = within_tolerance(y, ref, bound)
        assert ok, worst
    y = gpu_gemv(layer, torch.zeros((2, K), dtype=torch.bfloat16, device="cuda"), 2)
    assert np.all(y == 0)
    rng = np.random.default_rng(6)
    rand = dict(layer, w=rng.integers(-2**31, 2**31, layer["w"].shape, dtype=np.int64).astype(np.int32),
                zeros=rng.integers(-2**31, 2**31, layer["zeros"].shape, dtype=np.int64).astype(np.int32))
    check_gemv(rand, 2, config=43)
    act = synth.make_layer("gptq", 256, 512, config=43, matrix=1, act_order=True)
    check_gemv(act, 1, config=43)
    assert q4.q4_last_gemv_path() != "gemv_gptq_tc"
    assert q4.q4_last_error() == 0


def test_gemv_awq_tensor_core_edge_values():
    """x over 1e30 .. 1e-10 (one power-of-two scale per batch row and rank),
    an all-zero x (exactly 0), and every code and zero point in use."""
    N, K = 512, 2048
    layer = synth.make_layer("awq", N, K, config=41, matrix=0)
    for M in (1, 3):
        xf = np.random.default_rng(M).normal(0, 1e-10, (M, K)).astype(np.float32)
        xf[:, 7] = 1e30
        xf[:, 1500] = -3e20
        y = gpu_gemv(layer, x_device(xf), M)
        assert q4.q4_last_gemv_path() == "gemv_awq_tc"
        ref, bound = oracle.gemv(to_oracle(layer), xf)
        ok, worst = within_tolerance(y, ref, bound)
        assert ok, worst
    y = gpu_gemv(layer, torch.zeros((2, K), dtype=torch.bfloat16, device="cuda"), 2)
    assert np.all(y == 0)
    rng = np.random.default_rng(5)
    rand = dict(layer, w=rng.integers(-2**31, 2**31, layer["w"].shape, dtype=np.int64).astype(np.int32),
                zeros=rng.integers(-2**31, 2**31, layer["zeros"].shape, dtype=np.int64).astype(np.int32))
    check_gemv(rand, 2, config=41)
    assert q4.q4_last_error() == 0


def test_gemv_q4k_wide_dynamic_range_x():
    """f32 x spanning 1e30 to 1e-10: the hi + lo staging keeps the result
    within tolerance (tiny values fall below the scaled f16 range)."""
    N, K = 40, 4096
    layer = synth.make_layer("q4k", N, K, config=36, matrix=0)
    for M in (1, 3):
        xf = np.random.default_rng(M).normal(0, 1e-10, (M, K)).astype(np.float32)
        xf[:, 7] = 1e30
        xf[:, 1000] = -3e20
        y = gpu_gemv(layer, x_device(xf), M)
        ref, bound = oracle.gemv(to_oracle(layer), xf)
        ok, worst = within_tolerance(y, ref, bound)
        assert ok, worst


def test_gemv_nvfp4_wide_dynamic_range_x():
    """x whose range defeats the f16 staging (1e30 next to 1e-10): those warps
    fall back to f32 and the result is still within tolerance."""
    N, K = 40, 4096
    layer = synth.make_layer("nvfp4", N, K, config=31, matrix=0)
    for M in (1, 3):
        xf = np.random.default_rng(M).normal(0, 1e-10, (M, K)).astype(np.float32)
        xf[:, 7] = 1e30
        xf[:, 1000] = -3e20
        xbits = synth.f32_to_bf16_bits(xf)
        xr = oracle.bf16_bits_to_f32(xbits).reshape(M, K)
        y = gpu_gemv(layer, x_device(xbits), M)
        ref, bound = oracle.gemv(to_oracle(layer), xr)
        ok, worst = within_tolerance(y, ref, bound)
        assert ok, worst


@pytest.mark.parametrize("M", [1, 4])
def test_gemv_grouped_matches_oracle(M):
    """One launch over several NVFP4 members sharing K: shared and separate x,
    ragged N per member; then a mixed-format group (issued member by member)."""
    K = 2048
    layers = [synth.make_layer("nvfp4", N, K, config=32, matrix=i, row_scale=True)
              for i, N in enumerate((45, 16, 263, 7))]
    xb0, xf0 = synth.draw_x(M, K, config=32, matrix=9)
    xb1, xf1 = synth.draw_x(M, K, config=32, matrix=10)
    xs = [(xb0, xf0), (xb0, xf0), (xb1, xf1), (xb0, xf0)]
    devs = [to_device(L) for L in layers]
    xd = {id(xb0): x_device(xb0), id(xb1): x_device(xb1)}
    ys = [torch.full((M, L["N"]), float("nan"), device="cuda") for L in layers]
    auxes = [aux_for(L, d, x_dtype=torch.bfloat16) for L, d in zip(layers, devs)]
    descs = [("nvfp4", d["w"], d["scales"], a, xd[id(xb)], y, L["N"], K)
             for L, d, a, (xb, _), y in zip(layers, devs, auxes, xs, ys)]
    q4.q4_gemv_grouped(descs, M)
    torch.cuda.synchronize()
    for L, (_, xf), y in zip(layers, xs, ys):
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst
    # mixed formats fall back to one q4_gemv per member
    q = synth.make_layer("q4k", 20, K, config=32, matrix=7)
    dq = to_device(q)
    xq = x_device(xf0.astype(np.float32))
    yq = torch.full((M, 20), float("nan"), device="cuda")
    descs2 = [descs[0], ("q4k", dq["w"], None, aux_for(q, dq, x_dtype=torch.float32), xq, yq, 20, K)]
    ys[0].fill_(float("nan"))
    q4.q4_gemv_grouped(descs2, M)
    torch.cuda.synchronize()
    for L, xf, y in ((layers[0], xf0, ys[0]), (q, xf0, yq)):
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst


def test_gemv_pipeline_long_rows_and_tails():
    """R=2 tiles (K > 8192), a ragged last tile, one row, and N < grid."""
    for N, K in ((4099, 14336), (1, 14336), (3, 8448), (1029, 4096)):
        check_gemv(synth.make_layer("nvfp4", N, K, config=21, matrix=N % 7), 1)
    check_gemv(synth.make_layer("q4k", 517, 11008, config=21, matrix=9), 1)
    check_gemv(synth.make_layer("q40", 131, 11008, config=21, matrix=10), 1)
    assert q4.q4_last_error() == 0


@pytest.mark.parametrize("fmt", ALL_GEMV)
@pytest.mark.parametrize("M", [2, 4, 8])
def test_gemv_small_batch(fmt, M):
    N, K = shape_for(fmt)
    layer = synth.make_layer(fmt, N, K, config=22, matrix=M, row_scale=True)
    check_gemv(layer, M)


def test_gemv_general_paths():
    # NVFP4 with K % 32 == 16 and act-order GPTQ take the general kernel.
    check_gemv(synth.make_layer("nvfp4", 21, 1040, config=23, matrix=1), 1)
    check_gemv(synth.make_layer("gptq", 40, 512, config=23, matrix=2, act_order=True), 1)
    check_gemv(synth.make_layer("gptq", 40, 512, config=23, matrix=3, act_order=True), 3)
    check_gemv(synth.make_layer("nvfp4", 5, 16, config=23, matrix=4), 1)


@pytest.mark.parametrize("fmt", ALL_GEMV)
def test_gemv_random_bytes_edge(fmt):
    """Random codes everywhere; single row; the all-zero x gives exactly 0."""
    N, K = (8, 256) if fmt in ("gptq", "awq") else (1, 512)
    layer = synth.make_layer(fmt, N, K, config=24, matrix=1)
    check_gemv(layer, 1)
    d = to_device(layer)
    y = torch.full((1, N), 7.0, device="cuda")
    xz = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    q4.q4_gemv(fmt, d["w"], d["scales"], aux_for(layer, d, x_dtype=torch.bfloat16), xz, y, 1, N, K)
    torch.cuda.synchronize()
    assert torch.all(y == 0)


def test_gemv_one_hot_gives_exact_column():
    layer = synth.make_layer("nvfp4", 64, 4096, config=25, matrix=1)
    ref = oracle.dequant(to_oracle(layer))
    for k in (0, 17, 4095):
        x = torch.zeros((1, 4096), dtype=torch.bfloat16, device="cuda")
        x[0, k] = 1.0
        y = gpu_gemv(layer, x, 1)[0]
        assert np.array_equal(y, ref[:, k])      # exact; a -0.0 weight sums to +0.0


# Full-size workloads (the decode-GEMV study's layer shapes), every row.
FULL = [
    ("nvfp4", 1024, 4096, dict(), 0),                        # NVFP4 1024 x 4096
    ("q4k", 4096, 4096, dict(), 1),                          # Q4_K 4096 x 4096
    ("mxfp4", 4096, 11008, dict(outliers=True), 2),          # MXFP4 4096 x 11008
    ("q40", 4096, 11008, dict(outliers=True), 2),            # Q4_0 4096 x 11008
    ("gptq", 4096, 11008, dict(outliers=True), 2),
    ("awq", 4096, 11008, dict(outliers=True), 2),
    ("nvfp4", 14336, 4096, dict(row_scale=True), 5),         # MLP gate/up of the 4096x14336 set
    ("nvfp4", 4096, 14336, dict(row_scale=True), 5),         # MLP down
]


@pytest.mark.parametrize("fmt,N,K,kw,config", FULL)
def test_gemv_full_size_every_row(fmt, N, K, kw, config):
    layer = synth.make_layer(fmt, N, K, config=config, matrix=0, **kw)
    for M in (1, 4):
        for xdtype in ("bf16", "f32"):
            check_gemv(layer, M, config=config, xdtype=xdtype)


# ------------------------------------------------------------------ repack

def gpu_repack(layer, dst, perm=False):
    N, K = layer["N"], layer["K"]
    d = to_device(layer)
    group = 32 if layer["fmt"] == "q40" else layer["group"]
    if dst == "gptq":
        w = torch.empty((K // 8, N), dtype=torch.int32, device="cuda")
        z = torch.empty((K // group, N // 8), dtype=torch.int32, device="cuda")
    elif dst == "awq":
        w = torch.empty((K, N // 8), dtype=torch.int32, device="cuda")
        z = torch.empty((K // group, N // 8), dtype=torch.int32, device="cuda")
    elif dst == "logical":
        w = torch.empty((K, N), dtype=torch.uint8, device="cuda")
        z = torch.empty((K // group, N), dtype=torch.uint8, device="cuda")
    else:
        w = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
        z = None
    if dst in ("nvfp4", "nvfp4_splithalf"):
        s = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
    else:
        s = torch.empty((K // group, N), dtype=torch.int16, device="cuda")
    p = torch.empty((K,), dtype=torch.int32, device="cuda") if perm else None
    rc = q4.q4_repack(layer["fmt"], d["w"], d["scales"], aux_for(layer, d), dst, w, s, z, p, N, K,
                      check=False)
    torch.cuda.synchronize()
    out = [w.cpu().numpy(), s.cpu().numpy(), None if z is None else z.cpu().numpy(),
           None if p is None else p.cpu().numpy()]
    return rc, out


@pytest.mark.parametrize("src,dst", [("gptq", "awq"), ("awq", "gptq"), ("gptq", "logical"),
                                     ("logical", "gptq"), ("awq", "logical"), ("q40", "gptq"),
                                     ("q40", "awq"), ("q40", "logical"), ("gptq", "gptq"),
                                     ("nvfp4", "nvfp4_splithalf"), ("nvfp4_splithalf", "nvfp4")])
def test_repack_bit_exact(src, dst):
    N, K = (72, 512) if src != "q40" else (40, 512)
    layer = synth.make_layer(src, N, K, config=26, matrix=1, outliers=True)
    rc, (w, s, z, _) = gpu_repack(layer, dst)
    assert rc == q4.Q4_OK
    ew, es, ez, eperm = packing.repack(src, dst, N, K, layer["w"], layer["scales"], layer["zeros"],
                                       layer["group"])
    assert eperm is None
    assert np.array_equal(w.view(np.uint8), np.ascontiguousarray(ew).view(np.uint8))
    assert np.array_equal(s.view(np.uint8), np.ascontiguousarray(es).view(np.uint8))
    if ez is not None:
        assert np.array_equal(z.view(np.uint8), np.ascontiguousarray(ez).view(np.uint8))
    # the target dequantizes to the same weights, bit for bit (on the GPU too)
    tgt = dict(layer, fmt=dst, w=w, scales=s, zeros=z, group=32 if src == "q40" else layer["group"])
    if s.dtype == np.int16:
        tgt["scales"] = s.view(np.uint16)
    assert bits_equal(gpu_dequant(tgt).cpu().numpy(), oracle.dequant(to_oracle(layer)))


def test_repack_act_order_to_awq():
    N, K = 48, 1024
    layer = synth.make_layer("gptq", N, K, config=27, matrix=1, act_order=True)
    rc, (w, s, z, perm) = gpu_repack(layer, "awq", perm=True)
    assert rc == q4.Q4_OK
    ew, es, ez, eperm = packing.repack("gptq", "awq", N, K, layer["w"], layer["scales"], layer["zeros"],
                                       layer["group"], g_idx=layer["g_idx"])
    assert np.array_equal(perm, eperm)
    assert np.array_equal(w, ew) and np.array_equal(s.view(np.uint16), es) and np.array_equal(z, ez)


def test_repack_rejections():
    # a non-trivial g_idx without perm_out, and a zero the target cannot hold
    layer = synth.make_layer("gptq", 16, 512, config=28, matrix=1, act_order=True)
    rc, _ = gpu_repack(layer, "awq", perm=False)
    assert rc == q4.Q4_EINVAL
    lg = synth.make_layer("logical", 16, 256, config=28, matrix=2)
    lg["zeros"] = lg["zeros"].copy()
    lg["zeros"][0, 3] = 0
    rc, _ = gpu_repack(lg, "gptq")
    assert rc == q4.Q4_ERANGE
    lg["zeros"][0, 3] = 16
    rc, _ = gpu_repack(lg, "awq")
    assert rc == q4.Q4_ERANGE
    rc, _ = gpu_repack(lg, "gptq")
    assert rc == q4.Q4_OK


# ---------------------------------------------------------------- validate

@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "q4k", "q40", "gptq", "awq"])
def test_validate_counts_nan_scales(fmt):
    N, K = shape_for(fmt)
    layer = synth.make_layer(fmt, N, K, config=29, matrix=1)
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")

    def run(lay):
        d = to_device(lay)
        return q4.q4_validate(fmt, d["w"], d["scales"], aux_for(lay, d), N, K, cnt)
    assert run(layer) == q4.Q4_OK and int(cnt[0]) == 0
    bad = dict(layer)
    if fmt in ("nvfp4", "mxfp4"):
        s = layer["scales"].copy()
        s.flat[[0, 5, s.size - 1]] = 0xFF
        if fmt == "nvfp4":
            s.flat[7] = 0x7F
        bad["scales"] = s
        want = 4 if fmt == "nvfp4" else 3
        assert oracle.count_nan_scales(fmt, s) == want
    elif fmt in ("q4k", "q40"):
        w = layer["w"].copy()
        w[0, 0, 0:2] = np.array([np.float16(np.nan)]).view(np.uint8)
        w[-1, -1, 0:2] = np.array([np.float16(np.inf)]).view(np.uint8)
        bad["w"] = w
        want = 2
    else:
        s = layer["scales"].copy()
        s.flat[[1, 9]] = np.array([np.float16(np.nan)]).view(np.uint16)[0]
        bad["scales"] = s
        want = 2
    assert run(bad) == q4.Q4_ENAN and int(cnt[0]) == want
    if fmt == "nvfp4":
        d = to_device(layer)
        assert q4.q4_validate(fmt, d["w"], d["scales"], q4.make_aux(scale2=float("nan"), fmt=fmt),
                              N, K, cnt) == q4.Q4_ESCALE2
