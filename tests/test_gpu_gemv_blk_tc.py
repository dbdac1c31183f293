"""Batch-1 Q4_K and Q4_0 GEMV on the TMA-fed tensor-core kernel
(gemv_blk_tc) against the CPU oracle, through the C ABI, every row within
|y_gpu - y_ref| <= 1e-5 * sum|w||x| + 1e-6.

The shapes cover: a single 256-k unit (warps 1-7 idle), ragged last stages
(9, 17 and 43 units over 2048-k stages), ragged last 16-row tiles, more tiles
than CTAs (the ring runs across tile boundaries), and K = 14336, whose staged
x leaves too little shared memory for the ring (the register-fed kernel takes
it).  Edge cases: x spanning 1e-10 .. 1e30, all-zero x, random code and scale
bytes, one-hot x (exact columns), all-zero weights, repeated calls bit for
bit.  Groups of one format and one K sharing x run as one launch.  With bf16
x the kernel takes two batch rows per launch (B columns 2t and 2t + 1 carry
a row each), up to 8 rows in launches of two."""
import numpy as np
import pytest

import oracle
import synth

from _helpers import aux_for, oracle_gemv_all_rows, to_device, to_oracle, within_tolerance, x_device

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu

FMTS = ["q4k", "q40"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def run(layer, x, M=1):
    d = to_device(layer)
    N, K = layer["N"], layer["K"]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_gemv(layer["fmt"], d["w"], d["scales"], aux_for(layer, d, x_dtype=x.dtype), x, y, M, N, K)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check(layer, xf, x):
    y = run(layer, x, xf.shape[0])
    ref, bound = oracle_gemv_all_rows(to_oracle(layer), xf)
    ok, worst = within_tolerance(y, ref, bound)
    assert ok, f"worst error / tolerance = {worst}"
    return y


SHAPES = [(1, 256), (16, 256), (29, 1536), (263, 4096), (40, 11008), (5000, 2304), (4099, 4352)]


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_shapes(fmt, xdtype):
    for i, (N, K) in enumerate(SHAPES):
        layer = synth.make_layer(fmt, N, K, config=140, matrix=i, outliers=True)
        xb, xf = synth.draw_x(1, K, config=140, matrix=20 + i, dtype=xdtype)
        check(layer, xf, x_device(xb))
        assert q4.q4_last_gemv_path() == f"gemv_blk_tc_{fmt}"
    assert q4.q4_last_error() == q4.Q4_OK


@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_other_shapes_keep_the_register_fed_kernel(fmt):
    layer = synth.make_layer(fmt, 40, 14336, config=141, matrix=0)
    xb, xf = synth.draw_x(1, 14336, config=141, matrix=1, dtype="f32")
    check(layer, xf, x_device(xb))
    assert q4.q4_last_gemv_path() == f"gemv_mma_{fmt}"
    small = synth.make_layer(fmt, 40, 2048, config=141, matrix=2)
    xb, xf = synth.draw_x(2, 2048, config=141, matrix=3, dtype="f32")     # batch 2 with f32 x
    check(small, xf, x_device(xb))
    assert q4.q4_last_gemv_path() == f"gemv_mma_{fmt}"


@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_edge_values(fmt):
    N, K = 300, 2304
    layer = synth.make_layer(fmt, N, K, config=142, matrix=0)
    # x over 1e-10 .. 1e30 (the per-warp power-of-two scale and the hi + lo split)
    xf = np.random.default_rng(1).normal(0, 1e-10, (1, K)).astype(np.float32)
    xf[0, 7] = 1e30
    xf[0, 1501] = -3e20
    xf[0, 2300] = 5e-3
    check(layer, xf, x_device(xf))
    assert q4.q4_last_gemv_path() == f"gemv_blk_tc_{fmt}"
    # all-zero x gives exactly 0
    for xz in (torch.zeros((1, K), dtype=torch.bfloat16, device="cuda"), torch.zeros((1, K), device="cuda")):
        assert np.all(run(layer, xz) == 0)
    # random code, scale and min bytes with finite fp16 headers
    rng = np.random.default_rng(2)
    if fmt == "q4k":
        b = synth.random_bytes((N, K // 256, 144), 5)
        b[:, :, :4] = rng.uniform(-2, 2, (N, K // 256, 2)).astype(np.float16).view(np.uint8).reshape(N, K // 256, 4)
    else:
        b = synth.random_bytes((N, K // 32, 18), 6)
        b[:, :, :2] = rng.uniform(-2, 2, (N, K // 32)).astype(np.float16).view(np.uint8).reshape(N, K // 32, 2)
    rand = dict(layer, w=b)
    for xdtype in ("f32", "bf16"):
        xb, xf = synth.draw_x(1, K, config=142, matrix=3, dtype=xdtype)
        check(rand, xf, x_device(xb))
    # one-hot x: every product and sum is exact, so y is the dequantized column bit for bit
    ref = oracle.dequant(to_oracle(rand))
    for k in (0, 31, 32, 63, 64, 255, 256, 1000, K - 1):
        x = torch.zeros((1, K), device="cuda")
        x[0, k] = 1.0
        assert np.array_equal(run(rand, x)[0], ref[:, k]), k
    # all-zero weights (Q4_K: scales and mins 0; Q4_0: every code 8) give exactly 0
    z = b.copy()
    if fmt == "q4k":
        z[:, :, 4:16] = 0
    else:
        z[:, :, 2:] = 0x88
    xb, xf = synth.draw_x(1, K, config=142, matrix=4, dtype="f32")
    assert np.all(run(dict(layer, w=z), x_device(xb)) == 0)
    assert q4.q4_last_error() == q4.Q4_OK


@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_repeated_calls_bit_identical(fmt):
    N, K = 4096, 4096
    layer = synth.make_layer(fmt, N, K, config=143, matrix=0)
    xb, _ = synth.draw_x(1, K, config=143, matrix=1, dtype="f32")
    x = x_device(xb)
    first = run(layer, x)
    for _ in range(3):
        assert np.array_equal(run(layer, x).view(np.uint32), first.view(np.uint32))


@pytest.mark.parametrize("xdtype", ["f32", "bf16"])
@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_grouped_shared_x(fmt, xdtype):
    """q4_gemv_grouped over members of one format and one K that read the same
    x: one launch whose tile list runs through the members (ragged last
    tiles, a 17-row member), every row against the oracle and bit for bit
    equal to the members' own q4_gemv calls."""
    K = 2304
    Ns = (4096, 1024, 1000, 17, 520)
    layers = [synth.make_layer(fmt, N, K, config=144, matrix=i, outliers=True) for i, N in enumerate(Ns)]
    devs = [to_device(L) for L in layers]
    xb, xf = synth.draw_x(1, K, config=144, matrix=9, dtype=xdtype)
    x = x_device(xb)
    ys = [torch.full((1, N), float("nan"), dtype=torch.float32, device="cuda") for N in Ns]
    descs = [(fmt, d["w"], d["scales"], aux_for(L, d, x_dtype=x.dtype), x, y, L["N"], K)
             for L, d, y in zip(layers, devs, ys)]
    q4.q4_gemv_grouped(descs, 1)
    assert q4.q4_last_gemv_path() == f"gemv_blk_tc_{fmt}_group"
    torch.cuda.synchronize()
    for L, d, y in zip(layers, devs, ys):
        got = y.cpu().numpy()
        ref, bound = oracle_gemv_all_rows(to_oracle(L), xf)
        ok, worst = within_tolerance(got, ref, bound)
        assert ok, worst
        single = run(L, x)
        assert np.array_equal(single.view(np.uint32), got.view(np.uint32))
    assert q4.q4_last_error() == q4.Q4_OK


@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_groups_it_does_not_take(fmt):
    """Members with different x, or of different formats, run as their own
    q4_gemv calls (same results)."""
    K = 1024
    other = "q40" if fmt == "q4k" else "q4k"
    layers = [synth.make_layer(fmt, 64, K, config=145, matrix=0), synth.make_layer(other, 48, K, config=145, matrix=1)]
    devs = [to_device(L) for L in layers]
    xb, xf = synth.draw_x(1, K, config=145, matrix=2, dtype="f32")
    x = x_device(xb)
    x2 = x.clone()
    for xs in ((x, x), (x, x2)):
        ys = [torch.full((1, L["N"]), float("nan"), device="cuda") for L in layers]
        descs = [(L["fmt"], d["w"], d["scales"], aux_for(L, d, x_dtype=x.dtype), xx, y, L["N"], K)
                 for L, d, xx, y in zip(layers, devs, xs, ys)]
        q4.q4_gemv_grouped(descs, 1)
        assert not q4.q4_last_gemv_path().endswith("_group")
        torch.cuda.synchronize()
        for L, y in zip(layers, ys):
            ref, bound = oracle_gemv_all_rows(to_oracle(L), xf)
            ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
            assert ok, worst
    # same format, different x: also per member
    same = [synth.make_layer(fmt, 40, K, config=145, matrix=3 + i) for i in range(2)]
    dsame = [to_device(L) for L in same]
    ys = [torch.full((1, 40), float("nan"), device="cuda") for _ in same]
    descs = [(fmt, d["w"], d["scales"], aux_for(L, d, x_dtype=x.dtype), xx, y, 40, K)
             for L, d, xx, y in zip(same, dsame, (x, x2), ys)]
    q4.q4_gemv_grouped(descs, 1)
    assert q4.q4_last_gemv_path() == f"gemv_blk_tc_{fmt}"
    torch.cuda.synchronize()
    for L, y in zip(same, ys):
        ref, bound = oracle_gemv_all_rows(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [2, 3, 4, 5, 8])
def test_blk_tc_bf16_batches(fmt, M):
    """bf16 x at batch 2..8: launches of two rows (and one for an odd last
    row), each row with its own per-block scales; ragged tiles and stages,
    K = 11008 included (the two-row stage fits as the one-row stage does)."""
    for i, (N, K) in enumerate(((263, 4096), (40, 11008), (1029, 2304), (16, 256))):
        layer = synth.make_layer(fmt, N, K, config=146, matrix=i, outliers=True)
        xb, xf = synth.draw_x(M, K, config=146, matrix=20 + M, dtype="bf16")
        check(layer, xf, x_device(xb))
        assert q4.q4_last_gemv_path() == f"gemv_blk_tc_{fmt}"
    assert q4.q4_last_error() == q4.Q4_OK


@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_bf16_batch_rows_are_independent(fmt):
    """Each batch row of a two-row launch equals that row computed alone (same
    per-block scaling, same sums), bit for bit; edge rows: all zero, one-hot,
    and 1e30 next to 1e-10 noise in the other row."""
    N, K = 300, 2304
    layer = synth.make_layer(fmt, N, K, config=147, matrix=0)
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (4, K)).astype(np.float32)
    x[1] = 0.0
    x[2] = 0.0
    x[2, 700] = 1.0
    x[3] = rng.normal(0, 1e-10, K)
    x[3, 9] = 1e30
    xb = x.astype(np.float32).view(np.uint32)
    bits = ((xb + 0x7FFF + ((xb >> 16) & 1)) >> 16).astype(np.uint16)    # round to bf16
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    xd = x_device(bits)
    together = run(layer, xd, 4)
    for m in range(4):
        alone = run(layer, x_device(bits[m:m + 1]), 1)
        assert np.array_equal(alone[0].view(np.uint32), together[m].view(np.uint32)), m
    ref, bound = oracle_gemv_all_rows(to_oracle(layer), xf)
    ok, worst = within_tolerance(together, ref, bound)
    assert ok, worst
    assert np.all(together[1] == 0)


@pytest.mark.parametrize("fmt", FMTS)
def test_blk_tc_grouped_bf16_batch4(fmt):
    """A grouped call at batch 4 with bf16 x: two launches of two rows over the
    members' joint tile list, every row of every member against the oracle."""
    K = 4096
    Ns = (4096, 1000, 17)
    layers = [synth.make_layer(fmt, N, K, config=148, matrix=i) for i, N in enumerate(Ns)]
    devs = [to_device(L) for L in layers]
    xb, xf = synth.draw_x(4, K, config=148, matrix=9, dtype="bf16")
    x = x_device(xb)
    ys = [torch.full((4, N), float("nan"), dtype=torch.float32, device="cuda") for N in Ns]
    descs = [(fmt, d["w"], d["scales"], aux_for(L, d, x_dtype=x.dtype), x, y, L["N"], K)
             for L, d, y in zip(layers, devs, ys)]
    q4.q4_gemv_grouped(descs, 4)
    assert q4.q4_last_gemv_path() == f"gemv_blk_tc_{fmt}_group"
    torch.cuda.synchronize()
    for L, y in zip(layers, ys):
        ref, bound = oracle_gemv_all_rows(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst
