"""The integer-exact NVFP4 A16-Q8 contraction ([MUS7] 7.4.2) on the GPU,
through the C ABI, against the CPU oracle.

The lane is bit-reproducible by construction (an exact integer block sum and
a pinned f32 epilogue), so the bar is bit-exact equality with the oracle on
every output, at small ragged shapes, at the full 14336 x 4096 layer, and on
the edge cases: zero activation blocks, negative scale bytes, partial
1024-k chunks, N not a multiple of the warps per CTA, batches that span
several launches.  Batch 1 and 2 run the tensor-core kernel (exact f16 group
dots), larger batches the CUDA-core one: the batch-independence test checks
the two against each other bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth

from _helpers import oracle_gemv_all_rows, to_device, to_oracle, x_device

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def bits_equal(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


def gpu_a16q8(layer, xdev, M):
    d = to_device(layer)
    N, K = layer["N"], layer["K"]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(scale2=layer["scale2"], x_dtype=xdev.dtype, fmt="nvfp4")
    q4.q4_gemv_a16q8(d["w"], d["scales"], aux, xdev, y, M, N, K)
    torch.cuda.synchronize()
    # batch 1 and 2 (staged codes and three ring stages within shared memory) take the
    # tensor-core kernel; larger batches the CUDA-core one; both hold the same contract
    assert q4.q4_last_gemv_path() == ("gemv_a16q8_tc" if M <= 2 and K <= (14336 if M == 1 else 6144)
                                      else "gemv_a16q8")
    assert q4.q4_last_error() == q4.Q4_OK
    return y.cpu().numpy()


def draw(N, K, M, xdtype, config=30, matrix=0):
    layer = synth.make_layer("nvfp4", N, K, config=config, matrix=matrix, row_scale=True)
    xdev_host, xf = synth.draw_x(M, K, config=config, matrix=matrix, dtype=xdtype)
    return layer, xdev_host, xf


@pytest.mark.parametrize("N,K,M,xdtype", [
    (1024, 4096, 1, "bf16"),     # the 1024 x 4096 batch-1 layer
    (1000, 768, 1, "f32"),       # N % 8 != 0, K below one 1024-k chunk
    (333, 4352, 3, "bf16"),      # a partial last chunk after a full in-flight batch; batch 3 on the 4-row form
    (64, 2048, 8, "f32"),        # the 8-row form
    (40, 1280, 9, "bf16"),       # two launches (8 + 1 rows)
    (17, 256, 2, "bf16"),        # one block per row
])
def test_a16q8_bit_exact(N, K, M, xdtype):
    layer, xh, xf = draw(N, K, M, xdtype)
    ref = oracle.gemv_a16q8(to_oracle(layer), xf)
    got = gpu_a16q8(layer, x_device(xh), M)
    assert bits_equal(got, ref)


def test_a16q8_zero_blocks_and_negative_scales():
    N, K, M = 96, 2048, 2
    layer, xh, xf = draw(N, K, M, "f32", matrix=1)
    xf = xf.copy()
    xf[0, 256:512] = 0.0                      # an all-zero block: codes 0, scale 0
    xf[1, 1024:1280] = 0.0
    xf[1, 1300] = -0.0
    s = layer["scales"].copy()
    rng = np.random.default_rng(4)
    s[rng.random(s.shape) < 0.3] |= 0x80      # E4M3FN sign bit honoured
    layer = dict(layer, scales=s)
    ref = oracle.gemv_a16q8(to_oracle(layer), xf)
    got = gpu_a16q8(layer, x_device(xf), M)
    assert bits_equal(got, ref)


def test_a16q8_exact_inputs_give_the_exact_binary16_result():
    """Integer activations whose blocks peak at +-127 and scale bytes 1..8:
    every step is exact, so y is the binary16 rounding of the f64 GEMV."""
    N, K, M = 48, 1024, 3
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    w = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sb = rng.integers(1, 9, (N, K // 16)).astype(np.uint8)
    x = rng.integers(-126, 127, (M, K)).astype(np.float32)
    for m in range(M):
        for b in range(K // 256):
            x[m, b * 256 + rng.integers(0, 256)] = 127.0 * rng.choice([-1.0, 1.0])
    layer = {"fmt": "nvfp4", "N": N, "K": K, "w": w, "scales": sb, "zeros": None, "g_idx": None,
             "group": 128, "scale2": 0.125}
    y64, _ = oracle.gemv(to_oracle(layer), x)
    want = y64.astype(np.float32).astype(np.float16).astype(np.float32)
    assert bits_equal(gpu_a16q8(layer, x_device(x), M), want)


def test_a16q8_rows_do_not_depend_on_the_batch():
    N, K = 200, 3072
    layer, xh, _ = draw(N, K, 5, "bf16", matrix=2)
    xdev = x_device(xh)
    y5 = gpu_a16q8(layer, xdev, 5)
    for m in (0, 3, 4):
        assert bits_equal(gpu_a16q8(layer, xdev[m:m + 1].contiguous(), 1)[0], y5[m])
    assert bits_equal(gpu_a16q8(layer, xdev, 5), y5)      # repeated calls agree bit for bit


def test_a16q8_full_layer_14336x4096():
    N, K = 14336, 4096
    layer, xh, xf = draw(N, K, 1, "bf16", config=31)
    ref = oracle.gemv_a16q8(to_oracle(layer), xf)
    got = gpu_a16q8(layer, x_device(xh), 1)
    assert bits_equal(got, ref)
    # and it stays within the activation-quantization error of the exact GEMV
    y64, bound = oracle_gemv_all_rows(to_oracle(layer), xf[:, :K])
    err = np.abs(got.astype(np.float64) - y64)
    assert np.all(err <= 0.02 * bound + 1e-3)


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("xdtype", ["bf16", "f32"])
def test_a16q8_tensor_core_shapes(M, xdtype):
    """The tensor-core kernel on ragged shapes: a partial last 2048-k stage
    (K = 2304, 4352), one 256-k block, a 17-row last tile, more tiles than
    CTAs, K = 14336 at batch 1, extreme activation ranges; bit-exact."""
    shapes = [(4099, 2304), (17, 256), (5000, 4352), (300, 4096)]
    if M == 1:
        shapes.append((131, 14336))
    for i, (N, K) in enumerate(shapes):
        layer, xh, xf = draw(N, K, M, xdtype, config=32, matrix=i)
        ref = oracle.gemv_a16q8(to_oracle(layer), xf)
        assert bits_equal(gpu_a16q8(layer, x_device(xh), M), ref), (N, K)
    N, K = 64, 2048
    layer, _, _ = draw(N, K, M, xdtype, config=33)
    xf = np.random.default_rng(3).normal(0, 1e-10, (M, K)).astype(np.float32)
    xf[:, 5] = 1e30
    xf[:, 300] = -3e20
    xf[M - 1, 512:768] = 0.0
    ref = oracle.gemv_a16q8(to_oracle(layer), xf)
    assert bits_equal(gpu_a16q8(layer, x_device(xf), M), ref)
