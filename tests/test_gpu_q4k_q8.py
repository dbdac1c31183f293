"""The Q4_K x Q8 (W4A8) contraction ([W4K] section 7) on the GPU, through the
C ABI, bit-exact against the CPU oracle: ragged N, partial 4-block steps,
batches across launches, zero blocks, f32 and bf16 x, the full layer, the
largest codes, scales and activation codes.  Batch 1 and 2 (K up to 12288
and 10240) run the tensor-core kernel (exact sub-block sums from f16 MMAs),
other batches the CUDA-core one; a batch-independence test checks the two
against each other bit for bit."""
import numpy as np
import pytest

import oracle
import synth

from _helpers import x_device

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


def expected_path(M, K):
    return "gemv_q4k_q8_tc" if (M == 1 and K <= 12288) or (M == 2 and K <= 10240) else "gemv_q4k_q8"


def gpu_q4k_q8(w, xdev, M, N, K):
    wd = torch.from_numpy(np.ascontiguousarray(w)).cuda()
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(x_dtype=xdev.dtype, fmt="q4k")
    assert q4.q4_gemv_q4k_q8(wd, aux, xdev, y, M, N, K) == q4.Q4_OK
    torch.cuda.synchronize()
    assert q4.q4_last_gemv_path() == expected_path(M, K)
    assert q4.q4_last_error() == q4.Q4_OK
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K,M,xdtype", [
    (4096, 4096, 1, "f32"),      # the 4096 x 4096 Q4_K layer at batch 1
    (1000, 1280, 1, "bf16"),     # N % 8 != 0; 5 super-blocks: a partial 4-block step
    (333, 4608, 3, "f32"),       # 18 super-blocks: two in-flight batches; batch 3
    (64, 2048, 8, "bf16"),       # the 8-row form
    (40, 1024, 9, "f32"),        # two launches
    (17, 256, 2, "bf16"),
    (333, 4608, 2, "f32"),       # two rows on the tensor cores; 18 super-blocks: a partial last stage
    (4096, 11008, 1, "bf16"),    # K = 11008: 43 super-blocks, three ring stages
    (16, 12288, 1, "f32"),       # one tile at the largest K the tensor-core kernel takes
    (40, 14336, 1, "bf16"),      # past it: the CUDA-core kernel
])
def test_q4k_q8_bit_exact(N, K, M, xdtype):
    layer = synth.make_layer("q4k", N, K, config=70, matrix=0)
    xh, xf = synth.draw_x(M, K, config=70, matrix=1, dtype=xdtype)
    ref = oracle.gemv_q4k_q8(oracle.Tensor("q4k", N, K, layer["w"]), xf)
    assert bits_equal(gpu_q4k_q8(layer["w"], x_device(xh), M, N, K), ref)


def test_q4k_q8_zero_blocks_and_full_layer():
    N, K = 14336, 4096
    layer = synth.make_layer("q4k", N, K, config=71, matrix=0)
    _, xf = synth.draw_x(2, K, config=71, matrix=1, dtype="f32")
    xf = xf.copy()
    xf[0, 512:768] = 0.0
    ref = oracle.gemv_q4k_q8(oracle.Tensor("q4k", N, K, layer["w"]), xf)
    assert bits_equal(gpu_q4k_q8(layer["w"], x_device(xf), 2, N, K), ref)


def test_q4k_q8_largest_codes():
    """Every code 15, every 6-bit scale and minimum 63, activations at +-127
    codes: the largest sub-block sums (32 * 15 * 127) and I1 terms."""
    N, K, M = 48, 2048, 2
    layer = synth.make_layer("q4k", N, K, config=72, matrix=0)
    w = layer["w"].copy()                                    # [N][K/256][144]
    w[:, :, 4:] = 0xFF
    rng = np.random.default_rng(72)
    xf = (rng.choice([-1.0, 1.0], size=(M, K)) * rng.uniform(0.999, 1.0, size=(M, K))).astype(np.float32)
    xf[:, ::256] = np.where(xf[:, ::256] < 0, -1.0, 1.0)     # each block's largest magnitude first
    ref = oracle.gemv_q4k_q8(oracle.Tensor("q4k", N, K, w), xf)
    assert bits_equal(gpu_q4k_q8(w, x_device(xf), M, N, K), ref)


def test_q4k_q8_batch_independent():
    """The tensor-core kernel (batch 1 and 2) and the CUDA-core kernel (batch 5)
    give the same bits for the same rows of x."""
    N, K = 700, 3072
    layer = synth.make_layer("q4k", N, K, config=73, matrix=0)
    xh, _ = synth.draw_x(5, K, config=73, matrix=1, dtype="bf16")
    x5 = x_device(xh)
    y5 = gpu_q4k_q8(layer["w"], x5, 5, N, K)
    for m in range(5):
        y1 = gpu_q4k_q8(layer["w"], x5[m:m + 1].contiguous(), 1, N, K)
        assert bits_equal(y1[0], y5[m])
    y2 = gpu_q4k_q8(layer["w"], x5[3:5].contiguous(), 2, N, K)
    assert bits_equal(y2, y5[3:5])
