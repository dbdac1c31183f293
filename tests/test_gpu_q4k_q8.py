"""The Q4_K x Q8 (W4A8) contraction ([W4K] section 7) on the GPU, through the
C ABI, bit-exact against the CPU oracle: ragged N, partial 4-block steps,
batches across launches, zero blocks, f32 and bf16 x, the full layer."""
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


def gpu_q4k_q8(w, xdev, M, N, K):
    wd = torch.from_numpy(np.ascontiguousarray(w)).cuda()
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(x_dtype=xdev.dtype, fmt="q4k")
    q4.q4_gemv_q4k_q8(wd, aux, xdev, y, M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_last_gemv_path() == "gemv_q4k_q8"
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K,M,xdtype", [
    (4096, 4096, 1, "f32"),      # the 4096 x 4096 Q4_K layer at batch 1
    (1000, 1280, 1, "bf16"),     # N % 8 != 0; 5 super-blocks: a partial 4-block step
    (333, 4608, 3, "f32"),       # 18 super-blocks: two in-flight batches; batch 3
    (64, 2048, 8, "bf16"),       # the 8-row form
    (40, 1024, 9, "f32"),        # two launches
    (17, 256, 2, "bf16"),
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
