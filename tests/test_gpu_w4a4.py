"""The W4A4 contraction ([MUS7] 7.4.3) on the GPU, through the C ABI, bit-exact
against the CPU oracle: ragged N, K of one 64-k step, batches across
launches, negative weight scales, zero groups, f32 and bf16 x, the full layer."""
import numpy as np
import pytest

import oracle
import synth

from _helpers import to_device, to_oracle, x_device

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


def isi_for(xf):
    return float(np.float32(2688.0) / np.float32(np.abs(xf).max()))


def gpu_w4a4(layer, xdev, isi, M):
    d = to_device(layer)
    N, K = layer["N"], layer["K"]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    aux = q4.make_aux(scale2=layer["scale2"], x_dtype=xdev.dtype, fmt="nvfp4")
    q4.q4_gemv_w4a4(d["w"], d["scales"], aux, isi, xdev, y, M, N, K)
    torch.cuda.synchronize()
    assert q4.q4_last_gemv_path() == "gemv_w4a4"
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K,M,xdtype", [(1024, 4096, 1, "bf16"), (1000, 64, 1, "f32"), (333, 4352, 3, "bf16"),
                                          (64, 2048, 8, "f32"), (40, 1280, 9, "bf16"), (14336, 4096, 1, "bf16")])
def test_w4a4_bit_exact(N, K, M, xdtype):
    layer = synth.make_layer("nvfp4", N, K, config=90, matrix=0, row_scale=True)
    xh, xf = synth.draw_x(M, K, config=90, matrix=1, dtype=xdtype)
    isi = isi_for(xf)
    ref = oracle.gemv_w4a4(to_oracle(layer), xf, isi)
    assert bits_equal(gpu_w4a4(layer, x_device(xh), isi, M), ref)


def test_w4a4_zero_groups_and_negative_scales():
    N, K, M = 96, 512, 2
    layer = synth.make_layer("nvfp4", N, K, config=91, matrix=0)
    _, xf = synth.draw_x(M, K, config=91, matrix=1, dtype="f32")
    xf = xf.copy()
    xf[0, 32:48] = 0.0
    s = layer["scales"].copy()
    s[np.random.default_rng(2).random(s.shape) < 0.3] |= 0x80
    layer = dict(layer, scales=s)
    isi = isi_for(xf)
    assert bits_equal(gpu_w4a4(layer, x_device(xf), isi, M), oracle.gemv_w4a4(to_oracle(layer), xf, isi))
