"""W4A4 on the native block-scaled FP4 tensor cores, through the C ABI.

The activation quantizer with a given tensor scale (q4_quantize_nvfp4_scaled)
is bit-exact against the oracle's group rule (oracle.quantize_nvfp4_groups).
The contraction (q4_gemv_w4a4_tc) multiplies the stored E2M1 codes and E4M3
scales of both operands in tcgen05.mma.kind::mxf4nvf4.block_scale with f32
accumulation; it is checked against the f64 sum of the pinned weights times
the pinned activations x_hat = e2m1 * e4m3 * G (the oracle's own dequant of
the quantized activations): |y - y_ref| <= 1e-5 * sum|w||x_hat| + 1e-6."""
import numpy as np
import pytest

import oracle
import synth

from _helpers import aux_for, oracle_gemv_all_rows, to_device, to_oracle, within_tolerance

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def quantize_x(xf, G, bf16):
    M, K = xf.shape
    if bf16:
        bits = synth.f32_to_bf16_bits(xf)
        xd = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        xf = (bits.astype(np.uint32) << 16).view(np.float32).reshape(M, K)
    else:
        xd = torch.from_numpy(np.ascontiguousarray(xf, np.float32)).cuda()
    xq = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    xs = torch.empty((M, K // 16), dtype=torch.uint8, device="cuda")
    q4.q4_quantize_nvfp4_scaled(xd, q4.Q4_DT_BF16 if bf16 else q4.Q4_DT_F32, G, xq, xs, M, K)
    torch.cuda.synchronize()
    return xq, xs, xf


@pytest.mark.parametrize("N,K,M,bf16", [(1024, 4096, 1, True), (333, 2304, 3, False), (4099, 4096, 16, True),
                                        (200, 11008, 17, False), (64, 256, 40, True), (14336, 4096, 8, True)])
def test_w4a4_tc_matches_the_pinned_product(N, K, M, bf16):
    layer = synth.make_layer("nvfp4", N, K, config=140, matrix=0, row_scale=True)
    _, xf = synth.draw_x(M, K, config=140, matrix=1, dtype="f32")
    G = float(np.float32(np.abs(xf).max()) / np.float32(2688.0))        # x's own NVFP4 tensor scale
    xq, xs, xw = quantize_x(xf, G, bf16)
    rp, rs = oracle.quantize_nvfp4_groups(xw, G)
    assert np.array_equal(xq.cpu().numpy(), rp) and np.array_equal(xs.cpu().numpy(), rs)
    xhat = oracle.dequant(oracle.Tensor("nvfp4", M, K, rp, rs, scale2=G))
    d = to_device(layer)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_gemv_w4a4_tc(d["w"], d["scales"], aux_for(layer, d), xq, xs, G, y, M, N, K)
    assert q4.q4_last_gemv_path() == "gemv_w4a4_tc"
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    ref, bound = oracle_gemv_all_rows(to_oracle(layer), xhat)
    ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
    assert ok, worst


def test_w4a4_tc_rejects_bad_arguments():
    layer = synth.make_layer("nvfp4", 16, 256, config=141, matrix=0)
    d = to_device(layer)
    xq = torch.zeros((1, 128), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((1, 16), dtype=torch.uint8, device="cuda")
    y = torch.empty((1, 16), device="cuda")
    aux = aux_for(layer, d)
    assert q4.q4_gemv_w4a4_tc(d["w"], d["scales"], aux, xq, xs, float("nan"), y, 1, 16, 256,
                              check=False) == q4.Q4_ESCALE2
    assert q4.q4_gemv_w4a4_tc(d["w"], d["scales"], aux, xq, xs, 1.0, y, 1, 16, 128, check=False) == q4.Q4_EDIM
    assert q4.q4_quantize_nvfp4_scaled(y, q4.Q4_DT_F32, 0.0, xq, xs, 1, 16, check=False) == q4.Q4_ESCALE2
