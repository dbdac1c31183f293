"""GPU NVFP4 quantizer vs the oracle, bit for bit: payload, scale bytes and
scale2 on drawn weights (f32 and bf16, outliers, row scales), every E2M1
midpoint, saturation, zero groups and the all-zero tensor."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def gpu_quantize(W, bf16=False):
    N, K = W.shape
    if bf16:
        bits = synth.f32_to_bf16_bits(W)
        Wd = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        Wf = (bits.astype(np.uint32) << 16).view(np.float32)
    else:
        Wd, Wf = torch.from_numpy(np.ascontiguousarray(W, np.float32)).cuda(), W
    p = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
    s2 = torch.empty(4, dtype=torch.float32, device="cuda")
    q4.q4_quantize_nvfp4(Wd, q4.Q4_DT_BF16 if bf16 else q4.Q4_DT_F32, p, s, s2, N, K)
    torch.cuda.synchronize()
    return p.cpu().numpy(), s.cpu().numpy(), np.float32(s2[0].item()), Wf


@pytest.mark.parametrize("N,K,bf16", [(14336, 4096, False), (1000, 528, True), (7, 16, False)])
def test_quantize_bit_exact(N, K, bf16):
    W = synth.draw_weights(N, K, config=80, matrix=0, outliers=True, row_scale=True)
    p, s, s2, Wf = gpu_quantize(W, bf16)
    rp, rs, rs2 = oracle.quantize_nvfp4(Wf)
    assert np.float32(s2) == rs2 and np.array_equal(s, rs) and np.array_equal(p, rp)


def test_quantize_midpoints_saturation_and_zeros():
    # amax 2688 -> scale2 1; groups with amax 6 * 2^e get the exact scale 2^e, so
    # w / denom lands exactly on every E2M1 midpoint
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    W = np.zeros((4, 64), np.float32)
    W[0, 0] = 2688.0
    for e, row in ((0, 1), (-3, 2)):
        W[row, :8] = mids * 2.0 ** e
        W[row, 8:16] = -mids * 2.0 ** e
    W[3, 16], W[3, 17:32] = 6.0, -0.1                    # rounds to zero with the sign kept: code 8
    W[3, 32:48] = -1e-4                                  # scale rounds to 0: every code 0
    p, s, s2, _ = gpu_quantize(W)
    rp, rs, rs2 = oracle.quantize_nvfp4(W)
    assert s2 == rs2 == 1.0 and np.array_equal(s, rs) and np.array_equal(p, rp)
    pz, sz, s2z, _ = gpu_quantize(np.zeros((3, 32), np.float32))
    assert s2z == 1.0 and not pz.any() and not sz.any()
