"""GPU Q4_K fit vs the oracle's fit (oracle.quantize_q4k), byte for byte:
drawn weights (f32 and bf16, outliers, row scales, the 14336 x 4096 layer),
blocks built from codes that the fit must find again, zero and signed-zero
blocks, all-positive weights, and the decode of the result."""
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


def gpu_fit(W, bf16=False):
    N, K = W.shape
    if bf16:
        bits = synth.f32_to_bf16_bits(W)
        Wd = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        Wf = (bits.astype(np.uint32) << 16).view(np.float32)
    else:
        Wd, Wf = torch.from_numpy(np.ascontiguousarray(W, np.float32)).cuda(), np.asarray(W, np.float32)
    out = torch.full((N, K // 256, 144), 0xAB, dtype=torch.uint8, device="cuda")
    q4.q4_quantize_q4k(Wd, q4.Q4_DT_BF16 if bf16 else q4.Q4_DT_F32, out, N, K)
    torch.cuda.synchronize()
    return out.cpu().numpy(), Wf


@pytest.mark.parametrize("N,K,bf16,kw", [(14336, 4096, False, dict(row_scale=True)),
                                         (1000, 2560, True, dict(outliers=True)),
                                         (3, 256, False, dict())])
def test_q4k_fit_bit_exact(N, K, bf16, kw):
    W = synth.draw_weights(N, K, config=97, matrix=0, **kw)
    got, Wf = gpu_fit(W, bf16)
    assert np.array_equal(got, oracle.quantize_q4k(Wf))


def test_q4k_fit_special_blocks():
    rng = np.random.default_rng(3)
    W = np.zeros((6, 512), np.float32)
    W[1] = -0.0                                              # signed zeros: d = dmin = +0
    W[2] = np.abs(rng.standard_normal(512)).astype(np.float32) + 0.5       # all positive
    W[3] = -np.abs(rng.standard_normal(512)).astype(np.float32)            # all non-positive
    W[4, :256] = 1e-30                                       # tiny: binary16 subnormal or zero scales
    W[5] = rng.standard_normal(512).astype(np.float32) * 1e8              # large: d and dmin overflow to Inf
    got, Wf = gpu_fit(W)
    assert np.array_equal(got, oracle.quantize_q4k(Wf))
    assert not got[0].any() and not got[1].any()


def test_q4k_fit_round_trip_through_the_decoder():
    """GPU fit then GPU dequant: within the oracle fit's error bound of W."""
    N, K = 256, 1024
    W = synth.draw_weights(N, K, config=98, matrix=0)
    blocks, _ = gpu_fit(W)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    q4.q4_dequant("q4k", torch.from_numpy(blocks).cuda(), None, None, out, N, K)
    torch.cuda.synchronize()
    what = out.cpu().numpy()
    assert np.array_equal(what, oracle.dequant(oracle.Tensor("q4k", N, K, blocks)))
    assert np.max(np.abs(what - W)) < 0.01
