"""b-bit code streams and the act-order activation permutation on the GPU,
through the C ABI, byte-exact against the oracle's bit packer
(oracle.packing.pack_bits / unpack_bits): every width 1..8 on the page's
probes (patterned, random rng(0), all ones), the 3-bit codes that straddle
words at indices 10 and 21 ([BPA] "Odd widths: 3-bit, 2-bit and 6-bit"),
and the permutation a real act-order GPTQ -> AWQ repack returns."""
import numpy as np
import pytest

import oracle
from oracle import packing
import synth

from _helpers import aux_for, to_device, to_oracle, x_device

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def probes(n, bits):
    mask = (1 << bits) - 1
    return [((np.arange(n) * 7 + 3) % (mask + 1)).astype(np.uint8),
            np.random.default_rng(0).integers(0, mask + 1, n).astype(np.uint8),
            np.full(n, mask, np.uint8)]


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_pack_and_unpack_match_the_oracle(bits):
    n = 32 * 8 * 37                      # several blocks of the grid, a multiple of 32 bits
    for codes in probes(n, bits):
        ref = packing.pack_bits(codes, bits)
        cd = torch.from_numpy(codes).cuda()
        words = torch.zeros(n * bits // 32, dtype=torch.int32, device="cuda")
        q4.q4_pack_bits(cd, n, bits, words)
        back = torch.full((n,), 0xAA, dtype=torch.uint8, device="cuda")
        q4.q4_unpack_bits(words, n, bits, back)
        torch.cuda.synchronize()
        assert np.array_equal(words.cpu().numpy().view(np.uint32), ref)
        assert np.array_equal(back.cpu().numpy(), codes)


def test_three_bit_straddles_at_10_and_21():
    """Code 10 covers stream bits 30..32 and code 21 bits 63..65: each is cut
    by a word boundary.  Only those codes are set, to 7 and 5."""
    codes = np.zeros(32, np.uint8)
    codes[10], codes[21] = 7, 5
    cd = torch.from_numpy(codes).cuda()
    words = torch.zeros(3, dtype=torch.int32, device="cuda")
    q4.q4_pack_bits(cd, 32, 3, words)
    torch.cuda.synchronize()
    w = words.cpu().numpy().view(np.uint32)
    assert w.tolist() == [3 << 30, (1 << 0) | (1 << 31), 2]          # 7 = 0b111 split 2+1, 5 = 0b101 split 1+2
    assert np.array_equal(w, packing.pack_bits(codes, 3))


def test_pack_rejects_ragged_streams():
    cd = torch.zeros(64, dtype=torch.uint8, device="cuda")
    words = torch.zeros(8, dtype=torch.int32, device="cuda")
    assert q4.q4_pack_bits(cd, 33, 3, words, check=False) == q4.Q4_EDIM
    assert q4.q4_pack_bits(cd, 32, 9, words, check=False) == q4.Q4_EDIM


@pytest.mark.parametrize("xdtype", ["bf16", "f32"])
def test_permute_k_applies_the_act_order_permutation(xdtype):
    """GPTQ with act-order g_idx -> AWQ through q4_repack, which returns the
    source row of every target row; permuting x by it leaves the product
    unchanged: q4_gemv(AWQ target, x[perm]) == q4_gemv(GPTQ source, x)
    within the GEMV tolerance, and the permuted x equals numpy's gather."""
    N, K, M = 256, 1024, 3
    layer = synth.make_layer("gptq", N, K, config=90, matrix=0, act_order=True)
    d = to_device(layer)
    w = torch.empty((K, N // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((K // 128, N), dtype=torch.int16, device="cuda")
    z = torch.empty((K // 128, N // 8), dtype=torch.int32, device="cuda")
    perm = torch.empty(K, dtype=torch.int32, device="cuda")
    q4.q4_repack("gptq", d["w"], d["scales"], aux_for(layer, d), "awq", w, sc, z, perm, N, K)
    xb, xf = synth.draw_x(M, K, config=90, matrix=1, dtype=xdtype)
    x = x_device(xb)
    xp = torch.empty_like(x)
    q4.q4_permute_k(x, q4.Q4_DT_BF16 if xdtype == "bf16" else q4.Q4_DT_F32, perm, xp, M, K)
    torch.cuda.synchronize()
    p = perm.cpu().numpy()
    assert sorted(p.tolist()) == list(range(K)) and not np.array_equal(p, np.arange(K))
    assert torch.equal(xp.cpu(), x.cpu()[:, torch.from_numpy(p.astype(np.int64))])
    assert q4.q4_last_error() == q4.Q4_OK
    y_src = torch.empty((M, N), device="cuda")
    y_dst = torch.empty((M, N), device="cuda")
    q4.q4_gemv("gptq", d["w"], d["scales"], aux_for(layer, d, x_dtype=x.dtype), x, y_src, M, N, K)
    q4.q4_gemv("awq", w, sc, q4.make_aux(zeros=z, group=128, x_dtype=x.dtype, fmt="awq"), xp, y_dst, M, N, K)
    torch.cuda.synchronize()
    _, bound = oracle.gemv(to_oracle(layer), xf)               # sum |w||x|, the same for both orders
    assert np.all(np.abs(y_src.cpu().numpy() - y_dst.cpu().numpy()) <= 2 * oracle.gemv_tolerance(bound))


def test_permute_k_reports_an_index_out_of_range():
    K = 64
    x = torch.arange(2 * K, dtype=torch.float32, device="cuda").view(2, K)
    perm = torch.arange(K, dtype=torch.int32, device="cuda").flip(0).contiguous()
    perm[5] = K                                               # out of range: not read
    out = torch.full_like(x, -1.0)
    q4.q4_permute_k(x, q4.Q4_DT_F32, perm, out, 2, K)
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_ERANGE
    assert q4.q4_last_error() == q4.Q4_OK                    # reading clears it
    want = x.cpu()[:, torch.arange(K).flip(0)]
    want[:, 5] = 0.0
    assert torch.equal(out.cpu(), want)
