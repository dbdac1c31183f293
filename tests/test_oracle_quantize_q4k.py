"""Pins for the oracle's Q4_K fit (oracle.quantize_q4k, the write side of
Q4_K): the pages fix the decode, w = d*s_j*q - dmin*m_j, and the block layout
([FBTC] sections 5-6, [W4K] section 4), so the fit is pinned through the
oracle's independently pinned decoder and by closed forms:

  * a block built from codes, with every step exact, is found again byte for
    byte (fit(decode(B)) == B) -- this fixes the metadata packing, the code
    positions and the step order;
  * the zero block, all-positive sub-blocks (minimum 0) and saturation;
  * the reconstruction error bound of a min/max fit;
  * the binary16 encoder against all 65,536 patterns and numpy's cast.
No GPU needed."""
import numpy as np
import pytest

import oracle
import synth


def test_f16_bits_against_every_pattern_and_numpy():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = pats.view(np.float16).astype(np.float32)
    finite = np.isfinite(vals)
    got = np.array([oracle.f16_bits(float(v)) for v in vals[finite]], np.uint16)
    want = pats[finite].copy()
    want[want == 0x8000] = 0x8000                        # -0 keeps its sign
    assert np.array_equal(got, want)
    rng = np.random.default_rng(0)
    r = (rng.standard_normal(4000) * np.exp2(rng.integers(-30, 20, 4000))).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = r.astype(np.float16).view(np.uint16)
    assert np.array_equal(np.array([oracle.f16_bits(float(v)) for v in r], np.uint16), ref)


def built_block(rng, d_exp=-6, dmin_exp=-7):
    """A super-block whose fit is exact: fp16 powers of two d, dmin; every
    sub-block holds codes 0 and 15; max s_j = max m_j = 63 (so d and dmin are
    found again); all products and sums are exact in f32."""
    s = rng.integers(1, 64, 8)
    m = rng.integers(1, 64, 8)
    s[rng.integers(0, 8)] = 63
    m[rng.integers(0, 8)] = 63
    q = rng.integers(0, 16, (8, 32))
    q[:, 0], q[:, 1] = 0, 15
    rng.shuffle(q, axis=1)
    d, dmin = 2.0 ** d_exp, 2.0 ** dmin_exp
    w = (d * s[:, None] * q - dmin * m[:, None]).astype(np.float32)      # exact
    return w.reshape(256), s, m, q, d, dmin


def pack_by_hand(s, m, q, d, dmin):
    """The 144 bytes written from the layout rules directly (not the oracle)."""
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([np.float16(d)]).view(np.uint8)
    blk[2:4] = np.array([np.float16(dmin)]).view(np.uint8)
    for j in range(4):
        blk[4 + j] = s[j] | ((s[j + 4] >> 4) << 6)
        blk[8 + j] = m[j] | ((m[j + 4] >> 4) << 6)
        blk[12 + j] = (s[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    qq = q.reshape(256)
    for c in range(4):
        for lane in range(32):
            blk[16 + 32 * c + lane] = qq[64 * c + lane] | (qq[64 * c + 32 + lane] << 4)
    return blk


def test_fit_of_an_exact_block_returns_its_bytes():
    rng = np.random.default_rng(1)
    for trial in range(40):
        w, s, m, q, d, dmin = built_block(rng, d_exp=-6 - trial % 5, dmin_exp=-7 - trial % 3)
        want = pack_by_hand(s, m, q, d, dmin)
        # the pinned decoder reads the hand-packed block back to w
        t = oracle.Tensor("q4k", 1, 256, want.reshape(1, 1, 144))
        assert np.array_equal(oracle.dequant(t)[0], w)
        got = oracle.quantize_q4k(w.reshape(1, 256))
        assert np.array_equal(got.reshape(144), want), trial


def test_zero_block_and_all_positive_sub_blocks():
    assert not oracle.quantize_q4k(np.zeros((2, 512), np.float32)).any()
    rng = np.random.default_rng(2)
    w = rng.uniform(0.1, 1.0, (1, 256)).astype(np.float32)      # every sub-block positive: minimum 0
    blk = oracle.quantize_q4k(w)[0, 0]
    assert blk[2] == 0 and blk[3] == 0                           # dmin = 0
    t = oracle.Tensor("q4k", 1, 256, blk.reshape(1, 1, 144))
    assert np.all(oracle.dequant(t)[0] >= 0.0)


@pytest.mark.parametrize("kind", ["normal", "outliers", "positive"])
def test_reconstruction_error_bound(kind):
    """|w_hat - w| <= step/2 + 8 d + dmin (the rounding of the step, the code
    clamp and the rounding of the offset), step = d * s_j of the sub-block;
    also for all-positive weights, where the fit spans [0, max w]."""
    N, K = 64, 1024
    W = synth.draw_weights(N, K, config=95, matrix=0, outliers=kind == "outliers")
    if kind == "positive":
        W = np.abs(W) + np.float32(0.01)
    blocks = oracle.quantize_q4k(W)
    what = oracle.dequant(oracle.Tensor("q4k", N, K, blocks))
    for n in range(N):
        for b in range(K // 256):
            blk = blocks[n, b]
            d = float(np.array(blk[0:2]).view(np.float16)[0])
            dmin = float(np.array(blk[2:4]).view(np.float16)[0])
            B = blk[4:16].astype(int)
            for j in range(8):
                sj = (B[j] & 63) if j < 4 else (B[j + 4] & 15) | ((B[j - 4] >> 6) << 4)
                sl = slice(b * 256 + 32 * j, b * 256 + 32 * j + 32)
                err = np.abs(what[n, sl].astype(np.float64) - W[n, sl])
                assert np.all(err <= 0.5 * d * sj + 8 * d + dmin + 1e-7), (n, b, j, err.max(), d * sj)


def test_fit_agrees_with_the_write_side_generator_on_most_blocks():
    """Cross-check, not a pin: the synthetic generator fits in f64, the
    oracle in f32; the bytes agree except where an f32 rounding lands on the
    other side of a tie."""
    W = synth.draw_weights(32, 2048, config=96, matrix=0)
    a, b = oracle.quantize_q4k(W), synth.quantize_q4k(W)
    assert np.mean(a == b) > 0.999
