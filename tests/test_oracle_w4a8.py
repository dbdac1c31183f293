"""Pins for the oracle of the Q4_K x Q8 contraction ([W4K] section 7: Q4_K
weights as unsigned 4-bit codes, activations on the per-256 signed 8-bit
grid, exact integer sub-block sums, the scale / minimum-term / activation-
scale epilogue in f32).

Pinned against the page's worked W4A8 example (integer dot 3, code sum 3,
0.45 - 0.15 = 0.30), against the separately pinned f64 GEMV on inputs where
every step is exact, and by sign and power-of-two invariance.  No GPU needed.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def same_f32(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32),
                          np.asarray(b, np.float32).view(np.uint32))


def q4k_block(d, dmin, sc, mn, codes):
    """One 144-byte super-block from its fields: fp16 d, dmin; the 12 metadata
    bytes holding 6-bit sc[j], mn[j] (j < 4 in the low six bits of bytes j and
    j+4; j >= 4 split over bytes j+4 and the top bits of bytes j-4 and j);
    codes [256] with sub-block j = 32j .. 32j+31 at code byte 32(j//2) + l,
    low nibble for even j."""
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([np.float16(d)]).view(np.uint8)
    blk[2:4] = np.array([np.float16(dmin)]).view(np.uint8)
    for j in range(4):
        blk[4 + j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        blk[4 + j + 4] = mn[j] | ((mn[j + 4] >> 4) << 6)
        blk[4 + j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    codes = np.asarray(codes, np.uint8)
    for j in range(8):
        c, hi = divmod(j, 2)
        blk[16 + 32 * c:16 + 32 * c + 32] |= (codes[32 * j:32 * j + 32] << (4 * hi)).astype(np.uint8)
    return blk


def q4k_tensor(blocks, N, K):
    return oracle.Tensor("q4k", N, K, np.ascontiguousarray(np.asarray(blocks, np.uint8).reshape(N, -1)))


def test_block_packer_matches_the_pinned_dequant():
    rng = np.random.default_rng(1)
    sc, mn = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
    codes = rng.integers(0, 16, 256)
    row = oracle.dequant(q4k_tensor(q4k_block(0.5, 0.25, sc, mn, codes), 1, 256))[0]
    j = np.arange(256) // 32
    assert same_f32(row, (np.float32(0.5) * sc[j] * codes - np.float32(0.25) * mn[j]).astype(np.float32))


def test_worked_w4a8_example():
    with open(os.path.join(GOLD, "worked_examples.json")) as f:
        g = json.load(f)
    w, base = g["w4a8_q4k_dot"], g["q4k_subblock_dot"]
    assert base["d"] * base["s"] == pytest.approx(w["d_s"]) and base["dmin"] * base["m"] == pytest.approx(w["dmin_m"])
    sc, mn = [base["s"]] + [0] * 7, [base["m"]] + [0] * 7
    codes = np.zeros(256, np.int64)
    codes[:3] = w["q_w"]
    t = q4k_tensor(q4k_block(base["d"], base["dmin"], sc, mn, codes), 1, 256)
    # The page's activation scale s_x = 0.5 is the per-block grid of a block
    # whose first maximum is -127 * 0.5 (placed in sub-block 7, whose scale
    # and minimum are 0): then x = [0.5, -1, 2] quantizes to exactly q_x.
    x = np.zeros((1, 256), np.float32)
    x[0, :3] = w["x"]
    x[0, 255] = -127 * w["s_x"]
    q, s = oracle.q8_block(x[0])
    assert list(q[:3]) == w["q_x"] and s == w["s_x"]
    assert int(np.dot(w["q_w"], w["q_x"])) == w["int_dot"] and sum(w["q_x"]) == w["code_sum"]
    y = oracle.gemv_q4k_q8(t, x)[0, 0]
    assert abs(y - w["y"]) < 2e-3                                  # fp16 d and dmin
    assert w["terms"][0] - w["terms"][1] == pytest.approx(w["y"])
    # x is exactly on the grid, so the dequantize-then-multiply result agrees
    y64, _ = oracle.gemv(t, x)
    assert abs(y - y64[0, 0]) <= 1e-6


def exact_case(seed, K, smax, mmax, N=16, M=3):
    """Integer activations peaking at +-127 per block (codes = +-x), power-of-
    two d and dmin, scale / min ranges small enough that every integer and
    f32 step is exact; the result must equal the f64 GEMV, rounded to f32."""
    rng = np.random.default_rng(seed)
    blocks = []
    for _ in range(N):
        for _ in range(K // 256):
            blocks.append(q4k_block(2.0 ** -5, 2.0 ** -5, rng.integers(0, smax + 1, 8), rng.integers(0, mmax + 1, 8),
                                    rng.integers(0, 16, 256)))
    t = q4k_tensor(np.concatenate(blocks), N, K)
    x = rng.integers(-126, 127, (M, K)).astype(np.float32)
    for m in range(M):
        for b in range(K // 256):
            x[m, b * 256 + rng.integers(0, 256)] = 127.0 * rng.choice([-1.0, 1.0])
    return t, x


@pytest.mark.parametrize("seed,K,smax,mmax", [(0, 256, 15, 63), (1, 256, 15, 63), (2, 1024, 3, 15)])
def test_exact_case_equals_the_f64_gemv(seed, K, smax, mmax):
    t, x = exact_case(seed, K, smax, mmax)
    y64, _ = oracle.gemv(t, x)
    assert same_f32(oracle.gemv_q4k_q8(t, x), y64.astype(np.float32))


def realistic(seed, N=24, K=2048, M=2):
    layer = synth.make_layer("q4k", N, K, config=40, matrix=seed)
    x = np.random.default_rng(seed).standard_normal((M, K)).astype(np.float32)
    return oracle.Tensor("q4k", N, K, layer["w"]), x


def test_sign_and_power_of_two_invariance():
    t, x = realistic(3)
    y = oracle.gemv_q4k_q8(t, x)
    assert same_f32(oracle.gemv_q4k_q8(t, -x), -y)
    assert same_f32(oracle.gemv_q4k_q8(t, x * np.float32(8.0)), y * np.float32(8.0))


def test_within_the_activation_quantization_bound():
    t, x = realistic(4)
    y = oracle.gemv_q4k_q8(t, x).astype(np.float64)
    y64, bound = oracle.gemv(t, x)
    w = np.abs(oracle.dequant(t).astype(np.float64))
    _, s = oracle.q8_quantize(x)
    step = np.repeat(np.abs(s.astype(np.float64)), 256, axis=1)
    qbound = 0.5 * (step * (1 + 2.0 ** -20)) @ w.T
    assert np.all(np.abs(y - y64) <= qbound + 1e-4 * bound + 1e-6)


def test_rejects_other_formats():
    t, x = realistic(5, N=2, K=256, M=1)
    with pytest.raises(oracle.OracleError):
        oracle.gemv_q4k_q8(oracle.Tensor("nvfp4", 2, 256, np.zeros((2, 128), np.uint8),
                                         np.zeros((2, 16), np.uint8), scale2=1.0), x)
