"""Pins for the oracle of the integer-exact A16-Q8 lane ([MUS7] 7.4.2: NVFP4
weights, activations quantized per 256-value block to signed 8-bit codes, an
exact integer block sum and a four-step f32 epilogue).

Each pin compares against something other than the oracle itself: the
printed E2M1 codebook, torch's float8 decoder, numpy's binary16 rounding,
quantizer cases worked by hand from the definition, and a constructed case in
which every step is exact, so the result must equal the binary16 rounding of
the (separately pinned) f64 GEMV.  No GPU needed.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def same_f32(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32),
                          np.asarray(b, np.float32).view(np.uint32))


def pack_nvfp4(codes):
    """codes u8 [N][K] (0..15) -> payload [N][K/2], even k in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


# ------------------------------------------------------------ integer codes

def test_q1_is_twice_the_printed_e2m1_codebook():
    with open(os.path.join(GOLD, "e2m1_codebook.json")) as f:
        g = json.load(f)
    for code, value in zip(g["codes"], g["values"]):
        assert oracle.e2m1_q1(code) == 2 * value, code      # -0.0 -> 0
    assert oracle.e2m1_q1(8) == 0 and oracle.e2m1_q1(7) == 12 and oracle.e2m1_q1(15) == -12


def test_q9_exhaustive_against_torch_float8():
    for b in range(256):
        if b in (0x7F, 0xFF):
            with pytest.raises(oracle.OracleError):
                oracle.e4m3fn_q9(b)
            continue
        ref = torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        assert oracle.e4m3fn_q9(b) * 2.0 ** -9 == ref, hex(b)
    assert oracle.e4m3fn_q9(0x7E) == 448 * 512 and oracle.e4m3fn_q9(0x01) == 1


# ------------------------------------------------------ activation quantizer

def test_q8_block_integer_values_are_kept():
    rng = np.random.default_rng(5)
    x = rng.integers(-126, 127, 256).astype(np.float32)
    x[17] = -127.0                      # the first (and only) maximum is negative
    q, s = oracle.q8_block(x)           # iscale = -127 / -127 = 1
    assert np.array_equal(q, x.astype(np.int8)) and s == 1.0
    x[17] = 127.0                       # positive maximum: iscale = -1, codes negate
    q, s = oracle.q8_block(x)
    assert np.array_equal(q, (-x).astype(np.int8)) and s == -1.0


def test_q8_block_first_maximum_decides_the_sign():
    x = np.zeros(256, np.float32)
    x[3], x[5], x[9] = 127.0, -127.0, 5.0
    q, s = oracle.q8_block(x)           # first of equal magnitudes is +127
    assert s == -1.0 and q[3] == -127 and q[5] == 127 and q[9] == -5
    x[3], x[5] = -127.0, 127.0
    q, s = oracle.q8_block(x)
    assert s == 1.0 and q[3] == -127 and q[5] == 127 and q[9] == 5


def test_q8_block_rounds_half_to_even():
    x = np.zeros(256, np.float32)
    x[0] = -127.0                       # iscale = 1: the codes are x rounded
    vals = [62.5, 63.5, -62.5, 0.5, 1.5, -0.5, 2.5, 126.5, 3.25, -3.75]
    want = [62, 64, -62, 0, 2, 0, 2, 126, 3, -4]
    x[1:1 + len(vals)] = vals
    q, s = oracle.q8_block(x)
    assert s == 1.0 and list(q[1:1 + len(vals)]) == want


def test_q8_block_worked_by_hand():
    # x = [0.5, -1, 2] (the activation of [W4K] section 7's W4A8 example,
    # here on the per-block grid): first max 2, iscale = -63.5 (exact),
    # codes -31.75 -> -32, 63.5 -> 64 (tie, even), -127; scale 1/-63.5.
    x = np.zeros(256, np.float32)
    x[:3] = [0.5, -1.0, 2.0]
    q, s = oracle.q8_block(x)
    assert list(q[:3]) == [-32, 64, -127] and not q[3:].any()
    assert abs(float(s) - (-2.0 / 127.0)) <= 2.0 ** -30      # f32 rounding of -2/127
    assert np.float32(s) * np.float32(-63.5) == 1.0


def test_q8_block_zero_block():
    q, s = oracle.q8_block(np.zeros(256, np.float32))
    assert not q.any() and s == 0.0
    x = np.zeros(256, np.float32)
    x[7] = -0.0
    q, s = oracle.q8_block(x)
    assert not q.any() and s == 0.0


def test_q8_block_power_of_two_invariance_and_bounds():
    rng = np.random.default_rng(11)
    for _ in range(20):
        x = rng.standard_normal(256).astype(np.float32)
        q, s = oracle.q8_block(x)
        i = int(np.argmax(np.abs(x)))               # numpy's argmax takes the first
        assert q[i] == -127
        assert np.abs(q.astype(np.int32)).max() == 127
        err = np.abs(q.astype(np.float64) * float(s) - x.astype(np.float64))
        assert np.all(err <= 0.5 * abs(float(s)) * (1 + 2.0 ** -20))
        for j in (-3, 2, 5):
            q2, s2 = oracle.q8_block(x * np.float32(2.0 ** j))
            assert np.array_equal(q, q2) and s2 == s * np.float32(2.0 ** j)


# ---------------------------------------------------------- binary16 output

def test_f16_round_against_numpy():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        (rng.standard_normal(4000) * np.exp2(rng.uniform(-30, 18, 4000))).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -26, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 6.1e-5,
                  np.inf, -np.inf], np.float32)])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).astype(np.float32)
    assert same_f32(oracle.f16_round(x), want)


# ------------------------------------------------------------ the contraction

def exact_case(seed, N=24, K=1024, M=3):
    """Inputs on which every step of the lane is exact: integer activations
    with each block's first maximum at +-127 (codes = +-x, scale = -+1), scale
    bytes 1..8 (q9 <= 8) and negative ones, scale2 = 1/8, |T| < 2^24."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sbytes = rng.integers(1, 9, (N, K // 16)).astype(np.uint8)
    sbytes[rng.random((N, K // 16)) < 0.25] |= 0x80                # negative scales
    x = rng.integers(-126, 127, (M, K)).astype(np.float32)
    for m in range(M):
        for b in range(K // 256):
            x[m, b * 256 + rng.integers(0, 256)] = 127.0 * rng.choice([-1.0, 1.0])
    x[M - 1, 256:512] = 0.0                                         # one all-zero block
    t = oracle.Tensor("nvfp4", N, K, pack_nvfp4(codes), sbytes, scale2=0.125)
    return t, x


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_a16q8_exact_case_equals_binary16_of_the_f64_gemv(seed):
    t, x = exact_case(seed)
    y64, _ = oracle.gemv(t, x)
    assert np.all(np.abs(y64) * 8 * 1024 < 2 ** 24)     # the sum is exact in f32 too
    want = y64.astype(np.float32).astype(np.float16).astype(np.float32)
    assert same_f32(oracle.gemv_a16q8(t, x), want)


def realistic_case(seed, N=40, K=2048, M=2):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sbytes = rng.integers(0x20, 0x48, (N, K // 16)).astype(np.uint8)   # ~2^-3 .. 2^1
    x = rng.standard_normal((M, K)).astype(np.float32)
    t = oracle.Tensor("nvfp4", N, K, pack_nvfp4(codes), sbytes, scale2=0.0037)
    return t, x


def test_a16q8_sign_and_power_of_two_invariance():
    t, x = realistic_case(7)
    y = oracle.gemv_a16q8(t, x)
    assert same_f32(oracle.gemv_a16q8(t, -x), -y)
    y4 = oracle.gemv_a16q8(t, x * np.float32(4.0))
    normal = (np.abs(y) >= 2.0 ** -14) & (np.abs(y) * 4 < 65504)
    assert normal.mean() > 0.9
    assert same_f32(y4[normal], 4 * y[normal])


def test_a16q8_within_the_activation_quantization_bound():
    t, x = realistic_case(8)
    y = oracle.gemv_a16q8(t, x).astype(np.float64)
    y64, _ = oracle.gemv(t, x)
    w = oracle.dequant(t).astype(np.float64)
    _, s = oracle.q8_quantize(x)
    step = np.repeat(np.abs(s.astype(np.float64)), 256, axis=1)          # [M][K]
    bound = 0.5 * (step * (1 + 2.0 ** -20)) @ np.abs(w).T                 # activation rounding
    bound += np.abs(y64) * 2.0 ** -11 + 1e-6 * (np.abs(x) @ np.abs(w).T)  # binary16 + f32 steps
    assert np.all(np.abs(y - y64) <= bound)


def test_a16q8_rejects_other_formats_and_nan_scales():
    t, x = realistic_case(9, N=4, K=256, M=1)
    bad = t.scales.copy()
    bad[2, 3] = 0x7F
    with pytest.raises(oracle.OracleError):
        oracle.gemv_a16q8(oracle.Tensor("nvfp4", 4, 256, t.w, bad, scale2=t.scale2), x)
    with pytest.raises(oracle.OracleError):
        oracle.gemv_a16q8(oracle.Tensor("nvfp4", 4, 128, t.w[:, :64], t.scales[:, :8], scale2=1.0),
                          x[:, :128])
