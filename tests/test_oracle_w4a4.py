"""Pins for the oracle of the W4A4 contraction ([MUS7] 7.4.3): activations
quantized to NVFP4 per 16 with tensor scale 1/input_scale_inv, the exact
per-group integer product of the four encodings (denominator 2^-20), the f32
epilogue and the binary16 output.

Pinned by: idempotence of the activation quantizer on inputs that are already
NVFP4 (every step of the pinned rounding rules lands back on the same codes);
an all-exact case that must equal the binary16 rounding of the f64 GEMV;
sign and power-of-two invariance; the activation-quantization error bound.
No GPU needed.
"""
import numpy as np
import pytest

import oracle


def same_f32(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


def pack(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def nvfp4_exact_rows(rng, M, K, G, smax_byte):
    """Rows that are exactly NVFP4 with tensor scale G: every group holds a
    +-6 code, so the quantizer's group scale is recovered exactly."""
    codes = rng.integers(0, 16, (M, K)).astype(np.uint8)
    codes[:, ::16] = rng.choice([7, 15], size=(M, K // 16))          # +-6 in each group
    sb = rng.integers(1, smax_byte + 1, (M, K // 16)).astype(np.uint8)
    t = oracle.Tensor("nvfp4", M, K, pack(codes), sb, scale2=G)
    return oracle.dequant(t), pack(codes), sb


def test_activation_quantizer_is_idempotent_on_nvfp4_inputs():
    rng = np.random.default_rng(1)
    for G in (0.125, 1.0, 3.0):
        x, p, sb = nvfp4_exact_rows(rng, 5, 512, np.float32(G), 0x77)
        p2, sb2 = oracle.quantize_nvfp4_groups(x, G)
        assert np.array_equal(sb2, sb) and np.array_equal(p2, p)


def exact_case(seed, N=12, K=256, M=3):
    rng = np.random.default_rng(seed)
    wcodes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    wsb = rng.integers(1, 9, (N, K // 16)).astype(np.uint8)          # q9 <= 8
    wsb[rng.random(wsb.shape) < 0.25] |= 0x80                        # negative weight scales
    t = oracle.Tensor("nvfp4", N, K, pack(wcodes), wsb, scale2=0.25)
    G = np.float32(0.125)                                            # input_scale_inv = 8
    x, _, _ = nvfp4_exact_rows(rng, M, K, G, 8)
    return t, x, 8.0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_exact_case_equals_binary16_of_the_f64_gemv(seed):
    t, x, isi = exact_case(seed)
    y64, _ = oracle.gemv(t, x)              # x is already NVFP4: its quantization is exact
    want = y64.astype(np.float32).astype(np.float16).astype(np.float32)
    assert same_f32(oracle.gemv_w4a4(t, x, isi), want)


def realistic(seed, N=20, K=1024, M=2):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sb = rng.integers(0x20, 0x48, (N, K // 16)).astype(np.uint8)
    t = oracle.Tensor("nvfp4", N, K, pack(codes), sb, scale2=0.0037)
    x = rng.standard_normal((M, K)).astype(np.float32)
    isi = float(np.float32(2688.0 / np.abs(x).max()))                # the weight recipe's tensor scale, inverted
    return t, x, isi


def test_sign_and_power_of_two_invariance():
    t, x, isi = realistic(3)
    y = oracle.gemv_w4a4(t, x, isi)
    assert same_f32(oracle.gemv_w4a4(t, -x, isi), -y)
    y2 = oracle.gemv_w4a4(t, x * np.float32(2.0), isi / 2)
    normal = (np.abs(y) >= 2.0 ** -14) & (np.abs(y) * 2 < 65504)
    assert same_f32(y2[normal], 2 * y[normal])


def test_within_the_activation_quantization_bound():
    t, x, isi = realistic(4)
    G = np.float32(1.0) / np.float32(isi)
    p, sb = oracle.quantize_nvfp4_groups(x, G)
    x_hat = oracle.dequant(oracle.Tensor("nvfp4", x.shape[0], x.shape[1], p, sb, scale2=G)).astype(np.float64)
    w = oracle.dequant(t).astype(np.float64)
    y = oracle.gemv_w4a4(t, x, isi).astype(np.float64)
    y_q = x_hat @ w.T                                            # exact product of the quantized operands
    assert np.all(np.abs(y - y_q) <= np.abs(y_q) * 2.0 ** -11 + 1e-6 * (np.abs(x_hat) @ np.abs(w).T) + 1e-30)
    y64, _ = oracle.gemv(t, x)
    assert np.all(np.abs(y_q - y64) <= np.abs(x_hat - x) @ np.abs(w).T * (1 + 1e-9))


def test_rejects_bad_scale_and_format():
    t, x, _ = realistic(5, N=2, K=64, M=1)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(oracle.OracleError):
            oracle.gemv_w4a4(t, x, bad)
    with pytest.raises(oracle.OracleError):
        oracle.gemv_w4a4(oracle.Tensor("mxfp4", 2, 64, t.w, t.scales[:, :2]), x, 1.0)
