"""Pins for the oracle of the NVFP4 quantizer: E2M1 rounding with ModelOpt's
ties-to-even midpoints ([MUS7] 7.2), the worked rows of [FBTC] section 2,
E4M3FN nearest-even rounding against torch's float8 cast, and the
whole-tensor recipe by closed forms and a reconstruction bound.  No GPU.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_round_modelopt_midpoints():
    # each midpoint goes to the even code: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1,
    # 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    mids = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for m, want in mids.items():
        assert oracle.e2m1(oracle.e2m1_round(m)) == want, m
        assert oracle.e2m1(oracle.e2m1_round(-m)) == -want, m
        up, down = np.nextafter(np.float32(m), np.float32(10)), np.nextafter(np.float32(m), np.float32(0))
        grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
        i = max(k for k, g in enumerate(grid) if g < m)
        assert oracle.e2m1(oracle.e2m1_round(float(up))) == grid[i + 1]
        assert oracle.e2m1(oracle.e2m1_round(float(down))) == grid[i]
    for v in (6.0, 6.5, 7.0, 1e30):
        assert oracle.e2m1_round(v) == 7 and oracle.e2m1_round(-v) == 15
    assert oracle.e2m1_round(-0.1) == 8 and oracle.e2m1_round(0.0) == 0
    assert oracle.e2m1_round(-0.0) == 8          # the sign bit follows the value, zero included
    for c in range(16):                                  # every code is a fixed point
        assert oracle.e2m1_round(oracle.e2m1(c)) == c or (c == 8 and oracle.e2m1(c) == 0.0)


def test_e2m1_round_reproduces_the_printed_rows():
    with open(os.path.join(GOLD, "worked_examples.json")) as f:
        g = json.load(f)["e2m1_dot"]
    w = np.array(g["w"], np.float32)
    for case in g["cases"]:
        s = np.float32(case["scale"])
        got = [oracle.e2m1(oracle.e2m1_round(float(v / s))) * float(s) for v in w]
        assert got == case["w_hat"], case
        assert float(np.dot(np.float64(got), np.float64(g["x"]))) == case["y"]
    # [FBTC] section 2: 0.35 at scale 0.5 -> 0.25, at 0.125 -> 0.375; 1.7 at 0.125 clips to 0.75
    assert oracle.e2m1(oracle.e2m1_round(0.35 / 0.5)) * 0.5 == 0.25
    assert oracle.e2m1(oracle.e2m1_round(0.35 / 0.125)) * 0.125 == 0.375
    assert oracle.e2m1(oracle.e2m1_round(1.7 / 0.125)) * 0.125 == 0.75


def test_e4m3fn_round_against_torch_float8():
    rng = np.random.default_rng(2)
    v = np.concatenate([np.exp2(rng.uniform(-12, np.log2(448.0), 3000)),
                        rng.uniform(0, 2.0 ** -6, 500)]).astype(np.float32)
    v = np.concatenate([v, -v[:300]])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3fn_round(float(t)) for t in v], np.uint8)
    assert np.array_equal(got, ref)
    # every finite byte is a fixed point; ties to the even byte; saturation
    for b in range(0x7F):
        assert oracle.e4m3fn_round(oracle.e4m3fn(b)) == b
    assert oracle.e4m3fn_round(2.0 ** -10) == 0x00          # halfway 0 .. 2^-9
    assert oracle.e4m3fn_round(3 * 2.0 ** -10) == 0x02      # halfway 2^-9 .. 2^-8
    assert oracle.e4m3fn_round(1.0625) == 0x38              # halfway 1 .. 1.125
    for big in (448.0, 460.0, 464.0, 500.0, 1e9):
        assert oracle.e4m3fn_round(big) == 0x7E


def test_quantize_nvfp4_recipe_closed_forms():
    # a tensor whose amax is 2688 gives scale2 = 1; a group with amax 6 * 2^e
    # (e4m3-exact) gets that scale and its maximum element the code +-6
    W = np.zeros((2, 32), np.float32)
    W[0, 0] = 2688.0
    W[1, 16:32] = np.linspace(-24.0, 18.0, 16, dtype=np.float32)     # amax 24 -> scale 4
    p, s, s2 = oracle.quantize_nvfp4(W)
    assert s2 == 1.0
    assert s[0, 0] == 0x7E and (p[0, 0] & 15) == 7                   # 2688 / 448 = 6
    assert s[0, 1] == 0 and not p[0, 8:].any()                       # an all-zero group
    assert oracle.e4m3fn(int(s[1, 1])) == 4.0 and (p[1, 8] & 15) == 15   # -24 / 4 = -6
    p0, s0, s20 = oracle.quantize_nvfp4(np.zeros((3, 16), np.float32))
    assert s20 == 1.0 and not p0.any() and not s0.any()


def test_quantize_nvfp4_reconstruction_bound():
    W = synth.draw_weights(64, 256, config=50, matrix=0, outliers=True)
    p, s, s2 = oracle.quantize_nvfp4(W)
    t = oracle.Tensor("nvfp4", 64, 256, p, s, scale2=s2)
    w_hat = oracle.dequant(t).astype(np.float64)
    den = np.array([[oracle.e4m3fn(int(b)) for b in row] for row in s], np.float64) * float(s2)
    den = np.repeat(den, 16, axis=1)
    r = np.abs(W.astype(np.float64)) / den
    # half the E2M1 gap at |r| (0.25 below 2, 0.5 below 4, 1 above), times the denominator
    half_gap = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0)) * den
    assert np.all(np.abs(w_hat - W) <= half_gap * (1 + 1e-6) + 1e-30)
    assert float(s2) * 2688.0 == pytest.approx(float(np.abs(W).max()), rel=1e-6)


def test_quantize_nvfp4_agrees_with_the_input_generator():
    """The write-side generator implements the same recipe independently
    (vectorised numpy, closed-form rounding); the two agree bit for bit."""
    for cfg, (N, K) in enumerate([(16, 64), (33, 512), (8, 4096)]):
        W = synth.draw_weights(N, K, config=51 + cfg, matrix=0, outliers=True, row_scale=True)
        p, s, s2 = oracle.quantize_nvfp4(W)
        p2, s_2, s22 = synth.quantize_nvfp4(W)
        assert np.float32(s2) == np.float32(s22)
        assert np.array_equal(s, s_2) and np.array_equal(p, p2)
