"""The seeded workload encoders: deterministic, valid bytes, and the rounding
rules the pages fix for the write side.  No GPU needed."""
import numpy as np
import torch

import oracle
import synth


def test_e2m1_ties_to_even_midpoints():
    # ModelOpt's ties-to-even E2M1 rounding (Muser book, Chapter 7, section 7.2).
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.1, -0.25])
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -0.0, -0.0])
    got = [oracle.e2m1(int(c)) for c in synth.round_e2m1(mids)]
    assert np.array_equal(np.array(got), want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_e4m3_encoder_matches_torch_rounding():
    v = np.concatenate([np.random.default_rng(1).uniform(0, 448, 20000),
                        np.random.default_rng(2).uniform(0, 0.02, 5000),
                        [0.0, 2 ** -9, 2 ** -10, 3 * 2 ** -11, 448.0, 464.0 - 1e-3]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.round_e4m3fn(v), ref)
    assert synth.round_e4m3fn(np.array([1e6], np.float32))[0] == 0x7E


def test_encoders_deterministic_and_valid():
    W = synth.draw_weights(64, 512, config=0, matrix=0)
    assert np.array_equal(W, synth.draw_weights(64, 512, config=0, matrix=0))
    p, s, s2 = synth.quantize_nvfp4(W)
    assert p.shape == (64, 256) and s.shape == (64, 32) and s2 > 0
    assert not np.isin(s, [0x7F, 0xFF]).any()
    p2, s2b, _ = synth.quantize_nvfp4(W)
    assert np.array_equal(p, p2) and np.array_equal(s, s2b)
    _, e = synth.quantize_mxfp4(W)
    assert (e != 255).all()
    assert synth.quantize_q4k(W).shape == (64, 2, 144)
    assert synth.quantize_q40(W).shape == (64, 16, 18)
    codes, sb, z = synth.quantize_affine(W, 128)
    assert codes.max() <= 15 and z.min() >= 1 and z.max() <= 15


def test_quantizers_track_the_weights():
    """Coarse sanity on the write side: dequantized weights stay near W."""
    W = synth.draw_weights(32, 1024, config=0, matrix=3)
    p, s, s2 = synth.quantize_nvfp4(W)
    nv = oracle.dequant(oracle.Tensor("nvfp4", 32, 1024, p, s, scale2=s2))
    q4k = oracle.dequant(oracle.Tensor("q4k", 32, 1024, synth.quantize_q4k(W)))
    q40 = oracle.dequant(oracle.Tensor("q40", 32, 1024, synth.quantize_q40(W)))
    for Wh in (nv, q4k, q40):
        rel = np.linalg.norm(Wh - W) / np.linalg.norm(W)
        assert rel < 0.2, rel


def test_bf16_activation_rounding():
    bits, xf = synth.draw_x(2, 64, config=0, matrix=0)
    assert bits.dtype == np.uint16
    ref = torch.from_numpy(np.random.default_rng(synth.seed_for(0, 0, "x")).normal(0, 1, (2, 64))
                           .astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(xf, ref)
