"""Pins for the CPU oracle: it is checked against what the source pages and the
mathematics fix -- printed worked examples (tests/golden/, each cited),
library decoders for the same bit formats, closed forms, brute force and
invariants -- never against itself.  No GPU needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import packing

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def same_f32(a, b):
    """Bitwise f32 equality (distinguishes -0.0 from 0.0)."""
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32),
                          np.asarray(b, np.float32).view(np.uint32))


# ------------------------------------------------------------------ E2M1

def test_e2m1_codebook_matches_printed_table():
    g = gold("e2m1_codebook.json")
    got = [oracle.e2m1(c) for c in g["codes"]]
    assert same_f32(got, g["values"])
    assert oracle.e2m1(0b0101) == 3.0
    assert oracle.e2m1(7) == 6.0
    assert math.copysign(1.0, oracle.e2m1(8)) == -1.0 and oracle.e2m1(8) == 0.0


# --------------------------------------------------------------- E4M3FN

def test_e4m3fn_exhaustive_against_torch_float8():
    finite = 0
    for b in range(256):
        if b in (0x7F, 0xFF):
            with pytest.raises(oracle.OracleError):
                oracle.e4m3fn(b)
            continue
        ref = torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        assert same_f32([oracle.e4m3fn(b)], [ref]), hex(b)
        finite += 1
    assert finite == 254


def test_e4m3fn_printed_values():
    g = gold("worked_examples.json")["e4m3"]
    assert oracle.e4m3fn(0x38) == g["byte_0x38"]
    assert oracle.e4m3fn(g["exp5_frac2_byte"]) == g["exp5_frac2_value"]
    assert (g["exp5_frac2_byte"] >> 3) & 15 == 5 and g["exp5_frac2_byte"] & 7 == 2
    assert oracle.e2m1(0b0101) * oracle.e4m3fn(g["exp5_frac2_byte"]) * 1.0 == g["times3"]
    assert oracle.e4m3fn(g["max_byte"]) == g["max"]
    assert max(oracle.e4m3fn(b) for b in range(128) if b != 0x7F) == 448.0
    for b in g["nan_bytes"]:
        with pytest.raises(oracle.OracleError):
            oracle.e4m3fn(b)


# ----------------------------------------------------------------- E8M0

def test_e8m0_exhaustive_against_torch_e8m0():
    for b in range(255):
        ref = torch.tensor([b], dtype=torch.uint8).view(torch.float8_e8m0fnu).float().item()
        assert same_f32([oracle.e8m0(b)], [ref]), b
    with pytest.raises(oracle.OracleError):
        oracle.e8m0(255)


def test_e8m0_printed_values():
    g = gold("worked_examples.json")["e8m0"]
    assert oracle.e8m0(g["byte"]) == g["value"]
    assert g["code_value"] * oracle.e8m0(g["byte"]) == g["w_hat"]


# ------------------------------------------------------------ fp16, bf16

def test_half_exhaustive_against_numpy_float16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert same_f32(got[~nan], ref[~nan])


def test_bf16_widen_and_round_against_torch():
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.normal(0, 1, 5000), rng.normal(0, 1e-30, 100),
                           rng.normal(0, 1e30, 100), [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                                                      3.4e38, 1e-45]]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(vals), ref)
    for b in ref[:200]:
        assert same_f32([oracle.bf16(int(b))],
                        [torch.tensor([int(b)], dtype=torch.int32).to(torch.int16)
                         .view(torch.bfloat16).float().item()])


# --------------------------------------------------------- NVFP4 fixture

def test_nvfp4_fixture_row_bit_for_bit():
    g = gold("nvfp4_fixture_row.json")
    payload = np.frombuffer(bytes.fromhex(g["payload_hex"]), dtype=np.uint8).reshape(1, 8)
    t = oracle.Tensor("nvfp4", 1, 16, payload, np.array([[g["scale_byte"]]], np.uint8),
                      scale2=g["scale2"])
    row = oracle.dequant(t)[0]
    assert same_f32(row[:10], g["printed"])
    assert same_f32(row[10:], g["extension"])


def test_splithalf_group_bytes_pinned_by_hand():
    """One 16-group whose lanes all carry distinct codes, written out byte by
    byte from the split-half sentence: the split-half decoder must put low
    nibbles in lanes 0-7 and high nibbles in lanes 8-15, and the plain NVFP4
    decoder must read the same bytes as adjacent pairs."""
    g = gold("lane_orders.json")["nvfp4_splithalf_group"]
    payload = np.frombuffer(bytes.fromhex(g["bytes_hex"]), dtype=np.uint8).reshape(1, 8)
    scales = np.array([[g["scale_byte"]]], np.uint8)
    half = oracle.dequant(oracle.Tensor("nvfp4_splithalf", 1, 16, payload, scales, scale2=g["scale2"]))[0]
    assert same_f32(half, g["splithalf_w_hat"])
    pair = oracle.dequant(oracle.Tensor("nvfp4", 1, 16, payload, scales, scale2=g["scale2"]))[0]
    assert same_f32(pair, g["adjacent_pair_w_hat"])
    # the packer's split-half route reproduces the hand-written bytes
    hw, _, _, _ = packing.repack("nvfp4", "nvfp4_splithalf", 1, 16,
                                 packing.pack_nvfp4_codes(np.arange(16, dtype=np.uint8).reshape(1, 16)), scales)
    assert bytes(np.asarray(hw, np.uint8).ravel()) == bytes.fromhex(g["bytes_hex"])


def test_q40_block_bytes_pinned_by_hand():
    """A Q4_0 block whose low and high nibbles differ in every byte, written
    out from the page's byte rule: element j is the low nibble of byte j and
    element j + 16 its high nibble."""
    g = gold("lane_orders.json")["q4_0_block"]
    blk = np.frombuffer(bytes.fromhex(g["block_hex"]), dtype=np.uint8).reshape(1, 18)
    assert same_f32(oracle.dequant(oracle.Tensor("q40", 1, 32, blk))[0], g["w_hat"])
    # the packer writes the same bytes from the codes and d
    codes = np.array([[j for j in range(16)] + [15 - j for j in range(16)]], np.uint8)
    packed = packing.pack_q40(codes, np.array([[0x3800]], np.uint16))
    assert bytes(np.asarray(packed, np.uint8).ravel()) == bytes.fromhex(g["block_hex"])
    # one-hot x picks single elements: x = e_j gives w_hat[j] exactly
    for j in (0, 1, 15, 16, 17, 31):
        x = np.zeros((1, 32), np.float32)
        x[0, j] = 1.0
        assert oracle.gemv(oracle.Tensor("q40", 1, 32, blk), x)[0][0, 0] == g["w_hat"][j]


def test_fp4_small_examples():
    g = gold("worked_examples.json")["fp4_small"]
    inv = {oracle.e2m1(c): c for c in range(8)}
    inv.update({-oracle.e2m1(c): c | 8 for c in range(1, 8)})

    def payload(values, K):
        codes = np.zeros((1, K), np.uint8)
        codes[0, :len(values)] = [inv[v] for v in values]
        return packing.pack_nvfp4_codes(codes)

    nv = g["nvfp4"]
    t = oracle.Tensor("nvfp4", 1, 16, payload(nv["codes_values"], 16),
                      np.array([[nv["e4m3_byte"]]], np.uint8), scale2=nv["scale2"])
    assert same_f32(oracle.dequant(t)[0, :4], nv["w_hat"])
    mx = g["mxfp4"]
    t = oracle.Tensor("mxfp4", 1, 32, payload(mx["codes_values"], 32),
                      np.array([[mx["e8m0_byte"]]], np.uint8))
    assert same_f32(oracle.dequant(t)[0, :4], mx["w_hat"])


# ------------------------------------------------- worked dot products

def _e2m1_code(v):
    for c in range(16):
        if oracle.e2m1(c) == v and not (v == 0 and c == 8):
            return c
    raise KeyError(v)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_e2m1_worked_dot_products(fmt):
    g = gold("worked_examples.json")["e2m1_dot"]
    x = np.zeros((1, 32), np.float32)
    x[0, :4] = g["x"]
    assert sum(a * b for a, b in zip(g["w"], g["x"])) == pytest.approx(g["y_exact"])
    for case in g["cases"]:
        codes = np.zeros((1, 32), np.uint8)
        codes[0, :4] = [_e2m1_code(v / case["scale"]) for v in case["w_hat"]]
        pay = packing.pack_nvfp4_codes(codes)
        if fmt == "mxfp4":
            t = oracle.Tensor("mxfp4", 1, 32, pay, np.array([[case["e8m0"]]], np.uint8))
        else:
            e4 = {0.5: 0x30, 0.125: 0x20}[case["scale"]]
            t = oracle.Tensor("nvfp4", 1, 32, pay, np.array([[e4, e4]], np.uint8), scale2=1.0)
        assert same_f32(oracle.dequant(t)[0, :4], case["w_hat"])
        y, _ = oracle.gemv(t, x)
        assert y[0, 0] == case["y"]


def test_int4_toy_bytes_and_dot():
    g = gold("worked_examples.json")["int4_toy"]
    q = g["q"]
    assert q == [max(-8, min(7, round(w / g["scale"]))) for w in g["w"]]
    twos = [v & 15 for v in q]
    words = packing.pack_bits(twos + [0] * 4, 4)           # pad to one 32-bit word
    assert words.view(np.uint8)[:2].tobytes() == bytes.fromhex(g["bytes_hex"])
    assert list(packing.unpack_bits(words, 4, 4)) == twos
    # The same block as offset-binary codes (q + 8, zero 8) through GPTQ, AWQ and Q4_0.
    N, K = 8, 32
    codes = np.full((K, N), 8, np.uint8)
    codes[:4, 0] = [v + 8 for v in q]
    sbits = np.full((1, N), np.float16(g["scale"]).view(np.uint16), np.uint16)
    zeros = np.full((1, N), 8, np.uint8)
    x = np.zeros((1, K), np.float32)
    x[0, :4] = g["x"]
    for fmt in ("gptq", "awq"):
        w, s, z = packing.from_logical(fmt, codes, sbits, zeros)
        t = oracle.Tensor(fmt, N, K, w, s, z, group=32)
        assert same_f32(oracle.dequant(t, rows=[0])[0, :4], g["w_hat"])
        y, _ = oracle.gemv(t, x, rows=[0])
        assert y[0, 0] == g["y_hat"]
    blk = packing.pack_q40(codes.T.copy(), np.full((N, 1), np.float16(g["scale"]).view(np.uint16)))
    t = oracle.Tensor("q40", N, K, blk)
    assert same_f32(oracle.dequant(t, rows=[0])[0, :4], g["w_hat"])
    assert oracle.gemv(t, x, rows=[0])[0][0, 0] == g["y_hat"]


# ---------------------------------------------------------------- Q4_K

def _q4k_block(d, dmin, B, qs):
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([np.float16(d)]).view(np.uint8)
    blk[2:4] = np.array([np.float16(dmin)]).view(np.uint8)
    blk[4:16] = B
    blk[16:] = qs
    return blk


def _fixture_B():
    g = gold("worked_examples.json")["q4k_lanes"]
    B = np.zeros(12, np.uint8)
    (s0, m0), (s1, m1) = g["pairs"]
    B[0], B[1], B[4], B[5] = g["B0"], s1, m0, m1
    B[8] = g["B8"]
    assert B[0] & 63 == s0
    return B


def test_q4k_lanes_0_and_32():
    g = gold("worked_examples.json")["q4k_lanes"]
    qs = np.zeros(128, np.uint8)
    qs[0] = g["byte"]
    t = oracle.Tensor("q4k", 1, 256, _q4k_block(g["d"], g["dmin"], _fixture_B(), qs))
    row = oracle.dequant(t)[0]
    assert row[0] == g["lane0"] and row[32] == g["lane32"]
    assert row[1] == g["byte00_lane0"] and row[33] == g["byte00_lane32"]


def test_q4k_split_metadata_s4():
    g = gold("worked_examples.json")["q4k_lanes"]
    qs = np.zeros(128, np.uint8)
    qs[64] = 1                                           # sub-block 4: chunk 2, low nibble
    t = oracle.Tensor("q4k", 1, 256, _q4k_block(g["d"], g["dmin"], _fixture_B(), qs))
    row = oracle.dequant(t)[0]
    m4 = g["B8"] >> 4                                    # B[4]'s top bits are zero here
    assert row[128] == np.float32(g["d"] * g["s4"] * 1 - g["dmin"] * m4)
    assert row[129] == np.float32(-g["dmin"] * m4)


def test_q4k_all_256_destinations():
    """One nibble at a time: the lane that moves must be the printed map
    (payload 32c+l -> low 64c+l of sub-block 2c, high 64c+32+l of 2c+1), and
    its value must use that sub-block's own (distinct) scale and min."""
    sc = [5, 9, 13, 17, 33, 45, 50, 63]
    mn = [1, 2, 3, 4, 21, 37, 40, 59]
    B = np.zeros(12, np.uint8)
    for j in range(4):
        B[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        B[j + 4] = mn[j] | ((mn[j + 4] >> 4) << 6)
        B[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    d, dmin = 0.5, 0.25
    base = oracle.dequant(oracle.Tensor("q4k", 1, 256, _q4k_block(d, dmin, B, np.zeros(128, np.uint8))))[0]
    for j in range(8):
        assert np.all(base[32 * j:32 * j + 32] == np.float32(-dmin * mn[j]))
    seen = set()
    for p in range(128):
        for hi in (0, 1):
            qs = np.zeros(128, np.uint8)
            qs[p] = 15 << (4 * hi)
            row = oracle.dequant(oracle.Tensor("q4k", 1, 256, _q4k_block(d, dmin, B, qs)))[0]
            moved = np.nonzero(row != base)[0]
            c, l = divmod(p, 32)
            lane = 64 * c + 32 * hi + l
            j = 2 * c + hi
            assert list(moved) == [lane]
            assert row[lane] == np.float32(d * sc[j] * 15 - dmin * mn[j])
            seen.add(lane)
    assert seen == set(range(256))


def test_q4k_worked_subblock_dot():
    g = gold("worked_examples.json")["q4k_subblock_dot"]
    B = np.zeros(12, np.uint8)
    B[0], B[4] = g["s"], g["m"]
    qs = np.zeros(128, np.uint8)
    qs[:3] = g["q"]
    t = oracle.Tensor("q4k", 1, 256, _q4k_block(g["d"], g["dmin"], B, qs))
    row = oracle.dequant(t)[0]
    assert np.allclose(row[:3], g["w_hat"], atol=2e-3)
    x = np.zeros((1, 256), np.float32)
    x[0, :3] = g["x"]
    y, _ = oracle.gemv(t, x)
    assert abs(y[0, 0] - g["y"]) < 2e-3


# ------------------------------------------------------------ packers

def _probes(K, N):
    patterned = ((np.arange(K)[:, None] * 7 + np.arange(N)[None, :] * 3) % 16).astype(np.uint8)
    rand = np.random.default_rng(0).integers(0, 16, size=(K, N), dtype=np.uint8)
    return [patterned, rand, np.full((K, N), 15, np.uint8)]


def test_layout_probes_gptq_awq_q40():
    for probe in _probes(256, 256):
        qw = packing.pack_gptq_qweight(probe)
        assert qw.dtype == np.int32 and qw.shape == (32, 256)
        assert np.array_equal(packing.unpack_gptq_qweight(qw), probe)
        aw = packing.pack_awq_words(probe)
        assert aw.shape == (256, 32)
        assert np.array_equal(packing.unpack_awq_words(aw), probe)
        d = np.full((256, 8), 0x3C00, np.uint16)
        blocks = packing.pack_q40(probe.T.copy(), d)
        codes, _, _ = packing.q40_to_logical(blocks, 256, 256)
        assert np.array_equal(codes, probe)
    allf = packing.pack_gptq_qweight(np.full((8, 8), 15, np.uint8))
    assert np.all(allf == -1)                                   # top slot is the sign bit


def test_gptq_and_awq_slot_positions_printed():
    # GPTQ: logical row 8r+j sits at bits 4j of word r.
    for j in range(8):
        q = np.zeros((8, 8), np.uint8)
        q[j, 0] = 1
        assert packing.pack_gptq_qweight(q).view(np.uint32)[0, 0] == 1 << (4 * j)
    # AWQ: the reader's shifts for columns 0..7 are 0,16,4,20,8,24,12,28.
    printed_shift = [0, 16, 4, 20, 8, 24, 12, 28]
    for col in range(8):
        q = np.zeros((1, 8), np.uint8)
        q[0, col] = 1
        assert packing.pack_awq_words(q).view(np.uint32)[0, 0] == 1 << printed_shift[col]


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_pack_bits_round_trips(bits):
    rng = np.random.default_rng(0)
    n = 32 * 8
    for v in (rng.integers(0, 1 << bits, n), np.full(n, (1 << bits) - 1),
              (np.arange(n) * 7 + 3) % (1 << bits)):
        words = packing.pack_bits(v, bits)
        assert words.size == n * bits // 32
        assert np.array_equal(packing.unpack_bits(words, bits, n), v.astype(np.uint8))


def test_pack_bits_three_bit_straddles():
    # [BPA]: index 10 spans bits 30..32 (words 0 and 1); index 21 spans words 1 and 2.
    q = np.zeros(32, np.int64)
    q[10] = 0b111
    w = packing.pack_bits(q, 3)
    assert w[0] == 0xC0000000 and w[1] == 0x1 and w[2] == 0
    q = np.zeros(32, np.int64)
    q[21] = 0b111
    w = packing.pack_bits(q, 3)
    assert w[0] == 0 and w[1] == 0x80000000 and w[2] == 0x3


def test_gptq_zero_is_stored_minus_one():
    N, K = 8, 128
    codes = np.full((K, N), 9, np.uint8)
    sbits = np.full((1, N), np.float16(1.0).view(np.uint16), np.uint16)
    zeros = np.full((1, N), 8, np.uint8)
    w, s, z = packing.from_logical("gptq", codes, sbits, zeros)
    assert np.all(z.view(np.uint32) == 0x77777777)             # 8 stored as 7
    assert np.all(oracle.dequant(oracle.Tensor("gptq", N, K, w, s, z)) == 1.0)


# ------------------------------------------------- GEMV closed forms

def _random_tensor(fmt, N, K, seed):
    import synth
    W = synth.draw_weights(N, K, config=9, matrix=seed)
    if fmt == "nvfp4":
        p, s, s2 = synth.quantize_nvfp4(W)
        return oracle.Tensor(fmt, N, K, p, s, scale2=s2)
    if fmt == "mxfp4":
        p, s = synth.quantize_mxfp4(W)
        return oracle.Tensor(fmt, N, K, p, s)
    if fmt == "q4k":
        return oracle.Tensor(fmt, N, K, synth.quantize_q4k(W))
    if fmt == "q40":
        return oracle.Tensor(fmt, N, K, synth.quantize_q40(W))
    codes, sb, z = synth.quantize_affine(W, 128)
    w, s, zz = (synth.pack_gptq if fmt == "gptq" else synth.pack_awq)(codes, sb, z)
    return oracle.Tensor(fmt, N, K, w, s, zz, group=128)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "q4k", "q40", "gptq", "awq"])
def test_gemv_one_hot_and_ones(fmt):
    N, K = 16, 256
    t = _random_tensor(fmt, N, K, 1)
    W = oracle.dequant(t)
    for k in (0, 17, 255):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y, b = oracle.gemv(t, x)
        assert np.array_equal(y[0], W[:, k].astype(np.float64))
        assert np.array_equal(b[0], np.abs(W[:, k]).astype(np.float64))
    y, _ = oracle.gemv(t, np.ones((1, K), np.float32))
    assert np.allclose(y[0], [math.fsum(r) for r in W.astype(np.float64)], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("fmt", ["nvfp4", "q4k", "gptq"])
def test_gemv_brute_force_tiny(fmt):
    N, K = 8, 256
    t = _random_tensor(fmt, N, K, 2)
    x = np.random.default_rng(3).normal(size=(3, K)).astype(np.float32)
    W = oracle.dequant(t).astype(np.float64)
    ref = np.array([[math.fsum(W[n] * x[m].astype(np.float64)) for n in range(N)] for m in range(3)])
    y, _ = oracle.gemv(t, x)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    y2, _ = oracle.gemv(t, x, rows=[5, 1])
    assert np.array_equal(y2, y[:, [5, 1]])


def test_nan_scale_rejected():
    t = oracle.Tensor("nvfp4", 1, 16, np.zeros((1, 8), np.uint8), np.array([[0x7F]], np.uint8),
                      scale2=1.0)
    with pytest.raises(oracle.OracleError):
        oracle.dequant(t)
    assert oracle.count_nan_scales("nvfp4", np.array([0x7F, 0xFF, 0x7E, 0x00], np.uint8)) == 2
    assert oracle.count_nan_scales("mxfp4", np.array([0x7F, 0xFF, 0xFE], np.uint8)) == 1


# --------------------------------------------------------------- repack

def test_repack_oracle_preserves_dequant_bitwise():
    import synth
    N, K = 64, 512
    W = synth.draw_weights(N, K, config=9, matrix=7, outliers=True)
    codes, sb, z = synth.quantize_affine(W, 128)
    gw, gs, gz = synth.pack_gptq(codes, sb, z)
    ref = oracle.dequant(oracle.Tensor("gptq", N, K, gw, gs, gz))
    aw, as_, az, perm = packing.repack("gptq", "awq", N, K, gw, gs, gz)
    assert perm is None
    assert np.array_equal(oracle.dequant(oracle.Tensor("awq", N, K, aw, as_, az)), ref)
    bw, bs, bz, _ = packing.repack("awq", "gptq", N, K, aw, as_, az)
    assert np.array_equal(bw, gw) and np.array_equal(bs, gs) and np.array_equal(bz, gz)
    lw, ls, lz, _ = packing.repack("gptq", "logical", N, K, gw, gs, gz)
    assert np.array_equal(oracle.dequant(oracle.Tensor("logical", N, K, lw, ls, lz)), ref)
    q40 = synth.quantize_q40(W)
    ref0 = oracle.dequant(oracle.Tensor("q40", N, K, q40))
    qw, qs, qz, _ = packing.repack("q40", "gptq", N, K, q40)
    assert np.all(qz.view(np.uint32) == 0x77777777)
    assert np.array_equal(oracle.dequant(oracle.Tensor("gptq", N, K, qw, qs, qz, group=32)), ref0)
    p, s, s2 = synth.quantize_nvfp4(W)
    refn = oracle.dequant(oracle.Tensor("nvfp4", N, K, p, s, scale2=s2))
    hw, hs, _, _ = packing.repack("nvfp4", "nvfp4_splithalf", N, K, p, s)
    assert not np.array_equal(hw, p)
    assert np.array_equal(oracle.dequant(oracle.Tensor("nvfp4_splithalf", N, K, hw, hs, scale2=s2)), refn)
    back, _, _, _ = packing.repack("nvfp4_splithalf", "nvfp4", N, K, hw, hs)
    assert np.array_equal(back, p)


def test_repack_act_order_permutation():
    import synth
    N, K, G = 16, 512, 128
    W = synth.draw_weights(N, K, config=9, matrix=8)
    g_idx = synth.act_order_g_idx(K, G, seed=4)
    codes, sb, z = synth.quantize_affine(W, G, g_idx=g_idx)
    gw, gs, gz = synth.pack_gptq(codes, sb, z)
    src = oracle.dequant(oracle.Tensor("gptq", N, K, gw, gs, gz, g_idx=g_idx))
    aw, as_, az, perm = packing.repack("gptq", "awq", N, K, gw, gs, gz, g_idx=g_idx)
    assert perm is not None and sorted(perm) == list(range(K))
    assert np.all(np.diff(g_idx[perm]) >= 0)
    dst = oracle.dequant(oracle.Tensor("awq", N, K, aw, as_, az))
    assert np.array_equal(dst, src[:, perm])                    # same weights, K permuted


# ------------------------------------------- bf16-staged weights (tensor-core GEMM)

def _q4k_single_weight_block(d_bits):
    """One Q4_K super-block whose only nonzero weight is k = 0 with
    w_hat = d * sc_0 * q - dmin * m_0 = d (sc_0 = 1, m_0 = 0, q = 1, dmin = 0)."""
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([d_bits], np.uint16).view(np.uint8)
    blk[4] = 1          # sc_0 = B[0] & 63
    blk[16] = 0x01      # code byte 0, low nibble: k = 0
    return oracle.Tensor("q4k", 1, 256, blk.reshape(1, 1, 144))


@pytest.mark.parametrize("d, want", [
    (1 + 2**-8 + 2**-10, 1 + 2**-7),   # above the midpoint: rounds up
    (1 + 2**-8, 1.0),                  # exact tie, even neighbour below
    (1 + 2**-7 + 2**-8, 1 + 2**-6),    # exact tie, even neighbour above
    (1 + 2**-7, 1 + 2**-7),            # representable: unchanged
])
def test_bf16_weight_rounding_closed_form(d, want):
    """bf16 keeps 8 significant bits: these f16 weights sit on, between and at
    the midpoints of the bf16 grid near 1, so round-to-nearest-even is fixed
    by hand."""
    t = _q4k_single_weight_block(int(np.array([d], np.float16).view(np.uint16)[0]))
    assert oracle.dequant(t)[0, 0] == np.float32(d)
    x = np.zeros((2, 256), np.float32)
    x[0, 0] = 1.0
    x[1, 0] = -3.0
    y, b = oracle.gemm_bf16_weights(t, x)
    assert y[0, 0] == want and y[1, 0] == -3.0 * want
    assert b[1, 0] == 3.0 * want


def test_bf16_weights_equal_gemv_when_weights_are_bf16():
    """NVFP4 with a power-of-two scale2: w_hat = v*dec(s)*2^j has <= 6
    significant bits, so rounding to bf16 changes nothing and the result is
    the independent f64 GEMV's."""
    import synth
    W = synth.draw_weights(24, 512, config=0, matrix=9)
    p, s, _ = synth.quantize_nvfp4(W)
    t = oracle.Tensor("nvfp4", 24, 512, p, s, scale2=0.25)
    x = np.random.default_rng(4).normal(size=(3, 512)).astype(np.float32)
    y, b = oracle.gemm_bf16_weights(t, x)
    y0, b0 = oracle.gemv(t, x)
    assert np.allclose(y, y0, rtol=1e-13, atol=1e-15) and np.allclose(b, b0, rtol=1e-13)


def test_bf16_weights_against_torch_rounding():
    """The rounding step agrees with torch's own float32 -> bfloat16 cast on a
    random Q4_K tensor (rows subset included)."""
    t = _random_tensor("q4k", 12, 512, 5)
    x = np.random.default_rng(6).normal(size=(2, 512)).astype(np.float32)
    Wt = torch.from_numpy(oracle.dequant(t)).to(torch.bfloat16).to(torch.float64).numpy()
    ref = np.array([[math.fsum(Wt[n] * x[m].astype(np.float64)) for n in range(12)] for m in range(2)])
    y, _ = oracle.gemm_bf16_weights(t, x)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    y2, _ = oracle.gemm_bf16_weights(t, x, rows=[7, 0])
    assert np.allclose(y2, y[:, [7, 0]], rtol=1e-15, atol=0)
