"""The arithmetic the integer-exact tensor-core kernels rely on, checked on the
CPU (no GPU): the A16-Q8 lane ([MUS7] 7.4.2) and the Q4_K x Q8 (W4A8) lane
([W4K] section 7) form exact integers with f16 MMAs and f32 accumulators, then
read them back from f32 bits.

  * A16-Q8: E2M1 values times doubled 8-bit codes are integers, a 16-k group's
    sum stays below 2^15, so every partial sum is an exact f32.
  * W4A8: 4-bit codes as f16 subnormals (q 2^-24, 16 q 2^-24) and codes
    divided by 16 are exact f16 numbers; a 32-k sub-block's sum is an integer
    below 2^16 times 2^-24.
  * Both: 1.5 * 2^23 + n is exact in f32 for |n| < 2^22, and its bit pattern
    minus 0x4B400000 is n (the add that replaces a float-to-int conversion).
"""
import numpy as np

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)
MAGIC = np.float32(1.5 * 2 ** 23)


def magic_read(v32):
    """Bits of the f32 sum 1.5 * 2^23 + v, minus 0x4B400000."""
    s = (np.asarray(v32, np.float32) + MAGIC).astype(np.float32)
    return s.view(np.int32).astype(np.int64) - 0x4B400000


def test_magic_add_reads_every_integer_back():
    n = np.arange(-(1 << 16), (1 << 16) + 1, dtype=np.int64)
    assert np.array_equal(magic_read(n.astype(np.float32)), n)
    rng = np.random.default_rng(7)
    wide = rng.integers(-(1 << 22) + 1, 1 << 22, size=200000)
    assert np.array_equal(magic_read(wide.astype(np.float32)), wide)


def test_a16q8_group_sums_are_exact_integers():
    codes = np.arange(-127, 128, dtype=np.float64)               # the contract's 8-bit codes
    b = (2 * codes).astype(np.float16)                            # staged doubled: exact in f16
    assert np.array_equal(b.astype(np.float64), 2 * codes)
    a = np.concatenate([E2M1, -E2M1]).astype(np.float16)          # every E2M1 value is an f16 number
    prod = np.outer(a.astype(np.float64), b.astype(np.float64))
    assert np.array_equal(prod, np.round(prod))                   # q1 * q8: integers
    assert np.abs(prod).max() == 12 * 127 < 2 ** 11
    worst = 16 * np.abs(prod).max()                               # a 16-k group
    assert worst < 2 ** 15
    # f32 accumulation of any order of such products stays exact: partial sums are integers below 2^24
    rng = np.random.default_rng(3)
    for _ in range(2000):
        terms = rng.choice(prod.ravel(), size=16)
        acc = np.float32(0)
        for t in terms:
            acc = np.float32(acc + np.float32(t))
        assert float(acc) == terms.sum()
        assert magic_read(acc) == int(terms.sum())


def test_w4a8_subnormal_codes_and_sixteenth_codes_are_exact():
    q = np.arange(16)
    lo = q.astype(np.uint16).view(np.float16)                     # bits q: q * 2^-24 (f16 subnormal)
    hi = (q << 4).astype(np.uint16).view(np.float16)              # bits 16q: 16 q * 2^-24
    assert np.array_equal(lo.astype(np.float64), q * 2.0 ** -24)
    assert np.array_equal(hi.astype(np.float64), 16 * q * 2.0 ** -24)
    codes = np.arange(-128, 128, dtype=np.float64)
    sixteenth = (codes / 16).astype(np.float16)                   # high-nibble activations staged / 16
    assert np.array_equal(sixteenth.astype(np.float64), codes / 16)
    # both halves give q * q8 * 2^-24 exactly
    p_lo = np.outer(lo.astype(np.float64), codes)
    p_hi = np.outer(hi.astype(np.float64), sixteenth.astype(np.float64))
    assert np.array_equal(p_lo, p_hi)
    assert np.array_equal(p_lo * 2.0 ** 24, np.outer(q, codes))


def test_w4a8_sub_block_sum_read_by_one_fma():
    rng = np.random.default_rng(11)
    for worst in (False, True):
        for _ in range(500):
            q = np.full(32, 15) if worst else rng.integers(0, 16, 32)
            c = np.full(32, -127) if worst else rng.integers(-127, 128, 32)
            n = int((q * c).sum())
            assert abs(n) <= 32 * 15 * 127 < 2 ** 16
            d = np.float32(n * 2.0 ** -24)                        # the f32 accumulator: exact
            assert float(d) * 2 ** 24 == n
            # fma(D, 2^24, 1.5 * 2^23): the exact value is representable, so one rounding changes nothing
            exact = np.float64(d) * 2 ** 24 + 1.5 * 2 ** 23
            assert np.float64(np.float32(exact)) == exact
            assert int(np.float32(exact).view(np.int32)) - 0x4B400000 == n
