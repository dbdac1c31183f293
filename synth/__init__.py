"""Seeded synthetic workloads: weight/activation draws and the encoders that
turn them into packed 4-bit tensors.

This module is the *write side* only.  It draws random numbers, rounds them onto
a format's grid and lays the codes out in bytes.  It holds no decoder and no dot
product: the CUDA kernels and the CPU oracle each decode the bytes produced
here with their own code, and neither imports the other.

Recipes (the workload shapes of the decode-GEMV study):
  * W ~ N(0, 0.02) f32; optionally 1% of entries (seeded mask) x10 and each row
    scaled by U(0.5, 2); x ~ N(0, 1), rounded to bf16 nearest-even when bf16.
  * seed = 1000*config + 10*matrix_index + {0: W, 1: x, 2: outlier mask,
    3: row scale}; numpy ``default_rng`` (PCG64).
  * NVFP4: scale2 = f32(amax|W| / (448*6)); per 16 values the E4M3FN scale is
    the nearest-even E4M3FN of f32(amax_g/6/scale2), saturating at 448; the code
    is the nearest-even E2M1 value of w/(s*scale2), saturating at 6 (ModelOpt's
    ties-to-even rule); a negative value that rounds to zero keeps its sign.
  * MXFP4: E8M0 exponent e = clamp(floor(log2 amax_32) - 2, -127, 127), codes
    nearest-even E2M1 of w/2^e.
  * Q4_K: per 32-value sub-block lo = min(0, min w), scale = (max w - lo)/15,
    min = -lo; d = fp16(max scale/63), dmin = fp16(max min/63); 6-bit sc, m by
    nearest-even, codes nearest-even of (w + dmin*m)/(d*sc) clamped to 0..15.
  * Q4_0: d = fp16(-m/8), m the signed largest-magnitude value; q = rne(w/d)+8.
  * GPTQ / AWQ: asymmetric group-128 min/max: scale = fp16((max-min)/15),
    zero = clamp(rne(-min/scale), 1, 15), q = clamp(rne(w/scale)+zero, 0, 15).
"""
from __future__ import annotations

import numpy as np

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E2M1_MID = (E2M1_GRID[1:] + E2M1_GRID[:-1]) / 2
AWQ_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)


def seed_for(config: int, matrix: int, what: str) -> int:
    return 1000 * config + 10 * matrix + {"W": 0, "x": 1, "mask": 2, "rowscale": 3}[what]


def draw_weights(N, K, config=0, matrix=0, outliers=False, row_scale=False) -> np.ndarray:
    W = np.random.default_rng(seed_for(config, matrix, "W")).normal(0.0, 0.02, (N, K))
    W = W.astype(np.float32)
    if outliers:
        mask = np.random.default_rng(seed_for(config, matrix, "mask")).random((N, K)) < 0.01
        W[mask] *= np.float32(10.0)
    if row_scale:
        r = np.random.default_rng(seed_for(config, matrix, "rowscale")).uniform(0.5, 2.0, (N, 1))
        W *= r.astype(np.float32)
    return W


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Nearest-even rounding of finite f32 values to bfloat16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def draw_x(M, K, config=0, matrix=0, dtype="bf16"):
    """Activations ~ N(0,1).  Returns (array for the device, f32 values):
    bf16 bit patterns (uint16) or f32, and their exact f32 widening."""
    x = np.random.default_rng(seed_for(config, matrix, "x")).normal(0.0, 1.0, (M, K))
    x = x.astype(np.float32)
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x)
        return bits, (bits.astype(np.uint32) << 16).view(np.float32)
    return x, x


# --------------------------------------------------------------- encoders

def round_e2m1(r: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code for values r (any sign), ties to the even code,
    saturating at magnitude 6; negative values keep the sign bit.
    A value above midpoint i moves past grid point i; a value exactly on
    midpoint i goes up only when i is odd (grid i+1 has the even code)."""
    a = np.abs(np.asarray(r, dtype=np.float32))
    idx = np.zeros(a.shape, dtype=np.uint8)
    for i, mid in enumerate(_E2M1_MID.astype(np.float32)):
        idx += a > mid
        if i % 2 == 1:
            idx += a == mid
    return idx | (np.signbit(r).astype(np.uint8) << 3)


def round_e4m3fn(v: np.ndarray) -> np.ndarray:
    """Nearest-even E4M3FN byte for non-negative values, saturating at 448."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.int64)
    pos = v > 0
    _, ex = np.frexp(np.where(pos, v, 1.0))
    e = ex - 1                                     # v in [2^e, 2^(e+1))
    normal = pos & (e >= -6)
    m = np.rint((v / np.exp2(e.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    e = np.where(m == 8, e + 1, e)
    m = np.where(m == 8, 0, m)
    nb = ((e + 7) << 3) | m
    sub = pos & ~normal
    sb = np.rint(v * 512.0).astype(np.int64)       # multiples of 2^-9; 8 rolls into 0x08
    out = np.where(normal, nb, out)
    out = np.where(sub, sb, out)
    out = np.where(pos & ((out > 0x7E) | (v >= 448.0)), 0x7E, out)
    return out.astype(np.uint8)


def _e4m3_grid_value(b: np.ndarray) -> np.ndarray:
    """Grid value of the (non-negative, finite) E4M3 bytes this encoder emits."""
    b = b.astype(np.int64)
    e, m = (b >> 3) & 15, b & 7
    return np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * np.exp2(e - 7.0))


def _pack_nibbles_even_odd(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def quantize_nvfp4(W: np.ndarray):
    """-> (payload u8 [N][K/2], scales u8 [N][K/16], scale2 f32)."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    amax = np.float32(np.abs(W).max())
    scale2 = np.float32(amax / np.float32(448.0 * 6.0)) if amax > 0 else np.float32(1.0)
    g = W.reshape(N, K // 16, 16)
    amax_g = np.abs(g).max(axis=2)
    s_val = (amax_g / np.float32(6.0)) / scale2
    sb = round_e4m3fn(s_val.astype(np.float32))
    den = (_e4m3_grid_value(sb).astype(np.float32) * scale2).astype(np.float32)
    safe = np.where(den > 0, den, np.float32(1.0)).astype(np.float32)
    codes = round_e2m1(g / safe[:, :, None])
    codes[den <= 0] = 0
    codes = codes.reshape(N, K)
    return _pack_nibbles_even_odd(codes), sb, np.float32(scale2)


def quantize_mxfp4(W: np.ndarray):
    """-> (payload u8 [N][K/2], E8M0 scales u8 [N][K/32])."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    g = W.reshape(N, K // 32, 32)
    amax = np.abs(g).max(axis=2).astype(np.float64)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    e = np.clip(ex - 1 - 2, -127, 127)
    e = np.where(amax > 0, e, -127)
    codes = round_e2m1(g / np.exp2(e)[:, :, None]).reshape(N, K)
    return _pack_nibbles_even_odd(codes), (e + 127).astype(np.uint8)


def _fp16_bits(v: np.ndarray) -> np.ndarray:
    return np.asarray(v, dtype=np.float32).astype(np.float16).view(np.uint16)


def quantize_q4k(W: np.ndarray) -> np.ndarray:
    """-> Q4_K super-blocks u8 [N][K/256][144]: d@0, dmin@2, 12 B scales@4,
    128 B codes@16 (chunk c byte l: low = k 64c+l, high = k 64c+32+l)."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    nb = K // 256
    sub = W.reshape(N, nb, 8, 32).astype(np.float64)
    lo = np.minimum(0.0, sub.min(axis=3))
    scale = (sub.max(axis=3) - lo) / 15.0
    mins = -lo
    d = _fp16_bits(scale.max(axis=2) / 63.0)
    dmin = _fp16_bits(mins.max(axis=2) / 63.0)
    df = d.view(np.float16).astype(np.float64)
    dminf = dmin.view(np.float16).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(df[:, :, None] > 0, np.rint(scale / df[:, :, None]), 0.0)
        mn = np.where(dminf[:, :, None] > 0, np.rint(mins / dminf[:, :, None]), 0.0)
    sc = np.clip(sc, 0, 63).astype(np.int64)
    mn = np.clip(mn, 0, 63).astype(np.int64)
    step = df[:, :, None] * sc
    off = dminf[:, :, None] * mn
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(step[..., None] > 0, np.rint((sub + off[..., None]) / step[..., None]), 0.0)
    q = np.clip(q, 0, 15).astype(np.uint8)                      # [N, nb, 8, 32]
    out = np.zeros((N, nb, 144), dtype=np.uint8)
    out[:, :, 0] = d & 0xFF
    out[:, :, 1] = d >> 8
    out[:, :, 2] = dmin & 0xFF
    out[:, :, 3] = dmin >> 8
    B = np.zeros((N, nb, 12), dtype=np.int64)
    for j in range(4):
        B[:, :, j] = sc[:, :, j] | ((sc[:, :, j + 4] >> 4) << 6)
        B[:, :, j + 4] = mn[:, :, j] | ((mn[:, :, j + 4] >> 4) << 6)
        B[:, :, j + 8] = (sc[:, :, j + 4] & 15) | ((mn[:, :, j + 4] & 15) << 4)
    out[:, :, 4:16] = B.astype(np.uint8)
    for c in range(4):
        out[:, :, 16 + 32 * c:16 + 32 * c + 32] = q[:, :, 2 * c, :] | (q[:, :, 2 * c + 1, :] << 4)
    return out


def quantize_q40(W: np.ndarray) -> np.ndarray:
    """-> Q4_0 blocks u8 [N][K/32][18]."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    g = W.reshape(N, K // 32, 32).astype(np.float64)
    idx = np.abs(g).argmax(axis=2)
    m = np.take_along_axis(g, idx[:, :, None], axis=2)[:, :, 0]
    d = _fp16_bits(-m / 8.0)
    df = d.view(np.float16).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(df[:, :, None] != 0, np.rint(g / df[:, :, None]) + 8, 8)
    q = np.clip(q, 0, 15).astype(np.uint8)
    out = np.empty((N, K // 32, 18), dtype=np.uint8)
    out[:, :, 0] = d & 0xFF
    out[:, :, 1] = d >> 8
    out[:, :, 2:] = q[:, :, :16] | (q[:, :, 16:] << 4)
    return out


def quantize_affine(W: np.ndarray, group: int = 128, g_idx=None):
    """Asymmetric min/max quantization along K.  Returns the logical matrix:
    (codes u8 [K][N], fp16 scale bits u16 [groups][N], zeros u8 [groups][N])."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    Wt = W.T.astype(np.float64)                                 # [K][N]
    groups = K // group
    gi = (np.arange(K) // group) if g_idx is None else np.asarray(g_idx)
    gmin = np.full((groups, N), np.inf)
    gmax = np.full((groups, N), -np.inf)
    np.minimum.at(gmin, gi, Wt)
    np.maximum.at(gmax, gi, Wt)
    sbits = _fp16_bits((gmax - gmin) / 15.0)
    s = sbits.view(np.float16).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        z = np.where(s > 0, np.rint(-gmin / s), 8.0)
    z = np.clip(z, 1, 15).astype(np.int64)
    sk, zk = s[gi, :], z[gi, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sk > 0, np.rint(Wt / sk) + zk, zk)
    q = np.clip(q, 0, 15).astype(np.uint8)
    return q, sbits, z.astype(np.uint8)


def act_order_g_idx(K: int, group: int, seed: int) -> np.ndarray:
    """A non-monotonic g_idx with exactly ``group`` rows per group (act-order)."""
    perm = np.random.default_rng(seed).permutation(K)
    g = np.empty(K, dtype=np.int32)
    g[perm] = np.arange(K) // group
    return g


def pack_gptq(codes, sbits, zeros):
    """Logical (codes [K][N], scales, zeros 1..16) -> GPTQ (qweight int32
    [K/8][N], scales fp16 bits [groups][N], qzeros int32 [groups][N/8])."""
    K, N = codes.shape
    qw = np.zeros((K // 8, N), dtype=np.uint32)
    for j in range(8):
        qw |= codes[j::8, :].astype(np.uint32) << np.uint32(4 * j)
    st = (zeros.astype(np.int64) - 1) & 15
    qz = np.zeros((zeros.shape[0], N // 8), dtype=np.uint32)
    for s in range(8):
        qz |= st[:, s::8].astype(np.uint32) << np.uint32(4 * s)
    return qw.view(np.int32), sbits.copy(), qz.view(np.int32)


def pack_awq(codes, sbits, zeros):
    """Logical -> AWQ (qweight int32 [K][N/8], scales, qzeros int32 [groups][N/8])."""
    def words(a):
        R, N = a.shape
        o = np.zeros((R, N // 8), dtype=np.uint32)
        for p, col in enumerate(AWQ_ORDER):
            o |= a[:, col::8].astype(np.uint32) << np.uint32(4 * p)
        return o.view(np.int32)
    return words(codes), sbits.copy(), words(zeros)


def random_bytes(shape, seed, exclude=()):
    """Uniform random bytes (all nibble codes), resampling excluded values
    (e.g. the NaN scale encodings)."""
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 256, size=shape, dtype=np.uint8)
    for v in exclude:
        bad = b == v
        while bad.any():
            b[bad] = rng.integers(0, 256, size=int(bad.sum()), dtype=np.uint8)
            bad = np.isin(b, list(exclude))
    return b


def make_layer(fmt: str, N: int, K: int, config: int = 0, matrix: int = 0, outliers=False,
               row_scale=False, group: int = 128, act_order: bool = False, W=None) -> dict:
    """One packed weight tensor of ``fmt`` drawn by the recipe above.

    Returns host arrays: ``w`` (payload), ``scales``, ``zeros``, ``g_idx``
    (None unless act_order), plus ``scale2`` and ``group``; dtypes match the
    byte layouts (uint8 bytes, uint16 fp16 bits, int32 words)."""
    if W is None:
        W = draw_weights(N, K, config, matrix, outliers=outliers, row_scale=row_scale)
    out = {"fmt": fmt, "N": N, "K": K, "scale2": 1.0, "group": group, "zeros": None,
           "g_idx": None, "scales": None}
    if fmt in ("nvfp4", "nvfp4_splithalf"):
        p, s, s2 = quantize_nvfp4(W)
        if fmt == "nvfp4_splithalf":
            codes = np.empty((N, K), np.uint8)
            codes[:, 0::2], codes[:, 1::2] = p & 15, p >> 4
            g = codes.reshape(N, K // 16, 16)
            p = (g[:, :, :8] | (g[:, :, 8:] << 4)).reshape(N, K // 2).astype(np.uint8)
        out.update(w=p, scales=s, scale2=float(s2))
    elif fmt == "mxfp4":
        p, s = quantize_mxfp4(W)
        out.update(w=p, scales=s)
    elif fmt == "q4k":
        out.update(w=quantize_q4k(W))
    elif fmt == "q40":
        out.update(w=quantize_q40(W))
    elif fmt in ("gptq", "awq", "logical"):
        g_idx = act_order_g_idx(K, group, seed_for(config, matrix, "mask") + 7) if act_order else None
        codes, sb, z = quantize_affine(W, group, g_idx=g_idx)
        if fmt == "gptq":
            w, s, zz = pack_gptq(codes, sb, z)
        elif fmt == "awq":
            w, s, zz = pack_awq(codes, sb, z)
        else:
            w, s, zz = codes, sb, z
        out.update(w=w, scales=s, zeros=zz, g_idx=g_idx)
    else:
        raise ValueError(fmt)
    return out
