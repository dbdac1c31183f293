"""Reference bit packers and the repack-through-the-logical-matrix route.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Slow and unambiguous on
purpose: these are the oracle for the GPU repack kernels, as [BPA] "The packing
arithmetic" asks for a plain reference unpacker beside every fast one.

Layouts ([BPA] "Real layouts compared"; readings marked):
  * generic b-bit stream: element i occupies bits [i*b, (i+1)*b) of a
    little-endian sequence of 32-bit words; values may straddle two words.
  * GPTQ qweight int32 [K/8][N]: logical row 8r+j of column n at bits 4j of
    word (r, n).  qzeros int32 [groups][N/8]: column n at bits 4*(n%8) of word
    (g, n/8) (reading), stored as zero-1.
  * AWQ qweight int32 [K][N/8]: slot p (bits 4p) of word (k, c) holds logical
    column 8c + AWQ_ORDER[p].  qzeros: same interleave, no minus-one (reading).
  * Q4_0: 18-byte blocks (fp16 d, 16 code bytes; byte j = element j low,
    element j+16 high), w = d*(q-8).
  * logical matrix: u8 codes [K][N], fp16 scales [groups][N], u8 zeros
    [groups][N], w = scale*(q - zero) ([BPA] "Repacking between formats").
  * NVFP4 nibble orders: even/odd ([MUS7] 7.1: low nibble = even index) and
    split-half ([W4K] section 5: in each 16-group, low nibbles of the 8 bytes
    are lanes 0-7, high nibbles lanes 8-15).
"""
from __future__ import annotations

import numpy as np

AWQ_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)


# ----------------------------------------------------------- generic stream

def pack_bits(values, bits: int) -> np.ndarray:
    """Pack unsigned ``bits``-wide codes as one little-endian bit stream split
    into 32-bit words ([BPA] "The packing arithmetic").  The stream is built as
    a single Python integer, so straddling values need no special case."""
    values = [int(v) for v in np.asarray(values).ravel()]
    total = len(values) * bits
    if total % 32:
        raise ValueError("len(values) * bits must be a multiple of 32")
    mask = (1 << bits) - 1
    stream = 0
    for i, v in enumerate(values):
        if v < 0 or v > mask:
            raise ValueError(f"code {v} does not fit in {bits} bits")
        stream |= v << (i * bits)
    return np.array([(stream >> (32 * w)) & 0xFFFFFFFF for w in range(total // 32)],
                    dtype=np.uint32)


def unpack_bits(words, bits: int, n: int) -> np.ndarray:
    """Inverse of :func:`pack_bits` for the first ``n`` codes."""
    stream = 0
    for w, word in enumerate(np.asarray(words, dtype=np.uint32).ravel()):
        stream |= int(word) << (32 * w)
    mask = (1 << bits) - 1
    return np.array([(stream >> (i * bits)) & mask for i in range(n)], dtype=np.uint8)


# ------------------------------------------------------------- GPTQ / AWQ

def _u32(a):
    return np.asarray(a).astype(np.uint32)


def pack_gptq_qweight(q: np.ndarray) -> np.ndarray:
    """Logical codes [K][N] -> GPTQ qweight int32 [K/8][N] (packed along K)."""
    K, N = q.shape
    out = np.zeros((K // 8, N), dtype=np.uint32)
    for j in range(8):
        out |= _u32(q[j::8, :]) << np.uint32(4 * j)
    return out.view(np.int32)


def unpack_gptq_qweight(qw: np.ndarray) -> np.ndarray:
    R, N = qw.shape
    w = qw.view(np.uint32)
    q = np.empty((R * 8, N), dtype=np.uint8)
    for j in range(8):
        q[j::8, :] = (w >> np.uint32(4 * j)) & np.uint32(15)
    return q


def pack_gptq_qzeros(z: np.ndarray) -> np.ndarray:
    """Logical zeros [groups][N] (1..16) -> qzeros int32 [groups][N/8], each
    stored as zero-1 ([BPA]: AutoGPTQ subtracts one before storing)."""
    G, N = z.shape
    stored = (z.astype(np.int64) - 1) & 15
    out = np.zeros((G, N // 8), dtype=np.uint32)
    for s in range(8):
        out |= _u32(stored[:, s::8]) << np.uint32(4 * s)
    return out.view(np.int32)


def unpack_gptq_qzeros(qz: np.ndarray) -> np.ndarray:
    G, C = qz.shape
    w = qz.view(np.uint32)
    z = np.empty((G, C * 8), dtype=np.uint8)
    for s in range(8):
        z[:, s::8] = ((w >> np.uint32(4 * s)) & np.uint32(15)) + 1
    return z


def pack_awq_words(q: np.ndarray) -> np.ndarray:
    """[R][N] codes -> int32 [R][N/8] with AWQ's slot order (qweight, qzeros)."""
    R, N = q.shape
    out = np.zeros((R, N // 8), dtype=np.uint32)
    for p, col in enumerate(AWQ_ORDER):
        out |= _u32(q[:, col::8]) << np.uint32(4 * p)
    return out.view(np.int32)


def unpack_awq_words(words: np.ndarray) -> np.ndarray:
    R, C = words.shape
    w = words.view(np.uint32)
    q = np.empty((R, C * 8), dtype=np.uint8)
    for p, col in enumerate(AWQ_ORDER):
        q[:, col::8] = (w >> np.uint32(4 * p)) & np.uint32(15)
    return q


# -------------------------------------------------------------------- Q4_0

def q40_to_logical(blocks: np.ndarray, N: int, K: int):
    """Q4_0 bytes [N][K/32][18] -> (codes [K][N] u8, scale bits [K/32][N] u16,
    zeros [K/32][N] u8 = 8)."""
    b = np.asarray(blocks, dtype=np.uint8).reshape(N, K // 32, 18)
    d = (b[:, :, 0].astype(np.uint16) | (b[:, :, 1].astype(np.uint16) << 8))
    qs = b[:, :, 2:]
    codes = np.empty((N, K // 32, 32), dtype=np.uint8)
    codes[:, :, :16] = qs & 15
    codes[:, :, 16:] = qs >> 4
    codes = codes.reshape(N, K).T.copy()
    return codes, d.T.copy(), np.full((K // 32, N), 8, dtype=np.uint8)


def pack_q40(codes_nk: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """codes [N][K] (0..15) and fp16 bits [N][K/32] -> Q4_0 bytes [N][K/32][18]."""
    N, K = codes_nk.shape
    c = codes_nk.reshape(N, K // 32, 32).astype(np.uint8)
    out = np.empty((N, K // 32, 18), dtype=np.uint8)
    out[:, :, 0] = d_bits & 0xFF
    out[:, :, 1] = d_bits >> 8
    out[:, :, 2:] = c[:, :, :16] | (c[:, :, 16:] << 4)
    return out


# ------------------------------------------------------------ NVFP4 orders

def nvfp4_codes(payload: np.ndarray, N: int, K: int, split_half: bool = False) -> np.ndarray:
    """Payload bytes [N][K/2] -> E2M1 codes [N][K] in logical k order."""
    b = np.asarray(payload, dtype=np.uint8).reshape(N, K // 2)
    codes = np.empty((N, K), dtype=np.uint8)
    if not split_half:
        codes[:, 0::2] = b & 15
        codes[:, 1::2] = b >> 4
    else:
        g = b.reshape(N, K // 16, 8)
        c = codes.reshape(N, K // 16, 16)
        c[:, :, :8] = g & 15
        c[:, :, 8:] = g >> 4
    return codes


def pack_nvfp4_codes(codes: np.ndarray, split_half: bool = False) -> np.ndarray:
    """E2M1 codes [N][K] -> payload bytes [N][K/2] in the chosen nibble order."""
    N, K = codes.shape
    c = codes.astype(np.uint8)
    if not split_half:
        return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    g = c.reshape(N, K // 16, 16)
    return (g[:, :, :8] | (g[:, :, 8:] << 4)).reshape(N, K // 2).astype(np.uint8)


# ------------------------------------------------------- logical repacking

def to_logical(fmt: str, N: int, K: int, w, scales=None, zeros=None, group=128, g_idx=None):
    """Step 1-2 of [BPA] "Repacking between formats": unpack codes along the
    source's axis and order, normalise zero points (GPTQ adds back one).
    Returns (codes [K][N] u8, scale bits [groups][N] u16, zeros [groups][N] u8)."""
    if fmt == "gptq":
        codes = unpack_gptq_qweight(np.asarray(w, dtype=np.int32).reshape(K // 8, N))
        z = unpack_gptq_qzeros(np.asarray(zeros, dtype=np.int32).reshape(-1, N // 8))
        s = np.asarray(scales).view(np.uint16).reshape(-1, N)
        return codes, s.copy(), z
    if fmt == "awq":
        codes = unpack_awq_words(np.asarray(w, dtype=np.int32).reshape(K, N // 8))
        z = unpack_awq_words(np.asarray(zeros, dtype=np.int32).reshape(-1, N // 8))
        s = np.asarray(scales).view(np.uint16).reshape(-1, N)
        return codes, s.copy(), z
    if fmt == "q40":
        return q40_to_logical(w, N, K)
    if fmt == "logical":
        return (np.asarray(w, dtype=np.uint8).reshape(K, N).copy(),
                np.asarray(scales).view(np.uint16).reshape(-1, N).copy(),
                np.asarray(zeros, dtype=np.uint8).reshape(-1, N).copy())
    raise ValueError(f"no logical form for {fmt}")


def from_logical(fmt: str, codes, scale_bits, zeros):
    """Step 4 of [BPA] "Repacking between formats": pack along the target's axis
    and order and write its metadata.  Returns (w, scales, zeros) arrays.
    GPTQ cannot store a zero of 0 (stored zero-1 would wrap) and AWQ cannot
    store 16: both raise, the documented off-by-one failure mode."""
    codes = np.asarray(codes, dtype=np.uint8)
    zeros = np.asarray(zeros, dtype=np.uint8)
    if fmt == "gptq":
        if np.any(zeros < 1) or np.any(zeros > 16):
            raise ValueError("GPTQ zero outside 1..16")
        return pack_gptq_qweight(codes), scale_bits.copy(), pack_gptq_qzeros(zeros)
    if fmt == "awq":
        if np.any(zeros > 15):
            raise ValueError("AWQ zero outside 0..15")
        return pack_awq_words(codes), scale_bits.copy(), pack_awq_words(zeros)
    if fmt == "logical":
        return codes.copy(), scale_bits.copy(), zeros.copy()
    raise ValueError(f"cannot pack logical matrix as {fmt}")


def act_order_permutation(g_idx: np.ndarray) -> np.ndarray:
    """Step 3 of [BPA] "Repacking between formats": the K permutation that makes
    groups contiguous -- a stable sort of k by g_idx.  perm[k'] = source row."""
    g = np.asarray(g_idx, dtype=np.int64)
    return np.array(sorted(range(g.size), key=lambda k: (int(g[k]), k)), dtype=np.int32)


def repack(src: str, dst: str, N: int, K: int, w, scales=None, zeros=None, group=128,
           g_idx=None):
    """Repack ``src`` -> ``dst`` through the logical matrix.  Returns
    (w, scales, zeros, perm) where perm is None unless act-order rows had to be
    permuted (then row k' of the target is row perm[k'] of the source)."""
    if {src, dst} <= {"nvfp4", "nvfp4_splithalf"}:
        codes = nvfp4_codes(w, N, K, split_half=(src == "nvfp4_splithalf"))
        return (pack_nvfp4_codes(codes, split_half=(dst == "nvfp4_splithalf")),
                np.asarray(scales, dtype=np.uint8).copy(), None, None)
    codes, s, z = to_logical(src, N, K, w, scales, zeros, group, g_idx)
    perm = None
    if g_idx is not None and src in ("gptq", "logical"):
        g = np.asarray(g_idx, dtype=np.int64)
        if not np.array_equal(g, np.arange(K) // group):
            perm = act_order_permutation(g)
            codes = codes[perm, :]
    wt, st, zt = from_logical(dst, codes, s, z)
    return wt, st, zt, perm
