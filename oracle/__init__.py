"""CPU oracle for the 4-bit block formats -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library in
``bit_block_quantized_gb300``: the scalar decoders and the f64 GEMV live in
``q4_oracle.c`` (plain C, built with ``-ffp-contract=off``), the bit packers and
the repack-through-the-logical-matrix route in ``packing.py`` (numpy).

Citations name the source page and its section:
  [FBTC] "Four Bits, Three Contracts"; [W4K] "Why 4-Bit Quantization Is King";
  [BPA] "Bit Packing Architecture, in depth"; [MUS7] "Muser book, Chapter 7".
Every function is pinned by ``tests/test_oracle_pins.py`` or, for the A16-Q8,
W4A8, W4A4 and quantizer functions, by ``tests/test_oracle_{a16q8,w4a8,w4a4,quantize}.py``
(the Q4_K fit by ``tests/test_oracle_quantize_q4k.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import packing  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborc.so")
_lock = threading.Lock()
_lib = None

FMT = {"nvfp4": 1, "mxfp4": 2, "q4k": 3, "q40": 4, "gptq": 5, "awq": 6,
       "nvfp4_splithalf": 7, "logical": 8}


def build(force: bool = False) -> str:
    """Compile q4_oracle.c with the host C compiler (no CUDA involved)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Tensor(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("group", ctypes.c_int32),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("w", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p), ("g_idx", ctypes.c_void_p),
                ("scale2", ctypes.c_float)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_e2m1.restype = ctypes.c_float
            lib.orc_e2m1.argtypes = [ctypes.c_uint]
            lib.orc_e4m3fn.restype = ctypes.c_int
            lib.orc_e4m3fn.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_float)]
            lib.orc_e8m0.restype = ctypes.c_int
            lib.orc_e8m0.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_float)]
            lib.orc_half.restype = ctypes.c_float
            lib.orc_half.argtypes = [ctypes.c_uint16]
            lib.orc_bf16.restype = ctypes.c_float
            lib.orc_bf16.argtypes = [ctypes.c_uint16]
            lib.orc_round_bf16.restype = ctypes.c_uint16
            lib.orc_round_bf16.argtypes = [ctypes.c_float]
            lib.orc_dequant_rows.restype = ctypes.c_int
            lib.orc_dequant_rows.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_void_p]
            lib.orc_gemv_rows.restype = ctypes.c_int
            lib.orc_gemv_rows.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_void_p]
            lib.orc_round_bf16_array.restype = None
            lib.orc_round_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.orc_count_nan_scales.restype = ctypes.c_int64
            lib.orc_count_nan_scales.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64]
            lib.orc_e2m1_q1.restype = ctypes.c_int
            lib.orc_e2m1_q1.argtypes = [ctypes.c_uint]
            lib.orc_e4m3fn_q9.restype = ctypes.c_int
            lib.orc_e4m3fn_q9.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_int32)]
            lib.orc_q8_block.restype = None
            lib.orc_q8_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]
            lib.orc_f16_round.restype = ctypes.c_float
            lib.orc_f16_round.argtypes = [ctypes.c_float]
            lib.orc_gemv_a16q8_rows.restype = ctypes.c_int
            lib.orc_gemv_a16q8_rows.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_void_p, ctypes.c_int64,
                                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            lib.orc_gemv_q4k_q8_rows.restype = ctypes.c_int
            lib.orc_e2m1_round.restype = ctypes.c_uint
            lib.orc_e2m1_round.argtypes = [ctypes.c_float]
            lib.orc_e4m3fn_round.restype = ctypes.c_uint
            lib.orc_e4m3fn_round.argtypes = [ctypes.c_float]
            lib.orc_quantize_nvfp4.restype = None
            lib.orc_quantize_nvfp4_groups.restype = None
            lib.orc_quantize_nvfp4_groups.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                                      ctypes.c_void_p, ctypes.c_void_p]
            lib.orc_gemv_w4a4_rows.restype = ctypes.c_int
            lib.orc_gemv_w4a4_rows.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                               ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            lib.orc_quantize_nvfp4.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]
            lib.orc_gemv_q4k_q8_rows.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_void_p, ctypes.c_int64,
                                                 ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
            lib.orc_f16_bits.restype = ctypes.c_uint16
            lib.orc_f16_bits.argtypes = [ctypes.c_float]
            lib.orc_quantize_q4k.restype = None
            lib.orc_quantize_q4k.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
            _lib = lib
    return _lib


class OracleError(ValueError):
    pass


# ------------------------------------------------------------------ scalars

def e2m1(code: int) -> float:
    return float(_load().orc_e2m1(code))


def e4m3fn(byte: int) -> float:
    v = ctypes.c_float()
    if _load().orc_e4m3fn(byte, ctypes.byref(v)):
        raise OracleError(f"E4M3FN byte 0x{byte:02x} is a NaN encoding")
    return float(v.value)


def e8m0(byte: int) -> float:
    v = ctypes.c_float()
    if _load().orc_e8m0(byte, ctypes.byref(v)):
        raise OracleError(f"E8M0 byte 0x{byte:02x} is a NaN encoding")
    return float(v.value)


def half(bits: int) -> float:
    return float(_load().orc_half(bits))


def bf16(bits: int) -> float:
    return float(_load().orc_bf16(bits))


def round_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_round_bf16_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to f32 exactly (bf16 is the top half of f32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ tensors

class Tensor:
    """A packed weight tensor as host numpy arrays, in one of the formats.

    ``w``: payload bytes (any integer dtype, read as little-endian bytes);
    ``scales``: scale tensor bytes; ``zeros``: qzeros / logical zeros;
    ``g_idx``: optional int32 [K]; ``scale2``: NVFP4 tensor scale.
    """

    def __init__(self, fmt, N, K, w, scales=None, zeros=None, g_idx=None, group=128,
                 scale2=1.0):
        self.fmt = FMT[fmt] if isinstance(fmt, str) else int(fmt)
        self.N, self.K, self.group, self.scale2 = int(N), int(K), int(group), float(scale2)
        self.w = np.ascontiguousarray(w)
        self.scales = None if scales is None else np.ascontiguousarray(scales)
        self.zeros = None if zeros is None else np.ascontiguousarray(zeros)
        self.g_idx = None if g_idx is None else np.ascontiguousarray(g_idx, dtype=np.int32)

    def _c(self) -> _Tensor:
        p = lambda a: None if a is None else a.ctypes.data  # noqa: E731
        return _Tensor(self.fmt, self.group, self.N, self.K, p(self.w), p(self.scales),
                       p(self.zeros), p(self.g_idx), self.scale2)


def dequant(t: Tensor, rows=None) -> np.ndarray:
    """f32 [len(rows)][K] (all rows if ``rows`` is None) by the pinned rule."""
    lib = _load()
    ct = _Tensor.from_buffer_copy(t._c())
    if rows is None:
        out = np.empty((t.N, t.K), dtype=np.float32)
        rc = lib.orc_dequant_rows(ctypes.byref(ct), 0, t.N, out.ctypes.data)
    else:
        rows = list(rows)
        out = np.empty((len(rows), t.K), dtype=np.float32)
        rc = 0
        for i, n in enumerate(rows):
            rc = rc or lib.orc_dequant_rows(ctypes.byref(ct), int(n), 1, out[i].ctypes.data)
    if rc == 1:
        raise OracleError("a scale byte is a NaN encoding")
    if rc:
        raise OracleError(f"unknown format {t.fmt}")
    return out


def gemv(t: Tensor, x: np.ndarray, rows=None):
    """(y, bound): y[m][i] = sum_k w_hat[rows[i]][k] x[m][k] in f64, and
    bound[m][i] = sum_k |w_hat||x|.  ``x`` is f32 [M][K] (or [K])."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    M = x.shape[0]
    assert x.shape[1] == t.K
    rows = np.arange(t.N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    rows = np.ascontiguousarray(rows)
    y = np.empty((M, rows.size), dtype=np.float64)
    bound = np.empty((M, rows.size), dtype=np.float64)
    ct = _Tensor.from_buffer_copy(t._c())
    rc = _load().orc_gemv_rows(ctypes.byref(ct), x.ctypes.data, M, rows.ctypes.data, rows.size,
                               y.ctypes.data, bound.ctypes.data)
    if rc == 1:
        raise OracleError("a scale byte is a NaN encoding")
    if rc:
        raise OracleError(f"unknown format {t.fmt}")
    return y, bound


def gemm_bf16_weights(t: Tensor, x: np.ndarray, rows=None):
    """(y, bound) with every weight first rounded once to bf16.

    The small-batch tensor-core path stages weight tiles as bf16.  NVFP4's
    staged value v*dec(s) is exact there, but Q4_K's f32 weight
    fl(q*d*sc - dmin*m) ([FBTC] sections 5-6) generally is not; the reading
    for that path is w_bf16 = RNE_bf16(w_hat), then y = sum_k w_bf16 x in f64
    and bound = sum_k |w_bf16||x|.  ``x`` is f32 [M][K]; the result is
    [M][len(rows)] like :func:`gemv`."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float32)).astype(np.float64)
    assert x.shape[1] == t.K
    wb = bf16_bits_to_f32(round_bf16(dequant(t, rows))).astype(np.float64)
    return x @ wb.T, np.abs(x) @ np.abs(wb).T


def count_nan_scales(fmt, scales: np.ndarray) -> int:
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    return int(_load().orc_count_nan_scales(f, s.ctypes.data, s.size))


def gemv_tolerance(bound: np.ndarray) -> np.ndarray:
    """The GEMV acceptance bound: |y_gpu - y_ref| <= 1e-5 * sum|w_hat||x| + 1e-6."""
    return 1e-5 * bound + 1e-6


# ------------------------------------------- the integer-exact A16-Q8 lane
# [MUS7] 7.4.2: NVFP4 weights against activations quantized per 256-value
# block to signed 8-bit codes; the block contraction is an exact integer sum
# and only a pinned four-step f32 epilogue rounds.

def e2m1_q1(code: int) -> int:
    """E2M1 code as an integer number of halves (2 * v(code))."""
    return int(_load().orc_e2m1_q1(code))


def e4m3fn_q9(byte: int) -> int:
    """E4M3FN byte as an integer number of 2^-9 units."""
    v = ctypes.c_int32()
    if _load().orc_e4m3fn_q9(byte, ctypes.byref(v)):
        raise OracleError(f"E4M3FN byte 0x{byte:02x} is a NaN encoding")
    return int(v.value)


def q8_block(x: np.ndarray):
    """(codes int8 [256], scale f32) for one 256-value f32 activation block."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (256,)
    q = np.empty(256, dtype=np.int8)
    sc = ctypes.c_float()
    _load().orc_q8_block(x.ctypes.data, q.ctypes.data, ctypes.byref(sc))
    return q, np.float32(sc.value)


def q8_quantize(x: np.ndarray):
    """(codes int8 [M][K], scales f32 [M][K/256]) block by block."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    M, K = x.shape
    assert K % 256 == 0
    codes = np.empty((M, K), dtype=np.int8)
    scales = np.empty((M, K // 256), dtype=np.float32)
    for m in range(M):
        for b in range(K // 256):
            codes[m, b * 256:(b + 1) * 256], scales[m, b] = q8_block(x[m, b * 256:(b + 1) * 256])
    return codes, scales


def f16_round(x: np.ndarray) -> np.ndarray:
    """Each f32 rounded to the nearest binary16 value (ties to even), as f32."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    return np.array([lib.orc_f16_round(float(v)) for v in x.ravel()], dtype=np.float32).reshape(x.shape)


def gemv_a16q8(t: Tensor, x: np.ndarray, rows=None) -> np.ndarray:
    """y f32 [M][len(rows)] of the A16-Q8 contraction (NVFP4 only, K % 256 == 0);
    each value is the binary16-rounded total, widened to f32.  ``x`` is f32
    [M][K] (or [K])."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    M = x.shape[0]
    assert x.shape[1] == t.K
    rows = np.arange(t.N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    rows = np.ascontiguousarray(rows)
    y = np.empty((M, rows.size), dtype=np.float32)
    ct = _Tensor.from_buffer_copy(t._c())
    rc = _load().orc_gemv_a16q8_rows(ctypes.byref(ct), x.ctypes.data, M, rows.ctypes.data, rows.size,
                                     y.ctypes.data)
    if rc == 1:
        raise OracleError("a scale byte is a NaN encoding")
    if rc == 2:
        raise OracleError("the A16-Q8 contraction takes NVFP4 with K a multiple of 256")
    if rc:
        raise OracleError("out of memory")
    return y


def gemv_q4k_q8(t: Tensor, x: np.ndarray, rows=None) -> np.ndarray:
    """y f32 [M][len(rows)] of the Q4_K x Q8 contraction ([W4K] section 7):
    activations on the per-256 Q8 grid of :func:`q8_block`, exact integer
    sub-block sums, f32 epilogue per super-block.  ``x`` is f32 [M][K]."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    M = x.shape[0]
    assert x.shape[1] == t.K
    rows = np.arange(t.N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    rows = np.ascontiguousarray(rows)
    y = np.empty((M, rows.size), dtype=np.float32)
    ct = _Tensor.from_buffer_copy(t._c())
    rc = _load().orc_gemv_q4k_q8_rows(ctypes.byref(ct), x.ctypes.data, M, rows.ctypes.data, rows.size,
                                      y.ctypes.data)
    if rc == 2:
        raise OracleError("the Q4_K x Q8 contraction takes Q4_K with K a multiple of 256")
    if rc:
        raise OracleError("out of memory")
    return y


# ------------------------------------------------------ the NVFP4 quantizer

def e2m1_round(r: float) -> int:
    """Nearest E2M1 code (ties to the even code, saturating at 6, sign kept)."""
    return int(_load().orc_e2m1_round(float(r)))


def e4m3fn_round(v: float) -> int:
    """Nearest E4M3FN byte (ties to even, saturating at 448, sign kept)."""
    return int(_load().orc_e4m3fn_round(float(v)))


def quantize_nvfp4(W: np.ndarray):
    """(payload u8 [N][K/2], scales u8 [N][K/16], scale2 f32) of f32 W [N][K]."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % 16 == 0
    payload = np.empty((N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 16), dtype=np.uint8)
    s2 = ctypes.c_float()
    _load().orc_quantize_nvfp4(W.ctypes.data, N, K, payload.ctypes.data, scales.ctypes.data, ctypes.byref(s2))
    return payload, scales, np.float32(s2.value)


def quantize_nvfp4_groups(W: np.ndarray, scale2: float):
    """(payload, scales) of W [N][K] for a given tensor scale (the group rule of
    :func:`quantize_nvfp4`)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % 16 == 0
    payload = np.empty((N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 16), dtype=np.uint8)
    _load().orc_quantize_nvfp4_groups(W.ctypes.data, N, K, float(scale2), payload.ctypes.data, scales.ctypes.data)
    return payload, scales


def gemv_w4a4(t: Tensor, x: np.ndarray, input_scale_inv: float, rows=None) -> np.ndarray:
    """y f32 [M][len(rows)] of the W4A4 contraction ([MUS7] 7.4.3): x quantized
    to NVFP4 per 16 with tensor scale 1/input_scale_inv, exact per-group
    integer products, the f32 epilogue per group in order, binary16 output."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    M = x.shape[0]
    assert x.shape[1] == t.K
    rows = np.arange(t.N, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    rows = np.ascontiguousarray(rows)
    y = np.empty((M, rows.size), dtype=np.float32)
    ct = _Tensor.from_buffer_copy(t._c())
    rc = _load().orc_gemv_w4a4_rows(ctypes.byref(ct), x.ctypes.data, M, float(input_scale_inv), rows.ctypes.data,
                                    rows.size, y.ctypes.data)
    if rc == 1:
        raise OracleError("a scale byte is a NaN encoding")
    if rc == 2:
        raise OracleError("W4A4 takes NVFP4 weights and a finite input_scale_inv > 0")
    if rc:
        raise OracleError("out of memory")
    return y


# ------------------------------------------------------------ the Q4_K fit

def f16_bits(v: float) -> int:
    """binary16 encoding of f32 v rounded to nearest, ties to even."""
    return int(_load().orc_f16_bits(float(v)))


def quantize_q4k(W: np.ndarray) -> np.ndarray:
    """Q4_K super-blocks u8 [N][K/256][144] of f32 W [N][K] by the per-sub-block
    min/max fit of q4_oracle.c (orc_quantize_q4k)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert K % 256 == 0
    out = np.empty((N, K // 256, 144), dtype=np.uint8)
    _load().orc_quantize_q4k(W.ctypes.data, N, K, out.ctypes.data)
    return out
