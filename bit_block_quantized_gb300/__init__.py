"""Python binding of libq4.so: the same entry points as include/q4.h.

Argument marshalling only -- every step of decode, GEMV, dequant, repack and
validation runs in the library's CUDA kernels.  There is no CPU fallback: if
the shared library is missing, every call raises.

Pointer arguments accept torch tensors (their ``data_ptr()``), plain integers
(device addresses) or None.  ``stream`` defaults to torch's current stream.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libq4.so")

Q4_NVFP4, Q4_MXFP4, Q4_Q4K, Q4_Q40, Q4_GPTQ, Q4_AWQ, Q4_NVFP4_SPLITHALF, Q4_LOGICAL = range(1, 9)
FMT = {"nvfp4": Q4_NVFP4, "mxfp4": Q4_MXFP4, "q4k": Q4_Q4K, "q40": Q4_Q40, "gptq": Q4_GPTQ,
       "awq": Q4_AWQ, "nvfp4_splithalf": Q4_NVFP4_SPLITHALF, "logical": Q4_LOGICAL}
Q4_DT_F32, Q4_DT_BF16 = 0, 1
(Q4_OK, Q4_EINVAL, Q4_EDIM, Q4_EALIGN, Q4_ENAN, Q4_ESCALE2, Q4_ECUDA, Q4_EUNSUPPORTED,
 Q4_ERANGE, Q4_ETIMEOUT) = range(10)


class Aux(ctypes.Structure):
    """Mirror of ``q4_aux``."""
    _fields_ = [("scale2", ctypes.c_float), ("zeros", ctypes.c_void_p),
                ("g_idx", ctypes.c_void_p), ("group", ctypes.c_int32),
                ("x_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("flags", ctypes.c_uint32)]


Q4_FLAG_FP4_SLICES = 1


class GemvDesc(ctypes.Structure):
    """Mirror of ``q4_gemv_desc``."""
    _fields_ = [("fmt", ctypes.c_int), ("W_packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("aux", ctypes.POINTER(Aux)), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class Q4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({strerror(status)})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libq4.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with bit_block_quantized_gb300.build.build() "
                               "(or __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        AUXP = ctypes.POINTER(Aux)
        L.q4_gemv.argtypes = [I32, P, P, AUXP, P, P, I64, I64, I64, P]
        L.q4_dequant.argtypes = [I32, P, P, AUXP, P, I64, I64, P]
        L.q4_gemv_a16q8.argtypes = [P, P, AUXP, P, P, I64, I64, I64, P]
        L.q4_gemv_q4k_q8.argtypes = [P, AUXP, P, P, I64, I64, I64, P]
        L.q4_gemv_w4a4.argtypes = [P, P, AUXP, ctypes.c_float, P, P, I64, I64, I64, P]
        L.q4_gemv_w4a4_tc.argtypes = [P, P, AUXP, P, P, ctypes.c_float, P, I64, I64, I64, P]
        L.q4_quantize_nvfp4_scaled.argtypes = [P, I32, ctypes.c_float, P, P, I64, I64, P]
        L.q4_quantize_nvfp4.argtypes = [P, I32, P, P, P, I64, I64, P]
        L.q4_quantize_q4k.argtypes = [P, I32, P, I64, I64, P]
        L.q4_pack_bits.argtypes = [P, I64, I32, P, P]
        L.q4_unpack_bits.argtypes = [P, I64, I32, P, P]
        L.q4_permute_k.argtypes = [P, I32, P, P, I64, I64, P]
        L.q4_gemv_grouped.argtypes = [ctypes.POINTER(GemvDesc), I32, I64, P]
        L.q4_gemv_chain.argtypes = [ctypes.POINTER(GemvDesc), ctypes.POINTER(ctypes.c_int), I32, I64, P, P]
        L.q4_gemv_chain.restype = ctypes.c_int
        L.q4_repack.argtypes = [I32, P, P, AUXP, I32, P, P, P, P, I64, I64, P]
        L.q4_validate.argtypes = [I32, P, P, AUXP, I64, I64, P, P]
        L.q4_validate_noalloc.argtypes = [I32, P, P, AUXP, I64, I64, ctypes.POINTER(ctypes.c_int64), P]
        L.q4_validate_noalloc.restype = ctypes.c_int
        for f in ("q4_gemv", "q4_gemv_a16q8", "q4_gemv_grouped", "q4_dequant", "q4_repack", "q4_validate",
                  "q4_last_error", "q4_gemv_q4k_q8", "q4_gemv_w4a4", "q4_gemv_w4a4_tc", "q4_quantize_nvfp4_scaled", "q4_quantize_nvfp4", "q4_quantize_q4k", "q4_pack_bits", "q4_unpack_bits",
                  "q4_permute_k"):
            getattr(L, f).restype = ctypes.c_int
        L.q4_last_error.argtypes = []
        L.q4_set_wait_limit.argtypes = [I64]
        L.q4_set_wait_limit.restype = ctypes.c_int
        L.q4_strerror.restype = ctypes.c_char_p
        L.q4_last_gemv_path.restype = ctypes.c_char_p
        L.q4_strerror.argtypes = [I32]
        L.q4_packed_bytes.restype = ctypes.c_size_t
        L.q4_packed_bytes.argtypes = [I32, I64, I64]
        L.q4_version.restype = ctypes.c_char_p
        L.q4_version.argtypes = []
        _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _fmt(fmt):
    return FMT[fmt] if isinstance(fmt, str) else int(fmt)


def make_aux(scale2=0.0, zeros=None, g_idx=None, group=128, x_dtype=None, out_dtype=Q4_DT_F32,
             fmt=None, flags=0):
    """Build a ``q4_aux``.  x_dtype None picks the format default (bf16 for
    NVFP4/MXFP4, f32 otherwise); it may also be a torch dtype."""
    if x_dtype is None:
        x_dtype = Q4_DT_BF16 if _fmt(fmt or 0) in (Q4_NVFP4, Q4_MXFP4) else Q4_DT_F32
    elif not isinstance(x_dtype, int):
        import torch
        x_dtype = Q4_DT_BF16 if x_dtype == torch.bfloat16 else Q4_DT_F32
    if not isinstance(out_dtype, int):
        import torch
        out_dtype = Q4_DT_BF16 if out_dtype == torch.bfloat16 else Q4_DT_F32
    return Aux(float(scale2), _ptr(zeros), _ptr(g_idx), int(group), int(x_dtype), int(out_dtype), int(flags))


def _aux_ref(aux):
    return None if aux is None else ctypes.byref(aux)


def _check(rc: int, what: str):
    if rc != Q4_OK:
        raise Q4Error(rc, what)


# ------------------------------------------------------ the C entry points

def q4_gemv(fmt, W_packed, scales, aux, x, y, M, N, K, stream=None, check=True) -> int:
    rc = lib().q4_gemv(_fmt(fmt), _ptr(W_packed), _ptr(scales), _aux_ref(aux), _ptr(x), _ptr(y),
                       int(M), int(N), int(K), _stream(stream))
    if check:
        _check(rc, "q4_gemv")
    return rc


def q4_gemv_a16q8(W_packed, scales, aux, x, y, M, N, K, stream=None, check=True) -> int:
    """The integer-exact NVFP4 contraction with per-256 Q8 activations; y holds
    binary16-rounded values widened to f32."""
    rc = lib().q4_gemv_a16q8(_ptr(W_packed), _ptr(scales), _aux_ref(aux), _ptr(x), _ptr(y),
                             int(M), int(N), int(K), _stream(stream))
    if check:
        _check(rc, "q4_gemv_a16q8")
    return rc


def q4_gemv_q4k_q8(W_packed, aux, x, y, M, N, K, stream=None, check=True) -> int:
    """The Q4_K x Q8 (W4A8) contraction: exact integer sub-block sums, f32 y."""
    rc = lib().q4_gemv_q4k_q8(_ptr(W_packed), _aux_ref(aux), _ptr(x), _ptr(y), int(M), int(N), int(K),
                              _stream(stream))
    if check:
        _check(rc, "q4_gemv_q4k_q8")
    return rc


def q4_gemv_w4a4(W_packed, scales, aux, input_scale_inv, x, y, M, N, K, stream=None, check=True) -> int:
    """The integer-exact W4A4 contraction; y holds binary16 values widened to f32."""
    rc = lib().q4_gemv_w4a4(_ptr(W_packed), _ptr(scales), _aux_ref(aux), float(input_scale_inv), _ptr(x), _ptr(y),
                            int(M), int(N), int(K), _stream(stream))
    if check:
        _check(rc, "q4_gemv_w4a4")
    return rc


def q4_gemv_w4a4_tc(W_packed, scales, aux, xq, xs, x_scale2, y, M, N, K, stream=None, check=True) -> int:
    """W4A4 on the native block-scaled FP4 tensor cores; activations already NVFP4."""
    rc = lib().q4_gemv_w4a4_tc(_ptr(W_packed), _ptr(scales), _aux_ref(aux), _ptr(xq), _ptr(xs), float(x_scale2),
                               _ptr(y), int(M), int(N), int(K), _stream(stream))
    if check:
        _check(rc, "q4_gemv_w4a4_tc")
    return rc


def q4_quantize_nvfp4_scaled(x, x_dtype, scale2, payload, scales, M, K, stream=None, check=True) -> int:
    """NVFP4 groups of x [M][K] for a given tensor scale."""
    rc = lib().q4_quantize_nvfp4_scaled(_ptr(x), int(x_dtype), float(scale2), _ptr(payload), _ptr(scales), int(M),
                                        int(K), _stream(stream))
    if check:
        _check(rc, "q4_quantize_nvfp4_scaled")
    return rc


def q4_quantize_nvfp4(W, w_dtype, payload, scales, scale2, N, K, stream=None, check=True) -> int:
    """NVFP4 quantization of W [N][K]; scale2 is a device f32 word."""
    rc = lib().q4_quantize_nvfp4(_ptr(W), int(w_dtype), _ptr(payload), _ptr(scales), _ptr(scale2), int(N), int(K),
                                 _stream(stream))
    if check:
        _check(rc, "q4_quantize_nvfp4")
    return rc


def q4_quantize_q4k(W, w_dtype, out, N, K, stream=None, check=True) -> int:
    """Q4_K super-blocks [N][K/256][144] of W [N][K] by the min/max fit."""
    rc = lib().q4_quantize_q4k(_ptr(W), int(w_dtype), _ptr(out), int(N), int(K), _stream(stream))
    if check:
        _check(rc, "q4_quantize_q4k")
    return rc


def q4_pack_bits(codes, n, bits, words, stream=None, check=True) -> int:
    rc = lib().q4_pack_bits(_ptr(codes), int(n), int(bits), _ptr(words), _stream(stream))
    if check:
        _check(rc, "q4_pack_bits")
    return rc


def q4_unpack_bits(words, n, bits, codes, stream=None, check=True) -> int:
    rc = lib().q4_unpack_bits(_ptr(words), int(n), int(bits), _ptr(codes), _stream(stream))
    if check:
        _check(rc, "q4_unpack_bits")
    return rc


def q4_permute_k(x, x_dtype, perm, out, M, K, stream=None, check=True) -> int:
    rc = lib().q4_permute_k(_ptr(x), int(x_dtype), _ptr(perm), _ptr(out), int(M), int(K), _stream(stream))
    if check:
        _check(rc, "q4_permute_k")
    return rc


def q4_gemv_grouped(descs, M, stream=None, check=True) -> int:
    """``descs``: sequence of (fmt, W_packed, scales, aux, x, y, N, K) tuples."""
    arr = (GemvDesc * len(descs))()
    for i, (fmt, w, s, aux, x, y, N, K) in enumerate(descs):
        arr[i] = GemvDesc(_fmt(fmt), _ptr(w), _ptr(s), None if aux is None else ctypes.pointer(aux),
                          _ptr(x), _ptr(y), int(N), int(K))
    rc = lib().q4_gemv_grouped(arr, len(descs), int(M), _stream(stream))
    if check:
        _check(rc, "q4_gemv_grouped")
    return rc


def q4_gemv_chain(groups, M, sync=None, stream=None, check=True) -> int:
    """``groups``: sequence of groups, each a sequence of (fmt, W_packed,
    scales, aux, x, y, N, K) tuples; group g+1 runs after group g has written
    its outputs.  ``sync``: a device tensor of at least 2 uint32/int32 words,
    zero before its first use (required for more than one group)."""
    flat = [d for grp in groups for d in grp]
    arr = (GemvDesc * len(flat))()
    for i, (fmt, w, s, aux, x, y, N, K) in enumerate(flat):
        arr[i] = GemvDesc(_fmt(fmt), _ptr(w), _ptr(s), None if aux is None else ctypes.pointer(aux),
                          _ptr(x), _ptr(y), int(N), int(K))
    first = (ctypes.c_int * (len(groups) + 1))()
    for g, grp in enumerate(groups):
        first[g + 1] = first[g] + len(grp)
    rc = lib().q4_gemv_chain(arr, first, len(groups), int(M), _ptr(sync), _stream(stream))
    if check:
        _check(rc, "q4_gemv_chain")
    return rc


def q4_dequant(fmt, W_packed, scales, aux, out, N, K, stream=None, check=True) -> int:
    rc = lib().q4_dequant(_fmt(fmt), _ptr(W_packed), _ptr(scales), _aux_ref(aux), _ptr(out),
                          int(N), int(K), _stream(stream))
    if check:
        _check(rc, "q4_dequant")
    return rc


def q4_repack(src, src_w, src_scales, src_aux, dst, dst_w, dst_scales, dst_zeros, perm_out, N, K,
              stream=None, check=True) -> int:
    rc = lib().q4_repack(_fmt(src), _ptr(src_w), _ptr(src_scales), _aux_ref(src_aux), _fmt(dst),
                         _ptr(dst_w), _ptr(dst_scales), _ptr(dst_zeros), _ptr(perm_out),
                         int(N), int(K), _stream(stream))
    if check:
        _check(rc, "q4_repack")
    return rc


def q4_validate(fmt, W_packed, scales, aux, N, K, d_bad_count, stream=None) -> int:
    """Returns the status (Q4_OK, Q4_ENAN, Q4_ESCALE2, ...) without raising."""
    return lib().q4_validate(_fmt(fmt), _ptr(W_packed), _ptr(scales), _aux_ref(aux), int(N), int(K),
                             _ptr(d_bad_count), _stream(stream))


def q4_validate_noalloc(fmt, W_packed, scales, aux, N, K, stream=None):
    """The no-allocation scale scan: returns (status, count) with the count of
    NaN/Inf scale encodings read back into host memory."""
    n = ctypes.c_int64(-1)
    rc = lib().q4_validate_noalloc(_fmt(fmt), _ptr(W_packed), _ptr(scales), _aux_ref(aux), int(N), int(K),
                                   ctypes.byref(n), _stream(stream))
    return rc, int(n.value)


def q4_last_error() -> int:
    return lib().q4_last_error()


def q4_set_wait_limit(cycles: int) -> int:
    """Bounded-wait limit (SM clocks) of the TMA-fed kernels on the current
    device; cycles <= 0 restores the default (~1 s)."""
    return lib().q4_set_wait_limit(int(cycles))


def q4_last_gemv_path() -> str:
    """Kernel family of this thread's latest q4_gemv / q4_gemv_grouped call."""
    return lib().q4_last_gemv_path().decode()


def strerror(status: int) -> str:
    return lib().q4_strerror(int(status)).decode()


def q4_packed_bytes(fmt, N, K) -> int:
    return int(lib().q4_packed_bytes(_fmt(fmt), int(N), int(K)))


def version() -> str:
    return lib().q4_version().decode()
