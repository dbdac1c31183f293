"""The C-ABI library builds, loads and exports every symbol include/q4.h
declares; host-side argument checks reject bad calls before any launch.  No
GPU and no compute call."""
import ctypes
import json
import os
import re

import pytest

import bit_block_quantized_gb300 as q4
from bit_block_quantized_gb300 import build as q4build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    q4build.build()
    return q4.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "q4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("q4_gemv", "q4_dequant", "q4_repack", "q4_validate", "q4_last_error",
                     "q4_strerror", "q4_packed_bytes"):
        assert required in names


_LAYOUT_PROBE = r"""
#include <stdio.h>
#include <stddef.h>
#include "q4.h"
#define F(T, m) printf(#T " " #m " %zu\n", offsetof(T, m))
int main(void) {
    printf("q4_aux size %zu\n", sizeof(q4_aux));
    F(q4_aux, scale2); F(q4_aux, zeros); F(q4_aux, g_idx); F(q4_aux, group); F(q4_aux, x_dtype);
    F(q4_aux, out_dtype); F(q4_aux, flags);
    printf("q4_gemv_desc size %zu\n", sizeof(q4_gemv_desc));
    F(q4_gemv_desc, fmt); F(q4_gemv_desc, W_packed); F(q4_gemv_desc, scales); F(q4_gemv_desc, aux);
    F(q4_gemv_desc, x); F(q4_gemv_desc, y); F(q4_gemv_desc, N); F(q4_gemv_desc, K);
    return 0;
}
"""


def test_binding_structs_match_the_header(tmp_path):
    """The ctypes mirrors of q4_aux and q4_gemv_desc have the C layout (a C
    probe built against include/q4.h prints sizes and offsets)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src, exe = tmp_path / "layout.c", tmp_path / "layout"
    src.write_text(_LAYOUT_PROBE)
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    c = {}
    for line in subprocess.check_output([str(exe)], text=True).splitlines():
        t, m, v = line.split()
        c[(t, m)] = int(v)
    for T, name in ((q4.Aux, "q4_aux"), (q4.GemvDesc, "q4_gemv_desc")):
        assert ctypes.sizeof(T) == c[(name, "size")], name
        for field, _ in T._fields_:
            assert getattr(T, field).offset == c[(name, field)], (name, field)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_targets_sm103a_only():
    log = open(os.path.join(q4build.BUILD, "ptxas.log")).read() if os.path.exists(
        os.path.join(q4build.BUILD, "ptxas.log")) else ""
    assert "sm_103a" in " ".join(q4build.ARCH)
    if log:
        assert "for 'sm_103a'" in log


def test_packed_bytes_match_the_pages_arithmetic(lib):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "worked_examples.json")))["bytes"]
    N = K = 4096
    assert q4.q4_packed_bytes("nvfp4", N, K) - 4 == N * K * g["nvfp4_bits_per_weight"] / 8
    assert q4.q4_packed_bytes("mxfp4", N, K) == N * K * g["mxfp4_bits_per_weight"] / 8
    assert q4.q4_packed_bytes("mxfp4", 1, 32) == g["mxfp4_block_bytes"]
    assert q4.q4_packed_bytes("q4k", 1, 256) == g["q4k_block_bytes"]
    assert q4.q4_packed_bytes("q4k", N, K) == N * K * g["q4k_bits_per_weight"] / 8
    assert 7e9 * q4.q4_packed_bytes("q4k", 1, 256) / 256 / 1e9 == g["q4k_7b_gb"]
    assert q4.q4_packed_bytes("q40", 1, 32) == 18
    assert q4.q4_packed_bytes("gptq", 8, 128) == 8 * 64 + 8 * 2 + 4
    assert q4.q4_packed_bytes("nvfp4", 4, 15) == 0          # not a block multiple


def test_strerror_and_version(lib):
    assert q4.strerror(q4.Q4_OK) == "ok"
    assert "aligned" in q4.strerror(q4.Q4_EALIGN)
    assert "sm_103a" in q4.version()


# Fake, 16-byte aligned "device" addresses: every call below is rejected on
# the host before anything touches CUDA.
A, B, C, D = 0x10000, 0x20000, 0x30000, 0x40000


def gemv(fmt, aux, M=1, N=64, K=64, w=A, s=B, x=C, y=D):
    return q4.q4_gemv(fmt, w, s, aux, x, y, M, N, K, stream=0, check=False)


def test_host_side_rejections(lib):
    nv = q4.make_aux(scale2=0.5, fmt="nvfp4")
    assert gemv("nvfp4", nv, N=0) == q4.Q4_EDIM
    assert gemv("nvfp4", nv, K=40) == q4.Q4_EDIM
    assert gemv("nvfp4", nv, M=0) == q4.Q4_EDIM
    assert gemv("q4k", None, K=128) == q4.Q4_EDIM
    assert gemv("mxfp4", None, K=48) == q4.Q4_EDIM
    assert gemv("nvfp4", nv, w=0) == q4.Q4_EINVAL
    assert gemv("nvfp4", nv, w=A + 8) == q4.Q4_EALIGN
    assert gemv("nvfp4", nv, y=D + 4) == q4.Q4_EALIGN
    assert gemv("nvfp4", None) == q4.Q4_EINVAL                # NVFP4 needs scale2
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert gemv("nvfp4", q4.make_aux(scale2=bad, fmt="nvfp4")) == q4.Q4_ESCALE2
    assert gemv(99, None) == q4.Q4_EINVAL
    assert gemv("gptq", None, K=128) == q4.Q4_EINVAL          # zeros required
    gp = q4.make_aux(zeros=A, group=128)
    assert gemv("gptq", gp, N=12, K=128) == q4.Q4_EDIM        # N % 8
    assert gemv("gptq", gp, N=16, K=192) == q4.Q4_EDIM        # K % group
    assert gemv("nvfp4_splithalf", nv) == q4.Q4_EUNSUPPORTED
    assert gemv("logical", q4.make_aux(zeros=A), K=128) == q4.Q4_EUNSUPPORTED
    bad_dtype = q4.make_aux(scale2=1.0, x_dtype=7, fmt="nvfp4")
    assert gemv("nvfp4", bad_dtype) == q4.Q4_EINVAL
    assert q4.q4_dequant("q4k", A, None, None, B, 4, 100, stream=0, check=False) == q4.Q4_EDIM
    assert q4.q4_dequant("q40", A, None, None, 0, 4, 64, stream=0, check=False) == q4.Q4_EINVAL
    assert q4.q4_repack("q4k", A, None, None, "gptq", B, C, D, None, 8, 256, stream=0,
                        check=False) == q4.Q4_EUNSUPPORTED
    assert q4.q4_repack("gptq", A, B, q4.make_aux(zeros=C), "awq", B, C, D, None, 12, 256,
                        stream=0, check=False) == q4.Q4_EDIM
    assert q4.q4_validate("nvfp4", A, B, nv, 4, 64, 0, stream=0) == q4.Q4_EINVAL
    good = ("nvfp4", A, B, nv, C, D, 64, 64)
    assert q4.q4_gemv_grouped([good, ("nvfp4", A, B, nv, C, D + 4, 64, 64)], 1, stream=0,
                              check=False) == q4.Q4_EALIGN      # nothing launched
    assert q4.q4_gemv_grouped([good], 0, stream=0, check=False) == q4.Q4_EDIM
    assert q4.q4_gemv_grouped([], 1, stream=0, check=False) == q4.Q4_EINVAL
    # chains: a group barrier needs the caller's sync words; every member is
    # checked before anything is launched
    chain = q4.q4_gemv_chain
    assert chain([[good], [good]], 1, sync=None, stream=0, check=False) == q4.Q4_EINVAL
    assert chain([[good], [good]], 1, sync=0x50004, stream=0, check=False) == q4.Q4_EALIGN
    assert chain([[good], [("nvfp4", A, B, nv, C, D + 4, 64, 64)]], 1, sync=0x50000, stream=0,
                 check=False) == q4.Q4_EALIGN
    assert chain([[good]], 0, stream=0, check=False) == q4.Q4_EDIM
    assert chain([], 1, stream=0, check=False) == q4.Q4_EINVAL
    assert chain([[good], []], 1, sync=0x50000, stream=0, check=False) == q4.Q4_EINVAL


def test_a16q8_host_side_rejections(lib):
    nv = q4.make_aux(scale2=0.5, fmt="nvfp4")

    def call(aux=nv, M=1, N=64, K=256, w=A, s=B, x=C, y=D):
        return q4.q4_gemv_a16q8(w, s, aux, x, y, M, N, K, stream=0, check=False)

    assert call(K=128) == q4.Q4_EDIM                  # K % 256
    assert call(K=200_704) == q4.Q4_EDIM              # one row of codes exceeds the budget
    assert call(M=0) == q4.Q4_EDIM
    assert call(N=0) == q4.Q4_EDIM
    assert call(aux=None) == q4.Q4_EINVAL             # scale2 lives in aux
    assert call(aux=q4.make_aux(scale2=0.0, fmt="nvfp4")) == q4.Q4_ESCALE2
    assert call(aux=q4.make_aux(scale2=1.0, x_dtype=7, fmt="nvfp4")) == q4.Q4_EINVAL
    assert call(x=0) == q4.Q4_EINVAL
    assert call(x=C + 2) == q4.Q4_EALIGN
    assert call(s=B + 8) == q4.Q4_EALIGN
