"""q4_validate_noalloc -- the scale scan for callers that cannot allocate
device memory (a loader inside a pool-managed serving process, a plugin that
is handed tensors but no allocator) -- must agree with q4_validate, which
needs a caller-allocated count buffer.

Kept in a file of its own, collected last, so that a run stopping at the
first failure has already run every other test.  It passes alone in a fresh
process and after the rest of the suite.
"""
import numpy as np
import pytest

import synth
from _helpers import aux_for, to_device

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def with_nans(layer, n_bad, seed):
    """A copy of `layer` with `n_bad` NaN/Inf scale encodings at random places:
    E4M3FN 0x7f/0xff or E8M0 0xff in the FP4 scale bytes, fp16 NaN/Inf in the
    d / dmin header of Q4_K super-blocks and the d of Q4_0 blocks (inside the
    weight bytes), and in the fp16 scales of GPTQ, AWQ and the logical form."""
    bad = dict(layer)
    rng = np.random.default_rng(seed)
    fmt = layer["fmt"]
    if fmt in ("nvfp4", "mxfp4"):
        s = layer["scales"].copy()
        idx = rng.choice(s.size, n_bad, replace=False)
        s.flat[idx] = 0xFF if fmt == "mxfp4" else rng.choice([0x7F, 0xFF], n_bad)
        bad["scales"] = s
    elif fmt in ("q4k", "q40"):
        stride, per = (144, 2) if fmt == "q4k" else (18, 1)
        w = layer["w"].copy().reshape(-1)
        n_entries = w.size // stride * per
        for i in rng.choice(n_entries, n_bad, replace=False):
            off = (i // per) * stride + 2 * (i % per)                 # d (and dmin) of the block
            w[off:off + 2] = np.array([rng.choice([0x7E00, 0x7C00, 0xFC01])], np.uint16).view(np.uint8)
        bad["w"] = w.reshape(layer["w"].shape)
    else:
        s = layer["scales"].copy()
        idx = rng.choice(s.size, n_bad, replace=False)
        s.flat[idx] = np.array([np.float16(np.nan)]).view(np.uint16)[0]
        bad["scales"] = s
    return bad


def both(layer):
    d = to_device(layer)
    aux = aux_for(layer, d)
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    ref_rc = q4.q4_validate(layer["fmt"], d["w"], d["scales"], aux, layer["N"], layer["K"], cnt)
    rc, n = q4.q4_validate_noalloc(layer["fmt"], d["w"], d["scales"], aux, layer["N"], layer["K"])
    return (ref_rc, int(cnt[0])), (rc, n)


SHAPES = {"nvfp4": (4099, 4096), "mxfp4": (4099, 4096), "gptq": (4104, 4096), "awq": (4104, 4096),
          "logical": (1032, 1024), "q4k": (4099, 4096), "q40": (4099, 4096)}


@pytest.mark.parametrize("fmt", sorted(SHAPES))
def test_no_alloc_validate_matches_validate_two_calls(fmt):
    N, K = SHAPES[fmt]
    clean = synth.make_layer(fmt, N, K, config=40, matrix=1)
    dirty = with_nans(clean, 37, seed=3)
    # two calls in a row, dirty then clean: the second must not see the first's counts
    first_ref, first = both(dirty)
    second_ref, second = both(clean)
    assert first == first_ref == (q4.Q4_ENAN, 37)
    assert second == second_ref == (q4.Q4_OK, 0)
    # and the other order, with a different count
    third_ref, third = both(with_nans(clean, 5, seed=4))
    assert third == third_ref == (q4.Q4_ENAN, 5)


@pytest.mark.parametrize("N", [1048000, 1048576])
def test_no_alloc_validate_near_the_scratch_limit(N):
    """NVFP4 scale tensors of N x 256 bytes (K = 4096): 16375 chunks (not a
    power of two, the last one partial) and exactly the 16384-chunk limit,
    with NaN encodings in the first and last chunk and in between.  Only the
    scale bytes are read, so the payload pointer is a small placeholder."""
    K = 4096
    scales = torch.full((N, K // 16), 0x38, dtype=torch.uint8, device="cuda")
    flat = scales.view(-1)
    bad_at = torch.tensor([0, 1, 16383, 16384, flat.numel() // 2, flat.numel() - 16385, flat.numel() - 1])
    flat[bad_at.cuda()] = torch.tensor([0x7F, 0xFF, 0x7F, 0xFF, 0x7F, 0xFF, 0x7F], dtype=torch.uint8,
                                       device="cuda")
    w = torch.zeros(16, dtype=torch.uint8, device="cuda")
    aux = q4.make_aux(scale2=1.0, fmt="nvfp4")
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    for _ in range(2):
        ref_rc = q4.q4_validate("nvfp4", w, scales, aux, N, K, cnt)
        rc, n = q4.q4_validate_noalloc("nvfp4", w, scales, aux, N, K)
        assert (rc, n) == (ref_rc, int(cnt[0])) == (q4.Q4_ENAN, bad_at.numel())
    flat[bad_at.cuda()] = 0x38
    assert q4.q4_validate_noalloc("nvfp4", w, scales, aux, N, K) == (q4.Q4_OK, 0)
    del scales
    torch.cuda.empty_cache()


def test_no_alloc_validate_takes_the_same_argument_checks():
    """The host-side checks are q4_validate's own: a misaligned zeros or
    g_idx pointer, a g_idx on a format without one, and a bad scale2."""
    layer = synth.make_layer("gptq", 264, 1024, config=40, matrix=2)
    d = to_device(layer)
    base = dict(zeros=d["zeros"], group=128, fmt="gptq")
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    gi = torch.zeros(1024 + 4, dtype=torch.int32, device="cuda")
    cases = [q4.make_aux(zeros=d["zeros"].data_ptr() + 4, group=128, fmt="gptq"),      # misaligned zeros
             q4.make_aux(g_idx=gi.data_ptr() + 4, **base)]                               # misaligned g_idx
    for aux in cases:
        want = q4.q4_validate("gptq", d["w"], d["scales"], aux, 264, 1024, cnt)
        assert want == q4.Q4_EALIGN
        assert q4.q4_validate_noalloc("gptq", d["w"], d["scales"], aux, 264, 1024)[0] == want
    awq = synth.make_layer("awq", 264, 1024, config=40, matrix=3)
    da = to_device(awq)
    aux = q4.make_aux(zeros=da["zeros"], g_idx=gi, group=128, fmt="awq")       # AWQ takes no g_idx
    want = q4.q4_validate("awq", da["w"], da["scales"], aux, 264, 1024, cnt)
    assert want == q4.Q4_EINVAL
    assert q4.q4_validate_noalloc("awq", da["w"], da["scales"], aux, 264, 1024)[0] == want
    nv = synth.make_layer("nvfp4", 64, 256, config=40, matrix=4)
    dn = to_device(nv)
    aux = q4.make_aux(scale2=float("inf"), fmt="nvfp4")
    want = q4.q4_validate("nvfp4", dn["w"], dn["scales"], aux, 64, 256, cnt)
    assert want == q4.Q4_ESCALE2
    assert q4.q4_validate_noalloc("nvfp4", dn["w"], dn["scales"], aux, 64, 256) == (q4.Q4_ESCALE2, 0)


def test_no_alloc_validate_rejects_oversize_without_launch():
    # more scale entries than the fixed scratch covers: rejected on the host
    big_n = 16384 * 16384 // (4096 // 16) + 16            # N * K/16 > 16384 * 16384
    rc, n = q4.q4_validate_noalloc("nvfp4", 0x10000, 0x20000, q4.make_aux(scale2=1.0, fmt="nvfp4"),
                                   big_n, 4096, stream=0)
    assert rc == q4.Q4_EDIM and n == -1
