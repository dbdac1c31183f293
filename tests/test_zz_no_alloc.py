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
    """A copy of `layer` with `n_bad` NaN scale encodings at random places."""
    bad = dict(layer)
    rng = np.random.default_rng(seed)
    if layer["fmt"] in ("nvfp4", "mxfp4"):
        s = layer["scales"].copy()
        idx = rng.choice(s.size, n_bad, replace=False)
        s.flat[idx] = 0xFF if layer["fmt"] == "mxfp4" else rng.choice([0x7F, 0xFF], n_bad)
        bad["scales"] = s
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


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "gptq"])
def test_no_alloc_validate_matches_validate_two_calls(fmt):
    N, K = (4099, 4096) if fmt != "gptq" else (4104, 4096)
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


def test_no_alloc_validate_rejects_oversize_without_launch():
    # more scale entries than the fixed scratch covers: rejected on the host
    big_n = 16384 * 16384 // (4096 // 16) + 16            # N * K/16 > 16384 * 16384
    rc, n = q4.q4_validate_noalloc("nvfp4", 0x10000, 0x20000, q4.make_aux(scale2=1.0, fmt="nvfp4"),
                                   big_n, 4096, stream=0)
    assert rc == q4.Q4_EDIM and n == -1
