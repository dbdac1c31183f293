"""The TMA-fed NVFP4 decode-GEMV (batch 1..4, bf16 x, K % 256 == 0) through
the C ABI, against the CPU oracle: |y_gpu - y_ref| <= 1e-5 * sum|w||x| + 1e-6.

Shapes cover one 256-k chunk (7 of the 8 decode warps idle), a last stage
with only some chunks inside K, ragged 16-row tiles, more tiles than CTAs
(the ring wraps and the double-buffered tile reduction alternates), the
grouped launch over members that share x, the f32 fallback for activations
whose range defeats the f16 staging, and stream-order hazards against the
launch before (the next GEMV's weight prefetch runs before its dependency
wait).
"""
import numpy as np
import pytest

import oracle
import synth

from _helpers import aux_for, oracle_gemv_all_rows, to_device, to_oracle, within_tolerance, x_device

torch = pytest.importorskip("torch")
q4 = pytest.importorskip("bit_block_quantized_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_block_quantized_gb300 import build
    build.build()
    q4.lib()


def gemv(layer, d, x, M, y=None):
    N, K = layer["N"], layer["K"]
    if y is None:
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    aux = aux_for(layer, d, x_dtype=torch.bfloat16)
    assert q4.q4_gemv(layer["fmt"], d["w"], d["scales"], aux, x, y, M, N, K) == q4.Q4_OK
    return y


def tma_fits(K, M):
    """The kernel's shared-memory rule: the staged x (2 bytes per k and batch
    column, K rounded up to 2048-k stages), the partial sums and the fixed
    areas leave room for at least 3 ring stages of 18 KB in 112 KB."""
    mt = 1 if M == 1 else 2 if M == 2 else 4
    nst = -(-K // 2048)
    fixed = 1024 + 144 + 2 * 8 * 16 * mt * 4 + 8 * nst * 2 * 8 * mt * 4 * 8
    return (112 * 1024 - fixed) // 18432 >= 3


def expected_path(K, M):
    """Batch 1..4 runs on the TMA-fed kernel when its ring fits, else on the
    register-fed one (the FP4 tensor-core path is opt-in, tested apart)."""
    return "gemv_tma" if tma_fits(K, M) else "gemv_mma"


def check(layer, M, config, rows=None):
    d = to_device(layer)
    xbits, xf = synth.draw_x(M, layer["K"], config=config, matrix=5)
    y = gemv(layer, d, x_device(xbits), M)
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    assert q4.q4_last_gemv_path() == expected_path(layer["K"], M)
    yc = y.cpu().numpy()
    if rows is None:
        ref, bound = oracle_gemv_all_rows(to_oracle(layer), xf)
    else:
        ref, bound = oracle.gemv(to_oracle(layer), xf, rows=rows)
        yc = yc[:, rows]
    ok, worst = within_tolerance(yc, ref, bound)
    assert ok, f"worst error / tolerance = {worst}"


SHAPES = [(45, 4096), (16, 256), (7, 11008), (1, 2048), (300, 6144), (263, 14336), (33, 2304)]


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", SHAPES)
def test_tma_gemv_matches_oracle(N, K, M):
    check(synth.make_layer("nvfp4", N, K, config=50, matrix=M, row_scale=True), M, config=50 + M)


@pytest.mark.parametrize("M", [1, 4])
def test_tma_gemv_many_tiles_per_cta(M):
    """4099 rows = 257 tiles: more tiles than CTAs, a ragged last tile."""
    check(synth.make_layer("nvfp4", 4099, 4096, config=51, matrix=M, outliers=True), M, config=51)


def test_tma_gemv_wide_dynamic_range_x_falls_back_to_f32():
    N, K = 40, 6144
    layer = synth.make_layer("nvfp4", N, K, config=52, matrix=0)
    d = to_device(layer)
    for M in (1, 3):
        xf = np.random.default_rng(M).normal(0, 1e-10, (M, K)).astype(np.float32)
        xf[:, 7] = 1e30
        xf[:, 5000] = -3e20
        xbits = synth.f32_to_bf16_bits(xf)
        xr = oracle.bf16_bits_to_f32(xbits).reshape(M, K)
        y = gemv(layer, d, x_device(xbits), M).cpu().numpy()
        assert q4.q4_last_gemv_path() == expected_path(K, M)
        ref, bound = oracle.gemv(to_oracle(layer), xr)
        ok, worst = within_tolerance(y, ref, bound)
        assert ok, worst


def test_tma_gemv_one_hot_gives_exact_column():
    layer = synth.make_layer("nvfp4", 48, 4096, config=53, matrix=1)
    d = to_device(layer)
    ref = oracle.dequant(to_oracle(layer))
    for k in (0, 255, 256, 2047, 2048, 4095):
        x = torch.zeros((1, 4096), dtype=torch.bfloat16, device="cuda")
        x[0, k] = 1.0
        y = gemv(layer, d, x, 1).cpu().numpy()[0]
        assert np.array_equal(y, ref[:, k])


def test_tma_gemv_deterministic():
    layer = synth.make_layer("nvfp4", 1029, 14336, config=54, matrix=0)
    d = to_device(layer)
    xbits, _ = synth.draw_x(2, 14336, config=54, matrix=3)
    x = x_device(xbits)
    y0 = gemv(layer, d, x, 2).clone()
    for _ in range(3):
        assert torch.equal(gemv(layer, d, x, 2), y0)


@pytest.mark.parametrize("M", [1, 3])
def test_tma_grouped_shared_x(M):
    """Members that read the same x (gate/up, q/k/v) run as one TMA launch;
    a member with its own x sends the group to the register-fed kernels."""
    K = 4096
    layers = [synth.make_layer("nvfp4", N, K, config=55, matrix=i, row_scale=True)
              for i, N in enumerate((300, 17, 1024))]
    xb, xf = synth.draw_x(M, K, config=55, matrix=9)
    x = x_device(xb)
    devs = [to_device(L) for L in layers]
    ys = [torch.full((M, L["N"]), float("nan"), device="cuda") for L in layers]
    descs = [("nvfp4", d["w"], d["scales"], aux_for(L, d, x_dtype=torch.bfloat16), x, y, L["N"], K)
             for L, d, y in zip(layers, devs, ys)]
    assert q4.q4_gemv_grouped(descs, M) == q4.Q4_OK
    assert q4.q4_last_gemv_path() == "gemv_tma_group"
    torch.cuda.synchronize()
    for L, y in zip(layers, ys):
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst
    xb2, xf2 = synth.draw_x(M, K, config=55, matrix=10)
    x2 = x_device(xb2)
    descs[1] = descs[1][:4] + (x2,) + descs[1][5:]
    ys[1].fill_(float("nan"))
    assert q4.q4_gemv_grouped(descs, M) == q4.Q4_OK
    assert q4.q4_last_gemv_path() not in ("gemv_tma_group", "gemv_fp4tc_group")
    torch.cuda.synchronize()
    ref, bound = oracle.gemv(to_oracle(layers[1]), xf2)
    ok, worst = within_tolerance(ys[1].cpu().numpy(), ref, bound)
    assert ok, worst


@pytest.mark.parametrize("M", [1, 4])
def test_tma_grouped_mxfp4_shared_x(M):
    """MXFP4 members sharing x run as one TMA launch as well: each lane's scale
    word (loaded one stage ahead) comes from its tile's member, and a member
    whose scales leave the exact f16 range takes those stages in f32 with its
    own rows and scales.  Every row against the oracle, bit for bit equal to
    the members' own calls; a group mixing NVFP4 and MXFP4 runs per member."""
    K = 4096
    layers = [synth.make_layer("mxfp4", N, K, config=57, matrix=i, outliers=True)
              for i, N in enumerate((1000, 17, 2048, 300))]
    s = layers[2]["scales"].copy()
    s[5, 3] = 127 - 40                                  # 2^-40: that stage goes to the f32 path
    s[1500, :] = 127 + 20
    layers[2] = dict(layers[2], scales=s)
    xb, xf = synth.draw_x(M, K, config=57, matrix=9)
    x = x_device(xb)
    devs = [to_device(L) for L in layers]
    ys = [torch.full((M, L["N"]), float("nan"), device="cuda") for L in layers]
    descs = [("mxfp4", d["w"], d["scales"], aux_for(L, d, x_dtype=torch.bfloat16), x, y, L["N"], K)
             for L, d, y in zip(layers, devs, ys)]
    assert q4.q4_gemv_grouped(descs, M) == q4.Q4_OK
    assert q4.q4_last_gemv_path() == "gemv_tma_group"
    torch.cuda.synchronize()
    for L, d, y in zip(layers, devs, ys):
        got = y.cpu().numpy()
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(got, ref, bound)
        assert ok, worst
        single = gemv(L, d, x, M).cpu().numpy()
        assert np.array_equal(single.view(np.uint32), got.view(np.uint32))
    nv = synth.make_layer("nvfp4", 64, K, config=57, matrix=8)
    dn = to_device(nv)
    yn = torch.full((M, 64), float("nan"), device="cuda")
    mixed = [descs[0], ("nvfp4", dn["w"], dn["scales"], aux_for(nv, dn, x_dtype=torch.bfloat16), x, yn, 64, K)]
    assert q4.q4_gemv_grouped(mixed, M) == q4.Q4_OK
    assert q4.q4_last_gemv_path() != "gemv_tma_group"
    torch.cuda.synchronize()
    ref, bound = oracle.gemv(to_oracle(nv), xf)
    ok, worst = within_tolerance(yn.cpu().numpy(), ref, bound)
    assert ok, worst
    assert q4.q4_last_error() == q4.Q4_OK


def test_tma_chain_same_output_buffer():
    """Back-to-back launches overlap (programmatic dependent launch): each
    writes y only after the previous one has finished, so the last one wins."""
    K = 4096
    a = synth.make_layer("nvfp4", 2048, K, config=56, matrix=0)
    b = synth.make_layer("nvfp4", 2048, K, config=56, matrix=1)
    da, db = to_device(a), to_device(b)
    xb, _ = synth.draw_x(1, K, config=56, matrix=2)
    x = x_device(xb)
    want_a, want_b = gemv(a, da, x, 1).clone(), gemv(b, db, x, 1).clone()
    y = torch.empty((1, 2048), dtype=torch.float32, device="cuda")
    for last in (a, b, a):
        for L, dd in ((a, da), (b, db)) * 5:
            gemv(L, dd, x, 1, y)
        gemv(last, da if last is a else db, x, 1, y)
        torch.cuda.synchronize()
        assert torch.equal(y, want_a if last is a else want_b)


def test_tma_chain_reads_x_written_by_the_launch_before():
    """GEMV B reads the x that GEMV A, the launch just before it, writes: B's
    activation read waits for A.  A takes a one-hot x and scale2 = 1, so its
    f32 outputs are e2m1 * e4m3 products (at most 6 significant bits) whose
    low 16 bits are zero; B reads those bytes as bf16 pairs (0, y_A[n])."""
    N = 2048
    a = dict(synth.make_layer("nvfp4", N, 4096, config=57, matrix=0), scale2=1.0)
    b = synth.make_layer("nvfp4", 512, 2 * N, config=57, matrix=1)
    da, db = to_device(a), to_device(b)
    x = torch.zeros((1, 4096), dtype=torch.bfloat16, device="cuda")
    x[0, 5] = 1.0
    ya = torch.empty((1, N), dtype=torch.float32, device="cuda")
    yb = torch.empty((1, 512), dtype=torch.float32, device="cuda")
    xb_view = ya.view(torch.bfloat16)
    # reference: the two launches separated by a host synchronisation
    gemv(a, da, x, 1, ya)
    torch.cuda.synchronize()
    assert (ya.view(torch.int32) & 0xFFFF).eq(0).all().item()
    assert ya.abs().sum().item() > 0
    gemv(b, db, xb_view, 1, yb)
    torch.cuda.synchronize()
    want = yb.clone()
    ref, bound = oracle.gemv(to_oracle(b), xb_view.float().cpu().numpy())
    ok, worst = within_tolerance(want.cpu().numpy(), ref, bound)
    assert ok, worst
    for _ in range(5):
        ya.zero_()
        yb.fill_(float("nan"))
        gemv(a, da, x, 1, ya)
        gemv(b, db, xb_view, 1, yb)
        torch.cuda.synchronize()
        assert torch.equal(yb, want)


def test_tma_weights_written_by_the_launch_before():
    """Weights overwritten by an ordinary kernel on the same stream just
    before the GEMV: the GEMV sees the new weights."""
    K = 4096
    a = synth.make_layer("nvfp4", 1024, K, config=58, matrix=0)
    b = synth.make_layer("nvfp4", 1024, K, config=58, matrix=1)
    da, db = to_device(a), to_device(b)
    xb, _ = synth.draw_x(1, K, config=58, matrix=2)
    x = x_device(xb)
    want_b = gemv(b, db, x, 1).clone()
    w = da["w"].clone()
    s = da["scales"].clone()
    dw = dict(da, w=w, scales=s)
    y = torch.empty((1, 1024), dtype=torch.float32, device="cuda")
    for _ in range(3):
        w.copy_(da["w"])
        s.copy_(da["scales"])
        gemv(a, dw, x, 1, y)
        w.copy_(db["w"])
        s.copy_(db["scales"])
        gemv(b, dw, x, 1, y)
        torch.cuda.synchronize()
        assert torch.equal(y, want_b)


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_tma_full_size_every_row(N, K):
    """The 4096 x 14336 MLP set's two shapes at batch 1 to 4, every row."""
    layer = synth.make_layer("nvfp4", N, K, config=5, matrix=0, row_scale=True)
    for M in (1, 2, 3, 4):
        check(layer, M, config=5)


# ------------------------------------------------------------------ chains

def chain_member(layer, d, x, y):
    return ("nvfp4", d["w"], d["scales"], aux_for(layer, d, x_dtype=torch.bfloat16), x, y, layer["N"], layer["K"])


def sync_words():
    return torch.zeros(2, dtype=torch.int32, device="cuda")


def test_chain_matches_oracle():
    """gate + up (one x), then down (its own x), as one launch."""
    gate = synth.make_layer("nvfp4", 300, 4096, config=60, matrix=0, row_scale=True)
    up = synth.make_layer("nvfp4", 17, 4096, config=60, matrix=1, row_scale=True)
    down = synth.make_layer("nvfp4", 263, 14336, config=60, matrix=2, row_scale=True)
    xb0, xf0 = synth.draw_x(1, 4096, config=60, matrix=3)
    xb1, xf1 = synth.draw_x(1, 14336, config=60, matrix=4)
    x0, x1 = x_device(xb0), x_device(xb1)
    ds = [to_device(L) for L in (gate, up, down)]
    ys = [torch.full((1, L["N"]), float("nan"), device="cuda") for L in (gate, up, down)]
    sync = sync_words()
    q4.q4_gemv_chain([[chain_member(gate, ds[0], x0, ys[0]), chain_member(up, ds[1], x0, ys[1])],
                      [chain_member(down, ds[2], x1, ys[2])]], 1, sync=sync)
    assert q4.q4_last_gemv_path() == "gemv_tma_chain"
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    for L, xf, y in ((gate, xf0, ys[0]), (up, xf0, ys[1]), (down, xf1, ys[2])):
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst
    assert sync.cpu().tolist() == [0, 1]          # count reset, one barrier passed


@pytest.mark.parametrize("M", [1, 2, 4])
def test_chain_three_groups_of_different_K(M):
    Ks = (2048, 4096, 6144) if M < 4 else (2048, 4096, 4096)
    layers = [synth.make_layer("nvfp4", N, K, config=61, matrix=i, outliers=True)
              for i, (N, K) in enumerate(zip((129, 64, 40), Ks))]
    xs = [synth.draw_x(M, L["K"], config=61, matrix=10 + i) for i, L in enumerate(layers)]
    ds = [to_device(L) for L in layers]
    ys = [torch.full((M, L["N"]), float("nan"), device="cuda") for L in layers]
    xd = [x_device(b) for b, _ in xs]
    sync = sync_words()
    q4.q4_gemv_chain([[chain_member(L, d, x, y)] for L, d, x, y in zip(layers, ds, xd, ys)], M, sync=sync)
    assert q4.q4_last_gemv_path() == "gemv_tma_chain"
    torch.cuda.synchronize()
    assert q4.q4_last_error() == q4.Q4_OK
    for L, (_, xf), y in zip(layers, xs, ys):
        ref, bound = oracle.gemv(to_oracle(L), xf)
        ok, worst = within_tolerance(y.cpu().numpy(), ref, bound)
        assert ok, worst


def test_chain_later_group_reads_an_earlier_groups_output():
    """Group 1's x is a bf16 view of group 0's f32 y, inside one launch (the
    one-hot x and scale2 = 1 make y_A exact in bf16 pairs (0, y_A[n]))."""
    N = 2048
    a = dict(synth.make_layer("nvfp4", N, 4096, config=62, matrix=0), scale2=1.0)
    b = synth.make_layer("nvfp4", 512, 2 * N, config=62, matrix=1)
    da, db = to_device(a), to_device(b)
    x = torch.zeros((1, 4096), dtype=torch.bfloat16, device="cuda")
    x[0, 9] = 1.0
    ya = torch.empty((1, N), dtype=torch.float32, device="cuda")
    yb = torch.empty((1, 512), dtype=torch.float32, device="cuda")
    xv = ya.view(torch.bfloat16)
    gemv(a, da, x, 1, ya)
    torch.cuda.synchronize()
    assert (ya.view(torch.int32) & 0xFFFF).eq(0).all().item() and ya.abs().sum().item() > 0
    xb = xv.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, bound = oracle.gemv(to_oracle(b), oracle.bf16_bits_to_f32(xb).reshape(1, -1))
    sync = sync_words()
    groups = [[chain_member(a, da, x, ya)], [chain_member(b, db, xv, yb)]]
    want = None
    for _ in range(5):
        ya.zero_()
        yb.fill_(float("nan"))
        q4.q4_gemv_chain(groups, 1, sync=sync)
        assert q4.q4_last_gemv_path() == "gemv_tma_chain"
        torch.cuda.synchronize()
        if want is None:
            want = yb.clone()
            ok, worst = within_tolerance(want.cpu().numpy(), ref, bound)
            assert ok, worst
        assert torch.equal(yb, want)                   # the chain repeats bit for bit
    # the same chain replayed from a CUDA graph: the barrier words carry over
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        q4.q4_gemv_chain(groups, 1, sync=sync, stream=st)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            ya.zero_()
            yb.fill_(float("nan"))
            q4.q4_gemv_chain(groups, 1, sync=sync, stream=st)
        for _ in range(4):
            g.replay()
        torch.cuda.synchronize()
    assert torch.equal(yb, want)
    assert q4.q4_last_error() == q4.Q4_OK
    assert sync.cpu().tolist() == [0, 10]          # 5 + 1 calls and 4 replays


def test_chain_deterministic_and_falls_back_when_not_eligible():
    L0 = synth.make_layer("nvfp4", 1029, 4096, config=63, matrix=0)
    L1 = synth.make_layer("nvfp4", 300, 4096, config=63, matrix=1)
    d0, d1 = to_device(L0), to_device(L1)
    xb, xf = synth.draw_x(1, 4096, config=63, matrix=2)
    x = x_device(xb)
    y0, y1 = torch.empty((1, 1029), device="cuda"), torch.empty((1, 300), device="cuda")
    sync = sync_words()
    groups = [[chain_member(L0, d0, x, y0)], [chain_member(L1, d1, x, y1)]]
    q4.q4_gemv_chain(groups, 1, sync=sync)
    a0, a1 = y0.clone(), y1.clone()
    for _ in range(3):
        q4.q4_gemv_chain(groups, 1, sync=sync)
        assert torch.equal(y0, a0) and torch.equal(y1, a1)
    # an f32 x member is not eligible: the groups are issued one by one
    q = synth.make_layer("q4k", 64, 4096, config=63, matrix=3)
    dq = to_device(q)
    yq = torch.full((1, 64), float("nan"), device="cuda")
    xq = x_device(xf.astype(np.float32))
    qm = ("q4k", dq["w"], None, aux_for(q, dq, x_dtype=torch.float32), xq, yq, 64, 4096)
    q4.q4_gemv_chain([[chain_member(L0, d0, x, y0)], [qm]], 1, sync=sync)
    assert q4.q4_last_gemv_path() != "gemv_tma_chain"
    torch.cuda.synchronize()
    ref, bound = oracle.gemv(to_oracle(q), xf)
    ok, worst = within_tolerance(yq.cpu().numpy(), ref, bound)
    assert ok, worst
    # group 0 ran as its own batch-1 launch (another kernel, another rounding order)
    ref0, bound0 = oracle.gemv(to_oracle(L0), xf)
    ok, worst = within_tolerance(y0.cpu().numpy(), ref0, bound0)
    assert ok, worst
