// gemm_tc.cu -- small-batch decode-GEMM (M >= 9, bf16 activations) on the
// tcgen05 tensor cores: Y[m][n] = sum_k w_hat[n][k] * x[m][k].
//
// The batch is short, so the weights are the MMA's A operand (M = 128 weight
// rows per CTA = the 128 TMEM lanes) and the activations are B (the MMA's N =
// the batch, padded to 16, 32, 64 or 128 with zero rows by the TMA unit).
// A is produced by CUDA cores, so it is written straight into tensor memory
// (tcgen05.mma with A in TMEM): the decoded bf16 weights (4x the packed
// bytes) never pass through shared memory.  Roles per CTA (352 threads):
//
//   warps 0-7  decode, as two warpgroups that split every 64-k stage in
//              k halves: thread r of a warpgroup owns weight row n0+r (= TMEM
//              lane r), reads its packed bytes from the shared-memory slot,
//              decodes its 32 k to bf16 pairs and stores them with tcgen05.st
//              into its 16 columns of a TMEM A stage.  Warps 0-3 run the
//              epilogue.
//   warp 8     allocates TMEM; one thread issues tcgen05.mma and
//              tcgen05.commit (which frees A/X stages and signals the end).
//   warp 9     one thread streams the weight slots by TMA (128 rows x 256 k:
//              NVFP4 payload with a 128-byte swizzle plus its E4M3 scales,
//              or the Q4_K super-blocks) into a ring of 2-4 slots.
//   warp 10    one thread loads the X tiles by TMA (128-byte swizzle).
//
// K is split over the S CTAs of a thread-block cluster; their f32 partial
// tiles are summed in rank order through distributed shared memory, so the
// result does not depend on scheduling.
//
// What an A stage holds:
//   NVFP4  v(code) * dec(E4M3 scale), the first product of the pinned order
//          ([MUS7] 7.1-7.2): at most 6 significant bits, exact in bf16.  The
//          per-tensor scale2 multiplies the f32 accumulator in the epilogue.
//   Q4_K   RNE_bf16(fl(q * (d*sc) - dmin*m)) ([FBTC] sections 5-6): the f32
//          weight of the pinned rule, rounded once to bf16 for the MMA.
#include <cooperative_groups.h>
#include <mutex>

#include "q4_internal.cuh"
#include "tma_map.cuh"

namespace cg = cooperative_groups;

namespace q4 {
namespace {

// Sticky device-side error word (a bounded mbarrier wait that ran out).
__device__ int g_device_error;

constexpr int ROWS = 128;          // weight rows per CTA = MMA M = TMEM lanes
constexpr int BK = 64;             // k per pipeline (MMA) stage
constexpr int A_COLS = BK / 2;     // TMEM columns per A stage (one bf16 pair per column)
constexpr int SLOT_K = 256;        // k per weight slot = 4 stages
constexpr int PAYLOAD_BYTES = ROWS * 128;           // NVFP4: 128 rows x 128 payload bytes
constexpr int SLOT_BYTES = PAYLOAD_BYTES + ROWS * 16;  // + 16 scale bytes a row; Q4_K: 128 x 144 B
constexpr int DEC_WARPS = 8;
constexpr int W_MMA = DEC_WARPS, W_TMA_W = DEC_WARPS + 1, W_TMA_X = DEC_WARPS + 2;
constexpr int THREADS = (DEC_WARPS + 3) * 32;
constexpr int TMEM_COLS = 256;     // two CTAs per SM share the 512 columns
constexpr int SMEM_FLOOR = 80 * 1024;  // keeps a third CTA (which could get no TMEM) off the SM
static_assert(SLOT_BYTES == ROWS * 144, "an NVFP4 slot and a Q4_K slot have the same size");

// Both decode warpgroups work on every stage (each on half of its k range)
// and every role walks the stage and slot rings in order, so each waiter on
// a barrier sees all of its phases in turn -- mbarrier's parity test cannot
// tell a phase from the one two uses later.
template <int MB> struct Cfg {
    static constexpr int DCOLS = MB < 32 ? 32 : MB;           // accumulator columns
    static constexpr int NS = (TMEM_COLS - DCOLS) / A_COLS;   // A stages in TMEM = X stages
    static constexpr int B_BYTES = MB * BK * 2;               // one X tile: MB rows x 128 B
    static constexpr int XRING = NS * B_BYTES;
    // weight slots in flight (batch 16: 2 slots measured 20.6 us against 20.9 with 4,
    // the first slot of every CTA landing sooner)
    static constexpr int NW = MB == 64 ? 3 : 2;
    static constexpr int WRING = NW * SLOT_BYTES;
    static constexpr int USED = 1024 + WRING + XRING;
    static constexpr int SMEM = USED > SMEM_FLOOR ? USED : SMEM_FLOOR;
    static_assert(XRING >= MB * ROWS * 4, "the f32 partial tile reuses the X ring");
    static_assert(2 * SMEM <= 227 * 1024, "two CTAs per SM");
};

struct TcArgs {
    float *y;           // [M][N] f32 for this batch chunk
    int64_t N, K;
    int M;              // valid activation rows in this chunk (<= MB)
    int splits;         // CTAs per cluster, each owning K / splits
    int k_per_cta;
    float mult;         // epilogue multiplier: scale2 for NVFP4, 1 for Q4_K
    int ystore;         // 1: without a K split, y leaves through shared memory by one TMA store (maps.y)
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *dst) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(TMEM_COLS) : "memory");
}

// D (+)= A * B^T with A (128 x 16 bf16) in TMEM and B (MB x 16 bf16) in shared
// memory; `accumulate` = 0 overwrites D.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile("{ .reg .pred p;\n\t setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Instruction descriptor of kind::f16: f32 D, bf16 A and B, both K-major,
// N = MB, M = 128.
template <int MB> __device__ __forceinline__ constexpr uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(MB >> 3) << 17) | ((uint32_t)(ROWS >> 4) << 24);
}
// Shared-memory descriptor of a K-major operand in the 128-byte swizzle
// layout written by TMA: rows of 128 B, 8-row groups 1024 B apart.  A 16-k
// step inside the 64-k row is a 32-byte advance of the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// One tiled tensor store from shared memory (bulk group of this thread), and
// the wait until it has completed.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int c0, int c1, const void *src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(c0),
                 "r"(c1), "r"(smem_u32(src))
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// 16 consecutive TMEM columns of this thread's lane <- v[0..15]; waits until
// the stores are done.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                 "%12, %13, %14, %15, %16};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                 "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 16 consecutive TMEM columns of this thread's lane -> v[0..15].
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15}, [%16];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
                   "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]),
                   "=f"(v[15])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// Two f32 -> bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// Lane-wise (a + b) and (a * b + c) on f32 pairs, one rounding per lane.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{ .reg .b64 ra, rb;\n\t mov.b64 ra, {%2, %3};\n\t mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\t mov.b64 {%0, %1}, ra; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{ .reg .b64 ra, rb, rc;\n\t mov.b64 ra, {%2, %3};\n\t mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t fma.rn.f32x2 rc, ra, rb, rc;\n\t mov.b64 {%0, %1}, rc; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Bounded mbarrier wait shared by all roles: gives up after ~1 s, records
// Q4_ETIMEOUT and raises the CTA's abort flag; also gives up once another
// role has raised it.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > (1LL << 31)) {
            atomicExch(&g_device_error, Q4_ETIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------ NVFP4 decode
__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
    return v;
}

// Eight E2M1 codes of one payload word (byte j: k = 2j in the low nibble,
// 2j+1 in the high nibble) times one E4M3 block scale -> four bf16 pairs.
// `s2` holds two scales as exact f16 (cvt.rn.f16x2.e4m3x2); HI picks which.
// Per byte: the hardware convert gives both codes as exact f16, two
// mixed-precision FMAs form v * scale in f32 (exact: <= 6 significant bits),
// and one byte permute keeps the top halves of the two f32 -- their exact
// bf16 patterns.  Two ALU and two FMA-pipe instructions per weight pair.
#define Q4_NV_BYTE(B, OUT)                                                                                     \
    "cvt.rn.f16x2.e2m1x2 h, " B ";\n\t"                                                                        \
    "mov.b32 {c0, c1}, h;\n\t"                                                                                 \
    "fma.rn.f32.f16 f0, c0, sc, 0f00000000;\n\t"                                                               \
    "fma.rn.f32.f16 f1, c1, sc, 0f00000000;\n\t"                                                               \
    "prmt.b32 " OUT ", f0, f1, 0x7632;\n\t"
#define Q4_NV_WORD(SCALE_SEL)                                                                                  \
    asm("{\n\t .reg .b8 b0, b1, b2, b3;\n\t .reg .b16 s_lo, s_hi, sc, c0, c1;\n\t .reg .b32 h, f0, f1;\n\t"     \
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"                                                                    \
        "mov.b32 {s_lo, s_hi}, %5;\n\t"                                                                        \
        "mov.b16 sc, " SCALE_SEL ";\n\t" Q4_NV_BYTE("b0", "%0") Q4_NV_BYTE("b1", "%1") Q4_NV_BYTE("b2", "%2")   \
            Q4_NV_BYTE("b3", "%3") "}"                                                                         \
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])                                                       \
        : "r"(w), "r"(s2))
template <int HI>
__device__ __forceinline__ void nvfp4_word(uint32_t w, uint32_t s2, uint32_t *o) {
    if constexpr (HI)
        Q4_NV_WORD("s_hi");
    else
        Q4_NV_WORD("s_lo");
}
#undef Q4_NV_WORD
#undef Q4_NV_BYTE

// Half of a 64-k stage of one row: 16 payload bytes (32 codes, k = 32h ..
// 32h+31 of the stage) and the two E4M3 scales of its 16-k groups (s2, the
// low scale in the low byte) -> 16 bf16 pairs, column c holding k = 2c, 2c+1.
__device__ __forceinline__ void nvfp4_half(uint4 p, uint32_t s2, uint32_t (&o)[16]) {
    uint32_t sh;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(sh) : "h"((unsigned short)(s2 & 0xffffu)));
    nvfp4_word<0>(p.x, sh, o + 0);
    nvfp4_word<0>(p.y, sh, o + 4);
    nvfp4_word<1>(p.z, sh, o + 8);
    nvfp4_word<1>(p.w, sh, o + 12);
}

// ------------------------------------------------------------- Q4_K decode
// 6-bit scale and min of sub-block j from the 12 metadata bytes B0 (bytes
// 0-3), B1 (4-7), B2 (8-11), [FBTC] section 6.
__device__ __forceinline__ void q4k_sc_m(uint32_t B0, uint32_t B1, uint32_t B2, int j, uint32_t &sc, uint32_t &m) {
    if (j < 4) {
        sc = (B0 >> (8 * j)) & 63u;
        m = (B1 >> (8 * j)) & 63u;
    } else {
        const int s = 8 * (j - 4);
        sc = ((B2 >> s) & 15u) | (((B0 >> s) >> 6 & 3u) << 4);
        m = ((B2 >> s) >> 4 & 15u) | (((B1 >> s) >> 6 & 3u) << 4);
    }
}

// Four 4-bit codes (low nibble of each byte of L) -> two bf16 pairs of
// RNE_bf16(fl(q*step - off)): q is exact through the 2^23 + q construction,
// q*step is exact (<= 21 significant bits), so the one FMA rounding is the
// pinned f32 one, and the pack rounds that once to bf16.
__device__ __forceinline__ void q4k_quad(uint32_t L, float2 step, float2 noff, uint32_t *o) {
    const float2 m2 = make_float2(-8388608.0f, -8388608.0f);
    const float2 q01 = add2(make_float2(__uint_as_float(prmt(L, 0x4B000000u, 0x7440u)),
                                        __uint_as_float(prmt(L, 0x4B000000u, 0x7441u))),
                            m2);
    const float2 q23 = add2(make_float2(__uint_as_float(prmt(L, 0x4B000000u, 0x7442u)),
                                        __uint_as_float(prmt(L, 0x4B000000u, 0x7443u))),
                            m2);
    const float2 w01 = fma2(q01, step, noff), w23 = fma2(q23, step, noff);
    o[0] = pack_bf16x2(w01.x, w01.y);
    o[1] = pack_bf16x2(w23.x, w23.y);
}

// Half HI of chunk c (k = 64c .. 64c+63) of a super-block with header h
// (fp16 d, fp16 dmin, 12 metadata bytes): code byte i holds k = 64c + i in its
// low nibble (sub-block 2c, HI = 0) and k = 64c + 32 + i in its high nibble
// (sub-block 2c+1, HI = 1).  Output column p holds k = 2p, 2p+1 of the half.
__device__ __forceinline__ void q4k_half(uint4 h, uint4 q0, uint4 q1, int c, int hi, uint32_t (&o)[16]) {
    const float d = half_bits_f32(h.x), dmin = half_bits_f32(h.x >> 16);
    uint32_t sc, m;
    q4k_sc_m(h.y, h.z, h.w, 2 * c + hi, sc, m);
    const float step = d * (float)sc, off = dmin * (float)m;   // both exact
    const float2 s2 = make_float2(step, step), n2 = make_float2(-off, -off);
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const int shift = 4 * hi;
#pragma unroll
    for (int t = 0; t < 8; t++) q4k_quad((words[t] >> shift) & 0x0F0F0F0Fu, s2, n2, o + 2 * t);
}

// ------------------------------------------------------------ the kernel
struct Maps {
    CUtensorMap y;   // f32 [rows][N] of this batch chunk, box 128 n x MB rows (used when ystore)
    CUtensorMap x;   // bf16 [rows][K], box 64 k x MB rows, 128-byte swizzle
    CUtensorMap w;   // NVFP4 payload u8 [N][K/2] (box 128 x 128, 128-byte swizzle) or Q4_K u8 [N][K/256*144] (box 144 x 128)
    CUtensorMap s;   // NVFP4 scales u8 [N][K/16], box 16 x 128 (unused for Q4_K)
};

template <int FMT, int MB>
__global__ void __launch_bounds__(THREADS, 2)
    gemm_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ Maps maps) {
    using C = Cfg<MB>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t a_full[C::NS], a_empty[C::NS], w_full[C::NW], w_empty[C::NW], done_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    uint8_t *wring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *xring = wring + C::WRING;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / a.splits, rank = blockIdx.x % a.splits;
    const int n0 = tile * ROWS;
    const int kbeg = rank * a.k_per_cta;
    const int nst = a.k_per_cta / BK, nslots = a.k_per_cta / SLOT_K;
    volatile int *abort_flag = &abort_s;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; s++) {
            mbar_init(&a_full[s], DEC_WARPS + 1);  // one arrive per decode warp + the X-tile thread
            mbar_init(&a_empty[s], 1);         // one tcgen05.commit
        }
        for (int s = 0; s < C::NW; s++) {
            mbar_init(&w_full[s], 1);          // the weight thread's arrive + its bytes
            mbar_init(&w_empty[s], DEC_WARPS);     // one arrive per decode warp that read the slot
        }
        mbar_init(&done_bar, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) tmem_alloc(&tmem_base_s);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;
    bool aborted = false;

    if (warp < DEC_WARPS) {
        // ---------------------------------------------------------- decode
        const int h = warp >> 2;                 // warpgroup: k half of every stage
        const int r = threadIdx.x & (ROWS - 1);  // weight row in the tile = TMEM lane
        const uint32_t lane_base = tbase + ((uint32_t)(r & ~31) << 16) + C::DCOLS + h * (A_COLS / 2);
        for (int j = 0; j < nslots && !aborted; j++) {
            const int wi = j % C::NW;
            bool ok = wait_or_abort(&w_full[wi], (j / C::NW) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                aborted = true;
                break;
            }
            const uint32_t slot = smem_u32(wring + wi * SLOT_BYTES);
            uint4 meta;   // NVFP4: the row's 16 scale bytes; Q4_K: its super-block header
            if constexpr (FMT == Q4_NVFP4)
                meta = lds128(slot + PAYLOAD_BYTES + r * 16);
            else
                meta = lds128(slot + r * 144);
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int i = 4 * j + c;
                uint32_t o[16];
                if constexpr (FMT == Q4_NVFP4) {
                    // 16-byte chunk 2c+h of the row, at its 128-byte-swizzle position
                    const uint4 p = lds128(slot + r * 128 + (((uint32_t)(2 * c + h) ^ (uint32_t)(r & 7)) << 4));
                    const uint32_t s4 = c == 0 ? meta.x : c == 1 ? meta.y : c == 2 ? meta.z : meta.w;
                    nvfp4_half(p, s4 >> (16 * h), o);
                } else {
                    const uint32_t blk = slot + r * 144 + 16 + 32 * c;
                    q4k_half(meta, lds128(blk), lds128(blk + 16), c, h, o);
                }
                if (c == 3) {                        // the slot's bytes are all in this warp's registers
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&w_empty[wi]);
                }
                const int s = i % C::NS;
                ok = i < C::NS || wait_or_abort(&a_empty[s], ((i / C::NS) & 1) ^ 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {   // tcgen05.st is warp-collective
                    aborted = true;
                    break;
                }
                tc_fence_after();
                tmem_st16(lane_base + s * A_COLS, o);   // returns once this thread's stores are done
                tc_fence_before();
                __syncwarp();                           // ... and every lane's: one arrive per warp
                if (lane == 0) mbar_arrive(&a_full[s]);
            }
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            // One thread issues every MMA, and its loop is the kernel's critical
            // path (a tcgen05.mma of 128 x N x 16 costs ~94 issue cycles for
            // any N <= 128 even back to back): the loop is unrolled over the
            // ring so every descriptor is a constant offset from one base.
            constexpr uint32_t idesc = idesc_bf16<MB>();
            const uint64_t b0 = sw128_desc(smem_u32(xring));
            const uint32_t a0 = tbase + C::DCOLS;
            bool stop = false;
            for (int base = 0; base < nst && !stop; base += C::NS) {
                const uint32_t par = (uint32_t)(base / C::NS) & 1;
#pragma unroll
                for (int s = 0; s < C::NS; s++) {
                    if (base + s >= nst) break;
                    if (!wait_or_abort(&a_full[s], par, abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < BK / 16; k++)
                        mma_ts(tbase, a0 + s * A_COLS + k * 8, b0 + (uint64_t)((s * C::B_BYTES + k * 32) >> 4), idesc,
                               (base + s + k) != 0);
                    mma_commit(&a_empty[s]);
                }
            }
            mma_commit(&done_bar);
        }
        __syncwarp();
    } else if (warp == W_TMA_W) {
        // ---------------------------------------------------- weight slots
        if (lane == 0) {
            for (int j = 0; j < nslots; j++) {
                const int wi = j % C::NW;
                if (j >= C::NW && !wait_or_abort(&w_empty[wi], ((j / C::NW) & 1) ^ 1, abort_flag)) break;
                uint8_t *slot = wring + wi * SLOT_BYTES;
                mbar_arrive_expect_tx(&w_full[wi], SLOT_BYTES);
                if constexpr (FMT == Q4_NVFP4) {
                    tma_2d(slot, &maps.w, kbeg / 2 + j * (SLOT_K / 2), n0, &w_full[wi]);
                    tma_2d(slot + PAYLOAD_BYTES, &maps.s, kbeg / 16 + j * (SLOT_K / 16), n0, &w_full[wi]);
                } else {
                    tma_2d(slot, &maps.w, (kbeg / SLOT_K + j) * 144, n0, &w_full[wi]);
                }
            }
        }
        __syncwarp();
    } else if (warp == W_TMA_X) {
        // ------------------------------------------------------- X tiles
        if (lane == 0) {
            for (int i = 0; i < nst; i++) {
                const int s = i % C::NS;
                if (i >= C::NS && !wait_or_abort(&a_empty[s], ((i / C::NS) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(&a_full[s], C::B_BYTES);
                tma_2d(xring + s * C::B_BYTES, &maps.x, kbeg + i * BK, 0, &a_full[s]);
            }
        }
        __syncwarp();
    }

    // ---------------------------------------------------------- epilogue
    // [MB][128] f32 tile (the partial tile of a K split, or y on its way to the
    // TMA store); the X ring is idle once the MMAs are done
    float *red = reinterpret_cast<float *>(xring);
    if (warp < 4) {
        const int r = threadIdx.x;
        const int64_t n = (int64_t)n0 + r;
        bool ok = !aborted && wait_or_abort(&done_bar, 0, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            const uint32_t lane_d = tbase + ((uint32_t)(r & ~31) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < MB; c0 += 16) {
                float v[16];
                tmem_ld16(lane_d + c0, v);
                if (a.splits == 1 && a.ystore) {
#pragma unroll
                    for (int j = 0; j < 16; j++) red[(c0 + j) * ROWS + r] = v[j] * a.mult;
                } else if (a.splits == 1) {
                    if (n < a.N) {
#pragma unroll
                        for (int j = 0; j < 16; j++)
                            if (c0 + j < a.M) a.y[(int64_t)(c0 + j) * a.N + n] = v[j] * a.mult;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; j++) red[(c0 + j) * ROWS + r] = v[j];
                }
            }
        }
        tc_fence_before();
        if (a.splits == 1 && a.ystore) {
            // the tile's generic-proxy stores, then one TMA store of all of it
            // (rows past M and columns past N are clipped by the tensor map)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
            if (r == 0 && ok) tma_store_2d(&maps.y, n0, 0, red);
        }
    }
    if (a.splits > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();   // every partial tile of the cluster is in shared memory
        if (warp < 4 && !*abort_flag) {
            const int r = threadIdx.x;
            const int64_t n = (int64_t)n0 + r;
            const int cols = MB / a.splits;
            for (int c = rank * cols; c < (rank + 1) * cols; c++) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; q++) v[q] = q < a.splits ? cluster.map_shared_rank(red + c * ROWS + r, q)[0] : 0.0f;
                float acc = v[0];   // rank order, whatever the arrival order
#pragma unroll
                for (int q = 1; q < 8; q++)
                    if (q < a.splits) acc += v[q];
                if (c < a.M && n < a.N) a.y[(int64_t)c * a.N + n] = acc * a.mult;
            }
        }
        cluster.sync();   // no CTA leaves while its partial tile may still be read
    }
    if (*abort_flag) {
        // copies issued before the abort land within microseconds; do not
        // hand the shared memory back while one may still be in flight
        const long long t0 = clock64();
        while (clock64() - t0 < 2000000) {
        }
    }
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tbase);
    }
}

// ------------------------------------------------------------------ host
// One 2-D tiled tensor map: `inner` elements per row (contiguous), `rows`
// rows `pitch` bytes apart; boxes of box_inner x box_rows; reads past either
// edge return zeros.
bool encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base, int64_t inner, int64_t rows,
               int64_t pitch, int box_inner, int box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The weight maps of a tensor (independent of the batch chunk).
bool encode_weights(Maps *m, const Tensor &t) {
    if (t.fmt == Q4_NVFP4)
        return encode_2d(&m->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, t.w, t.K / 2, t.N, t.K / 2, SLOT_K / 2, ROWS,
                         CU_TENSOR_MAP_SWIZZLE_128B) &&
               encode_2d(&m->s, CU_TENSOR_MAP_DATA_TYPE_UINT8, t.scales, t.K / 16, t.N, t.K / 16, SLOT_K / 16, ROWS,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    const int64_t row_bytes = t.K / SLOT_K * 144;
    m->s = m->w;
    return encode_2d(&m->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, t.w, row_bytes, t.N, row_bytes, 144, ROWS,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

// X tiles of one batch chunk (bf16 [rows][K]): 64 k x MB rows, 128-byte
// swizzle; rows past `rows` read as zero.
bool encode_x(CUtensorMap *map, const void *x, int64_t K, int64_t rows, int MB) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, rows, K * 2, BK, MB, CU_TENSOR_MAP_SWIZZLE_128B);
}

// K slice per CTA: split K over up to 8 cluster ranks until the grid covers
// every SM once (batch tiles up to 32) or half of them (64 and 128, where the
// cluster's partial-tile exchange costs more than idle SMs), keeping every
// slice whole weight slots.  Measured on 14336 x 4096 (112 row tiles): split
// 2 at batch 16 (24.4 us against 27.7 at split 4), no split at batch 128
// (31.6 us against 40.9).
int pick_splits(int64_t tiles, int64_t K, int MB) {
    const int64_t sms = sm_count();
    const int64_t target = MB >= 64 ? sms / 2 : sms;
    int S = 1;
    while (S < 8 && tiles * S < target && K % (2 * S) == 0 && (K / (2 * S)) % SLOT_K == 0) S *= 2;
    return S;
}

template <int FMT, int MB>
cudaError_t launch_one(const TcArgs &args, const Maps &maps, int64_t tiles, cudaStream_t s) {
    auto kern = gemm_tc_kernel<FMT, MB>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<MB>::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * args.splits));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = Cfg<MB>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)args.splits;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args, maps);
}

template <int FMT>
cudaError_t launch_mb(int MB, const TcArgs &args, const Maps &maps, int64_t tiles, cudaStream_t s) {
    switch (MB) {
    case 16: return launch_one<FMT, 16>(args, maps, tiles, s);
    case 32: return launch_one<FMT, 32>(args, maps, tiles, s);
    case 64: return launch_one<FMT, 64>(args, maps, tiles, s);
    default: return launch_one<FMT, 128>(args, maps, tiles, s);
    }
}

}  // namespace

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool gemm_tc_eligible(const Tensor &t, q4_dtype x_dtype, int64_t M) {
    return M >= 9 && x_dtype == Q4_DT_BF16 && (t.fmt == Q4_NVFP4 || t.fmt == Q4_Q4K) && t.K % SLOT_K == 0 &&
           t.K <= (1LL << 30) && t.N <= (1LL << 30);
}

cudaError_t launch_gemm_tc(const Tensor &t, const void *x, q4_dtype x_dtype, float *y, int64_t M, cudaStream_t s,
                           bool *handled) {
    *handled = false;
    if (!gemm_tc_eligible(t, x_dtype, M)) return cudaSuccess;
    *handled = true;
    note_gemv_path("gemm_tc");
    const int64_t tiles = (t.N + ROWS - 1) / ROWS;
    Maps maps;
    if (!encode_weights(&maps, t)) return cudaErrorInvalidValue;
    for (int64_t m0 = 0; m0 < M; m0 += 128) {
        const int64_t rows = M - m0 < 128 ? M - m0 : 128;
        const int MB = rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
        const int S = pick_splits(tiles, t.K, MB);
        if (!encode_x(&maps.x, (const uint8_t *)x + m0 * t.K * 2, t.K, rows, MB)) return cudaErrorInvalidValue;
        TcArgs args;
        args.y = y + m0 * t.N;
        args.N = t.N;
        args.K = t.K;
        args.M = (int)rows;
        args.splits = S;
        args.k_per_cta = (int)(t.K / S);
        args.mult = t.fmt == Q4_NVFP4 ? t.scale2 : 1.0f;
        // without a K split the output tile leaves by one TMA store: rows of y
        // must be a multiple of 16 bytes apart
        args.ystore = (S == 1 && t.N % 4 == 0 &&
                       encode_2d(&maps.y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, y + m0 * t.N, t.N, rows, t.N * 4, ROWS, MB,
                                 CU_TENSOR_MAP_SWIZZLE_NONE))
                          ? 1
                          : 0;
        const cudaError_t e = t.fmt == Q4_NVFP4 ? launch_mb<Q4_NVFP4>(MB, args, maps, tiles, s)
                                                : launch_mb<Q4_Q4K>(MB, args, maps, tiles, s);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

int gemv_read_and_clear_error();
int gemv_tma_read_and_clear_error();
int pack_read_and_clear_error();
int fp4tc_read_and_clear_error();
int awq_read_and_clear_error();
int gptq_tc_read_and_clear_error();
int blk_tc_read_and_clear_error();
int a16tc_read_and_clear_error();
int k8tc_read_and_clear_error();

int read_and_clear_device_error() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    const int g = gemv_read_and_clear_error();
    const int tm = gemv_tma_read_and_clear_error();
    const int pk = pack_read_and_clear_error();
    const int f4 = fp4tc_read_and_clear_error();
    const int aw = awq_read_and_clear_error();
    const int gq = gptq_tc_read_and_clear_error();
    const int bt = blk_tc_read_and_clear_error();
    const int aq = a16tc_read_and_clear_error();
    const int kt = k8tc_read_and_clear_error();
    return v ? v : g ? g : tm ? tm : pk ? pk : f4 ? f4 : aw ? aw : gq ? gq : bt ? bt : aq ? aq : kt;
}

}  // namespace q4

extern "C" int q4_last_error(void) { return q4::read_and_clear_device_error(); }
