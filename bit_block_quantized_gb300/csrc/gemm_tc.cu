// gemm_tc.cu -- small-batch decode-GEMM (M >= 9, bf16 activations) on the
// tcgen05 tensor cores: Y[m][n] = sum_k w_hat[n][k] * x[m][k].
//
// The batch is short, so the weights are the MMA's A operand (M = 128 weight
// rows per CTA = the 128 TMEM lanes) and the activations are B (the MMA's N =
// the batch, padded to 16, 32, 64 or 128 with zero rows by the TMA unit).
// A is produced by CUDA cores, so it is written straight into tensor memory
// (tcgen05.mma with A in TMEM): the decoded bf16 weights (4x the packed
// bytes) never pass through shared memory, whose bandwidth would otherwise
// cap the decode rate.  Roles per CTA (192 threads):
//
//   warps 0-3  decode: thread r streams weight row n0+r from HBM, decodes 64
//              k per stage to bf16 pairs and stores them with tcgen05.st into
//              lane r of a TMEM A stage; then the epilogue.
//   warp 4     allocates TMEM; one thread issues tcgen05.mma and
//              tcgen05.commit (which frees A/B stages and signals the end).
//   warp 5     warms L2 with bulk prefetches of the CTA's weight slice, then
//              one thread loads the X tiles by TMA (128-byte swizzle).
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
#include <cuda.h>  // CUtensorMap and the encode signature; the function is fetched at run time

#include <cooperative_groups.h>
#include <mutex>

#include "q4_internal.cuh"

namespace cg = cooperative_groups;

namespace q4 {
namespace {

// Sticky device-side error word (a bounded mbarrier wait that ran out).
__device__ int g_device_error;

constexpr int ROWS = 128;          // weight rows per CTA = MMA M = TMEM lanes
constexpr int BK = 64;             // k per pipeline stage
constexpr int A_COLS = BK / 2;     // TMEM columns per A stage (one bf16 pair per column)
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 256;     // two CTAs per SM share the 512 columns
constexpr int SMEM_FLOOR = 80 * 1024;  // keeps a third CTA (which could get no TMEM) off the SM
#ifndef Q4_TC_PD
#define Q4_TC_PD 4
#endif
constexpr int PD = Q4_TC_PD;       // stages of weight bytes in registers per decode thread
static_assert(PD % 4 == 0, "the Q4_K decoder needs the chunk index of a stage to be static");

template <int MB> struct Cfg {
    static constexpr int DCOLS = MB < 32 ? 32 : MB;           // accumulator columns
    static constexpr int NS = (TMEM_COLS - DCOLS) / A_COLS;   // pipeline stages
    static constexpr int B_BYTES = MB * BK * 2;               // one X tile: MB rows x 128 B
    static constexpr int RING = NS * B_BYTES;
    static constexpr int SMEM = (RING + 1024 > SMEM_FLOOR) ? RING + 1024 : SMEM_FLOOR;
    static_assert(RING >= MB * ROWS * 4, "the f32 partial tile reuses the X ring");
};

struct TcArgs {
    const uint8_t *w;   // packed weights (NVFP4 payload [N][K/2] or Q4_K blocks [N][K/256][144])
    const uint8_t *s;   // NVFP4 E4M3 scales [N][K/16]; unused for Q4_K
    float *y;           // [M][N] f32 for this batch chunk
    int64_t N, K;
    int M;              // valid activation rows in this chunk (<= MB)
    int splits;         // CTAs per cluster, each owning K / splits
    int k_per_cta;
    float mult;         // epilogue multiplier: scale2 for NVFP4, 1 for Q4_K
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

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 32 consecutive TMEM columns of this thread's lane <- v[0..31].
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                 "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, "
                 "%31, %32};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                 "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
                 "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
                 "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
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
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
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
struct NvStage {
    uint4 a, b;   // 32 payload bytes: k0 .. k0+63 of one row
    uint32_t s;   // their four E4M3 block scales
};

// Eight E2M1 codes of one payload word (byte j: k = 2j in the low nibble,
// 2j+1 in the high nibble) times one block scale -> four bf16 pairs.
// S = bf16x2 of (scale * 2^112).  The hardware convert gives the magnitude
// codes as f16 whose low 9 bits are zero; shifted right by 3 each half is the
// bf16 pattern of |v| * 2^-112 (a normal number).  The sign bits of the
// nibbles (bits 3 and 7 of byte j) are placed at bits 15 and 31 by one byte
// permute, and the bf16 multiply by S restores the exponent and applies the
// block scale; every step is exact.
__device__ __forceinline__ void nvfp4_word(uint32_t w, uint32_t S, uint32_t *o) {
    uint32_t h0, h1, h2, h3;
    e2m1x8_h2(w & 0x77777777u, h0, h1, h2, h3);
    const uint32_t w4 = w << 4;
    o[0] = bf16x2_mul((h0 >> 3) | (prmt(w, w4, 0x0040u) & 0x80008000u), S);
    o[1] = bf16x2_mul((h1 >> 3) | (prmt(w, w4, 0x1050u) & 0x80008000u), S);
    o[2] = bf16x2_mul((h2 >> 3) | (prmt(w, w4, 0x2060u) & 0x80008000u), S);
    o[3] = bf16x2_mul((h3 >> 3) | (prmt(w, w4, 0x3070u) & 0x80008000u), S);
}

__device__ __forceinline__ void nvfp4_stage(const NvStage &st, uint32_t (&o)[32]) {
    const float k112 = 0x1p112f;
    const float2 f01 = e4m3x2_f32(st.s & 0xffffu), f23 = e4m3x2_f32(st.s >> 16);
    const uint32_t S0 = pack_bf16x2(f01.x * k112, f01.x * k112), S1 = pack_bf16x2(f01.y * k112, f01.y * k112);
    const uint32_t S2 = pack_bf16x2(f23.x * k112, f23.x * k112), S3 = pack_bf16x2(f23.y * k112, f23.y * k112);
    nvfp4_word(st.a.x, S0, o + 0);
    nvfp4_word(st.a.y, S0, o + 4);
    nvfp4_word(st.a.z, S1, o + 8);
    nvfp4_word(st.a.w, S1, o + 12);
    nvfp4_word(st.b.x, S2, o + 16);
    nvfp4_word(st.b.y, S2, o + 20);
    nvfp4_word(st.b.z, S3, o + 24);
    nvfp4_word(st.b.w, S3, o + 28);
}

// ------------------------------------------------------------- Q4_K decode
struct QkStage {
    uint4 h;       // super-block header: fp16 d, fp16 dmin, 12 scale/min bytes
    uint4 q0, q1;  // the 32 code bytes of one 64-weight chunk
};

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
// fl(q*step - off): q is exact through the 2^23 + q construction, q*step is
// exact (<= 21 significant bits), so the one FMA rounding is the pinned one.
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

// Chunk c of a super-block: code byte i holds k = 64c + i (low nibble,
// sub-block 2c) and k = 64c + 32 + i (high nibble, sub-block 2c+1).  Output
// column p holds k = 2p, 2p+1 of the chunk.
__device__ __forceinline__ void q4k_stage(const QkStage &st, int c, uint32_t (&o)[32]) {
    const float d = half_bits_f32(st.h.x), dmin = half_bits_f32(st.h.x >> 16);
    uint32_t sc0, m0, sc1, m1;
    q4k_sc_m(st.h.y, st.h.z, st.h.w, 2 * c, sc0, m0);
    q4k_sc_m(st.h.y, st.h.z, st.h.w, 2 * c + 1, sc1, m1);
    const float step0 = d * (float)sc0, off0 = dmin * (float)m0;
    const float step1 = d * (float)sc1, off1 = dmin * (float)m1;
    const float2 s0 = make_float2(step0, step0), n0 = make_float2(-off0, -off0);
    const float2 s1 = make_float2(step1, step1), n1 = make_float2(-off1, -off1);
    const uint32_t words[8] = {st.q0.x, st.q0.y, st.q0.z, st.q0.w, st.q1.x, st.q1.y, st.q1.z, st.q1.w};
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const uint32_t w = words[t];
        q4k_quad(w & 0x0F0F0F0Fu, s0, n0, o + 2 * t);             // k = 4t .. 4t+3
        q4k_quad((w >> 4) & 0x0F0F0F0Fu, s1, n1, o + 16 + 2 * t); // k = 32 + 4t ..
    }
}

// ------------------------------------------------------------ the kernel
template <int FMT> struct StageOf;
template <> struct StageOf<Q4_NVFP4> { using T = NvStage; };
template <> struct StageOf<Q4_Q4K> { using T = QkStage; };

template <int FMT>
__device__ __forceinline__ void load_stage(const TcArgs &a, const uint8_t *wrow, const uint8_t *srow, int i,
                                           typename StageOf<FMT>::T &st) {
    if constexpr (FMT == Q4_NVFP4) {
        st.a = ldg_stream16(wrow + 32 * i);
        st.b = ldg_stream16(wrow + 32 * i + 16);
        st.s = ldg_stream4(srow + 4 * i);
    } else {
        const uint8_t *blk = wrow + (i >> 2) * 144;
        st.h = ldg_stream16(blk);
        st.q0 = ldg_stream16(blk + 16 + 32 * (i & 3));
        st.q1 = ldg_stream16(blk + 32 + 32 * (i & 3));
    }
}

template <int FMT, int MB>
__global__ void __launch_bounds__(THREADS, 2)
    gemm_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tmx) {
    using C = Cfg<MB>;
    using Stage = typename StageOf<FMT>::T;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full_bar[C::NS], empty_bar[C::NS], done_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    uint8_t *xring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / a.splits, rank = blockIdx.x % a.splits;
    const int64_t n0 = (int64_t)tile * ROWS;
    const int64_t kbeg = (int64_t)rank * a.k_per_cta;
    const int nst = a.k_per_cta / BK;
    volatile int *abort_flag = &abort_s;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; s++) {
            mbar_init(&full_bar[s], ROWS + 1);   // 128 decode threads + the TMA thread (with its bytes)
            mbar_init(&empty_bar[s], 1);         // one tcgen05.commit
        }
        mbar_init(&done_bar, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 4) tmem_alloc(&tmem_base_s);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;
    bool aborted = false;

    if (warp < 4) {
        // ---------------------------------------------------------- decode
        const int r = threadIdx.x;
        const int64_t n = n0 + r;
        const bool valid = n < a.N;
        const uint8_t *wrow, *srow = nullptr;
        if constexpr (FMT == Q4_NVFP4) {
            wrow = a.w + (valid ? n : 0) * (a.K / 2) + kbeg / 2;
            srow = a.s + (valid ? n : 0) * (a.K / 16) + kbeg / 16;
        } else {
            wrow = a.w + ((valid ? n : 0) * (a.K / 256) + kbeg / 256) * 144;
        }
        const uint32_t lane_base = tbase + ((uint32_t)(r & ~31) << 16) + C::DCOLS;
        Stage ring[PD];
#pragma unroll
        for (int p = 0; p < PD; p++) {
            ring[p] = Stage{};
            if (valid && p < nst) load_stage<FMT>(a, wrow, srow, p, ring[p]);
        }
        for (int i0 = 0; i0 < nst && !aborted; i0 += PD) {
#pragma unroll
            for (int p = 0; p < PD; p++) {
                const int i = i0 + p;
                if (i < nst && !aborted) {
                    const Stage cur = ring[p];
                    if (valid && i + PD < nst) load_stage<FMT>(a, wrow, srow, i + PD, ring[p]);
                    uint32_t o[32];
                    if constexpr (FMT == Q4_NVFP4)
                        nvfp4_stage(cur, o);
                    else
                        q4k_stage(cur, p & 3, o);   // kbeg % 256 == 0 and PD % 4 == 0: chunk = p % 4
                    const int s = i % C::NS;
                    bool ok = i < C::NS || wait_or_abort(&empty_bar[s], ((i / C::NS) & 1) ^ 1, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);   // tcgen05.st is warp-collective
                    if (!ok) {
                        aborted = true;
                    } else {
                        tc_fence_after();
                        tmem_st32(lane_base + s * A_COLS, o);
                        tc_fence_before();
                        mbar_arrive(&full_bar[s]);
                    }
                }
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16<MB>();
            for (int i = 0; i < nst; i++) {
                const int s = i % C::NS;
                if (!wait_or_abort(&full_bar[s], (i / C::NS) & 1, abort_flag)) break;
                tc_fence_after();
                const uint32_t a_col = tbase + C::DCOLS + s * A_COLS;
                const uint32_t b_addr = smem_u32(xring + s * C::B_BYTES);
#pragma unroll
                for (int j = 0; j < BK / 16; j++)
                    mma_ts(tbase, a_col + j * 8, sw128_desc(b_addr + j * 32), idesc, (i | j) != 0);
                mma_commit(&empty_bar[s]);
            }
            mma_commit(&done_bar);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- L2 warm-up + TMA
        for (int r = lane; r < ROWS; r += 32) {
            const int64_t n = n0 + r;
            if (n >= a.N) break;
            if constexpr (FMT == Q4_NVFP4) {
                prefetch_l2(a.w + n * (a.K / 2) + kbeg / 2, (uint32_t)(a.k_per_cta / 2));
                prefetch_l2(a.s + n * (a.K / 16) + kbeg / 16, (uint32_t)(a.k_per_cta / 16));
            } else {
                prefetch_l2(a.w + (n * (a.K / 256) + kbeg / 256) * 144, (uint32_t)(a.k_per_cta / 256 * 144));
            }
        }
        if (lane == 0) {
            for (int i = 0; i < nst; i++) {
                const int s = i % C::NS;
                if (i >= C::NS && !wait_or_abort(&empty_bar[s], ((i / C::NS) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(&full_bar[s], C::B_BYTES);
                tma_2d(xring + s * C::B_BYTES, &tmx, (int)(kbeg + (int64_t)i * BK), 0, &full_bar[s]);
            }
        }
        __syncwarp();
    }

    // ---------------------------------------------------------- epilogue
    float *red = reinterpret_cast<float *>(xring);   // [MB][128] partial tile; the X ring is idle now
    if (warp < 4) {
        const int r = threadIdx.x;
        const int64_t n = n0 + r;
        bool ok = !aborted && wait_or_abort(&done_bar, 0, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            const uint32_t lane_d = tbase + ((uint32_t)(r & ~31) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < MB; c0 += 16) {
                float v[16];
                tmem_ld16(lane_d + c0, v);
                if (a.splits == 1) {
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
    }
    if (a.splits > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();   // every partial tile of the cluster is in shared memory
        if (warp < 4 && !*abort_flag) {
            const int r = threadIdx.x;
            const int64_t n = n0 + r;
            const int cols = MB / a.splits;
            for (int c = rank * cols; c < (rank + 1) * cols; c++) {
                float acc = 0.0f;
                for (int q = 0; q < a.splits; q++) acc += cluster.map_shared_rank(red, q)[c * ROWS + r];
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
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tbase);
    }
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

// Tensor map of one batch chunk of x (bf16 [rows][K]): 64 k x MB rows per
// box, 128-byte swizzle; rows past `rows` read as zero.
bool encode_x(CUtensorMap *map, const void *x, int64_t K, int64_t rows, int MB) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)MB};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K slice per CTA: split K over up to 8 cluster ranks until the grid holds
// about two CTAs per SM, keeping every slice >= 4 stages and (Q4_K) whole
// super-blocks.
int pick_splits(int64_t tiles, int64_t K, q4_fmt fmt) {
    const int64_t sms = sm_count();
    const int64_t unit = fmt == Q4_Q4K ? 256 : 4 * BK;
    int S = 1;
    while (S < 8 && tiles * S < 2 * sms && K % (2 * S) == 0 && (K / (2 * S)) % unit == 0) S *= 2;
    return S;
}

template <int FMT, int MB>
cudaError_t launch_one(const TcArgs &args, const CUtensorMap &map, int64_t tiles, cudaStream_t s) {
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
    return cudaLaunchKernelEx(&cfg, kern, args, map);
}

template <int FMT>
cudaError_t launch_mb(int MB, const TcArgs &args, const CUtensorMap &map, int64_t tiles, cudaStream_t s) {
    switch (MB) {
    case 16: return launch_one<FMT, 16>(args, map, tiles, s);
    case 32: return launch_one<FMT, 32>(args, map, tiles, s);
    case 64: return launch_one<FMT, 64>(args, map, tiles, s);
    default: return launch_one<FMT, 128>(args, map, tiles, s);
    }
}

}  // namespace

bool gemm_tc_eligible(const Tensor &t, q4_dtype x_dtype, int64_t M) {
    return M >= 9 && x_dtype == Q4_DT_BF16 && (t.fmt == Q4_NVFP4 || t.fmt == Q4_Q4K) && t.K % (4 * BK) == 0 &&
           t.K <= (1LL << 30) && (t.N + ROWS - 1) / ROWS * 8 <= (1LL << 31) - 1;
}

cudaError_t launch_gemm_tc(const Tensor &t, const void *x, q4_dtype x_dtype, float *y, int64_t M, cudaStream_t s,
                           bool *handled) {
    *handled = false;
    if (!gemm_tc_eligible(t, x_dtype, M)) return cudaSuccess;
    *handled = true;
    note_gemv_path("gemm_tc");
    const int64_t tiles = (t.N + ROWS - 1) / ROWS;
    const int S = pick_splits(tiles, t.K, t.fmt);
    for (int64_t m0 = 0; m0 < M; m0 += 128) {
        const int64_t rows = M - m0 < 128 ? M - m0 : 128;
        const int MB = rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
        CUtensorMap map;
        if (!encode_x(&map, (const uint8_t *)x + m0 * t.K * 2, t.K, rows, MB)) return cudaErrorInvalidValue;
        TcArgs args;
        args.w = t.w;
        args.s = t.scales;
        args.y = y + m0 * t.N;
        args.N = t.N;
        args.K = t.K;
        args.M = (int)rows;
        args.splits = S;
        args.k_per_cta = (int)(t.K / S);
        args.mult = t.fmt == Q4_NVFP4 ? t.scale2 : 1.0f;
        const cudaError_t e = t.fmt == Q4_NVFP4 ? launch_mb<Q4_NVFP4>(MB, args, map, tiles, s)
                                                : launch_mb<Q4_Q4K>(MB, args, map, tiles, s);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

int gemv_read_and_clear_error();

int read_and_clear_device_error() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    const int g = gemv_read_and_clear_error();
    return v ? v : g;
}

}  // namespace q4

extern "C" int q4_last_error(void) { return q4::read_and_clear_device_error(); }
