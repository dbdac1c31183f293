// gemv_fp4tc.cu -- batch-1 NVFP4 decode-GEMV on the native block-scaled FP4
// tensor cores (tcgen05.mma.kind::mxf4nvf4.block_scale), sm_103a.
//
// y[n] = scale2 * sum_k (e2m1 * e4m3)[n][k] * x[k]  ([MUS7] 7.1-7.2: the
// product e2m1 * e4m3 is exact and scale2 multiplies once).  The weights are
// never decoded on the CUDA cores: tensor TMA lands 128-row x 256-k slots of
// the packed payload in shared memory in the 128-byte-swizzled K-major form
// the MMA reads, and the MMA applies the E4M3 group scales itself (A scale
// factors in tensor memory).
//
// Activations.  bf16 x is not FP4, but every 16-value block of it is exactly
// a sum of 16 FP4 "slices": with t_b the block's top exponent + 1 (every
// |x| < 2^t_b), slice p holds each element's magnitude bits [t_b-2p-2, t_b-2p)
// as one E2M1 digit d in {0, 1, 2, 3} (codes 0, 2, 4, 5) with the element's
// sign.  Slice p is column p of the MMA's B (N = 16).  Column p is scaled by
// 2^(2p + 10 - T) (T = the top t_b over this CTA's k range), which gives every
// slice of block b the same UE4M3 scale 2^(t_b - T + 8): one B scale word per
// MMA, shared by all 16 columns.  The epilogue undoes the column shifts,
// adds the columns in slice order and multiplies by scale2.
//
// Residual blocks.  A 16-value block the slices cannot hold exactly -- an
// element more than 2^24 below its block's top (bits past slice 15), a block
// more than 2^17 below T (its scale would fall under UE4M3's 2^-9), or a
// subnormal or non-finite element -- gets zero slices; the scale warps then
// compute it on the CUDA cores from the weight bytes already in shared
// memory (exact e2m1 * e4m3 times x, f32), so every finite x is handled.
//
// Roles (192 threads): warp 0 streams the weight slots (TMA, L2 evict-first);
// warp 1 owns tensor memory and issues the MMAs (4 per slot, 64 k each);
// warps 2-5 slice x, move each slot's scale factors into tensor memory, run
// the residual blocks and the epilogue (warp w serves TMEM lanes 32*(w%4)..).
// Scale-factor layout in tensor memory (measured on the GB300 with a
// one-CTA probe): the factors of A row r for one MMA sit in lane r, column
// base + r/32, byte = 16-k block; each MMA's factors take 4 columns whose
// base must be a multiple of 4 (the layout tcgen05.cp .32x128b.warpx4 makes).
//
// Programmatic dependent launch: the producer streams weights before the
// previous launch has finished; x is read and y written only after
// griddepcontrol.wait.  Every wait is bounded (~1 s of SM clocks): a timeout
// records Q4_ETIMEOUT, the roles stop, bulk copies and MMAs in flight are
// waited for, tensor memory is freed, and the kernel returns.
#include <cooperative_groups.h>

#include "q4_internal.cuh"
#include "tma_map.cuh"

namespace q4 {

__device__ int g_fp4_error;
// Limit of the role waits, in SM clocks (the drains of bulk copies and MMAs
// before exit keep the full limit).
__device__ long long g_fp4_wait_limit = 1LL << 31;

namespace {

constexpr int ROWS = 128;                     // weight rows per tile = MMA M = TMEM lanes
constexpr int SLOT_K = 256;                   // k per ring slot: 4 MMAs of 64
constexpr int PAY = ROWS * 128;               // A payload box: 128 rows x 128 B, 128-byte swizzle
constexpr int SCB = ROWS * 16;                // A scale box: 128 rows x 16 B
constexpr int NW = 4;                         // ring slots
constexpr int P = 16;                         // MMA N: the slices, or up to 16 activation rows
constexpr int BPLANE = P * 128;               // one 256-k block of B, swizzled like A
constexpr int BSC = P * 16;                   // B scale box: 16 rows x 16 B
// Slot layouts.  Slices mode: A payload | A scales (18 KB).  Activation mode
// (x already NVFP4): A payload | B payload | A scales | B scales, padded to
// 21 KB; every slot and both payload boxes start on 1024-byte boundaries.
constexpr int SLOT_SL = PAY + SCB;
constexpr int XQ_BPAY = PAY, XQ_ASC = PAY + BPLANE, XQ_BSC = XQ_ASC + SCB;
constexpr int SLOT_XQ = 21 * 1024, TX_XQ = XQ_BSC + BSC;
constexpr int D_COL = 0, SFA_COL = 16, SFB_COL = SFA_COL + NW * 4 * 4;
constexpr int TMEM_COLS = 256;                // 16 + 64 + 64 columns used
constexpr int THREADS = 6 * 32;
constexpr int W_TMA = 0, W_MMA = 1;
constexpr int MAXG = 8;                       // matrices that share x in one launch
constexpr long long WAIT_LIMIT = 1LL << 31;   // ~1 s of SM clocks
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(P >> 3) << 17) | ((uint32_t)(ROWS >> 4) << 24);
static_assert(SLOT_SL % 1024 == 0 && SLOT_XQ % 1024 == 0 && XQ_BPAY % 1024 == 0, "swizzle atoms stay aligned");
static_assert(TX_XQ <= SLOT_XQ, "activation-mode slot");
static_assert(SFB_COL + NW * 4 * 4 <= TMEM_COLS, "tensor memory budget");

template <bool XQ> constexpr int slot_bytes() { return XQ ? SLOT_XQ : SLOT_SL; }

struct Fp4Args {
    float *y[MAXG];
    int64_t N[MAXG];
    float scale2[MAXG];
    int tile_start[MAXG + 1];     // first tile of each member; tile_start[count] = all tiles
    int count;
    const __nv_bfloat16 *x;       // slices mode: bf16 x [K]
    int M;                        // activation mode: rows of this launch (<= 16); y is [M][N]
    float x_scale2;               // activation mode: the activations' NVFP4 tensor scale
    int64_t K;
    int k_per_cta;                // the k range of one CTA (whole slots; the last rank's may be shorter)
    int splits;                   // CTAs of a cluster splitting K; partial rows summed in rank order
    int share;                    // slices mode, splits == 1: CTAs of a cluster (consecutive tiles) that
                                  // build the x slices together, each a 1/share part, pushed to the others
};
struct Fp4Maps {
    CUtensorMap w[MAXG];          // payload u8 [N][K/2], box 128 x 128, 128-byte swizzle
    CUtensorMap s[MAXG];          // scales u8 [N][K/16], box 16 x 128
    CUtensorMap xq, xs;           // activation mode: payload [M][K/2] (box 128 x 16, swizzled), scales [M][K/16]
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
__device__ __forceinline__ void mma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb, uint32_t acc) {
    asm volatile("{ .reg .pred p;\n\t setp.ne.b32 p, %5, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %6, [%3], [%4], p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(sfa), "r"(sfb), "r"(acc), "r"(IDESC)
                 : "memory");
}
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tst4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint64_t evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma2(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma2_plain(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
                 : "memory");
}
// Bulk copy of `bytes` (16-byte multiple, 16-byte aligned) from this CTA's
// shared memory to the same offset in cluster rank `peer`, counted on that
// rank's mbarrier `bar`.
__device__ __forceinline__ void push_to_peer(const void *src, uint32_t bytes, uint64_t *bar, uint32_t peer) {
    uint32_t dst, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(smem_u32(src)), "r"(peer));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_u32(bar)), "r"(peer));
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "r"(smem_u32(src)), "r"(bytes), "r"(rbar)
                 : "memory");
}
// Bounded wait that also gives up when another role has raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64(), limit = g_fp4_wait_limit;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            atomicExch(&g_fp4_error, Q4_ETIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}
// UE4M3 encoding of 2^u, u in [-9, 8].
__device__ __forceinline__ uint32_t ue4m3_pow2(int u) { return u >= -6 ? (uint32_t)(u + 7) << 3 : 1u << (u + 9); }

__device__ __forceinline__ void load16_bf16(const __nv_bfloat16 *p, uint32_t u[16]) {
    const uint4 a = *reinterpret_cast<const uint4 *>(p), b = *reinterpret_cast<const uint4 *>(p + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; i++) {
        u[2 * i] = w[i] & 0xffffu;
        u[2 * i + 1] = w[i] >> 16;
    }
}

// Top exponent + 1 of a block's normal finite elements (-1000 if none).
__device__ __forceinline__ int block_top(const uint32_t u[16]) {
    int t = -1000;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const int E = (int)((u[i] >> 7) & 0xffu);
        if (E != 0 && E != 255) t = max(t, E - 126);
    }
    return t;
}

// Slices p0 .. p1-1 of the 16-value bf16 block b of this CTA's k range (see
// the file header) into the B planes; the thread with p0 == 0 also writes the
// block's B scale byte: 2^(t_b - T + 8) in UE4M3, or 0 for a residual block
// (a value the slices never use: their smallest scale is 2^-9 = byte 1).
// Branch-free: each element's 8-bit significand m24 (top bit set) is shifted
// right by its distance below the block's top (shifts of 32 or more give 0);
// shifting back and comparing tells whether bits fell off the end.
__device__ void slice_block(const __nv_bfloat16 *xr, int b, int T, int p0, int p1, uint8_t *bplanes, uint8_t *sfb) {
    const uint4 qa = *reinterpret_cast<const uint4 *>(xr + b * 16), qb = *reinterpret_cast<const uint4 *>(xr + b * 16 + 8);
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    uint32_t E[16], u[16];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        u[2 * i] = w[i] & 0xffffu;
        u[2 * i + 1] = w[i] >> 16;
    }
    int tb_ = -1000;
    uint32_t special = 0u;                                               // a subnormal or non-finite element
#pragma unroll
    for (int i = 0; i < 16; i++) {
        E[i] = (u[i] >> 7) & 0xffu;
        const bool normal = E[i] - 1u < 254u;                             // biased exponent 1 .. 254
        tb_ = normal ? max(tb_, (int)E[i] - 126) : tb_;
        special |= (E[i] == 255u) | ((E[i] == 0u) & ((u[i] & 0x7fu) != 0u));
    }
    const int C = tb_ + 126;                                              // shift = C - E
    uint32_t A[16], lost = 0u, slo = 0u, shi = 0u;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const uint32_t m24 = (u[i] << 24) | 0x80000000u;                  // value bit j at word bit j + 32 - tb_
        const uint32_t sh = (uint32_t)(C - (int)E[i]);
        uint32_t a, back;
        asm("shr.b32 %0, %1, %2;" : "=r"(a) : "r"(m24), "r"(sh));
        asm("shl.b32 %0, %1, %2;" : "=r"(back) : "r"(a), "r"(sh));
        const bool normal = E[i] - 1u < 254u;
        A[i] = normal ? a : 0u;
        lost |= normal & (back != m24);
        if (i < 8) slo |= (u[i] >> 15) << (4 * i + 3);                    // the sign bit of each nibble
        else shi |= (u[i] >> 15) << (4 * (i - 8) + 3);
    }
    const bool resid = special | lost | (tb_ != -1000 && tb_ - T + 8 < -9);   // scale below UE4M3's 2^-9
    // transpose the 16 x 16 matrix of 2-bit cells: word q <- cell q of every element
#pragma unroll
    for (int stage = 0; stage < 4; stage++) {
        const int st = 8 >> stage;
        const uint32_t mask =
            stage == 0 ? 0x0000FFFFu : stage == 1 ? 0x00FF00FFu : stage == 2 ? 0x0F0F0F0Fu : 0x33333333u;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            if (i & st) continue;
            const uint32_t t2 = ((A[i] >> (2 * st)) ^ A[i + st]) & mask;
            A[i + st] ^= t2;
            A[i] ^= t2 << (2 * st);
        }
    }
    const int kk = b * 16, plane = kk / SLOT_K, c = (kk % SLOT_K) / 2;   // byte offset in the 128-B row
#pragma unroll
    for (int p = 0; p < P; p++) {
        if (p < p0 || p >= p1) continue;
        uint32_t h[2] = {0u, 0u};
        if (!resid) {
            const uint32_t Wd = A[15 - p];
#pragma unroll
            for (int q = 0; q < 2; q++) {
                uint32_t xx = q ? Wd >> 16 : Wd & 0xFFFFu;              // 2-bit digits -> one per nibble
                xx = (xx | (xx << 8)) & 0x00FF00FFu;
                xx = (xx | (xx << 4)) & 0x0F0F0F0Fu;
                xx = (xx | (xx << 2)) & 0x33333333u;
                h[q] = ((xx << 1) - ((xx >> 1) & xx & 0x11111111u)) | (q ? shi : slo);   // digit -> E2M1 code
            }
        }
        uint8_t *row = bplanes + plane * BPLANE + (p >> 3) * 1024 + (p & 7) * 128;
        *reinterpret_cast<uint2 *>(row + (((c >> 4) ^ (p & 7)) << 4) + (c & 15)) = make_uint2(h[0], h[1]);
    }
    if (p0 == 0) sfb[b] = resid ? 0u : (uint8_t)ue4m3_pow2(tb_ == -1000 ? 0 : tb_ - T + 8);
}

// Dynamic shared memory after the 1024-byte alignment: the ring, then
// (slices mode) the B planes and the B scale bytes, then the partial rows
// (P columns in activation mode, one in slices mode).
template <bool XQ> __host__ __device__ inline int64_t planes_off() { return (int64_t)NW * slot_bytes<XQ>(); }
__host__ __device__ inline int64_t sfb_off(int nslots) { return planes_off<false>() + (int64_t)nslots * BPLANE; }
template <bool XQ> __host__ __device__ inline int64_t red_off(int nslots) {
    return XQ ? planes_off<true>() : sfb_off(nslots) + nslots * 16;
}
template <bool XQ> int64_t smem_for(int nslots) { return 1024 + red_off<XQ>(nslots) + (XQ ? P : 1) * ROWS * 4; }

template <bool XQ>
__global__ void __launch_bounds__(THREADS, 2)
gemv_fp4tc_kernel(const __grid_constant__ Fp4Args a, const __grid_constant__ Fp4Maps maps) {
    constexpr int SLOT = slot_bytes<XQ>();
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[NW], empty[NW], sf_full[NW], done_bar, sliced_bar, slices_in, x_bar;
    __shared__ uint32_t tbase_s;
    __shared__ int abort_s, topT;
    uint8_t *wring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int rank = blockIdx.x % a.splits;
    const int kbeg = rank * a.k_per_cta;
    const int kcount = (int)min((int64_t)a.k_per_cta, a.K - kbeg);      // >= 256: every rank owns a slot
    const int nslots = kcount / SLOT_K, nblk = kcount / 16;
    const int max_slots = a.k_per_cta / SLOT_K;                          // the layout is the same on every rank
    // Slices mode: x of this CTA's range arrives by one bulk copy into the
    // ring's last slot, whose weights wait until the slices are built.
    const bool xstage = !XQ && kcount * 2 <= SLOT;
    const bool hold = xstage && nslots >= NW;
    uint8_t *xbuf = wring + (NW - 1) * SLOT;
    uint8_t *bplanes = wring + planes_off<XQ>();                         // slices mode: [nslots][16][128 B]
    uint8_t *sfb = wring + sfb_off(max_slots);                           // slices mode: [nblk] B scale bytes
    float *red = reinterpret_cast<float *>(wring + red_off<XQ>(max_slots));   // [XQ ? P : 1][ROWS]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / a.splits;
    int mb = 0;
    while (mb + 1 < a.count && tile >= a.tile_start[mb + 1]) mb++;
    const int64_t n0 = (int64_t)(tile - a.tile_start[mb]) * ROWS;
    volatile int *abort_flag = &abort_s;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NW; s++) {
            mbar_init(&full[s], 1);          // the producer's arrive + the slot's bytes
            mbar_init(&empty[s], 1);         // one tcgen05.commit
            mbar_init(&sf_full[s], 4);       // one arrive per scale warp
        }
        mbar_init(&done_bar, 1);
        mbar_init(&sliced_bar, 4);
        mbar_init(&slices_in, 1);            // this CTA's arrive + the bytes its cluster peers push
        mbar_init(&x_bar, 1);                // the x bulk copy
        if (!XQ && a.share > 1) {
            const int per = (a.k_per_cta / SLOT_K) / a.share;
            mbar_arrive_expect_tx(&slices_in, (uint32_t)((a.share - 1) * per * (BPLANE + 16)));
        }
        abort_s = 0;
        topT = -1000;
        fence_mbar_init();
    }
    __syncthreads();
    const int share = XQ ? 1 : a.share;
    if (share > 1) {
        // every peer's barriers are initialised before any slice is pushed
        namespace cg = cooperative_groups;
        cg::this_cluster().sync();
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // The weight stream starts at once.  Tensor memory may still be held by
    // the previous launch's CTAs on this SM, so its allocation (warp 1) and
    // the wait for it (bar 2: warps 1-5) come after the x slices are built.
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tbase_s)),
                     "n"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    }

    if (warp == W_TMA) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = evict_first();
            constexpr uint32_t TX = XQ ? TX_XQ : SLOT_SL;
            int issued = 0;
            const int pre = nslots < NW ? nslots : NW;
            const int first = hold ? NW - 1 : pre;
            // weights of the first slots before the dependency on the previous launch resolves
            for (int j = 0; j < first; j++) {
                const uint32_t slot = smem_u32(wring + j * SLOT);
                mbar_arrive_expect_tx(&full[j], TX);
                tma2(slot, &maps.w[mb], (kbeg + j * SLOT_K) / 2, (int)n0, &full[j], pol);
                tma2(slot + (XQ ? XQ_ASC : PAY), &maps.s[mb], (kbeg + j * SLOT_K) / 16, (int)n0, &full[j], pol);
                issued++;
            }
            if (XQ) {
                // the activations are the previous launch's output
                asm volatile("griddepcontrol.wait;" ::: "memory");
                for (int j = 0; j < pre; j++) {
                    const uint32_t slot = smem_u32(wring + j * SLOT);
                    tma2_plain(slot + XQ_BPAY, &maps.xq, (kbeg + j * SLOT_K) / 2, 0, &full[j]);
                    tma2_plain(slot + XQ_BSC, &maps.xs, (kbeg + j * SLOT_K) / 16, 0, &full[j]);
                }
            }
            bool go = true;
            if (hold) {
                // the last slot held x: its weights follow once the slices are built
                go = wait_or_abort(&sliced_bar, 0, abort_flag);
                if (go) {
                    const uint32_t slot = smem_u32(wring + (NW - 1) * SLOT);
                    mbar_arrive_expect_tx(&full[NW - 1], TX);
                    tma2(slot, &maps.w[mb], (kbeg + (NW - 1) * SLOT_K) / 2, (int)n0, &full[NW - 1], pol);
                    tma2(slot + PAY, &maps.s[mb], (kbeg + (NW - 1) * SLOT_K) / 16, (int)n0, &full[NW - 1], pol);
                    issued++;
                }
            }
            for (int j = pre; j < nslots && go; j++) {
                const int s = j % NW;
                if (!wait_or_abort(&empty[s], ((j / NW) & 1) ^ 1, abort_flag)) break;
                const uint32_t slot = smem_u32(wring + s * SLOT);
                mbar_arrive_expect_tx(&full[s], TX);
                tma2(slot, &maps.w[mb], (kbeg + j * SLOT_K) / 2, (int)n0, &full[s], pol);
                tma2(slot + (XQ ? XQ_ASC : PAY), &maps.s[mb], (kbeg + j * SLOT_K) / 16, (int)n0, &full[s], pol);
                if (XQ) {
                    tma2_plain(slot + XQ_BPAY, &maps.xq, (kbeg + j * SLOT_K) / 2, 0, &full[s]);
                    tma2_plain(slot + XQ_BSC, &maps.xs, (kbeg + j * SLOT_K) / 16, 0, &full[s]);
                }
                issued++;
            }
            // every copy issued has landed before the CTA may exit
            for (int q = issued > NW ? issued - NW : 0; q < issued; q++)
                if (!mbar_wait_bounded(&full[q % NW], (uint32_t)((q / NW) & 1), WAIT_LIMIT))
                    atomicExch(&g_fp4_error, Q4_ETIMEOUT);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ------------------------------------------------------- MMA issue
        asm volatile("bar.sync 2, 160;" ::: "memory");
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t tb = tbase_s;
        if (lane == 0) {
            bool ok = XQ || wait_or_abort(&sliced_bar, 0, abort_flag);
            const uint32_t bbase = smem_u32(bplanes);
            for (int j = 0; j < nslots && ok; j++) {
                const int s = j % NW;
                const uint32_t par = (uint32_t)(j / NW) & 1;
                ok = wait_or_abort(&full[s], par, abort_flag) && wait_or_abort(&sf_full[s], par, abort_flag);
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t abase = smem_u32(wring + s * SLOT);
                const uint32_t bb = XQ ? abase + XQ_BPAY : bbase + j * BPLANE;
#pragma unroll
                for (int q = 0; q < 4; q++)
                    mma_fp4(tb + D_COL, sw128_desc(abase + 32 * q), sw128_desc(bb + 32 * q),
                            tb + SFA_COL + (s * 4 + q) * 4, tb + SFB_COL + (s * 4 + q) * 4, (uint32_t)(j | q));
                commit(&empty[s]);
            }
            commit(&done_bar);
            // no MMA may still write tensor memory when it is freed
            if (!mbar_wait_bounded(&done_bar, 0, WAIT_LIMIT)) atomicExch(&g_fp4_error, Q4_ETIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------ x slices, scale factors (warps 2-5)
        const int t = threadIdx.x - 64;                                  // 0..127
        const __nv_bfloat16 *xr = a.x + kbeg;
        if (!XQ) {
            // L2 is the coherence point: lines fetched now still see the previous launch's writes
            for (int l = t; l < kcount / 64; l += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(xr + l * 64));
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");              // x (and y) belong to the previous launch
        int T = 0;
        if (!XQ) {
            const __nv_bfloat16 *xs = xr;                                // where the slicing reads x
            if (xstage) {
                if (t == 0) {
                    mbar_arrive_expect_tx(&x_bar, (uint32_t)(kcount * 2));
                    bulk_g2s(xbuf, xr, (uint32_t)(kcount * 2), &x_bar);
                }
                wait_or_abort(&x_bar, 0, abort_flag);
                xs = reinterpret_cast<const __nv_bfloat16 *>(xbuf);
            }
            int tmax = -1000;
            for (int b = t; b < nblk; b += 128) {
                uint32_t u[16];
                load16_bf16(xs + b * 16, u);
                tmax = max(tmax, block_top(u));
            }
            atomicMax(&topT, tmax);
            asm volatile("bar.sync 1, 128;" ::: "memory");
            T = topT == -1000 ? 0 : topT;                                // an all-zero range has no slices
            if (share == 1) {
                for (int b = t; b < nblk; b += 128) slice_block(xs, b, T, 0, P, bplanes, sfb);
            } else {
                // this rank's 1/share of the planes: lane = block, warp w = slices 4w .. 4w+3
                // (warp-uniform, so no lane idles through another's slices); then one thread
                // per peer sends the planes and the scale bytes by two bulk copies
                const int per = nslots / share, me = (int)(blockIdx.x % (unsigned)share);
                const int b0 = me * per * 16, nb = per * 16, sw = t >> 5;
                for (int bi = lane; bi < nb; bi += 32) slice_block(xs, b0 + bi, T, 4 * sw, 4 * sw + 4, bplanes, sfb);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (t >= 1 && t < share) {
                    const uint32_t peer = (uint32_t)((me + t) % share);
                    push_to_peer(bplanes + me * per * BPLANE, (uint32_t)(per * BPLANE), &slices_in, peer);
                    push_to_peer(sfb + b0, (uint32_t)(per * 16), &slices_in, peer);
                }
                if (!wait_or_abort(&slices_in, 0, abort_flag)) {
                    // a peer's slices did not arrive: nothing of this range is multiplied
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // slices -> the MMA's async proxy
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (lane == 0) mbar_arrive(&sliced_bar);
        }
        asm volatile("bar.sync 2, 160;" ::: "memory");                  // tensor memory allocated
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t tb = tbase_s;

        // ---- per slot: scale factors into tensor memory, residual blocks on the CUDA cores
        const int r = (warp & 3) * 32 + lane;                            // TMEM lane = weight row
        const uint32_t lane_addr = tb + ((uint32_t)((warp & 3) * 32) << 16);
        float resid_acc = 0.0f;
        for (int j = 0; j < nslots; j++) {
            const int s = j % NW;
            if (!wait_or_abort(&full[s], (uint32_t)(j / NW) & 1, abort_flag)) break;
            if (j >= NW && !wait_or_abort(&empty[s], ((j / NW) & 1) ^ 1, abort_flag)) break;   // slot j-NW's MMAs done
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint8_t *slot = wring + s * SLOT;
            const uint8_t *scl = slot + (XQ ? XQ_ASC : PAY);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                uint32_t v[4];
#pragma unroll
                for (int cc = 0; cc < 4; cc++) v[cc] = *reinterpret_cast<const uint32_t *>(scl + (lane + 32 * cc) * 16 + 4 * q);
                tst4(lane_addr + SFA_COL + (s * 4 + q) * 4, v[0], v[1], v[2], v[3]);
                uint32_t bsf;
                if (XQ) bsf = lane < P ? *reinterpret_cast<const uint32_t *>(slot + XQ_BSC + lane * 16 + 4 * q) : 0u;
                else bsf = lane < P ? reinterpret_cast<const uint32_t *>(sfb)[j * 4 + q] : 0u;
                tst4(lane_addr + SFB_COL + (s * 4 + q) * 4, bsf, 0u, 0u, 0u);
            }
            if (!XQ) {
                const uint4 sw = *reinterpret_cast<const uint4 *>(sfb + j * 16);   // this slot's 16 B scale bytes
                const uint32_t z = ((sw.x - 0x01010101u) & ~sw.x) | ((sw.y - 0x01010101u) & ~sw.y) |
                                   ((sw.z - 0x01010101u) & ~sw.z) | ((sw.w - 0x01010101u) & ~sw.w);
                if (z & 0x80808080u) {                                   // some byte is 0: a residual block
                    for (int bb = 0; bb < 16; bb++) {
                        if (sfb[j * 16 + bb] != 0) continue;
                        const int kk = j * SLOT_K + bb * 16, c = bb * 8;
                        const uint2 codes =
                            *reinterpret_cast<const uint2 *>(slot + r * 128 + (((c >> 4) ^ (r & 7)) << 4) + (c & 15));
                        const float sc = e4m3_f32(scl[r * 16 + bb]);
                        uint32_t u[16];
                        load16_bf16(xr + kk, u);
                        const uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float2 w2 = e2m1x2_f32((cw[i >> 3] >> (4 * (i & 7))) & 0xffu);
                            resid_acc = __fmaf_rn(__fmul_rn(w2.x, sc), __uint_as_float(u[i] << 16), resid_acc);
                            resid_acc = __fmaf_rn(__fmul_rn(w2.y, sc), __uint_as_float(u[i + 1] << 16), resid_acc);
                        }
                    }
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&sf_full[s]);
        }
        // ---- epilogue.  Slices: column p times 2^-(2p + 10 - T), in slice order, plus the
        // residual blocks.  Activation mode: column m is batch row m.
        float v[16];
#pragma unroll
        for (int p = 0; p < P; p++) v[p] = 0.0f;
        if (wait_or_abort(&done_bar, 0, abort_flag)) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]),
                  "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
                : "r"(lane_addr + D_COL)
                : "memory");
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        }
        if (XQ) {
#pragma unroll
            for (int p = 0; p < P; p++) red[p * ROWS + r] = v[p];
        } else {
            float acc = 0.0f;
#pragma unroll
            for (int p = 0; p < P; p++) acc += ldexpf(v[p], T - 2 * p - 10);
            red[r] = acc + resid_acc;
        }
    }
    const int ncols = XQ ? a.M : 1;
    const float outscale = XQ ? a.scale2[mb] * a.x_scale2 : a.scale2[mb];
    if (a.splits > 1) {
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();                                                  // every rank's partial rows are in place
        if (warp >= 2) {
            const int r = (warp & 3) * 32 + lane;
            if (r % a.splits == rank && n0 + r < a.N[mb]) {             // rows spread over the ranks
                for (int m = 0; m < ncols; m++) {
                    float acc = cluster.map_shared_rank(red, 0)[m * ROWS + r];
                    for (int q = 1; q < a.splits; q++) acc += cluster.map_shared_rank(red, q)[m * ROWS + r];   // rank order
                    a.y[mb][m * a.N[mb] + n0 + r] = acc * outscale;
                }
            }
        }
        cluster.sync();                                                  // no rank leaves while its rows may be read
    } else if (warp >= 2) {
        const int r = (warp & 3) * 32 + lane;
        if (n0 + r < a.N[mb])
            for (int m = 0; m < ncols; m++) a.y[mb][m * a.N[mb] + n0 + r] = red[m * ROWS + r] * outscale;
    }
    if (share > 1) {
        // no CTA leaves while a peer's pushes into it (or reads of its planes) may be in flight
        namespace cg = cooperative_groups;
        cg::this_cluster().sync();
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == W_MMA) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase_s), "n"(TMEM_COLS) : "memory");
    }
}

bool fp4_map(CUtensorMap *map, const void *base, int64_t inner, int64_t rows, int box_inner, int box_rows,
             CUtensorMapSwizzle swz) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)inner};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int64_t SMEM_LIMIT = 200 * 1024;

// A cluster of S CTAs splits K into ranges of `per` whole slots (the last
// rank's may be shorter, none empty): S grows until the grid covers the SMs
// (at most 8 ranks), then further while a range does not fit shared memory.
// Returns S (0 if nothing fits) and the slots per rank.
template <bool XQ> int splits_for(int tiles, int64_t K, int *per_out) {
    const int64_t slots = K / SLOT_K;
    auto per = [&](int S) { return (int)((slots + S - 1) / S); };
    auto ranks = [&](int S) { return (int)((slots + per(S) - 1) / per(S)); };   // no empty rank
    int S = 1;
    while (S < 8 && (int64_t)tiles * S < sm_count() && ranks(2 * S) == 2 * S) S *= 2;
    while (smem_for<XQ>(per(S)) > SMEM_LIMIT && S < 8 && ranks(2 * S) == 2 * S) S *= 2;
    if (smem_for<XQ>(per(S)) > SMEM_LIMIT) return 0;
    *per_out = per(S);
    return S;
}

// CTAs per slice-sharing cluster (slices mode, no K split): the largest of
// 8, 4, 2 that divides both the tile count and the slot count.
int share_for(int tiles, int nslots) {
    for (int c = 8; c > 1; c >>= 1)
        if (tiles % c == 0 && nslots % c == 0) return c;
    return 1;
}

template <bool XQ> cudaError_t run_fp4tc(const Fp4Args &a, const Fp4Maps &maps, int tiles, int S, cudaStream_t s) {
    auto kern = gemv_fp4tc_kernel<XQ>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * S), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem_for<XQ>(a.k_per_cta / SLOT_K);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    const int cluster = S > 1 ? S : (XQ ? 1 : a.share);
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = (unsigned)cluster;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a, maps);
}

// Fills the weight maps and tile list of `count` same-K NVFP4 members.
bool fill_members(const Tensor *ts, int count, Fp4Args &a, Fp4Maps &maps, float *const *ys, int *tiles) {
    int n = 0;
    for (int i = 0; i < count; i++) {
        const Tensor &t = ts[i];
        if (t.K != a.K || !fp4_map(&maps.w[i], t.w, t.K / 2, t.N, SLOT_K / 2, ROWS, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !fp4_map(&maps.s[i], t.scales, t.K / 16, t.N, SLOT_K / 16, ROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
        a.y[i] = ys[i];
        a.N[i] = t.N;
        a.scale2[i] = t.scale2;
        a.tile_start[i] = n;
        n += (int)((t.N + ROWS - 1) / ROWS);
    }
    a.tile_start[count] = n;
    *tiles = n;
    return true;
}

}  // namespace

// Batch 1 NVFP4 with bf16 x, K % 256 == 0, 16-byte aligned tensors, and the
// per-CTA slices within the shared-memory budget.
bool gemv_fp4tc_eligible(const Tensor &t, int64_t M) {
    if (t.fmt != Q4_NVFP4 || M != 1 || t.K % SLOT_K != 0 || t.K > (1LL << 30) || t.N > (1LL << 31)) return false;
    if ((((uintptr_t)t.w | (uintptr_t)t.scales) & 15) != 0 || encode_fn() == nullptr) return false;
    const int tiles = (int)((t.N + ROWS - 1) / ROWS);
    int per = 0;
    return splits_for<false>(tiles, t.K, &per) > 0;
}

// count (<= MAXG) eligible NVFP4 matrices with the same K that read the same x, one launch.
cudaError_t launch_gemv_fp4tc_group(const Tensor *ts, int count, const void *x, float *const *ys, cudaStream_t s) {
    if (count < 1 || count > MAXG) return cudaErrorInvalidValue;
    Fp4Maps maps;
    Fp4Args a = {};
    a.count = count;
    a.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    a.K = ts[0].K;
    a.M = 1;
    a.x_scale2 = 1.0f;
    int tiles = 0, per = 0;
    if (!fill_members(ts, count, a, maps, ys, &tiles)) return cudaErrorInvalidValue;
    const int S = splits_for<false>(tiles, a.K, &per);
    if (S == 0) return cudaErrorInvalidValue;
    a.splits = S;
    a.k_per_cta = per * SLOT_K;
    a.share = S == 1 ? share_for(tiles, per) : 1;
    return run_fp4tc<false>(a, maps, tiles, S, s);
}

cudaError_t launch_gemv_fp4tc(const Tensor &t, const void *x, float *y, cudaStream_t s) {
    return launch_gemv_fp4tc_group(&t, 1, x, &y, s);
}

// NVFP4 weights against NVFP4 activations xq [M][K/2], xs [M][K/16] with
// tensor scale x_scale2: y [M][N] f32, 16 activation rows per launch.
bool gemv_w4a4_tc_eligible(const Tensor &t) {
    if (t.fmt != Q4_NVFP4 || t.K % SLOT_K != 0 || t.K > (1LL << 30) || t.N > (1LL << 31)) return false;
    return (((uintptr_t)t.w | (uintptr_t)t.scales) & 15) == 0 && encode_fn() != nullptr;
}

cudaError_t launch_gemv_w4a4_tc(const Tensor &t, const uint8_t *xq, const uint8_t *xs, float x_scale2, float *y,
                                int64_t M, cudaStream_t s) {
    for (int64_t m0 = 0; m0 < M; m0 += P) {
        const int mc = (int)(M - m0 < P ? M - m0 : P);
        Fp4Maps maps;
        Fp4Args a = {};
        a.count = 1;
        a.K = t.K;
        a.M = mc;
        a.x_scale2 = x_scale2;
        float *ym = y + m0 * t.N;
        int tiles = 0, per = 0;
        if (!fill_members(&t, 1, a, maps, &ym, &tiles)) return cudaErrorInvalidValue;
        if (!fp4_map(&maps.xq, xq + m0 * (t.K / 2), t.K / 2, mc, SLOT_K / 2, P, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !fp4_map(&maps.xs, xs + m0 * (t.K / 16), t.K / 16, mc, SLOT_K / 16, P, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        const int S = splits_for<true>(tiles, t.K, &per);
        if (S == 0) return cudaErrorInvalidValue;
        a.splits = S;
        a.k_per_cta = per * SLOT_K;
        a.share = 1;
        const cudaError_t e = run_fp4tc<true>(a, maps, tiles, S, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int fp4tc_set_wait_limit(long long cycles) {
    return cudaMemcpyToSymbol(g_fp4_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int fp4tc_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fp4_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_fp4_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

}  // namespace q4
