// gemv_a16q8_tc.cu -- the integer-exact weight-only NVFP4 contraction of the
// Muser book, chapter 7, section 7.4.2 ([MUS7] 7.4.2), with the exact group
// dots on the tensor cores and the weights streamed by TMA.
//
// The contract is gemv_a16q8.cu's, bit for bit: activations quantized per
// 256-value block to signed 8-bit codes (signed first maximum m, iscale =
// -127/m, half-to-even, capped at 127, block scale 1/iscale); per output row
// and block T = sum_g q9(scale[n][g]) * sum_{k in g} q1(code[n][k]) * q8[k],
// an exact integer (q1 = E2M1 in halves, q9 = E4M3FN in units of 2^-9);
// then c = fma(float(T), 2^-10, 0), c = fma(c, act_scale, 0),
// c = fma(c, scale2, 0), total = fma(1, c, total) in block order, and the
// output is total rounded to binary16.
//
// Why the tensor cores give the same integers: the activation codes are
// staged doubled (2 q8, |2 q8| <= 254, exact in f16), so a 16-k group's sum
// e2m1 * 2 q8 has E2M1 values (multiples of 1/2, |v| <= 6, exact in f16)
// times even integers: integer products of at most 11 significant bits and
// partial sums below 2^15, which the f16 MMA's f32 accumulation holds
// exactly.  D is the group's q1 * q8 dot; adding 1.5 * 2^23 (exact) leaves it
// in the low mantissa bits, read as an integer with no conversion.
//
// Layout and roles are the NVFP4 TMA-fed GEMV's (gemv_tma.cu): a stage is 16
// rows x 2048 k (the payload as a chunk-major 3-D box with the 128-byte
// swizzle, the E4M3 scales as a 2-D box), one producer warp, eight decode
// warps, warp w on the 256-k block w of every stage.  The B operand is
// diagonal as in gemv_blk_tc.cu: lane (2t + m, t) supplies batch row m's codes
// for lane t's k slots, so D[row][2t + m] in lane (g, t) is row m's dot over
// lane t's own 16-k group; each group gets a fresh accumulator, its dot times
// q9 adds in 64 bits, the four lanes of a row add their block sums, and the
// block's pinned f32 steps go to a per-row list that one thread per row sums
// in block order at the end of the tile.  One or two batch rows per launch.
// Two CTAs share an SM, or three at batch 1 where three ring stages still fit
// in 74 KB (K <= 4352): more decode warps per scheduler, measured faster.
#include <cuda.h>

#include "q4_internal.cuh"
#include "tc_gemv_common.cuh"
#include "tma_map.cuh"

namespace q4 {

__device__ int g_a16tc_error;

namespace {

using namespace tc;

constexpr int AQ_WARPS = 8;
constexpr int AQ_THREADS = (AQ_WARPS + 1) * 32;
constexpr int AQ_ROWS = 16;
constexpr int AQ_KS = AQ_WARPS * 256;                 // k per stage
constexpr int AQ_PAY = AQ_ROWS * AQ_KS / 2;           // 16 KB of payload
constexpr int AQ_SC = AQ_ROWS * AQ_KS / 16;           // 2 KB of E4M3 scales
constexpr int AQ_STAGE = AQ_PAY + AQ_SC;
constexpr int AQ_MAX_NS = 6;
constexpr int AQ_XQ = 656;                            // staged codes per block and row: 4 x 144 B, padded to 16 mod 128
// Shared memory per CTA: two CTAs per SM, or three (batch 1 where three ring stages
// still fit: more decode warps per scheduler, measured faster) within 74 KB.
constexpr int aq_smem_cap(int ctas) { return ctas == 3 ? 74 * 1024 : 112 * 1024; }
constexpr long long AQ_WAIT = 1LL << 31;
static_assert(AQ_STAGE % 1024 == 0, "stages stay 1024-byte aligned");

struct AqMaps {
    CUtensorMap pay;   // u8 {128, N, K/256}, box {128, 16, 8}, 128-byte swizzle
    CUtensorMap sc;    // u8 {K/16, N}, box {128, 16}, 128-byte swizzle
};

struct AqArgs {
    const void *x;     // [MB][K] f32 or bf16
    float *y;          // [MB][N]
    int64_t N;
    int K, nb, nst, ntiles, NS;
    float scale2;
};

// After the ring: staged codes [8 warps][nst][MB][656] (lane quarter t at 144 t
// and batch row m at 656 m: 16 t + 16 m modulo 128), a 128-byte zero block at
// 80 mod 128, so the diagonal lanes' 16-byte loads and the zero block's never
// share banks; activation scales [8][nst][MB] f32, the q9 table [256] i32,
// block results [2][MB][16][nb | 1] f32 (an odd row stride: the lanes' stores
// and the row sums hit distinct banks).
struct AqLayout {
    int xs, zero, as, lut, cb, total;
};
__host__ __device__ inline AqLayout aq_layout(int NS, int nst, int nb, int mb) {
    AqLayout L;
    L.xs = NS * AQ_STAGE;
    L.zero = L.xs + AQ_WARPS * nst * mb * AQ_XQ + 80;
    L.as = L.zero + 128 + 48;
    L.lut = (L.as + AQ_WARPS * nst * mb * 4 + 15) / 16 * 16;
    L.cb = L.lut + 1024;
    L.total = L.cb + 2 * mb * AQ_ROWS * (nb | 1) * 4;
    return L;
}

__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar,
                                     uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ int64_t shfl_xor_i64(int64_t v, int mask) {
    return (int64_t)__shfl_xor_sync(0xffffffffu, (long long)v, mask);
}

// Eight consecutive x values as f32 (p 16-byte aligned).
__device__ __forceinline__ void aq_load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}
__device__ __forceinline__ void aq_load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <typename XT, int MB, int CTAS>
__global__ void __launch_bounds__(AQ_THREADS, CTAS)
gemv_a16q8_tc(const __grid_constant__ AqMaps maps, const __grid_constant__ AqArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[AQ_MAX_NS], empty[AQ_MAX_NS];
    __shared__ int abort_s;
    uint8_t *ring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int NS = a.NS, nst = a.nst, nb = a.nb;
    const AqLayout L = aq_layout(NS, nst, nb, MB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int my_tiles = (int)blockIdx.x < a.ntiles ? (a.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int J = my_tiles * nst;
    volatile int *abort_flag = &abort_s;
    int32_t *lut = reinterpret_cast<int32_t *>(ring + L.lut);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], AQ_WARPS);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 32) reinterpret_cast<uint32_t *>(ring + L.zero)[threadIdx.x] = 0u;
    if (threadIdx.x < 256) {       // E4M3FN byte -> q9 = (8+f) << (e-1), or f for exponent field 0; bit 7 the sign
        const uint32_t b = threadIdx.x, e = (b >> 3) & 15u, f = b & 7u;
        const int32_t mag = e == 0 ? (int32_t)f : (int32_t)((8u + f) << (e - 1u));
        lut[b] = (b & 0x80u) ? -mag : mag;
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == AQ_WARPS) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            int issued = 0;
            for (int j = 0; j < J; j++) {
                const int s = j % NS;
                if (j >= NS && !wait_or_abort(&empty[s], ((j / NS) & 1) ^ 1, abort_flag, &g_a16tc_error, AQ_WAIT)) break;
                const int tile = (int)blockIdx.x + (j / nst) * (int)gridDim.x, st = j % nst;
                const uint32_t dst = smem_u32(ring + s * AQ_STAGE);
                mbar_arrive_expect_tx(&full[s], AQ_STAGE);
                tma3(dst, &maps.pay, 0, tile * AQ_ROWS, st * AQ_WARPS, &full[s], pol);
                tma2(dst + AQ_PAY, &maps.sc, st * (AQ_KS / 16), tile * AQ_ROWS, &full[s], pol);
                issued++;
            }
            for (int q = issued > NS ? issued - NS : 0; q < issued; q++)
                if (!mbar_wait_bounded(&full[q % NS], (uint32_t)((q / NS) & 1), AQ_WAIT))
                    atomicExch(&g_a16tc_error, Q4_ETIMEOUT);
        }
        __syncwarp();
        return;
    }

    // ------------------------ activation quantization (this warp's blocks)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const XT *xp = reinterpret_cast<const XT *>(a.x);
    const uint32_t xs_w = smem_u32(ring + L.xs) + (uint32_t)(warp * nst * MB * AQ_XQ);
    float *as_w = reinterpret_cast<float *>(ring + L.as) + warp * nst * MB;
    for (int s0 = 0; s0 < nst; s0 += 2) {
        // two of the warp's blocks at a time: their loads and shuffle chains overlap
        float v[2][MB][8];
#pragma unroll
        for (int p = 0; p < 2; p++) {
            const int b = warp + AQ_WARPS * (s0 + p);
            const bool have = s0 + p < nst && b < nb;
#pragma unroll
            for (int m = 0; m < MB; m++) {
                if (have) {
                    aq_load8(xp + (int64_t)m * a.K + (int64_t)b * 256 + lane * 8, v[p][m]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; i++) v[p][m][i] = 0.0f;
                }
            }
        }
        float amax[2][MB], val[2][MB];
        int idx[2][MB];
#pragma unroll
        for (int p = 0; p < 2; p++)
#pragma unroll
            for (int m = 0; m < MB; m++) {
                amax[p][m] = 0.0f, val[p][m] = 0.0f, idx[p][m] = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const float av = fabsf(v[p][m][i]);
                    if (av > amax[p][m]) { amax[p][m] = av; val[p][m] = v[p][m][i]; idx[p][m] = lane * 8 + i; }
                }
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)          // largest magnitude, first index on ties
#pragma unroll
            for (int p = 0; p < 2; p++)
#pragma unroll
                for (int m = 0; m < MB; m++) {
                    const float oa = __shfl_xor_sync(0xffffffffu, amax[p][m], off);
                    const float ov = __shfl_xor_sync(0xffffffffu, val[p][m], off);
                    const int oi = __shfl_xor_sync(0xffffffffu, idx[p][m], off);
                    if (oa > amax[p][m] || (oa == amax[p][m] && oi < idx[p][m])) {
                        amax[p][m] = oa; val[p][m] = ov; idx[p][m] = oi;
                    }
                }
#pragma unroll
        for (int p = 0; p < 2; p++) {
            const int s = s0 + p, b = warp + AQ_WARPS * s;
            if (s >= nst || b >= nb) break;
#pragma unroll
            for (int m = 0; m < MB; m++) {
                const float iscale = __fdiv_rn(-127.0f, val[p][m]);
                const bool live = isfinite(iscale);     // zero (or vanishing) block: codes 0, scale 0
                uint32_t h[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    int c0 = live ? __float2int_rn(__fmul_rn(v[p][m][2 * i], iscale)) : 0;
                    int c1 = live ? __float2int_rn(__fmul_rn(v[p][m][2 * i + 1], iscale)) : 0;
                    c0 = (int)(int8_t)(uint8_t)((c0 > 127 ? 127 : c0) & 0xff);     // the 8-bit code the contract keeps
                    c1 = (int)(int8_t)(uint8_t)((c1 > 127 ? 127 : c1) & 0xff);
                    h[i] = h2bits(__int2half_rn(2 * c0), __int2half_rn(2 * c1));   // 2 q8: the MMA sums q1 q8
                }
                sts128(xs_w + (uint32_t)((s * MB + m) * AQ_XQ + (lane >> 3) * 144 + (lane & 7) * 16),
                       make_uint4(h[0], h[1], h[2], h[3]));
                if (lane == 0) as_w[s * MB + m] = live ? __fdiv_rn(1.0f, iscale) : 0.0f;
            }
        }
    }
    __syncwarp();

    // ------------------------------------------------ decode + multiply
    const int g = lane >> 2, t = lane & 3;
    const bool diag = MB == 1 ? g == 2 * t : (g >> 1) == t;              // supplies column g in lane t's slots
    const uint32_t xb0 = diag ? xs_w + (uint32_t)((g & 1) * AQ_XQ + t * 144) : smem_u32(ring + L.zero);
    const uint32_t xstep = diag ? (uint32_t)(MB * AQ_XQ) : 0u;
    const uint32_t ring_u = smem_u32(ring);
    // payload byte offsets of this lane's two 16-byte units in rows g and g + 8 of block `warp`
    const uint32_t offA0 = (uint32_t)((warp * 16 + g) * 128) + ((uint32_t)((2 * t) ^ g) << 4);
    const uint32_t offA1 = (uint32_t)((warp * 16 + g) * 128) + ((uint32_t)((2 * t + 1) ^ g) << 4);
    const uint32_t offS = (uint32_t)AQ_PAY + (uint32_t)(g * 128) + ((uint32_t)(warp ^ g) << 4) + 4 * t;
    constexpr uint32_t ROW8 = 8 * 128;
    float *cb = reinterpret_cast<float *>(ring + L.cb);
    const int nbp = nb | 1;                                                  // odd row stride: no bank conflicts
    bool ok = true;
    int buf = 0;
    for (int j = 0; j < J; j++) {
        const int s = j % NS, st = j % nst;
        const int b = warp + AQ_WARPS * st;
        if (ok) ok = wait_or_abort(&full[s], (uint32_t)((j / NS) & 1), abort_flag, &g_a16tc_error, AQ_WAIT);
        if (ok && b < nb) {
            const uint32_t stg = ring_u + (uint32_t)(s * AQ_STAGE);
            const uint32_t xa = xb0 + (uint32_t)st * xstep;
            const uint32_t sa = lds32(stg + offS), sb = lds32(stg + offS + ROW8);   // groups 4t .. 4t+3, rows g, g+8
            int32_t qa[4], qb[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                qa[q] = lut[(sa >> (8 * q)) & 0xffu];
                qb[q] = lut[(sb >> (8 * q)) & 0xffu];
            }
            int64_t T[MB][2] = {};
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint4 pa = lds128(stg + (h ? offA1 : offA0)), pb = lds128(stg + (h ? offA1 : offA0) + ROW8);
                const uint32_t wa[4] = {pa.x, pa.y, pa.z, pa.w}, wb[4] = {pb.x, pb.y, pb.z, pb.w};
                // the unit's two 16-k groups (words 0-1, 2-3), each a fresh accumulator, issued alternately
                float D[2][4] = {};
#pragma unroll
                for (int o = 0; o < 4; o++) {
                    const int wd = (o >> 1) | ((o & 1) << 1), gq = wd >> 1;   // words 0, 2, 1, 3
                    uint32_t av[4], cv[4];
                    e2m1x8_h2(wa[wd], av[0], av[1], av[2], av[3]);
                    e2m1x8_h2(wb[wd], cv[0], cv[1], cv[2], cv[3]);
                    const uint4 bx = lds128(xa + (uint32_t)(64 * h + 16 * wd));
                    mma16816(D[gq], make_uint4(av[0], cv[0], av[1], cv[1]), bx.x, bx.y);
                    mma16816(D[gq], make_uint4(av[2], cv[2], av[3], cv[3]), bx.z, bx.w);
                }
#pragma unroll
                for (int gq = 0; gq < 2; gq++) {
                    const int q = 2 * h + gq;
#pragma unroll
                    for (int m = 0; m < MB; m++) {
                        // D is the group's exact q1 * q8 dot (an integer below 2^15), read from the bits
                        // of 1.5 * 2^23 + D
                        const float da = __fadd_rn(D[gq][m], 0x1.8p23f), db = __fadd_rn(D[gq][2 + m], 0x1.8p23f);
                        T[m][0] += (int64_t)((int)__float_as_uint(da) - 0x4B400000) * qa[q];
                        T[m][1] += (int64_t)((int)__float_as_uint(db) - 0x4B400000) * qb[q];
                    }
                }
            }
            // the block: the four lanes of a row, then the pinned f32 steps
            float *cbb = cb + buf * MB * AQ_ROWS * nbp;
#pragma unroll
            for (int m = 0; m < MB; m++) {
                const float ascale = as_w[st * MB + m];
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    int64_t v = T[m][r];
                    v += shfl_xor_i64(v, 1);
                    v += shfl_xor_i64(v, 2);
                    float c = __fmaf_rn(__ll2float_rn((long long)v), 0x1p-10f, 0.0f);
                    c = __fmaf_rn(c, ascale, 0.0f);
                    c = __fmaf_rn(c, a.scale2, 0.0f);
                    if (t == 0) cbb[(m * AQ_ROWS + g + 8 * r) * nbp + b] = c;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (st == nst - 1) {
            // end of a tile: each row's block results in block order
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (threadIdx.x < MB * AQ_ROWS) {
                const int m = threadIdx.x / AQ_ROWS, rr = threadIdx.x % AQ_ROWS;
                const int64_t n = (int64_t)((int)blockIdx.x + (j / nst) * (int)gridDim.x) * AQ_ROWS + rr;
                if (n < a.N && ok) {
                    const float *row = cb + buf * MB * AQ_ROWS * nbp + (m * AQ_ROWS + rr) * nbp;
                    float total = 0.0f;
#pragma unroll 8
                    for (int bb = 0; bb < nb; bb++) total = __fmaf_rn(1.0f, row[bb], total);
                    a.y[(int64_t)m * a.N + n] = __half2float(__float2half_rn(total));
                }
            }
            buf ^= 1;
        }
    }
}

struct AqPlan {
    int nb, nst, NS, smem;
};

bool aq_plan(int64_t K, int mb, int ctas, AqPlan &p) {
    if (K % 256 != 0 || K <= 0 || K > (1LL << 24)) return false;
    p.nb = (int)(K / 256);
    p.nst = (p.nb + AQ_WARPS - 1) / AQ_WARPS;
    const AqLayout L0 = aq_layout(0, p.nst, p.nb, mb);
    const int ns = (aq_smem_cap(ctas) - 1024 - L0.total) / AQ_STAGE;
    if (ns < 3) return false;
    p.NS = ns < AQ_MAX_NS ? ns : AQ_MAX_NS;
    p.smem = 1024 + aq_layout(p.NS, p.nst, p.nb, mb).total;
    return true;
}

template <typename XT, int MB, int CTAS>
cudaError_t aq_run(const AqMaps &maps, const AqArgs &a, int smem, cudaStream_t s) {
    auto kern = gemv_a16q8_tc<XT, MB, CTAS>;
    static bool attr_set[64] = {};
    static int per_sm[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, aq_smem_cap(CTAS));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, AQ_THREADS, aq_smem_cap(CTAS)) != cudaSuccess || b < 1)
            b = 1;
        per_sm[dev & 63] = b;
        attr_set[dev & 63] = true;
    }
    int grid = per_sm[dev & 63] * sm_count();
    if (grid > a.ntiles) grid = a.ntiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(AQ_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps, a);
}

bool aq_encode(AqMaps &maps, const Tensor &t) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t pdims[3] = {128, (cuuint64_t)t.N, (cuuint64_t)(t.K / 256)};
    const cuuint64_t pstrides[2] = {(cuuint64_t)(t.K / 2), 128};
    const cuuint32_t pbox[3] = {128, (cuuint32_t)AQ_ROWS, (cuuint32_t)AQ_WARPS};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&maps.pay, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(t.w), pdims, pstrides, pbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const cuuint64_t sdims[2] = {(cuuint64_t)(t.K / 16), (cuuint64_t)t.N};
    const cuuint64_t sstrides[1] = {(cuuint64_t)(t.K / 16)};
    const cuuint32_t sbox[2] = {128, (cuuint32_t)AQ_ROWS};
    return enc(&maps.sc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(t.scales), sdims, sstrides, sbox,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// NVFP4 with K % 256 == 0, the tensors 16-byte aligned, M = 1 or 2 (one
// launch) with the staged codes and three ring stages within 112 KB.
bool gemv_a16q8_tc_eligible(const Tensor &t, int64_t M) {
    if (t.fmt != Q4_NVFP4 || M < 1 || M > 2 || t.K % 256 != 0 || t.N < 1 || t.N > (1LL << 30)) return false;
    if ((((uintptr_t)t.w | (uintptr_t)t.scales) & 15) != 0 || encode_fn() == nullptr) return false;
    AqPlan p;
    return aq_plan(t.K, (int)M, 2, p);
}

cudaError_t launch_gemv_a16q8_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    AqPlan p;
    AqMaps maps;
    const bool three = M == 1 && aq_plan(t.K, 1, 3, p);
    if (M < 1 || M > 2 || (!three && !aq_plan(t.K, (int)M, 2, p)) || !aq_encode(maps, t)) return cudaErrorInvalidValue;
    AqArgs a;
    a.x = x;
    a.y = y;
    a.N = t.N;
    a.K = (int)t.K;
    a.nb = p.nb;
    a.nst = p.nst;
    a.ntiles = (int)((t.N + AQ_ROWS - 1) / AQ_ROWS);
    a.NS = p.NS;
    a.scale2 = t.scale2;
    if (M == 2)
        return xd == Q4_DT_BF16 ? aq_run<__nv_bfloat16, 2, 2>(maps, a, p.smem, s)
                                : aq_run<float, 2, 2>(maps, a, p.smem, s);
    if (three)
        return xd == Q4_DT_BF16 ? aq_run<__nv_bfloat16, 1, 3>(maps, a, p.smem, s)
                                : aq_run<float, 1, 3>(maps, a, p.smem, s);
    return xd == Q4_DT_BF16 ? aq_run<__nv_bfloat16, 1, 2>(maps, a, p.smem, s) : aq_run<float, 1, 2>(maps, a, p.smem, s);
}

int a16tc_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_a16tc_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_a16tc_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

}  // namespace q4
