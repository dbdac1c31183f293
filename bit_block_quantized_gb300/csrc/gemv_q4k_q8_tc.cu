// gemv_q4k_q8_tc.cu -- the Q4_K x Q8 (W4A8) contraction of "Why 4-Bit
// Quantization Is King", section 7, with the exact sub-block sums on the
// tensor cores and the weights streamed by TMA.
//
// The contract is gemv_q4k_q8.cu's, bit for bit: activations quantized per
// 256-value block to signed 8-bit codes (signed first maximum m, iscale =
// -127/m, half-to-even, capped at 127, block scale 1/iscale), each 32-value
// sub-block's code sum bsum_j kept; per output row and super-block the exact
// integers I1 = sum_j sc_j * sum_{k in j} q[k] * q8[k] and
// I2 = sum_j m_j * bsum_j, then in f32 and in this order
// v = d * float(I1) - dmin * float(I2), c = v * act_scale, and
// total += c over the super-blocks in order.  Output f32.
//
// Why the tensor cores give the same integers: the unsigned codes enter the
// f16 MMA as subnormals, q * 2^-24 (low nibbles) or 16 q * 2^-24 (high
// nibbles, whose activation codes are staged divided by 16, a power of two),
// and the activation codes as f16 (|q8| <= 127).  Every product is
// q * q8 * 2^-24 exactly, and a sub-block's sum is an integer below 2^16
// times 2^-24, which the f32 accumulation holds without rounding; one FMA
// with 1.5 * 2^23 then reads the integer from the bits of the result.
//
// Layout and roles are the Q4_K TMA-fed GEMV's (gemv_blk_tc.cu): a stage is
// 16 rows x 2048 k (eight 144-byte super-blocks of each row, one 3-D box),
// one producer warp, eight decode warps, warp w on super-block w of every
// stage.  Lane (g, t) owns rows g and g + 8 and the 64-k chunk t (sub-blocks
// 2t, low nibbles, and 2t + 1, high nibbles); the B operand is diagonal, so
// D[row][2t + m] in lane (g, t) is batch row m's sum over lane t's own
// sub-block, with no shuffle and no fresh accumulator.  Each warp quantizes
// the activations of its own super-blocks.  The four lanes of a row add
// their integer parts; one lane per (row, batch row) takes the f32 steps and
// writes the super-block's value to a per-row list that one thread per row
// sums in super-block order at the end of the tile.  One or two batch rows
// per launch.
#include <cuda.h>

#include "q4_internal.cuh"
#include "tc_gemv_common.cuh"
#include "tma_map.cuh"

namespace q4 {

__device__ int g_k8tc_error;

namespace {

using namespace tc;

constexpr int KT_WARPS = 8;                          // decode warps = super-blocks per stage
constexpr int KT_THREADS = (KT_WARPS + 1) * 32;
constexpr int KT_UNIT = 144;                         // bytes of one super-block (256 k of one row)
constexpr int KT_ROWS = 16;
constexpr int KT_STAGE = KT_WARPS * KT_ROWS * KT_UNIT;   // 18432 bytes
constexpr int KT_MAX_NS = 6;
constexpr int KT_XU = 1024;                          // staged codes per super-block: 32 entries of 32 bytes
constexpr int KT_SMEM_CAP = 112 * 1024;              // two CTAs per SM
constexpr long long KT_WAIT = 1LL << 31;
static_assert(KT_STAGE % 1024 == 0, "stages stay 1024-byte aligned");

struct KtArgs {
    const void *x;   // [MB][K] f32 or bf16
    float *y;        // [MB][N]
    int64_t N;
    int K, nsb, nst, ntiles, NS;
};

// After the ring: staged codes [8 warps][nst][1024] (entry (chunk, word) at
// 32 (8 chunk + word): batch row m at 16 m, low-nibble codes at +0, high at
// +8), a 256-byte zero block at 64 mod 128, code sums [8][nst][MB][8] i32,
// activation scales [8][nst][MB] f32, super-block values [2][MB][16][nsb | 1]
// f32 (an odd row stride: the lanes' stores and the row sums hit distinct banks).
struct KtLayout {
    int xs, zero, bs, as, cb, total;
};
__host__ __device__ inline KtLayout kt_layout(int NS, int nst, int nsb, int mb) {
    KtLayout L;
    L.xs = NS * KT_STAGE;
    L.zero = L.xs + KT_WARPS * nst * KT_XU + 64;
    L.bs = L.zero + 256 + 64;
    L.as = L.bs + KT_WARPS * nst * mb * 8 * 4;
    L.cb = L.as + KT_WARPS * nst * mb * 4;
    L.total = L.cb + 2 * mb * KT_ROWS * (nsb | 1) * 4;
    return L;
}

__device__ __forceinline__ void kt_tma3(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar,
                                        uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void kt_sts64(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Eight consecutive x values as f32 (p 16-byte aligned).
__device__ __forceinline__ void kt_load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}
__device__ __forceinline__ void kt_load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// 6-bit scales and minima of sub-blocks 2t (low byte) and 2t + 1 (next byte)
// of one super-block, from its scale words B0 (bytes 4-7), B1 (8-11), B2
// (12-15): sub-block j < 4 takes the low 6 bits of scale bytes j and j + 4;
// j >= 4 the nibbles of byte j + 4 and the top two bits of bytes j - 4 and j.
__device__ __forceinline__ void kt_pair(uint32_t B0, uint32_t B1, uint32_t B2, int t, uint32_t &sc, uint32_t &mn) {
    const uint32_t p = 16u * (uint32_t)(t & 1);
    const uint32_t b0 = B0 >> p, b1 = B1 >> p, b2 = B2 >> p;
    const bool low = t < 2;
    sc = low ? (b0 & 0x3F3Fu) : ((b2 & 0x0F0Fu) | ((b0 >> 2) & 0x3030u));
    mn = low ? (b1 & 0x3F3Fu) : (((b2 >> 4) & 0x0F0Fu) | ((b1 >> 2) & 0x3030u));
}

// The integer n of D = n * 2^-24 (|n| < 2^22): n * 2^24 + 1.5 * 2^23 is exact
// in f32 and its low mantissa bits are n + 2^22.
__device__ __forceinline__ int kt_int(float D) {
    return (int)__float_as_uint(__fmaf_rn(D, 16777216.0f, 12582912.0f)) - 0x4B400000;
}

template <typename XT, int MB>
__global__ void __launch_bounds__(KT_THREADS, 2)
gemv_q4k_q8_tc(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ KtArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[KT_MAX_NS], empty[KT_MAX_NS];
    __shared__ int abort_s;
    uint8_t *ring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int NS = a.NS, nst = a.nst, nsb = a.nsb;
    const KtLayout L = kt_layout(NS, nst, nsb, MB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int my_tiles = (int)blockIdx.x < a.ntiles ? (a.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int J = my_tiles * nst;
    volatile int *abort_flag = &abort_s;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], KT_WARPS);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 64) reinterpret_cast<uint32_t *>(ring + L.zero)[threadIdx.x] = 0u;
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == KT_WARPS) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            int issued = 0;
            for (int j = 0; j < J; j++) {
                const int s = j % NS;
                if (j >= NS && !wait_or_abort(&empty[s], ((j / NS) & 1) ^ 1, abort_flag, &g_k8tc_error, KT_WAIT)) break;
                const int tile = (int)blockIdx.x + (j / nst) * (int)gridDim.x, st = j % nst;
                mbar_arrive_expect_tx(&full[s], KT_STAGE);
                kt_tma3(smem_u32(ring + s * KT_STAGE), &wmap, 0, tile * KT_ROWS, st * KT_WARPS, &full[s], pol);
                issued++;
            }
            for (int q = issued > NS ? issued - NS : 0; q < issued; q++)
                if (!mbar_wait_bounded(&full[q % NS], (uint32_t)((q / NS) & 1), KT_WAIT))
                    atomicExch(&g_k8tc_error, Q4_ETIMEOUT);
        }
        __syncwarp();
        return;
    }

    // ------------------------ activation quantization (this warp's super-blocks)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const XT *xp = reinterpret_cast<const XT *>(a.x);
    const uint32_t xs_w = smem_u32(ring + L.xs) + (uint32_t)(warp * nst * KT_XU);
    int32_t *bs_w = reinterpret_cast<int32_t *>(ring + L.bs) + warp * nst * MB * 8;
    float *as_w = reinterpret_cast<float *>(ring + L.as) + warp * nst * MB;
    {
        // lane l holds k = 8l .. 8l+7: chunk l >> 3, the low (0) or high (1) nibble half, code words i0, i0 + 1
        const int tq = lane >> 3, half = (lane >> 2) & 1, i0 = 2 * (lane & 3);
        const float f = half ? 0.0625f : 1.0f;
        // P of the warp's super-blocks at a time, their loads and shuffle chains overlapped: two,
        // but one for f32 x at batch 1 (measured faster: two f32 blocks hold 16 values per lane)
        constexpr int P = (sizeof(XT) == 4 && MB == 1) ? 1 : 2;
        for (int s0 = 0; s0 < nst; s0 += P) {
            float v[P][MB][8];
#pragma unroll
            for (int p = 0; p < P; p++) {
                const int u = warp + KT_WARPS * (s0 + p);
                const bool have = s0 + p < nst && u < nsb;
#pragma unroll
                for (int m = 0; m < MB; m++) {
                    if (have) {
                        kt_load8(xp + (int64_t)m * a.K + (int64_t)u * 256 + lane * 8, v[p][m]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; i++) v[p][m][i] = 0.0f;
                    }
                }
            }
            float amax[P][MB], val[P][MB];
            int idx[P][MB];
#pragma unroll
            for (int p = 0; p < P; p++)
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
            for (int off = 16; off > 0; off >>= 1)      // largest magnitude, first index on ties
#pragma unroll
                for (int p = 0; p < P; p++)
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
            for (int p = 0; p < P; p++) {
                const int s = s0 + p, u = warp + KT_WARPS * s;
                if (s >= nst || u >= nsb) break;
#pragma unroll
                for (int m = 0; m < MB; m++) {
                    const float iscale = __fdiv_rn(-127.0f, val[p][m]);
                    const bool live = isfinite(iscale);     // zero (or vanishing) block: codes 0, scale 0
                    int c[8], ssum = 0;
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        int ci = live ? __float2int_rn(__fmul_rn(v[p][m][i], iscale)) : 0;
                        ci = (int)(int8_t)(uint8_t)((ci > 127 ? 127 : ci) & 0xff);   // the 8-bit code the contract keeps
                        c[i] = ci;
                        ssum += ci;
                    }
                    ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);   // the sub-block's lanes 4j .. 4j+3
                    ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
#pragma unroll
                    for (int q = 0; q < 2; q++) {
                        const uint32_t h02 = h2bits(__float2half_rn((float)c[4 * q] * f), __float2half_rn((float)c[4 * q + 2] * f));
                        const uint32_t h13 = h2bits(__float2half_rn((float)c[4 * q + 1] * f), __float2half_rn((float)c[4 * q + 3] * f));
                        kt_sts64(xs_w + (uint32_t)(s * KT_XU + (tq * 8 + i0 + q) * 32 + m * 16 + half * 8), h02, h13);
                    }
                    if ((lane & 3) == 0) bs_w[(s * MB + m) * 8 + (lane >> 2)] = ssum;
                    if (lane == 0) as_w[s * MB + m] = live ? __fdiv_rn(1.0f, iscale) : 0.0f;
                }
            }
        }
    }
    __syncwarp();

    // ------------------------------------------------ decode + multiply
    const int g = lane >> 2, t = lane & 3;
    const bool diag = MB == 1 ? g == 2 * t : (g >> 1) == t;              // supplies B column g in lane t's slots
    const uint32_t xb = diag ? xs_w + (uint32_t)(t * 256 + (g & 1) * 16) : smem_u32(ring + L.zero) + (uint32_t)((g & 1) * 16);
    const uint32_t xstep = diag ? (uint32_t)KT_XU : 0u;
    const uint32_t ring_u = smem_u32(ring);
    float *cb = reinterpret_cast<float *>(ring + L.cb);
    const int nbp = nsb | 1;
    const int my_r = t & 1, my_m = t >> 1;                               // this lane's row g + 8 my_r, batch row my_m
    bool ok = true;
    int buf = 0;
    for (int j = 0; j < J; j++) {
        const int s = j % NS, st = j % nst;
        const int u = warp + KT_WARPS * st;
        if (ok) ok = wait_or_abort(&full[s], (uint32_t)((j / NS) & 1), abort_flag, &g_k8tc_error, KT_WAIT);
        if (ok && u < nsb) {
            const uint32_t rg = ring_u + (uint32_t)(s * KT_STAGE + warp * KT_ROWS * KT_UNIT + g * KT_UNIT);
            const uint32_t rg8 = rg + 8 * KT_UNIT;
            const uint32_t xa = xb + (uint32_t)st * xstep;
            const uint4 H0 = lds128(rg), H1 = lds128(rg8);
            const uint4 c0a = lds128(rg + 16 + 32 * t), c0b = lds128(rg + 32 + 32 * t);
            const uint4 c1a = lds128(rg8 + 16 + 32 * t), c1b = lds128(rg8 + 32 + 32 * t);
            const uint32_t w0[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
            const uint32_t w1[8] = {c1a.x, c1a.y, c1a.z, c1a.w, c1b.x, c1b.y, c1b.z, c1b.w};
            float Dl[4] = {0.f, 0.f, 0.f, 0.f}, Dh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint4 bx = lds128(xa + (uint32_t)(i * 32));
                const uint32_t s0 = w0[i] >> 8, s1 = w1[i] >> 8;
                mma16816(Dl, make_uint4(w0[i] & 0x000F000Fu, w1[i] & 0x000F000Fu, s0 & 0x000F000Fu, s1 & 0x000F000Fu),
                         bx.x, bx.y);
                mma16816(Dh, make_uint4(w0[i] & 0x00F000F0u, w1[i] & 0x00F000F0u, s0 & 0x00F000F0u, s1 & 0x00F000F0u),
                         bx.z, bx.w);
            }
            uint32_t sc0, mn0, sc1, mn1;
            kt_pair(H0.y, H0.z, H0.w, t, sc0, mn0);                      // row g
            kt_pair(H1.y, H1.z, H1.w, t, sc1, mn1);                      // row g + 8
            int I1 = 0, I2 = 0;
#pragma unroll
            for (int m = 0; m < MB; m++) {
                const int2 bsm = *reinterpret_cast<const int2 *>(bs_w + (st * MB + m) * 8 + 2 * t);
                // lane t's part of I1 and I2 for rows g and g + 8 (column 2t + m of the MMAs)
                int v1g = (int)(sc0 & 255u) * kt_int(Dl[m]) + (int)(sc0 >> 8) * kt_int(Dh[m]);
                int v1h = (int)(sc1 & 255u) * kt_int(Dl[2 + m]) + (int)(sc1 >> 8) * kt_int(Dh[2 + m]);
                int v2g = (int)(mn0 & 255u) * bsm.x + (int)(mn0 >> 8) * bsm.y;
                int v2h = (int)(mn1 & 255u) * bsm.x + (int)(mn1 >> 8) * bsm.y;
#pragma unroll
                for (int off = 1; off <= 2; off <<= 1) {                 // the four lanes of a row
                    v1g += __shfl_xor_sync(0xffffffffu, v1g, off);
                    v1h += __shfl_xor_sync(0xffffffffu, v1h, off);
                    v2g += __shfl_xor_sync(0xffffffffu, v2g, off);
                    v2h += __shfl_xor_sync(0xffffffffu, v2h, off);
                }
                if (m == my_m) {
                    I1 = my_r ? v1h : v1g;
                    I2 = my_r ? v2h : v2g;
                }
            }
            if (my_m < MB) {
                const uint32_t hx = my_r ? H1.x : H0.x;
                const float d = half_bits_f32(hx & 0xffffu), dmin = half_bits_f32(hx >> 16);
                const float p1 = __fmul_rn(d, __int2float_rn(I1)), p2 = __fmul_rn(dmin, __int2float_rn(I2));
                const float c = __fmul_rn(__fsub_rn(p1, p2), as_w[st * MB + my_m]);
                cb[(buf * MB * KT_ROWS + my_m * KT_ROWS + g + 8 * my_r) * nbp + u] = c;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (st == nst - 1) {
            // end of a tile: each row's super-block values in order
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (threadIdx.x < MB * KT_ROWS) {
                const int m = threadIdx.x / KT_ROWS, rr = threadIdx.x % KT_ROWS;
                const int64_t n = (int64_t)((int)blockIdx.x + (j / nst) * (int)gridDim.x) * KT_ROWS + rr;
                if (n < a.N && ok) {
                    const float *row = cb + (buf * MB * KT_ROWS + m * KT_ROWS + rr) * nbp;
                    float total = 0.0f;
#pragma unroll 8
                    for (int b = 0; b < nsb; b++) total = __fadd_rn(total, row[b]);
                    a.y[(int64_t)m * a.N + n] = total;
                }
            }
            buf ^= 1;
        }
    }
}

struct KtPlan {
    int nsb, nst, NS, smem;
};

bool kt_plan(int64_t K, int mb, KtPlan &p) {
    if (K % 256 != 0 || K <= 0 || K > (1LL << 24)) return false;
    p.nsb = (int)(K / 256);
    p.nst = (p.nsb + KT_WARPS - 1) / KT_WARPS;
    const KtLayout L0 = kt_layout(0, p.nst, p.nsb, mb);
    const int ns = (KT_SMEM_CAP - 1024 - L0.total) / KT_STAGE;
    if (ns < 3) return false;
    p.NS = ns < KT_MAX_NS ? ns : KT_MAX_NS;
    p.smem = 1024 + kt_layout(p.NS, p.nst, p.nsb, mb).total;
    return true;
}

template <typename XT, int MB>
cudaError_t kt_run(const CUtensorMap &map, const KtArgs &a, int smem, cudaStream_t s) {
    auto kern = gemv_q4k_q8_tc<XT, MB>;
    static bool attr_set[64] = {};
    static int per_sm[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KT_SMEM_CAP);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, KT_THREADS, KT_SMEM_CAP) != cudaSuccess || b < 1)
            b = 1;
        per_sm[dev & 63] = b;
        attr_set[dev & 63] = true;
    }
    int grid = per_sm[dev & 63] * sm_count();
    if (grid > a.ntiles) grid = a.ntiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(KT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, map, a);
}

// The weights as a 3-D tensor {144 bytes, N rows, K/256 super-blocks}: one
// box {144, 16, 8} is a stage.
bool kt_encode(CUtensorMap *map, const Tensor &t, int nsb) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)KT_UNIT, (cuuint64_t)t.N, (cuuint64_t)nsb};
    const cuuint64_t strides[2] = {(cuuint64_t)nsb * KT_UNIT, (cuuint64_t)KT_UNIT};
    const cuuint32_t box[3] = {(cuuint32_t)KT_UNIT, (cuuint32_t)KT_ROWS, (cuuint32_t)KT_WARPS};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(t.w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Q4_K with K % 256 == 0, the weights 16-byte aligned, M = 1 or 2 (one
// launch) with the staged codes and three ring stages within 112 KB.
bool gemv_q4k_q8_tc_eligible(const Tensor &t, int64_t M) {
    if (t.fmt != Q4_Q4K || M < 1 || M > 2 || t.K % 256 != 0 || t.N < 1 || t.N > (1LL << 30)) return false;
    if ((((uintptr_t)t.w) & 15) != 0 || encode_fn() == nullptr) return false;
    KtPlan p;
    return kt_plan(t.K, (int)M, p);
}

cudaError_t launch_gemv_q4k_q8_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    KtPlan p;
    CUtensorMap map;
    if (M < 1 || M > 2 || !kt_plan(t.K, (int)M, p) || !kt_encode(&map, t, p.nsb)) return cudaErrorInvalidValue;
    KtArgs a;
    a.x = x;
    a.y = y;
    a.N = t.N;
    a.K = (int)t.K;
    a.nsb = p.nsb;
    a.nst = p.nst;
    a.ntiles = (int)((t.N + KT_ROWS - 1) / KT_ROWS);
    a.NS = p.NS;
    if (M == 2)
        return xd == Q4_DT_BF16 ? kt_run<__nv_bfloat16, 2>(map, a, p.smem, s) : kt_run<float, 2>(map, a, p.smem, s);
    return xd == Q4_DT_BF16 ? kt_run<__nv_bfloat16, 1>(map, a, p.smem, s) : kt_run<float, 1>(map, a, p.smem, s);
}

int k8tc_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_k8tc_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_k8tc_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

}  // namespace q4
