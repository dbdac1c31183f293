// gemv_blk_tc.cu -- Q4_K and Q4_0 decode-GEMV at batch 1 on the tensor cores,
// weights streamed into shared memory by tensor TMA.
//
// Both formats store 256 k of one row in 144 bytes: a Q4_K super-block
// ([FBTC] sections 5-6: fp16 d, fp16 dmin, 12 bytes of 6-bit scales and
// mins, 128 code bytes whose low nibbles are k 64c + l and high nibbles
// 64c + 32 + l for byte 32c + l), or eight Q4_0 blocks of 18 bytes
// ([BPA] "Real layouts compared": fp16 d, then 16 code bytes whose low
// nibbles are elements 0-15 and high nibbles 16-31).  The weights form a
// 3-D tensor {144 bytes, N rows, K/256 units}; one TMA box {144, 16, 8} is a
// ring stage of 16 rows x 2048 k (18 KB), stored unit-major with rows 144
// bytes apart, so the lanes' 16-byte loads of two neighbouring rows fall in
// different banks.
//
// mma.sync m16n8k16 (f16 x f16 -> f32), weights as A (16 rows x 16 k).  Warp
// w takes unit w of every stage.  Lane (g, t) owns rows g and g + 8 and a
// quarter of the unit: for Q4_K the 32 code bytes of 64-k chunk t (sub-blocks
// 2t, low nibbles, and 2t + 1, high nibbles); for Q4_0 the blocks 2t and
// 2t + 1.  In every MMA lane t's four k slots carry four codes of its own
// quarter (one 32-bit code word: bytes 0 and 2 in slots 2t, 2t+1, bytes 1
// and 3 in slots 2t+8, 2t+9), and the B operand is "diagonal": column 2t
// (the f16 hi part of x) and column 2t + 1 (the lo part) are non-zero only
// in lane t's slots.  So D[row][2t] + D[row][2t + 1], which the MMA leaves in
// lane (g, t) itself, is the sum over lane t's own sub-block or block: a
// per-sub-block scale needs no shuffle and no fresh accumulator per 32 k.
//
// Codes become f16 with one LOP3 per two weights: for Q4_K the nibble itself
// as an f16 subnormal, q * 2^-24 (low nibbles) or 16q * 2^-24 (high nibbles,
// their x staged divided by 16), exact; the 2^24 rides on d.  Q4_K's min term
// dmin * m_j * sum(x over sub-block j) uses sub-block sums of the staged x.
// For Q4_0 the 1024 + q construction minus 1032 (or 1152 for high nibbles)
// gives q - 8 (or 16(q - 8)) exactly.
//
// x is staged per warp (the warp's own units only), each 32-k block scaled
// by a power of two from its own max |x| (undone in the block's epilogue)
// and split into f16 hi + lo (22 significant bits), in the order the B
// fragments read it; lanes outside the diagonal read a zero block.  Each 16-row tile's warp partials are summed in a fixed
// order.  Roles: warp 8 streams stages, warps 0-7 stage x and decode.  Two
// CTAs fit on an SM; tiles are dealt round-robin to a grid of at most two
// CTAs per SM.  One launch may serve a group of up to eight matrices of one
// format and one K that read the same x (a layer's q/k/v, gate/up): their
// tiles form one list, each stage taken through its member's tensor map.  Weights are requested before the programmatic dependency
// wait, x read and y written after it.  Every wait is bounded (~1 s): a
// timeout records Q4_ETIMEOUT, stops the roles, waits for issued copies and
// returns.
#include <cuda.h>

#include "q4_internal.cuh"
#include "tc_gemv_common.cuh"
#include "tma_map.cuh"

namespace q4 {

__device__ int g_blkt_error;
// Limit of the role waits in SM clocks (the producer's final drain of bulk
// copies keeps the full limit).
__device__ long long g_blkt_wait_limit = 1LL << 31;

namespace {

using namespace tc;

constexpr int BT_WARPS = 8;                        // decode warps = units per stage
constexpr int BT_THREADS = (BT_WARPS + 1) * 32;
constexpr int UNIT = 144;                          // bytes of 256 k of one row
constexpr int BT_ROWS = 16;
constexpr int STAGE = BT_WARPS * BT_ROWS * UNIT;   // 18432 bytes, a multiple of 1024
constexpr int MAX_NS = 6;
constexpr int XU = 1024;                           // staged x bytes per unit
constexpr int SMEM_CAP = 112 * 1024;               // two CTAs per SM
constexpr long long BT_WAIT = 1LL << 31;
static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned");

constexpr int BT_MAXM = 8;                         // matrices per launch (a group sharing x and K)

struct BtMaps {
    CUtensorMap w[BT_MAXM];                        // u8 {144, N_i, K/256}, box {144, 16, 8}
};

struct BtArgs {
    const void *x;                 // [K] f32 or bf16, shared by every member
    float *y[BT_MAXM];             // [N_i]
    int64_t N[BT_MAXM];
    int tile_start[BT_MAXM + 1];   // first 16-row tile of each member in the launch's tile list
    int nsb;                       // units (256 k) per row
    int nst;                       // stages per tile
    int ntiles;                    // tiles of all members
    int NS;                        // ring stages
};

// Member owning tile `tile` of the launch's tile list.
__device__ __forceinline__ int member_of(const BtArgs &a, int tile) {
    int m = 0;
#pragma unroll
    for (int i = 1; i < BT_MAXM; i++) m += tile >= a.tile_start[i] ? 1 : 0;
    return m;
}

// Shared-memory layout after the 1024-byte aligned ring: staged x [8 warps][nst][1024],
// a 256-byte zero block at an offset of 64 mod 128 (so its reads never share banks
// with a diagonal lane's), per 32-k block and batch row {x sum, x scale} pairs
// [8][nst][8][MB] x 2 f32, tile partials [2][MB][8][16] f32.
struct Layout {
    int xs, zero, sx, red, total;
};
__host__ __device__ inline Layout layout(int NS, int nst, int mb) {
    Layout L;
    L.xs = NS * STAGE;
    L.zero = L.xs + BT_WARPS * nst * XU + 64;
    L.sx = L.zero + 256 + 64;
    L.red = L.sx + BT_WARPS * nst * 64 * mb;
    L.total = L.red + 2 * mb * BT_WARPS * BT_ROWS * 4;
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
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Eight consecutive x values as f32 (p 16-byte aligned).
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Scale and min bytes of sub-blocks 2t (low byte) and 2t + 1 (next byte) of
// one Q4_K row, from the scale words B0 (bytes 0-3), B1 (4-7), B2 (8-11):
// sub-block j < 4 takes the low 6 bits of bytes j and j + 4; j >= 4 takes
// the nibbles of byte j + 4 and the top two bits of bytes j - 4 and j.
__device__ __forceinline__ void q4k_pair(uint32_t B0, uint32_t B1, uint32_t B2, int t, uint32_t &sc, uint32_t &mn) {
    const uint32_t p = 16u * (uint32_t)(t & 1);
    const uint32_t b0 = B0 >> p, b1 = B1 >> p, b2 = B2 >> p;
    const bool low = t < 2;                     // both forms, then a select: no divergent branch
    sc = low ? (b0 & 0x3F3Fu) : ((b2 & 0x0F0Fu) | ((b0 >> 2) & 0x3030u));
    mn = low ? (b1 & 0x3F3Fu) : (((b2 >> 4) & 0x0F0Fu) | ((b1 >> 2) & 0x3030u));
}

// step * (D_hi + D_lo) - off * S of one sub-block, where D_hi and D_lo are the
// code sums against the x hi and lo parts and S the sub-block's x sum.  The
// two products can be large and nearly cancel (a weight near 0 under a
// dominant x), so off * S is kept as an exact pair (p + e, by an FMA) and the
// cancelling subtraction happens inside one FMA: the rounding error stays
// relative to the sub-block's result, not to the cancelled terms.
__device__ __forceinline__ float q4k_sub(float step, float dh, float dl, float off, float S) {
    const float p = off * S, e = fmaf(off, S, -p);
    return fmaf(step, dl, fmaf(step, dh, -p)) - e;
}
// Steps and offsets of lane t's two sub-blocks of one row (header H = d | dmin,
// scale words): {step_2t, off_2t, step_2t+1, off_2t+1}, the steps carrying the
// 2^24 of the subnormal codes.  Formed before the row's MMAs, off their path.
__device__ __forceinline__ float4 q4k_terms(uint4 H, int t) {
    uint32_t sc, mn;
    q4k_pair(H.y, H.z, H.w, t, sc, mn);
    const float d24 = half_bits_f32(H.x) * 16777216.0f, dmin = half_bits_f32(H.x >> 16);
    return make_float4(d24 * (float)(sc & 255u), dmin * (float)(mn & 255u), d24 * (float)(sc >> 8),
                       dmin * (float)(mn >> 8));
}
// Lane t's two sub-blocks of one row, each in its own x scale:
// sv = {S_2t, 1/scale_2t, S_2t+1, 1/scale_2t+1}.
__device__ __forceinline__ float q4k_rows_term(float4 so, float l0, float l1, float h0, float h1, float4 sv) {
    const float lo = q4k_sub(so.x, l0, l1, so.y, sv.x);
    const float hi = q4k_sub(so.z, h0, h1, so.w, sv.z);
    return fmaf(hi, sv.w, lo * sv.y);
}

// MB = 1: one batch row, B columns 2t and 2t + 1 carrying its f16 hi and lo
// parts.  MB = 2 (bf16 x, whose 8 significant bits need no lo part): two batch
// rows, columns 2t and 2t + 1 carrying one row each, for the MMAs and the
// decode of one.
template <typename XT, bool Q4K, int MB>
__global__ void __launch_bounds__(BT_THREADS, 2)
gemv_blk_tc(const __grid_constant__ BtMaps maps, const __grid_constant__ BtArgs a) {
    static_assert(MB == 1 || (MB == 2 && sizeof(XT) == 2), "two rows per launch need bf16 x");
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[MAX_NS], empty[MAX_NS];
    __shared__ int abort_s;
    uint8_t *ring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int NS = a.NS, nst = a.nst;
    const Layout L = layout(NS, nst, MB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int my_tiles = (int)blockIdx.x < a.ntiles ? (a.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int J = my_tiles * nst;
    volatile int *abort_flag = &abort_s;
    const long long wait_limit = g_blkt_wait_limit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], BT_WARPS);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 64) reinterpret_cast<uint32_t *>(ring + L.zero)[threadIdx.x] = 0u;
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == BT_WARPS) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            int issued = 0;
            for (int j = 0; j < J; j++) {
                const int s = j % NS;
                if (j >= NS && !wait_or_abort(&empty[s], ((j / NS) & 1) ^ 1, abort_flag, &g_blkt_error, wait_limit)) break;
                const int tile = (int)blockIdx.x + (j / nst) * (int)gridDim.x, st = j % nst;
                const int mem = member_of(a, tile);
                mbar_arrive_expect_tx(&full[s], STAGE);
                tma3(smem_u32(ring + s * STAGE), &maps.w[mem], 0, (tile - a.tile_start[mem]) * BT_ROWS,
                     st * BT_WARPS, &full[s], pol);
                issued++;
            }
            for (int q = issued > NS ? issued - NS : 0; q < issued; q++)
                if (!mbar_wait_bounded(&full[q % NS], (uint32_t)((q / NS) & 1), BT_WAIT))
                    atomicExch(&g_blkt_error, Q4_ETIMEOUT);
        }
        __syncwarp();
        return;
    }

    // --------------------------------------- x staging (this warp's units)
    // Each 32-k block (Q4_K sub-block, Q4_0 block: four lanes' eight values)
    // gets its own power-of-two scale from its max |x|, so a value is lost to
    // the f16 range only when it is 2^-37 below its block's largest.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const XT *xp = reinterpret_cast<const XT *>(a.x);
    const uint32_t xs_w = smem_u32(ring + L.xs) + (uint32_t)(warp * nst * XU);
    float *sx_w = reinterpret_cast<float *>(ring + L.sx) + warp * nst * 16 * MB;
    {
        // lane l converts k = 8l .. 8l+7 of each unit: two code words' worth of B values
        int tq, half, i0;
        if (Q4K) {
            tq = lane >> 3;                      // 64-k chunk
            half = (lane >> 2) & 1;              // low / high nibbles
            i0 = 2 * (lane & 3);                 // code word within the chunk
        } else {
            const int b = lane >> 2;             // block
            half = (lane >> 1) & 1;
            tq = b >> 1;
            i0 = 4 * (b & 1) + 2 * (lane & 1);
        }
        for (int s = 0; s < nst; s++) {
            const int u = warp + BT_WARPS * s;
            if (u >= a.nsb) break;
#pragma unroll
            for (int m = 0; m < MB; m++) {
                float v[8];
                load8(xp + (int64_t)m * a.nsb * 256 + (int64_t)u * 256 + 8 * lane, v);
                float amax = 0.0f;
#pragma unroll
                for (int r = 0; r < 8; r++) amax = fmaxf(amax, fabsf(v[r]));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                float xscale = 1.0f, xinv = 1.0f;
                if (amax > 0.0f && amax < INFINITY) {
                    int ex = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;
                    ex = ex < -100 ? -100 : (ex > 100 ? 100 : ex);
                    xscale = __uint_as_float((uint32_t)(127 + 12 - ex) << 23);    // |x| * xscale < 2^13
                    xinv = __uint_as_float((uint32_t)(127 - 12 + ex) << 23);
                }
                const float sc = half ? xscale * 0.0625f : xscale;                // exact: powers of two
                float ssum = 0.0f;
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    const float f0 = v[4 * q] * sc, f1 = v[4 * q + 1] * sc, f2 = v[4 * q + 2] * sc,
                                f3 = v[4 * q + 3] * sc;
                    // B pairs (k, k+2) and (k+1, k+3) as f16
                    const __half2 h02 = __floats2half2_rn(f0, f2), h13 = __floats2half2_rn(f1, f3);
                    const float2 r02 = __half22float2(h02), r13 = __half22float2(h13);
                    // entry (tq, word i0 + q): [part 0: low-nibble half, high-nibble half][part 1: ...], 8 bytes
                    // each; part 0 holds x's hi terms (MB = 1) or row 0 (MB = 2), part 1 its lo terms or row 1
                    const uint32_t e = xs_w + (uint32_t)(s * XU + (tq * 8 + i0 + q) * 32 + half * 8 + m * 16);
                    sts64(e, *reinterpret_cast<const uint32_t *>(&h02), *reinterpret_cast<const uint32_t *>(&h13));
                    if (MB == 1) {
                        const __half2 l02 = __floats2half2_rn(f0 - r02.x, f2 - r02.y);
                        const __half2 l13 = __floats2half2_rn(f1 - r13.x, f3 - r13.y);
                        sts64(e + 16, *reinterpret_cast<const uint32_t *>(&l02), *reinterpret_cast<const uint32_t *>(&l13));
                        if (Q4K) {              // the staged values themselves: the numbers the MMA multiplies
                            const float2 s02 = __half22float2(l02), s13 = __half22float2(l13);
                            ssum += ((r02.x + s02.x) + (r02.y + s02.y)) + ((r13.x + s13.x) + (r13.y + s13.y));
                        }
                    } else if (Q4K) {
                        ssum += (r02.x + r02.y) + (r13.x + r13.y);
                    }
                }
                // the block's x sum in the units the MMA sees x in (Q4_K's min term) and its scale
                if (Q4K) {
                    if (half) ssum *= 16.0f;
                    ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
                    ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
                }
                if ((lane & 3) == 0) {
                    float *o = sx_w + ((s * 8 + (lane >> 2)) * MB + m) * 2;
                    o[0] = ssum;
                    o[1] = xinv;
                }
            }
        }
    }
    __syncwarp();

    // ------------------------------------------------ decode + multiply
    const int g = lane >> 2, t = lane & 3;
    const bool diag = (g >> 1) == t;                                     // supplies B column g in lane t's slots
    const uint32_t xb = diag ? xs_w + (uint32_t)(t * 256 + (g & 1) * 16) : smem_u32(ring + L.zero) + (uint32_t)((g & 1) * 16);
    const uint32_t xstep = diag ? XU : 0u;
    const uint32_t ring_u = smem_u32(ring);
    float *red = reinterpret_cast<float *>(ring + L.red);
    float acc[MB][2] = {};                                               // [batch row][rows g, g + 8]
    bool ok = true;
    int buf = 0;
    for (int j = 0; j < J; j++) {
        const int s = j % NS, st = j % nst;
        if (ok) ok = wait_or_abort(&full[s], (uint32_t)((j / NS) & 1), abort_flag, &g_blkt_error, wait_limit);
        if (ok && warp + BT_WARPS * st < a.nsb) {
            const uint32_t R = ring_u + (uint32_t)(s * STAGE + warp * BT_ROWS * UNIT);
            const uint32_t xa = xb + (uint32_t)st * xstep;
            const uint32_t rg = R + (uint32_t)(g * UNIT), rg8 = rg + 8 * UNIT;
            if constexpr (Q4K) {
                const uint4 H0 = lds128(rg), H1 = lds128(rg8);
                const float4 so0 = q4k_terms(H0, t), so1 = q4k_terms(H1, t);
                // x sums and scales of sub-blocks 2t, 2t + 1: {S, 1/scale} x 2 (MB = 1), or per block both rows
                const float4 sa = *reinterpret_cast<const float4 *>(sx_w + (st * 8 + 2 * t) * 2 * MB);
                const float4 sb = MB == 2 ? *reinterpret_cast<const float4 *>(sx_w + (st * 8 + 2 * t + 1) * 4) : sa;
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
                // sub-blocks 2t (low nibbles) and 2t + 1 (high nibbles) of rows g and g + 8
                if constexpr (MB == 1) {
                    acc[0][0] += q4k_rows_term(so0, Dl[0], Dl[1], Dh[0], Dh[1], sa);
                    acc[0][1] += q4k_rows_term(so1, Dl[2], Dl[3], Dh[2], Dh[3], sa);
                } else {
                    const float4 sv0 = make_float4(sa.x, sa.y, sb.x, sb.y), sv1 = make_float4(sa.z, sa.w, sb.z, sb.w);
                    acc[0][0] += q4k_rows_term(so0, Dl[0], 0.0f, Dh[0], 0.0f, sv0);
                    acc[1][0] += q4k_rows_term(so0, Dl[1], 0.0f, Dh[1], 0.0f, sv1);
                    acc[0][1] += q4k_rows_term(so1, Dl[2], 0.0f, Dh[2], 0.0f, sv0);
                    acc[1][1] += q4k_rows_term(so1, Dl[3], 0.0f, Dh[3], 0.0f, sv1);
                }
            } else {
                // blocks 2t (bytes 36t .. 36t+17) and 2t + 1 (36t+18 .. 36t+35) of rows g and g + 8
                uint32_t W0[9], W1[9];
#pragma unroll
                for (int c = 0; c < 9; c++) {
                    W0[c] = lds32(rg + (uint32_t)(36 * t + 4 * c));
                    W1[c] = lds32(rg8 + (uint32_t)(36 * t + 4 * c));
                }
                // d of blocks 2t and 2t + 1 of both rows, and the blocks' x scales (powers of two: exact)
                const float de0 = half_bits_f32(W0[0]), do0 = half_bits_f32(W0[4] >> 16);
                const float de1 = half_bits_f32(W1[0]), do1 = half_bits_f32(W1[4] >> 16);
                const float4 sa = *reinterpret_cast<const float4 *>(sx_w + (st * 8 + 2 * t) * 2 * MB);
                const float4 sb = MB == 2 ? *reinterpret_cast<const float4 *>(sx_w + (st * 8 + 2 * t + 1) * 4) : sa;
                const float e0s = de0 * sa.y, o0s = do0 * (MB == 1 ? sa.w : sb.y);
                const float e1s = de1 * sa.y, o1s = do1 * (MB == 1 ? sa.w : sb.y);
                uint32_t w0[8], w1[8];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    w0[c] = __funnelshift_r(W0[c], W0[c + 1], 16);     // block 2t: codes start 2 bytes into word 0
                    w1[c] = __funnelshift_r(W1[c], W1[c + 1], 16);
                    w0[4 + c] = W0[5 + c];                              // block 2t + 1: word-aligned codes
                    w1[4 + c] = W1[5 + c];
                }
                float DA[4] = {0.f, 0.f, 0.f, 0.f}, DB[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const uint4 bx = lds128(xa + (uint32_t)(i * 32));
                    const uint32_t s0 = w0[i] >> 8, s1 = w1[i] >> 8;
                    const uint4 al = make_uint4(hsub2_bits((w0[i] & 0x000F000Fu) | 0x64006400u, 0x64086408u),
                                                hsub2_bits((w1[i] & 0x000F000Fu) | 0x64006400u, 0x64086408u),
                                                hsub2_bits((s0 & 0x000F000Fu) | 0x64006400u, 0x64086408u),
                                                hsub2_bits((s1 & 0x000F000Fu) | 0x64006400u, 0x64086408u));
                    const uint4 ah = make_uint4(hsub2_bits((w0[i] & 0x00F000F0u) | 0x64006400u, 0x64806480u),
                                                hsub2_bits((w1[i] & 0x00F000F0u) | 0x64006400u, 0x64806480u),
                                                hsub2_bits((s0 & 0x00F000F0u) | 0x64006400u, 0x64806480u),
                                                hsub2_bits((s1 & 0x00F000F0u) | 0x64006400u, 0x64806480u));
                    if (i < 4) {
                        mma16816(DA, al, bx.x, bx.y);
                        mma16816(DA, ah, bx.z, bx.w);
                    } else {
                        mma16816(DB, al, bx.x, bx.y);
                        mma16816(DB, ah, bx.z, bx.w);
                    }
                }
                if constexpr (MB == 1) {
                    acc[0][0] = fmaf(e0s, DA[0] + DA[1], fmaf(o0s, DB[0] + DB[1], acc[0][0]));
                    acc[0][1] = fmaf(e1s, DA[2] + DA[3], fmaf(o1s, DB[2] + DB[3], acc[0][1]));
                } else {                      // column 2t + m is batch row m; row 1's scales sit at sa.w, sb.w
                    acc[0][0] = fmaf(e0s, DA[0], fmaf(o0s, DB[0], acc[0][0]));
                    acc[1][0] = fmaf(de0 * sa.w, DA[1], fmaf(do0 * sb.w, DB[1], acc[1][0]));
                    acc[0][1] = fmaf(e1s, DA[2], fmaf(o1s, DB[2], acc[0][1]));
                    acc[1][1] = fmaf(de1 * sa.w, DA[3], fmaf(do1 * sb.w, DB[3], acc[1][1]));
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (st == nst - 1) {
            // end of a tile: the four lanes of a row, then the eight warps in a fixed order
            float *rb = red + buf * MB * BT_WARPS * BT_ROWS;
#pragma unroll
            for (int m = 0; m < MB; m++) {
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    acc[m][r] += __shfl_xor_sync(0xffffffffu, acc[m][r], 1);
                    acc[m][r] += __shfl_xor_sync(0xffffffffu, acc[m][r], 2);
                }
                if (t == 0) {
                    rb[(m * BT_WARPS + warp) * BT_ROWS + g] = acc[m][0];
                    rb[(m * BT_WARPS + warp) * BT_ROWS + g + 8] = acc[m][1];
                }
                acc[m][0] = acc[m][1] = 0.0f;
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (threadIdx.x < MB * BT_ROWS) {
                const int m = threadIdx.x / BT_ROWS, rr = threadIdx.x % BT_ROWS;
                const int tile = (int)blockIdx.x + (j / nst) * (int)gridDim.x, mem = member_of(a, tile);
                const int64_t n = (int64_t)(tile - a.tile_start[mem]) * BT_ROWS + rr;
                if (n < a.N[mem]) {
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < BT_WARPS; w++) v += rb[(m * BT_WARPS + w) * BT_ROWS + rr];
                    a.y[mem][(int64_t)m * a.N[mem] + n] = v;
                }
            }
            buf ^= 1;
        }
    }
}

struct Plan {
    int nsb, nst, NS, smem;
};

bool plan_for(int64_t K, int mb, Plan &p) {
    if (K % 256 != 0 || K <= 0 || K > (1LL << 24)) return false;
    p.nsb = (int)(K / 256);
    p.nst = (p.nsb + BT_WARPS - 1) / BT_WARPS;
    const Layout L0 = layout(0, p.nst, mb);
    const int ns = (SMEM_CAP - 1024 - L0.total) / STAGE;
    if (ns < 3) return false;
    p.NS = ns < MAX_NS ? ns : MAX_NS;
    p.smem = 1024 + layout(p.NS, p.nst, mb).total;
    return true;
}

template <typename XT, bool Q4K, int MB>
cudaError_t blk_tc_run(const BtMaps &maps, const BtArgs &a, int smem, cudaStream_t s) {
    auto kern = gemv_blk_tc<XT, Q4K, MB>;
    static bool attr_set[64] = {};
    static int per_sm[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CAP);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, BT_THREADS, SMEM_CAP) != cudaSuccess || b < 1) b = 1;
        per_sm[dev & 63] = b;
        attr_set[dev & 63] = true;
    }
    int grid = per_sm[dev & 63] * sm_count();
    if (grid > a.ntiles) grid = a.ntiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(BT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps, a);
}

bool encode_units(CUtensorMap *map, const Tensor &t, int nsb) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)UNIT, (cuuint64_t)t.N, (cuuint64_t)nsb};
    const cuuint64_t strides[2] = {(cuuint64_t)nsb * UNIT, (cuuint64_t)UNIT};
    const cuuint32_t box[3] = {(cuuint32_t)UNIT, (cuuint32_t)BT_ROWS, (cuuint32_t)BT_WARPS};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(t.w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Q4_K or Q4_0, K % 256 == 0, weights 16-byte aligned, the staged x and three
// ring stages within 112 KB; batch 1 with f32 or bf16 x, batch 2..8 with bf16
// x (launches of two rows).
bool gemv_blk_tc_eligible(const Tensor &t, int64_t M, q4_dtype xd) {
    if ((t.fmt != Q4_Q4K && t.fmt != Q4_Q40) || M < 1 || M > 8 || t.N < 1 || t.N > (1LL << 30)) return false;
    if (M > 1 && xd != Q4_DT_BF16) return false;
    if ((((uintptr_t)t.w) & 15) != 0 || encode_fn() == nullptr) return false;
    Plan p;
    return plan_for(t.K, M > 1 ? 2 : 1, p);
}

// Up to BT_MAXM members of one format and one K (each eligible) that read the
// same x, batch rows M (f32 x: 1; bf16 x: up to 8): one launch per pair of
// rows (and one for an odd last row) whose tile list runs through the members
// in order.  Row m of x is at x + m K; row m of member i's output at ys[i] + m N_i.
cudaError_t launch_gemv_blk_tc_group(const Tensor *ts, int count, const void *x, q4_dtype xd, float *const *ys,
                                     int64_t M, cudaStream_t s) {
    Plan p1, p2;
    if (count < 1 || count > BT_MAXM || M < 1 || M > 8 || (M > 1 && xd != Q4_DT_BF16) || !plan_for(ts[0].K, 1, p1) ||
        (M > 1 && !plan_for(ts[0].K, 2, p2)))
        return cudaErrorInvalidValue;
    BtMaps maps;
    BtArgs base;
    int tiles = 0;
    for (int i = 0; i < BT_MAXM; i++) {
        const int m = i < count ? i : count - 1;     // unused slots repeat the last member (never reached)
        if (i < count) {
            if (ts[i].fmt != ts[0].fmt || ts[i].K != ts[0].K || !encode_units(&maps.w[i], ts[i], p1.nsb))
                return cudaErrorInvalidValue;
        } else {
            maps.w[i] = maps.w[m];
        }
        base.N[i] = ts[m].N;
        base.tile_start[i] = tiles;
        if (i < count) tiles += (int)((ts[i].N + BT_ROWS - 1) / BT_ROWS);
    }
    base.tile_start[BT_MAXM] = tiles;
    for (int i = count; i < BT_MAXM; i++) base.tile_start[i] = tiles;   // empty: member_of never picks them
    base.ntiles = tiles;
    const bool q4k = ts[0].fmt == Q4_Q4K;
    const int64_t xe = xd == Q4_DT_BF16 ? 2 : 4;
    for (int64_t m0 = 0; m0 < M; m0 += 2) {
        const int mb = M - m0 >= 2 ? 2 : 1;
        const Plan &p = mb == 2 ? p2 : p1;
        BtArgs a = base;
        a.x = static_cast<const char *>(x) + m0 * ts[0].K * xe;
        for (int i = 0; i < BT_MAXM; i++) a.y[i] = ys[i < count ? i : count - 1] + m0 * a.N[i];
        a.nsb = p.nsb;
        a.nst = p.nst;
        a.NS = p.NS;
        cudaError_t e;
        if (mb == 2)
            e = q4k ? blk_tc_run<__nv_bfloat16, true, 2>(maps, a, p.smem, s)
                    : blk_tc_run<__nv_bfloat16, false, 2>(maps, a, p.smem, s);
        else if (xd == Q4_DT_BF16)
            e = q4k ? blk_tc_run<__nv_bfloat16, true, 1>(maps, a, p.smem, s)
                    : blk_tc_run<__nv_bfloat16, false, 1>(maps, a, p.smem, s);
        else
            e = q4k ? blk_tc_run<float, true, 1>(maps, a, p.smem, s) : blk_tc_run<float, false, 1>(maps, a, p.smem, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv_blk_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    float *const ys[1] = {y};
    return launch_gemv_blk_tc_group(&t, 1, x, xd, ys, M, s);
}

int blk_tc_set_wait_limit(long long cycles) {
    return cudaMemcpyToSymbol(g_blkt_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int blk_tc_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_blkt_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_blkt_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

}  // namespace q4
