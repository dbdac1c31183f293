// gemv_mma.cu -- NVFP4 decode-GEMV for batch 1..8 with the dot products on the
// tensor cores (mma.sync m16n8k16, f16 x f16 -> f32).
//
// Why tensor cores for a bandwidth-bound GEMV: at HBM speed one GB300 SM must
// retire ~38 NVFP4 weights per clock.  Decoding a weight and multiplying it on
// the CUDA cores costs >= 2 instructions per weight (hardware E2M1 convert,
// half-word extracts, FMA), which is close to the whole issue budget.  Here
// the decode stays in registers and the multiply-accumulate moves to the MMA:
//   * the hardware convert cvt.rn.f16x2.e2m1x2 turns one payload byte (two
//     consecutive k) into exactly one f16x2 A-fragment register;
//   * one HMUL2 by the row's E4M3 block scale (also exact in f16: <= 6
//     significant bits, range 2^-10 .. 2688) folds (e2m1 * e4m3) into A, the
//     first product of the pinned order ([MUS7] 7.1-7.2);
//   * x is B: each activation row m is a column of the MMA, scaled by an
//     exact power of two into f16 (every bf16 value survives unless the
//     slice's dynamic range exceeds ~2^29, in which case the warp computes in
//     f32 on the CUDA cores instead);
//   * f32 accumulation in the MMA, then x 2^-e and x scale2 once per row.
// Columns 0..7 of the MMA are the batch (M <= 8): batch 1..8 cost the same
// weight traffic and decode work.
//
// Work split: a CTA owns one 16-row tile; its W warps split K into contiguous
// runs of 128-k blocks.  Lane (g, t) (g = lane/4, t = lane%4) streams the 16
// payload bytes of rows g and g+8 that hold k = 128b + 32t .. +31 (coalesced:
// 4 lanes cover 64 contiguous bytes of a row) plus their two E4M3 bytes, with
// all of the warp's loads issued before x is staged.  The MMA's 16-k columns
// are mapped to each lane's own k runs (the same permutation is applied to x
// in shared memory), so no lane ever moves a weight between registers.
#include "q4_internal.cuh"

namespace q4 {
namespace {

#ifndef Q4_MMA_MW
#define Q4_MMA_MW 8
#endif
constexpr int MW = Q4_MMA_MW;     // warps per CTA
#ifndef Q4_MMA_PD
#define Q4_MMA_PD 2
#endif
constexpr int PD = Q4_MMA_PD;     // 128-k blocks in flight per warp (register ring)
#ifndef Q4_MMA_NACC
#define Q4_MMA_NACC 4
#endif
constexpr int NACC = Q4_MMA_NACC; // independent accumulator sets (breaks the MMA chain)
constexpr size_t SMEM_MAX = 200 * 1024;

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 128-k block of rows g and g+8 for lane t: 16 payload bytes per row
// (k = 128b + 32t .. +31) and the two E4M3 scales of those 32 k.
struct Blk {
    uint4 p0, p1;
    uint32_t s0, s1;
};

// MXFP4 scale byte b -> 2^(b-127) as an f16x2 pair.  Every E2M1 multiple of
// 2^k is an f16 number exactly when k is in [-23, 13]; outside that range
// `ok` is cleared (the warp then recomputes its tile in f32).
__device__ __forceinline__ uint32_t e8m0_f16x2(uint32_t b, bool &ok) {
    const int k = (int)(b & 255u) - 127;
    ok = ok && k >= -23 && k <= 13;
    const uint32_t h = k >= -14 ? ((uint32_t)(k + 15) & 31u) << 10 : (k >= -24 ? 1u << (k + 24) : 0u);
    return h | (h << 16);
}

// A-fragment source for one payload word (8 k): four f16x2 of e2m1 * scale.
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t sc2, uint32_t (&a)[4]) {
    e2m1x8_h2(w, a[0], a[1], a[2], a[3]);
#pragma unroll
    for (int i = 0; i < 4; i++) a[i] = hmul2_u32(a[i], sc2);
}

// Four bf16 values (two words) times an exact power of two -> two f16x2
// words; `ok` stays true only if every value survives the f16 rounding.
__device__ __forceinline__ uint2 bf16x4_to_f16(uint2 v, float scale, bool &ok) {
    const float f0 = __uint_as_float(v.x << 16) * scale, f1 = __uint_as_float(v.x & 0xffff0000u) * scale;
    const float f2 = __uint_as_float(v.y << 16) * scale, f3 = __uint_as_float(v.y & 0xffff0000u) * scale;
    const __half2 h01 = __floats2half2_rn(f0, f1), h23 = __floats2half2_rn(f2, f3);
    const float2 c01 = __half22float2(h01), c23 = __half22float2(h23);
    ok = ok && c01.x == f0 && c01.y == f1 && c23.x == f2 && c23.y == f3;
    return make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
}

// x slice of one warp as exactly-scaled f16 B fragments, staged once per CTA:
// entry ((i*8 + j)*MT + m)*4 + t = x[m][128(b0+i) + 32t + 4j .. +3] * 2^e_m.
// Lane l serves column m = l % MT only.  Pass 1 loads 16-byte runs (8 k) of
// that row, all independent, keeps the column max and puts the raw bf16 bits
// straight into their two entries; the max is reduced over the lanes of the
// column; pass 2 converts the lane's own entries in place.
template <typename XT, int MT>
__device__ __forceinline__ bool stage_x(const XT *__restrict__ x, int64_t K, int M, int b0, int nbw, int lane,
                                        uint2 *xs, float (&inv)[MT]) {
    static_assert(sizeof(XT) == 2 && 32 % MT == 0, "bf16 activations, MT divides the warp");
    constexpr int LPC = 32 / MT;                // lanes per column
    const int m = lane % MT;
    const bool mv = m < M;
    const int nch = nbw * 16;                   // 16-byte runs in the warp's k range
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)(mv ? m : 0) * K + (int64_t)b0 * 128);
    uint32_t mx2 = 0;                           // packed |bf16| maximum (bit patterns order like values)
#pragma unroll 4
    for (int r = lane / MT; r < nch; r += LPC) {
        const uint4 v = mv ? __ldg(src + r) : make_uint4(0u, 0u, 0u, 0u);
        mx2 = __vmaxu2(mx2, __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                     __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu)));
        const int i = r >> 4, q = r & 15, t = q >> 2, j0 = (q & 3) * 2;
        xs[((i * 8 + j0) * MT + m) * 4 + t] = make_uint2(v.x, v.y);
        xs[((i * 8 + j0 + 1) * MT + m) * 4 + t] = make_uint2(v.z, v.w);
    }
    const uint32_t mxb = (mx2 & 0xffffu) > (mx2 >> 16) ? (mx2 & 0xffffu) : (mx2 >> 16);
    float amax = __uint_as_float(mxb << 16);
#pragma unroll
    for (int off = MT; off < 32; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float scale = 1.0f, iv = 1.0f;
    bool exact = true;
    if (amax > 0.0f) {
        const int ex = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;
        if (ex < -100 || ex > 100)
            exact = false;
        else {
            scale = __uint_as_float((uint32_t)(127 + 12 - ex) << 23);   // max |x * scale| < 2^13
            iv = __uint_as_float((uint32_t)(127 - 12 + ex) << 23);
        }
    }
#pragma unroll 4
    for (int r = lane / MT; r < nch; r += LPC) {
        const int i = r >> 4, q = r & 15, t = q >> 2, j0 = (q & 3) * 2;
        uint2 *e0 = xs + ((i * 8 + j0) * MT + m) * 4 + t, *e1 = xs + ((i * 8 + j0 + 1) * MT + m) * 4 + t;
        const uint2 c0 = bf16x4_to_f16(*e0, scale, exact), c1 = bf16x4_to_f16(*e1, scale, exact);
        *e0 = c0;
        *e1 = c1;
    }
#pragma unroll
    for (int mm = 0; mm < MT; mm++) inv[mm] = __shfl_sync(0xffffffffu, iv, mm);   // lane mm holds column mm
    exact = __all_sync(0xffffffffu, exact);
    __syncwarp();
    return exact;
}

// f32 CUDA-core path for one warp's k range of a 16-row tile (used only when
// the activations' dynamic range is too wide for exact f16 staging, or, for
// MXFP4, when a scale of the slice is outside the exact f16 range).
template <typename XT, int MT, int FMT>
__device__ __noinline__ void warp_rows_f32(const uint8_t *w, const uint8_t *scales, int64_t N, int64_t K,
                                           const XT *__restrict__ x, int M, int64_t n0, int b0, int b1, int lane,
                                           float *rw) {
    for (int rr = 0; rr < 16; rr++) {
        const int64_t n = n0 + rr;
        for (int m = 0; m < MT; m++) {
            float acc = 0.0f;
            if (n < N && m < M)
                for (int64_t k = (int64_t)b0 * 128 + lane; k < (int64_t)b1 * 128; k += 32) {
                    const uint32_t byte = w[n * (K >> 1) + (k >> 1)];
                    const float v = e2m1x2_f32((k & 1) ? (byte >> 4) : (byte & 15u)).x;
                    const float sc = FMT == Q4_NVFP4 ? e4m3_f32(scales[n * (K >> 4) + (k >> 4)])
                                                     : e8m0_f32(scales[n * (K >> 5) + (k >> 5)]);
                    acc = fmaf(v * sc, x_to_f32<XT>(x[(int64_t)m * K + k]), acc);
                }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) rw[rr * MT + m] = acc;
        }
    }
}

// A group of independent GEMVs that share K and the batch M (e.g. the q/k/v
// or gate/up projections of one decoder layer, which read the same x): their
// row tiles form one list so a single persistent launch streams all of them.
constexpr int MAXG = 8;
template <typename XT> struct Group {
    int count;
    int tile_start[MAXG + 1];                      // cumulative 16-row tiles
    const uint8_t *w[MAXG];
    const uint8_t *s[MAXG];
    const XT *x[MAXG];
    float *y[MAXG];
    int64_t N[MAXG];
    float scale2[MAXG];
};

#ifndef Q4_MMA_MINB
#define Q4_MMA_MINB 2
#endif

// Persistent CTAs: each takes tiles blockIdx.x, +gridDim.x, ... of the group's
// tile list; its MW warps split K into runs of nbw_max 128-k blocks (the last
// runs may be shorter).  A register ring of PD blocks per lane runs across
// tile (and member) boundaries, so the next tile's first loads are in flight
// while the current tile finishes; one barrier per tile hands the warp
// partials (double buffered) to a fixed-order final sum.  A warp restages its
// x slice only when the member's activation pointer changes.
// MODE 0: one matrix; 1: two matrices that read the same x (e.g. gate and
// up), the member chosen by one compare per tile; 2: any group.
template <typename XT, int MT, int MODE, int FMT>
__global__ void __launch_bounds__(MW * 32, MT >= 8 ? 1 : Q4_MMA_MINB)
    gemv_mma_nvfp4(const __grid_constant__ Group<XT> grp,
                                                                      int64_t K, int M, int nbw_max) {
    extern __shared__ __align__(16) uint8_t mma_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tt = lane & 3;
    const int nb = (int)(K >> 7);
    const int b0 = min(nb, warp * nbw_max), b1 = min(nb, (warp + 1) * nbw_max), nbw = b1 - b0;
    uint2 *xs = reinterpret_cast<uint2 *>(mma_smem) + (size_t)warp * nbw_max * 8 * MT * 4;
    float *red = reinterpret_cast<float *>(mma_smem + (size_t)MW * nbw_max * 8 * MT * 4 * sizeof(uint2));
    const int ntiles = MODE == 2 ? grp.tile_start[grp.count] : grp.tile_start[MODE == 1 ? 2 : 1];

    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int items = my_tiles * nbw_max;          // every warp walks the same item count

    // Load cursor: walks items (tile, block) in order with offset increments
    // only; a new tile recomputes its row offsets once.  Rows past N are
    // clamped to N-1 (valid memory; their results are never stored).  Scale
    // offsets are payload offsets / 8 (K/16 = (K/2)/8 bytes per row).
    const uint32_t rowb = (uint32_t)(K >> 1);
    const uint8_t *lw = grp.w[0], *ls = grp.s[0];
    bool lsec = false;                             // MODE 1: the load cursor is in the second matrix
    uint32_t ow0 = 0, ow_d = 0;
    int lc_i = 0, lc_tile = blockIdx.x, lc_p = 0;
    auto cursor_tile = [&](int tile) {
        lc_tile = tile;
        lc_i = 0;
        if (tile >= ntiles) return;
        int64_t Np, n0;
        if (MODE == 2) {
            while (lc_p + 1 < grp.count && tile >= grp.tile_start[lc_p + 1]) lc_p++;
            Np = grp.N[lc_p];
            lw = grp.w[lc_p];
            ls = grp.s[lc_p];
            n0 = (int64_t)(tile - grp.tile_start[lc_p]) * 16;
        } else if (MODE == 1) {
            lsec = tile >= grp.tile_start[1];
            Np = lsec ? grp.N[1] : grp.N[0];
            n0 = (int64_t)(tile - (lsec ? grp.tile_start[1] : 0)) * 16;
        } else {
            Np = grp.N[0];
            n0 = (int64_t)tile * 16;
        }
        const uint32_t r0 = (uint32_t)((n0 + g) < Np ? (n0 + g) : (Np - 1));
        const uint32_t r1 = (uint32_t)((n0 + g + 8) < Np ? (n0 + g + 8) : (Np - 1));
        ow0 = r0 * rowb + (uint32_t)b0 * 64 + 16 * tt;
        ow_d = (r1 - r0) * rowb;
    };
    cursor_tile(blockIdx.x);
    auto load_next = [&](Blk &r) {
        if (lc_tile < ntiles) {
            if (lc_i < nbw) {
                const uint8_t *bw = MODE == 2 ? lw : MODE == 1 ? (lsec ? grp.w[1] : grp.w[0]) : grp.w[0];
                const uint8_t *bs = MODE == 2 ? ls : MODE == 1 ? (lsec ? grp.s[1] : grp.s[0]) : grp.s[0];
                r.p0 = ldg_stream16(bw + ow0);
                r.p1 = ldg_stream16(bw + ow0 + ow_d);
                if (FMT == Q4_NVFP4) {   // two E4M3 scales per 32 k: payload offset / 8
                    r.s0 = ldg_stream2(bs + (ow0 >> 3));
                    r.s1 = ldg_stream2(bs + ((ow0 + ow_d) >> 3));
                } else {                 // one E8M0 scale per 32 k: payload offset / 16
                    r.s0 = ldg_stream1(bs + (ow0 >> 4));
                    r.s1 = ldg_stream1(bs + ((ow0 + ow_d) >> 4));
                }
            }
            ow0 += 64;
            if (++lc_i == nbw_max) cursor_tile(lc_tile + gridDim.x);
        }
    };
    Blk buf[PD];
#pragma unroll
    for (int q = 0; q < PD; q++) load_next(buf[q]);

    // Programmatic dependent launch: let the next kernel in the stream start
    // its own weight prefetch as SMs free up, and wait for the previous one
    // (which may have produced x) before reading activations.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float inv[MT];
#pragma unroll
    for (int m = 0; m < MT; m++) inv[m] = 1.0f;
    bool exact = true;
    bool sok = true;                                   // MXFP4: every scale of the tile in the exact range
    int staged = -1;                                   // member whose x is in shared memory
    const int mlane = g < M ? g : 0;
    const uint2 *xbase = xs + mlane * 4 + tt;

    float dacc[NACC][4];
#pragma unroll
    for (int a = 0; a < NACC; a++) dacc[a][0] = dacc[a][1] = dacc[a][2] = dacc[a][3] = 0.0f;
    int ci = 0, ctile = blockIdx.x, cp = 0, par = 0;   // compute cursor
    const uint2 *xb = xbase;
    for (int u0 = 0; u0 < items; u0 += PD) {
#pragma unroll
        for (int q = 0; q < PD; q++) {
            const int u = u0 + q;
            if (u < items) {
                const int i = ci;
                if (i == 0) {                          // a new tile: its member's x staged?
                    if (MODE == 2) {
                        while (cp + 1 < grp.count && ctile >= grp.tile_start[cp + 1]) cp++;
                        if (staged < 0 || grp.x[cp] != grp.x[staged]) {
                            staged = cp;
                            if (nbw > 0) exact = stage_x<XT, MT>(grp.x[cp], K, M, b0, nbw, lane, xs, inv);
                        }
                    } else if (staged < 0) {
                        staged = 0;
                        if (nbw > 0) exact = stage_x<XT, MT>(grp.x[0], K, M, b0, nbw, lane, xs, inv);
                    }
                }
                const Blk r = buf[q];
                load_next(buf[q]);
                if (i < nbw && exact) {
                    uint32_t sc0[2], sc1[2];
                    if (FMT == Q4_NVFP4) {
                        uint32_t h0, h1;
                        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"((uint16_t)r.s0));
                        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"((uint16_t)r.s1));
                        sc0[0] = prmt(h0, h0, 0x1010u);
                        sc0[1] = prmt(h0, h0, 0x3232u);
                        sc1[0] = prmt(h1, h1, 0x1010u);
                        sc1[1] = prmt(h1, h1, 0x3232u);
                    } else {
                        sc0[0] = sc0[1] = e8m0_f16x2(r.s0, sok);
                        sc1[0] = sc1[1] = e8m0_f16x2(r.s1, sok);
                    }
                    const uint32_t w0[4] = {r.p0.x, r.p0.y, r.p0.z, r.p0.w};
                    const uint32_t w1[4] = {r.p1.x, r.p1.y, r.p1.z, r.p1.w};
#pragma unroll
                    for (int w = 0; w < 4; w++) {
                        uint32_t a[4], c[4];
                        decode_word(w0[w], sc0[w >> 1], a);
                        decode_word(w1[w], sc1[w >> 1], c);
                        // lanes g >= M read column 0's x: MMA columns >= M are never stored
                        const uint2 bA = xb[(2 * w) * MT * 4], bB = xb[(2 * w + 1) * MT * 4];
                        mma16816(dacc[(2 * w) % NACC], a[0], c[0], a[1], c[1], bA.x, bA.y);
                        mma16816(dacc[(2 * w + 1) % NACC], a[2], c[2], a[3], c[3], bB.x, bB.y);
                    }
                }
                xb += 8 * MT * 4;
                const int ti = ctile;
                if (++ci == nbw_max) { ci = 0; ctile += gridDim.x; xb = xbase; }
                if (i == nbw_max - 1) {
                    // ---- end of tile `ti`: partials -> shared, one barrier, final sum
                    const int mb = MODE == 2 ? cp : MODE == 1 ? (ti >= grp.tile_start[1] ? 1 : 0) : 0;
                    const int64_t Np = grp.N[mb];
                    const int64_t n0 = (int64_t)(ti - grp.tile_start[mb]) * 16;
                    float *rw = red + (par * MW + warp) * 16 * MT;
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int a = 0; a < NACC; a++) {
                        d[0] += dacc[a][0]; d[1] += dacc[a][1]; d[2] += dacc[a][2]; d[3] += dacc[a][3];
                        dacc[a][0] = dacc[a][1] = dacc[a][2] = dacc[a][3] = 0.0f;
                    }
                    bool tile_ok = exact;
                    if (FMT != Q4_NVFP4) {
                        tile_ok = __all_sync(0xffffffffu, sok) && exact;
                        sok = true;
                    }
                    if (tile_ok) {
#pragma unroll
                        for (int mm = 0; mm < MT; mm++) {
                            if (mm == 2 * tt) { rw[g * MT + mm] = d[0] * inv[mm]; rw[(g + 8) * MT + mm] = d[2] * inv[mm]; }
                            if (mm == 2 * tt + 1) { rw[g * MT + mm] = d[1] * inv[mm]; rw[(g + 8) * MT + mm] = d[3] * inv[mm]; }
                        }
                    } else {
                        warp_rows_f32<XT, MT, FMT>(grp.w[mb], grp.s[mb], Np, K, grp.x[mb], M, n0, b0, b1, lane, rw);
                    }
                    __syncthreads();
                    const float *rt = red + par * MW * 16 * MT;
                    par ^= 1;
                    float *yp = grp.y[mb];
                    const float s2 = FMT == Q4_NVFP4 ? grp.scale2[mb] : 1.0f;
                    for (int e = threadIdx.x; e < 16 * MT; e += blockDim.x) {
                        const int rr = e / MT, m = e % MT;
                        const int64_t n = n0 + rr;
                        if (n < Np && m < M) {
                            float sum = 0.0f;
                            for (int w = 0; w < MW; w++) sum += rt[w * 16 * MT + e];
                            yp[(int64_t)m * Np + n] = sum * s2;
                        }
                    }
                }
            }
        }
    }
}

template <typename Kern> int max_blocks_mma(Kern k, size_t smem) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, MW * 32, smem) != cudaSuccess || b < 1) b = 1;
    return b;
}

size_t smem_bytes(int64_t K, int mt) {
    const int nb = (int)(K >> 7), nbw_max = (nb + MW - 1) / MW;
    return (size_t)MW * nbw_max * 8 * mt * 4 * sizeof(uint2) + 2 * (size_t)MW * 16 * mt * sizeof(float);
}

int mt_for(int64_t M) { return M == 1 ? 1 : (M == 2 ? 2 : (M <= 4 ? 4 : 8)); }

template <typename XT, int MT, int MODE, int FMT = Q4_NVFP4>
cudaError_t run_group(const Group<XT> &grp, int64_t K, int M, cudaStream_t s) {
    auto kern = gemv_mma_nvfp4<XT, MT, MODE, FMT>;
    const size_t smem = smem_bytes(K, MT);
    static bool attr_set[64] = {};
    static int bps_cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_MAX);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    const int nb = (int)(K >> 7), nbw_max = (nb + MW - 1) / MW;
    const int ntiles = grp.tile_start[grp.count];
    // occupancy measured once with the largest x area (smem only shrinks below it)
    if (!bps_cache[dev & 63]) bps_cache[dev & 63] = max_blocks_mma(kern, smem);
    int grid = bps_cache[dev & 63] * sm_count();
    if (grid > ntiles) grid = ntiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(MW * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, grp, K, M, nbw_max);
}

template <typename XT>
cudaError_t launch_group_x(const Tensor *ts, const void *const *xs, float *const *ys, int count, int64_t M,
                           cudaStream_t s) {
    Group<XT> grp = {};
    grp.count = count;
    grp.tile_start[0] = 0;
    for (int i = 0; i < count; i++) {
        grp.w[i] = ts[i].w;
        grp.s[i] = ts[i].scales;
        grp.x[i] = (const XT *)xs[i];
        grp.y[i] = ys[i];
        grp.N[i] = ts[i].N;
        grp.scale2[i] = ts[i].scale2;
        grp.tile_start[i + 1] = grp.tile_start[i] + (int)((ts[i].N + 15) / 16);
    }
    const int64_t K = ts[0].K;
    const int m = (int)M;
    if (ts[0].fmt == Q4_MXFP4) {   // single matrix only (groups are NVFP4)
        if (m == 1) return run_group<XT, 1, 0, Q4_MXFP4>(grp, K, m, s);
        if (m == 2) return run_group<XT, 2, 0, Q4_MXFP4>(grp, K, m, s);
        if (m <= 4) return run_group<XT, 4, 0, Q4_MXFP4>(grp, K, m, s);
        return run_group<XT, 8, 0, Q4_MXFP4>(grp, K, m, s);
    }
    if (count == 2 && xs[0] == xs[1]) {
        if (m == 1) return run_group<XT, 1, 1>(grp, K, m, s);
        if (m == 2) return run_group<XT, 2, 1>(grp, K, m, s);
        if (m <= 4) return run_group<XT, 4, 1>(grp, K, m, s);
        return run_group<XT, 8, 1>(grp, K, m, s);
    }
    if (count > 1) {
        if (m == 1) return run_group<XT, 1, 2>(grp, K, m, s);
        if (m == 2) return run_group<XT, 2, 2>(grp, K, m, s);
        if (m <= 4) return run_group<XT, 4, 2>(grp, K, m, s);
        return run_group<XT, 8, 2>(grp, K, m, s);
    }
    if (m == 1) return run_group<XT, 1, 0>(grp, K, m, s);
    if (m == 2) return run_group<XT, 2, 0>(grp, K, m, s);
    if (m <= 4) return run_group<XT, 4, 0>(grp, K, m, s);
    return run_group<XT, 8, 0>(grp, K, m, s);
}

}  // namespace

// Eligible: NVFP4, K % 128 == 0, x slice fits in shared memory.
bool gemv_mma_eligible(const Tensor &t, int64_t M) {
    return (t.fmt == Q4_NVFP4 || t.fmt == Q4_MXFP4) && M >= 1 && M <= 8 && t.K % 128 == 0 &&
           smem_bytes(t.K, mt_for(M)) <= SMEM_MAX &&
           t.N * (t.K / 2) < (int64_t(1) << 32) &&
           (((uintptr_t)t.w | (uintptr_t)t.scales) & 15) == 0;
}

// Several NVFP4 GEMVs with the same K and M in one launch (each eligible on
// its own; count <= MAXG; bf16 activations).
cudaError_t launch_gemv_mma_group(const Tensor *ts, const void *const *xs, float *const *ys, int count, int64_t M,
                                  cudaStream_t s) {
    if (count < 1 || count > MAXG) return cudaErrorInvalidValue;
    return launch_group_x<__nv_bfloat16>(ts, xs, ys, count, M, s);
}

cudaError_t launch_gemv_mma(const Tensor &t, const void *x, q4_dtype, float *y, int64_t M, cudaStream_t s) {
    return launch_gemv_mma_group(&t, &x, &y, 1, M, s);
}

}  // namespace q4
