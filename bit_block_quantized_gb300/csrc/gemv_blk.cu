// gemv_blk.cu -- Q4_K and Q4_0 decode-GEMV for batch 1..8 on the tensor
// cores (mma.sync m16n8k16, f16 x f16 -> f32) with one fresh accumulator per
// 32-k group (Q4_K sub-block, Q4_0 block), scaled on the CUDA cores.
//
// Q4_K weights are w = q * (d*sc_j) - dmin*m_j ([FBTC] sections 5-6).  The
// step d*sc_j has up to 17 significant bits, so it cannot ride in an f16 MMA
// operand exactly; the 4-bit code q can.  For each 16-row tile and 32-k
// sub-block j the MMA forms D_j = sum_k q*x (two k16 MMAs from a zero
// accumulator), and each lane adds step_j*D_j - off_j*S_j to its f32 sums,
// where S_j = sum_k x over the sub-block was formed when x was staged.
//
// Lane (g, t) owns rows g and g+8 of the tile.  The four lanes of a row take,
// for every k16 chunk, the four codes k = 4t..4t+3 of that chunk: one 32-bit
// load of the super-block's code bytes.  Inside the chunk the MMA's k slots
// (2t, 2t+1 | 2t+8, 2t+9) carry the actual k (4t, 4t+2 | 4t+1, 4t+3), so one
// LOP3 per A register turns the word's nibbles into exact f16 codes (the
// 1024 + q construction); x is staged in the same order.  The word's low
// nibbles feed k16 chunk s, its high nibbles chunk s + 2 of the same 64-k
// chunk.
//
// Q4_0 ([BPA] "Real layouts compared") uses the same 256-k unit: 8 blocks of
// 18 bytes (fp16 d, then 16 code bytes whose low nibbles are elements 0-15
// and high nibbles 16-31).  A holds q - 8 (exact), and each lane adds
// d_b * D_b per block; the code words of even blocks start 2 bytes off a
// 4-byte boundary and are assembled from two aligned words by a funnel shift.
//
// Activations (f32 or bf16) are staged once per CTA as hi + lo f16 pairs
// after an exact power-of-two column scale, so each value keeps 22 of its
// significand bits (relative error <= 2^-22, far inside the GEMV tolerance);
// two MMAs per chunk take the two parts.
#include "q4_internal.cuh"

namespace q4 {
namespace {

constexpr int BW = 8;                   // warps per CTA (split K by super-blocks)
constexpr size_t BLK_SMEM_MAX = 200 * 1024;

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two 4-bit codes (bits 0-3 and 16-19 of v) -> f16x2 of q - BIAS, exact.
template <int BIAS>
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t v) {
    const uint32_t mask = 0x000f000fu, magic = 0x64006400u;   // f16x2 (1024, 1024)
    const uint32_t base = BIAS == 8 ? 0x64086408u : 0x64006400u;  // f16x2 (1024 + BIAS)
    uint32_t h, d;
    asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(h) : "r"(v), "r"(mask), "r"(magic));   // (v & mask) | magic
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h), "r"(base));                     // (1024 + q) - (1024 + BIAS)
    return d;
}

// Per-warp staged activations for one super-block u, k16 chunk c, column m,
// lane t: entry ((u*16 + c)*MT + m)*4 + t holds the B fragment
// {x[k0+4t], x[k0+4t+2] | x[k0+4t+1], x[k0+4t+3]} (k0 = 256(sb0+u) + 16c) as
// f16 hi parts, and the same index of the lo array the remainders.  S holds
// the per-sub-block sums ((u*8 + j)*MT + m).
template <typename XT>
__device__ __forceinline__ float xval(const XT *x, int64_t i) {
    return x_to_f32<XT>(x[i]);
}

// Four consecutive activations (k, k+1, k+2, k+3) as f32, one vector load.
__device__ __forceinline__ float4 x4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ float4 x4(const __nv_bfloat16 *p) {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xffff0000u));
}

template <typename XT, int MT, bool SUMS>
__device__ void stage_x_blk(const XT *__restrict__ x, int64_t K, int M, int sb0, int nsb, int lane, uint2 *xh,
                            uint2 *xl, float *S, float (&inv)[MT]) {
    // column scale: max |x| over the warp's slice -> 2^(12 - e), exact
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; m++) amax[m] = 0.0f;
    const int nq = nsb * 64;                      // 4-value groups per column
#pragma unroll 4
    for (int i = lane; i < nq; i += 32) {
#pragma unroll
        for (int m = 0; m < MT; m++)
            if (m < M) {
                const float4 v = x4(x + (int64_t)m * K + (int64_t)sb0 * 256 + 4 * i);
                amax[m] = fmaxf(amax[m], fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
    }
    float scale[MT];
#pragma unroll
    for (int m = 0; m < MT; m++) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) amax[m] = fmaxf(amax[m], __shfl_xor_sync(0xffffffffu, amax[m], off));
        scale[m] = 1.0f;
        inv[m] = 1.0f;
        if (amax[m] > 0.0f && amax[m] < INFINITY) {
            int ex = (int)((__float_as_uint(amax[m]) >> 23) & 255u) - 127;
            ex = ex < -100 ? -100 : (ex > 100 ? 100 : ex);
            scale[m] = __uint_as_float((uint32_t)(127 + 12 - ex) << 23);
            inv[m] = __uint_as_float((uint32_t)(127 - 12 + ex) << 23);
        }
    }
    // fragments: entry e = ((u*16 + c)*MT + m)*4 + t holds x[k0 + 4t + {0, 2 | 1, 3}]
    const int entries = nsb * 16 * MT * 4;
#pragma unroll 4
    for (int e = lane; e < entries; e += 32) {
        const int t = e & 3, m = (e >> 2) % MT, c = (e / (4 * MT)) & 15, u = e / (64 * MT);
        uint2 hi = make_uint2(0u, 0u), lo = make_uint2(0u, 0u);
        if (m < M) {
            float sc = 1.0f;
#pragma unroll
            for (int mm = 0; mm < MT; mm++)
                if (mm == m) sc = scale[mm];
            const float4 v = x4(x + (int64_t)m * K + (int64_t)(sb0 + u) * 256 + 16 * c + 4 * t);
            const float v0 = v.x * sc, v1 = v.y * sc, v2 = v.z * sc, v3 = v.w * sc;
            const __half2 h02 = __floats2half2_rn(v0, v2), h13 = __floats2half2_rn(v1, v3);
            const float2 r02 = __half22float2(h02), r13 = __half22float2(h13);
            const __half2 l02 = __floats2half2_rn(v0 - r02.x, v2 - r02.y);
            const __half2 l13 = __floats2half2_rn(v1 - r13.x, v3 - r13.y);
            hi = make_uint2(*reinterpret_cast<const uint32_t *>(&h02), *reinterpret_cast<const uint32_t *>(&h13));
            lo = make_uint2(*reinterpret_cast<const uint32_t *>(&l02), *reinterpret_cast<const uint32_t *>(&l13));
        }
        xh[e] = hi;
        xl[e] = lo;
    }
    __syncwarp();
    if (!SUMS) return;
    // sub-block sums ((u*8 + j)*MT + m) of the staged values (hi + lo): the
    // same numbers the MMA multiplies
    const int nsum = nsb * 8 * MT;
    for (int e = lane; e < nsum; e += 32) {
        const int m = e % MT, j = (e / MT) & 7, u = e / (8 * MT);
        float sacc = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; h++)
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const int idx = ((u * 16 + 2 * j + h) * MT + m) * 4 + t;
                const uint2 vh = xh[idx], vl = xl[idx];
                const float2 a0 = __half22float2(*reinterpret_cast<const __half2 *>(&vh.x));
                const float2 a1 = __half22float2(*reinterpret_cast<const __half2 *>(&vh.y));
                const float2 b0 = __half22float2(*reinterpret_cast<const __half2 *>(&vl.x));
                const float2 b1 = __half22float2(*reinterpret_cast<const __half2 *>(&vl.y));
                sacc += ((a0.x + b0.x) + (a0.y + b0.y)) + ((a1.x + b1.x) + (a1.y + b1.y));
            }
        S[e] = sacc;
    }
    __syncwarp();
}

// 6-bit scale and min of sub-block j from the metadata words B0 (bytes 0-3),
// B1 (4-7), B2 (8-11) ([FBTC] section 6).
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

struct BlkArgs {
    const uint8_t *w;   // Q4_K blocks [N][K/256][144] or Q4_0 blocks [N][K/32][18]
    const void *x;      // [M][K] f32 or bf16
    float *y;           // [M][N]
    int64_t N, K;
    int M;
    int nsbw;           // super-blocks per warp
};

// One 256-k unit of rows g and g+8 for lane t.
//   Q4_K: header word t of each row (h0, h1) and the eight code words
//         (64-k chunk cc, half h) at bytes 16 + 32cc + 16h + 4t.
//   Q4_0: c[b] = code bytes 4t..4t+3 of block b (unit bytes 18b+2+4t ..),
//         h = the fp16 d of blocks 2t (low half) and 2t+1 (high half).
struct SB {
    uint32_t h0, h1;
    uint32_t c0[8], c1[8];
};

template <int FMT>
__device__ __forceinline__ void load_sb(const uint8_t *r0, const uint8_t *r1, int t, SB &s) {
    const uint32_t *w0 = reinterpret_cast<const uint32_t *>(r0), *w1 = reinterpret_cast<const uint32_t *>(r1);
    if constexpr (FMT == Q4_Q4K) {
        s.h0 = __ldg(w0 + t);
        s.h1 = __ldg(w1 + t);
#pragma unroll
        for (int q = 0; q < 8; q++) {
            s.c0[q] = __ldg(w0 + 4 + 4 * q + t);
            s.c1[q] = __ldg(w1 + 4 + 4 * q + t);
        }
    } else {
        // d of block 2t sits in the low half of word 9t, of block 2t+1 in the high half of word 9t+4
        s.h0 = (__ldg(w0 + 9 * t) & 0xffffu) | (__ldg(w0 + 9 * t + 4) & 0xffff0000u);
        s.h1 = (__ldg(w1 + 9 * t) & 0xffffu) | (__ldg(w1 + 9 * t + 4) & 0xffff0000u);
#pragma unroll
        for (int b = 0; b < 8; b++) {
            // code bytes 18b + 2 + 4t: word-aligned for odd b, 2 bytes past a word for even b
            if (b & 1) {
                s.c0[b] = __ldg(w0 + (18 * b + 2) / 4 + t);
                s.c1[b] = __ldg(w1 + (18 * b + 2) / 4 + t);
            } else {
                const int wi = (18 * b) / 4 + t;
                s.c0[b] = __funnelshift_r(__ldg(w0 + wi), __ldg(w0 + wi + 1), 16);
                s.c1[b] = __funnelshift_r(__ldg(w1 + wi), __ldg(w1 + wi + 1), 16);
            }
        }
    }
}

template <typename XT, int MT, int FMT>
__global__ void __launch_bounds__(BW * 32, 2) gemv_mma_blk(const __grid_constant__ BlkArgs a) {
    extern __shared__ __align__(16) uint8_t blk_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nsb = (int)(a.K >> 8);
    const int sb0 = min(nsb, warp * a.nsbw), sb1 = min(nsb, (warp + 1) * a.nsbw), nsbw = sb1 - sb0;
    const size_t xw = (size_t)a.nsbw * 16 * MT * 4;           // entries per warp
    uint2 *xh = reinterpret_cast<uint2 *>(blk_smem) + (size_t)warp * 2 * xw;
    uint2 *xl = xh + xw;
    float *S = reinterpret_cast<float *>(reinterpret_cast<uint2 *>(blk_smem) + (size_t)BW * 2 * xw) +
               (size_t)warp * a.nsbw * 8 * MT;
    float *red = reinterpret_cast<float *>(reinterpret_cast<uint2 *>(blk_smem) + (size_t)BW * 2 * xw) +
                 (size_t)BW * a.nsbw * 8 * MT;
    const int ntiles = (int)((a.N + 15) / 16);
    const int64_t row_bytes = (int64_t)nsb * 144;
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int items = my_tiles * a.nsbw;                      // every warp walks the same count

    // item i = (tile blockIdx.x + (i / nsbw_max) * gridDim.x, super-block i % nsbw_max)
    auto load_item = [&](int i, SB &s) {
        const int u = i % a.nsbw;
        if (u >= nsbw) return;
        const int64_t n0 = (int64_t)(blockIdx.x + (i / a.nsbw) * gridDim.x) * 16;
        const int64_t ra = n0 + g < a.N ? n0 + g : a.N - 1, rb = n0 + g + 8 < a.N ? n0 + g + 8 : a.N - 1;
        load_sb<FMT>(a.w + ra * row_bytes + (int64_t)(sb0 + u) * 144, a.w + rb * row_bytes + (int64_t)(sb0 + u) * 144,
                     t, s);
    };
    SB cur, nxt;
    if (items > 0) load_item(0, cur);        // weight bytes do not depend on the previous kernel

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float inv[MT];
    if (nsbw > 0) stage_x_blk<XT, MT, FMT == Q4_Q4K>((const XT *)a.x, a.K, a.M, sb0, nsbw, lane, xh, xl, S, inv);
    else {
#pragma unroll
        for (int m = 0; m < MT; m++) inv[m] = 1.0f;
    }
    const int mcol = g < MT ? g : 0;                  // B column of this lane
    const int c2a = 2 * t < MT ? 2 * t : 0, c2b = 2 * t + 1 < MT ? 2 * t + 1 : 0;

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < items; i++) {
        if (i + 1 < items) load_item(i + 1, nxt);
        const int u = i % a.nsbw;
        if (u < nsbw) {
            const uint2 *xhu = xh + (size_t)u * 16 * MT * 4 + mcol * 4 + t;
            const uint2 *xlu = xl + (size_t)u * 16 * MT * 4 + mcol * 4 + t;
            if constexpr (FMT == Q4_Q4K) {
                // the full 16-byte headers of rows g and g+8 (word t' from lane 4g + t')
                uint32_t H0[4], H1[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    H0[q] = __shfl_sync(0xffffffffu, cur.h0, (lane & ~3) | q);
                    H1[q] = __shfl_sync(0xffffffffu, cur.h1, (lane & ~3) | q);
                }
                // this lane's sub-blocks 2t and 2t+1 of both rows: step and offset
                float st[4], of[4];   // [row g: 2t, 2t+1 | row g+8: 2t, 2t+1]
                {
                    const float d0 = half_bits_f32(H0[0]), m0 = half_bits_f32(H0[0] >> 16);
                    const float d1 = half_bits_f32(H1[0]), m1 = half_bits_f32(H1[0] >> 16);
#pragma unroll
                    for (int q = 0; q < 2; q++) {
                        uint32_t sc, mn;
                        q4k_sc_m(H0[1], H0[2], H0[3], 2 * t + q, sc, mn);
                        st[q] = d0 * (float)sc;
                        of[q] = m0 * (float)mn;
                        q4k_sc_m(H1[1], H1[2], H1[3], 2 * t + q, sc, mn);
                        st[2 + q] = d1 * (float)sc;
                        of[2 + q] = m1 * (float)mn;
                    }
                }
                const float *Su = S + (size_t)u * 8 * MT;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    // sub-block j = k16 chunks 2j, 2j+1 = 64-k chunk j/2, nibble j%2,
                    // code words (j/2, 0) and (j/2, 1)
                    const int cc = j >> 1, sh = 4 * (j & 1);
                    float dj[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const uint32_t w0 = cur.c0[2 * cc + h] >> sh, w1 = cur.c1[2 * cc + h] >> sh;
                        const uint32_t a0 = codes_f16x2<0>(w0), a2 = codes_f16x2<0>(w0 >> 8);
                        const uint32_t a1 = codes_f16x2<0>(w1), a3 = codes_f16x2<0>(w1 >> 8);
                        const int c = 4 * cc + 2 * (j & 1) + h;   // k16 chunk of the super-block
                        const uint2 bh = xhu[(size_t)c * MT * 4], bl = xlu[(size_t)c * MT * 4];
                        mma16816(dj, a0, a1, a2, a3, bh.x, bh.y);
                        mma16816(dj, a0, a1, a2, a3, bl.x, bl.y);
                    }
                    // step and offset of sub-block j for rows g, g+8: lane 4g + j/2 computed them
                    const int src = (lane & ~3) | (j >> 1);
                    const float sg = __shfl_sync(0xffffffffu, (j & 1) ? st[1] : st[0], src);
                    const float og = __shfl_sync(0xffffffffu, (j & 1) ? of[1] : of[0], src);
                    const float sg8 = __shfl_sync(0xffffffffu, (j & 1) ? st[3] : st[2], src);
                    const float og8 = __shfl_sync(0xffffffffu, (j & 1) ? of[3] : of[2], src);
                    const float sa = Su[j * MT + c2a], sb = Su[j * MT + c2b];
                    acc[0] = fmaf(sg, dj[0], fmaf(-og, sa, acc[0]));
                    acc[1] = fmaf(sg, dj[1], fmaf(-og, sb, acc[1]));
                    acc[2] = fmaf(sg8, dj[2], fmaf(-og8, sa, acc[2]));
                    acc[3] = fmaf(sg8, dj[3], fmaf(-og8, sb, acc[3]));
                }
            } else {
#pragma unroll
                for (int b = 0; b < 8; b++) {
                    // block b = k16 chunks 2b (low nibbles) and 2b+1 (high nibbles)
                    float dj[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const uint32_t w0 = cur.c0[b] >> (4 * h), w1 = cur.c1[b] >> (4 * h);
                        const uint32_t a0 = codes_f16x2<8>(w0), a2 = codes_f16x2<8>(w0 >> 8);
                        const uint32_t a1 = codes_f16x2<8>(w1), a3 = codes_f16x2<8>(w1 >> 8);
                        const uint2 bh = xhu[(size_t)(2 * b + h) * MT * 4], bl = xlu[(size_t)(2 * b + h) * MT * 4];
                        mma16816(dj, a0, a1, a2, a3, bh.x, bh.y);
                        mma16816(dj, a0, a1, a2, a3, bl.x, bl.y);
                    }
                    // d of block b for rows g, g+8: lane 4g + b/2 loaded it (half b%2)
                    const int src = (lane & ~3) | (b >> 1);
                    const uint32_t dg = __shfl_sync(0xffffffffu, cur.h0, src) >> (16 * (b & 1));
                    const uint32_t dg8 = __shfl_sync(0xffffffffu, cur.h1, src) >> (16 * (b & 1));
                    const float fg = half_bits_f32(dg), fg8 = half_bits_f32(dg8);
                    acc[0] = fmaf(fg, dj[0], acc[0]);
                    acc[1] = fmaf(fg, dj[1], acc[1]);
                    acc[2] = fmaf(fg8, dj[2], acc[2]);
                    acc[3] = fmaf(fg8, dj[3], acc[3]);
                }
            }
        }
        if (i + 1 < items) cur = nxt;
        if (u == a.nsbw - 1) {
            // end of a tile: warp partials -> shared, one barrier, fixed-order sum over warps
            const int64_t n0 = (int64_t)(blockIdx.x + (i / a.nsbw) * gridDim.x) * 16;
            float *rw = red + warp * 16 * MT;
#pragma unroll
            for (int mm = 0; mm < MT; mm++) {
                if (mm == 2 * t) {
                    rw[g * MT + mm] = acc[0] * inv[mm];
                    rw[(g + 8) * MT + mm] = acc[2] * inv[mm];
                }
                if (mm == 2 * t + 1) {
                    rw[g * MT + mm] = acc[1] * inv[mm];
                    rw[(g + 8) * MT + mm] = acc[3] * inv[mm];
                }
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            __syncthreads();
            for (int e = threadIdx.x; e < 16 * MT; e += blockDim.x) {
                const int rr = e / MT, m = e % MT;
                const int64_t n = n0 + rr;
                if (n < a.N && m < a.M) {
                    float sum = 0.0f;
                    for (int w = 0; w < BW; w++) sum += red[w * 16 * MT + e];
                    a.y[(int64_t)m * a.N + n] = sum;
                }
            }
            __syncthreads();
        }
    }
}

// ------------------------------------------------------------------ GPTQ
// GPTQ ([BPA] "Real layouts compared"): qweight int32 [K/8][N] (word (kb, n)
// holds k = 8kb .. 8kb+7 of column n, nibble i = k % 8), scales f16 [K/G][N],
// qzeros int32 [K/G][N/8] holding z - 1; w = s * (q - z).  Here G = 128 and no
// act-order permutation.  Per 32-k super-chunk s, lane (g, t) loads word
// kb = 4s + t of rows g and g+8 (8 codes: k = 32s + 8t + i).  Two MMAs take
// them: X holds codes (0, 4 | 1, 5) and Y codes (2, 6 | 3, 7) of every word,
// so each nibble pair is one LOP3 away; x is staged in the same order.  Per
// 128-k group the lane adds s * (D - z * S), S the group's x sum.
template <typename XT, int MT>
__device__ void stage_x_gptq(const XT *__restrict__ x, int64_t K, int M, int gr0, int ngr, int lane, uint2 *xh,
                             uint2 *xl, float *S, float (&inv)[MT]) {
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; m++) amax[m] = 0.0f;
    const int nq = ngr * 32;                       // 4-value groups per column
#pragma unroll 4
    for (int i = lane; i < nq; i += 32) {
#pragma unroll
        for (int m = 0; m < MT; m++)
            if (m < M) {
                const float4 v = x4(x + (int64_t)m * K + (int64_t)gr0 * 128 + 4 * i);
                amax[m] = fmaxf(amax[m], fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
    }
    float scale[MT];
#pragma unroll
    for (int m = 0; m < MT; m++) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) amax[m] = fmaxf(amax[m], __shfl_xor_sync(0xffffffffu, amax[m], off));
        scale[m] = 1.0f;
        inv[m] = 1.0f;
        if (amax[m] > 0.0f && amax[m] < INFINITY) {
            int ex = (int)((__float_as_uint(amax[m]) >> 23) & 255u) - 127;
            ex = ex < -100 ? -100 : (ex > 100 ? 100 : ex);
            scale[m] = __uint_as_float((uint32_t)(127 + 12 - ex) << 23);
            inv[m] = __uint_as_float((uint32_t)(127 - 12 + ex) << 23);
        }
    }
    // entry e = ((sc*2 + which)*MT + m)*4 + t holds x[32sc + 8t + 2*which + {0, 4 | 1, 5}]
    const int entries = ngr * 4 * 2 * MT * 4;
#pragma unroll 2
    for (int e = lane; e < entries; e += 32) {
        const int t = e & 3, m = (e >> 2) % MT, which = (e / (4 * MT)) & 1, sc = e / (8 * MT);
        uint2 hi = make_uint2(0u, 0u), lo = make_uint2(0u, 0u);
        if (m < M) {
            float cs = 1.0f;
#pragma unroll
            for (int mm = 0; mm < MT; mm++)
                if (mm == m) cs = scale[mm];
            const XT *p = x + (int64_t)m * K + (int64_t)gr0 * 128 + 32 * sc + 8 * t;
            const float4 va = x4(p), vb = x4(p + 4);    // k + 0..3, k + 4..7
            const float v0 = (which ? va.z : va.x) * cs, v1 = (which ? va.w : va.y) * cs;
            const float v4 = (which ? vb.z : vb.x) * cs, v5 = (which ? vb.w : vb.y) * cs;
            const __half2 h04 = __floats2half2_rn(v0, v4), h15 = __floats2half2_rn(v1, v5);
            const float2 r04 = __half22float2(h04), r15 = __half22float2(h15);
            const __half2 l04 = __floats2half2_rn(v0 - r04.x, v4 - r04.y);
            const __half2 l15 = __floats2half2_rn(v1 - r15.x, v5 - r15.y);
            hi = make_uint2(*reinterpret_cast<const uint32_t *>(&h04), *reinterpret_cast<const uint32_t *>(&h15));
            lo = make_uint2(*reinterpret_cast<const uint32_t *>(&l04), *reinterpret_cast<const uint32_t *>(&l15));
        }
        xh[e] = hi;
        xl[e] = lo;
    }
    __syncwarp();
    // group sums (gr*MT + m) of the staged values
    const int nsum = ngr * MT;
    for (int e = lane; e < nsum; e += 32) {
        const int m = e % MT, gr = e / MT;
        float sacc = 0.0f;
        for (int q = 0; q < 8; q++)       // 4 super-chunks x {X, Y}
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const int idx = ((gr * 8 + q) * MT + m) * 4 + t;
                const uint2 vh = xh[idx], vl = xl[idx];
                const float2 a0 = __half22float2(*reinterpret_cast<const __half2 *>(&vh.x));
                const float2 a1 = __half22float2(*reinterpret_cast<const __half2 *>(&vh.y));
                const float2 b0 = __half22float2(*reinterpret_cast<const __half2 *>(&vl.x));
                const float2 b1 = __half22float2(*reinterpret_cast<const __half2 *>(&vl.y));
                sacc += ((a0.x + b0.x) + (a0.y + b0.y)) + ((a1.x + b1.x) + (a1.y + b1.y));
            }
        S[e] = sacc;
    }
    __syncwarp();
}

struct GptqArgs {
    const uint32_t *w;      // qweight [K/8][N]
    const uint16_t *s;      // scales [K/128][N] (f16 bits)
    const uint32_t *z;      // qzeros [K/128][N/8]
    const void *x;
    float *y;
    int64_t N, K;
    int M;
    int ngw;                // groups per warp
};

// One 128-k group of rows g and g+8 for lane t: the four code words of each
// row (super-chunks 0..3, word kb = 4*sc + t), its scale and zero word.
struct GG {
    uint32_t c0[4], c1[4];
    uint32_t s01;           // scales of rows g (low half) and g+8 (high half)
    uint32_t z0, z1;        // qzeros words holding rows g and g+8
};

__device__ __forceinline__ void load_gg(const GptqArgs &a, int64_t ra, int64_t rb, int64_t gr, int t, GG &q) {
    const int64_t kb0 = gr * 16;                   // 128 k = 16 words along K
#pragma unroll
    for (int sc = 0; sc < 4; sc++) {
        q.c0[sc] = __ldg(a.w + (kb0 + 4 * sc + t) * a.N + ra);
        q.c1[sc] = __ldg(a.w + (kb0 + 4 * sc + t) * a.N + rb);
    }
    q.s01 = (uint32_t)__ldg(a.s + gr * a.N + ra) | ((uint32_t)__ldg(a.s + gr * a.N + rb) << 16);
    q.z0 = __ldg(a.z + gr * (a.N >> 3) + (ra >> 3));
    q.z1 = __ldg(a.z + gr * (a.N >> 3) + (rb >> 3));
}

template <typename XT, int MT>
__global__ void __launch_bounds__(BW * 32, 2) gemv_mma_gptq(const __grid_constant__ GptqArgs a) {
    extern __shared__ __align__(16) uint8_t blk_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int ngroups = (int)(a.K >> 7);
    const int gr0 = min(ngroups, warp * a.ngw), gr1 = min(ngroups, (warp + 1) * a.ngw), ngr = gr1 - gr0;
    const size_t xw = (size_t)a.ngw * 8 * MT * 4;            // entries per warp
    uint2 *xh = reinterpret_cast<uint2 *>(blk_smem) + (size_t)warp * 2 * xw;
    uint2 *xl = xh + xw;
    float *S = reinterpret_cast<float *>(reinterpret_cast<uint2 *>(blk_smem) + (size_t)BW * 2 * xw) +
               (size_t)warp * a.ngw * MT;
    float *red = reinterpret_cast<float *>(reinterpret_cast<uint2 *>(blk_smem) + (size_t)BW * 2 * xw) +
                 (size_t)BW * a.ngw * MT;
    const int ntiles = (int)((a.N + 15) / 16);
    const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int items = my_tiles * a.ngw;

    auto load_item = [&](int i, GG &q) {
        const int u = i % a.ngw;
        if (u >= ngr) return;
        const int64_t n0 = (int64_t)(blockIdx.x + (i / a.ngw) * gridDim.x) * 16;
        // rows past N read row N - 8 + (g & 7) (N % 8 == 0): valid memory, never stored
        const int64_t ra = n0 + g < a.N ? n0 + g : a.N - 8 + g, rb = n0 + g + 8 < a.N ? n0 + g + 8 : a.N - 8 + g;
        load_gg(a, ra, rb, gr0 + u, t, q);
    };
    // two groups in flight ahead of the one being computed (register ring,
    // rotated by copies so no register array is indexed dynamically)
    GG cur, n1, n2;
    if (items > 0) load_item(0, cur);
    if (items > 1) load_item(1, n1);

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float inv[MT];
    if (ngr > 0) stage_x_gptq<XT, MT>((const XT *)a.x, a.K, a.M, gr0, ngr, lane, xh, xl, S, inv);
    else {
#pragma unroll
        for (int m = 0; m < MT; m++) inv[m] = 1.0f;
    }
    const int mcol = g < MT ? g : 0;
    const int c2a = 2 * t < MT ? 2 * t : 0, c2b = 2 * t + 1 < MT ? 2 * t + 1 : 0;

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < items; i++) {
        if (i + 2 < items) load_item(i + 2, n2);
        const int u = i % a.ngw;
        if (u < ngr) {
            const uint2 *xhu = xh + (size_t)u * 8 * MT * 4 + mcol * 4 + t;
            const uint2 *xlu = xl + (size_t)u * 8 * MT * 4 + mcol * 4 + t;
            float dj[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int sc = 0; sc < 4; sc++) {
                const uint32_t w0 = cur.c0[sc], w1 = cur.c1[sc];
#pragma unroll
                for (int which = 0; which < 2; which++) {
                    const int sh = 8 * which;          // X: nibbles (0,4 | 1,5); Y: (2,6 | 3,7)
                    const uint32_t a0 = codes_f16x2<0>(w0 >> sh), a2 = codes_f16x2<0>(w0 >> (sh + 4));
                    const uint32_t a1 = codes_f16x2<0>(w1 >> sh), a3 = codes_f16x2<0>(w1 >> (sh + 4));
                    const int c = sc * 2 + which;
                    const uint2 bh = xhu[(size_t)c * MT * 4], bl = xlu[(size_t)c * MT * 4];
                    mma16816(dj, a0, a1, a2, a3, bh.x, bh.y);
                    mma16816(dj, a0, a1, a2, a3, bl.x, bl.y);
                }
            }
            const float sg = half_bits_f32(cur.s01), sg8 = half_bits_f32(cur.s01 >> 16);
            const float zg = (float)(((cur.z0 >> (4 * g)) & 15u) + 1u);
            const float zg8 = (float)(((cur.z1 >> (4 * g)) & 15u) + 1u);
            const float Sa = S[u * MT + c2a], Sb = S[u * MT + c2b];
            acc[0] = fmaf(sg, fmaf(-zg, Sa, dj[0]), acc[0]);
            acc[1] = fmaf(sg, fmaf(-zg, Sb, dj[1]), acc[1]);
            acc[2] = fmaf(sg8, fmaf(-zg8, Sa, dj[2]), acc[2]);
            acc[3] = fmaf(sg8, fmaf(-zg8, Sb, dj[3]), acc[3]);
        }
        cur = n1;
        n1 = n2;
        if (u == a.ngw - 1) {
            const int64_t n0 = (int64_t)(blockIdx.x + (i / a.ngw) * gridDim.x) * 16;
            float *rw = red + warp * 16 * MT;
#pragma unroll
            for (int mm = 0; mm < MT; mm++) {
                if (mm == 2 * t) {
                    rw[g * MT + mm] = acc[0] * inv[mm];
                    rw[(g + 8) * MT + mm] = acc[2] * inv[mm];
                }
                if (mm == 2 * t + 1) {
                    rw[g * MT + mm] = acc[1] * inv[mm];
                    rw[(g + 8) * MT + mm] = acc[3] * inv[mm];
                }
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            __syncthreads();
            for (int e = threadIdx.x; e < 16 * MT; e += blockDim.x) {
                const int rr = e / MT, m = e % MT;
                const int64_t n = n0 + rr;
                if (n < a.N && m < a.M) {
                    float sum = 0.0f;
                    for (int w = 0; w < BW; w++) sum += red[w * 16 * MT + e];
                    a.y[(int64_t)m * a.N + n] = sum;
                }
            }
            __syncthreads();
        }
    }
}

size_t gptq_smem_bytes(int64_t K, int mt) {
    const int ng = (int)(K >> 7), ngw = (ng + BW - 1) / BW;
    return (size_t)BW * 2 * ngw * 8 * mt * 4 * sizeof(uint2) + (size_t)BW * ngw * mt * sizeof(float) +
           (size_t)BW * 16 * mt * sizeof(float);
}

template <typename XT, int MT>
cudaError_t run_gptq(const GptqArgs &a, cudaStream_t s) {
    auto kern = gemv_mma_gptq<XT, MT>;
    const size_t smem = gptq_smem_bytes(a.K, MT);
    static bool attr_set[64] = {};
    static int bps[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BLK_SMEM_MAX);
        if (e != cudaSuccess) return e;
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, BW * 32, smem) != cudaSuccess || b < 1) b = 1;
        bps[dev & 63] = b;
        attr_set[dev & 63] = true;
    }
    const int ntiles = (int)((a.N + 15) / 16);
    int grid = bps[dev & 63] * sm_count();
    if (grid > ntiles) grid = ntiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(BW * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

size_t blk_smem_bytes(int64_t K, int mt) {
    const int nsb = (int)(K >> 8), nsbw = (nsb + BW - 1) / BW;
    return (size_t)BW * 2 * nsbw * 16 * mt * 4 * sizeof(uint2) + (size_t)BW * nsbw * 8 * mt * sizeof(float) +
           (size_t)BW * 16 * mt * sizeof(float);
}

int blk_mt(int64_t M) { return M == 1 ? 1 : (M == 2 ? 2 : (M <= 4 ? 4 : 8)); }

template <typename XT, int MT, int FMT>
cudaError_t run_blk(const BlkArgs &a, cudaStream_t s) {
    auto kern = gemv_mma_blk<XT, MT, FMT>;
    const size_t smem = blk_smem_bytes(a.K, MT);
    static bool attr_set[64] = {};
    static int bps[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BLK_SMEM_MAX);
        if (e != cudaSuccess) return e;
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, BW * 32, smem) != cudaSuccess || b < 1) b = 1;
        bps[dev & 63] = b;
        attr_set[dev & 63] = true;
    }
    const int ntiles = (int)((a.N + 15) / 16);
    int grid = bps[dev & 63] * sm_count();
    if (grid > ntiles) grid = ntiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(BW * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

bool gemv_blk_eligible(const Tensor &t, int64_t M) {
    return (t.fmt == Q4_Q4K || t.fmt == Q4_Q40) && M >= 1 && M <= 8 && t.K % 256 == 0 && t.K <= (1LL << 30) &&
           blk_smem_bytes(t.K, blk_mt(M)) <= BLK_SMEM_MAX && (((uintptr_t)t.w) & 15) == 0;
}

bool gemv_gptq_eligible(const Tensor &t, int64_t M) {
    return t.fmt == Q4_GPTQ && t.g_idx == nullptr && t.group == 128 && M >= 1 && M <= 8 && t.K % 128 == 0 &&
           t.N % 8 == 0 && t.K <= (1LL << 30) && gptq_smem_bytes(t.K, blk_mt(M)) <= BLK_SMEM_MAX;
}

cudaError_t launch_gemv_gptq(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    GptqArgs a;
    a.w = reinterpret_cast<const uint32_t *>(t.w);
    a.s = reinterpret_cast<const uint16_t *>(t.scales);
    a.z = reinterpret_cast<const uint32_t *>(t.zeros);
    a.x = x;
    a.y = y;
    a.N = t.N;
    a.K = t.K;
    a.M = (int)M;
    a.ngw = (int)(((t.K >> 7) + BW - 1) / BW);
    const int mt = blk_mt(M);
    if (xd == Q4_DT_BF16) {
        if (mt == 1) return run_gptq<__nv_bfloat16, 1>(a, s);
        if (mt == 2) return run_gptq<__nv_bfloat16, 2>(a, s);
        if (mt == 4) return run_gptq<__nv_bfloat16, 4>(a, s);
        return run_gptq<__nv_bfloat16, 8>(a, s);
    }
    if (mt == 1) return run_gptq<float, 1>(a, s);
    if (mt == 2) return run_gptq<float, 2>(a, s);
    if (mt == 4) return run_gptq<float, 4>(a, s);
    return run_gptq<float, 8>(a, s);
}

namespace {
template <int FMT>
cudaError_t launch_blk_fmt(const BlkArgs &a, q4_dtype xd, cudaStream_t s) {
    const int mt = blk_mt(a.M);
    if (xd == Q4_DT_BF16) {
        if (mt == 1) return run_blk<__nv_bfloat16, 1, FMT>(a, s);
        if (mt == 2) return run_blk<__nv_bfloat16, 2, FMT>(a, s);
        if (mt == 4) return run_blk<__nv_bfloat16, 4, FMT>(a, s);
        return run_blk<__nv_bfloat16, 8, FMT>(a, s);
    }
    if (mt == 1) return run_blk<float, 1, FMT>(a, s);
    if (mt == 2) return run_blk<float, 2, FMT>(a, s);
    if (mt == 4) return run_blk<float, 4, FMT>(a, s);
    return run_blk<float, 8, FMT>(a, s);
}
}  // namespace

cudaError_t launch_gemv_blk(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    BlkArgs a;
    a.w = t.w;
    a.x = x;
    a.y = y;
    a.N = t.N;
    a.K = t.K;
    a.M = (int)M;
    a.nsbw = (int)(((t.K >> 8) + BW - 1) / BW);
    return t.fmt == Q4_Q4K ? launch_blk_fmt<Q4_Q4K>(a, xd, s) : launch_blk_fmt<Q4_Q40>(a, xd, s);
}

}  // namespace q4
