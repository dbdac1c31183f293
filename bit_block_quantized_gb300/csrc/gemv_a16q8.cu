// gemv_a16q8.cu -- the integer-exact weight-only NVFP4 contraction of the
// Muser book, chapter 7, section 7.4.2 ([MUS7] 7.4.2), on sm_103a.
//
// Activations are quantized per 256-value block to signed 8-bit codes (the
// signed first maximum m, iscale = -127/m, half-to-even, capped at 127, block
// scale 1/iscale).  Per output row and block the contraction
//     T = sum_g q9(scale[n][g]) * sum_{k in g} q1(code[n][k]) * q8[k]
// is an exact integer (q1 = E2M1 in halves, q9 = E4M3FN in units of 2^-9), so
// any summation order gives the same T.  Only the epilogue rounds, in four
// pinned f32 steps taken in block order:
//     c = fma(float(T), 2^-10, 0); c = fma(c, act_scale, 0);
//     c = fma(c, scale2, 0);       total = fma(1, c, total)
// and the output is total rounded to binary16 (stored widened to f32).
//
// Design (CUDA cores; HBM-bound like every batch-1 GEMV here):
//   * Each CTA first quantizes the whole activation chunk (MT rows x K) into
//     shared memory, one warp per 256-value block; no scratch memory and no
//     second launch.  x is tiny next to W and is read from L2 by every CTA.
//   * Warps then take output rows.  A lane streams 16 payload bytes (32
//     weights, two 16-value groups) per 1024-k chunk with 128-bit no-allocate
//     loads, four chunks in flight.
//   * Decode: a PRMT with the nibble codes as selectors picks q1 magnitudes
//     {0,1,2,3,4,6,8,12} from an 8-byte register table.  PRMT's sign-replicate
//     bit (selector bit 3 = the E2M1 sign bit) turns the negative codes into
//     0x00, and the same PRMT on code^8 yields the magnitudes of exactly the
//     negative codes, so dot = dp4a(pos, q8) - dp4a(neg, q8) with no per-byte
//     negation.  Fourteen instructions per eight weights.
//   * The per-group 32-bit dots times q9 (a 256-entry shared table) add in
//     64-bit; the eight lanes of a block reduce by shuffles, and the block
//     contributions enter the row total in block order.
#include <algorithm>

#include "q4_internal.cuh"

namespace q4 {
namespace {

constexpr int A8_WARPS = 8;
constexpr int A8_THREADS = A8_WARPS * 32;
constexpr int A8_INFLIGHT = 4;   // 1024-k chunks whose payload a lane loads before using any

// q1 magnitudes of E2M1 codes 0..7, one per byte: {0,1,2,3} and {4,6,8,12}.
constexpr uint32_t Q1_LUT_LO = 0x03020100u;
constexpr uint32_t Q1_LUT_HI = 0x0C080604u;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Signed dot of four E2M1 codes (selector nibbles sel[15:0], code i in bits
// 4i..4i+3) with four int8 activation codes, as q1 * q8 summed, added to acc.
__device__ __forceinline__ int dot4_e2m1_q8(uint32_t sel, uint32_t q8x4, int acc) {
    const uint32_t pos = prmt(Q1_LUT_LO, Q1_LUT_HI, sel);            // 0 for negative codes
    const uint32_t neg = prmt(Q1_LUT_LO, Q1_LUT_HI, sel ^ 0x8888u);  // 0 for non-negative codes
    acc = __dp4a((int)pos, (int)q8x4, acc);
    return acc - __dp4a((int)neg, (int)q8x4, 0);
}

// Exact dot of one 16-value group: payload words w0 (k .. k+7) and w1
// (k+8 .. k+15), activation codes qa = {k..k+3, k+4..k+7, k+8..k+11, k+12..k+15}.
__device__ __forceinline__ int group_dot(uint32_t w0, uint32_t w1, uint4 qa) {
    int acc = dot4_e2m1_q8(w0 & 0xffffu, qa.x, 0);
    acc = dot4_e2m1_q8(w0 >> 16, qa.y, acc);
    acc = dot4_e2m1_q8(w1 & 0xffffu, qa.z, acc);
    return dot4_e2m1_q8(w1 >> 16, qa.w, acc);
}

__device__ __forceinline__ int64_t shfl_xor_i64(int64_t v, int mask) {
    return (int64_t)__shfl_xor_sync(0xffffffffu, (long long)v, mask);
}

// Shared layout: q9 table [256] i32 | act_scale [MT][K/256] f32 | q8 [MT][K] i8.
__host__ __device__ inline int64_t a8_scale_off() { return 256 * 4; }
__host__ __device__ inline int64_t a8_q8_off(int mt, int64_t K) {
    return (a8_scale_off() + (int64_t)mt * (K / 256) * 4 + 15) / 16 * 16;
}
__host__ __device__ inline int64_t a8_smem_bytes(int mt, int64_t K) { return a8_q8_off(mt, K) + (int64_t)mt * K; }

template <typename XT> struct XLoad;
template <> struct XLoad<__nv_bfloat16> {      // eight bf16 -> f32, one 16-byte load
    static __device__ __forceinline__ void get(const __nv_bfloat16 *p, float v[8]) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <> struct XLoad<float> {              // eight f32, two 16-byte loads
    static __device__ __forceinline__ void get(const float *p, float v[8]) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        const float4 b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

// One CTA: quantize x rows [0, mrows) (mrows <= MT) into shared memory, then
// grid-stride over output rows, one warp per row.
template <int MT, typename XT>
__global__ void __launch_bounds__(A8_THREADS)
gemv_a16q8_kernel(const uint8_t *__restrict__ W, const uint8_t *__restrict__ S, float scale2,
                  const XT *__restrict__ x, float *__restrict__ y, int mrows, int64_t N, int64_t K) {
    extern __shared__ __align__(16) unsigned char smem[];
    int32_t *q9 = reinterpret_cast<int32_t *>(smem);
    float *act_scale = reinterpret_cast<float *>(smem + a8_scale_off());
    int8_t *q8 = reinterpret_cast<int8_t *>(smem + a8_q8_off(MT, K));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nb = K / 256;

    {   // E4M3FN byte -> q9 = (8+f) << (e-1), or f for exponent field 0; bit 7 the sign.
        const uint32_t b = threadIdx.x, e = (b >> 3) & 15u, f = b & 7u;
        const int32_t mag = e == 0 ? (int32_t)f : (int32_t)((8u + f) << (e - 1u));
        q9[b] = (b & 0x80u) ? -mag : mag;
    }

    // ---- activation quantization, one warp per (row m, block b)
    for (int64_t item = warp; item < (int64_t)mrows * nb; item += A8_WARPS) {
        const int64_t m = item / nb, b = item % nb;
        float v[8];
        XLoad<XT>::get(x + m * K + b * 256 + lane * 8, v);
        float amax = 0.0f, val = 0.0f;
        int idx = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float a = fabsf(v[i]);
            if (a > amax) { amax = a; val = v[i]; idx = lane * 8 + i; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {   // largest magnitude, first index on ties
            const float oa = __shfl_xor_sync(0xffffffffu, amax, off);
            const float ov = __shfl_xor_sync(0xffffffffu, val, off);
            const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
            if (oa > amax || (oa == amax && oi < idx)) { amax = oa; val = ov; idx = oi; }
        }
        const float iscale = __fdiv_rn(-127.0f, val);
        const bool live = isfinite(iscale);         // zero (or vanishing) block: codes 0, scale 0
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; i++) {
            int c = live ? __float2int_rn(__fmul_rn(v[i], iscale)) : 0;
            c = c > 127 ? 127 : c;
            packed[i >> 2] |= ((uint32_t)c & 0xffu) << (8 * (i & 3));
        }
        *reinterpret_cast<uint2 *>(q8 + m * K + b * 256 + lane * 8) = make_uint2(packed[0], packed[1]);
        if (lane == 0) act_scale[m * nb + b] = live ? __fdiv_rn(1.0f, iscale) : 0.0f;
    }
    __syncthreads();

    // ---- rows
    const int64_t nchunks = (K + 1023) / 1024;
    const int64_t total_warps = (int64_t)gridDim.x * A8_WARPS;
    const int sub = lane >> 3;                      // block of the lane inside a chunk
    for (int64_t n = (int64_t)blockIdx.x * A8_WARPS + warp; n < N; n += total_warps) {
        const uint8_t *wrow = W + n * (K / 2);
        const uint8_t *srow = S + n * (K / 16);
        float total[MT];
#pragma unroll
        for (int m = 0; m < MT; m++) total[m] = 0.0f;
        for (int64_t c0 = 0; c0 < nchunks; c0 += A8_INFLIGHT) {
            uint4 wv[A8_INFLIGHT];
            uint32_t sv[A8_INFLIGHT];
#pragma unroll
            for (int u = 0; u < A8_INFLIGHT; u++) {
                const int64_t k0 = (c0 + u) * 1024 + lane * 32;
                if (k0 < K) {
                    wv[u] = ldg_stream16(wrow + k0 / 2);
                    sv[u] = ldg_stream2(srow + k0 / 16);
                } else {
                    wv[u] = make_uint4(0u, 0u, 0u, 0u);
                    sv[u] = 0u;
                }
            }
#pragma unroll
            for (int u = 0; u < A8_INFLIGHT; u++) {
                const int64_t c = c0 + u;
                if (c >= nchunks) break;                       // warp-uniform
                const int64_t k0 = c * 1024 + lane * 32;
                const bool valid = k0 < K;                     // whole 256-k blocks: 8-lane uniform
                const int64_t blk = c * 4 + sub;
                const int32_t qa = q9[sv[u] & 0xffu], qb = q9[(sv[u] >> 8) & 0xffu];
#pragma unroll
                for (int m = 0; m < MT; m++) {
                    if (m >= mrows) break;
                    int64_t T = 0;
                    float s = 0.0f;
                    if (valid) {
                        const uint4 *q = reinterpret_cast<const uint4 *>(q8 + m * K + k0);
                        const int d0 = group_dot(wv[u].x, wv[u].y, q[0]);
                        const int d1 = group_dot(wv[u].z, wv[u].w, q[1]);
                        T = (int64_t)d0 * qa + (int64_t)d1 * qb;
                        s = act_scale[m * nb + blk];
                    }
                    T += shfl_xor_i64(T, 1);
                    T += shfl_xor_i64(T, 2);
                    T += shfl_xor_i64(T, 4);
                    float cc = __fmaf_rn(__ll2float_rn((long long)T), 0x1p-10f, 0.0f);
                    cc = __fmaf_rn(cc, s, 0.0f);
                    cc = __fmaf_rn(cc, scale2, 0.0f);
#pragma unroll
                    for (int j = 0; j < 4; j++) {              // block order: c*4 + j
                        const float cj = __shfl_sync(0xffffffffu, cc, j * 8);
                        if (c * 4 + j < nb) total[m] = __fmaf_rn(1.0f, cj, total[m]);
                    }
                }
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; m++)
                if (m < mrows) y[(int64_t)m * N + n] = __half2float(__float2half_rn(total[m]));
        }
    }
}

constexpr int A8_SMEM_LIMIT = 200 * 1024;   // the budget gemv_a16q8_chunk keeps every launch within

// Per device: the shared-memory attribute is set once (to the budget) and the
// blocks per SM of the latest shared-memory size are kept, so a repeated call
// costs no driver queries.  Any grid >= 1 gives the same result (grid-stride).
template <int MT, typename XT>
cudaError_t launch_mt(const Tensor &t, const XT *x, float *y, int mrows, cudaStream_t s) {
    const int64_t smem = a8_smem_bytes(MT, t.K);
    auto kern = gemv_a16q8_kernel<MT, XT>;
    static bool attr_set[64] = {};
    static int64_t cached_smem[64] = {};
    static int cached_per_sm[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    dev &= 63;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, A8_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int per_sm = cached_per_sm[dev];
    if (cached_smem[dev] != smem || per_sm < 1) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, A8_THREADS, (size_t)smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        cached_smem[dev] = smem;
        cached_per_sm[dev] = per_sm;
    }
    const int64_t want = (t.N + A8_WARPS - 1) / A8_WARPS;
    const int64_t grid = std::min<int64_t>(want, (int64_t)per_sm * sm_count());
    kern<<<(unsigned)grid, A8_THREADS, (size_t)smem, s>>>(t.w, t.scales, t.scale2, x, y, mrows, t.N, t.K);
    return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_chunk(const Tensor &t, const XT *x, float *y, int mrows, cudaStream_t s) {
    if (mrows > 4) return launch_mt<8, XT>(t, x, y, mrows, s);
    if (mrows > 2) return launch_mt<4, XT>(t, x, y, mrows, s);
    if (mrows > 1) return launch_mt<2, XT>(t, x, y, mrows, s);
    return launch_mt<1, XT>(t, x, y, mrows, s);
}

}  // namespace

// Activation rows per launch: min(M, 8), lowered until the template that
// serves it (MT = 8, 4, 2 or 1 rows) fits the shared-memory budget; 0 if not
// even one row of quantized activations fits.
int gemv_a16q8_chunk(int64_t M, int64_t K) {
    const int64_t limit = A8_SMEM_LIMIT;
    for (int rows = (int)std::min<int64_t>(M, 8); rows >= 1; rows--) {
        const int mt = rows > 4 ? 8 : rows > 2 ? 4 : rows;
        if (a8_smem_bytes(mt, K) <= limit) return rows;
    }
    return 0;
}

bool gemv_a16q8_tc_eligible(const Tensor &t, int64_t M);
cudaError_t launch_gemv_a16q8_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);

cudaError_t launch_gemv_a16q8(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    // batch 1 and 2: the same contract with the group dots on the tensor cores (gemv_a16q8_tc.cu)
    if (gemv_a16q8_tc_eligible(t, M)) {
        const cudaError_t e = launch_gemv_a16q8_tc(t, x, xd, y, M, s);
        if (e == cudaSuccess) note_gemv_path("gemv_a16q8_tc");
        return e;
    }
    const int chunk = gemv_a16q8_chunk(M, t.K);
    if (chunk == 0) return cudaErrorInvalidValue;
    for (int64_t m0 = 0; m0 < M; m0 += chunk) {
        const int mrows = (int)std::min<int64_t>(chunk, M - m0);
        cudaError_t e;
        if (xd == Q4_DT_BF16)
            e = launch_chunk<__nv_bfloat16>(t, reinterpret_cast<const __nv_bfloat16 *>(x) + m0 * t.K, y + m0 * t.N,
                                            mrows, s);
        else
            e = launch_chunk<float>(t, reinterpret_cast<const float *>(x) + m0 * t.K, y + m0 * t.N, mrows, s);
        if (e != cudaSuccess) return e;
    }
    note_gemv_path("gemv_a16q8");
    return cudaSuccess;
}

}  // namespace q4
