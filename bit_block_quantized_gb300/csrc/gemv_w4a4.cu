// gemv_w4a4.cu -- the W4A4 contraction of [MUS7] 7.4.3 on sm_103a (CUDA cores).
//
// Each CTA quantizes its activation rows (<= 8) to NVFP4 per 16 with the
// tensor scale G = 1/input_scale_inv: E4M3 scale = nearest-even of
// (amax/6)/G (saturating at 448), codes = nearest-even E2M1 of x/(scale*G),
// kept in shared memory as signed halves (q1, int8) plus the scale in units of
// 2^-9 (q9).  Rows: one LANE per output row ("lane = row"), 32 bytes (64
// weights, four groups) per step, so the per-group i64 products
// T_g = q9w * q9x * sum q1w * q1x and the ordered per-group epilogue
//   c = fma(fma(fma(float(T_g), 2^-20, 0), scale2, 0), G, 0); total = fma(1, c, total)
// stay in the lane with no shuffles; the activation reads are warp broadcasts.
// The epilogue's order makes each row one sequential chain, so rows are
// spread thin (two warps per CTA, many CTAs) and every lane keeps four steps
// (128 payload bytes) of its row in flight.
#include <algorithm>

#include "q4_internal.cuh"

namespace q4 {
namespace {

constexpr int W4_WARPS = 2;
constexpr int W4_AHEAD = 4;                    // 64-k steps loaded ahead per lane
constexpr int W4_THREADS = W4_WARPS * 32;
constexpr uint32_t W4_LUT_LO = 0x03020100u, W4_LUT_HI = 0x0C080604u;

__device__ __forceinline__ uint32_t w4_prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t w4_e4m3_round(float a) {      // nearest-even, saturating at 448
    if (a >= 448.0f) return 0x7eu;
    if (a < 0x1p-6f) return (uint32_t)rintf(a * 512.0f);
    const int e = (int)((__float_as_uint(a) >> 23) & 255u) - 127;
    const float m = rintf(__fmul_rn(a, __uint_as_float((uint32_t)(127 - e + 3) << 23)));
    uint32_t mi = (uint32_t)m, ee = (uint32_t)(e + 7);
    if (mi == 16u) { mi = 8u; ee += 1u; }
    const uint32_t b = (ee << 3) | (mi - 8u);
    return b > 0x7eu ? 0x7eu : b;
}
__device__ __forceinline__ float w4_e4m3_value(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, f = b & 7u;
    const float mag = e == 0 ? (float)f * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (f << 20));
    return (b & 0x80u) ? -mag : mag;
}
__device__ __forceinline__ int32_t w4_q9(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, f = b & 7u;
    const int32_t mag = e == 0 ? (int32_t)f : (int32_t)((8u + f) << (e - 1u));
    return (b & 0x80u) ? -mag : mag;
}
// Nearest-even E2M1 of r as signed halves (q1): {0,1,2,3,4,6,8,12}, sign of r.
__device__ __forceinline__ int w4_q1_round(float r) {
    const float a = fabsf(r);
    int v;
    if (a <= 0.25f) v = 0;
    else if (a < 0.75f) v = 1;
    else if (a <= 1.25f) v = 2;
    else if (a < 1.75f) v = 3;
    else if (a <= 2.5f) v = 4;
    else if (a < 3.5f) v = 6;
    else if (a <= 5.0f) v = 8;
    else v = 12;
    return signbit(r) ? -v : v;
}

// Shared layout: q9x [MT][K/16] i32 | q1x [MT][K] i8.
__host__ __device__ inline int64_t w4_q1_off(int mt, int64_t K) { return ((int64_t)mt * (K / 16) * 4 + 15) / 16 * 16; }
__host__ __device__ inline int64_t w4_smem_bytes(int mt, int64_t K) { return w4_q1_off(mt, K) + (int64_t)mt * K; }

template <int MT, typename XT>
__global__ void __launch_bounds__(W4_THREADS)
gemv_w4a4_kernel(const uint8_t *__restrict__ W, const uint8_t *__restrict__ S, float scale2, float G,
                 const XT *__restrict__ x, float *__restrict__ y, int mrows, int64_t N, int64_t K) {
    extern __shared__ __align__(16) unsigned char smem[];
    int32_t *q9x = reinterpret_cast<int32_t *>(smem);
    int8_t *q1x = reinterpret_cast<int8_t *>(smem + w4_q1_off(MT, K));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t ng = K / 16;

    // ---- activation quantization: one thread per 16-value group
    for (int64_t it = threadIdx.x; it < (int64_t)mrows * ng; it += W4_THREADS) {
        const int64_t m = it / ng, g = it % ng;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; i++) v[i] = x_to_f32(x[m * K + g * 16 + i]);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(v[i]));
        const uint32_t sb = w4_e4m3_round(__fdiv_rn(__fdiv_rn(amax, 6.0f), G));
        const float denom = __fmul_rn(w4_e4m3_value(sb), G);
        uint32_t pk[4] = {0u, 0u, 0u, 0u};
        if (denom > 0.0f) {
#pragma unroll
            for (int i = 0; i < 16; i++)
                pk[i >> 2] |= ((uint32_t)w4_q1_round(__fdiv_rn(v[i], denom)) & 0xffu) << (8 * (i & 3));
        }
        *reinterpret_cast<uint4 *>(q1x + m * K + g * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        q9x[m * ng + g] = w4_q9(sb);
    }
    __syncthreads();

    // ---- rows: one lane per output row, 64 weights (four groups) per step
    const int64_t total_lanes = (int64_t)gridDim.x * W4_THREADS;
    for (int64_t n = (int64_t)blockIdx.x * W4_THREADS + warp * 32 + lane; n - lane < N; n += total_lanes) {
        const bool live = n < N;                       // lanes past N follow the warp with no loads or stores
        const uint8_t *wrow = W + (live ? n : 0) * (K / 2);
        const uint8_t *srow = S + (live ? n : 0) * ng;
        float total[MT];
#pragma unroll
        for (int m = 0; m < MT; m++) total[m] = 0.0f;
        for (int64_t kb = 0; kb < K; kb += 64 * W4_AHEAD) {      // K % 64 == 0
            uint4 pa[W4_AHEAD], pb[W4_AHEAD];
            uint32_t psw[W4_AHEAD];
#pragma unroll
            for (int u = 0; u < W4_AHEAD; u++) {
                const int64_t k0 = kb + 64 * u;
                pa[u] = pb[u] = make_uint4(0u, 0u, 0u, 0u);
                psw[u] = 0u;
                if (live && k0 < K) {
                    pa[u] = ldg_stream16(wrow + k0 / 2);
                    pb[u] = ldg_stream16(wrow + k0 / 2 + 16);
                    psw[u] = ldg_stream4(srow + k0 / 16);
                }
            }
#pragma unroll
            for (int u = 0; u < W4_AHEAD; u++) {
            const int64_t k0 = kb + 64 * u;
            if (k0 >= K) break;                        // warp-uniform
            const uint4 a = pa[u], b = pb[u];
            const uint32_t sw = psw[u];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int m = 0; m < MT; m++) {
                if (m >= mrows) break;
                const uint4 *q = reinterpret_cast<const uint4 *>(q1x + m * K + k0);
#pragma unroll
                for (int g = 0; g < 4; g++) {
                    const uint4 qa = q[g];
                    const uint32_t qw[4] = {qa.x, qa.y, qa.z, qa.w};
                    int pos = 0, neg = 0;
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const uint32_t x0 = w[2 * g + h], x1 = x0 ^ 0x88888888u;
                        pos = __dp4a((int)w4_prmt(W4_LUT_LO, W4_LUT_HI, x0), (int)qw[2 * h], pos);
                        neg = __dp4a((int)w4_prmt(W4_LUT_LO, W4_LUT_HI, x1), (int)qw[2 * h], neg);
                        pos = __dp4a((int)w4_prmt(W4_LUT_LO, W4_LUT_HI, x0 >> 16), (int)qw[2 * h + 1], pos);
                        neg = __dp4a((int)w4_prmt(W4_LUT_LO, W4_LUT_HI, x1 >> 16), (int)qw[2 * h + 1], neg);
                    }
                    const int64_t T = (int64_t)(pos - neg) * w4_q9((sw >> (8 * g)) & 0xffu) *
                                      (int64_t)q9x[m * ng + k0 / 16 + g];
                    float c = __fmaf_rn(__ll2float_rn((long long)T), 0x1p-20f, 0.0f);
                    c = __fmaf_rn(c, scale2, 0.0f);
                    c = __fmaf_rn(c, G, 0.0f);
                    total[m] = __fmaf_rn(1.0f, c, total[m]);
                }
            }
            }
        }
        if (live) {
#pragma unroll
            for (int m = 0; m < MT; m++)
                if (m < mrows) y[(int64_t)m * N + n] = __half2float(__float2half_rn(total[m]));
        }
    }
}

template <int MT, typename XT>
cudaError_t w4_launch_mt(const Tensor &t, float G, const XT *x, float *y, int mrows, cudaStream_t s) {
    const int64_t smem = w4_smem_bytes(MT, t.K);
    auto kern = gemv_w4a4_kernel<MT, XT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, W4_THREADS, (size_t)smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t want = (t.N + W4_THREADS - 1) / W4_THREADS;
    const int64_t grid = std::min<int64_t>(want, (int64_t)per_sm * sm_count());
    kern<<<(unsigned)grid, W4_THREADS, (size_t)smem, s>>>(t.w, t.scales, t.scale2, G, x, y, mrows, t.N, t.K);
    return cudaGetLastError();
}

template <typename XT>
cudaError_t w4_launch_chunk(const Tensor &t, float G, const XT *x, float *y, int mrows, cudaStream_t s) {
    if (mrows > 4) return w4_launch_mt<8, XT>(t, G, x, y, mrows, s);
    if (mrows > 2) return w4_launch_mt<4, XT>(t, G, x, y, mrows, s);
    if (mrows > 1) return w4_launch_mt<2, XT>(t, G, x, y, mrows, s);
    return w4_launch_mt<1, XT>(t, G, x, y, mrows, s);
}

}  // namespace

int gemv_w4a4_chunk(int64_t M, int64_t K) {
    const int64_t limit = 200 * 1024;
    for (int rows = (int)std::min<int64_t>(M, 8); rows >= 1; rows--) {
        const int mt = rows > 4 ? 8 : rows > 2 ? 4 : rows;
        if (w4_smem_bytes(mt, K) <= limit) return rows;
    }
    return 0;
}

// input_scale_inv: finite and > 0 (checked by the caller); K % 64 == 0.
cudaError_t launch_gemv_w4a4(const Tensor &t, float input_scale_inv, const void *x, q4_dtype xd, float *y, int64_t M,
                             cudaStream_t s) {
    const float G = 1.0f / input_scale_inv;         // host IEEE division, as the definition
    const int chunk = gemv_w4a4_chunk(M, t.K);
    if (chunk == 0) return cudaErrorInvalidValue;
    for (int64_t m0 = 0; m0 < M; m0 += chunk) {
        const int mrows = (int)std::min<int64_t>(chunk, M - m0);
        cudaError_t e;
        if (xd == Q4_DT_BF16)
            e = w4_launch_chunk<__nv_bfloat16>(t, G, reinterpret_cast<const __nv_bfloat16 *>(x) + m0 * t.K,
                                               y + m0 * t.N, mrows, s);
        else
            e = w4_launch_chunk<float>(t, G, reinterpret_cast<const float *>(x) + m0 * t.K, y + m0 * t.N, mrows, s);
        if (e != cudaSuccess) return e;
    }
    note_gemv_path("gemv_w4a4");
    return cudaSuccess;
}

}  // namespace q4
