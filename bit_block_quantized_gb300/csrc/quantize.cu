// quantize.cu -- NVFP4 quantization on the GPU (the write side of the format):
// scale2 = amax(W) / (448 * 6) (1 for an all-zero W); per 16-value group the
// E4M3FN scale byte = nearest-even of (amax_group / 6) / scale2, saturating at
// 448; each code = nearest-even E2M1 of w / (dec(scale) * scale2), saturating
// at 6, the sign kept (a negative value that rounds to 0 is code 8); every
// step an IEEE f32 operation ([MUS7] 7.2 for the E2M1 rounding contract).
//
// q4_quantize_q4k: the per-sub-block min/max fit of Q4_K (below), one warp
// per 256-weight super-block.
//
// Four stream-ordered steps, no allocation: the caller's scale2 word is
// zeroed, holds the running amax (non-negative f32 bit patterns order like
// unsigned integers, so atomicMax on the bits is a float max), is turned into
// scale2 by one thread, and is read by the quantize kernel.  The quantize
// kernel gives each thread one 16-value group: 64 (f32) or 32 (bf16)
// contiguous input bytes, 8 payload bytes and one scale byte out.
#include <algorithm>

#include "q4_internal.cuh"

namespace q4 {
namespace {

template <typename WT> __device__ __forceinline__ float wload(const WT *p, int64_t i);
template <> __device__ __forceinline__ float wload<float>(const float *p, int64_t i) { return p[i]; }
template <> __device__ __forceinline__ float wload<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}

// 8 consecutive weights as f32 (one or two 16-byte loads; p 16-byte aligned).
template <typename WT> __device__ __forceinline__ void load8w(const WT *p, float v[8]);
template <> __device__ __forceinline__ void load8w<float>(const float *p, float v[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <> __device__ __forceinline__ void load8w<__nv_bfloat16>(const __nv_bfloat16 *p, float v[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Largest |w| over the tensor: runs of 8 weights (16-byte loads), four runs
// in flight per thread, then the scalar tail.
template <typename WT>
__global__ void amax_kernel(const WT *__restrict__ W, int64_t n, unsigned *amax_bits) {
    float m = 0.0f;
    const int64_t runs = n / 8, stride = (int64_t)gridDim.x * blockDim.x;
    int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; r + 3 * stride < runs; r += 4 * stride) {
        float v[4][8];
#pragma unroll
        for (int u = 0; u < 4; u++) load8w<WT>(W + (r + u * stride) * 8, v[u]);
#pragma unroll
        for (int u = 0; u < 4; u++)
#pragma unroll
            for (int i = 0; i < 8; i++) m = fmaxf(m, fabsf(v[u][i]));
    }
    for (; r < runs; r += stride) {
        float v[8];
        load8w<WT>(W + r * 8, v);
#pragma unroll
        for (int i = 0; i < 8; i++) m = fmaxf(m, fabsf(v[i]));
    }
    for (int64_t i = runs * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        m = fmaxf(m, fabsf(wload(W, i)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

__global__ void scale2_kernel(float *s2) {
    const float amax = *s2;
    *s2 = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
}

// E4M3FN byte -> value (finite bytes), exact in f32.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, f = b & 7u;
    const float mag = e == 0 ? (float)f * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (f << 20));
    return (b & 0x80u) ? -mag : mag;
}

// Nearest-even E4M3FN byte of a >= 0 (finite), saturating at 448 (0x7e).
// Values of binade [2^e, 2^(e+1)) sit on a grid of 2^(e-3) for e >= -6, and
// below 2^-6 on the subnormal grid 2^-9; the scaled quotient is exact, so
// rintf (ties to even) makes the one rounding, and a carry into the next
// binade lands on its first grid point.
__device__ __forceinline__ uint32_t e4m3_round(float a) {
    if (a >= 448.0f) return 0x7eu;
    if (a < 0x1p-6f) {
        const uint32_t q = (uint32_t)rintf(a * 512.0f);           // exact scaling; 8 = 2^-6 rolls into 0x08
        return q;
    }
    const int e = (int)((__float_as_uint(a) >> 23) & 255u) - 127;   // a in [2^e, 2^(e+1)), e in -6..8
    const float m = rintf(__fmul_rn(a, __uint_as_float((uint32_t)(127 - e + 3) << 23)));   // in [8, 16]
    uint32_t mi = (uint32_t)m, ee = (uint32_t)(e + 7);
    if (mi == 16u) { mi = 8u; ee += 1u; }
    const uint32_t b = (ee << 3) | (mi - 8u);
    return b > 0x7eu ? 0x7eu : b;
}

// Nearest-even E2M1 code of r (ModelOpt's midpoints), saturating at 6, sign kept.
__device__ __forceinline__ uint32_t e2m1_round(float r) {
    const float a = fabsf(r);
    uint32_t c;
    if (a <= 0.25f) c = 0;          // 0.25 -> 0 (even)
    else if (a < 0.75f) c = 1;      // 0.5
    else if (a <= 1.25f) c = 2;     // 0.75, 1.25 -> 1 (even)
    else if (a < 1.75f) c = 3;      // 1.5
    else if (a <= 2.5f) c = 4;      // 1.75, 2.5 -> 2
    else if (a < 3.5f) c = 5;       // 3
    else if (a <= 5.0f) c = 6;      // 3.5, 5 -> 4
    else c = 7;                     // 6 and above
    return c | (signbit(r) ? 8u : 0u);
}

template <typename WT>
__global__ void quantize_nvfp4_kernel(const WT *__restrict__ W, int64_t N, int64_t K, const float *s2p, float s2v,
                                      uint8_t *__restrict__ payload, uint8_t *__restrict__ scales) {
    const float scale2 = s2p ? *s2p : s2v;          // the tensor scale: computed on the device, or given
    const int64_t groups = N * (K / 16);
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += (int64_t)gridDim.x * blockDim.x) {
        float w[16];
        load8w<WT>(W + g * 16, w);
        load8w<WT>(W + g * 16 + 8, w + 8);
        float amax_g = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i++) amax_g = fmaxf(amax_g, fabsf(w[i]));
        const float sv = __fdiv_rn(__fdiv_rn(amax_g, 6.0f), scale2);
        const uint32_t sb = e4m3_round(sv);
        const float denom = __fmul_rn(e4m3_value(sb), scale2);
        uint32_t lo = 0u, hi = 0u;
        if (denom > 0.0f) {
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const uint32_t c = e2m1_round(__fdiv_rn(w[i], denom));
                if (i < 8) lo |= c << (4 * i);
                else hi |= c << (4 * (i - 8));
            }
        }
        *reinterpret_cast<uint2 *>(payload + g * 8) = make_uint2(lo, hi);
        scales[g] = (uint8_t)sb;
    }
}

template <typename WT>
cudaError_t launch_quantize_t(const WT *W, int64_t N, int64_t K, uint8_t *payload, uint8_t *scales, float *scale2,
                              cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(scale2, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    const int64_t n = N * K;
    const int64_t grid_a = std::min<int64_t>((n + 255) / 256, (int64_t)sms * 8);
    amax_kernel<WT><<<(unsigned)grid_a, 256, 0, s>>>(W, n, reinterpret_cast<unsigned *>(scale2));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    scale2_kernel<<<1, 1, 0, s>>>(scale2);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t groups = N * (K / 16);
    const int64_t grid_q = std::min<int64_t>((groups + 255) / 256, (int64_t)sms * 16);
    quantize_nvfp4_kernel<WT><<<(unsigned)grid_q, 256, 0, s>>>(W, N, K, scale2, 0.0f, payload, scales);
    return cudaGetLastError();
}

template <typename WT>
cudaError_t launch_quantize_scaled_t(const WT *W, int64_t N, int64_t K, float scale2, uint8_t *payload,
                                     uint8_t *scales, cudaStream_t s) {
    const int64_t groups = N * (K / 16);
    const int64_t grid_q = std::min<int64_t>((groups + 255) / 256, (int64_t)sm_count() * 16);
    quantize_nvfp4_kernel<WT><<<(unsigned)grid_q, 256, 0, s>>>(W, N, K, nullptr, scale2, payload, scales);
    return cudaGetLastError();
}

// ------------------------------------------------------------ Q4_K fit
// One warp per super-block of 256 weights: lane l holds k = 8l .. 8l+7, so
// sub-block j (32 weights) is lanes 4j .. 4j+3.  Per sub-block: lo = min(0,
// min w), scale = (max w - lo) / 15, min = -lo; d = fp16(max scale / 63),
// dmin = fp16(max min / 63); s_j = clamp(rint(scale / d), 0, 63), m_j =
// clamp(rint(min / dmin), 0, 63) (0 for a zero divisor); q = clamp(rint((w +
// dmin*m_j) / (d*s_j)), 0, 15) (0 for a zero step).  Each step is one IEEE
// f32 operation and rint rounds half to even.  The pages give only the
// decode, w = d*s_j*q - dmin*m_j ([FBTC] sections 5-6); the fit is the
// plainest one it supports.
template <typename WT> __device__ __forceinline__ void load8(const WT *p, float v[8]);
template <> __device__ __forceinline__ void load8<float>(const float *p, float v[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float v[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t clamp_rint(float v, float top) {
    const float r = rintf(v);
    return r < 0.0f ? 0u : r > top ? (uint32_t)top : (uint32_t)r;
}

template <typename WT>
__global__ void __launch_bounds__(256) quantize_q4k_kernel(const WT *__restrict__ W, int64_t nblocks, int64_t K,
                                                           uint8_t *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (blk >= nblocks) return;                                        // warp-uniform
    (void)K;
    float w[8];
    load8<WT>(W + blk * 256 + lane * 8, w);                            // row n, block b: (n * K/256 + b) * 256
    float lo = 0.0f, hi = w[0];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        lo = fminf(lo, w[i]);
        hi = fmaxf(hi, w[i]);
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {                          // the four lanes of the sub-block
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    const float scale = __fdiv_rn(__fsub_rn(hi, lo), 15.0f), mins = -lo;
    // the maxima start from +0 and take only larger values, so a signed zero
    // never reaches d or dmin
    float smax = scale > 0.0f ? scale : 0.0f, mmax = mins > 0.0f ? mins : 0.0f;
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {                         // over the eight sub-blocks
        smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, off));
        mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, off));
    }
    const unsigned short dbits = __half_as_ushort(__float2half_rn(__fdiv_rn(smax, 63.0f)));
    const unsigned short mbits = __half_as_ushort(__float2half_rn(__fdiv_rn(mmax, 63.0f)));
    const float d = __half2float(__ushort_as_half(dbits)), dmin = __half2float(__ushort_as_half(mbits));
    const uint32_t sj = d > 0.0f ? clamp_rint(__fdiv_rn(scale, d), 63.0f) : 0u;
    const uint32_t mj = dmin > 0.0f ? clamp_rint(__fdiv_rn(mins, dmin), 63.0f) : 0u;
    const float step = __fmul_rn(d, (float)sj), offv = __fmul_rn(dmin, (float)mj);
    uint32_t codes = 0u;                                               // nibble i = code of k = 8l + i
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const uint32_t q = step > 0.0f ? clamp_rint(__fdiv_rn(__fadd_rn(w[i], offv), step), 15.0f) : 0u;
        codes |= q << (4 * i);
    }
    uint8_t *o = out + blk * 144;
    // code byte 32c + p = k 64c + p (low nibble, sub-block 2c) | k 64c + 32 + p (high, sub-block 2c + 1):
    // lane l of an even sub-block pairs with lane l + 4
    const uint32_t partner = __shfl_down_sync(0xffffffffu, codes, 4);
    const int j = lane >> 2;
    if ((j & 1) == 0) {
        uint32_t lo4 = 0u, hi4 = 0u;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t byte = ((codes >> (4 * i)) & 15u) | (((partner >> (4 * i)) & 15u) << 4);
            if (i < 4) lo4 |= byte << (8 * i);
            else hi4 |= byte << (8 * (i - 4));
        }
        *reinterpret_cast<uint2 *>(o + 16 + 32 * (j >> 1) + 8 * (lane & 3)) = make_uint2(lo4, hi4);
    }
    // header: d, dmin, then the 12 packed bytes of the eight (s_j, m_j)
    uint32_t S[8], Mv[8];
#pragma unroll
    for (int jj = 0; jj < 8; jj++) {
        S[jj] = __shfl_sync(0xffffffffu, sj, 4 * jj);
        Mv[jj] = __shfl_sync(0xffffffffu, mj, 4 * jj);
    }
    if (lane == 0) {
        uint32_t B[12];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            B[jj] = S[jj] | ((S[jj + 4] >> 4) << 6);
            B[jj + 4] = Mv[jj] | ((Mv[jj + 4] >> 4) << 6);
            B[jj + 8] = (S[jj + 4] & 15u) | ((Mv[jj + 4] & 15u) << 4);
        }
        uint4 h;
        h.x = (uint32_t)dbits | ((uint32_t)mbits << 16);
        h.y = B[0] | (B[1] << 8) | (B[2] << 16) | (B[3] << 24);
        h.z = B[4] | (B[5] << 8) | (B[6] << 16) | (B[7] << 24);
        h.w = B[8] | (B[9] << 8) | (B[10] << 16) | (B[11] << 24);
        *reinterpret_cast<uint4 *>(o) = h;
    }
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const void *W, q4_dtype wd, int64_t N, int64_t K, uint8_t *payload, uint8_t *scales,
                                  float *scale2, cudaStream_t s) {
    if (wd == Q4_DT_BF16)
        return launch_quantize_t(reinterpret_cast<const __nv_bfloat16 *>(W), N, K, payload, scales, scale2, s);
    return launch_quantize_t(reinterpret_cast<const float *>(W), N, K, payload, scales, scale2, s);
}

cudaError_t launch_quantize_nvfp4_scaled(const void *W, q4_dtype wd, int64_t N, int64_t K, float scale2,
                                         uint8_t *payload, uint8_t *scales, cudaStream_t s) {
    if (wd == Q4_DT_BF16)
        return launch_quantize_scaled_t(reinterpret_cast<const __nv_bfloat16 *>(W), N, K, scale2, payload, scales, s);
    return launch_quantize_scaled_t(reinterpret_cast<const float *>(W), N, K, scale2, payload, scales, s);
}

cudaError_t launch_quantize_q4k(const void *W, q4_dtype wd, int64_t N, int64_t K, uint8_t *out, cudaStream_t s) {
    const int64_t nblocks = N * (K / 256);
    const unsigned grid = (unsigned)((nblocks + 7) / 8);
    if (wd == Q4_DT_BF16)
        quantize_q4k_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16 *>(W), nblocks,
                                                                K, out);
    else
        quantize_q4k_kernel<float><<<grid, 256, 0, s>>>(reinterpret_cast<const float *>(W), nblocks, K, out);
    return cudaGetLastError();
}

}  // namespace q4
