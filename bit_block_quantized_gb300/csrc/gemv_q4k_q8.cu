// gemv_q4k_q8.cu -- the Q4_K x Q8 (W4A8) contraction of "Why 4-Bit
// Quantization Is King", section 7, on sm_103a.
//
// Activations are quantized per 256-value block to signed 8-bit codes (the
// signed first maximum m, iscale = -127/m, half-to-even, capped at 127, block
// scale 1/iscale), and each 32-value sub-block's code sum is kept.  Per
// output row and 256-weight super-block two exact integers
//     I1 = sum_j sc_j * sum_{k in j} q[k] * q8[k]     I2 = sum_j m_j * bsum_j
// are formed from the unsigned 4-bit codes and the 6-bit sub-block scales and
// minima; then, in f32 and in this order,
//     v = d * float(I1) - dmin * float(I2);  c = v * act_scale;  total += c
// over the super-blocks in order.  Output f32.
//
// Design (CUDA cores): as the A16-Q8 lane.  Each CTA quantizes its activation
// rows into shared memory; warps take output rows; 8 lanes share a 144-byte
// super-block: each loads 16 code bytes (its 16 low-nibble k of one sub-block
// and 16 high-nibble k of the next, both contiguous in k) and the 16-byte
// header (a broadcast).  One mask and one shift per word give four unsigned
// codes for a dp4a with four activation codes.
#include <algorithm>

#include "q4_internal.cuh"

namespace q4 {
namespace {

constexpr int K8_WARPS = 8;
constexpr int K8_THREADS = K8_WARPS * 32;
constexpr int K8_INFLIGHT = 4;

__device__ __forceinline__ int64_t k8_shfl_xor_i64(int64_t v, int mask) {
    return (int64_t)__shfl_xor_sync(0xffffffffu, (long long)v, mask);
}

// Metadata byte i (0..11) of a super-block header held as a uint4 (bytes 4..15).
__device__ __forceinline__ uint32_t meta_byte(uint4 h, int i) {
    const uint32_t w = i < 4 ? h.y : (i < 8 ? h.z : h.w);
    return (w >> (8 * (i & 3))) & 0xffu;
}

// 6-bit scale and minimum of sub-block j (0..7).
__device__ __forceinline__ void scale_min(uint4 h, int j, int &sc, int &mn) {
    if (j < 4) {
        sc = (int)(meta_byte(h, j) & 63u);
        mn = (int)(meta_byte(h, j + 4) & 63u);
    } else {
        const uint32_t b = meta_byte(h, j + 4);
        sc = (int)((b & 15u) | ((meta_byte(h, j - 4) >> 6) << 4));
        mn = (int)((b >> 4) | ((meta_byte(h, j) >> 6) << 4));
    }
}

// Shared layout: act_scale [MT][K/256] f32 | bsum [MT][K/32] i32 | q8 [MT][K] i8.
__host__ __device__ inline int64_t k8_bsum_off(int mt, int64_t K) { return (int64_t)mt * (K / 256) * 4; }
__host__ __device__ inline int64_t k8_q8_off(int mt, int64_t K) {
    return (k8_bsum_off(mt, K) + (int64_t)mt * (K / 32) * 4 + 15) / 16 * 16;
}
__host__ __device__ inline int64_t k8_smem_bytes(int mt, int64_t K) { return k8_q8_off(mt, K) + (int64_t)mt * K; }

template <typename XT> struct K8Load;
template <> struct K8Load<__nv_bfloat16> {
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
template <> struct K8Load<float> {
    static __device__ __forceinline__ void get(const float *p, float v[8]) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        const float4 b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

template <int MT, typename XT>
__global__ void __launch_bounds__(K8_THREADS)
gemv_q4k_q8_kernel(const uint8_t *__restrict__ W, const XT *__restrict__ x, float *__restrict__ y, int mrows,
                   int64_t N, int64_t K) {
    extern __shared__ __align__(16) unsigned char smem[];
    float *act_scale = reinterpret_cast<float *>(smem);
    int32_t *bsum = reinterpret_cast<int32_t *>(smem + k8_bsum_off(MT, K));
    int8_t *q8 = reinterpret_cast<int8_t *>(smem + k8_q8_off(MT, K));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nb = K / 256;

    // ---- activation quantization, one warp per (row m, block b); lanes 4j..4j+3 hold sub-block j
    for (int64_t item = warp; item < (int64_t)mrows * nb; item += K8_WARPS) {
        const int64_t m = item / nb, b = item % nb;
        float v[8];
        K8Load<XT>::get(x + m * K + b * 256 + lane * 8, v);
        float amax = 0.0f, val = 0.0f;
        int idx = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float a = fabsf(v[i]);
            if (a > amax) { amax = a; val = v[i]; idx = lane * 8 + i; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oa = __shfl_xor_sync(0xffffffffu, amax, off);
            const float ov = __shfl_xor_sync(0xffffffffu, val, off);
            const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
            if (oa > amax || (oa == amax && oi < idx)) { amax = oa; val = ov; idx = oi; }
        }
        const float iscale = __fdiv_rn(-127.0f, val);
        const bool live = isfinite(iscale);
        uint32_t packed[2] = {0u, 0u};
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            int c = live ? __float2int_rn(__fmul_rn(v[i], iscale)) : 0;
            c = c > 127 ? 127 : c;
            s += c;
            packed[i >> 2] |= ((uint32_t)c & 0xffu) << (8 * (i & 3));
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        *reinterpret_cast<uint2 *>(q8 + m * K + b * 256 + lane * 8) = make_uint2(packed[0], packed[1]);
        if ((lane & 3) == 0) bsum[m * (K / 32) + b * 8 + (lane >> 2)] = s;
        if (lane == 0) act_scale[m * nb + b] = live ? __fdiv_rn(1.0f, iscale) : 0.0f;
    }
    __syncthreads();

    // ---- rows: 8 lanes per super-block, 4 super-blocks per warp step
    const int64_t nchunks = (nb + 3) / 4;
    const int64_t total_warps = (int64_t)gridDim.x * K8_WARPS;
    const int sub = lane >> 3, q = lane & 7;
    const int j0 = 2 * (q >> 1), j1 = j0 + 1, half = q & 1;
    for (int64_t n = (int64_t)blockIdx.x * K8_WARPS + warp; n < N; n += total_warps) {
        const uint8_t *wrow = W + n * nb * 144;
        float total[MT];
#pragma unroll
        for (int m = 0; m < MT; m++) total[m] = 0.0f;
        for (int64_t c0 = 0; c0 < nchunks; c0 += K8_INFLIGHT) {
            uint4 hv[K8_INFLIGHT], cv[K8_INFLIGHT];
#pragma unroll
            for (int u = 0; u < K8_INFLIGHT; u++) {
                const int64_t b = (c0 + u) * 4 + sub;
                if (b < nb) {
                    const uint8_t *blk = wrow + b * 144;
                    hv[u] = __ldg(reinterpret_cast<const uint4 *>(blk));
                    cv[u] = ldg_stream16(blk + 16 + 16 * q);
                } else {
                    hv[u] = make_uint4(0u, 0u, 0u, 0u);
                    cv[u] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < K8_INFLIGHT; u++) {
                const int64_t c = c0 + u;
                if (c >= nchunks) break;                     // warp-uniform
                const int64_t b = c * 4 + sub;
                const bool valid = b < nb;                   // 8-lane uniform
                int sc0, mn0, sc1, mn1, scq, mnq;
                scale_min(hv[u], j0, sc0, mn0);
                scale_min(hv[u], j1, sc1, mn1);
                scale_min(hv[u], q, scq, mnq);
                const float d = __half2float(__ushort_as_half((unsigned short)(hv[u].x & 0xffffu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hv[u].x >> 16)));
                const uint32_t cw[4] = {cv[u].x, cv[u].y, cv[u].z, cv[u].w};
#pragma unroll
                for (int m = 0; m < MT; m++) {
                    if (m >= mrows) break;
                    int I1 = 0, I2 = 0;
                    float s = 0.0f;
                    if (valid) {
                        const int8_t *qrow = q8 + m * K + b * 256;
                        const uint4 qa = *reinterpret_cast<const uint4 *>(qrow + 32 * j0 + 16 * half);
                        const uint4 qb = *reinterpret_cast<const uint4 *>(qrow + 32 * j1 + 16 * half);
                        const uint32_t qaw[4] = {qa.x, qa.y, qa.z, qa.w}, qbw[4] = {qb.x, qb.y, qb.z, qb.w};
                        int dot0 = 0, dot1 = 0;
#pragma unroll
                        for (int t = 0; t < 4; t++) {
                            dot0 = __dp4a((int)(cw[t] & 0x0f0f0f0fu), (int)qaw[t], dot0);
                            dot1 = __dp4a((int)((cw[t] >> 4) & 0x0f0f0f0fu), (int)qbw[t], dot1);
                        }
                        I1 = sc0 * dot0 + sc1 * dot1;
                        I2 = mnq * bsum[m * (K / 32) + b * 8 + q];
                        s = act_scale[m * nb + b];
                    }
                    I1 += __shfl_xor_sync(0xffffffffu, I1, 1);
                    I2 += __shfl_xor_sync(0xffffffffu, I2, 1);
                    I1 += __shfl_xor_sync(0xffffffffu, I1, 2);
                    I2 += __shfl_xor_sync(0xffffffffu, I2, 2);
                    I1 += __shfl_xor_sync(0xffffffffu, I1, 4);
                    I2 += __shfl_xor_sync(0xffffffffu, I2, 4);
                    const float p1 = __fmul_rn(d, __int2float_rn(I1));
                    const float p2 = __fmul_rn(dmin, __int2float_rn(I2));
                    const float cc = __fmul_rn(__fsub_rn(p1, p2), s);
#pragma unroll
                    for (int jj = 0; jj < 4; jj++) {
                        const float cj = __shfl_sync(0xffffffffu, cc, jj * 8);
                        if (c * 4 + jj < nb) total[m] = __fadd_rn(total[m], cj);
                    }
                }
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; m++)
                if (m < mrows) y[(int64_t)m * N + n] = total[m];
        }
    }
}

template <int MT, typename XT>
cudaError_t k8_launch_mt(const Tensor &t, const XT *x, float *y, int mrows, cudaStream_t s) {
    const int64_t smem = k8_smem_bytes(MT, t.K);
    auto kern = gemv_q4k_q8_kernel<MT, XT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, K8_THREADS, (size_t)smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t want = (t.N + K8_WARPS - 1) / K8_WARPS;
    const int64_t grid = std::min<int64_t>(want, (int64_t)per_sm * sm_count());
    kern<<<(unsigned)grid, K8_THREADS, (size_t)smem, s>>>(t.w, x, y, mrows, t.N, t.K);
    return cudaGetLastError();
}

template <typename XT>
cudaError_t k8_launch_chunk(const Tensor &t, const XT *x, float *y, int mrows, cudaStream_t s) {
    if (mrows > 4) return k8_launch_mt<8, XT>(t, x, y, mrows, s);
    if (mrows > 2) return k8_launch_mt<4, XT>(t, x, y, mrows, s);
    if (mrows > 1) return k8_launch_mt<2, XT>(t, x, y, mrows, s);
    return k8_launch_mt<1, XT>(t, x, y, mrows, s);
}

}  // namespace

int gemv_q4k_q8_chunk(int64_t M, int64_t K) {
    const int64_t limit = 200 * 1024;
    for (int rows = (int)std::min<int64_t>(M, 8); rows >= 1; rows--) {
        const int mt = rows > 4 ? 8 : rows > 2 ? 4 : rows;
        if (k8_smem_bytes(mt, K) <= limit) return rows;
    }
    return 0;
}

bool gemv_q4k_q8_tc_eligible(const Tensor &t, int64_t M);
cudaError_t launch_gemv_q4k_q8_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);

cudaError_t launch_gemv_q4k_q8(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    // batch 1 and 2: the same contract with the sub-block sums on the tensor cores (gemv_q4k_q8_tc.cu)
    if (gemv_q4k_q8_tc_eligible(t, M)) {
        const cudaError_t e = launch_gemv_q4k_q8_tc(t, x, xd, y, M, s);
        if (e == cudaSuccess) note_gemv_path("gemv_q4k_q8_tc");
        return e;
    }
    const int chunk = gemv_q4k_q8_chunk(M, t.K);
    if (chunk == 0) return cudaErrorInvalidValue;
    for (int64_t m0 = 0; m0 < M; m0 += chunk) {
        const int mrows = (int)std::min<int64_t>(chunk, M - m0);
        cudaError_t e;
        if (xd == Q4_DT_BF16)
            e = k8_launch_chunk<__nv_bfloat16>(t, reinterpret_cast<const __nv_bfloat16 *>(x) + m0 * t.K,
                                               y + m0 * t.N, mrows, s);
        else
            e = k8_launch_chunk<float>(t, reinterpret_cast<const float *>(x) + m0 * t.K, y + m0 * t.N, mrows, s);
        if (e != cudaSuccess) return e;
    }
    note_gemv_path("gemv_q4k_q8");
    return cudaSuccess;
}

}  // namespace q4
