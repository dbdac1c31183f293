// dequant.cu -- q4_dequant kernels: packed tensor -> f32 or bf16 [N][K] by the
// pinned per-format rule.  Write-bound (4 or 2 bytes out per weight), so each
// kernel is organised for coalesced stores; the packed reads are small.
#include "q4_internal.cuh"

namespace q4 {
namespace {

template <typename OT> __device__ __forceinline__ OT to_out(float v);
template <> __device__ __forceinline__ float to_out<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// NVFP4 / split-half NVFP4 / MXFP4: one thread per 16 output bytes (4 f32 or
// 8 bf16 values, a quarter or half of a 16-value group), so each warp store
// writes 512 contiguous bytes; the lanes of one group read its 8 payload
// bytes together.  NVFP4 order (e2m1 * e4m3fn) * scale2 ([MUS7] 7.2): the
// first product is exact, the second is the single rounding.
template <typename OT> __device__ __forceinline__ void store_chunk(OT *out, const float *v);
template <> __device__ __forceinline__ void store_chunk<float>(float *out, const float *v) {
    *reinterpret_cast<float4 *>(out) = make_float4(v[0], v[1], v[2], v[3]);
}
template <> __device__ __forceinline__ void store_chunk<__nv_bfloat16>(__nv_bfloat16 *out, const float *v) {
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        p[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(out) = make_uint4(p[0], p[1], p[2], p[3]);
}

template <int FMT, typename OT>
__global__ void dequant_fp4(const uint8_t *__restrict__ w, const uint8_t *__restrict__ scales,
                            float scale2, OT *__restrict__ out, int64_t nchunks) {
    constexpr int VPL = 16 / (int)sizeof(OT);   // values per thread
    constexpr int CPG = 16 / VPL;               // threads per 16-value group
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < nchunks;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = u / CPG;
        const int part = (int)(u % CPG);
        const uint2 p = *reinterpret_cast<const uint2 *>(w + 8 * g);
        const uint64_t bits = (uint64_t)p.x | ((uint64_t)p.y << 32);
        const float sc = (FMT == Q4_MXFP4) ? e8m0_f32(scales[g >> 1]) : e4m3_f32(scales[g]);
        float v[VPL];
        if (FMT == Q4_NVFP4_SPLITHALF) {
            // value j: low nibble of byte j (j < 8), high nibble of byte j - 8 ([W4K] section 5)
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int j = part * VPL + i;
                const uint32_t nib = (uint32_t)(bits >> (j < 8 ? 8 * j : 8 * (j - 8) + 4)) & 15u;
                v[i] = e2m1x2_f32(nib).x;
            }
        } else {
            // value j: nibble j (low nibble = even k); byte pairs decode together
#pragma unroll
            for (int b = 0; b < VPL / 2; b++) {
                const float2 c = e2m1x2_f32((uint32_t)(bits >> (8 * (part * VPL / 2 + b))) & 0xffu);
                v[2 * b] = c.x;
                v[2 * b + 1] = c.y;
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            if (FMT == Q4_MXFP4) {
                v[i] = __fmul_rn(v[i], sc);
            } else {
                const float prod = __fmul_rn(v[i], sc);
                v[i] = __fmul_rn(prod, scale2);
            }
        }
        store_chunk<OT>(out + VPL * u, v);
    }
}

// Q4_K: code byte b of 32-byte group c holds k = 64c + b (low nibble,
// sub-block 2c) and 64c + 32 + b (high nibble, sub-block 2c+1) ([FBTC]
// sections 5-6).  w = fma(q, d*s, -dmin*m) equals the pinned (d*s)*q - dmin*m:
// d*s*q is exact, one rounding.
__device__ __forceinline__ uint32_t byte_of(uint4 hdr, int i) {
    uint32_t word = i < 4 ? hdr.y : (i < 8 ? hdr.z : hdr.w);
    return (word >> (8 * (i & 3))) & 0xffu;
}

__device__ __forceinline__ void q4k_scale_min(uint4 hdr, int j, float &sc, float &mn) {
    uint32_t s, m;
    if (j < 4) {
        s = byte_of(hdr, j) & 63u;
        m = byte_of(hdr, j + 4) & 63u;
    } else {
        s = (byte_of(hdr, j + 4) & 15u) | ((byte_of(hdr, j - 4) >> 6) << 4);
        m = (byte_of(hdr, j + 4) >> 4) | ((byte_of(hdr, j) >> 6) << 4);
    }
    sc = (float)s;
    mn = (float)m;
}

template <typename OT>
__global__ void dequant_q4k(const uint8_t *__restrict__ w, OT *__restrict__ out, int64_t nchunks) {
    // one thread per 16 output bytes: VPL consecutive k of one sub-block
    constexpr int VPL = 16 / (int)sizeof(OT);
    constexpr int CPB = 256 / VPL;   // chunks per super-block
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < nchunks;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t blk = u / CPB;
        const int k0 = (int)(u % CPB) * VPL;            // within the super-block
        const int c = k0 >> 6, hi = (k0 >> 5) & 1, b0 = k0 & 31;
        const uint8_t *b = w + blk * 144;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(b);
        float sc, mn;
        q4k_scale_min(hdr, 2 * c + hi, sc, mn);
        const float step = __fmul_rn(half_bits_f32(hdr.x), sc), off = __fmul_rn(half_bits_f32(hdr.x >> 16), mn);
        uint32_t words[VPL / 4];
#pragma unroll
        for (int i = 0; i < VPL / 4; i++) words[i] = *reinterpret_cast<const uint32_t *>(b + 16 + 32 * c + b0 + 4 * i);
        float v[VPL];
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const uint32_t byte = (words[i >> 2] >> (8 * (i & 3))) & 0xffu;
            v[i] = __fmaf_rn((float)(hi ? byte >> 4 : byte & 15u), step, -off);
        }
        store_chunk<OT>(out + blk * 256 + k0, v);
    }
}

// Q4_0: one thread per 16 output bytes of an 18-byte block: fp16 d, byte j =
// element j (low) and j+16 (high); w = d*(q-8), exact ([BPA] "Real layouts
// compared").  The block is 2-byte aligned, so the codes are read as u16.
template <typename OT>
__global__ void dequant_q40(const uint8_t *__restrict__ w, OT *__restrict__ out, int64_t nchunks) {
    constexpr int VPL = 16 / (int)sizeof(OT);
    constexpr int CPB = 32 / VPL;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < nchunks;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bi = u / CPB;
        const int k0 = (int)(u % CPB) * VPL;
        const uint16_t *b = reinterpret_cast<const uint16_t *>(w + bi * 18);
        const float d = half_bits_f32(b[0]);
        const int hi = k0 >> 4, j0 = k0 & 15;
        float v[VPL];
#pragma unroll
        for (int i = 0; i < VPL; i += 2) {
            const uint32_t two = b[1 + (j0 + i) / 2];
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const uint32_t byte = (two >> (8 * e)) & 0xffu;
                v[i + e] = __fmul_rn(d, (float)((int)(hi ? byte >> 4 : byte & 15u) - 8));
            }
        }
        store_chunk<OT>(out + bi * 32 + k0, v);
    }
}

// 64x64 tile, transposed through shared memory: reads run along n (the packed
// axis), writes along k (the output row).
template <int FMT, typename OT>
__global__ void dequant_kmajor(Tensor t, OT *__restrict__ out) {
    __shared__ float tile[64][65];
    int64_t n0 = (int64_t)blockIdx.x * 64, k0 = (int64_t)blockIdx.y * 64;
    int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 256 threads: 64 x 4
    for (int kk = ty; kk < 64; kk += 4) {
        int64_t n = n0 + tx, k = k0 + kk;
        tile[kk][tx] = (n < t.N && k < t.K) ? elem_weight<FMT>(t, n, k) : 0.0f;
    }
    __syncthreads();
    for (int nn = ty; nn < 64; nn += 4) {
        int64_t n = n0 + nn, k = k0 + tx;
        if (n < t.N && k < t.K) out[n * t.K + k] = to_out<OT>(tile[tx][nn]);
    }
}

int grid_for(int64_t units, int threads) {
    int64_t blocks = (units + threads - 1) / threads;
    int64_t cap = (int64_t)sm_count() * 16;
    return (int)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

template <typename OT> cudaError_t dispatch(const Tensor &t, OT *out, cudaStream_t s) {
    const int T = 256;
    switch (t.fmt) {
    case Q4_NVFP4: {
        int64_t n = t.N * t.K * (int64_t)sizeof(OT) / 16;   // 16-byte output chunks
        dequant_fp4<Q4_NVFP4, OT><<<grid_for(n, T), T, 0, s>>>(t.w, t.scales, t.scale2, out, n);
        break;
    }
    case Q4_NVFP4_SPLITHALF: {
        int64_t n = t.N * t.K * (int64_t)sizeof(OT) / 16;
        dequant_fp4<Q4_NVFP4_SPLITHALF, OT><<<grid_for(n, T), T, 0, s>>>(t.w, t.scales, t.scale2, out, n);
        break;
    }
    case Q4_MXFP4: {
        int64_t n = t.N * t.K * (int64_t)sizeof(OT) / 16;
        dequant_fp4<Q4_MXFP4, OT><<<grid_for(n, T), T, 0, s>>>(t.w, t.scales, 1.0f, out, n);
        break;
    }
    case Q4_Q4K: {
        int64_t n = t.N * t.K * (int64_t)sizeof(OT) / 16;
        dequant_q4k<OT><<<grid_for(n, T), T, 0, s>>>(t.w, out, n);
        break;
    }
    case Q4_Q40: {
        int64_t n = t.N * t.K * (int64_t)sizeof(OT) / 16;
        dequant_q40<OT><<<grid_for(n, T), T, 0, s>>>(t.w, out, n);
        break;
    }
    case Q4_GPTQ:
    case Q4_AWQ:
    case Q4_LOGICAL: {
        dim3 grid((unsigned)((t.N + 63) / 64), (unsigned)((t.K + 63) / 64));
        if (t.fmt == Q4_GPTQ) dequant_kmajor<Q4_GPTQ, OT><<<grid, 256, 0, s>>>(t, out);
        else if (t.fmt == Q4_AWQ) dequant_kmajor<Q4_AWQ, OT><<<grid, 256, 0, s>>>(t, out);
        else dequant_kmajor<Q4_LOGICAL, OT><<<grid, 256, 0, s>>>(t, out);
        break;
    }
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant(const Tensor &t, void *out, q4_dtype out_dtype, cudaStream_t s) {
    if (out_dtype == Q4_DT_BF16) return dispatch<__nv_bfloat16>(t, (__nv_bfloat16 *)out, s);
    return dispatch<float>(t, (float *)out, s);
}

}  // namespace q4
