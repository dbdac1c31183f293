// q4_internal.cuh -- device decode helpers and the internal launch interface
// shared by the CUDA translation units of libq4.so (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q4.h"

namespace q4 {

// ------------------------------------------------------------------ decode
// E2M1 pair -> two f32 values, through the sm_100-family hardware convert
// (cvt.rn.f16x2.e2m1x2).  Bits [3:0] of `byte` land in .x, bits [7:4] in .y:
// the low nibble is the even k ([MUS7] 7.1).  Every E2M1 value is exact in
// f16 and f32.
__device__ __forceinline__ float2 e2m1x2_f32(uint32_t byte) {
    uint32_t h2;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// Same, left as the packed f16x2 bit pattern.
__device__ __forceinline__ uint32_t e2m1x2_h2(uint32_t byte) {
    uint32_t h2;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
    return h2;
}

// Four E2M1 pairs of one 32-bit payload word -> four f16x2 (byte b -> h[b];
// low nibble in the low half).  The byte split is a register-level unpack.
__device__ __forceinline__ void e2m1x8_h2(uint32_t w, uint32_t &h0, uint32_t &h1, uint32_t &h2, uint32_t &h3) {
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

// Mixed-precision FMA (sm_100 family): c + a*b with f16 a, b taken from the
// low (HI=0) or high (HI=1) halves of two f16x2 registers; the product is
// exact and the sum rounds once in f32, exactly like fmaf on the widened
// operands.
template <int HI>
__device__ __forceinline__ float fma_f16_f32(uint32_t a2, uint32_t b2, float c) {
    float d;
    if (HI)
        asm("{ .reg .b16 al, ah, bl, bh;\n\t mov.b32 {al, ah}, %1;\n\t mov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.f16 %0, ah, bh, %3; }"
            : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    else
        asm("{ .reg .b16 al, ah, bl, bh;\n\t mov.b32 {al, ah}, %1;\n\t mov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.f16 %0, al, bl, %3; }"
            : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    return d;
}

// Two E4M3FN bytes (low byte -> .x) -> f32, via cvt.rn.f16x2.e4m3x2; every
// finite E4M3FN value (subnormals included) is exact in f16.
__device__ __forceinline__ float2 e4m3x2_f32(uint32_t two_bytes) {
    uint32_t h2;
    uint16_t in = (uint16_t)two_bytes;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

__device__ __forceinline__ float e4m3_f32(uint32_t byte) { return e4m3x2_f32(byte & 0xffu).x; }

// E8M0 byte -> 2^(b-127) as an f32 bit pattern ([FBTC] section 3); b = 0 is
// the subnormal 2^-127, b = 255 (NaN encoding) yields a quiet NaN.
__device__ __forceinline__ float e8m0_f32(uint32_t b) {
    b &= 0xffu;
    uint32_t bits = b == 0u ? 0x00400000u : (b == 255u ? 0x7fc00000u : (b << 23));
    return __uint_as_float(bits);
}

__device__ __forceinline__ float half_bits_f32(uint32_t h) {
    return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

// Exact float of a small unsigned integer q < 2^23 minus `bias`, by the
// magic-number construction 2^23 + q (one LOP3-able OR and one FADD).
__device__ __forceinline__ float uint_minus(uint32_t q, float bias_plus_2p23) {
    return __uint_as_float(0x4b000000u | q) - bias_plus_2p23;
}

// Packed two-lane f32 FMA (sm_100 family): acc = a * b + acc, lane-wise, one
// rounding per lane exactly like two scalar fmaf calls.
__device__ __forceinline__ void ffma2(float2 &acc, float2 a, float2 b) {
    asm("{ .reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc; }"
        : "+f"(acc.x), "+f"(acc.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
}

template <typename XT> __device__ __forceinline__ float x_to_f32(XT v);
template <> __device__ __forceinline__ float x_to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float x_to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

// Read-only, no-L1-allocate streaming loads for the packed weights.
__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream4(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream2(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream1(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// AWQ slot of logical column j (inverse of the slot order 0,2,4,6,1,3,5,7).
__device__ __forceinline__ int awq_slot(int j) { return (j >> 1) + 4 * (j & 1); }

// --------------------------------------------- mbarrier + bulk-copy (TMA)
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Bounded wait: gives up after ~`limit_cycles` SM clocks and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long limit_cycles = 2000000000LL) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit_cycles) return false;
    }
    return true;
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes and both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------ launch interface
struct Tensor {
    q4_fmt fmt;
    const uint8_t *w;
    const uint8_t *scales;
    const uint8_t *zeros;
    const int32_t *g_idx;
    int32_t group;
    float scale2;
    int64_t N, K;
};

int sm_count();
// Host-side argument rules shared by every entry point (q4_api.cu): format
// known, 16-byte alignment, and the shape rule of each format.
bool known(q4_fmt f);
bool aligned16(const void *p);
int check_dims(q4_fmt f, int64_t N, int64_t K, int group);
// Every check on a packed weight tensor, then fills `t`.  The NVFP4 scale2
// check comes last (Q4_ESCALE2), so a caller that does not read scale2 may
// ignore that status.
int make_tensor(q4_fmt f, const void *W, const void *scales, const q4_aux *aux, int64_t N, int64_t K, Tensor &t,
                bool need_scale2 = true);
// Records, per host thread, which kernel family the latest q4_gemv /
// q4_gemv_grouped call launched (read back by q4_last_gemv_path).
void note_gemv_path(const char *name);
cudaError_t launch_dequant(const Tensor &t, void *out, q4_dtype out_dtype, cudaStream_t s);
cudaError_t launch_gemv(const Tensor &t, const void *x, q4_dtype x_dtype, float *y, int64_t M,
                        cudaStream_t s);
cudaError_t launch_gemm_tc(const Tensor &t, const void *x, q4_dtype x_dtype, float *y, int64_t M,
                           cudaStream_t s, bool *handled);
bool gemv_mma_eligible(const Tensor &t, int64_t M);
bool gemv_tma_eligible(const Tensor &t, int64_t M);
// Batch-1 NVFP4 on the native block-scaled FP4 tensor cores (gemv_fp4tc.cu).
bool gemv_fp4tc_eligible(const Tensor &t, int64_t M);
cudaError_t launch_gemv_fp4tc(const Tensor &t, const void *x, float *y, cudaStream_t s);
cudaError_t launch_gemv_fp4tc_group(const Tensor *ts, int count, const void *x, float *const *ys, cudaStream_t s);
// NVFP4 weights x NVFP4 activations on the same tensor-core kernel (W4A4).
bool gemv_w4a4_tc_eligible(const Tensor &t);
cudaError_t launch_gemv_w4a4_tc(const Tensor &t, const uint8_t *xq, const uint8_t *xs, float x_scale2, float *y,
                                int64_t M, cudaStream_t s);
cudaError_t launch_gemv_tma(const Tensor &t, const void *x, float *y, int64_t M, cudaStream_t s);
cudaError_t launch_gemv_tma_group(const Tensor *ts, const void *x, float *const *ys, int count, int64_t M,
                                  cudaStream_t s);
bool gemv_tma_chain_fits(const Tensor *ts, const int *first, int ngroups, int64_t M);
cudaError_t launch_gemv_tma_chain(const Tensor *ts, const void *const *xs, float *const *ys, const int *first,
                                  int ngroups, int64_t M, unsigned *sync, cudaStream_t s);
bool gemv_blk_eligible(const Tensor &t, int64_t M);
bool gemv_blk_tc_eligible(const Tensor &t, int64_t M, q4_dtype xd);
cudaError_t launch_gemv_blk_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);
cudaError_t launch_gemv_blk_tc_group(const Tensor *ts, int count, const void *x, q4_dtype xd, float *const *ys,
                                     int64_t M, cudaStream_t s);
cudaError_t launch_gemv_blk(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);
bool gemv_gptq_eligible(const Tensor &t, int64_t M);
// GPTQ group 128 (no g_idx) on the tensor cores, weights by tensor TMA (gemv_gptq_tc.cu).
bool gemv_gptq_tc_eligible(const Tensor &t, int64_t M);
cudaError_t launch_gemv_gptq_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);
// AWQ group 128 on the tensor cores, weights by tensor TMA (gemv_awq_tc.cu).
bool gemv_awq_tc_eligible(const Tensor &t, int64_t M);
cudaError_t launch_gemv_awq_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);
cudaError_t launch_gemv_gptq(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);
cudaError_t launch_gemv_mma(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);
cudaError_t launch_gemv_mma_group(const Tensor *ts, const void *const *xs, float *const *ys, int count, int64_t M,
                                  cudaStream_t s);
int launch_repack(q4_fmt src, const Tensor &t, q4_fmt dst, void *dst_w, void *dst_scales,
                  void *dst_zeros, int32_t *perm_out, cudaStream_t s);
int run_validate(const Tensor &t, int64_t *d_bad, cudaStream_t s);

// ------------------------------------------------- per-element decoders
// w_hat(n, k) for every format, f32, by the pinned rule: one weight at a time
// with byte loads (dequant's K-major tiles and the general-shape GEMV; not
// the bandwidth-bound path).
template <int FMT>
__device__ __forceinline__ float elem_weight(const Tensor &t, int64_t n, int64_t k) {
    const int64_t N = t.N, K = t.K;
    if (FMT == Q4_NVFP4 || FMT == Q4_NVFP4_SPLITHALF || FMT == Q4_MXFP4) {
        const uint8_t *row = t.w + n * (K >> 1);
        uint32_t code;
        if (FMT == Q4_NVFP4_SPLITHALF) {
            int lane = (int)(k & 15);
            uint32_t b = row[(k >> 4) * 8 + (lane & 7)];
            code = lane < 8 ? (b & 15u) : (b >> 4);
        } else {
            uint32_t b = row[k >> 1];
            code = (k & 1) ? (b >> 4) : (b & 15u);
        }
        float v = e2m1x2_f32(code).x;
        if (FMT == Q4_MXFP4) return __fmul_rn(v, e8m0_f32(t.scales[n * (K >> 5) + (k >> 5)]));
        float p = __fmul_rn(v, e4m3_f32(t.scales[n * (K >> 4) + (k >> 4)]));
        return __fmul_rn(p, t.scale2);
    } else if (FMT == Q4_Q4K) {
        const uint8_t *blk = t.w + (n * (K >> 8) + (k >> 8)) * 144;
        int i = (int)(k & 255), c = i >> 6, r = i & 63, hi = r >= 32;
        uint32_t b = blk[16 + 32 * c + (r & 31)];
        uint32_t q = hi ? (b >> 4) : (b & 15u);
        const uint8_t *B = blk + 4;
        int j = 2 * c + hi;
        uint32_t sc, mn;
        if (j < 4) {
            sc = B[j] & 63u;
            mn = B[j + 4] & 63u;
        } else {
            sc = (B[j + 4] & 15u) | ((uint32_t)(B[j - 4] >> 6) << 4);
            mn = (uint32_t)(B[j + 4] >> 4) | ((uint32_t)(B[j] >> 6) << 4);
        }
        float d = half_bits_f32(blk[0] | (blk[1] << 8)), dmin = half_bits_f32(blk[2] | (blk[3] << 8));
        float step = __fmul_rn(d, (float)sc), off = __fmul_rn(dmin, (float)mn);
        return __fmaf_rn((float)q, step, -off);
    } else if (FMT == Q4_Q40) {
        const uint8_t *blk = t.w + (n * (K >> 5) + (k >> 5)) * 18;
        int i = (int)(k & 31);
        uint32_t b = blk[2 + (i & 15)];
        uint32_t q = i < 16 ? (b & 15u) : (b >> 4);
        return __fmul_rn(half_bits_f32(blk[0] | (blk[1] << 8)), (float)((int)q - 8));
    } else {
        int64_t g = t.g_idx ? (int64_t)t.g_idx[k] : k / t.group;
        float s = half_bits_f32(reinterpret_cast<const uint16_t *>(t.scales)[g * N + n]);
        int q, z;
        if (FMT == Q4_GPTQ) {
            uint32_t word = reinterpret_cast<const uint32_t *>(t.w)[(k >> 3) * N + n];
            q = (int)((word >> (4 * (k & 7))) & 15u);
            uint32_t zw = reinterpret_cast<const uint32_t *>(t.zeros)[g * (N >> 3) + (n >> 3)];
            z = (int)((zw >> (4 * (n & 7))) & 15u) + 1;
        } else if (FMT == Q4_AWQ) {
            int p = awq_slot((int)(n & 7));
            uint32_t word = reinterpret_cast<const uint32_t *>(t.w)[k * (N >> 3) + (n >> 3)];
            q = (int)((word >> (4 * p)) & 15u);
            uint32_t zw = reinterpret_cast<const uint32_t *>(t.zeros)[g * (N >> 3) + (n >> 3)];
            z = (int)((zw >> (4 * p)) & 15u);
        } else {
            q = t.w[k * N + n];
            z = t.zeros[g * N + n];
        }
        return __fmul_rn(s, (float)(q - z));
    }
}

}  // namespace q4
