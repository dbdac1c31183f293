// repack.cu -- q4_repack and q4_validate kernels.
//
// Repacking goes through the logical matrix ([BPA] "Repacking between
// formats"): every output word is gathered from the source's logical codes
// (unpacked along the source's own axis and slot order), zero points are
// normalised (GPTQ stores zero-1), act-order g_idx is resolved into a K
// permutation, and codes are packed along the target's axis and order.  The
// kernels are output-driven gathers, so each output word is written once.
#include "q4_internal.cuh"

namespace q4 {
namespace {

// Sticky per-device flags of the last repack: bit 0 a zero the target cannot
// store, bit 1 an act-order group without exactly `group` rows, bit 2 a g_idx
// value out of range or a non-trivial g_idx without perm_out.
__device__ unsigned int g_repack_flags;

struct Src {
    q4_fmt fmt;
    const uint8_t *w, *scales, *zeros;
    int group;
    int64_t N, K;
};

// logical code of (k, n) in the source, 0..15
__device__ __forceinline__ uint32_t src_code(const Src &s, int64_t k, int64_t n) {
    if (s.fmt == Q4_GPTQ) {
        uint32_t w = reinterpret_cast<const uint32_t *>(s.w)[(k >> 3) * s.N + n];
        return (w >> (4 * (k & 7))) & 15u;
    }
    if (s.fmt == Q4_AWQ) {
        uint32_t w = reinterpret_cast<const uint32_t *>(s.w)[k * (s.N >> 3) + (n >> 3)];
        return (w >> (4 * awq_slot((int)(n & 7)))) & 15u;
    }
    if (s.fmt == Q4_Q40) {
        const uint8_t *blk = s.w + (n * (s.K >> 5) + (k >> 5)) * 18;
        int i = (int)(k & 31);
        uint32_t b = blk[2 + (i & 15)];
        return i < 16 ? (b & 15u) : (b >> 4);
    }
    return s.w[k * s.N + n];   // logical
}

// normalised logical zero of (group g, column n)
__device__ __forceinline__ int src_zero(const Src &s, int64_t g, int64_t n) {
    if (s.fmt == Q4_GPTQ) {
        uint32_t w = reinterpret_cast<const uint32_t *>(s.zeros)[g * (s.N >> 3) + (n >> 3)];
        return (int)((w >> (4 * (n & 7))) & 15u) + 1;
    }
    if (s.fmt == Q4_AWQ) {
        uint32_t w = reinterpret_cast<const uint32_t *>(s.zeros)[g * (s.N >> 3) + (n >> 3)];
        return (int)((w >> (4 * awq_slot((int)(n & 7)))) & 15u);
    }
    if (s.fmt == Q4_Q40) return 8;
    return s.zeros[g * s.N + n];
}

__device__ __forceinline__ uint16_t src_scale_bits(const Src &s, int64_t g, int64_t n) {
    if (s.fmt == Q4_Q40) {
        const uint8_t *blk = s.w + (n * (s.K >> 5) + g) * 18;
        return (uint16_t)(blk[0] | (blk[1] << 8));
    }
    return reinterpret_cast<const uint16_t *>(s.scales)[g * s.N + n];
}

__device__ __forceinline__ int64_t src_row(const int32_t *perm, int64_t k) {
    return perm ? (int64_t)perm[k] : k;
}

template <int DST>
__global__ void repack_codes(Src s, const int32_t *__restrict__ perm, void *__restrict__ dst) {
    const int64_t N = s.N, K = s.K;
    const int64_t units = (DST == Q4_GPTQ) ? (K >> 3) * N : (DST == Q4_AWQ ? K * (N >> 3) : K * N);
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        if (DST == Q4_GPTQ) {
            const int64_t r = u / N, n = u % N;
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) word |= src_code(s, src_row(perm, 8 * r + j), n) << (4 * j);
            reinterpret_cast<uint32_t *>(dst)[u] = word;
        } else if (DST == Q4_AWQ) {
            const int64_t k = u / (N >> 3), c = u % (N >> 3);
            const int64_t kr = src_row(perm, k);
            uint32_t word = 0;
#pragma unroll
            for (int p = 0; p < 8; p++) {
                const int col = (p < 4) ? 2 * p : 2 * (p - 4) + 1;   // slot order 0,2,4,6,1,3,5,7
                word |= src_code(s, kr, 8 * c + col) << (4 * p);
            }
            reinterpret_cast<uint32_t *>(dst)[u] = word;
        } else {
            const int64_t k = u / N, n = u % N;
            reinterpret_cast<uint8_t *>(dst)[u] = (uint8_t)src_code(s, src_row(perm, k), n);
        }
    }
}

// GPTQ <-> AWQ without act-order is a transpose of 8 x 8 nibble blocks: the
// GPTQ words (r, 8c .. 8c+7) hold codes k = 8r .. 8r+7 of columns 8c .. 8c+7
// (one column per word), the AWQ words (8r .. 8r+7, c) hold the same codes
// one row per word, columns in slot order 0,2,4,6,1,3,5,7.  Each thread
// moves one block: 32 contiguous bytes on the GPTQ side, eight coalesced
// words on the AWQ side, and three rounds of masked swaps transpose the
// nibbles in registers.  Feeding the GPTQ words in slot order makes the
// transposed rows come out in AWQ slot order.
__device__ __forceinline__ void transpose_nibbles8(uint32_t (&w)[8]) {
#pragma unroll
    for (int st = 0; st < 3; st++) {
        const int sh = 4 << st;                                     // 4, 8, 16
        const uint32_t mask = st == 0 ? 0x0F0F0F0Fu : st == 1 ? 0x00FF00FFu : 0x0000FFFFu;
        const int d = 1 << st;                                      // row distance 1, 2, 4
#pragma unroll
        for (int a = 0; a < 8; a++) {
            if (a & d) continue;
            const int b = a + d;
            const uint32_t t = ((w[a] >> sh) ^ w[b]) & mask;
            w[b] ^= t;
            w[a] ^= t << sh;
        }
    }
}

template <bool TO_AWQ>
__global__ void repack_gptq_awq(const uint32_t *__restrict__ src, uint32_t *__restrict__ dst, int64_t K,
                                int64_t N) {
    const int64_t C = N >> 3, units = (K >> 3) * C;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = u / C, c = u % C;
        uint32_t w[8];
        if (TO_AWQ) {
            const uint4 lo = *reinterpret_cast<const uint4 *>(src + r * N + 8 * c);
            const uint4 hi = *reinterpret_cast<const uint4 *>(src + r * N + 8 * c + 4);
            const uint32_t g[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int p = 0; p < 8; p++) w[p] = g[p < 4 ? 2 * p : 2 * (p - 4) + 1];   // slot p holds column col(p)
            transpose_nibbles8(w);
#pragma unroll
            for (int k = 0; k < 8; k++) dst[(8 * r + k) * C + c] = w[k];
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++) w[k] = src[(8 * r + k) * C + c];
            transpose_nibbles8(w);                                  // w[p] = GPTQ word of column col(p)
            uint32_t g[8];
#pragma unroll
            for (int n = 0; n < 8; n++) g[n] = w[awq_slot(n)];
            *reinterpret_cast<uint4 *>(dst + r * N + 8 * c) = make_uint4(g[0], g[1], g[2], g[3]);
            *reinterpret_cast<uint4 *>(dst + r * N + 8 * c + 4) = make_uint4(g[4], g[5], g[6], g[7]);
        }
    }
}

template <int DST>
__global__ void repack_meta(Src s, uint16_t *__restrict__ dst_scales, void *__restrict__ dst_zeros) {
    const int64_t N = s.N, G = s.K / s.group;
    const int64_t units = G * (N >> 3);   // one unit = 8 consecutive columns of one group
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = u / (N >> 3), c = u % (N >> 3);
        uint32_t word = 0;
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int64_t n = 8 * c + j;
            dst_scales[g * N + n] = src_scale_bits(s, g, n);
            const int z = src_zero(s, g, n);
            if (DST == Q4_GPTQ) {
                bad |= (z < 1 || z > 16);
                word |= (uint32_t)((z - 1) & 15) << (4 * j);
            } else if (DST == Q4_AWQ) {
                bad |= (z < 0 || z > 15);
                word |= (uint32_t)(z & 15) << (4 * awq_slot(j));
            } else {
                bad |= (z < 0 || z > 255);
                reinterpret_cast<uint8_t *>(dst_zeros)[g * N + n] = (uint8_t)z;
            }
        }
        if (DST != Q4_LOGICAL) reinterpret_cast<uint32_t *>(dst_zeros)[u] = word;
        if (bad) atomicOr(&g_repack_flags, 1u);
    }
}

// Act-order permutation: target row of source row k is its rank in a stable
// sort by g_idx; perm[rank] = k.  Each group must land on [g*G, (g+1)*G).
__global__ void act_order_perm(const int32_t *__restrict__ g_idx, int64_t K, int group,
                               int32_t *__restrict__ perm) {
    const int64_t ngroups = K / group;
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < K;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int gk = g_idx[k];
        if (gk < 0 || gk >= ngroups) {
            atomicOr(&g_repack_flags, 4u);
            continue;
        }
        int64_t rank = 0;
        for (int64_t j = 0; j < K; j++) {
            const int gj = g_idx[j];
            rank += (gj < gk) || (gj == gk && j < k);
        }
        if (rank / group != gk) atomicOr(&g_repack_flags, 2u);
        else perm[rank] = (int32_t)k;
    }
}

// Flags a g_idx that is not the trivial k / group.
__global__ void check_trivial_gidx(const int32_t *__restrict__ g_idx, int64_t K, int group) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < K;
         k += (int64_t)gridDim.x * blockDim.x)
        if (g_idx[k] != (int32_t)(k / group)) atomicOr(&g_repack_flags, 4u);
}

// NVFP4 nibble order within each 16-value group: even/odd <-> split-half.
template <bool TO_SPLIT>
__global__ void repack_nvfp4_order(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                   int64_t ngroups) {
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < ngroups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const uint2 in = *reinterpret_cast<const uint2 *>(src + 8 * g);
        uint32_t c[16];
#pragma unroll
        for (int b = 0; b < 8; b++) {
            const uint32_t byte = ((b < 4 ? in.x : in.y) >> (8 * (b & 3))) & 0xffu;
            if (TO_SPLIT) {   // even/odd source: low nibble = lane 2b, high = 2b+1
                c[2 * b] = byte & 15u;
                c[2 * b + 1] = byte >> 4;
            } else {          // split-half source: low nibble = lane b, high = b+8
                c[b] = byte & 15u;
                c[b + 8] = byte >> 4;
            }
        }
        uint32_t o[2] = {0u, 0u};
#pragma unroll
        for (int b = 0; b < 8; b++) {
            const uint32_t byte = TO_SPLIT ? (c[b] | (c[b + 8] << 4)) : (c[2 * b] | (c[2 * b + 1] << 4));
            o[b >> 2] |= byte << (8 * (b & 3));
        }
        *reinterpret_cast<uint2 *>(dst + 8 * g) = make_uint2(o[0], o[1]);
    }
}

int grid_for(int64_t units) {
    int64_t b = (units + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

// ------------------------------------------------------------- validate
__global__ void count_bad(q4_fmt fmt, const uint8_t *__restrict__ p, int64_t count,
                          unsigned long long *__restrict__ bad) {
    unsigned long long local = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (fmt == Q4_NVFP4 || fmt == Q4_NVFP4_SPLITHALF) {
            local += (p[i] & 0x7fu) == 0x7fu;               // E4M3FN NaN: 0x7f / 0xff
        } else if (fmt == Q4_MXFP4) {
            local += p[i] == 0xffu;                         // E8M0 NaN
        } else {
            uint32_t h;
            if (fmt == Q4_Q4K) {                            // d and dmin of block i/2
                const uint8_t *q = p + (i >> 1) * 144 + 2 * (i & 1);
                h = q[0] | (q[1] << 8);
            } else if (fmt == Q4_Q40) {
                const uint8_t *q = p + i * 18;
                h = q[0] | (q[1] << 8);
            } else {
                h = reinterpret_cast<const uint16_t *>(p)[i];
            }
            local += (h & 0x7c00u) == 0x7c00u;              // fp16 Inf or NaN
        }
    }
    for (int off = 16; off >= 1; off >>= 1) local += __shfl_xor_sync(0xffffffffu, local, off);
    if ((threadIdx.x & 31) == 0 && local) atomicAdd(bad, local);
}

}  // namespace

int launch_repack(q4_fmt src, const Tensor &t, q4_fmt dst, void *dst_w, void *dst_scales,
                  void *dst_zeros, int32_t *perm_out, cudaStream_t st) {
    const bool nv_src = (src == Q4_NVFP4 || src == Q4_NVFP4_SPLITHALF);
    const bool nv_dst = (dst == Q4_NVFP4 || dst == Q4_NVFP4_SPLITHALF);
    if (nv_src || nv_dst) {
        if (!(nv_src && nv_dst)) return Q4_EUNSUPPORTED;
        const int64_t ngroups = t.N * t.K / 16;
        if (src == dst) {
            if (cudaMemcpyAsync(dst_w, t.w, (size_t)(t.N * t.K / 2), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return Q4_ECUDA;
        } else if (dst == Q4_NVFP4_SPLITHALF) {
            repack_nvfp4_order<true><<<grid_for(ngroups), 256, 0, st>>>(t.w, (uint8_t *)dst_w, ngroups);
        } else {
            repack_nvfp4_order<false><<<grid_for(ngroups), 256, 0, st>>>(t.w, (uint8_t *)dst_w, ngroups);
        }
        if (cudaGetLastError() != cudaSuccess) return Q4_ECUDA;
        if (cudaMemcpyAsync(dst_scales, t.scales, (size_t)(t.N * t.K / 16), cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
            return Q4_ECUDA;
        return Q4_OK;
    }
    const bool src_ok = (src == Q4_GPTQ || src == Q4_AWQ || src == Q4_Q40 || src == Q4_LOGICAL);
    const bool dst_ok = (dst == Q4_GPTQ || dst == Q4_AWQ || dst == Q4_LOGICAL);
    if (!src_ok || !dst_ok) return Q4_EUNSUPPORTED;

    Src s{src, t.w, t.scales, t.zeros, src == Q4_Q40 ? 32 : t.group, t.N, t.K};
    // Reset the flags on the device: a copy from (pageable) host memory would
    // first wait for the stream, a second host round trip per call.
    void *flags_dev = nullptr;
    if (cudaGetSymbolAddress(&flags_dev, g_repack_flags) != cudaSuccess ||
        cudaMemsetAsync(flags_dev, 0, sizeof(unsigned int), st) != cudaSuccess)
        return Q4_ECUDA;
    const int32_t *perm = nullptr;
    if (t.g_idx && (src == Q4_GPTQ || src == Q4_LOGICAL)) {
        if (perm_out) {
            act_order_perm<<<grid_for(t.K), 256, 0, st>>>(t.g_idx, t.K, s.group, perm_out);
            perm = perm_out;
        } else {
            check_trivial_gidx<<<grid_for(t.K), 256, 0, st>>>(t.g_idx, t.K, s.group);
        }
    }
    const int64_t N = t.N, K = t.K;
    const int64_t code_units = (dst == Q4_GPTQ) ? (K / 8) * N : (dst == Q4_AWQ ? K * (N / 8) : K * N);
    const int64_t meta_units = (K / s.group) * (N / 8);
    if (dst == Q4_GPTQ) {
        if (src == Q4_AWQ && !perm)
            repack_gptq_awq<false><<<grid_for(code_units / 8), 256, 0, st>>>((const uint32_t *)t.w,
                                                                               (uint32_t *)dst_w, K, N);
        else
            repack_codes<Q4_GPTQ><<<grid_for(code_units), 256, 0, st>>>(s, perm, dst_w);
        repack_meta<Q4_GPTQ><<<grid_for(meta_units), 256, 0, st>>>(s, (uint16_t *)dst_scales, dst_zeros);
    } else if (dst == Q4_AWQ) {
        if (src == Q4_GPTQ && !perm)
            repack_gptq_awq<true><<<grid_for(code_units / 8), 256, 0, st>>>((const uint32_t *)t.w, (uint32_t *)dst_w,
                                                                              K, N);
        else
            repack_codes<Q4_AWQ><<<grid_for(code_units), 256, 0, st>>>(s, perm, dst_w);
        repack_meta<Q4_AWQ><<<grid_for(meta_units), 256, 0, st>>>(s, (uint16_t *)dst_scales, dst_zeros);
    } else {
        repack_codes<Q4_LOGICAL><<<grid_for(code_units), 256, 0, st>>>(s, perm, dst_w);
        repack_meta<Q4_LOGICAL><<<grid_for(meta_units), 256, 0, st>>>(s, (uint16_t *)dst_scales, dst_zeros);
    }
    if (cudaGetLastError() != cudaSuccess) return Q4_ECUDA;
    unsigned int flags = 0;
    if (cudaMemcpyFromSymbolAsync(&flags, g_repack_flags, sizeof(flags), 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return Q4_ECUDA;
    if (flags & 4u) return Q4_EINVAL;
    if (flags & 2u) return Q4_EDIM;
    if (flags & 1u) return Q4_ERANGE;
    return Q4_OK;
}

int run_validate(const Tensor &t, int64_t *d_bad, cudaStream_t st) {
    int64_t count;
    const uint8_t *p = t.scales;
    switch (t.fmt) {
    case Q4_NVFP4:
    case Q4_NVFP4_SPLITHALF: count = t.N * t.K / 16; break;
    case Q4_MXFP4: count = t.N * t.K / 32; break;
    case Q4_Q4K: count = t.N * (t.K / 256) * 2; p = t.w; break;
    case Q4_Q40: count = t.N * (t.K / 32); p = t.w; break;
    default: count = (t.K / t.group) * t.N; break;
    }
    if (cudaMemsetAsync(d_bad, 0, sizeof(int64_t), st) != cudaSuccess) return Q4_ECUDA;
    count_bad<<<grid_for(count), 256, 0, st>>>(t.fmt, p, count, (unsigned long long *)d_bad);
    if (cudaGetLastError() != cudaSuccess) return Q4_ECUDA;
    int64_t bad = 0;
    if (cudaMemcpyAsync(&bad, d_bad, sizeof(bad), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return Q4_ECUDA;
    return bad ? Q4_ENAN : Q4_OK;
}

}  // namespace q4
