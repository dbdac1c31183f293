// pack_bits.cu -- b-bit code streams ([BPA] "The packing arithmetic", and
// "Odd widths: 3-bit, 2-bit and 6-bit") and the activation permutation of an
// act-order repack ([BPA] "Repacking between formats"), on sm_103a.
//
// Stream: code i occupies bits [i*b, (i+1)*b) of one little-endian bit stream
// cut into 32-bit words, so a code may straddle two words (b = 3, 5, 6, 7).
// But 32 codes of b bits fill exactly b words, so a group of 32 codes never
// shares a word with the next group: one thread packs (or unpacks) a whole
// group with two 16-byte code loads and b word stores, the shifts fixed at
// compile time.  Pure integer bit movement.
#include "q4_internal.cuh"

namespace q4 {

__device__ int g_pack_error;

namespace {

// One thread per group of 32 codes -> words [g*B, g*B + B).
template <int B>
__global__ void __launch_bounds__(256) pack_groups_kernel(const uint8_t *__restrict__ codes, int64_t ngroups,
                                                          uint32_t *__restrict__ words) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= ngroups) return;
    const uint4 c0 = __ldg(reinterpret_cast<const uint4 *>(codes) + 2 * g);
    const uint4 c1 = __ldg(reinterpret_cast<const uint4 *>(codes) + 2 * g + 1);
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    constexpr uint32_t MASK = (1u << B) - 1u;
    uint32_t out[B];
    uint64_t acc = 0;
    int nb = 0, o = 0;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        acc |= (uint64_t)((cw[i >> 2] >> (8 * (i & 3))) & MASK) << nb;
        nb += B;
        if (nb >= 32) {
            out[o++] = (uint32_t)acc;
            acc >>= 32;
            nb -= 32;
        }
    }
    uint32_t *dst = words + g * B;
#pragma unroll
    for (int j = 0; j < B; j++) dst[j] = out[j];
}

// One thread per group of 32 codes <- words [g*B, g*B + B).
template <int B>
__global__ void __launch_bounds__(256) unpack_groups_kernel(const uint32_t *__restrict__ words, int64_t ngroups,
                                                            uint8_t *__restrict__ codes) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= ngroups) return;
    uint32_t in[B];
#pragma unroll
    for (int j = 0; j < B; j++) in[j] = __ldg(words + g * B + j);
    constexpr uint32_t MASK = (1u << B) - 1u;
    uint32_t cw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    uint64_t acc = in[0];
    int nb = 32, w = 1;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        if (nb < B) {                        // refill: the next word above the remaining bits
            acc |= (uint64_t)in[w++] << nb;
            nb += 32;
        }
        cw[i >> 2] |= ((uint32_t)acc & MASK) << (8 * (i & 3));
        acc >>= B;
        nb -= B;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(codes) + 2 * g;
    dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
}

// One thread per output word: the codes that overlap bits [32w, 32w + 32)
// (the words of a last, partial group).
__global__ void pack_bits_kernel(const uint8_t *__restrict__ codes, int64_t n, int bits, uint32_t *__restrict__ words,
                                 int64_t w0, int64_t nwords) {
    const int64_t w = w0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (w >= nwords) return;
    const int64_t lo = 32 * w, hi = lo + 32;                 // stream bits of this word
    uint32_t out = 0u;
    for (int64_t i = lo / bits; i * bits < hi && i < n; i++) {
        const uint32_t v = codes[i] & ((1u << bits) - 1u);
        const int64_t off = i * bits - lo;                   // may be negative for the first, straddling code
        out |= off >= 0 ? v << off : v >> (-off);
    }
    words[w] = out;
}

// One thread per code: its bits from one word, or two for a straddling code
// (the codes of a last, partial group).
__global__ void unpack_bits_kernel(const uint32_t *__restrict__ words, int64_t i0, int64_t n, int bits,
                                   uint8_t *__restrict__ codes) {
    const int64_t i = i0 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int64_t bit = i * bits, w = bit / 32;
    const int off = (int)(bit % 32);
    uint64_t two = words[w];
    if (off + bits > 32) two |= (uint64_t)words[w + 1] << 32;
    codes[i] = (uint8_t)((two >> off) & ((1u << bits) - 1u));
}

// x_perm[m][k] = x[m][perm[k]]: the activation side of an act-order repack
// (perm = the perm_out of q4_repack: the source row of each target row).
// An index outside [0, K) is not read: the element becomes 0 and the sticky
// error word records Q4_ERANGE (read by q4_last_error).
template <typename T>
__global__ void permute_k_kernel(const T *__restrict__ x, const int32_t *__restrict__ perm, T *__restrict__ out,
                                 int64_t M, int64_t K) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= M * K) return;
    const int64_t m = e / K, k = e % K;
    const int32_t src = perm[k];
    if (src < 0 || (int64_t)src >= K) {
        out[e] = T(0);
        atomicExch(&g_pack_error, Q4_ERANGE);
        return;
    }
    out[e] = x[m * K + src];
}

}  // namespace

int pack_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_pack_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_pack_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

template <int B> void pack_groups(const uint8_t *codes, int64_t ng, uint32_t *words, cudaStream_t s) {
    pack_groups_kernel<B><<<(unsigned)((ng + 255) / 256), 256, 0, s>>>(codes, ng, words);
}
template <int B> void unpack_groups(const uint32_t *words, int64_t ng, uint8_t *codes, cudaStream_t s) {
    unpack_groups_kernel<B><<<(unsigned)((ng + 255) / 256), 256, 0, s>>>(words, ng, codes);
}

cudaError_t launch_pack_bits(const uint8_t *codes, int64_t n, int bits, uint32_t *words, cudaStream_t s) {
    const int64_t nwords = n * bits / 32;            // the caller checks n * bits % 32 == 0
    const int64_t ng = n / 32, w0 = ng * bits;        // whole groups, then the words of the last partial one
    if (ng > 0) {
        switch (bits) {
        case 1: pack_groups<1>(codes, ng, words, s); break;
        case 2: pack_groups<2>(codes, ng, words, s); break;
        case 3: pack_groups<3>(codes, ng, words, s); break;
        case 4: pack_groups<4>(codes, ng, words, s); break;
        case 5: pack_groups<5>(codes, ng, words, s); break;
        case 6: pack_groups<6>(codes, ng, words, s); break;
        case 7: pack_groups<7>(codes, ng, words, s); break;
        default: pack_groups<8>(codes, ng, words, s); break;
        }
    }
    if (w0 < nwords)
        pack_bits_kernel<<<(unsigned)((nwords - w0 + 255) / 256), 256, 0, s>>>(codes, n, bits, words, w0, nwords);
    return cudaGetLastError();
}
cudaError_t launch_unpack_bits(const uint32_t *words, int64_t n, int bits, uint8_t *codes, cudaStream_t s) {
    const int64_t ng = n / 32, i0 = ng * 32;
    if (ng > 0) {
        switch (bits) {
        case 1: unpack_groups<1>(words, ng, codes, s); break;
        case 2: unpack_groups<2>(words, ng, codes, s); break;
        case 3: unpack_groups<3>(words, ng, codes, s); break;
        case 4: unpack_groups<4>(words, ng, codes, s); break;
        case 5: unpack_groups<5>(words, ng, codes, s); break;
        case 6: unpack_groups<6>(words, ng, codes, s); break;
        case 7: unpack_groups<7>(words, ng, codes, s); break;
        default: unpack_groups<8>(words, ng, codes, s); break;
        }
    }
    if (i0 < n) unpack_bits_kernel<<<(unsigned)((n - i0 + 255) / 256), 256, 0, s>>>(words, i0, n, bits, codes);
    return cudaGetLastError();
}
cudaError_t launch_permute_k(const void *x, q4_dtype xd, const int32_t *perm, void *out, int64_t M, int64_t K,
                             cudaStream_t s) {
    const unsigned grid = (unsigned)((M * K + 255) / 256);
    if (xd == Q4_DT_BF16)
        permute_k_kernel<uint16_t><<<grid, 256, 0, s>>>((const uint16_t *)x, perm, (uint16_t *)out, M, K);
    else
        permute_k_kernel<float><<<grid, 256, 0, s>>>((const float *)x, perm, (float *)out, M, K);
    return cudaGetLastError();
}

}  // namespace q4
