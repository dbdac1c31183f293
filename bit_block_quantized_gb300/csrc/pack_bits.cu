// pack_bits.cu -- b-bit code streams ([BPA] "The packing arithmetic", and
// "Odd widths: 3-bit, 2-bit and 6-bit") and the activation permutation of an
// act-order repack ([BPA] "Repacking between formats"), on sm_103a.
//
// Stream: code i occupies bits [i*b, (i+1)*b) of one little-endian bit stream
// cut into 32-bit words, so a code may straddle two words (b = 3, 5, 6, 7).
// Pure integer bit movement; one thread per output word or code.
#include "q4_internal.cuh"

namespace q4 {

__device__ int g_pack_error;

namespace {

// One thread per output word: the codes that overlap bits [32w, 32w + 32).
__global__ void pack_bits_kernel(const uint8_t *__restrict__ codes, int64_t n, int bits, uint32_t *__restrict__ words,
                                 int64_t nwords) {
    const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
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

// One thread per code: its bits from one word, or two for a straddling code.
__global__ void unpack_bits_kernel(const uint32_t *__restrict__ words, int64_t n, int bits,
                                   uint8_t *__restrict__ codes) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
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

cudaError_t launch_pack_bits(const uint8_t *codes, int64_t n, int bits, uint32_t *words, cudaStream_t s) {
    const int64_t nwords = n * bits / 32;            // the caller checks n * bits % 32 == 0
    pack_bits_kernel<<<(unsigned)((nwords + 255) / 256), 256, 0, s>>>(codes, n, bits, words, nwords);
    return cudaGetLastError();
}
cudaError_t launch_unpack_bits(const uint32_t *words, int64_t n, int bits, uint8_t *codes, cudaStream_t s) {
    unpack_bits_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(words, n, bits, codes);
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
