// validate_noalloc.cu -- q4_validate_noalloc: the fail-closed scale scan of
// q4_validate for callers that cannot allocate device memory.
//
// q4_validate needs a small device buffer for its NaN count, which the caller
// allocates.  Some callers cannot do that: a weight loader running inside a
// serving process whose device memory is owned by a pre-sized pool or arena,
// a plugin that is handed tensors but no allocator, or code that must not
// trigger cudaMalloc's implicit device synchronisation.  This variant keeps
// its scratch in a fixed array that lives in the library's own device memory
// for the life of the process, so it allocates nothing per call.
//
// Scratch layout (one copy per device): one partial count per chunk of
// CHUNK scale entries, then the total.  Every call overwrites the partials it
// uses and the total, so nothing has to be cleared between calls, but all
// calls share the one array: calls that overlap on the GPU (from two streams
// or two host threads) race on it and may report each other's counts.
#include <mutex>

#include "q4_internal.cuh"

namespace q4 {
namespace {

constexpr int CHUNK = 16384;                       // scale entries per block
constexpr int MAX_CHUNKS = Q4_VALIDATE_NOALLOC_MAX_CHUNKS;

// 128 KiB + 8 B per device, held until the process exits.
static __device__ __align__(256) unsigned long long g_noalloc_scratch[MAX_CHUNKS + 1];

// 1 if scale entry i of this tensor is a NaN/Inf encoding (same rules as
// q4_validate: E4M3FN 0x7f/0xff, E8M0 0xff, fp16 Inf/NaN in Q4_K/Q4_0 block
// headers and GPTQ/AWQ/logical scales).
__device__ __forceinline__ unsigned bad_entry(q4_fmt fmt, const uint8_t *p, int64_t i) {
    if (fmt == Q4_NVFP4 || fmt == Q4_NVFP4_SPLITHALF) return (p[i] & 0x7fu) == 0x7fu;
    if (fmt == Q4_MXFP4) return p[i] == 0xffu;
    uint32_t h;
    if (fmt == Q4_Q4K) {
        const uint8_t *q = p + (i >> 1) * 144 + 2 * (i & 1);
        h = q[0] | (q[1] << 8);
    } else if (fmt == Q4_Q40) {
        const uint8_t *q = p + i * 18;
        h = q[0] | (q[1] << 8);
    } else {
        h = reinterpret_cast<const uint16_t *>(p)[i];
    }
    return (h & 0x7c00u) == 0x7c00u;
}

// Block b counts chunk b and writes its partial (no atomics, no zeroing).
__global__ void __launch_bounds__(256) count_chunks(q4_fmt fmt, const uint8_t *__restrict__ p, int64_t count,
                                                    unsigned long long *__restrict__ scratch) {
    __shared__ unsigned int warp_sums[8];
    const int64_t base = (int64_t)blockIdx.x * CHUNK;
    unsigned int local = 0;
    for (int j = threadIdx.x; j < CHUNK; j += blockDim.x) {
        const int64_t i = base + j;
        if (i < count) local += bad_entry(fmt, p, i);
    }
    for (int off = 16; off >= 1; off >>= 1) local += __shfl_xor_sync(0xffffffffu, local, off);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = local;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int w = 0; w < 8; w++) s += warp_sums[w];
        scratch[blockIdx.x] = s;
    }
}

// One block sums the partials in a fixed order into scratch[MAX_CHUNKS].
__global__ void __launch_bounds__(1024) sum_chunks(int nchunks, unsigned long long *__restrict__ scratch) {
    __shared__ unsigned long long part[1024];
    unsigned long long s = 0;
    for (int c = threadIdx.x; c < nchunks; c += blockDim.x) s += scratch[c];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = 512; w >= 1; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) scratch[MAX_CHUNKS] = part[0];
}

// Device address of the scratch array, looked up once per device with that
// device current.  (In host code g_noalloc_scratch is only a host-side
// stand-in; a kernel must be given the address returned here.)
std::mutex g_setup_lock;
unsigned long long *g_scratch_addr[128];

cudaError_t scratch_for_current_device(unsigned long long **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_lock);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<unsigned long long *>(ptr);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace q4

using namespace q4;

extern "C" int q4_validate_noalloc(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux,
                                   int64_t N, int64_t K, int64_t *bad_count, void *stream) {
    // every host-side check of q4_validate (the same helper), then the scratch bound
    Tensor t;
    const int rc = make_tensor(fmt, W_packed, scales, aux, N, K, t);
    if (rc && rc != Q4_ESCALE2) return rc;
    int64_t count;
    const uint8_t *p;
    switch (fmt) {
    case Q4_NVFP4:
    case Q4_NVFP4_SPLITHALF: count = N * (K / 16); p = t.scales; break;
    case Q4_MXFP4: count = N * (K / 32); p = t.scales; break;
    case Q4_Q4K: count = N * (K / 256) * 2; p = t.w; break;      // d and dmin of every super-block
    case Q4_Q40: count = N * (K / 32); p = t.w; break;            // d of every block
    default: count = (K / t.group) * N; p = t.scales; break;      // GPTQ / AWQ / logical fp16 scales
    }
    // the fixed scratch bounds the problem: at most MAX_CHUNKS chunks of CHUNK entries
    if (count > (int64_t)Q4_VALIDATE_NOALLOC_MAX_CHUNKS * CHUNK) return Q4_EDIM;

    unsigned long long *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return Q4_ECUDA;
    cudaStream_t st = (cudaStream_t)stream;
    const int nchunks = (int)((count + CHUNK - 1) / CHUNK);
    count_chunks<<<nchunks, 256, 0, st>>>(fmt, p, count, scratch);
    sum_chunks<<<1, 1024, 0, st>>>(nchunks, scratch);
    if (cudaGetLastError() != cudaSuccess) return Q4_ECUDA;
    unsigned long long total = 0;
    if (cudaMemcpyAsync(&total, scratch + MAX_CHUNKS, sizeof(total), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return Q4_ECUDA;
    if (bad_count) *bad_count = (int64_t)total;
    if (total) return Q4_ENAN;
    return rc;                        // Q4_OK, or Q4_ESCALE2 for a bad NVFP4 scale2
}
