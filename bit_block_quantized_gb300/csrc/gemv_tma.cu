// gemv_tma.cu -- NVFP4 (and one-group MXFP4) decode-GEMV for batch 1..4, weights streamed into
// shared memory by the tensor-memory accelerator (TMA), dot products on the
// tensor cores (mma.sync m16n8k16, f16 x f16 -> f32).  One launch runs a
// chain of GEMV groups: the members of a group read the same x, and group
// g + 1 reads its x (and writes y) only after every member of the groups
// before it has written y, as if each group were its own launch.
//
// Why a TMA-fed kernel: at batch 1 the work is one pass over the packed
// weights, so the kernel must keep enough bytes in flight to cover the HBM
// latency (about 55 KB per SM at 7 TB/s) and must not lose the start and the
// end of each launch:
//   * one producer thread per CTA streams 16-row x 2048-k stages (16 KB of
//     payload + 2 KB of E4M3 scales, two tensor copies) into a ring of 3..8
//     stages.  It only reads weights, so it runs ahead across the group
//     boundaries of a chain: while the decode warps wait for the previous
//     group, the next group's weights are already landing;
//   * 8 consumer warps decode in registers: the hardware E2M1 convert gives
//     one f16x2 A register per payload byte, one f16x2 multiply by the E4M3
//     block scale makes it (e2m1 * e4m3) exactly ([MUS7] 7.1-7.2), x (scaled
//     by an exact power of two into f16) is the MMA's B, f32 accumulation,
//     x scale2 at the end.  Two CTAs per SM: the decode recipe sustains ~39
//     weights per SM clock on this GPU only with ~16 warps in flight;
//   * a chain's group boundary is a grid-wide barrier (a generation counter
//     in caller-owned memory, cooperative launch, bounded spin); a single
//     group needs none and is launched with programmatic dependent launch
//     (weights are read before the dependency wait, x and y after it).
//
// Shared-memory layout of a stage (1024-byte aligned, 128-byte swizzle):
//   payload: a 3-D box {128 bytes, 16 rows, 8 chunks of 256 k}; chunk c of
//            row r is the 128-byte line c*16 + r, whose 16-byte units are
//            permuted by XOR with (r & 7).  Warp w reads chunk w, lane
//            (g, t) the units 2t and 2t+1 (k = 64t .. 64t+63 of the chunk)
//            of rows g and g+8: a quarter-warp touches every bank once.
//   scales:  a 2-D box {128 bytes, 16 rows}; row r is line r (same swizzle),
//            lane (g, t) reads the 4 scale bytes of its 64 k.
// MXFP4 (one E8M0 scale per 32 k, [MUS7] 7.1's MX block) shares the payload
// layout; its scale rows (K/32 bytes) need not be 16-byte multiples, so no
// tensor map reads them: each lane loads the two scale bytes of its rows g
// and g+8 one stage ahead into registers.  A scale outside the range where
// every E2M1 multiple is an f16 number sends that warp's stage to the f32
// CUDA-core dot, which adds into the same partials.
// The staged x of warp w follows the same k order: entry
//   ((v*8 + j)*MT + m)*4 + t,  v = 2s + h,
//   = x[m][2048 s + 256 w + 64 t + 32 h + 4 j .. +3] * 2^e_m   (as f16).
#include <cuda.h>

#include "q4_internal.cuh"
#include "tma_map.cuh"

namespace q4 {
namespace {

__device__ int g_tma_error;
// Limit of the role waits and the chain's grid barrier, in SM clocks (the
// final drain of bulk copies keeps its own full limit).
__device__ long long g_tma_wait_limit = 1LL << 31;

#ifndef Q4_TMA_SMEM_KB
#define Q4_TMA_SMEM_KB 112
#endif
#ifndef Q4_TMA_CTAS_PER_SM
#define Q4_TMA_CTAS_PER_SM 2
#endif
#ifndef Q4_TMA_NACC
#define Q4_TMA_NACC 4
#endif
#ifndef Q4_TMA_CW
#define Q4_TMA_CW 8
#endif
#ifndef Q4_TMA_PREFETCH
#define Q4_TMA_PREFETCH 3
#endif
#ifndef Q4_TMA_L2_AHEAD
#define Q4_TMA_L2_AHEAD 0
#endif
constexpr int CW = Q4_TMA_CW;                  // consumer warps (a multiple of 8)
constexpr int THREADS = (CW + 1) * 32;         // + the producer warp
constexpr int KS = CW * 256;                   // k per ring stage = CW chunks of 256 k
constexpr int PAY_BYTES = 16 * KS / 2;         // 16 rows x 1024 payload bytes
constexpr int SC_BYTES = 16 * KS / 16;         // CW / 8 blocks of 16 rows x 128 scale bytes
constexpr int STAGE_BYTES = PAY_BYTES + SC_BYTES;
constexpr int MAX_STAGES = 8;
constexpr int MIN_STAGES = 3;
constexpr int PREFETCH_STAGES = Q4_TMA_PREFETCH;   // stages a CTA loads before its decode warps have staged x
constexpr int L2_AHEAD = Q4_TMA_L2_AHEAD;          // further stages it then only prefetches into L2
constexpr int MAXM = 8;                        // matrices per launch
constexpr int MAXP = 4;                        // groups per chain
constexpr size_t SMEM_CAP = Q4_TMA_SMEM_KB * 1024;   // 112 KB: two CTAs per SM
constexpr int NACC = Q4_TMA_NACC;
static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
static_assert(CW % 8 == 0, "scale blocks of 128 bytes (2048 k) per row");

struct Maps {
    CUtensorMap pay[MAXM];   // u8 {128, N, K/256}, strides {K/2, 128}: box {128, 16, 8}
    CUtensorMap sc[MAXM];    // u8 {K/16, N}, stride K/16: box {128, 16}
};

struct Args {
    float *y[MAXM];                 // [M][N_i]
    const uint8_t *mx_scales[MAXM]; // MXFP4 (a single group): E8M0 [N_i][K/32] of each member
    int64_t N[MAXM];
    float scale2[MAXM];
    int tile_start[MAXM];           // first 16-row tile of each member within its group
    const __nv_bfloat16 *x[MAXP];   // [M][K_p] of each group
    int K[MAXP];
    int nst[MAXP];                  // stages per tile = ceil(K_p / 2048)
    int ntiles[MAXP];               // tiles of each group
    int m0[MAXP + 1];               // first member of each group
    unsigned *sync;                 // {arrivals, generation}: the group barrier
    int ngroups;
    int M;
    int S;                          // ring stages
    int max_nst;
};

// MXFP4 scale byte b -> 2^(b-127) as an f16x2 pair, built from the exponent
// field alone: exact (and every E2M1 multiple an f16 number) for b - 127 in
// [-14, 13], the normal f16 powers; outside, `ok` clears and the stage takes
// the f32 path.
__device__ __forceinline__ uint32_t e8m0_h2(uint32_t b, bool &ok) {
    const uint32_t e = b & 255u;
    ok = ok && e - 113u <= 27u;
    const uint32_t h = (e - 112u) << 10;
    return h | (h << 16);
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// Weight copies carry an L2 evict-first policy: they are read exactly once,
// and should not push the activations and outputs out of L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, uint32_t bar,
                                       uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(pol)
        : "memory");
}
// L2-only prefetch of a tile: no shared memory, no completion to wait for.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(c0), "r"(c1),
                 "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar,
                                       uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar), "l"(pol)
        : "memory");
}

// Bounded mbarrier wait: gives up after the role-wait limit (~1 s of SM
// clocks unless q4_set_wait_limit shortened it; records Q4_ETIMEOUT and
// raises the CTA's abort flag), or at once when another role has raised the
// flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64(), limit = g_tma_wait_limit;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            atomicExch(&g_tma_error, Q4_ETIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier between two groups of a chain, called by one thread per
// CTA after a CTA barrier that orders the CTA's y stores before it.  The
// generation word makes it reusable across launches and graph replays: the
// last CTA to arrive resets the count and bumps the generation, the others
// wait for the bump.  The spin gives up after ~1 s (Q4_ETIMEOUT, abort flag).
__device__ void grid_barrier(unsigned *sync, volatile int *abort_flag) {
    unsigned *count = sync, *gen = sync + 1;
    __threadfence();
    const unsigned my_gen = ld_acquire(gen);
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
        atomicExch(count, 0u);
        __threadfence();
        atomicAdd(gen, 1u);
        return;
    }
    const long long t0 = clock64(), limit = g_tma_wait_limit;
    while (ld_acquire(gen) == my_gen) {
        if (*abort_flag) return;
        if (clock64() - t0 > limit) {
            atomicExch(&g_tma_error, Q4_ETIMEOUT);
            *abort_flag = 1;
            return;
        }
        __nanosleep(64);
    }
    __threadfence();
}


// Four bf16 values (two words) times an exact power of two -> two f16x2
// words; `ok` stays true only if every value survives the f16 rounding.
__device__ __forceinline__ uint2 bf16x4_to_f16(uint2 v, float scale, bool &ok) {
    const float f0 = __uint_as_float(v.x << 16) * scale, f1 = __uint_as_float(v.x & 0xffff0000u) * scale;
    const float f2 = __uint_as_float(v.y << 16) * scale, f3 = __uint_as_float(v.y & 0xffff0000u) * scale;
    const __half2 h01 = __floats2half2_rn(f0, f1), h23 = __floats2half2_rn(f2, f3);
    const float2 c01 = __half22float2(h01), c23 = __half22float2(h23);
    ok = ok && c01.x == f0 && c01.y == f1 && c23.x == f2 && c23.y == f3;
    return make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
}

// The x slice of consumer warp w (chunk w of every stage) as exactly-scaled
// f16 B fragments in the layout above.  Lane l serves column m = l % MT.
// Staging sits on the critical path of every launch (the decode warps wait
// for it once the launch before has finished), so when a lane's share is at
// most XR runs of 8 k it is one round trip: all loads issued at once into
// registers, the column maximum reduced over the lanes, then converted and
// stored.  Larger shares (batch 4 at large K) take two passes through shared
// memory.  The scale 2^(12-e) (e the largest exponent) keeps |x| < 2^13; a
// value that does not survive the f16 rounding sends the warp to the f32
// CUDA-core path.  Chunks past K are zeros (their weights are never read).
constexpr int XR = 8;

__device__ __forceinline__ uint32_t absmax8(uint4 v) {   // packed |bf16| maximum (bit patterns order like values)
    return __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu), __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu));
}

// Column scale from the packed maximum: x * 2^(12-e) keeps |x| < 2^13 in f16.
template <int MT>
__device__ __forceinline__ bool column_scale(uint32_t mx2, float &scale, float (&inv)[MT]) {
    const uint32_t mxb = (mx2 & 0xffffu) > (mx2 >> 16) ? (mx2 & 0xffffu) : (mx2 >> 16);
    float amax = __uint_as_float(mxb << 16);
#pragma unroll
    for (int off = MT; off < 32; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float iv = 1.0f;
    bool exact = true;
    scale = 1.0f;
    if (amax > 0.0f) {
        const int ex = (int)((__float_as_uint(amax) >> 23) & 255u) - 127;
        if (ex < -100 || ex > 100)
            exact = false;
        else {
            scale = __uint_as_float((uint32_t)(127 + 12 - ex) << 23);
            iv = __uint_as_float((uint32_t)(127 - 12 + ex) << 23);
        }
    }
#pragma unroll
    for (int mm = 0; mm < MT; mm++) inv[mm] = __shfl_sync(0xffffffffu, iv, mm);   // lane mm holds column mm
    return exact;
}

template <int MT>
__device__ __forceinline__ bool stage_x(const __nv_bfloat16 *__restrict__ x, int K, int M, int nst, int w, int lane,
                                        uint2 *xs, float (&inv)[MT]) {
    constexpr int LPC = 32 / MT;
    const int m = lane % MT;
    const bool mv = m < M;
    const int nrun = nst * 32;                  // 8-k runs of the warp's k set
    const __nv_bfloat16 *row = x + (int64_t)(mv ? m : 0) * K;
    uint32_t mx2 = 0;
    float scale;
    bool exact;
    if (nrun <= XR * LPC) {
        uint4 v[XR];
#pragma unroll
        for (int i = 0; i < XR; i++) {
            const int r = lane / MT + i * LPC;
            const int k = (r >> 5) * KS + w * 256 + (r & 31) * 8;
            // L2-coherent load: in a chain, x may have been written by an earlier group of this launch
            v[i] = (r < nrun && mv && k < K) ? __ldcg(reinterpret_cast<const uint4 *>(row + k))
                                             : make_uint4(0u, 0u, 0u, 0u);
            mx2 = __vmaxu2(mx2, absmax8(v[i]));
        }
        exact = column_scale<MT>(mx2, scale, inv);
#pragma unroll
        for (int i = 0; i < XR; i++) {
            const int r = lane / MT + i * LPC;
            if (r < nrun) {
                const int s = r >> 5, rr = r & 31;
                const int t = rr >> 3, h = (rr >> 2) & 1, j0 = (rr & 3) * 2, vb = 2 * s + h;
                xs[((vb * 8 + j0) * MT + m) * 4 + t] = bf16x4_to_f16(make_uint2(v[i].x, v[i].y), scale, exact);
                xs[((vb * 8 + j0 + 1) * MT + m) * 4 + t] = bf16x4_to_f16(make_uint2(v[i].z, v[i].w), scale, exact);
            }
        }
    } else {
#pragma unroll 4
        for (int r = lane / MT; r < nrun; r += LPC) {
            const int s = r >> 5, rr = r & 31;
            const int k = s * KS + w * 256 + rr * 8;
            const uint4 v = (mv && k < K) ? __ldcg(reinterpret_cast<const uint4 *>(row + k))
                                          : make_uint4(0u, 0u, 0u, 0u);
            mx2 = __vmaxu2(mx2, absmax8(v));
            const int t = rr >> 3, h = (rr >> 2) & 1, j0 = (rr & 3) * 2, vb = 2 * s + h;
            xs[((vb * 8 + j0) * MT + m) * 4 + t] = make_uint2(v.x, v.y);
            xs[((vb * 8 + j0 + 1) * MT + m) * 4 + t] = make_uint2(v.z, v.w);
        }
        exact = column_scale<MT>(mx2, scale, inv);
#pragma unroll 4
        for (int r = lane / MT; r < nrun; r += LPC) {
            const int s = r >> 5, rr = r & 31;
            const int t = rr >> 3, h = (rr >> 2) & 1, j0 = (rr & 3) * 2, vb = 2 * s + h;
            uint2 *e0 = xs + ((vb * 8 + j0) * MT + m) * 4 + t, *e1 = xs + ((vb * 8 + j0 + 1) * MT + m) * 4 + t;
            const uint2 c0 = bf16x4_to_f16(*e0, scale, exact), c1 = bf16x4_to_f16(*e1, scale, exact);
            *e0 = c0;
            *e1 = c1;
        }
    }
    exact = __all_sync(0xffffffffu, exact);
    __syncwarp();
    return exact;
}

// f32 CUDA-core dot of one warp's chunk (16 rows x 256 k) of a stage, used
// only when the activations' dynamic range is too wide for exact f16
// staging.  Adds the 16 x MT partial sums into `rw` (lane 0).
template <int MT, int FMT>
__device__ __noinline__ void chunk_f32(uint32_t stg, const __nv_bfloat16 *__restrict__ x, int K, int M, int k0, int w,
                                       int lane, float *rw, const uint8_t *__restrict__ mxs, int64_t n0, int64_t N) {
    for (int rr = 0; rr < 16; rr++) {
        const uint32_t word = lds32(stg + (uint32_t)((w * 16 + rr) * 128) +
                                    ((uint32_t)((lane >> 2) ^ (rr & 7)) << 4) + ((uint32_t)(lane & 3) << 2));
        float sc;
        if (FMT == Q4_NVFP4) {
            const uint32_t sb = lds8(stg + PAY_BYTES + (uint32_t)((w >> 3) * 2048 + rr * 128) +
                                     ((uint32_t)((w & 7) ^ (rr & 7)) << 4) + (uint32_t)(lane >> 1));
            sc = e4m3_f32(sb);
        } else {                 // rows past N carry zero payload: any scale
            sc = n0 + rr < N ? e8m0_f32(__ldg(mxs + (n0 + rr) * (K >> 5) + ((k0 + lane * 8) >> 5))) : 0.0f;
        }
        for (int m = 0; m < MT; m++) {
            float acc = 0.0f;
            if (m < M) {
                const __nv_bfloat16 *xr = x + (int64_t)m * K + k0 + lane * 8;
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const float2 v = e2m1x2_f32((word >> (4 * i)) & 0xffu);
                    acc = fmaf(v.x * sc, __bfloat162float(__ldcg(xr + i)), acc);
                    acc = fmaf(v.y * sc, __bfloat162float(__ldcg(xr + i + 1)), acc);
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) rw[rr * MT + m] += acc;
        }
    }
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory"); }

template <int MT, int FMT>
__global__ void __launch_bounds__(THREADS, Q4_TMA_CTAS_PER_SM)
    gemv_tma_fp4(const __grid_constant__ Maps maps, const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = a.S;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + (size_t)S * STAGE_BYTES);
    uint64_t *empty = full + MAX_STAGES;
    int *abort_s = reinterpret_cast<int *>(empty + MAX_STAGES);
    float *red = reinterpret_cast<float *>(abort_s + 4);               // [2][CW][16][MT]
    uint2 *xs_all = reinterpret_cast<uint2 *>(red + 2 * CW * 16 * MT);  // [CW][max_nst*2][8][MT][4]
    volatile int *abort_flag = abort_s;
    volatile int *x_staged = abort_s + 1;   // decode warps that have staged the first group's x

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&full[s], 1);      // the producer's arrive + the stage's bytes
            mbar_init(&empty[s], CW);    // one arrive per consumer warp
        }
        *abort_s = 0;
        *x_staged = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Let the next launch in the stream start its launch work (its producer
    // only reads weights before its own dependency wait).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == CW) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t ring = smem_u32(base);
            const uint64_t pol = evict_first_policy();
            int issued = 0, slot = 0, phase = 0;
            bool stop = false;
            for (int p = 0; p < a.ngroups && !stop; p++) {
                const int ntiles = a.ntiles[p], nst = a.nst[p], m_end = a.m0[p + 1];
                int member = a.m0[p];
                for (int tile = (int)blockIdx.x; tile < ntiles && !stop; tile += (int)gridDim.x) {
                    while (member + 1 < m_end && tile >= a.tile_start[member + 1]) member++;
                    const int row0 = (tile - a.tile_start[member]) * 16;
                    for (int st = 0; st < nst; st++) {
                        if (issued >= S && !wait_or_abort(&empty[slot], (uint32_t)(phase ^ 1), abort_flag)) {
                            stop = true;
                            break;
                        }
                        const uint32_t dst = ring + (uint32_t)(slot * STAGE_BYTES), bar = smem_u32(&full[slot]);
                        mbar_arrive_expect_tx(&full[slot], FMT == Q4_NVFP4 ? STAGE_BYTES : PAY_BYTES);
                        tma_3d(dst, &maps.pay[member], 0, row0, st * (KS / 256), bar, pol);
                        if (FMT == Q4_NVFP4) {
#pragma unroll
                            for (int sb = 0; sb < CW / 8; sb++)   // 128-byte scale boxes: the swizzle span
                                tma_2d(dst + PAY_BYTES + sb * 2048, &maps.sc[member], st * (KS / 16) + sb * 128, row0,
                                       bar, pol);
                        }
                        issued++;
                        if (++slot == S) { slot = 0; phase ^= 1; }
                        if (issued == PREFETCH_STAGES) {
                            // The next stages of this CTA's list into L2 only: their bytes move
                            // while the launch before finishes, without queueing in front of x.
                            int pt = tile, pst = st + 1, pm = member;
                            for (int q = 0; q < L2_AHEAD; q++, pst++) {
                                if (pst == nst) {
                                    pst = 0;
                                    pt += (int)gridDim.x;
                                    if (pt >= ntiles) break;
                                    while (pm + 1 < m_end && pt >= a.tile_start[pm + 1]) pm++;
                                }
                                const int prow0 = (pt - a.tile_start[pm]) * 16;
                                tma_prefetch_3d(&maps.pay[pm], 0, prow0, pst * (KS / 256));
                                if (FMT == Q4_NVFP4)
                                    for (int sb = 0; sb < CW / 8; sb++)
                                        tma_prefetch_2d(&maps.sc[pm], pst * (KS / 16) + sb * 128, prow0);
                            }
                            // Hold further copies until the decode warps have read x (or ~0.5 s,
                            // or an abort): a deeper prefetch queues their x loads behind this
                            // launch's weight stream while they cannot start without x.
                            const long long t0 = clock64();
                            while (*x_staged < CW && !*abort_flag && clock64() - t0 < (1LL << 30)) __nanosleep(64);
                        }
                    }
                }
            }
            // Every copy this thread issued has landed before the CTA may exit.
            for (int q = issued > S ? issued - S : 0; q < issued; q++)
                if (!mbar_wait_bounded(&full[q % S], (uint32_t)((q / S) & 1)))
                    atomicExch(&g_tma_error, Q4_ETIMEOUT);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // Warm L2 with this warp's slice of the first group's x while the launch
    // before may still be running: a prefetch only fills L2, the coherence
    // point, so a later write to x by that launch is still what the loads
    // after the dependency wait see.  Lane l covers 128-byte line l & 3 of
    // the warp's 512-byte run in stage l >> 2.
    {
        const int K0 = a.K[0];
        for (int m = 0; m < a.M; m++)
            for (int r = lane; r < a.nst[0] * 4; r += 32) {
                const int k = (r >> 2) * KS + warp * 256 + (r & 3) * 64;
                if (k < K0) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.x[0] + (int64_t)m * K0 + k));
            }
    }
    const int g = lane >> 2, tt = lane & 3;
    // MXFP4: lane l's 4 scale bytes of the warp's chunk in stage `st_` of tile
    // `tile_`: row l / 2, bytes 4 (l & 1) .. +3 of the chunk's 8 (scale byte j
    // of row n at n * K/32 + j; aligned since K % 256 == 0).  Weights: read
    // before the dependency wait like the payload.
    const int64_t mx_rs = a.K[0] >> 5;
    auto mx_word = [&](int tile_, int st_) -> uint32_t {
        if (FMT != Q4_MXFP4 || tile_ >= a.ntiles[0]) return 0x7f7f7f7fu;
        int m = 0;                       // the member holding tile_ (an MXFP4 launch is one group)
#pragma unroll
        for (int i = 1; i < MAXM; i++) m += (i < a.m0[1] && tile_ >= a.tile_start[i]) ? 1 : 0;
        const int64_t row = (int64_t)(tile_ - a.tile_start[m]) * 16 + (lane >> 1);
        const int col = st_ * 64 + warp * 8 + (lane & 1) * 4;
        if (col >= (int)mx_rs || row >= a.N[m]) return 0x7f7f7f7fu;
        return __ldg(reinterpret_cast<const unsigned *>(a.mx_scales[m] + row * mx_rs + col));   // 2^0 above
    };
    uint32_t mxv = mx_word((int)blockIdx.x, 0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    uint2 *xs = xs_all + (size_t)warp * a.max_nst * 2 * 8 * MT * 4;
    const uint32_t ring = smem_u32(base);
    // payload byte offsets of this lane's two units in rows g and g+8 of chunk `warp`
    const uint32_t offA0 = (uint32_t)((warp * 16 + g) * 128) + ((uint32_t)((2 * tt) ^ g) << 4);
    const uint32_t offA1 = (uint32_t)((warp * 16 + g) * 128) + ((uint32_t)((2 * tt + 1) ^ g) << 4);
    const uint32_t offS = (uint32_t)PAY_BYTES + (uint32_t)((warp >> 3) * 2048 + g * 128) +
                          ((uint32_t)((warp & 7) ^ g) << 4) + 4 * tt;
    constexpr uint32_t ROW8 = 8 * 128;   // rows g+8: same swizzle phase, 8 lines further
    const int mlane = g < a.M ? g : 0;

    float dacc[NACC][4];
#pragma unroll
    for (int i = 0; i < NACC; i++) dacc[i][0] = dacc[i][1] = dacc[i][2] = dacc[i][3] = 0.0f;
    int par = 0, slot = 0, phase = 0;
    uint32_t stg = ring;
    for (int p = 0; p < a.ngroups; p++) {
        if (p > 0) {
            // every CTA's y of the groups before this one is written before x is read
            consumer_sync();
            if (threadIdx.x == 0) grid_barrier(a.sync, abort_flag);
            consumer_sync();
        }
        const __nv_bfloat16 *x = a.x[p];
        const int K = a.K[p], nst = a.nst[p], ntiles = a.ntiles[p], m_end = a.m0[p + 1];
        float inv[MT];
        const bool exact = stage_x<MT>(x, K, a.M, nst, warp, lane, xs, inv);
        if (p == 0 && lane == 0) atomicAdd((int *)x_staged, 1);
        const uint2 *xbase = xs + mlane * 4 + tt;
        int mb = a.m0[p];
        for (int tile = (int)blockIdx.x; tile < ntiles; tile += (int)gridDim.x) {
            while (mb + 1 < m_end && tile >= a.tile_start[mb + 1]) mb++;   // this tile's member
            float *rw = red + (par * CW + warp) * 16 * MT;
            if (!exact || FMT == Q4_MXFP4) {     // MXFP4 stages may add f32 partials
                for (int e = lane; e < 16 * MT; e += 32) rw[e] = 0.0f;
                __syncwarp();
            }
            const uint2 *xb = xbase;
            for (int st = 0, k0 = warp * 256; st < nst; st++, k0 += KS) {
                const uint32_t mxcur = mxv;
                if (FMT == Q4_MXFP4)             // the next stage's scale word, one stage ahead
                    mxv = st + 1 < nst ? mx_word(tile, st + 1) : mx_word(tile + (int)gridDim.x, 0);
                const bool ok = wait_or_abort(&full[slot], (uint32_t)phase, abort_flag);
                if (ok && k0 < K) {
                    bool sok = true;
                    uint32_t mxs2[2][2];         // MXFP4: [h][row g / g+8] scale as f16x2
                    if (FMT == Q4_MXFP4) {
                        // the warp's 16 x 8 scale bytes through the slot's unused scale area
                        // (rows 68 bytes apart: the lanes' 2-byte reads hit distinct banks)
                        sts32(stg + PAY_BYTES + (uint32_t)((lane >> 1) * 68 + warp * 8 + (lane & 1) * 4), mxcur);
                        __syncwarp();
                        const uint32_t ra = lds16(stg + PAY_BYTES + (uint32_t)(g * 68 + warp * 8 + 2 * tt));
                        const uint32_t rb = lds16(stg + PAY_BYTES + (uint32_t)((g + 8) * 68 + warp * 8 + 2 * tt));
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            mxs2[h][0] = e8m0_h2(ra >> (8 * h), sok);
                            mxs2[h][1] = e8m0_h2(rb >> (8 * h), sok);
                        }
                        sok = __all_sync(0xffffffffu, sok);
                    }
                    if (exact && sok) {
                        const uint4 pa[2] = {lds128(stg + offA0), lds128(stg + offA1)};
                        const uint4 pb[2] = {lds128(stg + offA0 + ROW8), lds128(stg + offA1 + ROW8)};
                        uint32_t sa = 0, sb = 0;
                        if (FMT == Q4_NVFP4) sa = lds32(stg + offS), sb = lds32(stg + offS + ROW8);
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            uint32_t sca[2], scb[2];
                            if (FMT == Q4_NVFP4) {
                                uint32_t ha, hb;
                                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(ha) : "h"((uint16_t)(sa >> (16 * h))));
                                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hb) : "h"((uint16_t)(sb >> (16 * h))));
                                sca[0] = prmt(ha, ha, 0x1010u), sca[1] = prmt(ha, ha, 0x3232u);
                                scb[0] = prmt(hb, hb, 0x1010u), scb[1] = prmt(hb, hb, 0x3232u);
                            } else {                 // one scale per 32 k: the whole unit
                                sca[0] = sca[1] = mxs2[h][0];
                                scb[0] = scb[1] = mxs2[h][1];
                            }
                            const uint32_t wa[4] = {pa[h].x, pa[h].y, pa[h].z, pa[h].w};
                            const uint32_t wb[4] = {pb[h].x, pb[h].y, pb[h].z, pb[h].w};
                            const uint2 *xh = xb + h * 8 * MT * 4;
#pragma unroll
                            for (int wd = 0; wd < 4; wd++) {
                                uint32_t av[4], cv[4];
                                e2m1x8_h2(wa[wd], av[0], av[1], av[2], av[3]);
                                e2m1x8_h2(wb[wd], cv[0], cv[1], cv[2], cv[3]);
#pragma unroll
                                for (int i = 0; i < 4; i++) {
                                    av[i] = hmul2_u32(av[i], sca[wd >> 1]);
                                    cv[i] = hmul2_u32(cv[i], scb[wd >> 1]);
                                }
                                // lanes g >= M read column 0's x: MMA columns >= M are never stored
                                const uint2 bA = xh[(2 * wd) * MT * 4], bB = xh[(2 * wd + 1) * MT * 4];
                                mma16816(dacc[(2 * wd) % NACC], av[0], cv[0], av[1], cv[1], bA.x, bA.y);
                                mma16816(dacc[(2 * wd + 1) % NACC], av[2], cv[2], av[3], cv[3], bB.x, bB.y);
                            }
                        }
                    } else {
                        chunk_f32<MT, FMT>(stg, x, K, a.M, k0, warp, lane, rw, a.mx_scales[mb],
                                           (int64_t)(tile - a.tile_start[mb]) * 16, a.N[mb]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
                if (++slot == S) { slot = 0; phase ^= 1; stg = ring; } else stg += STAGE_BYTES;
                xb += 2 * 8 * MT * 4;
            }

            // ---- end of tile: warp partials -> shared, one consumer barrier, fixed-order sum
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < NACC; i++) {
                d[0] += dacc[i][0]; d[1] += dacc[i][1]; d[2] += dacc[i][2]; d[3] += dacc[i][3];
                dacc[i][0] = dacc[i][1] = dacc[i][2] = dacc[i][3] = 0.0f;
            }
            if (exact && FMT == Q4_NVFP4) {
#pragma unroll
                for (int mm = 0; mm < MT; mm++) {
                    if (mm == 2 * tt) { rw[g * MT + mm] = d[0] * inv[mm]; rw[(g + 8) * MT + mm] = d[2] * inv[mm]; }
                    if (mm == 2 * tt + 1) { rw[g * MT + mm] = d[1] * inv[mm]; rw[(g + 8) * MT + mm] = d[3] * inv[mm]; }
                }
            } else if (exact) {                  // MXFP4: add to the f32 stages' partials
                __syncwarp();
#pragma unroll
                for (int mm = 0; mm < MT; mm++) {
                    if (mm == 2 * tt) { rw[g * MT + mm] += d[0] * inv[mm]; rw[(g + 8) * MT + mm] += d[2] * inv[mm]; }
                    if (mm == 2 * tt + 1) { rw[g * MT + mm] += d[1] * inv[mm]; rw[(g + 8) * MT + mm] += d[3] * inv[mm]; }
                }
            }
            consumer_sync();
            const float *rt = red + par * CW * 16 * MT;
            par ^= 1;
            const int64_t Np = a.N[mb];
            const int64_t n0 = (int64_t)(tile - a.tile_start[mb]) * 16;
            float *yp = a.y[mb];
            const float s2 = a.scale2[mb];
            for (int e = threadIdx.x; e < 16 * MT; e += CW * 32) {
                const int rr = e / MT, m = e % MT;
                const int64_t n = n0 + rr;
                if (n < Np && m < a.M) {
                    float sum = 0.0f;
                    for (int w = 0; w < CW; w++) sum += rt[w * 16 * MT + e];
                    yp[(int64_t)m * Np + n] = sum * s2;
                }
            }
        }
    }
}

int mt_for(int64_t M) { return M == 1 ? 1 : (M == 2 ? 2 : 4); }

size_t fixed_smem(int64_t max_K, int mt) {
    const int64_t nst = (max_K + KS - 1) / KS;
    return 1024                                          // alignment slack
           + 2 * MAX_STAGES * sizeof(uint64_t) + 16       // barriers + abort word
           + 2 * (size_t)CW * 16 * mt * sizeof(float)     // partials (double buffered)
           + (size_t)CW * nst * 2 * 8 * mt * 4 * sizeof(uint2);
}

int stages_for(int64_t max_K, int mt) {
    const size_t f = fixed_smem(max_K, mt);
    if (f >= SMEM_CAP) return 0;
    const int s = (int)((SMEM_CAP - f) / STAGE_BYTES);
    return s > MAX_STAGES ? MAX_STAGES : s;
}

// Payload map: the rows of 128-byte chunks viewed as {128 bytes, N rows, K/256
// chunks}, so one box lands chunk-major and the swizzle separates the rows.
bool encode_payload(CUtensorMap *map, const Tensor &t) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)t.N, (cuuint64_t)(t.K / 256)};
    const cuuint64_t strides[2] = {(cuuint64_t)(t.K / 2), 128};
    const cuuint32_t box[3] = {128, 16, KS / 256};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(t.w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_scales(CUtensorMap *map, const Tensor &t) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(t.K / 16), (cuuint64_t)t.N};
    const cuuint64_t strides[1] = {(cuuint64_t)(t.K / 16)};
    const cuuint32_t box[2] = {128, 16};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(t.scales), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs that can be resident at once (a chain's group barrier waits on all of them).
template <typename Kern> int resident_ctas(Kern kern, size_t smem) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, THREADS, smem) != cudaSuccess || b < 1) b = 1;
    if (b > Q4_TMA_CTAS_PER_SM) b = Q4_TMA_CTAS_PER_SM;
    return b * sm_count();
}

template <int MT, int FMT>
cudaError_t run(const Maps &maps, const Args &args, int max_tiles, size_t smem, cudaStream_t s) {
    auto kern = gemv_tma_fp4<MT, FMT>;
    static bool attr_set[64] = {};
    static int grid_cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_CAP);
        if (e != cudaSuccess) return e;
        grid_cache[dev & 63] = resident_ctas(kern, SMEM_CAP);   // smem only shrinks below the cap
        attr_set[dev & 63] = true;
    }
    int grid = grid_cache[dev & 63];
    if (grid > max_tiles) grid = max_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = args.ngroups > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, maps, args);
}

}  // namespace

// Eligible: NVFP4 with bf16 x, K % 256 == 0, batch 1..4, and at least
// MIN_STAGES ring stages beside the staged x in 112 KB of shared memory.
bool gemv_tma_eligible(const Tensor &t, int64_t M) {
    if ((t.fmt != Q4_NVFP4 && t.fmt != Q4_MXFP4) || M < 1 || M > 4 || t.K % 256 != 0 || t.K > (1LL << 30) ||
        t.N > (1LL << 31))
        return false;
    if ((((uintptr_t)t.w | (uintptr_t)t.scales) & 15) != 0) return false;
    return stages_for(t.K, mt_for(M)) >= MIN_STAGES && encode_fn() != nullptr;
}

// A chain of GEMV groups in one launch: group p holds members
// [first[p], first[p+1]) of ts/ys, all eligible and sharing K; its x is xs[p].
bool gemv_tma_chain_fits(const Tensor *ts, const int *first, int ngroups, int64_t M) {
    if (ngroups < 1 || ngroups > MAXP || first[0] != 0 || first[ngroups] > MAXM) return false;
    int64_t max_K = 0;
    for (int p = 0; p < ngroups; p++) {
        if (first[p + 1] <= first[p]) return false;
        for (int i = first[p]; i < first[p + 1]; i++)
            if (!gemv_tma_eligible(ts[i], M) || ts[i].K != ts[first[p]].K) return false;
        // one format per launch (the kernel is instantiated per format); MXFP4 as a single group only
        for (int i = first[p]; i < first[p + 1]; i++)
            if (ts[i].fmt != ts[0].fmt) return false;
        if (ts[0].fmt == Q4_MXFP4 && ngroups > 1) return false;
        max_K = ts[first[p]].K > max_K ? ts[first[p]].K : max_K;
    }
    return stages_for(max_K, mt_for(M)) >= MIN_STAGES;
}

cudaError_t launch_gemv_tma_chain(const Tensor *ts, const void *const *xs, float *const *ys, const int *first,
                                  int ngroups, int64_t M, unsigned *sync, cudaStream_t s) {
    if (!gemv_tma_chain_fits(ts, first, ngroups, M) || (ngroups > 1 && !sync)) return cudaErrorInvalidValue;
    Maps maps;
    Args args = {};
    args.ngroups = ngroups;
    args.M = (int)M;
    args.sync = sync;
    int64_t max_K = 0;
    int max_tiles = 1;
    for (int p = 0; p < ngroups; p++) {
        args.x[p] = (const __nv_bfloat16 *)xs[p];
        args.K[p] = (int)ts[first[p]].K;
        args.nst[p] = (int)((ts[first[p]].K + KS - 1) / KS);
        args.m0[p] = first[p];
        args.max_nst = args.nst[p] > args.max_nst ? args.nst[p] : args.max_nst;
        max_K = ts[first[p]].K > max_K ? ts[first[p]].K : max_K;
        int tiles = 0;
        for (int i = first[p]; i < first[p + 1]; i++) {
            if (!encode_payload(&maps.pay[i], ts[i])) return cudaErrorInvalidValue;
            if (ts[i].fmt == Q4_NVFP4) {
                if (!encode_scales(&maps.sc[i], ts[i])) return cudaErrorInvalidValue;
            } else {
                maps.sc[i] = maps.pay[i];                 // never read: MXFP4 scales come through mx_scales
                args.mx_scales[i] = ts[i].scales;
            }
            args.y[i] = ys[i];
            args.N[i] = ts[i].N;
            args.scale2[i] = ts[i].scale2;
            args.tile_start[i] = tiles;
            tiles += (int)((ts[i].N + 15) / 16);
        }
        args.ntiles[p] = tiles;
        max_tiles = tiles > max_tiles ? tiles : max_tiles;
    }
    args.m0[ngroups] = first[ngroups];
    for (int i = first[ngroups]; i < MAXM; i++) maps.pay[i] = maps.sc[i] = maps.pay[0];   // never read
    const int mt = mt_for(M);
    args.S = stages_for(max_K, mt);
    if (args.S < MIN_STAGES) return cudaErrorInvalidValue;
    const size_t smem = fixed_smem(max_K, mt) + (size_t)args.S * STAGE_BYTES;
    if (ts[0].fmt == Q4_MXFP4) {
        if (mt == 1) return run<1, Q4_MXFP4>(maps, args, max_tiles, smem, s);
        if (mt == 2) return run<2, Q4_MXFP4>(maps, args, max_tiles, smem, s);
        return run<4, Q4_MXFP4>(maps, args, max_tiles, smem, s);
    }
    if (mt == 1) return run<1, Q4_NVFP4>(maps, args, max_tiles, smem, s);
    if (mt == 2) return run<2, Q4_NVFP4>(maps, args, max_tiles, smem, s);
    return run<4, Q4_NVFP4>(maps, args, max_tiles, smem, s);
}

// Several NVFP4 GEMVs that read the same x and share K and M, in one launch
// (count <= 8, each eligible on its own).
cudaError_t launch_gemv_tma_group(const Tensor *ts, const void *x, float *const *ys, int count, int64_t M,
                                  cudaStream_t s) {
    const int first[2] = {0, count};
    return launch_gemv_tma_chain(ts, &x, ys, first, 1, M, nullptr, s);
}

cudaError_t launch_gemv_tma(const Tensor &t, const void *x, float *y, int64_t M, cudaStream_t s) {
    return launch_gemv_tma_group(&t, x, &y, 1, M, s);
}

int gemv_tma_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tma_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_tma_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

int gemv_tma_set_wait_limit(long long cycles) {
    return cudaMemcpyToSymbol(g_tma_wait_limit, &cycles, sizeof(cycles)) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

}  // namespace q4
