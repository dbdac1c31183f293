// gemv_gptq_tc.cu -- GPTQ decode-GEMV on the tensor cores, weights streamed
// by tensor TMA ([BPA] "Real layouts compared": GPTQ qweight int32 [K/8][N]
// packed along K, k = 8r + j in bits 4j of word (r, n); fp16 scales
// [K/G][N]; qzeros int32 [K/G][N/8] packed along N, slot n % 8, stored as
// zero - 1; w = s * (q - z); group size 128 without act-order).
//
// mma.sync.m16n8k16 (f16 x f16 -> f32) with the WEIGHTS as A: the MMA's 16
// rows are 16 output columns of W (row g is column 2g, row g + 8 column
// 2g + 1 of the warp's 16, so one 8-byte shared load gives a lane both
// columns' words), its k16 is two word rows.  Lane (g, t) needs k = 2t, 2t+1
// and 2t+8, 2t+9: byte t of each word.  One byte permute copies byte t into
// both halves of a register, one LOP3 keeps the low nibble in the low half
// and the high nibble four bits up in the high half and ORs the f16 exponent
// of 1024, so the halves read 1024 + q_even and 1024 + 16 q_odd; one HSUB2
// of 1024 + z and 1024 + 16 z leaves q - z and 16 (q - z) exactly.  The
// odd-k x values are staged divided by 16 to match.  x fills B: the n8
// columns hold the f16 hi and lo terms of up to four batch rows (column
// 2m + h), so each lane's two D columns are one batch row's hi and lo.
// Each 128-k group (one ring stage) gets a fresh accumulator and the group
// epilogue multiplies by the columns' fp16 scales.
//
// A CTA owns 128 columns (warp w: columns 16w .. 16w+15) and a range of
// whole groups; the CTAs of a cluster split K and add their partial rows in
// rank order through distributed shared memory, so repeated calls agree bit
// for bit.  Roles: warp 8 streams the stages (TMA box 16 word rows x 128
// words, plus the group's scales and zero words by bulk copy); warps 0-7
// stage x, then decode and multiply.  Two CTAs fit on an SM.  Every wait is
// bounded (~1 s): a timeout records Q4_ETIMEOUT, stops the roles, waits for
// issued copies and returns.
#include <cooperative_groups.h>

#include <mutex>

#include "q4_internal.cuh"
#include "tc_gemv_common.cuh"
#include "tma_map.cuh"

namespace q4 {

__device__ int g_gptq_tc_error;

namespace {

namespace cg = cooperative_groups;
using namespace tc;

constexpr int GT_COLS = 128;                   // columns per CTA
constexpr int GT_G = 128;                      // group size = k per stage
constexpr int GT_ROWS = GT_G / 8;              // word rows per stage
constexpr int GT_WARPS = 8;                    // decode warps, 16 columns each
constexpr int GT_THREADS = (GT_WARPS + 1) * 32;
constexpr int GT_NS = 6;                       // ring stages
constexpr int W_BYTES = GT_ROWS * GT_COLS * 4; // 8 KB of weights per stage
constexpr int S_OFF = W_BYTES, S_BYTES = GT_COLS * 2;        // the group's fp16 scales
constexpr int Z_OFF = S_OFF + S_BYTES, Z_BYTES = GT_COLS / 2; // the group's zero words
constexpr int STAGE = 9 * 1024;
constexpr int MAXS = 8;                        // cluster ranks over K (the portable cluster size)
constexpr long long GT_WAIT = 1LL << 31;
static_assert(Z_OFF + Z_BYTES <= STAGE, "stage layout");

struct GptqArgs {
    const uint16_t *scales;   // [K/G][N]
    const uint32_t *zeros;    // [K/G][N/8]
    const void *x;            // [M][K], f32 or bf16
    float *y;                 // [M][N]
    int64_t N, K;
    int M;                    // <= 8 per launch
    int per;                  // groups per rank (the last rank's range may be shorter)
    int groups;               // K / G
};

// Dynamic shared memory: ring | B fragments [chunks][NB][32 lanes] uint2 | partial rows [MB][128].
template <typename XT, int MB>
__global__ void __maxnreg__(96)
gemv_gptq_tc(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ GptqArgs a) {
    constexpr int NB = (MB + 3) / 4;           // B tiles: four batch rows (hi, lo) per n8
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[GT_NS], empty[GT_NS];
    __shared__ int abort_s, xexp[MB];
    __shared__ float xscale[MB], xinv[MB];
    uint8_t *ring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
    const int tile = blockIdx.x / S;
    const int g0 = rank * a.per, ng = max(0, min(a.per, a.groups - g0));   // this rank's groups
    const int64_t k0 = (int64_t)g0 * GT_G;
    const int nch = ng * (GT_G / 16);
    uint2 *bfrag = reinterpret_cast<uint2 *>(ring + GT_NS * STAGE);                 // [a.per * 8][NB][32]
    float *part = reinterpret_cast<float *>(bfrag + (size_t)a.per * 8 * NB * 32);   // [MB][128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &abort_s;
    const int M = a.M;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GT_NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], GT_WARPS);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < MB) xexp[threadIdx.x] = -1000;
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == GT_WARPS) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            int issued = 0;
            for (int j = 0; j < ng; j++) {
                const int s = j % GT_NS;
                if (j >= GT_NS && !wait_or_abort(&empty[s], ((j / GT_NS) & 1) ^ 1, abort_flag, &g_gptq_tc_error, GT_WAIT))
                    break;
                uint8_t *st = ring + s * STAGE;
                const int64_t grp = g0 + j;
                mbar_arrive_expect_tx(&full[s], W_BYTES + S_BYTES + Z_BYTES);
                tma2(smem_u32(st), &wmap, tile * GT_COLS, (int)((k0 + (int64_t)j * GT_G) / 8), &full[s], pol);
                bulk_g2s(st + S_OFF, a.scales + grp * a.N + (int64_t)tile * GT_COLS, S_BYTES, &full[s]);
                bulk_g2s(st + Z_OFF, a.zeros + grp * (a.N >> 3) + (int64_t)tile * (GT_COLS / 8), Z_BYTES, &full[s]);
                issued++;
            }
            for (int q = issued > GT_NS ? issued - GT_NS : 0; q < issued; q++)
                if (!mbar_wait_bounded(&full[q % GT_NS], (uint32_t)((q / GT_NS) & 1), GT_WAIT))
                    atomicExch(&g_gptq_tc_error, Q4_ETIMEOUT);
        }
        __syncwarp();
    } else {
        // ---------------------------------- x staging (warps 0-7, 256 threads)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int t256 = threadIdx.x;
        {
            constexpr int VPC = 16 / (int)sizeof(XT);
            const int cpr = ng * GT_G / VPC, total = M * cpr;
#pragma unroll 4
            for (int i = t256; i < total; i += GT_WARPS * 32) {
                const int m = i / cpr, c = i - m * cpr;
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const XT *>(a.x) + (int64_t)m * a.K +
                                                                        k0 + (int64_t)c * VPC));
                const float mx = absmax16<XT>(v);
                if (mx > 0.0f) atomicMax(&xexp[m], (int)((__float_as_uint(mx) >> 23) & 255u) - 127);
            }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (t256 < MB) {
            // e in [-100, 127] keeps both powers of two normal (an all-zero or tiny x takes -100)
            const int e = min(127, max(-100, xexp[t256]));
            xscale[t256] = __uint_as_float((uint32_t)(127 + 14 - e) << 23);   // |x| * scale < 2^15
            xinv[t256] = __uint_as_float((uint32_t)(127 - 14 + e) << 23);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        // B fragments: lane (n, t) of chunk c, tile nb holds k = 2t, 2t+1 and 2t+8, 2t+9 of column n =
        // 2m + h (h = 0: hi terms, 1: lo terms) of batch row m = 4 nb + n / 2, odd k divided by 16;
        // one thread per (chunk, row m) reads the chunk's 16 values with 16-byte loads.  Rows m >= M
        // are zeros.
        for (int e = t256; e < nch * MB; e += GT_WARPS * 32) {
            const int c = e / MB, m = e - c * MB;
            __half hh[16], hl[16];
            if (m < M) {
                float v[16];
                load16<XT>(reinterpret_cast<const XT *>(a.x) + (int64_t)m * a.K + k0 + (int64_t)c * 16, v);
                const float sc = xscale[m];
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const float f = v[i] * sc * ((i & 1) ? 0.0625f : 1.0f);   // exact: powers of two
                    hh[i] = __float2half_rn(f);
                    hl[i] = __float2half_rn(f - __half2float(hh[i]));
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; i++) hh[i] = hl[i] = __float2half_rn(0.0f);
            }
            uint2 *dst = bfrag + ((size_t)c * NB + (m >> 2)) * 32 + (2 * (m & 3)) * 4;
#pragma unroll
            for (int t = 0; t < 4; t++) {
                dst[t] = make_uint2(h2bits(hh[2 * t], hh[2 * t + 1]), h2bits(hh[2 * t + 8], hh[2 * t + 9]));
                dst[4 + t] = make_uint2(h2bits(hl[2 * t], hl[2 * t + 1]), h2bits(hl[2 * t + 8], hl[2 * t + 9]));
            }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");

        // ------------------------------------------------ decode + multiply
        const int g = lane >> 2, t = lane & 3;
        const int c0 = warp * 16 + 2 * g;                                // columns c0 (row g), c0 + 1 (row g + 8)
        const uint32_t bsel = (uint32_t)t * 0x0101u;                      // byte t into bytes 0 and 2
        float acc[NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; nb++) acc[nb][0] = acc[nb][1] = 0.0f;
        const uint2 *bp = bfrag + lane;
        const uint32_t ring_u = smem_u32(ring);
        for (int j = 0; j < ng; j++) {
            const int s = j % GT_NS;
            if (!wait_or_abort(&full[s], (uint32_t)((j / GT_NS) & 1), abort_flag, &g_gptq_tc_error, GT_WAIT)) break;
            const uint8_t *sp = ring + s * STAGE;
            const uint32_t st = ring_u + (uint32_t)(s * STAGE) + (uint32_t)c0 * 4;
            // zero points of the two columns: word c0 / 8, slots c0 % 8 and c0 % 8 + 1, stored minus one
            const uint32_t zw = *reinterpret_cast<const uint32_t *>(sp + Z_OFF + (c0 >> 3) * 4);
            const uint32_t z0 = ((zw >> (4 * (c0 & 7))) & 15u) + 1u, z1 = ((zw >> (4 * (c0 & 7) + 4)) & 15u) + 1u;
            const uint32_t zz0 = (0x6400u + z0) | ((0x6400u + (z0 << 4)) << 16);
            const uint32_t zz1 = (0x6400u + z1) | ((0x6400u + (z1 << 4)) << 16);
            float D[NB][4];
#pragma unroll
            for (int nb = 0; nb < NB; nb++) D[nb][0] = D[nb][1] = D[nb][2] = D[nb][3] = 0.0f;
            const uint2 *bj = bp + (size_t)j * 8 * NB * 32;
#pragma unroll 4
            for (int ch = 0; ch < GT_G / 16; ch++) {
                const uint2 wr0 = lds64(st + (uint32_t)(2 * ch) * (GT_COLS * 4));      // word row 2ch: columns c0, c0+1
                const uint2 wr1 = lds64(st + (uint32_t)(2 * ch + 1) * (GT_COLS * 4));  // word row 2ch+1
                uint4 af;
                af.x = hsub2_bits((prmt(wr0.x, wr0.x, bsel) & 0x00F0000Fu) | 0x64006400u, zz0);   // row g, k 2t..
                af.y = hsub2_bits((prmt(wr0.y, wr0.y, bsel) & 0x00F0000Fu) | 0x64006400u, zz1);   // row g+8
                af.z = hsub2_bits((prmt(wr1.x, wr1.x, bsel) & 0x00F0000Fu) | 0x64006400u, zz0);   // row g, k 2t+8..
                af.w = hsub2_bits((prmt(wr1.y, wr1.y, bsel) & 0x00F0000Fu) | 0x64006400u, zz1);   // row g+8
#pragma unroll
                for (int nb = 0; nb < NB; nb++) {
                    const uint2 bf = bj[(ch * NB + nb) * 32];
                    mma16816(D[nb], af, bf.x, bf.y);
                }
            }
            // group epilogue: lane (g, t) holds batch row 4 nb + t (D columns 2t hi, 2t+1 lo) of columns c0, c0+1
            const uint32_t s2 = *reinterpret_cast<const uint32_t *>(sp + S_OFF + c0 * 2);
            const float sa = half_bits_f32(s2 & 0xffffu), sb = half_bits_f32(s2 >> 16);
#pragma unroll
            for (int nb = 0; nb < NB; nb++) {
                acc[nb][0] = fmaf(sa, D[nb][0] + D[nb][1], acc[nb][0]);
                acc[nb][1] = fmaf(sb, D[nb][2] + D[nb][3], acc[nb][1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
#pragma unroll
        for (int nb = 0; nb < NB; nb++) {
            const int m = 4 * nb + t;
            if (m < M) {
                part[m * GT_COLS + c0] = acc[nb][0] * xinv[m];
                part[m * GT_COLS + c0 + 1] = acc[nb][1] * xinv[m];
            }
        }
    }
    // partial rows of every rank, summed in rank order
    cluster.sync();
    if (warp < GT_WARPS) {
        for (int i = threadIdx.x; i < M * GT_COLS; i += GT_WARPS * 32) {
            const int m = i / GT_COLS, col = i % GT_COLS;
            if (col % S != rank) continue;                               // columns spread over the ranks
            float pv[MAXS];
#pragma unroll
            for (int q = 0; q < MAXS; q++) pv[q] = q < S ? cluster.map_shared_rank(part, q)[m * GT_COLS + col] : 0.0f;
            float v = 0.0f;
#pragma unroll
            for (int q = 0; q < MAXS; q++) v += pv[q];
            a.y[(int64_t)m * a.N + (int64_t)tile * GT_COLS + col] = v;
        }
    }
    cluster.sync();
}

int64_t gptq_tc_smem(int per, int MB) {
    const int NB = (MB + 3) / 4;
    return 1024 + (int64_t)GT_NS * STAGE + (int64_t)per * 8 * NB * 32 * 8 + (int64_t)MB * GT_COLS * 4;
}

// The fewest ranks whose shared memory fits: the fallback when no split has
// every cluster resident at once (more launch waves, same result).
bool gptq_tc_plan(int64_t K, int MB, int *S_out, int *per_out) {
    const int groups = (int)(K / GT_G);
    for (int S = 1; S <= MAXS && S <= groups; S++) {
        const int per = (groups + S - 1) / S;
        if (gptq_tc_smem(per, MB) <= 200 * 1024) {
            *S_out = (groups + per - 1) / per;
            *per_out = per;
            return true;
        }
    }
    return false;
}

std::mutex g_cap_lock;
struct CapEntry {
    const void *fn;
    int64_t smem;
    int cap;
};
CapEntry g_cap[64][3][MAXS];

int capacity(const void *fn, int mb_index, int S, int64_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_cap_lock);
    CapEntry &c = g_cap[dev & 63][mb_index][S - 1];
    if (c.fn == fn && c.smem == smem) return c.cap;
    c = CapEntry{fn, smem, cluster_capacity(fn, GT_THREADS, S, smem)};
    return c.cap;
}

template <typename XT, int MB>
cudaError_t gptq_tc_run(const CUtensorMap &map, GptqArgs a, cudaStream_t s) {
    auto kern = gemv_gptq_tc<XT, MB>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    // K split: the most CTAs for which every cluster is resident at once (one
    // wave), ranks of `per` whole groups, none empty
    const int tiles = (int)(a.N / GT_COLS), groups = (int)(a.K / GT_G);
    const int mbi = MB == 1 ? 0 : (MB == 4 ? 1 : 2);
    int S = 0, per = 0;
    int64_t best = 0;
    for (int c = 1; c <= MAXS && c <= groups; c++) {
        const int pc = (groups + c - 1) / c;
        if ((groups + pc - 1) / pc != c || gptq_tc_smem(pc, MB) > 200 * 1024) continue;
        if (tiles <= capacity((const void *)kern, mbi, c, gptq_tc_smem(pc, MB)) && (int64_t)tiles * c > best) {
            best = (int64_t)tiles * c;
            S = c;
            per = pc;
        }
    }
    if (S == 0 && !gptq_tc_plan(a.K, MB, &S, &per)) return cudaErrorInvalidValue;
    a.per = per;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * S), 1, 1);
    cfg.blockDim = dim3(GT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)gptq_tc_smem(per, MB);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, map, a);
}

}  // namespace

// GPTQ, group 128 without g_idx, N % 128 == 0, K % 128 == 0, 16-byte aligned tensors.
bool gemv_gptq_tc_eligible(const Tensor &t, int64_t M) {
    if (t.fmt != Q4_GPTQ || t.g_idx || t.group != GT_G || M < 1 || t.N % GT_COLS || t.K % GT_G) return false;
    if (t.K > (1LL << 30) || t.N > (1LL << 30) || encode_fn() == nullptr) return false;
    if ((((uintptr_t)t.w | (uintptr_t)t.scales | (uintptr_t)t.zeros) & 15) != 0) return false;
    int S = 0, per = 0;
    return gptq_tc_plan(t.K, M > 4 ? 8 : (M > 1 ? 4 : 1), &S, &per);
}

cudaError_t launch_gemv_gptq_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorInvalidValue;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)t.N, (cuuint64_t)(t.K / 8)};
    const cuuint64_t strides[1] = {(cuuint64_t)(t.N * 4)};
    const cuuint32_t box[2] = {(cuuint32_t)GT_COLS, (cuuint32_t)GT_ROWS};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t *>(t.w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t xe = xd == Q4_DT_BF16 ? 2 : 4;
    for (int64_t m0 = 0; m0 < M; m0 += 8) {
        const int mc = (int)(M - m0 < 8 ? M - m0 : 8);
        const int MB = mc > 4 ? 8 : (mc > 1 ? 4 : 1);
        GptqArgs a;
        a.scales = reinterpret_cast<const uint16_t *>(t.scales);
        a.zeros = reinterpret_cast<const uint32_t *>(t.zeros);
        a.x = static_cast<const char *>(x) + m0 * t.K * xe;
        a.y = y + m0 * t.N;
        a.N = t.N;
        a.K = t.K;
        a.M = mc;
        a.per = 0;
        a.groups = (int)(t.K / GT_G);
        cudaError_t e;
        if (xd == Q4_DT_BF16)
            e = MB == 1 ? gptq_tc_run<__nv_bfloat16, 1>(map, a, s)
                        : (MB == 4 ? gptq_tc_run<__nv_bfloat16, 4>(map, a, s) : gptq_tc_run<__nv_bfloat16, 8>(map, a, s));
        else
            e = MB == 1 ? gptq_tc_run<float, 1>(map, a, s)
                        : (MB == 4 ? gptq_tc_run<float, 4>(map, a, s) : gptq_tc_run<float, 8>(map, a, s));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int gptq_tc_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gptq_tc_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_gptq_tc_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

}  // namespace q4
