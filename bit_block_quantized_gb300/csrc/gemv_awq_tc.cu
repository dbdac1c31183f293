// gemv_awq_tc.cu -- AWQ decode-GEMV on the tensor cores, weights streamed by
// tensor TMA ([BPA] "Real layouts compared": AWQ qweight int32 [K][N/8], the
// eight 4-bit slots of a word holding columns 8c + {0,2,4,6,1,3,5,7}; fp16
// scales [K/G][N]; qzeros int32 [K/G][N/8] with the same interleave and no
// minus one; w = s * (q - z)).
//
// mma.sync.m16n8k16 (f16 x f16 -> f32) with the WEIGHTS as B: n8 = the eight
// columns of one AWQ word, so lane (g, t) needs the slot of column g from the
// words of four k rows.  The MMA's k order is permuted within each 16-k chunk
// so that those are rows t, t+4, t+8, t+12 of the chunk: with the 64-byte
// swizzle of the TMA box (16-byte unit u of row r stored at u ^ ((r >> 1) & 3))
// the four rows' units fall in different banks, and one conflict-free 16-byte
// shared load gives a lane its word of four consecutive column groups.  One byte permute and one LOP3 put the
// column's nibble of two rows into the two halves of an f16 pair as
// 1024 + q * 2^b (b = 0 or 4, the nibble's place in its byte, the same for
// every row of a lane), and one HSUB2 of 1024 + z * 2^b leaves (q - z) * 2^b
// exactly, so the accumulator never holds the large offset.  x fills A: rows
// m hold the f16 hi terms of batch row m, rows m + 8 its lo terms
// (x * 2^(14 - e_m) = hi + lo to 22 significant bits), in the same k order.
// Each 128-k group (one ring stage) gets a fresh accumulator; the group
// epilogue adds s * (D_hi + D_lo), and the output scale takes 2^(e_m - 14 - b).
//
// A CTA owns 128 columns (16 column groups) and a range of whole groups; warp
// w takes column groups 4 (w & 3) .. 4 (w & 3) + 3 over k rows 64 (w >> 2) ..
// 64 (w >> 2) + 63 of every stage.  The CTAs of a cluster split K and add
// their partial rows (and the two k halves) in a fixed order through
// distributed shared memory, so repeated calls agree bit for bit.  Roles:
// warp 8 streams the stages (TMA box 128 rows x 16 words, plus the group's
// scales and zeros by bulk copy); warps 0-7 stage x, then decode and multiply.
// Two CTAs fit on an SM.  Every wait is bounded (~1 s): a timeout records
// Q4_ETIMEOUT, stops the roles, waits for issued copies and returns.
#include <cooperative_groups.h>

#include <mutex>

#include "q4_internal.cuh"
#include "tc_gemv_common.cuh"
#include "tma_map.cuh"

namespace q4 {

__device__ int g_awq_error;

namespace {

namespace cg = cooperative_groups;
using namespace tc;

constexpr int AT_COLS = 128;                   // columns per CTA
constexpr int AT_CG = AT_COLS / 8;             // column groups (AWQ words) per CTA row
constexpr int AT_G = 128;                      // group size = k rows per stage
constexpr int AT_WARPS = 8;                    // decode warps
constexpr int AT_THREADS = (AT_WARPS + 1) * 32;
constexpr int AT_NS = 6;                       // ring stages
constexpr int W_BYTES = AT_G * AT_CG * 4;      // 8 KB of weights per stage
constexpr int S_OFF = W_BYTES, S_BYTES = AT_COLS * 2;       // the group's fp16 scales
constexpr int Z_OFF = S_OFF + S_BYTES, Z_BYTES = AT_CG * 4; // the group's zero words
constexpr int STAGE = 9 * 1024;                // 1024-byte aligned stages
constexpr int MAXS = 8;                        // cluster ranks over K (the portable cluster size)
constexpr long long AT_WAIT = 1LL << 31;
static_assert(Z_OFF + Z_BYTES <= STAGE, "stage layout");

struct AwqArgs {
    const uint16_t *scales;   // [K/G][N]
    const uint32_t *zeros;    // [K/G][N/8]
    const void *x;            // [M][K], f32 or bf16
    float *y;                 // [M][N]
    int64_t N, K;
    int M;                    // <= 8 per launch
    int per;                  // groups per rank (the last rank's range may be shorter)
    int groups;               // K / G
};

// Dynamic shared memory: ring | A fragments [chunks][M][4 lanes t] uint4 | partial rows [2 k halves][M][128].
template <typename XT, int MB>
__global__ void __maxnreg__(96)
gemv_awq_tc(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ AwqArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[AT_NS], empty[AT_NS];
    __shared__ int abort_s, xexp[MB];
    __shared__ float xscale[MB], xinv[MB];
    uint8_t *ring = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
    const int tile = blockIdx.x / S;
    const int g0 = rank * a.per, ng = max(0, min(a.per, a.groups - g0));   // this rank's groups
    const int64_t k0 = (int64_t)g0 * AT_G;
    const int nch = ng * (AT_G / 16);
    uint4 *afrag = reinterpret_cast<uint4 *>(ring + AT_NS * STAGE);      // [a.per * 8][MB][4]
    float *part = reinterpret_cast<float *>(afrag + (size_t)a.per * 8 * MB * 4);  // [2][MB][128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = &abort_s;
    const int M = a.M;

    if (threadIdx.x == 0) {
        for (int s = 0; s < AT_NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], AT_WARPS);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < MB) xexp[threadIdx.x] = -1000;
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == AT_WARPS) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            int issued = 0;
            for (int j = 0; j < ng; j++) {
                const int s = j % AT_NS;
                if (j >= AT_NS && !wait_or_abort(&empty[s], ((j / AT_NS) & 1) ^ 1, abort_flag, &g_awq_error, AT_WAIT)) break;
                uint8_t *st = ring + s * STAGE;
                const int64_t grp = g0 + j;
                mbar_arrive_expect_tx(&full[s], W_BYTES + S_BYTES + Z_BYTES);
                tma2(smem_u32(st), &wmap, tile * AT_CG, (int)(k0 + (int64_t)j * AT_G), &full[s], pol);
                bulk_g2s(st + S_OFF, a.scales + grp * a.N + (int64_t)tile * AT_COLS, S_BYTES, &full[s]);
                bulk_g2s(st + Z_OFF, a.zeros + grp * (a.N >> 3) + (int64_t)tile * AT_CG, Z_BYTES, &full[s]);
                issued++;
            }
            for (int q = issued > AT_NS ? issued - AT_NS : 0; q < issued; q++)
                if (!mbar_wait_bounded(&full[q % AT_NS], (uint32_t)((q / AT_NS) & 1), AT_WAIT))
                    atomicExch(&g_awq_error, Q4_ETIMEOUT);
        }
        __syncwarp();
    } else {
        // ---------------------------------- x staging (warps 0-7, 256 threads)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int t256 = threadIdx.x;
        {
            // row maxima from 16-byte loads (8 bf16 or 4 f32 values), several in flight per thread
            constexpr int VPC = 16 / (int)sizeof(XT);
            const int cpr = ng * AT_G / VPC, total = M * cpr;
#pragma unroll 4
            for (int i = t256; i < total; i += AT_WARPS * 32) {
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
        // fragments: lane (m, t) of chunk c holds k rows t, t+4 (a0 hi, a1 lo) and t+8, t+12 (a2 hi, a3 lo);
        // one thread per (chunk, row m) reads the chunk's 16 values with 16-byte loads
        for (int e = t256; e < nch * M; e += AT_WARPS * 32) {
            const int c = e / M, m = e - c * M;
            const XT *src = reinterpret_cast<const XT *>(a.x) + (int64_t)m * a.K + k0 + (int64_t)c * 16;
            float v[16];
            load16<XT>(src, v);
            const float sc = xscale[m];
            __half hh[16], hl[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const float f = v[i] * sc;                                 // exact: a power of two
                hh[i] = __float2half_rn(f);
                hl[i] = __float2half_rn(f - __half2float(hh[i]));
            }
            uint4 *dst = afrag + ((size_t)c * MB + m) * 4;
#pragma unroll
            for (int t = 0; t < 4; t++)
                dst[t] = make_uint4(h2bits(hh[t], hh[t + 4]), h2bits(hl[t], hl[t + 4]), h2bits(hh[t + 8], hh[t + 12]),
                                    h2bits(hl[t + 8], hl[t + 12]));
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");

        // ------------------------------------------------ decode + multiply
        const int g = lane >> 2, t = lane & 3;
        const int cgu = warp & 3, kh = warp >> 2;                        // column-group unit, k half
        const int sl = (g >> 1) + 4 * (g & 1);                           // AWQ slot of column g
        const uint32_t psel = (uint32_t)(sl >> 1) | ((uint32_t)(4 + (sl >> 1)) << 8);  // byte sl/2 of each word
        const uint32_t nsh = 4u * (uint32_t)(sl & 1);                    // the nibble's place in the byte
        const uint32_t nmask = 0x000F000Fu << nsh;
        float acc[4][2];
#pragma unroll
        for (int c = 0; c < 4; c++) acc[c][0] = acc[c][1] = 0.0f;
        const bool arow = g < M;
        // byte offsets of the lane's rows t + 4r of chunk 0 of its k half; the swizzle
        // phase (row >> 1) & 3 = ((t >> 1) + 2r) & 3 is the same in every chunk
        uint32_t roff[4];
#pragma unroll
        for (int r = 0; r < 4; r++)
            roff[r] = (uint32_t)((kh * 64 + t + 4 * r) * 64) + ((uint32_t)(cgu ^ (((t >> 1) + 2 * r) & 3)) << 4);
        const uint32_t zsh = 4u * (uint32_t)sl - nsh;                    // zero nibble -> bit nsh
        const uint4 *ap = afrag + ((size_t)(kh * 4) * MB + (arow ? g : 0)) * 4 + t;
        const uint32_t ring_u = smem_u32(ring);
        for (int j = 0; j < ng; j++) {
            const int s = j % AT_NS;
            if (!wait_or_abort(&full[s], (uint32_t)((j / AT_NS) & 1), abort_flag, &g_awq_error, AT_WAIT)) break;
            const uint8_t *sp = ring + s * STAGE;
            const uint32_t st = ring_u + (uint32_t)(s * STAGE);
            uint32_t zz[4];                                              // 1024 + z * 2^b in both halves
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const uint32_t zw = *reinterpret_cast<const uint32_t *>(sp + Z_OFF + (cgu * 4 + c) * 4);
                const uint32_t h = ((zw >> zsh) & (15u << nsh)) | 0x6400u;
                zz[c] = prmt(h, h, 0x1010u);
            }
            float D[4][4];
#pragma unroll
            for (int c = 0; c < 4; c++) D[c][0] = D[c][1] = D[c][2] = D[c][3] = 0.0f;
            const uint4 *apj = ap + (size_t)j * 8 * MB * 4;
#pragma unroll 2
            for (int ch = 0; ch < AT_G / 32; ch++) {
                uint4 w4[4];
#pragma unroll
                for (int r = 0; r < 4; r++) w4[r] = lds128(st + roff[r] + (uint32_t)(ch * 1024));
                const uint4 af = apj[ch * MB * 4];     // lanes g >= M read row 0: their MMA rows are never stored
                const uint32_t wr[4][4] = {{w4[0].x, w4[0].y, w4[0].z, w4[0].w}, {w4[1].x, w4[1].y, w4[1].z, w4[1].w},
                                           {w4[2].x, w4[2].y, w4[2].z, w4[2].w}, {w4[3].x, w4[3].y, w4[3].z, w4[3].w}};
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    // rows t, t+4 -> b0 and rows t+8, t+12 -> b1: (q - z) * 2^b of column g, exact in f16
                    const uint32_t b0 = hsub2_bits((prmt(wr[0][c], wr[1][c], psel) & nmask) | 0x64006400u, zz[c]);
                    const uint32_t b1 = hsub2_bits((prmt(wr[2][c], wr[3][c], psel) & nmask) | 0x64006400u, zz[c]);
                    mma16816(D[c], af, b0, b1);
                }
            }
            // group epilogue: lane (g, t) holds batch g, columns 2t and 2t+1 of each of its four groups
            if (arow) {
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const uint32_t s2 = *reinterpret_cast<const uint32_t *>(sp + S_OFF + ((cgu * 4 + c) * 8 + 2 * t) * 2);
#pragma unroll
                    for (int jj = 0; jj < 2; jj++)
                        acc[c][jj] = fmaf(half_bits_f32(s2 >> (16 * jj)), D[c][jj] + D[c][2 + jj], acc[c][jj]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // output columns 2t, 2t+1 sit in slots of nibble place 4 * (t & 1): undo that 2^b with the x scale
        if (arow) {
            const float oscale = xinv[g] * ((t & 1) ? 0.0625f : 1.0f);
#pragma unroll
            for (int c = 0; c < 4; c++)
#pragma unroll
                for (int jj = 0; jj < 2; jj++)
                    part[(kh * MB + g) * AT_COLS + (cgu * 4 + c) * 8 + 2 * t + jj] = acc[c][jj] * oscale;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        for (int i = t256; i < M * AT_COLS; i += AT_WARPS * 32) part[i] += part[MB * AT_COLS + i];   // k halves
    }
    // partial rows of every rank, summed in rank order
    cluster.sync();
    if (warp < AT_WARPS) {
        for (int i = threadIdx.x; i < M * AT_COLS; i += AT_WARPS * 32) {
            const int m = i / AT_COLS, col = i % AT_COLS;
            if (col % S != rank) continue;                               // columns spread over the ranks
            float pv[MAXS];
#pragma unroll
            for (int q = 0; q < MAXS; q++) pv[q] = q < S ? cluster.map_shared_rank(part, q)[m * AT_COLS + col] : 0.0f;
            float v = 0.0f;
#pragma unroll
            for (int q = 0; q < MAXS; q++) v += pv[q];
            a.y[(int64_t)m * a.N + (int64_t)tile * AT_COLS + col] = v;
        }
    }
    cluster.sync();
}

int64_t awq_smem(int per, int MB) {
    return 1024 + (int64_t)AT_NS * STAGE + (int64_t)per * 8 * MB * 4 * 16 + 2 * (int64_t)MB * AT_COLS * 4;
}

// The fewest ranks whose shared memory fits: the fallback when no split has
// every cluster resident at once (more launch waves, same result).
bool awq_plan(int64_t N, int64_t K, int MB, int *S_out, int *per_out) {
    (void)N;
    const int groups = (int)(K / AT_G);
    for (int S = 1; S <= MAXS && S <= groups; S++) {
        const int per = (groups + S - 1) / S;
        if (awq_smem(per, MB) <= 200 * 1024) {
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

// Clusters of S CTAs (with `smem` bytes of dynamic shared memory each) that
// can be resident at once on the current device, cached per kernel.
int awq_capacity(const void *fn, int mb_index, int S, int64_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_cap_lock);
    CapEntry &c = g_cap[dev & 63][mb_index][S - 1];
    if (c.fn == fn && c.smem == smem) return c.cap;
    c = CapEntry{fn, smem, cluster_capacity(fn, AT_THREADS, S, smem)};
    return c.cap;
}

template <typename XT, int MB>
cudaError_t awq_tc_run(const CUtensorMap &map, AwqArgs a, cudaStream_t s) {
    auto kern = gemv_awq_tc<XT, MB>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        // the largest shared-memory carveout, so that two CTAs fit on an SM
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    // K split: the most CTAs for which every cluster is resident at once (one
    // wave), ranks of `per` whole groups, none empty
    const int tiles = (int)(a.N / AT_COLS), groups = (int)(a.K / AT_G);
    const int mbi = MB == 1 ? 0 : (MB == 4 ? 1 : 2);
    int S = 0, per = 0;
    int64_t best = 0;
    for (int c = 1; c <= MAXS && c <= groups; c++) {
        const int pc = (groups + c - 1) / c;
        if ((groups + pc - 1) / pc != c || awq_smem(pc, MB) > 200 * 1024) continue;
        if (tiles <= awq_capacity((const void *)kern, mbi, c, awq_smem(pc, MB)) && (int64_t)tiles * c > best) {
            best = (int64_t)tiles * c;
            S = c;
            per = pc;
        }
    }
    if (S == 0 && !awq_plan(a.N, a.K, MB, &S, &per)) return cudaErrorInvalidValue;
    a.per = per;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * S), 1, 1);
    cfg.blockDim = dim3(AT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)awq_smem(per, MB);
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

// AWQ, group 128 without g_idx, N % 128 == 0, K % 128 == 0, 16-byte aligned tensors.
bool gemv_awq_tc_eligible(const Tensor &t, int64_t M) {
    if (t.fmt != Q4_AWQ || t.g_idx || t.group != AT_G || M < 1 || t.N % AT_COLS || t.K % AT_G) return false;
    if (t.K > (1LL << 30) || t.N > (1LL << 30) || encode_fn() == nullptr) return false;
    if ((((uintptr_t)t.w | (uintptr_t)t.scales | (uintptr_t)t.zeros) & 15) != 0) return false;
    int S = 0, per = 0;
    return awq_plan(t.N, t.K, M > 4 ? 8 : (M > 1 ? 4 : 1), &S, &per);
}

cudaError_t launch_gemv_awq_tc(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorInvalidValue;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)(t.N / 8), (cuuint64_t)t.K};
    const cuuint64_t strides[1] = {(cuuint64_t)(t.N / 8 * 4)};
    const cuuint32_t box[2] = {(cuuint32_t)AT_CG, (cuuint32_t)AT_G};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t *>(t.w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t xe = xd == Q4_DT_BF16 ? 2 : 4;
    for (int64_t m0 = 0; m0 < M; m0 += 8) {
        const int mc = (int)(M - m0 < 8 ? M - m0 : 8);
        const int MB = mc > 4 ? 8 : (mc > 1 ? 4 : 1);
        AwqArgs a;
        a.scales = reinterpret_cast<const uint16_t *>(t.scales);
        a.zeros = reinterpret_cast<const uint32_t *>(t.zeros);
        a.x = static_cast<const char *>(x) + m0 * t.K * xe;
        a.y = y + m0 * t.N;
        a.N = t.N;
        a.K = t.K;
        a.M = mc;
        a.per = 0;
        a.groups = (int)(t.K / AT_G);
        cudaError_t e;
        if (xd == Q4_DT_BF16)
            e = MB == 1 ? awq_tc_run<__nv_bfloat16, 1>(map, a, s)
                        : (MB == 4 ? awq_tc_run<__nv_bfloat16, 4>(map, a, s) : awq_tc_run<__nv_bfloat16, 8>(map, a, s));
        else
            e = MB == 1 ? awq_tc_run<float, 1>(map, a, s)
                        : (MB == 4 ? awq_tc_run<float, 4>(map, a, s) : awq_tc_run<float, 8>(map, a, s));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int awq_read_and_clear_error() {
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_awq_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_awq_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    return v;
}

}  // namespace q4
