/*
 * q4.h -- C ABI of libq4.so: fused 4-bit weight decode + GEMV/GEMM, dequant,
 * repack and validation for NVFP4, MXFP4, GGUF Q4_K and Q4_0, GPTQ and AWQ,
 * on one NVIDIA GB300 (sm_103a).
 *
 * Sources, cited as "page title, section":
 *   [FBTC] "Four Bits, Three Contracts" (shivasnotes.com/blog/6006)
 *   [W4K]  "Why 4-Bit Quantization Is King" (shivasnotes.com/blog/5996)
 *   [BPA]  "Bit Packing Architecture, in depth" (aicassindra.com quant_bit_packing)
 *   [MUS7] "Muser book, Chapter 7 - NVFP4: the native lane" (highperformanceailab.com)
 *
 * Conventions for every entry point
 *   - Logical weights W are [N out][K in]; activations x are [M][K] row-major;
 *     outputs y are [M][N] row-major f32:  y[m][n] = sum_k w_hat[n][k] * x[m][k].
 *   - Every pointer is a DEVICE pointer owned by the caller (e.g. allocated by
 *     torch).  The library allocates no device memory and keeps no pointer
 *     after a call returns.  Tensor base pointers must be 16-byte aligned
 *     (Q4_EALIGN otherwise).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on it unless documented as synchronous.
 *   - Arguments are checked on the host before any launch; a non-zero status
 *     means nothing was launched.  Padding to block/group multiples is the
 *     caller's job ([BPA] "Endianness, views and padding").
 *   - Scale bytes are NOT scanned for NaN encodings on every call: run
 *     q4_validate once when the weights are loaded ([MUS7] 7.3 fail-closed
 *     loader).  Results on unvalidated NaN scales are unspecified (no fault).
 *
 * Formats (byte layouts, little-endian)
 *   Q4_NVFP4  payload u8 [N][K/2], low nibble = even k; E4M3FN scales u8
 *             [N][K/16]; aux->scale2 f32 > 0.  w = (e2m1 * e4m3fn) * scale2,
 *             never regrouped ([MUS7] 7.1-7.2).  K % 16 == 0.
 *   Q4_MXFP4  payload as NVFP4; E8M0 scales u8 [N][K/32]; w = e2m1 * 2^(b-127)
 *             ([FBTC] section 3).  K % 32 == 0.
 *   Q4_Q4K    144-byte super-blocks [N][K/256]: fp16 d @0, fp16 dmin @2, 12 B of
 *             6-bit scales/mins @4, 128 code bytes @16; w = d*s_j*q - dmin*m_j;
 *             code byte 32c+l feeds k = 64c+l (low) and 64c+32+l (high)
 *             ([FBTC] sections 5-6).  `scales` ignored.  K % 256 == 0.
 *   Q4_Q40    18-byte blocks [N][K/32]: fp16 d, 16 code bytes, byte j = element
 *             j (low) and j+16 (high); w = d*(q-8) ([BPA] "Real layouts
 *             compared").  `scales` ignored.  K % 32 == 0.
 *   Q4_GPTQ   qweight i32 [K/8][N] (row 8r+j at bits 4j); scales fp16
 *             [K/G][N]; aux->zeros = qzeros i32 [K/G][N/8] (column n at bits
 *             4*(n%8), stored zero-1); optional aux->g_idx i32 [K]; w =
 *             scale*(q - zero) ([BPA]).  K % G == 0, N % 8 == 0.
 *   Q4_AWQ    qweight i32 [K][N/8], slot p holds column 8c+{0,2,4,6,1,3,5,7}[p];
 *             scales fp16 [K/G][N]; aux->zeros = qzeros i32 [K/G][N/8], same
 *             interleave, no minus-one ([BPA]).  K % G == 0, N % 8 == 0.
 *   Q4_NVFP4_SPLITHALF  NVFP4 with split-half nibble order in each 16-group:
 *             low nibbles of its 8 bytes = lanes 0-7, high = lanes 8-15 ([W4K]
 *             section 5).  Dequant and repack only.
 *   Q4_LOGICAL  the logical matrix of [BPA] "Repacking between formats": u8
 *             codes [K][N], fp16 scales [K/G][N], aux->zeros u8 [K/G][N];
 *             w = scale*(q - zero).  Dequant and repack only.
 */
#ifndef Q4_H
#define Q4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q4_NVFP4 = 1,
    Q4_MXFP4 = 2,
    Q4_Q4K = 3,
    Q4_Q40 = 4,
    Q4_GPTQ = 5,
    Q4_AWQ = 6,
    Q4_NVFP4_SPLITHALF = 7,
    Q4_LOGICAL = 8
} q4_fmt;

typedef enum { Q4_DT_F32 = 0, Q4_DT_BF16 = 1 } q4_dtype;

/* Status codes. */
enum {
    Q4_OK = 0,
    Q4_EINVAL = 1,       /* null pointer, unknown format/dtype, missing aux field */
    Q4_EDIM = 2,         /* M, N or K <= 0, or not a multiple of the format's block/group */
    Q4_EALIGN = 3,       /* a tensor pointer is not 16-byte aligned */
    Q4_ENAN = 4,         /* q4_validate found NaN scale encodings */
    Q4_ESCALE2 = 5,      /* NVFP4 scale2 not finite and > 0 ([MUS7] 7.2) */
    Q4_ECUDA = 6,        /* a CUDA launch or copy failed */
    Q4_EUNSUPPORTED = 7, /* format/operation pair not provided (e.g. GEMV on LOGICAL) */
    Q4_ERANGE = 8,       /* a value cannot be represented in the target (repack zeros) */
    Q4_ETIMEOUT = 9      /* a bounded device-side wait ran out (see q4_last_error) */
};

/* Per-call options.  Passing aux == NULL selects the defaults: x_dtype = bf16
 * for NVFP4/MXFP4 and f32 for the others, group = 128, no g_idx, out_dtype =
 * f32.  NVFP4 requires aux (for scale2); GPTQ/AWQ/LOGICAL require aux->zeros. */
typedef struct {
    float scale2;          /* NVFP4 per-tensor f32 scale; must be finite and > 0 */
    const void *zeros;     /* GPTQ/AWQ qzeros i32, LOGICAL u8 zeros */
    const int32_t *g_idx;  /* optional GPTQ/LOGICAL group of each k (values < K/group) */
    int32_t group;         /* GPTQ/AWQ/LOGICAL group size along K; <= 0 means 128 */
    q4_dtype x_dtype;      /* activation dtype for q4_gemv */
    q4_dtype out_dtype;    /* q4_dequant output dtype (bf16 = nearest-even of the f32 w) */
    uint32_t flags;        /* Q4_FLAG_* options; 0 = defaults */
} q4_aux;

/* q4_aux.flags: batch-1 NVFP4 GEMVs with bf16 x (q4_gemv, and
 * q4_gemv_grouped when every member sets it) run on the native block-scaled
 * FP4 tensor cores with x entered as its exact 2-bit FP4 slices (see
 * q4_gemv) instead of the TMA-fed decode kernel. */
#define Q4_FLAG_FP4_SLICES 1u

/* y[M][N] (f32) = x[M][K] . W^T.  The fused decode + dot of [W4K] section 1:
 * packed weights are streamed once from HBM, decoded on chip and accumulated
 * in f32; no dequantized matrix is written.  M <= 8 runs the bandwidth-bound
 * GEMV kernels.  With Q4_FLAG_FP4_SLICES, NVFP4 with bf16 x, M == 1 and
 * K % 256 == 0 runs on the native block-scaled FP4 tensor cores: TMA lands
 * the packed weights in shared memory, the MMA applies their E4M3 scales,
 * and x enters as its exact 2-bit FP4 slices (blocks the slices cannot hold
 * -- subnormal, non-finite, or more than 2^24 below their block's top -- are
 * added on the CUDA cores), so the result holds for every x.  Otherwise
 * NVFP4 with bf16 x, M <= 4 and K % 256 == 0 streams its
 * weights into shared memory by tensor TMA (weights are read before the
 * stream dependency on the previous launch resolves, x and y after it, so W
 * must not be written by a still-running kernel that released its dependents
 * early; the library's own kernels that do so only read weights).  GPTQ
 * and AWQ with group 128, no g_idx, N % 128 == 0 and K % 128 == 0 (any M, in
 * launches of up to 8 rows) run TMA-fed tensor-core kernels with the same
 * rule for W, its scales and zeros: codes minus zero points formed exactly
 * in f16 as an MMA operand, x as f16 hi + lo terms, K split over a
 * thread-block cluster and reduced in rank order (repeated calls agree bit
 * for bit).  Q4_K and Q4_0 with K % 256 == 0 and K <= 12288 (the staged x
 * and three 18 KB ring stages within 112 KB of shared memory), at M == 1 or,
 * with bf16 x, M <= 8 (launches of two rows), run a TMA-fed tensor-core kernel
 * with the same rule for W: 16 rows x 2048 k per stage, the codes as exact f16
 * MMA operands (Q4_K: q, its sub-block scale and min applied per lane in f32;
 * Q4_0: q - 8), repeated calls agreeing bit for bit.  M >= 9
 * with bf16 x on NVFP4 or Q4_K (K % 256 == 0) runs the
 * tcgen05 tensor-core kernel: weights decoded to bf16 straight into tensor
 * memory, x tiles by TMA, f32 accumulation in TMEM, K split over a cluster
 * and reduced in a fixed order (repeated calls agree bit for bit), batch in
 * chunks of 128.  NVFP4's staged e2m1*e4m3 product is exact in bf16; Q4_K's
 * f32 weight is rounded once to bf16 there, so its accuracy statement is
 * against RNE_bf16(w_hat).  Other M >= 9 cases run the general GEMV kernel.
 * Accuracy: within 1e-5 * sum_k |w||x| + 1e-6 of the exact f64 sum of the
 * pinned w_hat (bf16-rounded for the Q4_K tensor-core case).  The tensor-core
 * kernel's waits are bounded: a timeout is reported by q4_last_error.
 * Returns Q4_OK or a status; asynchronous on `stream`. */
int q4_gemv(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux,
            const void *x, float *y, int64_t M, int64_t N, int64_t K, void *stream);

/* One GEMV of a group (see q4_gemv_grouped). */
typedef struct {
    q4_fmt fmt;
    const void *W_packed;
    const void *scales;
    const q4_aux *aux;
    const void *x;         /* [M][K] */
    float *y;              /* [M][N] */
    int64_t N, K;
} q4_gemv_desc;

/* Several independent GEMVs with the same batch M, e.g. the projections of
 * one decoder layer that read the same activations (q/k/v, gate/up) -- the
 * grouping the pages' decode path applies per layer ([W4K] section 7d: one
 * token streams every weight once).  When every member is NVFP4 (or every
 * one MXFP4) with bf16 x and one x, all share K, count <= 8 and each takes
 * the TMA-fed tensor-core path, the group runs
 * as ONE persistent launch whose tile list spans all members (no launch gap
 * or ramp between them); so does a group whose members are all Q4_K (or all
 * Q4_0) with one K and one x, each taking q4_gemv's TMA-fed block kernel (one
 * launch per two batch rows); otherwise each member is issued as its own
 * q4_gemv.
 * Members must be independent: no y may alias another member's x or weights.
 * Same checks, accuracy and stream semantics as q4_gemv; if any member is
 * rejected nothing is launched. */
int q4_gemv_grouped(const q4_gemv_desc *descs, int count, int64_t M, void *stream);

/* A chain of GEMV groups with stream-order semantics, in one launch where
 * possible: group g is descs[first[g] .. first[g+1]-1] (first[0] = 0, ngroups
 * entries after it), its members read the same x and share K, and group g+1
 * reads its x and writes its y only after every member of groups 0..g has
 * written its y -- exactly as if each group were its own q4_gemv_grouped call
 * on `stream`, so a later group's x may be (a view of) an earlier group's y.
 * This is the decode sequence of one layer's projections (the pages' decode
 * path streams every weight of every layer once per token, [W4K] section 7d)
 * with the per-launch ramp and tail paid once.  When every member is NVFP4
 * with bf16 x, M <= 4, K % 256 == 0, ngroups <= 4 and count <= 8, the chain
 * runs as ONE cooperative launch whose CTAs meet at a grid-wide barrier
 * between groups while the next group's weights are already streaming;
 * otherwise the groups are issued one after the other as q4_gemv_grouped.
 * sync: caller-owned device memory of 2 uint32 words, zero before its first
 * use and not written by the caller afterwards; a launch that completes
 * without error leaves it ready for the next call (also across CUDA-graph
 * replays).  A launch whose barrier gave up (q4_last_error() returns
 * Q4_ETIMEOUT) leaves the count holding the CTAs that did arrive: the caller
 * must then set both words to zero again (e.g. cudaMemsetAsync) before the
 * next chain that uses them, or that chain may pass a barrier early or time
 * out.  Chains that may run at the same time (other streams) need their own
 * sync words.  May be NULL
 * when ngroups == 1.  Same checks, accuracy and stream semantics as
 * q4_gemv_grouped; if any member is rejected nothing is launched. */
int q4_gemv_chain(const q4_gemv_desc *descs, const int *first, int ngroups, int64_t M, uint32_t *sync,
                  void *stream);

/* The integer-exact weight-only NVFP4 contraction ([MUS7] 7.4.2): y[M][N]
 * from NVFP4 weights (layout as Q4_NVFP4; aux->scale2 required) and
 * activations x[M][K] (aux->x_dtype: bf16 or f32), in three pinned stages.
 *   1. Each activation row is cut into 256-value blocks.  A block's signed
 *      first maximum m (the first element of largest magnitude) gives
 *      iscale = -127/m; each code is the f32 product x*iscale rounded half to
 *      even and capped at 127, and the block scale is 1/iscale.  A block
 *      whose iscale is not finite (m zero, or so small that -127/m
 *      overflows) takes zero codes and scale 0.
 *   2. Per output row and block, T = sum over the block's 16 groups of
 *      q9(scale) * sum(q1(code) * q8) is an exact 64-bit integer (q1: E2M1 in
 *      halves; q9: E4M3FN in units of 2^-9), independent of summation order.
 *   3. In block order, in f32: c = fma(float(T), 2^-10, 0); c = fma(c,
 *      block scale, 0); c = fma(c, scale2, 0); total = fma(1, c, total).
 *      y = total rounded to binary16, stored widened to f32.
 * The result is therefore bit-reproducible: every run, batch size and
 * device gives the same bits.  K % 256 == 0 (Q4_EDIM otherwise); x must be
 * finite.  Each launch quantizes up to 8 activation rows into a 200 KiB
 * shared-memory budget (8 rows up to K = 24,832; fewer rows per launch above
 * that; K > 200,448 gets Q4_EDIM); larger M runs as several launches.
 * M = 1 (K up to 18,432) and M = 2 (K up to 8,192) run a TMA-fed kernel whose
 * f16 tensor-core MMA forms each group's q1 * q8 dot exactly (E2M1 halves
 * times 8-bit codes, partial sums below 2^15: no f32 rounding), the rest on
 * the CUDA cores; both give the same bits.
 * Allocates nothing; asynchronous on `stream`. */
int q4_gemv_a16q8(const void *W_packed, const void *scales, const q4_aux *aux, const void *x, float *y,
                  int64_t M, int64_t N, int64_t K, void *stream);

/* The Q4_K x Q8 (W4A8) contraction ([W4K] section 7: the W4A8 extension of
 * the section 4 Q4_K sub-block example, and the route of Q4_K weights against
 * 8-bit activation blocks): y[M][N] f32 from Q4_K weights (layout as Q4_Q4K;
 * aux may be NULL) and activations x[M][K] (aux->x_dtype, default f32).
 *   1. Activations go to the per-256 signed 8-bit grid of q4_gemv_a16q8
 *      (signed first maximum m, iscale = -127/m, codes nearest-even of
 *      x*iscale capped at 127, block scale 1/iscale); each 32-value
 *      sub-block's code sum is kept.
 *   2. Per output row and super-block, I1 = sum_j sc_j * sum q*q8 and
 *      I2 = sum_j m_j * (code sum of sub-block j) are exact integers.
 *   3. In f32 and in this order: v = d*float(I1) - dmin*float(I2), then
 *      c = v * block scale, then total += c over the super-blocks in order.
 * The page gives the algebra and the order of the steps in words; the
 * roundings above are this library's reading.  Bit-reproducible across
 * runs, batch sizes and devices.  K % 256 == 0 (Q4_EDIM otherwise); x must be
 * finite.  Up to 8 activation rows per launch in a 200 KiB shared-memory
 * budget; larger M runs as several launches.  M = 1 (K up to 12,288) and
 * M = 2 (K up to 10,240) run a TMA-fed kernel whose f16 tensor-core MMAs form
 * each 32-value sub-block's sum of q * q8 exactly (codes as f16 subnormals
 * times 8-bit activation codes, sums below 2^16 * 2^-24: no f32 rounding);
 * other shapes the CUDA cores; both give the same bits.  Allocates nothing;
 * asynchronous on `stream`. */
int q4_gemv_q4k_q8(const void *W_packed, const q4_aux *aux, const void *x, float *y, int64_t M, int64_t N,
                   int64_t K, void *stream);

/* The W4A4 contraction ([MUS7] 7.4.3): NVFP4 weights (layout as Q4_NVFP4;
 * aux->scale2 required) against activations x[M][K] (aux->x_dtype bf16 or
 * f32) that are themselves quantized to NVFP4 in 16-value groups.
 *   1. Activation tensor scale G = 1 / input_scale_inv (finite, > 0;
 *      Q4_ESCALE2 otherwise).  Each group takes the weights' own rule: E4M3
 *      scale = nearest-even of (amax/6)/G saturating at 448, codes =
 *      nearest-even E2M1 of x/(scale*G) (the midpoints of q4_quantize_nvfp4).
 *   2. Per output row and group, T_g = q9(weight scale) * q9(activation
 *      scale) * sum q1(w code) * q1(x code) is an exact 64-bit integer (q1:
 *      E2M1 in halves, q9: E4M3FN in units of 2^-9; denominator 2^-20).
 *   3. In group order, in f32: c = fma(float(T_g), 2^-20, 0); c = fma(c,
 *      scale2, 0); c = fma(c, G, 0); total = fma(1, c, total).  y = total
 *      rounded to binary16, stored widened to f32.
 * The section names the encodings, the integer product and the factors; the
 * per-group order of step 3 is this library's reading.  Bit-reproducible
 * across runs, batch sizes and devices.  K % 64 == 0; x finite.  Up to 8
 * activation rows per launch in a 200 KiB shared-memory budget.  Allocates
 * nothing; asynchronous on `stream`. */
int q4_gemv_w4a4(const void *W_packed, const void *scales, const q4_aux *aux, float input_scale_inv, const void *x,
                 float *y, int64_t M, int64_t N, int64_t K, void *stream);

/* W4A4 on the native block-scaled FP4 tensor cores ([MUS7] 7.4.3's producer
 * mode, where activations arrive already in NVFP4; [W4K] section 7: Blackwell
 * tensor cores consume the block-scaled FP4 layout directly).  Weights as
 * Q4_NVFP4 (aux->scale2 required); activations xq u8 [M][K/2] (even k in the
 * low nibble) with E4M3 scales xs u8 [M][K/16] and tensor scale x_scale2
 * (finite, > 0), e.g. from q4_quantize_nvfp4_scaled.  Both operands go to
 * tcgen05.mma.kind::mxf4nvf4.block_scale as they are stored: the MMA
 * multiplies E2M1 codes and applies both E4M3 scales exactly, accumulating
 * in f32; y[M][N] = accumulator * scale2 * x_scale2.  Accuracy: within
 * 1e-5 * sum_k |w||x_hat| + 1e-6 of the exact f64 sum over the pinned
 * weights and activations.  (q4_gemv_w4a4 is the integer-exact contract of
 * the section; this is the tensor-core lane.)  K % 256 == 0; 16 activation
 * rows per launch (larger M runs as several launches, each streaming the
 * weights).  Allocates nothing; asynchronous on `stream`. */
int q4_gemv_w4a4_tc(const void *W_packed, const void *scales, const q4_aux *aux, const void *xq, const void *xs,
                    float x_scale2, float *y, int64_t M, int64_t N, int64_t K, void *stream);

/* NVFP4 quantization of activations x[M][K] (f32 or bf16, finite) with a
 * GIVEN tensor scale (e.g. W4A4's 1 / input_scale_inv, [MUS7] 7.4.3): the
 * group rule of q4_quantize_nvfp4 (E4M3 scale = nearest-even of
 * (amax/6)/scale2 saturating at 448, E2M1 codes nearest-even of
 * x/(scale*scale2)) without the tensor-wide maximum.  payload [M][K/2],
 * scales [M][K/16].  K % 16 == 0; scale2 finite and > 0 (Q4_ESCALE2).
 * Bit-exact with the definition; one launch, asynchronous on `stream`. */
int q4_quantize_nvfp4_scaled(const void *x, q4_dtype x_dtype, float scale2, void *payload, void *scales, int64_t M,
                             int64_t K, void *stream);

/* NVFP4 quantization on the GPU, the write side of the format ([MUS7] 7.2):
 * W[N][K] (w_dtype f32 or bf16, finite) -> payload u8 [N][K/2] (even k in the
 * low nibble), E4M3FN scale bytes u8 [N][K/16] and the tensor scale.
 *   scale2 = amax(W) / (448 * 6) in f32 (1 if W is all zero), written to the
 *            DEVICE f32 word *scale2 (4-byte aligned; it holds the running
 *            maximum during the call, so nothing is allocated);
 *   per 16-value group: scale byte = nearest-even E4M3FN of
 *            (amax_group / 6) / scale2, saturating at 448 (never 0x7f);
 *   codes = nearest-even E2M1 of w / (dec(scale) * scale2), ties to the even
 *            code at the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5 and 5,
 *            saturating at 6, the sign kept (a negative value that rounds to
 *            zero is code 8); a group whose scale decodes to 0 is all code 0.
 * Every step is one IEEE f32 operation, so the result is bit-exact with the
 * definition.  K % 16 == 0.  Four stream-ordered launches; asynchronous on
 * `stream`. */
int q4_quantize_nvfp4(const void *W, q4_dtype w_dtype, void *payload, void *scales, float *scale2, int64_t N,
                      int64_t K, void *stream);

/* Q4_K quantization on the GPU (the write side of Q4_Q4K): W[N][K] (w_dtype
 * f32 or bf16, finite) -> 144-byte super-blocks out[N][K/256] in the Q4_Q4K
 * layout.  The pages fix the decode, w = d*s_j*q - dmin*m_j ([FBTC] sections
 * 5-6) but give no fitting recipe; this is the plainest per-sub-block
 * min/max fit that decode supports, every step one IEEE f32 operation:
 *   per 32-value sub-block j: lo = min(0, min w), scale_j = (max w - lo)/15,
 *                             min_j = -lo;
 *   d = binary16(max_j scale_j / 63), dmin = binary16(max_j min_j / 63),
 *       nearest even;
 *   s_j = clamp(rint(scale_j / d), 0, 63), m_j = clamp(rint(min_j / dmin), 0,
 *       63), 0 for a zero divisor;
 *   q = clamp(rint((w + dmin*m_j) / (d*s_j)), 0, 15), 0 for a zero step;
 * rint rounds half to even.  Bit-exact with that definition.  K % 256 == 0.
 * One launch; asynchronous on `stream`. */
int q4_quantize_q4k(const void *W, q4_dtype w_dtype, void *out, int64_t N, int64_t K, void *stream);

/* b-bit code streams ([BPA] "The packing arithmetic" and "Odd widths: 3-bit,
 * 2-bit and 6-bit"): code i (the low `bits` bits of codes[i], u8) occupies
 * bits [i*bits, (i+1)*bits) of one little-endian bit stream cut into 32-bit
 * words, so 3-, 5-, 6- and 7-bit codes may straddle two words.
 * q4_pack_bits writes words[n*bits/32]; q4_unpack_bits is its inverse.
 * 1 <= bits <= 8 and n * bits % 32 == 0 (Q4_EDIM otherwise).  Bit-exact;
 * asynchronous on `stream`. */
int q4_pack_bits(const uint8_t *codes, int64_t n, int bits, uint32_t *words, void *stream);
int q4_unpack_bits(const uint32_t *words, int64_t n, int bits, uint8_t *codes, void *stream);

/* The activation side of an act-order repack ([BPA] "Repacking between
 * formats": the weights' K permutation must be applied to the activations):
 * out[m][k] = x[m][perm[k]] for x[M][K] (x_dtype f32 or bf16), with perm the
 * perm_out of q4_repack (the source row of each target row).  out must not
 * alias x.  An index outside [0, K) is not read: that element becomes 0 and
 * q4_last_error() reports Q4_ERANGE.  Asynchronous on `stream`. */
int q4_permute_k(const void *x, q4_dtype x_dtype, const int32_t *perm, void *out, int64_t M, int64_t K,
                 void *stream);

/* out[N][K] = w_hat, f32 or bf16 per aux->out_dtype, by the pinned per-format
 * rule ([MUS7] 7.2 for NVFP4; the per-format sections cited above).  Bit-exact
 * with the definition.  Asynchronous on `stream`. */
int q4_dequant(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux,
               void *out, int64_t N, int64_t K, void *stream);

/* Repack through the logical matrix ([BPA] "Repacking between formats"):
 * unpack along the source's axis and order, normalise zero points (GPTQ +1),
 * resolve g_idx, pack along the target's.  Pairs provided:
 *   {GPTQ, AWQ, Q40, LOGICAL} -> {GPTQ, AWQ, LOGICAL}  (Q40 -> group 32, zero 8)
 *   NVFP4 <-> NVFP4_SPLITHALF                           (scales copied)
 * Outputs: dst_w, dst_scales (fp16 or E4M3 bytes), dst_zeros (GPTQ/AWQ i32,
 * LOGICAL u8; unused for NVFP4).  If src_aux->g_idx is not k/group (act-order),
 * rows are reordered so groups are contiguous (stable by k), every group must
 * hold exactly `group` rows (Q4_EDIM otherwise), and perm_out[K] (required)
 * receives the source row of each target row; the same permutation must be
 * applied to the layer's activations.  Otherwise perm_out may be NULL.
 * A GPTQ target cannot store zero 0 and an AWQ target cannot store 16: such a
 * tensor yields Q4_ERANGE after the call (the call then synchronizes on
 * `stream` to read the flag).  The result is bit-exact: q4_dequant of the
 * target equals q4_dequant of the source (with rows permuted if perm_out). */
int q4_repack(q4_fmt src, const void *src_w, const void *src_scales, const q4_aux *src_aux,
              q4_fmt dst, void *dst_w, void *dst_scales, void *dst_zeros, int32_t *perm_out,
              int64_t N, int64_t K, void *stream);

/* Fail-closed scan of the scale tensor ([MUS7] 7.3): counts NaN encodings
 * (E4M3FN 0x7f/0xff for NVFP4; E8M0 0xff for MXFP4; fp16 NaN/Inf in the d,
 * dmin of Q4_K/Q4_0 blocks and in GPTQ/AWQ scales) and checks NVFP4 scale2.
 * d_bad_count: caller-owned device int64 that receives the count.
 * SYNCHRONOUS on `stream`.  Returns Q4_OK, Q4_ENAN, Q4_ESCALE2 or a status. */
int q4_validate(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux,
                int64_t N, int64_t K, int64_t *d_bad_count, void *stream);

/* q4_validate without any device allocation by the caller.  The pages have
 * no counterpart; this exists for callers that cannot call cudaMalloc: a
 * loader inside a serving process whose device memory is owned by a
 * pre-sized pool or arena, a plugin handed tensors but no allocator, or code
 * that must avoid cudaMalloc's implicit synchronisation.  Same checks and
 * return codes as q4_validate; the count goes to a HOST int64 (`bad_count`,
 * may be NULL).  Its scratch is a fixed per-device array inside libq4.so
 * (Q4_VALIDATE_NOALLOC_MAX_CHUNKS x 8 B plus 8 B, held until the process
 * exits), one partial count per chunk of 16384 scale entries, so a tensor
 * may hold at most Q4_VALIDATE_NOALLOC_MAX_CHUNKS * 16384 scale entries
 * (268,435,456; an NVFP4 tensor of up to 2^32 weights); larger ones get
 * Q4_EDIM and nothing is launched.  The first call on a device looks up the
 * scratch address once with that device current; make that first call
 * before any stream capture.  Every call reuses the same array and overwrites
 * what it reads, so calls that overlap on the GPU (two streams or two host
 * threads) race and may report each other's counts.  SYNCHRONOUS on
 * `stream`; allocates nothing. */
#define Q4_VALIDATE_NOALLOC_MAX_CHUNKS 16384
int q4_validate_noalloc(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux,
                        int64_t N, int64_t K, int64_t *bad_count, void *stream);

/* Sticky device-side error of the current device (e.g. Q4_ETIMEOUT from a
 * bounded mbarrier wait in the tensor-core kernel, Q4_ERANGE from
 * q4_permute_k); reading it clears it.
 * Synchronizes the device. */
int q4_last_error(void);

/* Name of the kernel family the calling host thread's latest q4_gemv or
 * q4_gemv_grouped or q4_gemv_chain launched ("gemv_fp4tc",
 * "gemv_fp4tc_group", "gemv_tma", "gemv_tma_group",
 * "gemv_tma_chain", "gemm_tc", "gemv_mma", "gemv_mma_group", "gemv_mma_q4k",
 * "gemv_mma_q40", "gemv_mma_gptq", "gemv_rows_tma", "gemv_rows_m1",
 * "gemv_general", "gemv_kmajor", "gemv_awq_tc", "gemv_gptq_tc", "gemv_blk_tc_q4k",
 * "gemv_blk_tc_q40", "gemv_blk_tc_q4k_group", "gemv_blk_tc_q40_group"; "gemv_a16q8" or
 * "gemv_a16q8_tc" after q4_gemv_a16q8,
 * "gemv_q4k_q8" or "gemv_q4k_q8_tc" after q4_gemv_q4k_q8, "gemv_w4a4" after q4_gemv_w4a4,
 * "gemv_w4a4_tc" after q4_gemv_w4a4_tc; "" before
 * the first call).  A diagnostic with no counterpart in the pages: it lets a
 * caller (and the tests) confirm which path a shape takes.  Static storage. */
const char *q4_last_gemv_path(void);

/* Sets, for the current device, how long the bounded waits of the TMA-fed
 * kernels may spin before they give up: the waits between the roles of the
 * batch-1 FP4 tensor-core GEMV, of the batch 1-4 TMA GEMV and of the batch-1
 * Q4_K / Q4_0 TMA GEMV, and the grid barrier of q4_gemv_chain.  cycles <= 0 restores the default, 2^31 SM clocks
 * (about one second).  A wait that runs out records Q4_ETIMEOUT (read by
 * q4_last_error), the kernel's roles stop, the bulk copies and MMAs already
 * issued are waited for with the full limit, tensor memory is freed, and the
 * kernel returns: the context stays usable.  A diagnostic with no
 * counterpart in the pages, for exercising that path; synchronous; affects
 * every later launch on the device until reset. */
int q4_set_wait_limit(int64_t cycles);

/* Human-readable text of a status code (static storage). */
const char *q4_strerror(int status);

/* Bytes of the packed payload plus scale tensor (plus zeros for GPTQ/AWQ,
 * plus 4 for NVFP4's scale2) for an N x K tensor with group 128: the
 * algorithmic bytes a GEMV must stream.  0 for invalid sizes. */
size_t q4_packed_bytes(q4_fmt fmt, int64_t N, int64_t K);

/* Library version string. */
const char *q4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* Q4_H */
