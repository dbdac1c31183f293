/*
 * q4_oracle.c -- plain, slow CPU oracle for the 4-bit block formats.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the bench's CPU-baseline leg
 * do.  It shares no code, header, table or constant with the CUDA library.
 *
 * Every decoder is written from the bit-level definition the source pages give
 * (cited per function as "page title, section"), one weight at a time, in
 * scalar C.  Dequantized weights are f32 exactly as the pages pin them; GEMV
 * accumulates in f64.  Build with -ffp-contract=off so that no product/sum is
 * fused behind our back: the pinned orders below have one rounding each.
 *
 * Page titles used in citations:
 *   [FBTC]  "Four Bits, Three Contracts" (shivasnotes.com/blog/6006)
 *   [W4K]   "Why 4-Bit Quantization Is King" (shivasnotes.com/blog/5996)
 *   [BPA]   "Bit Packing Architecture, in depth" (aicassindra.com quant_bit_packing)
 *   [MUS7]  "Muser book, Chapter 7 - NVFP4: the native lane" (highperformanceailab.com)
 *
 * Parity status: every function below is pinned (printed worked examples,
 * library decoders, brute force, invariants) by tests/test_oracle_pins.py, and
 * the A16-Q8, W4A8, W4A4 and quantizer functions by test_oracle_a16q8.py,
 * test_oracle_w4a8.py, test_oracle_w4a4.py and test_oracle_quantize.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { F_NVFP4 = 1, F_MXFP4 = 2, F_Q4K = 3, F_Q40 = 4, F_GPTQ = 5, F_AWQ = 6,
       F_NVFP4_SPLITHALF = 7, F_LOGICAL = 8 };

/* ---------------------------------------------------------------- scalars */

/* E2M1 element, [FBTC] section 1 and [MUS7] 7.1: one sign bit, two exponent
 * bits (bias 1), one fraction bit.  Exponent field 0 is the subnormal/zero
 * case worth fraction * 0.5; otherwise 2^(e-1) * (1 + fraction/2).  Bit 3 is
 * the sign, so code 8 is negative zero. */
float orc_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, f = code & 1u;
    float mag;
    if (e == 0)
        mag = 0.5f * (float)f;
    else
        mag = ldexpf(1.0f + 0.5f * (float)f, (int)e - 1);
    return s ? -mag : mag;
}

/* E4M3FN scale byte, [FBTC] section 4 and [MUS7] 7.1: sign, four exponent bits
 * (bias 7), three fraction bits, no infinities; only 0x7f and 0xff are NaN.
 * Exponent field 0 is subnormal: fraction/8 * 2^(1-7).  Returns 1 for a NaN
 * encoding (the pages' loader refuses those), 0 otherwise. */
int orc_e4m3fn(unsigned byte, float *out)
{
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, f = byte & 7u;
    float mag;
    if (e == 15u && f == 7u) {
        *out = NAN;
        return 1;
    }
    if (e == 0)
        mag = ldexpf((float)f / 8.0f, 1 - 7);
    else
        mag = ldexpf(1.0f + (float)f / 8.0f, (int)e - 7);
    *out = s ? -mag : mag;
    return 0;
}

/* E8M0 scale byte, [FBTC] section 3: 2^(byte-127) for 0..254; 255 is NaN and
 * there is no zero.  Returns 1 for the NaN encoding. */
int orc_e8m0(unsigned byte, float *out)
{
    if (byte == 255u) {
        *out = NAN;
        return 1;
    }
    *out = ldexpf(1.0f, (int)byte - 127);
    return 0;
}

/* IEEE-754 binary16 (the fp16 d/dmin of Q4_K/Q4_0 and the GPTQ/AWQ scales),
 * decoded from the standard's definition: 5 exponent bits (bias 15), 10
 * fraction bits, exponent 0 subnormal, exponent 31 inf/NaN. */
float orc_half(uint16_t h)
{
    unsigned s = (h >> 15) & 1u, e = (h >> 10) & 31u, f = h & 1023u;
    float mag;
    if (e == 0)
        mag = ldexpf((float)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexpf(1.0f + (float)f / 1024.0f, (int)e - 15);
    return s ? -mag : mag;
}

/* bfloat16 is by definition the upper half of an IEEE binary32. */
float orc_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round an f32 to bfloat16, nearest-even; NaN stays a quiet NaN. */
uint16_t orc_round_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu, upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t rd32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* ---------------------------------------------------------------- tensors */

typedef struct {
    int32_t fmt;
    int32_t group;          /* GPTQ / AWQ / LOGICAL quantization group along K */
    int64_t N, K;           /* logical W is [N out][K in] */
    const uint8_t *w;       /* packed payload, little-endian bytes */
    const uint8_t *scales;  /* per-format scale tensor (unused for Q4_K, Q4_0) */
    const uint8_t *zeros;   /* GPTQ/AWQ qzeros (int32 words) or LOGICAL u8 zeros */
    const int32_t *g_idx;   /* optional [K] group index (GPTQ, LOGICAL); NULL = k/group */
    float scale2;           /* NVFP4 per-tensor f32 scale */
} orc_tensor;

/* NVFP4 weight (n,k), [MUS7] 7.1-7.2: payload [N][K/2] with the even index in
 * the low nibble, one E4M3FN scale per 16 values in [N][K/16], one f32 scale2;
 * the product order is pinned to (e2m1 * e4m3fn) * scale2 in f32.
 * Split-half variant, [W4K] section 5: inside each 16-value group the low
 * nibbles of the group's 8 bytes hold lanes 0-7 and the high nibbles lanes 8-15. */
static int nvfp4_weight(const orc_tensor *t, int64_t n, int64_t k, int split_half, float *out)
{
    const uint8_t *row = t->w + n * (t->K / 2);
    unsigned code;
    if (!split_half) {
        uint8_t b = row[k / 2];
        code = (k % 2 == 0) ? (b & 15u) : (b >> 4);
    } else {
        int64_t g = k / 16, lane = k % 16;
        uint8_t b = row[g * 8 + (lane % 8)];
        code = (lane < 8) ? (b & 15u) : (b >> 4);
    }
    float s;
    if (orc_e4m3fn(t->scales[n * (t->K / 16) + k / 16], &s))
        return 1;
    float p = orc_e2m1(code) * s;   /* exact: at most 2 x 4 significant bits */
    *out = p * t->scale2;           /* the single rounding of the pinned order */
    return 0;
}

/* MXFP4 weight (n,k), [FBTC] section 3: 32 E2M1 codes share one E8M0 scale.
 * Byte layout (a reading: the page fixes only group semantics): payload
 * [N][K/2] even index in the low nibble, scales [N][K/32]. */
static int mxfp4_weight(const orc_tensor *t, int64_t n, int64_t k, float *out)
{
    uint8_t b = t->w[n * (t->K / 2) + k / 2];
    unsigned code = (k % 2 == 0) ? (b & 15u) : (b >> 4);
    float s;
    if (orc_e8m0(t->scales[n * (t->K / 32) + k / 32], &s))
        return 1;
    *out = orc_e2m1(code) * s;
    return 0;
}

/* Q4_K 6-bit sub-block scale/min j from the 12 metadata bytes B,
 * [FBTC] section 6: j<4 keep the low six bits of B[j] / B[j+4]; j>=4 combine
 * four bits of B[j+4] with the top two bits of B[j-4] / B[j]. */
static void q4k_scale_min(const uint8_t *B, int j, unsigned *sc, unsigned *mn)
{
    if (j < 4) {
        *sc = B[j] & 63u;
        *mn = B[j + 4] & 63u;
    } else {
        *sc = (B[j + 4] & 15u) | ((unsigned)(B[j - 4] >> 6) << 4);
        *mn = (unsigned)(B[j + 4] >> 4) | ((unsigned)(B[j] >> 6) << 4);
    }
}

/* Q4_K weight (n,k), [FBTC] sections 5-6 and [W4K] section 4: 144-byte
 * super-block of 256 weights = fp16 d @0, fp16 dmin @2, 12 metadata bytes @4,
 * 128 code bytes @16 (byte order is a reading; the pages give field sizes).
 * Output position 64c+l takes the low nibble of code byte 32c+l (sub-block
 * 2c); 64c+32+l takes its high nibble (sub-block 2c+1).
 * w = (d*s_j)*q - dmin*m_j: both products are exact in f32, so the one
 * subtraction is the only rounding. */
static int q4k_weight(const orc_tensor *t, int64_t n, int64_t k, float *out)
{
    int64_t blocks_per_row = t->K / 256;
    const uint8_t *blk = t->w + (n * blocks_per_row + k / 256) * 144;
    int i = (int)(k % 256), c = i / 64, r = i % 64;
    int hi = r >= 32;
    uint8_t b = blk[16 + 32 * c + (r % 32)];
    unsigned q = hi ? (b >> 4) : (b & 15u);
    unsigned sc, mn;
    q4k_scale_min(blk + 4, 2 * c + hi, &sc, &mn);
    float d = orc_half(rd16(blk)), dmin = orc_half(rd16(blk + 2));
    float step = d * (float)sc;
    float off = dmin * (float)mn;
    float qs = step * (float)q;
    *out = qs - off;
    return 0;
}

/* Q4_0 weight (n,k), [BPA] "Real layouts compared": 18-byte block of 32 =
 * fp16 d then 16 code bytes; byte j holds element j (low nibble) and element
 * j+16 (high nibble); w = d * (q - 8). */
static int q40_weight(const orc_tensor *t, int64_t n, int64_t k, float *out)
{
    const uint8_t *blk = t->w + (n * (t->K / 32) + k / 32) * 18;
    int i = (int)(k % 32);
    uint8_t b = blk[2 + (i % 16)];
    unsigned q = (i < 16) ? (b & 15u) : (b >> 4);
    *out = orc_half(rd16(blk)) * (float)((int)q - 8);
    return 0;
}

static int64_t group_of(const orc_tensor *t, int64_t k)
{
    return t->g_idx ? (int64_t)t->g_idx[k] : k / t->group;
}

/* GPTQ weight (n,k), [BPA] "Real layouts compared": qweight int32 [K/8][N]
 * packed along K, row 8r+j at bits 4j; scales fp16 [groups][N]; qzeros int32
 * packed along N (slot n%8 at bits 4*(n%8), a reading: the page says only
 * "packed along the output dimension"), stored as zero-1; g_idx maps k to its
 * group.  Shifts are unsigned ([BPA] "Vectorised packers": the top slot holds
 * the sign bit).  w = scale * (q - zero). */
static int gptq_weight(const orc_tensor *t, int64_t n, int64_t k, float *out)
{
    int64_t N = t->N, g = group_of(t, k);
    uint32_t word = rd32(t->w + ((k / 8) * N + n) * 4);
    unsigned q = (word >> (4 * (k % 8))) & 15u;
    uint32_t zw = rd32(t->zeros + (g * (N / 8) + n / 8) * 4);
    int z = (int)((zw >> (4 * (n % 8))) & 15u) + 1;
    float s = orc_half(rd16(t->scales + (g * N + n) * 2));
    *out = s * (float)((int)q - z);
    return 0;
}

/* AWQ weight (n,k), [BPA] "Real layouts compared": qweight int32 [K][N/8]
 * packed along N with logical columns in slot order 0,2,4,6,1,3,5,7 (slot p
 * at bits 4p holds column AWQ_ORDER[p]).  qzeros int32 [K/group][N/8] use the
 * same interleave with no minus-one (a reading: the page describes qweight).
 * scales fp16 [K/group][N]. */
static const int AWQ_ORDER[8] = {0, 2, 4, 6, 1, 3, 5, 7};

static int awq_slot_of_column(int col)
{
    for (int p = 0; p < 8; p++)
        if (AWQ_ORDER[p] == col)
            return p;
    return -1;
}

static int awq_weight(const orc_tensor *t, int64_t n, int64_t k, float *out)
{
    int64_t N = t->N, g = k / t->group;
    int p = awq_slot_of_column((int)(n % 8));
    uint32_t word = rd32(t->w + (k * (N / 8) + n / 8) * 4);
    unsigned q = (word >> (4 * p)) & 15u;
    uint32_t zw = rd32(t->zeros + (g * (N / 8) + n / 8) * 4);
    int z = (int)((zw >> (4 * p)) & 15u);
    float s = orc_half(rd16(t->scales + (g * N + n) * 2));
    *out = s * (float)((int)q - z);
    return 0;
}

/* The logical matrix of [BPA] "Repacking between formats": u8 codes [K][N],
 * fp16 scales [groups][N], u8 zeros [groups][N], w = scale * (q - zero). */
static int logical_weight(const orc_tensor *t, int64_t n, int64_t k, float *out)
{
    int64_t N = t->N, g = group_of(t, k);
    int q = t->w[k * N + n];
    int z = t->zeros[g * N + n];
    float s = orc_half(rd16(t->scales + (g * N + n) * 2));
    *out = s * (float)(q - z);
    return 0;
}

static int weight_at(const orc_tensor *t, int64_t n, int64_t k, float *out)
{
    switch (t->fmt) {
    case F_NVFP4: return nvfp4_weight(t, n, k, 0, out);
    case F_NVFP4_SPLITHALF: return nvfp4_weight(t, n, k, 1, out);
    case F_MXFP4: return mxfp4_weight(t, n, k, out);
    case F_Q4K: return q4k_weight(t, n, k, out);
    case F_Q40: return q40_weight(t, n, k, out);
    case F_GPTQ: return gptq_weight(t, n, k, out);
    case F_AWQ: return awq_weight(t, n, k, out);
    case F_LOGICAL: return logical_weight(t, n, k, out);
    default: return 2;
    }
}

/* ------------------------------------------------------------- public API */

/* Dequantize logical rows [n0, n0+nrows) into out[nrows][K] (f32).
 * Returns 0, 1 if a scale byte is a NaN encoding, 2 for an unknown format. */
int orc_dequant_rows(const orc_tensor *t, int64_t n0, int64_t nrows, float *out)
{
    for (int64_t i = 0; i < nrows; i++)
        for (int64_t k = 0; k < t->K; k++) {
            int rc = weight_at(t, n0 + i, k, &out[i * t->K + k]);
            if (rc)
                return rc;
        }
    return 0;
}

/* y[m][i] = sum_k w_hat[rows[i]][k] * x[m][k] accumulated in f64, and
 * bound[m][i] = sum_k |w_hat| * |x| (the scale of the GEMV tolerance).
 * x is [M][K] f32 (bf16 activations are passed already widened, exactly).
 * The fused decode + dot of [W4K] section 1: the weight is reconstructed by
 * the pinned rule, then multiplied and accumulated in a wider type. */
int orc_gemv_rows(const orc_tensor *t, const float *x, int64_t M,
                  const int64_t *rows, int64_t nrows, double *y, double *bound)
{
    for (int64_t i = 0; i < nrows; i++) {
        for (int64_t m = 0; m < M; m++) {
            y[m * nrows + i] = 0.0;
            bound[m * nrows + i] = 0.0;
        }
        for (int64_t k = 0; k < t->K; k++) {
            float w;
            int rc = weight_at(t, rows[i], k, &w);
            if (rc)
                return rc;
            for (int64_t m = 0; m < M; m++) {
                double xv = (double)x[m * t->K + k];
                y[m * nrows + i] += (double)w * xv;
                bound[m * nrows + i] += fabs((double)w) * fabs(xv);
            }
        }
    }
    return 0;
}

/* Round an f32 array to bfloat16 bits (nearest-even), for the bf16 output of
 * dequantization. */
void orc_round_bf16_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_round_bf16(in[i]);
}

/* Count NaN scale encodings, the fail-closed check of [MUS7] 7.3. */
int64_t orc_count_nan_scales(int fmt, const uint8_t *scales, int64_t count)
{
    int64_t bad = 0;
    float v;
    for (int64_t i = 0; i < count; i++) {
        if (fmt == F_MXFP4)
            bad += orc_e8m0(scales[i], &v);
        else
            bad += orc_e4m3fn(scales[i], &v);
    }
    return bad;
}

/* ------------------------------------------ the integer-exact A16-Q8 lane */

/* E2M1 code as an integer count of halves: the weight encoding of the
 * weight-only contraction in [MUS7] 7.4.2.  The smallest nonzero E2M1 value
 * is 1/2, so every value is an integer multiple of it: 2*v(code), which is
 * f for exponent field 0 and (2+f) << (e-1) otherwise; bit 3 is the sign. */
int orc_e2m1_q1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, f = code & 1u;
    int mag = (e == 0) ? (int)f : (int)((2u + f) << (e - 1u));
    return s ? -mag : mag;
}

/* E4M3FN byte as an integer count of 2^-9 (the smallest subnormal), the
 * scale encoding of [MUS7] 7.4.2: f for exponent field 0, else
 * (1 + f/8) * 2^(e-7) / 2^-9 = (8+f) << (e-1); bit 7 is the sign.
 * Returns 1 for a NaN encoding (0x7f / 0xff). */
int orc_e4m3fn_q9(unsigned byte, int32_t *out)
{
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, f = byte & 7u;
    if (e == 15u && f == 7u) {
        *out = 0;
        return 1;
    }
    int32_t mag = (e == 0) ? (int32_t)f : (int32_t)((8u + f) << (e - 1u));
    *out = s ? -mag : mag;
    return 0;
}

/* One 256-value activation block onto the signed 8-bit grid, [MUS7] 7.4.2:
 * first_max is the signed value of the first element of largest magnitude,
 * iscale = -127 / first_max, each code is x * iscale (rounded to f32) rounded
 * half-to-even to an integer and capped at 127, and the block's scale is
 * 1 / iscale.  Reading: a block whose iscale is not finite (first_max zero,
 * or so small that -127 / first_max overflows) takes all-zero codes and
 * scale 0. */
void orc_q8_block(const float *x, int8_t *q, float *scale)
{
    float first_max = 0.0f, amax = 0.0f;
    for (int i = 0; i < 256; i++) {
        float a = fabsf(x[i]);
        if (a > amax) {
            amax = a;
            first_max = x[i];
        }
    }
    float iscale = -127.0f / first_max;
    if (!isfinite(iscale)) {
        for (int i = 0; i < 256; i++)
            q[i] = 0;
        *scale = 0.0f;
        return;
    }
    for (int i = 0; i < 256; i++) {
        float v = x[i] * iscale;
        long r = lrintf(v);             /* default rounding mode: half to even */
        q[i] = (int8_t)(r > 127 ? 127 : r);
    }
    *scale = 1.0f / iscale;
}

/* f32 -> nearest IEEE binary16 value (ties to even, gradual underflow,
 * overflow to infinity), returned widened to f32.  Written from the binary16
 * definition: values of binade [2^E, 2^(E+1)) sit on a grid of 2^(E-10), and
 * below 2^-14 on the subnormal grid 2^-24; the largest finite value is 65504.
 * The scaled quotient is exact in double, so nearbyint makes the one rounding. */
float orc_f16_round(float f)
{
    if (isnan(f))
        return f;
    double a = fabs((double)f);
    if (a == 0.0)
        return f;
    int ex;
    frexp(a, &ex);                      /* a = m * 2^ex, m in [0.5, 1) */
    int E = ex - 1;
    if (E > 15)
        return f > 0 ? INFINITY : -INFINITY;
    double quantum = ldexp(1.0, (E < -14 ? -14 : E) - 10);
    double r = nearbyint(a / quantum) * quantum;
    if (r > 65504.0)
        return f > 0 ? INFINITY : -INFINITY;
    return (float)(f > 0 ? r : -r);
}

/* The weight-only NVFP4 contraction of [MUS7] 7.4.2 for logical rows
 * rows[0..nrows) and activation rows x[0..M) (f32 [M][K], bf16 passed
 * widened).  Each activation row is first cut into 256-value blocks and
 * quantized by orc_q8_block.  For output row n and block b,
 *   T_b = sum over the block's 16 groups g of
 *         q9(scale[n][g]) * sum_{k in g} q1(code[n][k]) * q8[m][k]
 * is an exact 64-bit integer; its value is T_b * 2^-10 (halves times 2^-9)
 * in units of the block's activation scale.  The floating-point epilogue is
 * the page's four steps, in block order:
 *   c = fma(float(T_b), 2^-10, 0); c = fma(c, act_scale_b, 0);
 *   c = fma(c, scale2, 0);         total = fma(1, c, total)
 * and the output is total rounded to binary16 (stored widened, f32).
 * Returns 0; 1 if a scale byte is a NaN encoding; 2 if the tensor is not
 * NVFP4 or K is not a multiple of 256; 3 if memory runs out. */
int orc_gemv_a16q8_rows(const orc_tensor *t, const float *x, int64_t M,
                        const int64_t *rows, int64_t nrows, float *y)
{
    if (t->fmt != F_NVFP4 || t->K % 256 != 0)
        return 2;
    const int64_t K = t->K, nb = K / 256;
    int8_t *q8 = (int8_t *)malloc((size_t)(M * K));
    float *act_scale = (float *)malloc((size_t)(M * nb) * sizeof(float));
    if (!q8 || !act_scale) {
        free(q8);
        free(act_scale);
        return 3;
    }
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++)
            orc_q8_block(x + m * K + b * 256, q8 + m * K + b * 256, act_scale + m * nb + b);
    int rc = 0;
    for (int64_t i = 0; i < nrows && !rc; i++) {
        const int64_t n = rows[i];
        const uint8_t *row = t->w + n * (K / 2);
        const uint8_t *srow = t->scales + n * (K / 16);
        for (int64_t m = 0; m < M && !rc; m++) {
            float total = 0.0f;
            for (int64_t b = 0; b < nb; b++) {
                int64_t T = 0;
                for (int64_t g = b * 16; g < b * 16 + 16; g++) {
                    int32_t q9;
                    if (orc_e4m3fn_q9(srow[g], &q9)) {
                        rc = 1;
                        break;
                    }
                    int64_t dot = 0;
                    for (int64_t k = g * 16; k < g * 16 + 16; k++) {
                        uint8_t byte = row[k / 2];
                        unsigned code = (k % 2 == 0) ? (byte & 15u) : (byte >> 4);
                        dot += (int64_t)orc_e2m1_q1(code) * (int64_t)q8[m * K + k];
                    }
                    T += dot * (int64_t)q9;
                }
                if (rc)
                    break;
                float c = fmaf((float)T, 0x1p-10f, 0.0f);
                c = fmaf(c, act_scale[m * nb + b], 0.0f);
                c = fmaf(c, t->scale2, 0.0f);
                total = fmaf(1.0f, c, total);
            }
            y[m * nrows + i] = orc_f16_round(total);
        }
    }
    free(q8);
    free(act_scale);
    return rc;
}

/* The Q4_K x Q8 contraction of [W4K] section 7 ("W4A8" and the CKE
 * Q4_K x Q8_K route of 7b-7c): activations quantized per 256-value block
 * (orc_q8_block, the same signed-first-maximum grid), weights kept as the
 * unsigned 4-bit codes of each 32-value sub-block j.  Per super-block, two
 * exact integers:
 *   I1 = sum_j sc_j * sum_{k in j} q[k] * q8[k]     (scaled integer dot)
 *   I2 = sum_j m_j  * sum_{k in j} q8[k]            (minimum term, activation sums)
 * then, in f32 and in the order the section names the steps (a reading: the
 * section does not pin the rounding order):
 *   v = f32(d) * float(I1) - f32(dmin) * float(I2);  c = v * act_scale;
 *   total = total + c   (super-blocks in order).
 * Algebraically sum_k w_hat[k] * (q8[k] * act_scale), the section's
 * s_x (d s_j) sum q_w q_x - s_x (dmin m_j) sum q_x.  Output f32.
 * Returns 0; 2 if the tensor is not Q4_K; 3 if memory runs out. */
int orc_gemv_q4k_q8_rows(const orc_tensor *t, const float *x, int64_t M,
                         const int64_t *rows, int64_t nrows, float *y)
{
    if (t->fmt != F_Q4K || t->K % 256 != 0)
        return 2;
    const int64_t K = t->K, nb = K / 256;
    int8_t *q8 = (int8_t *)malloc((size_t)(M * K));
    float *act_scale = (float *)malloc((size_t)(M * nb) * sizeof(float));
    if (!q8 || !act_scale) {
        free(q8);
        free(act_scale);
        return 3;
    }
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++)
            orc_q8_block(x + m * K + b * 256, q8 + m * K + b * 256, act_scale + m * nb + b);
    for (int64_t i = 0; i < nrows; i++) {
        const int64_t n = rows[i];
        for (int64_t m = 0; m < M; m++) {
            float total = 0.0f;
            for (int64_t b = 0; b < nb; b++) {
                const uint8_t *blk = t->w + (n * nb + b) * 144;
                const int8_t *qx = q8 + m * K + b * 256;
                int64_t I1 = 0, I2 = 0;
                for (int j = 0; j < 8; j++) {
                    unsigned sc, mn;
                    q4k_scale_min(blk + 4, j, &sc, &mn);
                    int64_t dot = 0, bsum = 0;
                    for (int l = 0; l < 32; l++) {
                        /* sub-block j = 2c + hi: code byte 32c + l, k = 32j + l */
                        uint8_t byte = blk[16 + 32 * (j / 2) + l];
                        unsigned q = (j % 2) ? (byte >> 4) : (byte & 15u);
                        dot += (int64_t)q * qx[32 * j + l];
                        bsum += qx[32 * j + l];
                    }
                    I1 += (int64_t)sc * dot;
                    I2 += (int64_t)mn * bsum;
                }
                float d = orc_half(rd16(blk)), dmin = orc_half(rd16(blk + 2));
                float p1 = d * (float)I1;
                float p2 = dmin * (float)I2;
                float v = p1 - p2;
                float c = v * act_scale[m * nb + b];
                total = total + c;
            }
            y[m * nrows + i] = total;
        }
    }
    free(q8);
    free(act_scale);
    return 0;
}

/* ------------------------------------------------- the NVFP4 quantizer */

/* Nearest E2M1 code to r ([MUS7] 7.2: ModelOpt's midpoints, ties to the even
 * code), by search over the eight magnitudes; magnitudes above 6 saturate to
 * 6.  The sign bit follows r, so a negative value that rounds to zero keeps
 * it (code 8).  NaN is outside the definition. */
unsigned orc_e2m1_round(float r)
{
    double a = fabs((double)r);
    unsigned best = 0;
    double best_err = INFINITY;
    if (a >= 6.0)                       /* saturate (far values would tie in double) */
        return 7u | (signbit(r) ? 8u : 0u);
    for (unsigned c = 0; c < 8; c++) {
        double err = fabs(a - (double)orc_e2m1(c));
        if (err < best_err || (err == best_err && (c & 1u) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return best | (signbit(r) ? 8u : 0u);
}

/* Nearest E4M3FN byte to v, ties to the even byte (fraction bit 0 clear), by
 * search over the 127 non-negative finite encodings; magnitudes beyond 448
 * saturate to 448 (0x7e), so no NaN encoding is produced.  The sign bit
 * follows v. */
unsigned orc_e4m3fn_round(float v)
{
    double a = fabs((double)v);
    unsigned best = 0;
    double best_err = INFINITY;
    if (a >= 448.0)
        return 0x7eu | (signbit(v) ? 0x80u : 0u);
    for (unsigned b = 0; b <= 0x7eu; b++) {
        float s;
        orc_e4m3fn(b, &s);
        double err = fabs(a - (double)s);
        if (err < best_err || (err == best_err && (b & 1u) == 0)) {
            best = b;
            best_err = err;
        }
    }
    return best | (signbit(v) ? 0x80u : 0u);
}

/* NVFP4 groups of W [N][K] (f32, finite, K % 16 == 0) for a given tensor
 * scale: per 16-value group, scale byte = E4M3FN nearest-even of
 * (amax_group / 6) / scale2, saturating at 448; each code = E2M1 nearest-even
 * of w / (dec(scale byte) * scale2), every step an f32 operation; a group
 * whose scale decodes to 0 takes code 0 throughout.  Payload with the even k
 * in the low nibble ([MUS7] 7.1). */
void orc_quantize_nvfp4_groups(const float *W, int64_t N, int64_t K, float scale2, uint8_t *payload,
                               uint8_t *scales)
{
    for (int64_t n = 0; n < N; n++)
        for (int64_t g = 0; g < K / 16; g++) {
            const float *w = W + n * K + g * 16;
            float amax_g = 0.0f;
            for (int i = 0; i < 16; i++)
                if (fabsf(w[i]) > amax_g)
                    amax_g = fabsf(w[i]);
            float sv = amax_g / 6.0f;
            sv = sv / scale2;
            unsigned sb = orc_e4m3fn_round(sv);
            float s;
            orc_e4m3fn(sb, &s);
            float denom = s * scale2;
            scales[n * (K / 16) + g] = (uint8_t)sb;
            for (int i = 0; i < 16; i += 2) {
                unsigned c0 = 0, c1 = 0;
                if (denom > 0.0f) {
                    c0 = orc_e2m1_round(w[i] / denom);
                    c1 = orc_e2m1_round(w[i + 1] / denom);
                }
                payload[n * (K / 2) + g * 8 + i / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
}

/* NVFP4 quantization of W [N][K] by the recipe the weights of this build are
 * stated in: scale2 = amax(W) / (448 * 6) in f32 (1 for an all-zero W), then
 * the groups as above. */
void orc_quantize_nvfp4(const float *W, int64_t N, int64_t K, uint8_t *payload, uint8_t *scales,
                        float *scale2_out)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < N * K; i++)
        if (fabsf(W[i]) > amax)
            amax = fabsf(W[i]);
    const float scale2 = amax > 0.0f ? amax / 2688.0f : 1.0f;
    *scale2_out = scale2;
    orc_quantize_nvfp4_groups(W, N, K, scale2, payload, scales);
}

/* The W4A4 contraction of [MUS7] 7.4.3.  Each activation row is quantized to
 * NVFP4 in groups of 16 with the tensor scale G = 1 / input_scale_inv (f32),
 * by the same rule as the weights (orc_quantize_nvfp4_groups).  Per group g of
 * output row n the product of the four integer encodings
 *   T_g = q9(sw) * q9(sx) * sum_{k in g} q1(w_k) * q1(x_k)
 * is exact in 64 bits with denominator 2^-20 (halves x halves x 2^-9 x 2^-9).
 * Epilogue per group, in group order (a reading: the section names the
 * factors, the per-group i64 sum and the binary16 output):
 *   c = fma(float(T_g), 2^-20, 0); c = fma(c, scale2, 0); c = fma(c, G, 0);
 *   total = fma(1, c, total)
 * and y = total rounded to binary16 (stored widened, f32).
 * Returns 0; 1 for a NaN weight-scale encoding; 2 for a non-NVFP4 tensor or
 * an input_scale_inv that is not finite and > 0; 3 if memory runs out. */
int orc_gemv_w4a4_rows(const orc_tensor *t, const float *x, int64_t M, float input_scale_inv,
                       const int64_t *rows, int64_t nrows, float *y)
{
    if (t->fmt != F_NVFP4 || !(input_scale_inv > 0.0f) || !isfinite(input_scale_inv))
        return 2;
    const int64_t K = t->K, ng = K / 16;
    const float G = 1.0f / input_scale_inv;
    uint8_t *xp = (uint8_t *)malloc((size_t)(M * K / 2));
    uint8_t *xs = (uint8_t *)malloc((size_t)(M * ng));
    if (!xp || !xs) {
        free(xp);
        free(xs);
        return 3;
    }
    orc_quantize_nvfp4_groups(x, M, K, G, xp, xs);
    int rc = 0;
    for (int64_t i = 0; i < nrows && !rc; i++) {
        const int64_t n = rows[i];
        const uint8_t *wrow = t->w + n * (K / 2), *srow = t->scales + n * ng;
        for (int64_t m = 0; m < M && !rc; m++) {
            const uint8_t *xrow = xp + m * (K / 2), *xsrow = xs + m * ng;
            float total = 0.0f;
            for (int64_t g = 0; g < ng; g++) {
                int32_t q9w, q9x;
                if (orc_e4m3fn_q9(srow[g], &q9w)) {
                    rc = 1;
                    break;
                }
                orc_e4m3fn_q9(xsrow[g], &q9x);       /* produced by the quantizer: never NaN */
                int64_t dot = 0;
                for (int64_t k = g * 16; k < g * 16 + 16; k++) {
                    unsigned cw = (k % 2 == 0) ? (wrow[k / 2] & 15u) : (wrow[k / 2] >> 4);
                    unsigned cx = (k % 2 == 0) ? (xrow[k / 2] & 15u) : (xrow[k / 2] >> 4);
                    dot += (int64_t)orc_e2m1_q1(cw) * (int64_t)orc_e2m1_q1(cx);
                }
                int64_t T = dot * (int64_t)q9w * (int64_t)q9x;
                float c = fmaf((float)T, 0x1p-20f, 0.0f);
                c = fmaf(c, t->scale2, 0.0f);
                c = fmaf(c, G, 0.0f);
                total = fmaf(1.0f, c, total);
            }
            y[m * nrows + i] = orc_f16_round(total);
        }
    }
    free(xp);
    free(xs);
    return rc;
}

/* ------------------------------------------------ the Q4_K fit (write side) */

/* binary16 bit pattern of f32 f rounded to nearest, ties to even (the value
 * is orc_f16_round's; this returns its encoding). */
uint16_t orc_f16_bits(float f)
{
    float r = orc_f16_round(f);
    uint16_t sign = signbit(r) ? 0x8000u : 0u;
    double a = fabs((double)r);
    if (isnan(r))
        return 0x7e00u;
    if (isinf(r))
        return sign | 0x7c00u;
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);
    int E = ex - 1;
    if (E < -14)                                  /* subnormal: a multiple of 2^-24 */
        return sign | (uint16_t)nearbyint(a / ldexp(1.0, -24));
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)(nearbyint(a / ldexp(1.0, E - 10)) - 1024.0);
}

/* Q4_K super-blocks of W [N][K] (f32, finite, K % 256 == 0) by a per-sub-block
 * min/max fit.  The pages give the decode, w = d*s_j*q - dmin*m_j ([FBTC]
 * sections 5-6, [W4K] section 4), but no fitting recipe; this one is the
 * plainest that the decode supports, every step one f32 operation:
 *   per sub-block j of 32:  lo_j = min(0, min w),  scale_j = (max w - lo_j) / 15,
 *                           min_j = -lo_j;
 *   d = fp16(max_j scale_j / 63),  dmin = fp16(max_j min_j / 63)  (nearest even);
 *   s_j = clamp(rint(scale_j / d), 0, 63) and m_j = clamp(rint(min_j / dmin), 0, 63)
 *         (0 when the divisor is 0);
 *   q = clamp(rint((w + dmin*m_j) / (d*s_j)), 0, 15)  (0 when d*s_j is 0);
 * rint rounds half to even.  The 12 metadata bytes are the inverse of the
 * decode's unpacking: for j < 4, B[j] = s_j | (s_{j+4} >> 4) << 6 and
 * B[j+4] = m_j | (m_{j+4} >> 4) << 6; B[j+8] = (s_{j+4} & 15) | (m_{j+4} & 15) << 4.
 * Code byte 32c + l holds k = 64c + l (low nibble) and 64c + 32 + l (high). */
void orc_quantize_q4k(const float *W, int64_t N, int64_t K, uint8_t *out)
{
    const int64_t nb = K / 256;
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            const float *w = W + n * K + b * 256;
            uint8_t *blk = out + (n * nb + b) * 144;
            float scale[8], mins[8], smax = 0.0f, mmax = 0.0f;
            for (int j = 0; j < 8; j++) {
                float lo = 0.0f, hi = w[32 * j];
                for (int i = 0; i < 32; i++) {
                    if (w[32 * j + i] < lo)
                        lo = w[32 * j + i];
                    if (w[32 * j + i] > hi)
                        hi = w[32 * j + i];
                }
                scale[j] = (hi - lo) / 15.0f;
                mins[j] = -lo;
                if (scale[j] > smax)
                    smax = scale[j];
                if (mins[j] > mmax)
                    mmax = mins[j];
            }
            const uint16_t dbits = orc_f16_bits(smax / 63.0f), mbits = orc_f16_bits(mmax / 63.0f);
            const float d = orc_half(dbits), dmin = orc_half(mbits);
            unsigned s[8], m[8];
            for (int j = 0; j < 8; j++) {
                float a = d > 0.0f ? nearbyintf(scale[j] / d) : 0.0f;
                float c = dmin > 0.0f ? nearbyintf(mins[j] / dmin) : 0.0f;
                s[j] = a < 0.0f ? 0u : a > 63.0f ? 63u : (unsigned)a;
                m[j] = c < 0.0f ? 0u : c > 63.0f ? 63u : (unsigned)c;
            }
            blk[0] = (uint8_t)(dbits & 0xffu);
            blk[1] = (uint8_t)(dbits >> 8);
            blk[2] = (uint8_t)(mbits & 0xffu);
            blk[3] = (uint8_t)(mbits >> 8);
            for (int j = 0; j < 4; j++) {
                blk[4 + j] = (uint8_t)(s[j] | ((s[j + 4] >> 4) << 6));
                blk[4 + j + 4] = (uint8_t)(m[j] | ((m[j + 4] >> 4) << 6));
                blk[4 + j + 8] = (uint8_t)((s[j + 4] & 15u) | ((m[j + 4] & 15u) << 4));
            }
            uint8_t q[256];
            for (int j = 0; j < 8; j++) {
                const float step = d * (float)s[j], off = dmin * (float)m[j];
                for (int i = 0; i < 32; i++) {
                    float v = step > 0.0f ? nearbyintf((w[32 * j + i] + off) / step) : 0.0f;
                    q[32 * j + i] = (uint8_t)(v < 0.0f ? 0 : v > 15.0f ? 15 : (int)v);
                }
            }
            for (int c = 0; c < 4; c++)
                for (int l = 0; l < 32; l++)
                    blk[16 + 32 * c + l] = (uint8_t)(q[64 * c + l] | (q[64 * c + 32 + l] << 4));
        }
}
