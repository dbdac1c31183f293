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
 * Parity status: every function below is pinned by tests/test_oracle_pins.py
 * (printed worked examples, library decoders, brute force, invariants).
 */
#include <math.h>
#include <stdint.h>
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
