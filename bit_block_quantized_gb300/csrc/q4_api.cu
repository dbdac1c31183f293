// q4_api.cu -- the extern "C" boundary of libq4.so: host-side argument checks
// (nothing is launched on a bad argument), then dispatch to the kernels.
#include <cmath>
#include <cstdio>

#include "q4_internal.cuh"

namespace q4 {

namespace {
thread_local const char *g_last_path = "";
}  // namespace

void note_gemv_path(const char *name) { g_last_path = name; }

// The integer-exact A16-Q8 lane (gemv_a16q8.cu): activation rows per launch
// (0 if K does not fit the shared-memory budget) and the launcher.
int gemv_a16q8_chunk(int64_t M, int64_t K);
cudaError_t launch_gemv_a16q8(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);

// The Q4_K x Q8 (W4A8) contraction (gemv_q4k_q8.cu), the NVFP4 quantizer
// (quantize.cu) and the b-bit packers (pack_bits.cu).
int gemv_q4k_q8_chunk(int64_t M, int64_t K);
cudaError_t launch_gemv_q4k_q8(const Tensor &t, const void *x, q4_dtype xd, float *y, int64_t M, cudaStream_t s);
cudaError_t launch_quantize_nvfp4(const void *W, q4_dtype wd, int64_t N, int64_t K, uint8_t *payload, uint8_t *scales,
                                  float *scale2, cudaStream_t s);
int gemv_w4a4_chunk(int64_t M, int64_t K);
cudaError_t launch_gemv_w4a4(const Tensor &t, float input_scale_inv, const void *x, q4_dtype xd, float *y, int64_t M,
                             cudaStream_t s);
cudaError_t launch_quantize_q4k(const void *W, q4_dtype wd, int64_t N, int64_t K, uint8_t *out, cudaStream_t s);
cudaError_t launch_quantize_nvfp4_scaled(const void *W, q4_dtype wd, int64_t N, int64_t K, float scale2,
                                         uint8_t *payload, uint8_t *scales, cudaStream_t s);
cudaError_t launch_pack_bits(const uint8_t *codes, int64_t n, int bits, uint32_t *words, cudaStream_t s);
cudaError_t launch_unpack_bits(const uint32_t *words, int64_t n, int bits, uint8_t *codes, cudaStream_t s);
cudaError_t launch_permute_k(const void *x, q4_dtype xd, const int32_t *perm, void *out, int64_t M, int64_t K,
                             cudaStream_t s);

// Role-wait limits of the bounded-wait kernels (gemv_tma.cu, gemv_fp4tc.cu, gemv_blk_tc.cu).
int gemv_tma_set_wait_limit(long long cycles);
int fp4tc_set_wait_limit(long long cycles);
int blk_tc_set_wait_limit(long long cycles);

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    return n;
}

bool known(q4_fmt f) { return f >= Q4_NVFP4 && f <= Q4_LOGICAL; }
bool aligned16(const void *p) { return p && (((uintptr_t)p) & 15u) == 0; }
bool kmajor_fmt(q4_fmt f) { return f == Q4_GPTQ || f == Q4_AWQ || f == Q4_LOGICAL; }
bool uses_scale_tensor(q4_fmt f) { return f != Q4_Q4K && f != Q4_Q40; }

int group_of(const q4_aux *aux) { return (aux && aux->group > 0) ? aux->group : 128; }

// Shape rules of each format (block / group multiples; [BPA] padding note).
int check_dims(q4_fmt f, int64_t N, int64_t K, int group) {
    if (N <= 0 || K <= 0) return Q4_EDIM;
    switch (f) {
    case Q4_NVFP4:
    case Q4_NVFP4_SPLITHALF: return K % 16 ? Q4_EDIM : Q4_OK;
    case Q4_MXFP4:
    case Q4_Q40: return K % 32 ? Q4_EDIM : Q4_OK;
    case Q4_Q4K: return K % 256 ? Q4_EDIM : Q4_OK;
    case Q4_GPTQ: return (K % 8 || K % group || N % 8) ? Q4_EDIM : Q4_OK;
    case Q4_AWQ:
    case Q4_LOGICAL: return (K % group || N % 8) ? Q4_EDIM : Q4_OK;
    default: return Q4_EINVAL;
    }
}

// Common checks for a packed weight tensor; fills `t`.  The NVFP4 scale2
// check comes last so a caller that does not read scale2 may ignore it.
int make_tensor(q4_fmt f, const void *W, const void *scales, const q4_aux *aux, int64_t N, int64_t K,
                Tensor &t, bool need_scale2) {
    if (!known(f)) return Q4_EINVAL;
    const int group = group_of(aux);
    int rc = check_dims(f, N, K, group);
    if (rc) return rc;
    if (!W) return Q4_EINVAL;
    if (!aligned16(W)) return Q4_EALIGN;
    if (uses_scale_tensor(f)) {
        if (!scales) return Q4_EINVAL;
        if (!aligned16(scales)) return Q4_EALIGN;
    }
    if (kmajor_fmt(f)) {
        if (!aux || !aux->zeros) return Q4_EINVAL;
        if (!aligned16(aux->zeros)) return Q4_EALIGN;
    }
    if (aux && aux->g_idx) {
        if (f != Q4_GPTQ && f != Q4_LOGICAL) return Q4_EINVAL;
        if (!aligned16(aux->g_idx)) return Q4_EALIGN;
    }
    t.fmt = f;
    t.w = (const uint8_t *)W;
    t.scales = (const uint8_t *)scales;
    t.zeros = aux ? (const uint8_t *)aux->zeros : nullptr;
    t.g_idx = aux ? aux->g_idx : nullptr;
    t.group = group;
    t.scale2 = aux ? aux->scale2 : 1.0f;
    t.N = N;
    t.K = K;
    if (need_scale2 && (f == Q4_NVFP4 || f == Q4_NVFP4_SPLITHALF)) {
        if (!aux) return Q4_EINVAL;
        if (!std::isfinite(aux->scale2) || !(aux->scale2 > 0.0f)) return Q4_ESCALE2;
    }
    return Q4_OK;
}

namespace {

q4_dtype default_x_dtype(q4_fmt f) { return (f == Q4_NVFP4 || f == Q4_MXFP4) ? Q4_DT_BF16 : Q4_DT_F32; }

}  // namespace
}  // namespace q4

using namespace q4;

extern "C" {

int q4_gemv(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux, const void *x, float *y,
            int64_t M, int64_t N, int64_t K, void *stream) {
    Tensor t;
    int rc = make_tensor(fmt, W_packed, scales, aux, N, K, t);
    if (rc) return rc;
    if (M <= 0) return Q4_EDIM;
    if (fmt == Q4_NVFP4_SPLITHALF || fmt == Q4_LOGICAL) return Q4_EUNSUPPORTED;
    if (!x || !y) return Q4_EINVAL;
    if (!aligned16(x) || !aligned16(y)) return Q4_EALIGN;
    const q4_dtype xd = aux ? aux->x_dtype : default_x_dtype(fmt);
    if (xd != Q4_DT_F32 && xd != Q4_DT_BF16) return Q4_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    if (fmt == Q4_NVFP4 && M == 1 && xd == Q4_DT_BF16 && (aux->flags & Q4_FLAG_FP4_SLICES) &&
        gemv_fp4tc_eligible(t, M)) {
        note_gemv_path("gemv_fp4tc");
        return launch_gemv_fp4tc(t, x, y, s) == cudaSuccess ? Q4_OK : Q4_ECUDA;
    }
    bool handled = false;
    cudaError_t e = cudaSuccess;
    if (M > 8) e = launch_gemm_tc(t, x, xd, y, M, s, &handled);
    if (e == cudaSuccess && !handled) e = launch_gemv(t, x, xd, y, M, s);
    return e == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_gemv_grouped(const q4_gemv_desc *descs, int count, int64_t M, void *stream) {
    if (!descs || count <= 0) return Q4_EINVAL;
    if (M <= 0) return Q4_EDIM;
    Tensor ts[8];
    const void *xs[8];
    float *ys[8];
    bool one_launch = count <= 8;
    bool tma = count <= 8;                     // every member NVFP4 on the TMA kernel, one shared x
    bool fp4tc = count <= 8 && M == 1;         // every member NVFP4 at batch 1 on the FP4 tensor cores
    bool blk = count <= 8 && M <= 8;           // every member Q4_K (or every one Q4_0) on the block kernel, one x
    q4_dtype xd0 = Q4_DT_F32;
    for (int i = 0; i < count; i++) {          // check every member before launching any
        const q4_gemv_desc &d = descs[i];
        Tensor t;
        const int rc = make_tensor(d.fmt, d.W_packed, d.scales, d.aux, d.N, d.K, t);
        if (rc) return rc;
        if (d.fmt == Q4_NVFP4_SPLITHALF || d.fmt == Q4_LOGICAL) return Q4_EUNSUPPORTED;
        if (!d.x || !d.y) return Q4_EINVAL;
        if (!aligned16(d.x) || !aligned16(d.y)) return Q4_EALIGN;
        const q4_dtype xd = d.aux ? d.aux->x_dtype : default_x_dtype(d.fmt);
        if (xd != Q4_DT_F32 && xd != Q4_DT_BF16) return Q4_EINVAL;
        if (i == 0) xd0 = xd;
        if (i < 8) {
            ts[i] = t;
            xs[i] = d.x;
            ys[i] = d.y;
        }
        one_launch = one_launch && d.fmt == Q4_NVFP4 && xd == Q4_DT_BF16 && d.K == descs[0].K && M <= 8 &&
                     gemv_mma_eligible(t, M);
        tma = tma && (d.fmt == Q4_NVFP4 || d.fmt == Q4_MXFP4) && d.fmt == descs[0].fmt && xd == Q4_DT_BF16 &&
              d.K == descs[0].K && d.x == descs[0].x && gemv_tma_eligible(t, M);
        fp4tc = fp4tc && d.fmt == Q4_NVFP4 && xd == Q4_DT_BF16 && d.K == descs[0].K && d.x == descs[0].x &&
                (d.aux->flags & Q4_FLAG_FP4_SLICES) && gemv_fp4tc_eligible(t, M);
        blk = blk && (d.fmt == Q4_Q4K || d.fmt == Q4_Q40) && d.fmt == descs[0].fmt && xd == xd0 &&
              d.K == descs[0].K && d.x == descs[0].x && gemv_blk_tc_eligible(t, M, xd);
    }
    if (blk && count > 1) {
        note_gemv_path(descs[0].fmt == Q4_Q4K ? "gemv_blk_tc_q4k_group" : "gemv_blk_tc_q40_group");
        return launch_gemv_blk_tc_group(ts, count, descs[0].x, xd0, ys, M, (cudaStream_t)stream) == cudaSuccess
                   ? Q4_OK
                   : Q4_ECUDA;
    }
    if (fp4tc) {
        note_gemv_path(count == 1 ? "gemv_fp4tc" : "gemv_fp4tc_group");
        return launch_gemv_fp4tc_group(ts, count, descs[0].x, ys, (cudaStream_t)stream) == cudaSuccess ? Q4_OK
                                                                                                  : Q4_ECUDA;
    }
    if (tma) {
        note_gemv_path(count == 1 ? "gemv_tma" : "gemv_tma_group");
        return launch_gemv_tma_group(ts, descs[0].x, ys, count, M, (cudaStream_t)stream) == cudaSuccess ? Q4_OK
                                                                                                  : Q4_ECUDA;
    }
    if (one_launch) {
        note_gemv_path("gemv_mma_group");
        return launch_gemv_mma_group(ts, xs, ys, count, M, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
    }
    for (int i = 0; i < count; i++) {
        const q4_gemv_desc &d = descs[i];
        const int rc = q4_gemv(d.fmt, d.W_packed, d.scales, d.aux, d.x, d.y, M, d.N, d.K, stream);
        if (rc) return rc;
    }
    return Q4_OK;
}

int q4_gemv_chain(const q4_gemv_desc *descs, const int *first, int ngroups, int64_t M, uint32_t *sync,
                  void *stream) {
    if (!descs || !first || ngroups <= 0) return Q4_EINVAL;
    if (M <= 0) return Q4_EDIM;
    if (first[0] != 0) return Q4_EINVAL;
    for (int g = 0; g < ngroups; g++)
        if (first[g + 1] <= first[g]) return Q4_EINVAL;
    const int count = first[ngroups];
    if (ngroups > 1 && !sync) return Q4_EINVAL;
    if (sync && (((uintptr_t)sync) & 7u) != 0) return Q4_EALIGN;
    Tensor ts[8];
    const void *xs[4];
    float *ys[8];
    bool one_launch = count <= 8 && ngroups <= 4;
    for (int g = 0; g < ngroups; g++) {
        for (int i = first[g]; i < first[g + 1]; i++) {   // check every member before launching any
            const q4_gemv_desc &d = descs[i];
            Tensor t;
            const int rc = make_tensor(d.fmt, d.W_packed, d.scales, d.aux, d.N, d.K, t);
            if (rc) return rc;
            if (d.fmt == Q4_NVFP4_SPLITHALF || d.fmt == Q4_LOGICAL) return Q4_EUNSUPPORTED;
            if (!d.x || !d.y) return Q4_EINVAL;
            if (!aligned16(d.x) || !aligned16(d.y)) return Q4_EALIGN;
            const q4_dtype xd = d.aux ? d.aux->x_dtype : default_x_dtype(d.fmt);
            if (xd != Q4_DT_F32 && xd != Q4_DT_BF16) return Q4_EINVAL;
            one_launch = one_launch && xd == Q4_DT_BF16 && d.x == descs[first[g]].x && d.K == descs[first[g]].K;
            if (one_launch) {
                ts[i] = t;
                ys[i] = d.y;
            }
        }
        if (one_launch) xs[g] = descs[first[g]].x;
    }
    if (one_launch && gemv_tma_chain_fits(ts, first, ngroups, M)) {
        note_gemv_path(ngroups == 1 ? (count == 1 ? "gemv_tma" : "gemv_tma_group") : "gemv_tma_chain");
        return launch_gemv_tma_chain(ts, xs, ys, first, ngroups, M, sync, (cudaStream_t)stream) == cudaSuccess
                   ? Q4_OK
                   : Q4_ECUDA;
    }
    for (int g = 0; g < ngroups; g++) {
        const int rc = q4_gemv_grouped(descs + first[g], first[g + 1] - first[g], M, stream);
        if (rc) return rc;
    }
    return Q4_OK;
}

const char *q4_last_gemv_path(void) { return q4::g_last_path; }

int q4_set_wait_limit(int64_t cycles) {
    const long long c = cycles > 0 ? (long long)cycles : (1LL << 31);
    const int a = gemv_tma_set_wait_limit(c), b = fp4tc_set_wait_limit(c), d = blk_tc_set_wait_limit(c);
    return a ? a : b ? b : d;
}

int q4_gemv_a16q8(const void *W_packed, const void *scales, const q4_aux *aux, const void *x, float *y, int64_t M,
                  int64_t N, int64_t K, void *stream) {
    Tensor t;
    const int rc = make_tensor(Q4_NVFP4, W_packed, scales, aux, N, K, t);   // aux is non-null past this
    if (rc) return rc;
    if (M <= 0 || K % 256) return Q4_EDIM;
    if (!x || !y) return Q4_EINVAL;
    if (!aligned16(x) || !aligned16(y)) return Q4_EALIGN;
    const q4_dtype xd = aux->x_dtype;
    if (xd != Q4_DT_F32 && xd != Q4_DT_BF16) return Q4_EINVAL;
    if (gemv_a16q8_chunk(M, K) == 0) return Q4_EDIM;
    return launch_gemv_a16q8(t, x, xd, y, M, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_gemv_q4k_q8(const void *W_packed, const q4_aux *aux, const void *x, float *y, int64_t M, int64_t N,
                   int64_t K, void *stream) {
    Tensor t;
    const int rc = make_tensor(Q4_Q4K, W_packed, nullptr, aux, N, K, t);
    if (rc) return rc;
    if (M <= 0) return Q4_EDIM;
    if (!x || !y) return Q4_EINVAL;
    if (!aligned16(x) || !aligned16(y)) return Q4_EALIGN;
    const q4_dtype xd = aux ? aux->x_dtype : Q4_DT_F32;
    if (xd != Q4_DT_F32 && xd != Q4_DT_BF16) return Q4_EINVAL;
    if (gemv_q4k_q8_chunk(M, K) == 0) return Q4_EDIM;
    return launch_gemv_q4k_q8(t, x, xd, y, M, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_gemv_w4a4(const void *W_packed, const void *scales, const q4_aux *aux, float input_scale_inv, const void *x,
                 float *y, int64_t M, int64_t N, int64_t K, void *stream) {
    Tensor t;
    const int rc = make_tensor(Q4_NVFP4, W_packed, scales, aux, N, K, t);   // aux is non-null past this
    if (rc) return rc;
    if (M <= 0 || K % 64) return Q4_EDIM;
    if (!std::isfinite(input_scale_inv) || !(input_scale_inv > 0.0f)) return Q4_ESCALE2;
    if (!x || !y) return Q4_EINVAL;
    if (!aligned16(x) || !aligned16(y)) return Q4_EALIGN;
    const q4_dtype xd = aux->x_dtype;
    if (xd != Q4_DT_F32 && xd != Q4_DT_BF16) return Q4_EINVAL;
    if (gemv_w4a4_chunk(M, K) == 0) return Q4_EDIM;
    return launch_gemv_w4a4(t, input_scale_inv, x, xd, y, M, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_quantize_nvfp4(const void *W, q4_dtype w_dtype, void *payload, void *scales, float *scale2, int64_t N,
                      int64_t K, void *stream) {
    if (N <= 0 || K <= 0 || K % 16) return Q4_EDIM;
    if (!W || !payload || !scales || !scale2) return Q4_EINVAL;
    if (!aligned16(W) || !aligned16(payload) || !aligned16(scales) || (((uintptr_t)scale2) & 3u)) return Q4_EALIGN;
    if (w_dtype != Q4_DT_F32 && w_dtype != Q4_DT_BF16) return Q4_EINVAL;
    return launch_quantize_nvfp4(W, w_dtype, N, K, (uint8_t *)payload, (uint8_t *)scales, scale2,
                                 (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_quantize_nvfp4_scaled(const void *x, q4_dtype x_dtype, float scale2, void *payload, void *scales, int64_t M,
                             int64_t K, void *stream) {
    if (M <= 0 || K <= 0 || K % 16) return Q4_EDIM;
    if (!x || !payload || !scales) return Q4_EINVAL;
    if (!aligned16(x) || !aligned16(payload) || !aligned16(scales)) return Q4_EALIGN;
    if (x_dtype != Q4_DT_F32 && x_dtype != Q4_DT_BF16) return Q4_EINVAL;
    if (!std::isfinite(scale2) || !(scale2 > 0.0f)) return Q4_ESCALE2;
    return launch_quantize_nvfp4_scaled(x, x_dtype, M, K, scale2, (uint8_t *)payload, (uint8_t *)scales,
                                        (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_gemv_w4a4_tc(const void *W_packed, const void *scales, const q4_aux *aux, const void *xq, const void *xs,
                    float x_scale2, float *y, int64_t M, int64_t N, int64_t K, void *stream) {
    Tensor t;
    const int rc = make_tensor(Q4_NVFP4, W_packed, scales, aux, N, K, t);
    if (rc) return rc;
    if (M <= 0 || K % 256) return Q4_EDIM;
    if (!std::isfinite(x_scale2) || !(x_scale2 > 0.0f)) return Q4_ESCALE2;
    if (!xq || !xs || !y) return Q4_EINVAL;
    if (!aligned16(xq) || !aligned16(xs) || !aligned16(y)) return Q4_EALIGN;
    if (!gemv_w4a4_tc_eligible(t)) return Q4_EUNSUPPORTED;
    note_gemv_path("gemv_w4a4_tc");
    return launch_gemv_w4a4_tc(t, (const uint8_t *)xq, (const uint8_t *)xs, x_scale2, y, M, (cudaStream_t)stream) ==
                   cudaSuccess
               ? Q4_OK
               : Q4_ECUDA;
}

int q4_quantize_q4k(const void *W, q4_dtype w_dtype, void *out, int64_t N, int64_t K, void *stream) {
    if (N <= 0 || K <= 0 || K % 256) return Q4_EDIM;
    if (!W || !out) return Q4_EINVAL;
    if (!aligned16(W) || !aligned16(out)) return Q4_EALIGN;
    if (w_dtype != Q4_DT_F32 && w_dtype != Q4_DT_BF16) return Q4_EINVAL;
    return launch_quantize_q4k(W, w_dtype, N, K, (uint8_t *)out, (cudaStream_t)stream) == cudaSuccess ? Q4_OK
                                                                                                    : Q4_ECUDA;
}

int q4_pack_bits(const uint8_t *codes, int64_t n, int bits, uint32_t *words, void *stream) {
    if (bits < 1 || bits > 8 || n <= 0 || (n * bits) % 32) return Q4_EDIM;
    if (!codes || !words) return Q4_EINVAL;
    if (!aligned16(codes) || !aligned16(words)) return Q4_EALIGN;
    return launch_pack_bits(codes, n, bits, words, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_unpack_bits(const uint32_t *words, int64_t n, int bits, uint8_t *codes, void *stream) {
    if (bits < 1 || bits > 8 || n <= 0 || (n * bits) % 32) return Q4_EDIM;
    if (!codes || !words) return Q4_EINVAL;
    if (!aligned16(codes) || !aligned16(words)) return Q4_EALIGN;
    return launch_unpack_bits(words, n, bits, codes, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_permute_k(const void *x, q4_dtype x_dtype, const int32_t *perm, void *out, int64_t M, int64_t K,
                 void *stream) {
    if (M <= 0 || K <= 0) return Q4_EDIM;
    if (!x || !perm || !out) return Q4_EINVAL;
    if (!aligned16(x) || !aligned16(perm) || !aligned16(out)) return Q4_EALIGN;
    if (x_dtype != Q4_DT_F32 && x_dtype != Q4_DT_BF16) return Q4_EINVAL;
    if (x == out) return Q4_EINVAL;
    return launch_permute_k(x, x_dtype, perm, out, M, K, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_dequant(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux, void *out, int64_t N,
               int64_t K, void *stream) {
    Tensor t;
    int rc = make_tensor(fmt, W_packed, scales, aux, N, K, t);
    if (rc) return rc;
    if (!out) return Q4_EINVAL;
    if (!aligned16(out)) return Q4_EALIGN;
    const q4_dtype od = aux ? aux->out_dtype : Q4_DT_F32;
    if (od != Q4_DT_F32 && od != Q4_DT_BF16) return Q4_EINVAL;
    return launch_dequant(t, out, od, (cudaStream_t)stream) == cudaSuccess ? Q4_OK : Q4_ECUDA;
}

int q4_repack(q4_fmt src, const void *src_w, const void *src_scales, const q4_aux *src_aux, q4_fmt dst,
              void *dst_w, void *dst_scales, void *dst_zeros, int32_t *perm_out, int64_t N, int64_t K,
              void *stream) {
    Tensor t;
    int rc = make_tensor(src, src_w, src_scales, src_aux, N, K, t, /*need_scale2=*/false);
    if (rc) return rc;
    if (!known(dst)) return Q4_EINVAL;
    const int group = (src == Q4_Q40) ? 32 : t.group;
    rc = check_dims(dst, N, K, group);
    if (rc) return rc;
    if (!dst_w || !dst_scales) return Q4_EINVAL;
    if (!aligned16(dst_w) || !aligned16(dst_scales)) return Q4_EALIGN;
    if (kmajor_fmt(dst)) {
        if (!dst_zeros) return Q4_EINVAL;
        if (!aligned16(dst_zeros)) return Q4_EALIGN;
    }
    if (perm_out && !aligned16(perm_out)) return Q4_EALIGN;
    return launch_repack(src, t, dst, dst_w, dst_scales, dst_zeros, perm_out, (cudaStream_t)stream);
}

int q4_validate(q4_fmt fmt, const void *W_packed, const void *scales, const q4_aux *aux, int64_t N, int64_t K,
                int64_t *d_bad_count, void *stream) {
    Tensor t;
    const int rc = make_tensor(fmt, W_packed, scales, aux, N, K, t);
    if (rc && rc != Q4_ESCALE2) return rc;
    if (!d_bad_count) return Q4_EINVAL;
    if (!aligned16(d_bad_count)) return Q4_EALIGN;
    const int v = run_validate(t, d_bad_count, (cudaStream_t)stream);
    return v != Q4_OK ? v : rc;      // NaN scale bytes first, then a bad scale2
}

const char *q4_strerror(int status) {
    switch (status) {
    case Q4_OK: return "ok";
    case Q4_EINVAL: return "invalid argument (null pointer, unknown format or dtype, missing aux field)";
    case Q4_EDIM: return "invalid dimensions (non-positive, or not a multiple of the format's block/group)";
    case Q4_EALIGN: return "a tensor pointer is not 16-byte aligned";
    case Q4_ENAN: return "NaN scale encodings found";
    case Q4_ESCALE2: return "NVFP4 scale2 must be finite and > 0";
    case Q4_ECUDA: return "CUDA launch or copy failed";
    case Q4_EUNSUPPORTED: return "format/operation pair not provided";
    case Q4_ERANGE: return "a zero point cannot be stored in the target format";
    case Q4_ETIMEOUT: return "a bounded device-side wait timed out";
    default: return "unknown status";
    }
}

size_t q4_packed_bytes(q4_fmt fmt, int64_t N, int64_t K) {
    if (check_dims(fmt, N, K, 128) != Q4_OK) return 0;
    const int64_t G = K / 128;
    switch (fmt) {
    case Q4_NVFP4:
    case Q4_NVFP4_SPLITHALF: return (size_t)(N * K / 2 + N * K / 16 + 4);
    case Q4_MXFP4: return (size_t)(N * K / 2 + N * K / 32);
    case Q4_Q4K: return (size_t)(N * (K / 256) * 144);
    case Q4_Q40: return (size_t)(N * (K / 32) * 18);
    case Q4_GPTQ:
    case Q4_AWQ: return (size_t)(N * K / 2 + G * N * 2 + G * (N / 8) * 4);
    case Q4_LOGICAL: return (size_t)(N * K + G * N * 2 + G * N);
    default: return 0;
    }
}

const char *q4_version(void) { return "q4 0.1 sm_103a"; }

}  // extern "C"
