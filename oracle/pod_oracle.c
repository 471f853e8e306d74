/*
 * POD paged-attention ORACLE: plain, slow, fp64, single file of C.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do. It shares no code, header, table or helper
 * with the CUDA path.
 *
 * What it computes is the plain definition of softmax attention over a paged
 * KV cache, written out one (query token, qo head) at a time:
 *
 *  - Paged KV cache, NHD layout [num_pages, 2, page_size, num_kv_heads, head_dim],
 *    addressed through kv_indptr / kv_indices / last_page_len
 *    (POD walkthrough, the two wrapper docstring examples and "plan 内部做了什么":
 *    kv_len = (pages - 1) * page_size + last_page_len).
 *  - GQA: qo head h reads kv head h / (num_qo_heads / num_kv_heads)
 *    (POD walkthrough, "plan/run 生命周期": num_qo_heads must be a multiple
 *    of num_kv_heads; unequal counts mean grouped-query attention).
 *  - Bottom-right causal diagonal: query row i of a request with q_len rows
 *    and kv_len keys sits at key position p = kv_len - q_len + i and may see
 *    keys 0..p (flashinfer.cudnn page, "Decode 能力矩阵与参数", q_len_per_req row).
 *  - window_left counts the keys strictly before the diagonal; the diagonal is
 *    attended too, so key t is allowed iff t >= p - window_left; -1 disables it
 *    (flashinfer.cudnn page, "Decode 能力矩阵与参数", window paragraph).
 *  - Sinks: one extra logit per qo head in the softmax denominator with a zero
 *    value row (flashinfer.cudnn page, "Decode 能力矩阵与参数", sinks row).
 *    Reading taken here: the sink is already a logit (not multiplied by
 *    sm_scale) and it does not enter the LSE.
 *  - LSE in base 2: lse = log2(sum over allowed keys of exp(sm_scale * q.k))
 *    (flashinfer.cudnn page, "LSE 契约").
 *  - Merge of split partials (o_i, lse_i): weights 2^(lse_i - max), the
 *    property that lets base-2 LSE feed a cascade merge (same section).
 *  - KV layout (FlashInfer guide, "快速上手", kv_layout: NHD or HND orders
 *    the dimensions of the k/v tensors): NHD pages are [2, page_size, Hk, d],
 *    HND pages [2, Hk, page_size, d]; the page pool is [num_pages, ...] either way.
 *  - ALiBi (same section, pos_encoding_mode ALIBI; per-head slopes are an
 *    input): the logit of key t for query row i gains slope[h] * (t - p),
 *    p the row's bottom-right diagonal position (the published ALiBi bias
 *    -m * distance, with the distance measured from the diagonal).
 *  - Logits soft cap (same section, logits_soft_cap: cap * tanh(x / cap), 0
 *    = off): x is the scaled logit sm_scale * q.k. With both, the ALiBi bias
 *    is added after the cap (a reading: the pages do not combine them).
 *  - ROPE_LLAMA (same section, pos_encoding_mode, rope_scale default 1,
 *    rope_theta default 1e4): q and each key are rotated before the dot
 *    product by the rotary embedding of their positions (p for the query,
 *    t for key t; values are not rotated). Reading taken here: the LLaMA
 *    half-split pairing, element j with j + d/2, turned by the angle
 *    (pos / rope_scale) * rope_theta^(-2j/d) (rotary position embedding
 *    with position interpolation by rope_scale).
 *  - Custom mask (POD walkthrough, "run 参数详解", prefill parameters
 *    custom_mask_p / packed_custom_mask_p, packed with little bit order; a
 *    custom mask takes precedence over causal): one boolean per (query row,
 *    key) of each request, the requests' [q_len, kv_len] row-major matrices
 *    laid end to end, eight to a byte, the first element in the least
 *    significant bit. Readings taken here: a set bit allows the key;
 *    window_left still applies; a row the mask leaves without keys has
 *    out = 0 and lse = -inf.
 *
 * Inputs are the same rounded fp16/bf16 values the GPU reads, widened to
 * double by decoders written from the IEEE-754 binary16 and bfloat16 bit
 * layouts. An FP8 (E4M3) cache is read as its codes decoded from the E4M3
 * bit layout times a per-tensor scale for K and one for V: attention over the
 * dequantized cache, which is what folding the K scale into the softmax scale
 * and multiplying the output by the V scale compute. Nothing is blocked, fused or reordered: keys are visited in order
 * 0..kv_len-1.
 *
 * Parity pins (tests under tests/, run on the CPU): brute-force dense attention
 * on tiny inputs, page-permutation and page-size invariance, split/merge
 * identity, the hand-worked two-token example, closed forms (q = 0,
 * window_left = 0, kv_len = 1, equal keys), GQA head duplication, exhaustive
 * checks of the two 16-bit decoders; for the custom mask, brute force over
 * the bits numpy unpacks, single-bit masks (out = v_t) and the triangular and
 * all-ones masks against the causal and non-causal rules; for HND pages,
 * bit-identity with NHD and brute force over an HND gather; for ALiBi, brute
 * force, the geometric-series lse of q = 0 and slope 0; for the soft cap,
 * brute force, two saturated keys and a cap far above every logit; for
 * ROPE_LLAMA, closed-form logits cos/sin((p - t) f) of unit vectors, a
 * request shifted five positions later, and position 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_EMPTY_ROW 2

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);    /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float x;
    memcpy(&x, &u, sizeof(x));
    return (double)x;
}

static double widen(uint16_t v, int dtype)
{
    return dtype == 0 ? oracle_f16_to_f64(v) : oracle_bf16_to_f64(v);
}

/* FP8 E4M3 (the "fn" variant: 1 sign, 4 exponent bits with bias 7, 3 fraction
 * bits, no infinities, S.1111.111 is NaN). */
double oracle_e4m3_to_f64(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int f = c & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) {
        v = ldexp((double)f, -9);                /* subnormal: f/8 * 2^-6 */
    } else {
        v = ldexp((double)(8 + f), e - 10);      /* (1 + f/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

/* one K or V element: 16-bit codes of `dtype`, or e4m3 codes times `scale`
 * when kv_fp8 is set */
static double kv_elem(const void* kv, int64_t idx, int dtype, int kv_fp8, double scale)
{
    if (kv_fp8) return oracle_e4m3_to_f64(((const uint8_t*)kv)[idx]) * scale;
    return widen(((const uint16_t*)kv)[idx], dtype);
}

/* kv_len of request r from its page table (POD walkthrough, plan step 1). */
int64_t oracle_kv_len(const int32_t* kv_indptr, const int32_t* last_page_len,
                      int r, int page_size)
{
    int64_t pages = (int64_t)kv_indptr[r + 1] - kv_indptr[r];
    if (pages <= 0) return 0;
    return (pages - 1) * (int64_t)page_size + last_page_len[r];
}

void oracle_seq_lens(const int32_t* kv_indptr, const int32_t* last_page_len,
                     int batch, int page_size, int32_t* kv_len_out)
{
    for (int r = 0; r < batch; ++r)
        kv_len_out[r] = (int32_t)oracle_kv_len(kv_indptr, last_page_len, r, page_size);
}

/* Element offset of the K (kv = 0) or V (kv = 1) row of (page, slot, head). */
static int64_t row_offset(int kv_layout, int64_t page, int kv, int64_t slot, int hk,
                          int page_size, int Hk, int d)
{
    if (kv_layout == 1) /* HND */
        return (((page * 2 + kv) * Hk + hk) * (int64_t)page_size + slot) * (int64_t)d;
    return (((page * 2 + kv) * (int64_t)page_size + slot) * Hk + hk) * (int64_t)d;
}

/* Rotary embedding of x[0..d) at position pos, pairs (j, j + d/2). */
static void rope_rotate(double* x, int d, double pos, double rope_scale, double rope_theta)
{
    int half = d / 2;
    for (int j = 0; j < half; ++j) {
        double ang = (pos / rope_scale) * pow(rope_theta, -2.0 * (double)j / (double)d);
        double c = cos(ang), sn = sin(ang);
        double a = x[j], b = x[j + half];
        x[j] = a * c - b * sn;
        x[j + half] = b * c + a * sn;
    }
}

/* Bit `pos` of a little-bit-order packed array. */
static int mask_bit(const uint8_t* packed, int64_t pos)
{
    return (packed[pos >> 3] >> (int)(pos & 7)) & 1;
}

static int find_request(const int32_t* q_indptr, int batch, int64_t token)
{
    for (int r = 0; r < batch; ++r)
        if (token >= q_indptr[r] && token < q_indptr[r + 1]) return r;
    return -1;
}

/*
 * Attention for a list of selected (token, qo head) pairs of one half.
 *   q   : [rows, H, d] 16-bit codes       kv : [num_pages, 2, ps, Hk, d] codes
 *   sel_token[n], sel_head[n]             : which outputs to compute
 *   key_lo/key_hi (may be NULL)           : extra restriction key in [lo, hi)
 *                                           per selection (split-KV partials)
 *   sinks (may be NULL)                   : fp32 [H] extra logit per qo head
 *   packed_mask (may be NULL)             : custom mask bits (see the header);
 *                                           when given, causal is not applied
 *   out [n, d], lse [n]                   : fp64 results
 * Returns the first error code met (rows are still filled where possible).
 */
int oracle_attention_rows_ext(const uint16_t* q, const void* kv, int dtype,
                              int kv_fp8, double k_scale, double v_scale,
                              const int32_t* q_indptr, const int32_t* kv_indptr,
                              const int32_t* kv_indices, const int32_t* last_page_len,
                              int batch, int num_pages,
                              int H, int Hk, int d, int page_size, int kv_layout,
                              int causal, int window_left, double sm_scale,
                              double soft_cap, const float* alibi_slopes,
                              int rope, double rope_scale, double rope_theta,
                              const float* sinks, const uint8_t* packed_mask,
                              int64_t n_sel, const int64_t* sel_token, const int32_t* sel_head,
                              const int64_t* key_lo, const int64_t* key_hi,
                              double* out, double* lse, int nthreads)
{
    if (H <= 0 || Hk <= 0 || H % Hk != 0 || d <= 0 || page_size <= 0) return ORACLE_BAD_ARG;
    if (kv_layout != 0 && kv_layout != 1) return ORACLE_BAD_ARG;
    if (rope && (d % 2 != 0 || !(rope_scale > 0.0) || !(rope_theta > 0.0))) return ORACLE_BAD_ARG;
    int group = H / Hk;
    int status = ORACLE_OK;
    (void)nthreads;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t s = 0; s < n_sel; ++s) {
        int64_t token = sel_token[s];
        int h = sel_head[s];
        double* o = out + s * (int64_t)d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        lse[s] = -INFINITY;
        int r = find_request(q_indptr, batch, token);
        if (r < 0 || h < 0 || h >= H) {
#pragma omp atomic write
            status = ORACLE_BAD_ARG;
            continue;
        }
        int64_t q_len = (int64_t)q_indptr[r + 1] - q_indptr[r];
        int64_t i = token - q_indptr[r];
        int64_t kv_len = oracle_kv_len(kv_indptr, last_page_len, r, page_size);
        int64_t p = kv_len - q_len + i;          /* bottom-right diagonal */
        int hk = h / group;                       /* GQA mapping */
        /* first bit of this request's mask: the earlier requests' q_len * kv_len */
        int64_t mask_row = 0;
        if (packed_mask) {
            for (int rr = 0; rr < r; ++rr)
                mask_row += ((int64_t)q_indptr[rr + 1] - q_indptr[rr]) *
                            oracle_kv_len(kv_indptr, last_page_len, rr, page_size);
            mask_row += i * kv_len;
        }

        double* qv = (double*)malloc(sizeof(double) * (size_t)d);
        double* kr = (double*)malloc(sizeof(double) * (size_t)d);
        double* logit = (double*)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
        char* allowed = (char*)malloc((size_t)(kv_len > 0 ? kv_len : 1));
        for (int e = 0; e < d; ++e)
            qv[e] = widen(q[(token * H + h) * (int64_t)d + e], dtype);
        if (rope) rope_rotate(qv, d, (double)p, rope_scale, rope_theta);

        /* logits of the allowed keys */
        double m = -INFINITY;
        int64_t n_allowed = 0;
        for (int64_t t = 0; t < kv_len; ++t) {
            int ok = 1;
            if (packed_mask) {
                if (!mask_bit(packed_mask, mask_row + t)) ok = 0;
            } else if (causal && t > p) {
                ok = 0;
            }
            if (window_left >= 0 && t < p - window_left) ok = 0;
            if (key_lo && t < key_lo[s]) ok = 0;
            if (key_hi && t >= key_hi[s]) ok = 0;
            allowed[t] = (char)ok;
            if (!ok) continue;
            int64_t page = kv_indices[kv_indptr[r] + t / page_size];
            int64_t slot = t % page_size;
            if (page < 0 || page >= num_pages) {
                allowed[t] = 0;
#pragma omp atomic write
                status = ORACLE_BAD_ARG;
                continue;
            }
            int64_t k0 = row_offset(kv_layout, page, 0, slot, hk, page_size, Hk, d);
            for (int e = 0; e < d; ++e) kr[e] = kv_elem(kv, k0 + e, dtype, kv_fp8, k_scale);
            if (rope) rope_rotate(kr, d, (double)t, rope_scale, rope_theta);
            double dot = 0.0;
            for (int e = 0; e < d; ++e) dot += qv[e] * kr[e];
            if (soft_cap > 0.0)
                logit[t] = soft_cap * tanh(sm_scale * dot / soft_cap);
            else
                logit[t] = sm_scale * dot;
            if (alibi_slopes) logit[t] += (double)alibi_slopes[h] * (double)(t - p);
            if (logit[t] > m) m = logit[t];
            ++n_allowed;
        }
        if (n_allowed == 0) {
            /* out = 0, lse = -inf; only the custom mask may empty a row */
            if (!packed_mask) {
#pragma omp atomic write
                status = ORACLE_EMPTY_ROW;
            }
            free(qv); free(kr); free(logit); free(allowed);
            continue;
        }
        /* explicit softmax with an optional sink logit in the denominator */
        double z = 0.0;
        for (int64_t t = 0; t < kv_len; ++t)
            if (allowed[t]) z += exp(logit[t] - m);
        double denom = z;
        if (sinks) denom += exp((double)sinks[h] - m);
        for (int64_t t = 0; t < kv_len; ++t) {
            if (!allowed[t]) continue;
            int64_t page = kv_indices[kv_indptr[r] + t / page_size];
            int64_t slot = t % page_size;
            int64_t v0 = row_offset(kv_layout, page, 1, slot, hk, page_size, Hk, d);
            double w = exp(logit[t] - m) / denom;
            for (int e = 0; e < d; ++e) o[e] += w * kv_elem(kv, v0 + e, dtype, kv_fp8, v_scale);
        }
        lse[s] = (m + log(z)) / log(2.0);
        free(qv); free(kr); free(logit); free(allowed);
    }
    return status;
}

/* oracle_attention_rows_ext with the NHD layout, no soft cap and no ALiBi. */
int oracle_attention_rows_masked(const uint16_t* q, const void* kv, int dtype,
                                 int kv_fp8, double k_scale, double v_scale,
                                 const int32_t* q_indptr, const int32_t* kv_indptr,
                                 const int32_t* kv_indices, const int32_t* last_page_len,
                                 int batch, int num_pages,
                                 int H, int Hk, int d, int page_size,
                                 int causal, int window_left, double sm_scale,
                                 const float* sinks, const uint8_t* packed_mask,
                                 int64_t n_sel, const int64_t* sel_token, const int32_t* sel_head,
                                 const int64_t* key_lo, const int64_t* key_hi,
                                 double* out, double* lse, int nthreads)
{
    return oracle_attention_rows_ext(q, kv, dtype, kv_fp8, k_scale, v_scale, q_indptr, kv_indptr,
                                     kv_indices, last_page_len, batch, num_pages, H, Hk, d,
                                     page_size, 0, causal, window_left, sm_scale, 0.0, NULL,
                                     0, 1.0, 1e4, sinks, packed_mask, n_sel, sel_token, sel_head,
                                     key_lo,
                                     key_hi, out, lse, nthreads);
}

/* oracle_attention_rows_masked without a custom mask. */
int oracle_attention_rows_kv(const uint16_t* q, const void* kv, int dtype,
                             int kv_fp8, double k_scale, double v_scale,
                             const int32_t* q_indptr, const int32_t* kv_indptr,
                             const int32_t* kv_indices, const int32_t* last_page_len,
                             int batch, int num_pages,
                             int H, int Hk, int d, int page_size,
                             int causal, int window_left, double sm_scale,
                             const float* sinks,
                             int64_t n_sel, const int64_t* sel_token, const int32_t* sel_head,
                             const int64_t* key_lo, const int64_t* key_hi,
                             double* out, double* lse, int nthreads)
{
    return oracle_attention_rows_masked(q, kv, dtype, kv_fp8, k_scale, v_scale, q_indptr,
                                        kv_indptr, kv_indices, last_page_len, batch, num_pages,
                                        H, Hk, d, page_size, causal, window_left, sm_scale, sinks,
                                        NULL, n_sel, sel_token, sel_head, key_lo, key_hi, out, lse,
                                        nthreads);
}

/* The 16-bit cache of `dtype`: oracle_attention_rows_kv without FP8. */
int oracle_attention_rows(const uint16_t* q, const uint16_t* kv, int dtype,
                          const int32_t* q_indptr, const int32_t* kv_indptr,
                          const int32_t* kv_indices, const int32_t* last_page_len,
                          int batch, int num_pages,
                          int H, int Hk, int d, int page_size,
                          int causal, int window_left, double sm_scale,
                          const float* sinks,
                          int64_t n_sel, const int64_t* sel_token, const int32_t* sel_head,
                          const int64_t* key_lo, const int64_t* key_hi,
                          double* out, double* lse, int nthreads)
{
    return oracle_attention_rows_kv(q, kv, dtype, 0, 1.0, 1.0, q_indptr, kv_indptr, kv_indices,
                                    last_page_len, batch, num_pages, H, Hk, d, page_size, causal,
                                    window_left, sm_scale, sinks, n_sel, sel_token, sel_head,
                                    key_lo, key_hi, out, lse, nthreads);
}

/*
 * Merge n partial results of the same (row, head) computed over disjoint key
 * sets. Partial i is a normalised output o_i with Z_i = 2^lse_i the sum of
 * exponentials of its keys (no sink). The merged output is
 *   o = sum_i Z_i o_i / (sum_i Z_i + [sink] exp(sink)),  lse = log2 sum_i Z_i,
 * evaluated with every Z_i divided by 2^M, M = max_i lse_i.
 *   o_parts [n, d], lse_parts [n]  ->  o [d], *lse
 */
void oracle_merge(int n, int d, const double* o_parts, const double* lse_parts,
                  int has_sink, double sink, double* o, double* lse)
{
    double M = -INFINITY;
    for (int i = 0; i < n; ++i) if (lse_parts[i] > M) M = lse_parts[i];
    double wsum = 0.0;
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    for (int i = 0; i < n; ++i) {
        double w = pow(2.0, lse_parts[i] - M);
        wsum += w;
        for (int e = 0; e < d; ++e) o[e] += w * o_parts[(int64_t)i * d + e];
    }
    double lse_all = M + log2(wsum);       /* log2 sum_t exp(s_t) over all parts */
    double denom = wsum;                     /* = sum_t exp(s_t) / 2^M */
    if (has_sink) denom += exp(sink - M * log(2.0));
    for (int e = 0; e < d; ++e) o[e] /= denom;
    *lse = lse_all;
}
