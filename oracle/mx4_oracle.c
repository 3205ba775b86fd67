/*
 * mx4_oracle.c -- plain, slow fp64 CPU oracle for the paged MXFP4 index-K scorer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: it is used by tests/, by __graft_entry__.smoke() and by the
 * cpu_baseline / --impl reference legs of bench.py.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * What it computes, and where the sources say so:
 *
 *   aiter #7061 "MiniMax-M3 index score: MXFP4 index-cache prefill scorer",
 *   section "Format": MXFP4 is e2m1 data with one e8m0 scale per 32 elements;
 *   a page of 128 tokens is [128 x 64 B data][128 x 4 B scale] = 8704 B, read
 *   through two views k_data [pages,128,64] and k_scale [pages,128,4] that
 *   each carry their own byte page stride.  The same section fixes the value
 *   of a cached element as  e2m1 x 2^(byte-127)  and the block score as the
 *   max over live tokens of the dot with Q.
 *
 *   Same page, section "Kernels": a bf16 query is rounded to e4m3 before the
 *   product; an e4m3 query is used as stored; the causal mask is shared with
 *   the fp8 scorer.
 *
 *   aiter #5518 "[FlyDSL][gfx950] explicit page strides and 64-bit rebase for
 *   FP4 MQA logits", section "Summary": the block table stride is in int32
 *   elements and physical page offsets are 64-bit; the per-token ("MQA
 *   logits") output keeps -inf for masked tokens (section "Correctness").
 *
 * Readings where the pages are silent:
 *   - nibble order: element 2i is the low nibble of byte i, 2i+1 the high one;
 *   - scale byte g of a token covers elements 32g .. 32g+31;
 *   - token i of a page sits at byte i*64 of the data view, i*4 of the scale view;
 *   - bf16 -> e4m3 is round-to-nearest-even with saturation to +-448
 *     ("satfinite"), signed zero kept, subnormals kept;
 *   - live limit of a prefill row: L = min(seq_len, prefix_len + row_pos + 1);
 *     a decode row: L = seq_len;
 *   - pages j with 128*j >= L score -inf (also pages past the request's own
 *     length but below ceil(max_seq_len/128));
 *   - sm_scale multiplies every token's dot before the max.
 *
 * Arithmetic is fp64 throughout.  With e4m3 Q (multiples of 2^-9, |q|<=448),
 * e2m1 K (multiples of 1/2, |k|<=6) and scale bytes >= 122, every product is a
 * multiple of 2^-15 below 2^12 in magnitude and a 128-term sum is exact in fp64,
 * so for such inputs the pre-scale dot is the exact real number.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_HEADS 64
#define ORC_DIM 128
#define ORC_PAGE 128
#define ORC_TOKEN_DATA_BYTES 64
#define ORC_TOKEN_SCALE_BYTES 4

/* ---------------------------------------------------------------- codecs -- */

/* e2m1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.
 * Magnitudes of codes 0..7, from the format definition. */
static const double ORC_E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code)
{
    double m = ORC_E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* e8m0: the byte is a biased power-of-two exponent, value 2^(byte-127).
 * Bytes 0 and 255 are outside the contract (aiter #7061, "Format"). */
double orc_e8m0_value(int byte)
{
    return ldexp(1.0, byte - 127);
}

/* e4m3 (fn variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * subnormal step 2^-9, largest finite 448, S.1111.111 is NaN, no infinity. */
double orc_e4m3_value(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

double orc_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a real value to e4m3: nearest representable value, ties to the
 * even mantissa, magnitudes at or above 448 saturate to 448, sign of zero
 * kept.  NaN maps to 0x7F (never produced by the generators). */
int orc_e4m3_from_double(double x)
{
    int sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x), q, n, fl, frac, r, v;
    int e, E, mant;

    if (isnan(x))
        return 0x7F;
    if (a >= 448.0)
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    frexp(a, &e);          /* a = f * 2^e with f in [0.5, 1) */
    E = e - 1;             /* floor(log2(a)) */
    if (E < -6)
        E = -6;            /* below the normal range the quantum stays 2^-9 */
    q = ldexp(1.0, E - 3); /* spacing of e4m3 values in this binade */
    n = a / q;             /* exact: q is a power of two */
    fl = floor(n);
    frac = n - fl;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    v = r * q;
    if (v == 0.0)
        return sign;
    /* encode v */
    frexp(v, &e);
    E = e - 1;
    if (E < -6) {
        mant = (int)ldexp(v, 9); /* subnormal: v = m * 2^-9 */
        return sign | mant;
    }
    mant = (int)(ldexp(v, 3 - E)) - 8;
    return sign | ((E + 7) << 3) | mant;
}

int orc_bf16_to_e4m3(uint16_t bits)
{
    return orc_e4m3_from_double(orc_bf16_value(bits));
}

/* Vector helpers for the Python side. */
void orc_bf16_to_e4m3_n(const uint16_t *in, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)orc_bf16_to_e4m3(in[i]);
}

void orc_e4m3_values_n(const uint8_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_value(in[i]);
}

/* ----------------------------------------------------------- the scorer -- */

/* Value of element d of token i in physical page p: e2m1 code times its
 * group's e8m0 scale (aiter #7061, "Format"). */
static double orc_k_value(const uint8_t *k_data, const uint8_t *k_scale,
                          int64_t sd, int64_t ss, int64_t p, int i, int d)
{
    uint8_t byte = k_data[p * sd + (int64_t)i * ORC_TOKEN_DATA_BYTES + d / 2];
    int code = (d & 1) ? (byte >> 4) : (byte & 15);
    uint8_t sbyte = k_scale[p * ss + (int64_t)i * ORC_TOKEN_SCALE_BYTES + d / 32];
    return orc_e2m1_value(code) * orc_e8m0_value(sbyte);
}

/* fp8 index cache (the format the MXFP4 cache replaces; aiter #7061, summary:
 * 128 B per token for fp8 against 68 B for MXFP4, and "Format": MXFP4 values
 * dequantised to e4m3 are exact for scale bytes 119..133).  READING: a page
 * of 128 tokens x 128 e4m3 bytes, token i at byte i*128, element d at byte d,
 * no scale; pages `sd` bytes apart. */
static double orc_k_value_fp8(const uint8_t *k, int64_t sd, int64_t p, int i, int d)
{
    return orc_e4m3_value(k[p * sd + (int64_t)i * ORC_DIM + d]);
}

/* Query value of (row, head, d).  mode 0: the e4m3 value the scorer uses
 * (bf16 rounded to e4m3, or the stored e4m3 byte).  mode 1: the unrounded
 * bf16 value, used only for the cosine context figure. */
static double orc_q_value(const void *q, int q_is_e4m3, int unquantized,
                          int64_t row, int h, int d)
{
    int64_t idx = (row * ORC_HEADS + h) * ORC_DIM + d;
    if (q_is_e4m3)
        return orc_e4m3_value(((const uint8_t *)q)[idx]);
    if (unquantized)
        return orc_bf16_value(((const uint16_t *)q)[idx]);
    return orc_e4m3_value(orc_bf16_to_e4m3(((const uint16_t *)q)[idx]));
}

/* Request that owns global query row r (prefill), or -1. */
static int orc_request_of_row(const int32_t *cu, int num_seqs, int64_t r)
{
    for (int b = 0; b < num_seqs; ++b)
        if (cu[b] <= r && r < cu[b + 1])
            return b;
    return -1;
}

/* Live limit of a row: tokens t < L are visible to it. */
int64_t orc_live_limit(int decode, const int32_t *cu, const int32_t *seq_lens,
                       const int32_t *prefix_lens, int b, int64_t r)
{
    int64_t seq = seq_lens[b];
    int64_t lim;
    if (decode)
        return seq;
    lim = (int64_t)prefix_lens[b] + (r - cu[b]) + 1;
    return lim < seq ? lim : seq;
}

/*
 * Score the query rows listed in rows[0..n_rows).
 *
 * decode = 0: prefill.  Rows are global rows of q; cu_seqlens_q[num_seqs+1]
 *             assigns them to requests; prefix_lens gives each request's
 *             cached prefix.
 * decode = 1: decode.   Row r is request r (one query row each); cu_seqlens_q
 *             and prefix_lens are ignored and L = seq_len.
 *
 * scores (optional): [n_rows, 64, P] with P = ceil(max_seq_len/128):
 *     max over live t in page j of sm_scale * sum_d Q[r,h,d] * K[t,d], else -inf.
 * logits (optional): [n_rows, 64, max_seq_len]:
 *     sm_scale * sum_d Q[r,h,d] * K[t,d] for t < L, else -inf.
 *
 * Returns 0, or -1 if a row is not in any request, -2 if a live token maps
 * to a page id outside [0, num_pool_pages), -3 on a bad argument.
 */
static int orc_score_impl(int decode, const void *q, int q_is_e4m3, int unquantized, int k_fp8,
                          const uint8_t *k_data, const uint8_t *k_scale,
                          int64_t k_data_page_stride, int64_t k_scale_page_stride,
                          const int32_t *block_table, int64_t block_table_stride,
                          const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                          const int32_t *prefix_lens, int num_seqs, int max_seq_len,
                          double sm_scale, int64_t num_pool_pages,
                          const int64_t *rows, int64_t n_rows,
                          double *scores, double *logits, int num_threads)
{
    const int64_t P = ((int64_t)max_seq_len + ORC_PAGE - 1) / ORC_PAGE;
    int status = 0;

    if (max_seq_len < 0 || num_seqs < 0 || n_rows < 0 || !q || !k_data || (!k_fp8 && !k_scale)
        || !block_table || !seq_lens || (!decode && (!cu_seqlens_q || !prefix_lens)))
        return -3;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int b = decode ? (int)r : orc_request_of_row(cu_seqlens_q, num_seqs, r);
        int64_t L, t;
        double qv[ORC_HEADS][ORC_DIM], kv[ORC_DIM];

        for (int h = 0; h < ORC_HEADS; ++h) {
            if (scores)
                for (int64_t j = 0; j < P; ++j)
                    scores[(ri * ORC_HEADS + h) * P + j] = -INFINITY;
            if (logits)
                for (t = 0; t < max_seq_len; ++t)
                    logits[(ri * ORC_HEADS + h) * (int64_t)max_seq_len + t] = -INFINITY;
        }
        if (b < 0 || b >= num_seqs) {
#pragma omp atomic write
            status = -1;
            continue;
        }
        L = orc_live_limit(decode, cu_seqlens_q, seq_lens, prefix_lens, b, r);
        if (L > max_seq_len)
            L = max_seq_len;
        for (int h = 0; h < ORC_HEADS; ++h)
            for (int d = 0; d < ORC_DIM; ++d)
                qv[h][d] = orc_q_value(q, q_is_e4m3, unquantized, r, h, d);

        for (t = 0; t < L; ++t) {
            int64_t j = t / ORC_PAGE;
            int i = (int)(t % ORC_PAGE);
            int64_t p = block_table[(int64_t)b * block_table_stride + j];
            if (p < 0 || (num_pool_pages > 0 && p >= num_pool_pages)) {
#pragma omp atomic write
                status = -2;
                break;
            }
            for (int d = 0; d < ORC_DIM; ++d)
                kv[d] = k_fp8 ? orc_k_value_fp8(k_data, k_data_page_stride, p, i, d)
                              : orc_k_value(k_data, k_scale, k_data_page_stride,
                                            k_scale_page_stride, p, i, d);
            for (int h = 0; h < ORC_HEADS; ++h) {
                double dot = 0.0, val;
                for (int d = 0; d < ORC_DIM; ++d)
                    dot += qv[h][d] * kv[d];
                val = sm_scale * dot;
                if (logits)
                    logits[(ri * ORC_HEADS + h) * (int64_t)max_seq_len + t] = val;
                if (scores) {
                    double *s = &scores[(ri * ORC_HEADS + h) * P + j];
                    if (val > *s)
                        *s = val;
                }
            }
        }
    }
    return status;
}

/* MXFP4 index cache: the scorer as specified. */
int orc_score(int decode, const void *q, int q_is_e4m3, int unquantized,
              const uint8_t *k_data, const uint8_t *k_scale,
              int64_t k_data_page_stride, int64_t k_scale_page_stride,
              const int32_t *block_table, int64_t block_table_stride,
              const int32_t *cu_seqlens_q, const int32_t *seq_lens,
              const int32_t *prefix_lens, int num_seqs, int max_seq_len,
              double sm_scale, int64_t num_pool_pages,
              const int64_t *rows, int64_t n_rows,
              double *scores, double *logits, int num_threads)
{
    return orc_score_impl(decode, q, q_is_e4m3, unquantized, 0, k_data, k_scale, k_data_page_stride,
                          k_scale_page_stride, block_table, block_table_stride, cu_seqlens_q, seq_lens,
                          prefix_lens, num_seqs, max_seq_len, sm_scale, num_pool_pages, rows, n_rows,
                          scores, logits, num_threads);
}

/* fp8 index cache: the same scorer with K read as plain e4m3 bytes. */
int orc_score_fp8(int decode, const void *q, int q_is_e4m3, int unquantized,
                  const uint8_t *k_fp8, int64_t k_page_stride,
                  const int32_t *block_table, int64_t block_table_stride,
                  const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                  const int32_t *prefix_lens, int num_seqs, int max_seq_len,
                  double sm_scale, int64_t num_pool_pages,
                  const int64_t *rows, int64_t n_rows,
                  double *scores, double *logits, int num_threads)
{
    return orc_score_impl(decode, q, q_is_e4m3, unquantized, 1, k_fp8, NULL, k_page_stride, 0,
                          block_table, block_table_stride, cu_seqlens_q, seq_lens, prefix_lens,
                          num_seqs, max_seq_len, sm_scale, num_pool_pages, rows, n_rows, scores,
                          logits, num_threads);
}

/* Number of live (row, token) pairs over the listed rows: the causal mask
 * alone, for closed-form checks of the live limit. */
int64_t orc_live_pairs(int decode, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                       const int32_t *prefix_lens, int num_seqs, int max_seq_len,
                       const int64_t *rows, int64_t n_rows)
{
    int64_t total = 0;
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int b = decode ? (int)r : orc_request_of_row(cu_seqlens_q, num_seqs, r);
        int64_t L;
        if (b < 0 || b >= num_seqs)
            continue;
        L = orc_live_limit(decode, cu_seqlens_q, seq_lens, prefix_lens, b, r);
        if (L > max_seq_len)
            L = max_seq_len;
        if (L > 0)
            total += L;
    }
    return total;
}

/* ------------------------------------------------------- the page writer -- */
/*
 * Quantising a bf16 index key into an MXFP4 page slot.  The pages say only
 * that the index key is quantised straight into the 8704 B pool page (ATOM
 * #2770 "MiniMax-M3.1 MXFP4 sparse KV cache and index cache", section "How it
 * works", item "Write") with a per-1x32 MXFP4 quantiser (aiter #7061,
 * section "Tests": the cache is built with per_1x32_f4_quant).  They do not
 * state the rounding rule.  READING, from the OCP Microscaling Formats (MX)
 * v1.0 conversion rule:
 *   - shared exponent of a 32-element group: E = floor(log2(amax)) - 2, where
 *     2 is the largest exponent of e2m1 (its top value 6 = 1.5 x 2^2);
 *   - scale byte = E + 127, clamped to [1, 254] (the scorer's contract
 *     excludes bytes 0 and 255); an all-zero group takes byte 127;
 *   - element = x / 2^(byte-127) rounded to the nearest e2m1 value, ties to
 *     the even code, magnitudes past 6 saturate to 6, sign kept (also for a
 *     result of zero).
 * Inputs are finite (bf16 Inf/NaN are outside the contract).
 */

/* Round a real value to an e2m1 code: nearest of {0,.5,1,1.5,2,3,4,6} in
 * magnitude, ties to the even code, saturating at 6, sign bit kept. */
int orc_e2m1_from_double(double x)
{
    int sign = signbit(x) ? 8 : 0;
    double a = fabs(x), q, n, fl, frac, r, v;
    int e, E;

    if (a >= 6.0)
        return sign | 7;
    if (a == 0.0)
        return sign;
    frexp(a, &e);
    E = e - 1;             /* floor(log2(a)) */
    if (E < 0)
        E = 0;             /* below 1 the spacing stays 1/2 (subnormal 0.5) */
    q = ldexp(1.0, E - 1); /* spacing of e2m1 values in this binade */
    n = a / q;
    fl = floor(n);
    frac = n - fl;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    v = r * q;             /* at most 6: 5.x rounds to 4 or 6 */
    if (v == 0.0)
        return sign;
    if (v < 1.0)
        return sign | 1;                       /* 0.5 */
    frexp(v, &e);
    E = e - 1;                                 /* 0, 1 or 2 */
    return sign | ((E + 1) << 1) | (int)(ldexp(v, 1 - E) - 2.0);
}

/* One 32-element group: its scale byte and 32 codes (code i for element i). */
int orc_quantize_group(const double *x, uint8_t *codes)
{
    double amax = 0.0;
    int e, byte;
    for (int i = 0; i < 32; ++i)
        if (fabs(x[i]) > amax)
            amax = fabs(x[i]);
    if (amax == 0.0) {
        byte = 127;
    } else {
        frexp(amax, &e);
        byte = (e - 1) - 2 + 127;
        if (byte < 1)
            byte = 1;
        if (byte > 254)
            byte = 254;
    }
    for (int i = 0; i < 32; ++i)
        codes[i] = (uint8_t)orc_e2m1_from_double(x[i] / ldexp(1.0, byte - 127));
    return byte;
}

/*
 * Write num_tokens bf16 keys (row t at k + t*k_row_stride elements, 128
 * elements each) into the page slots named by slot_mapping: slot s is token
 * s % 128 of physical page s / 128.  Token i of page p keeps its 64 code bytes
 * at k_data[p*sd + i*64] (element 2c in the low nibble of byte c, 2c+1 in the
 * high nibble) and its 4 scale bytes at k_scale[p*ss + i*4] (byte g for
 * elements 32g..32g+31).  Negative slots are skipped (padding); a slot whose
 * page is outside [0, num_pool_pages) (when num_pool_pages > 0) is skipped
 * and counted.  Returns the number of such out-of-pool slots.
 */
int64_t orc_write_index_k(const uint16_t *k, int64_t num_tokens, int64_t k_row_stride,
                          const int64_t *slot_mapping, uint8_t *k_data, uint8_t *k_scale,
                          int64_t sd, int64_t ss, int64_t num_pool_pages)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        int64_t p = s / ORC_PAGE, i = s % ORC_PAGE;
        if (num_pool_pages > 0 && p >= num_pool_pages) {
            ++bad;
            continue;
        }
        uint8_t *dst = k_data + p * sd + i * ORC_TOKEN_DATA_BYTES;
        uint8_t *sdst = k_scale + p * ss + i * ORC_TOKEN_SCALE_BYTES;
        for (int g = 0; g < 4; ++g) {
            double x[32];
            uint8_t codes[32];
            for (int j = 0; j < 32; ++j)
                x[j] = orc_bf16_value(k[t * k_row_stride + 32 * g + j]);
            sdst[g] = (uint8_t)orc_quantize_group(x, codes);
            for (int c = 0; c < 16; ++c)
                dst[16 * g + c] = (uint8_t)(codes[2 * c] | (codes[2 * c + 1] << 4));
        }
    }
    return bad;
}

/* ---------------------------------------------------- top-k page selection -- */
/*
 * The step after the scorer: each query row reads at most `topk` pages of its
 * request, chosen from the block scores (ATOM #2770 "MiniMax-M3.1 MXFP4 sparse
 * KV cache and index cache", "How it works": the index scores feed the
 * selection and the emit of a page-level block table, one page a block for
 * 128-token pages; the local block and the tail page are always selected; a
 * row reads at most topk pages).  READINGS where the pages are silent:
 *   - the 64 index heads form kv_groups contiguous groups; a page's value for
 *     a group is the max of its block scores over the group's heads;
 *   - live pages of a row are j < ceil(L/128) with L the scorer's live limit;
 *     the last min(local, live) of them are always selected;
 *   - the other topk - forced slots go to the live pages with the largest
 *     values, ties to the lower page index;
 *   - the emit lists the selected pages' physical ids (block_table) in
 *     ascending page order, then -1 up to topk; count = number selected;
 *   - tokens (optional) = the live tokens of the selected pages: the valid
 *     context of the emitted list, read in list order, for the attention
 *     step (page j holds min(128, L - 128 j) live tokens).
 * Values are the fp32 block scores as given; every comparison is exact.
 */
static int orc_cmp_desc_value_asc_index(const void *pa, const void *pb)
{
    const double *a = (const double *)pa, *b = (const double *)pb;
    if (a[0] > b[0]) return -1;
    if (a[0] < b[0]) return 1;
    return (a[1] < b[1]) ? -1 : (a[1] > b[1]);
}

/*
 * scores [n_rows_total, 64, P] fp32 (P = ceil(max_seq_len/128)); rows as for
 * orc_score.  sel [n_rows, kv_groups, topk] int32, count [n_rows, kv_groups],
 * tokens [n_rows, kv_groups] int32 or NULL.
 * Returns 0, or -1 for a row outside every request, -3 for bad arguments.
 */
int orc_topk(int decode, const float *scores, int max_seq_len,
             const int32_t *block_table, int64_t block_table_stride,
             const int32_t *cu_seqlens_q, const int32_t *seq_lens, const int32_t *prefix_lens,
             int num_seqs, int topk, int local, int kv_groups,
             const int64_t *rows, int64_t n_rows, int32_t *sel, int32_t *count, int32_t *tokens)
{
    const int64_t P = ((int64_t)max_seq_len + ORC_PAGE - 1) / ORC_PAGE;
    int status = 0;
    if (topk < 1 || local < 0 || local > topk || kv_groups < 1 || ORC_HEADS % kv_groups != 0 || !scores
        || !sel || !count || !block_table || !seq_lens || (!decode && (!cu_seqlens_q || !prefix_lens)))
        return -3;
    const int hg = ORC_HEADS / kv_groups;
    double *cand = (double *)malloc(sizeof(double) * 2 * (size_t)(P > 0 ? P : 1));
    char *pick = (char *)malloc((size_t)(P > 0 ? P : 1));
    if (!cand || !pick) {
        free(cand);
        free(pick);
        return -3;
    }
    for (int64_t ri = 0; ri < n_rows; ++ri) {
        int64_t r = rows[ri];
        int b = decode ? (int)r : orc_request_of_row(cu_seqlens_q, num_seqs, r);
        for (int g = 0; g < kv_groups; ++g) {
            int32_t *out = sel + (ri * kv_groups + g) * (int64_t)topk;
            int64_t L, nl, forced, n_c = 0, n_sel = 0, n_tok = 0;
            for (int i = 0; i < topk; ++i)
                out[i] = -1;
            count[ri * kv_groups + g] = 0;
            if (tokens)
                tokens[ri * kv_groups + g] = 0;
            if (b < 0 || b >= num_seqs) {
                status = -1;
                continue;
            }
            L = orc_live_limit(decode, cu_seqlens_q, seq_lens, prefix_lens, b, r);
            if (L > max_seq_len)
                L = max_seq_len;
            nl = L > 0 ? (L + ORC_PAGE - 1) / ORC_PAGE : 0;
            forced = local < nl ? local : nl;
            for (int64_t j = 0; j < nl; ++j)
                pick[j] = (j >= nl - forced);
            /* candidates: the live pages before the forced tail */
            for (int64_t j = 0; j < nl - forced; ++j) {
                double v = -INFINITY;
                for (int h = g * hg; h < (g + 1) * hg; ++h) {
                    double s = scores[(r * ORC_HEADS + h) * P + j];
                    if (s > v)
                        v = s;
                }
                cand[2 * n_c] = v;
                cand[2 * n_c + 1] = (double)j;
                ++n_c;
            }
            qsort(cand, (size_t)n_c, 2 * sizeof(double), orc_cmp_desc_value_asc_index);
            for (int64_t i = 0; i < n_c && i < topk - forced; ++i)
                pick[(int64_t)cand[2 * i + 1]] = 1;
            for (int64_t j = 0; j < nl; ++j)
                if (pick[j]) {
                    out[n_sel++] = block_table[(int64_t)b * block_table_stride + j];
                    n_tok += (L - ORC_PAGE * j < ORC_PAGE) ? L - ORC_PAGE * j : ORC_PAGE;
                }
            count[ri * kv_groups + g] = (int32_t)n_sel;
            if (tokens)
                tokens[ri * kv_groups + g] = (int32_t)n_tok;
        }
    }
    free(cand);
    free(pick);
    return status;
}

/* -------------------------------------- sparse paged-attention decode -- */
/*
 * Decode attention over the pages a row selected, with K and V in MXFP4
 * (aiter pa_decode MXFP4, as described in ATOM #2770 "MiniMax-M3.1 MXFP4
 * sparse KV cache and index cache", commit "pa_decode MXFP4": K and V are
 * e2m1 data plus one e8m0 byte per 32 elements along head_dim, read through
 * data/scale views with their own page and head strides; the fp8 query is
 * used as stored; invalid tokens get a -inf score; (token, kv head) pairs are
 * folded into rows that each read at most topk pages).  Definition, per row
 * r and query head h of the row's group of G heads:
 *     s[t]   = softmax_scale * sum_d q[r,h,d] * K[t,d]      (t valid)
 *     out    = sum_t softmax(s)[t] * V[t,:]
 * READINGS: head_dim 128 for K and V; the row's tokens are those of its
 * block-table pages in list order, the first context_len of them valid (the
 * selection lists pages in ascending order with the tail page last);
 * page p of kv head k holds token i's K codes at k_data + p*kd_ps + k*kd_hs +
 * i*64 and scales at k_scale + p*ks_ps + k*ks_hs + i*4 (V the same); a row
 * with no valid token outputs zeros.  fp64 here; the stored output is bf16.
 */
int orc_pa_decode(const uint8_t *q, int64_t n_rows, int kv_heads, int groups,
                  const uint8_t *k_data, const uint8_t *k_scale, int64_t kd_ps, int64_t kd_hs,
                  int64_t ks_ps, int64_t ks_hs,
                  const uint8_t *v_data, const uint8_t *v_scale, int64_t vd_ps, int64_t vd_hs,
                  int64_t vs_ps, int64_t vs_hs,
                  const int32_t *block_table, int64_t bt_stride, const int32_t *context_lens,
                  double softmax_scale, int64_t num_pool_pages, double *out, int num_threads)
{
    int status = 0;
    if (n_rows < 0 || kv_heads < 1 || groups < 1 || !q || !k_data || !k_scale || !v_data || !v_scale
        || !block_table || !context_lens || !out)
        return -3;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int kh = 0; kh < kv_heads; ++kh) {
            const int64_t row = r * kv_heads + kh;
            const int64_t ctx = context_lens[row];
            double *o = out + row * groups * ORC_DIM;
            for (int64_t i = 0; i < (int64_t)groups * ORC_DIM; ++i)
                o[i] = 0.0;
            if (ctx <= 0)
                continue;
            double *s = (double *)malloc(sizeof(double) * (size_t)ctx * (size_t)groups);
            double kv[ORC_DIM];
            if (!s) {
#pragma omp atomic write
                status = -3;
                continue;
            }
            for (int64_t t = 0; t < ctx; ++t) {
                int64_t p = block_table[row * bt_stride + t / ORC_PAGE];
                int i = (int)(t % ORC_PAGE);
                if (p < 0 || (num_pool_pages > 0 && p >= num_pool_pages)) {
#pragma omp atomic write
                    status = -2;
                    p = 0;
                }
                for (int d = 0; d < ORC_DIM; ++d)
                    kv[d] = orc_k_value(k_data + kh * kd_hs, k_scale + kh * ks_hs, kd_ps, ks_ps, p, i, d);
                for (int h = 0; h < groups; ++h) {
                    double dot = 0.0;
                    for (int d = 0; d < ORC_DIM; ++d)
                        dot += orc_e4m3_value(q[(row * groups + h) * ORC_DIM + d]) * kv[d];
                    s[t * groups + h] = softmax_scale * dot;
                }
            }
            for (int h = 0; h < groups; ++h) {
                double m = -INFINITY, sum = 0.0;
                for (int64_t t = 0; t < ctx; ++t)
                    if (s[t * groups + h] > m)
                        m = s[t * groups + h];
                for (int64_t t = 0; t < ctx; ++t) {
                    s[t * groups + h] = exp(s[t * groups + h] - m);
                    sum += s[t * groups + h];
                }
                for (int64_t t = 0; t < ctx; ++t)
                    s[t * groups + h] /= sum;
            }
            for (int64_t t = 0; t < ctx; ++t) {
                int64_t p = block_table[row * bt_stride + t / ORC_PAGE];
                int i = (int)(t % ORC_PAGE);
                if (p < 0 || (num_pool_pages > 0 && p >= num_pool_pages))
                    p = 0;
                for (int d = 0; d < ORC_DIM; ++d)
                    kv[d] = orc_k_value(v_data + kh * vd_hs, v_scale + kh * vs_hs, vd_ps, vs_ps, p, i, d);
                for (int h = 0; h < groups; ++h)
                    for (int d = 0; d < ORC_DIM; ++d)
                        o[h * ORC_DIM + d] += s[t * groups + h] * kv[d];
            }
            free(s);
        }
    }
    return status;
}
