/*
 * mx4_index.h -- C ABI of the paged MXFP4 index-K scorer for GB300 (sm_103a).
 *
 * The scorer of a sparse-attention indexer: for every query row, head and
 * 128-token page of the request's context it writes the largest causal-masked,
 * sm_scale-scaled logit of the page (a "block score"), or -inf when the page
 * has no live token.  An optional per-token mode writes the logits
 * themselves.
 *
 * Sources (each entry point cites the passage that defines it):
 *   [P1] aiter #7061, "MiniMax-M3 index score: MXFP4 index-cache prefill
 *        scorer": sections "Format", "Kernels", "Tests".
 *   [P2] ATOM #2770, "MiniMax-M3.1 MXFP4 sparse KV cache and index cache":
 *        section "How it works" and the pa_decode MXFP4 commit message.
 *   [P3] aiter #5518, "[FlyDSL][gfx950] explicit page strides and 64-bit
 *        rebase for FP4 MQA logits": sections "Summary", decode auto-CTA
 *        table, "Correctness / regression".
 *
 * Shapes and layouts (H = 64 heads, D = 128, 128-token pages):
 *   q            [total_rows, 64, 128], contiguous; bf16 (q_is_e4m3 = 0) or
 *                e4m3 bytes (q_is_e4m3 = 1).  16-byte aligned.
 *   k_data       page p's e2m1 codes at k_data + p * k_data_page_stride:
 *                [128 tokens][64 bytes]; element 2i in the low nibble of byte
 *                i, element 2i+1 in the high nibble.  32-byte aligned;
 *                k_data_page_stride >= 8192 and a multiple of 32 (a GB300
 *                TMA rule for 4-bit data).
 *   k_scale      page p's e8m0 bytes at k_scale + p * k_scale_page_stride:
 *                [128 tokens][4 bytes], byte g scales elements 32g..32g+31.
 *                16-byte aligned; k_scale_page_stride >= 512, multiple of 16.
 *                The single-region page of [P1] is k_scale = k_data + 8192
 *                with both strides 8704.
 *   block_table  int32 [num_seqs, block_table_stride] physical page ids;
 *                entries at or past ceil(seq_len/128) are never read.
 *   out          fp32 [total_rows, 64, ceil(max_seq_len/128)] block scores,
 *                or [total_rows, 64, max_seq_len] per-token logits.  Every
 *                cell of every existing row is written (no pre-fill needed).
 *                16-byte aligned.
 *
 * Ownership: every pointer is a borrowed device pointer owned by the caller.
 * The library allocates no device memory; its only device state is one
 * status word in a static device variable of the loaded module.
 *
 * Streams: calls enqueue on `stream` (a cudaStream_t; NULL = legacy default
 * stream), never synchronise, and read no device data on the host, so a
 * sequence of calls can be captured in a CUDA graph after a first
 * (warm-up) call on the device.  The scorer, writer and attention kernels
 * are launched as programmatic dependent launches: their set-up (barriers,
 * tensor memory, descriptor prefetch) may overlap the end of the previous
 * kernel of the stream, but every global read and write waits for that
 * kernel to complete, so stream order semantics are unchanged.
 *
 * Errors: host-checkable faults return a status before anything is
 * launched.  A call with no output cell (num_seqs, max_seq_len or, for
 * prefill, max_query_len equal to 0) returns MX4_OK at once; its pointers
 * are not checked.  Faults only the device can see (a page id outside
 * [0, num_pool_pages) for a live page, an internal wait that ran out) set
 * bits of the device status word and leave the affected outputs undefined;
 * read them with mx4_index_get_device_status.  No C++ exception crosses
 * this ABI.
 */
#ifndef MX4_INDEX_H
#define MX4_INDEX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MX4_ABI_VERSION 2

typedef enum {
    MX4_OK = 0,
    MX4_ERR_INVALID_ARG = 1, /* null pointer, negative size, narrow view or table, bad sm_scale */
    MX4_ERR_MISALIGNED = 2,  /* pointer or stride alignment rule broken */
    MX4_ERR_UNSUPPORTED = 3, /* size outside what the kernels support */
    MX4_ERR_CUDA = 4         /* a CUDA runtime/driver call failed */
} mx4_status;

/* Device status bits (mx4_index_get_device_status). */
#define MX4_DEV_BAD_PAGE 0x1u /* a live page id (scorer) or a slot's page (writer) was outside [0, num_pool_pages) */
#define MX4_DEV_TIMEOUT 0x2u  /* an internal wait gave up; the kernel returned early */
/* With MX4_DEV_TIMEOUT, bit (8 + site) names the wait that gave up: site 0 =
 * producer waiting for a free smem stage, 1 = MMA waiting for the query tile,
 * 2 = MMA waiting for a page's bytes, 3 = MMA waiting for a free
 * accumulator, 4 = epilogue waiting for a free query buffer, 5 = epilogue
 * waiting for an accumulator; attention: 6 = copy issue, 7 = MMA issue,
 * 8 = softmax or widening warps; 9 = a CTA leaving while a copy it armed
 * had not landed.  Diagnostic only. */

/*
 * Block scores for ragged prefill (causal) rows.  [P1] "Kernels":
 * score_prefill_flydsl_fp4(idx_q, k_data, k_scale, block_table, cu_seqlens_q,
 * seq_lens, prefix_lens, max_query_len, max_seq_len, sm_scale, out); [P1]
 * "Format" for the page, the value e2m1 x 2^(byte-127) and the block score
 * (max over live tokens of the dot with Q); [P3] "Summary" for the page
 * strides (bytes), the block-table stride (int32 elements) and 64-bit page
 * offsets.
 *
 * Row r of request b (cu_seqlens_q[b] <= r < cu_seqlens_q[b+1]) sees token t
 * iff t < min(seq_lens[b], prefix_lens[b] + (r - cu_seqlens_q[b]) + 1).
 * out[r, h, j] = sm_scale * max over live t in [128j, 128j+128) of
 *                sum_d Q8[r,h,d] * e2m1(K[t,d]) * 2^(S[t,d/32]-127),
 * accumulated in fp32 on the tensor cores; -inf if page j has no live token.
 * Q8 is the bf16 query rounded to e4m3 (nearest even, saturating to +-448),
 * or the e4m3 query as stored.
 *
 * Appended scalars (not on the page, needed to size a launch without reading
 * device memory): num_seqs = B (cu_seqlens_q has B+1 entries),
 * block_table_stride in int32 elements (>= ceil(max_seq_len/128)),
 * num_pool_pages = pages addressable through both views (>= 1, < 2^31).
 * max_query_len must be >= every request's row count and max_seq_len >=
 * every seq_len.  sm_scale must be finite and > 0.
 */
mx4_status mx4_index_score_prefill(const void *q, int q_is_e4m3, const uint8_t *k_data,
                                   const uint8_t *k_scale, int64_t k_data_page_stride,
                                   int64_t k_scale_page_stride, const int32_t *block_table,
                                   const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                   const int32_t *prefix_lens, int max_query_len,
                                   int max_seq_len, float sm_scale, float *out, void *stream,
                                   int num_seqs, int64_t block_table_stride,
                                   int64_t num_pool_pages);

/*
 * Block scores for decode: one query row per request (q [num_seqs, 64, 128]),
 * token t live iff t < seq_lens[b].  Same arithmetic and output rule as the
 * prefill call.  [P2] "How it works" (decode scoring inside the CUDA graph)
 * and [P3] decode auto-CTA table: the context of each request is split over
 * several CTAs by a grid chosen on the host from num_seqs and max_seq_len
 * only, so the launch is stable under graph replay.
 */
mx4_status mx4_index_score_decode(const void *q, int q_is_e4m3, const uint8_t *k_data,
                                  const uint8_t *k_scale, int64_t k_data_page_stride,
                                  int64_t k_scale_page_stride, const int32_t *block_table,
                                  const int32_t *seq_lens, int max_seq_len, float sm_scale,
                                  float *out, void *stream, int num_seqs,
                                  int64_t block_table_stride, int64_t num_pool_pages);

/*
 * Per-token logits for prefill rows ([P3] "Summary": paged MXFP4 MQA logits;
 * "Correctness": -inf masks retained).  logits[r, h, t] = sm_scale *
 * sum_d Q8[r,h,d] * K[t,d] for live t, -inf for every other t < max_seq_len.
 * logits is fp32 [total_rows, 64, max_seq_len].  Arguments as for
 * mx4_index_score_prefill.
 */
mx4_status mx4_index_logits_prefill(const void *q, int q_is_e4m3, const uint8_t *k_data,
                                    const uint8_t *k_scale, int64_t k_data_page_stride,
                                    int64_t k_scale_page_stride, const int32_t *block_table,
                                    const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                    const int32_t *prefix_lens, int max_query_len,
                                    int max_seq_len, float sm_scale, float *logits,
                                    void *stream, int num_seqs, int64_t block_table_stride,
                                    int64_t num_pool_pages);

/*
 * Per-token logits for decode rows: logits fp32 [num_seqs, 64, max_seq_len],
 * -inf for t >= seq_lens[b].  Arguments as for mx4_index_score_decode.
 */
mx4_status mx4_index_logits_decode(const void *q, int q_is_e4m3, const uint8_t *k_data,
                                   const uint8_t *k_scale, int64_t k_data_page_stride,
                                   int64_t k_scale_page_stride, const int32_t *block_table,
                                   const int32_t *seq_lens, int max_seq_len, float sm_scale,
                                   float *logits, void *stream, int num_seqs,
                                   int64_t block_table_stride, int64_t num_pool_pages);

/*
 * The same scorer over an fp8 index cache, the format the MXFP4 cache
 * replaces ([P1] summary: 128 B per token for fp8 against 68 B for MXFP4;
 * [P1] "Kernels": the fp8 and MXFP4 scorers share tiling, Q staging, causal
 * mask, folds and stores and differ only in the K side).  READING of the
 * fp8 page: 128 tokens x 128 e4m3 bytes, token i at byte i*128 of the page,
 * element d at byte d, no scale; logit = sm_scale * sum_d Q8 * e4m3(K).
 *
 *   k_fp8          page p at k_fp8 + p * k_page_stride; 16-byte aligned,
 *                  k_page_stride >= 16384 and a multiple of 16.
 * Every other argument, the outputs, ownership, streams and errors are as
 * for the MXFP4 calls above (k_scale and its stride do not exist here).
 */
mx4_status mx4_index_score_prefill_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8,
                                       int64_t k_page_stride, const int32_t *block_table,
                                       const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                       const int32_t *prefix_lens, int max_query_len, int max_seq_len,
                                       float sm_scale, float *out, void *stream, int num_seqs,
                                       int64_t block_table_stride, int64_t num_pool_pages);

mx4_status mx4_index_score_decode_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8,
                                      int64_t k_page_stride, const int32_t *block_table,
                                      const int32_t *seq_lens, int max_seq_len, float sm_scale, float *out,
                                      void *stream, int num_seqs, int64_t block_table_stride,
                                      int64_t num_pool_pages);

mx4_status mx4_index_logits_prefill_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8,
                                        int64_t k_page_stride, const int32_t *block_table,
                                        const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                        const int32_t *prefix_lens, int max_query_len, int max_seq_len,
                                        float sm_scale, float *logits, void *stream, int num_seqs,
                                        int64_t block_table_stride, int64_t num_pool_pages);

mx4_status mx4_index_logits_decode_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8,
                                       int64_t k_page_stride, const int32_t *block_table,
                                       const int32_t *seq_lens, int max_seq_len, float sm_scale,
                                       float *logits, void *stream, int num_seqs,
                                       int64_t block_table_stride, int64_t num_pool_pages);

/*
 * Top-k page selection, the step after the scorer ([P2] "How it works": the
 * index scores feed the selection and the emit of a page-level block table,
 * one page a block for 128-token pages, with the local and tail blocks always
 * selected; a row reads at most topk pages).  READINGS where the sources are
 * silent: the 64 index heads form kv_groups contiguous groups (64/kv_groups
 * heads each); a page's value for a group is the max of its block scores over
 * those heads; a row's live pages are j < ceil(L/128) with the scorer's live
 * limit L; the last min(local_pages, live) live pages are always selected and
 * the other topk - forced slots go to the largest values, ties to the lower
 * page index.
 *
 *   scores      fp32 [total_rows, 64, ceil(max_seq_len/128)], the scorer's
 *               block scores (device, 4-byte aligned).
 *   sel         int32 [total_rows, kv_groups, topk]: physical page ids of the
 *               selected pages in ascending page order, then -1.
 *   count       int32 [total_rows, kv_groups]: pages selected.
 *   sel_tokens  int32 [total_rows, kv_groups] or NULL: the live tokens of the
 *               selected pages (128 for each but the row's last live page,
 *               which holds L - 128 (ceil(L/128) - 1)); this is the context
 *               the attention step reads from the emitted list in order
 *               (mx4_sparse_pa_decode's context_lens).
 *   topk >= 1, 0 <= local_pages <= topk, kv_groups divides 64,
 *   ceil(max_seq_len/128) <= 16384 (MX4_ERR_UNSUPPORTED beyond).
 * The request arguments (block_table, cu_seqlens_q, seq_lens, prefix_lens,
 * max_query_len, num_seqs, block_table_stride) are those of the scorer call
 * that produced `scores`.  Every row that exists is written; a call with no
 * row returns MX4_OK at once.  Comparisons are exact (fp32 values, -0 equal
 * to +0), so the selection is deterministic.
 */
mx4_status mx4_index_topk_prefill(const float *scores, const int32_t *block_table, const int32_t *cu_seqlens_q,
                                  const int32_t *seq_lens, const int32_t *prefix_lens, int max_query_len,
                                  int max_seq_len, int topk, int local_pages, int kv_groups, int32_t *sel,
                                  int32_t *count, int32_t *sel_tokens, void *stream, int num_seqs,
                                  int64_t block_table_stride);

mx4_status mx4_index_topk_decode(const float *scores, const int32_t *block_table, const int32_t *seq_lens,
                                 int max_seq_len, int topk, int local_pages, int kv_groups, int32_t *sel,
                                 int32_t *count, int32_t *sel_tokens, void *stream, int num_seqs,
                                 int64_t block_table_stride);

/*
 * Sparse paged-attention decode over MXFP4 K and V: each row (a decode token
 * and one KV head) attends over the pages its block table lists.  [P2] "How
 * it works" (sparse attention: (token, kv head) folded into rows, each row
 * reads at most topk pages) and the pa_decode MXFP4 commit message (K and V
 * as e2m1 + one e8m0 byte per 32 elements along head_dim through data/scale
 * views with page and head strides; the e4m3 query used as stored; invalid
 * tokens get a -inf score and a zero V; V widened to bf16, P bf16):
 *     s[t] = softmax_scale * sum_d q[h,d] K[t,d],  out[h,:] = softmax(s) V
 * over the row's valid tokens: the first context_lens[row] tokens of its
 * listed pages, in list order (the top-k emit lists pages in ascending order
 * with the partial tail page last).
 *
 *   q              e4m3 bytes [num_rows, kv_heads, groups, 128], 16-byte
 *                  aligned; groups <= 16.
 *   K / V views    page p of KV head k: codes at data + p * page_stride +
 *                  k * head_stride (128 tokens x 64 B), scales at scale +
 *                  p * page_stride + k * head_stride (128 tokens x 4 B).
 *                  K codes 32-byte aligned with strides multiple of 32; K
 *                  scales, V codes and V scales 16-byte aligned with strides
 *                  multiple of 16; head strides >= 8192 / 512, page strides
 *                  >= kv_heads * head stride.  A [pages, kv_heads, 8704] pool
 *                  has data = pool, scale = pool + 8192, page stride
 *                  kv_heads * 8704, head stride 8704 for both.
 *   block_table    int32 [num_rows, kv_heads, block_table_width] page ids;
 *                  entries past ceil(context_len / 128) are never read;
 *                  block_table_width <= 24 (MX4_ERR_UNSUPPORTED beyond).
 *   context_lens   int32 [num_rows, kv_heads]; clamped to [0, width*128].
 *   out            bf16 [num_rows, kv_heads, groups, 128]; a row with no
 *                  valid token is written with zeros.
 * A listed page id outside [0, num_pool_pages) reads page 0 and sets
 * MX4_DEV_BAD_PAGE.  Pointers are caller-owned device memory; no allocation;
 * num_rows == 0 returns MX4_OK at once.
 */
mx4_status mx4_sparse_pa_decode(const uint8_t *q, int64_t num_rows, int kv_heads, int groups,
                                const uint8_t *k_data, const uint8_t *k_scale, int64_t k_data_page_stride,
                                int64_t k_data_head_stride, int64_t k_scale_page_stride,
                                int64_t k_scale_head_stride, const uint8_t *v_data, const uint8_t *v_scale,
                                int64_t v_data_page_stride, int64_t v_data_head_stride,
                                int64_t v_scale_page_stride, int64_t v_scale_head_stride,
                                const int32_t *block_table, int block_table_width, const int32_t *context_lens,
                                float softmax_scale, void *out, int64_t num_pool_pages, void *stream);

/*
 * The query-preparation step on its own: n bf16 values (raw bits) rounded to
 * e4m3 bytes, nearest even, saturating to +-448, signed zero kept ([P1]
 * "Kernels": a bf16 query is rounded to e4m3 in-kernel; the scorers above do
 * this inside the kernel with the same device function).  Both pointers are
 * device pointers; n >= 0.
 */
mx4_status mx4_quantize_q_e4m3(const uint16_t *q_bf16, uint8_t *q_e4m3, int64_t n, void *stream);

/*
 * Index-K page writer: quantise num_tokens bf16 keys into MXFP4 page slots.
 * [P2] "How it works", item "Write": the index key is quantised straight
 * into its 8704 B pool page, no bf16 stage; [P1] "Tests": the cache is built
 * by a per-1x32 MXFP4 quantiser; [P1] "Format" for the page.  The rounding
 * rule is not stated by the sources; this call implements the OCP MX v1.0
 * conversion: per 32-element group, scale byte = floor(log2 amax) - 2 + 127
 * clamped to [1, 254] (127 for an all-zero group), each element rounded to
 * the nearest e2m1 value of x / 2^(byte-127), ties to the even code,
 * saturating at 6, its sign bit kept.
 *
 *   k             bf16 bits, key of token t = 128 elements at
 *                 k + t * k_row_stride (elements); k_row_stride >= 128.
 *                 2-byte aligned (rows 16-byte aligned take 128-bit loads).
 *   slot_mapping  int64 [num_tokens]: slot s = token s % 128 of page s / 128;
 *                 a negative slot is padding and writes nothing.
 *   k_data, k_scale, strides   the page views of the scorer calls: token i
 *                 of page p gets its 64 code bytes at k_data + p *
 *                 k_data_page_stride + 64 i and its 4 scale bytes at k_scale
 *                 + p * k_scale_page_stride + 4 i.  k_data 16-byte aligned,
 *                 k_data_page_stride >= 8192 and a multiple of 16; k_scale
 *                 4-byte aligned, k_scale_page_stride >= 512 and a multiple
 *                 of 4.
 *   num_pool_pages  > 0: a slot whose page is >= num_pool_pages is skipped
 *                 and sets MX4_DEV_BAD_PAGE; <= 0: unchecked.
 *
 * All pointers are caller-owned device pointers.  num_tokens == 0 returns
 * MX4_OK without checking pointers.  Bytes of slots not named are not
 * touched; two tokens naming one slot race (either result may remain).
 * Keys must be finite (Inf/NaN give unspecified codes, no fault).
 */
mx4_status mx4_index_k_write(const void *k, int64_t num_tokens, int64_t k_row_stride,
                             const int64_t *slot_mapping, uint8_t *k_data, uint8_t *k_scale,
                             int64_t k_data_page_stride, int64_t k_scale_page_stride,
                             int64_t num_pool_pages, void *stream);

/*
 * Read the current device's status word (MX4_DEV_* bits, ORed by every call
 * since the last read) after synchronising `stream`, then clear it.
 */
mx4_status mx4_index_get_device_status(void *stream, uint32_t *status_out);

/* Human-readable name of a status code; never NULL. */
const char *mx4_status_string(int status);

/* MX4_ABI_VERSION of the loaded library. */
int mx4_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MX4_INDEX_H */
