// topk_kernel.cuh -- top-k page selection after the block scorer.
//
// Each query row reads at most `topk` pages of its request (ATOM #2770
// "MiniMax-M3.1 MXFP4 sparse KV cache and index cache", "How it works": the
// index scores feed the selection and the emit of a page-level block table,
// one page a block for 128-token pages, with the local and tail blocks always
// selected).  Per (row, head group):
//   value[j]  = max of the group's block scores of live page j
//   forced    = the last min(local, live) live pages
//   chosen    = the topk - forced other live pages with the largest values,
//               ties to the lower page index
//   emit      = physical ids of forced + chosen in ascending page order,
//               -1 up to topk, and the count.
//
// One CTA per (row, group) work item, grid-stride.  The values become
// order-preserving 32-bit keys in shared memory; an exact MSB-first radix
// select (4 passes of 8 bits, shared-memory histograms) finds the m-th
// largest key T and how many keys equal to T are taken; one ordered pass over
// contiguous per-thread page ranges (a block-wide exclusive scan) ranks the
// ties by page index and compacts the selected pages in ascending order.
// Reading the block scores is the bulk of the work: 4 B per (head, page).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace mx4 {

constexpr int kTopkThreads = 256;
constexpr int kTopkMaxPages = 16384;   // ceil(max_seq_len / 128) supported (2M tokens)

struct TopkParams {
    const float *scores;           // [rows, 64, P]
    const int32_t *block_table;
    const int32_t *cu_seqlens_q;   // prefill only
    const int32_t *seq_lens;
    const int32_t *prefix_lens;    // prefill only
    int32_t *sel;                  // [rows, groups, topk]
    int32_t *count;                // [rows, groups]
    int64_t bt_stride;
    int64_t num_items;             // num_seqs * rows_per_seq * groups
    int num_seqs;
    int rows_per_seq;              // max_query_len (1 for decode)
    int max_seq_len;
    int num_pages;                 // P
    int topk;
    int local;
    int groups;
    int vec;                       // scores 16-byte aligned and P % 4 == 0: float4 loads
};

// Order-preserving map of a float to a 32-bit key (larger float, larger
// key); -0 is folded into +0 so equal values have equal keys.
__device__ __forceinline__ uint32_t topk_key(float v)
{
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread (256 threads); also
// returns the total.  `buf` holds 8 ints of shared memory.
__device__ __forceinline__ int topk_block_scan(int x, int *buf, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) buf[warp] = inc;
    __syncthreads();
    int base = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
        const int t = buf[w];
        if (w < warp) base += t;
        total += t;
    }
    __syncthreads();   // buf may be reused by the caller
    return base + inc - x;
}

template <bool kDecode>
// (at least 4 resident blocks per SM: up to 64 registers a thread)
__global__ void __launch_bounds__(kTopkThreads, 4) mx4_topk_kernel(const __grid_constant__ TopkParams p)
{
    extern __shared__ uint32_t topk_smem[];
    uint32_t *keys = topk_smem;                                 // [num_pages]
    __shared__ int hist[256];
    __shared__ int scan_buf[8];
    __shared__ uint32_t sel_prefix;
    __shared__ int sel_remaining;

    const int tid = threadIdx.x;
    const int hg = 64 / p.groups;
    for (int64_t item = blockIdx.x; item < p.num_items; item += gridDim.x) {
        const int g = static_cast<int>(item % p.groups);
        const int64_t rest = item / p.groups;
        const int pos = static_cast<int>(rest % p.rows_per_seq);
        const int b = static_cast<int>(rest / p.rows_per_seq);
        int64_t row;
        int64_t L;
        if (kDecode) {
            row = b;
            L = p.seq_lens[b];
        } else {
            const int qs = p.cu_seqlens_q[b];
            if (pos >= p.cu_seqlens_q[b + 1] - qs) continue;     // uniform over the block
            row = qs + pos;
            const int64_t c = static_cast<int64_t>(p.prefix_lens[b]) + pos + 1;
            L = c < p.seq_lens[b] ? c : p.seq_lens[b];
        }
        if (L > p.max_seq_len) L = p.max_seq_len;
        if (L < 0) L = 0;
        const int nl = static_cast<int>((L + 127) / 128);                 // live pages
        const int forced = p.local < nl ? p.local : nl;
        const int nc = nl - forced;                                       // candidates
        const int want = p.topk - forced < nc ? p.topk - forced : nc;     // candidates to take

        // --- values: max over the group's heads, as keys ---
        // (a warp reads 32 consecutive pages of one head per load; the head
        // loop is unrolled so many independent loads are in flight)
        const float *src = p.scores + (row * 64 + static_cast<int64_t>(g) * hg) * p.num_pages;
        if (p.vec) {
            const int64_t hstride = p.num_pages >> 2;                // float4 per head
            const int nq = (nc + 3) >> 2;
            for (int qd = tid; qd < nq; qd += kTopkThreads) {
                const float4 *s4 = reinterpret_cast<const float4 *>(src) + qd;
                float4 m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll 16
                for (int h = 0; h < hg; ++h) {
                    const float4 x = __ldg(s4 + h * hstride);
                    m.x = fmaxf(m.x, x.x);
                    m.y = fmaxf(m.y, x.y);
                    m.z = fmaxf(m.z, x.z);
                    m.w = fmaxf(m.w, x.w);
                }
                // pages past nc (up to the quad's end, < P) get keys never read
                keys[4 * qd + 0] = topk_key(m.x);
                keys[4 * qd + 1] = topk_key(m.y);
                keys[4 * qd + 2] = topk_key(m.z);
                keys[4 * qd + 3] = topk_key(m.w);
            }
        } else {
            for (int j = tid; j < nc; j += kTopkThreads) {
                float m = -INFINITY;
#pragma unroll 16
                for (int h = 0; h < hg; ++h) m = fmaxf(m, __ldg(src + static_cast<int64_t>(h) * p.num_pages + j));
                keys[j] = topk_key(m);
            }
        }
        __syncthreads();

        // --- radix select of the want-th largest key (only when some are left out) ---
        uint32_t T = 0;
        int take_eq = 0;
        const bool all = want >= nc;
        if (!all && want > 0) {
            if (tid == 0) {
                sel_prefix = 0;
                sel_remaining = want;
            }
            uint32_t mask = 0;
            for (int shift = 24; shift >= 0; shift -= 8) {
                hist[tid] = 0;
                __syncthreads();
                const uint32_t prefix = sel_prefix;
                for (int j = tid; j < nc; j += kTopkThreads) {
                    const uint32_t k = keys[j];
                    if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFF], 1);
                }
                __syncthreads();
                if (tid < 32) {
                    // lane l holds buckets 255-8l .. 248-8l (descending)
                    int c[8], s = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        c[i] = hist[255 - 8 * tid - i];
                        s += c[i];
                    }
                    int inc = s;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, inc, o);
                        if (tid >= o) inc += y;
                    }
                    const int rem = sel_remaining;
                    const int before = inc - s;             // keys in higher buckets of earlier lanes
                    const unsigned hit = __ballot_sync(0xffffffffu, inc >= rem);
                    const int first = __ffs(hit) - 1;     // the lane whose range reaches rem
                    if (tid == first) {
                        // walk this lane's 8 buckets downwards to the one
                        // that reaches rem (unrolled: c stays in registers)
                        int acc = before, pick = 7;
                        bool found = false;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (!found && acc + c[i] >= rem) {
                                pick = i;
                                found = true;
                            } else if (!found) {
                                acc += c[i];
                            }
                        }
                        const uint32_t digit = 255u - 8u * tid - pick;
                        sel_prefix = prefix | (digit << shift);
                        sel_remaining = rem - acc;
                    }
                }
                __syncthreads();
                mask |= 0xFFu << shift;
            }
            T = sel_prefix;
            take_eq = sel_remaining;                 // keys equal to T to take, lowest pages first
        }

        // --- ordered compaction of the selected pages ---
        // thread t owns pages [t*C, (t+1)*C) of [0, nl)
        const int C = (nl + kTopkThreads - 1) / kTopkThreads;
        const int j0 = tid * C;
        const int j1 = j0 + C < nl ? j0 + C : nl;
        int n_eq = 0;
        if (!all && want > 0)
            for (int j = j0; j < j1 && j < nc; ++j) n_eq += keys[j] == T;
        int tot_eq;
        int eq_before = topk_block_scan(n_eq, scan_buf, tot_eq);
        // page j is taken when it is in the forced tail, or all candidates
        // are taken, or its key beats T, or it is one of the first take_eq
        // pages (in page order) whose key equals T
        const bool pick_some = !all && want > 0;
        int n_sel = 0;
        {
            int r = eq_before;
            for (int j = j0; j < j1; ++j) {
                bool take = j >= nc || all;
                if (!take && pick_some) {
                    const uint32_t k = keys[j];
                    take = k > T || (k == T && r < take_eq);
                    r += k == T;
                }
                n_sel += take;
            }
        }
        int tot_sel;
        int out_pos = topk_block_scan(n_sel, scan_buf, tot_sel);
        int32_t *dst = p.sel + (row * p.groups + g) * static_cast<int64_t>(p.topk);
        const int32_t *bt = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
        {
            int r = eq_before;
            for (int j = j0; j < j1; ++j) {
                bool take = j >= nc || all;
                if (!take && pick_some) {
                    const uint32_t k = keys[j];
                    take = k > T || (k == T && r < take_eq);
                    r += k == T;
                }
                if (take) dst[out_pos++] = bt[j];
            }
        }
        for (int i = tot_sel + tid; i < p.topk; i += kTopkThreads) dst[i] = -1;
        if (tid == 0) p.count[row * p.groups + g] = tot_sel;
        __syncthreads();   // keys and hist are reused by the next item
    }
}

}  // namespace mx4
