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
//               -1 up to topk, the count and (optionally) the live tokens of
//               the selected pages, the context the attention step reads.
//
// One CTA per (row, group) work item, grid-stride; or, when there are fewer
// items than two per SM, one cluster of kTopkSplit CTAs per item, each CTA
// computing the keys of a quarter of the pages (a row's score reads are then
// spread over four SMs).  With at most kTopkFastWant = 32 chosen pages of at
// most 4 x 256 candidates the select has two stages: each CTA sorts its
// (key, page) ranks one a thread in warp bitonic sorts and keeps the 32
// largest through a merge tree; rank 0 merges the four lists and takes the
// first `want`.  Otherwise the CTAs store their keys into rank 0's
// shared memory and rank 0 alone selects, as one CTA does.  The values become
// order-preserving 32-bit keys in shared memory; an exact MSB-first radix
// select (4 passes of 8 bits, shared-memory histograms fed by warp-aggregated
// atomics) finds the m-th largest key T and how many keys equal to T are
// taken; one ordered pass over contiguous per-thread page ranges (a
// block-wide exclusive scan) ranks the ties by page index and compacts the
// selected pages in ascending order.  Reading the block scores is the bulk of
// the work: 4 B per (head, page).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace mx4 {

constexpr int kTopkThreads = 256;
constexpr int kTopkSplit = 4;          // CTAs (one cluster) per item when items are few
constexpr int kTopkMaxPages = 16384;   // ceil(max_seq_len / 128) supported (2M tokens)
constexpr int kTopkFastWant = 32;      // cluster path: two-stage select up to this many chosen pages

struct TopkParams {
    const float *scores;           // [rows, 64, P]
    const int32_t *block_table;
    const int32_t *cu_seqlens_q;   // prefill only
    const int32_t *seq_lens;
    const int32_t *prefix_lens;    // prefill only
    int32_t *sel;                  // [rows, groups, topk]
    int32_t *count;                // [rows, groups]
    int32_t *tokens;               // [rows, groups] or null: live tokens of the selected pages
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

// Ranks of the two-stage select: (key << 32) | (2^32 - 1 - page), so the
// larger rank comes first in the selection order (key descending, ties to the
// lower page); 0 marks an empty slot, below every page's rank.
__device__ __forceinline__ uint64_t topk_rank(uint32_t key, int page)
{
    return (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(page));
}

// Bitonic sort of one value a lane, descending over the warp's lanes.
__device__ __forceinline__ uint64_t topk_warp_sort_desc(uint64_t x)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t y = __shfl_xor_sync(0xffffffffu, x, j);
            // the lower lane of a pair keeps the larger value in runs that
            // end descending ((lane & k) == 0; every lane in the last run)
            const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0 || k == 32);
            x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
        }
    }
    return x;
}

// The 32 largest of two descending warp lists a and b (lane i gives a[i] and
// b[31 - i], a bitonic run), descending.
__device__ __forceinline__ uint64_t topk_warp_merge_desc(uint64_t a, uint64_t b_rev)
{
    const int lane = threadIdx.x & 31;
    uint64_t x = a > b_rev ? a : b_rev;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const uint64_t y = __shfl_xor_sync(0xffffffffu, x, j);
        x = (lane & j) == 0 ? (x > y ? x : y) : (x < y ? x : y);
    }
    return x;
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

// kSplit == 1: grid-stride over items.  kSplit > 1: launched as clusters of
// kSplit CTAs, exactly one item per cluster (grid = items x kSplit).
// (at least 4 resident blocks per SM: up to 64 registers a thread)
template <bool kDecode, int kSplit>
__global__ void __launch_bounds__(kTopkThreads, 4) mx4_topk_kernel(const __grid_constant__ TopkParams p)
{
    extern __shared__ __align__(16) uint32_t topk_smem[];
    uint32_t *keys = topk_smem;                                 // [num_pages], 16-byte aligned
    __shared__ int hist[256];
    __shared__ int scan_buf[8];
    __shared__ uint32_t sel_prefix;
    __shared__ int sel_remaining;
    __shared__ int sel_done;
    // cluster path, two-stage select: the warps' sorted lists (two buffers,
    // one per merge level), and in rank 0 every rank's 32 largest
    __shared__ uint64_t run[2][kTopkThreads];
    __shared__ uint64_t cand[kTopkSplit * 32];

    const int tid = threadIdx.x;
    const int hg = 64 / p.groups;
    const uint32_t rank = kSplit > 1 ? cluster_ctarank() : 0u;
    const int64_t first = kSplit > 1 ? static_cast<int64_t>(blockIdx.x / kSplit) : static_cast<int64_t>(blockIdx.x);
    const int64_t step = kSplit > 1 ? p.num_items : static_cast<int64_t>(gridDim.x);
    for (int64_t item = first; item < p.num_items; item += step) {
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
        if (kSplit > 1) {
            // Rank r takes the r-th share of the quads (pages); four slices
            // of 64 threads split the heads, so each thread keeps all its
            // loads in flight at once, and fold their maxima into this CTA's
            // keys with atomicMax (keys start at 0, below every value's key);
            // the other ranks then copy their share into rank 0's keys.
            const int sl = tid >> 6, st = tid & 63;
            const int hper = (hg + 3) >> 2;
            const int h0 = sl * hper < hg ? sl * hper : hg;
            const int h1 = h0 + hper < hg ? h0 + hper : hg;
            const uint32_t keys0 = cluster_map(static_cast<uint32_t>(__cvta_generic_to_shared(keys)), 0);
            // few chosen pages of at most 4 x 256 candidates: the two-stage
            // select below, else rank 0 selects over all the keys
            const bool fast = want > 0 && want < nc && want <= kTopkFastWant && nc <= kTopkSplit * kTopkThreads;
            int pj0 = 0, pj1 = 0;                        // this rank's candidate pages
            // Rank 0's shared memory may be written only once every CTA of the
            // cluster is known to have started: arrive here, wait just before
            // the remote stores, so the barrier overlaps the score reads.
            cluster_arrive_relaxed();
            if (p.vec) {
                const int64_t hstride = p.num_pages >> 2;            // float4 per head
                const int nq = (nc + 3) >> 2;
                const int share = (nq + kSplit - 1) / kSplit;
                const int q0 = static_cast<int>(rank) * share < nq ? static_cast<int>(rank) * share : nq;
                const int q1 = q0 + share < nq ? q0 + share : nq;
                for (int j = 4 * q0 + tid; j < 4 * q1; j += kTopkThreads) keys[j] = 0u;   // (P % 4 == 0)
                __syncthreads();
                for (int qd = q0 + st; qd < q1; qd += 64) {
                    const float4 *s4 = reinterpret_cast<const float4 *>(src) + qd;
                    float4 m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll 16
                    for (int h = h0; h < h1; ++h) {
                        const float4 x = __ldg(s4 + h * hstride);
                        m.x = fmaxf(m.x, x.x);
                        m.y = fmaxf(m.y, x.y);
                        m.z = fmaxf(m.z, x.z);
                        m.w = fmaxf(m.w, x.w);
                    }
                    atomicMax(&keys[4 * qd + 0], topk_key(m.x));
                    atomicMax(&keys[4 * qd + 1], topk_key(m.y));
                    atomicMax(&keys[4 * qd + 2], topk_key(m.z));
                    atomicMax(&keys[4 * qd + 3], topk_key(m.w));
                }
                __syncthreads();
                pj0 = 4 * q0;
                pj1 = 4 * q1 < nc ? 4 * q1 : nc;
                if (!fast) {
                    cluster_wait();
                    if (rank != 0)
                        for (int qd = q0 + tid; qd < q1; qd += kTopkThreads)
                            st_cluster_v4_u32(keys0 + 16u * qd, keys[4 * qd], keys[4 * qd + 1], keys[4 * qd + 2],
                                              keys[4 * qd + 3]);
                }
            } else {
                const int share = (nc + kSplit - 1) / kSplit;
                const int j0 = static_cast<int>(rank) * share < nc ? static_cast<int>(rank) * share : nc;
                const int j1 = j0 + share < nc ? j0 + share : nc;
                for (int j = j0 + tid; j < j1; j += kTopkThreads) keys[j] = 0u;
                __syncthreads();
                for (int j = j0 + st; j < j1; j += 64) {
                    float m = -INFINITY;
#pragma unroll 16
                    for (int h = h0; h < h1; ++h) m = fmaxf(m, __ldg(src + static_cast<int64_t>(h) * p.num_pages + j));
                    atomicMax(&keys[j], topk_key(m));
                }
                __syncthreads();
                pj0 = j0;
                pj1 = j1;
                if (!fast) {
                    cluster_wait();
                    if (rank != 0)
                        for (int j = j0 + tid; j < j1; j += kTopkThreads) st_cluster_u32(keys0 + 4u * j, keys[j]);
                }
            }
            if (fast) {
                // Two-stage select, first stage: this rank's 32 largest
                // candidate ranks, from one a thread over its pages [pj0, pj1):
                // each warp sorts its 32, three merge levels keep the 32
                // largest of all.  Every page of the row's top want (want <=
                // 32) is among its CTA's 32 largest.
                const int lane = tid & 31, warp = tid >> 5;
                const int jt = pj0 + tid;
                uint64_t x = topk_warp_sort_desc(jt < pj1 ? topk_rank(keys[jt], jt) : 0ull);
                run[0][tid] = x;
                __syncthreads();
#pragma unroll
                for (int lv = 0, n = kTopkThreads / 64; n >= 1; ++lv, n >>= 1) {
                    if (warp < n) {
                        x = topk_warp_merge_desc(run[lv & 1][64 * warp + lane], run[lv & 1][64 * warp + 63 - lane]);
                        if (n > 1) run[(lv + 1) & 1][32 * warp + lane] = x;
                    }
                    if (n > 1) __syncthreads();
                }
                cluster_wait();
                if (warp == 0)
                    st_cluster_u64(cluster_map(static_cast<uint32_t>(__cvta_generic_to_shared(cand)), 0) +
                                       8u * (32u * rank + lane),
                                   x);
            }
            // every rank's keys (or chosen pages) have landed in rank 0
            // (release / acquire); the other ranks are done with the item
            cluster_sync();
            if (rank != 0) continue;
            if (fast) {
                // second stage (rank 0): the 32 largest of the four ranks'
                // lists; the first want of them are the chosen pages, each
                // placed by how many chosen pages lie below it
                const int lane = tid & 31, warp = tid >> 5;
                static_assert(kTopkSplit == 4, "two merge levels");
                if (warp < 2) run[0][32 * warp + lane] =
                    topk_warp_merge_desc(cand[64 * warp + lane], cand[64 * warp + 63 - lane]);
                __syncthreads();
                int32_t *dst = p.sel + (row * p.groups + g) * static_cast<int64_t>(p.topk);
                const int32_t *bt = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
                if (warp == 0) {
                    const uint64_t x = topk_warp_merge_desc(run[0][lane], run[0][63 - lane]);
                    const int pg = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(x));
                    const bool chosen = lane < want;
                    int below = 0;
#pragma unroll
                    for (int s2 = 0; s2 < 32; ++s2) {
                        const int q = __shfl_sync(0xffffffffu, pg, s2);
                        below += (s2 < want) & (q < pg);
                    }
                    if (chosen) dst[below] = bt[pg];
                    // the row's last live page (the only partial one) is
                    // taken when it is forced or chosen
                    const bool last_taken = forced > 0 || __any_sync(0xffffffffu, chosen && pg == nl - 1);
                    if (lane == 0) {
                        p.count[row * p.groups + g] = want + forced;
                        if (p.tokens) {
                            const int64_t full = 128 * static_cast<int64_t>(want + forced);
                            p.tokens[row * p.groups + g] =
                                static_cast<int32_t>(last_taken ? full - (128 * static_cast<int64_t>(nl) - L) : full);
                        }
                    }
                }
                // then the forced tail in page order, and -1 up to topk
                for (int f = tid; f < forced; f += kTopkThreads) dst[want + f] = bt[nc + f];
                for (int f = want + forced + tid; f < p.topk; f += kTopkThreads) dst[f] = -1;
                __syncthreads();   // shared state is reused by the next item
                continue;
            }
        } else {
            if (p.vec) {
                const int64_t hstride = p.num_pages >> 2;            // float4 per head
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
        }

        // --- radix select of the want-th largest key (only when some are left out) ---
        uint32_t T = 0, Tmask = 0xFFFFFFFFu;
        int take_eq = 0;
        const bool all = want >= nc;
        if (!all && want > 0) {
            if (tid == 0) {
                sel_prefix = 0;
                sel_remaining = want;
                sel_done = 0;
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
                        int acc = before, pick = 7, picked = c[7];
                        bool found = false;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (!found && acc + c[i] >= rem) {
                                pick = i;
                                picked = c[i];
                                found = true;
                            } else if (!found) {
                                acc += c[i];
                            }
                        }
                        const uint32_t digit = 255u - 8u * tid - pick;
                        sel_prefix = prefix | (digit << shift);
                        sel_remaining = rem - acc;
                        // every key of the chosen bucket is taken: the
                        // prefix alone decides, no further pass
                        sel_done = rem - acc == picked ? 1 : 0;
                    }
                }
                __syncthreads();
                mask |= 0xFFu << shift;
                if (sel_done) break;                 // (uniform: read after the barrier)
            }
            T = sel_prefix;
            Tmask = mask;
            take_eq = sel_remaining;                 // keys equal to T (under Tmask) to take, lowest pages first
        }

        // --- ordered compaction of the selected pages ---
        // thread t owns pages [t*C, (t+1)*C) of [0, nl)
        const int C = (nl + kTopkThreads - 1) / kTopkThreads;
        const int j0 = tid * C;
        const int j1 = j0 + C < nl ? j0 + C : nl;
        int n_eq = 0;
        if (!all && want > 0)
            for (int j = j0; j < j1 && j < nc; ++j) n_eq += (keys[j] & Tmask) == T;
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
                    const uint32_t k = keys[j] & Tmask;
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
        bool last_taken = false;     // the row's last live page (the only partial one) was selected
        {
            int r = eq_before;
            for (int j = j0; j < j1; ++j) {
                bool take = j >= nc || all;
                if (!take && pick_some) {
                    const uint32_t k = keys[j] & Tmask;
                    take = k > T || (k == T && r < take_eq);
                    r += k == T;
                }
                if (take) dst[out_pos++] = bt[j];
                if (j == nl - 1) last_taken = take;
            }
        }
        for (int i = tot_sel + tid; i < p.topk; i += kTopkThreads) dst[i] = -1;
        if (tid == 0) p.count[row * p.groups + g] = tot_sel;
        // every selected page is full except the last live one, which holds
        // L - 128 (nl - 1) live tokens; its owner (thread 0 when nothing is
        // live) writes the count
        if (p.tokens && (nl == 0 ? tid == 0 : (nl - 1 >= j0 && nl - 1 < j1))) {
            const int64_t full = 128 * static_cast<int64_t>(tot_sel);
            p.tokens[row * p.groups + g] =
                static_cast<int32_t>(last_taken ? full - (128 * static_cast<int64_t>(nl) - L) : full);
        }
        __syncthreads();   // keys and hist are reused by the next item
    }
}

}  // namespace mx4
