// attn_rows_kernel.cuh -- the sparse paged-attention decode of
// attn_kernel.cuh for launches in which clusters take several rows each.
//
// The same computation (ATOM #2770 "MiniMax-M3.1 MXFP4 sparse KV cache and
// index cache", commit "pa_decode MXFP4"; the arithmetic, the lazy per-head
// weight offsets, the page split over a 2-CTA cluster and the combine are
// those of attn_kernel.cuh) with the work of a CTA spread over more warps,
// so that one row's end overlaps the next row's pages:
//   warps 0-3 and 16-19  two softmax groups, the even and the odd pages of
//            each row (the PV warps' split), each with its own offsets,
//            weight sums, P^T buffers and, per row parity, accumulator;
//   warps 20-23  the epilogue: for each row, once both groups have handed
//            over their sums and offsets and the row's PV products are done,
//            it merges the groups, reads the accumulators, runs the cluster
//            combine and writes the output, while the groups go on with the
//            next row;
//   warps 4, 5, 10, 15, 6-9, 11-14  copies, QK, PV and V widening as in
//            attn_kernel.cuh.
// 768 threads; setmaxnreg gives the softmax warpgroups 104 registers, the
// copy, MMA and widening warpgroups 64, the epilogue 80.  Measured against
// the one-group kernel: faster when clusters stream several rows
// (pa-decode-4kvh 37.7 -> 35.3 us), slower for one row a cluster (pa-decode
// 11.8 -> 12.1 us), so the host picks it only when there are more rows than
// clusters.  It runs in two forms: rows split over a 2-CTA cluster as in
// attn_kernel.cuh (kSplit = 2), or whole rows on single CTAs (kSplit = 1:
// twice the units, no combine, half the row transitions a CTA; 256 rows of
// 16 pages: 32.7 -> 30.1 us); the host takes the one with fewer pages a CTA.
//
// Every barrier is waited for in each of its phases, in order, by the one
// role that waits on it, and none can complete a phase ahead of that role:
// each group's P^T buffers have their own ready and free barriers; V^T
// readiness (widening) and P^T readiness (softmax) are separate; a row's
// accumulators, sums and offsets are kept per row parity with row_ready /
// acc_free / pv_done barriers, and a group waits acc_free for the row two
// before its first P^T of a row (or at the row's end when it has no page).
#pragma once

#include "attn_kernel.cuh"

namespace mx4 {

constexpr int kArThreads = 768;
constexpr int kArKStages = 3;
constexpr int kArVStages = 3;           // (3 x 32 KB V^T and two groups' P^T leave no room for a fourth)
constexpr int kArPtBufs = 2;            // P^T operand buffers of each softmax group
// TMEM: scores as attn_kernel.cuh, then [row parity][page parity]
// accumulators, K scales, unit Q scales
constexpr uint32_t kArAccCol = kAttnSlots * kAttnN;                 // 192
constexpr uint32_t kArSfaCol = kArAccCol + 4 * kAttnN;              // 256
constexpr uint32_t kArSfbCol = kArSfaCol + 4 * kAttnSlots;          // 304
static_assert(kArSfbCol + 4 <= 512, "attention TMEM budget (rows kernel)");
static_assert(kArKStages == kArVStages, "the copy warp arms K and V stage s together");
static_assert(kAttnMaxPages <= 32, "the copy warp holds a whole row's page ids one per lane (kSplit = 1)");

struct ArSmem {
    static constexpr uint32_t kK = 0;                                    // K pages, 16 KB each
    static constexpr uint32_t kKs = kK + kArKStages * kTileBytes;      // K scales
    static constexpr uint32_t kV = kKs + kArKStages * kScaleBytes;     // V codes, natural order
    static constexpr uint32_t kVs = kV + kArVStages * kDataBytes;      // V scales
    static constexpr uint32_t kVt = ((kVs + kArVStages * kScaleBytes) + 1023) & ~1023u;   // kAttnPvBufs x 32 KB
    static constexpr uint32_t kPt = kVt + kAttnPvBufs * 32768;           // [group][2] x 4.5 KB
    static constexpr uint32_t kQ = (kPt + 2 * kArPtBufs * kPtBytes + 1023) & ~1023u;   // 2 x (16 x 128 B), by row parity
    static constexpr uint32_t kUnit = kQ + 2 * 2048;                     // 512 B of 0x7F
    static constexpr uint32_t kRed = kUnit + 512;                        // [group][2][16 heads][4 warps] warp maxima
    static constexpr uint32_t kPsum = kRed + 2 * 2 * 16 * 4 * 4;         // [row parity][group][16 heads][4 warps] sums
    static constexpr uint32_t kMo = kPsum + 2 * 2 * 16 * 4 * 4;          // [row parity][group][16 heads] offsets
    // per head: the two groups' sums and offsets, the CTA's, the groups' factors
    static constexpr uint32_t kFin = kMo + 2 * 2 * 16 * 4;
    static constexpr uint32_t kComb = kFin + 8 * 16 * 4;                 // 2 x from the peer (by row parity)
    static constexpr uint32_t kBars = kComb + 2 * (128 * 8 * 4 + 2 * 16 * 4);
    // kfull[3] kempty[3] vfull[3] vempty[3] qready[2] qfree[2] sready[12] vtready[3] pvfree[3] pv_done[2] qk_done
    // comb_ready[2] pv_fin[2] row_ready[2] acc_free[2] ptready[2][2] ptfree[2][2]
    static constexpr uint32_t kNumBars =
        2 * kArKStages + 2 * kArVStages + 4 + kAttnSlots + 2 * kAttnPvBufs + 11 + 4 * kArPtBufs;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kAlloc = kEnd + 1024;
};
static_assert(ArSmem::kAlloc <= 227 * 1024, "attention shared memory budget (rows kernel)");
static_assert(ArSmem::kComb % 16 == 0 && ArSmem::kRed % 16 == 0 && ArSmem::kPsum % 16 == 0 &&
                  ArSmem::kMo % 16 == 0 && ArSmem::kQ % 1024 == 0 && ArSmem::kBars % 8 == 0,
              "attention shared memory alignment (rows kernel)");

// Named barrier `id` over the 4 warps of a warpgroup (1 and 2: the softmax
// groups, 3: the epilogue).  A named barrier counts whole warps, so each warp reconverges first (a
// bounded wait before it may have let its lanes leave at different times).
__device__ __forceinline__ void epi_bar_sync(uint32_t id)
{
    __syncwarp();
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// The same barrier, also ANDing a predicate across the group, so that all
// four warps leave a loop at the same iteration.
__device__ __forceinline__ bool epi_bar_and(uint32_t id, bool pred)
{
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %2, 0;\n\t"
        "bar.red.and.pred q, %1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// The same barrier, ORing a predicate across the group.
__device__ __forceinline__ bool epi_bar_or(uint32_t id, bool pred)
{
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %2, 0;\n\t"
        "bar.red.or.pred q, %1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// kSplit: CTAs a row is split over (2: a cluster of 2 launched with the
// cluster attribute, the halves combined through distributed shared memory;
// 1: a CTA takes whole rows and writes their output itself).
template <int kSplit>
__global__ void __launch_bounds__(kArThreads, 1)
    mx4_attn_rows_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_ks,
                         const __grid_constant__ AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kSplit == 2 ? cluster_ctarank() : 0u;   // this CTA's half of each row's pages
    const int64_t item0 = blockIdx.x / kSplit;             // this cluster's first row (row * kv_heads + kv head)
    const int64_t nclus = gridDim.x / kSplit;              // rows item0, item0 + nclus, ...

    auto bar = [&](int i) { return sbase + ArSmem::kBars + 8u * i; };
    auto kfull = [&](int i) { return bar(i); };
    auto kempty = [&](int i) { return bar(kArKStages + i); };
    auto vfull = [&](int i) { return bar(2 * kArKStages + i); };
    auto vempty = [&](int i) { return bar(2 * kArKStages + kArVStages + i); };
    constexpr int kB0 = 2 * kArKStages + 2 * kArVStages;
    auto qready = [&](int i) { return bar(kB0 + i); };              // Q buffer i staged
    auto qfree = [&](int i) { return bar(kB0 + 2 + i); };           // Q buffer i no longer read
    auto sready = [&](int i) { return bar(kB0 + 4 + i); };          // slot i's scores are in TMEM
    auto vtready = [&](int i) { return bar(kB0 + 4 + kAttnSlots + i); };             // V^T buffer i written
    auto pvfree = [&](int i) { return bar(kB0 + 4 + kAttnSlots + kAttnPvBufs + i); };
    const uint32_t bar_rows = bar(kB0 + 4 + kAttnSlots + 2 * kAttnPvBufs);
    // per row parity, each completing once per row of its parity and
    // waited for in every phase by one role: the row's PV products done,
    // both softmax groups' sums and offsets written, the row's accumulators
    // read by the epilogue
    auto pv_done = [&](int i) { return bar_rows + 8u * i; };
    const uint32_t qk_done = bar_rows + 16;
    auto comb_ready = [&](int i) { return bar_rows + 24 + 8u * i; }; // the peer's push for a row of parity i
    auto pv_fin = [&](int i) { return bar_rows + 40 + 8u * i; };     // a PV warp's products all done
    auto row_ready = [&](int i) { return bar_rows + 56 + 8u * i; };
    auto acc_free = [&](int i) { return bar_rows + 72 + 8u * i; };
    const uint32_t pv_done0 = bar_rows;
    // P^T buffer i of softmax group x written / read by its PV warp's
    // products (each barrier is waited for in every phase, in order, by the
    // one role that waits on it, and cannot complete a phase ahead of it)
    auto ptready = [&](int x, int i) { return pv_done0 + 88 + 8u * (kArPtBufs * x + i); };
    auto ptfree = [&](int x, int i) { return pv_done0 + 88 + 8u * (2 * kArPtBufs + kArPtBufs * x + i); };
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + ArSmem::kAbort);

    if (threadIdx.x == 0) {
        // arrivals: TMA / commits count 1; the 4 warps of a softmax group
        // arrive on qready (group 0) and their ptready, the 8 widening warps
        // on vempty and vtready;
        // pv_done takes two a row: a commit from each PV warp that had pages
        // in the row, the softmax arriving for one that had none (so that
        // neither runs a phase ahead of the softmax's wait)
        for (int i = 0; i < kArKStages; ++i) {
            mbar_init(kfull(i), 1);
            mbar_init(kempty(i), 1);
        }
        for (int i = 0; i < kArVStages; ++i) {
            mbar_init(vfull(i), 1);
            mbar_init(vempty(i), kAttnWidenWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qready(i), 4);
            mbar_init(qfree(i), 1);
        }
        for (int i = 0; i < kAttnSlots; ++i) mbar_init(sready(i), 1);
        for (int i = 0; i < kAttnPvBufs; ++i) {
            mbar_init(vtready(i), kAttnWidenWarps);
            mbar_init(pvfree(i), 1);
        }
        for (int x = 0; x < 2; ++x)
            for (int i = 0; i < kArPtBufs; ++i) {
                mbar_init(ptready(x, i), 4);
                mbar_init(ptfree(x, i), 1);
            }
        mbar_init(pv_done(0), 2);
        mbar_init(pv_done(1), 2);
        mbar_init(row_ready(0), 8);
        mbar_init(row_ready(1), 8);
        mbar_init(acc_free(0), 4);
        mbar_init(acc_free(1), 4);
        mbar_init(qk_done, 1);
        mbar_init(pv_fin(0), 1);
        mbar_init(pv_fin(1), 1);
        // completed by the bytes the peer pushes (st.async complete_tx);
        // re-armed for the row after next once a push has been read
        for (int i = 0; i < 2; ++i) {
            mbar_init(comb_ready(i), 1);
            mbar_arrive_expect_tx(comb_ready(i), kCombBytes);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_ks);
    }
    if (warp == 5) {
        tmem_alloc(sbase + ArSmem::kTmemSlot, 512);
        tmem_relinquish();
    }
    // The set-up above touches no global memory, so under a programmatic
    // dependent launch it overlaps the previous kernel's tail; every global
    // access follows the wait.
    griddep_launch_dependents();
    griddep_wait();
    tc_fence_before();
    __syncthreads();
    // the peer's barriers are initialised before anyone pushes into them
    if (kSplit == 2) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<uint32_t *>(smem + ArSmem::kTmemSlot);

    // Registers: the softmax warpgroups (warps 0-3, 16-19) take 104 a
    // thread, the copy, MMA and widening warpgroups (4-15) give theirs down
    // to 64, the epilogue warpgroup (20-23) keeps the 80 the block launched
    // with: 2 x 128 x 104 + 3 x 128 x 64 + 128 x 80 = 61,440 = 768 x 80.
    // Each setmaxnreg heads the code of its warpgroups.
    if (warp < 4 || (warp >= 16 && warp < 20)) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 104;" ::: "memory");
        // ------------------------------------------------------------- softmax --
        // Group 0 (warps 0-3) takes the CTA's even pages and group 1 (warps
        // 16-19) its odd ones (the PV warps' split): each keeps its own
        // per-head offsets, weight sums and PV accumulator.  At a row's end
        // group 1 hands its sums and offsets to group 0 and goes on; group 0
        // merges the two halves and runs the cluster combine.
        const int grp = warp >= 16 ? 1 : 0;
        const uint32_t bid = 1u + static_cast<uint32_t>(grp);   // the group's named barrier
        const int m = threadIdx.x & 127;                 // TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float *mos = reinterpret_cast<float *>(smem + ArSmem::kMo);
        const int tok_m = token_of_col(m);               // token of lane m within each page
        const int G = p.groups;
        float *red = reinterpret_cast<float *>(smem + ArSmem::kRed) + grp * (2 * 16 * 4);
        float *psum = reinterpret_cast<float *>(smem + ArSmem::kPsum);
        // Q of a row (16 rows x 128 B, SW128) into buffer qb, then qready
        auto stage_q = [&](int64_t item, int qb) {
            const int h = m >> 3, c = m & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < G) v = *reinterpret_cast<const uint4 *>(p.q + ((item * G + h) << 7) + c * 16);
            *reinterpret_cast<uint4 *>(smem + ArSmem::kQ + qb * 2048 + (h >> 3) * 1024 + (h & 7) * 128 +
                                       ((c ^ (h & 7)) << 4)) = v;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready(qb));
        };
        if (grp == 0) {
            reinterpret_cast<uint32_t *>(smem + ArSmem::kUnit)[m] = 0x7F7F7F7Fu;   // before the first qready
            stage_q(item0, 0);
        }
        // scores in log2 units: x = s * softmax_scale * log2(e)
        const float sl = p.softmax_scale * 1.4426950408889634f;
        const int hl = lane & 15;
        bool ok = true;
        int g = 0;                                       // the CTA's pages so far
        int k = 0;                                       // rows done
        int nx = 0;                                      // the group's pages so far
        PageRing<kArPtBufs> prg;                       // the group's P^T buffers
        PageRing<kAttnSlots> srg;
        // (the named-barrier syncs below run on every path, so the four
        // warps of a group always pass the same number of them)
        for (int64_t item = item0; item < p.num_items; item += nclus, ++k) {
            const AttnItem it = attn_item(p, item, rank, kSplit);
            // the next row's Q, one row ahead, once QK is done with the buffer
            if (grp == 0 && item + nclus < p.num_items) {
                const int kn = k + 1;
                if (kn < 2 || __all_sync(0xffffffffu, wait_bounded(qfree(static_cast<int>(kn & 1)),
                                                                   static_cast<uint32_t>((kn >> 1) - 1) & 1u,
                                                                   abort_flag, kSiteAttnEpi)))
                    stage_q(item + nclus, static_cast<int>(kn & 1));
            }
            const int g0 = g;
            // the group's per-head weight offsets (the same in its every
            // thread) and this thread's per-head sums of its tokens' bf16
            // weights
            float mo[kAttnN], S[kAttnN];
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) {
                mo[h] = h < G ? kAttnNoOffset : kAttnMuted;
                S[h] = 0.0f;
            }
            int mine = 0;                                // the group's pages of the row so far
            const int pr = k & 1;                        // the row's accumulators, sums and offsets
            const uint32_t acc_col = kArAccCol + kAttnN * static_cast<uint32_t>(2 * pr + grp);
            // the same of the row two before must have been read by the
            // epilogue before this row's first product of the group
            // overwrites them
            bool await_free = k >= 2;
            const uint32_t free_par = static_cast<uint32_t>((k >> 1) - 1) & 1u;
            for (int j = 0; j < it.npages && ok; ++j, ++g, srg.next()) {
                if ((g & 1) != grp) continue;
                const int pb = prg.idx;
                const uint32_t slot = static_cast<uint32_t>(srg.idx);
                // the page's scores, and the group's P^T buffer back from
                // the product of its page two before
                const bool okw = __all_sync(0xffffffffu,
                                            wait2_bounded(sready(srg.idx), srg.ph, nx >= kArPtBufs, ptfree(grp, pb),
                                                          prg.ph ^ 1u, abort_flag, kSiteAttnEpi));
                const bool valid = (it.pbase + j) * kPage + tok_m < it.ctx;
                // (a page past whose end the context stops has invalid tokens)
                const bool full = (it.pbase + j + 1) * kPage <= it.ctx;
                const uint32_t s_addr = tmem_base + lane_addr + kAttnSCol + kAttnN * slot;
                // y = score in log2 units minus the head's offset (-inf for an
                // invalid token): one fma a score
                float y[16];
                bool need = false;
                if (okw) {
                    tc_fence_after();
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(s_addr, v);
#pragma unroll
                    for (int h = 0; h < kAttnN; ++h) y[h] = fmaf(__uint_as_float(v[h]), sl, -mo[h]);
                    if (!full) {
#pragma unroll
                        for (int h = 0; h < kAttnN; ++h) y[h] = valid ? y[h] : -INFINITY;
                    }
                    float ym[8];
#pragma unroll
                    for (int h = 0; h < 8; ++h) ym[h] = fmaxf(y[2 * h], y[2 * h + 1]);
#pragma unroll
                    for (int h = 0; h < 4; ++h) ym[h] = fmaxf(ym[2 * h], ym[2 * h + 1]);
                    need = fmaxf(fmaxf(ym[0], ym[1]), fmaxf(ym[2], ym[3])) > kAttnOffsetSlack;
                }
                // One barrier a page: the four warps leave together after a
                // failed wait, and raise the offsets together when a score
                // passed its head's offset by more than the slack (always on
                // the group's first page of a row).
                if (epi_bar_or(bid, need || !okw)) {
                    // the scores themselves again, into y (y lost them
                    // against the old offsets)
                    if (okw) {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(s_addr, v);
#pragma unroll
                        for (int h = 0; h < kAttnN; ++h) y[h] = valid ? __uint_as_float(v[h]) * sl : -INFINITY;
                    }
                    // the warp's max of each head (lanes 2 h, 2 h + 1 hold head h)
                    const float wm = okw ? warp_max16(y, lane) : 0.0f;
                    if ((lane & 1) == 0) red[((j & 1) * 16 + (lane >> 1)) * 4 + (warp & 3)] = wm;
                    ok = epi_bar_and(bid, okw);
                    if (!ok) break;
                    // the page's max of head hl over the four warps; each
                    // head's offset becomes the larger of it and the old one,
                    // and what was summed against the old offset is rescaled
                    const float4 r4 = reinterpret_cast<const float4 *>(red)[(j & 1) * 16 + hl];
                    const float mh = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
                    float f[kAttnN];
#pragma unroll
                    for (int h = 0; h < kAttnN; ++h) {
                        const float mn = fmaxf(mo[h], __shfl_sync(0xffffffffu, mh, h));
                        f[h] = ex2_approx(mo[h] - mn);
                        mo[h] = mn;
                        S[h] *= f[h];
                    }
                    if (mine > 0) {
                        // the group's accumulator, once the product of its
                        // previous page (in the other P^T buffer) has
                        // completed; the next one is issued only after this
                        // page's P^T, below
                        const bool okp = __all_sync(
                            0xffffffffu, wait_bounded(ptfree(grp, pb ^ 1), pb ? prg.ph : prg.ph ^ 1u, abort_flag,
                                                      kSiteAttnEpi));
                        ok = epi_bar_and(bid, okp);
                        if (!ok) break;
                        tc_fence_after();
                        uint32_t a[16];
                        tmem_ld_32x32b_x16(tmem_base + lane_addr + acc_col, a);
#pragma unroll
                        for (int h = 0; h < kAttnN; ++h) a[h] = __float_as_uint(__uint_as_float(a[h]) * f[h]);
                        tmem_st_32x32b_x16(tmem_base + lane_addr + acc_col, a);
                        tc_fence_before();
                    }
                    // y against the new offsets (-inf stays -inf)
#pragma unroll
                    for (int h = 0; h < kAttnN; ++h) y[h] -= mo[h];
                }
                // the weights 2^y (0 for an invalid token and for a head past
                // `groups`): their sums in fp32, the operand in bf16
                uint32_t w[8];
#pragma unroll
                for (int h2 = 0; h2 < 8; ++h2) {
                    const float p0 = ex2_approx(y[2 * h2]), p1 = ex2_approx(y[2 * h2 + 1]);
                    S[2 * h2] += p0;
                    S[2 * h2 + 1] += p1;
                    const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                    w[h2] = *reinterpret_cast<const uint32_t *>(&pb);
                }
                uint8_t *pt = smem + ArSmem::kPt + (kArPtBufs * grp + pb) * kPtBytes + pt_offset(tok_m);
                *reinterpret_cast<uint4 *>(pt) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(pt + kPtSbo) = make_uint4(w[4], w[5], w[6], w[7]);
                // P^T visible to the tensor core
                fence_proxy_async_smem();
                if (await_free) {
                    // (a wait that runs out leaves only this row's output
                    // wrong: the status word reports it)
                    (void)__all_sync(0xffffffffu, wait_bounded(acc_free(pr), free_par, abort_flag, kSiteAttnEpi));
                    await_free = false;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ptready(grp, pb));
                ++mine;
                ++nx;
                prg.next();
            }
            // The group's per-head weight sums (each warp's) and offsets, for
            // the epilogue, which finishes the row while the groups go on
            // with the next one.
            const float wsum = warp_sum16(S, lane);          // lanes 2 h, 2 h + 1 hold head h
            if (await_free)      // (no page of this group in the row)
                (void)__all_sync(0xffffffffu, wait_bounded(acc_free(pr), free_par, abort_flag, kSiteAttnEpi));
            if ((lane & 1) == 0) psum[((pr * 2 + grp) * 16 + (lane >> 1)) * 4 + (warp & 3)] = ok ? wsum : 0.0f;
            if ((warp & 3) == 0 && lane < kAttnN) {
                float om = 0.0f;
#pragma unroll
                for (int h = 0; h < kAttnN; ++h) om = lane == h ? mo[h] : om;
                mos[(pr * 2 + grp) * 16 + lane] = om;
            }
            // the row's PV products: a PV warp without pages in the row does
            // not commit, the softmax group of its parity arrives in its
            // place (every row's phase is waited for, so the parities stay
            // in step)
            const bool has_pages = it.npages >= 2 || (it.npages == 1 && (g0 & 1) == grp);
            if (m == 0 && !has_pages) mbar_arrive(pv_done(pr));
            __syncwarp();
            if (lane == 0) mbar_arrive(row_ready(pr));
        }
    } else if (warp >= 20) {
        // ------------------------------------------------------------ epilogue --
        // Warps 20-23 finish each row while the softmax groups go on with
        // the next: the two groups' per-head sums and offsets merged, their
        // accumulators once the row's PV products are done, the cluster
        // combine and the output.  Thread m reads TMEM lane m (head dim m).
        const int m = threadIdx.x - 640;
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int G = p.groups;
        const float *psum = reinterpret_cast<const float *>(smem + ArSmem::kPsum);
        const float *mos = reinterpret_cast<const float *>(smem + ArSmem::kMo);
        // per head h: [h] / [16 + h] the even group's sum / offset, [32 + h] /
        // [48 + h] the odd group's, [64 + h] / [80 + h] the CTA's, [96 + h] /
        // [112 + h] the groups' factors
        float *fin = reinterpret_cast<float *>(smem + ArSmem::kFin);
        int64_t g = 0;
        int64_t k = 0;
        for (int64_t item = item0; item < p.num_items; item += nclus, ++k) {
            const AttnItem it = attn_item(p, item, rank, kSplit);
            const int pr = static_cast<int>(k & 1);
            const uint32_t par = static_cast<uint32_t>(k >> 1) & 1u;
            const int64_t g0 = g;
            g += it.npages;
            // (made the group's, so that all four warps take the same path)
            const bool okw = __all_sync(0xffffffffu, wait_bounded(row_ready(pr), par, abort_flag, kSiteAttnEpi)) &&
                             __all_sync(0xffffffffu, wait_bounded(pv_done(pr), par, abort_flag, kSiteAttnEpi));
            const bool ok = epi_bar_and(3u, okw);
            if (m < kAttnN) {
                // per head: the CTA's offset (the larger of the groups' with
                // weight), the groups' factors and the CTA's weight sum
                const float4 a4 = reinterpret_cast<const float4 *>(psum)[(pr * 2 + 0) * 16 + m];
                const float4 b4 = reinterpret_cast<const float4 *>(psum)[(pr * 2 + 1) * 16 + m];
                const float s0 = ok ? (a4.x + a4.y) + (a4.z + a4.w) : 0.0f, o0 = mos[(pr * 2 + 0) * 16 + m];
                const float s1 = ok ? (b4.x + b4.y) + (b4.z + b4.w) : 0.0f, o1 = mos[(pr * 2 + 1) * 16 + m];
                const float M = s0 > 0.0f ? (s1 > 0.0f && o1 > o0 ? o1 : o0) : o1;
                const float f0 = s0 > 0.0f ? ex2_approx(o0 - M) : 0.0f;
                const float f1 = s1 > 0.0f ? ex2_approx(o1 - M) : 0.0f;
                fin[64 + m] = s0 * f0 + s1 * f1;
                fin[80 + m] = M;
                fin[96 + m] = f0;
                fin[112 + m] = f1;
            }
            epi_bar_sync(3u);
            // lane m of the accumulators holds head dim m of every head: the
            // even pages' and the odd pages' products (each only if the row
            // had such a page)
            float acc[kAttnN];
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) acc[h] = 0.0f;
            if (ok && it.npages > 0) {
                tc_fence_after();
                uint32_t a[2][16];
                const uint32_t acc_row = tmem_base + lane_addr + kArAccCol + 2u * kAttnN * static_cast<uint32_t>(pr);
                tmem_ld2_32x32b_x16(acc_row, acc_row + kAttnN, a[0], a[1]);
                const bool use_even = it.npages >= 2 || (g0 & 1) == 0;
                const bool use_odd = it.npages >= 2 || (g0 & 1) == 1;
#pragma unroll
                for (int h = 0; h < kAttnN; ++h)
                    acc[h] = (use_even ? __uint_as_float(a[0][h]) * fin[96 + h] : 0.0f) +
                             (use_odd ? __uint_as_float(a[1][h]) * fin[112 + h] : 0.0f);
            }
            // the row's sums, offsets and accumulators are read: the softmax
            // groups may reuse them for the row after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free(pr));
            // Combine the two halves: rank r finalises heads 8r .. 8r+7.
            // Each CTA pushes the peer's heads of its accumulator ([dim][8
            // heads]) and its 16 sums and offsets into the peer's buffer of
            // this row's parity with st.async, whose bytes complete the
            // peer's comb_ready; it then waits for its own, rescales both
            // halves to the larger offset, adds, normalises and stores bf16
            // (a half with no weight contributes nothing).
            if (kSplit == 1) {
                // a whole row: this CTA's sums and accumulators are the row's
                __nv_bfloat16 *o = p.out + (item * G) * kDim;
#pragma unroll
                for (int h = 0; h < kAttnN; ++h) {
                    const float sum = fin[64 + h];
                    if (ok && h < G) o[h * kDim + m] = __float2bfloat16_rn(sum > 0.0f ? __fdividef(acc[h], sum) : 0.0f);
                }
                epi_bar_sync(3u);        // fin is rewritten for the next row
            } else {
                const int cb = static_cast<int>(k & 1);
                const uint32_t peer = rank ^ 1u;
                const uint32_t pc = cluster_map(sbase + ArSmem::kComb + cb * kCombBytes, peer);
                const uint32_t pbar = cluster_map(comb_ready(cb), peer);
                float a8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) a8[i] = peer ? acc[8 + i] : acc[i];
                st_async_v4_u32(pc + 32u * m, __float_as_uint(a8[0]), __float_as_uint(a8[1]),
                                __float_as_uint(a8[2]), __float_as_uint(a8[3]), pbar);
                st_async_v4_u32(pc + 32u * m + 16u, __float_as_uint(a8[4]), __float_as_uint(a8[5]),
                                __float_as_uint(a8[6]), __float_as_uint(a8[7]), pbar);
                if (m < 2 * kAttnN) st_async_u32(pc + 4096u + 4u * m, __float_as_uint(fin[64 + m]), pbar);
                const bool comb_ok = __all_sync(0xffffffffu, wait_bounded(comb_ready(cb), static_cast<uint32_t>(k >> 1) & 1u,
                                                                         abort_flag, kSiteAttnEpi));
                if (comb_ok) {
                    const float *cm = reinterpret_cast<const float *>(smem + ArSmem::kComb + cb * kCombBytes);
                    const float4 c0 = reinterpret_cast<const float4 *>(cm)[2 * m];
                    const float4 c1 = reinterpret_cast<const float4 *>(cm)[2 * m + 1];
                    const float a1[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    __nv_bfloat16 *o = p.out + (item * G) * kDim;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int h = 8 * static_cast<int>(rank) + i;
                        // this thread's own values of head h (static register indexes)
                        const float a0 = rank ? acc[8 + i] : acc[i];
                        const float s0 = fin[64 + h], m0 = fin[80 + h];
                        const float s1 = cm[1024 + h], m1 = cm[1024 + kAttnN + h];
                        const float mx = s1 > 0.0f && m1 > m0 ? m1 : m0;
                        const float f0 = s0 > 0.0f ? ex2_approx(m0 - mx) : 0.0f;
                        const float f1 = s1 > 0.0f ? ex2_approx(m1 - mx) : 0.0f;
                        const float av = a0 * f0 + a1[i] * f1, sum = s0 * f0 + s1 * f1;
                        if (h < G) o[h * kDim + m] = __float2bfloat16_rn(sum > 0.0f ? __fdividef(av, sum) : 0.0f);
                    }
                }
                // every thread has read this buffer and fin: the buffer's
                // barrier is re-armed for the row after next (only once its
                // phase has completed; after a wait that ran out the CTA is
                // aborting and every later wait gives up at once)
                epi_bar_sync(3u);
                if (m == 0 && comb_ok) mbar_arrive_expect_tx(comb_ready(cb), kCombBytes);
            }
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
        if (warp == 4) {
            // ------------------------------------------------------------ copies --
            // K page g once QK of page g - 4 is done, V page g once the widening
            // of page g - 4 is done; they run ahead into the next rows.  Lane j
            // holds the row's j-th page id, and the next row's context and ids
            // are loaded while this row's pages stream.
            const uint64_t policy = l2_policy_evict_first();
            int64_t g = 0;
            bool ok = true;
            auto load_ids = [&](int64_t item, const AttnItem &it) {
                int32_t id = 0;
                if (lane < it.npages) {
                    const int64_t raw = p.block_table[item * p.width + it.pbase + lane];
                    if (raw < 0 || raw >= p.num_pool_pages)
                        atomicOr(&g_mx4_device_status, 0x1u);
                    else
                        id = static_cast<int32_t>(raw);
                }
                return id;
            };
            AttnItem it = attn_item(p, item0, rank, kSplit);
            int32_t id = load_ids(item0, it);
            PageRing<kArKStages> krg;
            for (int64_t item = item0; item < p.num_items && ok; item += nclus) {
                AttnItem nit{};
                int32_t nid = 0;
                bool fetched = false;
                auto fetch_next = [&]() {
                    if (!fetched && item + nclus < p.num_items) {
                        nit = attn_item(p, item + nclus, rank, kSplit);
                        nid = load_ids(item + nclus, nit);
                    }
                    fetched = true;
                };
                for (int j = 0; j < it.npages; ++j) {
                    const int s = krg.idx;
                    if (!(ok = __all_sync(0xffffffffu, wait2_bounded(kempty(s), krg.ph ^ 1u, true, vempty(s), krg.ph ^ 1u,
                                                                     abort_flag, kSiteAttnProducer))))
                        break;
                    const int64_t pg = __shfl_sync(0xffffffffu, id, j);
                    if (elect_one()) {
                        mbar_arrive_expect_tx(kfull(s), kDataBytes + kScaleBytes);
                        tma_load_5d(sbase + ArSmem::kK + s * kTileBytes, &tmap_k, kfull(s), 0, 0, 0, it.kvh,
                                    static_cast<int>(pg), policy);
                        tma_load_3d(sbase + ArSmem::kKs + s * kScaleBytes, &tmap_ks, kfull(s), 0, it.kvh,
                                    static_cast<int>(pg), policy);
                        mbar_arrive_expect_tx(vfull(s), kDataBytes + kScaleBytes);
                        bulk_load(sbase + ArSmem::kV + s * kDataBytes, p.v_data + pg * p.vd_ps + it.kvh * p.vd_hs,
                                  kDataBytes, vfull(s), policy);
                        bulk_load(sbase + ArSmem::kVs + s * kScaleBytes, p.v_scale + pg * p.vs_ps + it.kvh * p.vs_hs,
                                  kScaleBytes, vfull(s), policy);
                    }
                    __syncwarp();
                    ++g;
                    krg.next();
                    // the next row's context and ids once the first stages are
                    // issued (the warp waits for stages after that anyway)
                    if (j == kArKStages - 1) fetch_next();
                }
                fetch_next();
                it = nit;
                id = nid;
            }
            // no copy may be in flight when the CTA exits: the last use of each
            // stage this warp armed completes (bounded)
            if (lane == 0) {
                const int64_t n = g < kArKStages ? g : kArKStages;
                for (int64_t i = 0; i < n; ++i) {
                    const int64_t gg = g - 1 - i;
                    const uint32_t ph = static_cast<uint32_t>(gg / kArKStages) & 1u;
                    if (!drain_bounded(kfull(static_cast<int>(gg % kArKStages)), ph)) break;
                    if (!drain_bounded(vfull(static_cast<int>(gg % kArKStages)), ph)) break;
                }
            }
            __syncwarp();
        } else if (warp == 5 || warp == 10 || warp == 15) {
            // ----------------------------------------------------------------- MMA --
            // Separate issuing warps, so that neither kind of product waits
            // behind the other: warp 5 issues the QK products as the K pages
            // land, warps 15 and 10 the PV products of the even and odd pages as
            // V^T and P^T are written.  Each waits for its own products to
            // complete before the CTA frees TMEM.
            if (lane == 0) {
                bool ok = true;
                int64_t g = 0;
                int64_t k = 0;                                 // rows done
                uint32_t done_b = qk_done;
                if (warp == 5) {
                    const uint32_t sfb = tmem_base + kArSfbCol;
                    PageRing<kArKStages> krg;
                    PageRing<kAttnSlots> srg;
                    for (int64_t item = item0; item < p.num_items && ok; item += nclus, ++k) {
                        const AttnItem it = attn_item(p, item, rank, kSplit);
                        const int qb = static_cast<int>(k & 1);
                        if (!(ok = wait_bounded(qready(qb), static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                                kSiteAttnMma)))
                            break;
                        tc_fence_after();
                        if (k == 0) tc_cp_32x128b_warpx4(sfb, smem_desc(sbase + ArSmem::kUnit, 16, 128, 0));
                        const uint64_t qdesc = smem_desc(sbase + ArSmem::kQ + qb * 2048u, 16, 1024, 2);
                        for (int j = 0; j < it.npages; ++j, ++g, krg.next(), srg.next()) {
                            const int s = krg.idx;
                            const uint32_t slot = static_cast<uint32_t>(srg.idx);
                            if (!(ok = wait_bounded(kfull(s), krg.ph, abort_flag, kSiteAttnMma))) break;
                            tc_fence_after();
                            const uint32_t sfa = tmem_base + kArSfaCol + 4u * slot;
                            tc_cp_32x128b_warpx4(sfa, smem_desc(sbase + ArSmem::kKs + s * kScaleBytes, 16, 128, 0));
                            const uint64_t kdesc = smem_desc(sbase + ArSmem::kK + s * kTileBytes, 16, 1024, 2);
                            const uint32_t d = tmem_base + kAttnSCol + kAttnN * slot;
#pragma unroll
                            for (uint32_t kb = 0; kb < 4; ++kb)
                                tc_mma_mx_ss(d, kdesc + 2 * kb, qdesc + 2 * kb, attn_idesc_qk(kb), sfa, sfb,
                                             kb > 0 ? 1u : 0u);
                            tc_commit(kempty(s));
                            tc_commit(sready(slot));
                        }
                        tc_commit(qfree(qb));
                    }
                } else {
                    // page g waits here only after page g - 2 was ready, hence
                    // page g - 3 (the previous phase of its buffer's barrier) too
                    const int64_t mine = warp == 15 ? 0 : 1;
                    done_b = pv_fin(static_cast<int>(mine));
                    PageRing<kAttnPvBufs> brg;
                    PageRing<kArPtBufs> prg;
                    for (int64_t item = item0; item < p.num_items && ok; item += nclus, ++k) {
                        const AttnItem it = attn_item(p, item, rank, kSplit);
                        int issued = 0;
                        const uint32_t d = tmem_base + kArAccCol + kAttnN * static_cast<uint32_t>(2 * (k & 1) + mine);
                        for (int j = 0; j < it.npages; ++j, ++g, brg.next()) {
                            if ((g & 1) != mine) continue;
                            // the row's first product overwrites the accumulator
                            const uint32_t acc_in = issued > 0 ? 1u : 0u;
                            ++issued;
                            const int b = brg.idx;
                            const int pb = prg.idx;
                            if (!(ok = wait_bounded(vtready(b), brg.ph, abort_flag, kSiteAttnMma) &&
                                       wait_bounded(ptready(static_cast<int>(mine), pb), prg.ph, abort_flag,
                                                    kSiteAttnMma)))
                                break;
                            tc_fence_after();
                            const uint32_t vt = sbase + ArSmem::kVt + b * 32768u;
                            const uint32_t pt = sbase + ArSmem::kPt + (kArPtBufs * static_cast<uint32_t>(mine) +
                                                                         static_cast<uint32_t>(pb)) * kPtBytes;
#pragma unroll
                            for (uint32_t ks = 0; ks < 8; ++ks) {
                                // K step of 16 tokens: two 8-token groups of each operand
                                const uint64_t a = smem_desc(vt + ks * 4096u, 2048, 128, 0);
                                const uint64_t bd = smem_desc(pt + ks * (2 * kPtLbo), kPtLbo, kPtSbo, 0);
                                tc_mma_f16_ss(d, a, bd, kAttnIdescPv, ks > 0 ? 1u : acc_in);
                            }
                            tc_commit(pvfree(b));
                            tc_commit(ptfree(static_cast<int>(mine), pb));
                            prg.next();
                        }
                        if (ok && issued > 0) tc_commit(pv_done(static_cast<int>(k & 1)));   // the row's PV products done
                    }
                }
                // every product issued above completes before TMEM is read or
                // freed (a barrier of this warp's own, waited for here only)
                tc_commit(done_b);
                const uint64_t t1 = globaltimer_ns();
                while (!mbar_try_wait(done_b, 0) && globaltimer_ns() - t1 < kWaitLimitNs) {
                }
            }
            __syncwarp();
        } else if (warp >= 6 && warp < 16) {
            // ---------------------------------------------------------- V widening --
            // warps 6-9 and 11-14 (warps 10 and 15 are PV issuers)
            int64_t g = 0;
            bool ok = true;
            PageRing<kAttnPvBufs> brg;
            PageRing<kArVStages> krg;
            for (int64_t item = item0; item < p.num_items && ok; item += nclus) {
                const AttnItem it = attn_item(p, item, rank, kSplit);
                for (int j = 0; j < it.npages; ++j, ++g, brg.next(), krg.next()) {
                    const int b = brg.idx, vs = krg.idx;
                    // (a buffer's first use waits for no PV product)
                    if (!(ok = __all_sync(0xffffffffu, wait2_bounded(vfull(vs), krg.ph, g >= kAttnPvBufs, pvfree(b),
                                                                     brg.ph ^ 1u, abort_flag, kSiteAttnEpi))))
                        break;
                    attn_widen(smem + ArSmem::kV + vs * kDataBytes, smem + ArSmem::kVs + vs * kScaleBytes,
                               smem + ArSmem::kVt + b * 32768, warp < 10 ? warp - 6 : warp - 7, lane,
                               it.ctx - (it.pbase + j) * kPage);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(vtready(b));
                        mbar_arrive(vempty(vs));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
    // neither CTA leaves while the other may still write into its shared memory
    if (kSplit == 2) cluster_sync();
}

}  // namespace mx4
