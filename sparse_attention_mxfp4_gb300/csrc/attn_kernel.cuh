// attn_kernel.cuh -- sparse paged-attention decode over MXFP4 K and V.
//
// Each row (a decode token and one KV head) attends over the pages it
// selected (ATOM #2770 "MiniMax-M3.1 MXFP4 sparse KV cache and index cache",
// commit "pa_decode MXFP4": K and V are e2m1 data plus one e8m0 byte per 32
// elements along head_dim; the e4m3 query is used as stored; QK is a mixed
// fp4 x fp8 block-scaled product; V is widened to bf16 exactly and P stays
// bf16; invalid tokens get a -inf score and a zero V, so tail garbage cannot
// leak):
//     s[t] = softmax_scale * sum_d q[h,d] K[t,d],  out[h,:] = softmax(s) V.
//
// One 2-CTA cluster per row, 512 threads a CTA, each CTA taking half of the
// row's pages with its own softmax max; at the end each CTA finalises 8 of
// the 16 heads, reading the peer's partial output, weight sums and maxima
// from the peer's shared memory (rescaled to the row's max, added,
// normalised); per CTA:
//   warp 4   K copies: per page, the K codes (4-D token-permuting TMA view
//            plus a KV-head dimension, the scorer's smem form) and K scales.
//   warp 10  V copies: the V codes and scales as two plain bulk copies per
//            page (natural token order: V is not an MMA operand in MXFP4
//            form), from the start, four pages deep.
//   warp 5   MMA: QK per page with tcgen05.mma kind::mxf8f6f4 block_scale,
//            A = the K page (M = 128 tokens, e2m1, its e8m0 scales copied to a
//            per-page TMEM slot), B = the Q tile (N = 16 heads, e4m3, unit
//            scales), D = the page's 16 score columns in TMEM (all pages kept).
//            Then PV per page with kind::f16: A = V^T (M = 128 head dims,
//            K = 128 token positions, bf16), B = P^T (N = 16 heads, bf16,
//            MN-major), D = the output accumulator (16 columns), accumulated
//            over pages.
//   warps 0-3 softmax: thread m reads TMEM lane m (token 4(m%32)+m/32 of each
//            page) as each page's QK product completes, takes the per-head
//            max over valid tokens (shuffles across lanes, shared memory
//            across warps), then per page writes P^T (bf16, at the thread's
//            token position: two 16-byte stores) for the PV MMA and sums the
//            bf16 P; finally the combine above and out = acc / sum (bf16).
//   warps 6-9, 11-14 widen each page's V into V^T (bf16) in the same
//            token-position order, one (position pair, 32-dim scale group)
//            cell a thread.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "score_kernel.cuh"

namespace mx4 {

// warps 0-3 softmax (P^T), 4 K copies, 5 MMA, 6-9 and 11-14 V widening,
// 10 V copies, 15 idle (the block is 16 warps so that 4 sit on each SM
// sub-partition: 128 registers a thread)
constexpr int kAttnThreads = 512;
constexpr int kAttnWidenWarps = 8;
constexpr int kAttnMaxPages = 24;       // pages a row may list
constexpr int kAttnSplit = 2;           // CTAs (one cluster) per row: each takes half of the row's pages
constexpr int kAttnCtaPages = (kAttnMaxPages + kAttnSplit - 1) / kAttnSplit;   // scores kept in TMEM
constexpr int kAttnN = 16;              // query heads per KV head (fewer are zero-padded)
constexpr int kAttnKStages = 4;
constexpr int kAttnVStages = 4;        // V pages load from the start, alongside the K pages
constexpr int kAttnPvBufs = 3;         // V^T / P^T operand buffers: widening runs up to 3 pages ahead of PV
constexpr uint32_t kAttnSCol = 0;                                    // page j: 16 columns at 16 j
constexpr uint32_t kAttnOutCol = kAttnCtaPages * kAttnN;              // 192
constexpr uint32_t kAttnSfaCol = kAttnOutCol + kAttnN;                // 208: 4 per page
constexpr uint32_t kAttnSfbCol = kAttnSfaCol + 4 * kAttnCtaPages;     // 256
static_assert(kAttnSfbCol + 4 <= 512, "attention TMEM budget");

enum AttnSite : uint32_t { kSiteAttnProducer = 6, kSiteAttnMma = 7, kSiteAttnEpi = 8 };

struct AttnParams {
    const uint8_t *q;                 // e4m3 [rows, kv_heads, groups, 128]
    const uint8_t *v_data;
    const uint8_t *v_scale;
    int64_t vd_ps, vd_hs, vs_ps, vs_hs;
    const int32_t *block_table;       // [rows, kv_heads, width]
    const int32_t *context_lens;      // [rows, kv_heads]
    __nv_bfloat16 *out;               // [rows, kv_heads, groups, 128]
    int64_t num_pool_pages;
    int kv_heads;
    int groups;
    int width;
    float softmax_scale;
};

struct AttnSmem {
    static constexpr uint32_t kK = 0;                                    // K pages, 16 KB each
    static constexpr uint32_t kKs = kK + kAttnKStages * kTileBytes;      // K scales
    static constexpr uint32_t kV = kKs + kAttnKStages * kScaleBytes;     // V codes, natural order
    static constexpr uint32_t kVs = kV + kAttnVStages * kDataBytes;      // V scales
    static constexpr uint32_t kVt = ((kVs + kAttnVStages * kScaleBytes) + 1023) & ~1023u;   // 3 x 32 KB
    static constexpr uint32_t kPt = kVt + kAttnPvBufs * 32768;           // 3 x 4 KB
    static constexpr uint32_t kQ = kPt + kAttnPvBufs * 4096;             // 16 x 128 B
    static constexpr uint32_t kUnit = kQ + 2048;                         // 512 B of 0x7F
    static constexpr uint32_t kRed = kUnit + 512;                        // 4 warps x 16 floats
    static constexpr uint32_t kComb = kRed + 4 * 16 * 4;                 // the peer's 8 heads x 128 (staged)
    static constexpr uint32_t kCombS = kComb + 128 * 8 * 4;              // this CTA's 16 sums, then 16 maxima
    static constexpr uint32_t kBars = kCombS + 2 * 16 * 4;
    // kfull[4] kempty[4] vfull[4] vempty[4] qready sready[12] pvready[3] pvfree[3] pv_done comb_ready
    static constexpr uint32_t kNumBars = 2 * kAttnKStages + 2 * kAttnVStages + 1 + kAttnCtaPages + 2 * kAttnPvBufs + 2;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kPid = kAbort + 4;                         // page ids of the row
    static constexpr uint32_t kEnd = kPid + 4 * kAttnMaxPages;
    static constexpr uint32_t kAlloc = kEnd + 1024;
};
static_assert(AttnSmem::kAlloc <= 227 * 1024, "attention shared memory budget");

// Instruction descriptors.  QK (kind::mxf8f6f4): A = E2M1 (5, bits 7..9),
// B = E4M3 (0, bits 10..12), N = 16, M = 128, UE8M0 scales (bit 23), scale
// ids of K block k in bits 4..5 (B) and 29..30 (A).  PV (kind::f16): F32
// accumulator (1, bits 4..5), A = B = BF16 (1), A K-major, B MN-major (bit
// 16), N = 16, M = 128.
__device__ __forceinline__ uint32_t attn_idesc_qk(uint32_t k)
{
    constexpr uint32_t kBase = (5u << 7) | (0u << 10) | ((16u >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
    return kBase | (k << 4) | (k << 29);
}
constexpr uint32_t kAttnIdescPv =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// P^T as an MN-major operand without swizzling: for token position k and
// head h, byte 256 (k / 8) + 128 (h / 8) + 16 (k % 8) + 2 (h % 8).  Each
// 8 x 8 core matrix (8 positions x 8 heads, 16 bytes a position) is 128
// contiguous bytes; the two head halves of a group of 8 positions follow each
// other (stride 128 B along N) and groups follow every 256 B (along K).  One
// MMA (K = 16) takes two groups.
__device__ __forceinline__ uint32_t pt_offset(int k) { return 256u * (k >> 3) + 16u * (k & 7); }

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// prmt.b32 in its default mode: result byte i is byte (sel >> 4i) & 7 of
// {b, a} (a = bytes 0..3), or that byte's sign bit replicated when bit 3 of
// the selector nibble is set.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Bounded spin on a barrier that the peer CTA completes remotely (cluster-
// scope acquire, non-blocking tests); on timeout it records the site and
// aborts like wait_bounded.
__device__ __forceinline__ bool wait_cluster_bounded(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                                     uint32_t site)
{
    const bool stall = stalled_here(site);
    if (!stall && mbar_test_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (!stall && mbar_test_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_mx4_device_status, 0x2u | (0x100u << site));
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// Widen one eighth of a V page (natural layout in smem: 64 code bytes and 4
// scale bytes per token) into the bf16 V^T operand tile, whose K positions
// follow the token order of the QK product (position m holds token
// 4(m%32) + m/32).  The 256 threads of the 8 widening warps each take one
// (position pair, 32-dim scale group) cell: lane l = 8q + 4s + qd of warp
// slot wi takes group qd and the pair
// pr = 32 (wi % 2) + (q + 16 s + 4 qd + 4 (wi / 2)) mod 32 (positions 2 pr,
// 2 pr + 1 = tokens ta, ta + 4), so that (checked exhaustively on the CPU)
//   - each 16-byte code load of a quarter-warp touches 8 distinct 16-byte
//     bank groups,
//   - at every store the 32 lanes write 32 distinct banks.
// Conversion without a table: an e2m1 code s|E|m (E two bits) placed as
// bf16 bits (E m) << 6 | s << 15 is the bf16 number 2^-126 times its value
// (a subnormal for E = 0, exact), so one packed multiply by 2^(b-1) (bf16
// bits (b + 126) << 7; b = the token's e8m0 byte) gives the scaled value;
// when some lane has b > 128 that factor overflows bf16, and the warp
// multiplies by 2^126 and 2^(b-127) instead.  Tokens at or past `valid` get
// a zero factor.  Each pair lands in one 4-byte store (adjacent K positions
// of one V^T row).
__device__ __forceinline__ void attn_widen(const uint8_t *vc, const uint8_t *vsc, uint8_t *vt, int wi, int lane,
                                           int valid)
{
    const int qd = lane & 3;
    const int pr = 32 * (wi & 1) + (((lane >> 3) + 16 * ((lane >> 2) & 1) + 4 * qd + 4 * (wi >> 1)) & 31);
    const int k0 = 2 * pr;                                   // K position of the pair's first token
    const int ta = token_of_col(k0), tb = ta + 4;            // its two tokens
    const uint4 a = *reinterpret_cast<const uint4 *>(vc + ta * 64 + qd * 16);
    const uint4 c = *reinterpret_cast<const uint4 *>(vc + tb * 64 + qd * 16);
    const uint32_t b0 = ta < valid ? vsc[ta * 4 + qd] : 0u;
    const uint32_t b1 = tb < valid ? vsc[tb * 4 + qd] : 0u;
    const bool one_step = __all_sync(0xffffffffu, b0 <= 128u && b1 <= 128u);
    uint32_t fbits;
    if (one_step)
        fbits = (ta < valid ? (b0 + 126u) << 7 : 0u) | (tb < valid ? (b1 + 126u) << 23 : 0u);
    else    // 2^(b-127); byte 0 is the subnormal 2^-127 (bits 0x40)
        fbits = (ta < valid ? (b0 ? b0 << 7 : 0x40u) : 0u) | (tb < valid ? (b1 ? b1 << 23 : 0x400000u) : 0u);
    const __nv_bfloat162 fac = *reinterpret_cast<const __nv_bfloat162 *>(&fbits);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wc[4] = {c.x, c.y, c.z, c.w};
    // v[i]: head dim 32 qd + i of both tokens (ta in the low half); the
    // multiply by 0x1040 adds the non-overlapping copies x << 6 and x << 12
    uint32_t v[32];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t ae = wa[w] & 0x0F0F0F0Fu, ce = wc[w] & 0x0F0F0F0Fu;                  // even dims
        const uint32_t ao = (wa[w] >> 4) & 0x0F0F0F0Fu, co = (wc[w] >> 4) & 0x0F0F0F0Fu;    // odd dims
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // byte j of each token in bytes 0 and 2, zeros in bytes 1 and 3
            const uint32_t sel = static_cast<uint32_t>(j | ((8 + j) << 4) | ((4 + j) << 8) | ((12 + j) << 12));
            v[8 * w + 2 * j] = (prmt(ae, ce, sel) * 0x1040u) & 0x81C081C0u;
            v[8 * w + 2 * j + 1] = (prmt(ao, co, sel) * 0x1040u) & 0x81C081C0u;
        }
    }
    // the store address of head dim 32 qd + 8 r + e is row[e] + 1024 r
    const uint32_t cch = static_cast<uint32_t>((k0 & 63) >> 3);    // the pair's 16-byte chunk in a row
    uint8_t *base = vt + (k0 >> 6) * 16384 + (k0 & 7) * 2 + qd * 4096;   // rows 32 qd ..
    uint8_t *row[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) row[e] = base + e * 128 + ((cch ^ static_cast<uint32_t>(e)) << 4);
    if (one_step) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            *reinterpret_cast<__nv_bfloat162 *>(row[i & 7] + (i >> 3) * 1024) =
                __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&v[i]), fac);
    } else {
        const uint32_t k126 = 0x7E807E80u;                             // 2^126 in both halves
        const __nv_bfloat162 two126 = *reinterpret_cast<const __nv_bfloat162 *>(&k126);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            *reinterpret_cast<__nv_bfloat162 *>(row[i & 7] + (i >> 3) * 1024) =
                __hmul2(__hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&v[i]), two126), fac);
    }
}

__global__ void __cluster_dims__(kAttnSplit, 1, 1) __launch_bounds__(kAttnThreads, 1)
    mx4_attn_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_ks,
                    const __grid_constant__ AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x / kAttnSplit;          // row * kv_heads + kv head
    const int kvh = static_cast<int>(item % p.kv_heads);
    const uint32_t rank = cluster_ctarank();               // this CTA's half of the row's pages

    auto bar = [&](int i) { return sbase + AttnSmem::kBars + 8u * i; };
    auto kfull = [&](int i) { return bar(i); };
    auto kempty = [&](int i) { return bar(kAttnKStages + i); };
    auto vfull = [&](int i) { return bar(2 * kAttnKStages + i); };
    auto vempty = [&](int i) { return bar(2 * kAttnKStages + kAttnVStages + i); };
    constexpr int kB0 = 2 * kAttnKStages + 2 * kAttnVStages;
    const uint32_t qready = bar(kB0);
    auto sready = [&](int j) { return bar(kB0 + 1 + j); };          // page j's scores are in TMEM
    auto pvready = [&](int i) { return bar(kB0 + 1 + kAttnCtaPages + i); };
    auto pvfree = [&](int i) { return bar(kB0 + 1 + kAttnCtaPages + kAttnPvBufs + i); };
    const uint32_t pv_done = bar(kB0 + 1 + kAttnCtaPages + 2 * kAttnPvBufs);
    const uint32_t comb_ready = pv_done + 8;               // the peer has staged its partial results
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + AttnSmem::kAbort);
    int32_t *pids = reinterpret_cast<int32_t *>(smem + AttnSmem::kPid);

    if (threadIdx.x == 0) {
        // arrivals: TMA / commits count 1; the 4 softmax warps arrive on
        // qready and pvready, the 8 widening warps on vempty and pvready
        for (int i = 0; i < kAttnKStages; ++i) {
            mbar_init(kfull(i), 1);
            mbar_init(kempty(i), 1);
        }
        for (int i = 0; i < kAttnVStages; ++i) {
            mbar_init(vfull(i), 1);
            mbar_init(vempty(i), kAttnWidenWarps);
        }
        // pvready: the 4 softmax warps (P^T) and the 8 widening warps (V^T)
        mbar_init(qready, 4);
        for (int j = 0; j < kAttnCtaPages; ++j) mbar_init(sready(j), 1);
        for (int i = 0; i < kAttnPvBufs; ++i) {
            mbar_init(pvready(i), 4 + kAttnWidenWarps);
            mbar_init(pvfree(i), 1);
        }
        mbar_init(pv_done, 1);
        mbar_init(comb_ready, 4);               // the peer's 4 softmax warps (remote)
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_ks);
    }
    if (warp == 5) {
        tmem_alloc(sbase + AttnSmem::kTmemSlot, 512);
        tmem_relinquish();
    }
    // The set-up above touches no global memory, so under a programmatic
    // dependent launch it overlaps the previous kernel's tail; every global
    // access follows the wait.
    griddep_launch_dependents();
    griddep_wait();

    int ctx = p.context_lens[item];
    if (ctx > p.width * kPage) ctx = p.width * kPage;
    if (ctx < 0) ctx = 0;
    const int npages_all = (ctx + kPage - 1) / kPage;
    const int half = (npages_all + 1) / 2;
    const int pbase = rank == 0 ? 0 : half;                // first page of this CTA
    const int npages = rank == 0 ? half : npages_all - half;   // pages of this CTA

    if (threadIdx.x < kAttnMaxPages) {
        int32_t id = 0;
        if (static_cast<int>(threadIdx.x) >= pbase && static_cast<int>(threadIdx.x) < pbase + npages) {
            const int64_t raw = p.block_table[item * p.width + threadIdx.x];
            if (raw < 0 || raw >= p.num_pool_pages)
                atomicOr(&g_mx4_device_status, 0x1u);
            else
                id = static_cast<int32_t>(raw);
        }
        pids[threadIdx.x] = id;
    }
    tc_fence_before();
    __syncthreads();
    // the peer's barriers are initialised before anyone arrives on them remotely
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<uint32_t *>(smem + AttnSmem::kTmemSlot);

    if (warp == 4 || warp == 10) {
        // ------------------------------------------------------------ copies --
        // warp 4: the K pages (TMA); warp 10: the V pages (bulk copies), from
        // the start so they overlap the QK phase
        const uint64_t policy = l2_policy_evict_first();
        const bool is_k = warp == 4;
        const int nst = is_k ? kAttnKStages : kAttnVStages;
        int issued = 0;
        for (int j = 0; j < npages; ++j) {
            const int s = j % nst, u = j / nst;
            const uint32_t empty_b = is_k ? kempty(s) : vempty(s);
            if (!__all_sync(0xffffffffu, wait_bounded(empty_b, (u & 1) ^ 1u, abort_flag, kSiteAttnProducer)))
                break;
            if (elect_one()) {
                const int64_t pg = pids[pbase + j];
                if (is_k) {
                    mbar_arrive_expect_tx(kfull(s), kDataBytes + kScaleBytes);
                    tma_load_5d(sbase + AttnSmem::kK + s * kTileBytes, &tmap_k, kfull(s), 0, 0, 0, kvh,
                                static_cast<int>(pg), policy);
                    tma_load_3d(sbase + AttnSmem::kKs + s * kScaleBytes, &tmap_ks, kfull(s), 0, kvh,
                                static_cast<int>(pg), policy);
                } else {
                    mbar_arrive_expect_tx(vfull(s), kDataBytes + kScaleBytes);
                    bulk_load(sbase + AttnSmem::kV + s * kDataBytes, p.v_data + pg * p.vd_ps + kvh * p.vd_hs,
                              kDataBytes, vfull(s), policy);
                    bulk_load(sbase + AttnSmem::kVs + s * kScaleBytes, p.v_scale + pg * p.vs_ps + kvh * p.vs_hs,
                              kScaleBytes, vfull(s), policy);
                }
            }
            __syncwarp();
            ++issued;
        }
        // no copy may be in flight when the CTA exits: the last use of each
        // stage this warp armed completes (bounded)
        if (lane == 0) {
            const int n = issued < nst ? issued : nst;
            for (int i = 0; i < n; ++i) {
                const int j = issued - 1 - i;
                const uint32_t full_b = is_k ? kfull(j % nst) : vfull(j % nst);
                if (!drain_bounded(full_b, (j / nst) & 1)) break;
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA --
        bool ok = __all_sync(0xffffffffu, wait_bounded(qready, 0, abort_flag, kSiteAttnMma));
        const uint32_t sfb = tmem_base + kAttnSfbCol;
        const uint64_t qdesc = smem_desc(sbase + AttnSmem::kQ, 16, 1024, 2);
        if (ok) {
            tc_fence_after();
            if (elect_one()) tc_cp_32x128b_warpx4(sfb, smem_desc(sbase + AttnSmem::kUnit, 16, 128, 0));
            __syncwarp();
        }
        for (int j = 0; j < npages && ok; ++j) {
            const int s = j % kAttnKStages, u = j / kAttnKStages;
            if (!__all_sync(0xffffffffu, wait_bounded(kfull(s), u & 1, abort_flag, kSiteAttnMma))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (elect_one()) {
                const uint32_t sfa = tmem_base + kAttnSfaCol + 4u * j;
                tc_cp_32x128b_warpx4(sfa, smem_desc(sbase + AttnSmem::kKs + s * kScaleBytes, 16, 128, 0));
                const uint64_t kdesc = smem_desc(sbase + AttnSmem::kK + s * kTileBytes, 16, 1024, 2);
                const uint32_t d = tmem_base + kAttnSCol + kAttnN * j;
#pragma unroll
                for (uint32_t k = 0; k < 4; ++k)
                    tc_mma_mx_ss(d, kdesc + 2 * k, qdesc + 2 * k, attn_idesc_qk(k), sfa, sfb, k > 0 ? 1u : 0u);
                tc_commit(kempty(s));
                tc_commit(sready(j));
            }
            __syncwarp();
        }
        for (int j = 0; j < npages && ok; ++j) {
            const int b = j % kAttnPvBufs, u = j / kAttnPvBufs;
            if (!__all_sync(0xffffffffu, wait_bounded(pvready(b), u & 1, abort_flag, kSiteAttnMma))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (elect_one()) {
                const uint32_t vt = sbase + AttnSmem::kVt + b * 32768u;
                const uint32_t pt = sbase + AttnSmem::kPt + b * 4096u;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    // K step of 16 positions: 32 B inside a 128-byte atom row of
                    // V^T (next K-atom after 4 steps); two 256-byte groups of P^T
                    // (leading offset 256 B along K, stride offset 128 B along N)
                    const uint64_t a = smem_desc(vt + (ks >> 2) * 16384u + (ks & 3) * 32u, 16, 1024, 2);
                    const uint64_t bd = smem_desc(pt + ks * 512u, 256, 128, 0);
                    tc_mma_f16_ss(tmem_base + kAttnOutCol, a, bd, kAttnIdescPv, (j > 0 || ks > 0) ? 1u : 0u);
                }
                tc_commit(pvfree(b));
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(pv_done);
        __syncwarp();
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(pv_done, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ---------------------------------------------------------- V widening --
        // warps 6-9 and 11-14 widen one eighth of each page each (warp 10
        // is the V copy warp above, warp 15 has no role)
        if (warp == 15) goto done;
        for (int j = 0; j < npages; ++j) {
            const int b = j % kAttnPvBufs, u = j / kAttnPvBufs;
            const int vs = j % kAttnVStages;
            if (!__all_sync(0xffffffffu,
                            (u == 0 || wait_bounded(pvfree(b), (u - 1) & 1, abort_flag, kSiteAttnEpi)) &&
                                wait_bounded(vfull(vs), (j / kAttnVStages) & 1, abort_flag, kSiteAttnEpi)))
                break;
            attn_widen(smem + AttnSmem::kV + vs * kDataBytes, smem + AttnSmem::kVs + vs * kScaleBytes,
                       smem + AttnSmem::kVt + b * 32768, warp < 10 ? warp - 6 : warp - 7, lane,
                       ctx - (pbase + j) * kPage);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(pvready(b));
                mbar_arrive(vempty(vs));
            }
        }
    } else {
        // ------------------------------------------------------------- softmax --
        const int m = threadIdx.x;                       // TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
        const int tok_m = token_of_col(m);               // token of lane m within each page
        const int G = p.groups;
        {
            // Q tile (16 rows x 128 B, SW128) and the unit scale block
            const int h = m >> 3, c = m & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < G) v = *reinterpret_cast<const uint4 *>(p.q + ((item * G + h) << 7) + c * 16);
            *reinterpret_cast<uint4 *>(smem + AttnSmem::kQ + (h >> 3) * 1024 + (h & 7) * 128 + ((c ^ (h & 7)) << 4)) = v;
            reinterpret_cast<uint32_t *>(smem + AttnSmem::kUnit)[m] = 0x7F7F7F7Fu;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready);
        }
        float M[kAttnN], S[kAttnN];
#pragma unroll
        for (int h = 0; h < kAttnN; ++h) {
            M[h] = -INFINITY;
            S[h] = 0.0f;
        }
        // pass A: this CTA's per-head max over its valid tokens, page by page
        // as the QK products complete
        bool ok = true;
        for (int j = 0; j < npages; ++j) {
            if (!__all_sync(0xffffffffu, wait_bounded(sready(j), 0, abort_flag, kSiteAttnEpi))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[16];
            tmem_ld_32x32b_x16(tmem_base + lane_addr + kAttnSCol + kAttnN * j, v);
            if ((pbase + j) * kPage + tok_m < ctx) {
#pragma unroll
                for (int h = 0; h < kAttnN; ++h) M[h] = fmaxf(M[h], __uint_as_float(v[h]) * p.softmax_scale);
            }
        }
        // (the named-barrier syncs below run on every path, so the four
        // warps always pass the same number of them)
        float *red = reinterpret_cast<float *>(smem + AttnSmem::kRed);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) M[h] = fmaxf(M[h], __shfl_xor_sync(0xffffffffu, M[h], o));
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) red[warp * kAttnN + h] = M[h];
        }
        epi_bar_sync();
#pragma unroll
        for (int h = 0; h < kAttnN; ++h)
            M[h] = fmaxf(fmaxf(red[h], red[kAttnN + h]), fmaxf(red[2 * kAttnN + h], red[3 * kAttnN + h]));
        epi_bar_sync();
        // pass B: per page P^T and V^T for the PV MMA
        constexpr float kLog2e = 1.4426950408889634f;
        for (int j = 0; j < npages && ok; ++j) {
            const int b = j % kAttnPvBufs, u = j / kAttnPvBufs;
            if (!__all_sync(0xffffffffu,
                            u == 0 || wait_bounded(pvfree(b), (u - 1) & 1, abort_flag, kSiteAttnEpi))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // P^T at this lane's token position m (token tok_m): its 16 heads
            // as two 16-byte stores
            {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem_base + lane_addr + kAttnSCol + kAttnN * j, v);
                const bool valid = (pbase + j) * kPage + tok_m < ctx;
                uint32_t w[8];
#pragma unroll
                for (int h2 = 0; h2 < 8; ++h2) {
                    float p0 = 0.0f, p1 = 0.0f;
                    if (valid && 2 * h2 < G)
                        p0 = exp2f((__uint_as_float(v[2 * h2]) * p.softmax_scale - M[2 * h2]) * kLog2e);
                    if (valid && 2 * h2 + 1 < G)
                        p1 = exp2f((__uint_as_float(v[2 * h2 + 1]) * p.softmax_scale - M[2 * h2 + 1]) * kLog2e);
                    const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                    S[2 * h2] += __low2float(pb);
                    S[2 * h2 + 1] += __high2float(pb);
                    w[h2] = *reinterpret_cast<const uint32_t *>(&pb);
                }
                uint8_t *pt = smem + AttnSmem::kPt + b * 4096 + pt_offset(m);
                *reinterpret_cast<uint4 *>(pt) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(pt + 128) = make_uint4(w[4], w[5], w[6], w[7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(pvready(b));
        }
        // the normaliser: sum of the bf16 weights over all lanes
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) S[h] += __shfl_xor_sync(0xffffffffu, S[h], o);
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) red[warp * kAttnN + h] = S[h];
        }
        epi_bar_sync();
#pragma unroll
        for (int h = 0; h < kAttnN; ++h) S[h] = (red[h] + red[kAttnN + h]) + (red[2 * kAttnN + h] + red[3 * kAttnN + h]);
        // output: lane m holds head dim m of every head
        if (ok && npages > 0)
            ok = __all_sync(0xffffffffu, wait_bounded(pv_done, 0, abort_flag, kSiteAttnEpi));
        uint32_t acc[16];
        if (ok && npages > 0) {
            tc_fence_after();
            tmem_ld_32x32b_x16(tmem_base + lane_addr + kAttnOutCol, acc);
        } else {
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) acc[h] = 0u;
        }
        // Combine the two halves: rank r finalises heads 8r .. 8r+7.  Each
        // CTA stages the peer's heads of its accumulator (head-major) and
        // all its sums and maxima in its own shared memory, arrives on the
        // peer's comb_ready (release, cluster scope), waits for the peer's
        // arrival on its own, then reads the peer's staged values (one
        // coalesced 128-byte cluster load per warp and head), rescales both
        // halves to the row's max, adds, normalises and stores bf16 (a half
        // with no weight contributes nothing).
        {
            float *cm = reinterpret_cast<float *>(smem + AttnSmem::kComb);
#pragma unroll
            for (int h = 0; h < kAttnN; ++h)
                if ((h >> 3) != static_cast<int>(rank)) cm[(h & 7) * 128 + m] = __uint_as_float(acc[h]);
            if (threadIdx.x < kAttnN) {
                float *cs = reinterpret_cast<float *>(smem + AttnSmem::kCombS);
                float sv = 0.0f, mv = 0.0f;
#pragma unroll
                for (int h = 0; h < kAttnN; ++h) {
                    sv = h == m ? S[h] : sv;
                    mv = h == m ? M[h] : mv;
                }
                cs[m] = sv;
                cs[kAttnN + m] = mv;
            }
            fence_cluster();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(cluster_map(comb_ready, rank ^ 1u));
            if (__all_sync(0xffffffffu, wait_cluster_bounded(comb_ready, 0, abort_flag, kSiteAttnEpi))) {
                const uint32_t pm = cluster_map(sbase + AttnSmem::kComb + 4u * m, rank ^ 1u);
                const uint32_t ps = cluster_map(sbase + AttnSmem::kCombS, rank ^ 1u);
                float a1[8], s1[8], m1[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    a1[i] = ld_cluster_f32(pm + 512u * i);
                    s1[i] = ld_cluster_f32(ps + 4u * (8 * rank + i));
                    m1[i] = ld_cluster_f32(ps + 4u * (kAttnN + 8 * rank + i));
                }
                __nv_bfloat16 *o = p.out + (item * G) * kDim;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    // this thread's own values of head 8 rank + i (static register indexes)
                    const float a0 = __uint_as_float(rank ? acc[8 + i] : acc[i]);
                    const float s0 = rank ? S[8 + i] : S[i], m0 = rank ? M[8 + i] : M[i];
                    const float mx = s1[i] > 0.0f && m1[i] > m0 ? m1[i] : m0;
                    const float f0 = s0 > 0.0f ? exp2f((m0 - mx) * kLog2e) : 0.0f;
                    const float f1 = s1[i] > 0.0f ? exp2f((m1[i] - mx) * kLog2e) : 0.0f;
                    const float a = a0 * f0 + a1[i] * f1, sum = s0 * f0 + s1[i] * f1;
                    const int h = 8 * static_cast<int>(rank) + i;
                    if (h < G) o[h * kDim + m] = __float2bfloat16_rn(sum > 0.0f ? __fdividef(a, sum) : 0.0f);
                }
            }
        }
    }

done:
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
    // neither CTA leaves while the other may still write into its shared memory
    cluster_sync();
}

}  // namespace mx4
