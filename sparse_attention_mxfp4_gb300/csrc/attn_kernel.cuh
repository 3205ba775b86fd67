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
// 2-CTA clusters, 512 threads a CTA; a cluster takes rows c, c + C, c + 2C,
// ... (C clusters, at most as many as fit on the GPU at once), each CTA half
// of each row's pages, so that one row's tail overlaps the next row's
// copies.  The pages stream against per-head weight offsets o (x the score
// in log2 units): P = bf16(2^(x - o)), summed per thread and multiplied
// into V by the tensor core as each page's QK product lands.  An offset
// moves up only when some score passes it by more than 2^8 (always on the
// row's first page): then the weight sums and the PV accumulators are
// rescaled by 2^(o_old - o_new) in place.  With sigma = sum P and D = sum P V,
//     out = D / sigma,
// which is the softmax above up to the bf16 rounding of the weights (each
// weight is rounded once, whatever the offset); the two CTAs then combine
// their halves the same way (rescaled to the larger offset), each finalising
// 8 of the 16 heads from the partial output, weight sums and offsets that
// the peer pushed into its shared memory.  Per CTA:
//   warp 4   copies: per page, the K codes (4-D token-permuting TMA view
//            plus a KV-head dimension, the scorer's smem form) and K scales,
//            and the V codes and scales as two plain bulk copies (natural
//            token order), four pages deep each.
//   warp 5   QK MMAs (one thread): per page as soon as its K page lands,
//            tcgen05.mma kind::mxf8f6f4 block_scale, A = the K page (M = 128
//            tokens, e2m1, its e8m0 scales copied to a per-page TMEM slot),
//            B = the Q tile (N = 16 heads, e4m3, unit scales), D = the page's
//            16 score columns.
//   warps 15, 10  PV MMAs (one thread each, even and odd pages): per page as
//            soon as its operands are written, kind::f16, A = V^T (M = 128
//            head dims, K = 128 tokens, bf16, MN-major), B = P^T (N = 16
//            heads, bf16, MN-major), D = the warp's 16 accumulator columns.
//            A warp issues one of these small MMAs every hundred-odd cycles,
//            so the PV products of a page take two warps to keep up.
//   warps 0-3 softmax: thread m reads TMEM lane m (token 4(m%32)+m/32 of each
//            page) as each page's QK product completes, tests its scores
//            against the offsets (one barrier a page; the exact page max
//            only when an offset moves), writes P^T (bf16, at the token's
//            position: two 16-byte stores) and adds its weights to its
//            per-head sums; at the row's end the sums over the CTA, the two
//            accumulators and the cluster combine.
//   warps 6-9, 11-14 widen each page's V into V^T (bf16, natural token
//            order), two (token, 32-dim scale group) cells a thread.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "score_kernel.cuh"

namespace mx4 {

// warps 0-3 softmax (P^T), 4 copies, 5 QK MMAs, 6-9 and 11-14 V widening,
// 10 and 15 PV MMAs (the block is 16 warps so that 4 sit on each SM
// sub-partition: 128 registers a thread)
constexpr int kAttnThreads = 512;
constexpr int kAttnWidenWarps = 8;
constexpr int kAttnMaxPages = 24;       // pages a row may list
constexpr int kAttnSplit = 2;           // CTAs (one cluster) per row: each takes half of the row's pages
constexpr int kAttnCtaPages = (kAttnMaxPages + kAttnSplit - 1) / kAttnSplit;   // pages a CTA takes of a row
constexpr int kAttnSlots = kAttnCtaPages;   // TMEM score / accumulator slots, a ring over the CTA's pages
constexpr int kAttnN = 16;              // query heads per KV head (fewer are zero-padded)
constexpr int kAttnKStages = 4;
constexpr int kAttnVStages = 4;         // V pages load from the start, alongside the K pages
constexpr int kAttnPvBufs = 3;          // V^T / P^T operand buffers: widening runs up to 3 pages ahead of PV
// The CTA's g-th page (counted over all its rows) uses score slot
// g % kAttnSlots.  A QK product into a slot comes only after the softmax has
// read the scores of the page 7 before it (K and V copies go in step, V
// waits on the widening, the widening on PV, PV on the softmax), so 12 slots
// are never overwritten early.  The PV products of the even and of the odd
// pages accumulate in one accumulator each; a row's first product of each
// overwrites it, and comes only after the softmax has read the row before.
constexpr uint32_t kAttnSCol = 0;                                     // scores of slot i: 16 columns at 16 i
constexpr uint32_t kAttnAccCol = kAttnSlots * kAttnN;                 // 192: even-page and odd-page accumulators
constexpr uint32_t kAttnSfaCol = kAttnAccCol + 2 * kAttnN;            // 224: K scales, 4 per slot
constexpr uint32_t kAttnSfbCol = kAttnSfaCol + 4 * kAttnSlots;        // 272: unit Q scales
static_assert(kAttnSfbCol + 4 <= 512, "attention TMEM budget");
// Weight offsets: a head's offset moves up only when a score passes it by
// more than this (log2 units), so every weight stays below 2^8.
constexpr float kAttnOffsetSlack = 8.0f;
constexpr float kAttnNoOffset = -3.0e38f;   // a row's offsets before its first score (below every finite one)
// the offset of a head past `groups`: its zero query row scores 0, which this
// offset turns into a weight of 0 and never raises
constexpr float kAttnMuted = 3.0e38f;
static_assert(kAttnKStages == kAttnVStages, "one copy warp runs the K and V stages in step");
static_assert(kAttnCtaPages <= 32, "the copy warp holds a row's page ids one per lane");

enum AttnSite : uint32_t { kSiteAttnProducer = 6, kSiteAttnMma = 7, kSiteAttnEpi = 8 };

// P^T operand layout steps (see pt_offset below)
constexpr uint32_t kPtLbo = 144;
constexpr uint32_t kPtSbo = 2304;
constexpr uint32_t kPtBytes = 2 * kPtSbo;               // one P^T buffer

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
    int64_t num_items;                // rows * kv_heads
};

struct AttnSmem {
    static constexpr uint32_t kK = 0;                                    // K pages, 16 KB each
    static constexpr uint32_t kKs = kK + kAttnKStages * kTileBytes;      // K scales
    static constexpr uint32_t kV = kKs + kAttnKStages * kScaleBytes;     // V codes, natural order
    static constexpr uint32_t kVs = kV + kAttnVStages * kDataBytes;      // V scales
    static constexpr uint32_t kVt = ((kVs + kAttnVStages * kScaleBytes) + 1023) & ~1023u;   // 3 x 32 KB
    static constexpr uint32_t kPt = kVt + kAttnPvBufs * 32768;           // 3 x 4.5 KB
    static constexpr uint32_t kQ = (kPt + kAttnPvBufs * kPtBytes + 1023) & ~1023u;   // 2 x (16 x 128 B), by row parity
    static constexpr uint32_t kUnit = kQ + 2 * 2048;                     // 512 B of 0x7F
    static constexpr uint32_t kRed = kUnit + 512;                        // [2][16 heads][4 warps] warp maxima
    static constexpr uint32_t kPsum = kRed + 2 * 16 * 4 * 4;             // [16 heads][4 warps] weight sums
    static constexpr uint32_t kFin = kPsum + 16 * 4 * 4;                 // this CTA's 16 sums, then 16 offsets
    static constexpr uint32_t kComb = kFin + 2 * 16 * 4;                 // 2 x from the peer (by row parity)
    static constexpr uint32_t kBars = kComb + 2 * (128 * 8 * 4 + 2 * 16 * 4);
    // kfull[4] kempty[4] vfull[4] vempty[4] qready[2] qfree[2] sready[12] pvready[3] pvfree[3] pv_done qk_done
    // comb_ready[2] pv_fin[2]
    static constexpr uint32_t kNumBars = 2 * kAttnKStages + 2 * kAttnVStages + 4 + kAttnSlots + 2 * kAttnPvBufs + 6;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kAlloc = kEnd + 1024;
};
static_assert(AttnSmem::kAlloc <= 227 * 1024, "attention shared memory budget");
static_assert(AttnSmem::kComb % 16 == 0 && AttnSmem::kRed % 16 == 0 && AttnSmem::kPsum % 16 == 0 &&
                  AttnSmem::kQ % 1024 == 0 && AttnSmem::kBars % 8 == 0,
              "attention shared memory alignment");

// Instruction descriptors.  QK (kind::mxf8f6f4): A = E2M1 (5, bits 7..9),
// B = E4M3 (0, bits 10..12), N = 16, M = 128, UE8M0 scales (bit 23), scale
// ids of K block k in bits 4..5 (B) and 29..30 (A).  PV (kind::f16): F32
// accumulator (1, bits 4..5), A = B = BF16 (1), A MN-major (bit 15), B
// MN-major (bit 16), N = 16, M = 128.
__device__ __forceinline__ uint32_t attn_idesc_qk(uint32_t k)
{
    constexpr uint32_t kBase = (5u << 7) | (0u << 10) | ((16u >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
    return kBase | (k << 4) | (k << 29);
}
constexpr uint32_t kAttnIdescPv =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// Both PV operands are MN-major without swizzling: an 8 x 8 core matrix is
// 8 tokens of 16 bytes (8 bf16 along M or N), 128 contiguous bytes; core
// matrices follow each other every SBO bytes along M / N (the stride
// offset) and every LBO bytes along K (the leading offset):
//   P^T (N = 16 heads):  byte 144 (t / 8) + 2304 (h / 8) + 16 (t % 8) + 2 (h % 8), LBO 144, SBO 2304
//   V^T (M = 128 dims):  byte 2048 (t / 8) + 128 (d / 8) + 16 (t % 8) + 2 (d % 8), LBO 2048, SBO 128
// One MMA (K = 16) takes two groups of 8 tokens of each.  The 144-byte step
// of P^T (a 16-byte gap after each core matrix) keeps the softmax threads'
// 16-byte stores free of bank conflicts: the 8 lanes of a quarter warp hold
// tokens 8 (4 q + j / 2) + 4 (j % 2) + w, whose stores then fall in 8
// distinct 16-byte bank groups (with a 256-byte step they fell in 2).  The
// steps are kPtLbo and kPtSbo.
__device__ __forceinline__ uint32_t pt_offset(int t) { return kPtLbo * (t >> 3) + 16u * (t & 7); }

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Named barrier 1 over the 4 softmax warps that also ANDs a predicate
// across them, so that all four leave a loop at the same iteration.
__device__ __forceinline__ bool epi_bar_and(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// Named barrier 1 over the 4 softmax warps that also ORs a predicate across
// them.
__device__ __forceinline__ bool epi_bar_or(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// prmt.b32 in its default mode: result byte i is byte (sel >> 4i) & 7 of
// {b, a} (a = bytes 0..3), or that byte's sign bit replicated when bit 3 of
// the selector nibble is set.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Sum 16 per-head values over the 32 lanes of a warp by halving: at each of
// the first four exchanges a lane keeps half of its heads and sends the other
// half to its partner, so lane l ends with head (l >> 1) & 15 (bits 4..1 of
// l), summed over all 32 lanes after the fifth.
__device__ __forceinline__ float warp_sum16(const float (&x)[16], int lane)
{
    float a[8], b[4], c[2];
    const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4, u1 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (u4 ? x[i + 8] : x[i]) + __shfl_xor_sync(0xffffffffu, u4 ? x[i] : x[i + 8], 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = (u3 ? a[i + 4] : a[i]) + __shfl_xor_sync(0xffffffffu, u3 ? a[i] : a[i + 4], 8);
#pragma unroll
    for (int i = 0; i < 2; ++i) c[i] = (u2 ? b[i + 2] : b[i]) + __shfl_xor_sync(0xffffffffu, u2 ? b[i] : b[i + 2], 4);
    const float d = (u1 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, u1 ? c[0] : c[1], 2);
    return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

// Maximum of 16 per-head values over the 32 lanes of a warp by halving, as
// warp_sum16: lane l ends with head (l >> 1) & 15 (NaN inputs are ignored,
// like fmaxf).
__device__ __forceinline__ float warp_max16(const float (&x)[16], int lane)
{
    float a[8], b[4], c[2];
    const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4, u1 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = fmaxf(u4 ? x[i + 8] : x[i], __shfl_xor_sync(0xffffffffu, u4 ? x[i] : x[i + 8], 16));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        b[i] = fmaxf(u3 ? a[i + 4] : a[i], __shfl_xor_sync(0xffffffffu, u3 ? a[i] : a[i + 4], 8));
#pragma unroll
    for (int i = 0; i < 2; ++i)
        c[i] = fmaxf(u2 ? b[i + 2] : b[i], __shfl_xor_sync(0xffffffffu, u2 ? b[i] : b[i + 2], 4));
    const float d = fmaxf(u1 ? c[1] : c[0], __shfl_xor_sync(0xffffffffu, u1 ? c[0] : c[1], 2));
    return fmaxf(d, __shfl_xor_sync(0xffffffffu, d, 1));
}

// Wait for bar0 and, when need1, bar1 as well: one probe of both first (one
// round trip), then bounded waits as wait_bounded.
__device__ __forceinline__ bool wait2_bounded(uint32_t bar0, uint32_t parity0, bool need1, uint32_t bar1,
                                              uint32_t parity1, volatile uint32_t *abort_flag, uint32_t site)
{
    if (!stalled_here(site) && (need1 ? mbar_try_wait2(bar0, parity0, bar1, parity1) : mbar_try_wait(bar0, parity0)))
        return true;
    return wait_bounded(bar0, parity0, abort_flag, site) && (!need1 || wait_bounded(bar1, parity1, abort_flag, site));
}

// Bytes each CTA pushes into its peer for the combine: 128 dims x 8 heads of
// the partial output, then 16 weight sums and 16 maxima.
constexpr uint32_t kCombBytes = 128 * 8 * 4 + 2 * 16 * 4;

// Widen a V page (natural layout in smem: 64 code bytes and 4 scale bytes
// per token) into the bf16 V^T operand.  The 256 threads of the 8 widening
// warps each take two (token, 32-dim scale group) cells: lane l = 8 q + i of
// warp slot wi takes the tokens t = 8 (wi + 8 r) + i (r = 0, 1) in group
// g = (i / 2 + q) % 4, so that the 16-byte code loads of a quarter-warp
// touch 8 distinct 16-byte bank groups (their (t % 2, g) all differ) and so
// do its 16-byte stores (their t % 8 all differ); the four quarters cover a
// token's four groups.  Conversion without a table: an e2m1 code s|E|m (E
// two bits) placed as bf16 bits (E m) << 6 | s << 15 is the bf16 number
// 2^-126 times its value (a subnormal for E = 0, exact), so one packed
// multiply by 2^(b-1) (bf16 bits (b + 126) << 7; b = the cell's e8m0 byte)
// gives the scaled value; when some lane has b > 128 that factor overflows
// bf16, and the warp multiplies by 2^126 and 2^(b-127) instead.  Tokens at
// or past `valid` get a zero factor.  A cell's 32 dims are 16 pairs of
// neighbours (the low and high nibble of one code byte, under one scale),
// stored as four 16-byte rows of 8 dims.
__device__ __forceinline__ void attn_widen(const uint8_t *vc, const uint8_t *vsc, uint8_t *vt, int wi, int lane,
                                           int valid)
{
    const int i = lane & 7, q = lane >> 3;
    const int g = ((i >> 1) + q) & 3;
    int t[2];
    uint4 c[2];
    uint32_t sb[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        t[r] = 8 * (wi + 8 * r) + i;
        c[r] = *reinterpret_cast<const uint4 *>(vc + t[r] * 64 + g * 16);
        sb[r] = t[r] < valid ? vsc[t[r] * 4 + g] : 0u;
    }
    const bool one_step = __all_sync(0xffffffffu, sb[0] <= 128u && sb[1] <= 128u);
    const uint32_t k126 = 0x7E807E80u;                             // 2^126 in both halves
    const __nv_bfloat162 two126 = *reinterpret_cast<const __nv_bfloat162 *>(&k126);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        uint32_t fb;
        if (one_step)
            fb = t[r] < valid ? (sb[r] + 126u) << 7 : 0u;
        else    // 2^(b-127); byte 0 is the subnormal 2^-127 (bits 0x40)
            fb = t[r] < valid ? (sb[r] ? sb[r] << 7 : 0x40u) : 0u;
        fb |= fb << 16;
        const __nv_bfloat162 fac = *reinterpret_cast<const __nv_bfloat162 *>(&fb);
        const uint32_t wd[4] = {c[r].x, c[r].y, c[r].z, c[r].w};
        uint8_t *dst = vt + 2048 * (t[r] >> 3) + 16 * (t[r] & 7) + 512 * g;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            // code byte jb of word w: dims 32 g + 8 w + 2 jb (low nibble) and
            // 32 g + 8 w + 2 jb + 1 (high nibble); the multiply by 0x1040 adds
            // the non-overlapping copies x << 6 and x << 12
            const uint32_t lo = wd[w] & 0x0F0F0F0Fu, hi = (wd[w] >> 4) & 0x0F0F0F0Fu;
            uint32_t o[4];
#pragma unroll
            for (int jb = 0; jb < 4; ++jb) {
                const uint32_t sel = static_cast<uint32_t>(jb | ((8 + jb) << 4) | ((4 + jb) << 8) | ((12 + jb) << 12));
                const uint32_t x = (prmt(lo, hi, sel) * 0x1040u) & 0x81C081C0u;
                __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&x);
                if (!one_step) v = __hmul2(v, two126);
                v = __hmul2(v, fac);
                o[jb] = *reinterpret_cast<const uint32_t *>(&v);
            }
            *reinterpret_cast<uint4 *>(dst + 128 * w) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// One row's share for this CTA: the clamped context, its pages and the KV
// head.  Every role reads it for itself (a cached load of context_lens).
struct AttnItem {
    int ctx, npages, pbase, kvh;
};

__device__ __forceinline__ AttnItem attn_item(const AttnParams &p, int64_t item, uint32_t rank, int split = kAttnSplit)
{
    AttnItem it;
    int ctx = p.context_lens[item];
    if (ctx > p.width * kPage) ctx = p.width * kPage;
    if (ctx < 0) ctx = 0;
    const int all = (ctx + kPage - 1) / kPage;
    const int half = split == 1 ? all : (all + 1) / 2;
    it.ctx = ctx;
    it.pbase = rank == 0 ? 0 : half;
    it.npages = rank == 0 ? half : all - half;
    it.kvh = static_cast<int>(item % p.kv_heads);
    return it;
}

// Position in a ring of N stages / buffers / slots and the parity of the
// pass over it, advanced once per page (no division on the page counter).
template <int N>
struct PageRing {
    int idx = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next()
    {
        if (++idx == N) {
            idx = 0;
            ph ^= 1u;
        }
    }
};

__global__ void __cluster_dims__(kAttnSplit, 1, 1) __launch_bounds__(kAttnThreads, 1)
    mx4_attn_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_ks,
                    const __grid_constant__ AttnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();               // this CTA's half of each row's pages
    const int64_t item0 = blockIdx.x / kAttnSplit;         // this cluster's first row (row * kv_heads + kv head)
    const int64_t nclus = gridDim.x / kAttnSplit;          // rows item0, item0 + nclus, ...

    auto bar = [&](int i) { return sbase + AttnSmem::kBars + 8u * i; };
    auto kfull = [&](int i) { return bar(i); };
    auto kempty = [&](int i) { return bar(kAttnKStages + i); };
    auto vfull = [&](int i) { return bar(2 * kAttnKStages + i); };
    auto vempty = [&](int i) { return bar(2 * kAttnKStages + kAttnVStages + i); };
    constexpr int kB0 = 2 * kAttnKStages + 2 * kAttnVStages;
    auto qready = [&](int i) { return bar(kB0 + i); };              // Q buffer i staged
    auto qfree = [&](int i) { return bar(kB0 + 2 + i); };           // Q buffer i no longer read
    auto sready = [&](int i) { return bar(kB0 + 4 + i); };          // slot i's scores are in TMEM
    auto pvready = [&](int i) { return bar(kB0 + 4 + kAttnSlots + i); };
    auto pvfree = [&](int i) { return bar(kB0 + 4 + kAttnSlots + kAttnPvBufs + i); };
    const uint32_t pv_done = bar(kB0 + 4 + kAttnSlots + 2 * kAttnPvBufs);   // a row's PV products done
    const uint32_t qk_done = pv_done + 8;
    auto comb_ready = [&](int i) { return pv_done + 16 + 8u * i; }; // the peer's push for a row of parity i
    auto pv_fin = [&](int i) { return pv_done + 32 + 8u * i; };     // a PV warp's products all done
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + AttnSmem::kAbort);

    if (threadIdx.x == 0) {
        // arrivals: TMA / commits count 1; the 4 softmax warps arrive on
        // qready and pvready, the 8 widening warps on vempty and pvready;
        // pvfree takes a commit from each PV warp (each issues half of every
        // page's products); pv_done takes two a row: a commit from each PV
        // warp when the row has pages, else two arrivals of the softmax (so
        // that neither runs a phase ahead of the softmax's wait)
        for (int i = 0; i < kAttnKStages; ++i) {
            mbar_init(kfull(i), 1);
            mbar_init(kempty(i), 1);
        }
        for (int i = 0; i < kAttnVStages; ++i) {
            mbar_init(vfull(i), 1);
            mbar_init(vempty(i), kAttnWidenWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qready(i), 4);
            mbar_init(qfree(i), 1);
        }
        for (int i = 0; i < kAttnSlots; ++i) mbar_init(sready(i), 1);
        for (int i = 0; i < kAttnPvBufs; ++i) {
            mbar_init(pvready(i), 4 + kAttnWidenWarps);
            mbar_init(pvfree(i), 2);
        }
        mbar_init(pv_done, 2);
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
        tmem_alloc(sbase + AttnSmem::kTmemSlot, 512);
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
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<uint32_t *>(smem + AttnSmem::kTmemSlot);

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
        AttnItem it = attn_item(p, item0, rank);
        int32_t id = load_ids(item0, it);
        PageRing<kAttnKStages> krg;
        for (int64_t item = item0; item < p.num_items && ok; item += nclus) {
            AttnItem nit{};
            int32_t nid = 0;
            bool fetched = false;
            auto fetch_next = [&]() {
                if (!fetched && item + nclus < p.num_items) {
                    nit = attn_item(p, item + nclus, rank);
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
                    tma_load_5d(sbase + AttnSmem::kK + s * kTileBytes, &tmap_k, kfull(s), 0, 0, 0, it.kvh,
                                static_cast<int>(pg), policy);
                    tma_load_3d(sbase + AttnSmem::kKs + s * kScaleBytes, &tmap_ks, kfull(s), 0, it.kvh,
                                static_cast<int>(pg), policy);
                    mbar_arrive_expect_tx(vfull(s), kDataBytes + kScaleBytes);
                    bulk_load(sbase + AttnSmem::kV + s * kDataBytes, p.v_data + pg * p.vd_ps + it.kvh * p.vd_hs,
                              kDataBytes, vfull(s), policy);
                    bulk_load(sbase + AttnSmem::kVs + s * kScaleBytes, p.v_scale + pg * p.vs_ps + it.kvh * p.vs_hs,
                              kScaleBytes, vfull(s), policy);
                }
                __syncwarp();
                ++g;
                krg.next();
                // the next row's context and ids once the first stages are
                // issued (the warp waits for stages after that anyway)
                if (j == kAttnKStages - 1) fetch_next();
            }
            fetch_next();
            it = nit;
            id = nid;
        }
        // no copy may be in flight when the CTA exits: the last use of each
        // stage this warp armed completes (bounded)
        if (lane == 0) {
            const int64_t n = g < kAttnKStages ? g : kAttnKStages;
            for (int64_t i = 0; i < n; ++i) {
                const int64_t gg = g - 1 - i;
                const uint32_t ph = static_cast<uint32_t>(gg / kAttnKStages) & 1u;
                if (!drain_bounded(kfull(static_cast<int>(gg % kAttnKStages)), ph)) break;
                if (!drain_bounded(vfull(static_cast<int>(gg % kAttnKStages)), ph)) break;
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
                const uint32_t sfb = tmem_base + kAttnSfbCol;
                PageRing<kAttnKStages> krg;
                PageRing<kAttnSlots> srg;
                for (int64_t item = item0; item < p.num_items && ok; item += nclus, ++k) {
                    const AttnItem it = attn_item(p, item, rank);
                    const int qb = static_cast<int>(k & 1);
                    if (!(ok = wait_bounded(qready(qb), static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                            kSiteAttnMma)))
                        break;
                    tc_fence_after();
                    if (k == 0) tc_cp_32x128b_warpx4(sfb, smem_desc(sbase + AttnSmem::kUnit, 16, 128, 0));
                    const uint64_t qdesc = smem_desc(sbase + AttnSmem::kQ + qb * 2048u, 16, 1024, 2);
                    for (int j = 0; j < it.npages; ++j, ++g, krg.next(), srg.next()) {
                        const int s = krg.idx;
                        const uint32_t slot = static_cast<uint32_t>(srg.idx);
                        if (!(ok = wait_bounded(kfull(s), krg.ph, abort_flag, kSiteAttnMma))) break;
                        tc_fence_after();
                        const uint32_t sfa = tmem_base + kAttnSfaCol + 4u * slot;
                        tc_cp_32x128b_warpx4(sfa, smem_desc(sbase + AttnSmem::kKs + s * kScaleBytes, 16, 128, 0));
                        const uint64_t kdesc = smem_desc(sbase + AttnSmem::kK + s * kTileBytes, 16, 1024, 2);
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
                // Both PV warps take every page, warp 15 its first 64 tokens
                // (K steps 0-3) into the first accumulator and warp 10 its
                // last 64 into the second, so that a page's products take
                // half the issue time; the accumulators are added at the
                // row's end.
                const int64_t mine = warp == 15 ? 0 : 1;
                done_b = pv_fin(static_cast<int>(mine));
                PageRing<kAttnPvBufs> brg;
                for (int64_t item = item0; item < p.num_items && ok; item += nclus, ++k) {
                    const AttnItem it = attn_item(p, item, rank);
                    const uint32_t d = tmem_base + kAttnAccCol + kAttnN * static_cast<uint32_t>(mine);
                    for (int j = 0; j < it.npages; ++j, ++g, brg.next()) {
                        const int b = brg.idx;
                        if (!(ok = wait_bounded(pvready(b), brg.ph, abort_flag, kSiteAttnMma))) break;
                        tc_fence_after();
                        const uint32_t vt = sbase + AttnSmem::kVt + b * 32768u;
                        const uint32_t pt = sbase + AttnSmem::kPt + b * kPtBytes;
#pragma unroll
                        for (uint32_t i = 0; i < 4; ++i) {
                            // K step of 16 tokens: two 8-token groups of each operand
                            const uint32_t ks = 4u * static_cast<uint32_t>(mine) + i;
                            const uint64_t a = smem_desc(vt + ks * 4096u, 2048, 128, 0);
                            const uint64_t bd = smem_desc(pt + ks * (2 * kPtLbo), kPtLbo, kPtSbo, 0);
                            // (the row's first product overwrites the accumulator)
                            tc_mma_f16_ss(d, a, bd, kAttnIdescPv, (i > 0 || j > 0) ? 1u : 0u);
                        }
                        tc_commit(pvfree(b));
                    }
                    if (ok && it.npages > 0) tc_commit(pv_done);   // this warp's PV products of the row are done
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
    } else if (warp >= 6) {
        // ---------------------------------------------------------- V widening --
        // warps 6-9 and 11-14 (warps 10 and 15 are PV issuers)
        int64_t g = 0;
        bool ok = true;
        PageRing<kAttnPvBufs> brg;
        PageRing<kAttnVStages> krg;
        for (int64_t item = item0; item < p.num_items && ok; item += nclus) {
            const AttnItem it = attn_item(p, item, rank);
            for (int j = 0; j < it.npages; ++j, ++g, brg.next(), krg.next()) {
                const int b = brg.idx, vs = krg.idx;
                // (a buffer's first use waits for no PV product)
                if (!(ok = __all_sync(0xffffffffu, wait2_bounded(vfull(vs), krg.ph, g >= kAttnPvBufs, pvfree(b),
                                                                 brg.ph ^ 1u, abort_flag, kSiteAttnEpi))))
                    break;
                attn_widen(smem + AttnSmem::kV + vs * kDataBytes, smem + AttnSmem::kVs + vs * kScaleBytes,
                           smem + AttnSmem::kVt + b * 32768, warp < 10 ? warp - 6 : warp - 7, lane,
                           it.ctx - (it.pbase + j) * kPage);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(pvready(b));
                    mbar_arrive(vempty(vs));
                }
            }
        }
    } else {
        // ------------------------------------------------------------- softmax --
        const int m = threadIdx.x;                       // TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
        const int tok_m = token_of_col(m);               // token of lane m within each page
        const int G = p.groups;
        float *red = reinterpret_cast<float *>(smem + AttnSmem::kRed);
        float *psum = reinterpret_cast<float *>(smem + AttnSmem::kPsum);
        float *fin = reinterpret_cast<float *>(smem + AttnSmem::kFin);
        // Q of a row (16 rows x 128 B, SW128) into buffer qb, then qready
        auto stage_q = [&](int64_t item, int qb) {
            const int h = m >> 3, c = m & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < G) v = *reinterpret_cast<const uint4 *>(p.q + ((item * G + h) << 7) + c * 16);
            *reinterpret_cast<uint4 *>(smem + AttnSmem::kQ + qb * 2048 + (h >> 3) * 1024 + (h & 7) * 128 +
                                       ((c ^ (h & 7)) << 4)) = v;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready(qb));
        };
        reinterpret_cast<uint32_t *>(smem + AttnSmem::kUnit)[m] = 0x7F7F7F7Fu;   // before the first qready
        stage_q(item0, 0);
        // scores in log2 units: x = s * softmax_scale * log2(e)
        const float sl = p.softmax_scale * 1.4426950408889634f;
        const int hl = lane & 15;
        bool ok = true;
        int64_t g = 0;
        int64_t k = 0;                                   // rows done
        PageRing<kAttnPvBufs> brg;
        PageRing<kAttnSlots> srg;
        // (the named-barrier syncs below run on every path, so the four
        // warps always pass the same number of them)
        for (int64_t item = item0; item < p.num_items; item += nclus, ++k) {
            const AttnItem it = attn_item(p, item, rank);
            // the next row's Q, one row ahead, once QK is done with the buffer
            if (item + nclus < p.num_items) {
                const int64_t kn = k + 1;
                if (kn < 2 || __all_sync(0xffffffffu, wait_bounded(qfree(static_cast<int>(kn & 1)),
                                                                   static_cast<uint32_t>((kn >> 1) - 1) & 1u,
                                                                   abort_flag, kSiteAttnEpi)))
                    stage_q(item + nclus, static_cast<int>(kn & 1));
            }
            // the row's per-head weight offsets (the same in every thread)
            // and this thread's per-head sums of its tokens' bf16 weights
            float mo[kAttnN], S[kAttnN];
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) {
                mo[h] = h < G ? kAttnNoOffset : kAttnMuted;
                S[h] = 0.0f;
            }
            for (int j = 0; j < it.npages && ok; ++j, ++g, brg.next(), srg.next()) {
                const int b = brg.idx;
                const uint32_t slot = static_cast<uint32_t>(srg.idx);
                const bool okw = __all_sync(0xffffffffu, wait2_bounded(sready(srg.idx), srg.ph, g >= kAttnPvBufs,
                                                                       pvfree(b), brg.ph ^ 1u, abort_flag, kSiteAttnEpi));
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
                // a row's first page).
                if (epi_bar_or(need || !okw)) {
                    // the scores themselves again, into y (y lost them against
                    // the old offsets)
                    if (okw) {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(s_addr, v);
#pragma unroll
                        for (int h = 0; h < kAttnN; ++h) y[h] = valid ? __uint_as_float(v[h]) * sl : -INFINITY;
                    }
                    // the warp's max of each head (lanes 2 h, 2 h + 1 hold head h)
                    const float wm = okw ? warp_max16(y, lane) : 0.0f;
                    if ((lane & 1) == 0) red[((j & 1) * 16 + (lane >> 1)) * 4 + warp] = wm;
                    ok = epi_bar_and(okw);
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
                    if (j > 0) {
                        // the PV accumulators, once every product issued so
                        // far has completed: both PV warps' commits of page
                        // g - 1 (each tracks all of its warp's earlier
                        // products); the next product is issued only after
                        // this page's P^T, below
                        const int b1 = b > 0 ? b - 1 : kAttnPvBufs - 1;
                        const uint32_t ph1 = b > 0 ? brg.ph : brg.ph ^ 1u;
                        const bool okp = __all_sync(0xffffffffu, wait_bounded(pvfree(b1), ph1, abort_flag, kSiteAttnEpi));
                        ok = epi_bar_and(okp);
                        if (!ok) break;
                        tc_fence_after();
                        uint32_t a[2][16];
                        tmem_ld2_32x32b_x16(tmem_base + lane_addr + kAttnAccCol,
                                            tmem_base + lane_addr + kAttnAccCol + kAttnN, a[0], a[1]);
                        uint32_t o[32];
#pragma unroll
                        for (int h = 0; h < kAttnN; ++h) {
                            o[h] = __float_as_uint(__uint_as_float(a[0][h]) * f[h]);
                            o[kAttnN + h] = __float_as_uint(__uint_as_float(a[1][h]) * f[h]);
                        }
                        tmem_st_32x32b_x32(tmem_base + lane_addr + kAttnAccCol, o);
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
                uint8_t *pt = smem + AttnSmem::kPt + b * kPtBytes + pt_offset(tok_m);
                *reinterpret_cast<uint4 *>(pt) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(pt + kPtSbo) = make_uint4(w[4], w[5], w[6], w[7]);
                // P^T visible to the tensor core
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(pvready(b));
            }
            // the CTA's weight sum and offset per head (threads 0-15)
            {
                const float wsum = warp_sum16(S, lane);      // lanes 2 h, 2 h + 1 hold head h
                if ((lane & 1) == 0) psum[(lane >> 1) * 4 + warp] = wsum;
            }
            epi_bar_sync();
            if (m < kAttnN) {
                float om = 0.0f;
#pragma unroll
                for (int h = 0; h < kAttnN; ++h) om = m == h ? mo[h] : om;
                const float4 s4 = reinterpret_cast<const float4 *>(psum)[m];
                fin[m] = ok ? (s4.x + s4.y) + (s4.z + s4.w) : 0.0f;
                fin[kAttnN + m] = om;
            }
            // this row's PV products: in a row without pages the PV warps do
            // not commit, the softmax arrives in their place (every row's
            // phase is waited for, so the parities stay in step)
            if (m == 0 && it.npages == 0) {
                mbar_arrive(pv_done);
                mbar_arrive(pv_done);
            }
            // (the result is made the group's: a warp whose wait ran out must
            // not run fewer named barriers than the others in the next row)
            const bool pv_ok = !ok || __all_sync(0xffffffffu, wait_bounded(pv_done, static_cast<uint32_t>(k) & 1u,
                                                                           abort_flag, kSiteAttnEpi));
            ok = epi_bar_and(ok && pv_ok);
            epi_bar_sync();
            // lane m of the accumulators holds head dim m of every head: the
            // products of the pages' first and last 64 tokens
            float acc[kAttnN];
#pragma unroll
            for (int h = 0; h < kAttnN; ++h) acc[h] = 0.0f;
            if (ok && it.npages > 0) {
                tc_fence_after();
                uint32_t a[2][16];
                tmem_ld2_32x32b_x16(tmem_base + lane_addr + kAttnAccCol, tmem_base + lane_addr + kAttnAccCol + kAttnN,
                                    a[0], a[1]);
#pragma unroll
                for (int h = 0; h < kAttnN; ++h) acc[h] = __uint_as_float(a[0][h]) + __uint_as_float(a[1][h]);
            }
            // Combine the two halves: rank r finalises heads 8r .. 8r+7.
            // Each CTA pushes the peer's heads of its accumulator ([dim][8
            // heads]) and its 16 sums and maxima into the peer's buffer of
            // this row's parity with st.async, whose bytes complete the
            // peer's comb_ready; it then waits for its own, rescales both
            // halves to the row's max, adds, normalises and stores bf16 (a
            // half with no weight contributes nothing).
            {
                const int cb = static_cast<int>(k & 1);
                const uint32_t peer = rank ^ 1u;
                const uint32_t pc = cluster_map(sbase + AttnSmem::kComb + cb * kCombBytes, peer);
                const uint32_t pbar = cluster_map(comb_ready(cb), peer);
                float a8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) a8[i] = peer ? acc[8 + i] : acc[i];
                st_async_v4_u32(pc + 32u * m, __float_as_uint(a8[0]), __float_as_uint(a8[1]),
                                __float_as_uint(a8[2]), __float_as_uint(a8[3]), pbar);
                st_async_v4_u32(pc + 32u * m + 16u, __float_as_uint(a8[4]), __float_as_uint(a8[5]),
                                __float_as_uint(a8[6]), __float_as_uint(a8[7]), pbar);
                if (m < 2 * kAttnN) st_async_u32(pc + 4096u + 4u * m, __float_as_uint(fin[m]), pbar);
                const bool comb_ok = __all_sync(0xffffffffu, wait_bounded(comb_ready(cb), static_cast<uint32_t>(k >> 1) & 1u,
                                                                         abort_flag, kSiteAttnEpi));
                if (comb_ok) {
                    const float *cm = reinterpret_cast<const float *>(smem + AttnSmem::kComb + cb * kCombBytes);
                    const float4 c0 = reinterpret_cast<const float4 *>(cm)[2 * m];
                    const float4 c1 = reinterpret_cast<const float4 *>(cm)[2 * m + 1];
                    const float a1[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    __nv_bfloat16 *o = p.out + (item * G) * kDim;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int h = 8 * static_cast<int>(rank) + i;
                        // this thread's own values of head h (static register indexes)
                        const float a0 = rank ? acc[8 + i] : acc[i];
                        const float s0 = fin[h], m0 = fin[kAttnN + h];
                        const float s1 = cm[1024 + h], m1 = cm[1024 + kAttnN + h];
                        const float mx = s1 > 0.0f && m1 > m0 ? m1 : m0;
                        const float f0 = s0 > 0.0f ? ex2_approx(m0 - mx) : 0.0f;
                        const float f1 = s1 > 0.0f ? ex2_approx(m1 - mx) : 0.0f;
                        const float a = a0 * f0 + a1[i] * f1, sum = s0 * f0 + s1 * f1;
                        if (h < G) o[h * kDim + m] = __float2bfloat16_rn(sum > 0.0f ? __fdividef(a, sum) : 0.0f);
                    }
                }
                // every thread has read this buffer and fin: the buffer's
                // barrier is re-armed for the row after next (only once its
                // phase has completed; after a wait that ran out the CTA is
                // aborting and every later wait gives up at once)
                epi_bar_sync();
                if (m == 0 && comb_ok) mbar_arrive_expect_tx(comb_ready(cb), kCombBytes);
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
    cluster_sync();
}

}  // namespace mx4
