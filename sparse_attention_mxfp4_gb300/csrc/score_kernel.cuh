// score_kernel.cuh -- the paged MXFP4 index-K scorer kernel for sm_103a.
//
// One persistent CTA per SM walks a contiguous range of work units.  A unit
// is (request, tile of query rows, chunk of kChunk pages).  A tile is R query
// rows x 64 heads = 128 rows of the MMA A operand (R = 2 for prefill, 1 for
// decode, where lanes 64..127 stay zero).
//
// Roles (warp-specialised, 480 threads, three independent pipeline lanes
// that take the units in rotation; the constants below give the warp numbers):
//   epilogue warpgroup (one per lane): warpgroup 0 also loads Q, rounds bf16
//              -> e4m3 in registers and stores it into TMEM as the MMA's A
//              operand (thread m owns TMEM lane m); per page each thread reads
//              its fp32 accumulator row from TMEM (tcgen05.ld.red returns the
//              page max of a fully live page in the load itself), applies the
//              causal mask on partial pages and sm_scale, stages the unit's 8
//              page maxima in smem and writes them as one 32-byte sector (or
//              emits per-token logits).
//   lane warp (one per lane), TMA side: per live page, look up the physical
//              page id in the block table and issue two TMA loads: the 8 KB of
//              e2m1 codes (unpacked in flight to the 16 KB padded layout the
//              tensor core reads) and the 512 B of e8m0 scales.
//   lane warp, MMA side: copies the page's scales into TMEM (tcgen05.cp)
//              and issues 4 block-scaled MMAs (K = 32 each) of
//              kind::mxf8f6f4: A = Q from TMEM (e4m3, unit scale), B = K page
//              from smem (e2m1 with its e8m0 bytes), D = 128 x 128 fp32 in TMEM.
//              Only B is read from shared memory, so the operand traffic is
//              16 KB per 128x128x128 MMA group.
//
// Token order inside the B tile: MMA column n holds token 4*(n%32) + n/32.
// The 4-D tensor map that gathers the page performs this permutation, and it
// makes the page's raw [128][4] scale block exactly the scale-factor layout
// the tensor core expects (32 lanes x 4 columns x 4 bytes), so scales need no
// reshuffle.  The page max is order-free; the mask and the per-token stores
// use the permuted index.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace mx4 {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kPage = 128;
constexpr int kDataBytes = 8192;                // packed e2m1 codes per page
constexpr int kScaleBytes = 512;                // e8m0 bytes per page
constexpr int kTileBytes = 128 * 128;           // one page in the padded 4-bit smem form
// The CTA runs three independent pipeline lanes; a CTA's units go to them in
// rotation.  Each lane has its own lane warp (TMA loads and MMAs), epilogue
// warpgroup, smem stages, TMEM scale buffers and TMEM accumulator, so every
// mbarrier has one waiting and one arriving side that walk its phases in
// order (a parity wait never runs two phases ahead of its barrier, where the
// parity test could not tell it from done), and each epilogue warpgroup
// writes whole 8-page units (full 32-byte sectors of the output).  With one
// accumulator per lane, a lane's page period is the serial chain MMA issue ->
// MMA completion -> epilogue TMEM read -> accumulator release; three lanes
// overlap three such chains on the tensor pipe.  The lanes share only the
// double-buffered query tile.
constexpr int kLanes = 3;
constexpr int kStagesPerLane = 4;               // smem pages in flight per lane
constexpr int kStages = kLanes * kStagesPerLane;
// TMEM scale-factor buffers for B per lane.  They need no barrier of their
// own: a lane's MMA warp copies page j+1's scales only after the epilogue has
// released the accumulator of page j, i.e. after page j's MMAs (and all
// earlier ones of the lane, the readers of the buffer being overwritten)
// completed.
constexpr int kSfbPerLane = 2;
constexpr int kSfbBufs = kLanes * kSfbPerLane;
constexpr int kDBufs = kLanes;                  // one TMEM accumulator per lane
constexpr int kChunk = 8;                       // pages per work unit
// Warp roles: warps 4l .. 4l+3 are the epilogue warpgroup of lane l (warp w
// reads TMEM lane quadrant w % 4; lane 0's group also loads the query tiles),
// then one lane warp per lane that issues both the lane's TMA page loads and
// its MMAs (the first lane warp owns the TMEM allocation).
constexpr int kEpiSets = kLanes;
constexpr int kMmaWarps = kLanes;
constexpr int kLaneWarp0 = 4 * kEpiSets;                 // 12
constexpr int kThreads = 32 * (kLaneWarp0 + kMmaWarps);  // 15 warps: at most 4 per SM sub-partition
constexpr int kLookahead = kStagesPerLane - 1;           // TMA pages in flight ahead of the MMA stream
constexpr uint32_t kTmemCols = 512;
// TMEM columns: D[lanes] x 128 | A (query tile, e4m3) [2] x 32 | SFA[lanes] x 4 | SFB[lanes x 2] x 4
constexpr uint32_t kTmemACol = kDBufs * 128;
constexpr uint32_t kTmemSfaCol = kTmemACol + 2 * 32;
constexpr uint32_t kTmemSfbCol = kTmemSfaCol + 4 * kMmaWarps;
// Transaction bytes of one page: the 4-bit TMA load counts the packed
// global bytes (8192), not the 16 KB it writes in the padded smem form.
constexpr uint32_t kStageTxBytes = kDataBytes + kScaleBytes;
// fp8 index cache: one 16 KB page of 128 tokens x 128 e4m3 bytes, no scales.
constexpr uint32_t kFp8PageBytes = 128 * 128;
// Every mbarrier wait gives up after this long (1 s; a test build of the
// library sets a shorter limit to make its stalled waits run out quickly).
#ifndef MX4_WAIT_LIMIT_NS
#define MX4_WAIT_LIMIT_NS 1000000000ull
#endif
constexpr uint64_t kWaitLimitNs = MX4_WAIT_LIMIT_NS;

static_assert(kTmemSfbCol + 4 * kSfbBufs <= kTmemCols, "TMEM budget");

// Instruction descriptor of kind::mxf8f6f4 with block scaling:
// A = E4M3 (0, bits 7..9), B = E2M1 (5, bits 10..12) for the MXFP4 cache or
// E4M3 (0) for the fp8 cache, both K-major, N >> 3 in bits 17..22, scale type
// UE8M0 (bit 23), M >> 4 in bits 24..28, B scale-factor id in bits 4..5, A
// scale-factor id in bits 29..30 (the id picks byte k of each 32-bit scale
// word for the k-th 32-element block).  The fp8 cache runs with unit scales
// on both sides.
template <bool kFp8>
__device__ __forceinline__ uint32_t idesc_for_k(uint32_t k)
{
    constexpr uint32_t kBase = (0u << 7) | ((kFp8 ? 0u : 5u) << 10) | ((128u >> 3) << 17) | (1u << 23) |
                               ((128u >> 4) << 24);
    return kBase | (k << 4) | (k << 29);
}

// Device status word of this module (MX4_DEV_* bits), ORed by the kernels
// and read back and cleared by the host.
__device__ unsigned int g_mx4_device_status;

struct ScoreParams {
    const void *q;
    const int32_t *block_table;
    const int32_t *cu_seqlens_q;   // prefill only
    const int32_t *seq_lens;
    const int32_t *prefix_lens;    // prefill only
    float *out;
    int64_t bt_stride;
    int64_t num_pool_pages;
    int64_t num_units;
    int64_t out_row_stride;        // floats per (row, head) line of out
    int num_seqs;
    int max_seq_len;
    int num_out_pages;
    int tiles_per_seq;
    int chunks_per_tile;
    int q_is_e4m3;
    float sm_scale;
};

// Shared memory carve-up (offsets from a 1024-aligned base).
struct SmemLayout {
    static constexpr uint32_t kData = 0;                                   // kStages x 16 KB
    static constexpr uint32_t kScale = kData + kStages * kTileBytes;       // kStages x 512 B
    static constexpr uint32_t kSfa = kScale + kStages * kScaleBytes;       // 512 B of 0x7F
    static constexpr uint32_t kOut = kSfa + kScaleBytes;                   // lanes x 128 x kChunk floats
    static constexpr uint32_t kBars = kOut + kLanes * 128 * kChunk * 4;
    // barriers: full[kStages], empty[kStages], dfull[kDBufs],
    //           dempty[kDBufs], qfull[2], qempty[2], final[kMmaWarps]
    static constexpr uint32_t kNumBars = 2 * kStages + 2 * kDBufs + 4 + kMmaWarps;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kAlloc = kEnd + 1024;                        // + alignment slack
};
static_assert(SmemLayout::kAlloc <= 227 * 1024, "shared memory budget");

// One tile: R query rows (R = 2 prefill, 1 decode) x 64 heads = 128 A rows.
struct TileInfo {
    int64_t tile;      // global tile id = b * tiles_per_seq + t (-1: none)
    int64_t row0;      // first global query row of the tile
    int b;
    int nrows;         // rows of the tile (0 = tile does not exist)
    int pos0;          // position of the tile's first row within its request
    int live_end;      // pages [0, live_end) hold a live token for some row
    int L[2];          // live limit of each row of the tile
};

template <bool kDecode>
__device__ __forceinline__ int live_limit(const ScoreParams &p, int b, int row_pos)
{
    int64_t seq = p.seq_lens[b];
    int64_t lim;
    if (kDecode) {
        lim = seq;
    } else {
        int64_t c = static_cast<int64_t>(p.prefix_lens[b]) + row_pos + 1;
        lim = c < seq ? c : seq;
    }
    if (lim > p.max_seq_len) lim = p.max_seq_len;
    if (lim < 0) lim = 0;
    return static_cast<int>(lim);
}

template <bool kDecode>
__device__ __forceinline__ TileInfo tile_info(const ScoreParams &p, int64_t tile)
{
    constexpr int R = kDecode ? 1 : 2;
    TileInfo ti;
    ti.tile = tile;
    ti.b = static_cast<int>(tile / p.tiles_per_seq);
    const int t = static_cast<int>(tile - static_cast<int64_t>(ti.b) * p.tiles_per_seq);
    if (kDecode) {
        ti.row0 = ti.b;
        ti.nrows = 1;
        ti.pos0 = 0;
    } else {
        const int qs = p.cu_seqlens_q[ti.b];
        const int ql = p.cu_seqlens_q[ti.b + 1] - qs;
        ti.pos0 = t * R;
        ti.nrows = ql - ti.pos0;
        if (ti.nrows > R) ti.nrows = R;
        if (ti.nrows < 0) ti.nrows = 0;
        ti.row0 = static_cast<int64_t>(qs) + ti.pos0;
    }
    ti.L[0] = ti.L[1] = 0;
    ti.live_end = 0;
    if (ti.nrows > 0) {
        ti.L[0] = live_limit<kDecode>(p, ti.b, ti.pos0);
        ti.L[1] = ti.nrows > 1 ? live_limit<kDecode>(p, ti.b, ti.pos0 + 1) : ti.L[0];
        const int Lmax = ti.L[0] > ti.L[1] ? ti.L[0] : ti.L[1];
        ti.live_end = (Lmax + kPage - 1) / kPage;
    }
    return ti;
}

// Wait sites, recorded as status bit (8 + site) when a wait gives up.
enum WaitSite : uint32_t {
    kSiteProducerEmpty = 0,
    kSiteMmaQFull = 1,
    kSiteMmaFull = 2,
    kSiteMmaDEmpty = 3,
    kSiteEpiQEmpty = 4,
    kSiteEpiDFull = 5,
    // 6..8: the attention kernel's wait sites
    kSiteDrain = 9,    // an armed copy had not landed when the CTA was leaving
};

#ifdef MX4_STALL_TEST
// Test build only (never in the product library): the waits at one site of
// one CTA treat their barrier as never completing, as if the arriving side had
// stalled, so that the time limit and the abort path can be exercised without
// hanging anything.  Set from the host by mx4_test_set_stall; site -1 = off.
__device__ int g_mx4_stall_site = -1;
__device__ int g_mx4_stall_cta = 0;
__device__ __forceinline__ bool stalled_here(uint32_t site)
{
    return static_cast<int>(site) == g_mx4_stall_site && static_cast<int>(blockIdx.x) == g_mx4_stall_cta;
}
// Whether some wait of this CTA is stalled (its fast probes are skipped).
__device__ __forceinline__ bool stall_in_cta()
{
    return g_mx4_stall_site >= 0 && static_cast<int>(blockIdx.x) == g_mx4_stall_cta;
}
// The waits that depend on a stalled one run out too, some of them having
// started earlier; they get four times the limit, so that the stalled site is
// the one the status word names.
__device__ __forceinline__ uint64_t wait_limit_ns(uint32_t site)
{
    return stall_in_cta() && !stalled_here(site) ? 4 * kWaitLimitNs : kWaitLimitNs;
}
#else
__device__ __forceinline__ constexpr bool stalled_here(uint32_t) { return false; }
__device__ __forceinline__ constexpr bool stall_in_cta() { return false; }
__device__ __forceinline__ constexpr uint64_t wait_limit_ns(uint32_t) { return kWaitLimitNs; }
#endif

// Bounded wait: true when the phase completed; false after the time limit or
// when another role has aborted (then the status word carries the reason:
// bit 1 = timeout, bit 8 + site = where the wait gave up).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                             uint32_t site)
{
    const bool stall = stalled_here(site);
    const uint64_t limit = wait_limit_ns(site);
    if (!stall && mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (!stall && mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit) {
            atomicOr(&g_mx4_device_status, 0x2u | (0x100u << site));
            *abort_flag = 1;
            return false;
        }
    }
}

// Wait for a copy this CTA armed to land before the CTA exits (its shared
// memory must not be written after that).  Bounded like every other wait;
// when it gives up, the status word records it (timeout + site 9), because a
// copy may then still be in flight.
__device__ __forceinline__ bool drain_bounded(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_mx4_device_status, 0x2u | (0x100u << kSiteDrain));
            return false;
        }
    }
    return true;
}

template <bool kDecode>
__device__ __forceinline__ bool tile_has_rows(const ScoreParams &p, int64_t tile)
{
    if (kDecode) return true;
    const int b = static_cast<int>(tile / p.tiles_per_seq);
    const int t = static_cast<int>(tile - static_cast<int64_t>(b) * p.tiles_per_seq);
    return p.cu_seqlens_q[b + 1] - p.cu_seqlens_q[b] > t * 2;
}

// Round this thread's query row (A row m = row m/64 of the tile, head m%64)
// to e4m3 and store it into TMEM lane m, 32 columns of 4 bytes (element 4c+i
// in byte i of column c).  Rows past the tile's end are zero.
template <bool kDecode>
__device__ __forceinline__ void load_q_tile_tmem(const ScoreParams &p, const TileInfo &ti, uint32_t taddr,
                                                 int m)
{
    const int ri = m / kHeads;
    const int h = m % kHeads;
    uint32_t w[32];
    if (ri < ti.nrows) {
        const int64_t line = (ti.row0 + ri) * kHeads + h;
        if (p.q_is_e4m3) {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.q) + line * kDim);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 x = __ldg(src + c);
                w[4 * c + 0] = x.x;
                w[4 * c + 1] = x.y;
                w[4 * c + 2] = x.z;
                w[4 * c + 3] = x.w;
            }
        } else {
            const uint4 *src =
                reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) + line * kDim);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint2 e = bf16x8_to_e4m3x8(__ldg(src + c));
                w[2 * c + 0] = e.x;
                w[2 * c + 1] = e.y;
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) w[c] = 0u;
    }
    tmem_st_32x32b_x32(taddr, w);
}

// Walks a CTA's contiguous unit range as (tile, chunk) without a division
// per unit.
struct UnitCursor {
    int64_t tile;
    int chunk;
    int64_t left;   // units remaining, this one included
};

__device__ __forceinline__ UnitCursor cursor_begin(const ScoreParams &p, int64_t u_begin, int64_t u_end)
{
    UnitCursor c;
    c.tile = u_begin / p.chunks_per_tile;
    c.chunk = static_cast<int>(u_begin - c.tile * p.chunks_per_tile);
    c.left = u_end - u_begin;
    return c;
}

__device__ __forceinline__ void cursor_next(const ScoreParams &p, UnitCursor &c)
{
    --c.left;
    if (++c.chunk == p.chunks_per_tile) {
        c.chunk = 0;
        ++c.tile;
    }
}

// Position in a ring of N slots and the parity of the slot's current use.
struct Ring {
    int idx = 0;
    uint32_t ph = 0;
};

template <int N>
__device__ __forceinline__ void ring_next(Ring &r)
{
    if (++r.idx == N) {
        r.idx = 0;
        r.ph ^= 1u;
    }
}

// Whose turn a unit is: the units of tiles with query rows go to the lanes
// in rotation.
struct LaneTurn {
    int next = 0;
    __device__ __forceinline__ bool take(int me)
    {
        const bool mine = next == me;
        next = next + 1 == kLanes ? 0 : next + 1;
        return mine;
    }
};

// MMA column n holds token 4*(n%32) + n/32.
__device__ __forceinline__ int token_of_col(int n) { return ((n & 31) << 2) | (n >> 5); }

// kFp8: the cache holds 128 e4m3 bytes per token (tmap_k is a UINT8 view of
// the same 4-D shape, tmap_s is unused); otherwise MXFP4 codes and scales.
template <bool kDecode, bool kLogits, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    mx4_score_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_s,
                     const __grid_constant__ ScoreParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Every role walks the same units in the same order; the units of tiles
    // with query rows go to the lanes in rotation.  Lane l's page stages
    // are l*kStagesPerLane.., its scale buffers l*kSfbPerLane.., its
    // accumulator l.
    auto bar = [&](int i) { return sbase + SmemLayout::kBars + 8u * i; };
    auto full_bar = [&](int i) { return bar(i); };
    auto empty_bar = [&](int i) { return bar(kStages + i); };
    auto dfull_bar = [&](int i) { return bar(2 * kStages + i); };
    auto dempty_bar = [&](int i) { return bar(2 * kStages + kDBufs + i); };
    auto qfull_bar = [&](int i) { return bar(2 * kStages + 2 * kDBufs + i); };
    auto qempty_bar = [&](int i) { return bar(2 * kStages + 2 * kDBufs + 2 + i); };
    auto final_bar = [&](int i) { return bar(2 * kStages + 2 * kDBufs + 4 + i); };
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + SmemLayout::kAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SmemLayout::kTmemSlot);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        for (int i = 0; i < kDBufs; ++i) {
            mbar_init(dfull_bar(i), 1);
            mbar_init(dempty_bar(i), 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull_bar(i), 4);
            mbar_init(qempty_bar(i), kMmaWarps);
        }
        for (int i = 0; i < kMmaWarps; ++i) mbar_init(final_bar(i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 128) {
        // unit scale for A: e8m0 byte 127 = 2^0 in every slot
        reinterpret_cast<uint32_t *>(smem + SmemLayout::kSfa)[threadIdx.x] = 0x7F7F7F7Fu;
        fence_proxy_async_smem();
    }
    if (warp == kLaneWarp0 && lane == 0) {
        prefetch_tmap(&tmap_k);
        if (!kFp8) prefetch_tmap(&tmap_s);
    }
    if (warp == kLaneWarp0) {
        tmem_alloc(sbase + SmemLayout::kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The set-up above touches no global memory, so under a programmatic
    // dependent launch it overlaps the previous kernel's last CTAs; every
    // global read and write comes after the wait.  The next kernel may start
    // its own set-up as this grid's CTAs retire.
    griddep_launch_dependents();
    griddep_wait();

    const int64_t u_begin = static_cast<int64_t>(blockIdx.x) * p.num_units / gridDim.x;
    const int64_t u_end = static_cast<int64_t>(blockIdx.x + 1) * p.num_units / gridDim.x;

    if (warp >= kLaneWarp0) {
        // -------------------------------------------- lane warps (TMA + MMA) --
        // Lane warp ln runs its lane's two page streams.  The TMA stream looks
        // up each page id in the block table (lane i of the warp holds the id
        // of the unit's i-th page, fetched one unit ahead so the lookup latency
        // overlaps the copies) and issues two TMA loads into the lane's smem
        // stage ring, kLookahead pages ahead of the MMA stream.  The MMA stream
        // copies the page's scales into a TMEM scale buffer (tcgen05.cp), issues
        // 4 block-scaled MMAs (K = 32 each) into the lane's accumulator and one
        // commit.  The tcgen05 operations of one thread run in issue order, so
        // the MMAs see the copied scales without a commit/wait in between.
        // Each page's TMA loads are issued right after the MMAs of the page
        // before it, into the stage that page's predecessor used: by then the
        // epilogue has read that predecessor's accumulator, so the stage is
        // free or about to be, and the copy stays off the MMA -> epilogue ->
        // MMA chain.
        const int ln = warp - kLaneWarp0;
        const uint64_t policy = kDecode ? l2_policy_evict_first() : l2_policy_evict_last();

        // next unit of this lane at or after c with live pages: tile info, first
        // page, page count; t rotates over the units with rows (it picks the lane)
        auto next_unit = [&](UnitCursor &c, TileInfo &t, LaneTurn &turn, int &j0, int &n) -> bool {
            for (; c.left > 0; cursor_next(p, c)) {
                if (c.tile != t.tile) t = tile_info<kDecode>(p, c.tile);
                if (t.nrows <= 0) continue;
                if (!turn.take(ln)) continue;
                j0 = c.chunk * kChunk;
                const int j1 = j0 + kChunk < p.num_out_pages ? j0 + kChunk : p.num_out_pages;
                const int jc = j1 < t.live_end ? j1 : t.live_end;
                n = jc - j0;
                if (n > 0) return true;
            }
            return false;
        };
        // Start the load of the ids of pages j0 .. j0+n-1 (n >= 1) of tile t's
        // request into lane i's `raw`.  Lanes past n re-read the last id, so the
        // load is unconditional: nothing here consumes the value and the warp
        // does not wait for it.
        auto fetch_id = [&](const TileInfo &t, int j0, int n, int &raw) {
            raw = p.block_table[static_cast<int64_t>(t.b) * p.bt_stride + j0 + (lane < n ? lane : n - 1)];
        };
        // First use of a fetched id (one unit later): range check.
        auto checked_id = [&](int raw, int n) -> int {
            int pid = 0;
            if (lane < n) {
                if (raw < 0 || raw >= p.num_pool_pages)
                    atomicOr(&g_mx4_device_status, 0x1u);
                else
                    pid = raw;
            }
            return pid;
        };

        // TMA stream state: current unit (cursor, tile, turn, pages) and the
        // prefetched next one
        UnitCursor tc_cur = cursor_begin(p, u_begin, u_end);
        TileInfo tc_ti;
        tc_ti.tile = -1;
        LaneTurn tc_turn;
        int tc_j0 = 0, tc_n = 0, tc_i = 0;
        bool tc_have = next_unit(tc_cur, tc_ti, tc_turn, tc_j0, tc_n);
        int tc_raw = 0;
        if (tc_have) fetch_id(tc_ti, tc_j0, tc_n, tc_raw);
        int tc_pid = checked_id(tc_raw, tc_n);
        UnitCursor nx_cur = tc_cur;
        TileInfo nx_ti = tc_ti;
        LaneTurn nx_turn = tc_turn;
        int nx_j0 = 0, nx_n = 0;
        bool nx_have = false;
        int nx_raw = 0;
        auto prefetch_next = [&]() {
            nx_cur = tc_cur;
            cursor_next(p, nx_cur);
            nx_ti = tc_ti;
            nx_turn = tc_turn;
            nx_have = next_unit(nx_cur, nx_ti, nx_turn, nx_j0, nx_n);
            if (nx_have) fetch_id(nx_ti, nx_j0, nx_n, nx_raw);
        };
        if (tc_have) prefetch_next();
        Ring pst;
        // issue the TMA stream's next page (if any); false on abort
        // Issue the TMA stream's next page into its stage, which the caller
        // has seen free, and advance the stream.
        auto issue_page = [&]() {
            const int id = __shfl_sync(0xffffffffu, tc_pid, tc_i);
            const int stage = ln * kStagesPerLane + pst.idx;
            if (elect_one()) {
                mbar_arrive_expect_tx(full_bar(stage), kFp8 ? kFp8PageBytes : kStageTxBytes);
                tma_load_4d(sbase + SmemLayout::kData + stage * kTileBytes, &tmap_k, full_bar(stage), 0, 0, 0, id,
                            policy);
                if (!kFp8)
                    tma_load_2d(sbase + SmemLayout::kScale + stage * kScaleBytes, &tmap_s, full_bar(stage), 0, id,
                                policy);
            }
            __syncwarp();
            ring_next<kStagesPerLane>(pst);
            if (++tc_i == tc_n) {
                tc_cur = nx_cur;
                tc_ti = nx_ti;
                tc_turn = nx_turn;
                tc_j0 = nx_j0;
                tc_n = nx_n;
                tc_have = nx_have;
                tc_i = 0;
                tc_pid = checked_id(nx_raw, tc_n);
                if (tc_have) prefetch_next();
            }
        };
        // Wait (bounded) for the next page's stage, then issue it; false on abort.
        auto issue_next_page = [&]() -> bool {
            if (!tc_have) return true;
            if (!__all_sync(0xffffffffu, wait_bounded(empty_bar(ln * kStagesPerLane + pst.idx), pst.ph ^ 1u,
                                                      abort_flag, kSiteProducerEmpty)))
                return false;
            issue_page();
            return true;
        };

        // this warp's copy of the unit scale of A (e8m0 127 everywhere)
        const uint32_t tmem_sfa = tmem_base + kTmemSfaCol + 4u * ln;
        if (elect_one()) tc_cp_32x128b_warpx4(tmem_sfa, smem_desc(sbase + SmemLayout::kSfa, 16, 128, 0));
        __syncwarp();
        const uint64_t bdesc0 = smem_desc(sbase + SmemLayout::kData, 16, 1024, 2);
        const uint64_t sdesc0 = smem_desc(sbase + SmemLayout::kScale, 16, 128, 0);
        const uint32_t d_tmem = tmem_base + ln * 128u;
        bool ok = true;
        for (int i = 0; i < kLookahead && ok; ++i) ok = issue_next_page();
        Ring st, sf, dr;
        int64_t qcount = 0;
        LaneTurn uc;
        uint32_t a_tmem = tmem_base + kTmemACol;
        TileInfo ti;
        ti.tile = -1;
        bool holding_q = false;
        for (UnitCursor c = cursor_begin(p, u_begin, u_end); c.left > 0 && ok; cursor_next(p, c)) {
            if (c.tile != ti.tile) {
                ti = tile_info<kDecode>(p, c.tile);
                if (ti.nrows > 0) {
                    // the previous query tile's buffer is free once its MMAs retire
                    if (holding_q && elect_one()) tc_commit(qempty_bar(static_cast<int>((qcount - 1) & 1)));
                    __syncwarp();
                    const int64_t qi = qcount++;
                    a_tmem = tmem_base + kTmemACol + static_cast<uint32_t>(qi & 1) * 32u;
                    holding_q = true;
                    if (!__all_sync(0xffffffffu, wait_bounded(qfull_bar(static_cast<int>(qi & 1)),
                                                              static_cast<uint32_t>((qi >> 1) & 1), abort_flag,
                                                              kSiteMmaQFull))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
            }
            if (ti.nrows <= 0) continue;
            if (!uc.take(ln)) continue;
            const int j0 = c.chunk * kChunk;
            const int j1 = j0 + kChunk < p.num_out_pages ? j0 + kChunk : p.num_out_pages;
            const int jc = j1 < ti.live_end ? j1 : ti.live_end;
            for (int j = j0; j < jc; ++j) {
                const int stage = ln * kStagesPerLane + st.idx;
                const int sfb = ln * kSfbPerLane + sf.idx;
                // The page's bytes, a free accumulator and, when the TMA stream
                // has a page left, a free stage for it (released when the MMAs
                // of the page before this one completed): one probe round trip
                // when all are ready, bounded waits otherwise.
                const bool tma_next = tc_have;
                const uint32_t e_bar = empty_bar(ln * kStagesPerLane + pst.idx);
                const uint32_t e_par = pst.ph ^ 1u;
                const bool ready = !stall_in_cta() &&
                                   (tma_next ? mbar_try_wait3(full_bar(stage), st.ph, dempty_bar(ln), dr.ph ^ 1u,
                                                              e_bar, e_par)
                                             : mbar_try_wait2(full_bar(stage), st.ph, dempty_bar(ln), dr.ph ^ 1u));
                if (!__all_sync(0xffffffffu, ready) &&
                    !__all_sync(0xffffffffu,
                                wait_bounded(full_bar(stage), st.ph, abort_flag, kSiteMmaFull) &&
                                    wait_bounded(dempty_bar(ln), dr.ph ^ 1u, abort_flag, kSiteMmaDEmpty) &&
                                    (!tma_next || wait_bounded(e_bar, e_par, abort_flag, kSiteProducerEmpty)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    // fp8 pages carry no scales: B uses the unit scales of A
                    uint32_t tmem_sfb = tmem_sfa;
                    if (!kFp8) {
                        tmem_sfb = tmem_base + kTmemSfbCol + 4u * sfb;
                        // descriptor start addresses count 16-byte units
                        tc_cp_32x128b_warpx4(tmem_sfb, sdesc0 + static_cast<uint64_t>(stage * (kScaleBytes >> 4)));
                    }
                    const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(stage * (kTileBytes >> 4));
                    // K block k: +32 bytes of B (2 units of 16 B), +8 TMEM columns of A
                    tc_mma_mx_ts(d_tmem, a_tmem, bdesc, idesc_for_k<kFp8>(0), tmem_sfa, tmem_sfb, 0u);
                    tc_mma_mx_ts(d_tmem, a_tmem + 8u, bdesc + 2, idesc_for_k<kFp8>(1), tmem_sfa, tmem_sfb, 1u);
                    tc_mma_mx_ts(d_tmem, a_tmem + 16u, bdesc + 4, idesc_for_k<kFp8>(2), tmem_sfa, tmem_sfb, 1u);
                    tc_mma_mx_ts(d_tmem, a_tmem + 24u, bdesc + 6, idesc_for_k<kFp8>(3), tmem_sfa, tmem_sfb, 1u);
                    tc_commit(dfull_bar(ln));
                }
                __syncwarp();
                ring_next<kStagesPerLane>(st);
                ring_next<kSfbPerLane>(sf);
                ring_next<1>(dr);
                if (tma_next) issue_page();
            }
        }
        // Do not leave while copies into this CTA's smem may be in flight:
        // every armed stage of this lane completes (bounded) before the CTA
        // exits; then all MMAs retire before TMEM is released.
        if (lane == 0) {
            for (int i = 0; i < kStagesPerLane; ++i) {
                // stages before pst.idx were armed in phase ph, the others in ph^1 (if ever)
                const uint32_t par = (i < pst.idx) ? pst.ph : (pst.ph ^ 1u);
                if (!drain_bounded(full_bar(ln * kStagesPerLane + i), par)) break;
            }
        }
        __syncwarp();
        if (elect_one()) tc_commit(final_bar(ln));
        __syncwarp();
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(final_bar(ln), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue --
        // Warpgroup `set` (warps 4*set .. 4*set+3) reads lane `set`'s
        // accumulator; warpgroup 0 also loads the query tiles.
        const int set = warp / 4;
        const int quad = warp % 4;
        const int m = quad * 32 + lane;            // A row / TMEM lane 0..127
        const int ri = m / kHeads;                 // row within the tile
        const int h = m % kHeads;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t d_taddr = tmem_base + lane_addr + set * 128u;
        // this thread's staged page maxima of the current unit, page-major
        // (page i of the unit at stg[128 i]): the per-page stores of a warp
        // fill 32 consecutive words, free of bank conflicts
        float *stg = reinterpret_cast<float *>(smem + SmemLayout::kOut) + set * 128 * kChunk + m;
        const float sm_scale = p.sm_scale;
        Ring dr;
        int st_idx = 0;
        int64_t qcount = 0;
        LaneTurn uc;
        TileInfo ti;
        ti.tile = -1;

        // Load the query tile of `t` into A buffer qi & 1 once the MMAs of the
        // tile that used that buffer before have retired (warpgroup 0 only).
        auto q_load = [&](const TileInfo &t, int64_t qi) -> bool {
            const int buf = static_cast<int>(qi & 1);
            // warp-uniform outcome, so the .sync.aligned operations below never diverge
            if (!__all_sync(0xffffffffu, wait_bounded(qempty_bar(buf), static_cast<uint32_t>(((qi >> 1) & 1) ^ 1),
                                                      abort_flag, kSiteEpiQEmpty)))
                return false;
            tc_fence_after();
            load_q_tile_tmem<kDecode>(p, t, tmem_base + lane_addr + kTmemACol + buf * 32u, m);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(qfull_bar(buf));
            return true;
        };

        bool ok = true;
        for (UnitCursor c = cursor_begin(p, u_begin, u_end);
             c.left > 0 && ok && !__any_sync(0xffffffffu, *abort_flag != 0); cursor_next(p, c)) {
            if (c.tile != ti.tile) {
                const TileInfo nt_info = tile_info<kDecode>(p, c.tile);
                if (nt_info.nrows <= 0) continue;   // keeps ti: units of this tile are skipped below
                ti = nt_info;
                if (set == 0) {
                    if (qcount == 0 && !q_load(ti, 0)) break;
                    const int64_t qi = qcount++;
                    // prefetch the next tile with rows in this CTA's range
                    int64_t nt = c.tile + 1;
                    while (nt * p.chunks_per_tile < u_end && !tile_has_rows<kDecode>(p, nt)) ++nt;
                    if (nt * p.chunks_per_tile < u_end) {
                        if (!q_load(tile_info<kDecode>(p, nt), qi + 1)) break;
                    }
                }
            }
            if (!uc.take(set)) continue;
            const int j0 = c.chunk * kChunk;
            const int j1 = j0 + kChunk < p.num_out_pages ? j0 + kChunk : p.num_out_pages;
            const bool has_row = ri < ti.nrows;     // uniform per warp
            const int L = has_row ? (ri == 0 ? ti.L[0] : ti.L[1]) : 0;
            const int64_t line = (ti.row0 + ri) * kHeads + h;
            float *row_out = p.out + line * p.out_row_stride;
            for (int j = j0; j < j1; ++j) {
                const int lim = L - j * kPage;   // live tokens of page j for this row
                if (j < ti.live_end) {
                    if (!__all_sync(0xffffffffu, wait_bounded(dfull_bar(set), dr.ph, abort_flag, kSiteEpiDFull))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the page's MMAs have completed, so its smem stage can be
                    // refilled at once
                    if (quad == 0 && lane == 0) mbar_arrive(empty_bar(set * kStagesPerLane + st_idx));
                    if (++st_idx == kStagesPerLane) st_idx = 0;
                    if (has_row) {
                        // the accumulator is read in two 64-column halves (15
                        // warps per CTA leave 128 registers per thread)
                        uint32_t v[64];
                        if (!kLogits) {
                            float mx;
                            if (lim >= kPage) {
                                // a rolled loop: the two loads reuse one set of
                                // destination registers
                                mx = -INFINITY;
#pragma unroll 1
                                for (int hh = 0; hh < 2; ++hh)
                                    mx = fmaxf(mx, tmem_ld_max_32x32b_x64(d_taddr + 64u * hh, v));
                            } else {
                                mx = -INFINITY;
#pragma unroll
                                for (int hh = 0; hh < 2; ++hh) {
                                    tmem_ld_32x32b_x64(d_taddr + 64u * hh, v);
#pragma unroll
                                    for (int n = 0; n < 64; ++n)
                                        if (token_of_col(64 * hh + n) < lim) mx = fmaxf(mx, __uint_as_float(v[n]));
                                }
                            }
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(dempty_bar(set));
                            stg[128 * (j - j0)] = mx * sm_scale;
                        } else {
                            float *dst = row_out + static_cast<int64_t>(j) * kPage;
                            const int valid = p.max_seq_len - j * kPage;   // columns that exist
                            const bool vec = (p.out_row_stride & 1) == 0 && valid >= kPage;
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                tmem_ld_32x32b_x64(d_taddr + 64u * hh, v);
                                if (hh == 1) {
                                    tc_fence_before();
                                    __syncwarp();
                                    if (lane == 0) mbar_arrive(dempty_bar(set));
                                }
                                // column 64hh + g holds token 4g + 2hh, column
                                // 64hh + 32 + g token 4g + 2hh + 1
#pragma unroll
                                for (int g = 0; g < 32; ++g) {
                                    const int t0 = 4 * g + 2 * hh;
                                    float2 o;
                                    o.x = (t0 < lim) ? __uint_as_float(v[g]) * sm_scale : -INFINITY;
                                    o.y = (t0 + 1 < lim) ? __uint_as_float(v[g + 32]) * sm_scale : -INFINITY;
                                    if (vec) {
                                        __stcs(reinterpret_cast<float2 *>(dst + t0), o);
                                    } else {
                                        if (t0 < valid) dst[t0] = o.x;
                                        if (t0 + 1 < valid) dst[t0 + 1] = o.y;
                                    }
                                }
                            }
                        }
                    } else {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(dempty_bar(set));
                    }
                    ring_next<1>(dr);
                } else if (has_row) {
                    // no row of the tile sees this page: nothing was computed
                    if (!kLogits) {
                        stg[128 * (j - j0)] = -INFINITY;
                    } else {
                        float *dst = row_out + static_cast<int64_t>(j) * kPage;
                        const int valid = p.max_seq_len - j * kPage;
                        for (int cc = 0; cc < kPage && cc < valid; ++cc) dst[cc] = -INFINITY;
                    }
                }
            }
            if (!ok) break;
            if (!kLogits && has_row) {
                // the whole unit (up to 8 pages, one 32-byte sector) at once
                float *dst = row_out + j0;
                const int n = j1 - j0;
                if (n == kChunk && (p.out_row_stride & 3) == 0) {
                    __stcs(reinterpret_cast<float4 *>(dst), make_float4(stg[0], stg[128], stg[256], stg[384]));
                    __stcs(reinterpret_cast<float4 *>(dst) + 1, make_float4(stg[512], stg[640], stg[768], stg[896]));
                } else if (n == kChunk && (p.out_row_stride & 1) == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        __stcs(reinterpret_cast<float2 *>(dst) + i, make_float2(stg[256 * i], stg[256 * i + 128]));
                } else {
                    for (int i = 0; i < n; ++i) dst[i] = stg[128 * i];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kLaneWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Standalone query preparation: bf16 -> e4m3, 8 values per thread-step.
// `vec` = 1 when in is 16-byte and out 8-byte aligned.
__global__ void mx4_quantize_q_kernel(const uint16_t *__restrict__ in, uint8_t *__restrict__ out, int64_t n,
                                      int vec)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t n8 = vec ? n / 8 : 0;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8; i += stride) {
        const uint4 x = reinterpret_cast<const uint4 *>(in)[i];
        reinterpret_cast<uint2 *>(out)[i] = bf16x8_to_e4m3x8(x);
    }
    for (int64_t i = n8 * 8 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
        const float f = __uint_as_float(static_cast<uint32_t>(in[i]) << 16);
        out[i] = static_cast<uint8_t>(f32x2_to_e4m3x2(f, 0.0f) & 0xFF);
    }
}

}  // namespace mx4
