// score_kernel.cuh -- the paged MXFP4 index-K scorer kernel for sm_103a.
//
// One persistent CTA per SM walks a contiguous range of work units.  A unit
// is (request, tile of query rows, chunk of kChunk pages).  A tile is R query
// rows x 64 heads = 128 rows of the MMA A operand (R = 2 for prefill, 1 for
// decode, where lanes 64..127 stay zero).
//
// Roles (warp-specialised, 192 threads):
//   warps 0-3  epilogue: load Q (bf16 -> e4m3 in registers) into a swizzled
//              smem A tile; per page read the fp32 accumulator from TMEM,
//              apply the causal mask, take the page max (or emit per-token
//              logits), scale by sm_scale and store.
//   warp 4     producer: per live page, look up the physical page id in the
//              block table and issue two TMA loads: the 8 KB of e2m1 codes
//              (unpacked in flight to the 16 KB padded layout the tensor core
//              reads) and the 512 B of e8m0 scales.
//   warp 5     MMA issuer: copies the page's scales into TMEM (tcgen05.cp)
//              and issues 4 block-scaled MMAs (K = 32 each) of
//              kind::mxf8f6f4: A = Q (e4m3, unit scale), B = K page (e2m1 with
//              its e8m0 bytes), D = 128 x 128 fp32 in TMEM.
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
constexpr int kTileBytes = 128 * 128;           // one 128 x 128 operand tile in smem (8-bit slots)
constexpr int kStages = 8;                      // smem pipeline depth (pages in flight)
constexpr int kDBufs = 3;                       // TMEM accumulator buffers
constexpr int kSfbBufs = 4;                     // TMEM scale-factor buffers for B
constexpr int kChunk = 8;                       // pages per work unit
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSfaCol = kDBufs * 128;          // 384
constexpr uint32_t kTmemSfbCol = kTmemSfaCol + 4;       // 388
// Transaction bytes of one page: the 4-bit TMA load counts the packed
// global bytes (8192), not the 16 KB it writes in the padded smem form.
constexpr uint32_t kStageTxBytes = kDataBytes + kScaleBytes;
constexpr uint64_t kWaitLimitNs = 1000000000ull;        // 1 s per wait

// Instruction descriptor of kind::mxf8f6f4 with block scaling:
// A = E4M3 (0, bits 7..9), B = E2M1 (5, bits 10..12), both K-major,
// N >> 3 in bits 17..22, scale type UE8M0 (bit 23), M >> 4 in bits 24..28,
// B scale-factor id in bits 4..5, A scale-factor id in bits 29..30.
constexpr uint32_t kIdescBase = (0u << 7) | (5u << 10) | ((128u >> 3) << 17) | (1u << 23) |
                                ((128u >> 4) << 24);

__device__ __forceinline__ uint32_t idesc_for_k(uint32_t k) { return kIdescBase | (k << 4) | (k << 29); }

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
    static constexpr uint32_t kQ = kData + kStages * kTileBytes;           // 2 x 16 KB
    static constexpr uint32_t kScale = kQ + 2 * kTileBytes;                // kStages x 512 B
    static constexpr uint32_t kSfa = kScale + kStages * kScaleBytes;       // 512 B of 0x7F
    static constexpr uint32_t kStage = kSfa + kScaleBytes;                 // 128 x kChunk floats
    static constexpr uint32_t kBars = kStage + 128 * kChunk * 4;
    // barriers: full[kStages], empty[kStages], dfull[kDBufs], dempty[kDBufs],
    //           qfull[2], qempty[2], final
    static constexpr uint32_t kNumBars = 2 * kStages + 2 * kDBufs + 4 + 1;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kEnd = kAbort + 4;
    static constexpr uint32_t kAlloc = kEnd + 1024;                        // + alignment slack
};

struct Unit {
    int64_t tile;      // global tile id = b * tiles_per_seq + t
    int64_t row0;      // first global query row of the tile
    int b;
    int nrows;         // rows of the tile (0 = tile does not exist)
    int pos0;          // position of the tile's first row within its request
    int j0, j1;        // page range of the unit [j0, j1)
    int live_end;      // pages [0, live_end) hold a live token for some row
    int L0;            // live limit of the tile's first row
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
__device__ __forceinline__ Unit decode_unit(const ScoreParams &p, int64_t u)
{
    constexpr int R = kDecode ? 1 : 2;
    Unit w;
    w.tile = u / p.chunks_per_tile;
    const int chunk = static_cast<int>(u - w.tile * p.chunks_per_tile);
    w.b = static_cast<int>(w.tile / p.tiles_per_seq);
    const int t = static_cast<int>(w.tile - static_cast<int64_t>(w.b) * p.tiles_per_seq);
    int first_pos;
    if (kDecode) {
        w.row0 = w.b;
        w.nrows = 1;
        first_pos = 0;
    } else {
        const int qs = p.cu_seqlens_q[w.b];
        const int ql = p.cu_seqlens_q[w.b + 1] - qs;
        first_pos = t * R;
        w.nrows = ql - first_pos;
        if (w.nrows > R) w.nrows = R;
        if (w.nrows < 0) w.nrows = 0;
        w.row0 = static_cast<int64_t>(qs) + first_pos;
    }
    w.pos0 = first_pos;
    w.j0 = chunk * kChunk;
    w.j1 = w.j0 + kChunk < p.num_out_pages ? w.j0 + kChunk : p.num_out_pages;
    if (w.nrows > 0) {
        w.L0 = live_limit<kDecode>(p, w.b, first_pos);
        const int Llast = live_limit<kDecode>(p, w.b, first_pos + w.nrows - 1);
        w.live_end = (Llast + kPage - 1) / kPage;
    } else {
        w.L0 = 0;
        w.live_end = 0;
    }
    return w;
}

// Wait sites, recorded as status bit (8 + site) when a wait gives up.
enum WaitSite : uint32_t {
    kSiteProducerEmpty = 0,
    kSiteMmaQFull = 1,
    kSiteMmaFull = 2,
    kSiteMmaDEmpty = 3,
    kSiteEpiQEmpty = 4,
    kSiteEpiDFull = 5,
};

// Bounded wait: true when the phase completed; false after the time limit or
// when another role has aborted (then the status word carries the reason:
// bit 1 = timeout, bit 8 + site = where the wait gave up).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                             unsigned int *status, uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, 0x2u | (0x100u << site));
            *abort_flag = 1;
            return false;
        }
    }
}

template <bool kDecode>
__device__ __forceinline__ bool tile_has_rows(const ScoreParams &p, int64_t tile)
{
    if (kDecode) return true;
    const int b = static_cast<int>(tile / p.tiles_per_seq);
    const int t = static_cast<int>(tile - static_cast<int64_t>(b) * p.tiles_per_seq);
    return p.cu_seqlens_q[b + 1] - p.cu_seqlens_q[b] > t * 2;
}

// Write one tile of Q (R rows x 64 heads, rounded to e4m3) into the swizzled
// K-major smem A layout: row m at (m/8)*1024 + (m%8)*128, 16-byte chunk c
// stored at chunk position c ^ (m%8).  Thread m owns A row m.
template <bool kDecode>
__device__ __forceinline__ void load_q_tile(const ScoreParams &p, int64_t tile, uint8_t *qbuf, int m)
{
    constexpr int R = kDecode ? 1 : 2;
    const int b = static_cast<int>(tile / p.tiles_per_seq);
    const int t = static_cast<int>(tile - static_cast<int64_t>(b) * p.tiles_per_seq);
    int64_t row0;
    int nrows;
    if (kDecode) {
        row0 = b;
        nrows = 1;
    } else {
        const int qs = p.cu_seqlens_q[b];
        const int ql = p.cu_seqlens_q[b + 1] - qs;
        nrows = ql - t * R;
        if (nrows > R) nrows = R;
        row0 = static_cast<int64_t>(qs) + t * R;
    }
    const int ri = m / kHeads;
    const int h = m % kHeads;
    uint4 chunks[8];
    if (ri < nrows) {
        const int64_t line = (row0 + ri) * kHeads + h;
        if (p.q_is_e4m3) {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.q) + line * kDim);
#pragma unroll
            for (int c = 0; c < 8; ++c) chunks[c] = __ldg(src + c);
        } else {
            const uint4 *src =
                reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.q) + line * kDim);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint2 lo = bf16x8_to_e4m3x8(__ldg(src + 2 * c));
                const uint2 hi = bf16x8_to_e4m3x8(__ldg(src + 2 * c + 1));
                chunks[c] = make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) chunks[c] = make_uint4(0, 0, 0, 0);
    }
    uint8_t *row = qbuf + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(row + ((c ^ (m & 7)) << 4)) = chunks[c];
}

__device__ __forceinline__ float fmax3(float a, float b, float c) { return fmaxf(a, fmaxf(b, c)); }

// MMA column n holds token 4*(n%32) + n/32.
__device__ __forceinline__ int token_of_col(int n) { return ((n & 31) << 2) | (n >> 5); }

template <bool kDecode, bool kLogits>
__global__ void __launch_bounds__(kThreads, 1)
    mx4_score_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_s,
                     const __grid_constant__ ScoreParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto bar = [&](int i) { return sbase + SmemLayout::kBars + 8u * i; };
    auto full_bar = [&](int s) { return bar(s); };
    auto empty_bar = [&](int s) { return bar(kStages + s); };
    auto dfull_bar = [&](int d) { return bar(2 * kStages + d); };
    auto dempty_bar = [&](int d) { return bar(2 * kStages + kDBufs + d); };
    auto qfull_bar = [&](int q) { return bar(2 * kStages + 2 * kDBufs + q); };
    auto qempty_bar = [&](int q) { return bar(2 * kStages + 2 * kDBufs + 2 + q); };
    const uint32_t final_bar = bar(2 * kStages + 2 * kDBufs + 4);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + SmemLayout::kAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SmemLayout::kTmemSlot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int d = 0; d < kDBufs; ++d) {
            mbar_init(dfull_bar(d), 1);
            mbar_init(dempty_bar(d), 4);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(qfull_bar(q), 4);
            mbar_init(qempty_bar(q), 1);
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < 128) {
        // unit scale for A: e8m0 byte 127 = 2^0 in every slot
        reinterpret_cast<uint32_t *>(smem + SmemLayout::kSfa)[threadIdx.x] = 0x7F7F7F7Fu;
        fence_proxy_async_smem();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_s);
    }
    if (warp == 5) {
        tmem_alloc(sbase + SmemLayout::kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int64_t u_begin = static_cast<int64_t>(blockIdx.x) * p.num_units / gridDim.x;
    const int64_t u_end = static_cast<int64_t>(blockIdx.x + 1) * p.num_units / gridDim.x;

    if (warp == 4) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int64_t u = u_begin; u < u_end && !*abort_flag; ++u) {
                const Unit w = decode_unit<kDecode>(p, u);
                if (w.nrows <= 0) continue;
                const int jc = w.j1 < w.live_end ? w.j1 : w.live_end;
                for (int j = w.j0; j < jc; ++j) {
                    int64_t pid = p.block_table[static_cast<int64_t>(w.b) * p.bt_stride + j];
                    if (pid < 0 || pid >= p.num_pool_pages) {
                        atomicOr(&g_mx4_device_status, 0x1u);
                        pid = 0;
                    }
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, &g_mx4_device_status, kSiteProducerEmpty)) break;
                    mbar_arrive_expect_tx(full_bar(s), kStageTxBytes);
                    tma_load_4d(sbase + SmemLayout::kData + s * kTileBytes, &tmap_k, full_bar(s), 0, 0, 0,
                                static_cast<int>(pid));
                    tma_load_2d(sbase + SmemLayout::kScale + s * kScaleBytes, &tmap_s, full_bar(s), 0,
                                static_cast<int>(pid));
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Do not leave while copies into this CTA's smem may be in flight:
            // every armed stage completes (bounded) before the CTA exits.
            for (int i = 0; i < kStages; ++i) {
                // stages < s were armed in phase ph, the others in ph^1 (if ever)
                const uint32_t par = (i < s) ? ph : (ph ^ 1u);
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(full_bar(i), par) && globaltimer_ns() - t0 < 2000000ull) {
                }
            }
        }
    } else if (warp == 5) {
        // ----------------------------------------------------- MMA issuer --
        if (lane == 0) {
            const uint32_t tmem_sfa = tmem_base + kTmemSfaCol;
            tc_cp_32x128b_warpx4(tmem_sfa, smem_desc(sbase + SmemLayout::kSfa, 16, 128, 0));
            int s = 0, d = 0, x = 0;
            uint32_t ph = 0, dph = 0;
            int64_t cur_tile = -1, qcount = 0;
            uint32_t qbuf = 0;
            for (int64_t u = u_begin; u < u_end && !*abort_flag; ++u) {
                const Unit w = decode_unit<kDecode>(p, u);
                if (w.nrows <= 0) continue;
                if (w.tile != cur_tile) {
                    if (cur_tile >= 0) tc_commit(qempty_bar(static_cast<int>((qcount - 1) & 1)));
                    cur_tile = w.tile;
                    const int64_t qi = qcount++;
                    qbuf = static_cast<uint32_t>(qi & 1);
                    if (!wait_bounded(qfull_bar(qbuf), static_cast<uint32_t>((qi >> 1) & 1), abort_flag, &g_mx4_device_status,
                                      kSiteMmaQFull))
                        break;
                    tc_fence_after();
                }
                const int jc = w.j1 < w.live_end ? w.j1 : w.live_end;
                bool ok = true;
                for (int j = w.j0; j < jc; ++j) {
                    if (!wait_bounded(full_bar(s), ph, abort_flag, &g_mx4_device_status, kSiteMmaFull) ||
                        !wait_bounded(dempty_bar(d), dph ^ 1u, abort_flag, &g_mx4_device_status, kSiteMmaDEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tmem_sfb = tmem_base + kTmemSfbCol + 4u * x;
                    tc_cp_32x128b_warpx4(tmem_sfb, smem_desc(sbase + SmemLayout::kScale + s * kScaleBytes, 16, 128, 0));
                    const uint32_t a_addr = sbase + SmemLayout::kQ + qbuf * kTileBytes;
                    const uint32_t b_addr = sbase + SmemLayout::kData + s * kTileBytes;
                    const uint32_t d_tmem = tmem_base + d * 128u;
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k) {
                        tc_mma_mx_ss(d_tmem, smem_desc(a_addr + 32u * k, 16, 1024, 2),
                                     smem_desc(b_addr + 32u * k, 16, 1024, 2), idesc_for_k(k), tmem_sfa, tmem_sfb,
                                     k > 0 ? 1u : 0u);
                    }
                    tc_commit(empty_bar(s));
                    tc_commit(dfull_bar(d));
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++d == kDBufs) {
                        d = 0;
                        dph ^= 1u;
                    }
                    if (++x == kSfbBufs) x = 0;
                }
                if (!ok) break;
            }
            // all MMAs and copies retire before TMEM is released
            tc_commit(final_bar);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(final_bar, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue --
        const int m = threadIdx.x;                 // A row / TMEM lane 0..127
        const int ri = m / kHeads;                 // row within the tile
        const int h = m % kHeads;
        const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
        float *stage = reinterpret_cast<float *>(smem + SmemLayout::kStage) + m * kChunk;
        const float sm_scale = p.sm_scale;
        int d = 0;
        uint32_t dph = 0;
        int64_t cur_tile = -1, qcount = 0;

        auto q_load = [&](int64_t tile, int64_t qi) -> bool {
            const int buf = static_cast<int>(qi & 1);
            // warp-uniform outcome, so the .sync.aligned operations below never diverge
            if (!__all_sync(0xffffffffu, wait_bounded(qempty_bar(buf), static_cast<uint32_t>(((qi >> 1) & 1) ^ 1),
                                                      abort_flag, &g_mx4_device_status, kSiteEpiQEmpty)))
                return false;
            load_q_tile<kDecode>(p, tile, smem + SmemLayout::kQ + buf * kTileBytes, m);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qfull_bar(buf));
            return true;
        };

        for (int64_t u = u_begin; u < u_end && !__any_sync(0xffffffffu, *abort_flag != 0); ++u) {
            const Unit w = decode_unit<kDecode>(p, u);
            if (w.nrows <= 0) continue;
            if (w.tile != cur_tile) {
                if (qcount == 0 && !q_load(w.tile, 0)) break;
                cur_tile = w.tile;
                const int64_t qi = qcount++;
                // prefetch the next tile with rows in this CTA's range
                int64_t nt = w.tile + 1;
                while (nt * p.chunks_per_tile < u_end && !tile_has_rows<kDecode>(p, nt)) ++nt;
                if (nt * p.chunks_per_tile < u_end) {
                    if (!q_load(nt, qi + 1)) break;
                }
            }
            const bool has_row = ri < w.nrows;
            const int L = has_row ? (ri == 0 ? w.L0 : live_limit<kDecode>(p, w.b, w.pos0 + ri)) : 0;
            const int64_t line = (w.row0 + ri) * kHeads + h;
            bool ok = true;
            for (int j = w.j0; j < w.j1; ++j) {
                const int lim = L - j * kPage;   // live tokens of page j for this row
                if (j < w.live_end) {
                    if (!__all_sync(0xffffffffu, wait_bounded(dfull_bar(d), dph, abort_flag, &g_mx4_device_status, kSiteEpiDFull))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t v[128];
                    tmem_ld_32x32b_x128(tmem_base + lane_addr + d * 128u, v);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dempty_bar(d));
                    if (++d == kDBufs) {
                        d = 0;
                        dph ^= 1u;
                    }
                    if (!has_row) continue;
                    if (!kLogits) {
                        float mx;
                        if (lim >= kPage) {
                            float a = __uint_as_float(v[0]), b2 = __uint_as_float(v[1]);
#pragma unroll
                            for (int n = 2; n < 128; n += 2) {
                                a = fmaxf(a, __uint_as_float(v[n]));
                                b2 = fmaxf(b2, __uint_as_float(v[n + 1]));
                            }
                            mx = fmaxf(a, b2);
                        } else {
                            mx = -INFINITY;
#pragma unroll
                            for (int n = 0; n < 128; ++n)
                                if (token_of_col(n) < lim) mx = fmaxf(mx, __uint_as_float(v[n]));
                        }
                        stage[j - w.j0] = mx * sm_scale;
                    } else {
                        float *dst = p.out + line * p.out_row_stride + static_cast<int64_t>(j) * kPage;
                        const int valid = p.max_seq_len - j * kPage;   // columns that exist
                        const bool vec = (p.out_row_stride & 3) == 0 && valid >= kPage;
#pragma unroll
                        for (int g = 0; g < 32; ++g) {
                            float4 o;
                            o.x = (4 * g + 0 < lim) ? __uint_as_float(v[g]) * sm_scale : -INFINITY;
                            o.y = (4 * g + 1 < lim) ? __uint_as_float(v[g + 32]) * sm_scale : -INFINITY;
                            o.z = (4 * g + 2 < lim) ? __uint_as_float(v[g + 64]) * sm_scale : -INFINITY;
                            o.w = (4 * g + 3 < lim) ? __uint_as_float(v[g + 96]) * sm_scale : -INFINITY;
                            if (vec) {
                                *reinterpret_cast<float4 *>(dst + 4 * g) = o;
                            } else {
                                if (4 * g + 0 < valid) dst[4 * g + 0] = o.x;
                                if (4 * g + 1 < valid) dst[4 * g + 1] = o.y;
                                if (4 * g + 2 < valid) dst[4 * g + 2] = o.z;
                                if (4 * g + 3 < valid) dst[4 * g + 3] = o.w;
                            }
                        }
                    }
                } else if (has_row) {
                    // no row of the tile sees this page: nothing was computed
                    if (!kLogits) {
                        stage[j - w.j0] = -INFINITY;
                    } else {
                        float *dst = p.out + line * p.out_row_stride + static_cast<int64_t>(j) * kPage;
                        const int valid = p.max_seq_len - j * kPage;
                        for (int c = 0; c < kPage && c < valid; ++c) dst[c] = -INFINITY;
                    }
                }
            }
            if (!ok) break;
            if (!kLogits && has_row) {
                float *dst = p.out + line * p.out_row_stride + w.j0;
                const int n = w.j1 - w.j0;
                if (n == kChunk && (p.out_row_stride & 3) == 0) {
                    const float4 *src = reinterpret_cast<const float4 *>(stage);
                    reinterpret_cast<float4 *>(dst)[0] = src[0];
                    reinterpret_cast<float4 *>(dst)[1] = src[1];
                } else if (n == kChunk && (p.out_row_stride & 1) == 0) {
                    const float2 *src = reinterpret_cast<const float2 *>(stage);
#pragma unroll
                    for (int i = 0; i < 4; ++i) reinterpret_cast<float2 *>(dst)[i] = src[i];
                } else {
                    for (int i = 0; i < n; ++i) dst[i] = stage[i];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
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
