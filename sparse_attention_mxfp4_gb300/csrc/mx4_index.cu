// mx4_index.cu -- C ABI of the paged MXFP4 index-K scorer (declared in
// include/mx4_index.h): argument validation, TMA tensor-map encoding, grid
// choice and kernel launch.  No allocation, no synchronisation, no device
// reads on the host path of the scoring calls.
#include "mx4_index.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "score_kernel.cuh"
#include "writer_kernel.cuh"
#include "topk_kernel.cuh"
#include "attn_kernel.cuh"
#include "attn_rows_kernel.cuh"

namespace {

using mx4::ScoreParams;
using mx4::SmemLayout;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

constexpr int kMaxDevices = 64;

struct DeviceState {
    int sm_count = 0;
    bool topk_attr_set[2] = {false, false};
    bool attn_attr_set = false;
    int attn_clusters = 0;          // single-group attention clusters resident at once on the device
    int attn_rows_clusters = 0;     // two-group attention kernel: 2-CTA clusters resident at once
    int attn_rows_ctas = 0;         // two-group attention kernel: single CTAs resident at once
    bool smem_attr_set[8] = {false, false, false, false, false, false, false, false};
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

template <bool kDecode, bool kLogits, bool kFp8>
constexpr int kernel_index()
{
    return (kDecode ? 1 : 0) + (kLogits ? 2 : 0) + (kFp8 ? 4 : 0);
}

// Per-device one-time setup: SM count and the dynamic smem opt-in.
// Launch with clusters of `cluster` CTAs (when > 1) and, when `pdl`, with
// programmatic stream serialization: such kernels wait for the previous
// kernel of the stream before their first global access, so their set-up
// overlaps its tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                      unsigned cluster, bool pdl, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <bool kDecode, bool kLogits, bool kFp8>
mx4_status device_setup(int *sm_count)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &st = g_dev[dev];
    if (st.sm_count == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return MX4_ERR_CUDA;
        st.sm_count = n;
    }
    constexpr int ki = kernel_index<kDecode, kLogits, kFp8>();
    if (!st.smem_attr_set[ki]) {
        if (cudaFuncSetAttribute(mx4::mx4_score_kernel<kDecode, kLogits, kFp8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SmemLayout::kAlloc)) != cudaSuccess)
            return MX4_ERR_CUDA;
        st.smem_attr_set[ki] = true;
    }
    *sm_count = st.sm_count;
    return MX4_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Host cache of encoded tensor maps.  A map depends only on the view it
// describes (device, kind, base pointer, strides, extents), so a call that
// repeats a view (the usual case: the same pool every step) copies the
// 128-byte map instead of encoding it again.  Least-recently-used eviction
// over a small table; guarded by its own mutex.
enum TmapKind : int { kMapKData = 0, kMapKFp8 = 1, kMapKScale = 2, kMapAttnK = 3, kMapAttnKs = 4 };

struct TmapKey {
    int dev;
    int kind;
    const void *ptr;
    int64_t s0, s1, pages, heads;
    bool operator==(const TmapKey &o) const
    {
        return dev == o.dev && kind == o.kind && ptr == o.ptr && s0 == o.s0 && s1 == o.s1 && pages == o.pages &&
               heads == o.heads;
    }
};

constexpr int kTmapCacheSize = 64;

struct TmapEntry {
    TmapKey key;
    CUtensorMap map;
    uint64_t used = 0;   // 0 = empty slot
};

std::mutex g_tmap_mutex;
TmapEntry g_tmap[kTmapCacheSize];
uint64_t g_tmap_clock = 0;

// The cached map for `key`, or encode(&map) on a miss (false if encoding failed).
template <typename Encode>
bool cached_tmap(const TmapKey &key, CUtensorMap *out, Encode encode)
{
    std::lock_guard<std::mutex> lock(g_tmap_mutex);
    int victim = 0;
    for (int i = 0; i < kTmapCacheSize; ++i) {
        if (g_tmap[i].used != 0 && g_tmap[i].key == key) {
            g_tmap[i].used = ++g_tmap_clock;
            *out = g_tmap[i].map;
            return true;
        }
        if (g_tmap[i].used < g_tmap[victim].used) victim = i;
    }
    if (!encode(out)) return false;
    g_tmap[victim].key = key;
    g_tmap[victim].map = *out;
    g_tmap[victim].used = ++g_tmap_clock;
    return true;
}

int current_device()
{
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

// Page data view as a 4-D tensor of 4-bit elements:
//   dim0: 128 elements of one token (64 B), dim1: n0 in [0,32) (stride 256 B),
//   dim2: n1 in [0,4) (stride 64 B), dim3: page id (stride = page stride).
// A box {128, 32, 4, 1} lands token 4*n0 + n1 in smem row n0 + 32*n1, each
// 16-element group padded to 16 B (the tensor core's 4-bit operand form) and
// 128-byte swizzled.
bool encode_kdata_map(CUtensorMap *m, const uint8_t *k_data, int64_t stride, int64_t pages)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {128, 32, 4, static_cast<cuuint64_t>(pages)};
    const cuuint64_t strides[3] = {256, 64, static_cast<cuuint64_t>(stride)};
    const cuuint32_t box[4] = {128, 32, 4, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<uint8_t *>(k_data), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp8 page view, the same 4-D shape over bytes: dim0: the 128 e4m3 bytes of
// one token, dim1: n0 (stride 512 B), dim2: n1 (stride 128 B), dim3: page.
// The box lands token 4*n0 + n1 in smem row n0 + 32*n1 (128 B rows,
// 128-byte swizzled), the same row order as the MXFP4 view.
bool encode_kfp8_map(CUtensorMap *m, const uint8_t *k, int64_t stride, int64_t pages)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {128, 32, 4, static_cast<cuuint64_t>(pages)};
    const cuuint64_t strides[3] = {512, 128, static_cast<cuuint64_t>(stride)};
    const cuuint32_t box[4] = {128, 32, 4, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t *>(k), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Page scale view: 128 words (4 e8m0 bytes of one token each) per page.
bool encode_kscale_map(CUtensorMap *m, const uint8_t *k_scale, int64_t stride, int64_t pages)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(pages)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride)};
    const cuuint32_t box[2] = {128, 1};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t *>(k_scale), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Args {
    const void *q;
    int q_is_e4m3;
    const uint8_t *k_data;
    const uint8_t *k_scale;
    int64_t sd, ss;
    const int32_t *block_table;
    const int32_t *cu_seqlens_q;
    const int32_t *seq_lens;
    const int32_t *prefix_lens;
    int max_query_len;
    int max_seq_len;
    float sm_scale;
    float *out;
    cudaStream_t stream;
    int num_seqs;
    int64_t bt_stride;
    int64_t num_pool_pages;
    bool fp8 = false;   // k_data is an fp8 cache (k_scale, ss unused)
};

// True when the call has no output cell (no request, no query row or no
// page): such a call succeeds without touching any pointer.
bool empty_call(const Args &a, bool decode)
{
    return a.num_seqs == 0 || a.max_seq_len == 0 || (!decode && a.max_query_len == 0);
}

mx4_status validate(const Args &a, bool decode)
{
    if (a.q_is_e4m3 != 0 && a.q_is_e4m3 != 1) return MX4_ERR_INVALID_ARG;
    if (a.num_seqs < 0 || a.max_seq_len < 0 || (!decode && a.max_query_len < 0)) return MX4_ERR_INVALID_ARG;
    if (!(std::isfinite(a.sm_scale) && a.sm_scale > 0.0f)) return MX4_ERR_INVALID_ARG;
    if (empty_call(a, decode)) return MX4_OK;
    if (!a.q || !a.k_data || (!a.fp8 && !a.k_scale) || !a.block_table || !a.seq_lens || !a.out)
        return MX4_ERR_INVALID_ARG;
    if (!decode && (!a.cu_seqlens_q || !a.prefix_lens)) return MX4_ERR_INVALID_ARG;
    if (a.fp8 ? a.sd < static_cast<int64_t>(mx4::kFp8PageBytes)
              : (a.sd < mx4::kDataBytes || a.ss < mx4::kScaleBytes))
        return MX4_ERR_INVALID_ARG;   // narrow views
    if (a.num_pool_pages < 1) return MX4_ERR_INVALID_ARG;
    if (a.num_pool_pages > INT32_MAX) return MX4_ERR_UNSUPPORTED;
    const int64_t P = (static_cast<int64_t>(a.max_seq_len) + mx4::kPage - 1) / mx4::kPage;
    if (a.bt_stride < P || a.bt_stride < 0) return MX4_ERR_INVALID_ARG;                  // narrow table
    if (a.sd >= (int64_t(1) << 40) || a.ss >= (int64_t(1) << 40)) return MX4_ERR_UNSUPPORTED;
    if (a.fp8) {
        if (!aligned(a.k_data, 16) || (a.sd % 16) != 0) return MX4_ERR_MISALIGNED;
    } else {
        if (!aligned(a.k_data, 32) || (a.sd % 32) != 0) return MX4_ERR_MISALIGNED;
        if (!aligned(a.k_scale, 16) || (a.ss % 16) != 0) return MX4_ERR_MISALIGNED;
    }
    if (!aligned(a.q, 16) || !aligned(a.out, 16)) return MX4_ERR_MISALIGNED;
    if (!aligned(a.block_table, 4) || !aligned(a.seq_lens, 4)) return MX4_ERR_MISALIGNED;
    if (!decode && (!aligned(a.cu_seqlens_q, 4) || !aligned(a.prefix_lens, 4))) return MX4_ERR_MISALIGNED;
    return MX4_OK;
}

template <bool kDecode, bool kLogits, bool kFp8 = false>
mx4_status launch(const Args &a)
{
    mx4_status st = validate(a, kDecode);
    if (st != MX4_OK || empty_call(a, kDecode)) return st;
    const int P = static_cast<int>((static_cast<int64_t>(a.max_seq_len) + mx4::kPage - 1) / mx4::kPage);
    const int rows_per_tile = kDecode ? 1 : 2;
    const int tiles_per_seq = kDecode ? 1 : (a.max_query_len + rows_per_tile - 1) / rows_per_tile;
    if (a.num_seqs == 0 || P == 0 || tiles_per_seq == 0) return MX4_OK;   // no output cell exists
    const int chunks_per_tile = (P + mx4::kChunk - 1) / mx4::kChunk;
    const int64_t num_units = static_cast<int64_t>(a.num_seqs) * tiles_per_seq * chunks_per_tile;

    int sm_count = 0;
    st = device_setup<kDecode, kLogits, kFp8>(&sm_count);
    if (st != MX4_OK) return st;

    alignas(64) CUtensorMap tmap_k;
    alignas(64) CUtensorMap tmap_s;
    const int dev = current_device();
    if (kFp8) {
        const TmapKey kk{dev, kMapKFp8, a.k_data, a.sd, 0, a.num_pool_pages, 0};
        if (!cached_tmap(kk, &tmap_k, [&](CUtensorMap *m) { return encode_kfp8_map(m, a.k_data, a.sd, a.num_pool_pages); }))
            return MX4_ERR_CUDA;
        tmap_s = tmap_k;   // unused by the fp8 kernel
    } else {
        const TmapKey kd{dev, kMapKData, a.k_data, a.sd, 0, a.num_pool_pages, 0};
        const TmapKey ks{dev, kMapKScale, a.k_scale, a.ss, 0, a.num_pool_pages, 0};
        if (!cached_tmap(kd, &tmap_k, [&](CUtensorMap *m) { return encode_kdata_map(m, a.k_data, a.sd, a.num_pool_pages); }) ||
            !cached_tmap(ks, &tmap_s, [&](CUtensorMap *m) { return encode_kscale_map(m, a.k_scale, a.ss, a.num_pool_pages); }))
            return MX4_ERR_CUDA;
    }

    ScoreParams p{};
    p.q = a.q;
    p.block_table = a.block_table;
    p.cu_seqlens_q = a.cu_seqlens_q;
    p.seq_lens = a.seq_lens;
    p.prefix_lens = a.prefix_lens;
    p.out = a.out;
    p.bt_stride = a.bt_stride;
    p.num_pool_pages = a.num_pool_pages;
    p.num_units = num_units;
    p.out_row_stride = kLogits ? a.max_seq_len : P;
    p.num_seqs = a.num_seqs;
    p.max_seq_len = a.max_seq_len;
    p.num_out_pages = P;
    p.tiles_per_seq = tiles_per_seq;
    p.chunks_per_tile = chunks_per_tile;
    p.q_is_e4m3 = a.q_is_e4m3;
    p.sm_scale = a.sm_scale;

    // Host-known grid: one persistent CTA per SM (fewer when there are fewer
    // units); each CTA takes a contiguous, equal share of the units.
    const int64_t grid = num_units < sm_count ? num_units : sm_count;
    cudaGetLastError();   // clear a stale error so the check below is ours
    if (launch_ex(mx4::mx4_score_kernel<kDecode, kLogits, kFp8>, static_cast<unsigned>(grid), mx4::kThreads,
                  SmemLayout::kAlloc, a.stream, 1, true, tmap_k, tmap_s, p) != cudaSuccess)
        return MX4_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? MX4_OK : MX4_ERR_CUDA;
}

template <bool kDecode>
mx4_status topk_launch(const float *scores, const int32_t *block_table, const int32_t *cu_seqlens_q,
                       const int32_t *seq_lens, const int32_t *prefix_lens, int max_query_len, int max_seq_len,
                       int topk, int local_pages, int kv_groups, int32_t *sel, int32_t *count, int32_t *tokens,
                       void *stream, int num_seqs, int64_t block_table_stride)
{
    if (num_seqs < 0 || max_seq_len < 0 || (!kDecode && max_query_len < 0)) return MX4_ERR_INVALID_ARG;
    if (topk < 1 || local_pages < 0 || local_pages > topk) return MX4_ERR_INVALID_ARG;
    if (kv_groups < 1 || kv_groups > 64 || 64 % kv_groups != 0) return MX4_ERR_INVALID_ARG;
    if (num_seqs == 0 || (!kDecode && max_query_len == 0)) return MX4_OK;       // no row exists
    if (!scores || !block_table || !seq_lens || !sel || !count) return MX4_ERR_INVALID_ARG;
    if (!kDecode && (!cu_seqlens_q || !prefix_lens)) return MX4_ERR_INVALID_ARG;
    const int64_t P = (static_cast<int64_t>(max_seq_len) + mx4::kPage - 1) / mx4::kPage;
    if (P > mx4::kTopkMaxPages) return MX4_ERR_UNSUPPORTED;
    if (block_table_stride < P) return MX4_ERR_INVALID_ARG;
    if (!aligned(scores, 4) || !aligned(sel, 4) || !aligned(count, 4) || !aligned(tokens, 4) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return MX4_ERR_MISALIGNED;
    if (!kDecode && (!aligned(cu_seqlens_q, 4) || !aligned(prefix_lens, 4))) return MX4_ERR_MISALIGNED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX4_ERR_CUDA;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState &st = g_dev[dev];
        if (st.sm_count == 0) {
            int n = 0;
            if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
                return MX4_ERR_CUDA;
            st.sm_count = n;
        }
        if (!st.topk_attr_set[kDecode ? 1 : 0]) {
            if (cudaFuncSetAttribute(mx4::mx4_topk_kernel<kDecode, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     mx4::kTopkMaxPages * 4) != cudaSuccess ||
                cudaFuncSetAttribute(mx4::mx4_topk_kernel<kDecode, mx4::kTopkSplit>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, mx4::kTopkMaxPages * 4) != cudaSuccess)
                return MX4_ERR_CUDA;
            st.topk_attr_set[kDecode ? 1 : 0] = true;
        }
        sms = st.sm_count;
    }
    mx4::TopkParams p{};
    p.scores = scores;
    p.block_table = block_table;
    p.cu_seqlens_q = cu_seqlens_q;
    p.seq_lens = seq_lens;
    p.prefix_lens = prefix_lens;
    p.sel = sel;
    p.count = count;
    p.tokens = tokens;
    p.bt_stride = block_table_stride;
    p.num_seqs = num_seqs;
    p.rows_per_seq = kDecode ? 1 : max_query_len;
    p.max_seq_len = max_seq_len;
    p.num_pages = static_cast<int>(P);
    p.topk = topk;
    p.local = local_pages;
    p.groups = kv_groups;
    p.vec = aligned(scores, 16) && (P % 4) == 0;
    p.num_items = static_cast<int64_t>(num_seqs) * p.rows_per_seq * kv_groups;
    const size_t smem = static_cast<size_t>(P > 0 ? P : 1) * 4;
    cudaGetLastError();
    if (p.num_items < 2LL * sms) {
        // few items: one cluster of kTopkSplit CTAs per item, so a row's
        // score reads are spread over kTopkSplit SMs
        // (a plain launch: with a programmatic dependent launch the decode
        // selection measured slower)
        if (launch_ex(mx4::mx4_topk_kernel<kDecode, mx4::kTopkSplit>,
                      static_cast<unsigned>(p.num_items * mx4::kTopkSplit), mx4::kTopkThreads, smem,
                      static_cast<cudaStream_t>(stream), mx4::kTopkSplit, false, p) != cudaSuccess)
            return MX4_ERR_CUDA;
    } else {
        // one CTA per (row, group) item, at most 8 resident per SM, grid-stride
        const int64_t grid = p.num_items < 8LL * sms ? p.num_items : 8LL * sms;
        mx4::mx4_topk_kernel<kDecode, 1><<<static_cast<unsigned>(grid), mx4::kTopkThreads, smem,
                                           static_cast<cudaStream_t>(stream)>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? MX4_OK : MX4_ERR_CUDA;
}

// Attention K views: the scorer's 4-D token-permuting view of a page's codes
// with a KV-head dimension (5-D), and the scale words per (head, page) (3-D).
bool encode_attn_k_map(CUtensorMap *m, const uint8_t *k_data, int64_t ps, int64_t hs, int heads, int64_t pages)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[5] = {128, 32, 4, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(pages)};
    const cuuint64_t strides[4] = {256, 64, static_cast<cuuint64_t>(hs), static_cast<cuuint64_t>(ps)};
    const cuuint32_t box[5] = {128, 32, 4, 1, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 5, const_cast<uint8_t *>(k_data), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_attn_ks_map(CUtensorMap *m, const uint8_t *k_scale, int64_t ps, int64_t hs, int heads, int64_t pages)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(pages)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hs), static_cast<cuuint64_t>(ps)};
    const cuuint32_t box[3] = {128, 1, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t *>(k_scale), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

mx4_status mx4_index_score_prefill(const void *q, int q_is_e4m3, const uint8_t *k_data, const uint8_t *k_scale,
                                   int64_t k_data_page_stride, int64_t k_scale_page_stride,
                                   const int32_t *block_table, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                   const int32_t *prefix_lens, int max_query_len, int max_seq_len, float sm_scale,
                                   float *out, void *stream, int num_seqs, int64_t block_table_stride,
                                   int64_t num_pool_pages)
{
    const Args a{q,           q_is_e4m3,     k_data,       k_scale,   k_data_page_stride, k_scale_page_stride,
                 block_table, cu_seqlens_q,  seq_lens,     prefix_lens, max_query_len,    max_seq_len,
                 sm_scale,    out,           static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
                 num_pool_pages};
    return launch<false, false>(a);
}

mx4_status mx4_index_score_decode(const void *q, int q_is_e4m3, const uint8_t *k_data, const uint8_t *k_scale,
                                  int64_t k_data_page_stride, int64_t k_scale_page_stride,
                                  const int32_t *block_table, const int32_t *seq_lens, int max_seq_len,
                                  float sm_scale, float *out, void *stream, int num_seqs,
                                  int64_t block_table_stride, int64_t num_pool_pages)
{
    const Args a{q,           q_is_e4m3, k_data,   k_scale, k_data_page_stride, k_scale_page_stride,
                 block_table, nullptr,   seq_lens, nullptr, 1,                  max_seq_len,
                 sm_scale,    out,       static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
                 num_pool_pages};
    return launch<true, false>(a);
}

mx4_status mx4_index_logits_prefill(const void *q, int q_is_e4m3, const uint8_t *k_data, const uint8_t *k_scale,
                                    int64_t k_data_page_stride, int64_t k_scale_page_stride,
                                    const int32_t *block_table, const int32_t *cu_seqlens_q,
                                    const int32_t *seq_lens, const int32_t *prefix_lens, int max_query_len,
                                    int max_seq_len, float sm_scale, float *logits, void *stream, int num_seqs,
                                    int64_t block_table_stride, int64_t num_pool_pages)
{
    const Args a{q,           q_is_e4m3,    k_data,   k_scale,     k_data_page_stride, k_scale_page_stride,
                 block_table, cu_seqlens_q, seq_lens, prefix_lens, max_query_len,      max_seq_len,
                 sm_scale,    logits,       static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
                 num_pool_pages};
    return launch<false, true>(a);
}

mx4_status mx4_index_logits_decode(const void *q, int q_is_e4m3, const uint8_t *k_data, const uint8_t *k_scale,
                                   int64_t k_data_page_stride, int64_t k_scale_page_stride,
                                   const int32_t *block_table, const int32_t *seq_lens, int max_seq_len,
                                   float sm_scale, float *logits, void *stream, int num_seqs,
                                   int64_t block_table_stride, int64_t num_pool_pages)
{
    const Args a{q,           q_is_e4m3, k_data,   k_scale, k_data_page_stride, k_scale_page_stride,
                 block_table, nullptr,   seq_lens, nullptr, 1,                  max_seq_len,
                 sm_scale,    logits,    static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
                 num_pool_pages};
    return launch<true, true>(a);
}

mx4_status mx4_index_score_prefill_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8, int64_t k_page_stride,
                                       const int32_t *block_table, const int32_t *cu_seqlens_q,
                                       const int32_t *seq_lens, const int32_t *prefix_lens, int max_query_len,
                                       int max_seq_len, float sm_scale, float *out, void *stream, int num_seqs,
                                       int64_t block_table_stride, int64_t num_pool_pages)
{
    Args a{q,           q_is_e4m3,    k_fp8,    nullptr,     k_page_stride, 0,
           block_table, cu_seqlens_q, seq_lens, prefix_lens, max_query_len, max_seq_len,
           sm_scale,    out,          static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
           num_pool_pages};
    a.fp8 = true;
    return launch<false, false, true>(a);
}

mx4_status mx4_index_score_decode_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8, int64_t k_page_stride,
                                      const int32_t *block_table, const int32_t *seq_lens, int max_seq_len,
                                      float sm_scale, float *out, void *stream, int num_seqs,
                                      int64_t block_table_stride, int64_t num_pool_pages)
{
    Args a{q,           q_is_e4m3, k_fp8,    nullptr, k_page_stride, 0,
           block_table, nullptr,   seq_lens, nullptr, 1,             max_seq_len,
           sm_scale,    out,       static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
           num_pool_pages};
    a.fp8 = true;
    return launch<true, false, true>(a);
}

mx4_status mx4_index_logits_prefill_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8, int64_t k_page_stride,
                                        const int32_t *block_table, const int32_t *cu_seqlens_q,
                                        const int32_t *seq_lens, const int32_t *prefix_lens, int max_query_len,
                                        int max_seq_len, float sm_scale, float *logits, void *stream, int num_seqs,
                                        int64_t block_table_stride, int64_t num_pool_pages)
{
    Args a{q,           q_is_e4m3,    k_fp8,    nullptr,     k_page_stride, 0,
           block_table, cu_seqlens_q, seq_lens, prefix_lens, max_query_len, max_seq_len,
           sm_scale,    logits,       static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
           num_pool_pages};
    a.fp8 = true;
    return launch<false, true, true>(a);
}

mx4_status mx4_index_logits_decode_fp8(const void *q, int q_is_e4m3, const uint8_t *k_fp8, int64_t k_page_stride,
                                       const int32_t *block_table, const int32_t *seq_lens, int max_seq_len,
                                       float sm_scale, float *logits, void *stream, int num_seqs,
                                       int64_t block_table_stride, int64_t num_pool_pages)
{
    Args a{q,           q_is_e4m3, k_fp8,    nullptr, k_page_stride, 0,
           block_table, nullptr,   seq_lens, nullptr, 1,             max_seq_len,
           sm_scale,    logits,    static_cast<cudaStream_t>(stream), num_seqs, block_table_stride,
           num_pool_pages};
    a.fp8 = true;
    return launch<true, true, true>(a);
}

mx4_status mx4_index_topk_prefill(const float *scores, const int32_t *block_table, const int32_t *cu_seqlens_q,
                                  const int32_t *seq_lens, const int32_t *prefix_lens, int max_query_len,
                                  int max_seq_len, int topk, int local_pages, int kv_groups, int32_t *sel,
                                  int32_t *count, int32_t *sel_tokens, void *stream, int num_seqs,
                                  int64_t block_table_stride)
{
    return topk_launch<false>(scores, block_table, cu_seqlens_q, seq_lens, prefix_lens, max_query_len, max_seq_len,
                              topk, local_pages, kv_groups, sel, count, sel_tokens, stream, num_seqs,
                              block_table_stride);
}

mx4_status mx4_index_topk_decode(const float *scores, const int32_t *block_table, const int32_t *seq_lens,
                                 int max_seq_len, int topk, int local_pages, int kv_groups, int32_t *sel,
                                 int32_t *count, int32_t *sel_tokens, void *stream, int num_seqs,
                                 int64_t block_table_stride)
{
    return topk_launch<true>(scores, block_table, nullptr, seq_lens, nullptr, 1, max_seq_len, topk, local_pages,
                             kv_groups, sel, count, sel_tokens, stream, num_seqs, block_table_stride);
}

mx4_status mx4_sparse_pa_decode(const uint8_t *q, int64_t num_rows, int kv_heads, int groups,
                                const uint8_t *k_data, const uint8_t *k_scale, int64_t k_data_page_stride,
                                int64_t k_data_head_stride, int64_t k_scale_page_stride,
                                int64_t k_scale_head_stride, const uint8_t *v_data, const uint8_t *v_scale,
                                int64_t v_data_page_stride, int64_t v_data_head_stride,
                                int64_t v_scale_page_stride, int64_t v_scale_head_stride,
                                const int32_t *block_table, int block_table_width, const int32_t *context_lens,
                                float softmax_scale, void *out, int64_t num_pool_pages, void *stream)
{
    if (num_rows < 0 || kv_heads < 1 || groups < 1 || block_table_width < 0) return MX4_ERR_INVALID_ARG;
    if (!(std::isfinite(softmax_scale) && softmax_scale > 0.0f)) return MX4_ERR_INVALID_ARG;
    if (num_rows == 0) return MX4_OK;
    if (groups > mx4::kAttnN || block_table_width > mx4::kAttnMaxPages) return MX4_ERR_UNSUPPORTED;
    if (!q || !k_data || !k_scale || !v_data || !v_scale || !block_table || !context_lens || !out)
        return MX4_ERR_INVALID_ARG;
    if (num_pool_pages < 1) return MX4_ERR_INVALID_ARG;
    // rows x KV heads items, kept within the range the per-item indexing was checked for
    if (num_pool_pages > INT32_MAX || num_rows > INT32_MAX / (static_cast<int64_t>(kv_heads) * mx4::kAttnSplit))
        return MX4_ERR_UNSUPPORTED;
    // views: a page of one head holds 8192 code bytes and 512 scale bytes
    const int64_t strides[8] = {k_data_page_stride, k_data_head_stride, k_scale_page_stride, k_scale_head_stride,
                                v_data_page_stride, v_data_head_stride, v_scale_page_stride, v_scale_head_stride};
    for (int64_t st : strides)
        if (st < 0 || st >= (int64_t(1) << 40)) return MX4_ERR_INVALID_ARG;
    if (k_data_head_stride < mx4::kDataBytes || k_scale_head_stride < mx4::kScaleBytes ||
        v_data_head_stride < mx4::kDataBytes || v_scale_head_stride < mx4::kScaleBytes ||
        k_data_page_stride < k_data_head_stride * kv_heads || k_scale_page_stride < k_scale_head_stride * kv_heads ||
        v_data_page_stride < v_data_head_stride * kv_heads || v_scale_page_stride < v_scale_head_stride * kv_heads)
        return MX4_ERR_INVALID_ARG;                                    // narrow views
    if (!aligned(k_data, 32) || k_data_page_stride % 32 || k_data_head_stride % 32) return MX4_ERR_MISALIGNED;
    if (!aligned(k_scale, 16) || k_scale_page_stride % 16 || k_scale_head_stride % 16) return MX4_ERR_MISALIGNED;
    if (!aligned(v_data, 16) || v_data_page_stride % 16 || v_data_head_stride % 16) return MX4_ERR_MISALIGNED;
    if (!aligned(v_scale, 16) || v_scale_page_stride % 16 || v_scale_head_stride % 16) return MX4_ERR_MISALIGNED;
    if (!aligned(q, 16) || !aligned(out, 2) || !aligned(block_table, 4) || !aligned(context_lens, 4))
        return MX4_ERR_MISALIGNED;

    int dev = 0;
    int max_clusters = 0, rows_clusters = 0, rows_ctas = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX4_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState &st = g_dev[dev];
        if (!st.attn_attr_set) {
            if (cudaFuncSetAttribute(mx4::mx4_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(mx4::AttnSmem::kAlloc)) != cudaSuccess ||
                cudaFuncSetAttribute(mx4::mx4_attn_rows_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(mx4::ArSmem::kAlloc)) != cudaSuccess ||
                cudaFuncSetAttribute(mx4::mx4_attn_rows_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(mx4::ArSmem::kAlloc)) != cudaSuccess)
                return MX4_ERR_CUDA;
            // how many 2-CTA clusters of each kernel fit on the device at once
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(mx4::kAttnSplit, 1, 1);
            cfg.blockDim = dim3(mx4::kAttnThreads, 1, 1);
            cfg.dynamicSmemBytes = mx4::AttnSmem::kAlloc;
            int n = 0, nr = 0;
            if (cudaOccupancyMaxActiveClusters(&n, mx4::mx4_attn_kernel, &cfg) != cudaSuccess || n < 1)
                return MX4_ERR_CUDA;
            // (the two-group kernel takes its cluster shape from the launch)
            cudaLaunchAttribute cl;
            cl.id = cudaLaunchAttributeClusterDimension;
            cl.val.clusterDim.x = mx4::kAttnSplit;
            cl.val.clusterDim.y = 1;
            cl.val.clusterDim.z = 1;
            cfg.blockDim = dim3(mx4::kArThreads, 1, 1);
            cfg.dynamicSmemBytes = mx4::ArSmem::kAlloc;
            cfg.attrs = &cl;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&nr, mx4::mx4_attn_rows_kernel<2>, &cfg) != cudaSuccess || nr < 1)
                return MX4_ERR_CUDA;
            int per_sm = 0, sms = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mx4::mx4_attn_rows_kernel<1>, mx4::kArThreads,
                                                              mx4::ArSmem::kAlloc) != cudaSuccess ||
                per_sm < 1 || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                sms < 1)
                return MX4_ERR_CUDA;
            st.attn_clusters = n;
            st.attn_rows_clusters = nr;
            st.attn_rows_ctas = per_sm * sms;
            st.attn_attr_set = true;
        }
        max_clusters = st.attn_clusters;
        rows_clusters = st.attn_rows_clusters;
        rows_ctas = st.attn_rows_ctas;
    }
    alignas(64) CUtensorMap tmap_k;
    alignas(64) CUtensorMap tmap_ks;
    const TmapKey kk{dev, kMapAttnK, k_data, k_data_page_stride, k_data_head_stride, num_pool_pages, kv_heads};
    const TmapKey ks{dev, kMapAttnKs, k_scale, k_scale_page_stride, k_scale_head_stride, num_pool_pages, kv_heads};
    if (!cached_tmap(kk, &tmap_k, [&](CUtensorMap *m) {
            return encode_attn_k_map(m, k_data, k_data_page_stride, k_data_head_stride, kv_heads, num_pool_pages);
        }) ||
        !cached_tmap(ks, &tmap_ks, [&](CUtensorMap *m) {
            return encode_attn_ks_map(m, k_scale, k_scale_page_stride, k_scale_head_stride, kv_heads, num_pool_pages);
        }))
        return MX4_ERR_CUDA;
    mx4::AttnParams p{};
    p.q = q;
    p.v_data = v_data;
    p.v_scale = v_scale;
    p.vd_ps = v_data_page_stride;
    p.vd_hs = v_data_head_stride;
    p.vs_ps = v_scale_page_stride;
    p.vs_hs = v_scale_head_stride;
    p.block_table = block_table;
    p.context_lens = context_lens;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.num_pool_pages = num_pool_pages;
    p.kv_heads = kv_heads;
    p.groups = groups;
    p.width = block_table_width;
    p.softmax_scale = softmax_scale;
    p.num_items = num_rows * kv_heads;
    // Persistent launches: cluster (or CTA) c takes the (row, KV head) items
    // c, c + n, ... .  When every 2-CTA cluster gets at most one item, the
    // single-group kernel runs.  With more items than that, the two-group
    // kernel overlaps one item's end with the next one's pages, either on
    // 2-CTA clusters (each CTA half of every item's pages) or on single CTAs
    // (whole items, no combine): of the two, the one with fewer pages a CTA,
    // counted as ceil(items / units) x the pages a unit takes of an item, and
    // on a tie the one with single CTAs (half the item transitions).
    cudaGetLastError();
    cudaError_t e;
    const int64_t items = p.num_items;
    if (items <= max_clusters) {
        e = launch_ex(mx4::mx4_attn_kernel, static_cast<unsigned>(items * mx4::kAttnSplit), mx4::kAttnThreads,
                      mx4::AttnSmem::kAlloc, static_cast<cudaStream_t>(stream), 1, true, tmap_k, tmap_ks, p);
    } else if (2 * ((items + rows_ctas - 1) / rows_ctas) <= (items + rows_clusters - 1) / rows_clusters) {
        const int64_t ctas = items < rows_ctas ? items : rows_ctas;
        e = launch_ex(mx4::mx4_attn_rows_kernel<1>, static_cast<unsigned>(ctas), mx4::kArThreads, mx4::ArSmem::kAlloc,
                      static_cast<cudaStream_t>(stream), 1, true, tmap_k, tmap_ks, p);
    } else {
        const int64_t clusters = items < rows_clusters ? items : rows_clusters;
        e = launch_ex(mx4::mx4_attn_rows_kernel<2>, static_cast<unsigned>(clusters * mx4::kAttnSplit),
                      mx4::kArThreads, mx4::ArSmem::kAlloc, static_cast<cudaStream_t>(stream),
                      static_cast<unsigned>(mx4::kAttnSplit), true, tmap_k, tmap_ks, p);
    }
    if (e != cudaSuccess) return MX4_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? MX4_OK : MX4_ERR_CUDA;
}

mx4_status mx4_quantize_q_e4m3(const uint16_t *q_bf16, uint8_t *q_e4m3, int64_t n, void *stream)
{
    if (n < 0) return MX4_ERR_INVALID_ARG;
    if (n == 0) return MX4_OK;
    if (!q_bf16 || !q_e4m3) return MX4_ERR_INVALID_ARG;
    if (!aligned(q_bf16, 2)) return MX4_ERR_MISALIGNED;
    const int vec = aligned(q_bf16, 16) && aligned(q_e4m3, 8);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MX4_ERR_CUDA;
    const int64_t work = vec ? (n + 7) / 8 : n;
    int64_t blocks = (work + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    cudaGetLastError();
    mx4::mx4_quantize_q_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        q_bf16, q_e4m3, n, vec);
    return cudaGetLastError() == cudaSuccess ? MX4_OK : MX4_ERR_CUDA;
}

mx4_status mx4_index_k_write(const void *k, int64_t num_tokens, int64_t k_row_stride,
                             const int64_t *slot_mapping, uint8_t *k_data, uint8_t *k_scale,
                             int64_t k_data_page_stride, int64_t k_scale_page_stride, int64_t num_pool_pages,
                             void *stream)
{
    if (num_tokens < 0) return MX4_ERR_INVALID_ARG;
    if (num_tokens == 0) return MX4_OK;
    if (!k || !slot_mapping || !k_data || !k_scale) return MX4_ERR_INVALID_ARG;
    if (k_row_stride < mx4::kDim) return MX4_ERR_INVALID_ARG;
    if (k_data_page_stride < mx4::kDataBytes || k_scale_page_stride < mx4::kScaleBytes) return MX4_ERR_INVALID_ARG;
    if (!aligned(k, 2) || !aligned(slot_mapping, 8)) return MX4_ERR_MISALIGNED;
    if (!aligned(k_data, 16) || (k_data_page_stride % 16) != 0) return MX4_ERR_MISALIGNED;
    if (!aligned(k_scale, 4) || (k_scale_page_stride % 4) != 0) return MX4_ERR_MISALIGNED;
    if (num_tokens > (INT64_MAX / 4) / k_row_stride) return MX4_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MX4_ERR_CUDA;
    mx4::WriteParams p;
    p.k = static_cast<const uint16_t *>(k);
    p.slot_mapping = slot_mapping;
    p.k_data = k_data;
    p.k_scale = k_scale;
    p.num_tokens = num_tokens;
    p.k_row_stride = k_row_stride;
    p.k_data_page_stride = k_data_page_stride;
    p.k_scale_page_stride = k_scale_page_stride;
    p.num_pool_pages = num_pool_pages;
    p.vec = aligned(k, 16) && (k_row_stride % 8) == 0;
    // four threads per token; at most 8 resident 256-thread blocks per SM,
    // the rest of the tokens by a grid-stride loop
    int64_t blocks = (num_tokens * 4 + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    cudaGetLastError();
    if (launch_ex(mx4::mx4_write_index_k_kernel, static_cast<unsigned>(blocks), 256, 0,
                  static_cast<cudaStream_t>(stream), 1, true, p) != cudaSuccess)
        return MX4_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? MX4_OK : MX4_ERR_CUDA;
}

mx4_status mx4_index_get_device_status(void *stream, uint32_t *status_out)
{
    if (!status_out) return MX4_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MX4_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, mx4::g_mx4_device_status, sizeof v) != cudaSuccess) return MX4_ERR_CUDA;
    if (cudaMemcpyToSymbol(mx4::g_mx4_device_status, &zero, sizeof zero) != cudaSuccess) return MX4_ERR_CUDA;
    *status_out = v;
    return MX4_OK;
}

const char *mx4_status_string(int status)
{
    switch (status) {
    case MX4_OK: return "MX4_OK";
    case MX4_ERR_INVALID_ARG: return "MX4_ERR_INVALID_ARG";
    case MX4_ERR_MISALIGNED: return "MX4_ERR_MISALIGNED";
    case MX4_ERR_UNSUPPORTED: return "MX4_ERR_UNSUPPORTED";
    case MX4_ERR_CUDA: return "MX4_ERR_CUDA";
    default: return "MX4_ERR_UNKNOWN";
    }
}

int mx4_abi_version(void) { return MX4_ABI_VERSION; }

#ifdef MX4_STALL_TEST
// Test build only (compiled with -DMX4_STALL_TEST; not part of the product
// library or its header): make the waits at `site` (the MX4_DEV_TIMEOUT site
// numbers) in CTA `cta` of the following launches never see their barrier
// complete; site -1 turns it off.  Synchronous.
mx4_status mx4_test_set_stall(int site, int cta)
{
    if (cudaMemcpyToSymbol(mx4::g_mx4_stall_site, &site, sizeof site) != cudaSuccess ||
        cudaMemcpyToSymbol(mx4::g_mx4_stall_cta, &cta, sizeof cta) != cudaSuccess)
        return MX4_ERR_CUDA;
    return MX4_OK;
}
#endif

}  // extern "C"
