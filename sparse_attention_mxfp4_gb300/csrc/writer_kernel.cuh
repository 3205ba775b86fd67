// writer_kernel.cuh -- quantise bf16 index keys into MXFP4 pool page slots.
//
// The index key of each new token goes straight into its 8704 B pool page
// (ATOM #2770 "MiniMax-M3.1 MXFP4 sparse KV cache and index cache", "How it
// works", item "Write"): per 32-element group one e8m0 scale byte and 32
// e2m1 codes (aiter #7061 "MiniMax-M3 index score: MXFP4 index-cache prefill
// scorer", "Format").  The pages name a per-1x32 quantiser without its
// rounding rule; this kernel implements the OCP MX v1.0 conversion:
//   byte = clamp(floor(log2 amax) - 2 + 127, 1, 254), 127 for an all-zero group,
//   code = e2m1 round-to-nearest-even of x / 2^(byte-127), saturating at 6,
//   sign bit copied from x (also when the magnitude rounds to zero).
//
// Work split: four threads per token, one per 32-element group.  A thread
// reads its group's 64 bytes, takes the maximum magnitude on the bf16 bit
// patterns (for finite values the order of |x| is the order of the low 15
// bits), converts 32 elements with the hardware e2m1x2 conversion and stores
// its 16 code bytes; the quad's four scale bytes are gathered by shuffles into
// one 32-bit store.  The kernel is bound by HBM bandwidth: 256 B read and
// 68 B written per token (plus the 8 B slot).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace mx4 {

struct WriteParams {
    const uint16_t *k;             // bf16 bits, row t at k + t * k_row_stride
    const int64_t *slot_mapping;   // [num_tokens]; < 0 = padding
    uint8_t *k_data;
    uint8_t *k_scale;
    int64_t num_tokens;
    int64_t k_row_stride;          // elements
    int64_t k_data_page_stride;    // bytes
    int64_t k_scale_page_stride;   // bytes
    int64_t num_pool_pages;        // <= 0: unchecked
    int vec;                       // rows 16-byte aligned: 128-bit loads
};

// Two magnitudes -> one byte of e2m1 codes (lo in bits 0..3, hi in 4..7),
// round to nearest even, saturating at 6.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi)
{
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;
}

// 8 bf16 elements (bits) -> 4 code bytes in a 32-bit word, each magnitude
// multiplied by inv_scale (an exact power of two) before the conversion and
// the element's sign bit copied into bit 3 of its nibble.
__device__ __forceinline__ uint32_t bf16x8_to_e2m1x8(uint4 x, float inv_scale)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float((w[i] & 0x7FFFu) << 16) * inv_scale;
        const float hi = __uint_as_float(w[i] & 0x7FFF0000u) * inv_scale;
        uint32_t b = f32x2_to_e2m1x2(lo, hi);
        b |= ((w[i] >> 15) & 1u) << 3;     // sign of the even element
        b |= ((w[i] >> 31) & 1u) << 7;     // sign of the odd element
        out |= b << (8 * i);
    }
    return out;
}

__device__ __forceinline__ uint32_t absmax_bits(uint4 x, uint32_t m)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = max(m, w[i] & 0x7FFFu);
        m = max(m, (w[i] >> 16) & 0x7FFFu);
    }
    return m;
}

__global__ void __launch_bounds__(256) mx4_write_index_k_kernel(const __grid_constant__ WriteParams p)
{
    // programmatic dependent launch: every global access follows the wait
    griddep_launch_dependents();
    griddep_wait();
    // Warp-uniform trip count: every lane reaches the shuffles below.
    const int64_t n_threads = p.num_tokens * 4;
    const int64_t n_round = (n_threads + 31) & ~int64_t(31);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < n_round; gi += stride) {
        const int64_t t = gi >> 2;
        const int g = static_cast<int>(gi & 3);
        bool write = false;
        int64_t page = 0, tok = 0;
        uint4 x[4] = {};
        if (gi < n_threads) {
            // the key row is read together with its slot (a padding row is
            // read too and then ignored), so the two loads overlap
            const int64_t slot = __ldg(p.slot_mapping + t);
            const uint16_t *src = p.k + t * p.k_row_stride + 32 * g;
            if (p.vec) {
                const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] = __ldcs(s4 + i);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        v[j] = static_cast<uint32_t>(__ldcs(src + 8 * i + 2 * j)) |
                               (static_cast<uint32_t>(__ldcs(src + 8 * i + 2 * j + 1)) << 16);
                    x[i] = make_uint4(v[0], v[1], v[2], v[3]);
                }
            }
            if (slot >= 0) {
                page = slot >> 7;
                tok = slot & 127;
                if (p.num_pool_pages > 0 && page >= p.num_pool_pages) {
                    if (g == 0) atomicOr(&g_mx4_device_status, 0x1u);
                } else {
                    write = true;
                }
            }
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = absmax_bits(x[i], amax);
        // floor(log2 amax) = biased exponent - 127 for normal amax; the clamp
        // to byte 1 also covers subnormal maxima (exponent field 0..2)
        const int e_field = static_cast<int>(amax >> 7);
        const uint32_t byte = amax == 0 ? 127u : static_cast<uint32_t>(e_field - 2 < 1 ? 1 : e_field - 2);
        const float inv_scale = __uint_as_float((254u - byte) << 23);   // 2^(127 - byte), byte <= 252
        uint4 codes;
        codes.x = bf16x8_to_e2m1x8(x[0], inv_scale);
        codes.y = bf16x8_to_e2m1x8(x[1], inv_scale);
        codes.z = bf16x8_to_e2m1x8(x[2], inv_scale);
        codes.w = bf16x8_to_e2m1x8(x[3], inv_scale);
        uint32_t sw = byte << (8 * g);
        sw |= __shfl_xor_sync(0xffffffffu, sw, 1);
        sw |= __shfl_xor_sync(0xffffffffu, sw, 2);
        if (write) {
            uint8_t *dst = p.k_data + page * p.k_data_page_stride + tok * 64 + 16 * g;
            *reinterpret_cast<uint4 *>(dst) = codes;
            if (g == 0)
                *reinterpret_cast<uint32_t *>(p.k_scale + page * p.k_scale_page_stride + tok * 4) = sw;
        }
    }
}

}  // namespace mx4
