// Paged-cache helpers shared by the kernels: the table entry of a page (full
// tables and window-bounded rings), the block id of a 16-token box, and the
// per-token int8 quantisation of new K/V rows.
#pragma once

#include "common.cuh"

namespace mqa {

constexpr int32_t kNoBlock = INT32_MIN;  // "box not needed" (never a table entry we accept)

// Table entry of page p: with ring > 0 (a window-bounded cache) page p lives in
// entry p % ring.
__device__ __forceinline__ int table_entry(int page, int ring) { return ring > 0 ? page % ring : page; }

// Block id of box c of tile T (kNoBlock when the box lies outside [lo, L)).
__device__ __forceinline__ int32_t fetch_box_block(const int32_t *table, int page_size, int T, int c, int lo, int L,
                                                   int ring)
{
    const int t0 = T * kTileTokens + c * kChunkTokens;
    return (t0 + kChunkTokens > lo && t0 < L) ? __ldg(table + table_entry(t0 / page_size, ring)) : kNoBlock;
}

// Per-token symmetric int8 quantisation (the int8 KV cache of the "Character.AI
// best practices" blog, section "quantisation for training and serving"; the
// per-token scheme is this library's reading): scale = max|x| / 127 and
// code = clamp(round half to even(x / scale), -127, 127), both in IEEE fp32 (no
// reciprocal, no fast-math); an all-zero vector stores scale 0 and codes 0.
// kv_quant_scale takes the vector's max|x|; kv_quant8 packs 8 codes of a lane's
// slice (byte i = code of x[i]).
__device__ __forceinline__ float kv_quant_scale(float amax) { return __fdiv_rn(amax, 127.0f); }

__device__ __forceinline__ uint2 kv_quant8(const float (&x)[8], float s)
{
    uint32_t packed[2] = {0u, 0u};
    if (s != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int c = __float2int_rn(__fdiv_rn(x[i], s));
            c = max(-127, min(127, c));
            packed[i >> 2] |= (uint32_t)(c & 0xff) << (8 * (i & 3));
        }
    }
    return make_uint2(packed[0], packed[1]);
}

// The 8 values of a 16-byte slice of a bf16 row, widened exactly to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 raw, float (&x)[8])
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

}  // namespace mqa
