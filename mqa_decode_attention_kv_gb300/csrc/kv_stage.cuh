// One pipeline stage of int8 K/V: a 64-token tile fetched with TMA.
//
// Stage layout: K codes [64 rows][D] then V codes [64 rows][D], each written by
// four 16-row TMA boxes with the 128-byte (D=128) or 64-byte (D=64) swizzle;
// fp32 scales land in a separate [2][64] array (K then V).  A box is fetched
// only if its 16 tokens overlap the key range [lo, L) and its block id is
// inside the pool; bit c of *stage_mask records whether box c arrived.
#pragma once

#include "common.cuh"

namespace mqa {

constexpr int32_t kNoBlock = INT32_MIN;  // "box not needed" (never a table entry we accept)

template <int D>
struct KvStage {
    static constexpr int CODE_BYTES = kTileTokens * D;  // K (or V) codes of one tile
    static constexpr int CODE_PAIR = 2 * CODE_BYTES;     // K then V
    static constexpr uint32_t SWZ_MASK = (D == 128) ? 7u : 3u;
};

// Byte offset of (row, col) inside a K or V tile region written by TMA with
// the swizzle of the code maps (the region base is 1024-byte aligned).
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t col)
{
    const uint32_t o = row * D + col;
    return o ^ (((o >> 7) & KvStage<D>::SWZ_MASK) << 4);
}

// Physical block ids of the four 16-token boxes of tile T (tokens [64T, 64T+64)):
// kNoBlock for a box outside the key range [lo, L).  The loads are independent, so a
// caller can issue them a tile ahead of use.
// With ring > 0 (a window-bounded cache) page p lives in table entry p % ring.
__device__ __forceinline__ int table_entry(int page, int ring) { return ring > 0 ? page % ring : page; }

__device__ __forceinline__ void fetch_tile_blocks(const int32_t *table, int page_size, int T, int lo, int L,
                                                  int ring, int32_t (&ids)[kChunksPerTile])
{
#pragma unroll
    for (int c = 0; c < kChunksPerTile; ++c) {
        const int t0 = T * kTileTokens + c * kChunkTokens;
        ids[c] = (t0 + kChunkTokens > lo && t0 < L) ? __ldg(table + table_entry(t0 / page_size, ring)) : kNoBlock;
    }
}

// Issue the copies of tile T into a stage from block ids fetched by
// fetch_tile_blocks (kNoBlock = not needed); called by a single thread.  Ids outside
// the pool are reported in dev_status and their boxes skipped.
template <int D>
__device__ __forceinline__ void issue_kv_tile_ids(const CUtensorMap &k_map, const CUtensorMap &v_map,
                                                  const float *k_scale, const float *v_scale,
                                                  const int32_t (&ids)[kChunksPerTile], int num_blocks,
                                                  int page_size, int32_t *dev_status, uint8_t *codes_dst,
                                                  float *scales_dst, uint64_t *bar, uint32_t *stage_mask, int T)
{
    uint8_t *kdst = codes_dst;
    uint8_t *vdst = codes_dst + KvStage<D>::CODE_BYTES;
    float *ksdst = scales_dst;
    float *vsdst = scales_dst + kTileTokens;
    int32_t rowbase[kChunksPerTile];
    uint32_t mask = 0, bytes = 0;
#pragma unroll
    for (int c = 0; c < kChunksPerTile; ++c) {
        const int t0 = T * kTileTokens + c * kChunkTokens;
        rowbase[c] = -1;
        if (ids[c] >= 0 && ids[c] < num_blocks) {
            rowbase[c] = ids[c] * page_size + (t0 % page_size);
            mask |= 1u << c;
            bytes += 2 * kChunkTokens * D + 2 * kChunkTokens * 4;
        } else if (ids[c] != kNoBlock) {
            set_status(dev_status, MQA_DEV_BAD_BLOCK);
        }
    }
    *stage_mask = mask;
    mbar_arrive_expect_tx(bar, bytes);
    int run_c = -1, run_n = 0;
#pragma unroll
    for (int c = 0; c <= kChunksPerTile; ++c) {
        const bool have = c < kChunksPerTile && rowbase[c] >= 0;
        if (have) {
            tma_load_2d(kdst + c * kChunkTokens * D, &k_map, 0, rowbase[c], bar);
            tma_load_2d(vdst + c * kChunkTokens * D, &v_map, 0, rowbase[c], bar);
        }
        // scales: boxes whose slots are contiguous (same page) share one bulk copy
        const bool extends = have && run_n > 0 && rowbase[c] == rowbase[run_c] + run_n * kChunkTokens;
        if (!extends && run_n > 0) {
            const uint32_t nb = run_n * kChunkTokens * 4;
            bulk_load(ksdst + run_c * kChunkTokens, k_scale + rowbase[run_c], nb, bar);
            bulk_load(vsdst + run_c * kChunkTokens, v_scale + rowbase[run_c], nb, bar);
            run_n = 0;
        }
        if (have) {
            if (run_n == 0)
                run_c = c;
            ++run_n;
        }
    }
}

// fetch + issue in one step (block-table latency not hidden)
template <int D>
__device__ __forceinline__ void issue_kv_tile(const CUtensorMap &k_map, const CUtensorMap &v_map,
                                              const float *k_scale, const float *v_scale, const int32_t *table,
                                              int num_blocks, int page_size, int32_t *dev_status,
                                              uint8_t *codes_dst, float *scales_dst, uint64_t *bar,
                                              uint32_t *stage_mask, int T, int lo, int L, int ring)
{
    int32_t ids[kChunksPerTile];
    fetch_tile_blocks(table, page_size, T, lo, L, ring, ids);
    issue_kv_tile_ids<D>(k_map, v_map, k_scale, v_scale, ids, num_blocks, page_size, dev_status, codes_dst,
                         scales_dst, bar, stage_mask, T);
}


// One warp's share of a tile: box c (16 tokens) of tile T, issued by the warp's
// lane 0 from a block id fetched earlier (kNoBlock = not needed).  Arrives once
// on `bar` (initialised for kChunksPerTile arrivals) with the box's transaction
// bytes, and records in *box_ok whether the box is coming.
template <int D>
__device__ __forceinline__ void issue_kv_box(const CUtensorMap &k_map, const CUtensorMap &v_map,
                                             const float *k_scale, const float *v_scale, int32_t id,
                                             int num_blocks, int page_size, int32_t *dev_status,
                                             uint8_t *codes_dst, float *scales_dst, uint64_t *bar,
                                             uint32_t *box_ok, int T, int c)
{
    const int t0 = T * kTileTokens + c * kChunkTokens;
    const bool ok = id >= 0 && id < num_blocks;
    if (!ok && id != kNoBlock)
        set_status(dev_status, MQA_DEV_BAD_BLOCK);
    *box_ok = ok ? 1u : 0u;
    if (!ok) {
        mbar_arrive_expect_tx(bar, 0);
        return;
    }
    const int row = id * page_size + (t0 % page_size);
    mbar_arrive_expect_tx(bar, 2 * kChunkTokens * D + 2 * kChunkTokens * 4);
    tma_load_2d(codes_dst + c * kChunkTokens * D, &k_map, 0, row, bar);
    tma_load_2d(codes_dst + KvStage<D>::CODE_BYTES + c * kChunkTokens * D, &v_map, 0, row, bar);
    bulk_load(scales_dst + c * kChunkTokens, k_scale + row, kChunkTokens * 4, bar);
    bulk_load(scales_dst + kTileTokens + c * kChunkTokens, v_scale + row, kChunkTokens * 4, bar);
}

// Block id of box c of tile T (kNoBlock when the box lies outside [lo, L)).
__device__ __forceinline__ int32_t fetch_box_block(const int32_t *table, int page_size, int T, int c, int lo, int L,
                                                   int ring)
{
    const int t0 = T * kTileTokens + c * kChunkTokens;
    return (t0 + kChunkTokens > lo && t0 < L) ? __ldg(table + table_entry(t0 / page_size, ring)) : kNoBlock;
}

}  // namespace mqa
