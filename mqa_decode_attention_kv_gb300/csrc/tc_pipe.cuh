// Pipeline helpers shared by the tcgen05 kernels (decode and prefill): bounded
// mbarrier waits with a CTA abort flag, named barriers, tensor-core issue from
// tensor memory, descriptor arithmetic.
#pragma once

#include "common.cuh"
#include "kv_stage.cuh"
#include "tc.cuh"

namespace mqa {

// Bounded wait that also gives up once another role has raised the abort
// flag; a wait that runs out raises it.  Returns false when giving up.
__device__ __forceinline__ bool wait_phase_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag);

__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    return mbar_try_wait(bar, parity) || wait_phase_slow(bar, parity, abort_flag);
}

// For a wait that is usually satisfied already: a test of the phase first
// (mbarrier.test_wait costs ~37 cycles against ~57 for try_wait on GB300).
__device__ __forceinline__ bool wait_done(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    return mbar_test(bar, parity) || wait_phase(bar, parity, abort_flag);
}

// The polling loop (inlined: a called function could not serve warpgroups that
// run with different register counts).
__device__ __forceinline__ bool wait_phase_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier over n threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// A: tensor memory, B: shared memory descriptor.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred pa;\n\tsetp.ne.u32 pa, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// Shared-memory descriptor plus a byte offset (the address field counts 16 B).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// The CTA-wide barrier of the teardown.  Every role ends with its own copy of
// the teardown (the roles run with different register counts and never rejoin).
__device__ __forceinline__ void bar_all() { asm volatile("bar.sync 0;" ::: "memory"); }

// Packed fp32 pairs (one instruction for two lanes of arithmetic) and a 3-input maximum.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Key blocks of the tcgen05 kernels: 128 tokens (two 64-token tiles) of head_dim 128.
constexpr int kBlockTokens = 128, kBlockD = 128;

// Cache row of the first token of box c of tile T in block `id`, or -1 when
// the box is not fetched (kNoBlock, or an id outside the pool: reported).
template <class Args>
__device__ __forceinline__ int box_row(const Args &a, int32_t id, int T, int c)
{
    const bool ok = id >= 0 && id < a.num_blocks;
    if (!ok && id != kNoBlock)
        set_status(a.dev_status, MQA_DEV_BAD_BLOCK);
    return ok ? id * a.page_size + (T * kTileTokens + c * kChunkTokens) % a.page_size : -1;
}

// Block id of box c (16 tokens) of tile t (64 tokens, 0 .. TILES-1) of the block at
// position p (fields b, blk, t_first, lo, L) of TILES tiles; kNoBlock when the box
// lies outside [lo, L).
template <int TILES = 2, class Args, class Pos>
__device__ __forceinline__ int32_t fetch_tile_box_id(const Args &a, const Pos &p, int t, int c)
{
    const int T = p.t_first + TILES * p.blk + t;
    return T <= (p.L - 1) / kTileTokens
               ? fetch_box_block(a.block_table + (size_t)p.b * a.max_blocks, a.page_size, T, c, p.lo, p.L, a.ring)
               : kNoBlock;
}

// Both tiles of the block at p into ring stage `stage`, their token scales into
// `scl` ([2][SCL_STRIDE] fp32: K, V).  Lane 4t + c holds the id of box c of tile t.
// A tile inside [lo, L) on one 64-token page goes as one 64-row copy per tensor
// (and one 256-byte copy per scale row), any other tile as its 16-row boxes
// that overlap [lo, L) (and 64-byte scale copies).  `part` 0 issues the K codes
// and scales, 1 the V ones, -1 both: two warps may share a block (one part
// each), each arriving once per tile on bars[t] with its byte count; the part-0
// (or only) warp records in oks[4t + c] whether box c comes.  The copies are
// spread over the lanes: one copy instruction takes a thread a few hundred
// cycles to issue, and the lanes' and warps' issues overlap.
template <int SCL_STRIDE = kBlockTokens, class Args, class Pos>
__device__ __forceinline__ void issue_block(const Args &a, const Pos &p, int lane, int32_t idc, uint8_t *stage,
                                            float *scl, uint64_t *bars, uint32_t *oks, int part = -1)
{
    constexpr int D = kBlockD, CODES = kBlockTokens * kBlockD;
    const int tb = lane >> 2, c = lane & 3;  // lanes 0-7: tile tb, box c
    const int Tb = p.t_first + 2 * p.blk + (tb & 1);
    const int row = lane < 8 ? box_row(a, idc, Tb, c) : -1;
    const uint32_t okall = __ballot_sync(0xffffffffu, row >= 0);
    // per tile t: whole_t, and row_t = the cache row of its first token (both tiles in
    // registers; a lane picks its tile's with a select, never an indexed array)
    const int row_0 = __shfl_sync(0xffffffffu, row, 0), row_1 = __shfl_sync(0xffffffffu, row, 4);
    const int T0 = p.t_first + 2 * p.blk;
    const bool p64 = a.page_size == kTileTokens;
    const bool whole_0 = p64 && (okall & 0xfu) == 0xfu && T0 * kTileTokens >= p.lo && (T0 + 1) * kTileTokens <= p.L;
    const bool whole_1 =
        p64 && ((okall >> 4) & 0xfu) == 0xfu && (T0 + 1) * kTileTokens >= p.lo && (T0 + 2) * kTileTokens <= p.L;
    if (lane < 8 && part <= 0)
        oks[lane] = row >= 0 ? 1u : 0u;
    __syncwarp();  // the flags are written before the arrival (a tile with nothing to fetch completes on it)
    if (lane < 2) {
        const uint32_t per_part = (uint32_t)__popc((okall >> (4 * lane)) & 0xfu) * kChunkTokens * (D + 4);
        mbar_arrive_expect_tx(bars + lane, part < 0 ? 2u * per_part : per_part);
    }
    __syncwarp();
    const int p_lo = part < 0 ? 0 : part, p_hi = part < 0 ? 1 : part;
    // whole tiles: lane 8 + 4t + 2q + k issues part q's codes (k = 0) or scales (k = 1) of tile t
    if (lane >= 8 && lane < 16) {
        const int t = (lane - 8) >> 2, q = ((lane - 8) >> 1) & 1, k = lane & 1;
        const int r0 = t ? row_1 : row_0;
        if ((t ? whole_1 : whole_0) && q >= p_lo && q <= p_hi) {
            if (k == 0)
                tma_load_2d(stage + q * CODES + t * kTileTokens * D, q ? &a.v_map64 : &a.k_map64, 0, r0, bars + t);
            else
                bulk_load(scl + q * SCL_STRIDE + t * kTileTokens, (q ? a.v_scale : a.k_scale) + r0, kTileTokens * 4, bars + t);
        }
    }
    // other tiles: lane 4t + c issues box c's codes and scales of the part(s)
    if (lane < 8 && row >= 0 && !(tb ? whole_1 : whole_0)) {
        const int box = lane;
        for (int q = p_lo; q <= p_hi; ++q) {
            tma_load_2d(stage + q * CODES + box * kChunkTokens * D, q ? &a.v_map : &a.k_map, 0, row, bars + tb);
            bulk_load(scl + q * SCL_STRIDE + box * kChunkTokens, (q ? a.v_scale : a.k_scale) + row, kChunkTokens * 4,
                      bars + tb);
        }
    }
}

// head_dim 64 read as rows of two tokens: a block is 128 rows of 128 bytes (256
// tokens, four 64-token tiles), each 16-token box one 8-row copy per tensor
// through maps over [num_blocks * page_size / 2][128] (a box never crosses a
// page: 16 tokens divide both page sizes).  Lane c < 16 holds the id of box c
// (tile c / 4, box c % 4 of it) and issues its codes and scales; token scales go
// to scl[c * 16 ..] (K) and scl[scl_stride + c * 16 ..] (V).  Barrier bars[h]
// takes boxes 8h .. 8h+7 (rows 64h .. 64h+63); oks[c] records whether box c comes.
template <class Args, class Pos>
__device__ __forceinline__ void issue_block_pairs(const Args &a, const Pos &p, int lane, int32_t idc,
                                                  uint8_t *stage, float *scl, int scl_stride, uint64_t *bars,
                                                  uint32_t *oks)
{
    constexpr int CODES = kBlockTokens * kBlockD, BOX_BYTES = 8 * kBlockD;
    const int T = p.t_first + 4 * p.blk + (lane >> 2);
    const int row = lane < 16 ? box_row(a, idc, T, lane & 3) : -1;  // cache row (token) of the box's first token
    const uint32_t okall = __ballot_sync(0xffffffffu, row >= 0);
    if (lane < 16)
        oks[lane] = row >= 0 ? 1u : 0u;
    __syncwarp();  // the flags are written before the arrival
    if (lane < 2) {
        const uint32_t n = (uint32_t)__popc((okall >> (8 * lane)) & 0xffu);
        mbar_arrive_expect_tx(bars + lane, n * 2u * kChunkTokens * (kBlockD / 2 + 4));
    }
    __syncwarp();
    if (lane < 16 && row >= 0) {
        uint64_t *bar = bars + (lane >> 3);
        tma_load_2d(stage + lane * BOX_BYTES, &a.k_map, 0, row >> 1, bar);
        tma_load_2d(stage + CODES + lane * BOX_BYTES, &a.v_map, 0, row >> 1, bar);
        bulk_load(scl + lane * kChunkTokens, a.k_scale + row, kChunkTokens * 4, bar);
        bulk_load(scl + scl_stride + lane * kChunkTokens, a.v_scale + row, kChunkTokens * 4, bar);
    }
}

}  // namespace mqa
