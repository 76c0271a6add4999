// Decode attention on the 5th-generation tensor cores (tcgen05), head_dim 128,
// groups of 32 query heads: one persistent, warp-specialised kernel.
//
// Work.  The call's (sequence b, head group g, 128-token key block) triples
// form one list, ordered by b, then g, then block.  In the balanced mode CTA c
// of the first G' = min(G, N) CTAs takes the contiguous share
// [c*N/G', (c+1)*N/G') of the N list entries (never empty), so every CTA
// streams the same number of blocks (+-1) whatever the length mix and
// its pipeline runs across sequence boundaries without draining.  A piece of
// a (b, g) pair that lies inside one share is the whole pair: its output is
// written directly (bf16).  A pair cut by share boundaries leaves an fp32
// partial (O, lse) per piece in slot 0 (the share's first piece) or 1 (its
// last) of the CTA that computed it, and the CTA holding its last piece
// writes a merge descriptor; a second kernel merges every cut pair, a CTA per
// (pair, 8 heads).  Each CTA rewrites both of its descriptor slots on every
// call, so the workspace needs no zeroing.  In the whole-sequence mode CTA c
// computes pair c alone and needs no workspace.
//
// Roles (14 warps, one CTA per SM):
//   warps 0-3   converters.  Thread t owns token row t of every block.  Waits
//               for its tile of the ring, converts the K codes to fp16 (kept
//               with their exponent bias +1152) straight into tensor memory
//               (the A operand of S^T = K Q^T) and the V codes to fp16 in
//               place in the ring stage (the A operand of O^T += V^T P'), and
//               copies the token's scales (landed with the codes) and
//               validity into the block's scale slot.  At a piece's first
//               block it also converts Q (bulk-copied a piece ahead) into the
//               B operand of S^T = K Q^T, scaled by one exact power of two,
//               and sums it per head for the bias.
//   warps 4-11  softmax.  Thread (t, half) reads token t's 16 scores of its
//               head half from tensor memory, takes the K bias off, applies
//               the K scale, exponentiates against a per-head reference
//               maximum that only moves when a score exceeds it by more than
//               2^8 (then O is rescaled in tensor memory: rare), and writes
//               P' = p * s_v * 2^(6-E) (fp16; 2^E a running power-of-two bound
//               of the V scales, so P' stays below 2^14).  At a piece's last
//               block it normalises O and stores the output or partial.
//   warp 12     lane 0 issues every tcgen05.mma and commit; the warp owns the
//               tensor-memory allocation.
//   warp 13     TMA: block ids a block ahead, the codes and scales of each
//               block into a ring stage once its O^T update has completed.
//
// Every int8 code is converted exactly once (exponent-bias trick, exact), the
// scores and O accumulate in fp32 tensor memory, and every wait is bounded:
// a wait that runs out raises a CTA-wide abort flag that makes all roles
// leave, and the call reports MQA_DEV_TIMEOUT.
#include <atomic>
#include <cfloat>
#include <math.h>

#include "common.cuh"
#include "kv_stage.cuh"
#include "launch.h"
#include "tc.cuh"

namespace mqa {
namespace {

struct TcCfg {
    static constexpr int D = 128;
    static constexpr int NH = 32;                    // heads per group (MMA N)
    static constexpr int BT = 128;                   // tokens per block (M of S^T, K of O^T)
    static constexpr int BOXES = BT / kChunkTokens;  // 8 TMA boxes of 16 tokens
    static constexpr int RING = 5;                   // ring stages (codes in flight, then fp16 V)
    static constexpr int DEPTH = 3;                  // blocks in flight between roles (S, K, P, scales)
    static constexpr int THREADS = 448;              // 4 converter + 8 softmax warps, MMA warp, TMA warp
    static constexpr int CODES = BT * D;             // int8 bytes of K (or V) of a block
    static constexpr int STAGE = 2 * CODES;          // K codes, V codes; then fp16 V in place
    // shared memory (offsets from a 1024-aligned base)
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_QH = OFF_RING + RING * STAGE;      // [2] fp16 Q [32 h][128 d], core layout (piece parity)
    static constexpr int OFF_QRAW = OFF_QH + 2 * NH * D * 2;    // bf16 Q [32 h][128 d] as copied (next piece)
    static constexpr int OFF_PH = OFF_QRAW + NH * D * 2;        // [DEPTH] fp16 P' [128 tok][32 h], core layout
    static constexpr int OFF_SC = OFF_PH + DEPTH * BT * NH * 2;  // [DEPTH][3][128] fp32: K scale, V scale, valid
    static constexpr int OFF_RED = OFF_SC + DEPTH * 3 * BT * 4;  // softmax group: [4 warps][32] + [4] fp32
    static constexpr int OFF_MREF = OFF_RED + 160 * 4;          // softmax group: reference maxima [32], factors [32]
    static constexpr int OFF_CRED = OFF_MREF + 64 * 4;          // converter group: [4] fp32, gh[4]
    static constexpr int OFF_OK = OFF_CRED + 16 * 4;            // [RING][8] box arrived
    static constexpr int OFF_SCL = OFF_OK + RING * BOXES * 4;   // [RING][2][128] fp32 K, V token scales (TMA)
    static constexpr int OFF_QB = OFF_SCL + RING * 2 * BT * 4;  // [4 pieces][4 warps][32] fp32 partial sums of Q
    static constexpr int OFF_BS = OFF_QB + 4 * 4 * NH * 4;      // [32] fp32 K bias of the piece's scores
    static constexpr int OFF_MISC = OFF_BS + NH * 4;            // tmem base, abort flag, start position
    static constexpr int OFF_MBAR = OFF_MISC + 256;
    static constexpr int NBAR = 4 * RING + 5 * DEPTH + 4;  // tiles, 5 x DEPTH hand-offs, O free [2], Q full / free
    static constexpr int SMEM_BYTES = OFF_MBAR + 8 * NBAR + 1024;
    // tensor memory columns: S^T [DEPTH][32], O^T [2][32], fp16 K [DEPTH][64]
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0, O_COL = DEPTH * NH, K_COL = O_COL + 2 * NH;
    // core-matrix strides (bytes): V rows = tokens, Q rows = heads, P rows = tokens.  The fp16
    // V of converter warp w's tokens 32w .. 32w+31 overwrites the 8 KB of codes they came
    // from: 8-token groups 0, 1 of the warp at K-half offset 4096w, groups 2, 3 at V-half
    // offset 4096w, each group 16 core matrices (8 d each) of 128 B.
    static constexpr uint32_t V_SR = 16 * 128;  // next 8 tokens (inside a 16-token MMA step)
    static constexpr uint32_t V_SC = 128;       // next 8 d
    static constexpr uint32_t Q_SR = 16 * 128;  // next 8 heads
    static constexpr uint32_t Q_SC = 128;       // next 8 d
    static constexpr uint32_t P_SR = 4 * 128;   // next 8 tokens
    static constexpr uint32_t P_SC = 128;       // next 8 heads
};
static_assert(TcCfg::SMEM_BYTES <= 227 * 1024, "shared memory budget");
// 128-byte-swizzled TMA destinations and descriptor bases on 1024 B; bulk copies, vector
// loads and stores on 16 B; mbarriers on 8 B
static_assert(TcCfg::OFF_RING % 1024 == 0 && TcCfg::STAGE % 1024 == 0 && TcCfg::OFF_QH % 1024 == 0 &&
                  TcCfg::OFF_PH % 1024 == 0, "1024-byte alignment");
static_assert(TcCfg::OFF_QRAW % 16 == 0 && TcCfg::OFF_SC % 16 == 0 && TcCfg::OFF_RED % 16 == 0 &&
                  TcCfg::OFF_MREF % 16 == 0 && TcCfg::OFF_CRED % 16 == 0 && TcCfg::OFF_OK % 16 == 0 &&
                  TcCfg::OFF_SCL % 16 == 0 && TcCfg::OFF_QB % 16 == 0 && TcCfg::OFF_BS % 16 == 0 &&
                  TcCfg::OFF_MISC % 16 == 0 && TcCfg::OFF_MBAR % 8 == 0,
              "16-byte alignment");
static_assert(TcCfg::K_COL + TcCfg::DEPTH * 64 <= TcCfg::TMEM_COLS, "tensor memory budget");

// Mbarrier wait with a suspend hint: a waiting warp sleeps until the phase
// completes instead of polling (eight warps polling would crowd the shared-
// memory pipe that the converters, the TMA and the tensor core use).
__device__ __forceinline__ bool mbar_poll(uint64_t *bar, uint32_t parity) { return mbar_try_wait(bar, parity); }

// Bounded wait that also gives up once another role has raised the abort
// flag; a wait that runs out raises it.  Returns false when giving up.
__device__ __noinline__ bool wait_phase_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag);

__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    return mbar_poll(bar, parity) || wait_phase_slow(bar, parity, abort_flag);
}

// The polling loop, out of line: the many wait sites stay small.
__device__ __noinline__ bool wait_phase_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 16; ++i)
            if (mbar_poll(bar, parity))
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

// Parity of the phase of a two-buffer hand-off barrier that carries item i.
__device__ __forceinline__ uint32_t ph2(int i) { return (uint32_t)(i >> 1) & 1u; }
// Buffer and phase parity of block i on a DEPTH-buffer hand-off (i >= 0).
__device__ __forceinline__ int bufd(int i) { return i % TcCfg::DEPTH; }
__device__ __forceinline__ uint32_t phd(int i) { return (uint32_t)(i / TcCfg::DEPTH) & 1u; }

// Reduce 16 per-head values over the 32 lanes of a warp with 16 shuffles (the
// butterfly below over each half-warp, then one exchange between the halves):
// lane L returns the reduction of head L % 16.  v is consumed.
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce16(float (&v)[16], int lane)
{
#pragma unroll
    for (int s = 8; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int k = 0; k < s; ++k) {
            const float send = up ? v[k] : v[k + s];
            const float keep = up ? v[k + s] : v[k];
            const float got = __shfl_xor_sync(0xffffffffu, send, s);
            v[k] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    const float other = __shfl_xor_sync(0xffffffffu, v[0], 16);
    return MAX ? fmaxf(v[0], other) : v[0] + other;
}

// Reduce 32 per-head values over the 32 lanes of a warp with 31 shuffles (a
// butterfly that halves the values each lane keeps at every step): lane L
// returns the reduction of head L.  v is consumed.
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane)
{
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int k = 0; k < s; ++k) {
            const float send = up ? v[k] : v[k + s];
            const float keep = up ? v[k + s] : v[k];
            const float got = __shfl_xor_sync(0xffffffffu, send, s);
            v[k] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
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

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Key blocks of a sequence of length L: the 64-token tiles from the one
// holding the window start to the one holding L-1, paired into 128-token
// blocks (the last block may hold a single tile).  0 for an invalid length.
__device__ __forceinline__ int seq_blocks(int L, int window, int max_seq_len, int &t_first, int &lo)
{
    t_first = 0;
    lo = 0;
    if (L < 1 || L > max_seq_len)
        return 0;
    lo = (window > 0 && L > window) ? L - window : 0;
    t_first = lo / kTileTokens;
    const int t_last = (L - 1) / kTileTokens;
    return (t_last - t_first + 2) >> 1;
}

// Position in the (sequence, head group, block) list.
struct Cursor {
    int b, g, blk;      // sequence, head group, block of the sequence
    int nblk;           // blocks of sequence b
    int t_first, lo, L; // first tile, window start, length of sequence b
};

// Load sequence b's shape into the cursor; then skip sequences without blocks.
__device__ __forceinline__ void cursor_seek(Cursor &c, const DecodeArgs &a)
{
    while (c.b < a.batch) {
        c.L = __ldg(a.seq_lens + c.b);
        c.nblk = seq_blocks(c.L, a.window, a.max_seq_len, c.t_first, c.lo);
        if (c.nblk > 0)
            return;
        ++c.b;
        c.g = 0;
        c.blk = 0;
    }
}

__device__ __forceinline__ void cursor_next(Cursor &c, const DecodeArgs &a, int groups)
{
    if (++c.blk < c.nblk)
        return;
    c.blk = 0;
    if (++c.g < groups)
        return;
    c.g = 0;
    ++c.b;
    cursor_seek(c, a);
}

// The CTA whose share holds list entry x (the largest c with floor(c*N/G) <= x).
__device__ __forceinline__ int cta_of(long long x, long long N, int G)
{
    return (int)(((x + 1) * G - 1) / N);
}

// Cache row of the first token of box c of tile T in block `id`, or -1 when
// the box is not fetched (kNoBlock, or an id outside the pool: reported).
__device__ __forceinline__ int box_row(const DecodeArgs &a, int32_t id, int T, int c)
{
    const bool ok = id >= 0 && id < a.num_blocks;
    if (!ok && id != kNoBlock)
        set_status(a.dev_status, MQA_DEV_BAD_BLOCK);
    return ok ? id * a.page_size + (T * kTileTokens + c * kChunkTokens) % a.page_size : -1;
}

// Block id of box c (16 tokens) of tile t (64 tokens, 0 or 1) of the block at
// cursor position p; kNoBlock when the box lies outside [lo, L).
__device__ __forceinline__ int32_t fetch_tile_box_id(const DecodeArgs &a, const Cursor &p, int t, int c)
{
    const int T = p.t_first + 2 * p.blk + t;
    return T <= (p.L - 1) / kTileTokens
               ? fetch_box_block(a.block_table + (size_t)p.b * a.max_blocks, a.page_size, T, c, p.lo, p.L)
               : kNoBlock;
}

// Both tiles of the block at p into ring stage `stage`, their token scales into
// `scl` ([2][128] fp32: K, V), issued by the TMA warp (every lane calls; lane
// 4t + c holds the id of box c of tile t).  A tile inside [lo, L) on one
// 64-token page goes as one 64-row copy per tensor (and one 256-byte copy per
// scale row), any other tile as its 16-row boxes that overlap [lo, L) (and
// 64-byte scale copies).  One arrival per tile on bars[t] with its byte count;
// box_ok[4t + c] records whether box c comes.
__device__ __forceinline__ void issue_block(const DecodeArgs &a, const Cursor &p, int lane, int32_t idc,
                                            uint8_t *stage, float *scl, uint64_t *bars, uint32_t *oks)
{
    constexpr int D = TcCfg::D;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int T = p.t_first + 2 * p.blk + t;
        const int c = lane - 4 * t;
        const bool mine = c >= 0 && c < 4;
        const int row = mine ? box_row(a, idc, T, c) : -1;
        const uint32_t okmask = (__ballot_sync(0xffffffffu, row >= 0) >> (4 * t)) & 0xfu;
        const int row0 = __shfl_sync(0xffffffffu, row, 4 * t);
        const bool whole = a.page_size == kTileTokens && okmask == 0xfu && T * kTileTokens >= p.lo &&
                           T * kTileTokens + kTileTokens <= p.L;
        if (mine)
            oks[4 * t + c] = row >= 0 ? 1u : 0u;
        __syncwarp();  // the flags are written before the arrival (a tile with nothing to fetch completes on it)
        if (lane == 0)
            mbar_arrive_expect_tx(bars + t, 2u * (uint32_t)__popc(okmask) * kChunkTokens * (D + 4));
        __syncwarp();
        if (whole) {
            if (lane == 0) {
                tma_load_2d(stage + t * kTileTokens * D, &a.k_map64, 0, row0, bars + t);
                tma_load_2d(stage + TcCfg::CODES + t * kTileTokens * D, &a.v_map64, 0, row0, bars + t);
                bulk_load(scl + t * kTileTokens, a.k_scale + row0, kTileTokens * 4, bars + t);
                bulk_load(scl + TcCfg::BT + t * kTileTokens, a.v_scale + row0, kTileTokens * 4, bars + t);
            }
        } else if (row >= 0) {
            const int box = 4 * t + c;
            tma_load_2d(stage + box * kChunkTokens * D, &a.k_map, 0, row, bars + t);
            tma_load_2d(stage + TcCfg::CODES + box * kChunkTokens * D, &a.v_map, 0, row, bars + t);
            bulk_load(scl + box * kChunkTokens, a.k_scale + row, kChunkTokens * 4, bars + t);
            bulk_load(scl + TcCfg::BT + box * kChunkTokens, a.v_scale + row, kChunkTokens * 4, bars + t);
        }
    }
}

// Four codes (byte i = code c_i) -> lo = {c0, c1} + kBias, hi = {c2, c3} + kBias as f16x2,
// exact: the exponent-bias conversion (0x64xx = 1024 + byte, on the codes offset by 128)
// without its final subtraction.  K enters S^T = K Q^T this way; the bias adds
// kBias * sum_d Q[h][d] to every score of head h, which the softmax warps take off in fp32.
constexpr float kBias = 1152.f;
__device__ __forceinline__ void i8x4_to_f16x2x2_biased(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t t = w ^ 0x80808080u;
    lo = __byte_perm(t, 0x64646464u, 0x5140);
    hi = __byte_perm(t, 0x64646464u, 0x7362);
}

// Shared-memory descriptor plus a byte offset (the address field counts 16 B).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// O^T += V^T(j) P'(j) for block j into the O buffer of its piece (MMA thread).
// Returns false when a wait gave up.
__device__ __forceinline__ bool issue_pv(int j, uint32_t first_bits, int &piece, int &n_pv, uint32_t tmem,
                                         uint64_t vdesc0, uint64_t pdesc0, uint64_t *pready, uint64_t *vready,
                                         uint64_t *ofree, uint64_t *odone, uint64_t *sfree, volatile int *abort_flag)
{
    using C = TcCfg;
    constexpr uint32_t IDESC_PV = umma_idesc_f16(128, C::NH, true, true);
    const int jb = bufd(j);
    if (!wait_phase(pready + jb, phd(j), abort_flag) || !wait_phase(vready + jb, phd(j), abort_flag))
        return false;
    const bool first = (first_bits >> (j & 31)) & 1u;
    if (first) {
        ++piece;
        // the O buffer of piece - 2 must have been read by its epilogue
        if (piece >= 2 && !wait_phase(ofree + (piece & 1), ph2(piece - 2), abort_flag))
            return false;
    }
    tc_fence_after();
    const uint32_t o_col = C::O_COL + (uint32_t)(piece & 1) * C::NH;
    // V: fp16 in place in ring stage j % RING; 16-token step kk = token groups 2kk, 2kk+1 of
    // converter warp kk / 2, in the K half (kk even) or the V half (kk odd)
    const uint64_t vd = desc_add(vdesc0, (j % C::RING) * C::STAGE), pd = desc_add(pdesc0, jb * C::BT * C::NH * 2);
#pragma unroll
    for (int kk = 0; kk < C::BT / 16; ++kk)
        umma_f16(tmem + o_col, desc_add(vd, (kk & 1) * C::CODES + (kk >> 1) * 4096), desc_add(pd, kk * 2 * C::P_SR),
                 IDESC_PV, !first || kk > 0);
    umma_commit(odone + jb);
    umma_commit(sfree + (j % C::RING));  // the stage's V is read: the TMA warp may refill it
    ++n_pv;
    return true;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Partial-output row of piece s (0 = the pair's first piece, in CTA c_lo) of a
// merged pair: CTA c_lo + s, slot slot_lo for s == 0 else 0, head jh.
__device__ __forceinline__ size_t merge_row(int c_lo, int s, int slot_lo, int jh)
{
    return (size_t)(2 * (c_lo + s) + (s == 0 ? slot_lo : 0)) * TcCfg::NH + jh;
}

}  // namespace

__global__ void __launch_bounds__(TcCfg::THREADS, 1) decode_tc_kernel(const __grid_constant__ DecodeArgs a)
{
    using C = TcCfg;
    constexpr int D = C::D, NH = C::NH, RING = C::RING, BT = C::BT;
    constexpr int BAR_SM = 1;  // named barrier of the softmax warps
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qh = base + C::OFF_QH;
    uint8_t *qraw = base + C::OFF_QRAW;
    uint8_t *ph = base + C::OFF_PH;
    float *sc = reinterpret_cast<float *>(base + C::OFF_SC);
    float *red = reinterpret_cast<float *>(base + C::OFF_RED);
    float *mref = reinterpret_cast<float *>(base + C::OFF_MREF);  // [32] per-head reference (log2 domain)
    float *ofac_s = mref + NH;                                     // [32] per-head O rescale factors
    float *cred = reinterpret_cast<float *>(base + C::OFF_CRED);
    uint32_t *box_ok = reinterpret_cast<uint32_t *>(base + C::OFF_OK);
    float *scl = reinterpret_cast<float *>(base + C::OFF_SCL);  // [RING][2][128] token scales, with the codes
    float *qpart = reinterpret_cast<float *>(base + C::OFF_QB);  // [4][4][32] per-warp sums of the fp16 Q
    float *bsum = reinterpret_cast<float *>(base + C::OFF_BS);   // [32] kBias * sum_d Q of the piece
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 4);
    int *start_pos = reinterpret_cast<int *>(base + C::OFF_MISC + 16);          // b, g, blk, n
    long long *share = reinterpret_cast<long long *>(base + C::OFF_MISC + 32);  // first entry, N, CTAs
    static_assert(32 + 3 * 8 <= 64, "misc layout");
    uint64_t *tfull = reinterpret_cast<uint64_t *>(base + C::OFF_MBAR);  // [RING][2] tile codes landed (TMA)
    uint64_t *tfree = tfull + 2 * RING;         // [RING] stage free: O^T of its block done (tensor core)
    uint64_t *kready = tfree + 2 * RING;        // [DEPTH] K in tensor memory, scales, Q (4 converter warps)
    uint64_t *vready = kready + C::DEPTH;       // [DEPTH] fp16 V in shared memory     (4 converter warps)
    uint64_t *pready = vready + C::DEPTH;       // [DEPTH] P' written, S read          (8 softmax warps)
    uint64_t *sfull = pready + C::DEPTH;        // [DEPTH] S^T = K Q^T done            (tensor core)
    uint64_t *odone = sfull + C::DEPTH;         // [DEPTH] O^T += V^T P' done          (tensor core)
    uint64_t *ofree = odone + C::DEPTH;         // [2] a piece's O read by its epilogue (8 softmax warps)
    uint64_t *qfull = ofree + 2;                // raw Q of the next piece landed      (bulk copy)
    uint64_t *qfree = qfull + 1;                // raw Q read by every converter warp  (4 converter warps)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int groups = (a.num_q_heads + NH - 1) / NH;
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    const bool balanced = a.persistent != 0;

    // ---- set-up: barriers and tensor memory (no inputs needed: overlaps the length reads below)
    if (tid == 0) {
        for (int s = 0; s < 2 * RING; ++s) {
            mbar_init(tfull + s, 1);
            mbar_init(tfree + s, 1);
        }
        for (int s = 0; s < C::DEPTH; ++s) {
            mbar_init(kready + s, 4);
            mbar_init(vready + s, 4);
            mbar_init(pready + s, 8);
            mbar_init(sfull + s, 1);
            mbar_init(odone + s, 1);
        }
        for (int s = 0; s < 2; ++s)
            mbar_init(ofree + s, 8);
        mbar_init(qfull, 1);
        mbar_init(qfree, 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 12)
        tmem_alloc(tmem_slot, C::TMEM_COLS);
    // ---- this CTA's share of the (sequence, group, block) list
    if (balanced && a.batch <= C::THREADS) {
        // one pass (a sequence per thread): its blocks, the block-wide prefix and total
        int *wsum = reinterpret_cast<int *>(red);
        int nb = 0;
        if (tid < a.batch) {
            int tf, lo;
            nb = seq_blocks(__ldg(a.seq_lens + tid), a.window, a.max_seq_len, tf, lo);
            if (nb == 0 && tid % G == cta) {
                set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + (size_t)tid * a.num_q_heads * D);
                for (int k = 0; k < a.num_q_heads * D / 8; ++k)
                    dst[k] = make_uint4(0, 0, 0, 0);
            }
        }
        int x = nb;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off)
                x += y;
        }
        if (lane == 31)
            wsum[warp] = x;
        __syncthreads();
        long long pre = 0, total = 0;
        for (int w = 0; w < C::THREADS / 32; ++w) {
            if (w < warp)
                pre += wsum[w];
            total += wsum[w];
        }
        const long long NB = total * groups;
        const int Ge = (int)(NB < G ? NB : G);
        const long long first = cta < Ge ? NB * cta / Ge : 0, last = cta < Ge ? NB * (cta + 1) / Ge : 0;
        const long long incl = (pre + x) * groups, excl = (pre + x - nb) * groups;
        if (tid == 0) {
            share[0] = first;
            share[1] = NB;
            share[2] = Ge;
            start_pos[3] = (int)(last - first);
        }
        if (nb > 0 && last > first && excl <= first && first < incl) {
            const int r = (int)(first - excl);
            start_pos[0] = tid;
            start_pos[1] = r / nb;
            start_pos[2] = r % nb;
        }
        __syncthreads();
    } else if (balanced) {
        int *wsum = reinterpret_cast<int *>(red);
        // pass 1: blocks per group over all sequences; sequences without blocks
        // (invalid length) get a zero output from CTA b % G and a status bit
        long long mine = 0;
        for (int bb = tid; bb < a.batch; bb += C::THREADS) {
            int tf, lo;
            const int L = __ldg(a.seq_lens + bb);
            const int nb = seq_blocks(L, a.window, a.max_seq_len, tf, lo);
            mine += nb;
            if (nb == 0 && bb % G == cta) {
                set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + (size_t)bb * a.num_q_heads * D);
                for (int k = 0; k < a.num_q_heads * D / 8; ++k)
                    dst[k] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            mine += __shfl_xor_sync(0xffffffffu, mine, off);
        if (lane == 0)
            reinterpret_cast<long long *>(wsum)[warp] = mine;
        __syncthreads();
        long long NB = 0;
        for (int w = 0; w < C::THREADS / 32; ++w)
            NB += reinterpret_cast<long long *>(wsum)[w];
        NB *= groups;
        // shares over Ge = min(G, N) CTAs, so that every share is non-empty and the
        // pieces of a cut pair lie in consecutive CTAs; CTAs from Ge on have none
        const int Ge = (int)(NB < G ? NB : G);
        const long long first = cta < Ge ? NB * cta / Ge : 0, last = cta < Ge ? NB * (cta + 1) / Ge : 0;
        if (tid == 0) {
            share[0] = first;
            share[1] = NB;
            share[2] = Ge;
            start_pos[3] = (int)(last - first);
        }
        __syncthreads();
        // pass 2: the sequence holding entry `first` (its prefix of blocks x groups
        // is <= first < prefix + its blocks x groups)
        long long run = 0;
        for (int b0 = 0; b0 < a.batch && last > first; b0 += C::THREADS) {
            const int bb = b0 + tid;
            int tf, lo, nb = 0;
            if (bb < a.batch)
                nb = seq_blocks(__ldg(a.seq_lens + bb), a.window, a.max_seq_len, tf, lo);
            int x = nb;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off)
                    x += y;
            }
            __syncthreads();  // wsum reuse
            if (lane == 31)
                wsum[warp] = x;
            __syncthreads();
            long long pre = run;
            int chunk = 0;
            for (int w = 0; w < C::THREADS / 32; ++w) {
                if (w < warp)
                    pre += wsum[w];
                chunk += wsum[w];
            }
            const long long incl = (pre + x) * groups, excl = (pre + x - nb) * groups;
            if (nb > 0 && excl <= first && first < incl) {
                const int r = (int)(first - excl);
                start_pos[0] = bb;
                start_pos[1] = r / nb;
                start_pos[2] = r % nb;
            }
            run += chunk;
        }
        __syncthreads();
    } else {
        // whole-sequence mode: CTA c computes (sequence c / groups, group c % groups)
        if (tid == 0) {
            const int bb = cta / groups, gg = cta % groups;
            int tf, lo;
            const int nb = seq_blocks(__ldg(a.seq_lens + bb), a.window, a.max_seq_len, tf, lo);
            start_pos[0] = bb;
            start_pos[1] = gg;
            start_pos[2] = 0;
            start_pos[3] = nb;
            share[0] = 0;
            share[1] = 0;
            share[2] = G;
            if (nb == 0)
                set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
        }
        __syncthreads();
        if (start_pos[3] == 0) {
            const int bb = cta / groups, gg = cta % groups;
            for (int r = tid; r < NH * D / 8; r += C::THREADS) {
                const int h = gg * NH + r / (D / 8);
                if (h < a.num_q_heads)
                    reinterpret_cast<uint4 *>(a.out + ((size_t)bb * a.num_q_heads + h) * D)[r % (D / 8)] =
                        make_uint4(0, 0, 0, 0);
            }
        }
    }
    const int n = start_pos[3];
    if (balanced && tid == 0) {
        // both merge slots of this CTA start empty on every call (set below if needed)
        a.merge_desc[(2 * cta) * 8] = -1;
        a.merge_desc[(2 * cta + 1) * 8] = -1;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (n <= 0) {  // uniform: nothing to compute
        if (warp == 12)
            tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }
    const long long list_first = share[0], list_n = share[1];
    const int Ge = (int)share[2];  // CTAs with a share (balanced mode)
    Cursor c0;
    c0.b = start_pos[0];
    c0.g = start_pos[1];
    c0.blk = start_pos[2];
    cursor_seek(c0, a);  // loads the shape of sequence c0.b (which has blocks)
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's tensor-memory lanes
    constexpr uint32_t IDESC_QK = umma_idesc_f16(128, NH, false, false);

    if (warp < 4) {
        // ================================================================ converters
        const int tok = tid;  // token row of every block = tensor-memory lane
        const int my_tile = warp >> 1;            // warps 0, 1 read tile 0 of a block; warps 2, 3 tile 1
        Cursor cur = c0;
        int q_issued = 0;
        {
            // the first piece's Q (bf16, 32 heads x 256 B, contiguous)
            if (warp == 0 && lane == 0) {
                mbar_arrive_expect_tx(qfull, NH * D * 2);
                bulk_load(qraw, a.q + ((size_t)c0.b * a.num_q_heads + c0.g * NH) * D, NH * D * 2, qfull);
            }
            q_issued = 1;
        }
        int piece = -1;
        int i = 0;
        for (; i < n; ++i) {
            const int r = i % RING, buf = bufd(i);
            uint8_t *st = base + C::OFF_RING + r * C::STAGE;
            const bool first = (i == 0) || cur.blk == 0;
            bool ok = wait_phase(tfull + 2 * r + my_tile, (uint32_t)(i / RING) & 1u, abort_flag);
            if (i >= C::DEPTH) {
                // scale slot [buf] free once softmax(i-DEPTH) is done, and with it K buffer [buf]:
                // the softmax warps arrive only after they saw S^T(i-DEPTH), which read K(i-DEPTH),
                // complete, so this one wait orders the tensor core's reads before the stores below
                ok = ok && wait_phase(pready + buf, phd(i - C::DEPTH), abort_flag);
            }
            if (first) {
                ok = ok && wait_phase(qfull, (uint32_t)(piece + 1) & 1u, abort_flag);  // this piece's raw Q
                if (i >= 2)  // fp16 Q buffer (piece parity) was last read by piece-2's S^T, done by S^T(i-2)
                    ok = ok && wait_phase(sfull + bufd(i - 2), phd(i - 2), abort_flag);
            }
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after();
            if (first) {
                // ---- Q of this piece, scaled by one power of two 2^e (exact in fp16): lane =
                // head; pass 1 takes the max over the 32 x 128 values (chunks read in a
                // lane-rotated order: no bank conflicts), pass 2 converts this warp's d range
                ++piece;
                const uint8_t *qrow = qraw + lane * D * 2;
                float m = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const uint4 qv = *reinterpret_cast<const uint4 *>(qrow + 16 * ((k + lane) & 15));
                    const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[t] << 16)),
                                           fabsf(__uint_as_float(w4[t] & 0xffff0000u))));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                int e = 0;
                if (m > 0.f && isfinite(m)) {
                    int x;
                    frexpf(m, &x);
                    e = min(120, max(-120, 14 - x));
                }
                const float f = exp2i(e);
                float qsum = 0.f;  // this warp's d range of head `lane`, as the tensor core sees it
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int c = 4 * warp + ((t + lane) & 3);  // 8-d chunk: d = 8c .. 8c+7
                    const uint4 qv = *reinterpret_cast<const uint4 *>(qrow + 16 * c);
                    const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
                    uint32_t hv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        hv[u] = pack_half2(__uint_as_float(w4[u] << 16) * f, __uint_as_float(w4[u] & 0xffff0000u) * f);
                        const __half2 h2 = *reinterpret_cast<const __half2 *>(&hv[u]);
                        qsum += __low2float(h2);
                        qsum += __high2float(h2);
                    }
                    *reinterpret_cast<uint4 *>(qh + (piece & 1) * NH * D * 2 + core_off(lane, 8 * c, C::Q_SR, C::Q_SC)) =
                        make_uint4(hv[0], hv[1], hv[2], hv[3]);
                }
                qpart[((piece & 3) * 4 + warp) * NH + lane] = qsum;  // 4 slots, as for the score factor
                if (warp == 0 && lane == 0)
                    cred[4 + (piece & 3)] = a.q_scale_log2 * exp2i(-e);  // log2-domain factor of raw scores
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(qfree);  // this warp has read the raw Q
                // the next piece's Q, once every warp has read this one (only if this CTA has it)
                const int i_next = i + (cur.nblk - cur.blk);
                if (warp == 0 && i_next < n) {
                    Cursor nx = cur;
                    nx.blk = cur.nblk - 1;
                    cursor_next(nx, a, groups);
                    if (!__all_sync(0xffffffffu, wait_phase(qfree, (uint32_t)piece & 1u, abort_flag)))
                        break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(qfull, NH * D * 2);
                        bulk_load(qraw, a.q + ((size_t)nx.b * a.num_q_heads + nx.g * NH) * D, NH * D * 2, qfull);
                    }
                    ++q_issued;
                }
            }
            // ---- this token's K codes (all chunks loaded before the conversion)
            uint4 kc[D / 16];
            {
                const uint8_t *krow = st + tok * D;
#pragma unroll
                for (int j = 0; j < D / 16; ++j)
                    kc[j] = *reinterpret_cast<const uint4 *>(krow + ((uint32_t)(j ^ (tok & 7)) << 4));
            }
            {
                const int pos = (cur.t_first + 2 * cur.blk) * kTileTokens + tok;
                const bool fetched = box_ok[r * C::BOXES + (tok >> 4)] != 0;
                const bool valid = fetched && pos >= cur.lo && pos < cur.L;
                const float *sr = scl + r * 2 * BT;  // landed with the codes
                float *scb = sc + buf * 3 * BT;
                scb[tok] = fetched ? sr[tok] : 0.f;
                scb[BT + tok] = fetched ? sr[BT + tok] : 0.f;
                scb[2 * BT + tok] = valid ? 1.f : 0.f;
            }
            // ---- K: 128 codes -> fp16 pairs in tensor memory (lane tok, 64 columns)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t kr[32];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint4 kv = kc[4 * half + jj];
                    i8x4_to_f16x2x2_biased(kv.x, kr[8 * jj + 0], kr[8 * jj + 1]);
                    i8x4_to_f16x2x2_biased(kv.y, kr[8 * jj + 2], kr[8 * jj + 3]);
                    i8x4_to_f16x2x2_biased(kv.z, kr[8 * jj + 4], kr[8 * jj + 5]);
                    i8x4_to_f16x2x2_biased(kv.w, kr[8 * jj + 6], kr[8 * jj + 7]);
                }
                tmem_st32(tmem + lane_base + C::K_COL + (uint32_t)buf * 64 + 32 * half, kr);
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(kready + buf);
            // ---- V: fp16 in place over this warp's 8 KB of codes in stage r (every lane's
            // rows are in registers once the warp passes the barrier): the MN-major A operand
            // of O^T += V^T P', token group g = lane / 8 of the warp at (g < 2 ? K half :
            // V half) + 4096 warp + 2048 (g % 2), row lane % 8 of its 16 core matrices.
            uint4 vc[D / 16];
            {
                const uint8_t *vrow = st + C::CODES + tok * D;
#pragma unroll
                for (int j = 0; j < D / 16; ++j)
                    vc[j] = *reinterpret_cast<const uint4 *>(vrow + ((uint32_t)(j ^ (tok & 7)) << 4));
            }
            __syncwarp();
            {
                const int g = lane >> 3;
                uint8_t *vb = st + (g >> 1) * C::CODES + warp * 4096 + (g & 1) * 2048 + (lane & 7) * 16;
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    uint32_t v8[8];
                    i8x4_to_f16x2x2(vc[j].x, v8[0], v8[1]);
                    i8x4_to_f16x2x2(vc[j].y, v8[2], v8[3]);
                    i8x4_to_f16x2x2(vc[j].z, v8[4], v8[5]);
                    i8x4_to_f16x2x2(vc[j].w, v8[6], v8[7]);
                    *reinterpret_cast<uint4 *>(vb + (2 * j) * C::V_SC) = make_uint4(v8[0], v8[1], v8[2], v8[3]);
                    *reinterpret_cast<uint4 *>(vb + (2 * j + 1) * C::V_SC) = make_uint4(v8[4], v8[5], v8[6], v8[7]);
                }
            }
            // vready[buf] may take block i's arrivals only once the MMA thread has consumed
            // block i-DEPTH's phase (O^T(i-DEPTH) done): else its wait on that phase could be lapped
            if (i >= C::DEPTH && !__all_sync(0xffffffffu, wait_phase(odone + buf, phd(i - C::DEPTH), abort_flag))) {
                ++i;
                break;
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(vready + buf);
            cursor_next(cur, a, groups);
        }
        if (*abort_flag && lane == 0 && warp == 0 && q_issued > piece + 1)
            mbar_wait_bounded(qfull, (uint32_t)(q_issued - 1) & 1u);  // the Q copy still in flight (bounded)
    } else if (warp == 13) {
        // ================================================================ TMA producer
        // ring stage j % RING takes block j once O^T of block j - RING has read its V;
        // lane 4t + c fetches the block id of box c of tile t a block ahead
        if (lane == 0) {
            const bool p64 = a.page_size == kTileTokens;
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(p64 ? &a.k_map64 : &a.k_map))
                         : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(p64 ? &a.v_map64 : &a.v_map))
                         : "memory");
        }
        Cursor pre = c0;
        int32_t idc = lane < 8 ? fetch_tile_box_id(a, pre, lane >> 2, lane & 3) : kNoBlock;
        int j = 0;
        for (; j < n; ++j) {
            const int r = j % RING;
            if (j >= RING &&
                !__all_sync(0xffffffffu, wait_phase(tfree + r, (uint32_t)(j / RING - 1) & 1u, abort_flag)))
                break;
            Cursor nx = pre;
            cursor_next(nx, a, groups);
            const int32_t id_next = (lane < 8 && j + 1 < n) ? fetch_tile_box_id(a, nx, lane >> 2, lane & 3) : kNoBlock;
            issue_block(a, pre, lane, idc, base + C::OFF_RING + r * C::STAGE, scl + r * 2 * BT, tfull + 2 * r,
                        box_ok + r * C::BOXES);
            idc = id_next;
            pre = nx;
        }
        if (*abort_flag && lane == 0) {
            // let the copies still in flight land before the CTA leaves (bounded): the last
            // block issued into each stage
            for (int jj = max(0, j - RING); jj < j; ++jj)
                for (int t = 0; t < 2; ++t)
                    mbar_wait_bounded(tfull + 2 * (jj % RING) + t, (uint32_t)(jj / RING) & 1u);
        }
    } else if (warp == 12) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            // descriptors of the shared-memory operands at their buffers' starts
            const uint64_t qdesc0 = umma_sdesc(smem_u32(qh), C::Q_SC, C::Q_SR);
            const uint64_t vdesc0 = umma_sdesc(smem_u32(base + C::OFF_RING), C::V_SR, C::V_SC);
            const uint64_t pdesc0 = umma_sdesc(smem_u32(ph), C::P_SR, C::P_SC);
            Cursor cur = c0;
            int n_qk = 0, n_pv = 0, piece = -1, qpiece = -1;
            uint32_t first_bits = 0;  // bit (j & 31): block j starts a piece
            bool ok = true;
            for (int i = 0; i < n && ok; ++i) {
                const int buf = bufd(i);
                const bool first = i == 0 || cur.blk == 0;
                if (first) {
                    first_bits |= 1u << (i & 31);
                    ++qpiece;
                } else {
                    first_bits &= ~(1u << (i & 31));
                }
                // S^T(i) = K(i) Q^T: K from tensor memory, Q (this piece's buffer) from shared
                // memory.  The S buffer [buf] was read by softmax(i-DEPTH), waited for before
                // O^T(i-DEPTH) was issued.
                if (!wait_phase(kready + buf, phd(i), abort_flag))
                    break;
                tc_fence_after();
                const uint64_t qd = desc_add(qdesc0, (uint32_t)(qpiece & 1) * NH * D * 2);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_f16_ts(tmem + C::S_COL + (uint32_t)buf * NH, tmem + C::K_COL + (uint32_t)buf * 64 + 8 * kk,
                                desc_add(qd, kk * 2 * C::Q_SC), IDESC_QK, kk > 0);
                umma_commit(sfull + buf);
                ++n_qk;
                if (i >= 1)
                    ok = issue_pv(i - 1, first_bits, piece, n_pv, tmem, vdesc0, pdesc0, pready, vready, ofree, odone,
                                  tfree, abort_flag);
                cursor_next(cur, a, groups);
            }
            if (ok && n_qk == n)
                issue_pv(n - 1, first_bits, piece, n_pv, tmem, vdesc0, pdesc0, pready, vready, ofree, odone, tfree,
                         abort_flag);
            if (*abort_flag) {
                // let the tensor core finish what was issued (bounded)
                if (n_qk > 0)
                    mbar_wait_bounded(sfull + bufd(n_qk - 1), phd(n_qk - 1));
                if (n_pv > 0)
                    mbar_wait_bounded(odone + bufd(n_pv - 1), phd(n_pv - 1));
            }
        }
    } else {
        // ================================================================ softmax
        // thread (token tok, head half hh): warps 4-7 take heads 0-15 of their tokens,
        // warps 8-11 heads 16-31; tensor-memory lanes by warp % 4
        constexpr int NHH = NH / 2;
        const int sw = warp - 4, hh = sw >> 2, tok = 32 * (warp & 3) + lane;
        // per head: this token's sum of p.  The reference maxima (log2 domain),
        // the same in every softmax thread, live in mref (shared memory).
        float l_acc[NHH];
        int E_run = -100;         // running power-of-two bound of the V scales
        float gh = 0.f;           // log2-domain factor of the raw scores of the piece
        int piece = -1, piece_first_i = 0;
        bool piece_from_start = false;
        Cursor cur = c0;
        for (int i = 0; i < n; ++i) {
            const int buf = bufd(i);
            const bool first = (i == 0) || cur.blk == 0;
            const bool last = (i == n - 1) || cur.blk == cur.nblk - 1;
            if (first) {
                ++piece;
                piece_first_i = i;
                piece_from_start = cur.blk == 0;
                E_run = -100;
#pragma unroll
                for (int j = 0; j < NHH; ++j)
                    l_acc[j] = 0.f;
            }
            bool ok = wait_phase(kready + buf, phd(i), abort_flag);
            // the scales (and the piece's Q factor) are in place once K(i) is
            const float *scb = sc + buf * 3 * BT;
            const float ksv = scb[tok], vsv = scb[BT + tok];
            const bool valid = scb[2 * BT + tok] != 0.f;
            if (first)
                gh = cred[4 + (piece & 3)];  // 4 slots: the converters run up to DEPTH blocks ahead
            float mr[NHH];  // the reference maxima of this thread's heads, in registers while they hold
            if (!first) {
#pragma unroll
                for (int q = 0; q < NHH / 4; ++q) {
                    const float4 m4 = reinterpret_cast<const float4 *>(mref + NHH * hh)[q];
                    mr[4 * q] = m4.x;
                    mr[4 * q + 1] = m4.y;
                    mr[4 * q + 2] = m4.z;
                    mr[4 * q + 3] = m4.w;
                }
            }
            ok = ok && wait_phase(sfull + buf, phd(i), abort_flag);
            tc_fence_after();
            uint32_t sr[NHH];
            tmem_ld16(tmem + lane_base + C::S_COL + (uint32_t)buf * NH + NHH * hh, sr);
            tmem_wait_ld();
            {
                // take the K codes' bias off the scores: kBias * sum_d Q[h][d] per head, summed in
                // a fixed order at the piece's first block (and kept for its later blocks)
                float bq[NHH];
                if (first) {
                    const float4 *qp = reinterpret_cast<const float4 *>(qpart + (piece & 3) * 4 * NH + NHH * hh);
#pragma unroll
                    for (int q = 0; q < NHH / 4; ++q) {
                        const float4 p0 = qp[q], p1 = qp[NH / 4 + q], p2 = qp[NH / 2 + q], p3 = qp[3 * NH / 4 + q];
                        bq[4 * q] = kBias * (((p0.x + p1.x) + p2.x) + p3.x);
                        bq[4 * q + 1] = kBias * (((p0.y + p1.y) + p2.y) + p3.y);
                        bq[4 * q + 2] = kBias * (((p0.z + p1.z) + p2.z) + p3.z);
                        bq[4 * q + 3] = kBias * (((p0.w + p1.w) + p2.w) + p3.w);
                    }
                    if ((sw & 3) == 0 && lane == 0) {
#pragma unroll
                        for (int j = 0; j < NHH; ++j)
                            bsum[NHH * hh + j] = bq[j];  // read from the next block on, after the barrier below
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < NHH / 4; ++q) {
                        const float4 b4 = reinterpret_cast<const float4 *>(bsum + NHH * hh)[q];
                        bq[4 * q] = b4.x;
                        bq[4 * q + 1] = b4.y;
                        bq[4 * q + 2] = b4.z;
                        bq[4 * q + 3] = b4.w;
                    }
                }
#pragma unroll
                for (int j = 0; j < NHH; ++j)
                    sr[j] = __float_as_uint(__uint_as_float(sr[j]) - bq[j]);
            }
            const float kg = ksv * gh;  // raw score -> log2 domain
            // a piece's first block always moves the references (they start at -inf)
            bool need = valid && (first || !(vsv <= exp2i(E_run)));
            if (!first) {
#pragma unroll
                for (int j = 0; j < NHH; ++j)
                    need |= valid && !(fmaf(__uint_as_float(sr[j]), kg, -mr[j]) <= 8.f);
            }
            if (named_bar_or(BAR_SM, 256, need || !ok)) {
                if (named_bar_or(BAR_SM, 256, !ok))
                    break;  // abort (every softmax thread leaves here together)
                // rare: move the references to the block maxima (and the V-scale bound)
                {
                    float mv[NHH];
#pragma unroll
                    for (int j = 0; j < NHH; ++j)
                        mv[j] = valid ? __uint_as_float(sr[j]) * kg : -INFINITY;
                    const float wm = warp_transpose_reduce16<true>(mv, lane);  // head lane % 16's warp max
                    if (lane < NHH)
                        red[sw * NHH + lane] = wm;
                }
                float vm = valid ? vsv : 0.f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                if (lane == 0)
                    red[8 * NHH + sw] = vm;
                named_bar(BAR_SM, 256);
                float vmax = red[8 * NHH];
#pragma unroll
                for (int k = 1; k < 8; ++k)
                    vmax = fmaxf(vmax, red[8 * NHH + k]);
                const int E_new = max(E_run, ceil_log2_pow(vmax));
                const int dE = E_run - E_new;
                const float escale = dE < -126 ? 0.f : exp2i(dE);
                // warp 4 moves the references (lane = head, over the 4 warps of its half)
                if (sw == 0) {
                    const int h = lane, base4 = 4 * (h >> 4) * NHH + (h & 15);
                    const float bm = fmaxf(fmaxf(red[base4], red[base4 + NHH]),
                                           fmaxf(red[base4 + 2 * NHH], red[base4 + 3 * NHH]));
                    const float mo = first ? -INFINITY : mref[h];
                    const float mn = fmaxf(mo, bm);
                    mref[h] = mn;
                    ofac_s[h] = (mn == -INFINITY) ? 1.f : fast_exp2(mo - mn);
                }
                named_bar(BAR_SM, 256);
#pragma unroll
                for (int j = 0; j < NHH; ++j)
                    l_acc[j] *= ofac_s[NHH * hh + j];
                E_run = E_new;
                if (!first) {
                    // O of this piece, once O^T(i-1) has landed: row d = tok, this thread's 16 heads
                    wait_phase(odone + bufd(i - 1), phd(i - 1), abort_flag);
                    tc_fence_after();
                    const uint32_t o_col = C::O_COL + (uint32_t)(piece & 1) * NH + NHH * hh;
                    uint32_t orr[16];
                    tmem_ld16(tmem + lane_base + o_col, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        orr[j] = __float_as_uint(__uint_as_float(orr[j]) * (ofac_s[NHH * hh + j] * escale));
                    tmem_st16(tmem + lane_base + o_col, orr);
                    tmem_wait_st();
                }
                named_bar(BAR_SM, 256);  // reductions read before red is reused
#pragma unroll
                for (int q = 0; q < NHH / 4; ++q) {
                    const float4 m4 = reinterpret_cast<const float4 *>(mref + NHH * hh)[q];
                    mr[4 * q] = m4.x;
                    mr[4 * q + 1] = m4.y;
                    mr[4 * q + 2] = m4.z;
                    mr[4 * q + 3] = m4.w;
                }
            }
            // ---- P' = 2^(score - ref) * s_v * 2^(6-E) as fp16: row tok, heads 16hh .. 16hh+15 of P'[buf]
            if (i >= C::DEPTH)  // P' buffer [buf] free once O^T(i-DEPTH) is done
                wait_phase(odone + buf, phd(i - C::DEPTH), abort_flag);
            const float vf = valid ? vsv * exp2i(6 - E_run) : 0.f;
            uint8_t *pb = ph + buf * BT * NH * 2;
#pragma unroll
            for (int q = 0; q < NHH / 8; ++q) {
                uint32_t pk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j0 = 8 * q + 2 * k;
                    const float p0 = valid ? fast_exp2(fmaf(__uint_as_float(sr[j0]), kg, -mr[j0])) : 0.f;
                    const float p1 = valid ? fast_exp2(fmaf(__uint_as_float(sr[j0 + 1]), kg, -mr[j0 + 1])) : 0.f;
                    l_acc[j0] += p0;
                    l_acc[j0 + 1] += p1;
                    pk[k] = pack_half2(p0 * vf, p1 * vf);
                }
                *reinterpret_cast<uint4 *>(pb + core_off(tok, NHH * hh + 8 * q, C::P_SR, C::P_SC)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(pready + buf);
            if (last) {
                // ---- epilogue of the piece: l per head over the 128 token rows, normalise O
                wait_phase(odone + buf, phd(i), abort_flag);  // O^T(i) landed
                tc_fence_after();
                {
                    float lv[NHH];
#pragma unroll
                    for (int j = 0; j < NHH; ++j)
                        lv[j] = l_acc[j];
                    const float ws = warp_transpose_reduce16<false>(lv, lane);  // head lane % 16's warp sum
                    if (lane < NHH)
                        red[sw * NHH + lane] = ws;
                }
                const bool whole_pair = piece_from_start && cur.blk == cur.nblk - 1;
                const int slot = piece_first_i == 0 ? 0 : 1;
                named_bar(BAR_SM, 256);
                if (sw == 0) {
                    // head lane: l, the output factor 2^(E-6) / l and (for a partial) the lse
                    const int h = lane, base4 = 4 * (h >> 4) * NHH + (h & 15);
                    const float l = red[base4] + red[base4 + NHH] + red[base4 + 2 * NHH] + red[base4 + 3 * NHH];
                    ofac_s[h] = l > 0.f ? __fdividef(exp2i(E_run - 6), l) : 0.f;
                    if (!whole_pair && cur.g * NH + h < a.num_q_heads)
                        a.lse[(size_t)(2 * cta + slot) * NH + h] =
                            l > 0.f ? (mref[h] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                }
                const uint32_t o_col = C::O_COL + (uint32_t)(piece & 1) * NH + NHH * hh;
                uint32_t ov[NHH];
                tmem_ld16(tmem + lane_base + o_col, ov);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(ofree + (piece & 1));
                named_bar(BAR_SM, 256);  // ofac_s ready
                const int nh = min(NH, a.num_q_heads - cur.g * NH);  // heads of this group that exist
                if (whole_pair) {
                    __nv_bfloat16 *dst = a.out + ((size_t)cur.b * a.num_q_heads + cur.g * NH + NHH * hh) * D + tok;
#pragma unroll
                    for (int j = 0; j < NHH; ++j)
                        if (NHH * hh + j < nh)
                            dst[(size_t)j * D] = __float2bfloat16_rn(__uint_as_float(ov[j]) * ofac_s[NHH * hh + j]);
                } else {
                    float *dst = a.o_partial + ((size_t)(2 * cta + slot) * NH + NHH * hh) * D + tok;
#pragma unroll
                    for (int j = 0; j < NHH; ++j)
                        dst[(size_t)j * D] = __uint_as_float(ov[j]) * ofac_s[NHH * hh + j];
                }
                if (!whole_pair && cur.blk == cur.nblk - 1 && sw == 0 && lane == 0) {
                    // the pair's last piece: describe the pair for the merge kernel
                    const long long g0 = list_first + i - cur.blk, g1 = g0 + cur.nblk - 1;
                    const int c_lo = cta_of(g0, list_n, Ge), c_hi = cta_of(g1, list_n, Ge);
                    int *m = a.merge_desc + (2 * cta + slot) * 8;
                    m[0] = cur.b;
                    m[1] = cur.g;
                    m[2] = c_lo;
                    m[3] = c_hi;
                    m[4] = (list_n * c_lo / Ge == g0) ? 0 : 1;  // slot of the pair in CTA c_lo
                }
                named_bar(BAR_SM, 256);  // red and ofac_s are reused by the next piece
            }
            cursor_next(cur, a, groups);
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (aborted && tid == 0)
        set_status(a.dev_status, MQA_DEV_TIMEOUT);
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Merge the pieces of one cut (sequence, head group) pair, 8 heads per CTA:
// warp k takes head 8 blockIdx.y + k, lane d = 4 lane .. 4 lane + 3.  The
// flash-decoding combine: M = max lse, w = exp(lse - M), out = sum w o / sum w.
// A cut pair's last piece always opens its CTA's share, so its descriptor is in
// slot 0 of CTA blockIdx.x.
__global__ void __launch_bounds__(256) decode_tc_merge_kernel(const __grid_constant__ DecodeArgs a)
{
    constexpr int NH = TcCfg::NH, D = TcCfg::D;
    const int *m = a.merge_desc + (2 * blockIdx.x) * 8;
    const int b = __ldg(m);
    if (b < 0)
        return;
    const int g = __ldg(m + 1), c_lo = __ldg(m + 2), c_hi = __ldg(m + 3), slot_lo = __ldg(m + 4);
    const int np = c_hi - c_lo + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jh = blockIdx.y * 8 + warp, h = g * NH + jh;
    if (h >= a.num_q_heads)
        return;
    float M = -INFINITY;
    for (int p = lane; p < np; p += 32)
        M = fmaxf(M, __ldg(a.lse + merge_row(c_lo, p, slot_lo, jh)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < np; p0 += 8) {
        float wgt[8];
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = min(p0 + u, np - 1);
            const size_t row = merge_row(c_lo, p, slot_lo, jh);
            const float ls = __ldg(a.lse + row);
            wgt[u] = (p0 + u >= np || ls == -INFINITY || M == -INFINITY) ? 0.f : __expf(ls - M);
            x[u] = __ldg(reinterpret_cast<const float4 *>(a.o_partial + row * D) + lane);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            den += wgt[u];
            acc.x += wgt[u] * x[u].x;
            acc.y += wgt[u] * x[u].y;
            acc.z += wgt[u] * x[u].z;
            acc.w += wgt[u] * x[u].w;
        }
    }
    const float f = den > 0.f ? 1.f / den : 0.f;
    uint2 o;
    o.x = pack_bf16x2(acc.x * f, acc.y * f);
    o.y = pack_bf16x2(acc.z * f, acc.w * f);
    *reinterpret_cast<uint2 *>(a.out + ((size_t)b * a.num_q_heads + h) * D + 4 * lane) = o;
}

cudaError_t launch_decode_tc(const DecodeArgs &a, cudaStream_t s)
{
    static std::atomic<int> attr_set{0};
    if (!attr_set.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             TcCfg::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_set.store(1, std::memory_order_release);
    }
    decode_tc_kernel<<<a.persist_ctas, TcCfg::THREADS, TcCfg::SMEM_BYTES, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !a.persistent)
        return e;
    decode_tc_merge_kernel<<<dim3(a.persist_ctas, TcCfg::NH / 8), 256, 0, s>>>(a);
    return cudaGetLastError();
}

int decode_tc_ctas_per_sm()
{
    int n = 0;
    cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM_BYTES);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_tc_kernel, TcCfg::THREADS, TcCfg::SMEM_BYTES) !=
        cudaSuccess)
        n = 1;
    return n < 1 ? 1 : n;
}

}  // namespace mqa
