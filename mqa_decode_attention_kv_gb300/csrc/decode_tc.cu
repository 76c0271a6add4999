// Decode attention on the 5th-generation tensor cores (tcgen05): one persistent
// kernel with worker warpgroups.  A key block is 128 rows of 128 code bytes
// (tensor-memory lanes): 128 tokens at head_dim 128, 256 tokens at head_dim 64
// (two tokens a row; see TcMode).  A head group is 32 query heads at head_dim
// 128 (fewer heads leave zero-query columns) and 16 at head_dim 64.
//
// Work.  The call's (sequence b, head group g, key block) triples
// form one list, ordered by b, then g, then block.  In the balanced mode CTA c
// of the first G' = min(G, N) CTAs takes the contiguous share
// [c*N/G', (c+1)*N/G') of the N list entries (never empty), so every CTA
// streams the same number of blocks (+-1) whatever the length mix and its
// pipeline runs across sequence boundaries without draining.  A piece of a
// (b, g) pair that lies inside one share is the whole pair: its output is
// written directly (bf16).  A pair cut by share boundaries leaves an fp32
// partial (O, lse) per piece in slot 0 (the share's first piece) or 1 (its
// last) of the CTA that computed it, and the CTA holding its last piece writes
// a merge descriptor; a second kernel merges every cut pair, a CTA per (pair,
// 8 heads).  Each CTA rewrites both of its descriptor slots on every call, so
// the workspace needs no zeroing.  In the whole-pair mode CTA c computes pair
// c alone and needs no workspace.
//
// Roles (12 warps, one CTA per SM):
//   warps 0-7   two worker warpgroups.  Worker group w takes the CTA's blocks
//               i with i % 2 == w, whole: thread t owns row t (= tensor
//               memory lane t).  Per block it converts the K codes to fp16
//               (kept with their exponent bias +1152) straight into its K
//               buffer in tensor memory (the A operand of S^T = K Q^T), the V
//               codes to fp16 in place in the ring stage (the A operand of
//               O^T += V^T P'), then reads its row's 32 scores, takes the K
//               bias off, applies the K scale and writes
//               P' = 2^(score - ref) * s_v * 2^(6-E) (fp16) for the MMA.  Each
//               group keeps its own per-head reference maxima (moved only when
//               a score passes them by more than 2^8, or at the group's first
//               block of a piece), its own power-of-two bound 2^E of the V
//               scales, its own row sums and its own O accumulator in tensor
//               memory; the group that computes a piece's last block merges
//               both groups' (O, ref, sum, E) into the piece's result.  The
//               group that computes a piece's first block converts its Q
//               (bulk-copied a piece ahead) into the B operand of S^T, scaled
//               by one exact power of two, and sums it per head for the bias.
//   warps 8-11  the control warpgroup (its registers go to the workers):
//               lane 0 of warp 8 (group 0) and of warp 10 (group 1) issue
//               their group's tcgen05.mma and commits, S^T(i) as soon as K(i)
//               is in tensor memory and O^T_w += V^T(i) P'(i) once P'(i) is
//               written; warp 8 owns the tensor-memory allocation.  Warp 9
//               is the TMA producer: block ids a block ahead, the codes and
//               scales of each block into a ring stage once the O^T update
//               that read the stage's previous block has completed.  Warp 11
//               idles.
//
// Every int8 code is converted exactly once (exponent-bias trick, exact), the
// scores and O accumulate in fp32 tensor memory.  Every wait is bounded: a
// wait that runs out raises a CTA-wide abort flag; every role then leaves at
// its next exit point (the worker groups all together, at a barrier that ORs
// the flag), copies and MMAs still in flight are drained first, and the call
// reports MQA_DEV_TIMEOUT.
//
// The kernel is launched with programmatic stream serialisation: barrier and
// tensor-memory set-up overlap the previous kernel on the stream, and every
// global access comes after griddep_wait().
#include <atomic>
#include <cfloat>
#include <math.h>

#include "common.cuh"
#include "kv_stage.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace mqa {
namespace {

struct TcCfg {
    static constexpr int D = 128;
    static constexpr int NH = 32;                    // heads per group (MMA N)
    static constexpr int BT = 128;                   // rows per block (M of S^T, K of O^T)
    static constexpr int SCL_TOK = 2 * BT;           // token scales per stage and tensor (up to 256 tokens)
    static constexpr int BOXES = SCL_TOK / kChunkTokens;  // box flags per stage (16 tokens a box)
    static constexpr int NW = 2;                     // worker warpgroups
    static constexpr int RING = 5;                   // ring stages (codes in flight, then fp16 V)
    // a control warpgroup after the workers: the MMA warp, the TMA warp and two idle warps
    static constexpr int MMA_WARP = 4 * NW, TMA_WARP = 4 * NW + 1;
    static constexpr int THREADS = 32 * (4 * NW + 4);
    // registers per thread: at launch (one CTA per SM), then moved from the control group to
    // the workers with setmaxnreg; the split must fit what the CTA was launched with
    static constexpr int REG_LAUNCH = (65536 / THREADS) / 8 * 8;
    static constexpr int REG_CTRL = 88;
    static constexpr int REG_WORK = ((REG_LAUNCH * THREADS - 128 * REG_CTRL) / (128 * NW)) / 8 * 8;
    static constexpr int CODES = BT * D;             // int8 bytes of K (or V) of a block
    static constexpr int STAGE = 2 * CODES;          // K codes, V codes; then fp16 V in place
    // shared memory (offsets from a 1024-aligned base)
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_QH = OFF_RING + RING * STAGE;     // [2 slots] fp16 Q [32 h][128 d], core layout
    static constexpr int QH_SLOT = NH * D * 2;                 // one slot of fp16 Q
    static constexpr int OFF_QRAW = OFF_QH + 2 * QH_SLOT;      // bf16 Q [<= 32 h][<= 128 d] as copied (next piece)
    static constexpr int OFF_PH = OFF_QRAW + NH * D * 2;       // [NW] fp16 P' [128 tok][32 h], core layout
    static constexpr int OFF_SCL = OFF_PH + NW * BT * NH * 2;  // [RING][2][SCL_TOK] fp32 K, V token scales (TMA)
    static constexpr int OFF_OK = OFF_SCL + RING * 2 * SCL_TOK * 4;  // [RING][BOXES] box arrived
    // per worker group: red [4 warps][32], vred [4], mref [32], fac [NW][32]
    static constexpr int WG_RED = 0, WG_VRED = 512, WG_MREF = 528, WG_FAC = 656;
    static constexpr int WG_BYTES = (WG_FAC + NW * NH * 4 + 15) / 16 * 16;
    static constexpr int OFF_WG = OFF_OK + RING * BOXES * 4;
    // per piece slot (2): bias [32], gh, then per group: ref [32], sum [32], E
    static constexpr int SL_BIAS = 0, SL_GH = 128, SL_GRP = 144, SL_GRP_BYTES = 272;
    static constexpr int SLOT_BYTES = (SL_GRP + NW * SL_GRP_BYTES + 15) / 16 * 16;
    static constexpr int OFF_SLOT = OFF_WG + NW * WG_BYTES;
    static constexpr int OFF_MISC = OFF_SLOT + 2 * SLOT_BYTES;  // tmem base, abort flag, start position, share
    static constexpr int OFF_MBAR = OFF_MISC + 256;
    static constexpr int NBAR = 3 * RING + 5 * NW + 7;
    static constexpr int SMEM_BYTES = OFF_MBAR + 8 * NBAR + 1024;
    // tensor memory columns: S^T [NW][32], O^T [NW][2][32], fp16 K [NW][64]
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0, O_COL = NW * NH, K_COL = O_COL + 2 * NW * NH;
    // core-matrix strides (bytes): V rows = tokens, Q rows = heads, P rows = tokens.  The fp16
    // V of token group warp j (tokens 32j .. 32j+31) overwrites the 8 KB of codes they came
    // from: 8-token groups 0, 1 of the warp at K-half offset 4096j, groups 2, 3 at V-half
    // offset 4096j, each group 16 core matrices (8 d each) of 128 B.
    static constexpr uint32_t V_SR = 16 * 128;  // next 8 tokens (inside a 16-token MMA step)
    static constexpr uint32_t V_SC = 128;       // next 8 d
    static constexpr uint32_t Q_SR = 16 * 128;  // next 8 heads
    static constexpr uint32_t Q_SC = 128;       // next 8 d
    static constexpr uint32_t P_SR = 4 * 128;   // next 8 tokens
    static constexpr uint32_t P_SC = 128;       // next 8 heads
};
static_assert(TcCfg::SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(TcCfg::RING >= TcCfg::NW + 1, "the ring must hold every group's block and one more");
static_assert(TcCfg::NW <= 3, "the control warpgroup has one MMA issuer per worker group, besides the TMA warp");
static_assert(TcCfg::REG_WORK <= 256 && TcCfg::REG_WORK >= TcCfg::REG_LAUNCH &&
                  128 * (TcCfg::NW * TcCfg::REG_WORK + TcCfg::REG_CTRL) <= TcCfg::REG_LAUNCH * TcCfg::THREADS,
              "register split within the launch allocation");
// 128-byte-swizzled TMA destinations and descriptor bases on 1024 B; bulk copies, vector
// loads and stores on 16 B; mbarriers on 8 B
static_assert(TcCfg::OFF_RING % 1024 == 0 && TcCfg::STAGE % 1024 == 0 && TcCfg::OFF_QH % 1024 == 0 &&
                  TcCfg::OFF_PH % 1024 == 0,
              "1024-byte alignment");
static_assert(TcCfg::OFF_QRAW % 16 == 0 && TcCfg::OFF_SCL % 16 == 0 && TcCfg::OFF_OK % 16 == 0 &&
                  TcCfg::OFF_WG % 16 == 0 && TcCfg::WG_BYTES % 16 == 0 && TcCfg::WG_MREF % 16 == 0 &&
                  TcCfg::WG_FAC % 16 == 0 && TcCfg::OFF_SLOT % 16 == 0 && TcCfg::SLOT_BYTES % 16 == 0 &&
                  TcCfg::SL_GRP % 16 == 0 && TcCfg::SL_GRP_BYTES % 16 == 0 && TcCfg::OFF_MISC % 16 == 0 &&
                  TcCfg::OFF_MBAR % 8 == 0,
              "16-byte alignment");
static_assert(TcCfg::K_COL + TcCfg::NW * 64 <= TcCfg::TMEM_COLS, "tensor memory budget");

// The two row formats of a key block (128 rows of 128 code bytes = tensor-memory lanes):
// head_dim 128, a row is one token; head_dim 64, a row is two consecutive tokens (the
// cache's bytes as they lie: the second token's codes are columns 64-127).  With pairs
// the 32 MMA columns are (token of the row, head): columns 0-15 hold heads 0-15 of
// the row's first token, columns 16-31 the same heads of its second; the B operand Q
// of S^T = K Q^T holds head h's query in columns 0-63 of column h and 64-127 of column
// h + 16 (zeros elsewhere), so each column scores one token, and O^T += V^T P' leaves
// the first token's sums in rows 0-63 of columns 0-15 and the second's in rows 64-127
// of columns 16-31 (the other quadrants are discarded).  Each column keeps its own
// softmax state; the epilogue merges the two columns of a head.  Groups with fewer
// heads than columns (8 or 16 query heads) leave the rest of their columns at a zero
// query, computed and discarded.
template <bool PAIR>
struct TcMode {
    static constexpr int TPR = PAIR ? 2 : 1;                        // tokens per row
    static constexpr int DH = TcCfg::D / TPR;                       // head_dim
    static constexpr int NHG = TcCfg::NH / TPR;                     // query heads per group
    static constexpr int TILES = 2 * TPR;                           // 64-token tiles per block
    static constexpr int BOXES = TcCfg::BT * TPR / kChunkTokens;    // 16-token boxes per block
    static_assert(BOXES <= TcCfg::BOXES && TcCfg::BT * TPR <= TcCfg::SCL_TOK, "stage flags and scales");
};

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

// Key blocks of a sequence of length L: the 64-token tiles from the one
// holding the window start to the one holding L-1, grouped TILES to a block
// (the last block may hold fewer).  0 for an invalid length.
template <int TILES>
__device__ __forceinline__ int seq_blocks(int L, int window, int max_seq_len, int &t_first, int &lo)
{
    t_first = 0;
    lo = 0;
    if (L < 1 || L > max_seq_len)
        return 0;
    lo = (window > 0 && L > window) ? L - window : 0;
    t_first = lo / kTileTokens;
    const int t_last = (L - 1) / kTileTokens;
    return (t_last - t_first + TILES) / TILES;
}

// Position in the (sequence, head group, block) list.
struct Cursor {
    int b, g, blk;      // sequence, head group, block of the sequence
    int nblk;           // blocks of sequence b
    int t_first, lo, L; // first tile, window start, length of sequence b
};

// Load sequence b's shape into the cursor; then skip sequences without blocks.
template <int TILES>
__device__ __forceinline__ void cursor_seek(Cursor &c, const DecodeArgs &a)
{
    while (c.b < a.batch) {
        c.L = __ldg(a.seq_lens + c.b);
        c.nblk = seq_blocks<TILES>(c.L, a.window, a.max_seq_len, c.t_first, c.lo);
        if (c.nblk > 0)
            return;
        ++c.b;
        c.g = 0;
        c.blk = 0;
    }
}

template <int TILES>
__device__ __forceinline__ void cursor_next(Cursor &c, const DecodeArgs &a, int groups)
{
    if (++c.blk < c.nblk)
        return;
    c.blk = 0;
    if (++c.g < groups)
        return;
    c.g = 0;
    ++c.b;
    cursor_seek<TILES>(c, a);
}

// The CTA whose share holds list entry x (the largest c with floor(c*N/G) <= x).
__device__ __forceinline__ int cta_of(long long x, long long N, int G)
{
    return (int)(((x + 1) * G - 1) / N);
}

// Four codes (byte i = code c_i) -> lo = {c0, c1} + kBias, hi = {c2, c3} + kBias as f16x2,
// exact: the exponent-bias conversion (0x64xx = 1024 + byte, on the codes offset by 128)
// without its final subtraction.  K enters S^T = K Q^T this way; the bias adds
// kBias * sum_d Q[h][d] to every score of head h, which the worker groups take off in fp32.
constexpr float kBias = 1152.f;
__device__ __forceinline__ void i8x4_to_f16x2x2_biased(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t t = w ^ 0x80808080u;
    lo = __byte_perm(t, 0x64646464u, 0x5140);
    hi = __byte_perm(t, 0x64646464u, 0x7362);
}

// Partial-output row of piece s (0 = the pair's first piece, in CTA c_lo) of a
// merged pair: CTA c_lo + s, slot slot_lo for s == 0 else 0, head jh; a slot
// holds hs rows (the heads of a group that exist).
__device__ __forceinline__ size_t merge_row(int c_lo, int s, int slot_lo, int jh, int hs)
{
    return (size_t)(2 * (c_lo + s) + (s == 0 ? slot_lo : 0)) * hs + jh;
}

// Whether worker group w computes a block of the piece whose blocks are list
// positions [i0, i0 + nb) (block i goes to group i % NW).
__device__ __forceinline__ bool group_in_piece(int w, int i0, int nb)
{
    return nb >= TcCfg::NW || ((w - i0 % TcCfg::NW + TcCfg::NW) % TcCfg::NW) < nb;
}

}  // namespace

__device__ __forceinline__ void regs_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(TcCfg::REG_WORK));
}
__device__ __forceinline__ void regs_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(TcCfg::REG_CTRL));
}

template <bool PAIR>
__global__ void __launch_bounds__(TcCfg::THREADS, 1) decode_tc_kernel(const __grid_constant__ DecodeArgs a)
{
    using C = TcCfg;
    using MD = TcMode<PAIR>;
    // D, NH: a row's code bytes and the MMA columns; DH, NHG: head_dim and query heads per group
    constexpr int D = C::D, NH = C::NH, RING = C::RING, BT = C::BT, NW = C::NW;
    constexpr int DH = MD::DH, NHG = MD::NHG, TPR = MD::TPR, TILES = MD::TILES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qh = base + C::OFF_QH;
    uint8_t *qraw = base + C::OFF_QRAW;
    uint8_t *ph = base + C::OFF_PH;
    uint32_t *box_ok = reinterpret_cast<uint32_t *>(base + C::OFF_OK);
    float *scl = reinterpret_cast<float *>(base + C::OFF_SCL);  // [RING][2][SCL_TOK] token scales, with the codes
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 4);
    volatile int *q_issued = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 8);  // raw Q copies issued
    int *start_pos = reinterpret_cast<int *>(base + C::OFF_MISC + 16);          // b, g, blk, n
    long long *share = reinterpret_cast<long long *>(base + C::OFF_MISC + 32);  // first entry, N, CTAs
    static_assert(32 + 3 * 8 <= 64, "misc layout");
    uint64_t *tfull = reinterpret_cast<uint64_t *>(base + C::OFF_MBAR);  // [RING][2] tile codes landed (TMA)
    uint64_t *tfree = tfull + 2 * RING;  // [RING] stage free: O^T of its block done   (tensor core)
    uint64_t *kready = tfree + RING;     // [NW] K in tensor memory (+ Q of a new piece) (4 warps)
    uint64_t *vready = kready + NW;      // [NW] fp16 V in shared memory                (4 warps)
    uint64_t *pready = vready + NW;      // [NW] P' written, S read                     (4 warps)
    uint64_t *sfull = pready + NW;       // [NW] S^T = K Q^T done                       (tensor core)
    uint64_t *odone = sfull + NW;        // [NW] O^T += V^T P' done                     (tensor core)
    uint64_t *qready = odone + NW;       // [2] the piece slot's Q, bias, factor ready  (4 warps)
    uint64_t *pdone = qready + 2;        // [2] every group is done with the piece      (4 NW warps)
    uint64_t *sfree = pdone + 2;         // [2] the piece's epilogue read slot and O    (4 warps)
    uint64_t *qfull = sfree + 2;         // raw Q of the next piece landed              (bulk copy)
    static_assert(3 * C::RING + 5 * C::NW + 7 == C::NBAR, "barrier count");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int groups = (a.num_q_heads + NHG - 1) / NHG;
    const int HS = min(a.num_q_heads, NHG);  // partial-output rows per slot: the heads of a group
    const int G = gridDim.x;
    const int cta = blockIdx.x;
    const bool balanced = a.persistent != 0;

    // ---- set-up: barriers and tensor memory (touches no global memory: overlaps the previous kernel)
    if (tid == 0) {
        for (int s = 0; s < 2 * RING; ++s)
            mbar_init(tfull + s, 1);
        for (int s = 0; s < RING; ++s)
            mbar_init(tfree + s, 1);
        for (int w = 0; w < NW; ++w) {
            mbar_init(kready + w, 4);
            mbar_init(vready + w, 4);
            mbar_init(pready + w, 4);
            mbar_init(sfull + w, 1);
            mbar_init(odone + w, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(qready + s, 4);
            mbar_init(pdone + s, 4 * NW);
            mbar_init(sfree + s, 4);
        }
        mbar_init(qfull, 1);
        *abort_flag = 0;
        *q_issued = 0;
        fence_mbar_init();
    }
    if (warp == C::MMA_WARP)
        tmem_alloc(tmem_slot, C::TMEM_COLS);
    if (warp == C::TMA_WARP && lane == 0) {
        const bool p64 = !PAIR && a.page_size == kTileTokens;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(p64 ? &a.k_map64 : &a.k_map))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(p64 ? &a.v_map64 : &a.v_map))
                     : "memory");
    }
    if (warp == C::THREADS / 32 - 1) {
        // while the previous kernel may still run: warm L2 with the lengths and, in whole-pair
        // mode, this CTA's block-table row and query rows (the first three things it reads)
        for (int off = lane * 128; off < a.batch * 4; off += 32 * 128)
            prefetch_l2(reinterpret_cast<const char *>(a.seq_lens) + off);
        if (!balanced) {
            const int bb = cta / groups, gg = cta % groups;
            const char *row = reinterpret_cast<const char *>(a.block_table + (size_t)bb * a.max_blocks);
            for (int off = lane * 128; off < a.max_blocks * 4 && off < 64 * 128; off += 32 * 128)
                prefetch_l2(row + off);
            const char *qp = reinterpret_cast<const char *>(a.q + ((size_t)bb * a.num_q_heads + gg * NHG) * DH);
            for (int off = lane * 128; off < min(NHG, a.num_q_heads - gg * NHG) * DH * 2; off += 32 * 128)
                prefetch_l2(qp + off);
        }
    }
    // the previous kernel's writes (the cache slot just appended, q, out, the workspace) are visible from here
    griddep_wait();
    griddep_launch_dependents();
    // ---- this CTA's share of the (sequence, group, block) list
    int *wsum = reinterpret_cast<int *>(base + C::OFF_WG);  // scratch of the scans (worker-group area)
    if (balanced && a.batch <= C::THREADS) {
        // one pass (a sequence per thread): its blocks, the block-wide prefix and total
        int nb = 0;
        if (tid < a.batch) {
            int tf, lo;
            nb = seq_blocks<TILES>(__ldg(a.seq_lens + tid), a.window, a.max_seq_len, tf, lo);
            if (nb == 0 && tid % G == cta) {
                set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + (size_t)tid * a.num_q_heads * DH);
                for (int k = 0; k < a.num_q_heads * DH / 8; ++k)
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
        // pass 1: blocks per group over all sequences; sequences without blocks
        // (invalid length) get a zero output from CTA b % G and a status bit
        long long mine = 0;
        for (int bb = tid; bb < a.batch; bb += C::THREADS) {
            int tf, lo;
            const int L = __ldg(a.seq_lens + bb);
            const int nb = seq_blocks<TILES>(L, a.window, a.max_seq_len, tf, lo);
            mine += nb;
            if (nb == 0 && bb % G == cta) {
                set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + (size_t)bb * a.num_q_heads * DH);
                for (int k = 0; k < a.num_q_heads * DH / 8; ++k)
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
                nb = seq_blocks<TILES>(__ldg(a.seq_lens + bb), a.window, a.max_seq_len, tf, lo);
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
        // whole-pair mode: CTA c computes (sequence c / groups, group c % groups)
        if (tid == 0) {
            const int bb = cta / groups, gg = cta % groups;
            int tf, lo;
            const int nb = seq_blocks<TILES>(__ldg(a.seq_lens + bb), a.window, a.max_seq_len, tf, lo);
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
            for (int r = tid; r < NHG * DH / 8; r += C::THREADS) {
                const int h = gg * NHG + r / (DH / 8);
                if (h < a.num_q_heads)
                    reinterpret_cast<uint4 *>(a.out + ((size_t)bb * a.num_q_heads + h) * DH)[r % (DH / 8)] =
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
    __syncthreads();  // also: the scans' scratch is free for the worker groups
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (n <= 0) {  // uniform: nothing to compute
        if (warp == C::MMA_WARP)
            tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }
    const long long list_first = share[0], list_n = share[1];
    const int Ge = (int)share[2];  // CTAs with a share (balanced mode)
    Cursor c0;
    c0.b = start_pos[0];
    c0.g = start_pos[1];
    c0.blk = start_pos[2];
    cursor_seek<TILES>(c0, a);  // loads the shape of sequence c0.b (which has blocks)
    // registers: the control warpgroup gives most of its share to the worker groups
    if (warp < 4 * NW)
        regs_inc();
    else
        regs_dec();

    if (warp < 4 * NW) {
        // ================================================================ worker groups
        const int w = warp >> 2, wj = warp & 3;
        const int tok = 32 * wj + lane;                        // row of every block = tensor-memory lane
        const uint32_t lane_base = (uint32_t)(32 * wj) << 16;  // this warp's tensor-memory lanes
        const int BAR_WG = 1 + w;                              // named barrier of this group
        uint8_t *wg = base + C::OFF_WG + w * C::WG_BYTES;
        float *red = reinterpret_cast<float *>(wg + C::WG_RED);    // [4 warps][32]
        float *vred = reinterpret_cast<float *>(wg + C::WG_VRED);  // [4]
        float *mref = reinterpret_cast<float *>(wg + C::WG_MREF);  // [32] reference maxima (log2 domain)
        float *fac = reinterpret_cast<float *>(wg + C::WG_FAC);    // [NW][32] factors
        uint8_t *pw = ph + w * BT * NH * 2;                        // this group's P'
        const uint32_t s_col = C::S_COL + (uint32_t)w * NH, k_col = C::K_COL + (uint32_t)w * 64;
        if (w == 0 && wj == 0 && lane == 0) {
            // the first piece's Q (bf16, the group's heads x head_dim, contiguous): group 0 converts it
            const uint32_t qb = (uint32_t)min(NHG, a.num_q_heads - c0.g * NHG) * DH * 2;
            *q_issued = 1;
            mbar_arrive_expect_tx(qfull, qb);
            bulk_load(qraw, a.q + ((size_t)c0.b * a.num_q_heads + c0.g * NHG) * DH, qb, qfull);
        }
        Cursor cur = c0;
        float l_acc[NH];  // this token's sum of p per head, for the current piece
#pragma unroll
        for (int h = 0; h < NH; ++h)
            l_acc[h] = 0.f;
        const float *bias = nullptr;  // kBias * sum_d Q[h][d] of the current piece (its slot)
        int E_run = -100;       // running power-of-two bound of the V scales (group-uniform)
        float gh = 0.f;         // log2-domain factor of the raw scores of the piece
        int piece = -1, piece_i0 = 0;
        bool piece_from_start = false, took = false;  // took: this group computed a block of the piece
        int jw = 0;                                   // blocks this group computed so far
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            const bool first = (i == 0) || cur.blk == 0;
            const bool last = (i == n - 1) || cur.blk == cur.nblk - 1;
            const bool mine = (i % NW) == w;
            if (first) {
                ++piece;
                piece_i0 = i;
                piece_from_start = cur.blk == 0;
                took = false;
                const int s = piece & 1;
                uint8_t *slot = base + C::OFF_SLOT + s * C::SLOT_BYTES;
                if (mine) {
                    // ---- this group converts the piece's Q into slot s (free once piece-2's
                    // epilogue read it) and sums it per column; lane = column, whose head is
                    // lane % NHG (heads past the group's last read as zero)
                    if (piece >= 2)
                        ok &= wait_phase(sfree + s, (uint32_t)((piece - 2) >> 1) & 1u, abort_flag);
                    ok &= wait_phase(qfull, (uint32_t)piece & 1u, abort_flag);
                    const int hc = lane % NHG;
                    const bool hreal = hc < min(NHG, a.num_q_heads - cur.g * NHG);
                    const uint8_t *qrow = qraw + hc * DH * 2;
                    float m = 0.f;
                    if (hreal) {
#pragma unroll
                        for (int k = 0; k < DH / 8; ++k) {
                            const uint4 qv = *reinterpret_cast<const uint4 *>(qrow + 16 * ((k + lane) & (DH / 8 - 1)));
                            const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t)
                                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[t] << 16)),
                                                   fabsf(__uint_as_float(w4[t] & 0xffff0000u))));
                        }
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
                    float qsum = 0.f;  // this warp's range of column `lane`, as the tensor core sees it
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int c = 4 * wj + ((t + lane) & 3);  // 8-wide chunk of the row: 8c .. 8c+7
                        // with pairs, chunks 0-7 face a row's first token, 8-15 its second
                        const bool live = hreal && (!PAIR || (c >> 3) == lane / NHG);
                        uint4 qv = make_uint4(0u, 0u, 0u, 0u);
                        if (live)
                            qv = *reinterpret_cast<const uint4 *>(qrow + 16 * (c % (DH / 8)));
                        const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
                        uint32_t hv[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            hv[u] = pack_half2(__uint_as_float(w4[u] << 16) * f,
                                               __uint_as_float(w4[u] & 0xffff0000u) * f);
                            const __half2 h2 = *reinterpret_cast<const __half2 *>(&hv[u]);
                            qsum += __low2float(h2);
                            qsum += __high2float(h2);
                        }
                        *reinterpret_cast<uint4 *>(qh + s * C::QH_SLOT + core_off(lane, 8 * c, C::Q_SR, C::Q_SC)) =
                            make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    }
                    red[wj * NH + lane] = qsum;
                    fence_proxy_async();  // fp16 Q for the tensor core; raw Q reads before its next copy
                    named_bar(BAR_WG, 128);
                    if (wj == 0) {
                        float *sb = reinterpret_cast<float *>(slot + C::SL_BIAS);
                        sb[lane] = kBias * (((red[lane] + red[NH + lane]) + red[2 * NH + lane]) + red[3 * NH + lane]);
                        if (lane == 0)
                            *reinterpret_cast<float *>(slot + C::SL_GH) = a.q_scale_log2 * exp2i(-e);
                        // the next piece's Q, now that every warp of the group has read this one
                        const int i_next = i + (cur.nblk - cur.blk);
                        if (lane == 0 && i_next < n && ok && !*abort_flag) {
                            Cursor nx = cur;
                            nx.blk = cur.nblk - 1;
                            cursor_next<TILES>(nx, a, groups);
                            const uint32_t qb = (uint32_t)min(NHG, a.num_q_heads - nx.g * NHG) * DH * 2;
                            *q_issued = *q_issued + 1;  // before the arrival that publishes it
                            mbar_arrive_expect_tx(qfull, qb);
                            bulk_load(qraw, a.q + ((size_t)nx.b * a.num_q_heads + nx.g * NHG) * DH, qb, qfull);
                        }
                    }
                    named_bar(BAR_WG, 128);  // red reuse; the slot's bias and factor written
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(qready + s);
                } else {
                    ok &= wait_phase(qready + s, (uint32_t)(piece >> 1) & 1u, abort_flag);
                }
                // this piece's Q factor and bias (the slot stays until the piece's epilogue)
                gh = *reinterpret_cast<const float *>(slot + C::SL_GH);
                bias = reinterpret_cast<const float *>(slot + C::SL_BIAS);
            }
            if (mine) {
                // ============================================ block i: K, V, softmax
                const int r = i % RING;
                const int pj = jw & 1;  // phase parity of this group's per-block barriers
                uint8_t *st = base + C::OFF_RING + r * C::STAGE;
                ok &= wait_done(tfull + 2 * r + (wj >> 1), (uint32_t)(i / RING) & 1u, abort_flag);
                tc_fence_after();
                const uint8_t *crow = st + tok * D;  // this row's codes (K, then V at + CODES)
                // the row's token(s): pos0 (and pos0 + 1 with pairs), in one box
                const int pos0 = (cur.t_first + TILES * cur.blk) * kTileTokens + TPR * tok;
                const bool fetched = box_ok[r * C::BOXES + ((TPR * tok) >> 4)] != 0;
                const bool valid0 = fetched && pos0 >= cur.lo && pos0 < cur.L;
                const bool valid1 = PAIR && fetched && pos0 + 1 >= cur.lo && pos0 + 1 < cur.L;
                const float *sct = scl + r * 2 * C::SCL_TOK + TPR * tok;
                const float ksv0 = fetched ? sct[0] : 0.f, vsv0 = fetched ? sct[C::SCL_TOK] : 0.f;
                const float ksv1 = PAIR && fetched ? sct[1] : 0.f;
                const float vsv1 = PAIR && fetched ? sct[C::SCL_TOK + 1] : 0.f;
                // ---- K: 128 codes -> fp16 pairs in tensor memory (lane tok, 64 columns); the
                // group's K buffer was last read by S^T of its previous block, which it waited for.
                // (A loop, not unrolled: the kernel's instruction footprint is a bottleneck of its own.)
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint4 kc[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        kc[jj] = *reinterpret_cast<const uint4 *>(crow + ((uint32_t)((4 * half + jj) ^ (tok & 7)) << 4));
                    uint32_t kr[32];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint4 kv = kc[jj];
                        i8x4_to_f16x2x2_biased(kv.x, kr[8 * jj + 0], kr[8 * jj + 1]);
                        i8x4_to_f16x2x2_biased(kv.y, kr[8 * jj + 2], kr[8 * jj + 3]);
                        i8x4_to_f16x2x2_biased(kv.z, kr[8 * jj + 4], kr[8 * jj + 5]);
                        i8x4_to_f16x2x2_biased(kv.w, kr[8 * jj + 6], kr[8 * jj + 7]);
                    }
                    tmem_st32(tmem + lane_base + k_col + 32 * half, kr);
                }
                // this token's V codes, in flight while the K stores complete
                uint4 vc[D / 16];
#pragma unroll
                for (int j = 0; j < D / 16; ++j)
                    vc[j] = *reinterpret_cast<const uint4 *>(crow + C::CODES + ((uint32_t)(j ^ (tok & 7)) << 4));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(kready + w);
                // ---- V: fp16 in place over this warp's 8 KB of codes in stage r (every lane's
                // rows are in registers): the MN-major A operand of O^T += V^T P', token group
                // g = lane / 8 of the warp at (g < 2 ? K half : V half) + 4096 wj + 2048 (g % 2),
                // row lane % 8 of its 16 core matrices
                __syncwarp();
                {
                    const int g = lane >> 3;
                    uint8_t *vb = st + (g >> 1) * C::CODES + wj * 4096 + (g & 1) * 2048 + (lane & 7) * 16;
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
                // O^T of this group's previous block done: its P' buffer and O are free, and the MMA
                // thread has consumed that block's vready / pready phases (no phase can be lapped)
                if (jw >= 1)
                    ok &= wait_done(odone + w, (uint32_t)(pj ^ 1), abort_flag);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(vready + w);
                // ---- scores of this row: S^T(i) row tok, 32 columns
                ok &= wait_done(sfull + w, (uint32_t)pj, abort_flag);
                tc_fence_after();
                uint32_t sr[NH];
                tmem_ld32(tmem + lane_base + s_col, sr);
                tmem_wait_ld();
                // raw score -> log2 domain; with pairs columns 16-31 score the row's second token
                const float kg0 = ksv0 * gh, kg1 = ksv1 * gh;
                float x[NH];
                float dmax0 = -INFINITY, dmax1 = -INFINITY;
#pragma unroll
                for (int q = 0; q < NH / 4; ++q) {
                    const float4 b4 = reinterpret_cast<const float4 *>(bias)[q];
                    const float kg = (PAIR && q >= NH / 8) ? kg1 : kg0;
                    x[4 * q] = (__uint_as_float(sr[4 * q]) - b4.x) * kg;
                    x[4 * q + 1] = (__uint_as_float(sr[4 * q + 1]) - b4.y) * kg;
                    x[4 * q + 2] = (__uint_as_float(sr[4 * q + 2]) - b4.z) * kg;
                    x[4 * q + 3] = (__uint_as_float(sr[4 * q + 3]) - b4.w) * kg;
                }
#pragma unroll
                for (int q = 0; q < NH / 4; ++q) {
                    const float4 m4 = reinterpret_cast<const float4 *>(mref)[q];
                    const float dq = fmaxf(fmaxf(x[4 * q] - m4.x, x[4 * q + 1] - m4.y),
                                           fmaxf(x[4 * q + 2] - m4.z, x[4 * q + 3] - m4.w));
                    if (PAIR && q >= NH / 8)
                        dmax1 = fmaxf(dmax1, dq);
                    else
                        dmax0 = fmaxf(dmax0, dq);
                }
                // a group's first block of a piece always moves the references (they start at -inf)
                const bool need = !took || (valid0 && (!(dmax0 <= 8.f) || !(vsv0 <= exp2i(E_run)))) ||
                                  (valid1 && (!(dmax1 <= 8.f) || !(vsv1 <= exp2i(E_run))));
                ok &= *abort_flag == 0;
                if (named_bar_or(BAR_WG, 128, need || !ok)) {
                    if (named_bar_or(BAR_WG, 128, !ok))
                        break;  // abort: the whole group leaves here together
                    // rare: move the references to the block maxima (and the V-scale bound)
                    {
                        float mv[NH];
#pragma unroll
                        for (int h = 0; h < NH; ++h)
                            mv[h] = ((PAIR && h >= NH / 2) ? valid1 : valid0) ? x[h] : -INFINITY;
                        red[wj * NH + lane] = warp_transpose_reduce<true>(mv, lane);  // head lane's warp max
                    }
                    float vm = fmaxf(valid0 ? vsv0 : 0.f, valid1 ? vsv1 : 0.f);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                    if (lane == 0)
                        vred[wj] = vm;
                    named_bar(BAR_WG, 128);
                    if (wj == 0) {
                        const int h = lane;
                        const float bm = fmaxf(fmaxf(red[h], red[NH + h]), fmaxf(red[2 * NH + h], red[3 * NH + h]));
                        const float mo = took ? mref[h] : -INFINITY;
                        const float mn = fmaxf(mo, bm);
                        mref[h] = mn;
                        fac[h] = (mn == -INFINITY) ? 1.f : fast_exp2(mo - mn);
                    }
                    const float vmax = fmaxf(fmaxf(vred[0], vred[1]), fmaxf(vred[2], vred[3]));
                    named_bar(BAR_WG, 128);
                    const int E_new = max(took ? E_run : -100, ceil_log2_pow(vmax));
                    const float escale = took ? exp2i(max(E_run - E_new, -126)) : 1.f;
                    if (took) {
                        // this group's O of the piece (its previous O^T update is done, waited
                        // above): row tok, 32 columns
                        const uint32_t o_col = C::O_COL + (uint32_t)(w * 2 + (piece & 1)) * NH;
                        uint32_t orr[NH];
                        tmem_ld32(tmem + lane_base + o_col, orr);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < NH / 4; ++q) {
                            const float4 f4 = reinterpret_cast<const float4 *>(fac)[q];
                            l_acc[4 * q] *= f4.x;
                            l_acc[4 * q + 1] *= f4.y;
                            l_acc[4 * q + 2] *= f4.z;
                            l_acc[4 * q + 3] *= f4.w;
                            orr[4 * q] = __float_as_uint(__uint_as_float(orr[4 * q]) * (f4.x * escale));
                            orr[4 * q + 1] = __float_as_uint(__uint_as_float(orr[4 * q + 1]) * (f4.y * escale));
                            orr[4 * q + 2] = __float_as_uint(__uint_as_float(orr[4 * q + 2]) * (f4.z * escale));
                            orr[4 * q + 3] = __float_as_uint(__uint_as_float(orr[4 * q + 3]) * (f4.w * escale));
                        }
                        tmem_st32(tmem + lane_base + o_col, orr);
                        tmem_wait_st();
                    } else {
#pragma unroll
                        for (int h = 0; h < NH; ++h)
                            l_acc[h] = 0.f;
                    }
                    E_run = E_new;
                    named_bar(BAR_WG, 128);  // red, vred and fac are reused
                }
                took = true;
                // ---- P' = 2^(score - ref) * s_v * 2^(6-E) as fp16: row tok of this group's P'
                const float ef = exp2i(6 - E_run);
                const float vf0 = valid0 ? vsv0 * ef : 0.f, vf1 = valid1 ? vsv1 * ef : 0.f;
#pragma unroll
                for (int q = 0; q < NH / 8; ++q) {
                    const bool valid = (PAIR && q >= NH / 16) ? valid1 : valid0;
                    const float vf = (PAIR && q >= NH / 16) ? vf1 : vf0;
                    const float4 ma = reinterpret_cast<const float4 *>(mref)[2 * q];
                    const float4 mb = reinterpret_cast<const float4 *>(mref)[2 * q + 1];
                    const float mq[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
                    uint32_t pk[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int h0 = 8 * q + 2 * k;
                        const float p0 = valid ? fast_exp2(x[h0] - mq[2 * k]) : 0.f;
                        const float p1 = valid ? fast_exp2(x[h0 + 1] - mq[2 * k + 1]) : 0.f;
                        l_acc[h0] += p0;
                        l_acc[h0 + 1] += p1;
                        pk[k] = pack_half2(p0 * vf, p1 * vf);
                    }
                    *reinterpret_cast<uint4 *>(pw + core_off(tok, 8 * q, C::P_SR, C::P_SC)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(pready + w);
                ++jw;
            }
            if (last) {
                // ============================================ end of the piece
                const int s = piece & 1;
                uint8_t *slot = base + C::OFF_SLOT + s * C::SLOT_BYTES;
                if (took) {
                    // this group's last O^T update of the piece has completed (its issuer's commit):
                    // after pdone, the epilogue may read every group's O
                    ok &= wait_phase(odone + w, (uint32_t)((jw - 1) & 1), abort_flag);
                    // this group's row sums over its 128 tokens (l_acc is consumed: the next piece
                    // starts from zero), its references and E
                    red[wj * NH + lane] = warp_transpose_reduce<false>(l_acc, lane);
                    named_bar(BAR_WG, 128);
                    if (wj == 0) {
                        float *gs = reinterpret_cast<float *>(slot + C::SL_GRP + w * C::SL_GRP_BYTES);
                        gs[lane] = mref[lane];
                        gs[NH + lane] = ((red[lane] + red[NH + lane]) + red[2 * NH + lane]) + red[3 * NH + lane];
                        if (lane == 0)
                            reinterpret_cast<int *>(gs)[2 * NH] = E_run;
                    }
                    named_bar(BAR_WG, 128);  // red reuse
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(pdone + s);
                if (mine) {
                    // this group computed the piece's last block: merge every group's share (every
                    // participant's O^T updates completed before it arrived on pdone)
                    ok &= wait_phase(pdone + s, (uint32_t)(piece >> 1) & 1u, abort_flag);
                    tc_fence_after();
                    const int nb = i - piece_i0 + 1;
                    const bool whole_pair = piece_from_start && cur.blk == cur.nblk - 1;
                    const int oslot = piece_i0 == 0 ? 0 : 1;
                    if (wj == 0) {
                        // column lane: the merged reference, sum, and every group's output factor
                        const int h = lane;
                        float M = -INFINITY;
#pragma unroll
                        for (int u = 0; u < NW; ++u)
                            if (group_in_piece(u, piece_i0, nb))
                                M = fmaxf(M, reinterpret_cast<const float *>(slot + C::SL_GRP + u * C::SL_GRP_BYTES)[h]);
                        // (a group without a block in this piece left nothing in the slot: its
                        // entries are not read at all, stale bits may be NaN)
                        float Ls = 0.f, wu[NW];
#pragma unroll
                        for (int u = 0; u < NW; ++u) {
                            const float *gs = reinterpret_cast<const float *>(slot + C::SL_GRP + u * C::SL_GRP_BYTES);
                            wu[u] = 0.f;
                            if (group_in_piece(u, piece_i0, nb) && M != -INFINITY) {
                                wu[u] = fast_exp2(gs[h] - M);
                                Ls += wu[u] * gs[NH + h];
                            }
                        }
                        // with pairs, columns h and h ^ 16 are one head (a row's two tokens):
                        // their reference Mt and sum Lt are shared, sh weighs this column's part
                        float Mt = M, Lt = Ls, sh = 1.f;
                        if (PAIR) {
                            const float Mo = __shfl_xor_sync(0xffffffffu, M, 16);
                            const float Lo = __shfl_xor_sync(0xffffffffu, Ls, 16);
                            Mt = fmaxf(M, Mo);
                            sh = M == -INFINITY ? 0.f : fast_exp2(M - Mt);
                            Lt = Ls * sh + (Mo == -INFINITY ? 0.f : Lo * fast_exp2(Mo - Mt));
                        }
#pragma unroll
                        for (int u = 0; u < NW; ++u) {
                            float f = 0.f;
                            if (Lt > 0.f && wu[u] > 0.f) {
                                const int Eu =
                                    reinterpret_cast<const int *>(slot + C::SL_GRP + u * C::SL_GRP_BYTES)[2 * NH];
                                f = __fdividef(wu[u] * sh * exp2i(Eu - 6), Lt);
                            }
                            fac[u * NH + h] = f;
                        }
                        if (!whole_pair && h < NHG && cur.g * NHG + h < a.num_q_heads)
                            a.lse[(size_t)(2 * cta + oslot) * HS + h] =
                                Lt > 0.f ? (Mt + __log2f(Lt)) * 0.69314718055994531f : -INFINITY;
                    }
                    named_bar(BAR_WG, 128);
                    float acc[NH];
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        acc[h] = 0.f;
#pragma unroll
                    for (int u = 0; u < NW; ++u) {
                        if (!group_in_piece(u, piece_i0, nb))
                            continue;  // group-uniform
                        uint32_t ov[NH];
                        tmem_ld32(tmem + lane_base + C::O_COL + (uint32_t)(u * 2 + s) * NH, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < NH / 4; ++q) {
                            const float4 f4 = reinterpret_cast<const float4 *>(fac + u * NH)[q];
                            acc[4 * q] += f4.x * __uint_as_float(ov[4 * q]);
                            acc[4 * q + 1] += f4.y * __uint_as_float(ov[4 * q + 1]);
                            acc[4 * q + 2] += f4.z * __uint_as_float(ov[4 * q + 2]);
                            acc[4 * q + 3] += f4.w * __uint_as_float(ov[4 * q + 3]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(sfree + s);  // slot s and the groups' O buffers s are free
                    const int nh = min(NHG, a.num_q_heads - cur.g * NHG);  // heads of this group that exist
                    if (PAIR) {
                        // a head's two columns meet: row d + 64 (the second tokens' sums, columns
                        // 16-31) hands them to row d through this group's P' buffer (free: the
                        // group's last O^T update of the piece has completed)
                        float *xb = reinterpret_cast<float *>(pw);  // [64 d][16 heads]
                        if (tok >= DH) {
#pragma unroll
                            for (int q = 0; q < NHG / 4; ++q)
                                reinterpret_cast<float4 *>(xb + (tok - DH) * NHG)[q] =
                                    make_float4(acc[NHG + 4 * q], acc[NHG + 4 * q + 1], acc[NHG + 4 * q + 2],
                                                acc[NHG + 4 * q + 3]);
                        }
                        named_bar(BAR_WG, 128);
                        if (tok < DH) {
#pragma unroll
                            for (int q = 0; q < NHG / 4; ++q) {
                                const float4 o4 = reinterpret_cast<const float4 *>(xb + tok * NHG)[q];
                                acc[4 * q] += o4.x;
                                acc[4 * q + 1] += o4.y;
                                acc[4 * q + 2] += o4.z;
                                acc[4 * q + 3] += o4.w;
                            }
                        }
                    }
                    if (tok < DH) {
                        if (whole_pair) {
                            __nv_bfloat16 *dst = a.out + ((size_t)cur.b * a.num_q_heads + cur.g * NHG) * DH + tok;
#pragma unroll
                            for (int h = 0; h < NHG; ++h)
                                if (h < nh)
                                    dst[(size_t)h * DH] = __float2bfloat16_rn(acc[h]);
                        } else {
                            float *dst = a.o_partial + ((size_t)(2 * cta + oslot) * HS) * DH + tok;
#pragma unroll
                            for (int h = 0; h < NHG; ++h)
                                if (h < nh)
                                    dst[(size_t)h * DH] = acc[h];
                        }
                    }
                    if (!whole_pair && cur.blk == cur.nblk - 1 && wj == 0 && lane == 0) {
                        // the pair's last piece: describe the pair for the merge kernel
                        const long long g0 = list_first + i - cur.blk, g1 = g0 + cur.nblk - 1;
                        const int c_lo = cta_of(g0, list_n, Ge), c_hi = cta_of(g1, list_n, Ge);
                        int *m = a.merge_desc + (2 * cta + oslot) * 8;
                        m[0] = cur.b;
                        m[1] = cur.g;
                        m[2] = c_lo;
                        m[3] = c_hi;
                        m[4] = (list_n * c_lo / Ge == g0) ? 0 : 1;  // slot of the pair in CTA c_lo
                    }
                    named_bar(BAR_WG, 128);  // fac is reused
                }
                // the next piece starts from empty sums (its first block sets the references)
#pragma unroll
                for (int h = 0; h < NH; ++h)
                    l_acc[h] = 0.f;
                E_run = -100;
            }
            cursor_next<TILES>(cur, a, groups);
        }
        // ---- teardown (workers): tid 0 reports a timeout and lets the last raw Q copy land
        tc_fence_before();
        bar_all();
        if (tid == 0 && *abort_flag) {
            set_status(a.dev_status, MQA_DEV_TIMEOUT);
            const int qi = *q_issued;
            if (qi > 0)
                mbar_wait_drain(qfull, (uint32_t)(qi - 1) & 1u);
        }
        return;
    } else if (warp == C::TMA_WARP) {
        // ================================================================ TMA producer
        // ring stage j % RING takes block j once O^T of block j - RING has read its V;
        // lane 4t + c fetches the block id of box c of tile t a block ahead
        Cursor pre = c0;
        int32_t idc = lane < MD::BOXES ? fetch_tile_box_id<TILES>(a, pre, lane >> 2, lane & 3) : kNoBlock;
        int j = 0;
        for (; j < n; ++j) {
            const int r = j % RING;
            if (j >= RING &&
                !__all_sync(0xffffffffu, wait_phase(tfree + r, (uint32_t)(j / RING - 1) & 1u, abort_flag)))
                break;
            Cursor nx = pre;
            cursor_next<TILES>(nx, a, groups);
            const int32_t id_next =
                (lane < MD::BOXES && j + 1 < n) ? fetch_tile_box_id<TILES>(a, nx, lane >> 2, lane & 3) : kNoBlock;
            if (PAIR)
                issue_block_pairs(a, pre, lane, idc, base + C::OFF_RING + r * C::STAGE, scl + r * 2 * C::SCL_TOK,
                                  C::SCL_TOK, tfull + 2 * r, box_ok + r * C::BOXES);
            else
                issue_block<C::SCL_TOK>(a, pre, lane, idc, base + C::OFF_RING + r * C::STAGE,
                                        scl + r * 2 * C::SCL_TOK, tfull + 2 * r, box_ok + r * C::BOXES);
            idc = id_next;
            pre = nx;
        }
        if (*abort_flag && lane == 0) {
            // let the copies still in flight land before the CTA leaves: the last block
            // issued into each stage
            for (int jj = max(0, j - RING); jj < j; ++jj)
                for (int t = 0; t < 2; ++t)
                    mbar_wait_drain(tfull + 2 * (jj % RING) + t, (uint32_t)(jj / RING) & 1u);
        }
        tc_fence_before();
        bar_all();
        return;
    } else {
        // ================================================================ MMA issuers
        // one issuing thread per worker group (warps MMA_WARP, then the warps after the TMA
        // warp): S^T(i) once the group's K(i) is in tensor memory, O^T_w += V^T(i) P'(i) once its
        // P' and V are.  Each issuer's commits track only its own MMAs, so the groups' products
        // never queue behind one another.
        const int w = warp == C::MMA_WARP ? 0 : warp - C::TMA_WARP;
        if (w < NW && lane == 0) {
            constexpr uint32_t IDESC_QK = umma_idesc_f16(128, NH, false, false);
            constexpr uint32_t IDESC_PV = umma_idesc_f16(128, NH, true, true);
            // descriptors of the shared-memory operands at their buffers' starts
            const uint64_t qdesc0 = umma_sdesc(smem_u32(qh), C::Q_SC, C::Q_SR);
            const uint64_t vdesc0 = umma_sdesc(smem_u32(base + C::OFF_RING), C::V_SR, C::V_SC);
            const uint64_t pd = desc_add(umma_sdesc(smem_u32(ph), C::P_SR, C::P_SC), w * BT * NH * 2);
            const uint32_t s_col = C::S_COL + (uint32_t)w * NH, k_col = C::K_COL + (uint32_t)w * 64;
            Cursor c = c0;
            int piece = -1, o_piece = -1, jw = 0, n_s = 0, n_pv = 0;
            for (int i = 0; i < n; ++i) {
                if (i == 0 || c.blk == 0)
                    ++piece;
                if (i % NW == w) {
                    const uint32_t pj = (uint32_t)jw & 1u;
                    // S^T(i) = K(i) Q^T: K from the group's tensor memory, Q (the piece's slot) from
                    // shared memory; the group read its S buffer's previous contents before K(i)
                    if (!wait_done(kready + w, pj, abort_flag))
                        break;
                    tc_fence_after();
                    const uint64_t qd = desc_add(qdesc0, (uint32_t)(piece & 1) * C::QH_SLOT);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_f16_ts(tmem + s_col, tmem + k_col + 8 * kk, desc_add(qd, kk * 2 * C::Q_SC), IDESC_QK,
                                    kk > 0);
                    umma_commit(sfull + w);
                    ++n_s;
                    if (!wait_done(pready + w, pj, abort_flag) || !wait_done(vready + w, pj, abort_flag))
                        break;
                    // the group's first update of a piece overwrites O buffer piece & 1, last read by
                    // the epilogue of piece - 2
                    const bool fresh = o_piece != piece;
                    if (fresh && piece >= 2 &&
                        !wait_phase(sfree + (piece & 1), (uint32_t)((piece - 2) >> 1) & 1u, abort_flag))
                        break;
                    o_piece = piece;
                    tc_fence_after();
                    const uint32_t o_col = C::O_COL + (uint32_t)(w * 2 + (piece & 1)) * NH;
                    // V: fp16 in place in ring stage i % RING; 16-token step kk = token groups 2kk,
                    // 2kk+1 of warp kk / 2, in the K half (kk even) or the V half (kk odd)
                    const uint64_t vd = desc_add(vdesc0, (i % RING) * C::STAGE);
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        umma_f16(tmem + o_col, desc_add(vd, (kk & 1) * C::CODES + (kk >> 1) * 4096),
                                 desc_add(pd, kk * 2 * C::P_SR), IDESC_PV, !fresh || kk > 0);
                    umma_commit(odone + w);
                    umma_commit(tfree + (i % RING));  // the stage's V is read: the TMA warp may refill it
                    ++n_pv;
                    ++jw;
                }
                cursor_next<TILES>(c, a, groups);
            }
            if (*abort_flag) {
                // let the tensor core finish what this thread issued: its last commit covers it all
                if (n_pv > 0)
                    mbar_wait_drain(odone + w, (uint32_t)(n_pv - 1) & 1u);
                if (n_s > 0)
                    mbar_wait_drain(sfull + w, (uint32_t)(n_s - 1) & 1u);
            }
        }
        // ---- teardown (issuers and the idle warp): the workers saw every MMA complete; the
        // MMA warp frees the tensor memory
        tc_fence_before();
        bar_all();
        if (warp == C::MMA_WARP) {
            tc_fence_after();
            tmem_dealloc(tmem, C::TMEM_COLS);
        }
        return;
    }
}

// Merge the pieces of one cut (sequence, head group) pair, 8 heads per CTA:
// warp k takes head 8 blockIdx.y + k of the group, lane d = 4 lane .. 4 lane + 3.
// The flash-decoding combine: M = max lse, w = exp(lse - M), out = sum w o / sum w.
// A cut pair's last piece always opens its CTA's share, so its descriptor is in
// slot 0 of CTA blockIdx.x.
template <bool PAIR>
__global__ void __launch_bounds__(256) decode_tc_merge_kernel(const __grid_constant__ DecodeArgs a)
{
    constexpr int NHG = TcMode<PAIR>::NHG, D = TcMode<PAIR>::DH;
    griddep_wait();
    griddep_launch_dependents();
    const int *m = a.merge_desc + (2 * blockIdx.x) * 8;
    const int b = __ldg(m);
    if (b < 0)
        return;
    const int g = __ldg(m + 1), c_lo = __ldg(m + 2), c_hi = __ldg(m + 3), slot_lo = __ldg(m + 4);
    const int np = c_hi - c_lo + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = min(a.num_q_heads, NHG);
    const int jh = blockIdx.y * 8 + warp, h = g * NHG + jh;
    if (jh >= hs || h >= a.num_q_heads)
        return;
    float M = -INFINITY;
    for (int p = lane; p < np; p += 32)
        M = fmaxf(M, __ldg(a.lse + merge_row(c_lo, p, slot_lo, jh, hs)));
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
            const size_t row = merge_row(c_lo, p, slot_lo, jh, hs);
            const float ls = __ldg(a.lse + row);
            wgt[u] = (p0 + u >= np || ls == -INFINITY || M == -INFINITY) ? 0.f : __expf(ls - M);
            x[u] = 4 * lane < D ? __ldg(reinterpret_cast<const float4 *>(a.o_partial + row * D) + lane)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
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
    if (4 * lane >= D)
        return;
    uint2 o;
    o.x = pack_bf16x2(acc.x * f, acc.y * f);
    o.y = pack_bf16x2(acc.z * f, acc.w * f);
    *reinterpret_cast<uint2 *>(a.out + ((size_t)b * a.num_q_heads + h) * D + 4 * lane) = o;
}

namespace {

template <bool PAIR>
cudaError_t launch_decode_tc_t(const DecodeArgs &a, cudaStream_t s)
{
    static std::atomic<int> attr_set{0};
    if (!attr_set.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             TcCfg::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        // the kernel moves registers between its warpgroups (setmaxnreg): the split must fit
        // the registers it is launched with, or a group would wait for registers forever
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, decode_tc_kernel<PAIR>);
        if (e != cudaSuccess)
            return e;
        if (fa.numRegs != TcCfg::REG_LAUNCH)
            return cudaErrorInvalidConfiguration;
        attr_set.store(1, std::memory_order_release);
    }
    cudaError_t e =
        launch_pdl(decode_tc_kernel<PAIR>, dim3(a.persist_ctas), dim3(TcCfg::THREADS), TcCfg::SMEM_BYTES, s, a);
    if (e != cudaSuccess || !a.persistent)
        return e;
    const int hs = a.num_q_heads < TcMode<PAIR>::NHG ? a.num_q_heads : TcMode<PAIR>::NHG;
    return launch_pdl(decode_tc_merge_kernel<PAIR>, dim3(a.persist_ctas, (hs + 7) / 8), dim3(256), 0, s, a);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs &a, int head_dim, cudaStream_t s)
{
    return head_dim == 64 ? launch_decode_tc_t<true>(a, s) : launch_decode_tc_t<false>(a, s);
}

int decode_tc_ctas_per_sm()
{
    int n = 0;
    cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM_BYTES);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_tc_kernel<false>, TcCfg::THREADS,
                                                      TcCfg::SMEM_BYTES) != cudaSuccess)
        n = 1;
    return n < 1 ? 1 : n;
}

}  // namespace mqa
