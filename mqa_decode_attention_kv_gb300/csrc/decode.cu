// Decode attention over the int8 paged cache (one query token per sequence,
// all query heads of the shared K/V head in one CTA), with optional split-KV.
//
// Design (sm_103a):
//  * Work unit: one CTA = (split, sequence, group of up to 32 query heads).  It
//    walks the 64-token tiles of its key range through a STAGES-deep ring of
//    shared-memory stages.  A tile is four 16-token boxes; each box (K codes,
//    V codes: one 16-row TMA box each from 2-D tensor maps over
//    [num_blocks*page, d] int8 with the 128-byte (d=128) or 64-byte (d=64)
//    swizzle; K and V scales: two linear bulk copies) has its own mbarrier.
//  * Warps are independent: warp w owns 16 query heads (one m16 tile) and a
//    token group (two boxes of every tile for 32 heads, one box for <= 16
//    heads).  It computes S = Q K^T, the online softmax and O += P V for its
//    heads over its tokens entirely in registers: the QK^T accumulator fragment
//    is reused as the A operand of PV, so nothing goes through shared memory
//    and there is no CTA-wide barrier in the main loop.  The last warp to finish
//    with a box refills it (shared-memory counter), so no warp waits on a
//    producer.  The token groups' partial results are merged once at the end.
//  * MQA makes the query heads the M dimension of a dense contraction: QK^T and
//    PV run on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate).
//    int8 codes become fp16 operands in registers with an exact exponent-bias
//    conversion.  The K scale multiplies the fp32 score column; the V scale is
//    folded into the probability before it is rounded to fp16
//    (P' = p * s_v * 2^(14-E), 2^E a running power-of-two bound of the V scales,
//    so P' stays inside fp16's range whatever the data; O is rescaled when E
//    grows, like the online-softmax rescale).  Q is scaled per head by a power
//    of two only, which is exact in fp16; sm_scale*log2(e) multiplies the fp32
//    scores.
//  * Output: bf16 directly (one split) or fp32 partial O and natural-log lse per
//    split, merged by the combine kernel.
//  * Every wait is bounded; bad block ids / sequence lengths are reported in
//    dev_status and the affected tokens are skipped.
#include <atomic>
#include <cfloat>
#include <math.h>

#include "common.cuh"
#include "kv_stage.cuh"
#include "launch.h"
#include "split_merge.cuh"

namespace mqa {
namespace {

template <int D, int HT>
struct DecodeCfg {
    static constexpr int HG = HT / 16;            // head groups (warps sharing a token group)
    static constexpr int TG = 4 / HG;             // token groups
    static constexpr int BPW = kChunksPerTile / TG;  // boxes per warp per tile
    static constexpr int KSTEPS = D / 16;         // k16 steps of QK^T
    static constexpr int SEG = D / 4;             // bytes of a K row owned by one lane (per quad position)
    static constexpr int NT = D / 8;              // n8 tiles of PV (d)
    static constexpr int VB = D / 8;              // bytes of a V row owned by one lane
    static constexpr int STAGES = 4;
    static constexpr int CODE_BYTES = kTileTokens * D;               // K (or V) codes of a tile
    static constexpr int STAGE_CODES = 2 * CODE_BYTES;                // K then V
    // shared memory carve-up (offsets from a 1024-aligned base)
    static constexpr int OFF_CODES = 0;
    static constexpr int OFF_SCALES = STAGES * STAGE_CODES;                     // [STAGES][2][64] fp32
    static constexpr int OFF_OK = OFF_SCALES + STAGES * 2 * kTileTokens * 4;     // [STAGES][4] u32 box arrived
    static constexpr int OFF_CNT = OFF_OK + STAGES * 4 * 4;                      // [STAGES][4] consumers done
    static constexpr int OFF_ISS = OFF_CNT + STAGES * 4 * 4;                     // [STAGES][4] last tile issued
    static constexpr int OFF_STAT = OFF_ISS + STAGES * 4 * 4;                    // [4 warps][16 rows] (m, l)
    static constexpr int OFF_E = OFF_STAT + 4 * 16 * 8;                          // [4 warps] int
    static constexpr int OFF_FLAG = OFF_E + 16;                                  // int
    static constexpr int OFF_MBAR = (OFF_FLAG + 4 + 7) / 8 * 8;                  // [STAGES][4] u64
    static constexpr int SMEM_BYTES = OFF_MBAR + 8 * 4 * STAGES + 1024;          // + alignment slack
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(HT == 16 || HT == 32, "head tile");
    // the epilogue stages the O partials of token groups 1.. in the code ring
    static_assert((TG - 1) * HG * 16 * D * 4 <= STAGES * STAGE_CODES, "epilogue buffer");
};

// This lane's query fragments for the 16 heads h16..h16+15 (A operand of
// QK^T, k-index permuted so that quad position c owns d in
// [c*D/4, (c+1)*D/4)), scaled by 2^e_h (exact in fp16);
// gexp = sm_scale*log2(e)*2^-e_h for rows g and g+8.
template <int D>
__device__ __forceinline__ void load_q16(const DecodeArgs &a, int b, int h16, int lane, uint32_t (&qf)[D / 16][4],
                                         float (&gexp)[2])
{
    constexpr int SEG = D / 4;
    const int g = lane >> 2, c = lane & 3;
    uint32_t w[2][D / 8];
    float amax[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int h = h16 + g + 8 * hf;
        const bool ok = h < a.num_q_heads;
        const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.num_q_heads + h) * D + c * SEG);
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
            const uint4 v = ok ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
            const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                w[hf][4 * j + k] = vv[k];
                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(vv[k] << 16)), fabsf(__uint_as_float(vv[k] & 0xffff0000u))));
            }
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        amax[hf] = m;
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        // e chosen so that max|q| * 2^e lies in [2^13, 2^14)
        int e = 0;
        if (amax[hf] > 0.f && isfinite(amax[hf])) {
            int x;
            frexpf(amax[hf], &x);
            e = 14 - x;
            e = e < -120 ? -120 : (e > 120 ? 120 : e);
        }
        // q * 2^e is exact in fp16 (bf16 carries 8 significant bits); the softmax
        // scale is applied in fp32 to the scores instead
        gexp[hf] = a.q_scale_log2 * exp2i(-e);
        const float f = exp2i(e);
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt) {
            const uint32_t w01 = w[hf][2 * kt], w23 = w[hf][2 * kt + 1];
            qf[kt][hf] = pack_half2(__uint_as_float(w01 << 16) * f, __uint_as_float(w01 & 0xffff0000u) * f);
            qf[kt][2 + hf] = pack_half2(__uint_as_float(w23 << 16) * f, __uint_as_float(w23 & 0xffff0000u) * f);
        }
    }
}

template <int D, int HT>
__global__ void __launch_bounds__(128, 3) decode_kernel(const __grid_constant__ DecodeArgs a)
{
    using C = DecodeCfg<D, HT>;
    constexpr int S = C::STAGES, BPW = C::BPW, HG = C::HG, NT = C::NT;
    griddep_wait();  // the previous kernel's writes (cache slots, q, tickets) are visible from here
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t *box_ok = reinterpret_cast<uint32_t *>(base + C::OFF_OK);
    int *cnt = reinterpret_cast<int *>(base + C::OFF_CNT);
    int *issued = reinterpret_cast<int *>(base + C::OFF_ISS);
    float2 *stat = reinterpret_cast<float2 *>(base + C::OFF_STAT);
    int *ebuf = reinterpret_cast<int *>(base + C::OFF_E);
    volatile int *flag = reinterpret_cast<int *>(base + C::OFF_FLAG);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(base + C::OFF_MBAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int hg = warp % HG, tg = warp / HG;
    const int split = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * HT;
    const int h16 = h0 + hg * 16;
    const bool split_mode = a.num_splits > 1;

    // ---- key range of this CTA (in 64-token tiles)
    const int L = __ldg(a.seq_lens + b);
    const int lo = (L >= 1 && a.window > 0 && L > a.window) ? L - a.window : 0;
    const int t_first = lo / kTileTokens;
    const int t_last = (L - 1) / kTileTokens;
    const bool bad = L < 1 || L > a.max_seq_len ||
                     (t_last - t_first + 1) > a.tiles_per_split * a.num_splits;
    const int tb = t_first + split * a.tiles_per_split;
    const int te = min(tb + a.tiles_per_split, t_last + 1);
    if (bad || tb >= te) {
        if (bad && threadIdx.x == 0 && split == 0)
            set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
        // empty split: lse = -inf; invalid sequence: also a zero output (nobody merges it)
        for (int r = threadIdx.x; r < HT; r += blockDim.x) {
            const int h = h0 + r;
            if (h >= a.num_q_heads)
                continue;
            if (split_mode)
                a.lse[((size_t)b * a.num_splits + split) * a.num_q_heads + h] = -INFINITY;
            if (!split_mode || (bad && split == 0)) {
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)b * a.num_q_heads + h) * D);
                for (int j = 0; j < D / 8; ++j)
                    dst[j] = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int n_tiles = te - tb;
    const int32_t *table = a.block_table + (size_t)b * a.max_blocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S * kChunksPerTile; ++s) {
            mbar_init(mbar + s, 1);
            cnt[s] = 0;
            issued[s] = -1;
        }
        *flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // prologue: warp w issues box w of the first STAGES tiles
    if (lane == 0)
        for (int i = 0; i < n_tiles && i < S; ++i) {
            issued[i * kChunksPerTile + warp] = i;
            issue_kv_box<D>(a.k_map, a.v_map, a.k_scale, a.v_scale,
                            fetch_box_block(table, a.page_size, tb + i, warp, lo, L, a.ring), a.num_blocks, a.page_size,
                            a.dev_status, base + C::OFF_CODES + i * C::STAGE_CODES,
                            reinterpret_cast<float *>(base + C::OFF_SCALES) + i * 2 * kTileTokens,
                            mbar + i * kChunksPerTile + warp, box_ok + i * kChunksPerTile + warp, tb + i, warp);
        }

    uint32_t qf[C::KSTEPS][4];
    float gexp[2];
    load_q16<D>(a, b, h16, lane, qf, gexp);

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // l_run: this lane's share
    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[nt][k] = 0.f;
    int E_run = -100;
    // lane-constant swizzled offsets: row g of a box (K) and rows 2c, 2c+1 (V);
    // adding multiples of 8 rows leaves the swizzle phase unchanged
    uint32_t koff[C::SEG / 16];
#pragma unroll
    for (int j = 0; j < C::SEG / 16; ++j)
        koff[j] = swz<D>(g, c * C::SEG + 16 * j);
    const uint32_t voff0 = swz<D>(2 * c, C::VB * g);
    const uint32_t voff1 = swz<D>(2 * c + 1, C::VB * g);
    bool timed_out = false;

    for (int i = 0; i < n_tiles; ++i) {
        const int stage = i % S;
        const int T = tb + i;
        const uint8_t *kst = base + C::OFF_CODES + stage * C::STAGE_CODES;
        const uint8_t *vst = kst + C::CODE_BYTES;
        const float *ks = reinterpret_cast<const float *>(base + C::OFF_SCALES) + stage * 2 * kTileTokens;
        const float *vs = ks + kTileTokens;
        // block ids of my boxes of tile i+S, for the refill if this warp finishes a box last
        int32_t id_pf[BPW];
#pragma unroll
        for (int j = 0; j < BPW; ++j)
            id_pf[j] = (lane == 0 && i + S < n_tiles)
                           ? fetch_box_block(table, a.page_size, T + S, tg * BPW + j, lo, L, a.ring) : kNoBlock;
        bool okj[BPW];
#pragma unroll
        for (int j = 0; j < BPW; ++j) {
            const int bx = tg * BPW + j;
            if (!mbar_wait_bounded(mbar + stage * kChunksPerTile + bx, (uint32_t)(i / S) & 1u))
                timed_out = true;
            okj[j] = box_ok[stage * kChunksPerTile + bx] != 0;
        }
        if (__any_sync(0xffffffffu, timed_out)) {
            *flag = 1;
            break;
        }

        // ---- S = Q K^T for my boxes (tokens 16 bx + 8 s + g of the tile)
        float acc[BPW][2][4];
#pragma unroll
        for (int j = 0; j < BPW; ++j)
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    acc[j][s][k] = 0.f;
#pragma unroll
        for (int j = 0; j < BPW; ++j) {
            if (!okj[j])
                continue;
            const int bx = tg * BPW + j;
            uint32_t kw[2][C::KSTEPS];
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int q = 0; q < C::SEG / 16; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(kst + (16 * bx + 8 * s) * D + koff[q]);
                    kw[s][4 * q] = v.x;
                    kw[s][4 * q + 1] = v.y;
                    kw[s][4 * q + 2] = v.z;
                    kw[s][4 * q + 3] = v.w;
                }
#pragma unroll
            for (int kt = 0; kt < C::KSTEPS; ++kt)
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    uint32_t b0, b1;
                    i8x4_to_f16x2x2(kw[s][kt], b0, b1);
                    mma_f16_16816(acc[j][s], qf[kt], b0, b1);
                }
        }

        // ---- scores y = S' * s_k (C fragment: tokens 16 bx + 8 s + 2c + e), masks
        float ksv[BPW][2][2], vsv[BPW][2][2];
        bool valid[BPW][2][2];
        float svm = 0.f;
#pragma unroll
        for (int j = 0; j < BPW; ++j) {
            const int bx = tg * BPW + j;
            const int tok0 = T * kTileTokens + 16 * bx;
            const bool full = okj[j] && tok0 >= lo && tok0 + 16 <= L;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const float2 kk = *reinterpret_cast<const float2 *>(ks + 16 * bx + 8 * s + 2 * c);
                const float2 vv = *reinterpret_cast<const float2 *>(vs + 16 * bx + 8 * s + 2 * c);
                ksv[j][s][0] = kk.x;
                ksv[j][s][1] = kk.y;
                vsv[j][s][0] = vv.x;
                vsv[j][s][1] = vv.y;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int pos = tok0 + 8 * s + 2 * c + e;
                    valid[j][s][e] = full || (okj[j] && pos >= lo && pos < L);
                    if (valid[j][s][e])
                        svm = fmaxf(svm, vsv[j][s][e]);
                }
            }
        }
        svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 1));
        svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 2));
        const int E_new = max(E_run, ceil_log2_pow(svm));
        float y[BPW][2][4];
        float m_new[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < BPW; ++j)
#pragma unroll
                for (int s = 0; s < 2; ++s)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float v = valid[j][s][e] ? acc[j][s][2 * hf + e] * ksv[j][s][e] : -INFINITY;
                        y[j][s][2 * hf + e] = v;
                        m = fmaxf(m, v);
                    }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m_new[hf] = fmaxf(m_run[hf], m);
        }
        // online-softmax rescale, only when the running max or the V-scale bound moved
        const bool changed = __any_sync(0xffffffffu, (m_new[0] != m_run[0]) | (m_new[1] != m_run[1]) | (E_new != E_run));
        if (changed) {
            const int dE = E_run - E_new;
            const float escale = dE < -126 ? 0.f : exp2i(dE);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const bool none = m_new[hf] == -INFINITY;
                const float al = none ? 1.f : fast_exp2((m_run[hf] - m_new[hf]) * gexp[hf]);
                l_run[hf] *= al;
                const float osc = al * escale;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    o[nt][2 * hf] *= osc;
                    o[nt][2 * hf + 1] *= osc;
                }
                m_run[hf] = m_new[hf];
            }
            E_run = E_new;
        }
        const float vfac = exp2i(14 - E_run);

        // ---- P' = p * s_v * 2^(14-E) as the A fragments of PV (one k16 step per box)
        uint32_t pa[BPW][4];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const float gh = gexp[hf];
            const float negm = m_run[hf] == -INFINITY ? 0.f : -m_run[hf] * gh;
            float lsum = 0.f;
#pragma unroll
            for (int j = 0; j < BPW; ++j) {
                float pp[2][2];
#pragma unroll
                for (int s = 0; s < 2; ++s)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float p = fast_exp2(fmaf(y[j][s][2 * hf + e], gh, negm));
                        lsum += p;
                        pp[s][e] = valid[j][s][e] ? p * (vsv[j][s][e] * vfac) : 0.f;
                    }
                pa[j][hf] = pack_half2(pp[0][0], pp[0][1]);      // a0a1 / a2a3: tokens 2c, 2c+1
                pa[j][2 + hf] = pack_half2(pp[1][0], pp[1][1]);  // a4a5 / a6a7: tokens 2c+8, 2c+9
            }
            l_run[hf] += lsum;
        }

        // ---- O += P' V (B fragment: V rows 16 bx + 2c + {0,1,8,9}, d = (D/8) g + nt)
#pragma unroll
        for (int j = 0; j < BPW; ++j) {
            if (!okj[j])
                continue;
            const int bx = tg * BPW + j;
            const uint8_t *vrow = vst + (16 * bx) * D;
            uint32_t vw[4][C::VB / 4];
            if constexpr (C::VB == 16) {
                const uint4 r0 = *reinterpret_cast<const uint4 *>(vrow + voff0);
                const uint4 r1 = *reinterpret_cast<const uint4 *>(vrow + voff1);
                const uint4 r2 = *reinterpret_cast<const uint4 *>(vrow + 8 * D + voff0);
                const uint4 r3 = *reinterpret_cast<const uint4 *>(vrow + 8 * D + voff1);
                const uint4 rr[4] = {r0, r1, r2, r3};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    vw[r][0] = rr[r].x;
                    vw[r][1] = rr[r].y;
                    vw[r][2] = rr[r].z;
                    vw[r][3] = rr[r].w;
                }
            } else {
                const uint2 r0 = *reinterpret_cast<const uint2 *>(vrow + voff0);
                const uint2 r1 = *reinterpret_cast<const uint2 *>(vrow + voff1);
                const uint2 r2 = *reinterpret_cast<const uint2 *>(vrow + 8 * D + voff0);
                const uint2 r3 = *reinterpret_cast<const uint2 *>(vrow + 8 * D + voff1);
                const uint2 rr[4] = {r0, r1, r2, r3};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    vw[r][0] = rr[r].x;
                    vw[r][1] = rr[r].y;
                }
            }
#pragma unroll
            for (int q = 0; q < C::VB / 4; ++q) {
                uint32_t bl[4], bh[4];
                i8x4x2_interleave_to_f16x2(vw[0][q], vw[1][q], bl);
                i8x4x2_interleave_to_f16x2(vw[2][q], vw[3][q], bh);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16_16816(o[4 * q + k], pa[j], bl[k], bh[k]);
            }
        }

        // ---- release my boxes; the last of the HG consumers refills with tile i+S
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < BPW; ++j) {
                const int bx = tg * BPW + j;
                const int slot = stage * kChunksPerTile + bx;
                const int done = (HG == 1) ? 0 : atomicAdd(cnt + slot, 1);
                if (done == HG - 1) {
                    if (HG > 1)
                        atomicExch(cnt + slot, 0);
                    if (i + S < n_tiles) {
                        issued[slot] = i + S;
                        fence_proxy_async();
                        issue_kv_box<D>(a.k_map, a.v_map, a.k_scale, a.v_scale, id_pf[j], a.num_blocks,
                                        a.page_size, a.dev_status, base + C::OFF_CODES + stage * C::STAGE_CODES,
                                        reinterpret_cast<float *>(base + C::OFF_SCALES) + stage * 2 * kTileTokens,
                                        mbar + slot, box_ok + slot, T + S, bx);
                    }
                }
            }
        }
    }

    // ---- epilogue: total l per row, merge the token groups, normalise, store
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 1);
        l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 2);
    }
    __syncthreads();  // every warp is done with the stage ring
    if (*flag) {
        // a TMA wait ran out: report and let copies still in flight land (bounded)
        if (threadIdx.x == 0) {
            set_status(a.dev_status, MQA_DEV_TIMEOUT);
            for (int s = 0; s < S * kChunksPerTile; ++s)
                if (issued[s] >= 0)
                    mbar_wait_drain(mbar + s, (uint32_t)(issued[s] / S) & 1u);
        }
        return;
    }
    float4 *obuf = reinterpret_cast<float4 *>(base + C::OFF_CODES);  // the code ring is idle now
    if constexpr (C::TG > 1) {
        if (tg > 0) {
            float4 *dst = obuf + ((tg - 1) * HG + hg) * NT * 32;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                dst[nt * 32 + lane] = make_float4(o[nt][0], o[nt][1], o[nt][2], o[nt][3]);
            if (c == 0) {
                stat[warp * 16 + g] = make_float2(m_run[0], l_run[0]);
                stat[warp * 16 + g + 8] = make_float2(m_run[1], l_run[1]);
            }
            if (lane == 0)
                ebuf[warp] = E_run;
        }
        __syncthreads();
    }
    if (tg == 0) {
        if constexpr (C::TG > 1) {
        // merge: num = sum_t O_t 2^(E_t-14) 2^((m_t-M) gh), den = sum_t l_t 2^((m_t-M) gh)
        float M[2] = {m_run[0], m_run[1]};
#pragma unroll
        for (int t = 1; t < C::TG; ++t)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
                M[hf] = fmaxf(M[hf], stat[(t * HG + hg) * 16 + g + 8 * hf].x);
        float wself[2], den[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const float ws = M[hf] == -INFINITY ? 0.f : fast_exp2((m_run[hf] - M[hf]) * gexp[hf]);
            den[hf] = l_run[hf] * ws;
            wself[hf] = ws * exp2i(E_run - 14);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            o[nt][0] *= wself[0];
            o[nt][1] *= wself[0];
            o[nt][2] *= wself[1];
            o[nt][3] *= wself[1];
        }
#pragma unroll
        for (int t = 1; t < C::TG; ++t) {
            const int wt = t * HG + hg;
            const float2 s0 = stat[wt * 16 + g], s1 = stat[wt * 16 + g + 8];
            const int Et = ebuf[wt];
            float wt_[2];
            const float2 ss[2] = {s0, s1};
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float w = (M[hf] == -INFINITY || ss[hf].x == -INFINITY)
                                    ? 0.f : fast_exp2((ss[hf].x - M[hf]) * gexp[hf]);
                den[hf] += ss[hf].y * w;
                wt_[hf] = w * exp2i(Et - 14);
            }
            const float4 *src = obuf + ((t - 1) * HG + hg) * NT * 32;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float4 v = src[nt * 32 + lane];
                o[nt][0] += v.x * wt_[0];
                o[nt][1] += v.y * wt_[0];
                o[nt][2] += v.z * wt_[1];
                o[nt][3] += v.w * wt_[1];
            }
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            m_run[hf] = M[hf];
            l_run[hf] = den[hf];
        }
        } else {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const float s = exp2i(E_run - 14);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                o[nt][2 * hf] *= s;
                o[nt][2 * hf + 1] *= s;
            }
        }
    }
    // store: this lane holds d in [(D/4) c, (D/4) (c+1)) of rows g and g+8, ordered (e, nt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int h = h16 + g + 8 * hf;
        if (h >= a.num_q_heads || h >= h0 + HT)
            continue;
        const float l = l_run[hf];
        const float f = l > 0.f ? 1.f / l : 0.f;
        const int d0 = (D / 4) * c;
        if (split_mode) {
            const size_t rowoff = ((size_t)b * a.num_splits + split) * a.num_q_heads + h;
            float4 *dst = reinterpret_cast<float4 *>(a.o_partial + rowoff * D + d0);
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int q = 0; q < NT / 4; ++q)
                    dst[e * (NT / 4) + q] = make_float4(o[4 * q][2 * hf + e] * f, o[4 * q + 1][2 * hf + e] * f,
                                                        o[4 * q + 2][2 * hf + e] * f, o[4 * q + 3][2 * hf + e] * f);
            if (c == 0)
                a.lse[rowoff] = l > 0.f ? (m_run[hf] * gexp[hf] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)b * a.num_q_heads + h) * D + d0);
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int q = 0; q < NT / 8; ++q) {
                    __nv_bfloat162 p[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        p[k] = __floats2bfloat162_rn(o[8 * q + 2 * k][2 * hf + e] * f,
                                                     o[8 * q + 2 * k + 1][2 * hf + e] * f);
                    dst[e * (NT / 8) + q] = *reinterpret_cast<uint4 *>(p);
                }
        }
    }
    }  // tg == 0

    // ---- fused split-KV merge: the last of this sequence's split CTAs to finish
    // (atomic ticket) merges every split's partial result from L2
    if (split_mode && a.counters != nullptr) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int n_active = (t_last - t_first + 1 + a.tiles_per_split - 1) / a.tiles_per_split;
            const int ticket = atomicAdd(a.counters + (size_t)b * gridDim.z + blockIdx.z, 1);
            *flag = (ticket == n_active - 1) ? 2 : 0;
        }
        __syncthreads();
        if (*flag == 2) {
            __threadfence();
            const int n_active = (t_last - t_first + 1 + a.tiles_per_split - 1) / a.tiles_per_split;
            merge_splits<D, HT>(a, b, h0, n_active);
        }
    }
}

template <int D, int HT>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t s)
{
    using C = DecodeCfg<D, HT>;
    static std::atomic<int> attr_set{0};  // idempotent; racing first calls set the same value
    if (!attr_set.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, HT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(decode_kernel<D, HT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        attr_set.store(1, std::memory_order_release);
    }
    dim3 grid(a.num_splits, a.batch, (a.num_q_heads + HT - 1) / HT);
    return launch_pdl(decode_kernel<D, HT>, grid, dim3(128), C::SMEM_BYTES, s, a);
}

template <int D, int HT>
int ctas_per_sm_t()
{
    using C = DecodeCfg<D, HT>;
    int n = 0;
    cudaFuncSetAttribute(decode_kernel<D, HT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    cudaFuncSetAttribute(decode_kernel<D, HT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, HT>, 128, C::SMEM_BYTES) != cudaSuccess)
        n = 1;
    return n < 1 ? 1 : n;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, int head_dim, cudaStream_t s)
{
    if (decode_uses_tc(head_dim, a.num_q_heads))
        return launch_decode_tc(a, s);
    const bool small = a.num_q_heads <= 16;
    if (head_dim == 128)
        return small ? launch_decode_t<128, 16>(a, s) : launch_decode_t<128, 32>(a, s);
    return small ? launch_decode_t<64, 16>(a, s) : launch_decode_t<64, 32>(a, s);
}

int decode_ctas_per_sm(int head_dim, int num_q_heads)
{
    if (decode_uses_tc(head_dim, num_q_heads))
        return decode_tc_ctas_per_sm();
    const bool small = num_q_heads <= 16;
    if (head_dim == 128)
        return small ? ctas_per_sm_t<128, 16>() : ctas_per_sm_t<128, 32>();
    return small ? ctas_per_sm_t<64, 16>() : ctas_per_sm_t<64, 32>();
}

}  // namespace mqa
