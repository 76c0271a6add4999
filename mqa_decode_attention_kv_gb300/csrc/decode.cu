// Decode attention over the int8 paged cache (one query token per sequence,
// all query heads of the shared K/V head in one CTA), with optional split-KV.
//
// Design (sm_103a):
//  * Work unit: one CTA = (split, sequence, head group of up to 32 heads).  It
//    walks 64-token tiles of its key range through a STAGES-deep ring of shared
//    memory stages.  Thread 0 fills a stage with TMA: four 16-row boxes of K
//    codes and four of V codes (2-D tensor maps over [num_blocks*page, d] int8,
//    128-byte (d=128) or 64-byte (d=64) swizzle) plus linear bulk copies of the
//    fp32 scales; an mbarrier with transaction counts signals arrival.  Boxes
//    that fall outside [window start, L) are not fetched.
//  * MQA makes the query heads the M dimension of a dense contraction, so QK^T
//    and PV run on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate).
//    int8 codes become fp16 operands in registers with an exact exponent-bias
//    conversion; they never go back to shared memory.
//      QK^T: warp w owns the 16 tokens of box w of the tile, for all heads.
//      PV:   warp w owns a 32-wide slice of d (d=128) -- or a slice and half of
//            the tokens (d=64) -- for all heads; P is exchanged through shared
//            memory in mma A-fragment order.
//  * Scales: the K scale multiplies the fp32 score column; the V scale is folded
//    into the probability before it is rounded to fp16 (P' = p * s_v * 2^(14-E),
//    with 2^E a running power-of-two bound of the V scales, so P' stays inside
//    fp16's range whatever the data; O is rescaled when E grows, exactly like the
//    online-softmax rescale).  Q is pre-scaled per head by sm_scale*log2(e) and a
//    power of two so that it also uses fp16's full precision.
//  * Online softmax (running max m and sum l per head) as in FlashAttention:
//    tile row maxima are combined across warps in shared memory.
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

namespace mqa {
namespace {

template <int D, int HT>
struct DecodeCfg {
    static constexpr int MT = HT / 16;            // m16 tiles over heads
    static constexpr int KSTEPS = D / 16;         // k16 steps of QK^T
    static constexpr int SEG = D / 4;             // bytes of a K row owned by one lane (per quad position)
    static constexpr int NSLICE = D / 32;         // 32-wide d slices of PV
    static constexpr int GROUPS = 4 / NSLICE;     // token groups of PV
    static constexpr int PV_STEPS = 4 / GROUPS;   // PV k-steps per warp per tile
    static constexpr int STAGES = 4;
    static constexpr int CODE_BYTES = kTileTokens * D;              // K (or V) codes of a tile
    static constexpr int STAGE_CODES = 2 * CODE_BYTES;               // K then V
    // shared memory carve-up (offsets from a 1024-aligned base)
    static constexpr int OFF_CODES = 0;
    static constexpr int OFF_SCALES = STAGES * STAGE_CODES;              // [STAGES][2][64] fp32
    static constexpr int OFF_PBUF = OFF_SCALES + STAGES * 2 * kTileTokens * 4;  // [4][MT][32][4] u32
    static constexpr int OFF_REDMAX = OFF_PBUF + 4 * MT * 32 * 16;       // [4][HT] fp32
    static constexpr int OFF_REDL = OFF_REDMAX + 4 * HT * 4;             // [4][HT] fp32
    static constexpr int OFF_REDSV = OFF_REDL + 4 * HT * 4;              // [4] fp32
    static constexpr int OFF_MASK = OFF_REDSV + 16;                      // [STAGES] u32
    static constexpr int OFF_FLAG = OFF_MASK + 4 * STAGES;               // int
    static constexpr int OFF_MBAR = (OFF_FLAG + 4 + 7) / 8 * 8;          // [STAGES] u64
    static constexpr int SMEM_BYTES = OFF_MBAR + 8 * STAGES + 1024;      // + alignment slack
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(HT == 16 || HT == 32, "head tile");
    // the d=64 epilogue stages partial O of the second token group in the code ring
    static_assert(GROUPS == 1 || HT * D * 4 <= STAGES * STAGE_CODES, "epilogue buffer");
};

// Load this lane's query fragments (A operand of QK^T, k-index permuted so that
// lane quad position c owns d in [c*D/4, (c+1)*D/4)), scaled by
// sm_scale*log2(e)*2^e_h and rounded to fp16; gexp = 2^-e_h per row.
template <int D, int HT>
__device__ __forceinline__ void load_q(const DecodeArgs &a, int b, int h0, int lane,
                                       uint32_t (&qf)[HT / 16][D / 16][4], float (&gexp)[HT / 16][2])
{
    using C = DecodeCfg<D, HT>;
    const int g = lane >> 2, c = lane & 3;
    uint32_t w[C::MT][2][D / 8];
    float amax[C::MT][2];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int h = h0 + mt * 16 + g + 8 * hf;
            const bool ok = h < a.num_q_heads && (mt * 16 + g + 8 * hf) < HT;
            const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.num_q_heads + h) * D + c * C::SEG);
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const uint4 v = ok ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
                const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    w[mt][hf][4 * j + k] = vv[k];
                    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(vv[k] << 16)),
                                       fabsf(__uint_as_float(vv[k] & 0xffff0000u))));
                }
            }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            amax[mt][hf] = m;
        }
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            // e chosen so that max|q| * sm_scale*log2(e) * 2^e lies in (2^13, 2^14]
            const float sm = amax[mt][hf] * a.q_scale_log2;
            int e = 0;
            if (sm > 0.f && isfinite(sm)) {
                int x;
                frexpf(sm, &x);
                e = 14 - x;
                e = e < -120 ? -120 : (e > 120 ? 120 : e);
            }
            gexp[mt][hf] = exp2i(-e);
            const float f = a.q_scale_log2 * exp2i(e);
#pragma unroll
            for (int kt = 0; kt < C::KSTEPS; ++kt) {
                const uint32_t w01 = w[mt][hf][2 * kt], w23 = w[mt][hf][2 * kt + 1];
                const uint32_t lo = pack_half2(__uint_as_float(w01 << 16) * f, __uint_as_float(w01 & 0xffff0000u) * f);
                const uint32_t hi = pack_half2(__uint_as_float(w23 << 16) * f, __uint_as_float(w23 & 0xffff0000u) * f);
                qf[mt][kt][hf] = lo;       // a0a1 (row g) / a2a3 (row g+8): columns 2c, 2c+1
                qf[mt][kt][2 + hf] = hi;   // a4a5 (row g) / a6a7 (row g+8): columns 2c+8, 2c+9
            }
        }
}

template <int D, int HT>
__global__ void __launch_bounds__(128, 3) decode_kernel(const __grid_constant__ DecodeArgs a)
{
    using C = DecodeCfg<D, HT>;
    constexpr int MT = C::MT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t *pbuf = reinterpret_cast<uint32_t *>(base + C::OFF_PBUF);
    float *red_max = reinterpret_cast<float *>(base + C::OFF_REDMAX);
    float *red_l = reinterpret_cast<float *>(base + C::OFF_REDL);
    float *red_sv = reinterpret_cast<float *>(base + C::OFF_REDSV);
    uint32_t *stage_mask = reinterpret_cast<uint32_t *>(base + C::OFF_MASK);
    volatile int *flag = reinterpret_cast<int *>(base + C::OFF_FLAG);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(base + C::OFF_MBAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int split = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * HT;
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
        // empty split (or invalid sequence): lse = -inf, or zero output
        for (int r = threadIdx.x; r < HT; r += blockDim.x) {
            const int h = h0 + r;
            if (h >= a.num_q_heads)
                continue;
            if (split_mode) {
                a.lse[((size_t)b * a.num_splits + split) * a.num_q_heads + h] = -INFINITY;
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((size_t)b * a.num_q_heads + h) * D);
                for (int j = 0; j < D / 8; ++j)
                    dst[j] = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int n_tiles = te - tb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s)
            mbar_init(mbar + s, 1);
        *flag = 0;
        fence_mbar_init();
        const int npro = n_tiles < C::STAGES ? n_tiles : C::STAGES;
        for (int i = 0; i < npro; ++i)
            issue_kv_tile<D>(a.k_map, a.v_map, a.k_scale, a.v_scale, a.block_table + (size_t)b * a.max_blocks,
                              a.num_blocks, a.page_size, a.dev_status,
                              base + C::OFF_CODES + i * C::STAGE_CODES,
                              reinterpret_cast<float *>(base + C::OFF_SCALES) + i * 2 * kTileTokens, mbar + i,
                              stage_mask + i, tb + i, lo, L);
    }

    uint32_t qf[MT][C::KSTEPS][4];
    float gexp[MT][2];
    load_q<D, HT>(a, b, h0, lane, qf, gexp);

    float m_run[MT][2], l_run[MT][2];
    float o[MT][4][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            m_run[mt][hf] = -INFINITY;
            l_run[mt][hf] = 0.f;
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                o[mt][nt][k] = 0.f;
    }
    int E_run = -100;
    __syncthreads();  // barriers initialised, stage masks of the prologue written

    const int slice = warp % C::NSLICE, grp = warp / C::NSLICE;
    int i = 0;
    for (; i < n_tiles; ++i) {
        const int stage = i % C::STAGES;
        if (!mbar_wait_bounded(mbar + stage, (uint32_t)(i / C::STAGES) & 1u))
            *flag = 1;
        const uint8_t *kst = base + C::OFF_CODES + stage * C::STAGE_CODES;
        const uint8_t *vst = kst + C::CODE_BYTES;
        const float *ks = reinterpret_cast<const float *>(base + C::OFF_SCALES) + stage * 2 * kTileTokens;
        const float *vs = ks + kTileTokens;
        const uint32_t mask = stage_mask[stage];
        const int T = tb + i;

        // ---- S = Q K^T for the 16 tokens of box `warp`
        const int t = warp;
        const bool box_ok = (mask >> t) & 1u;
        float acc[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    acc[mt][s][k] = 0.f;
        if (box_ok) {
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int row = 16 * t + 8 * s + g;
                uint32_t kw[C::KSTEPS];
#pragma unroll
                for (int j = 0; j < C::SEG / 16; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(kst + swz<D>(row, c * C::SEG + 16 * j));
                    kw[4 * j] = v.x;
                    kw[4 * j + 1] = v.y;
                    kw[4 * j + 2] = v.z;
                    kw[4 * j + 3] = v.w;
                }
#pragma unroll
                for (int kt = 0; kt < C::KSTEPS; ++kt) {
                    uint32_t b0, b1;
                    i8x4_to_f16x2x2(kw[kt], b0, b1);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        mma_f16_16816(acc[mt][s], qf[mt][kt], b0, b1);
                }
            }
        }

        // ---- scale by s_k, mask, per-row tile maxima
        const int tok0 = T * kTileTokens + 16 * t + 2 * c;  // absolute position of (s=0, e=0)
        float ksv[2][2], vsv[2][2];
        bool valid[2][2];
        float svmax = 0.f;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const float2 kk = *reinterpret_cast<const float2 *>(ks + 16 * t + 8 * s + 2 * c);
            const float2 vv = *reinterpret_cast<const float2 *>(vs + 16 * t + 8 * s + 2 * c);
            ksv[s][0] = kk.x;
            ksv[s][1] = kk.y;
            vsv[s][0] = vv.x;
            vsv[s][1] = vv.y;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int pos = tok0 + 8 * s + e;
                valid[s][e] = box_ok && pos >= lo && pos < L;
                if (valid[s][e])
                    svmax = fmaxf(svmax, vsv[s][e]);
            }
        }
        float y[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float m = -INFINITY;
#pragma unroll
                for (int s = 0; s < 2; ++s)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float v = valid[s][e] ? acc[mt][s][2 * hf + e] * ksv[s][e] : -INFINITY;
                        y[mt][s][2 * hf + e] = v;
                        m = fmaxf(m, v);
                    }
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                if (c == 0)
                    red_max[t * HT + mt * 16 + g + 8 * hf] = m;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            svmax = fmaxf(svmax, __shfl_xor_sync(0xffffffffu, svmax, off));
        if (lane == 0)
            red_sv[t] = svmax;
        __syncthreads();  // ---- A: tile maxima visible; stage (i-1) free
        if (*flag)
            break;
        if (threadIdx.x == 0 && i >= 1 && i - 1 + C::STAGES < n_tiles)
        {
            const int st = (i - 1) % C::STAGES;
            issue_kv_tile<D>(a.k_map, a.v_map, a.k_scale, a.v_scale, a.block_table + (size_t)b * a.max_blocks,
                             a.num_blocks, a.page_size, a.dev_status, base + C::OFF_CODES + st * C::STAGE_CODES,
                             reinterpret_cast<float *>(base + C::OFF_SCALES) + st * 2 * kTileTokens, mbar + st,
                             stage_mask + st, tb + i - 1 + C::STAGES, lo, L);
        }

        // ---- online softmax update (each thread for its rows)
        const float sv_tile = fmaxf(fmaxf(red_sv[0], red_sv[1]), fmaxf(red_sv[2], red_sv[3]));
        const int E_new = max(E_run, ceil_log2_pow(sv_tile));
        const float vfac = exp2i(14 - E_new);
        const int dE = E_run - E_new;
        const float escale = dE < -126 ? 0.f : exp2i(dE);
        E_run = E_new;
        float oscale[MT][2];
        uint32_t pf[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int row = mt * 16 + g + 8 * hf;
                const float mt_ = fmaxf(fmaxf(red_max[row], red_max[HT + row]),
                                        fmaxf(red_max[2 * HT + row], red_max[3 * HT + row]));
                const float m_new = fmaxf(m_run[mt][hf], mt_);
                const float gh = gexp[mt][hf];
                const bool none = m_new == -INFINITY;
                const float alpha = none ? 1.f : fast_exp2((m_run[mt][hf] - m_new) * gh);
                const float negmg = none ? 0.f : -m_new * gh;
                m_run[mt][hf] = m_new;
                float lsum = l_run[mt][hf] * alpha;
                oscale[mt][hf] = alpha * escale;
                float pp[2][2];
#pragma unroll
                for (int s = 0; s < 2; ++s)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float p = fast_exp2(fmaf(y[mt][s][2 * hf + e], gh, negmg));
                        lsum += p;
                        pp[s][e] = valid[s][e] ? p * (vsv[s][e] * vfac) : 0.f;
                    }
                l_run[mt][hf] = lsum;
                pf[mt][hf] = pack_half2(pp[0][0], pp[0][1]);      // a0a1 / a2a3: tokens 2c, 2c+1
                pf[mt][2 + hf] = pack_half2(pp[1][0], pp[1][1]);  // a4a5 / a6a7: tokens 2c+8, 2c+9
            }
            *reinterpret_cast<uint4 *>(pbuf + ((t * MT + mt) * 32 + lane) * 4) =
                make_uint4(pf[mt][0], pf[mt][1], pf[mt][2], pf[mt][3]);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                o[mt][nt][0] *= oscale[mt][0];
                o[mt][nt][1] *= oscale[mt][0];
                o[mt][nt][2] *= oscale[mt][1];
                o[mt][nt][3] *= oscale[mt][1];
            }
        __syncthreads();  // ---- B: P' fragments visible

        // ---- O += P' V for this warp's d slice (and token group)
#pragma unroll
        for (int tt = 0; tt < C::PV_STEPS; ++tt) {
            const int t2 = grp * C::PV_STEPS + tt;
            if (!((mask >> t2) & 1u))
                continue;
            uint32_t af[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const uint4 v = *reinterpret_cast<const uint4 *>(pbuf + ((t2 * MT + mt) * 32 + lane) * 4);
                af[mt][0] = v.x;
                af[mt][1] = v.y;
                af[mt][2] = v.z;
                af[mt][3] = v.w;
            }
            const uint32_t col = 32 * slice + 4 * g;
            const uint32_t r0 = 16 * t2 + 2 * c;
            const uint32_t w0 = *reinterpret_cast<const uint32_t *>(vst + swz<D>(r0, col));
            const uint32_t w1 = *reinterpret_cast<const uint32_t *>(vst + swz<D>(r0 + 1, col));
            const uint32_t w2 = *reinterpret_cast<const uint32_t *>(vst + swz<D>(r0 + 8, col));
            const uint32_t w3 = *reinterpret_cast<const uint32_t *>(vst + swz<D>(r0 + 9, col));
            uint32_t bl[4], bh[4];
            i8x4x2_interleave_to_f16x2(w0, w1, bl);
            i8x4x2_interleave_to_f16x2(w2, w3, bh);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    mma_f16_16816(o[mt][nt], af[mt], bl[nt], bh[nt]);
        }
    }

    if (*flag) {
        // a TMA wait ran out: report, let our own copies in flight land (bounded), leave
        if (threadIdx.x == 0) {
            set_status(a.dev_status, MQA_DEV_TIMEOUT);
            // tiles issued so far: 0..STAGES-1 by the prologue, then tile i-1+STAGES at iteration i >= 1
            const int issued_end = min(n_tiles, i >= 1 ? i + C::STAGES - 1 : C::STAGES);
            for (int j = i; j < issued_end; ++j)
                mbar_wait_bounded(mbar + (j % C::STAGES), (uint32_t)(j / C::STAGES) & 1u);
        }
        return;
    }

    // ---- epilogue: total l per row, merge token groups (d=64), normalise, store
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float l = l_run[mt][hf];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (c == 0)
                red_l[warp * HT + mt * 16 + g + 8 * hf] = l;
        }
    float *obuf = reinterpret_cast<float *>(base + C::OFF_CODES);  // the code ring is idle now
    if constexpr (C::GROUPS == 2) {
        if (grp == 1) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        obuf[((mt * 4 + nt) * 4 + k) * 64 + slice * 32 + lane] = o[mt][nt][k];
        }
    }
    __syncthreads();
    if (grp != 0)
        return;
    if constexpr (C::GROUPS == 2) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o[mt][nt][k] += obuf[((mt * 4 + nt) * 4 + k) * 64 + slice * 32 + lane];
    }
    const float ofac = exp2i(E_run - 14);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int row = mt * 16 + g + 8 * hf;
            const int h = h0 + row;
            if (row >= HT || h >= a.num_q_heads)
                continue;
            const float l = red_l[row] + red_l[HT + row] + red_l[2 * HT + row] + red_l[3 * HT + row];
            const float f = l > 0.f ? ofac / l : 0.f;
            float v[8];  // d = 32*slice + 8c + (4e + nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
                    v[4 * e + nt] = o[mt][nt][2 * hf + e] * f;
            const int d0 = 32 * slice + 8 * c;
            if (split_mode) {
                const size_t rowoff = ((size_t)b * a.num_splits + split) * a.num_q_heads + h;
                float4 *dst = reinterpret_cast<float4 *>(a.o_partial + rowoff * D + d0);
                dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                dst[1] = make_float4(v[4], v[5], v[6], v[7]);
                if (slice == 0 && c == 0)
                    a.lse[rowoff] = l > 0.f ? (m_run[mt][hf] * gexp[mt][hf] + __log2f(l)) * 0.69314718055994531f
                                            : -INFINITY;
            } else {
                __nv_bfloat162 p[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    p[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
                *reinterpret_cast<uint4 *>(a.out + ((size_t)b * a.num_q_heads + h) * D + d0) =
                    *reinterpret_cast<uint4 *>(p);
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
        attr_set.store(1, std::memory_order_release);
    }
    dim3 grid(a.num_splits, a.batch, (a.num_q_heads + HT - 1) / HT);
    decode_kernel<D, HT><<<grid, 128, C::SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

template <int D, int HT>
int ctas_per_sm_t()
{
    using C = DecodeCfg<D, HT>;
    int n = 0;
    cudaFuncSetAttribute(decode_kernel<D, HT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, HT>, 128, C::SMEM_BYTES) != cudaSuccess)
        n = 1;
    return n < 1 ? 1 : n;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, int head_dim, cudaStream_t s)
{
    const bool small = a.num_q_heads <= 16;
    if (head_dim == 128)
        return small ? launch_decode_t<128, 16>(a, s) : launch_decode_t<128, 32>(a, s);
    return small ? launch_decode_t<64, 16>(a, s) : launch_decode_t<64, 32>(a, s);
}

int decode_ctas_per_sm(int head_dim, int num_q_heads)
{
    const bool small = num_q_heads <= 16;
    if (head_dim == 128)
        return small ? ctas_per_sm_t<128, 16>() : ctas_per_sm_t<128, 32>();
    return small ? ctas_per_sm_t<64, 16>() : ctas_per_sm_t<64, 32>();
}

}  // namespace mqa
