// Chunked causal prefill attention on the 5th-generation tensor cores
// (tcgen05), head_dim 64 or 128, over the int8 paged cache (prefix-shared
// blocks allowed).
//
// Two kernels.  kv_tile_images_kernel converts, once per sequence, every
// 64-key tile its queries can see into an fp16 image laid out exactly as the
// tensor core reads it (K with its codes' exponent bias, V exact), plus a
// record of the tile's K and V scales (a negative K scale marks a key that no
// query of the sequence sees or whose block id is bad), its largest V scale
// and whether all 64 keys are valid; one extra all-invalid tile closes each
// sequence.  Every CTA of the attention kernel then bulk-copies the images of
// its blocks: the 128 / (query tokens per CTA) CTAs of a sequence share one
// conversion instead of each converting every block.
//
// A CTA owns M = 128 consecutive query rows of one sequence: 128 / H query
// tokens times all H heads (MQA: every row reads the same K/V; the rows of
// tokens t and heads h are contiguous in q and out).  It walks the 128-key
// blocks its rows need, from the earliest row's window start to the last
// row's position.  Per block j:
//   S(j)  = Q K(j)^T     M = 128 rows, N = 128 keys, K = d: Q in tensor
//                        memory (A), K as fp16 in shared memory (B);
//   P'(j) = 2^(s - m) * s_v * 2^(6-E) per row and key (fp16, in tensor memory
//                        in place of S(j));
//   O    += P'(j) V(j)   M = 128 rows, N = 128 d, K = keys: P' in tensor
//                        memory (A), V as fp16 converted in place in its
//                        ring stage (B).
// Scores and O accumulate in fp32 tensor memory.
//
// Roles (20 warps, one CTA per SM):
//   warps 0-15  softmax, four warpgroups: quarter q takes keys 32 q .. 32 q + 31
//               of every block, thread r of each quarter owns query row r
//               (tensor-memory lane r).  Quarter 0 converts the row of Q to fp16
//               times one exact power of two into tensor memory.  Per block a
//               thread reads its 32 scores, takes off the K codes' exponent
//               bias (kBias * sum_d Q~[r][d]), applies the K scales and the
//               row's causal / window mask and writes P' for its keys.  The
//               row keeps one reference maximum (moved only when a score
//               passes it by more than 2^8; the quarters agree through a
//               barrier that ORs the need) and one power-of-two bound 2^E of
//               the V scales.  At the end each quarter normalises its D / 4
//               columns of the row of O.
//   warp 16     lane 0 issues every tcgen05.mma and commit, S(j) one block
//               ahead of O += P'(j-1) V(j-1); the warp owns the tensor memory.
//   warp 17     bulk copies: the two tile images and records of each block
//               into a ring stage once the O update that read the stage's
//               previous block has completed.
//   warps 18-19 idle (their registers go to the softmax warps).
//
// Every wait is bounded: a wait that runs out raises a CTA abort flag, every
// role leaves at its next check (the softmax warps all together, at the
// barrier that ORs the flag), copies and MMAs in flight are drained, and the
// call reports MQA_DEV_TIMEOUT.  Launched with programmatic stream
// serialisation: every global access comes after griddep_wait().
#include <atomic>
#include <math.h>

#include "common.cuh"
#include "kv_stage.cuh"
#include "launch.h"
#include "tc.cuh"
#include "tc_pipe.cuh"

namespace mqa {
namespace {

// A tile image (head_dim D): fp16 K [64 keys][D] in the core layout of the
// K-major B operand of S (8-key row groups D / 8 * 128 B apart, 8-d column groups
// 128 B apart), then fp16 V as two pieces of 64 * D bytes of the MN-major B
// operand of O (see PfCfg).
template <int D>
constexpr int tile_img_bytes() { return 2 * kTileTokens * D * 2; }
// A tile record: fp32 K scales [64], V scales [64], then the largest V scale of the
// valid keys, an all-valid flag (int) and two pad words.
constexpr int kTileRec = (2 * kTileTokens + 4) * 4;      // 528

template <int D_>
struct PfCfg {
    static constexpr int D = D_;                 // head_dim: 64 or 128
    static constexpr int IMG = tile_img_bytes<D>();
    static constexpr int RS = D / 8 * 128;       // bytes between 8-row groups of the K and V layouts
    static constexpr int M = 128;                // query rows per CTA
    static constexpr int BK = kBlockTokens;      // keys per block
    static constexpr int RING = D == 64 ? 4 : 3;  // (head_dim 64: also keeps one CTA per SM)
    static constexpr int QT = 4;                 // softmax warpgroups: each takes a quarter of a block's keys
    static constexpr int THREADS = 128 * QT + 128;
    static constexpr int MMA_WARP = 4 * QT, TMA_WARP = 4 * QT + 1;
    static constexpr int BAR_SM = 1;  // named barrier of the two softmax warpgroups
    static constexpr int REG_LAUNCH = (65536 / THREADS) / 8 * 8;  // 168
    static constexpr int REG_CTRL = 56;
    static constexpr int REG_WORK = ((REG_LAUNCH * THREADS - 128 * REG_CTRL) / (128 * QT)) / 8 * 8;
    static constexpr int CODES = BK * D;  // bytes of one V half (see the V layout below)
    static constexpr int V_W = 2 * RS;    // bytes of a 32-key group inside a V half
    // a ring stage: fp16 K of the block (its two tile images' K parts), fp16 V (their V
    // pieces), the two tile records
    static constexpr int ST_K = 0, ST_V = BK * D * 2, ST_REC = 2 * BK * D * 2;
    static constexpr int STAGE = (ST_REC + 2 * kTileRec + 1023) / 1024 * 1024;
    // shared memory
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_XM = OFF_RING + RING * STAGE;        // [2 parity][QT][128] row maxima / sums
    static constexpr int OFF_QG = OFF_XM + 2 * QT * M * 4;        // [2][128] g, bg of every row (quarter 0)
    static constexpr int OFF_MISC = OFF_QG + 2 * M * 4;           // tmem base, abort flag
    static constexpr int OFF_MBAR = OFF_MISC + 64;
    static constexpr int NBAR = 3 * RING + 6;
    static constexpr int SMEM_BYTES = OFF_MBAR + 8 * NBAR + 1024;
    // tensor memory: Q (fp16 pairs) | O | S [2]; P'(j) (fp16 pairs) replaces S(j) in its own
    // buffer once read: keys 0-63 at columns 0-31 of the buffer, keys 64-127 at 64-95
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t Q_COL = 0, O_COL = 64, S_COL = 192;
    // core-matrix strides: K rows = keys (K-major B of S); V rows = keys (MN-major B of O): key
    // 32 w + 8 g + i (w < 4, g < 4, i < 8) in half g / 2 (CODES bytes apart) at V_W w + RS (g % 2)
    // + 16 i, so a 16-key MMA step kk reads half kk % 2 at V_W (kk / 2); tile t of the block
    // holds w = 2t, 2t + 1, i.e. 64 * D bytes at 64 * D * t of each half
    static constexpr uint32_t K_SR = RS;   // next 8 keys
    static constexpr uint32_t K_SC = 128;  // next 8 d
    static constexpr uint32_t V_SR = RS;   // next 8 keys (inside a 16-key MMA step)
    static constexpr uint32_t V_SC = 128;  // next 8 d
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(STAGE % 1024 == 0 && ST_V % 1024 == 0, "1024-byte alignment");
    static_assert(ST_REC % 16 == 0 && kTileRec % 16 == 0 && IMG % 64 == 0 && OFF_XM % 16 == 0 && OFF_MISC % 16 == 0 &&
                      OFF_MBAR % 8 == 0,
                  "16-byte alignment");
    static_assert(O_COL + D <= S_COL && S_COL + 2 * 128 <= TMEM_COLS && Q_COL + D / 2 <= O_COL, "tensor memory");
    static_assert(128 * (QT * REG_WORK + REG_CTRL) <= REG_LAUNCH * THREADS && REG_WORK >= REG_LAUNCH,
                  "register split within the launch allocation");
};

constexpr float kBiasK = 1152.f;  // K codes enter the tensor core as code + 1152 (exact in fp16)

// A sequence's shape as both kernels read it: length L, query rows [q0, q0 + qlen),
// the window start klo of its first query, its first tile tf and the nt tiles from
// there to the one holding L - 1 (records 0 .. nt - 1, record nt all-invalid).
// False for a sequence without query rows or with lengths the launch does not
// allow (the attention kernel's CTA 0 reports those).
__device__ __forceinline__ bool pf_seq_shape(const PrefillArgs &a, int b, int &L, int &q0, int &qlen, int &klo,
                                             int &tf, int &nt)
{
    L = __ldg(a.seq_lens + b);
    q0 = __ldg(a.cu_q + b);
    const int q1 = __ldg(a.cu_q + b + 1);
    qlen = q1 - q0;
    if (L < 1 || L > a.max_seq_len || qlen < 1 || qlen > L || qlen > a.max_q_len || q0 < 0 || q1 > a.total_q)
        return false;
    klo = a.window > 0 ? max(0, L - qlen - a.window + 1) : 0;
    tf = klo / kTileTokens;
    nt = (L - 1) / kTileTokens - tf + 1;
    return nt + 1 <= a.tiles_max;
}

__device__ __forceinline__ void pf_regs_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PfCfg<128>::REG_WORK));
}
__device__ __forceinline__ void pf_regs_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PfCfg<128>::REG_CTRL));
}
static_assert(PfCfg<64>::REG_WORK == PfCfg<128>::REG_WORK && PfCfg<64>::REG_CTRL == PfCfg<128>::REG_CTRL,
              "one register split");

}  // namespace

template <int D_>
__global__ void __launch_bounds__(PfCfg<D_>::THREADS, 1) prefill_tc_kernel(const __grid_constant__ PrefillArgs a)
{
    using C = PfCfg<D_>;
    constexpr int D = C::D, RING = C::RING, BK = C::BK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + C::OFF_MISC + 4);
    uint64_t *tfull = reinterpret_cast<uint64_t *>(base + C::OFF_MBAR);  // [RING][2] tile images landed (copies)
    uint64_t *tfree = tfull + 2 * RING;  // [RING] stage free: O update of its block done (tensor core)
    uint64_t *sfull = tfree + RING;      // [2] S(j) done                                   (tensor core)
    uint64_t *pready = sfull + 2;        // P'(j) written, S(j) read                       (16 softmax warps)
    uint64_t *odone = pready + 1;        // O += P'(j) V(j) done                           (tensor core)
    uint64_t *qready = odone + 1;        // Q in tensor memory                             (4 softmax warps)
    uint64_t *ofinal = qready + 1;       // the last O update done (once per CTA)          (tensor core)
    static_assert(3 * C::RING + 6 == C::NBAR, "barrier count");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.num_q_heads;
    const int tpc = C::M / H;  // query tokens per CTA

    // ---- set-up (no global memory: overlaps the previous kernel)
    if (tid == 0) {
        for (int s = 0; s < 2 * RING; ++s)
            mbar_init(tfull + s, 1);
        for (int s = 0; s < RING; ++s)
            mbar_init(tfree + s, 1);
        for (int s = 0; s < 2; ++s)
            mbar_init(sfull + s, 1);
        mbar_init(pready, 4 * C::QT);
        mbar_init(odone, 1);
        mbar_init(qready, 4);
        mbar_init(ofinal, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::MMA_WARP)
        tmem_alloc(tmem_slot, C::TMEM_COLS);
    griddep_wait();
    griddep_launch_dependents();

    // ---- this CTA's tile: CTA x takes tile x of the list of every sequence's
    // ceil(q_len / tpc) tiles (a mixed batch of decode rows, q_len = 1, and long
    // prefill chunks launches no idle CTA per sequence); a block-wide scan of cu_q
    __shared__ int pf_scan[C::THREADS / 32 + 2];
    {
        if (tid == 0)
            pf_scan[C::THREADS / 32] = -1;
        long long run = 0;
        const long long x = blockIdx.x;
        for (int b0 = 0; b0 < a.batch; b0 += C::THREADS) {
            const int bb = b0 + tid;
            int nt = 0;
            if (bb < a.batch) {
                const int ql = __ldg(a.cu_q + bb + 1) - __ldg(a.cu_q + bb);
                nt = ql > 0 ? (ql + tpc - 1) / tpc : 0;
            }
            int incl = nt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off)
                    incl += y;
            }
            __syncthreads();  // pf_scan reuse
            if (lane == 31)
                pf_scan[warp] = incl;
            __syncthreads();
            long long pre = run, chunk = 0;
            for (int w = 0; w < C::THREADS / 32; ++w) {
                if (w < warp)
                    pre += pf_scan[w];
                chunk += pf_scan[w];
            }
            const long long lo_t = pre + incl - nt;
            if (nt > 0 && lo_t <= x && x < lo_t + nt) {
                pf_scan[C::THREADS / 32] = bb;
                pf_scan[C::THREADS / 32 + 1] = (int)(x - lo_t);
            }
            run += chunk;
        }
        __syncthreads();
    }
    const bool past_end = pf_scan[C::THREADS / 32] < 0;  // beyond the last tile: leaves below
    const int b = past_end ? 0 : pf_scan[C::THREADS / 32];
    const int t_begin = past_end ? 0 : pf_scan[C::THREADS / 32 + 1] * tpc;
    if (blockIdx.x == 0) {
        // one CTA reports bad lengths and query counts of the whole batch (a sequence with
        // q_len <= 0 gets no tile)
        for (int bb = tid; bb < a.batch; bb += C::THREADS) {
            const int Lb = __ldg(a.seq_lens + bb);
            const int qa = __ldg(a.cu_q + bb), qb = __ldg(a.cu_q + bb + 1);
            if (Lb < 1 || Lb > a.max_seq_len)
                set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
            else if (qb - qa > Lb || qa < 0 || qb < qa || qb > a.total_q || qb - qa > a.max_q_len)
                set_status(a.dev_status, MQA_DEV_BAD_CU);
        }
    }

    // ---- this CTA's rows and keys (every thread computes the same)
    int L, q0, qlen, klo_seq, tf, nt;
    const bool good = pf_seq_shape(a, b, L, q0, qlen, klo_seq, tf, nt);
    const int ntok = (!good || past_end) ? 0 : min(qlen, t_begin + tpc) - t_begin;  // query tokens of this CTA
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (ntok <= 0) {  // uniform: nothing to compute
        if (warp == C::MMA_WARP)
            tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }
    const int i0 = L - qlen + t_begin;     // position of the CTA's first query token
    const int i_last = i0 + ntok - 1;      // and of its last
    const int W = a.window;
    const int klo = W > 0 ? max(0, i0 - W + 1) : 0;       // keys the earliest row may see
    const int lo_max = W > 0 ? max(0, i_last - W + 1) : 0; // the window start of the latest row
    const int t_first = klo / kTileTokens;
    const int nb = (i_last / kTileTokens - t_first + 2) >> 1;  // 128-key blocks
    // block j holds tiles t_first + 2j, +1: the sequence's records t_first + 2j - tf, +1 (the
    // second of the last block may be the all-invalid record nt)

    if (warp < C::MMA_WARP)
        pf_regs_inc();
    else
        pf_regs_dec();

    if (warp < C::MMA_WARP) {
        // ================================================================ softmax
        // four warpgroups: quarter qt takes keys 32 qt .. 32 qt + 31 of every block for all 128
        // rows; thread r of each quarter owns query row r (tensor-memory lane r).  Every quarter
        // keeps the same reference per row; they agree on moving it through a barrier that ORs
        // the need (rare), and quarter 0 rescales O.
        const int qt = warp >> 2;  // quarter: keys 32 qt .. 32 qt + 31 of every block
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int t = r / H;
        const bool rvalid = t < ntok;
        const int ipos = i0 + t;
        const int lo_r = W > 0 ? max(0, ipos - W + 1) : 0;
        const size_t qrow = ((size_t)(q0 + t_begin) * H + r) * D;
        float* xm = reinterpret_cast<float *>(base + C::OFF_XM);  // [2 parity][QT][128]
        // ---- Q row: fp16 times 2^e (exact); quarter 0 writes it to tensor memory.  g turns a raw
        // score into the log2 domain, bg = kBias * sum_d Q~ * g takes the K codes' bias off
        float g, bg;
        float *qgb = reinterpret_cast<float *>(base + C::OFF_QG);
        if (qt == 0) {
            // quarter 0 converts the rows and publishes g, bg for the other quarters; two passes
            // over the row (the second from L1): its largest magnitude, then the conversion 64 d
            // at a time (the softmax threads run with ~100 registers)
            const uint4 *qg = reinterpret_cast<const uint4 *>(a.q + qrow);
            float mx = 0.f;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = rvalid ? __ldg(qg + c) : make_uint4(0, 0, 0, 0);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[u] << 16)), fabsf(__uint_as_float(w4[u] & 0xffff0000u))));
            }
            int e = 0;
            if (mx > 0.f && isfinite(mx)) {
                int x;
                frexpf(mx, &x);
                e = min(120, max(-120, 14 - x));
            }
            const float f = exp2i(e);
            g = a.q_scale_log2 * exp2i(-e);
            float qsum = 0.f;
#pragma unroll
            for (int half = 0; half < D / 64; ++half) {
                uint32_t hq[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = rvalid ? __ldg(qg + 8 * half + c) : make_uint4(0, 0, 0, 0);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        hq[4 * c + u] = pack_half2(__uint_as_float(w4[u] << 16) * f, __uint_as_float(w4[u] & 0xffff0000u) * f);
                        const __half2 h2 = *reinterpret_cast<const __half2 *>(&hq[4 * c + u]);
                        qsum += __low2float(h2);
                        qsum += __high2float(h2);
                    }
                }
                tmem_st32(tmem + lane_base + C::Q_COL + 32 * half, hq);
            }
            bg = kBiasK * qsum * g;
            qgb[r] = g;
            qgb[C::M + r] = bg;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(qready);
        }
        named_bar(C::BAR_SM, 128 * C::QT);  // g, bg of every row published
        g = qgb[r];
        bg = qgb[C::M + r];
        // the row's state, the same in every quarter: reference m (log2 domain), V-scale bound 2^E,
        // and c = 6 - E - m, which turns a masked score into the exponent of p * 2^(6-E);
        // lp: this quarter's sum of p * 2^(6-E)
        float m_run = -INFINITY, cexp = 0.f, lp = 0.f;
        int E_run = -100;
        bool ok = true;
        int j = 0;
        for (; j < nb; ++j) {
            const int b2 = j & 1, rs = j % RING;
            // (the copies and S(j) have usually completed long before: tests first)
            ok &= wait_done(tfull + 2 * rs, (uint32_t)(j / RING) & 1u, abort_flag);
            ok &= wait_done(tfull + 2 * rs + 1, (uint32_t)(j / RING) & 1u, abort_flag);
            ok &= wait_done(sfull + b2, (uint32_t)(j >> 1) & 1u, abort_flag);
            tc_fence_after();
            // this quarter's keys are half qt % 2 of the block's tile qt / 2: its record
            const uint8_t *recs = base + C::OFF_RING + rs * C::STAGE + C::ST_REC;
            const uint8_t *rec_t = recs + (qt >> 1) * kTileRec;
            const float *ks = reinterpret_cast<const float *>(rec_t) + 32 * (qt & 1);
            const float *vs = ks + kTileTokens;
            const int kb = (t_first + 2 * j) * kTileTokens + 32 * qt;  // first key of this quarter
            // every row sees every key of the quarter, and every key of its tile is valid
            const bool full = kb >= lo_max && kb + 31 <= i0 &&
                              reinterpret_cast<const int *>(rec_t)[2 * kTileTokens + 1] != 0 && rvalid;
            // ---- exponent arguments y = x + c (x the masked log2-domain score, -inf when masked),
            // as fp32 pairs: y = ((S g - b g) k_s) + c
            uint64_t y2[16];
            float ymx[2] = {-INFINITY, -INFINITY};  // independent partial maxima
            {
                uint32_t sr[32];
                tmem_ld32(tmem + lane_base + C::S_COL + (uint32_t)b2 * BK + 32 * qt, sr);
                tmem_wait_ld();
                const uint64_t g2 = f2pack(g, g), nbg2 = f2pack(-bg, -bg), c2 = f2pack(cexp, cexp);
                {
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 k4 = reinterpret_cast<const float4 *>(ks)[c4];
                        const uint32_t *sv = &sr[4 * c4];
                        const int c = 4 * c4;  // first key (of the quarter) of the four
                        uint64_t ya = fma2(fma2(f2pack(__uint_as_float(sv[0]), __uint_as_float(sv[1])), g2, nbg2),
                                           f2pack(k4.x, k4.y), c2);
                        uint64_t yb = fma2(fma2(f2pack(__uint_as_float(sv[2]), __uint_as_float(sv[3])), g2, nbg2),
                                           f2pack(k4.z, k4.w), c2);
                        float y0, y1, y2v, y3;
                        f2unpack(ya, y0, y1);
                        f2unpack(yb, y2v, y3);
                        if (!full) {
                            const int key = kb + c;
                            y0 = (rvalid && k4.x >= 0.f && key >= lo_r && key <= ipos) ? y0 : -INFINITY;
                            y1 = (rvalid && k4.y >= 0.f && key + 1 >= lo_r && key + 1 <= ipos) ? y1 : -INFINITY;
                            y2v = (rvalid && k4.z >= 0.f && key + 2 >= lo_r && key + 2 <= ipos) ? y2v : -INFINITY;
                            y3 = (rvalid && k4.w >= 0.f && key + 3 >= lo_r && key + 3 <= ipos) ? y3 : -INFINITY;
                            ya = f2pack(y0, y1);
                            yb = f2pack(y2v, y3);
                        }
                        y2[c / 2] = ya;
                        y2[c / 2 + 1] = yb;
                        ymx[0] = max3f(ymx[0], y0, y1);
                        ymx[1] = max3f(ymx[1], y2v, y3);
                    }
                }
            }
            const float ymax = fmaxf(ymx[0], ymx[1]);
            const float vmx = fmaxf(reinterpret_cast<const float *>(recs)[2 * kTileTokens],
                                    reinterpret_cast<const float *>(recs + kTileRec)[2 * kTileTokens]);
            // the reference holds while every y <= 14 - E (p <= 2^8) and the V bound covers the block;
            // a row without a reference yet moves at its first key
            const bool need = (m_run == -INFINITY && ymax != -INFINITY) || !(ymax <= 14.f - (float)E_run) ||
                              !(vmx <= exp2i(E_run));
            ok &= *abort_flag == 0;
            if (named_bar_or(C::BAR_SM, 128 * C::QT, need || !ok)) {
                if (named_bar_or(C::BAR_SM, 128 * C::QT, !ok))
                    break;  // abort: every quarter leaves here together
                // ---- rare: the row's reference and V bound move (every quarter computes the same)
                float *xmp = xm + b2 * C::QT * C::M;
                xmp[qt * C::M + r] = ymax - cexp;  // this quarter's largest masked score (log2 domain)
                named_bar(C::BAR_SM, 128 * C::QT);
                float xmax = xmp[r];
#pragma unroll
                for (int u = 1; u < C::QT; ++u)
                    xmax = fmaxf(xmax, xmp[u * C::M + r]);
                const float m_new = fmaxf(m_run, xmax);
                const int E_new = max(E_run, ceil_log2_pow(vmx));
                const float c_new = m_new == -INFINITY ? 0.f : (float)(6 - E_new) - m_new;
                // old terms in the new units: 2^(m - m') 2^(E - E')
                const float factor = m_run == -INFINITY ? 0.f : fast_exp2((m_run - m_new) + (float)(E_run - E_new));
                lp *= factor;
                if (qt == 0) {
                    // O of the previous blocks (its last update done: waited here) to the new units
                    const bool resc = j >= 1 && m_run != -INFINITY && factor != 1.f;
                    if (__any_sync(0xffffffffu, resc)) {
                        if (j >= 1)
                            ok &= wait_phase(odone, (uint32_t)(j - 1) & 1u, abort_flag);
                        tc_fence_after();
                        const float of = resc ? factor : 1.f;
#pragma unroll 1
                        for (int q8 = 0; q8 < D / 16; ++q8) {
                            uint32_t orr[16];
                            tmem_ld16(tmem + lane_base + C::O_COL + 16 * q8, orr);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                orr[c] = __float_as_uint(__uint_as_float(orr[c]) * of);
                            tmem_st16(tmem + lane_base + C::O_COL + 16 * q8, orr);
                        }
                        tmem_wait_st();
                    }
                }
                const uint64_t dc2 = f2pack(c_new - cexp, c_new - cexp);
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    y2[c] = add2(y2[c], dc2);
                m_run = m_new;
                E_run = E_new;
                cexp = c_new;
            }
            // ---- P' = 2^y * s_v (fp16) in place of this quarter's scores in S buffer b2, keys
            // 2c, 2c + 1 of the quarter in its column c (the O update that read this buffer's
            // previous P' was issued before S(j), which it holds now)
            const bool live = m_run != -INFINITY;
            uint32_t pk[16];
            uint64_t ls2 = 0;  // (0.f, 0.f): independent partial sums
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 v4 = reinterpret_cast<const float4 *>(vs)[c4];
                float y0, y1, y2v, y3;
                f2unpack(y2[2 * c4], y0, y1);
                f2unpack(y2[2 * c4 + 1], y2v, y3);
                const uint64_t pa = live ? f2pack(fast_exp2(y0), fast_exp2(y1)) : 0ull;
                const uint64_t pb = live ? f2pack(fast_exp2(y2v), fast_exp2(y3)) : 0ull;
                ls2 = add2(ls2, add2(pa, pb));
                float q0, q1, q2v, q3;
                f2unpack(mul2(pa, f2pack(v4.x, v4.y)), q0, q1);
                f2unpack(mul2(pb, f2pack(v4.z, v4.w)), q2v, q3);
                pk[2 * c4] = pack_half2(q0, q1);
                pk[2 * c4 + 1] = pack_half2(q2v, q3);
            }
            {
                float la, lb;
                f2unpack(ls2, la, lb);
                lp += la + lb;
            }
            tmem_st16(tmem + lane_base + C::S_COL + (uint32_t)b2 * BK + 32 * qt, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(pready);
        }
        // ---- epilogue: out = O / (sum of p * 2^(6-E)), quarter qt writing d = D/4 qt .. D/4 qt + D/4 - 1
        if (j == nb) {
            float *ls2 = xm + (nb & 1) * C::QT * C::M;  // parity slot the last block did not use
            ls2[qt * C::M + r] = lp;
            named_bar(C::BAR_SM, 128 * C::QT);
            float lt = 0.f;
#pragma unroll
            for (int u = 0; u < C::QT; ++u)
                lt += ls2[u * C::M + r];
            ok &= wait_phase(ofinal, 0u, abort_flag);  // the CTA's last O update
            tc_fence_after();
            const float of = lt > 0.f ? 1.f / lt : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + qrow + (D / 4) * qt);
            constexpr int NC = D / 4;  // columns of this quarter: 32 or 16
            uint32_t orr[NC];
            if constexpr (NC == 32)
                tmem_ld32(tmem + lane_base + C::O_COL + NC * qt, orr);
            else
                tmem_ld16(tmem + lane_base + C::O_COL + NC * qt, orr);
            tmem_wait_ld();
            if (rvalid) {
#pragma unroll
                for (int c = 0; c < NC / 8; ++c)
                    dst[c] = make_uint4(
                        pack_bf16x2(__uint_as_float(orr[8 * c + 0]) * of, __uint_as_float(orr[8 * c + 1]) * of),
                        pack_bf16x2(__uint_as_float(orr[8 * c + 2]) * of, __uint_as_float(orr[8 * c + 3]) * of),
                        pack_bf16x2(__uint_as_float(orr[8 * c + 4]) * of, __uint_as_float(orr[8 * c + 5]) * of),
                        pack_bf16x2(__uint_as_float(orr[8 * c + 6]) * of, __uint_as_float(orr[8 * c + 7]) * of));
            }
        }
        tc_fence_before();
        bar_all();
        if (tid == 0 && *abort_flag)
            set_status(a.dev_status, MQA_DEV_TIMEOUT);
        return;
    } else if (warp == C::TMA_WARP) {
        // ================================================================ image copies
        // block j into ring stage j % RING once the O update of block j - RING has read it:
        // lane 4t + k copies tile t's K image (k = 0), V pieces (k = 1, 2) or record (k = 3)
        const int t = (lane >> 2) & 1, k = lane & 3;
        int j = 0;
        for (; j < nb; ++j) {
            const int r = j % RING;
            if (j >= RING &&
                !__all_sync(0xffffffffu, wait_phase(tfree + r, (uint32_t)(j / RING - 1) & 1u, abort_flag)))
                break;
            uint8_t *st = base + C::OFF_RING + r * C::STAGE;
            const size_t rec = (size_t)b * a.tiles_max + (t_first + 2 * j + t - tf);  // < tiles_max (pf_seq_shape)
            if (lane < 2)
                mbar_arrive_expect_tx(tfull + 2 * r + lane, C::IMG + kTileRec);
            __syncwarp();
            if (lane < 8) {
                uint64_t *bar = tfull + 2 * r + t;
                const uint8_t *img = a.img + rec * C::IMG;
                if (k == 0)
                    bulk_load(st + C::ST_K + t * (C::IMG / 2), img, C::IMG / 2, bar);
                else if (k < 3)
                    bulk_load(st + C::ST_V + (k - 1) * C::CODES + t * (C::IMG / 4), img + (C::IMG / 4) * (k + 1),
                              C::IMG / 4, bar);
                else
                    bulk_load(st + C::ST_REC + t * kTileRec, a.srec + rec * kTileRec, kTileRec, bar);
            }
        }
        if (*abort_flag && lane == 0) {
            // the copies still in flight land before the CTA leaves
            for (int jj = max(0, j - RING); jj < j; ++jj)
                for (int tt = 0; tt < 2; ++tt)
                    mbar_wait_drain(tfull + 2 * (jj % RING) + tt, (uint32_t)(jj / RING) & 1u);
        }
        tc_fence_before();
        bar_all();
        return;
    } else {
        // ================================================================ MMA issuer (and idle warps)
        if (warp == C::MMA_WARP && lane == 0) {
            constexpr uint32_t IDESC_S = umma_idesc_f16(128, BK, false, false);
            constexpr uint32_t IDESC_O = umma_idesc_f16(128, D, false, true);
            const uint64_t kdesc0 = umma_sdesc(smem_u32(base + C::OFF_RING + C::ST_K), C::K_SC, C::K_SR);
            const uint64_t vdesc0 = umma_sdesc(smem_u32(base + C::OFF_RING + C::ST_V), C::V_SR, C::V_SC);
            int n_s = 0, n_o = 0;
            // O += P'(k) V(k): P' from S buffer k & 1 (keys 16kk .. 16kk+15 at column
            // 32 (kk / 2) + 8 (kk % 2)), V (fp16 in ring stage k % RING) from shared memory;
            // 16-key step kk = key groups 2kk, 2kk+1: half kk % 2 at V_W (kk / 2)
            auto issue_o = [&](int k) -> bool {
                if (!wait_phase(pready, (uint32_t)k & 1u, abort_flag))
                    return false;
                tc_fence_after();
                const uint64_t vd = desc_add(vdesc0, (k % RING) * C::STAGE);
                const uint32_t pcol = C::S_COL + (uint32_t)(k & 1) * BK;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_f16_ts(tmem + C::O_COL, tmem + pcol + 32 * (kk >> 1) + 8 * (kk & 1),
                                desc_add(vd, (kk & 1) * C::CODES + (kk >> 1) * C::V_W), IDESC_O, k > 0 || kk > 0);
                umma_commit(odone);
                umma_commit(tfree + (k % RING));  // the stage's V is read: the TMA warp may refill it
                ++n_o;
                return true;
            };
            bool ok = wait_phase(qready, 0u, abort_flag);
            for (int j = 0; j < nb && ok; ++j) {
                const int b2 = j & 1;
                // S(j) = Q K(j)^T into S buffer b2: its last contents, P'(j-2), were read by the O
                // update issued in the previous step (the tensor core runs this thread's MMAs in order)
                if (!wait_phase(tfull + 2 * (j % RING), (uint32_t)(j / RING) & 1u, abort_flag) ||
                    !wait_phase(tfull + 2 * (j % RING) + 1, (uint32_t)(j / RING) & 1u, abort_flag))
                    break;
                tc_fence_after();
                const uint64_t kd = desc_add(kdesc0, (uint32_t)(j % RING) * C::STAGE);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_f16_ts(tmem + C::S_COL + (uint32_t)b2 * BK, tmem + C::Q_COL + 8 * kk,
                                desc_add(kd, kk * 2 * C::K_SC), IDESC_S, kk > 0);
                umma_commit(sfull + b2);
                ++n_s;
                if (j >= 1)
                    ok = issue_o(j - 1);
            }
            if (ok && n_s == nb && issue_o(nb - 1))
                umma_commit(ofinal);
            if (*abort_flag) {
                if (n_o > 0)
                    mbar_wait_drain(odone, (uint32_t)(n_o - 1) & 1u);
                if (n_s > 0)
                    mbar_wait_drain(sfull + ((n_s - 1) & 1), (uint32_t)((n_s - 1) >> 1) & 1u);
            }
        }
        tc_fence_before();
        bar_all();
        if (warp == C::MMA_WARP) {
            tc_fence_after();
            tmem_dealloc(tmem, C::TMEM_COLS);
        }
        return;
    }
}

// Tile record blockIdx.x of sequence blockIdx.y: 256 threads, 64 keys.  Keys
// from the window start of the sequence's first query to L - 1 are valid
// (their block ids inside the pool); any other key gets code 0, K scale -1
// and V scale 0, and record nt (past the sequence's last tile) is all such
// keys.  Codes are converted exactly: K to code + 1152 (the exponent-bias
// form of its byte; the attention kernel takes the bias off), V to the code.
template <int D>
__global__ void __launch_bounds__(256) kv_tile_images_kernel(const __grid_constant__ PrefillArgs a)
{
    using C = PfCfg<D>;
    griddep_wait();  // the appended keys are visible from here
    griddep_launch_dependents();
    const int b = blockIdx.y, idx = blockIdx.x, tid = threadIdx.x;
    int L, q0, qlen, klo, tf, nt;
    if (!pf_seq_shape(a, b, L, q0, qlen, klo, tf, nt) || idx > nt)
        return;
    const int T = tf + idx;
    uint8_t *img = a.img + ((size_t)b * a.tiles_max + idx) * C::IMG;
    float *rec = reinterpret_cast<float *>(a.srec + ((size_t)b * a.tiles_max + idx) * kTileRec);
    __shared__ int s_row[kTileTokens];  // cache row of each key, -1 = not valid
    __shared__ float s_vmax[2];
    __shared__ int s_all[2];
    if (tid < kTileTokens) {
        const int pos = T * kTileTokens + tid;
        int row = -1;
        if (idx < nt && pos >= klo && pos < L) {
            const int id = __ldg(a.block_table + (size_t)b * a.max_blocks + table_entry(pos / a.page_size, a.ring));
            if (id >= 0 && id < a.num_blocks)
                row = id * a.page_size + pos % a.page_size;
            else
                set_status(a.dev_status, MQA_DEV_BAD_BLOCK);
        }
        s_row[tid] = row;
        const float vs = row >= 0 ? __ldg(a.v_scale + row) : 0.f;
        rec[tid] = row >= 0 ? __ldg(a.k_scale + row) : -1.f;
        rec[kTileTokens + tid] = vs;
        float vm = vs;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
        const bool all = __all_sync(0xffffffffu, row >= 0);
        if ((tid & 31) == 0) {
            s_vmax[tid >> 5] = vm;
            s_all[tid >> 5] = all ? 1 : 0;
        }
    }
    __syncthreads();
    if (tid == 0) {
        rec[2 * kTileTokens] = fmaxf(s_vmax[0], s_vmax[1]);
        reinterpret_cast<int *>(rec)[2 * kTileTokens + 1] = s_all[0] & s_all[1];
        rec[2 * kTileTokens + 2] = 0.f;
        rec[2 * kTileTokens + 3] = 0.f;
    }
    // K part: 16-byte piece at byte o holds key 8 (o / RS) + (o / 16) % 8, d = 8 ((o % RS) / 128) ..
    for (int c = tid; c < C::IMG / 32; c += 256) {
        const uint32_t o = 16u * c;
        const int key = (int)(o / C::RS) * 8 + (int)((o >> 4) & 7);
        const int d0 = (int)((o % C::RS) >> 7) * 8;
        const int row = s_row[key];
        const uint2 w = row >= 0 ? __ldg(reinterpret_cast<const uint2 *>(a.k_codes + (size_t)row * D + d0))
                                 : make_uint2(0u, 0u);
        const uint32_t t0 = w.x ^ 0x80808080u, t1 = w.y ^ 0x80808080u;
        *reinterpret_cast<uint4 *>(img + o) =
            make_uint4(__byte_perm(t0, 0x64646464u, 0x5140), __byte_perm(t0, 0x64646464u, 0x7362),
                       __byte_perm(t1, 0x64646464u, 0x5140), __byte_perm(t1, 0x64646464u, 0x7362));
    }
    // V part: piece h (64 D bytes) holds the keys 32 w + 8 g + i with g / 2 == h, the 16-byte piece
    // at byte p of it key 32 (p / V_W) + 8 (2 h + (p / RS) % 2) + (p / 16) % 8, d = 8 ((p % RS) / 128) ..
    for (int c = tid; c < C::IMG / 32; c += 256) {
        const uint32_t o = 16u * c;
        const int h = (int)(o / (C::IMG / 4));
        const uint32_t p = o % (C::IMG / 4);
        const int key = (int)(p / C::V_W) * 32 + (2 * h + (int)((p / C::RS) & 1)) * 8 + (int)((p >> 4) & 7);
        const int d0 = (int)((p % C::RS) >> 7) * 8;
        const int row = s_row[key];
        const uint2 w = row >= 0 ? __ldg(reinterpret_cast<const uint2 *>(a.v_codes + (size_t)row * D + d0))
                                 : make_uint2(0u, 0u);
        uint32_t v[4];
        i8x4_to_f16x2x2(w.x, v[0], v[1]);
        i8x4_to_f16x2x2(w.y, v[2], v[3]);
        *reinterpret_cast<uint4 *>(img + C::IMG / 2 + o) = make_uint4(v[0], v[1], v[2], v[3]);
    }
}

namespace {

template <int D>
cudaError_t launch_prefill_tc_t(const PrefillArgs &a, cudaStream_t s)
{
    using C = PfCfg<D>;
    static std::atomic<int> attr_set{0};
    if (!attr_set.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        // the kernel moves registers between its warpgroups (setmaxnreg): the split must fit the
        // registers it is launched with, or a group would wait for registers forever
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<D>);
        if (e != cudaSuccess)
            return e;
        if (fa.numRegs != C::REG_LAUNCH)
            return cudaErrorInvalidConfiguration;
        attr_set.store(1, std::memory_order_release);
    }
    // an upper bound of the tiles (sum over sequences of ceil(q_len / tpc)); CTAs past the
    // last tile leave at once
    const int tpc = C::M / a.num_q_heads;
    const long long tiles = ((long long)a.total_q + tpc - 1) / tpc + a.batch;
    if (tiles > 0x7fffffffll)
        return cudaErrorInvalidConfiguration;
    cudaError_t e = launch_pdl(kv_tile_images_kernel<D>, dim3((unsigned)a.tiles_max, (unsigned)a.batch, 1),
                               dim3(256), 0, s, a);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(prefill_tc_kernel<D>, dim3((unsigned)tiles, 1, 1), dim3(C::THREADS), C::SMEM_BYTES, s, a);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, int head_dim, cudaStream_t s)
{
    return head_dim == 64 ? launch_prefill_tc_t<64>(a, s) : launch_prefill_tc_t<128>(a, s);
}

// Tile records per sequence a prefill of this shape needs (its tiles plus the all-invalid one):
// see pf_seq_shape.
int prefill_tiles_max(int max_seq_len, int window, int max_q_len)
{
    long long t = ((long long)max_seq_len - 1) / kTileTokens + 1;
    if (window > 0) {
        const long long w = ((long long)window + max_q_len - 2) / kTileTokens + 2;
        t = w < t ? w : t;
    }
    return (int)(t + 1);
}

size_t prefill_tile_image_bytes(int head_dim) { return head_dim == 64 ? tile_img_bytes<64>() : tile_img_bytes<128>(); }
size_t prefill_tile_record_bytes() { return kTileRec; }

}  // namespace mqa
