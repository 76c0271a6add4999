// Decode attention on the 5th-generation tensor cores (tcgen05), head_dim 128,
// 32 query heads per CTA.
//
// Per CTA (one split of one sequence, 8 warps, one CTA per SM):
//  * keys arrive as 128-token blocks (two 64-token tiles = eight 16-token
//    boxes) through a ring of RING blocks: per box one TMA tiled load of K
//    codes, one of V codes (2-D maps over [num_blocks*page, 128] int8,
//    128-byte swizzle) and two 64-byte bulk copies of the scales, each box on
//    its own mbarrier; boxes outside [window start, L) are not fetched;
//  * every int8 code is converted exactly once (exponent-bias trick, exact) into
//    fp16 operand tiles in shared memory, K and V in one "core matrix" layout
//    (8 token rows x 8 d, 16-byte rows) that serves as the K-major A operand of
//    QK^T and as the MN-major A operand of PV;
//  * MQA puts all 32 heads of a token into one row of a dense contraction:
//      S^T[128 tokens x 32 heads]  = K[128 x 128] . Q^T      (tcgen05, TMEM)
//      O^T[128 d x 32 heads]     += V^T[128 x 128] . P      (tcgen05, TMEM)
//    one thread issues the MMAs; the accumulators live in tensor memory;
//  * softmax: thread (token t, head half) reads its token's 16 scores with
//    tcgen05.ld, applies the K scale, and exponentiates against a per-head
//    reference maximum that only moves when a score exceeds it by more than
//    2^8 (then the CTA rescales O in tensor memory and l in registers: rare);
//    the V scale is folded into P' = p * s_v * 2^(6-E), 2^E a running
//    power-of-two bound of the V scales, so fp16 P' never overflows;
//  * output: bf16 directly, or fp32 partial O and lse per split (merged by the
//    last split CTA for <= 16 splits, else by the combine kernel).
#include <atomic>
#include <cfloat>
#include <math.h>

#include "common.cuh"
#include "kv_stage.cuh"
#include "launch.h"
#include "split_merge.cuh"
#include "tc.cuh"

namespace mqa {
namespace {

struct TcCfg {
    static constexpr int D = 128;
    static constexpr int NH = 32;                 // heads per CTA (MMA N)
    static constexpr int BT = 128;                // tokens per block (MMA M of QK^T, K of PV)
    static constexpr int BOXES = BT / kChunkTokens;  // 8
    static constexpr int RING = 3;                // blocks in flight
    static constexpr int THREADS = 256;
    static constexpr int CODES = BT * D;          // int8 bytes of K (or V) of a block
    static constexpr int STAGE = 2 * CODES + 1024;  // K codes, V codes, K and V scales (1 KB)
    // shared memory (offsets from a 1024-aligned base)
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_KH = OFF_RING + RING * STAGE;    // fp16 K [128 tok][128 d], core layout
    static constexpr int OFF_VH = OFF_KH + BT * D * 2;        // fp16 V, same layout
    static constexpr int OFF_QH = OFF_VH + BT * D * 2;        // fp16 Q [32 h][128 d], core layout
    static constexpr int OFF_PH = OFF_QH + NH * D * 2;        // fp16 P' [128 tok][32 h], core layout
    static constexpr int OFF_RED = OFF_PH + BT * NH * 2;      // 256 fp32: reductions across warps
    static constexpr int OFF_OK = OFF_RED + 256 * 4;          // [RING][8] box arrived
    static constexpr int OFF_MISC = OFF_OK + RING * BOXES * 4;  // tmem base, flags
    static constexpr int OFF_MBAR = OFF_MISC + 64;            // [RING][8] + S + O
    static constexpr int SMEM_BYTES = OFF_MBAR + 8 * (RING * BOXES + 2) + 1024;
    static constexpr uint32_t TMEM_COLS = 128;    // S (2 x 32) + O (32), power of two
    // core-matrix strides (bytes): K/V tiles rows = tokens, Q rows = heads, P rows = tokens
    static constexpr uint32_t KV_SR = 16 * 128;   // next 8 tokens
    static constexpr uint32_t KV_SC = 128;        // next 8 d
    static constexpr uint32_t Q_SR = 16 * 128;    // next 8 heads
    static constexpr uint32_t Q_SC = 128;
    static constexpr uint32_t P_SR = 4 * 128;     // next 8 tokens
    static constexpr uint32_t P_SC = 128;         // next 8 heads
};

// One box of a ring block: K and V codes (16 rows x 128 B each, TMA with
// 128-byte swizzle) and their 16 + 16 scales.
__device__ __forceinline__ void issue_block_box(const DecodeArgs &a, int32_t id, uint8_t *stage, uint64_t *bar,
                                                uint32_t *box_ok, int T, int c, int box)
{
    constexpr int D = TcCfg::D;
    const int t0 = T * kTileTokens + c * kChunkTokens;
    const bool ok = id >= 0 && id < a.num_blocks;
    if (!ok && id != kNoBlock)
        set_status(a.dev_status, MQA_DEV_BAD_BLOCK);
    *box_ok = ok ? 1u : 0u;
    if (!ok) {
        mbar_arrive_expect_tx(bar, 0);
        return;
    }
    const int row = id * a.page_size + (t0 % a.page_size);
    float *ks = reinterpret_cast<float *>(stage + 2 * TcCfg::CODES);
    mbar_arrive_expect_tx(bar, 2 * kChunkTokens * D + 2 * kChunkTokens * 4);
    tma_load_2d(stage + box * kChunkTokens * D, &a.k_map, 0, row, bar);
    tma_load_2d(stage + TcCfg::CODES + box * kChunkTokens * D, &a.v_map, 0, row, bar);
    bulk_load(ks + box * kChunkTokens, a.k_scale + row, kChunkTokens * 4, bar);
    bulk_load(ks + TcCfg::BT + box * kChunkTokens, a.v_scale + row, kChunkTokens * 4, bar);
}

}  // namespace

__global__ void __launch_bounds__(TcCfg::THREADS, 1) decode_tc_kernel(const __grid_constant__ DecodeArgs a)
{
    using C = TcCfg;
    constexpr int D = C::D, NH = C::NH, RING = C::RING;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *kh = base + C::OFF_KH;
    uint8_t *vh = base + C::OFF_VH;
    uint8_t *qh = base + C::OFF_QH;
    uint8_t *ph = base + C::OFF_PH;
    float *red = reinterpret_cast<float *>(base + C::OFF_RED);
    uint32_t *box_ok = reinterpret_cast<uint32_t *>(base + C::OFF_OK);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + C::OFF_MISC);
    volatile int *flag = reinterpret_cast<int *>(base + C::OFF_MISC + 8);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(base + C::OFF_MBAR);  // [RING][8] boxes
    uint64_t *mbar_s = mbar + RING * C::BOXES;
    uint64_t *mbar_o = mbar_s + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tok = 32 * (warp & 3) + lane;  // token row of a block = tensor-memory lane
    const int hh = warp >> 2;                // head half: heads 16hh .. 16hh+15 of the CTA
    const int split = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * NH;
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
        if (bad && tid == 0 && split == 0)
            set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
        for (int r = tid; r < NH; r += blockDim.x) {
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
    const int n_blocks = (n_tiles + 1) / 2;
    const int32_t *table = a.block_table + (size_t)b * a.max_blocks;

    // ---- set-up: barriers, tensor memory, the first RING blocks in flight
    if (tid == 0) {
        for (int s = 0; s < RING * C::BOXES + 2; ++s)
            mbar_init(mbar + s, 1);
        *flag = 0;
        fence_mbar_init();
    }
    if (warp == 0)
        tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // warp w produces box w of every block: tile (w / 4) of the block, box (w % 4) of the tile
    const int my_tile = warp >> 2, my_c = warp & 3;
    if (lane == 0)
        for (int j = 0; j < n_blocks && j < RING; ++j) {
            const int T = tb + 2 * j + my_tile;
            const int32_t id = T < te ? fetch_box_block(table, a.page_size, T, my_c, lo, L) : kNoBlock;
            issue_block_box(a, id, base + C::OFF_RING + j * C::STAGE, mbar + j * C::BOXES + warp,
                            box_ok + j * C::BOXES + warp, T, my_c, warp);
        }

    // ---- Q: 32 heads x 128 d, scaled by one power of two 2^e (exact in fp16), into
    // the core-matrix layout of the QK^T B operand (rows = heads, K-major)
    {
        // thread covers head (tid >> 3), d = 16*(tid & 7) .. +15
        const int qr = tid >> 3, qc = (tid & 7) * 16;
        const int h = h0 + qr;
        uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
        if (h < a.num_q_heads) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.num_q_heads + h) * D + qc);
            v0 = __ldg(src);
            v1 = __ldg(src + 1);
        }
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xffff0000u))));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0)
            red[warp] = m;
        __syncthreads();
        m = red[0];
#pragma unroll
        for (int k = 1; k < 8; ++k)
            m = fmaxf(m, red[k]);
        int e = 0;
        if (m > 0.f && isfinite(m)) {
            int x;
            frexpf(m, &x);
            e = 14 - x;
            e = e < -120 ? -120 : (e > 120 ? 120 : e);
        }
        const float f = exp2i(e);
        uint32_t hv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            hv[k] = pack_half2(__uint_as_float(w[k] << 16) * f, __uint_as_float(w[k] & 0xffff0000u) * f);
        *reinterpret_cast<uint4 *>(qh + core_off(qr, qc, C::Q_SR, C::Q_SC)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4 *>(qh + core_off(qr, qc + 8, C::Q_SR, C::Q_SC)) =
            make_uint4(hv[4], hv[5], hv[6], hv[7]);
        if (tid == 0)
            red[8] = a.q_scale_log2 * exp2i(-e);  // log2-domain factor of the raw scores
    }
    fence_proxy_async();
    __syncthreads();
    const float gh = red[8];

    float m_ref[16], l_acc[16];  // heads 16hh + j: reference max (raw-score units), this thread's sum of p
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        m_ref[j] = -INFINITY;
        l_acc[j] = 0.f;
    }
    int E_run = -100;       // running power-of-two bound of the V scales
    bool o_valid = false;   // O has been written by a first PV
    const uint32_t tl = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's tensor-memory lanes
    constexpr uint32_t O_COL = 64;
    constexpr uint32_t IDESC_QK = umma_idesc_f16(128, NH, false, false);
    constexpr uint32_t IDESC_PV = umma_idesc_f16(128, NH, true, true);
    const uint32_t kh_u = smem_u32(kh), vh_u = smem_u32(vh), qh_u = smem_u32(qh), ph_u = smem_u32(ph);
    int blk = 0;
    int n_issued = min(n_blocks, RING);  // blocks whose boxes are in flight or landed
    int n_qk = 0, n_pv = 0;              // MMA groups issued (same in every thread)
    for (; blk < n_blocks; ++blk) {
        const int r = blk % RING;
        uint8_t *st = base + C::OFF_RING + r * C::STAGE;
        const float *ks = reinterpret_cast<const float *>(st + 2 * C::CODES);
        const float *vs = ks + C::BT;
        const int mybox = tok >> 4;
        // block id of my box of block blk + RING, fetched ahead of its issue
        int32_t id_next = kNoBlock;
        const int T_next = tb + 2 * (blk + RING) + my_tile;
        if (lane == 0 && blk + RING < n_blocks && T_next < te)
            id_next = fetch_box_block(table, a.page_size, T_next, my_c, lo, L);
        if (!mbar_wait_bounded(mbar + r * C::BOXES + mybox, (uint32_t)(blk / RING) & 1u))
            *flag = 1;
        const bool ok = box_ok[r * C::BOXES + mybox] != 0;
        const int pos = (tb + 2 * blk) * kTileTokens + tok;
        const bool valid = ok && pos >= lo && pos < L;
        // the previous PV reads V, P and writes O: wait before touching them
        if (blk > 0) {
            if (!mbar_wait_bounded(mbar_o, (uint32_t)(blk - 1) & 1u))
                *flag = 1;
            tc_fence_after();
        }
        // ---- convert this token's K and V codes, d in [64hh, 64hh+64), to fp16 (exact)
        {
            const uint8_t *krow = st + tok * D;
            const uint8_t *vrow = st + C::CODES + tok * D;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 4 * hh + q;  // 16-byte chunk of the row (d = 16j .. 16j+15)
                const uint32_t so = (uint32_t)(j ^ (tok & 7)) << 4;
                const uint4 kv = *reinterpret_cast<const uint4 *>(krow + so);
                const uint4 vv = *reinterpret_cast<const uint4 *>(vrow + so);
                uint32_t k8[8], v8[8];
                i8x4_to_f16x2x2(kv.x, k8[0], k8[1]);
                i8x4_to_f16x2x2(kv.y, k8[2], k8[3]);
                i8x4_to_f16x2x2(kv.z, k8[4], k8[5]);
                i8x4_to_f16x2x2(kv.w, k8[6], k8[7]);
                i8x4_to_f16x2x2(vv.x, v8[0], v8[1]);
                i8x4_to_f16x2x2(vv.y, v8[2], v8[3]);
                i8x4_to_f16x2x2(vv.z, v8[4], v8[5]);
                i8x4_to_f16x2x2(vv.w, v8[6], v8[7]);
                const uint32_t o0 = core_off(tok, 16 * j, C::KV_SR, C::KV_SC);
                const uint32_t o1 = core_off(tok, 16 * j + 8, C::KV_SR, C::KV_SC);
                *reinterpret_cast<uint4 *>(kh + o0) = make_uint4(k8[0], k8[1], k8[2], k8[3]);
                *reinterpret_cast<uint4 *>(kh + o1) = make_uint4(k8[4], k8[5], k8[6], k8[7]);
                *reinterpret_cast<uint4 *>(vh + o0) = make_uint4(v8[0], v8[1], v8[2], v8[3]);
                *reinterpret_cast<uint4 *>(vh + o1) = make_uint4(v8[4], v8[5], v8[6], v8[7]);
            }
        }
        const float ksv = ks[tok], vsv = vs[tok];
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();  // B1: fp16 K/V ready; ring slot r fully read
        if (*flag)
            break;
        tc_fence_after();
        if (blk + RING < n_blocks) {
            if (lane == 0)
                issue_block_box(a, T_next < te ? id_next : kNoBlock, st, mbar + r * C::BOXES + warp,
                                box_ok + r * C::BOXES + warp, T_next, my_c, warp);
            ++n_issued;
        }
        // ---- S^T = K Q^T on the tensor cores
        const uint32_t s_col = (uint32_t)(blk & 1) * NH;
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_f16(tmem + s_col, umma_sdesc(kh_u + kk * 2 * C::KV_SC, C::KV_SC, C::KV_SR),
                         umma_sdesc(qh_u + kk * 2 * C::Q_SC, C::Q_SC, C::Q_SR), IDESC_QK, kk > 0);
            umma_commit(mbar_s);
        }
        ++n_qk;
        if (!mbar_wait_bounded(mbar_s, (uint32_t)blk & 1u))
            *flag = 1;
        tc_fence_after();
        uint32_t sr[16];
        tmem_ld16(tmem + tl + s_col + 16 * hh, sr);
        tmem_wait_ld();
        // ---- softmax against the reference maxima
        float y[16], dd[16];
        bool need = valid && !(vsv <= exp2i(E_run));
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            y[j] = valid ? __uint_as_float(sr[j]) * ksv : -INFINITY;
            dd[j] = valid ? fmaf(y[j], gh, -m_ref[j] * gh) : -INFINITY;
            need |= valid && !(dd[j] <= 8.f);
        }
        if (__syncthreads_or(need)) {  // B2 (rare after the first block): move the references
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float m = y[j];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                if (lane == 0)
                    red[warp * 16 + j] = m;
            }
            float vm = valid ? vsv : 0.f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
            if (lane == 0)
                red[128 + warp] = vm;
            __syncthreads();
            float vmax = red[128];
#pragma unroll
            for (int k = 1; k < 8; ++k)
                vmax = fmaxf(vmax, red[128 + k]);
            const int E_new = max(E_run, ceil_log2_pow(vmax));
            const int dE = E_run - E_new;
            const float escale = dE < -126 ? 0.f : exp2i(dE);
            float fo[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float bm = red[(4 * hh) * 16 + j];
#pragma unroll
                for (int k = 1; k < 4; ++k)
                    bm = fmaxf(bm, red[(4 * hh + k) * 16 + j]);
                const float mn = fmaxf(m_ref[j], bm);
                const float fl = (mn == -INFINITY) ? 1.f : fast_exp2((m_ref[j] - mn) * gh);
                l_acc[j] *= fl;
                fo[j] = fl * escale;
                m_ref[j] = mn;
                dd[j] = valid ? fmaf(y[j], gh, -mn * gh) : -INFINITY;
            }
            E_run = E_new;
            if (o_valid) {
                // O^T row tok (a d index), columns = heads 16hh..16hh+15
                uint32_t orr[16];
                tmem_ld16(tmem + tl + O_COL + 16 * hh, orr);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    orr[j] = __float_as_uint(__uint_as_float(orr[j]) * fo[j]);
                tmem_st16(tmem + tl + O_COL + 16 * hh, orr);
                tmem_wait_st();
            }
        }
        // ---- P' = 2^dd * s_v * 2^(6-E) as fp16 row tok of P (heads 16hh..16hh+15)
        const float vf = valid ? vsv * exp2i(6 - E_run) : 0.f;
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float p0 = fast_exp2(dd[2 * k]), p1 = fast_exp2(dd[2 * k + 1]);
            l_acc[2 * k] += p0;
            l_acc[2 * k + 1] += p1;
            pk[k] = pack_half2(p0 * vf, p1 * vf);
        }
        *reinterpret_cast<uint4 *>(ph + core_off(tok, 16 * hh, C::P_SR, C::P_SC)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4 *>(ph + core_off(tok, 16 * hh + 8, C::P_SR, C::P_SC)) =
            make_uint4(pk[4], pk[5], pk[6], pk[7]);
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();  // B3: P' ready (and any O rescale done)
        if (*flag)
            break;
        tc_fence_after();
        // ---- O^T += V^T P' on the tensor cores (A = V, B = P', both MN-major)
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < C::BT / 16; ++kk)
                umma_f16(tmem + O_COL, umma_sdesc(vh_u + kk * 2 * C::KV_SR, C::KV_SR, C::KV_SC),
                         umma_sdesc(ph_u + kk * 2 * C::P_SR, C::P_SR, C::P_SC), IDESC_PV, o_valid || kk > 0);
            umma_commit(mbar_o);
        }
        ++n_pv;
        o_valid = true;
    }

    const bool timed_out = *flag != 0;
    if (timed_out) {
        // a bounded wait ran out: report; let copies and MMAs in flight land (bounded)
        if (tid == 0) {
            set_status(a.dev_status, MQA_DEV_TIMEOUT);
            // only what was issued: each barrier's last phase (an older parity would alias)
            for (int j = blk; j < n_issued; ++j)
                for (int w = 0; w < C::BOXES; ++w)
                    mbar_wait_bounded(mbar + (j % RING) * C::BOXES + w, (uint32_t)(j / RING) & 1u);
            if (n_qk > 0)
                mbar_wait_bounded(mbar_s, (uint32_t)(n_qk - 1) & 1u);
            if (n_pv > 0)
                mbar_wait_bounded(mbar_o, (uint32_t)(n_pv - 1) & 1u);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0)
            tmem_dealloc(tmem, C::TMEM_COLS);
        return;
    }
    if (!mbar_wait_bounded(mbar_o, (uint32_t)(n_blocks - 1) & 1u) && tid == 0)
        set_status(a.dev_status, MQA_DEV_TIMEOUT);
    tc_fence_after();

    // ---- epilogue: l per head over the block's 128 token rows, normalise O, store
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        float v = l_acc[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0)
            red[warp * 16 + j] = v;
    }
    __syncthreads();
    uint32_t ov[16];
    tmem_ld16(tmem + tl + O_COL + 16 * hh, ov);  // O^T row d = tok, heads 16hh..16hh+15
    tmem_wait_ld();
    const float ofac = exp2i(E_run - 6);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int h = h0 + 16 * hh + j;
        if (h >= a.num_q_heads)
            continue;
        const float l = red[(4 * hh) * 16 + j] + red[(4 * hh + 1) * 16 + j] + red[(4 * hh + 2) * 16 + j] +
                        red[(4 * hh + 3) * 16 + j];
        const float val = l > 0.f ? __uint_as_float(ov[j]) * (ofac / l) : 0.f;
        if (split_mode) {
            const size_t rowoff = ((size_t)b * a.num_splits + split) * a.num_q_heads + h;
            a.o_partial[rowoff * D + tok] = val;
            if (tok == 0)
                a.lse[rowoff] = l > 0.f ? (m_ref[j] * gh + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
            a.out[((size_t)b * a.num_q_heads + h) * D + tok] = __float2bfloat16_rn(val);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tmem, C::TMEM_COLS);

    // ---- fused split-KV merge: the last of this sequence's split CTAs merges them
    if (split_mode && a.counters != nullptr) {
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int n_active = (t_last - t_first + 1 + a.tiles_per_split - 1) / a.tiles_per_split;
            const int ticket = atomicAdd(a.counters + (size_t)b * gridDim.z + blockIdx.z, 1);
            *flag = (ticket == n_active - 1) ? 2 : 0;
        }
        __syncthreads();
        if (*flag == 2 && warp < 4) {
            __threadfence();
            const int n_active = (t_last - t_first + 1 + a.tiles_per_split - 1) / a.tiles_per_split;
            merge_splits<D, NH>(a, b, h0, n_active);
        }
    }
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
    dim3 grid(a.num_splits, a.batch, (a.num_q_heads + TcCfg::NH - 1) / TcCfg::NH);
    decode_tc_kernel<<<grid, TcCfg::THREADS, TcCfg::SMEM_BYTES, s>>>(a);
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
