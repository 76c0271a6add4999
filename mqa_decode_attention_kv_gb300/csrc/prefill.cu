// Chunked causal prefill attention over the int8 paged cache (prefix-shared
// blocks allowed), warp-level tensor-core version for head_dim 64 (head_dim
// 128 runs on the tcgen05 kernel of prefill_tc.cu).
//
// A CTA owns 64 query rows -- QT = 64/num_q_heads consecutive query tokens of
// one sequence times all heads (MQA: every row reads the same K/V) -- and walks
// the 64-token key tiles its rows need.  Per tile:
//   1. TMA brings the int8 K/V codes and fp32 scales into a STAGES-deep ring
//      (same boxes and swizzle as the decode kernel);
//   2. the CTA converts the codes once to fp16 (exact) into a swizzled fp16
//      tile shared by its four warps;
//   3. each warp (16 rows) computes S = Q K^T and O += P' V with mma.sync
//      (fp16 operands from ldmatrix, fp32 accumulators), applying the K scale to
//      the score columns and folding the V scale into P' exactly as in decode.
// Rows mask keys outside [max(0, i-W+1), i] (causal + window).
#include <atomic>
#include <math.h>

#include "common.cuh"
#include "kv_stage.cuh"
#include "launch.h"

namespace mqa {
namespace {

template <int D>
struct PrefillCfg {
    static constexpr int ROWS = 64;                 // query rows per CTA (4 warps x 16)
    static constexpr int KSTEPS = D / 16;
    static constexpr int DT = D / 8;                // n8 tiles of the output
    static constexpr int STAGES = 3;
    static constexpr int OFF_CODES = 0;
    static constexpr int OFF_HALF = STAGES * KvStage<D>::CODE_PAIR;          // fp16 K tile, then V tile
    static constexpr int HALF_BYTES = kTileTokens * D * 2;                    // one fp16 tile
    static constexpr int OFF_SCALES = OFF_HALF + 2 * HALF_BYTES;              // [STAGES][2][64] fp32
    static constexpr int OFF_MASK = OFF_SCALES + STAGES * 2 * kTileTokens * 4;
    static constexpr int OFF_FLAG = OFF_MASK + 4 * STAGES;
    static constexpr int OFF_MBAR = (OFF_FLAG + 4 + 7) / 8 * 8;
    static constexpr int SMEM_BYTES = OFF_MBAR + 8 * STAGES + 1024;
};

// byte offset of fp16 element (row, d) of a [64][D] tile: 64-column (128-byte)
// blocks, each [64 rows][128 B] with 16-byte chunks XOR-swizzled by row.
template <int D>
__device__ __forceinline__ uint32_t hoff(uint32_t row, uint32_t d)
{
    return (d >> 6) * (kTileTokens * 128) + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4) + (d & 7) * 2;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <int D>
__global__ void __launch_bounds__(128, 2) prefill_kernel(const __grid_constant__ PrefillArgs a)
{
    using C = PrefillCfg<D>;
    griddep_wait();  // the append of this chunk's K/V (and q) before it on the stream
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *khalf = base + C::OFF_HALF;
    uint8_t *vhalf = khalf + C::HALF_BYTES;
    uint32_t *stage_mask = reinterpret_cast<uint32_t *>(base + C::OFF_MASK);
    volatile int *flag = reinterpret_cast<int *>(base + C::OFF_FLAG);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(base + C::OFF_MBAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int b = blockIdx.y;
    const int H = a.num_q_heads;
    const int QT = C::ROWS / H > 0 ? C::ROWS / H : 1;      // query tokens per CTA
    const int HPB = H < C::ROWS ? H : C::ROWS;              // heads per CTA row block
    const int hgroups = H / HPB;                             // > 1 only when H > 64
    const int tblk = blockIdx.x / hgroups, hg = blockIdx.x % hgroups;

    const int L = __ldg(a.seq_lens + b);
    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    const int qlen = q1 - q0;
    const int t_begin = tblk * QT;
    if (L < 1 || L > a.max_seq_len || qlen > L || q0 < 0 || qlen < 0 || q1 > a.total_q) {
        if (threadIdx.x == 0)
            set_status(a.dev_status, (L < 1 || L > a.max_seq_len) ? MQA_DEV_BAD_SEQLEN : MQA_DEV_BAD_CU);
        return;
    }
    if (t_begin >= qlen)
        return;

    const int t_end = min(qlen, t_begin + QT);
    const int first_pos = L - qlen + t_begin, last_pos = L - qlen + t_end - 1;
    const int klo = a.window > 0 ? max(0, first_pos - a.window + 1) : 0;
    const int tb = klo / kTileTokens, te = last_pos / kTileTokens + 1;
    const int n_tiles = te - tb;
    const int Lkeys = last_pos + 1;  // keys beyond the last query are never fetched

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s)
            mbar_init(mbar + s, 1);
        *flag = 0;
        fence_mbar_init();
        for (int i = 0; i < n_tiles && i < C::STAGES; ++i)
            issue_kv_tile<D>(a.k_map, a.v_map, a.k_scale, a.v_scale, a.block_table + (size_t)b * a.max_blocks,
                             a.num_blocks, a.page_size, a.dev_status, base + C::OFF_CODES + i * KvStage<D>::CODE_PAIR,
                             reinterpret_cast<float *>(base + C::OFF_SCALES) + i * 2 * kTileTokens, mbar + i,
                             stage_mask + i, tb + i, klo, Lkeys, a.ring);
    }

    // ---- this thread's two rows (g and g+8 of the warp's 16)
    int pos[2], lo[2];
    bool rvalid[2];
    uint32_t qf[C::KSTEPS][4];
    float gexp[2];
    size_t orow[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int r = warp * 16 + g + 8 * hf;
        const int t = t_begin + r / HPB;
        const int h = hg * HPB + r % HPB;
        rvalid[hf] = (r / HPB) < QT && t < t_end;
        pos[hf] = L - qlen + t;
        lo[hf] = a.window > 0 ? max(0, pos[hf] - a.window + 1) : 0;
        orow[hf] = ((size_t)(q0 + t) * H + h) * D;
    }
    {
        // query fragments: natural k order, scaled by 2^e per row (exact in fp16)
        uint32_t w[2][D / 2];
        float amax[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float m = 0.f;
#pragma unroll
            for (int kt = 0; kt < C::KSTEPS; ++kt) {
                const int d0 = 16 * kt + 2 * c;
                uint32_t lo32 = 0, hi32 = 0;
                if (rvalid[hf]) {
                    lo32 = __ldg(reinterpret_cast<const uint32_t *>(a.q + orow[hf] + d0));
                    hi32 = __ldg(reinterpret_cast<const uint32_t *>(a.q + orow[hf] + d0 + 8));
                }
                w[hf][2 * kt] = lo32;
                w[hf][2 * kt + 1] = hi32;
                m = fmaxf(m, fmaxf(fmaxf(fabsf(__uint_as_float(lo32 << 16)), fabsf(__uint_as_float(lo32 & 0xffff0000u))),
                                   fmaxf(fabsf(__uint_as_float(hi32 << 16)), fabsf(__uint_as_float(hi32 & 0xffff0000u)))));
            }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            amax[hf] = m;
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const float sm = amax[hf];
            int e = 0;
            if (sm > 0.f && isfinite(sm)) {
                int x;
                frexpf(sm, &x);
                e = 14 - x;
                e = e < -120 ? -120 : (e > 120 ? 120 : e);
            }
            gexp[hf] = a.q_scale_log2 * exp2i(-e);  // q * 2^e is exact in fp16
            const float f = exp2i(e);
#pragma unroll
            for (int kt = 0; kt < C::KSTEPS; ++kt) {
                const uint32_t lo32 = w[hf][2 * kt], hi32 = w[hf][2 * kt + 1];
                qf[kt][hf] = pack_half2(__uint_as_float(lo32 << 16) * f, __uint_as_float(lo32 & 0xffff0000u) * f);
                qf[kt][2 + hf] = pack_half2(__uint_as_float(hi32 << 16) * f, __uint_as_float(hi32 & 0xffff0000u) * f);
            }
        }
    }

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[C::DT][4];
#pragma unroll
    for (int nt = 0; nt < C::DT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[nt][k] = 0.f;
    int E_run = -100;
    __syncthreads();

    const uint32_t khalf_u = smem_u32(khalf), vhalf_u = smem_u32(vhalf);
    int i = 0;
    for (; i < n_tiles; ++i) {
        const int stage = i % C::STAGES;
        if (!mbar_wait_bounded(mbar + stage, (uint32_t)(i / C::STAGES) & 1u))
            *flag = 1;
        const uint8_t *kst = base + C::OFF_CODES + stage * KvStage<D>::CODE_PAIR;
        const uint8_t *vst = kst + KvStage<D>::CODE_BYTES;
        const float *ks = reinterpret_cast<const float *>(base + C::OFF_SCALES) + stage * 2 * kTileTokens;
        const float *vs = ks + kTileTokens;
        const uint32_t mask = stage_mask[stage];
        const int T = tb + i;

        // ---- convert the tile's codes to fp16 (all boxes: stale codes are finite)
        constexpr int CH = D / 16;  // 16-byte code chunks per row
#pragma unroll
        for (int it = 0; it < (kTileTokens * CH) / 128; ++it) {
            const int qid = threadIdx.x + 128 * it;
            const int r = qid / CH, j = qid % CH;
            const uint4 kv = *reinterpret_cast<const uint4 *>(kst + swz<D>(r, 16 * j));
            const uint4 vv = *reinterpret_cast<const uint4 *>(vst + swz<D>(r, 16 * j));
            uint32_t kh[8], vh[8];
            i8x4_to_f16x2x2(kv.x, kh[0], kh[1]);
            i8x4_to_f16x2x2(kv.y, kh[2], kh[3]);
            i8x4_to_f16x2x2(kv.z, kh[4], kh[5]);
            i8x4_to_f16x2x2(kv.w, kh[6], kh[7]);
            i8x4_to_f16x2x2(vv.x, vh[0], vh[1]);
            i8x4_to_f16x2x2(vv.y, vh[2], vh[3]);
            i8x4_to_f16x2x2(vv.z, vh[4], vh[5]);
            i8x4_to_f16x2x2(vv.w, vh[6], vh[7]);
            *reinterpret_cast<uint4 *>(khalf + hoff<D>(r, 16 * j)) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
            *reinterpret_cast<uint4 *>(khalf + hoff<D>(r, 16 * j + 8)) = make_uint4(kh[4], kh[5], kh[6], kh[7]);
            *reinterpret_cast<uint4 *>(vhalf + hoff<D>(r, 16 * j)) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
            *reinterpret_cast<uint4 *>(vhalf + hoff<D>(r, 16 * j + 8)) = make_uint4(vh[4], vh[5], vh[6], vh[7]);
        }
        // scales of this thread's score columns: keys 8nt + 2c + {0,1}
        float ksv[8][2], vsv[8][2];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float2 kk = *reinterpret_cast<const float2 *>(ks + 8 * nt + 2 * c);
            const float2 vv = *reinterpret_cast<const float2 *>(vs + 8 * nt + 2 * c);
            ksv[nt][0] = kk.x;
            ksv[nt][1] = kk.y;
            vsv[nt][0] = vv.x;
            vsv[nt][1] = vv.y;
        }
        __syncthreads();  // fp16 tile ready; int8 stage consumed
        if (*flag)
            break;
        if (threadIdx.x == 0 && i + C::STAGES < n_tiles)
            issue_kv_tile<D>(a.k_map, a.v_map, a.k_scale, a.v_scale, a.block_table + (size_t)b * a.max_blocks,
                             a.num_blocks, a.page_size, a.dev_status,
                             base + C::OFF_CODES + stage * KvStage<D>::CODE_PAIR,
                             reinterpret_cast<float *>(base + C::OFF_SCALES) + stage * 2 * kTileTokens, mbar + stage,
                             stage_mask + stage, tb + i + C::STAGES, klo, Lkeys, a.ring);

        // ---- S = Q K^T (16 rows x 64 keys per warp)
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                s[nt][k] = 0.f;
#pragma unroll
        for (int kt = 0; kt < C::KSTEPS; ++kt)
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                // matrices: (keys 16np..+7, d lo), (same keys, d hi), (keys +8, d lo), (keys +8, d hi)
                const int key = 16 * np + 8 * (lane >> 4) + (lane & 7);
                const int d = 16 * kt + 8 * ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(khalf_u + hoff<D>(key, d), b0, b1, b2, b3);
                mma_f16_16816(s[2 * np], qf[kt], b0, b1);
                mma_f16_16816(s[2 * np + 1], qf[kt], b2, b3);
            }

        // ---- mask, scale, online softmax
        float svmax = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = T * kTileTokens + 8 * nt + 2 * c + e;
                const bool inbox = (mask >> (nt >> 1)) & 1u;
                if (inbox && key < Lkeys && key >= klo)
                    svmax = fmaxf(svmax, vsv[nt][e]);
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            svmax = fmaxf(svmax, __shfl_xor_sync(0xffffffffu, svmax, off));
        const int E_new = max(E_run, ceil_log2_pow(svmax));
        const float vfac = exp2i(14 - E_new);
        const int dE = E_run - E_new;
        const float escale = dE < -126 ? 0.f : exp2i(dE);
        E_run = E_new;
        uint32_t pa[4][4];  // A fragments of P' for the 4 key steps of 16
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float m = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = T * kTileTokens + 8 * nt + 2 * c + e;
                    const bool ok = rvalid[hf] && ((mask >> (nt >> 1)) & 1u) && key >= lo[hf] && key <= pos[hf];
                    const float y = ok ? s[nt][2 * hf + e] * ksv[nt][e] : -INFINITY;
                    s[nt][2 * hf + e] = y;
                    m = fmaxf(m, y);
                }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const float m_new = fmaxf(m_run[hf], m);
            const bool none = m_new == -INFINITY;
            const float alpha = none ? 1.f : fast_exp2((m_run[hf] - m_new) * gexp[hf]);
            const float negmg = none ? 0.f : -m_new * gexp[hf];
            m_run[hf] = m_new;
            float lsum = 0.f;
            float pp[8][2];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float y = s[nt][2 * hf + e];
                    const float p = fast_exp2(fmaf(y, gexp[hf], negmg));
                    lsum += p;
                    pp[nt][e] = y == -INFINITY ? 0.f : p * (vsv[nt][e] * vfac);
                }
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
            l_run[hf] = l_run[hf] * alpha + lsum;
            const float osc = alpha * escale;
#pragma unroll
            for (int nt = 0; nt < C::DT; ++nt) {
                o[nt][2 * hf] *= osc;
                o[nt][2 * hf + 1] *= osc;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                pa[kk][hf] = pack_half2(pp[2 * kk][0], pp[2 * kk][1]);          // keys 16kk + 2c (+1)
                pa[kk][2 + hf] = pack_half2(pp[2 * kk + 1][0], pp[2 * kk + 1][1]);  // keys 16kk + 8 + 2c (+1)
            }
        }

        // ---- O += P' V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int dp = 0; dp < C::DT / 2; ++dp) {
                // matrices: (keys lo, d 16dp..+7), (keys hi, same d), (keys lo, d +8), (keys hi, d +8)
                const int key = 16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7);
                const int d = 16 * dp + 8 * (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vhalf_u + hoff<D>(key, d), b0, b1, b2, b3);
                mma_f16_16816(o[2 * dp], pa[kk], b0, b1);
                mma_f16_16816(o[2 * dp + 1], pa[kk], b2, b3);
            }
        __syncthreads();  // all warps done with the fp16 tile
    }

    if (*flag) {
        if (threadIdx.x == 0) {
            set_status(a.dev_status, MQA_DEV_TIMEOUT);
            for (int j = i; j < n_tiles && j < i + C::STAGES; ++j)
                mbar_wait_drain(mbar + (j % C::STAGES), (uint32_t)(j / C::STAGES) & 1u);
        }
        return;
    }

    // ---- normalise and store bf16
    const float ofac = exp2i(E_run - 14);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        if (!rvalid[hf])
            continue;
        const float f = l_run[hf] > 0.f ? ofac / l_run[hf] : 0.f;
        __nv_bfloat16 *dst = a.out + orow[hf];
#pragma unroll
        for (int nt = 0; nt < C::DT; ++nt)
            *reinterpret_cast<__nv_bfloat162 *>(dst + 8 * nt + 2 * c) =
                __floats2bfloat162_rn(o[nt][2 * hf] * f, o[nt][2 * hf + 1] * f);
    }
}

template <int D>
cudaError_t launch_prefill_t(const PrefillArgs &a, cudaStream_t s)
{
    using C = PrefillCfg<D>;
    static std::atomic<int> attr_set{0};
    if (!attr_set.load(std::memory_order_acquire)) {
        cudaError_t e =
            cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_set.store(1, std::memory_order_release);
    }
    const int H = a.num_q_heads;
    const int QT = C::ROWS / H > 0 ? C::ROWS / H : 1;
    const int hgroups = H > C::ROWS ? H / C::ROWS : 1;
    dim3 grid((unsigned)(((a.max_q_len + QT - 1) / QT) * hgroups), (unsigned)a.batch, 1);
    return launch_pdl(prefill_kernel<D>, grid, dim3(128), C::SMEM_BYTES, s, a);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, int head_dim, cudaStream_t s)
{
    // head_dim 128 runs on the tcgen05 kernel (prefill_tc.cu); head_dim 64 here
    return head_dim == 128 ? launch_prefill_tc(a, s) : launch_prefill_t<64>(a, s);
}

}  // namespace mqa
