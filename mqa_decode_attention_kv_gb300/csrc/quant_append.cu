// kv_quant_append kernel: per-token symmetric int8 quantisation of new K/V
// rows and their scatter into paged cache slots.
//
// One group of head_dim/8 lanes handles one vector (K or V of one token): each
// lane loads 16 bytes (8 bf16), the group reduces max|x| with shuffles, and
// each lane writes 8 codes (8 bytes) with kv_quant8 (IEEE fp32 division and
// round-half-even conversion; the decode kernel's fused append uses the same
// functions, so both write the same bits).
#include "common.cuh"
#include "kv_stage.cuh"
#include "launch.h"

namespace mqa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) quant_append_kernel(AppendArgs a)
{
    constexpr int kLanesPerVec = D / 8;               // 16 (d=128) or 8 (d=64)
    constexpr int kVecsPerWarp = 32 / kLanesPerVec;   // 2 or 4
    constexpr int kTokensPerWarp = kVecsPerWarp / 2;  // K and V of a token
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int vec = lane / kLanesPerVec;              // which vector of the warp
    const int sub = lane % kLanesPerVec;              // 16-byte slice of the vector
    const int token = warp * kTokensPerWarp + (vec >> 1);
    const bool is_v = (vec & 1) != 0;
    const bool active = token < a.num_tokens;
    // while the previous kernel may still run: warm L2 with what this token's lanes read next
    // (hints only: every load below comes after griddep_wait and sees what that kernel writes).
    // The guessed sequence b = token is the one-token-per-sequence append of a decode step.
    if (active && sub == 0) {
        const int g = min(token, a.batch - 1);
        prefetch_l2(a.cu_new + token);
        prefetch_l2(a.seq_lens + g);
        prefetch_l2((is_v ? a.v_new : a.k_new) + (size_t)token * D);
        const char *row = reinterpret_cast<const char *>(a.block_table + (size_t)g * a.max_blocks);
        for (int off = 0; off < a.max_blocks * 4 && off < 16 * 128; off += 128)
            prefetch_l2(row + off);
    }
    griddep_wait();  // the previous kernel on the stream (which may read the slots written here) is done
    griddep_launch_dependents();
    if (warp * kTokensPerWarp >= a.num_tokens)
        return;

    // sequence of this token: the b with cu_new[b] <= token < cu_new[b+1]; one new token per
    // sequence (b = token) is tested first with two independent loads
    int b = 0;
    if (active) {
        const int g = min(token, a.batch - 1);
        if (__ldg(a.cu_new + g) <= token && token < __ldg(a.cu_new + g + 1)) {
            b = g;
        } else {
            int lo = 0, hi = a.batch - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(a.cu_new + mid) <= token)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            b = lo;
        }
    }

    // load 8 bf16 values
    uint4 raw = make_uint4(0, 0, 0, 0);
    const __nv_bfloat16 *src = is_v ? a.v_new : a.k_new;
    if (active)
        raw = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)token * D) + sub);
    float x[8];
    bf16x8_to_f32(raw, x);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int off = kLanesPerVec / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (!active)
        return;

    // destination slot
    const int32_t c0 = __ldg(a.cu_new + b), c1 = __ldg(a.cu_new + b + 1);
    const int32_t L = __ldg(a.seq_lens + b);
    const int32_t pos = L - (c1 - c0) + (token - c0);
    // a window-bounded cache holds ring pages: more new tokens than that would overwrite one another
    if (pos < 0 || pos >= L || c1 < c0 || (a.ring > 0 && c1 - c0 > a.ring * a.page_size)) {
        if (sub == 0)
            set_status(a.dev_status, MQA_DEV_BAD_CU);
        return;
    }
    const int32_t lb = table_entry(pos / a.page_size, a.ring);
    if (lb >= a.max_blocks) {
        if (sub == 0)
            set_status(a.dev_status, MQA_DEV_BAD_SEQLEN);
        return;
    }
    const int32_t blk = __ldg(a.block_table + (size_t)b * a.max_blocks + lb);
    if (blk < 0 || blk >= a.num_blocks) {
        if (sub == 0)
            set_status(a.dev_status, MQA_DEV_BAD_BLOCK);
        return;
    }
    const size_t slot = (size_t)blk * a.page_size + (pos % a.page_size);

    const float s = kv_quant_scale(amax);
    int8_t *codes = is_v ? a.v_codes : a.k_codes;
    reinterpret_cast<uint2 *>(codes + slot * D)[sub] = kv_quant8(x, s);
    if (sub == 0)
        (is_v ? a.v_scale : a.k_scale)[slot] = s;
}

}  // namespace

cudaError_t launch_quant_append(const AppendArgs &a, cudaStream_t s)
{
    if (a.num_tokens <= 0)
        return cudaSuccess;
    const int threads = 256;
    const int tokens_per_warp = (a.head_dim == 128) ? 1 : 2;
    const long long warps = ((long long)a.num_tokens + tokens_per_warp - 1) / tokens_per_warp;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    if (a.head_dim == 128)
        return launch_pdl(quant_append_kernel<128>, dim3((unsigned)blocks), dim3(threads), 0, s, a);
    return launch_pdl(quant_append_kernel<64>, dim3((unsigned)blocks), dim3(threads), 0, s, a);
}

}  // namespace mqa
