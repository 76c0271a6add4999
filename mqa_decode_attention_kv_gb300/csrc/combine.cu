// split_kv_combine kernel: merge split-KV partial outputs with their
// log-sum-exps (flash-decoding).  One warp per (sequence, head): lanes own
// head_dim/32 consecutive elements of d; splits whose lse is -inf are skipped
// without reading their partial output.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace mqa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ o_partial,
                                                     const float *__restrict__ lse, int32_t batch,
                                                     int32_t num_splits, int32_t num_q_heads,
                                                     __nv_bfloat16 *__restrict__ out)
{
    constexpr int V = D / 32;  // elements per lane (4 or 2)
    const int lane = threadIdx.x & 31;
    const int pair = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (pair >= batch * num_q_heads)
        return;
    const int b = pair / num_q_heads, h = pair % num_q_heads;
    const size_t stride = (size_t)num_q_heads;  // between consecutive splits of one (b, h)
    const float *l = lse + (size_t)b * num_splits * num_q_heads + h;
    float M = -INFINITY;
    for (int s = lane; s < num_splits; s += 32)
        M = fmaxf(M, __ldg(l + s * stride));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        const float *o = o_partial + ((size_t)b * num_splits * num_q_heads + h) * D + lane * V;
        for (int s = 0; s < num_splits; ++s) {
            const float ls = __ldg(l + s * stride);
            if (ls == -INFINITY)
                continue;
            const float w = __expf(ls - M);
            den += w;
            const float *src = o + (size_t)s * stride * D;
            if constexpr (V == 4) {
                const float4 x = __ldg(reinterpret_cast<const float4 *>(src));
                acc[0] += w * x.x;
                acc[1] += w * x.y;
                acc[2] += w * x.z;
                acc[3] += w * x.w;
            } else {
                const float2 x = __ldg(reinterpret_cast<const float2 *>(src));
                acc[0] += w * x.x;
                acc[1] += w * x.y;
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16 *dst = out + ((size_t)b * num_q_heads + h) * D + lane * V;
    if constexpr (V == 4) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&p0);
        u.y = *reinterpret_cast<uint32_t *>(&p1);
        *reinterpret_cast<uint2 *>(dst) = u;
    } else {
        *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    }
}

}  // namespace

cudaError_t launch_combine(const float *o_partial, const float *lse, int32_t batch, int32_t num_splits,
                           int32_t num_q_heads, int32_t head_dim, __nv_bfloat16 *out, cudaStream_t s)
{
    const long long pairs = (long long)batch * num_q_heads;
    if (pairs == 0)
        return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((pairs * 32 + threads - 1) / threads);
    if (head_dim == 128)
        combine_kernel<128><<<blocks, threads, 0, s>>>(o_partial, lse, batch, num_splits, num_q_heads, out);
    else
        combine_kernel<64><<<blocks, threads, 0, s>>>(o_partial, lse, batch, num_splits, num_q_heads, out);
    return cudaGetLastError();
}

}  // namespace mqa
