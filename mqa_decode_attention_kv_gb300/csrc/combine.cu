// split_kv_combine kernel: merge split-KV partial outputs with their
// log-sum-exps (flash-decoding).
//
// One CTA of four warps per (sequence, head).  The CTA first finds
// M = max_s lse_s, then each warp accumulates w_s * o_s over the splits
// s = warp, warp+4, ... (up to sixteen independent loads in flight per lane),
// and the four partial sums are added in shared memory.  Splits whose lse is
// -inf are skipped without reading their partial output.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace mqa {
namespace {

constexpr int kCombineWarps = 4;

template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ o_partial,
                                                     const float *__restrict__ lse, int32_t num_splits,
                                                     int32_t num_q_heads, __nv_bfloat16 *__restrict__ out)
{
    constexpr int V = D / 32;  // fp32 elements per lane (4 or 2)
    griddep_wait();  // the partials of the decode kernel before it on the stream
    griddep_launch_dependents();
    __shared__ float red[kCombineWarps];
    __shared__ float part[kCombineWarps][D];
    __shared__ float dens[kCombineWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y, h = blockIdx.x;
    const size_t stride = (size_t)num_q_heads;  // between consecutive splits of one (b, h)
    const float *l = lse + (size_t)b * num_splits * num_q_heads + h;
    const float *o = o_partial + ((size_t)b * num_splits * num_q_heads + h) * D + lane * V;

    float M = -INFINITY;
    for (int s = threadIdx.x; s < num_splits; s += blockDim.x)
        M = fmaxf(M, __ldg(l + s * stride));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0)
        red[warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));

    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        // a warp's splits s = warp + 4u: up to U partial rows loaded in one batch
        constexpr int U = 16;
        for (int s0 = warp; s0 < num_splits; s0 += kCombineWarps * U) {
            float ls[U];
            float x[U][V];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int s = s0 + u * kCombineWarps;
                ls[u] = s < num_splits ? __ldg(l + s * stride) : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int s = s0 + u * kCombineWarps;
                if (ls[u] != -INFINITY) {
                    if constexpr (V == 4) {
                        const float4 t = __ldg(reinterpret_cast<const float4 *>(o + (size_t)s * stride * D));
                        x[u][0] = t.x;
                        x[u][1] = t.y;
                        x[u][2] = t.z;
                        x[u][3] = t.w;
                    } else {
                        const float2 t = __ldg(reinterpret_cast<const float2 *>(o + (size_t)s * stride * D));
                        x[u][0] = t.x;
                        x[u][1] = t.y;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < V; ++k)
                        x[u][k] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float w = ls[u] == -INFINITY ? 0.f : __expf(ls[u] - M);
                den += w;
#pragma unroll
                for (int k = 0; k < V; ++k)
                    acc[k] += w * x[u][k];
            }
        }
    }
#pragma unroll
    for (int k = 0; k < V; ++k)
        part[warp][lane * V + k] = acc[k];
    if (lane == 0)
        dens[warp] = den;
    __syncthreads();
    if (warp != 0)
        return;
    const float dsum = dens[0] + dens[1] + dens[2] + dens[3];
    const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
    float r[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        r[k] = (part[0][lane * V + k] + part[1][lane * V + k] + part[2][lane * V + k] + part[3][lane * V + k]) * inv;
    __nv_bfloat16 *dst = out + ((size_t)b * num_q_heads + h) * D + lane * V;
    if constexpr (V == 4) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(r[0], r[1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(r[2], r[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&p0);
        u.y = *reinterpret_cast<uint32_t *>(&p1);
        *reinterpret_cast<uint2 *>(dst) = u;
    } else {
        *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(r[0], r[1]);
    }
}

}  // namespace

cudaError_t launch_combine(const float *o_partial, const float *lse, int32_t batch, int32_t num_splits,
                           int32_t num_q_heads, int32_t head_dim, __nv_bfloat16 *out, cudaStream_t s)
{
    if (batch == 0)
        return cudaSuccess;
    dim3 grid((unsigned)num_q_heads, (unsigned)batch);
    if (head_dim == 128)
        return launch_pdl(combine_kernel<128>, grid, dim3(32 * kCombineWarps), 0, s, o_partial, lse, num_splits,
                          num_q_heads, out);
    return launch_pdl(combine_kernel<64>, grid, dim3(32 * kCombineWarps), 0, s, o_partial, lse, num_splits,
                      num_q_heads, out);
}

}  // namespace mqa
