// Fused split-KV merge shared by the decode kernels: the last split CTA of a
// (sequence, head group) merges every split's partial output from L2.
#pragma once

#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace mqa {

// Merge the partial results of one sequence's n (<= kMaxFusedSplits) splits for
// the heads [h0, h0+HT): warp w takes heads h0+w, h0+w+4, ...  All the warp's
// lse values are loaded in one batch (lane s holds split s), then the partial
// rows of two heads at a time, every split's row in flight together.
template <int D, int HT>
__device__ __forceinline__ void merge_splits(const DecodeArgs &a, int b, int h0, int n)
{
    constexpr int V = D / 32;
    constexpr int R = HT / 4;  // heads per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float w[R], inv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int h = h0 + warp + 4 * r;
        const size_t base = (size_t)b * a.num_splits * a.num_q_heads + h;
        w[r] = (h < a.num_q_heads && lane < n) ? __ldcg(a.lse + base + (size_t)lane * a.num_q_heads) : -INFINITY;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float M = w[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        w[r] = (w[r] == -INFINITY || M == -INFINITY) ? 0.f : __expf(w[r] - M);
        float den = w[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            den += __shfl_xor_sync(0xffffffffu, den, off);
        inv[r] = den > 0.f ? 1.f / den : 0.f;
    }
#pragma unroll
    for (int r0 = 0; r0 < R; r0 += 2) {
        float x[2][kMaxFusedSplits][V];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int h = h0 + warp + 4 * (r0 + u);
            const size_t base = (size_t)b * a.num_splits * a.num_q_heads + h;
#pragma unroll
            for (int s = 0; s < kMaxFusedSplits; ++s) {
                const bool ok = h < a.num_q_heads && s < n;
                const float *src = a.o_partial + (base + (size_t)s * a.num_q_heads) * D + lane * V;
                if constexpr (V == 4) {
                    const float4 t = ok ? __ldcg(reinterpret_cast<const float4 *>(src)) : make_float4(0, 0, 0, 0);
                    x[u][s][0] = t.x;
                    x[u][s][1] = t.y;
                    x[u][s][2] = t.z;
                    x[u][s][3] = t.w;
                } else {
                    const float2 t = ok ? __ldcg(reinterpret_cast<const float2 *>(src)) : make_float2(0, 0);
                    x[u][s][0] = t.x;
                    x[u][s][1] = t.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int h = h0 + warp + 4 * (r0 + u);
            float acc[V];
#pragma unroll
            for (int k = 0; k < V; ++k)
                acc[k] = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxFusedSplits; ++s) {
                const float ws = __shfl_sync(0xffffffffu, w[r0 + u], s);
#pragma unroll
                for (int k = 0; k < V; ++k)
                    acc[k] += ws * x[u][s][k];
            }
            if (h >= a.num_q_heads)
                continue;
            __nv_bfloat16 *dst = a.out + ((size_t)b * a.num_q_heads + h) * D + lane * V;
            const float f = inv[r0 + u];
            if constexpr (V == 4) {
                __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0] * f, acc[1] * f);
                __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2] * f, acc[3] * f);
                uint2 q;
                q.x = *reinterpret_cast<uint32_t *>(&p0);
                q.y = *reinterpret_cast<uint32_t *>(&p1);
                *reinterpret_cast<uint2 *>(dst) = q;
            } else {
                *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(acc[0] * f, acc[1] * f);
            }
        }
    }
}

}  // namespace mqa
