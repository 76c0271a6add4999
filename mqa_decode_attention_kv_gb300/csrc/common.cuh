// Device helpers shared by the kernels of libmqa_kv (sm_103a only).
//
// Inline PTX wrappers for mbarriers, programmatic dependent launch, L2 prefetch
// and TMA (cp.async.bulk / cp.async.bulk.tensor); the exact int8 -> fp16
// conversion; power-of-two and exponential helpers.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mqa_kv.h"

namespace mqa {

// ---------------------------------------------------------------- constants
constexpr int kTileTokens = 64;   // tokens per pipeline stage
constexpr int kChunkTokens = 16;  // rows per TMA box (a box never crosses a page: P in {16, 64})
constexpr int kChunksPerTile = kTileTokens / kChunkTokens;
// Bounded waits.  A pipeline wait (one role waiting for another) gives up after
// kWaitLimitNs and reports MQA_DEV_TIMEOUT; a drain (a CTA that gave up waiting
// for its own copies and MMAs in flight before it leaves) uses kDrainLimitNs.
// MQA_TEST_WAIT_LIMIT_NS builds a test-only library whose pipeline waits give
// up almost at once, to exercise the abort path; drains keep their limit.
#ifdef MQA_TEST_WAIT_LIMIT_NS
constexpr unsigned long long kWaitLimitNs = MQA_TEST_WAIT_LIMIT_NS;
constexpr uint32_t kTryWaitSuspendNs = 0;
#else
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kTryWaitSuspendNs = 1000000;  // let a waiting thread sleep instead of spinning
#endif
constexpr unsigned long long kDrainLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kDrainSuspendNs = 1000000;

// ---------------------------------------------------------------- addressing
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(int32_t *dev_status, int32_t bits)
{
    if (dev_status != nullptr)
        atomicOr(dev_status, bits);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kTryWaitSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Whether phase `parity` of `bar` has completed (does not wait).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` with the drain limit: a CTA that is leaving early
// waits this long for its own asynchronous copies and MMAs before it gives up.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait_hint(bar, parity, kDrainSuspendNs))
        return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_hint(bar, parity, kDrainSuspendNs))
                return true;
        if (global_timer_ns() - t0 > kDrainLimitNs)
            return false;
    }
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialisation: a kernel may
// start while its predecessor on the stream is still running.  griddep_wait()
// blocks until the predecessor grid has completed and its memory is visible;
// every kernel calls it before its first access to global memory.
// griddep_launch_dependents() lets the successor start its own set-up early.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Hint: bring the line holding p into L2 (no data returns to the thread).  L2 is
// the point of coherence, so this may run before griddep_wait(): a line the
// predecessor writes afterwards is updated there, never served stale.
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- TMA
// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Linear bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- int8 -> fp16
// Exponent-bias ("magic number") conversion, as described for int8 weights in
// Kim et al., "Who Says Elephants Can't Run: Bringing Large Scale MoE Models
// into Cloud Scale Production" (2022): placing the biased byte u = x + 128 in
// the low mantissa bits of the fp16 pattern 0x6400 (= 1024) gives exactly
// 1024 + u; subtracting 1152 leaves x.  Every int8 is exact in fp16.
__device__ __forceinline__ uint32_t hsub2_1152(uint32_t v)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x64806480u));
    return r;
}

// Four codes packed in w (byte i = code i) -> lo = {c0, c1}, hi = {c2, c3} as f16x2.
__device__ __forceinline__ void i8x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t t = w ^ 0x80808080u;
    lo = hsub2_1152(__byte_perm(t, 0x64646464u, 0x5140));
    hi = hsub2_1152(__byte_perm(t, 0x64646464u, 0x7362));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 2^e for an integer e in [-126, 127], built from the exponent field (exact).
__device__ __forceinline__ float exp2i(int e)
{
    return __int_as_float((e + 127) << 23);
}

// Smallest integer E with x <= 2^E for finite x > 0 (clamped to [-100, 127]);
// -100 for x <= 0 or subnormal x.
__device__ __forceinline__ int ceil_log2_pow(float x)
{
    const uint32_t u = __float_as_uint(x);
    const int e = int((u >> 23) & 0xff);
    if (x <= 0.f || e == 0)
        return -100;
    const bool pow2 = (u & 0x7fffff) == 0;
    int r = e - 127 + (pow2 ? 0 : 1);
    return r < -100 ? -100 : (r > 127 ? 127 : r);
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace mqa
