// mqa_decode_attn_noalloc: decode attention for callers that cannot allocate
// device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// while a CUDA graph is being captured by a framework that forbids new device
// allocations, serving loops that reserve their whole memory budget up front
// and must not touch the allocator again, plugins and foreign-language runtimes
// that have no handle on the process's CUDA allocator, and real-time paths
// where cudaMalloc's implicit device synchronisation is not acceptable.  This
// entry point gives them split-KV decode without a workspace argument: the
// split partials live in one file-scope device array of fixed size that every
// GPU loading this library holds until the process exits.
#include <atomic>
#include <cstdint>

#include "mqa_kv.h"
#include <cuda_runtime.h>

namespace {

// Largest workspace this entry point can use (32 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

// The shared scratch array.  In host code `g_noalloc_scratch` names a host-side
// stand-in, not device memory: only the address from cudaGetSymbolAddress may
// be handed to a kernel.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this set-up).
int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return MQA_ERR_CUDA;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MQA_ERR_CUDA;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return MQA_OK;
}

}  // namespace

extern "C" int mqa_decode_attn_noalloc(const mqa_kv_cache *caches, int32_t num_caches, const int32_t *layer_to_kv,
                                       int32_t num_layers, int32_t layer, int32_t window, const mqa_batch *batch,
                                       const void *q, void *out, int32_t num_q_heads, float sm_scale,
                                       int32_t num_splits, int32_t *dev_status, void *stream)
{
    if (caches == nullptr || layer_to_kv == nullptr || batch == nullptr || num_layers < 1 || layer < 0 ||
        layer >= num_layers || num_splits < 0 || num_splits > MQA_MAX_SPLITS)
        return MQA_ERR_INVALID_ARG;
    const int32_t k = layer_to_kv[layer];
    if (k < 0 || k >= num_caches)
        return MQA_ERR_INVALID_ARG;
    const int32_t head_dim = caches[k].head_dim;
    int32_t splits = num_splits;
    if (splits == 0) {
        // the automatic plan, narrowed until its workspace fits the scratch array
        // (one split needs no workspace at all)
        const int s = mqa_decode_auto_splits(batch, window, num_q_heads, head_dim, caches[k].page_size);
        if (s < 0)
            return s;
        splits = s;
        while (splits > 1 &&
               mqa_decode_workspace_size(batch->batch, num_q_heads, head_dim, splits) > kNoAllocScratchBytes)
            --splits;
    } else if (mqa_decode_workspace_size(batch->batch, num_q_heads, head_dim, splits) > kNoAllocScratchBytes) {
        return MQA_ERR_WORKSPACE;  // the requested split count needs more than the 32 MiB scratch array
    }
    void *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != MQA_OK)
        return rc;
    return mqa_decode_attn(caches, num_caches, layer_to_kv, num_layers, layer, window, batch, q, out, num_q_heads,
                           sm_scale, splits, scratch, kNoAllocScratchBytes, dev_status, stream);
}
