// Host-memory prefix cache: a page-granular prefix tree of cached KV pages in
// pinned host memory, indexed by a rolling hash of the prefix tokens, with LRU
// eviction of leaf pages and gather / scatter kernels that move whole pages
// between the pool and the device caches.  The behaviour (what is cached, what
// a match returns, which page is evicted) is specified in
// include/mqa_prefix_cache.h.
#include <cstdlib>
#include <cstring>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "mqa_kv.h"
#include "mqa_prefix_cache.h"

namespace {

constexpr uint64_t kHashMul = 0x100000001b3ull;

struct PcNode {
    int64_t parent;             // node id, -1 for a page at depth 0
    uint64_t key;               // rolling hash of the tokens up to the end of this page
    int64_t slot;               // host pool slot
    uint64_t stamp;             // last match / insert that touched this page
    int32_t children;           // cached successor pages
    std::vector<int32_t> tokens;  // the page's tokens (hits are confirmed on them)
};

// Copy jobs of one launch: page pairs passed by value (no device-side index arrays).
constexpr int kJobsPerLaunch = 256;
struct PcJobs {
    int8_t *k_codes[MQA_PC_MAX_CACHES];
    int8_t *v_codes[MQA_PC_MAX_CACHES];
    float *k_scale[MQA_PC_MAX_CACHES];
    float *v_scale[MQA_PC_MAX_CACHES];
    uint8_t *pool;         // device address of the pinned pool
    int64_t slot_bytes;
    int32_t page_size, head_dim, n;
    int32_t to_pool;       // 1: device -> pool, 0: pool -> device
    int32_t block[kJobsPerLaunch];
    int64_t slot[kJobsPerLaunch];
};

// One CTA per (page, cache): the page's K codes, V codes, K scales, V scales.
__global__ void __launch_bounds__(256) pc_copy_kernel(const __grid_constant__ PcJobs j)
{
    const int i = blockIdx.x, c = blockIdx.y;
    const int P = j.page_size, D = j.head_dim;
    const int64_t code_bytes = (int64_t)P * D;
    uint8_t *slot = j.pool + j.slot[i] * j.slot_bytes + (int64_t)c * (2 * code_bytes + 8 * P);
    uint8_t *parts_pool[4] = {slot, slot + code_bytes, slot + 2 * code_bytes, slot + 2 * code_bytes + 4 * P};
    const int64_t row = (int64_t)j.block[i] * P;
    uint8_t *parts_dev[4] = {reinterpret_cast<uint8_t *>(j.k_codes[c] + row * D),
                             reinterpret_cast<uint8_t *>(j.v_codes[c] + row * D),
                             reinterpret_cast<uint8_t *>(j.k_scale[c] + row),
                             reinterpret_cast<uint8_t *>(j.v_scale[c] + row)};
    const int64_t bytes[4] = {code_bytes, code_bytes, 4 * P, 4 * P};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint4 *src = reinterpret_cast<const uint4 *>(j.to_pool ? parts_dev[p] : parts_pool[p]);
        uint4 *dst = reinterpret_cast<uint4 *>(j.to_pool ? parts_pool[p] : parts_dev[p]);
        for (int64_t k = threadIdx.x; k < bytes[p] / 16; k += blockDim.x)
            dst[k] = src[k];
    }
}

}  // namespace

struct mqa_prefix_cache {
    int32_t page_size, head_dim, num_caches, pinned;
    int64_t capacity, slot_bytes;
    uint8_t *pool = nullptr;      // host address
    uint8_t *pool_dev = nullptr;  // device address of the same memory (pinned pools)
    std::vector<PcNode> nodes;    // node id -> node (free ids are reused)
    std::vector<int64_t> free_ids;
    std::vector<int64_t> free_slots;
    std::unordered_multimap<uint64_t, int64_t> index;  // rolling prefix hash -> node id
    std::set<std::pair<uint64_t, int64_t>> leaves;     // (stamp, node id) of pages without successors
    uint64_t clock = 0;
    int64_t n_match_calls = 0, n_matched = 0, n_inserted = 0, n_evicted = 0;

    // the cached page following node `parent` (-1: the root) whose prefix hash is key and
    // whose tokens are tok[0, page_size), or -1
    int64_t find(int64_t parent, uint64_t key, const int32_t *tok) const
    {
        auto range = index.equal_range(key);
        for (auto it = range.first; it != range.second; ++it) {
            const PcNode &nd = nodes[it->second];
            if (nd.parent == parent && std::memcmp(nd.tokens.data(), tok, sizeof(int32_t) * page_size) == 0)
                return it->second;
        }
        return -1;
    }

    void touch(int64_t id, uint64_t t)
    {
        PcNode &nd = nodes[id];
        if (nd.children == 0) {
            leaves.erase({nd.stamp, id});
            leaves.insert({t, id});
        }
        nd.stamp = t;
    }

    // evict the least recently used leaf older than `now`; false when there is none
    bool evict_one(uint64_t now)
    {
        if (leaves.empty() || leaves.begin()->first >= now)
            return false;
        const int64_t id = leaves.begin()->second;
        leaves.erase(leaves.begin());
        PcNode &nd = nodes[id];
        auto range = index.equal_range(nd.key);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second == id) {
                index.erase(it);
                break;
            }
        free_slots.push_back(nd.slot);
        if (nd.parent >= 0) {
            PcNode &pa = nodes[nd.parent];
            if (--pa.children == 0)
                leaves.insert({pa.stamp, nd.parent});
        }
        nd.tokens.clear();
        nd.tokens.shrink_to_fit();
        free_ids.push_back(id);
        ++n_evicted;
        return true;
    }
};

namespace {

bool shape_ok(int32_t page_size, int32_t head_dim)
{
    return (page_size == 16 || page_size == 64) && (head_dim == 64 || head_dim == 128);
}

int copy_pages(mqa_prefix_cache *pc, const mqa_kv_cache *caches, int32_t num_caches, const int32_t *blocks,
               const int64_t *slots, int64_t n, int to_pool, void *stream)
{
    if (pc == nullptr || n < 0 || (n > 0 && (caches == nullptr || blocks == nullptr || slots == nullptr)))
        return MQA_ERR_INVALID_ARG;
    if (!pc->pinned)
        return MQA_ERR_UNSUPPORTED;
    if (num_caches != pc->num_caches)
        return MQA_ERR_INVALID_ARG;
    if (n == 0)
        return MQA_OK;
    PcJobs j;
    std::memset(&j, 0, sizeof j);
    for (int c = 0; c < num_caches; ++c) {
        const mqa_kv_cache &cc = caches[c];
        if (cc.page_size != pc->page_size || cc.head_dim != pc->head_dim || cc.k_codes == nullptr ||
            cc.v_codes == nullptr || cc.k_scale == nullptr || cc.v_scale == nullptr || cc.num_blocks < 1)
            return MQA_ERR_INVALID_ARG;
        if (((reinterpret_cast<uintptr_t>(cc.k_codes) | reinterpret_cast<uintptr_t>(cc.v_codes) |
              reinterpret_cast<uintptr_t>(cc.k_scale) | reinterpret_cast<uintptr_t>(cc.v_scale)) & 15u) != 0)
            return MQA_ERR_INVALID_ARG;
        j.k_codes[c] = cc.k_codes;
        j.v_codes[c] = cc.v_codes;
        j.k_scale[c] = cc.k_scale;
        j.v_scale[c] = cc.v_scale;
    }
    for (int64_t i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= pc->capacity)
            return MQA_ERR_INVALID_ARG;
        for (int c = 0; c < num_caches; ++c)
            if (blocks[i] < 0 || blocks[i] >= caches[c].num_blocks)
                return MQA_ERR_INVALID_ARG;
    }
    j.pool = pc->pool_dev;
    j.slot_bytes = pc->slot_bytes;
    j.page_size = pc->page_size;
    j.head_dim = pc->head_dim;
    j.to_pool = to_pool;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int64_t i0 = 0; i0 < n; i0 += kJobsPerLaunch) {
        const int m = (int)(n - i0 < kJobsPerLaunch ? n - i0 : kJobsPerLaunch);
        j.n = m;
        for (int i = 0; i < m; ++i) {
            j.block[i] = blocks[i0 + i];
            j.slot[i] = slots[i0 + i];
        }
        pc_copy_kernel<<<dim3((unsigned)m, (unsigned)num_caches), 256, 0, s>>>(j);
        if (cudaGetLastError() != cudaSuccess)
            return MQA_ERR_CUDA;
    }
    return MQA_OK;
}

}  // namespace

extern "C" {

int mqa_pc_create(int32_t page_size, int32_t head_dim, int32_t num_caches, int64_t host_pages, int32_t pinned,
                  mqa_prefix_cache **out)
{
    if (out == nullptr)
        return MQA_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_caches < 1 || num_caches > MQA_PC_MAX_CACHES || host_pages < 1)
        return MQA_ERR_INVALID_ARG;
    if (!shape_ok(page_size, head_dim))
        return MQA_ERR_UNSUPPORTED;
    mqa_prefix_cache *pc = new (std::nothrow) mqa_prefix_cache();
    if (pc == nullptr)
        return MQA_ERR_INVALID_ARG;
    pc->page_size = page_size;
    pc->head_dim = head_dim;
    pc->num_caches = num_caches;
    pc->pinned = pinned != 0;
    pc->capacity = host_pages;
    pc->slot_bytes = (int64_t)num_caches * page_size * (2 * head_dim + 8);
    const size_t bytes = (size_t)pc->slot_bytes * (size_t)host_pages;
    if (pc->pinned) {
        void *p = nullptr;
        if (cudaHostAlloc(&p, bytes, cudaHostAllocMapped) != cudaSuccess) {
            delete pc;
            return MQA_ERR_CUDA;
        }
        void *d = nullptr;
        if (cudaHostGetDevicePointer(&d, p, 0) != cudaSuccess) {
            cudaFreeHost(p);
            delete pc;
            return MQA_ERR_CUDA;
        }
        pc->pool = static_cast<uint8_t *>(p);
        pc->pool_dev = static_cast<uint8_t *>(d);
    } else {
        pc->pool = static_cast<uint8_t *>(std::malloc(bytes));
        if (pc->pool == nullptr) {
            delete pc;
            return MQA_ERR_INVALID_ARG;
        }
    }
    pc->free_slots.reserve((size_t)host_pages);
    for (int64_t s = host_pages - 1; s >= 0; --s)
        pc->free_slots.push_back(s);  // slot 0 first
    *out = pc;
    return MQA_OK;
}

void mqa_pc_destroy(mqa_prefix_cache *pc)
{
    if (pc == nullptr)
        return;
    if (pc->pinned)
        cudaFreeHost(pc->pool);
    else
        std::free(pc->pool);
    delete pc;
}

int64_t mqa_pc_match(mqa_prefix_cache *pc, const int32_t *tokens, int64_t n_tokens, int64_t *slots,
                     int64_t max_pages)
{
    if (pc == nullptr || n_tokens < 0 || max_pages < 0 || (n_tokens > 0 && tokens == nullptr) ||
        (max_pages > 0 && slots == nullptr))
        return MQA_ERR_INVALID_ARG;
    ++pc->n_match_calls;
    const int P = pc->page_size;
    const int64_t pages = n_tokens / P;
    std::vector<int64_t> path;
    uint64_t h = 0;
    int64_t parent = -1;
    for (int64_t k = 0; k < pages; ++k) {
        const int32_t *tok = tokens + k * P;
        for (int t = 0; t < P; ++t)
            h = h * kHashMul + (uint64_t)(uint32_t)tok[t] + 1u;
        const int64_t id = pc->find(parent, h, tok);
        if (id < 0)
            break;
        path.push_back(id);
        parent = id;
    }
    const uint64_t now = ++pc->clock;
    for (size_t k = 0; k < path.size(); ++k) {
        pc->touch(path[k], now);
        if ((int64_t)k < max_pages)
            slots[k] = pc->nodes[path[k]].slot;
    }
    pc->n_matched += (int64_t)path.size();
    return (int64_t)path.size();
}

int64_t mqa_pc_insert(mqa_prefix_cache *pc, const int32_t *tokens, int64_t n_tokens, int64_t *page_index,
                      int64_t *slots, int64_t max_new)
{
    if (pc == nullptr || n_tokens < 0 || max_new < 0 || (n_tokens > 0 && tokens == nullptr) ||
        (max_new > 0 && (page_index == nullptr || slots == nullptr)))
        return MQA_ERR_INVALID_ARG;
    const int P = pc->page_size;
    const int64_t pages = n_tokens / P;
    const uint64_t now = ++pc->clock;
    uint64_t h = 0;
    int64_t parent = -1, added = 0;
    for (int64_t k = 0; k < pages; ++k) {
        const int32_t *tok = tokens + k * P;
        for (int t = 0; t < P; ++t)
            h = h * kHashMul + (uint64_t)(uint32_t)tok[t] + 1u;
        int64_t id = pc->find(parent, h, tok);
        if (id >= 0) {
            pc->touch(id, now);
            parent = id;
            continue;
        }
        if (added >= max_new)
            break;
        if (pc->free_slots.empty() && !pc->evict_one(now))
            break;  // every cached page lies on this path
        const int64_t slot = pc->free_slots.back();
        pc->free_slots.pop_back();
        if (!pc->free_ids.empty()) {
            id = pc->free_ids.back();
            pc->free_ids.pop_back();
        } else {
            id = (int64_t)pc->nodes.size();
            pc->nodes.emplace_back();
        }
        PcNode &nd = pc->nodes[id];
        nd.parent = parent;
        nd.key = h;
        nd.slot = slot;
        nd.stamp = now;
        nd.children = 0;
        nd.tokens.assign(tok, tok + P);
        pc->index.insert({h, id});
        pc->leaves.insert({now, id});
        if (parent >= 0) {
            PcNode &pa = pc->nodes[parent];
            if (pa.children++ == 0)
                pc->leaves.erase({pa.stamp, parent});
        }
        page_index[added] = k;
        slots[added] = slot;
        ++added;
        parent = id;
    }
    pc->n_inserted += added;
    return added;
}

int mqa_pc_offload(mqa_prefix_cache *pc, const mqa_kv_cache *caches, int32_t num_caches, const int32_t *src_blocks,
                   const int64_t *slots, int64_t n, void *stream)
{
    return copy_pages(pc, caches, num_caches, src_blocks, slots, n, 1, stream);
}

int mqa_pc_upload(mqa_prefix_cache *pc, const mqa_kv_cache *caches, int32_t num_caches, const int64_t *slots,
                  const int32_t *dst_blocks, int64_t n, void *stream)
{
    return copy_pages(pc, caches, num_caches, dst_blocks, slots, n, 0, stream);
}

int mqa_pc_stats(const mqa_prefix_cache *pc, int64_t *out)
{
    if (pc == nullptr || out == nullptr)
        return MQA_ERR_INVALID_ARG;
    out[0] = (int64_t)pc->index.size();
    out[1] = (int64_t)pc->free_slots.size();
    out[2] = pc->capacity;
    out[3] = pc->n_match_calls;
    out[4] = pc->n_matched;
    out[5] = pc->n_inserted;
    out[6] = pc->n_evicted;
    out[7] = pc->slot_bytes;
    return MQA_OK;
}

}  // extern "C"
