// C ABI of libmqa_kv: argument validation, split planning, tensor-map set-up
// and kernel launches.  Every call validates on the host before touching the
// GPU, so bad arguments return a negative status and launch nothing.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "launch.h"

using namespace mqa;

namespace {

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool head_dim_ok(int d) { return d == 64 || d == 128; }
bool heads_ok(int h) { return h == 8 || h == 16 || h == 32 || h == 64; }
bool page_ok(int p) { return p == 16 || p == 64; }

int check_cache(const mqa_kv_cache *c)
{
    if (c == nullptr || c->k_codes == nullptr || c->v_codes == nullptr || c->k_scale == nullptr ||
        c->v_scale == nullptr)
        return MQA_ERR_INVALID_ARG;
    if (!head_dim_ok(c->head_dim) || !page_ok(c->page_size))
        return MQA_ERR_UNSUPPORTED;
    if (c->num_blocks < 1 || (int64_t)c->num_blocks * c->page_size > INT32_MAX)
        return MQA_ERR_INVALID_ARG;
    if (!aligned16(c->k_codes) || !aligned16(c->v_codes) || !aligned16(c->k_scale) || !aligned16(c->v_scale))
        return MQA_ERR_INVALID_ARG;
    return MQA_OK;
}

int check_batch(const mqa_batch *bt, int page_size)
{
    if (bt == nullptr || bt->batch < 0 || bt->batch > 65535)  // one grid row per sequence
        return MQA_ERR_INVALID_ARG;
    if (bt->batch == 0)
        return MQA_OK;
    if (bt->block_table == nullptr || bt->seq_lens == nullptr || bt->max_blocks < 1 || bt->max_seq_len < 1)
        return MQA_ERR_INVALID_ARG;
    if (bt->ring_blocks < 0 || bt->ring_blocks > bt->max_blocks)
        return MQA_ERR_INVALID_ARG;
    // a full table maps every page; a ring keeps only the most recent ones
    if (bt->ring_blocks == 0 && (int64_t)bt->max_seq_len > (int64_t)bt->max_blocks * page_size)
        return MQA_ERR_INVALID_ARG;
    if (bt->seq_lens_host != nullptr)
        for (int b = 0; b < bt->batch; ++b)
            if (bt->seq_lens_host[b] < 1 || bt->seq_lens_host[b] > bt->max_seq_len)
                return MQA_ERR_INVALID_ARG;
    return MQA_OK;
}

// The cache a layer reads, after validating the layer -> cache map.
int pick_cache(const mqa_kv_cache *caches, int32_t num_caches, const int32_t *layer_to_kv, int32_t num_layers,
               int32_t layer, const mqa_kv_cache **out)
{
    if (caches == nullptr || layer_to_kv == nullptr || num_caches < 1 || num_layers < 1 || layer < 0 ||
        layer >= num_layers)
        return MQA_ERR_INVALID_ARG;
    const int32_t k = layer_to_kv[layer];
    if (k < 0 || k >= num_caches)
        return MQA_ERR_INVALID_ARG;
    *out = caches + k;
    return check_cache(*out);
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// 2-D map over int8 codes viewed as [num_blocks*page_size rows][head_dim cols],
// boxes of box_rows rows x head_dim (16 by default; 64 for whole pages of 64),
// swizzled so that the kernels' fragment loads are free of shared-memory bank
// conflicts.
int make_code_map(CUtensorMap *m, const int8_t *codes, int num_blocks, int page_size, int head_dim,
                  int box_rows = kChunkTokens)
{
    EncodeTiledFn f = encode_fn();
    if (f == nullptr)
        return MQA_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)num_blocks * (cuuint64_t)page_size};
    const cuuint64_t strides[1] = {(cuuint64_t)head_dim};
    const cuuint32_t box[2] = {(cuuint32_t)head_dim, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(codes), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MQA_OK : MQA_ERR_CUDA;
}

// ---------------------------------------------------------------- planning
int sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 0;
    if (dev < 64) {
        int v = cached[dev].load(std::memory_order_relaxed);
        if (v > 0)
            return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev < 64)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

int tc_ctas_per_sm()
{
    static std::atomic<int> cached{0};
    int v = cached.load(std::memory_order_relaxed);
    if (v <= 0) {
        v = decode_tc_ctas_per_sm();
        cached.store(v, std::memory_order_relaxed);
    }
    return v;
}

// 64-token tiles touched by the decode keys max(0, L-W) .. L-1.
int tiles_for(int L, int W)
{
    const int lo = (W > 0 && L > W) ? L - W : 0;
    return (L - 1) / kTileTokens - lo / kTileTokens + 1;
}

// Upper bound of tiles_for(L, W) over 1 <= L <= Lmax.
int tiles_bound(int Lmax, int W)
{
    const int all = (Lmax + kTileTokens - 1) / kTileTokens;
    if (W <= 0 || Lmax <= W)
        return all;
    const int win = (W - 1) / kTileTokens + 2;
    return win < all ? win : all;
}

// Head groups of a (sequence): 32 query heads each at head_dim 128, 16 at head_dim 64.
int head_groups(int32_t heads, int32_t head_dim)
{
    const int g = decode_heads_per_group(head_dim);
    return (heads + g - 1) / g;
}

// Key blocks of the decode kernel: 128 tokens (head_dim 128) or 256 (head_dim 64,
// two tokens a row), i.e. 2 or 4 of the 64-token tiles.
int blocks_of_tiles(int tiles, int head_dim)
{
    const int t = head_dim == 64 ? 4 : 2;
    return (tiles + t - 1) / t;
}

// The balanced (persistent) decode: CTAs it runs at most (one per SM).
int tc_max_ctas()
{
    const int sms = sm_count();
    if (sms <= 0)
        return 0;
    const int g = sms * tc_ctas_per_sm();
    return g < kTcMaxCtas ? g : kTcMaxCtas;
}

// Whether the automatic plan runs one CTA per (sequence, head group) instead of
// balanced shares.  Cutting a pair between CTAs costs far more than its blocks
// (the pieces' epilogues and reference moves, the merge kernel): measured on
// GB300, a 24-layer step ran 17% faster with whole pairs on its local layers
// (8-9 blocks a pair, 7.2 blocks a balanced share) and 2.5x slower with them on
// its long global layers.  Whole pairs win when waves x the longest pair stays
// within kWholeSlack blocks of the balanced share.  Lengths come from the host
// copy when given, else from max_seq_len.
constexpr int kWholeSlack = 6;

bool tc_whole_pairs(const mqa_batch *bt, int window, int heads, int head_dim)
{
    const long long g = tc_max_ctas();
    if (g <= 0 || bt->batch <= 0)
        return false;
    const long long groups = head_groups(heads, head_dim), pairs = (long long)bt->batch * groups;
    long long nb = 0, maxb = 0;
    if (bt->seq_lens_host != nullptr) {
        for (int b = 0; b < bt->batch; ++b) {
            const long long t = blocks_of_tiles(tiles_for(bt->seq_lens_host[b], window), head_dim);
            nb += t;
            maxb = t > maxb ? t : maxb;
        }
    } else {
        maxb = blocks_of_tiles(tiles_bound(bt->max_seq_len, window), head_dim);
        nb = maxb * bt->batch;
    }
    nb *= groups;
    const long long ctas = g < nb ? g : nb;
    if (ctas <= 0)
        return true;
    const long long waves = (pairs + g - 1) / g;
    return waves * maxb * ctas <= nb + kWholeSlack * ctas;  // waves * maxb <= share + slack
}

// The split count whose workspace holds the partials of every resident CTA (two
// slots of a head group's rows per CTA).
int tc_auto_splits(int batch, int heads, int head_dim)
{
    const long long g = tc_max_ctas();
    const long long pairs = (long long)batch * head_groups(heads, head_dim);
    long long s = (2 * g + pairs - 1) / pairs;
    if (s < 2)
        s = 2;
    return (int)(s > MQA_MAX_SPLITS ? MQA_MAX_SPLITS : s);
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

size_t lse_offset(int32_t batch, int32_t heads, int32_t head_dim, int32_t splits)
{
    return round256((size_t)batch * splits * heads * head_dim * sizeof(float));
}

size_t descs_offset(int32_t batch, int32_t heads, int32_t head_dim, int32_t splits)
{
    return round256(lse_offset(batch, heads, head_dim, splits) + (size_t)batch * splits * heads * sizeof(float));
}


// A window-bounded cache (ring of R pages) serves only reads inside its resident
// pages: the R most recent pages of a sequence hold any run of up to
// (R - 1) * page keys that ends at its last token, i.e. R >= (keys - 1) / page + 2.
bool ring_covers(const mqa_batch *bt, int32_t window, int32_t extra_keys, int page_size)
{
    if (bt->ring_blocks == 0)
        return true;
    if (window <= 0)
        return false;
    return (int64_t)bt->ring_blocks >= ((int64_t)window + extra_keys - 1) / page_size + 2;
}

}  // namespace

extern "C" {

const char *mqa_status_str(int status)
{
    switch (status) {
    case MQA_OK:
        return "ok";
    case MQA_ERR_INVALID_ARG:
        return "invalid argument";
    case MQA_ERR_UNSUPPORTED:
        return "unsupported shape";
    case MQA_ERR_WORKSPACE:
        return "workspace missing or too small";
    case MQA_ERR_CUDA:
        return "CUDA error";
    default:
        return "unknown status";
    }
}

int kv_quant_append(const mqa_kv_cache *cache, const mqa_batch *batch, const int32_t *cu_new,
                    int32_t num_new_tokens, const void *k_new, const void *v_new, int32_t *dev_status, void *stream)
{
    int rc = check_cache(cache);
    if (rc != MQA_OK)
        return rc;
    if (batch == nullptr || num_new_tokens < 0)
        return MQA_ERR_INVALID_ARG;
    if (num_new_tokens == 0)
        return MQA_OK;
    if (batch->batch < 1)
        return MQA_ERR_INVALID_ARG;
    rc = check_batch(batch, cache->page_size);
    if (rc != MQA_OK)
        return rc;
    if (cu_new == nullptr || k_new == nullptr || v_new == nullptr || !aligned16(k_new) || !aligned16(v_new))
        return MQA_ERR_INVALID_ARG;
    AppendArgs a;
    a.k_codes = cache->k_codes;
    a.v_codes = cache->v_codes;
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.num_blocks = cache->num_blocks;
    a.page_size = cache->page_size;
    a.head_dim = cache->head_dim;
    a.block_table = batch->block_table;
    a.seq_lens = batch->seq_lens;
    a.cu_new = cu_new;
    a.batch = batch->batch;
    a.max_blocks = batch->max_blocks;
    a.ring = batch->ring_blocks;
    a.num_tokens = num_new_tokens;
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.dev_status = dev_status;
    return launch_quant_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MQA_OK : MQA_ERR_CUDA;
}

size_t mqa_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t head_dim, int32_t num_splits)
{
    if (num_splits <= 1 || batch <= 0 || num_q_heads <= 0 || head_dim <= 0)
        return 0;
    // partials, log-sum-exps, then the merge descriptors of up to kTcMaxCtas CTAs
    return descs_offset(batch, num_q_heads, head_dim, num_splits) + (size_t)2 * kTcMaxCtas * 8 * sizeof(int32_t);
}

int mqa_decode_auto_splits(const mqa_batch *batch, int32_t window, int32_t num_q_heads, int32_t head_dim,
                           int32_t page_size)
{
    if (!head_dim_ok(head_dim) || !heads_ok(num_q_heads) || !page_ok(page_size))
        return MQA_ERR_UNSUPPORTED;
    if (window < 0)
        return MQA_ERR_INVALID_ARG;
    int rc = check_batch(batch, page_size);
    if (rc != MQA_OK)
        return rc;
    if (batch->batch == 0)
        return 1;
    if (tc_max_ctas() <= 0)
        return MQA_ERR_CUDA;
    return tc_whole_pairs(batch, window, num_q_heads, head_dim) ? 1 : tc_auto_splits(batch->batch, num_q_heads, head_dim);
}

int mqa_decode_attn(const mqa_kv_cache *caches, int32_t num_caches, const int32_t *layer_to_kv, int32_t num_layers,
                    int32_t layer, int32_t window, const mqa_batch *batch, const void *q, void *out,
                    int32_t num_q_heads, float sm_scale, int32_t num_splits, void *workspace,
                    size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    const mqa_kv_cache *cache = nullptr;
    int rc = pick_cache(caches, num_caches, layer_to_kv, num_layers, layer, &cache);
    if (rc != MQA_OK)
        return rc;
    if (!heads_ok(num_q_heads))
        return MQA_ERR_UNSUPPORTED;
    if (window < 0 || num_splits < 0 || num_splits > MQA_MAX_SPLITS || !(std::isfinite(sm_scale) && sm_scale > 0.f))
        return MQA_ERR_INVALID_ARG;
    rc = check_batch(batch, cache->page_size);
    if (rc != MQA_OK)
        return rc;
    if (!ring_covers(batch, window, 0, cache->page_size))
        return MQA_ERR_INVALID_ARG;
    if (batch->batch == 0)
        return MQA_OK;
    if (q == nullptr || out == nullptr || !aligned16(q) || !aligned16(out))
        return MQA_ERR_INVALID_ARG;
    const int D = cache->head_dim;
    // num_splits 1 = one CTA per (sequence, head group); otherwise balanced shares
    // over the CTAs whose partials fit the split count's workspace (the automatic
    // count fits every resident CTA)
    int splits = num_splits;
    if (splits == 0)
        splits = tc_whole_pairs(batch, window, num_q_heads, D) ? 1 : tc_auto_splits(batch->batch, num_q_heads, D);
    DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    const long long pairs = (long long)batch->batch * head_groups(num_q_heads, D);
    if (splits > 1) {
        const size_t need = mqa_decode_workspace_size(batch->batch, num_q_heads, D, splits);
        if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
            return MQA_ERR_WORKSPACE;
        const long long g = tc_max_ctas();
        if (g <= 0)
            return MQA_ERR_CUDA;
        // CTA c keeps its partials in rows [2c, 2c + 2) x (heads of a group) of head_dim
        // floats (and as many log-sum-exps): the regions sized for `splits` hold
        // batch x splits x heads rows, i.e. pairs x splits / 2 CTAs
        a.o_partial = static_cast<float *>(workspace);
        a.lse = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                          lse_offset(batch->batch, num_q_heads, D, splits));
        a.merge_desc = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) +
                                                   descs_offset(batch->batch, num_q_heads, D, splits));
        const long long fit = pairs * splits / 2;
        a.persistent = 1;
        a.persist_ctas = (int)(g < fit ? g : fit);
    } else {
        if (pairs > INT32_MAX)
            return MQA_ERR_INVALID_ARG;
        a.persistent = 0;
        a.persist_ctas = (int)pairs;
    }
    if (D == 64) {
        // two tokens a row: the codes as [num_blocks * page_size / 2][128], 8-row boxes (16 tokens)
        if ((rc = make_code_map(&a.k_map, cache->k_codes, cache->num_blocks, cache->page_size / 2, 128, 8)) != MQA_OK)
            return rc;
        if ((rc = make_code_map(&a.v_map, cache->v_codes, cache->num_blocks, cache->page_size / 2, 128, 8)) != MQA_OK)
            return rc;
    } else {
        if ((rc = make_code_map(&a.k_map, cache->k_codes, cache->num_blocks, cache->page_size, D)) != MQA_OK)
            return rc;
        if ((rc = make_code_map(&a.v_map, cache->v_codes, cache->num_blocks, cache->page_size, D)) != MQA_OK)
            return rc;
        if (cache->page_size == kTileTokens) {
            // whole 64-token tiles (= pages) in one copy per tensor
            if ((rc = make_code_map(&a.k_map64, cache->k_codes, cache->num_blocks, cache->page_size, D,
                                    kTileTokens)) != MQA_OK)
                return rc;
            if ((rc = make_code_map(&a.v_map64, cache->v_codes, cache->num_blocks, cache->page_size, D,
                                    kTileTokens)) != MQA_OK)
                return rc;
        }
    }
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.block_table = batch->block_table;
    a.seq_lens = batch->seq_lens;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.dev_status = dev_status;
    a.batch = batch->batch;
    a.max_blocks = batch->max_blocks;
    a.num_blocks = cache->num_blocks;
    a.page_size = cache->page_size;
    a.max_seq_len = batch->max_seq_len;
    a.ring = batch->ring_blocks;
    a.num_q_heads = num_q_heads;
    a.window = window;
    a.q_scale_log2 = sm_scale * 1.4426950408889634f;
    return launch_decode_tc(a, D, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MQA_OK : MQA_ERR_CUDA;
}

int split_kv_combine(const float *o_partial, const float *lse, int32_t batch, int32_t num_splits,
                     int32_t num_q_heads, int32_t head_dim, void *out, void *stream)
{
    if (!head_dim_ok(head_dim) || !heads_ok(num_q_heads))
        return MQA_ERR_UNSUPPORTED;
    if (batch < 0 || num_splits < 1 || num_splits > MQA_MAX_SPLITS)
        return MQA_ERR_INVALID_ARG;
    if (batch == 0)
        return MQA_OK;
    if (o_partial == nullptr || lse == nullptr || out == nullptr || !aligned16(o_partial) || !aligned16(out))
        return MQA_ERR_INVALID_ARG;
    return launch_combine(o_partial, lse, batch, num_splits, num_q_heads, head_dim,
                          static_cast<__nv_bfloat16 *>(out), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MQA_OK
               : MQA_ERR_CUDA;
}

size_t mqa_prefill_workspace_size(int32_t batch, int32_t max_seq_len, int32_t window, int32_t max_q_len,
                                  int32_t head_dim)
{
    if (!head_dim_ok(head_dim) || batch <= 0 || max_seq_len <= 0 || max_q_len <= 0 || window < 0)
        return 0;
    const size_t recs = (size_t)batch * prefill_tiles_max(max_seq_len, window, max_q_len);
    return round256(recs * prefill_tile_image_bytes(head_dim)) + recs * prefill_tile_record_bytes();
}

int mqa_prefill_attn(const mqa_kv_cache *caches, int32_t num_caches, const int32_t *layer_to_kv,
                     int32_t num_layers, int32_t layer, int32_t window, const mqa_batch *batch,
                     const int32_t *cu_q, int32_t total_q, int32_t max_q_len, const void *q, void *out,
                     int32_t num_q_heads, float sm_scale, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, void *stream)
{
    const mqa_kv_cache *cache = nullptr;
    int rc = pick_cache(caches, num_caches, layer_to_kv, num_layers, layer, &cache);
    if (rc != MQA_OK)
        return rc;
    if (!heads_ok(num_q_heads))
        return MQA_ERR_UNSUPPORTED;
    if (window < 0 || total_q < 0 || max_q_len < 0 || !(std::isfinite(sm_scale) && sm_scale > 0.f))
        return MQA_ERR_INVALID_ARG;
    rc = check_batch(batch, cache->page_size);
    if (rc != MQA_OK)
        return rc;
    if (batch->batch == 0 || total_q == 0)
        return MQA_OK;
    if (max_q_len < 1 || max_q_len > batch->max_seq_len)
        return MQA_ERR_INVALID_ARG;
    if (!ring_covers(batch, window, max_q_len - 1, cache->page_size))
        return MQA_ERR_INVALID_ARG;
    if (cu_q == nullptr || q == nullptr || out == nullptr || !aligned16(q) || !aligned16(out))
        return MQA_ERR_INVALID_ARG;
    const int D = cache->head_dim;
    PrefillArgs a;
    std::memset(&a, 0, sizeof a);
    a.k_codes = cache->k_codes;
    a.v_codes = cache->v_codes;
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.block_table = batch->block_table;
    a.seq_lens = batch->seq_lens;
    a.cu_q = cu_q;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.dev_status = dev_status;
    a.batch = batch->batch;
    a.max_blocks = batch->max_blocks;
    a.num_blocks = cache->num_blocks;
    a.page_size = cache->page_size;
    a.max_seq_len = batch->max_seq_len;
    a.ring = batch->ring_blocks;
    a.num_q_heads = num_q_heads;
    a.window = window;
    a.total_q = total_q;
    a.max_q_len = max_q_len;
    a.q_scale_log2 = sm_scale * 1.4426950408889634f;
    // the tile images and records: [batch][tiles_max] each
    const size_t need = mqa_prefill_workspace_size(batch->batch, batch->max_seq_len, window, max_q_len, D);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
        return MQA_ERR_WORKSPACE;
    a.tiles_max = prefill_tiles_max(batch->max_seq_len, window, max_q_len);
    a.img = static_cast<uint8_t *>(workspace);
    a.srec = a.img + round256((size_t)batch->batch * a.tiles_max * prefill_tile_image_bytes(D));
    return launch_prefill_tc(a, D, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MQA_OK : MQA_ERR_CUDA;
}

}  // extern "C"
