// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mqa {

// Launch with programmatic stream serialisation: the kernel may start (and run
// its set-up) while the previous kernel on the stream finishes; every kernel
// of this library calls griddep_wait() before its first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct AppendArgs {
    int8_t *k_codes, *v_codes;
    float *k_scale, *v_scale;
    int32_t num_blocks, page_size, head_dim;
    const int32_t *block_table, *seq_lens, *cu_new;
    int32_t batch, max_blocks;
    int32_t ring;                      // > 0: window-bounded cache, page p in table entry p % ring
    int32_t num_tokens;
    const __nv_bfloat16 *k_new, *v_new;
    int32_t *dev_status;
};
cudaError_t launch_quant_append(const AppendArgs &a, cudaStream_t s);

struct DecodeArgs {
    // 2-D maps over the int8 codes: head_dim 128, [num_blocks*page_size][128] in 16-row
    // boxes (k_map64, v_map64: 64-row boxes, page_size 64 only); head_dim 64, two tokens
    // a row, [num_blocks*page_size/2][128] in 8-row boxes
    CUtensorMap k_map, v_map;
    CUtensorMap k_map64, v_map64;
    const float *k_scale, *v_scale;
    const int32_t *block_table, *seq_lens;
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;                // bf16 output (whole pairs directly; cut pairs by the merge kernel)
    float *o_partial, *lse;            // partials of pairs cut between CTAs (balanced mode)
    int32_t *dev_status;
    int32_t batch, max_blocks, num_blocks, page_size, max_seq_len;
    int32_t ring;                      // > 0: window-bounded cache, page p in table entry p % ring
    int32_t num_q_heads, window;
    float q_scale_log2;                // sm_scale * log2(e)
    // persistent != 0 = balanced shares of the (sequence, head group, block) list
    // over persist_ctas CTAs (partials in o_partial / lse rows [2 * persist_ctas]
    // [heads of a group]); 0 = one CTA per (sequence, head group), persist_ctas =
    // batch * head groups.  A head group is 32 query heads (head_dim 128) or 16
    // (head_dim 64).
    int32_t persistent, persist_ctas;
    int32_t *merge_desc;               // [2 * persist_ctas][8]: cut pairs to merge (written by every call)
};
// Decode attention on the tcgen05 kernel (head_dim 64 or 128), then, in balanced
// mode, the kernel that merges the pairs cut between CTAs.
cudaError_t launch_decode_tc(const DecodeArgs &a, int head_dim, cudaStream_t s);
constexpr int kTcMaxCtas = 1024;   // balanced decode: at most this many CTAs (merge slots: 2 each)
int decode_tc_ctas_per_sm();
inline int decode_heads_per_group(int head_dim) { return head_dim == 64 ? 16 : 32; }

cudaError_t launch_combine(const float *o_partial, const float *lse, int32_t batch, int32_t num_splits,
                           int32_t num_q_heads, int32_t head_dim, __nv_bfloat16 *out, cudaStream_t s);

struct PrefillArgs {
    const int8_t *k_codes, *v_codes;   // read by the tile-image pass
    const float *k_scale, *v_scale;
    const int32_t *block_table, *seq_lens, *cu_q;
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    int32_t *dev_status;
    int32_t batch, max_blocks, num_blocks, page_size, max_seq_len;
    int32_t ring;                      // > 0: window-bounded cache, page p in table entry p % ring
    int32_t num_q_heads, window, total_q, max_q_len;
    float q_scale_log2;
    // the workspace's fp16 tile images [batch][tiles_max] and their scale records
    uint8_t *img, *srec;
    int32_t tiles_max;
};
// The tile-image pass, then the tcgen05 attention kernel (head_dim 64 or 128).
cudaError_t launch_prefill_tc(const PrefillArgs &a, int head_dim, cudaStream_t s);
int prefill_tiles_max(int max_seq_len, int window, int max_q_len);
size_t prefill_tile_image_bytes(int head_dim);
size_t prefill_tile_record_bytes();

}  // namespace mqa
