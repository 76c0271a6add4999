/*
 * mqa_oracle.c -- plain, slow, single-threaded CPU oracle for int8 paged MQA.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes, and where each step comes from:
 *
 *  - quantise (oracle_quantize_token): symmetric per-token int8 with one fp32
 *    scale per token for K and one for V.  The pages say only that the KV cache
 *    is int8 ("Character.AI best practices" blog, section "training and serving
 *    quantisation": weights, activations and the attention KV cache in int8);
 *    the per-token symmetric scheme (scale = max|x|/127, round half to even,
 *    clamp to +-127) is the reading stated for this library.  All steps in IEEE
 *    fp32 with round-to-nearest-even.
 *  - paged store (oracle_quant_append): the logical token position p of
 *    sequence b lives in physical block block_table[b][p / page] at row
 *    p % page -- a pure re-addressing (LLM-inference workshop transcript,
 *    01:01:35-01:03:22, PagedAttention: logical blocks mapped to physical ones).
 *    A window-bounded cache (ring_blocks = R > 0) keeps only the R most recent
 *    pages of a sequence: page p / page lives in table entry (p / page) % R,
 *    and a later page overwrites the entry of the page R before it (the local
 *    layers of the "Character.AI inference article", secret 1, attend over a
 *    1024-token window only, so older keys need not stay resident).  A key
 *    is resident iff its page is one of the R most recent of the sequence.
 *  - attention (oracle_attention): multi-query attention -- every query head
 *    attends to the one shared K/V head ("Character.AI inference article",
 *    secret 1, "use MQA everywhere"; workshop 00:44:39-00:45:08).  A local layer
 *    with window W lets the query at position i see keys j with i-W < j <= i
 *    (article, secret 1, "hybrid attention horizon": local layers attend over
 *    a sliding 1024-token window); W = 0 means global (j <= i).  Scores
 *    s_j = sm_scale * <q, k^_j> and out = sum_j e^{s_j-m} v^_j / sum_j e^{s_j-m}
 *    in fp64 over dequantised x^ = code * scale, plus lse = m + ln(sum).  The
 *    tiled online softmax of FlashAttention (workshop 00:48:51-00:49:13) yields
 *    this same value; the oracle does not tile.
 *  - combine (oracle_combine): the log-sum-exp merge of partial results over
 *    disjoint key ranges, the same identity the online softmax relies on.
 *
 * Pinned by the "not gpu" tests (tie cases, closed forms, torch fp64 SDPA on
 * tiny inputs, a dense brute-force loop, and invariants); no function here is
 * unpinned.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -shared -fPIC
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Quantise one token vector of d bf16 values.  scale = fl32(amax / 127);
 * code = clamp(round_half_even(fl32(x / scale)), -127, 127); an all-zero
 * vector gives scale 0 and codes 0. */
void oracle_quantize_token(const uint16_t *x, int32_t d, int8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int32_t k = 0; k < d; ++k) {
        float a = fabsf(bf16_to_f32(x[k]));
        if (a > amax)
            amax = a;
    }
    volatile float s = amax / 127.0f; /* one IEEE fp32 division */
    *scale = s;
    if (s == 0.0f) {
        memset(codes, 0, (size_t)d);
        return;
    }
    for (int32_t k = 0; k < d; ++k) {
        volatile float r = bf16_to_f32(x[k]) / s; /* fp32 division by the stored scale */
        float c = nearbyintf(r);                  /* default mode: to nearest, ties to even */
        if (c > 127.0f)
            c = 127.0f;
        if (c < -127.0f)
            c = -127.0f;
        codes[k] = (int8_t)c;
    }
}

/* Quantise the new tokens of every sequence and store them in the paged cache.
 * Sequence b appends cu_new[b+1]-cu_new[b] tokens that occupy the LAST
 * positions of its seq_lens[b] tokens.  k_new / v_new are bf16 [T, d].
 * Returns ORACLE_EINVAL (and writes nothing more) on any out-of-range index. */
int oracle_quant_append(int8_t *k_codes, int8_t *v_codes, float *k_scale, float *v_scale,
                        int32_t num_blocks, int32_t page_size, int32_t d,
                        const int32_t *block_table, int32_t max_blocks,
                        const int32_t *seq_lens, int32_t batch, const int32_t *cu_new,
                        const uint16_t *k_new, const uint16_t *v_new, int32_t ring_blocks)
{
    if (ring_blocks < 0 || ring_blocks > max_blocks)
        return ORACLE_EINVAL;
    for (int32_t b = 0; b < batch; ++b) {
        int32_t n = cu_new[b + 1] - cu_new[b];
        int32_t first = seq_lens[b] - n;
        if (n < 0 || first < 0)
            return ORACLE_EINVAL;
        if (ring_blocks > 0 && (int64_t)n > (int64_t)ring_blocks * page_size)
            return ORACLE_EINVAL; /* the call's own tokens would overwrite one another */
        for (int32_t t = 0; t < n; ++t) {
            int32_t pos = first + t;
            int32_t lb = pos / page_size;
            if (ring_blocks > 0)
                lb %= ring_blocks;
            if (lb >= max_blocks)
                return ORACLE_EINVAL;
            int32_t blk = block_table[(int64_t)b * max_blocks + lb];
            if (blk < 0 || blk >= num_blocks)
                return ORACLE_EINVAL;
            int64_t slot = (int64_t)blk * page_size + pos % page_size;
            int64_t row = (int64_t)cu_new[b] + t;
            oracle_quantize_token(k_new + row * d, d, k_codes + slot * d, k_scale + slot);
            oracle_quantize_token(v_new + row * d, d, v_codes + slot * d, v_scale + slot);
        }
    }
    return ORACLE_OK;
}

/* Dequantise one cached token row: x^_k = (double)code_k * (double)scale. */
static void dequant_row(const int8_t *codes, float scale, int32_t d, double *dst)
{
    for (int32_t k = 0; k < d; ++k)
        dst[k] = (double)codes[k] * (double)scale;
}

/* Exact softmax attention of query rows over one paged int8 cache.
 *
 * Row r is the query of sequence row_seq[r] at absolute position row_pos[r]
 * (decode: seq_lens[b]-1; prefill: seq_lens[b]-q_len+t).  Its keys are the
 * positions j with lo <= j <= row_pos[r], lo = max(0, pos-window+1) for a
 * local layer (window > 0) and 0 for a global one, further restricted to
 * [key_begin, key_end) when key_end >= 0 (used to form split-KV partials).
 *
 * q is bf16 [rows, num_q_heads, d]; out is fp64 [rows, num_q_heads, d];
 * lse is fp64 [rows, num_q_heads] (natural log; -inf for an empty key set,
 * whose out is 0).  If probs is not NULL, probs[(r*H + h)*probs_stride + j]
 * receives the attention weight of key j (entries outside the key set are
 * left untouched).  scratch must hold (max keys of any row)*H + (H+1)*d doubles. */
int oracle_attention(const int8_t *k_codes, const int8_t *v_codes,
                     const float *k_scale, const float *v_scale,
                     int32_t num_blocks, int32_t page_size, int32_t d,
                     const int32_t *block_table, int32_t max_blocks,
                     const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                     const uint16_t *q, int32_t rows, const int32_t *row_seq,
                     const int32_t *row_pos, int32_t window, double sm_scale,
                     int32_t key_begin, int32_t key_end,
                     double *out, double *lse, double *probs, int64_t probs_stride,
                     double *scratch, int32_t ring_blocks)
{
    const int32_t H = num_q_heads;
    if (ring_blocks < 0 || ring_blocks > max_blocks)
        return ORACLE_EINVAL;
    for (int32_t r = 0; r < rows; ++r) {
        const int32_t b = row_seq[r];
        const int32_t i = row_pos[r];
        if (b < 0 || b >= batch || i < 0 || i >= seq_lens[b])
            return ORACLE_EINVAL;
        int32_t lo = (window > 0) ? (i - window + 1) : 0;
        if (lo < 0)
            lo = 0;
        int32_t hi = i + 1; /* exclusive */
        if (key_end >= 0) {
            if (key_begin > lo)
                lo = key_begin;
            if (key_end < hi)
                hi = key_end;
        }
        const int32_t n = hi > lo ? hi - lo : 0;
        double *s = scratch;              /* [n][H] scores */
        double *kh = scratch + (int64_t)n * H; /* [d] one dequantised K or V row */
        double *qd = kh + d;              /* [H][d] query as double */
        for (int32_t h = 0; h < H; ++h)
            for (int32_t k = 0; k < d; ++k)
                qd[(int64_t)h * d + k] = (double)bf16_to_f32(q[((int64_t)r * H + h) * d + k]);
        double *o = out + (int64_t)r * H * d;
        memset(o, 0, sizeof(double) * (size_t)H * (size_t)d);
        if (n == 0) {
            for (int32_t h = 0; h < H; ++h)
                lse[(int64_t)r * H + h] = -INFINITY;
            continue;
        }
        /* scores s_j = sm_scale * <q_h, k^_j> */
        for (int32_t jj = 0; jj < n; ++jj) {
            const int32_t j = lo + jj;
            int32_t lb = j / page_size;
            if (ring_blocks > 0) {
                /* resident only among the sequence's ring_blocks most recent pages */
                if (lb <= (seq_lens[b] - 1) / page_size - ring_blocks)
                    return ORACLE_EINVAL;
                lb %= ring_blocks;
            }
            if (lb >= max_blocks)
                return ORACLE_EINVAL;
            const int32_t blk = block_table[(int64_t)b * max_blocks + lb];
            if (blk < 0 || blk >= num_blocks)
                return ORACLE_EINVAL;
            const int64_t slot = (int64_t)blk * page_size + j % page_size;
            dequant_row(k_codes + slot * d, k_scale[slot], d, kh);
            for (int32_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int32_t k = 0; k < d; ++k)
                    acc += qd[(int64_t)h * d + k] * kh[k];
                s[(int64_t)jj * H + h] = sm_scale * acc;
            }
        }
        /* per head: m = max_j s_j, weights e^{s_j - m}, denominator */
        for (int32_t h = 0; h < H; ++h) {
            double m = -INFINITY;
            for (int32_t jj = 0; jj < n; ++jj)
                if (s[(int64_t)jj * H + h] > m)
                    m = s[(int64_t)jj * H + h];
            double den = 0.0;
            for (int32_t jj = 0; jj < n; ++jj) {
                double e = exp(s[(int64_t)jj * H + h] - m);
                s[(int64_t)jj * H + h] = e;
                den += e;
            }
            for (int32_t jj = 0; jj < n; ++jj) {
                s[(int64_t)jj * H + h] /= den;
                if (probs)
                    probs[((int64_t)r * H + h) * probs_stride + lo + jj] = s[(int64_t)jj * H + h];
            }
            lse[(int64_t)r * H + h] = m + log(den);
        }
        /* out_h = sum_j p_hj v^_j */
        for (int32_t jj = 0; jj < n; ++jj) {
            const int32_t j = lo + jj;
            const int32_t lb = ring_blocks > 0 ? (j / page_size) % ring_blocks : j / page_size;
            const int32_t blk = block_table[(int64_t)b * max_blocks + lb];
            const int64_t slot = (int64_t)blk * page_size + j % page_size;
            dequant_row(v_codes + slot * d, v_scale[slot], d, kh);
            for (int32_t h = 0; h < H; ++h) {
                const double p = s[(int64_t)jj * H + h];
                for (int32_t k = 0; k < d; ++k)
                    o[(int64_t)h * d + k] += p * kh[k];
            }
        }
    }
    return ORACLE_OK;
}

/* Merge S partial results over disjoint key ranges.  parts is fp64 [S][n][d],
 * part_lse is fp64 [S][n] (natural log, -inf = empty part).  For each of the n
 * (row, head) pairs: M = max_s lse_s, w_s = e^{lse_s - M},
 * out = sum_s w_s part_s / sum_s w_s, lse = M + ln sum_s w_s.  All parts empty:
 * out = 0, lse = -inf. */
void oracle_combine(const double *parts, const double *part_lse, int32_t S, int64_t n,
                    int32_t d, double *out, double *lse)
{
    for (int64_t x = 0; x < n; ++x) {
        double M = -INFINITY;
        for (int32_t s = 0; s < S; ++s)
            if (part_lse[(int64_t)s * n + x] > M)
                M = part_lse[(int64_t)s * n + x];
        double *o = out + x * d;
        for (int32_t k = 0; k < d; ++k)
            o[k] = 0.0;
        if (M == -INFINITY) {
            lse[x] = -INFINITY;
            continue;
        }
        double den = 0.0;
        for (int32_t s = 0; s < S; ++s) {
            double ls = part_lse[(int64_t)s * n + x];
            if (ls == -INFINITY)
                continue;
            double w = exp(ls - M);
            den += w;
            const double *p = parts + ((int64_t)s * n + x) * d;
            for (int32_t k = 0; k < d; ++k)
                o[k] += w * p[k];
        }
        for (int32_t k = 0; k < d; ++k)
            o[k] /= den;
        lse[x] = M + log(den);
    }
}
