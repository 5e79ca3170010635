/* eagle3_f32.h - fp32 building blocks for small models: the tiny lossless configuration (a
 * 4-layer Llama-style target with d = 64 and 16-dim heads, and its EAGLE-3 head) runs its target
 * and draft layers on these, and its acceptance and compaction on eagle3_accept and
 * eagle3_compact_kv.
 *
 * Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", appendix C
 * (bias-free linear layers, RMSNorm, rotate-half RoPE, grouped-query attention, SwiGLU MLP) and
 * section VIII (the draft decoder layer); "Advanced speculative decoding: tree drafts and EAGLE",
 * section "Implementation" (tree rows attend to the cache plus their ancestors).
 *
 * Every output row is computed on its own, in an order fixed by the row's own data: a dot product
 * runs over k in order, a row reduction is a fixed tree over a fixed lane assignment, attention
 * visits the row's keys in sequence order (cache positions, then the visible new rows by index).
 * So a row computed inside a batch or a tree pass is bitwise equal to the same row computed alone
 * (vanilla decoding), which is what makes greedy speculative decoding reproduce vanilla greedy
 * decoding token for token.  These kernels are plain SIMT code meant for small shapes.
 *
 * Conventions as in eagle3.h: caller-owned device memory, asynchronous on `stream`, argument
 * errors returned before any launch.
 */
#ifndef EAGLE3_F32_H
#define EAGLE3_F32_H

#include "eagle3.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[m, n] = epilogue(x[m, k] W[n, k]^T), W in nn.Linear [out, in] layout.
 *   EAGLE3_F32_EPI_NONE      out = x W^T
 *   EAGLE3_F32_EPI_RESIDUAL  out = residual + x W^T (residual may be out itself)
 *   EAGLE3_F32_EPI_SWIGLU    out = silu(x W^T) * (x W2^T)
 * Row pitches (elements) of x, out and residual default to k, n and n when 0. */
enum { EAGLE3_F32_EPI_NONE = 0, EAGLE3_F32_EPI_RESIDUAL = 1, EAGLE3_F32_EPI_SWIGLU = 2 };
typedef struct {
    int64_t m, n, k;
    int32_t epilogue;
    int64_t ld_x, ld_out, ld_res;
    const float *x;
    const float *w;
    const float *w2;         /* SWIGLU only */
    const float *residual;   /* RESIDUAL only */
    float *out;
} eagle3_f32_linear_args_t;
eagle3_status_t eagle3_f32_linear(const eagle3_f32_linear_args_t *args, eagle3_stream_t stream);

/* out[r, :] = w * x[g, :] / sqrt(mean(x[g, :]^2) + eps), g = gather ? gather[r] : r.
 * Row pitches ld_x / ld_out in elements (0 = dim). */
eagle3_status_t eagle3_f32_rmsnorm(int64_t rows, int64_t dim, const float *x, int64_t ld_x, const int32_t *gather,
                                   const float *w, float eps, float *out, int64_t ld_out, eagle3_stream_t stream);

/* Rotate-half RoPE in place: x[r, h, :] for h < heads, row pitch ld (elements), at position pos[r];
 * inv_j = theta^(-2j/D) is computed in double and rounded to float, angle = float(pos * inv_j). */
eagle3_status_t eagle3_f32_rope(int64_t rows, int32_t heads, int32_t head_dim, float *x, int64_t ld,
                                const int32_t *pos, float theta, eagle3_stream_t stream);

/* out[r, :] = table[idx[r], :] (embedding lookup); ld_out in elements (0 = dim). */
eagle3_status_t eagle3_f32_gather(int64_t rows, int64_t dim, const float *table, const int32_t *idx, float *out,
                                  int64_t ld_out, eagle3_stream_t stream);

/* out[r] = argmax_v logits[r, v] (ties to the lowest index; the same total order as eagle3_accept). */
eagle3_status_t eagle3_f32_argmax(int64_t rows, int64_t vocab, const float *logits, int32_t *out,
                                  eagle3_stream_t stream);

/* Attention of T new rows over a cache plus the new rows they may see.  Row i, query head h
 * (KV head g = h / (Hq/Hkv)) attends, in this order, to cache positions 0..cache_len-1 and to the
 * new rows j whose bit is set in visible[i]; softmax of q.k * scale in fp32, weighted sum of v.
 * Keys and queries arrive rotated.  T <= 64, head_dim <= 128, cache_len + T <= 65536. */
typedef struct {
    int32_t n_rows;          /* T */
    int32_t n_heads;         /* Hq, a multiple of n_kv_heads */
    int32_t n_kv_heads;      /* Hkv */
    int32_t head_dim;        /* D */
    int32_t cache_len;       /* L */
    int32_t s_max;           /* cache capacity in positions */
    float scale;             /* 0 = 1/sqrt(D) */
    int64_t ld_q;            /* elements between rows of q (0 = Hq * D) */
    int64_t ld_kv;           /* elements between rows of k_new / v_new (0 = Hkv * D) */
    const float *q;          /* [T, Hq, D] */
    const float *k_new;      /* [T, Hkv, D] */
    const float *v_new;
    const float *k_cache;    /* [Hkv, s_max, D] */
    const float *v_cache;
    const uint64_t *visible; /* [T] */
    float *out;              /* [T, Hq, D] */
} eagle3_f32_attn_args_t;
eagle3_status_t eagle3_f32_attn(const eagle3_f32_attn_args_t *args, eagle3_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
