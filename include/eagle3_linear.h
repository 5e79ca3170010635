/*
 * eagle3_linear.h - the tensor-core linear layer of libeagle3 (building block).
 *
 * Defines: the bias-free nn.Linear projections of "EAGLE-3: Engineering Implementation of LLM
 * Inference Acceleration", section VIII and appendix C (fc 3k -> k, q/k/v from 2k, o, SwiGLU
 * gate/up/down, lm_head), out = x W^T, used by the draft head and by the target layers that
 * verify a tree.  bf16 inputs, fp32 accumulation on the tcgen05 tensor cores, fused epilogues:
 *   EAGLE3_EPI_BF16           out (bf16) = x W^T
 *   EAGLE3_EPI_F32            out (fp32) = x W^T                    (logits)
 *   EAGLE3_EPI_BF16_RESIDUAL  out (bf16) = residual + x W^T         (residual stream; out may be
 *                                                                    the residual buffer itself)
 *   EAGLE3_EPI_SWIGLU         out (bf16) = silu(x W^T) * (x W2^T)   (W = gate, W2 = up, both [n, k])
 *   EAGLE3_EPI_BF16_ROPE      out (bf16) = x W^T with rotate-half RoPE applied (in fp32, before the
 *                             rounding) to the columns [0, rope_cols) taken as 128-wide heads: row r
 *                             sits at position pos = rope_base[r / rope_rows_per_seq] + rope_depth[r]
 *                             and, per head, column pair (j, j + 64), j < 64, becomes
 *                             (x_j cos a_j - x_{j+64} sin a_j, x_{j+64} cos a_j + x_j sin a_j) with
 *                             a_j = fp32(pos * inv_j), inv_j = theta^(-2j/128) computed in double and
 *                             rounded to float ("EAGLE-3: Engineering Implementation of LLM Inference
 *                             Acceleration", appendix C: rotate-half RoPE; "Advanced speculative
 *                             decoding: tree drafts and EAGLE", section "Implementation": a tree
 *                             node sits at prefix length + depth).  This is the q / k part of a fused
 *                             QKV projection leaving already rotated; the k-split plans are not used
 *                             and the output must be 16-byte aligned with a pitch of whole 16 bytes.
 * Shapes: x [m, k] (row pitch ld_x), W and W2 [n, k] (row pitch ld_w), out [m, n] (pitch ld_out),
 * residual [m, n] (pitch ld_res); a pitch of 0 means dense.  k and every pitch must be multiples of
 * 8 elements and x, W, W2 must start on 16-byte boundaries.  All pointers are caller-owned device
 * memory.  When the k dimension is split across CTAs (few rows, or long k with a partial last
 * wave), fp32 partials go to the caller's workspace (eagle3_linear_workspace_size bytes) and are
 * added in a fixed order (split order, or CTA order for a stream-K plan).  The split points come
 * from the shape and the device's SM count, so results are reproducible on a given GPU model and
 * agree with any other order within fp32 rounding.  Errors: as in eagle3.h.
 */
#ifndef EAGLE3_LINEAR_H
#define EAGLE3_LINEAR_H

#include "eagle3.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EAGLE3_EPI_BF16 = 0,
    EAGLE3_EPI_F32 = 1,
    EAGLE3_EPI_BF16_RESIDUAL = 2,
    EAGLE3_EPI_SWIGLU = 3,
    EAGLE3_EPI_BF16_ROPE = 4
} eagle3_epilogue_t;

typedef struct {
    int32_t m, n, k;            /* rows of x, rows of W (= output columns), contraction length   */
    int32_t epilogue;           /* eagle3_epilogue_t                                              */
    int32_t splits;             /* k splits; 0 = choose from the shape                            */
    int64_t ld_x, ld_w, ld_out, ld_res;   /* row pitches in elements, 0 = dense                   */
    const uint16_t *x;          /* [m, k] bf16                                                    */
    const uint16_t *w;          /* [n, k] bf16                                                    */
    const uint16_t *w2;         /* [n, k] bf16 (SWIGLU only)                                      */
    void *out;                  /* [m, n] bf16 or fp32                                            */
    const uint16_t *residual;   /* [m, n] bf16 (BF16_RESIDUAL only)                               */
    int32_t *dev_status;        /* optional EAGLE3_DEV_* word                                     */
    /* BF16_ROPE only (ignored otherwise) */
    int32_t rope_cols;          /* rotated columns, a multiple of 128, <= n                        */
    int32_t rope_rows_per_seq;  /* rows of one sequence (row r belongs to sequence r / this)       */
    float rope_theta;           /* > 0                                                            */
    const int32_t *rope_base;   /* [ceil(m / rope_rows_per_seq)] base position per sequence        */
    const int32_t *rope_depth;  /* [m] offset per row                                             */
    /* F32 only (NULL otherwise): [m] row-maximum words.  Each is raised (atomic max) to the order
       key of the largest output of its row, so a reader of the row (e.g. a top-k with a
       normaliser that subtracts the row maximum) needs no pass of its own to find it.  The order key
       of x maps its fp32 bit pattern b to b ^ 0x80000000 for x >= 0 (sign bit clear) and to ~b
       otherwise, so unsigned order is float order.  The caller sets the words to 0 beforehand.   */
    uint32_t *row_max;
    /* RMSNorm folded into the neighbouring projections ("EAGLE-3: Engineering Implementation of
       LLM Inference Acceleration", appendix C: RMSNorm(x) = x * rsqrt(mean(x^2) + eps) * g before
       every projection that reads the residual stream).  Since
           RMSNorm(x) W^T = diag(rsqrt(mean(x^2) + eps)) (x W'^T),  W' = W diag(g),
       a projection may read the un-normalised stream x with the norm weight folded into its
       weights and scale each output row afterwards, given the row's sum of squares, which the
       projection that produced x can emit on the way out.
       row_ssq (BF16 / BF16_RESIDUAL only; NULL otherwise): [ceil(n / 256)][m] fp32 out: for each
         row and each block of 256 output columns, the sum of squares of the bf16 outputs as stored
         (in a fixed order; blocks are whole-row sums when added in block order).
       row_ssq_in (optional): [ssq_blocks][m] fp32, such sums of the rows of x: each output row's
         accumulator is multiplied by rsqrt((sum over blocks in order) / ssq_dim + ssq_eps) before
         the epilogue (before the residual add, the rotation, the SwiGLU or the fp32 store).
       Either option rules out the k-split plans with a separate reduction (a k-split caller
       request returns EAGLE3_ERR_UNSUPPORTED).                                                  */
    float *row_ssq;
    const float *row_ssq_in;
    int32_t ssq_blocks;         /* >= 1 with row_ssq_in                                            */
    int32_t ssq_dim;            /* >= 1 with row_ssq_in: the length of the rows of x               */
    float ssq_eps;              /* >= 0                                                            */
} eagle3_linear_args_t;

size_t eagle3_linear_workspace_size(const eagle3_linear_args_t *args);
eagle3_status_t eagle3_linear(const eagle3_linear_args_t *args, void *workspace, size_t workspace_bytes,
                              eagle3_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE3_LINEAR_H */
