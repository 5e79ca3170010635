/*
 * eagle3_ttt.h - the training-time-test attention of the EAGLE-3 draft layer (the attention of
 * the draft's training; the training itself needs data and is not part of this library).
 *
 * Conventions as in eagle3.h: asynchronous on the stream, host-detected errors returned before any
 * launch, caller-owned device memory, scratch in a caller workspace.
 */
#ifndef EAGLE3_TTT_H
#define EAGLE3_TTT_H

#include "eagle3.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------------------------------
 * eagle3_ttt_attn - attention of one training-time-test step over all simulated steps.
 *
 * Defines: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections VII.5
 * (Figure 6's mask) and VIII.2 (forward_ttt): the query at position i attends causally to the
 * native step's keys 0..i and, of every simulated step s >= 1, to that step's key at position i
 * alone (the diagonal, a per-position dot product).  For batch row b, position i, query head h
 * (KV head g = h / (Hq / Hkv)):
 *   out[b,i,h] = sum over keys j in {k[0,b,0..i]} U {k[s,b,i] : 1 <= s < n_steps} of
 *                softmax_j(q[b,i,h] . k_j * sm_scale) v_j.
 * q and k carry their rotary embedding already; bf16 in and out, fp32 softmax and accumulation.
 *
 * Design: the causal part runs on the tree-attention kernel of eagle3_verify_attn: the positions
 * are cut into chunks of C = min(64, 256 / (Hq / Hkv)) positions, each chunk a chain "tree" whose
 * prefix (the positions before the chunk) is read through an identity block table over the native
 * keys; its log-sum-exp then lets one more kernel fold the diagonal keys in.  seq_len must be a
 * multiple of C (EAGLE3_ERR_UNSUPPORTED otherwise); head_dim 128; Hq / Hkv in {1, 2, 4, 8}.
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t batch;            /* Bt >= 0                                                       */
    int32_t seq_len;          /* T, a multiple of the chunk C                                  */
    int32_t n_heads;          /* Hq                                                            */
    int32_t n_kv_heads;       /* Hkv                                                           */
    int32_t head_dim;         /* D = 128                                                       */
    int32_t n_steps;          /* S >= 1: the native step and S - 1 simulated steps             */
    float sm_scale;           /* 0 = 1 / sqrt(D)                                               */
    const uint16_t *q;        /* [Bt, T, Hq, D] bf16                                           */
    const uint16_t *k;        /* [S, Bt, T, Hkv, D] bf16: step 0 native, then simulated steps  */
    const uint16_t *v;        /* [S, Bt, T, Hkv, D] bf16                                       */
    uint16_t *out;            /* [Bt, T, Hq, D] bf16                                           */
    int32_t *dev_status;      /* optional                                                      */
} eagle3_ttt_attn_args_t;

size_t eagle3_ttt_attn_workspace_size(const eagle3_ttt_attn_args_t *args);
eagle3_status_t eagle3_ttt_attn(const eagle3_ttt_attn_args_t *args, void *workspace, size_t workspace_bytes,
                                eagle3_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE3_TTT_H */
