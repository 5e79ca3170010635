/*
 * eagle3_chain.h - ragged chain verification in the layout of a serving engine's batch: requests
 * with different numbers of draft tokens laid end to end, their index bookkeeping, and a chain
 * rejection sampler whose recovered tokens are Gumbel-max draws.
 *
 * Conventions as in eagle3.h: asynchronous on the given stream, host-detected errors returned
 * before any launch, device-detected conditions OR-ed into the optional dev_status word, all
 * pointers caller-owned device memory, nothing allocated.
 */
#ifndef EAGLE3_CHAIN_H
#define EAGLE3_CHAIN_H

#include "eagle3.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bit OR-ed into *dev_status: a request's counts are inconsistent (a negative draft count, fewer
 * scheduled tokens than drafts + 1, or more drafts than the output rows hold); its outputs are
 * left untouched (bookkeeping) or filled with -1 (sampler). */
#define EAGLE3_DEV_BAD_COUNTS 0x20

/* ------------------------------------------------------------------------------------------------
 * eagle3_spec_decode_metadata - index bookkeeping of a ragged verify batch.
 *
 * Defines: "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
 * "SpecDecodeMetadata: Index Bookkeeping": the requests' scheduled tokens are laid end to end
 * (cu_num_scheduled_tokens[r] is the running end of request r); a request with d_r draft tokens
 * needs the target's logits at its last d_r + 1 scheduled positions: d_r of them verify its drafts
 * and the last gives its bonus token.  The logits rows are those positions in request order, so
 * request r's rows start at row0_r = (cu_num_draft_tokens[r] - d_r) + r.
 *
 * Outputs (int32): cu_num_draft_tokens[r] = d_0 + ... + d_r;
 *   logits_indices[row0_r + j] = cu_num_scheduled_tokens[r] - d_r - 1 + j,  j = 0..d_r;
 *   target_logits_indices[cu_num_draft_tokens[r] - d_r + j] = row0_r + j,   j < d_r;
 *   bonus_logits_indices[r] = row0_r + d_r;  num_rows[0] = sum_r (d_r + 1).
 * A batch whose rows exceed max_rows sets EAGLE3_DEV_CAPACITY and writes only the rows below it;
 * an inconsistent request sets EAGLE3_DEV_BAD_COUNTS.  One CTA; R up to 2^20.
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t n_requests;                       /* R >= 0                                              */
    int32_t max_rows;                         /* capacity of logits_indices and target_logits_indices */
    const int32_t *cu_num_scheduled_tokens;   /* [R]                                                 */
    const int32_t *num_draft_tokens;          /* [R] d_r                                             */
    int32_t *cu_num_draft_tokens;             /* [R] out                                             */
    int32_t *logits_indices;                  /* [max_rows] out                                      */
    int32_t *target_logits_indices;           /* [max_rows] out                                      */
    int32_t *bonus_logits_indices;            /* [R] out                                             */
    int32_t *num_rows;                        /* [1] out                                             */
    int32_t *dev_status;                      /* optional                                            */
} eagle3_spec_decode_metadata_args_t;

eagle3_status_t eagle3_spec_decode_metadata(const eagle3_spec_decode_metadata_args_t *args,
                                            eagle3_stream_t stream);

/* ------------------------------------------------------------------------------------------------
 * eagle3_chain_verify - chain rejection sampling over a ragged batch, Gumbel-max recovered tokens.
 *
 * Defines: "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section "Rejection
 * Sampling": request r verifies its d_r chained drafts against the target distributions of its
 * rows; a greedy request keeps draft i while it equals the argmax of row i and otherwise emits that
 * argmax; a random request keeps draft i when a uniform draw u < p_i(draft i) (the draft's own
 * probability is taken as 1) and otherwise emits a token drawn from p_i with the draft's entry
 * removed, renormalised, by the Gumbel-max rule argmax_x p_i(x) / E_x with E_x ~ Exp(1); when every
 * draft is kept, a bonus token comes from the last row (greedy: its argmax).  "EAGLE-3: Engineering
 * Implementation of LLM Inference Acceleration", sections X.3-X.6: this emits exactly the target's
 * distribution.
 *
 * Arithmetic (identical in the library's CPU oracle): p = the deterministic fixed-point softmax of
 * eagle3.h (W_x = floor(EXP((z_x - max z) / T) * 2^31), S = sum W); keep iff U32 * S < 2^32 * W_d
 * (exact integers); the Gumbel-max score is fp32(W_x) / E_x (fp32 round-to-nearest division, ties
 * to the lower id) with E_x = EXP_NOISE(w): u = (2 (w >> 9) + 1) * 2^-24, E = -ln u computed as
 * (24 - e) ln 2 - ln m for u * 2^24 = 2^e m, m in [sqrt(1/2), sqrt(2)), ln m by the atanh series.
 * Philox4x32-10, key = seed: the accept word of draft i of request r is word 0 of counter
 * (0x7fffffff, 256 r + i, step low, step high); the noise word of token x in row i is word (x & 3)
 * of counter (x >> 2, 256 r + i, step low, step high).
 *
 * Layout: logits [rows, V] fp32 with request r's d_r + 1 rows starting at row0_r (as in
 * eagle3_spec_decode_metadata: its d_r verification rows, then its bonus row); draft_tokens flat,
 * request r's at [cu_num_draft_tokens[r] - d_r, cu_num_draft_tokens[r]).  Output row r (width
 * max_drafts + 1): the kept drafts, then the recovered or bonus token, then -1.  A request with
 * d_r > max_drafts or a draft token outside [0, V) is skipped (row of -1, num_accepted -1) and
 * flagged (EAGLE3_DEV_BAD_COUNTS / EAGLE3_DEV_BAD_TOKEN).  d_r <= 255.
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t n_requests;                   /* R in [0, 2^24]: one 8-CTA cluster per request           */
    int32_t vocab;                        /* V in [1, 2^22]                                          */
    int32_t max_drafts;                   /* K: output rows hold K + 1 tokens; 0 <= K <= 255          */
    float temperature;                    /* T > 0 for random requests                              */
    uint64_t seed;                        /* Philox key                                              */
    uint64_t step;                        /* counter words 2, 3 (ignored when step_counter is set)   */
    const float *logits;                  /* [rows, V]                                               */
    const int32_t *draft_tokens;          /* [sum d_r]                                               */
    const int32_t *cu_num_draft_tokens;   /* [R]                                                     */
    const int32_t *is_greedy;             /* [R] nonzero: greedy request; NULL: every request random */
    int32_t *output_tokens;               /* [R, K + 1] out                                          */
    int32_t *num_accepted;                /* [R] out (optional)                                      */
    int32_t *dev_status;                  /* optional                                                */
    uint64_t *step_counter;               /* optional device step, read and then incremented         */
} eagle3_chain_verify_args_t;

eagle3_status_t eagle3_chain_verify(const eagle3_chain_verify_args_t *args, eagle3_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE3_CHAIN_H */
