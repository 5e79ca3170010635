/*
 * eagle3.h - C ABI of libeagle3, one EAGLE-3 draft-and-verify step on one GPU.
 *
 * Every entry point is asynchronous on the given CUDA stream and returns an
 * eagle3_status_t.  Argument, shape and capacity errors are detected on the
 * host, before anything is launched, and returned synchronously.  Errors that
 * only the device can see (a malformed parent array, a token id out of range,
 * a wait that ran out of time) are OR-ed into the caller's optional device
 * word `dev_status` (EAGLE3_DEV_* bits); the call itself still returns
 * EAGLE3_OK.  A failed launch returns EAGLE3_ERR_CUDA.
 *
 * Memory: every pointer in an argument struct is caller-owned DEVICE memory
 * unless its comment says otherwise.  The library allocates nothing; calls
 * that need scratch space take a caller-owned device workspace whose size the
 * matching *_workspace_size() function returns (0 means none is needed).
 * Tensors are dense, row-major, with the innermost dimension last, and must
 * start on a 16-byte boundary.  bf16 values are passed as uint16_t bit
 * patterns.  The library keeps no state between calls except cached device
 * attributes; calls on different streams do not share memory.
 *
 * Tree conventions (all entry points): a draft tree of N <= 64 nodes is a
 * parent array `parents[N]` with parents[0] = -1 (node 0 is the root, the
 * token the target produced last step) and 0 <= parents[i] < i.  Node i
 * attends to every cached prefix position, to the nodes on its path from the
 * root and to itself, and sits at position prefix_len + depth(i).
 */
#ifndef EAGLE3_H
#define EAGLE3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *eagle3_stream_t; /* identical to cudaStream_t; NULL = legacy default stream */

typedef enum {
    EAGLE3_OK = 0,
    EAGLE3_ERR_INVALID_ARGUMENT = 1, /* null pointer, misaligned pointer, negative or inconsistent size */
    EAGLE3_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. head_dim != 128, N > 64)      */
    EAGLE3_ERR_CAPACITY = 3,         /* prefix + tree would not fit the cache (S_max)                 */
    EAGLE3_ERR_BAD_TREE = 4,         /* host-visible tree parameters are inconsistent                */
    EAGLE3_ERR_CUDA = 5,             /* a CUDA runtime call or kernel launch failed                   */
    EAGLE3_ERR_WORKSPACE = 6         /* workspace missing or smaller than *_workspace_size()          */
} eagle3_status_t;

/* Bits OR-ed into *dev_status by the kernels (device-detected conditions). */
#define EAGLE3_DEV_BAD_TREE   0x1 /* parents[0] != -1 or parents[i] not in [0, i): that sequence is skipped  */
#define EAGLE3_DEV_BAD_TOKEN  0x2 /* a token id outside [0, vocab): that sequence is skipped                 */
#define EAGLE3_DEV_CAPACITY   0x4 /* a per-sequence length exceeded the bound given on the host              */
#define EAGLE3_DEV_TIMEOUT    0x8 /* a bounded wait inside a kernel gave up; outputs of that block are void */
#define EAGLE3_DEV_PATH_TRUNC 0x10 /* an accepted path was longer than max_path: it was cut                 */

const char *eagle3_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int eagle3_version(void);

/* ------------------------------------------------------------------------------------------------
 * eagle3_accept - lossless acceptance of a verified draft tree.
 *
 * Defines: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections III.5
 * and X.3-X.6 (a drafted token x survives when a uniform draw falls below p(x)/q(x), capped at 1;
 * after a rejection the replacement comes from max(0, p - q) renormalised; when every draft
 * survives, one extra token comes from the last target distribution), "Advanced speculative decoding: tree drafts and EAGLE", section "Implementation"
 * (greedy walk: follow the child whose token equals the target argmax) and exercise 2 (multiple
 * candidates per node: try the children in turn, replacing p by the residual after each
 * rejection), and "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
 * "Rejection Sampling" (output rows of accepted drafts then the correction or bonus token,
 * padded with -1).
 *
 * Modes:
 *   EAGLE3_ACCEPT_GREEDY   temperature 0: pred = argmax of the node's target logits (fp32 total
 *                          order of bit patterns, lowest id on ties); move to the lowest-index child
 *                          whose token == pred; stop when there is none.  next_root = last pred.
 *   EAGLE3_ACCEPT_TOPK     temperature T > 0 with children chosen deterministically (top-k of the
 *                          draft): q is the point mass on each child, so child x is accepted with
 *                          probability p_cur(x) and rejected children are removed from p.
 *   EAGLE3_ACCEPT_SAMPLED  temperature T > 0 with children drawn without replacement from the
 *                          draft's distribution q = softmax(draft_logits / T): recursive rejection
 *                          sampling with the residual max(0, p - q) and q renormalised after each
 *                          removed child.
 * Probabilities are the deterministic fixed-point softmax: W_i = floor(EXP((z_i - max z) / T) *
 * 2^31) with a specified fp32 EXP, p_i = W_i / sum W; every comparison is exact integer
 * arithmetic.  Random words come from Philox4x32-10 (Salmon et al., SC'11) with key = seed and
 * counter = (slot + 256 * node, b, step low, step high): U32 = word 0 for the accept test of the
 * s-th child (slot s), R64 = word1:word2 for the residual / bonus draw (slot 64).
 * ---------------------------------------------------------------------------------------------- */
typedef enum {
    EAGLE3_ACCEPT_GREEDY = 0,
    EAGLE3_ACCEPT_TOPK = 1,
    EAGLE3_ACCEPT_SAMPLED = 2
} eagle3_accept_mode_t;

typedef struct {
    int32_t mode;               /* eagle3_accept_mode_t                                               */
    int32_t batch;              /* B >= 0                                                              */
    int32_t n_nodes;            /* N in [1, 64]                                                        */
    int32_t vocab;              /* V in [1, 2^22]                                                      */
    int32_t max_path;           /* width W of path / emitted rows, >= 1 (a path of depth d needs d+1)  */
    float temperature;          /* T > 0 for TOPK / SAMPLED; ignored for GREEDY                        */
    uint64_t seed;              /* Philox key                                                          */
    uint64_t step;              /* draft-and-verify cycle counter (Philox counter words 2, 3)          */
    const float *target_logits; /* [B, N, V] fp32: target logits at every tree node                   */
    const float *draft_logits;  /* [B, N, V] fp32: draft logits at every node (SAMPLED only, else NULL)*/
    const int32_t *tokens;      /* [B, N] token of each node (node 0's entry is not read)              */
    const int32_t *parents;     /* [B, N] parent arrays                                                */
    int32_t *accept_len;        /* [B] out: number of accepted draft nodes n (path has n+1 nodes)      */
    int32_t *path;              /* [B, W] out: node ids root..last accepted, then -1                   */
    int32_t *emitted;           /* [B, W] out: tokens of path[1..n], then next_root, then -1           */
    int32_t *next_root;         /* [B] out: correction / bonus token (the next step's root)           */
    int32_t *dev_status;        /* [1] optional device word for EAGLE3_DEV_* bits (may be NULL)       */
    uint64_t *step_counter;     /* [1] optional device word: when not NULL the Philox step is read from
                                   it (the `step` field is ignored) and it is incremented after the
                                   call, so a captured CUDA graph draws fresh numbers on every replay */
} eagle3_accept_args_t;

size_t eagle3_accept_workspace_size(const eagle3_accept_args_t *args);
eagle3_status_t eagle3_accept(const eagle3_accept_args_t *args, void *workspace, size_t workspace_bytes,
                              eagle3_stream_t stream);

/* ------------------------------------------------------------------------------------------------
 * eagle3_accept_lazy - eagle3_accept with a lazy target LM head: target logits only for the nodes
 * the walk visits.
 *
 * Defines: "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section "Rejection
 * Sampling" (the target's distribution is needed only where a decision is taken) with the walk of
 * eagle3_accept.  The walk visits one node per level; level by level the library gathers the
 * final-normed hidden state of every sequence's current node, computes its logits
 * (x W_lm^T, fp32, on the tensor cores, M = batch) and advances the walk by one node, until every
 * sequence has stopped (at most max_path levels; a level in which no sequence is still walking
 * launches kernels that return at once).  Results are those of eagle3_accept on the logits of the
 * visited nodes as computed here.  Modes GREEDY and TOPK (SAMPLED needs the draft logits of the
 * visited nodes too: EAGLE3_ERR_UNSUPPORTED).  accept.target_logits is not read.
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    eagle3_accept_args_t accept; /* as for eagle3_accept (target_logits unused)                      */
    int32_t hidden;              /* d, a multiple of 8                                               */
    const uint16_t *hidden_states; /* [B, N, d] bf16: every tree node's final-normed hidden state    */
    const uint16_t *lm_head;     /* [V, d] bf16                                                      */
    float *dbg_level_logits;     /* optional [max_path, B, V] fp32: each level's logits row per
                                    sequence (rows of sequences that had stopped are not defined)    */
} eagle3_accept_lazy_args_t;

size_t eagle3_accept_lazy_workspace_size(const eagle3_accept_lazy_args_t *args);
eagle3_status_t eagle3_accept_lazy(const eagle3_accept_lazy_args_t *args, void *workspace,
                                   size_t workspace_bytes, eagle3_stream_t stream);

/* ------------------------------------------------------------------------------------------------
 * eagle3_compact_kv - copy the accepted path's K/V into contiguous cache slots.
 *
 * Defines: "Advanced speculative decoding: tree drafts and EAGLE", section "Implementation" (the
 * verify pass already produced the path nodes' K/V at their final positions, so they are copied
 * into the cache instead of recomputed, and the other nodes are discarded) and "EAGLE-3: Engineering Implementation of LLM
 * Inference Acceleration", section XI.4 (the target cache keeps exactly the committed positions).
 *
 * For each sequence b with L = prefix_len[b] and n = accept_len[b]: for j = 0..n, every layer and
 * KV head, cache slot L + j <- tree row path[b, j]; slot_map[b, j] = L + j (then -1); optional aux
 * rows are gathered in path order; finally prefix_len[b] = L + n + 1.  Copies are bit-exact.
 * Source and destination must not overlap (the tree K/V live in their own buffers).
 * Sequences with L + n + 1 > s_max or a path entry outside [0, N) are skipped and flagged.
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t n_layers;            /* >= 1                                                              */
    int32_t batch;               /* B >= 0                                                            */
    int32_t n_nodes;             /* N in [1, 64]                                                      */
    int32_t n_kv_heads;          /* Hkv >= 1                                                          */
    int32_t head_dim;            /* D >= 1                                                            */
    int32_t elem_bytes;          /* 2 (bf16) or 4 (fp32)                                              */
    int32_t s_max;               /* cache capacity in positions                                       */
    int32_t max_path;            /* width W of path / slot_map rows                                   */
    int64_t cache_layer_stride;  /* elements between consecutive layers of k_cache / v_cache          */
    int64_t tree_layer_stride;   /* elements between consecutive layers of tree_k / tree_v            */
    int64_t tree_node_stride;    /* elements between consecutive nodes of tree_k / tree_v; 0 = Hkv*D */
    void *k_cache;               /* [layers][B, Hkv, s_max, D]                                        */
    void *v_cache;               /* [layers][B, Hkv, s_max, D]                                        */
    const void *tree_k;          /* [layers][B, N, Hkv, D] node pitch tree_node_stride (rotated keys) */
    const void *tree_v;          /* [layers][B, N, Hkv, D] node pitch tree_node_stride                */
    const int32_t *path;         /* [B, W] from eagle3_accept                                         */
    const int32_t *accept_len;   /* [B]                                                               */
    int32_t *prefix_len;         /* [B] in: L; out: L + n + 1                                         */
    int32_t *slot_map;           /* [B, W] out                                                        */
    int32_t *committed;          /* [B] optional out: n + 1 positions committed (0 if skipped); this is
                                    the next draft catch-up row count                                */
    int32_t aux_dim;             /* A: elements per aux row; 0 = no aux gather                        */
    const void *aux_tree;        /* [B, N, A] (elem_bytes each) or NULL                               */
    void *aux_out;               /* [B, W, A] or NULL                                                 */
    int32_t *dev_status;         /* optional                                                          */
    /* Paged cache (as in eagle3_verify_attn): when block_table is set, each layer of k_cache /
       v_cache is a pool [n_slots, Hkv, D] (layers cache_layer_stride elements apart), position p of
       sequence b is slot block_table[b * max_blocks + p / block_size] * block_size + p % block_size,
       slot_map receives those slots, and a sequence fits when L + n + 1 <= max_blocks * block_size
       with every page id it writes inside [0, n_slots / block_size); s_max is then not used.     */
    const int32_t *block_table;  /* [B, max_blocks] page ids, or NULL (contiguous cache)               */
    int32_t max_blocks;          /* columns of block_table                                             */
    int32_t block_size;          /* positions per page, >= 1                                           */
    int32_t n_slots;             /* slots in each layer's pool                                         */
} eagle3_compact_args_t;

eagle3_status_t eagle3_compact_kv(const eagle3_compact_args_t *args, eagle3_stream_t stream);

/* ------------------------------------------------------------------------------------------------
 * eagle3_verify_attn - tree-masked verify attention for one layer (bf16, GQA, head_dim 128).
 *
 * Defines: "Advanced speculative decoding: tree drafts and EAGLE", sections "Why trees" and
 * "Implementation" (forward_with_mask: every node attends to the whole cached prefix and to the
 * tree nodes its mask row allows - itself and its ancestors - at position prefix_len + depth) and
 * "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", appendix C (rotate-half
 * RoPE with inv_j = theta^(-2j/D); grouped-query attention; scores scaled by sm_scale).
 *
 * For each sequence b (L = prefix_len[b]), node i and query head h (KV head g = h / (Hq/Hkv)):
 *   out[b,i,h] = sum_j softmax_j(q_i . k_j * sm_scale) v_j over keys j in
 *                {cache positions 0..L-1} U {tree nodes that are i or an ancestor of i}.
 * q and tree_k arrive un-rotated; the kernel applies RoPE at position L + depth(i) to both, and
 * writes the rotated tree keys back into tree_k (so eagle3_compact_kv copies rotated keys).  The
 * cache holds rotated keys.  fp32 softmax and accumulation; out in bf16.  lse (optional) gets the
 * natural-log sum of exp of the scaled scores.
 * The prefix is split across CTAs (split-KV) by a plan made from max_prefix_len (a host bound on
 * every prefix_len[b]); partial results are merged by a second kernel in a fixed order.
 * Cache slots at positions >= prefix_len are read in whole 128-key tiles and multiplied by a zero
 * weight, so they must hold finite values (zero-initialise a cache once; compaction only ever
 * writes finite rows).
 * Node pitches let q / tree_k / tree_v be views into one fused QKV projection output
 * [B * N, (Hq + 2 Hkv) * D]; rotating tree_k twice (calling twice on the same buffers) rotates the
 * keys twice, so each verify pass must start from freshly projected keys.
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t batch;              /* B >= 0                                                             */
    int32_t n_nodes;            /* N in [1, 64]                                                       */
    int32_t n_heads;            /* Hq, a multiple of n_kv_heads                                       */
    int32_t n_kv_heads;         /* Hkv                                                                */
    int32_t head_dim;           /* D; 128 is supported                                                */
    int32_t s_max;              /* cache capacity; max_prefix_len + N <= s_max is required            */
    int32_t max_prefix_len;     /* host bound on prefix_len[b]                                        */
    int32_t num_splits;         /* 0 = choose automatically                                           */
    int64_t q_node_stride;      /* elements between consecutive nodes of q; 0 = Hq * D (dense)        */
    int64_t kv_node_stride;     /* elements between consecutive nodes of tree_k / tree_v; 0 = Hkv * D */
    float rope_theta;           /* e.g. 500000                                                        */
    float sm_scale;             /* 0 = 1/sqrt(D)                                                      */
    const uint16_t *q;          /* [B, N, Hq, D] bf16 (node pitch q_node_stride), un-rotated           */
    uint16_t *tree_k;           /* [B, N, Hkv, D] bf16 (node pitch kv_node_stride), rotated in place   */
    const uint16_t *tree_v;     /* [B, N, Hkv, D] bf16 (node pitch kv_node_stride)                    */
    const uint16_t *k_cache;    /* [B, Hkv, s_max, D] bf16, rotated keys                              */
    const uint16_t *v_cache;    /* [B, Hkv, s_max, D] bf16                                            */
    const int32_t *parents;     /* [B, N]                                                             */
    const int32_t *prefix_len;  /* [B]                                                                */
    uint16_t *out;              /* [B, N, Hq, D] bf16                                                 */
    float *lse;                 /* [B, N, Hq] fp32 or NULL                                            */
    int32_t *dev_status;        /* optional                                                           */
    int32_t qk_rotated;         /* 1: q and tree_k arrive already rotated at prefix_len + depth (e.g.
                                   from eagle3_linear's EAGLE3_EPI_BF16_ROPE); neither is rotated
                                   again and tree_k is not written.  Needs (Hq / Hkv) to divide 128
                                   and a q node pitch of whole 16 bytes (else EAGLE3_ERR_UNSUPPORTED) */
    /* Paged cache ("Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", "EagleProposer:
       Draft Model Management": slot = block_table[pos / block_size] * block_size + pos % block_size).
       When block_table is set, k_cache / v_cache are a pool of n_slots slots of [Hkv, D] each
       ([n_slots, Hkv, D] bf16, n_slots = pages * block_size) and position p of sequence b is slot
       block_table[b * max_blocks + p / block_size] * block_size + p % block_size; s_max is then not
       used.  block_size must be a multiple of 64 and max_blocks * block_size >= max_prefix_len.
       Only the entries of positions < prefix_len[b] are read; page ids outside [0, n_slots /
       block_size) read as zeros.                                                              */
    const int32_t *block_table;  /* [B, max_blocks] page ids, or NULL (contiguous cache)               */
    int32_t max_blocks;          /* columns of block_table                                             */
    int32_t block_size;          /* positions per page                                                 */
    int32_t n_slots;             /* slots in the pool                                                  */
} eagle3_verify_attn_args_t;

size_t eagle3_verify_attn_workspace_size(const eagle3_verify_attn_args_t *args);
eagle3_status_t eagle3_verify_attn(const eagle3_verify_attn_args_t *args, void *workspace,
                                   size_t workspace_bytes, eagle3_stream_t stream);

/* eagle3_verify_attn_noalloc - eagle3_verify_attn for callers that cannot allocate device memory.
 * The pages have no counterpart: this exists for callers whose device memory is all handed to
 * another owner (a serving runtime's preallocated pool, a process that must not call cudaMalloc
 * while a step is being captured into a CUDA graph), so they cannot provide a workspace.
 * Same arguments, semantics and results as eagle3_verify_attn; the split-KV partials go to a
 * 32 MiB scratch array that the library places in device memory (every GPU that loads the library
 * holds it until the process exits).  The call allocates nothing: no cudaMalloc / cudaFree.
 *  - The first call on each device looks up the scratch address (cudaGetSymbolAddress) with that
 *    device current; make that first call before any stream capture.  The address is kept per
 *    device together with the CUDA context it was looked up in; after cudaDeviceReset (or any
 *    other destruction of that context) the next call looks it up again, so that call too should
 *    come before any stream capture.
 *  - A split plan that needs more than 32 MiB (batch * n_nodes * n_heads * splits * 520 bytes)
 *    returns EAGLE3_ERR_WORKSPACE before launching; pass a smaller num_splits to fit.
 *  - All calls share the one scratch array: calls that can overlap on the GPU (different streams,
 *    no ordering between them) race on it.  Nothing in it needs to start at zero: every partial
 *    is written before it is read, and a call never reads an earlier call's contents. */
eagle3_status_t eagle3_verify_attn_noalloc(const eagle3_verify_attn_args_t *args, eagle3_stream_t stream);


/* ------------------------------------------------------------------------------------------------
 * eagle3_draft_tree - EAGLE-3 draft head and its dynamic top-k draft tree.
 *
 * Defines: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections VIII-IX
 * (fc: bias-free Linear(3d -> d) fusing the three aux target states of a committed position;
 * one decoder layer over two streams - input_norm(e) and hidden_norm(x) concatenated to 2d feed
 * q/k/v, the residual stream is x, SwiGLU MLP - then final norm and LM head; the embedding is the
 * target's), section XI (catch-up of committed positions (g_i, e_{t_{i+1}}) into the draft cache,
 * then drafting rows (a, e_token) one position further per depth), sections IV.3 / XI.6 and
 * "EAGLE-3: Training-Time Test for Speculative Decoding", "Dynamic Draft Trees" (expand, then
 * rerank by cumulative log-probability).
 *
 * One call: (1) catch-up: rows i < tc[b] of sequence b are (g = fc(aux[b,i]), e = embed[next_tokens
 * [b,i]]) at positions draft_len[b] + i, causal over the draft cache; their rotated K/V are
 * appended to the draft cache and draft_len[b] += tc[b] (= L, the target prefix length).  The last
 * catch-up row (whose token is the root) gives the depth-1 logits.  (2) depth t = 2..depth: the
 * top_k best depth-(t-1) candidates (score desc, creation asc) each run one draft row (x = a of its
 * parent's row, e = its token) at position L - 1 + (t - 1), attending to the draft cache, to its
 * ancestors' rows and to itself; each row's top_k tokens become candidates with score = parent
 * score + logq (ties in top-k go to the lower token id).  logq is the deterministic fixed-point
 * log-softmax at T = 1 (see eagle3_accept).  (3) the n_nodes - 1 best candidates by (score desc,
 * depth asc, creation asc) - ancestor-closed - are emitted after the root in (depth asc, score
 * desc, creation asc) order, with creation = frontier rank * top_k + child rank.
 * Weights are bf16 [out, in]; q/k/v rows are stacked in w_qkv ((Hq + 2 Hkv) * D rows).  head_dim
 * 128; top_k <= 16; (depth - 1) * top_k <= 64; n_nodes - 1 <= top_k + (depth - 1) * top_k^2.
 *
 * Reduced draft vocabulary ("EAGLE-3: Engineering Implementation of LLM Inference Acceleration",
 * sections VIII.5-VIII.6: the draft's own LM head projects onto a subset of Vd target tokens, and
 * a draft-to-target map gives each draft id its target id): with draft_vocab = Vd > 0 and d2t set,
 * lm_head is [Vd, d], top-k and logq run over the Vd draft logits (ties to the lower draft id) and
 * every candidate token is d2t[draft id], a target id; d2t holds the subset's target ids in
 * increasing order.  A mapped id outside [0, vocab) sets EAGLE3_DEV_BAD_TOKEN.  For SAMPLED
 * acceptance, scatter the draft logits into the target vocabulary with -inf elsewhere (those
 * tokens then have q = 0).
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    const uint16_t *w_fc;        /* [d, 3d]                                                          */
    const uint16_t *embed;       /* [V, d] token embedding (the target's table)                      */
    const uint16_t *input_norm;  /* [d] RMSNorm weight of the embedding stream                       */
    const uint16_t *hidden_norm; /* [d] RMSNorm weight of the feature stream                         */
    const uint16_t *w_qkv;       /* [(Hq + 2 Hkv) * D, 2d]                                           */
    const uint16_t *w_o;         /* [d, Hq * D]                                                      */
    const uint16_t *post_norm;   /* [d]                                                              */
    const uint16_t *w_gate;      /* [F, d]                                                           */
    const uint16_t *w_up;        /* [F, d]                                                           */
    const uint16_t *w_down;      /* [d, F]                                                           */
    const uint16_t *final_norm;  /* [d]                                                              */
    const uint16_t *lm_head;     /* [V, d], or [Vd, d] with a reduced draft vocabulary               */
} eagle3_draft_weights_t;

typedef struct {
    int32_t batch;               /* B                                                                */
    int32_t hidden;              /* d                                                                */
    int32_t n_heads, n_kv_heads, head_dim;   /* Hq, Hkv, D (= 128)                                    */
    int32_t ffn;                 /* F                                                                */
    int32_t vocab;               /* V                                                                */
    int32_t depth;               /* tree depth (>= 1)                                                */
    int32_t top_k;               /* children per expanded node (1..16)                               */
    int32_t n_nodes;             /* nodes emitted including the root (2..64)                         */
    int32_t tc_max;              /* catch-up rows per sequence in aux / next_tokens (1..64)          */
    int32_t s_max;               /* draft cache capacity                                             */
    int32_t max_draft_len;       /* host bound on draft_len[b]; max_draft_len + tc_max <= s_max      */
    float rope_theta;            /* e.g. 500000                                                      */
    float rms_eps;               /* e.g. 1e-5                                                        */
    const uint16_t *aux;         /* [B, tc_max, 3d] bf16 aux target states of the committed positions */
    const int32_t *next_tokens;  /* [B, tc_max]: token after each committed position; row tc[b]-1 holds the root */
    const int32_t *tc;           /* [B] catch-up rows per sequence, 1..tc_max                        */
    uint16_t *draft_k_cache;     /* [B, Hkv, s_max, D] bf16, rotated keys                            */
    uint16_t *draft_v_cache;     /* [B, Hkv, s_max, D] bf16                                          */
    int32_t *draft_len;          /* [B] in: cached positions; out: + tc[b]                           */
    int32_t *tokens;             /* [B, n_nodes] out: node tokens (node 0 = root)                    */
    int32_t *parents;            /* [B, n_nodes] out                                                 */
    int32_t *depth_out;          /* [B, n_nodes] out                                                 */
    uint64_t *anc_mask;          /* [B, n_nodes] out: bit j set <=> node j is the node or an ancestor */
    float *score;                /* [B, n_nodes] out: cumulative logq (root 0)                       */
    float *dbg_logits;           /* optional [depth, top_k * B, Vd] fp32: every draft row's logits;
                                    depth 1 uses rows 0..B-1 (row b), depth t rows r * B + b for
                                    frontier rank r; may be NULL                                    */
    int32_t *dev_status;         /* optional                                                         */
    int32_t draft_vocab;         /* Vd: rows of lm_head, 1..V; 0 = V (no reduced vocabulary)          */
    const int32_t *d2t;          /* [Vd] target id of each draft id, or NULL (identity; Vd must be V) */
} eagle3_draft_tree_args_t;

size_t eagle3_draft_tree_workspace_size(const eagle3_draft_tree_args_t *args);
eagle3_status_t eagle3_draft_tree(const eagle3_draft_weights_t *weights, const eagle3_draft_tree_args_t *args,
                                  void *workspace, size_t workspace_bytes, eagle3_stream_t stream);

/* ------------------------------------------------------------------------------------------------
 * eagle3_rmsnorm - RMSNorm rows (building block of the target layers that verify a tree).
 *
 * Defines: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", appendix C (RMSNorm:
 * w * x * rsqrt(mean(x^2) + eps), statistics in fp32) and section IX.6 / "Speculative Decoding
 * (EAGLE3) in the vLLM Neuron Framework", "Auxiliary Hidden State Extraction" (the aux taps are the
 * hidden states entering a decoder layer, i.e. the input of its first norm).
 * out[r] = w * norm(in[src(r)]), src(r) = gather[r] when gather is given (an embedding lookup:
 * `in` is then the [V, d] table and gather holds token ids) else r.  When tap_out is given, the
 * un-normalised input row is also copied to tap_out[r] (pitch ld_tap).  bf16 in / out.
 * ---------------------------------------------------------------------------------------------- */
typedef struct {
    int32_t rows, dim;
    int32_t n_src;               /* rows of `in` (for gather bounds); 0 = rows                       */
    float eps;
    int64_t ld_in, ld_out, ld_tap;   /* pitches in elements, 0 = dim                                 */
    const uint16_t *in;
    const uint16_t *w;           /* [dim]                                                            */
    const int32_t *gather;       /* [rows] or NULL                                                   */
    uint16_t *out;
    uint16_t *tap_out;           /* or NULL                                                          */
    int32_t *dev_status;
} eagle3_rmsnorm_args_t;

eagle3_status_t eagle3_rmsnorm(const eagle3_rmsnorm_args_t *args, eagle3_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE3_H */
