// Internal interface of the tree-attention kernel shared by eagle3_verify_attn and the draft head.
#pragma once

#include "common.cuh"

namespace e3 {

// Tree attention over a cached prefix plus tree slots.  Query slots [q_lo, q_hi) attend to the
// prefix keys 0..prefix_len[b]-1 and to the slots j < q_hi whose bit is set in anc[i]; their
// keys are rotated in place (slots below q_lo hold keys rotated by an earlier call).  Either
// `parents` (slot 0 the root, positions prefix_len + depth) or (`anc`, `pos`) describe the slots.
// Element (b, slot i, head h) of q / k / v lives at base + b * sb + i * si + h * 128; output row
// of query slot i at out + b * o_sb + (i - q_lo) * o_si + h * 128.
struct AttnLaunch {
    int B, n_slots, q_lo, q_hi, Hq, Hkv, S, max_prefix, num_splits;
    float rope_theta, sm_scale;
    const __nv_bfloat16 *q;
    int64_t q_sb, q_si;
    __nv_bfloat16 *k;
    int64_t k_sb, k_si;
    const __nv_bfloat16 *v;
    int64_t v_sb, v_si;
    __nv_bfloat16 *out;
    int64_t o_sb, o_si;
    const __nv_bfloat16 *k_cache, *v_cache;
    const int32_t *parents;
    const uint64_t *anc;
    const int32_t *pos;
    int anc_sb, pos_sb;
    const int32_t *prefix_len;
    float *lse;
    int32_t *dev_status;
    int qk_rotated = 0;              // q and the tree keys arrive rotated (no RoPE, no tree_k write)
    // bounded waits give up after this many clocks; a test of the timeout path shortens it
    long long wait_limit = WAIT_LIMIT_CYCLES;
    // test of the timeout path only: the K producer never loads this prefix tile (local index
    // within the CTA's split), so the wait for it runs out; -1 = off
    int stall_tile = -1;
    // paged cache: k_cache / v_cache are a pool [n_slots, Hkv, 128]; position p of sequence b is
    // slot block_table[b * bt_stride + p / block_size] * block_size + p % block_size (64 | block_size);
    // pool_slots = slots in the pool
    const int32_t *block_table = nullptr;
    int bt_stride = 0, block_size = 0, pool_slots = 0;
};

size_t tree_attn_workspace(const AttnLaunch &a);
eagle3_status_t tree_attn_launch(const AttnLaunch &a, void *workspace, size_t ws_bytes, cudaStream_t stream);

}  // namespace e3
