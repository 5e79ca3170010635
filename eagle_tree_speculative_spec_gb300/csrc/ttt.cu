// eagle3_ttt_attn: the training-time-test attention of the EAGLE-3 draft layer.
//
// Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections VII.5
// (Figure 6: the native step is causal, every simulated step contributes only the key at the
// query's own position) and VIII.2 (forward_ttt: the diagonal scores are per-position dot
// products, concatenated to the causal scores under one softmax).
//
// Design: the causal part is tree attention (tree_attn_launch, the tcgen05 kernel behind
// eagle3_verify_attn).  The positions of a sequence are cut into chunks of C positions; chunk c is
// a "sequence" whose prefix is the native keys before it (64c positions, read through an identity
// block table over the native keys, so nothing is copied) and whose tree is the chain of its own C
// positions, with q and the keys taken as already rotated.  That kernel also returns each row's
// log-sum-exp; a second kernel, one warp per (position, head), computes the diagonal scores of the
// simulated steps and merges them into the causal result with an online softmax.
#include "attn.cuh"
#include "eagle3_ttt.h"

namespace e3 {
namespace {

constexpr int HD = 128;

int ttt_chunk(int rep) { return rep > 4 ? 256 / rep : 64; }

struct Geometry {
    int rep, C, chunks, max_blocks;
    int page;   // positions per page of the identity block table: 128 when T allows (whole-tile boxes), else 64
    size_t o_bt, o_par, o_pre, o_lse, o_attn, total;
};

Geometry geometry(const eagle3_ttt_attn_args_t *a) {
    Geometry g;
    g.rep = a->n_heads / a->n_kv_heads;
    g.C = ttt_chunk(g.rep);
    g.chunks = a->batch * (a->seq_len / g.C);
    g.page = a->seq_len % 128 == 0 ? 128 : 64;
    g.max_blocks = a->seq_len / g.page;
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t o = at;
        at += (bytes + 255) / 256 * 256;
        return o;
    };
    g.o_bt = take((size_t)g.chunks * g.max_blocks * 4);
    g.o_par = take((size_t)g.chunks * g.C * 4);
    g.o_pre = take((size_t)g.chunks * 4);
    g.o_lse = take((size_t)a->batch * a->seq_len * a->n_heads * 4);
    g.o_attn = at;
    g.total = at;
    return g;
}

// per chunk: identity block table over its sequence's native keys, a chain parent array, prefix 64 c
__global__ void ttt_setup_kernel(int T, int C, int max_blocks, int chunks, int32_t *bt, int32_t *par, int32_t *pre) {
    const int ch = blockIdx.x;
    if (ch >= chunks) return;
    const int per_seq = T / C, b = ch / per_seq, c = ch % per_seq;
    for (int j = threadIdx.x; j < max_blocks; j += blockDim.x) bt[(size_t)ch * max_blocks + j] = b * max_blocks + j;
    for (int n = threadIdx.x; n < C; n += blockDim.x) par[(size_t)ch * C + n] = n - 1;
    if (threadIdx.x == 0) pre[ch] = c * C;
}

struct MergeParams {
    int rows;                        // Bt * T * Hq (position-major, heads inner)
    int Hq, Hkv, rep, S;
    int64_t step_stride;             // elements between steps of k / v
    float scale;
    const __nv_bfloat16 *q, *k, *v;
    __nv_bfloat16 *out;              // in: causal result; out: merged
    const float *lse;                // natural-log sum of exp of the causal scores
};

E3_DEV float4 ld_bf16x4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// one warp per (position, head): lane l holds dimensions 4l..4l+3
__global__ void ttt_merge_kernel(const MergeParams m) {
    pdl_wait();
    pdl_trigger();
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= m.rows) return;
    const int h = w % m.Hq, pos = w / m.Hq, g = h / m.rep;
    const size_t qoff = (size_t)w * HD + 4 * lane;
    const float4 q = ld_bf16x4(m.q + qoff);
    const float4 o = ld_bf16x4(m.out + qoff);
    float M = m.lse[w];                 // the causal part enters with weight exp(lse)
    float den = 1.0f;
    float4 num = o;
    for (int s = 1; s < m.S; ++s) {
        const size_t koff = (size_t)s * m.step_stride + ((size_t)pos * m.Hkv + g) * HD + 4 * lane;
        const float4 k = ld_bf16x4(m.k + koff);
        float d = q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w;
#pragma unroll
        for (int x = 16; x; x >>= 1) d += __shfl_xor_sync(0xffffffffu, d, x);
        d *= m.scale;
        if (d > M) {                    // online softmax: rescale what is there
            const float c = __expf(M - d);
            num.x *= c;
            num.y *= c;
            num.z *= c;
            num.w *= c;
            den *= c;
            M = d;
        }
        const float e = __expf(d - M);
        const float4 v = ld_bf16x4(m.v + koff);
        num.x += e * v.x;
        num.y += e * v.y;
        num.z += e * v.z;
        num.w += e * v.w;
        den += e;
    }
    const float inv = 1.0f / den;
    __nv_bfloat162 lo = __floats2bfloat162_rn(num.x * inv, num.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(num.z * inv, num.w * inv);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&lo);
    u.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(m.out + qoff) = u;
}

eagle3_status_t ttt_validate(const eagle3_ttt_attn_args_t *a) {
    if (!a || a->batch < 0 || a->seq_len < 1 || a->n_heads < 1 || a->n_kv_heads < 1 || a->n_steps < 1 ||
        a->sm_scale < 0.0f || a->n_heads % a->n_kv_heads)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    const int rep = a->n_heads / a->n_kv_heads;
    if (a->head_dim != HD || (rep != 1 && rep != 2 && rep != 4 && rep != 8) || a->seq_len % 64)
        return EAGLE3_ERR_UNSUPPORTED;
    if (a->batch == 0) return EAGLE3_OK;
    const void *ptrs[] = {a->q, a->k, a->v, a->out};
    for (const void *p : ptrs)
        if (!p || ((uintptr_t)p & 15)) return EAGLE3_ERR_INVALID_ARGUMENT;
    return EAGLE3_OK;
}

AttnLaunch causal_launch(const eagle3_ttt_attn_args_t *a, const Geometry &g, uint8_t *ws) {
    AttnLaunch l;
    const int T = a->seq_len, Hq = a->n_heads, Hkv = a->n_kv_heads;
    l.B = g.chunks;
    l.n_slots = g.C;
    l.q_lo = 0;
    l.q_hi = g.C;
    l.Hq = Hq;
    l.Hkv = Hkv;
    l.S = 0;
    l.max_prefix = T - g.C;
    l.num_splits = 0;
    l.rope_theta = 10000.0f;   // not used: q and the keys arrive rotated
    l.sm_scale = a->sm_scale > 0.0f ? a->sm_scale : 1.0f / sqrtf((float)HD);
    l.q = (const __nv_bfloat16 *)a->q;
    l.q_si = (int64_t)Hq * HD;
    l.q_sb = l.q_si * g.C;
    l.k = (__nv_bfloat16 *)a->k;   // read only: with rotated keys the kernel writes nothing back
    l.k_si = (int64_t)Hkv * HD;
    l.k_sb = l.k_si * g.C;
    l.v = (const __nv_bfloat16 *)a->v;
    l.v_si = l.k_si;
    l.v_sb = l.k_sb;
    l.out = (__nv_bfloat16 *)a->out;
    l.o_si = l.q_si;
    l.o_sb = l.q_sb;
    l.k_cache = (const __nv_bfloat16 *)a->k;   // step 0 as a pool of Bt * T slots
    l.v_cache = (const __nv_bfloat16 *)a->v;
    l.parents = ws ? (const int32_t *)(ws + g.o_par) : nullptr;
    l.anc = nullptr;
    l.pos = nullptr;
    l.anc_sb = l.pos_sb = 0;
    l.prefix_len = ws ? (const int32_t *)(ws + g.o_pre) : nullptr;
    l.lse = ws ? (float *)(ws + g.o_lse) : nullptr;
    l.dev_status = a->dev_status;
    l.qk_rotated = 1;
    l.block_table = ws ? (const int32_t *)(ws + g.o_bt) : (const int32_t *)nullptr;
    l.bt_stride = g.max_blocks;
    l.block_size = g.page;
    l.pool_slots = a->batch * T;
    return l;
}

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" size_t eagle3_ttt_attn_workspace_size(const eagle3_ttt_attn_args_t *a) {
    if (ttt_validate(a) != EAGLE3_OK || a->batch == 0) return 0;
    const Geometry g = geometry(a);
    return g.total + tree_attn_workspace(causal_launch(a, g, nullptr)) + 256;
}

extern "C" eagle3_status_t eagle3_ttt_attn(const eagle3_ttt_attn_args_t *a, void *workspace, size_t ws_bytes,
                                           eagle3_stream_t stream_) {
    const eagle3_status_t st = ttt_validate(a);
    if (st != EAGLE3_OK || a->batch == 0) return st;
    const Geometry g = geometry(a);
    if (!workspace || ws_bytes < eagle3_ttt_attn_workspace_size(a)) return EAGLE3_ERR_WORKSPACE;
    uint8_t *ws = (uint8_t *)(((uintptr_t)workspace + 255) & ~(uintptr_t)255);
    cudaStream_t stream = (cudaStream_t)stream_;
    ttt_setup_kernel<<<g.chunks, 64, 0, stream>>>(a->seq_len, g.C, g.max_blocks, g.chunks, (int32_t *)(ws + g.o_bt),
                                                  (int32_t *)(ws + g.o_par), (int32_t *)(ws + g.o_pre));
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    const AttnLaunch l = causal_launch(a, g, ws);
    const size_t attn_ws = ws_bytes - (size_t)(ws - (uint8_t *)workspace) - g.o_attn;
    const eagle3_status_t s2 = tree_attn_launch(l, ws + g.o_attn, attn_ws, stream);
    if (s2 != EAGLE3_OK) return s2;
    if (a->n_steps > 1) {
        MergeParams m;
        m.rows = a->batch * a->seq_len * a->n_heads;
        m.Hq = a->n_heads;
        m.Hkv = a->n_kv_heads;
        m.rep = g.rep;
        m.S = a->n_steps;
        m.step_stride = (int64_t)a->batch * a->seq_len * a->n_kv_heads * HD;
        m.scale = l.sm_scale;
        m.q = (const __nv_bfloat16 *)a->q;
        m.k = (const __nv_bfloat16 *)a->k;
        m.v = (const __nv_bfloat16 *)a->v;
        m.out = (__nv_bfloat16 *)a->out;
        m.lse = (const float *)(ws + g.o_lse);
        if (launch_pdl(ttt_merge_kernel, dim3((unsigned)((m.rows + 3) / 4)), dim3(128), 0, stream, m) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}
