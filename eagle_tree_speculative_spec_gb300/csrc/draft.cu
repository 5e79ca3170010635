// eagle3_draft_tree: the EAGLE-3 draft head and its dynamic top-k tree; eagle3_rmsnorm.
//
// Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections VIII
// (two-stream draft decoder layer, frozen embedding, final norm + LM head, pre-norm recurrent
// state), IX (fc over the concatenated aux states), XI (catch-up, drafting positions, cache
// rollback), IV.3 / XI.6 (EAGLE-2 dynamic tree: expand by draft confidence, prune at the end) and
// appendix C (RMSNorm, RoPE); "EAGLE-3: Training-Time Test for Speculative Decoding", "Dynamic
// Draft Trees Spend Verification Where It Can Pay Off"; "Advanced speculative decoding: tree
// drafts and EAGLE" (top-k children per node, node 0 is the root).
//
// Data flow of one call (rows of a draft step are ordered rank-major, row = r * B + b, so the rows
// of one depth are one contiguous block and each projection is a single tensor-core GEMM):
//   catch-up   fc GEMM -> prologue (two RMSNorms, concat) -> QKV GEMM -> tree attention (chain
//              over the draft cache) -> O GEMM (+x) -> RMSNorm -> SwiGLU GEMM -> down GEMM (+x1)
//              -> append rotated K/V to the draft cache -> final RMSNorm of the root row -> LM
//              head (fp32 logits) -> row top-k + fixed-point log-normaliser -> candidates
//   depth 2..D the same layer for the top_k frontier rows of the previous depth, attending to the
//              draft cache plus their ancestors' rows in a K/V pool; selection of the next frontier
//   final      rerank of all candidates, emission of tokens / parents / depth / masks / scores
// Every selection decision compares fp32 scores built with the same RN operations as the CPU
// oracle, so for the same logits the tree is bit-identical.
#include <algorithm>
#include <cooperative_groups.h>

#include "../../include/eagle3_linear.h"
#include "attn.cuh"
#include "tc.cuh"

namespace e3 {
namespace {

constexpr int KMAX = 16;
constexpr int HD = 128;
constexpr int MAX_SLOTS = 64;

// ------------------------------------------------------------------------------------------------
// RMSNorm helpers: one CTA of 128 threads per row.
// ------------------------------------------------------------------------------------------------
constexpr int NT_NORM = 128;

E3_DEV float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    return t;
}

// out = w * x * rsqrt(mean(x^2) + eps), fp32 statistics, bf16 out
E3_DEV void norm_row(const __nv_bfloat16 *x, const __nv_bfloat16 *w, __nv_bfloat16 *out, int dim, float eps,
                     __nv_bfloat16 *tap, float *red) {
    float ss = 0.0f;
    for (int i = threadIdx.x; i < dim; i += blockDim.x) {
        const float v = __bfloat162float(x[i]);
        ss += v * v;
    }
    const float r = rsqrtf(block_sum(ss, red) / (float)dim + eps);
    for (int i = threadIdx.x; i < dim; i += blockDim.x) {
        const __nv_bfloat16 xv = x[i];
        out[i] = __float2bfloat16_rn(__bfloat162float(w[i]) * (__bfloat162float(xv) * r));
        if (tap) tap[i] = xv;
    }
}

// Vectorised variant: the row is read once with 16-byte loads (CH chunks of 8 values per thread),
// kept in registers for the scale pass.  Needs dim % 8 == 0 and 16-byte aligned rows.
template <int CH>
E3_DEV void norm_row_vec(const __nv_bfloat16 *x, const __nv_bfloat16 *w, __nv_bfloat16 *out, int dim, float eps,
                         __nv_bfloat16 *tap, float *red) {
    const int nchunk = dim >> 3;
    uint4 xv[CH];
    float ss = 0.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int ch = threadIdx.x + c * (int)blockDim.x;
        if (ch < nchunk) {
            xv[c] = *reinterpret_cast<const uint4 *>(x + ch * 8);
            const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&xv[c]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float v = __bfloat162float(h[e]);
                ss += v * v;
            }
        }
    }
    const float r = rsqrtf(block_sum(ss, red) / (float)dim + eps);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int ch = threadIdx.x + c * (int)blockDim.x;
        if (ch < nchunk) {
            const uint4 wv = *reinterpret_cast<const uint4 *>(w + ch * 8);
            const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(&xv[c]);
            const __nv_bfloat16 *wh = reinterpret_cast<const __nv_bfloat16 *>(&wv);
            uint4 o;
            __nv_bfloat16 *oh = reinterpret_cast<__nv_bfloat16 *>(&o);
#pragma unroll
            for (int e = 0; e < 8; ++e) oh[e] = __float2bfloat16_rn(__bfloat162float(wh[e]) * (__bfloat162float(h[e]) * r));
            *reinterpret_cast<uint4 *>(out + ch * 8) = o;
            if (tap) *reinterpret_cast<uint4 *>(tap + ch * 8) = xv[c];
        }
    }
}

// chooses the vector path when the row and its pointers allow it
E3_DEV void norm_row_any(const __nv_bfloat16 *x, const __nv_bfloat16 *w, __nv_bfloat16 *out, int dim, float eps,
                         __nv_bfloat16 *tap, float *red) {
    const bool vec = (dim % 8 == 0) &&
                     (((uintptr_t)x | (uintptr_t)w | (uintptr_t)out | (uintptr_t)(tap ? tap : out)) & 15) == 0;
    const int per = (dim / 8 + (int)blockDim.x - 1) / (int)blockDim.x;
    if (vec && per <= 1) norm_row_vec<1>(x, w, out, dim, eps, tap, red);
    else if (vec && per <= 2) norm_row_vec<2>(x, w, out, dim, eps, tap, red);
    else if (vec && per <= 4) norm_row_vec<4>(x, w, out, dim, eps, tap, red);
    else if (vec && per <= 8) norm_row_vec<8>(x, w, out, dim, eps, tap, red);
    else norm_row(x, w, out, dim, eps, tap, red);
}

struct NormParams {
    int rows, dim, n_src;
    float eps;
    int64_t ld_in, ld_out, ld_tap;
    const __nv_bfloat16 *in, *w;
    const int32_t *gather;
    __nv_bfloat16 *out, *tap;
    int32_t *dev_status;
};

__global__ void __launch_bounds__(NT_NORM) rmsnorm_kernel(const NormParams p) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[NT_NORM / 32];
    const int r = blockIdx.x;
    int src = p.gather ? p.gather[r] : r;
    if (src < 0 || src >= p.n_src) {
        if (threadIdx.x == 0) flag(p.dev_status, EAGLE3_DEV_BAD_TOKEN);
        src = 0;
    }
    norm_row_any(p.in + (size_t)src * p.ld_in, p.w, p.out + (size_t)r * p.ld_out, p.dim, p.eps,
                 p.tap ? p.tap + (size_t)r * p.ld_tap : nullptr, red);
}

// Draft prologue: a2k[r] = [input_norm(embed[tok[r]]) ; hidden_norm(x[r])], optionally x copied
// to xres[r].  Catch-up rows past tc[b] use token 0 (their outputs are never read).
struct PrologueParams {
    int rows, d, vocab, tc_max;
    float eps;
    const __nv_bfloat16 *embed, *w_in, *w_hid;
    const int32_t *tokens;         // [rows]
    const int32_t *tc;             // catch-up validity (rows = b * tc_max + i) or null
    const __nv_bfloat16 *x;        // x rows base
    const int32_t *x_row;          // [rows] absolute row of x, or null (row r)
    __nv_bfloat16 *a2k, *xres;
    int32_t *dev_status;
};

__global__ void __launch_bounds__(NT_NORM) draft_prologue_kernel(const PrologueParams p) {
    __shared__ float red[NT_NORM / 32];
    const int r = blockIdx.x;
    int tok = p.tokens[r];
    bool valid = true;
    if (p.tc) valid = (r % p.tc_max) < p.tc[r / p.tc_max];
    if (!valid) tok = 0;
    if (tok < 0 || tok >= p.vocab) {
        if (threadIdx.x == 0) flag(p.dev_status, EAGLE3_DEV_BAD_TOKEN);
        tok = 0;
    }
    const __nv_bfloat16 *x = p.x + (size_t)(p.x_row ? p.x_row[r] : r) * p.d;
    __nv_bfloat16 *o = p.a2k + (size_t)r * 2 * p.d;
    norm_row_any(p.embed + (size_t)tok * p.d, p.w_in, o, p.d, p.eps, nullptr, red);
    norm_row_any(x, p.w_hid, o + p.d, p.d, p.eps, p.xres ? p.xres + (size_t)r * p.d : nullptr, red);
}

// ------------------------------------------------------------------------------------------------
// Row top-k (k <= 16) by (logit desc, token asc) and the fixed-point log-normaliser at T = 1.
// ------------------------------------------------------------------------------------------------
constexpr int NT_TOPK = 256;      // threads per CTA, cluster kernel and one-wave row counts
constexpr int NT_TOPK_NARROW = 128; // threads per CTA when the rows overflow one wave of NT_TOPK CTAs

E3_DEV uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const uint64_t t = __shfl_xor_sync(0xffffffffu, v, o);
        v = t > v ? t : v;
    }
    return v;
}

// merge the 32 sorted lists held by the lanes into the top-k of their union (all lanes get it)
E3_DEV void warp_merge(uint64_t (&best)[KMAX], uint64_t (&res)[KMAX], int k) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        const uint64_t m = warp_max_u64(best[0]);
        res[j] = j < k ? m : 0ull;
        if (best[0] == m && m != 0ull) {   // packed values are unique: exactly one lane pops
#pragma unroll
            for (int q = 0; q < KMAX - 1; ++q) best[q] = best[q + 1];
            best[KMAX - 1] = 0ull;
        }
    }
}

E3_DEV void insert_best(uint64_t (&best)[KMAX], uint64_t v) {
    if (v <= best[KMAX - 1]) return;
#pragma unroll
    for (int q = 0; q < KMAX; ++q) {
        if (v > best[q]) {
            const uint64_t t = best[q];
            best[q] = v;
            v = t;
        }
    }
}

// Row top-k by (value desc, index asc) and the row's fixed-point normaliser.  One CTA per row, or
// a cluster of CTAs per row when rows are few.  Each warp keeps its current top-k in shared
// memory and the packed key of its k-th best as a threshold: an element below the threshold
// cannot enter the top-k, so it costs one compare (one per four elements: their NaN-propagating
// maximum); the rest are appended (ballot-compacted) to a per-warp buffer that is merged into the
// list only when it fills up.  For a row in random order about k ln(n / k) elements pass.  The
// normaliser pass weighs two elements per paired-fp32 instruction, bit-identical to one at a time.
constexpr int TK_CAP = 256;   // candidate buffer per warp (two float4 groups of a warp)

// merge a warp's candidate buffer into its list (KMAX entries, the first k meaningful); returns
// the new k-th best (0 while fewer than k candidates have been seen)
E3_DEV uint64_t warp_flush(uint64_t *list, const uint64_t *cand, int cnt, int k, int lane) {
    uint64_t best[KMAX];
#pragma unroll
    for (int q = 0; q < KMAX; ++q) best[q] = 0ull;
#pragma unroll
    for (int t = 0; t < (KMAX + TK_CAP + 31) / 32; ++t) {
        const int i = lane + 32 * t;
        if (i < KMAX + cnt) insert_best(best, i < KMAX ? list[i] : cand[i - KMAX]);
    }
    __syncwarp();
    uint64_t res[KMAX];
    warp_merge(best, res, k);
    if (lane == 0)
#pragma unroll
        for (int q = 0; q < KMAX; ++q) list[q] = res[q];
    __syncwarp();
    return list[k - 1];   // (selecting res[k - 1] in registers would demote res to local memory)
}

// max of four floats in two instructions, NaN if any is NaN
E3_DEV float max4_nan(float4 v) {
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(v.x), "f"(v.y), "f"(v.z));
    asm("max.NaN.f32 %0, %0, %1;" : "+f"(r) : "f"(v.w));
    return r;
}

template <int NT> struct TopkSmem {
    uint64_t buf[NT / 32][TK_CAP];
    uint64_t wres[NT / 32][KMAX];
    uint64_t fin[KMAX];
    uint64_t sred[NT / 32];
    uint64_t s_cta;                 // this CTA's share of the normaliser (cluster version)
};

// The CTA's warps' lists merged into sm.fin and the per-thread normaliser terms summed (the sum is
// returned, valid in thread 0)
template <int NT> E3_DEV uint64_t topk_finish(TopkSmem<NT> &sm, uint64_t s, int k) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sm.sred[warp] = s;
    __syncthreads();
    if (warp == 0) {
        uint64_t best[KMAX], res[KMAX];
#pragma unroll
        for (int q = 0; q < KMAX; ++q) best[q] = lane < NT / 32 ? sm.wres[lane][q] : 0ull;
        warp_merge(best, res, k);
        if (lane == 0)
#pragma unroll
            for (int q = 0; q < KMAX; ++q) sm.fin[q] = res[q];
    }
    uint64_t S = 0;
    if (threadIdx.x == 0)
        for (int w = 0; w < NT / 32; ++w) S += sm.sred[w];
    __syncthreads();
    return S;
}

// Top-k candidates of the slice [lo, hi) of row z into sm.fin (sorted, KMAX entries, the first k
// meaningful; 0 = none) and, in the same pass over the slice, its fixed-point normaliser terms with
// m = the row maximum (known beforehand: the LM head's epilogue published it): the CTA's sum is
// returned (valid in thread 0).
template <int NT> E3_DEV uint64_t topk_slice(TopkSmem<NT> &sm, const float *z, int lo, int hi, int k, float m) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    if (lane < KMAX) sm.wres[warp][lane] = 0ull;
    __syncwarp();
    uint64_t tau = 0ull;             // packed key of the warp's k-th best so far (0: fewer than k)
    float tau_f = key_to_float(0u);  // a NaN: every value passes `!(v < tau_f)`
    int cnt = 0;                     // warp-uniform fill of buf[warp]
    uint64_t s = 0;                  // normaliser terms of this thread's elements
    auto flush = [&]() {
        tau = warp_flush(sm.wres[warp], sm.buf[warp], cnt, k, lane);
        tau_f = key_to_float((uint32_t)(tau >> 32));
        cnt = 0;
    };
    // one element per lane: append it when it can still enter the top-k (all lanes call this)
    auto offer = [&](float v, uint32_t idx, bool valid) {
        bool pass = valid && !(v < tau_f);
        uint64_t key = 0ull;
        if (pass) {
            key = pack_argmax(v, idx);
            pass = key > tau;
        }
        const uint32_t msk = __ballot_sync(0xffffffffu, pass);
        if (pass) sm.buf[warp][cnt + __popc(msk & lt_mask)] = key;
        cnt += __popc(msk);
    };
    const float *zs = z + lo;
    const int n = hi - lo;
    const bool vec = ((((uintptr_t)zs) & 15) == 0);
    const int n4 = vec ? n / 4 : 0;
    constexpr int U = 4;   // float4 loads in flight per thread
    const int n4u = n4 / (U * NT) * (U * NT);   // float4 groups every lane has
    for (int j0 = threadIdx.x; j0 < n4u; j0 += U * NT) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = __ldg(reinterpret_cast<const float4 *>(zs) + j0 + u * NT);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            // each weight is up to 2^31: widen before adding
            const uint2 w01 = dsm_weight_pair(v[u].x, v[u].y, m, 1.0f), w23 = dsm_weight_pair(v[u].z, v[u].w, m, 1.0f);
            s += ((uint64_t)w01.x + w01.y) + ((uint64_t)w23.x + w23.y);
            // some element is not below the threshold <=> their maximum is not (a NaN propagates, and
            // passes, as it does element by element)
            const bool any = !(max4_nan(v[u]) < tau_f);
            if (!__any_sync(0xffffffffu, any)) continue;
            if (cnt + 4 * 32 > TK_CAP) flush();
            const uint32_t j = (uint32_t)lo + 4u * (uint32_t)(j0 + u * NT);
            offer(v[u].x, j, true);
            offer(v[u].y, j + 1, true);
            offer(v[u].z, j + 2, true);
            offer(v[u].w, j + 3, true);
        }
    }
    // the rest, one element per lane per round, with warp-uniform trip counts
    for (int base = 4 * n4u; base < n; base += NT) {
        const int i = base + threadIdx.x;
        const bool valid = i < n;
        const float v = valid ? __ldg(zs + i) : 0.0f;
        if (valid) s += dsm_weight(dsm_scaled(v, m, 1.0f));
        if (cnt + 32 > TK_CAP) flush();
        offer(v, (uint32_t)(lo + i), valid);
    }
    if (cnt > 0) flush();
    return topk_finish(sm, s, k);
}

// Output of a row's top-k: token ids (through the draft-to-target map when there is one) and logq.
struct TopkOut {
    int32_t *tok;
    float *lq;
    const int32_t *d2t;   // [V] target id of each draft id (V: the row length), or NULL
    int v_target;         // bound of the mapped ids
    int32_t *dev_status;
};

E3_DEV void topk_write(const uint64_t *fin, uint64_t S, float m, int row, int V, int k, const TopkOut &o) {
    if (threadIdx.x < k) {
        const float ln_s = dsm_log31(S);
        const uint64_t e = fin[threadIdx.x];
        const float zx = key_to_float((uint32_t)(e >> 32));
        const uint32_t idx = unpack_idx(e);
        int32_t tok = (int32_t)idx;
        if (o.d2t) {
            tok = idx < (uint32_t)V ? __ldg(o.d2t + idx) : -1;
            if (tok < 0 || tok >= o.v_target) flag(o.dev_status, EAGLE3_DEV_BAD_TOKEN);
        }
        o.tok[(size_t)row * k + threadIdx.x] = tok;
        o.lq[(size_t)row * k + threadIdx.x] = __fsub_rn(dsm_scaled(zx, m, 1.0f), ln_s);
    }
}

// One CTA of NT threads per row (many rows).  row_max[row] holds the order key of the row's maximum.
template <int NT>
__global__ void __launch_bounds__(NT)
    topk_kernel(const float *logits, int64_t ld, int V, int k, const uint32_t *row_max, const TopkOut o) {
    __shared__ TopkSmem<NT> sm;
    __shared__ uint64_t S;
    const int row = blockIdx.x;
    const float *z = logits + (size_t)row * ld;
    const float m = key_to_float(__ldg(row_max + row));
    const uint64_t s = topk_slice(sm, z, 0, V, k, m);
    if (threadIdx.x == 0) S = s;
    __syncthreads();
    topk_write(sm.fin, S, m, row, V, k, o);
}

// One CTA of NT threads per row, the row streamed through a shared-memory ring: thread 0 issues
// bulk copies of TKR_CHUNK-float chunks (TKR_STAGES in flight), every warp scans each chunk from
// shared memory as it lands.  The bytes in flight per CTA no longer depend on registers (the
// register-fed loop keeps four 16-byte loads per thread in flight), so a wave of rows streams
// at a higher rate.  Same selection and normaliser arithmetic as topk_slice, so the result is
// bit-identical.  Needs a row length and a row pitch that are multiples of 4 floats, 16-byte
// aligned logits.  All waits are bounded (EAGLE3_DEV_TIMEOUT, the CTA drains its copies).
constexpr int TKR_CHUNK = 2048;    // floats per stage (8 KB)
constexpr int TKR_STAGES = 4;
constexpr uint32_t TKR_RING_BYTES = TKR_STAGES * TKR_CHUNK * 4;

template <int NT>
__global__ void __launch_bounds__(NT)
    topk_ring_kernel(const float *logits, int64_t ld, int V, int k, const uint32_t *row_max, const TopkOut o) {
    extern __shared__ __align__(128) float ring[];   // [TKR_STAGES][TKR_CHUNK]
    __shared__ TopkSmem<NT> sm;
    __shared__ uint64_t full[TKR_STAGES], empty[TKR_STAGES];
    __shared__ uint64_t S;
    __shared__ int abort_flag;
    pdl_wait();
    pdl_trigger();
    volatile int *abort = &abort_flag;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int row = blockIdx.x;
    const float *z = logits + (size_t)row * ld;
    const float m = key_to_float(__ldg(row_max + row));
    const int nch = (V + TKR_CHUNK - 1) / TKR_CHUNK;
    auto chunk_len = [&](int c) { return min(TKR_CHUNK, V - c * TKR_CHUNK); };
    auto issue = [&](int c) {   // thread 0
        const int s = c % TKR_STAGES;
        const uint32_t bytes = (uint32_t)chunk_len(c) * 4u;
        tc::mbar_expect_tx(&full[s], bytes);
        tc::bulk_load(ring + (size_t)s * TKR_CHUNK, z + (size_t)c * TKR_CHUNK, bytes, &full[s]);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < TKR_STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], NT / 32);
        }
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (lane < KMAX) sm.wres[warp][lane] = 0ull;
    __syncthreads();
    int issued = 0;   // thread 0: chunks whose copy has been issued
    if (threadIdx.x == 0)
        for (; issued < min(nch, TKR_STAGES); ++issued) issue(issued);

    uint64_t tau = 0ull;
    float tau_f = key_to_float(0u);
    int cnt = 0;
    uint64_t s = 0;
    bool ok = true;
    auto flush = [&]() {
        tau = warp_flush(sm.wres[warp], sm.buf[warp], cnt, k, lane);
        tau_f = key_to_float((uint32_t)(tau >> 32));
        cnt = 0;
    };
    auto offer = [&](float v, uint32_t idx, bool valid) {
        bool pass = valid && !(v < tau_f);
        uint64_t key = 0ull;
        if (pass) {
            key = pack_argmax(v, idx);
            pass = key > tau;
        }
        const uint32_t msk = __ballot_sync(0xffffffffu, pass);
        if (pass) sm.buf[warp][cnt + __popc(msk & lt_mask)] = key;
        cnt += __popc(msk);
    };
    for (int c = 0; c < nch; ++c) {
        const int st = c % TKR_STAGES;
        const uint32_t ph = (uint32_t)(c / TKR_STAGES) & 1u;
        int got = 0;
        if (lane == 0) got = (ok && tc::mbar_wait(&full[st], ph, abort)) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) ok = false;
        const int n = chunk_len(c), n4 = n / 4;
        const float4 *src = reinterpret_cast<const float4 *>(ring + (size_t)st * TKR_CHUNK);
        if (ok) {
            // every lane of a warp runs the same number of rounds (the offers are warp-collective)
            for (int j0 = warp * 32; j0 < n4; j0 += NT) {
                const int j = j0 + lane;
                const bool valid = j < n4;
                const float4 v = valid ? src[j] : make_float4(0.f, 0.f, 0.f, 0.f);
                if (valid) {
                    const uint2 w01 = dsm_weight_pair(v.x, v.y, m, 1.0f), w23 = dsm_weight_pair(v.z, v.w, m, 1.0f);
                    s += ((uint64_t)w01.x + w01.y) + ((uint64_t)w23.x + w23.y);
                }
                const bool any = valid && !(max4_nan(v) < tau_f);
                if (!__any_sync(0xffffffffu, any)) continue;
                if (cnt + 4 * 32 > TK_CAP) flush();
                const uint32_t e = (uint32_t)(c * TKR_CHUNK) + 4u * (uint32_t)j;
                offer(v.x, e, valid);
                offer(v.y, e + 1, valid);
                offer(v.z, e + 2, valid);
                offer(v.w, e + 3, valid);
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[st]);
        // thread 0 refills the stage once every warp has scanned it
        if (threadIdx.x == 0 && issued < nch && issued == c + TKR_STAGES) {
            if (ok && tc::mbar_wait(&empty[st], ph, abort))
                issue(issued++);
            else
                ok = false;
        }
    }
    if (cnt > 0) flush();
    if (!ok && lane == 0) flag(o.dev_status, EAGLE3_DEV_TIMEOUT);
    if (threadIdx.x == 0) {   // no copy may still be in flight when the CTA exits
        for (int c = max(0, issued - TKR_STAGES); c < issued; ++c) {
            const long long t0 = clock64();
            while (!tc::mbar_try(&full[c % TKR_STAGES], (uint32_t)(c / TKR_STAGES) & 1u) &&
                   clock64() - t0 < WAIT_LIMIT_CYCLES) {
            }
        }
    }
    const uint64_t tot = topk_finish(sm, s, k);
    if (threadIdx.x == 0) S = tot;
    __syncthreads();
    topk_write(sm.fin, S, m, row, V, k, o);
}

// A cluster of TOPK_CL CTAs per row (few rows): CTA r scans slice r, the slices' top-k lists and
// normaliser sums are combined through distributed shared memory in rank order.
constexpr int TOPK_CL = 8;
__global__ void __cluster_dims__(TOPK_CL, 1, 1) __launch_bounds__(NT_TOPK)
    topk_cluster_kernel(const float *logits, int64_t ld, int V, int k, const uint32_t *row_max, const TopkOut o) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ TopkSmem<NT_TOPK> sm;
    __shared__ uint64_t fin_all[KMAX];
    const int rank = (int)cluster.block_rank(), row = blockIdx.x / TOPK_CL;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *z = logits + (size_t)row * ld;
    const float m = key_to_float(__ldg(row_max + row));
    const int slice = ((V + TOPK_CL - 1) / TOPK_CL + 3) / 4 * 4;   // a multiple of 4 elements
    const int lo = min(V, rank * slice), hi = min(V, lo + slice);
    const uint64_t s = topk_slice(sm, z, lo, hi, k, m);
    if (threadIdx.x == 0) sm.s_cta = s;
    cluster.sync();
    if (rank == 0) {
        if (warp == 0) {
            uint64_t best[KMAX], res[KMAX];
            const uint64_t *src = cluster.map_shared_rank(sm.fin, lane < TOPK_CL ? lane : 0);
#pragma unroll
            for (int q = 0; q < KMAX; ++q) best[q] = lane < TOPK_CL ? src[q] : 0ull;
            warp_merge(best, res, k);
            if (lane == 0)
#pragma unroll
                for (int q = 0; q < KMAX; ++q) fin_all[q] = res[q];
        }
        __shared__ uint64_t S;
        if (threadIdx.x == 0) {
            uint64_t t = 0;
            for (int r = 0; r < TOPK_CL; ++r) t += *cluster.map_shared_rank(&sm.s_cta, r);
            S = t;
        }
        __syncthreads();
        topk_write(fin_all, S, m, row, V, k, o);
    }
    cluster.sync();   // no CTA leaves while its shared memory may still be read
}

// ------------------------------------------------------------------------------------------------
// Candidate table and selection (one CTA per sequence).
// ------------------------------------------------------------------------------------------------
struct Tree {
    int B, K, depth, n_nodes, maxc, tc_max, rows_c;   // rows_c = B * tc_max (a-buffer rows of catch-up)
    float *c_score;          // [B, maxc]
    int32_t *c_tok, *c_par, *c_dc;   // c_dc = depth << 16 | creation
    int32_t *n_cand;         // [B]
    int32_t *frontier;       // [B, KMAX] candidate ids in rank order
    int32_t *row_tok, *row_x;        // [K * B] next depth rows (rank-major)
    uint64_t *pool_anc;      // [B, MAX_SLOTS]
    int32_t *pool_pos;       // [B, MAX_SLOTS]
    const int32_t *root_row; // [B] a-buffer row of the root (last catch-up row)
    const int32_t *draft_len;
    const int32_t *topk_tok;
    const float *topk_lq;
    const int32_t *next_tokens, *tc;
    int32_t *out_tok, *out_par, *out_depth;
    uint64_t *out_anc;
    float *out_score;
    int32_t *dev_status;
};

E3_DEV uint32_t score_key(float s) { return order_key(__fadd_rn(s, 0.0f)); }   // -0 -> +0

// rank of entry i among n by `key` (unique keys, descending): count of larger keys
template <class KF>
E3_DEV int rank_desc(int i, int n, KF key) {
    const uint64_t ki = key(i);
    int r = 0;
    for (int j = 0; j < n; ++j) r += key(j) > ki;
    return r;
}

// Choose the next frontier among the candidates [c0, c0 + n) (all of depth t) and describe the
// rows of depth t + 1 (frontier of depth t) for the next iteration.
E3_DEV void make_frontier(const Tree &T, int b, int t, int c0, int n, int32_t *sfront) {
    const float *sc = T.c_score + (size_t)b * T.maxc;
    const int32_t *dc = T.c_dc + (size_t)b * T.maxc;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int r = rank_desc(i, n, [&](int j) {
            return ((uint64_t)score_key(sc[c0 + j]) << 32) | (uint64_t)(0xFFFFu - (uint32_t)(dc[c0 + j] & 0xFFFF));
        });
        if (r < T.K) sfront[r] = c0 + i;
    }
    __syncthreads();
    const int L = T.draft_len[b];
    for (int r = threadIdx.x; r < T.K && r < n; r += blockDim.x) {
        const int f = sfront[r];
        const int slot = (t - 1) * T.K + r;                       // pool slot of this frontier row
        int pslot = -1;                                          // pool slot of its parent's row
        int xrow = T.root_row[b];
        if (t >= 2) {
            const int prank = (dc[f] & 0xFFFF) / T.K;            // the row that produced it
            pslot = (t - 2) * T.K + prank;
            xrow = T.rows_c + pslot * T.B + b;
        }
        T.frontier[(size_t)b * KMAX + r] = f;
        T.row_tok[(size_t)r * T.B + b] = T.c_tok[(size_t)b * T.maxc + f];
        T.row_x[(size_t)r * T.B + b] = xrow;
        T.pool_anc[(size_t)b * MAX_SLOTS + slot] =
            (pslot >= 0 ? T.pool_anc[(size_t)b * MAX_SLOTS + pslot] : 0ull) | (1ull << slot);
        T.pool_pos[(size_t)b * MAX_SLOTS + slot] = L - 1 + t;
    }
}

// Depth-t candidates from the top-k of the rows of depth t (t = 1: the root row of sequence b;
// t >= 2: frontier rank r of depth t - 1 at row r * B + b), then the next frontier.
__global__ void select_step_kernel(const Tree T, int t) {
    __shared__ int32_t sfront[KMAX];
    const int b = blockIdx.x;
    const int K = T.K;
    const int base = t == 1 ? 0 : T.n_cand[b];
    const int nrows = t == 1 ? 1 : K;
    const int n = nrows * K;
    float *sc = T.c_score + (size_t)b * T.maxc;
    for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
        const int r = idx / K, c = idx % K;
        const size_t trow = t == 1 ? (size_t)b : (size_t)r * T.B + b;
        const float lq = T.topk_lq[trow * K + c];
        const int id = base + idx;
        int par = -1;
        float s = lq;
        if (t >= 2) {
            par = T.frontier[(size_t)b * KMAX + r];
            s = __fadd_rn(sc[par], lq);
        }
        sc[id] = s;
        T.c_tok[(size_t)b * T.maxc + id] = T.topk_tok[trow * K + c];
        T.c_par[(size_t)b * T.maxc + id] = par;
        T.c_dc[(size_t)b * T.maxc + id] = (t << 16) | (r * K + c);
    }
    __syncthreads();
    if (threadIdx.x == 0) T.n_cand[b] = base + n;
    if (t < T.depth) make_frontier(T, b, t, base, n, sfront);
}

// Final rerank: top n_nodes - 1 of all candidates, emitted after the root.
__global__ void select_final_kernel(const Tree T) {
    extern __shared__ uint8_t sm_raw[];
    int32_t *chosen = (int32_t *)sm_raw;                       // [n_nodes - 1] by final rank
    int32_t *order = chosen + MAX_SLOTS;                       // [n_nodes - 1] node order
    int16_t *node_of = (int16_t *)(order + MAX_SLOTS);        // [maxc]
    const int b = blockIdx.x;
    const int n = T.n_cand[b], keep = min(T.n_nodes - 1, n);
    const float *sc = T.c_score + (size_t)b * T.maxc;
    const int32_t *dc = T.c_dc + (size_t)b * T.maxc;
    auto key1 = [&](int j) {
        return ((uint64_t)score_key(sc[j]) << 32) | ((uint64_t)(15 - (dc[j] >> 16)) << 16) |
               (uint64_t)(0xFFFFu - (uint32_t)(dc[j] & 0xFFFF));
    };
    for (int j = threadIdx.x; j < T.maxc; j += blockDim.x) node_of[j] = -1;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int r = rank_desc(i, n, key1);
        if (r < keep) chosen[r] = i;
    }
    __syncthreads();
    auto key2 = [&](int q) {
        const int j = chosen[q];
        return ((uint64_t)(15 - (dc[j] >> 16)) << 48) | ((uint64_t)score_key(sc[j]) << 16) |
               (uint64_t)(0xFFFFu - (uint32_t)(dc[j] & 0xFFFF));
    };
    for (int q = threadIdx.x; q < keep; q += blockDim.x) {
        const int r = rank_desc(q, keep, key2);
        order[r] = chosen[q];
        node_of[chosen[q]] = (int16_t)(r + 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const size_t o = (size_t)b * T.n_nodes;
        const int root = T.next_tokens[(size_t)b * T.tc_max + max(0, T.tc[b] - 1)];
        T.out_tok[o] = root;
        T.out_par[o] = -1;
        T.out_depth[o] = 0;
        T.out_score[o] = 0.0f;
        T.out_anc[o] = 1ull;
        bool bad = false;
        for (int m = 1; m <= keep; ++m) {
            const int j = order[m - 1];
            const int pc = T.c_par[(size_t)b * T.maxc + j];
            int pn = pc < 0 ? 0 : node_of[pc];
            if (pn < 0 || pn >= m) {
                bad = true;
                pn = 0;
            }
            T.out_tok[o + m] = T.c_tok[(size_t)b * T.maxc + j];
            T.out_par[o + m] = pn;
            T.out_depth[o + m] = dc[j] >> 16;
            T.out_score[o + m] = sc[j];
            T.out_anc[o + m] = T.out_anc[o + pn] | (1ull << m);
        }
        for (int m = keep + 1; m < T.n_nodes; ++m) {   // fewer candidates than nodes: pad with the root
            T.out_tok[o + m] = root;
            T.out_par[o + m] = 0;
            T.out_depth[o + m] = 1;
            T.out_score[o + m] = -INFINITY;
            T.out_anc[o + m] = 1ull | (1ull << m);
        }
        if (bad) flag(T.dev_status, EAGLE3_DEV_BAD_TREE);
    }
}

// Catch-up bookkeeping: chain masks / positions of the catch-up rows and the root row index.
__global__ void catchup_meta_kernel(int B, int tc_max, const int32_t *draft_len, const int32_t *tc,
                                    uint64_t *cu_anc, int32_t *cu_pos, int32_t *root_row, int32_t *dev_status) {
    const int b = blockIdx.x;
    for (int i = threadIdx.x; i < tc_max; i += blockDim.x) {
        cu_anc[(size_t)b * tc_max + i] = i >= 63 ? ~0ull : ((1ull << (i + 1)) - 1ull);
        cu_pos[(size_t)b * tc_max + i] = draft_len[b] + i;
    }
    if (threadIdx.x == 0) {
        int t = tc[b];
        if (t < 1 || t > tc_max) {
            flag(dev_status, EAGLE3_DEV_CAPACITY);
            t = max(1, min(t, tc_max));
        }
        root_row[b] = b * tc_max + t - 1;
    }
}

// Append the catch-up rows' rotated K and V to the draft cache, then advance draft_len.
__global__ void append_kv_kernel(int B, int tc_max, int Hkv, int S, int qkv_w, int k_off, int v_off,
                                 const __nv_bfloat16 *qkv, __nv_bfloat16 *kc, __nv_bfloat16 *vc, int32_t *draft_len,
                                 const int32_t *tc, int max_len, int32_t *dev_status) {
    const int b = blockIdx.x;
    const int L = draft_len[b];
    const int t = max(1, min(tc[b], tc_max));
    const bool ok = L >= 0 && L + t <= S && L <= max_len;
    if (ok) {
        const int chunks = t * Hkv * (HD / 8);
        for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
            const int i = c / (Hkv * (HD / 8)), g = (c / (HD / 8)) % Hkv, d8 = (c % (HD / 8)) * 8;
            const __nv_bfloat16 *src = qkv + (size_t)(b * tc_max + i) * qkv_w;
            const size_t dst = (((size_t)b * Hkv + g) * S + (size_t)(L + i)) * HD + d8;
            *reinterpret_cast<uint4 *>(kc + dst) = *reinterpret_cast<const uint4 *>(src + k_off + g * HD + d8);
            *reinterpret_cast<uint4 *>(vc + dst) = *reinterpret_cast<const uint4 *>(src + v_off + g * HD + d8);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (ok) draft_len[b] = L + t;
        else flag(dev_status, EAGLE3_DEV_CAPACITY);
    }
}

// ------------------------------------------------------------------------------------------------
// Host orchestration.
// ------------------------------------------------------------------------------------------------
struct Layout {
    size_t off[32];
    size_t total;
    int n = 0;
    size_t add(size_t bytes) {
        const size_t o = total;
        total += (bytes + 255) & ~(size_t)255;
        off[n++] = o;
        return o;
    }
};

struct Dims {
    int B, d, Hq, Hkv, F, V, Vd, K, depth, N, tc_max, S, max_len;
    int qkv_w, Rc, Rd, R, P, maxc, lm_rows;
};

Dims dims_of(const eagle3_draft_tree_args_t *a) {
    Dims m;
    m.B = a->batch;
    m.d = a->hidden;
    m.Hq = a->n_heads;
    m.Hkv = a->n_kv_heads;
    m.F = a->ffn;
    m.V = a->vocab;
    m.Vd = a->draft_vocab > 0 ? a->draft_vocab : a->vocab;
    m.K = a->top_k;
    m.depth = a->depth;
    m.N = a->n_nodes;
    m.tc_max = a->tc_max;
    m.S = a->s_max;
    m.max_len = a->max_draft_len;
    m.qkv_w = (m.Hq + 2 * m.Hkv) * HD;
    m.Rc = m.B * m.tc_max;
    m.Rd = m.K * m.B;
    m.R = std::max(m.Rc, m.Rd);
    m.P = (m.depth - 1) * m.K;
    m.maxc = m.K + (m.depth - 1) * m.K * m.K;
    m.lm_rows = std::max(m.B, m.Rd);
    return m;
}

eagle3_status_t draft_validate(const eagle3_draft_tree_args_t *a) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->batch < 0 || a->hidden < 8 || a->n_heads < 1 || a->n_kv_heads < 1 || a->ffn < 8 || a->vocab < 1 ||
        a->depth < 1 || a->top_k < 1 || a->n_nodes < 2 || a->tc_max < 1 || a->s_max < 1 || a->max_draft_len < 0)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->n_heads % a->n_kv_heads || a->hidden % 8 || a->ffn % 8) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->head_dim != HD || a->top_k > KMAX || a->depth > 8 || a->n_nodes > 64 || a->tc_max > 64)
        return EAGLE3_ERR_UNSUPPORTED;
    if ((a->depth - 1) * a->top_k > MAX_SLOTS) return EAGLE3_ERR_UNSUPPORTED;
    if (a->top_k * (a->n_heads / a->n_kv_heads) > 256 || a->tc_max * (a->n_heads / a->n_kv_heads) > 256)
        return EAGLE3_ERR_UNSUPPORTED;
    if (a->draft_vocab < 0 || a->draft_vocab > a->vocab) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->draft_vocab > 0 && a->draft_vocab != a->vocab && !a->d2t) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->top_k > (a->draft_vocab > 0 ? a->draft_vocab : a->vocab)) return EAGLE3_ERR_UNSUPPORTED;
    if ((int64_t)a->max_draft_len + a->tc_max > a->s_max) return EAGLE3_ERR_CAPACITY;
    if (a->batch == 0) return EAGLE3_OK;
    if (!a->aux || !a->next_tokens || !a->tc || !a->draft_k_cache || !a->draft_v_cache || !a->draft_len ||
        !a->tokens || !a->parents || !a->depth_out || !a->anc_mask || !a->score)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    return EAGLE3_OK;
}

eagle3_linear_args_t lin(int m, int n, int k, int epi, const void *x, const void *w, void *out, const void *res = nullptr,
                         const void *w2 = nullptr, int32_t *st = nullptr) {
    eagle3_linear_args_t l = {};
    l.m = m;
    l.n = n;
    l.k = k;
    l.epilogue = epi;
    l.splits = 0;
    l.ld_x = l.ld_w = l.ld_out = l.ld_res = 0;
    l.x = (const uint16_t *)x;
    l.w = (const uint16_t *)w;
    l.w2 = (const uint16_t *)w2;
    l.out = out;
    l.residual = (const uint16_t *)res;
    l.dev_status = st;
    return l;
}

struct Plan {
    Layout lay;
    size_t o_g, o_a2k, o_xres, o_qkvc, o_pool, o_attn, o_x1, o_h, o_act, o_abuf, o_nrm, o_logits, o_ttok, o_tlq;
    size_t o_rmax;   // [depth][lm_rows] row-maximum keys of each LM-head call (zeroed at the call's start)
    size_t o_cs, o_ct, o_cp, o_cd, o_ncand, o_front, o_rtok, o_rx, o_panc, o_ppos, o_canc, o_cpos, o_root, o_gws,
        o_aws;
    size_t gws, aws;
};

AttnLaunch catchup_attn(const Dims &m, const eagle3_draft_tree_args_t *a, uint8_t *ws, const Plan &pl) {
    AttnLaunch l;
    l.B = m.B;
    l.n_slots = m.tc_max;
    l.q_lo = 0;
    l.q_hi = m.tc_max;
    l.Hq = m.Hq;
    l.Hkv = m.Hkv;
    l.S = m.S;
    l.max_prefix = m.max_len;
    l.num_splits = 0;
    l.rope_theta = a->rope_theta;
    l.sm_scale = 1.0f / sqrtf((float)HD);
    __nv_bfloat16 *qkv = (__nv_bfloat16 *)(ws + pl.o_qkvc);
    l.q = qkv;
    l.q_si = m.qkv_w;
    l.q_sb = (int64_t)m.tc_max * m.qkv_w;
    l.k = qkv + (size_t)m.Hq * HD;
    l.k_si = l.q_si;
    l.k_sb = l.q_sb;
    l.v = qkv + (size_t)(m.Hq + m.Hkv) * HD;
    l.v_si = l.q_si;
    l.v_sb = l.q_sb;
    l.out = (__nv_bfloat16 *)(ws + pl.o_attn);
    l.o_si = (int64_t)m.Hq * HD;
    l.o_sb = (int64_t)m.tc_max * m.Hq * HD;
    l.k_cache = (const __nv_bfloat16 *)a->draft_k_cache;
    l.v_cache = (const __nv_bfloat16 *)a->draft_v_cache;
    l.parents = nullptr;
    l.anc = (const uint64_t *)(ws + pl.o_canc);
    l.pos = (const int32_t *)(ws + pl.o_cpos);
    l.anc_sb = l.pos_sb = m.tc_max;
    l.prefix_len = a->draft_len;
    l.lse = nullptr;
    l.dev_status = a->dev_status;
    return l;
}

AttnLaunch depth_attn(const Dims &m, const eagle3_draft_tree_args_t *a, uint8_t *ws, const Plan &pl, int t) {
    AttnLaunch l;
    l.B = m.B;
    l.n_slots = m.P;
    l.q_lo = (t - 2) * m.K;
    l.q_hi = (t - 1) * m.K;
    l.Hq = m.Hq;
    l.Hkv = m.Hkv;
    l.S = m.S;
    l.max_prefix = m.max_len + m.tc_max;
    l.num_splits = 0;
    l.rope_theta = a->rope_theta;
    l.sm_scale = 1.0f / sqrtf((float)HD);
    __nv_bfloat16 *pool = (__nv_bfloat16 *)(ws + pl.o_pool);
    l.q = pool;
    l.q_sb = m.qkv_w;
    l.q_si = (int64_t)m.B * m.qkv_w;
    l.k = pool + (size_t)m.Hq * HD;
    l.k_sb = l.q_sb;
    l.k_si = l.q_si;
    l.v = pool + (size_t)(m.Hq + m.Hkv) * HD;
    l.v_sb = l.q_sb;
    l.v_si = l.q_si;
    l.out = (__nv_bfloat16 *)(ws + pl.o_attn);
    l.o_sb = (int64_t)m.Hq * HD;
    l.o_si = (int64_t)m.B * m.Hq * HD;
    l.k_cache = (const __nv_bfloat16 *)a->draft_k_cache;
    l.v_cache = (const __nv_bfloat16 *)a->draft_v_cache;
    l.parents = nullptr;
    l.anc = (const uint64_t *)(ws + pl.o_panc);
    l.pos = (const int32_t *)(ws + pl.o_ppos);
    l.anc_sb = l.pos_sb = MAX_SLOTS;
    l.prefix_len = a->draft_len;
    l.lse = nullptr;
    l.dev_status = a->dev_status;
    return l;
}

Plan make_plan(const Dims &m, const eagle3_draft_tree_args_t *a) {
    Plan pl;
    Layout &L = pl.lay;
    L.total = 0;
    const size_t bf = 2;
    pl.o_g = L.add((size_t)m.Rc * m.d * bf);
    pl.o_a2k = L.add((size_t)m.R * 2 * m.d * bf);
    pl.o_xres = L.add((size_t)m.Rd * m.d * bf);
    pl.o_qkvc = L.add((size_t)m.Rc * m.qkv_w * bf);
    pl.o_pool = L.add((size_t)std::max(1, m.P) * m.B * m.qkv_w * bf);
    pl.o_attn = L.add((size_t)m.R * m.Hq * HD * bf);
    pl.o_x1 = L.add((size_t)m.R * m.d * bf);
    pl.o_h = L.add((size_t)m.R * m.d * bf);
    pl.o_act = L.add((size_t)m.R * m.F * bf);
    pl.o_abuf = L.add((size_t)(m.Rc + std::max(1, m.P) * m.B) * m.d * bf);
    pl.o_nrm = L.add((size_t)m.lm_rows * m.d * bf);
    pl.o_logits = L.add(a->dbg_logits ? 16 : (size_t)m.lm_rows * m.Vd * 4);
    pl.o_ttok = L.add((size_t)m.lm_rows * m.K * 4);
    pl.o_tlq = L.add((size_t)m.lm_rows * m.K * 4);
    pl.o_rmax = L.add((size_t)m.depth * m.lm_rows * 4);
    pl.o_cs = L.add((size_t)m.B * m.maxc * 4);
    pl.o_ct = L.add((size_t)m.B * m.maxc * 4);
    pl.o_cp = L.add((size_t)m.B * m.maxc * 4);
    pl.o_cd = L.add((size_t)m.B * m.maxc * 4);
    pl.o_ncand = L.add((size_t)m.B * 4);
    pl.o_front = L.add((size_t)m.B * KMAX * 4);
    pl.o_rtok = L.add((size_t)m.Rd * 4);
    pl.o_rx = L.add((size_t)m.Rd * 4);
    pl.o_panc = L.add((size_t)m.B * MAX_SLOTS * 8);
    pl.o_ppos = L.add((size_t)m.B * MAX_SLOTS * 4);
    pl.o_canc = L.add((size_t)m.B * m.tc_max * 8);
    pl.o_cpos = L.add((size_t)m.B * m.tc_max * 4);
    pl.o_root = L.add((size_t)m.B * 4);
    // GEMM split-K workspace: the largest any projection of this call asks for
    size_t g = 0;
    const int shapes[][4] = {{m.Rc, m.d, 3 * m.d, EAGLE3_EPI_BF16},       {m.R, m.qkv_w, 2 * m.d, EAGLE3_EPI_BF16},
                             {m.R, m.d, m.Hq * HD, EAGLE3_EPI_BF16_RESIDUAL}, {m.R, m.F, m.d, EAGLE3_EPI_SWIGLU},
                             {m.R, m.d, m.F, EAGLE3_EPI_BF16_RESIDUAL},   {m.B, m.Vd, m.d, EAGLE3_EPI_F32},
                             {m.Rd, m.Vd, m.d, EAGLE3_EPI_F32},            {m.Rd, m.qkv_w, 2 * m.d, EAGLE3_EPI_BF16},
                             {m.Rd, m.d, m.Hq * HD, EAGLE3_EPI_BF16_RESIDUAL}, {m.Rd, m.F, m.d, EAGLE3_EPI_SWIGLU},
                             {m.Rd, m.d, m.F, EAGLE3_EPI_BF16_RESIDUAL},  {m.Rc, m.qkv_w, 2 * m.d, EAGLE3_EPI_BF16},
                             {m.Rc, m.d, m.Hq * HD, EAGLE3_EPI_BF16_RESIDUAL}, {m.Rc, m.F, m.d, EAGLE3_EPI_SWIGLU},
                             {m.Rc, m.d, m.F, EAGLE3_EPI_BF16_RESIDUAL}};
    // sizing only: any non-null 16-byte aligned address passes the checks (nothing is dereferenced)
    const uint16_t *dummy = reinterpret_cast<const uint16_t *>((uintptr_t)256);
    for (auto &s : shapes) {
        eagle3_linear_args_t l = lin(s[0], s[1], s[2], s[3], dummy, dummy, (void *)dummy, dummy, dummy);
        g = std::max(g, eagle3_linear_workspace_size(&l));
    }
    pl.gws = g;
    pl.o_gws = L.add(g + 16);
    size_t at = 0;
    uint8_t *fake = nullptr;
    at = std::max(at, tree_attn_workspace(catchup_attn(m, a, fake, pl)));
    for (int t = 2; t <= m.depth; ++t) at = std::max(at, tree_attn_workspace(depth_attn(m, a, fake, pl, t)));
    pl.aws = at;
    pl.o_aws = L.add(at + 16);
    return pl;
}

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" size_t eagle3_draft_tree_workspace_size(const eagle3_draft_tree_args_t *a) {
    if (draft_validate(a) != EAGLE3_OK || a->batch == 0) return 0;
    const Dims m = dims_of(a);
    return make_plan(m, a).lay.total + 256;
}

#define E3_TRY(x)                                     \
    do {                                              \
        const eagle3_status_t _s = (x);               \
        if (_s != EAGLE3_OK) return _s;               \
    } while (0)
#define E3_LAUNCHED()                                                   \
    do {                                                                \
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA; \
    } while (0)

extern "C" eagle3_status_t eagle3_draft_tree(const eagle3_draft_weights_t *W, const eagle3_draft_tree_args_t *a,
                                             void *workspace, size_t ws_bytes, eagle3_stream_t stream_) {
    E3_TRY(draft_validate(a));
    if (a->batch == 0) return EAGLE3_OK;
    if (!W || !W->w_fc || !W->embed || !W->input_norm || !W->hidden_norm || !W->w_qkv || !W->w_o || !W->post_norm ||
        !W->w_gate || !W->w_up || !W->w_down || !W->final_norm || !W->lm_head)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    const Dims m = dims_of(a);
    const Plan pl = make_plan(m, a);
    if (!workspace || ws_bytes < pl.lay.total + 256) return EAGLE3_ERR_WORKSPACE;
    uint8_t *ws = (uint8_t *)(((uintptr_t)workspace + 255) & ~(uintptr_t)255);
    cudaStream_t st = (cudaStream_t)stream_;
    auto P = [&](size_t o) { return (void *)(ws + o); };
    void *gws = P(pl.o_gws);
    void *aws = P(pl.o_aws);
    const int d = m.d, B = m.B, K = m.K;
    __nv_bfloat16 *abuf = (__nv_bfloat16 *)P(pl.o_abuf);
    float *logits_base = a->dbg_logits ? a->dbg_logits : (float *)P(pl.o_logits);

    NormParams np;
    np.dim = d;
    np.eps = a->rms_eps;
    np.gather = nullptr;
    np.tap = nullptr;
    np.ld_tap = 0;
    np.dev_status = a->dev_status;

    // row-maximum words of every LM-head call start at zero (below every order key but a negative NaN's)
    if (cudaMemsetAsync(P(pl.o_rmax), 0, (size_t)m.depth * m.lm_rows * 4, st) != cudaSuccess) return EAGLE3_ERR_CUDA;
    // ---------------------------------------------------------------- catch-up rows
    catchup_meta_kernel<<<B, 64, 0, st>>>(B, m.tc_max, a->draft_len, a->tc, (uint64_t *)P(pl.o_canc),
                                          (int32_t *)P(pl.o_cpos), (int32_t *)P(pl.o_root), a->dev_status);
    E3_LAUNCHED();
    {
        eagle3_linear_args_t l = lin(m.Rc, d, 3 * d, EAGLE3_EPI_BF16, a->aux, W->w_fc, P(pl.o_g), nullptr, nullptr,
                                     a->dev_status);
        E3_TRY(eagle3_linear(&l, gws, pl.gws, stream_));
    }
    PrologueParams pp;
    pp.d = d;
    pp.vocab = m.V;
    pp.tc_max = m.tc_max;
    pp.eps = a->rms_eps;
    pp.embed = (const __nv_bfloat16 *)W->embed;
    pp.w_in = (const __nv_bfloat16 *)W->input_norm;
    pp.w_hid = (const __nv_bfloat16 *)W->hidden_norm;
    pp.dev_status = a->dev_status;
    pp.rows = m.Rc;
    pp.tokens = a->next_tokens;
    pp.tc = a->tc;
    pp.x = (const __nv_bfloat16 *)P(pl.o_g);
    pp.x_row = nullptr;
    pp.a2k = (__nv_bfloat16 *)P(pl.o_a2k);
    pp.xres = nullptr;
    draft_prologue_kernel<<<m.Rc, NT_NORM, 0, st>>>(pp);
    E3_LAUNCHED();

    auto layer_tail = [&](int rows, const void *x_res, void *a_out) -> eagle3_status_t {
        // attention output -> O (+x) -> post norm -> SwiGLU -> down (+x1) = a
        eagle3_linear_args_t l1 = lin(rows, d, m.Hq * HD, EAGLE3_EPI_BF16_RESIDUAL, P(pl.o_attn), W->w_o, P(pl.o_x1),
                                      x_res, nullptr, a->dev_status);
        E3_TRY(eagle3_linear(&l1, gws, pl.gws, stream_));
        NormParams n2 = np;
        n2.rows = rows;
        n2.n_src = rows;
        n2.ld_in = n2.ld_out = d;
        n2.in = (const __nv_bfloat16 *)P(pl.o_x1);
        n2.w = (const __nv_bfloat16 *)W->post_norm;
        n2.out = (__nv_bfloat16 *)P(pl.o_h);
        rmsnorm_kernel<<<rows, NT_NORM, 0, st>>>(n2);
        E3_LAUNCHED();
        eagle3_linear_args_t l2 = lin(rows, m.F, d, EAGLE3_EPI_SWIGLU, P(pl.o_h), W->w_gate, P(pl.o_act), nullptr,
                                      W->w_up, a->dev_status);
        E3_TRY(eagle3_linear(&l2, gws, pl.gws, stream_));
        eagle3_linear_args_t l3 = lin(rows, d, m.F, EAGLE3_EPI_BF16_RESIDUAL, P(pl.o_act), W->w_down, a_out, P(pl.o_x1),
                                      nullptr, a->dev_status);
        return eagle3_linear(&l3, gws, pl.gws, stream_);
    };
    auto lm_head = [&](int rows, const __nv_bfloat16 *a_rows, const int32_t *gather, float *logits,
                       int depth_t) -> eagle3_status_t {
        NormParams n3 = np;
        n3.rows = rows;
        n3.n_src = gather ? m.Rc : rows;
        n3.ld_in = n3.ld_out = d;
        n3.in = a_rows;
        n3.gather = gather;
        n3.w = (const __nv_bfloat16 *)W->final_norm;
        n3.out = (__nv_bfloat16 *)P(pl.o_nrm);
        rmsnorm_kernel<<<rows, NT_NORM, 0, st>>>(n3);
        E3_LAUNCHED();
        eagle3_linear_args_t l = lin(rows, m.Vd, d, EAGLE3_EPI_F32, P(pl.o_nrm), W->lm_head, logits, nullptr, nullptr,
                                     a->dev_status);
        // the epilogue publishes each row's maximum, so the top-k reads the logits once
        uint32_t *rmax = (uint32_t *)P(pl.o_rmax) + (size_t)(depth_t - 1) * m.lm_rows;
        l.row_max = rmax;
        E3_TRY(eagle3_linear(&l, gws, pl.gws, stream_));
        // few rows: a cluster per row, so that the scan of the vocabulary is spread over the SMs;
        // more rows than one wave of NT_TOPK-thread CTAs holds: narrower CTAs, so that all rows are
        // in flight at once (the scan is bound by the loads each SM keeps in flight)
        const int sms = device_sm_count();
        static PerDevice<int> topk_per_sm;
        const int per_sm = topk_per_sm.get([] {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, topk_kernel<NT_TOPK>, NT_TOPK, 0) != cudaSuccess)
                n = 0;
            return n > 0 ? n : 1;
        });
        const int wave = sms * per_sm;
        const TopkOut o = {(int32_t *)P(pl.o_ttok), (float *)P(pl.o_tlq), a->d2t, m.V, a->dev_status};
        // the shared-memory ring needs 16-byte rows: rows of a multiple of 4 floats, aligned logits
        const bool ring_ok = m.Vd % 4 == 0 && ((uintptr_t)logits & 15) == 0;
        if ((int64_t)rows * TOPK_CL <= 4LL * sms)   // up to ~4 cluster CTAs per SM (the B = 64 root rows)
            topk_cluster_kernel<<<rows * TOPK_CL, NT_TOPK, 0, st>>>(logits, m.Vd, m.Vd, K, rmax, o);
        else if (ring_ok)
            topk_ring_kernel<NT_TOPK_NARROW><<<rows, NT_TOPK_NARROW, TKR_RING_BYTES, st>>>(logits, m.Vd, m.Vd, K, rmax,
                                                                                          o);
        else if (rows <= wave)
            topk_kernel<NT_TOPK><<<rows, NT_TOPK, 0, st>>>(logits, m.Vd, m.Vd, K, rmax, o);
        else
            topk_kernel<NT_TOPK_NARROW><<<rows, NT_TOPK_NARROW, 0, st>>>(logits, m.Vd, m.Vd, K, rmax, o);
        E3_LAUNCHED();
        return EAGLE3_OK;
    };

    {
        eagle3_linear_args_t l = lin(m.Rc, m.qkv_w, 2 * d, EAGLE3_EPI_BF16, P(pl.o_a2k), W->w_qkv, P(pl.o_qkvc), nullptr,
                                     nullptr, a->dev_status);
        E3_TRY(eagle3_linear(&l, gws, pl.gws, stream_));
        E3_TRY(tree_attn_launch(catchup_attn(m, a, ws, pl), aws, pl.aws, st));
        E3_TRY(layer_tail(m.Rc, P(pl.o_g), abuf));
        append_kv_kernel<<<B, 256, 0, st>>>(B, m.tc_max, m.Hkv, m.S, m.qkv_w, m.Hq * HD, (m.Hq + m.Hkv) * HD,
                                            (const __nv_bfloat16 *)P(pl.o_qkvc), (__nv_bfloat16 *)a->draft_k_cache,
                                            (__nv_bfloat16 *)a->draft_v_cache, a->draft_len, a->tc, m.max_len,
                                            a->dev_status);
        E3_LAUNCHED();
        E3_TRY(lm_head(B, abuf, (const int32_t *)P(pl.o_root), logits_base, 1));
    }

    Tree T;
    T.B = B;
    T.K = K;
    T.depth = m.depth;
    T.n_nodes = m.N;
    T.maxc = m.maxc;
    T.tc_max = m.tc_max;
    T.rows_c = m.Rc;
    T.c_score = (float *)P(pl.o_cs);
    T.c_tok = (int32_t *)P(pl.o_ct);
    T.c_par = (int32_t *)P(pl.o_cp);
    T.c_dc = (int32_t *)P(pl.o_cd);
    T.n_cand = (int32_t *)P(pl.o_ncand);
    T.frontier = (int32_t *)P(pl.o_front);
    T.row_tok = (int32_t *)P(pl.o_rtok);
    T.row_x = (int32_t *)P(pl.o_rx);
    T.pool_anc = (uint64_t *)P(pl.o_panc);
    T.pool_pos = (int32_t *)P(pl.o_ppos);
    T.root_row = (const int32_t *)P(pl.o_root);
    T.draft_len = a->draft_len;
    T.topk_tok = (const int32_t *)P(pl.o_ttok);
    T.topk_lq = (const float *)P(pl.o_tlq);
    T.next_tokens = a->next_tokens;
    T.tc = a->tc;
    T.out_tok = a->tokens;
    T.out_par = a->parents;
    T.out_depth = a->depth_out;
    T.out_anc = a->anc_mask;
    T.out_score = a->score;
    T.dev_status = a->dev_status;
    select_step_kernel<<<B, 256, 0, st>>>(T, 1);
    E3_LAUNCHED();

    // ---------------------------------------------------------------- depth rows
    for (int t = 2; t <= m.depth; ++t) {
        const int rows = m.Rd;
        PrologueParams q = pp;
        q.rows = rows;
        q.tokens = T.row_tok;
        q.tc = nullptr;
        q.x = abuf;
        q.x_row = T.row_x;
        q.xres = (__nv_bfloat16 *)P(pl.o_xres);
        draft_prologue_kernel<<<rows, NT_NORM, 0, st>>>(q);
        E3_LAUNCHED();
        __nv_bfloat16 *pool_rows = (__nv_bfloat16 *)P(pl.o_pool) + (size_t)(t - 2) * rows * m.qkv_w;
        eagle3_linear_args_t l = lin(rows, m.qkv_w, 2 * d, EAGLE3_EPI_BF16, P(pl.o_a2k), W->w_qkv, pool_rows, nullptr,
                                     nullptr, a->dev_status);
        E3_TRY(eagle3_linear(&l, gws, pl.gws, stream_));
        E3_TRY(tree_attn_launch(depth_attn(m, a, ws, pl, t), aws, pl.aws, st));
        __nv_bfloat16 *a_rows = abuf + (size_t)(m.Rc + (t - 2) * rows) * d;
        E3_TRY(layer_tail(rows, P(pl.o_xres), a_rows));
        float *logits = logits_base + (a->dbg_logits ? (size_t)(t - 1) * rows * m.Vd : 0);
        E3_TRY(lm_head(rows, a_rows, nullptr, logits, t));
        select_step_kernel<<<B, 256, 0, st>>>(T, t);
        E3_LAUNCHED();
    }
    const size_t fsm = 2 * MAX_SLOTS * 4 + (size_t)m.maxc * 2 + 16;
    select_final_kernel<<<B, 256, fsm, st>>>(T);
    E3_LAUNCHED();
    return EAGLE3_OK;
}

extern "C" eagle3_status_t eagle3_rmsnorm(const eagle3_rmsnorm_args_t *a, eagle3_stream_t stream) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->rows < 0 || a->dim < 1 || a->n_src < 0 || a->ld_in < 0 || a->ld_out < 0 || a->ld_tap < 0 || !(a->eps >= 0.0f))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->rows == 0) return EAGLE3_OK;
    if (!a->in || !a->w || !a->out) return EAGLE3_ERR_INVALID_ARGUMENT;
    NormParams p;
    p.rows = a->rows;
    p.dim = a->dim;
    p.n_src = a->n_src ? a->n_src : a->rows;
    p.eps = a->eps;
    p.ld_in = a->ld_in ? a->ld_in : a->dim;
    p.ld_out = a->ld_out ? a->ld_out : a->dim;
    p.ld_tap = a->ld_tap ? a->ld_tap : a->dim;
    p.in = (const __nv_bfloat16 *)a->in;
    p.w = (const __nv_bfloat16 *)a->w;
    p.gather = a->gather;
    p.out = (__nv_bfloat16 *)a->out;
    p.tap = (__nv_bfloat16 *)a->tap_out;
    p.dev_status = a->dev_status;
    if (launch_pdl(rmsnorm_kernel, dim3(a->rows), dim3(NT_NORM), 0, (cudaStream_t)stream, p) != cudaSuccess)
        return EAGLE3_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}
