// Ragged chain verification: the index bookkeeping of a batch of requests with different numbers
// of draft tokens, and a chain rejection sampler whose recovered tokens are Gumbel-max draws.
//
// Sources: "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", sections
// "SpecDecodeMetadata: Index Bookkeeping" (rows of a ragged batch) and "Rejection Sampling" (keep
// draft i while u < p_i(draft), recover from p_i without the draft by argmax p / E with Exp(1)
// noise, bonus from the last row; greedy requests compare with the argmax); "EAGLE-3: Engineering
// Implementation of LLM Inference Acceleration", sections X.3-X.6 (the emitted tokens follow the
// target distribution).
//
// Design: the bookkeeping is one CTA running a chunked block-wide scan over the requests.  The
// sampler runs one thread-block cluster of CLC CTAs per request: CTA r of the cluster reads its
// slice of every visited row with 16-byte loads (a row maximum pass, then one pass for the
// fixed-point normaliser or one for the Gumbel-max draw, which makes one Philox block per four
// tokens, keyed by the four tokens' index in the row).  The slices' maxima, sums and argmax keys
// are combined through distributed shared memory in rank order, so every CTA holds the same values
// and takes the same decisions.  Only the rows of the drafts up to the first rejection are read.
#include <cooperative_groups.h>

#include "common.cuh"
#include "eagle3_chain.h"

namespace cg = cooperative_groups;

namespace e3 {
namespace {

// ---------------------------------------------------------------------------------------------
// Bookkeeping
// ---------------------------------------------------------------------------------------------
constexpr int NT_META = 1024;

__global__ void __launch_bounds__(NT_META) spec_meta_kernel(const eagle3_spec_decode_metadata_args_t a) {
    __shared__ int32_t warp_sum[NT_META / 32];
    __shared__ int32_t chunk_total;
    __shared__ int32_t flags;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) flags = 0;
    __syncthreads();
    int carry = 0;   // drafts of the requests before this chunk
    for (int base = 0; base < a.n_requests; base += NT_META) {
        const int r = base + tid;
        int d = r < a.n_requests ? a.num_draft_tokens[r] : 0;
        bool bad = d < 0;
        if (bad) d = 0;
        // inclusive block scan of d
        int x = d;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sum[lane] = w;   // inclusive over warps
            if (lane == 31) chunk_total = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? warp_sum[warp - 1] : 0);
        if (r < a.n_requests) {
            const int cu_d = carry + incl;
            const int row0 = (cu_d - d) + r;
            const int end = a.cu_num_scheduled_tokens[r];
            const int start = r > 0 ? a.cu_num_scheduled_tokens[r - 1] : 0;
            bad = bad || end - start < d + 1;
            a.cu_num_draft_tokens[r] = cu_d;
            if (bad) {
                atomicOr(&flags, EAGLE3_DEV_BAD_COUNTS);
            } else {
                for (int j = 0; j <= d; ++j) {
                    const int row = row0 + j;
                    if (row < a.max_rows) {
                        a.logits_indices[row] = end - d - 1 + j;
                        if (j < d) a.target_logits_indices[cu_d - d + j] = row;   // cu_d - d + j <= row
                    } else {
                        atomicOr(&flags, EAGLE3_DEV_CAPACITY);
                    }
                }
                a.bonus_logits_indices[r] = row0 + d;
            }
        }
        carry += chunk_total;
        __syncthreads();   // warp_sum / chunk_total are rewritten by the next chunk
    }
    if (tid == 0) {
        a.num_rows[0] = carry + a.n_requests;
        if (flags) flag(a.dev_status, flags);
    }
}

// ---------------------------------------------------------------------------------------------
// Sampler
// ---------------------------------------------------------------------------------------------
constexpr int CLC = 8;     // CTAs per cluster (one cluster per request)
constexpr int NT = 256;    // threads per CTA
constexpr int NW = NT / 32;
constexpr uint32_t ACCEPT_C0 = 0x7fffffffu;

struct CParams {
    int R, V, K;
    float inv_t;
    uint64_t seed, step;
    const float *logits;
    const int32_t *drafts, *cu, *greedy;
    int32_t *out, *n_acc, *dev_status;
    const uint64_t *step_counter;
};

struct CSmem {
    uint64_t part[NW];
    uint64_t bcast;
    uint64_t cl[2];   // this CTA's partial of the cluster-wide reduction (double-buffered by parity)
};

// block-wide reductions of one value per thread; the result is returned to every thread
E3_DEV uint64_t block_max_u64(CSmem &s, uint64_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const uint64_t y = __shfl_xor_sync(0xffffffffu, v, o);
        v = y > v ? y : v;
    }
    if ((threadIdx.x & 31) == 0) s.part[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t m = 0;
        for (int w = 0; w < NW; ++w) m = s.part[w] > m ? s.part[w] : m;
        s.bcast = m;
    }
    __syncthreads();
    const uint64_t r = s.bcast;
    __syncthreads();
    return r;
}

E3_DEV uint64_t block_sum_u64(CSmem &s, uint64_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) s.part[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t t = 0;
        for (int w = 0; w < NW; ++w) t += s.part[w];   // integer sum: exact in any order
        s.bcast = t;
    }
    __syncthreads();
    const uint64_t r = s.bcast;
    __syncthreads();
    return r;
}

// The cluster-wide maximum / sum of one value per CTA (every thread passes its CTA's value; every
// thread gets the result): each CTA publishes its value, one cluster barrier, every thread reads the
// CLC values in rank order.  Partials alternate between two slots, so one barrier per reduction
// suffices: a slot is rewritten two reductions later, after every CTA has passed the barrier in
// between, i.e. after every CTA has read it.
template <bool MAX>
E3_DEV uint64_t cluster_reduce_u64(CSmem &s, cg::cluster_group &cluster, uint32_t &par, uint64_t v) {
    if (threadIdx.x == 0) s.cl[par] = v;
    cluster.sync();
    uint64_t acc = 0;
#pragma unroll
    for (int r = 0; r < CLC; ++r) {
        const uint64_t x = *cluster.map_shared_rank(&s.cl[par], r);
        acc = MAX ? (x > acc ? x : acc) : acc + x;
    }
    par ^= 1u;
    return acc;
}

// f(j, x0, z[x0 .. x0+3]) over this CTA's slice of a row: the float4 groups j in [j_lo, j_hi) of
// tokens 4j .. 4j+3 (one 16-byte load when the row allows)
template <typename F>
E3_DEV void for_row4(const float *z, int V, int j_lo, int j_hi, F f) {
    const bool vec = (((uintptr_t)z) & 15) == 0;
    for (int j = j_lo + (int)threadIdx.x; j < j_hi; j += NT) {
        float v[4];
        const int x0 = 4 * j;
        if (vec && x0 + 4 <= V) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(z) + j);
            v[0] = q.x;
            v[1] = q.y;
            v[2] = q.z;
            v[3] = q.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = x0 + e < V ? __ldg(z + x0 + e) : 0.0f;
        }
        f(j, x0, v);
    }
}

__global__ void __cluster_dims__(CLC, 1, 1) __launch_bounds__(NT) chain_verify_kernel(const CParams p) {
    __shared__ CSmem s;
    __shared__ int bad;
    pdl_wait();
    pdl_trigger();
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const bool writer = rank == 0;          // the CTA that writes the request's outputs
    const int r = blockIdx.x / CLC;
    const int end = p.cu[r], start = r > 0 ? p.cu[r - 1] : 0, d = end - start;
    int32_t *out = p.out + (size_t)r * (p.K + 1);
    const uint64_t step = p.step_counter ? *p.step_counter : p.step;
    if (threadIdx.x == 0) bad = (d < 0 || d > p.K) ? EAGLE3_DEV_BAD_COUNTS : 0;
    __syncthreads();
    if (!bad)
        for (int i = threadIdx.x; i < d; i += NT) {
            const int t = p.drafts[start + i];
            if (t < 0 || t >= p.V) atomicOr(&bad, EAGLE3_DEV_BAD_TOKEN);
        }
    __syncthreads();
    if (bad) {   // every CTA of the cluster sees the same counts and tokens: all leave here
        if (writer) {
            for (int i = threadIdx.x; i <= p.K; i += NT) out[i] = -1;
            if (threadIdx.x == 0) {
                if (p.n_acc) p.n_acc[r] = -1;
                flag(p.dev_status, bad);
            }
        }
        return;
    }
    // this CTA's slice of every row: float4 groups [j_lo, j_hi)
    const int n4 = (p.V + 3) / 4, per = (n4 + CLC - 1) / CLC;
    const int j_lo = min(n4, rank * per), j_hi = min(n4, j_lo + per);
    uint32_t par = 0;
    const int row0 = start + r;            // (cu_num_draft_tokens[r] - d) + r
    const bool greedy = p.greedy && p.greedy[r];
    const uint32_t k0 = (uint32_t)p.seed, k1 = (uint32_t)(p.seed >> 32);
    int n = d;                              // accepted drafts
    for (int i = 0; i <= d; ++i) {
        const float *z = p.logits + (size_t)(row0 + i) * p.V;
        const int dt = i < d ? p.drafts[start + i] : -1;
        if (greedy) {
            uint64_t best = 0;
            for_row4(z, p.V, j_lo, j_hi, [&](int, int x0, const float(&v)[4]) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (x0 + e < p.V) {
                        const uint64_t k = pack_argmax(v[e], (uint32_t)(x0 + e));
                        best = k > best ? k : best;
                    }
            });
            const int pred = (int)unpack_idx(cluster_reduce_u64<true>(s, cluster, par, block_max_u64(s, best)));
            if (i < d && dt == pred) {
                if (writer && threadIdx.x == 0) out[i] = dt;
                continue;
            }
            if (writer && threadIdx.x == 0) out[i] = pred;
            n = i;
            break;
        }
        // row maximum (total order of fp32 bit patterns)
        uint32_t mk = 0;
        for_row4(z, p.V, j_lo, j_hi, [&](int, int x0, const float(&v)[4]) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (x0 + e < p.V) mk = max(mk, order_key(v[e]));
        });
        const float m = key_to_float((uint32_t)cluster_reduce_u64<true>(s, cluster, par, block_max_u64(s, mk)));
        if (i < d) {
            uint64_t sum = 0;
            for_row4(z, p.V, j_lo, j_hi, [&](int, int x0, const float(&v)[4]) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (x0 + e < p.V) sum += dsm_weight(dsm_scaled(v[e], m, p.inv_t));
            });
            // integer sums: exact whatever the order of the slices
            const uint64_t S = cluster_reduce_u64<false>(s, cluster, par, block_sum_u64(s, sum));
            const uint64_t Wd = dsm_weight(dsm_scaled(__ldg(z + dt), m, p.inv_t));
            const uint32_t u32 = philox4x32_10(ACCEPT_C0, 256u * (uint32_t)r + (uint32_t)i, (uint32_t)step,
                                               (uint32_t)(step >> 32), k0, k1).x0;
            if ((unsigned __int128)u32 * S < ((unsigned __int128)Wd << 32)) {
                if (writer && threadIdx.x == 0) out[i] = dt;
                continue;
            }
        }
        // rejected (or every draft kept): the Gumbel-max draw over the row, the draft's entry removed
        uint64_t best = 0;
        for_row4(z, p.V, j_lo, j_hi, [&](int j, int x0, const float(&v)[4]) {
            const U4 w = philox4x32_10((uint32_t)j, 256u * (uint32_t)r + (uint32_t)i, (uint32_t)step,
                                       (uint32_t)(step >> 32), k0, k1);
            const uint32_t words[4] = {w.x0, w.x1, w.x2, w.x3};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int x = x0 + e;
                if (x >= p.V) continue;
                const uint32_t W = x == dt ? 0u : dsm_weight(dsm_scaled(v[e], m, p.inv_t));
                const float g = __fdiv_rn(__uint2float_rn(W), dsm_exp_noise(words[e]));
                const uint64_t k = pack_argmax(g, (uint32_t)x);
                best = k > best ? k : best;
            }
        });
        const int tok = (int)unpack_idx(cluster_reduce_u64<true>(s, cluster, par, block_max_u64(s, best)));
        if (writer && threadIdx.x == 0) out[i] = tok;
        n = i;
        break;
    }
    if (writer) {
        for (int i = n + 1 + threadIdx.x; i <= p.K; i += NT) out[i] = -1;
        if (threadIdx.x == 0 && p.n_acc) p.n_acc[r] = n;
    }
    cluster.sync();   // last use of remote shared memory: every CTA passes before any leaves
}

__global__ void chain_step_increment_kernel(uint64_t *counter) { *counter += 1; }

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" eagle3_status_t eagle3_spec_decode_metadata(const eagle3_spec_decode_metadata_args_t *a,
                                                       eagle3_stream_t stream) {
    if (!a || a->n_requests < 0 || a->n_requests > (1 << 20) || a->max_rows < 0) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->n_requests == 0) return EAGLE3_OK;
    if (!a->cu_num_scheduled_tokens || !a->num_draft_tokens || !a->cu_num_draft_tokens || !a->bonus_logits_indices ||
        !a->num_rows || (a->max_rows > 0 && (!a->logits_indices || !a->target_logits_indices)))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    spec_meta_kernel<<<1, NT_META, 0, (cudaStream_t)stream>>>(*a);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}

extern "C" eagle3_status_t eagle3_chain_verify(const eagle3_chain_verify_args_t *a, eagle3_stream_t stream) {
    if (!a || a->n_requests < 0 || a->n_requests > (1 << 24) || a->vocab < 1 || a->vocab > (1 << 22) ||
        a->max_drafts < 0 || a->max_drafts > 255)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->n_requests == 0) return EAGLE3_OK;
    if (!a->logits || !a->cu_num_draft_tokens || !a->output_tokens || (a->max_drafts > 0 && !a->draft_tokens))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (!(a->temperature > 0.0f)) return EAGLE3_ERR_INVALID_ARGUMENT;
    CParams p;
    p.R = a->n_requests;
    p.V = a->vocab;
    p.K = a->max_drafts;
    p.inv_t = 1.0f / a->temperature;   // fp32 round-to-nearest, as the oracle's fp32(1 / T)
    p.seed = a->seed;
    p.step = a->step;
    p.logits = a->logits;
    p.drafts = a->draft_tokens;
    p.cu = a->cu_num_draft_tokens;
    p.greedy = a->is_greedy;
    p.out = a->output_tokens;
    p.n_acc = a->num_accepted;
    p.dev_status = a->dev_status;
    p.step_counter = a->step_counter;
    if (launch_pdl(chain_verify_kernel, dim3(a->n_requests * CLC), dim3(NT), 0, (cudaStream_t)stream, p) != cudaSuccess)
        return EAGLE3_ERR_CUDA;
    if (a->step_counter) {
        chain_step_increment_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(a->step_counter);
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}
