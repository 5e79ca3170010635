// eagle3_accept: lossless acceptance of a verified draft tree (greedy walk, or rejection
// sampling with residual resampling and a bonus token).
//
// Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", sections III.5
// and X.3-X.6; "Advanced speculative decoding: tree drafts and EAGLE", section "Implementation"
// and exercise 2; "Speculative Decoding (EAGLE3) in the vLLM Neuron Framework", section
// "Rejection Sampling".
//
// Design: one thread-block cluster of CL CTAs per sequence.  CTA r of the cluster owns the
// vocabulary slice [r*chunk, (r+1)*chunk) of every row it touches, so each level of the walk
// reads one target row (and one draft row in SAMPLED mode) with the whole cluster in parallel.
// Row-wide maxima and integer sums go through distributed shared memory (each CTA publishes its
// partial, one cluster barrier, every CTA reads all partials in rank order), so every CTA holds
// the same scalars and takes the same decisions; only the CTA that owns the final residual draw
// keeps running after the walk ends.  Only the rows of visited nodes are read.  All decisions
// are integer: the weights come from the deterministic fixed-point softmax in common.cuh, the
// accept tests and residual draws use 128-bit products.
#include <cooperative_groups.h>

#include "common.cuh"
#include "eagle3_linear.h"

namespace cg = cooperative_groups;

namespace e3 {
namespace {

constexpr int CL = 8;      // CTAs per cluster (one cluster per sequence)
constexpr int NT = 256;    // threads per CTA
constexpr int NW = NT / 32;
constexpr int MAXN = 64;

struct Params {
    int mode, B, N, V, W;
    float inv_t;
    uint64_t seed, step;
    const float *zt, *zd;
    const int32_t *tokens, *parents;
    int32_t *accept_len, *path, *emitted, *next_root, *dev_status;
    uint32_t *ws_p, *ws_q;   // [B, V] each, SAMPLED only
    const uint64_t *step_counter;   // when set, the step is read from device memory
    // one level of the walk (the lazy LM head): the target logits of each sequence's current node
    // are row b of zt ([B, V]); the walk state lives in st_* and path rows; a sequence that moves to
    // a child saves its state and counts itself in *moved; one that stops writes its outputs
    int level_mode;
    int32_t *st_node, *st_plen, *st_done, *moved;
    const int32_t *level_active;     // sequences still walking before this level (0: nothing to do)
};

struct Smem {
    int32_t parents[MAXN];
    int32_t tokens[MAXN];
    int32_t path[MAXN];
    int32_t rej_tok[MAXN];
    uint64_t slot[2][2];                 // published partials (double-buffered), 2 values each
    uint64_t warp_part[NW][2];
    uint64_t bcast[4];
    int32_t flag;
};

// ---- reductions over a CTA, then over the cluster ------------------------------------------
enum Op { MAX = 0, SUM = 1 };

template <int OP>
E3_DEV uint64_t combine(uint64_t a, uint64_t b) {
    return OP == MAX ? (a > b ? a : b) : a + b;
}

template <int OP>
E3_DEV uint64_t warp_reduce(uint64_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = combine<OP>(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Reduce two values per thread across the cluster.  Returns the cluster result in out[0..1];
// `parts` (optional, [CL]) receives each CTA's partial of value 0, in rank order.
template <int OP>
E3_DEV void cluster_reduce2(Smem &s, int &phase, uint64_t v0, uint64_t v1, uint64_t out[2],
                            uint64_t *parts, const cg::cluster_group &cluster) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v0 = warp_reduce<OP>(v0);
    v1 = warp_reduce<OP>(v1);
    if (lane == 0) {
        s.warp_part[warp][0] = v0;
        s.warp_part[warp][1] = v1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t a = s.warp_part[0][0], b = s.warp_part[0][1];
        for (int w = 1; w < NW; ++w) {
            a = combine<OP>(a, s.warp_part[w][0]);
            b = combine<OP>(b, s.warp_part[w][1]);
        }
        s.slot[phase][0] = a;
        s.slot[phase][1] = b;
    }
    cluster.sync();
    uint64_t a = 0, b = 0;
#pragma unroll
    for (int r = 0; r < CL; ++r) {
        const uint64_t *rs = cluster.map_shared_rank(&s.slot[phase][0], r);
        const uint64_t x0 = rs[0], x1 = rs[1];
        if (parts) parts[r] = x0;
        a = r ? combine<OP>(a, x0) : x0;
        b = r ? combine<OP>(b, x1) : x1;
    }
    out[0] = a;
    out[1] = b;
    phase ^= 1;
}

// ---- per-slice loops (float4 when the slice start is 16-byte aligned) ----------------------
template <class F>
E3_DEV void for_slice(const float *row, int lo, int hi, F f) {
    if (((reinterpret_cast<uintptr_t>(row + lo)) & 15) == 0) {
        const int n4 = (hi - lo) >> 2;
        const float4 *r4 = reinterpret_cast<const float4 *>(row + lo);
#pragma unroll 4
        for (int j = threadIdx.x; j < n4; j += NT) {
            const float4 v = __ldg(r4 + j);
            const int i = lo + 4 * j;
            f(i, v.x);
            f(i + 1, v.y);
            f(i + 2, v.z);
            f(i + 3, v.w);
        }
        for (int i = lo + 4 * n4 + threadIdx.x; i < hi; i += NT) f(i, __ldg(row + i));
    } else {
#pragma unroll 4
        for (int i = lo + threadIdx.x; i < hi; i += NT) f(i, __ldg(row + i));
    }
}

E3_DEV int bitlen128(unsigned __int128 v) {
    const uint64_t hi = (uint64_t)(v >> 64), lo = (uint64_t)v;
    return hi ? 64 + bitlen64(hi) : bitlen64(lo);
}

E3_DEV void write_outputs(const Params &p, int b, const int32_t *path, int plen, int next_root) {
    int *prow = p.path + (size_t)b * p.W, *erow = p.emitted + (size_t)b * p.W;
    const int n = plen - 1;
    for (int j = threadIdx.x; j < p.W; j += NT) {
        prow[j] = j < plen ? path[j] : -1;
        erow[j] = j < n ? p.tokens[(size_t)b * p.N + path[j + 1]] : (j == n ? next_root : -1);
    }
    if (threadIdx.x == 0) {
        p.accept_len[b] = n;
        p.next_root[b] = next_root;
    }
}

// Smallest k in this CTA's slice with (offset + W[lo] + ... + W[k]) > target, for weights given
// by wfn(i, z_i).  Each thread scans a contiguous run; a block scan of the run sums picks the run.
template <class WF>
E3_DEV int slice_inverse_cdf(Smem &s, const float *row, int lo, int hi, uint64_t offset,
                             uint64_t target, WF wfn) {
    const int len = hi - lo;
    const int per = (len + NT - 1) / NT;
    const int a = lo + threadIdx.x * per, e = min(hi, a + per);
    uint64_t mine = 0;
    for (int i = a; i < e; ++i) mine += wfn(i, row ? __ldg(row + i) : 0.0f);
    // inclusive block scan of run sums (warp shuffles, then warp totals)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s.warp_part[warp][0] = inc;
    if (threadIdx.x == 0) s.flag = -1;
    __syncthreads();
    uint64_t before = offset;
    for (int w = 0; w < warp; ++w) before += s.warp_part[w][0];
    before += inc - mine;   // exclusive prefix of this thread's run
    if (mine && before <= target && target < before + mine) {
        uint64_t run = before;
        for (int i = a; i < e; ++i) {
            run += wfn(i, row ? __ldg(row + i) : 0.0f);
            if (run > target) {
                s.flag = i;
                break;
            }
        }
    }
    __syncthreads();
    return s.flag;
}

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT) accept_kernel(const Params p) {
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ Smem s;
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / CL;
    const int N = p.N, V = p.V;
    const uint64_t step = p.step_counter ? *p.step_counter : p.step;
    int phase = 0;
    if (p.level_mode && (*p.level_active == 0 || p.st_done[b])) return;   // uniform across the cluster

    // ---- tree into shared memory, validated identically by every CTA
    if (threadIdx.x == 0) s.flag = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += NT) {
        const int par = p.parents[(size_t)b * N + i];
        const int tok = i ? p.tokens[(size_t)b * N + i] : 0;
        s.parents[i] = par;
        s.tokens[i] = tok;
        if ((i == 0 && par != -1) || (i > 0 && (par < 0 || par >= i))) atomicOr(&s.flag, EAGLE3_DEV_BAD_TREE);
        if (i > 0 && (tok < 0 || tok >= V)) atomicOr(&s.flag, EAGLE3_DEV_BAD_TOKEN);
    }
    __syncthreads();
    if (s.flag) {
        if (rank == 0) {
            if (threadIdx.x == 0) flag(p.dev_status, s.flag);
            for (int j = threadIdx.x; j < p.W; j += NT) {
                p.path[(size_t)b * p.W + j] = j == 0 ? 0 : -1;
                p.emitted[(size_t)b * p.W + j] = -1;
            }
            if (threadIdx.x == 0) {
                p.accept_len[b] = 0;
                p.next_root[b] = -1;
                if (p.level_mode) p.st_done[b] = 1;
            }
        }
        return;   // uniform across the cluster: no cluster barrier has been used yet
    }

    const int chunk = (((V + CL - 1) / CL) + 3) & ~3;
    const int lo = min(V, rank * chunk), hi = min(V, lo + chunk);
    int node = 0, plen = 1;
    if (threadIdx.x == 0) s.path[0] = 0;
    if (p.level_mode) {   // resume the walk where the previous level left it
        node = p.st_node[b];
        plen = p.st_plen[b];
        for (int j = threadIdx.x; j < plen; j += NT) s.path[j] = p.path[(size_t)b * p.W + j];
        __syncthreads();
    }
    uint64_t parts[CL];
    uint64_t red[2];
    // a move to a child: the full walk continues with it; one level saves the state and stops here
    auto advance = [&](int next) -> bool {
        if (!p.level_mode) return false;
        cluster.sync();   // no CTA leaves while another may still read its slots
        if (rank == 0 && threadIdx.x == 0) {
            p.st_node[b] = next;
            p.st_plen[b] = plen + 1;
            p.path[(size_t)b * p.W + plen] = next;
            atomicAdd(p.moved, 1);
        }
        return true;
    };

    for (;;) {
        const size_t row_off = p.level_mode ? (size_t)b * V : ((size_t)b * N + node) * (size_t)V;
        const float *zt = p.zt + row_off;

        if (p.mode == EAGLE3_ACCEPT_GREEDY) {
            uint64_t best = 0;
            for_slice(zt, lo, hi, [&](int i, float z) {
                const uint64_t k = pack_argmax(z, (uint32_t)i);
                best = k > best ? k : best;
            });
            cluster_reduce2<MAX>(s, phase, best, 0, red, nullptr, cluster);
            const int pred = (int)unpack_idx(red[0]);
            int next = -1;
            for (int c = node + 1; c < N; ++c)
                if (s.parents[c] == node && s.tokens[c] == pred) {
                    next = c;
                    break;
                }
            if (next >= 0 && plen < p.W) {
                if (advance(next)) return;
                node = next;
                if (threadIdx.x == 0) s.path[plen] = next;
                ++plen;
                continue;
            }
            cluster.sync();   // no CTA leaves while another may still read its slots
            if (next >= 0 && threadIdx.x == 0 && rank == 0) flag(p.dev_status, EAGLE3_DEV_PATH_TRUNC);
            if (rank == 0) {
                __syncthreads();
                write_outputs(p, b, s.path, plen, pred);
                if (p.level_mode && threadIdx.x == 0) p.st_done[b] = 1;
            }
            return;
        }

        // ---------------- TOPK / SAMPLED: deterministic fixed-point softmax of the row(s)
        const bool sampled = p.mode == EAGLE3_ACCEPT_SAMPLED;
        const float *zd = sampled ? p.zd + row_off : nullptr;
        uint32_t *wsp = sampled ? p.ws_p + (size_t)b * V : nullptr;
        uint32_t *wsq = sampled ? p.ws_q + (size_t)b * V : nullptr;
        uint32_t kp = 0, kq = 0;
        for_slice(zt, lo, hi, [&](int, float z) { kp = max(kp, order_key(z)); });
        if (sampled) for_slice(zd, lo, hi, [&](int, float z) { kq = max(kq, order_key(z)); });
        cluster_reduce2<MAX>(s, phase, kp, kq, red, nullptr, cluster);
        const float mp = key_to_float((uint32_t)red[0]), mq = key_to_float((uint32_t)red[1]);
        const float inv_t = p.inv_t;

        uint64_t sp = 0, sq = 0;
        if (!sampled) {
            for_slice(zt, lo, hi, [&](int, float z) { sp += dsm_weight(dsm_scaled(z, mp, inv_t)); });
        } else {
            for_slice(zt, lo, hi, [&](int i, float z) {
                const uint32_t w = dsm_weight(dsm_scaled(z, mp, inv_t));
                wsp[i] = w;
                sp += w;
            });
            for_slice(zd, lo, hi, [&](int i, float z) {
                const uint32_t w = dsm_weight(dsm_scaled(z, mq, inv_t));
                wsq[i] = w;
                sq += w;
            });
        }
        cluster_reduce2<SUM>(s, phase, sp, sq, red, parts, cluster);
        uint64_t Sp = red[0], Sq = red[1];

        int nrej = 0, next = -1, sib = 0;
        for (int c = node + 1; c < N && next < 0; ++c) {
            if (s.parents[c] != node) continue;
            const int x = s.tokens[c];
            const U4 rnd = accept_draw(p.seed, step, b, node, sib);
            ++sib;
            if (!sampled) {
                bool gone = false;
                for (int j = 0; j < nrej; ++j) gone |= s.rej_tok[j] == x;
                const uint64_t wx = gone ? 0 : dsm_weight(dsm_scaled(__ldg(zt + x), mp, inv_t));
                if ((unsigned __int128)rnd.x0 * Sp < ((unsigned __int128)wx << 32)) {
                    next = c;
                    break;
                }
                Sp -= wx;
                if (threadIdx.x == 0) s.rej_tok[nrej] = x;
                ++nrej;
                __syncthreads();
                continue;
            }
            // SAMPLED: current weights live in the workspace (published by the last barrier)
            const uint64_t wpx = *((volatile uint32_t *)wsp + x), wqx = *((volatile uint32_t *)wsq + x);
            if (Sq > 0 && (unsigned __int128)rnd.x0 * wqx * Sp < (((unsigned __int128)wpx * Sq) << 32)) {
                next = c;
                break;
            }
            const bool owner_x = x >= lo && x < hi;
            if (Sq > 0) {
                // residual r_i = max(0, Wp_i * Sq - Wq_i * Sp); requantise to 31 bits
                uint32_t mbits = 0;
                for (int i = lo + threadIdx.x; i < hi; i += NT) {
                    const unsigned __int128 a = (unsigned __int128)wsp[i] * Sq, q = (unsigned __int128)wsq[i] * Sp;
                    if (a > q) mbits = max(mbits, (uint32_t)bitlen128(a - q));
                }
                cluster_reduce2<MAX>(s, phase, mbits, 0, red, nullptr, cluster);
                const int mb = (int)red[0];
                if (mb > 0) {
                    const int sh = mb > FIX_BITS ? mb - FIX_BITS : 0;
                    uint64_t part = 0;
                    for (int i = lo + threadIdx.x; i < hi; i += NT) {
                        const unsigned __int128 a = (unsigned __int128)wsp[i] * Sq, q = (unsigned __int128)wsq[i] * Sp;
                        const uint32_t w = a > q ? (uint32_t)((a - q) >> sh) : 0u;
                        wsp[i] = w;
                        part += w;
                        if (i == x) wsq[i] = 0;   // remove x from q after its last use
                    }
                    cluster_reduce2<SUM>(s, phase, part, 0, red, parts, cluster);
                    Sp = red[0];
                    Sq -= wqx;
                    continue;
                }
            }
            // no residual update: remove x from q and publish before the next read
            if (owner_x && threadIdx.x == 0) wsq[x] = 0;
            Sq -= wqx;
            cluster.sync();
        }

        if (next >= 0 && plen < p.W) {
            if (advance(next)) return;
            node = next;
            if (threadIdx.x == 0) s.path[plen] = next;
            ++plen;
            continue;
        }
        if (next >= 0 && threadIdx.x == 0 && rank == 0) flag(p.dev_status, EAGLE3_DEV_PATH_TRUNC);

        // ---------------- all children rejected (or a leaf): residual / bonus draw
        const U4 rnd = accept_draw(p.seed, step, b, node, SLOT_RESIDUAL);
        const uint64_t r64 = ((uint64_t)rnd.x1 << 32) | rnd.x2;
        const uint64_t target = (uint64_t)(((unsigned __int128)r64 * Sp) >> 64);
        // slice sums of the current weights (TOPK: minus the rejected children in each slice)
        uint64_t off = 0;
        int owner = CL - 1;
        for (int r = 0; r < CL; ++r) {
            uint64_t sum_r = parts[r];
            if (!sampled) {
                const int rlo = min(V, r * chunk), rhi = min(V, rlo + chunk);
                for (int j = 0; j < nrej; ++j) {
                    const int x = s.rej_tok[j];
                    bool dup = false;
                    for (int k = 0; k < j; ++k) dup |= s.rej_tok[k] == x;
                    if (!dup && x >= rlo && x < rhi) sum_r -= dsm_weight(dsm_scaled(__ldg(zt + x), mp, inv_t));
                }
            }
            if (target < off + sum_r) {
                owner = r;
                break;
            }
            off += sum_r;
        }
        cluster.sync();   // last use of remote shared memory: everyone passes before anyone leaves
        if (rank != owner) return;
        int tok;
        if (!sampled) {
            tok = slice_inverse_cdf(s, zt, lo, hi, off, target, [&](int i, float z) -> uint64_t {
                for (int j = 0; j < nrej; ++j)
                    if (s.rej_tok[j] == i) return 0;
                return dsm_weight(dsm_scaled(z, mp, inv_t));
            });
        } else {
            tok = slice_inverse_cdf(s, nullptr, lo, hi, off, target,
                                    [&](int i, float) -> uint64_t { return wsp[i]; });
        }
        write_outputs(p, b, s.path, plen, tok);
        if (p.level_mode && threadIdx.x == 0) p.st_done[b] = 1;
        return;
    }
}

__global__ void step_increment_kernel(uint64_t *counter) { *counter += 1; }

// ---- lazy LM head: the level loop's small kernels ------------------------------------------
// every walk starts at the root: state, path rows, the moved counter
__global__ void lazy_init_kernel(int B, int W, int32_t *st_node, int32_t *st_plen, int32_t *st_done, int32_t *path,
                                 int32_t *moved) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b == 0) *moved = B;   // level 0: every sequence walks
    if (b >= B) return;
    st_node[b] = 0;
    st_plen[b] = 1;
    st_done[b] = 0;
    path[(size_t)b * W] = 0;
}

// before a level: the sequences still walking (those that moved in the previous level) become the
// level's active count, and the move counter restarts
__global__ void lazy_level_kernel(int32_t *moved, int32_t *active) {
    *active = *moved;
    *moved = 0;
}

// the final-normed hidden state of every walking sequence's current node, as the GEMM's rows
__global__ void lazy_gather_kernel(int N, int d, const __nv_bfloat16 *hs, const int32_t *st_node,
                                   const int32_t *st_done, const int32_t *active, __nv_bfloat16 *x) {
    const int b = blockIdx.x;
    if (*active == 0 || st_done[b]) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(hs + ((size_t)b * N + st_node[b]) * d);
    uint4 *dst = reinterpret_cast<uint4 *>(x + (size_t)b * d);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
}

struct LazyLayout {
    size_t x, z, node, plen, done, moved, active, gemm, total;
};

LazyLayout lazy_layout(const eagle3_accept_lazy_args_t *a, size_t gemm_ws) {
    LazyLayout l;
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t o = at;
        at += (bytes + 255) / 256 * 256;
        return o;
    };
    const size_t B = (size_t)a->accept.batch;
    l.x = take(B * a->hidden * 2);
    l.z = take(B * a->accept.vocab * 4);
    l.node = take(B * 4);
    l.plen = take(B * 4);
    l.done = take(B * 4);
    l.moved = take(4);
    l.active = take(4);
    l.gemm = take(gemm_ws);
    l.total = at + 256;
    return l;
}

eagle3_linear_args_t lazy_linear(const eagle3_accept_lazy_args_t *a, const void *x, void *z) {
    eagle3_linear_args_t l = {};
    l.m = a->accept.batch;
    l.n = a->accept.vocab;
    l.k = a->hidden;
    l.epilogue = EAGLE3_EPI_F32;
    l.x = (const uint16_t *)x;
    l.w = a->lm_head;
    l.out = z;
    l.dev_status = a->accept.dev_status;
    return l;
}

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" size_t eagle3_accept_workspace_size(const eagle3_accept_args_t *a) {
    if (!a || a->mode != EAGLE3_ACCEPT_SAMPLED || a->batch <= 0 || a->vocab <= 0) return 0;
    return (size_t)2 * (size_t)a->batch * (size_t)a->vocab * sizeof(uint32_t);
}

extern "C" eagle3_status_t eagle3_accept(const eagle3_accept_args_t *a, void *workspace, size_t ws_bytes,
                                         eagle3_stream_t stream) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->mode < EAGLE3_ACCEPT_GREEDY || a->mode > EAGLE3_ACCEPT_SAMPLED) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->batch < 0 || a->n_nodes < 1 || a->vocab < 1 || a->max_path < 1) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->n_nodes > MAXN || a->vocab > (1 << 22)) return EAGLE3_ERR_UNSUPPORTED;
    if (a->batch == 0) return EAGLE3_OK;
    if (!a->target_logits || !a->tokens || !a->parents || !a->accept_len || !a->path || !a->emitted ||
        !a->next_root)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    const bool sampled = a->mode == EAGLE3_ACCEPT_SAMPLED;
    if (sampled && !a->draft_logits) return EAGLE3_ERR_INVALID_ARGUMENT;
    float inv_t = 1.0f;
    if (a->mode != EAGLE3_ACCEPT_GREEDY) {
        if (!(a->temperature > 0.0f) || !(a->temperature < 3.0e38f)) return EAGLE3_ERR_INVALID_ARGUMENT;
        inv_t = 1.0f / a->temperature;
    }
    const size_t need = eagle3_accept_workspace_size(a);
    if (need && (!workspace || ws_bytes < need)) return EAGLE3_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 15) != 0) return EAGLE3_ERR_INVALID_ARGUMENT;

    Params p;
    p.mode = a->mode;
    p.B = a->batch;
    p.N = a->n_nodes;
    p.V = a->vocab;
    p.W = a->max_path;
    p.inv_t = inv_t;
    p.seed = a->seed;
    p.step = a->step;
    p.zt = a->target_logits;
    p.zd = sampled ? a->draft_logits : nullptr;
    p.tokens = a->tokens;
    p.parents = a->parents;
    p.accept_len = a->accept_len;
    p.path = a->path;
    p.emitted = a->emitted;
    p.next_root = a->next_root;
    p.dev_status = a->dev_status;
    p.ws_p = sampled ? (uint32_t *)workspace : nullptr;
    p.ws_q = sampled ? (uint32_t *)workspace + (size_t)a->batch * a->vocab : nullptr;
    p.step_counter = a->step_counter;
    p.level_mode = 0;
    p.st_node = p.st_plen = p.st_done = p.moved = nullptr;
    p.level_active = nullptr;
    accept_kernel<<<dim3(a->batch * CL), dim3(NT), 0, (cudaStream_t)stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (a->step_counter) {
        // stream-ordered after every CTA of the acceptance kernel has read the counter
        step_increment_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(a->step_counter);
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    return EAGLE3_OK;
}

namespace e3 {
eagle3_status_t linear_launch(const eagle3_linear_args_t *a, void *workspace, size_t ws_bytes, cudaStream_t stream,
                              const int32_t *skip_if_zero);
}

static eagle3_status_t lazy_validate(const eagle3_accept_lazy_args_t *a) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    const eagle3_accept_args_t *c = &a->accept;
    if (c->mode == EAGLE3_ACCEPT_SAMPLED) return EAGLE3_ERR_UNSUPPORTED;
    if (c->mode != EAGLE3_ACCEPT_GREEDY && c->mode != EAGLE3_ACCEPT_TOPK) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (c->batch < 0 || c->n_nodes < 1 || c->vocab < 1 || c->max_path < 1 || a->hidden < 8 || a->hidden % 8)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (c->n_nodes > MAXN || c->vocab > (1 << 22)) return EAGLE3_ERR_UNSUPPORTED;
    if (c->mode == EAGLE3_ACCEPT_TOPK && (!(c->temperature > 0.0f) || !(c->temperature < 3.0e38f)))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (c->batch == 0) return EAGLE3_OK;
    if (!c->tokens || !c->parents || !c->accept_len || !c->path || !c->emitted || !c->next_root ||
        !a->hidden_states || !a->lm_head || (((uintptr_t)a->hidden_states | (uintptr_t)a->lm_head) & 15))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    return EAGLE3_OK;
}

extern "C" size_t eagle3_accept_lazy_workspace_size(const eagle3_accept_lazy_args_t *a) {
    if (lazy_validate(a) != EAGLE3_OK || a->accept.batch == 0) return 0;
    const uint16_t *dummy = reinterpret_cast<const uint16_t *>((uintptr_t)256);   // sizing only
    eagle3_accept_lazy_args_t t = *a;
    t.lm_head = dummy;
    eagle3_linear_args_t l = lazy_linear(&t, dummy, (void *)dummy);
    return lazy_layout(a, eagle3_linear_workspace_size(&l)).total;
}

extern "C" eagle3_status_t eagle3_accept_lazy(const eagle3_accept_lazy_args_t *a, void *workspace, size_t ws_bytes,
                                              eagle3_stream_t stream_) {
    const eagle3_status_t st = lazy_validate(a);
    if (st != EAGLE3_OK || a->accept.batch == 0) return st;
    const eagle3_accept_args_t *c = &a->accept;
    const size_t need = eagle3_accept_lazy_workspace_size(a);
    if (!workspace || ws_bytes < need) return EAGLE3_ERR_WORKSPACE;
    uint8_t *ws = (uint8_t *)(((uintptr_t)workspace + 255) & ~(uintptr_t)255);
    cudaStream_t stream = (cudaStream_t)stream_;
    const int B = c->batch, W = c->max_path;
    const eagle3_linear_args_t probe = lazy_linear(a, ws, ws);
    const LazyLayout L = lazy_layout(a, eagle3_linear_workspace_size(&probe));
    auto P = [&](size_t o) { return (void *)(ws + o); };
    int32_t *st_node = (int32_t *)P(L.node), *st_plen = (int32_t *)P(L.plen), *st_done = (int32_t *)P(L.done);
    int32_t *moved = (int32_t *)P(L.moved), *active = (int32_t *)P(L.active);
    lazy_init_kernel<<<(B + 127) / 128, 128, 0, stream>>>(B, W, st_node, st_plen, st_done, c->path, moved);
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;

    Params p;
    p.mode = c->mode;
    p.B = B;
    p.N = c->n_nodes;
    p.V = c->vocab;
    p.W = W;
    p.inv_t = c->mode == EAGLE3_ACCEPT_GREEDY ? 1.0f : 1.0f / c->temperature;
    p.seed = c->seed;
    p.step = c->step;
    p.zt = (const float *)P(L.z);
    p.zd = nullptr;
    p.tokens = c->tokens;
    p.parents = c->parents;
    p.accept_len = c->accept_len;
    p.path = c->path;
    p.emitted = c->emitted;
    p.next_root = c->next_root;
    p.dev_status = c->dev_status;
    p.ws_p = p.ws_q = nullptr;
    p.step_counter = c->step_counter;
    p.level_mode = 1;
    p.st_node = st_node;
    p.st_plen = st_plen;
    p.st_done = st_done;
    p.moved = moved;
    p.level_active = active;
    const eagle3_linear_args_t lin = lazy_linear(a, P(L.x), P(L.z));
    for (int level = 0; level < W; ++level) {
        lazy_level_kernel<<<1, 1, 0, stream>>>(moved, active);
        lazy_gather_kernel<<<B, 128, 0, stream>>>(c->n_nodes, a->hidden, (const __nv_bfloat16 *)a->hidden_states,
                                                 st_node, st_done, active, (__nv_bfloat16 *)P(L.x));
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
        const eagle3_status_t s2 = linear_launch(&lin, P(L.gemm), L.total - L.gemm, stream, active);
        if (s2 != EAGLE3_OK) return s2;
        if (a->dbg_level_logits &&
            cudaMemcpyAsync(a->dbg_level_logits + (size_t)level * B * c->vocab, P(L.z), (size_t)B * c->vocab * 4,
                            cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
        accept_kernel<<<dim3(B * CL), dim3(NT), 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    if (c->step_counter) {
        step_increment_kernel<<<1, 1, 0, stream>>>(c->step_counter);
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    return EAGLE3_OK;
}
