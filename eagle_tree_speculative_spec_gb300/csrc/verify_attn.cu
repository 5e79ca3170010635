// eagle3_verify_attn: tree-masked verify attention (bf16, GQA, head_dim 128), split-KV.
//
// Sources: "Advanced speculative decoding: tree drafts and EAGLE", sections "Why trees" and
// "Implementation" (forward_with_mask: each node sees the whole prefix plus itself and its
// ancestors; position = prefix length + depth); "EAGLE-3: Engineering Implementation of LLM
// Inference Acceleration", appendix C (rotate-half RoPE, GQA, 1/sqrt(D) scaling).
//
// One CTA per (sequence b, KV head g, split s).  The N tree nodes times the Hq/Hkv query heads
// that share KV head g form up to 256 query rows (row = node * rep + head), so the whole GQA
// group streams each K/V tile once.  Each of the 8 warps owns 32 rows.  K/V tiles of 64 keys are
// double-buffered in shared memory with cp.async; S = Q K^T and O += P V run on the bf16 tensor
// cores (mma.m16n8k16, fp32 accumulate) with an online softmax in the log2 domain.  The last split
// also processes the tree tile: tree keys are rotated in-kernel at L + depth, written back, and
// masked with the ancestor bitmask built from the parent array.  With more than one split the
// partial (O, m, l) go to the workspace and a second kernel merges them in split order.
#include "attn.cuh"

namespace e3 {
namespace {

constexpr int D = 128;
constexpr int ROWS = 256;           // query rows per CTA (N * rep <= 256)
constexpr int BK = 64;              // keys per tile
constexpr int NWARP = 8;
constexpr int NT = NWARP * 32;
constexpr int LDS = D + 8;          // padded smem row (bf16 elements): conflict-free ldmatrix
constexpr float LOG2E_F = 1.4426950408889634f;

struct Params {
    int B, n_slots, q_lo, q_hi, Hq, Hkv, S, splits, tiles_per_split, rep, max_prefix;
    float scale_log2;               // sm_scale * log2(e)
    float inv_freq[D / 2];
    // element (b, slot i, head h) lives at base + b * sb + i * si + h * D
    const __nv_bfloat16 *q;
    int64_t q_sb, q_si;
    __nv_bfloat16 *k;               // tree keys; slots [q_lo, q_hi) are rotated in place
    int64_t k_sb, k_si;
    const __nv_bfloat16 *v;
    int64_t v_sb, v_si;
    __nv_bfloat16 *out;             // query slot i -> row (i - q_lo)
    int64_t o_sb, o_si;
    const __nv_bfloat16 *k_cache, *v_cache;   // [B, Hkv, S, D]
    const int32_t *parents;         // [B, n_slots] or null: then anc / pos are given
    const uint64_t *anc;            // [B, anc_sb] ancestor-or-self bits over slots
    const int32_t *pos;             // [B, pos_sb] RoPE positions of the slots
    int anc_sb, pos_sb;
    const int32_t *prefix_len;
    float *lse;                     // [B, nq, Hq] or null
    float *part_o, *part_ml;        // [splits][B][nq][Hq][D], [splits][B][nq][Hq][2]
    int32_t *dev_status;
};

struct __align__(16) Smem {
    __nv_bfloat16 q[ROWS * LDS];
    __nv_bfloat16 k[2][BK * LDS];
    __nv_bfloat16 v[2][BK * LDS];
    uint64_t anc[64];
    int32_t pos[64];
    int32_t bad;
};

E3_DEV void cp_async16(void *smem, const void *gmem, bool pred) {
    const uint32_t s = smem_u32(smem);
    const int n = pred ? 16 : 0;   // zero-fill when out of range
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
E3_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
E3_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

E3_DEV void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
E3_DEV void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
E3_DEV void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
E3_DEV uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Rotate one 128-wide row (rotate-half RoPE) at position pos, fp32 math, bf16 out.
E3_DEV void rope_row(const __nv_bfloat16 *src, __nv_bfloat16 *dst_smem, __nv_bfloat16 *dst_global,
                     int pos, const float *inv_freq, int lane) {
    // lane handles pairs j = lane, lane + 32 (j < 64) and their partners j + 64
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int j = lane + 32 * u;
        const float x1 = __bfloat162float(src[j]), x2 = __bfloat162float(src[j + 64]);
        float sn, cs;
        sincosf(__fmul_rn((float)pos, inv_freq[j]), &sn, &cs);
        const __nv_bfloat16 o1 = __float2bfloat16_rn(x1 * cs - x2 * sn);
        const __nv_bfloat16 o2 = __float2bfloat16_rn(x2 * cs + x1 * sn);
        dst_smem[j] = o1;
        dst_smem[j + 64] = o2;
        if (dst_global) {
            dst_global[j] = o1;
            dst_global[j + 64] = o2;
        }
    }
}

__global__ void __launch_bounds__(NT, 1) verify_attn_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rep = p.rep, nk = p.q_hi, nq = p.q_hi - p.q_lo, nrows = nq * rep;
    const bool last = split == p.splits - 1;

    int L = p.prefix_len[b];
    if (L < 0 || L > p.max_prefix) {
        if (tid == 0 && split == 0 && g == 0) flag(p.dev_status, EAGLE3_DEV_CAPACITY);
        L = max(0, min(L, p.max_prefix));
    }
    // ---- tree slots: ancestor-or-self bits and RoPE positions
    if (tid == 0) {
        if (p.parents) {
            int bad = 0, depth[64];
            for (int i = 0; i < nk; ++i) {
                const int par = p.parents[(size_t)b * p.n_slots + i];
                if ((i == 0 && par != -1) || (i > 0 && (par < 0 || par >= i))) {
                    bad = 1;
                    depth[i] = 0;
                    s.anc[i] = 1ull << i;
                } else {
                    depth[i] = i ? depth[par] + 1 : 0;
                    s.anc[i] = (i ? s.anc[par] : 0ull) | (1ull << i);
                }
                s.pos[i] = L + depth[i];
            }
            s.bad = bad;
            if (bad && split == 0 && g == 0) flag(p.dev_status, EAGLE3_DEV_BAD_TREE);
        } else {
            for (int i = 0; i < nk; ++i) {
                s.anc[i] = p.anc[(size_t)b * p.anc_sb + i] & (nk >= 64 ? ~0ull : ((1ull << nk) - 1));
                s.pos[i] = p.pos[(size_t)b * p.pos_sb + i];
            }
            s.bad = 0;
        }
    }
    __syncthreads();

    // ---- prefix key range of this split
    const int t_lo = split * p.tiles_per_split;
    const int k_lo = min(L, t_lo * BK);
    const int k_hi = last ? L : min(L, (t_lo + p.tiles_per_split) * BK);
    const int n_tiles = (k_hi - k_lo + BK - 1) / BK + (last ? 1 : 0);   // + the tree tile

    // ---- Q rows (rotated) into smem; zero padding rows
    for (int r = warp; r < ROWS; r += NWARP) {
        __nv_bfloat16 *dst = s.q + r * LDS;
        if (r < nrows) {
            const int i = p.q_lo + r / rep, hh = r % rep;
            const __nv_bfloat16 *src = p.q + (size_t)b * p.q_sb + (size_t)i * p.q_si + ((size_t)g * rep + hh) * D;
            rope_row(src, dst, nullptr, s.pos[i], p.inv_freq, lane);
        } else {
            for (int j = lane; j < D; j += 32) dst[j] = __float2bfloat16_rn(0.0f);
        }
    }

    const __nv_bfloat16 *kc = p.k_cache + ((size_t)b * p.Hkv + g) * (size_t)p.S * D;
    const __nv_bfloat16 *vc = p.v_cache + ((size_t)b * p.Hkv + g) * (size_t)p.S * D;

    auto load_tile = [&](int t, int buf) {
        // prefix tiles: cp.async from the cache; the tree tile is written by the warps below
        const int key0 = k_lo + t * BK;
        for (int c = tid; c < BK * (D / 8); c += NT) {
            const int kr = c / (D / 8), kc8 = (c % (D / 8)) * 8;
            const bool ok = key0 + kr < k_hi;
            const size_t off = (size_t)(ok ? key0 + kr : 0) * D + kc8;
            cp_async16(s.k[buf] + kr * LDS + kc8, kc + off, ok);
            cp_async16(s.v[buf] + kr * LDS + kc8, vc + off, ok);
        }
    };
    const int n_prefix_tiles = n_tiles - (last ? 1 : 0);
    auto stage_tree_tile = [&](int buf) {
        // tree slots [0, q_hi): keys of the query slots are rotated here and written back once
        // (by the last split only), earlier slots were rotated when they were queries; rows past
        // q_hi are zero
        for (int i = warp; i < BK; i += NWARP) {
            __nv_bfloat16 *kd = s.k[buf] + i * LDS, *vd = s.v[buf] + i * LDS;
            if (i < nk) {
                __nv_bfloat16 *kg = p.k + (size_t)b * p.k_sb + (size_t)i * p.k_si + (size_t)g * D;
                const __nv_bfloat16 *vg = p.v + (size_t)b * p.v_sb + (size_t)i * p.v_si + (size_t)g * D;
                if (i >= p.q_lo) {
                    // each lane reads elements lane + 32u (u < 4) and writes back the same four,
                    // so the in-place rotation has no cross-lane hazard
                    __nv_bfloat16 tmp[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) tmp[u] = kg[lane + 32 * u];
                    const float pos = (float)s.pos[i];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {   // pairs (j, j + 64), j = lane + 32u
                        const int j = lane + 32 * u;
                        const float x1 = __bfloat162float(tmp[u]), x2 = __bfloat162float(tmp[u + 2]);
                        float sn, cs;
                        sincosf(__fmul_rn(pos, p.inv_freq[j]), &sn, &cs);
                        const __nv_bfloat16 o1 = __float2bfloat16_rn(x1 * cs - x2 * sn);
                        const __nv_bfloat16 o2 = __float2bfloat16_rn(x2 * cs + x1 * sn);
                        kd[j] = o1;
                        kd[j + 64] = o2;
                        kg[j] = o1;
                        kg[j + 64] = o2;
                    }
                } else {
                    for (int j = lane; j < D; j += 32) kd[j] = kg[j];
                }
                for (int j = lane; j < D; j += 32) vd[j] = vg[j];
            } else {
                for (int j = lane; j < D; j += 32) {
                    kd[j] = __float2bfloat16_rn(0.0f);
                    vd[j] = __float2bfloat16_rn(0.0f);
                }
            }
        }
    };

    // ---- accumulators: 2 m16 tiles per warp; O over 16 n8 tiles of D; running max / sum
    float o[2][16][4];
    float m_run[2][2], l_run[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.0f;
        m_run[mt][0] = m_run[mt][1] = -INFINITY;
        l_run[mt][0] = l_run[mt][1] = 0.0f;
    }
    const int row_base = warp * 32;

    if (n_tiles > 0) {
        if (n_prefix_tiles > 0) load_tile(0, 0);
        cp_async_commit();
    }
    for (int t = 0; t < n_tiles; ++t) {
        const int buf = t & 1;
        const bool tree_tile = last && t == n_tiles - 1;
        if (t + 1 < n_tiles) {
            if (t + 1 < n_prefix_tiles) load_tile(t + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        if (tree_tile) stage_tree_tile(buf);
        __syncthreads();

        const int key0 = tree_tile ? 0 : k_lo + t * BK;
        const int key_end = tree_tile ? nk : k_hi;
        // ---- S = Q K^T for 32 rows x 64 keys
        float sc[2][8][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[mt][nt][e] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const __nv_bfloat16 *qa = s.q + (row_base + mt * 16 + (lane & 15)) * LDS + kk * 16 + (lane >> 4) * 8;
                ldsm_x4(a[mt][0], a[mt][1], a[mt][2], a[mt][3], qa);
            }
#pragma unroll
            for (int np = 0; np < 4; ++np) {   // pairs of n8 tiles (16 keys)
                uint32_t b0, b1, b2, b3;
                const int krow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const __nv_bfloat16 *kb = s.k[buf] + krow * LDS + kk * 16 + ((lane >> 3) & 1) * 8;
                ldsm_x4(b0, b1, b2, b3, kb);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma_bf16(sc[mt][2 * np], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b0, b1);
                    mma_bf16(sc[mt][2 * np + 1], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b2, b3);
                }
            }
        }
        // ---- mask, online softmax (log2 domain), P in bf16
        uint32_t pa[2][4][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = row_base + mt * 16 + (lane >> 2) + hr * 8;
                const uint64_t bits = (tree_tile && row < nrows) ? s.anc[p.q_lo + row / rep] : 0ull;
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = key0 + nt * 8 + (lane & 3) * 2 + e;
                        const int local = nt * 8 + (lane & 3) * 2 + e;
                        bool ok = key < key_end;
                        if (tree_tile) ok = ok && ((bits >> local) & 1ull);
                        float v = sc[mt][nt][hr * 2 + e] * p.scale_log2;
                        v = ok ? v : -INFINITY;
                        sc[mt][nt][hr * 2 + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[mt][hr], mx);
                const float m_use = m_new == -INFINITY ? 0.0f : m_new;
                const float corr = exp2f(m_run[mt][hr] - m_use);
                m_run[mt][hr] = m_new;
                float sum = 0.0f;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = exp2f(sc[mt][nt][hr * 2 + e] - m_use);
                        sc[mt][nt][hr * 2 + e] = pv;
                        sum += pv;
                    }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                l_run[mt][hr] = l_run[mt][hr] * corr + sum;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    o[mt][nt][hr * 2] *= corr;
                    o[mt][nt][hr * 2 + 1] *= corr;
                }
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                pa[mt][kk][0] = pack_bf16(sc[mt][2 * kk][0], sc[mt][2 * kk][1]);
                pa[mt][kk][1] = pack_bf16(sc[mt][2 * kk][2], sc[mt][2 * kk][3]);
                pa[mt][kk][2] = pack_bf16(sc[mt][2 * kk + 1][0], sc[mt][2 * kk + 1][1]);
                pa[mt][kk][3] = pack_bf16(sc[mt][2 * kk + 1][2], sc[mt][2 * kk + 1][3]);
            }
        }
        // ---- O += P V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // 16 keys per step
#pragma unroll
            for (int np = 0; np < 8; ++np) {   // pairs of n8 tiles of D
                uint32_t b0, b1, b2, b3;
                const int vrow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const __nv_bfloat16 *vb = s.v[buf] + vrow * LDS + np * 16 + (lane >> 4) * 8;
                ldsm_x4_t(b0, b1, b2, b3, vb);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma_bf16(o[mt][2 * np], pa[mt][kk][0], pa[mt][kk][1], pa[mt][kk][2], pa[mt][kk][3], b0, b1);
                    mma_bf16(o[mt][2 * np + 1], pa[mt][kk][0], pa[mt][kk][1], pa[mt][kk][2], pa[mt][kk][3], b2, b3);
                }
            }
        }
        __syncthreads();   // buffer `buf` is reloaded two iterations later
    }

    // ---- epilogue: final output (one split) or partials
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int row = row_base + mt * 16 + (lane >> 2) + hr * 8;
            if (row >= nrows) continue;
            const int qi = row / rep, h = g * rep + row % rep;
            const size_t prow = ((size_t)b * nq + qi) * p.Hq + h;      // partial / lse row
            if (p.splits == 1) {
                __nv_bfloat16 *orow = p.out + (size_t)b * p.o_sb + (size_t)qi * p.o_si + (size_t)h * D;
                const float inv_l = l_run[mt][hr] > 0.0f ? 1.0f / l_run[mt][hr] : 0.0f;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const int d = nt * 8 + (lane & 3) * 2;
                    *reinterpret_cast<__nv_bfloat162 *>(orow + d) =
                        __floats2bfloat162_rn(o[mt][nt][hr * 2] * inv_l, o[mt][nt][hr * 2 + 1] * inv_l);
                }
                if (p.lse && (lane & 3) == 0)
                    p.lse[prow] = (m_run[mt][hr] + log2f(l_run[mt][hr])) * 0.6931471805599453f;
            } else {
                const size_t rows = (size_t)p.B * nq * p.Hq;
                float *po = p.part_o + ((size_t)split * rows + prow) * D;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const int d = nt * 8 + (lane & 3) * 2;
                    *reinterpret_cast<float2 *>(po + d) = make_float2(o[mt][nt][hr * 2], o[mt][nt][hr * 2 + 1]);
                }
                if ((lane & 3) == 0) {
                    float *pm = p.part_ml + ((size_t)split * rows + prow) * 2;
                    pm[0] = m_run[mt][hr];
                    pm[1] = l_run[mt][hr];
                }
            }
        }
}

// Merge split partials in split order: one warp per (b, query slot, head) row.
__global__ void verify_combine_kernel(const Params p) {
    const int nq = p.q_hi - p.q_lo;
    const int rows = p.B * nq * p.Hq;
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const size_t stride = (size_t)rows;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.part_ml[((size_t)s * stride + row) * 2]);
    const float Mu = M == -INFINITY ? 0.0f : M;
    float acc[4] = {0, 0, 0, 0}, l = 0.0f;
    for (int s = 0; s < p.splits; ++s) {
        const float *pm = p.part_ml + ((size_t)s * stride + row) * 2;
        const float w = exp2f(pm[0] - Mu);
        l += w * pm[1];
        const float4 v = *reinterpret_cast<const float4 *>(p.part_o + ((size_t)s * stride + row) * D + lane * 4);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
    }
    const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
    const int h = row % p.Hq, qi = (row / p.Hq) % nq, b = row / (p.Hq * nq);
    __nv_bfloat16 *dst = p.out + (size_t)b * p.o_sb + (size_t)qi * p.o_si + (size_t)h * D + lane * 4;
    *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(acc[0] * inv_l, acc[1] * inv_l);
    *reinterpret_cast<__nv_bfloat162 *>(dst + 2) = __floats2bfloat162_rn(acc[2] * inv_l, acc[3] * inv_l);
    if (p.lse && lane == 0) p.lse[row] = (M + log2f(l)) * 0.6931471805599453f;
}

int plan_splits(int ctas, int max_prefix, int requested, int sm_count) {
    const int tiles = (max_prefix + BK - 1) / BK;
    if (requested > 0) return max(1, min(requested, max(1, tiles)));
    if (ctas >= sm_count || tiles <= 2) return 1;
    int s = (sm_count + ctas - 1) / ctas;       // fill the GPU once
    s = min(s, max(1, tiles / 2));              // at least two tiles per split
    return max(1, s);
}

int sm_count_cached() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

}  // namespace

size_t tree_attn_workspace(const AttnLaunch &a) {
    const int splits = plan_splits(a.B * a.Hkv, a.max_prefix, a.num_splits, sm_count_cached());
    if (splits == 1 || a.B == 0) return 0;
    const size_t rows = (size_t)a.B * (a.q_hi - a.q_lo) * a.Hq;
    return (size_t)splits * rows * (D + 2) * sizeof(float);
}

eagle3_status_t tree_attn_launch(const AttnLaunch &a, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (a.B == 0 || a.q_hi <= a.q_lo) return EAGLE3_OK;
    const int splits = plan_splits(a.B * a.Hkv, a.max_prefix, a.num_splits, sm_count_cached());
    const size_t need = tree_attn_workspace(a);
    if (need && (!workspace || ws_bytes < need || ((uintptr_t)workspace & 15))) return EAGLE3_ERR_WORKSPACE;
    Params p;
    p.B = a.B;
    p.n_slots = a.n_slots;
    p.q_lo = a.q_lo;
    p.q_hi = a.q_hi;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.S = a.S;
    p.rep = a.Hq / a.Hkv;
    p.splits = splits;
    const int tiles = (a.max_prefix + BK - 1) / BK;
    p.tiles_per_split = max(1, (tiles + splits - 1) / splits);
    p.max_prefix = a.max_prefix;
    p.scale_log2 = a.sm_scale * LOG2E_F;
    for (int j = 0; j < D / 2; ++j) p.inv_freq[j] = (float)pow((double)a.rope_theta, -2.0 * j / D);
    p.q = a.q;
    p.q_sb = a.q_sb;
    p.q_si = a.q_si;
    p.k = a.k;
    p.k_sb = a.k_sb;
    p.k_si = a.k_si;
    p.v = a.v;
    p.v_sb = a.v_sb;
    p.v_si = a.v_si;
    p.out = a.out;
    p.o_sb = a.o_sb;
    p.o_si = a.o_si;
    p.k_cache = a.k_cache;
    p.v_cache = a.v_cache;
    p.parents = a.parents;
    p.anc = a.anc;
    p.pos = a.pos;
    p.anc_sb = a.anc_sb;
    p.pos_sb = a.pos_sb;
    p.prefix_len = a.prefix_len;
    p.lse = a.lse;
    p.dev_status = a.dev_status;
    const size_t rows = (size_t)a.B * (a.q_hi - a.q_lo) * a.Hq;
    p.part_o = splits > 1 ? (float *)workspace : nullptr;
    p.part_ml = splits > 1 ? (float *)workspace + (size_t)splits * rows * D : nullptr;

    const size_t smem = sizeof(Smem);
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(verify_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return EAGLE3_ERR_CUDA;
        attr_done = true;
    }
    verify_attn_kernel<<<dim3(splits, a.Hkv, a.B), NT, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (splits > 1) {
        verify_combine_kernel<<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    return EAGLE3_OK;
}

}  // namespace e3

using namespace e3;

static eagle3_status_t verify_validate(const eagle3_verify_attn_args_t *a) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->batch < 0 || a->n_nodes < 1 || a->n_heads < 1 || a->n_kv_heads < 1 || a->head_dim < 1 ||
        a->s_max < 1 || a->max_prefix_len < 0 || a->num_splits < 0 || a->q_node_stride < 0 || a->kv_node_stride < 0)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->n_heads % a->n_kv_heads) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->head_dim != D || a->n_nodes > 64) return EAGLE3_ERR_UNSUPPORTED;
    if (a->n_nodes * (a->n_heads / a->n_kv_heads) > ROWS) return EAGLE3_ERR_UNSUPPORTED;
    if ((int64_t)a->max_prefix_len + a->n_nodes > a->s_max) return EAGLE3_ERR_CAPACITY;
    if (!(a->rope_theta > 0.0f) || a->sm_scale < 0.0f) return EAGLE3_ERR_INVALID_ARGUMENT;
    if ((a->q_node_stride && (a->q_node_stride < (int64_t)a->n_heads * D || a->q_node_stride % 8)) ||
        (a->kv_node_stride && (a->kv_node_stride < (int64_t)a->n_kv_heads * D || a->kv_node_stride % 8)))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->batch == 0) return EAGLE3_OK;
    const void *ptrs[] = {a->q, a->tree_k, a->tree_v, a->k_cache, a->v_cache, a->out};
    for (const void *ptr : ptrs)
        if (!ptr || ((uintptr_t)ptr & 15)) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (!a->parents || !a->prefix_len) return EAGLE3_ERR_INVALID_ARGUMENT;
    return EAGLE3_OK;
}

static AttnLaunch verify_launch(const eagle3_verify_attn_args_t *a) {
    AttnLaunch l;
    l.B = a->batch;
    l.n_slots = a->n_nodes;
    l.q_lo = 0;
    l.q_hi = a->n_nodes;
    l.Hq = a->n_heads;
    l.Hkv = a->n_kv_heads;
    l.S = a->s_max;
    l.max_prefix = a->max_prefix_len;
    l.num_splits = a->num_splits;
    l.rope_theta = a->rope_theta;
    l.sm_scale = a->sm_scale > 0.0f ? a->sm_scale : 1.0f / sqrtf((float)D);
    const int64_t qs = a->q_node_stride ? a->q_node_stride : (int64_t)a->n_heads * D;
    const int64_t kvs = a->kv_node_stride ? a->kv_node_stride : (int64_t)a->n_kv_heads * D;
    l.q = (const __nv_bfloat16 *)a->q;
    l.q_si = qs;
    l.q_sb = qs * a->n_nodes;
    l.k = (__nv_bfloat16 *)a->tree_k;
    l.k_si = kvs;
    l.k_sb = kvs * a->n_nodes;
    l.v = (const __nv_bfloat16 *)a->tree_v;
    l.v_si = kvs;
    l.v_sb = kvs * a->n_nodes;
    l.out = (__nv_bfloat16 *)a->out;
    l.o_si = (int64_t)a->n_heads * D;
    l.o_sb = l.o_si * a->n_nodes;
    l.k_cache = (const __nv_bfloat16 *)a->k_cache;
    l.v_cache = (const __nv_bfloat16 *)a->v_cache;
    l.parents = a->parents;
    l.anc = nullptr;
    l.pos = nullptr;
    l.anc_sb = l.pos_sb = 0;
    l.prefix_len = a->prefix_len;
    l.lse = a->lse;
    l.dev_status = a->dev_status;
    return l;
}

extern "C" size_t eagle3_verify_attn_workspace_size(const eagle3_verify_attn_args_t *a) {
    if (verify_validate(a) != EAGLE3_OK || a->batch == 0) return 0;
    return tree_attn_workspace(verify_launch(a));
}

extern "C" eagle3_status_t eagle3_verify_attn(const eagle3_verify_attn_args_t *a, void *workspace,
                                              size_t ws_bytes, eagle3_stream_t stream) {
    const eagle3_status_t st = verify_validate(a);
    if (st != EAGLE3_OK || a->batch == 0) return st;
    return tree_attn_launch(verify_launch(a), workspace, ws_bytes, (cudaStream_t)stream);
}
