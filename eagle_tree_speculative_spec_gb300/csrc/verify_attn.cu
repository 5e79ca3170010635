// eagle3_verify_attn: tree-masked verify attention (bf16, GQA, head_dim 128), split-KV, on the
// tcgen05 tensor cores with TMEM accumulators.
//
// Sources: "Advanced speculative decoding: tree drafts and EAGLE", sections "Why trees" and
// "Implementation" (forward_with_mask: each node sees the whole prefix plus itself and its
// ancestors; position = prefix length + depth); "EAGLE-3: Engineering Implementation of LLM
// Inference Acceleration", appendix C (rotate-half RoPE, GQA, 1/sqrt(D) scaling).
//
// One CTA per (sequence b, KV head g, split s).  The query slots times the Hq/Hkv heads that share
// KV head g form up to 256 query rows (row = slot * rep + head), i.e. up to two 128-row M tiles,
// so the whole GQA group streams each K/V tile from HBM once.  Warp roles:
//   warp 0        TMA: 64-key K and V tiles of the prefix (128B-swizzled) into a 3-stage ring
//   warps 1, 11   tcgen05.mma issuers, one per M tile so that the two tiles' chains do not wait on
//                 each other: S = Q K^T (M 128, N 64) into a double-buffered TMEM tile, then
//                 O += P V (M 128, N 128; P read from TMEM, V an MN-major smem operand); a K or V
//                 stage is released when both issuers have committed
//   warps 2..9    softmax, four warps per M tile, one thread per query row: the row's 64 scores
//                 come out of TMEM into registers (no shuffles), masked, exponentiated in the log2
//                 domain and written back over the same TMEM columns as packed bf16 P; O is
//                 rescaled in TMEM only when the running maximum grows by more than 8 (the result
//                 is the same, the intermediate weights stay below 2^8)
//   warp 10       TMA: V tiles (K and V have separate rings)
// The last split also processes the tree tile: the query slots' keys are rotated in-kernel at
// their positions and written back, then masked with the ancestor bitmask.  With more than one
// split the partial (O, m, l) go to the workspace and a second kernel merges them in split order.
// All waits are bounded; a timeout sets EAGLE3_DEV_TIMEOUT and the CTA drains and exits.
#include <cudaTypedefs.h>

#include "attn.cuh"
#include "tc.cuh"

namespace e3 {
namespace {

constexpr int D = 128;
constexpr int ROWS = 256;           // query rows per CTA (two M tiles)
constexpr int MT = 128;             // rows per M tile
constexpr int BK = 64;              // keys per tile
constexpr int ST = 4;               // K and V stages (each its own ring)
constexpr int NWARP = 12;             // 0: K loads, 1 and 11: MMA (one per M tile), 2..9: softmax, 10: V loads
constexpr int NT = NWARP * 32;
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int ROPE_TABLE_POS = 32;    // positions in the per-CTA angle table (16 KB of float2)

constexpr uint32_t Q_TILE = MT * D * 2;          // 32 KB: two 64-column blocks of 16 KB
constexpr uint32_t KV_TILE = BK * D * 2;         // 16 KB: two 64-column blocks of 8 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = OFF_Q + 2 * Q_TILE;
constexpr uint32_t OFF_TREE = OFF_KV + ST * 2 * KV_TILE;
constexpr uint32_t SMEM_DYN = OFF_TREE + 2 * KV_TILE + 1024;   // + alignment slack
static_assert(SMEM_DYN + 1024 <= 232448, "shared memory budget");
static_assert(ROPE_TABLE_POS * (D / 2) * sizeof(float2) <= KV_TILE, "angle table fits the tree-V tile");

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
    const int32_t *parents;         // [B, n_slots] or null: then anc / pos are given
    const uint64_t *anc;            // [B, anc_sb] ancestor-or-self bits over slots
    const int32_t *pos;             // [B, pos_sb] RoPE positions of the slots
    int anc_sb, pos_sb;
    const int32_t *prefix_len;
    float *lse;                     // [B, nq, Hq] or null
    float *part_o, *part_ml;        // [splits][B][nq][Hq][D], [splits][B][nq][Hq][2]
    int32_t *dev_status;
};

struct SmemStatic {
    uint64_t k_full[ST], k_empty[ST], v_full[ST], v_empty[ST];
    // every per-tile barrier is double-buffered by tile parity: a producer may run one tile ahead
    // of its consumer, and a phase that completes twice before it is awaited would be lost
    uint64_t s_full[2][2], p_full[2][2], pv_done[2][2], mma_done[2];
    uint64_t q_ready;               // the softmax warps have staged Q (and the tree tile)
    uint64_t anc[64];
    int32_t pos[64];
    int32_t par[64];
    uint32_t tmem_base;
    int abort_flag;
};

// 2^x on the special-function unit (flushes subnormal results to zero)
E3_DEV float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// warp-uniform bounded wait (lane 0 polls, the outcome is broadcast)
E3_DEV bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Rows are staged 16 bytes at a time: a 128-wide bf16 row is two 64-column blocks of eight 16-byte
// chunks, and a 128-byte swizzle keeps each chunk contiguous.  Lane group c (0..7) of a row owns
// chunk c of both blocks, i.e. the rotate-half pairs (8c + e, 64 + 8c + e), e = 0..7.
E3_DEV uint4 ld16(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint4 *>(p); }

E3_DEV void st_chunk(uint8_t *tile, int row, int chunk, uint32_t block_bytes, uint4 v) {
    *reinterpret_cast<uint4 *>(tile + tc::sw128_offset(row, chunk * 8, block_bytes)) = v;
}

// cos / sin of pos * inv_freq[8c + e], e = 0..7
E3_DEV void rope_angles(float pos, const float *inv_freq, int c, float cs[8], float sn[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sincosf(__fmul_rn(pos, inv_freq[8 * c + e]), &sn[e], &cs[e]);
}

// rotate-half RoPE of chunk pair c of one row: (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin)
E3_DEV void rope_chunks(uint4 &lo, uint4 &hi, const float cs[8], const float sn[8]) {
    const __nv_bfloat162 *a = reinterpret_cast<const __nv_bfloat162 *>(&lo);
    const __nv_bfloat162 *bb = reinterpret_cast<const __nv_bfloat162 *>(&hi);
    uint4 o1, o2;
    __nv_bfloat162 *r1 = reinterpret_cast<__nv_bfloat162 *>(&o1);
    __nv_bfloat162 *r2 = reinterpret_cast<__nv_bfloat162 *>(&o2);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x1 = __bfloat1622float2(a[e]), x2 = __bfloat1622float2(bb[e]);
        const float c0 = cs[2 * e], c1 = cs[2 * e + 1], s0 = sn[2 * e], s1 = sn[2 * e + 1];
        r1[e] = __floats2bfloat162_rn(x1.x * c0 - x2.x * s0, x1.y * c1 - x2.y * s1);
        r2[e] = __floats2bfloat162_rn(x2.x * c0 + x1.x * s0, x2.y * c1 + x1.y * s1);
    }
    lo = o1;
    hi = o2;
}

__global__ void __launch_bounds__(NT, 1)
    verify_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ SmemStatic ss;
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    volatile int *abort = &ss.abort_flag;
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rep = p.rep, nk = p.q_hi, nq = p.q_hi - p.q_lo, nrows = nq * rep;
    const int n_mt = (nrows + MT - 1) / MT;
    const bool last = split == p.splits - 1;

    int L = p.prefix_len[b];
    if (L < 0 || L > p.max_prefix) {
        if (tid == 0 && split == 0 && g == 0) flag(p.dev_status, EAGLE3_DEV_CAPACITY);
        L = max(0, min(L, p.max_prefix));
    }
    const int t_lo = split * p.tiles_per_split;
    const int k_lo = min(L, t_lo * BK);
    const int k_hi = last ? L : min(L, (t_lo + p.tiles_per_split) * BK);
    const int n_prefix = (k_hi - k_lo + BK - 1) / BK;
    const int n_tiles = n_prefix + (last ? 1 : 0);

    // ---- phase A: barriers, TMEM, raw tree description into shared memory
    if (tid == 0) {
        for (int s = 0; s < ST; ++s) {
            tc::mbar_init(&ss.k_full[s], 1);
            tc::mbar_init(&ss.k_empty[s], n_mt);
            tc::mbar_init(&ss.v_full[s], 1);
            tc::mbar_init(&ss.v_empty[s], n_mt);
        }
        for (int m = 0; m < 2; ++m) {
            for (int u = 0; u < 2; ++u) tc::mbar_init(&ss.s_full[m][u], 1);
            tc::mbar_init(&ss.p_full[m][0], 4);
            tc::mbar_init(&ss.p_full[m][1], 4);
            tc::mbar_init(&ss.pv_done[m][0], 1);
            tc::mbar_init(&ss.pv_done[m][1], 1);
        }
        tc::mbar_init(&ss.mma_done[0], 1);
        tc::mbar_init(&ss.mma_done[1], 1);
        tc::mbar_init(&ss.q_ready, 8);
        ss.abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(&ss.tmem_base, 512);
    if (warp == 2 || warp == 3) {
        const int i = tid - 64;
        if (i < nk) {
            if (p.parents) {
                ss.par[i] = p.parents[(size_t)b * p.n_slots + i];
            } else {
                ss.anc[i] = p.anc[(size_t)b * p.anc_sb + i] & (nk >= 64 ? ~0ull : ((1ull << nk) - 1));
                ss.pos[i] = p.pos[(size_t)b * p.pos_sb + i];
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = ss.tmem_base;

    if (warp == 0 || warp == 10) {
        // ------------------------------------------------------------------ TMA producers
        // warp 0 streams K tiles, warp 10 V tiles; each has its own ring so that a K stage is
        // refilled as soon as its S MMA is done, long before the V of the same tile is used
        if (lane == 0 && n_prefix > 0) {
            const bool is_k = warp == 0;
            const CUtensorMap *map = is_k ? &tm_k : &tm_v;
            uint64_t *full = is_k ? ss.k_full : ss.v_full;
            uint64_t *empty = is_k ? ss.k_empty : ss.v_empty;
            uint8_t *ring = sm + OFF_KV + (is_k ? 0 : ST * KV_TILE);
            tc::prefetch_tmap(map);
            const int row0 = ((b * p.Hkv + g) * p.S) + k_lo;
            uint32_t issued = 0, last_par = 0;
            for (int j = 0; j < n_prefix; ++j) {
                const int s = j % ST;
                const uint32_t ph = (uint32_t)(j / ST) & 1u;
                if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort)) {
                    flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
                    break;
                }
                uint8_t *dst = ring + s * KV_TILE;
                tc::mbar_expect_tx(&full[s], KV_TILE);
                const int y = row0 + j * BK;
                tc::tma_load_2d(dst, map, 0, y, &full[s]);
                tc::tma_load_2d(dst + KV_TILE / 2, map, 64, y, &full[s]);
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | (ph << s);
            }
            // no TMA write may be in flight when the CTA exits (bounded)
            for (int s = 0; s < ST; ++s) {
                if (!((issued >> s) & 1u)) continue;
                const long long t0 = clock64();
                while (!tc::mbar_try(&full[s], (last_par >> s) & 1u) && clock64() - t0 < WAIT_LIMIT_CYCLES) {
                }
            }
        }
    } else if (warp == 1 || warp == 11) {
        // ------------------------------------------------------------------ MMA issuers
        const int m = warp == 1 ? 0 : 1;
        if (lane == 0 && n_tiles > 0 && m < n_mt) {
            constexpr uint32_t IDESC_S = tc::idesc_bf16(MT, BK);
            constexpr uint32_t IDESC_PV = tc::idesc_bf16_bmn(MT, D);
            bool ok = true;
            auto k_tile = [&](int j) -> uint8_t * {
                return j < n_prefix ? sm + OFF_KV + (j % ST) * KV_TILE : sm + OFF_TREE;
            };
            auto v_tile = [&](int j) -> uint8_t * {
                return j < n_prefix ? sm + OFF_KV + (ST + j % ST) * KV_TILE : sm + OFF_TREE + KV_TILE;
            };
            // Q and the tree tile are written by the softmax warps (generic proxy, fenced)
            if (!tc::mbar_wait(&ss.q_ready, 0, abort)) ok = false;
            auto issue_s = [&](int j) {
                if (j < n_prefix) {
                    if (!tc::mbar_wait(&ss.k_full[j % ST], (uint32_t)(j / ST) & 1u, abort)) {
                        ok = false;
                        return;
                    }
                }
                // the S/P buffer j & 1 last held P(j - 2), read by P V(j - 2): that MMA was issued earlier
                // by this thread, and tcgen05.mma operations from one thread execute in issue order,
                // so S(j) cannot overwrite P(j - 2) before it has been read; no wait is needed
                tc::fence_after();
                const uint32_t kaddr = smem_u32(k_tile(j));
                const uint32_t qaddr = smem_u32(sm + OFF_Q + m * Q_TILE);
                const uint32_t d_s = tmem + 256u + (uint32_t)(m * 128 + (j & 1) * 64);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t blk = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
                    tc::mma_bf16_ss(d_s, tc::desc_sw128(qaddr + blk * (Q_TILE / 2) + kk * 32),
                                    tc::desc_sw128(kaddr + blk * (KV_TILE / 2) + kk * 32), IDESC_S, k > 0 ? 1u : 0u);
                }
                tc::mma_commit(&ss.s_full[m][j & 1]);
                if (j < n_prefix) tc::mma_commit(&ss.k_empty[j % ST]);   // K stage free once S is done
            };
            // two S tiles in flight; each iteration: P V of tile j as soon as its P is ready, then S(j + 2)
            if (ok) issue_s(0);
            if (n_tiles > 1 && ok) issue_s(1);
            for (int j = 0; j < n_tiles && ok; ++j) {
                if (j < n_prefix && !tc::mbar_wait(&ss.v_full[j % ST], (uint32_t)(j / ST) & 1u, abort)) {
                    ok = false;
                    break;
                }
                const uint32_t vaddr = smem_u32(v_tile(j));
                if (!tc::mbar_wait(&ss.p_full[m][j & 1], (uint32_t)(j >> 1) & 1u, abort)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t t_p = tmem + 256u + (uint32_t)(m * 128 + (j & 1) * 64);   // P over S
                const uint32_t d_o = tmem + (uint32_t)(m * 128);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    tc::mma_bf16_ts(d_o, t_p + (uint32_t)(kk * 8),
                                    tc::desc_mn_sw128(vaddr + kk * 2048, KV_TILE / 2, 1024), IDESC_PV,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(&ss.pv_done[m][j & 1]);
                if (j < n_prefix) tc::mma_commit(&ss.v_empty[j % ST]);
                if (j + 2 < n_tiles) issue_s(j + 2);
            }
            if (!ok) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            tc::mma_commit(&ss.mma_done[m]);
            const long long t0 = clock64();
            while (!tc::mbar_try(&ss.mma_done[m], 0) && clock64() - t0 < WAIT_LIMIT_CYCLES) {
            }
        }
    } else {
        // ------------------------------------------------------------------ softmax warps
        const int w8 = warp - 2;
        // ancestor-or-self bits and positions: slot i walks its own parent chain (parents < i)
        if (p.parents && w8 < 2) {
            const int i = tid - 64;
            if (i < nk) {
                auto invalid = [&](int j) {
                    const int pj = ss.par[j];
                    return j == 0 ? pj != -1 : (pj < 0 || pj >= j);
                };
                uint64_t bits = 1ull << i;
                int d = 0, j = i;
                const bool bad = invalid(i);
                while (j > 0 && !invalid(j)) {
                    j = ss.par[j];
                    bits |= 1ull << j;
                    ++d;
                }
                ss.anc[i] = bits;
                ss.pos[i] = L + d;
                if (bad && split == 0 && g == 0) flag(p.dev_status, EAGLE3_DEV_BAD_TREE);
            }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");   // the eight softmax warps only
        {
            const int c = lane & 7, sub = lane >> 3;
            // RoPE angles: the slots of a tree share few positions (prefix length + depth), so
            // cos / sin of every position in [pos_lo, pos_lo + span) are computed once per CTA into
            // the tree-V tile area (free until the tree V rows are staged below); a position
            // outside the table is computed directly.  Same arguments, so the same values.
            int pos_lo = 0x7fffffff, pos_hi = -1;
            for (int i = 0; i < nk; ++i) {
                pos_lo = min(pos_lo, ss.pos[i]);
                pos_hi = max(pos_hi, ss.pos[i]);
            }
            const int span = min(pos_hi - pos_lo + 1, ROPE_TABLE_POS);
            float2 *table = reinterpret_cast<float2 *>(sm + OFF_TREE + KV_TILE);
            for (int e = tid - 64; e < span * (D / 2); e += 256) {
                float sn, cs;
                sincosf(__fmul_rn((float)(pos_lo + e / (D / 2)), p.inv_freq[e % (D / 2)]), &sn, &cs);
                table[e] = make_float2(cs, sn);
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            auto angles = [&](int pos, float cs[8], float sn[8]) {
                const int d = pos - pos_lo;
                if (d >= 0 && d < span) {
                    const float4 *t4 = reinterpret_cast<const float4 *>(table + d * (D / 2) + 8 * c);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 v = t4[u];
                        cs[2 * u] = v.x;
                        sn[2 * u] = v.y;
                        cs[2 * u + 1] = v.z;
                        sn[2 * u + 1] = v.w;
                    }
                } else {
                    rope_angles((float)pos, p.inv_freq, c, cs, sn);
                }
            };
            // tree rows of the last split: issued first, used after the Q rows
            uint4 kl[2], kh[2], vl[2], vh[2];
            if (last) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int i = w8 * 4 + sub + 32 * t;
                    if (i < nk) {
                        const __nv_bfloat16 *kg = p.k + (size_t)b * p.k_sb + (size_t)i * p.k_si + (size_t)g * D;
                        const __nv_bfloat16 *vg = p.v + (size_t)b * p.v_sb + (size_t)i * p.v_si + (size_t)g * D;
                        kl[t] = ld16(kg + 8 * c);
                        kh[t] = ld16(kg + 64 + 8 * c);
                        vl[t] = ld16(vg + 8 * c);
                        vh[t] = ld16(vg + 64 + 8 * c);
                    }
                }
            }
            // Q rows (row = slot * rep + head), rotated at the slot's position.  Warp w8 takes the
            // slots w8 + 8 t (t < 8, i.e. all of them, nq <= 64), lane group `sub` the heads
            // sub + 4 h; all of a warp's loads are issued before the first is used.
            for (int hh = sub, h4 = 0; h4 * 4 < rep; hh += 4, ++h4) {
                uint4 lo[8], hi[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int sl = w8 + 8 * t;
                    if (sl < nq && hh < rep) {
                        const __nv_bfloat16 *src = p.q + (size_t)b * p.q_sb + (size_t)(p.q_lo + sl) * p.q_si +
                                                   ((size_t)g * rep + hh) * D;
                        lo[t] = ld16(src + 8 * c);
                        hi[t] = ld16(src + 64 + 8 * c);
                    }
                }
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int sl = w8 + 8 * t;
                    if (sl < nq && hh < rep) {
                        float cs[8], sn[8];
                        angles(ss.pos[p.q_lo + sl], cs, sn);
                        rope_chunks(lo[t], hi[t], cs, sn);
                        const int r = sl * rep + hh;
                        uint8_t *tile = sm + OFF_Q + (r / MT) * Q_TILE;
                        st_chunk(tile, r % MT, c, Q_TILE / 2, lo[t]);
                        st_chunk(tile, r % MT, c + 8, Q_TILE / 2, hi[t]);
                    }
                }
            }
            // zero rows of the last M tile
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int k = (tid - 64); k < (n_mt * MT - nrows) * 16; k += 256) {
                const int r = nrows + k / 16, ch = k % 16;
                st_chunk(sm + OFF_Q + (r / MT) * Q_TILE, r % MT, ch, Q_TILE / 2, z);
            }
            if (last) {
                // the tree tile: keys of the query slots rotated (and written back), others copied;
                // then the values, over the angle table
                uint8_t *tk = sm + OFF_TREE, *tv = sm + OFF_TREE + KV_TILE;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int i = w8 * 4 + sub + 32 * t;
                    if (i < nk) {
                        __nv_bfloat16 *kg = p.k + (size_t)b * p.k_sb + (size_t)i * p.k_si + (size_t)g * D;
                        uint4 klo = kl[t], khi = kh[t];
                        if (i >= p.q_lo) {
                            float cs[8], sn[8];
                            angles(ss.pos[i], cs, sn);
                            rope_chunks(klo, khi, cs, sn);
                            *reinterpret_cast<uint4 *>(kg + 8 * c) = klo;
                            *reinterpret_cast<uint4 *>(kg + 64 + 8 * c) = khi;
                        }
                        st_chunk(tk, i, c, KV_TILE / 2, klo);
                        st_chunk(tk, i, c + 8, KV_TILE / 2, khi);
                    } else {
                        st_chunk(tk, i, c, KV_TILE / 2, z);
                        st_chunk(tk, i, c + 8, KV_TILE / 2, z);
                    }
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");   // every table read is done
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int i = w8 * 4 + sub + 32 * t;
                    if (i < nk) {
                        st_chunk(tv, i, c, KV_TILE / 2, vl[t]);
                        st_chunk(tv, i, c + 8, KV_TILE / 2, vh[t]);
                    } else {
                        st_chunk(tv, i, c, KV_TILE / 2, z);
                        st_chunk(tv, i, c + 8, KV_TILE / 2, z);
                    }
                }
            }
            tc::fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor cores
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ss.q_ready);
        }
        const int m = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int rl = quarter * 32 + lane;              // row within the M tile
        const int row = m * MT + rl;
        if (m < n_mt) {
            const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
            const uint64_t bits = row < nrows ? ss.anc[p.q_lo + row / rep] : 0ull;
            float m_run = -INFINITY, l_run = 0.0f;
            bool ok = true;
            for (int j = 0; j < n_tiles; ++j) {
                const int u = j & 1;
                if (!warp_wait(&ss.s_full[m][u], (uint32_t)(j >> 1) & 1u, abort)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                float sc[64];
                {
                    float a[32], c[32];
                    tc::tmem_ld32(t_lane + 256u + (uint32_t)(m * 128 + u * 64), a);
                    tc::tmem_ld32(t_lane + 256u + (uint32_t)(m * 128 + u * 64 + 32), c);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        sc[i] = a[i];
                        sc[32 + i] = c[i];
                    }
                }
                const bool tree = j == n_prefix;         // the last split's final tile
                const int key0 = k_lo + j * BK;
                const bool full = !tree && key0 + BK <= k_hi;  // every key of the tile is visible
                // scale (and mask) with four independent max chains
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (full) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        sc[i] *= p.scale_log2;
                        mq[i & 3] = fmaxf(mq[i & 3], sc[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const bool valid = tree ? (i < nk && ((bits >> i) & 1ull)) : (key0 + i < k_hi);
                        sc[i] = valid ? sc[i] * p.scale_log2 : -INFINITY;
                        mq[i & 3] = fmaxf(mq[i & 3], sc[i]);
                    }
                }
                const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                const bool need = (m_run == -INFINITY) ? (mx > -INFINITY) : (mx > m_run + RESCALE_LOG2);
                const bool any_need = __any_sync(0xffffffffu, need);
                if (any_need && j > 0) {
                    // O is about to be rescaled: the previous P V must be finished first
                    if (!warp_wait(&ss.pv_done[m][(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                }
                if (any_need) {
                    const float m_new = need ? fmaxf(m_run, mx) : m_run;
                    const float corr = need ? (m_run == -INFINITY ? 0.0f : fast_exp2(m_run - m_new)) : 1.0f;
                    if (j > 0) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            float o[32];
                            tc::tmem_ld32(t_lane + (uint32_t)(m * 128 + c * 32), o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= corr;
                            tc::tmem_st32(t_lane + (uint32_t)(m * 128 + c * 32), o);
                        }
                    }
                    l_run *= corr;
                    m_run = m_new;
                }
                const float mu = m_run == -INFINITY ? 0.0f : m_run;
                // exponentials and the row sum (four chains), packed to bf16 pairs
                uint32_t pk[32];
                float sq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float p0 = fast_exp2(sc[2 * e] - mu), p1 = fast_exp2(sc[2 * e + 1] - mu);
                    sq[e & 3] += p0 + p1;
                    __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                    pk[e] = *reinterpret_cast<uint32_t *>(&h);
                }
                const float sum = (sq[0] + sq[1]) + (sq[2] + sq[3]);
                // P over the S columns it came from (the next S into this buffer waits for P V)
                tc::tmem_st32u(t_lane + 256u + (uint32_t)(m * 128 + u * 64), pk);
                l_run += sum;
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ss.p_full[m][j & 1]);
            }
            if (!ok && lane == 0) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            // ---- epilogue: O / l
            float o[D];
            bool have = false;
            if (ok && n_tiles > 0 &&
                warp_wait(&ss.pv_done[m][(n_tiles - 1) & 1], (uint32_t)((n_tiles - 1) >> 1) & 1u, abort)) {
                tc::fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float t[32];
                    tc::tmem_ld32(t_lane + (uint32_t)(m * 128 + c * 32), t);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[c * 32 + i] = t[i];
                }
                have = true;
            }
            if (!have) {
                m_run = -INFINITY;
                l_run = 0.0f;
#pragma unroll
                for (int i = 0; i < D; ++i) o[i] = 0.0f;
            }
            if (row < nrows) {
                const int qi = row / rep, h = g * rep + row % rep;
                const size_t prow_i = ((size_t)b * nq + qi) * p.Hq + h;
                if (p.splits == 1) {
                    __nv_bfloat16 *dst = p.out + (size_t)b * p.o_sb + (size_t)qi * p.o_si + (size_t)h * D;
                    const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
#pragma unroll
                    for (int c = 0; c < D; c += 8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 hv = __floats2bfloat162_rn(o[c + 2 * e] * inv_l, o[c + 2 * e + 1] * inv_l);
                            w[e] = *reinterpret_cast<uint32_t *>(&hv);
                        }
                        *reinterpret_cast<uint4 *>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (p.lse) p.lse[prow_i] = (m_run + log2f(l_run)) * 0.6931471805599453f;
                } else {
                    const size_t rows_all = (size_t)p.B * nq * p.Hq;
                    float *po = p.part_o + ((size_t)split * rows_all + prow_i) * D;
#pragma unroll
                    for (int c = 0; c < D; c += 4) *reinterpret_cast<float4 *>(po + c) = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
                    float *pm = p.part_ml + ((size_t)split * rows_all + prow_i) * 2;
                    pm[0] = m_run;
                    pm[1] = l_run;
                }
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

// [rows, 128] bf16 cache viewed as a 2-D tensor; 64 x 64 boxes, 128-byte swizzle
bool make_cache_map(CUtensorMap *m, const void *base, int64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)BK};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int plan_splits(int ctas, int max_prefix, int requested, int sm_count) {
    const int tiles = (max_prefix + BK - 1) / BK;
    if (requested > 0) return max(1, min(requested, max(1, tiles)));
    if (ctas >= sm_count || tiles <= 2) return 1;
    int s = sm_count / ctas;                    // at most one wave
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

// A launch covers sequences [b0, b0 + nb) with `splits` KV splits.  When the (sequence, KV head)
// blocks fill some waves of the GPU and leave a tail smaller than half a wave, the full waves run
// unsplit and the tail sequences are split over the SMs the tail would leave idle.
struct Part {
    int b0, nb, splits;
};

int plan_parts(const AttnLaunch &a, Part parts[2]) {
    const int sms = sm_count_cached();
    const int items = a.B * a.Hkv;
    if (a.num_splits == 0 && items > sms && items % sms) {
        const int b0 = (items / sms) * sms / a.Hkv;
        const int tail = (a.B - b0) * a.Hkv;
        if (b0 > 0 && b0 < a.B && 2 * tail <= sms) {
            parts[0] = {0, b0, 1};
            parts[1] = {b0, a.B - b0, plan_splits(tail, a.max_prefix, 0, sms)};
            return 2;
        }
    }
    parts[0] = {0, a.B, plan_splits(items, a.max_prefix, a.num_splits, sms)};
    return 1;
}

size_t part_workspace(const AttnLaunch &a, const Part &pt) {
    if (pt.splits == 1 || pt.nb == 0) return 0;
    const size_t rows = (size_t)pt.nb * (a.q_hi - a.q_lo) * a.Hq;
    return (size_t)pt.splits * rows * (D + 2) * sizeof(float);
}

eagle3_status_t launch_part(const AttnLaunch &a, const Part &pt, void *workspace, cudaStream_t stream) {
    const int splits = pt.splits;
    const size_t b0 = (size_t)pt.b0;
    const int nq = a.q_hi - a.q_lo;
    Params p;
    p.B = pt.nb;
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
    p.q = a.q + b0 * a.q_sb;
    p.q_sb = a.q_sb;
    p.q_si = a.q_si;
    p.k = a.k + b0 * a.k_sb;
    p.k_sb = a.k_sb;
    p.k_si = a.k_si;
    p.v = a.v + b0 * a.v_sb;
    p.v_sb = a.v_sb;
    p.v_si = a.v_si;
    p.out = a.out + b0 * a.o_sb;
    p.o_sb = a.o_sb;
    p.o_si = a.o_si;
    p.parents = a.parents ? a.parents + b0 * a.n_slots : nullptr;
    p.anc = a.anc ? a.anc + b0 * a.anc_sb : nullptr;
    p.pos = a.pos ? a.pos + b0 * a.pos_sb : nullptr;
    p.anc_sb = a.anc_sb;
    p.pos_sb = a.pos_sb;
    p.prefix_len = a.prefix_len + b0;
    p.lse = a.lse ? a.lse + b0 * nq * a.Hq : nullptr;
    p.dev_status = a.dev_status;
    const size_t rows = (size_t)pt.nb * nq * a.Hq;
    p.part_o = splits > 1 ? (float *)workspace : nullptr;
    p.part_ml = splits > 1 ? (float *)workspace + (size_t)splits * rows * D : nullptr;

    CUtensorMap mk, mv;
    const size_t cache_off = b0 * a.Hkv * a.S * D;
    const int64_t cache_rows = (int64_t)pt.nb * a.Hkv * a.S;
    if (!make_cache_map(&mk, a.k_cache + cache_off, cache_rows) ||
        !make_cache_map(&mv, a.v_cache + cache_off, cache_rows))
        return EAGLE3_ERR_CUDA;
    verify_attn_kernel<<<dim3(splits, a.Hkv, pt.nb), NT, SMEM_DYN, stream>>>(mk, mv, p);
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (splits > 1) {
        verify_combine_kernel<<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    return EAGLE3_OK;
}

}  // namespace

size_t tree_attn_workspace(const AttnLaunch &a) {
    if (a.B == 0) return 0;
    Part parts[2];
    const int n = plan_parts(a, parts);
    size_t need = 0;
    for (int i = 0; i < n; ++i) need = std::max(need, part_workspace(a, parts[i]));   // parts run in order
    return need;
}

eagle3_status_t tree_attn_launch(const AttnLaunch &a, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (a.B == 0 || a.q_hi <= a.q_lo) return EAGLE3_OK;
    const size_t need = tree_attn_workspace(a);
    if (need && (!workspace || ws_bytes < need || ((uintptr_t)workspace & 15))) return EAGLE3_ERR_WORKSPACE;
    // rows of q / tree k / tree v / out are moved 16 bytes at a time
    const int64_t strides[] = {a.q_sb, a.q_si, a.k_sb, a.k_si, a.v_sb, a.v_si, a.o_sb, a.o_si};
    for (int64_t st : strides)
        if (st % 8) return EAGLE3_ERR_INVALID_ARGUMENT;
    const void *row_bases[] = {a.q, a.k, a.v, a.out};
    for (const void *r : row_bases)
        if ((uintptr_t)r & 15) return EAGLE3_ERR_INVALID_ARGUMENT;
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(verify_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_DYN) !=
            cudaSuccess)
            return EAGLE3_ERR_CUDA;
        attr_done = true;
    }
    Part parts[2];
    const int n = plan_parts(a, parts);
    for (int i = 0; i < n; ++i) {
        const eagle3_status_t st = launch_part(a, parts[i], workspace, stream);
        if (st != EAGLE3_OK) return st;
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

// ------------------------------------------------------------------------------------------------
// eagle3_verify_attn_noalloc: the same attention for callers that cannot allocate device memory
// (for example a runtime that hands all device memory to its own pool before the first step, or
// code that must not allocate while it is being captured into a CUDA graph).  The split-KV
// partials live in a file-scope device array of fixed size instead of a caller workspace.
// ------------------------------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)32 << 20;   // 32 MiB, held by every device that loads the library
__device__ __align__(256) uint8_t g_verify_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Host code cannot use the array's name as a device address: look the address up once per device
// (with that device current) and keep it.
void *noalloc_scratch_address() {
    static std::mutex mu;
    static void *addr[128] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" eagle3_status_t eagle3_verify_attn_noalloc(const eagle3_verify_attn_args_t *a, eagle3_stream_t stream) {
    const eagle3_status_t st = verify_validate(a);
    if (st != EAGLE3_OK || a->batch == 0) return st;
    void *scratch = noalloc_scratch_address();     // first call on a device: address lookup
    if (!scratch) return EAGLE3_ERR_CUDA;
    const AttnLaunch l = verify_launch(a);
    if (tree_attn_workspace(l) > NOALLOC_SCRATCH_BYTES) return EAGLE3_ERR_WORKSPACE;
    return tree_attn_launch(l, scratch, NOALLOC_SCRATCH_BYTES, (cudaStream_t)stream);
}
