// eagle3_verify_attn: tree-masked verify attention (bf16, GQA, head_dim 128), split-KV, on the
// tcgen05 tensor cores with TMEM accumulators.
//
// Sources: "Advanced speculative decoding: tree drafts and EAGLE", sections "Why trees" and
// "Implementation" (forward_with_mask: each node sees the whole prefix plus itself and its
// ancestors; position = prefix length + depth); "EAGLE-3: Engineering Implementation of LLM
// Inference Acceleration", appendix C (rotate-half RoPE, GQA, 1/sqrt(D) scaling).
//
// One CTA per (sequence b, KV head g, split s, half h).  The query slots times the Hq/Hkv heads
// that share KV head g form the query rows (row = slot * rep + head); when they are more than one
// 128-row M tile, the slots are cut into two halves and each half is its own CTA (adjacent blocks,
// so the second read of every K/V tile comes from L2).  Warp roles:
//   warp 0        TMA: 128-key K tiles of the prefix (128B-swizzled) into a 3-stage ring
//   warp 10       TMA: V tiles into a 2-stage ring
//   warp 1        S = Q K^T (M 128, N 128) into one of three TMEM buffers; S(j) waits only for its
//                 K tile and for P V(j - 3), which read the buffer last
//   warp 11       O += P V (M 128, N 128; P read from TMEM, V an MN-major smem operand)
//   warps 2..9    Q staging (rotated, 16-byte chunks), then the softmax: two
//                 warps per TMEM lane quarter, each taking half of a row's 128 scores; the two halves
//                 exchange their row maxima through shared memory once per tile.  Scores are
//                 exponentiated in the log2 domain and written back over the same TMEM columns as
//                 packed bf16 P; O is rescaled in TMEM only when the running maximum grows by more
//                 than 8 (the result is the same, the intermediate weights stay below 2^8)
// A kernel before this one rotates the query slots' keys in tree_k at their positions (prefix
// length + depth); the last split then also streams the tree tile (64 rows of tree_k / tree_v, by
// TMA like the prefix) and masks it with the ancestor bitmask.  Thread 0 issues the first K tiles
// as soon as it has initialised their barriers.  With more than one split the partial (O, m, l) go
// to the workspace and another kernel merges them in split order.  Queries and tree keys that
// arrive already rotated (qk_rotated: the QKV projection applied RoPE, always with a parent array)
// run on the persistent kernel further below, which loads Q by 4-D TMA boxes and needs neither the
// key rotation nor the staging.
// All waits are bounded; a timeout sets EAGLE3_DEV_TIMEOUT and the CTA drains and exits.
#include <cudaTypedefs.h>

#include "attn.cuh"
#include "eagle3_testing.h"
#include "tc.cuh"

namespace e3 {
namespace {

constexpr int D = 128;
constexpr int MT = 128;             // query rows per CTA (one M tile)
constexpr int BK = 128;             // keys per prefix tile
constexpr int BKT = 64;             // keys of the tree tile
constexpr int ST_K = 3;             // K stages
constexpr int ST_V = 2;             // V stages
constexpr int NS = 3;               // S / P buffers in TMEM
constexpr int NWARP = 12;           // 0: K loads, 1: S MMAs, 2..9: softmax, 10: V loads, 11: P V MMAs
constexpr int NT = NWARP * 32;
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr int ROPE_TABLE_POS = 32;    // positions in the per-CTA angle table (16 KB of float2)

constexpr uint32_t Q_TILE = MT * D * 2;          // 32 KB: two 64-column blocks of 16 KB
constexpr uint32_t KV_TILE = BK * D * 2;         // 32 KB: two 64-column blocks of 16 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + Q_TILE;                 // K ring; the tree tile (64 keys) uses the first
constexpr uint32_t OFF_V = OFF_K + ST_K * KV_TILE;         // V ring    half of each 64-column block of a stage
constexpr uint32_t OFF_TABLE = OFF_V + KV_TILE;            // RoPE angles while Q is staged (V stage 1)
constexpr uint32_t SMEM_DYN = OFF_V + ST_V * KV_TILE + 1024;   // + alignment slack
// TMEM columns: O at [0, 128); S / P buffer u at TM_S + 128 u
constexpr uint32_t TM_S = 128;
static_assert(SMEM_DYN + 1024 <= 232448, "shared memory budget");
static_assert(ROPE_TABLE_POS * (D / 2) * sizeof(float2) <= KV_TILE, "angle table fits a V stage");
static_assert(TM_S + NS * BK <= 512, "TMEM budget");

struct Params {
    int B, n_slots, q_lo, q_hi, Hq, Hkv, S, splits, tiles_per_split, rep, max_prefix;
    int halves;                     // CTAs per (sequence, KV head, split): 1 or 2
    int tree_slot_inner;            // tree maps: slots are the middle dimension (else the outer)
    int s_mid;                      // with two halves, the first half's query slots are [q_lo, q_lo + s_mid)
    int qk_rotated;                 // q and the tree keys arrive rotated: Q is loaded by TMA as is
    int stall_tile;                 // timeout-path test only: this prefix tile is never loaded (-1 off)
    const int32_t *block_table;     // paged cache (slot pool [n_slots, Hkv, 128]) or null (contiguous)
    int bt_stride, block_size, n_pages;
    int pool_box;                   // slots per box of the pool's tensor map: 128 (block_size % 128 == 0) or 64
    long long wait_limit;           // clocks after which a bounded wait gives up
    float scale_log2;               // sm_scale * log2(e)
    float inv_freq[D / 2];
    // element (b, slot i, head h) lives at base + b * sb + i * si + h * D
    const __nv_bfloat16 *q;
    int64_t q_sb, q_si;
    __nv_bfloat16 *k;               // tree keys; slots [q_lo, q_hi) are rotated in place (second kernel)
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
    uint64_t k_full[ST_K], k_empty[ST_K], v_full[ST_V], v_empty[ST_V];
    // per S / P buffer u (tiles u, u + 3, ...): a phase can never complete twice before it is
    // awaited, because S(j + 3) waits for P V(j), which waits for P(j)
    uint64_t s_full[NS], p_full[NS], pv_done[NS];
    uint64_t s_done, pv_mma_done;
    uint64_t q_ready;               // the softmax warps have staged Q (and the tree tile)
    uint64_t anc[64];
    int32_t pos[64];
    int32_t par[64];
    float mx_x[2][2][MT];           // [tile parity][column half][row]: each half's row maximum
    float l_x[2][MT];               // [column half][row]: each half's row sum, at the end
    uint32_t tmem_base;
    int abort_flag;
};

// 2^x on the special-function unit (flushes subnormal results to zero)
E3_DEV float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction
E3_DEV float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Visibility of a row's half tile as a bit mask: bit i set when column col0 + i (i < hw) is a key the
// row sees: on the tree tile an ancestor-or-self slot below nk (anc_bits: the row's slot bits), on a
// prefix tile a key below k_hi (key0: the key of column col0).  Built once per tile, so the per-score
// test is a fixed-position bit test.
E3_DEV uint64_t visible_mask(bool tree, uint64_t anc_bits, int col0, int nk, int key0, int k_hi, int hw) {
    const int n = min(hw, tree ? nk - col0 : k_hi - key0);   // columns in range
    uint64_t m = n >= 64 ? ~0ull : (n <= 0 ? 0ull : ((1ull << n) - 1ull));
    if (tree) m &= anc_bits >> col0;                         // col0 < 64 on the tree tile
    return m;
}

// warp-uniform bounded wait (lane 0 polls, the outcome is broadcast)
E3_DEV bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort, long long limit) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, limit) ? 1 : 0;
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
                       const __grid_constant__ CUtensorMap tm_tk, const __grid_constant__ CUtensorMap tm_tv,
                       const Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ SmemStatic ss;
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    volatile int *abort = &ss.abort_flag;
    pdl_wait();   // the previous kernel's outputs (q / tree_k / caches) before any global access
    pdl_trigger();
    const int half = blockIdx.x % p.halves, split = blockIdx.x / p.halves, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rep = p.rep, nk = p.q_hi, nq = p.q_hi - p.q_lo;
    // this CTA's query slots [s_lo, s_hi) and rows (row = (slot - s_lo) * rep + head)
    const int s_lo = p.q_lo + (half ? p.s_mid : 0);
    const int s_hi = p.halves == 1 ? p.q_hi : (half ? p.q_hi : p.q_lo + p.s_mid);
    const int nrows = (s_hi - s_lo) * rep;
    const bool last = split == p.splits - 1;

    int L = p.prefix_len[b];
    if (L < 0 || L > p.max_prefix) {
        if (tid == 0 && split == 0 && g == 0 && half == 0) flag(p.dev_status, EAGLE3_DEV_CAPACITY);
        L = max(0, min(L, p.max_prefix));
    }
    const int t_lo = split * p.tiles_per_split;
    const int k_lo = min(L, t_lo * BK);
    const int k_hi = last ? L : min(L, (t_lo + p.tiles_per_split) * BK);
    const int n_prefix = (k_hi - k_lo + BK - 1) / BK;
    const int n_tiles = n_prefix + (last ? 1 : 0);
    // one 128-key prefix tile of K or V into a stage (two 64-column blocks of 16 KB).  Contiguous
    // cache: two 128-row boxes of the [B * Hkv * S, 128] view.  Paged cache: two 128-slot boxes of
    // the [n_slots, Hkv, 128] pool when pages hold a multiple of 128 positions (a tile, which starts
    // at a multiple of 128, stays inside one page), else four 64-slot boxes (a 64-aligned run stays
    // inside one page); runs past the prefix, or on a page id outside the pool, start at a negative
    // slot and read as zeros.
    const int row0 = ((b * p.Hkv + g) * p.S) + k_lo;
    auto load_prefix_tile = [&](uint8_t *dst, const CUtensorMap *map, int j, uint64_t *bar) {
        if (!p.block_table) {
            const int y = row0 + j * BK;
            tc::tma_load_2d(dst, map, 0, y, bar);
            tc::tma_load_2d(dst + KV_TILE / 2, map, 64, y, bar);
            return;
        }
        const int32_t *bt = p.block_table + (size_t)b * p.bt_stride;
        if (p.pool_box == BK) {
            const int pos = k_lo + j * BK;
            int slot = -BK;
            if (pos < L) {
                const int page = __ldg(bt + pos / p.block_size);
                if (page >= 0 && page < p.n_pages) slot = page * p.block_size + pos % p.block_size;
            }
            tc::tma_load_3d(dst, map, 0, g, slot, bar);
            tc::tma_load_3d(dst + KV_TILE / 2, map, 64, g, slot, bar);
            return;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int pos = k_lo + j * BK + 64 * h;
            int slot = -64;
            if (pos < L) {
                const int page = __ldg(bt + pos / p.block_size);
                if (page >= 0 && page < p.n_pages) slot = page * p.block_size + pos % p.block_size;
            }
            tc::tma_load_3d(dst + h * 8192, map, 0, g, slot, bar);
            tc::tma_load_3d(dst + KV_TILE / 2 + h * 8192, map, 64, g, slot, bar);
        }
    };

    // ---- phase A: barriers, TMEM, raw tree description into shared memory.  Thread 0, which is also
    // the K producer, issues the first K tiles (and Q when it arrives rotated) as soon as their
    // barriers exist, so that the loads are in flight during the rest of phase A.
    int npre = 0;                   // K tiles issued in phase A
    if (tid == 0) {
        for (int s = 0; s < ST_K; ++s) {
            tc::mbar_init(&ss.k_full[s], 1);
            tc::mbar_init(&ss.k_empty[s], 1);
        }
        for (int s = 0; s < ST_V; ++s) {
            tc::mbar_init(&ss.v_full[s], 1);
            tc::mbar_init(&ss.v_empty[s], 1);
        }
        for (int u = 0; u < NS; ++u) {
            tc::mbar_init(&ss.s_full[u], 1);
            tc::mbar_init(&ss.p_full[u], 8);
            tc::mbar_init(&ss.pv_done[u], 1);
        }
        tc::mbar_init(&ss.s_done, 1);
        tc::mbar_init(&ss.pv_mma_done, 1);
        tc::mbar_init(&ss.q_ready, 8);   // the eight staging warps
        ss.abort_flag = 0;
        tc::fence_barrier_init();
        if (n_tiles > 0) {
            npre = min(ST_K, n_prefix);   // fresh stages: nothing to wait for
            for (int j = 0; j < npre; ++j) {
                if (j == p.stall_tile) continue;   // timeout-path test: this tile never arrives
                uint8_t *dst = sm + OFF_K + j * KV_TILE;
                tc::mbar_expect_tx(&ss.k_full[j], KV_TILE);
                load_prefix_tile(dst, &tm_k, j, &ss.k_full[j]);
            }
        }
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

    auto k_tile = [&](int j) -> uint8_t * { return sm + OFF_K + (j % ST_K) * KV_TILE; };
    auto v_tile = [&](int j) -> uint8_t * { return sm + OFF_V + (j % ST_V) * KV_TILE; };

    if (warp == 0 || warp == 10) {
        // ------------------------------------------------------------------ TMA producers
        // warp 0 streams K tiles, warp 10 V tiles: the prefix from the cache, then (last split)
        // the tree tile, 64 rows of this KV head's tree keys / values (rotated beforehand)
        if (lane == 0 && n_tiles > 0) {
            const bool is_k = warp == 0;
            const int stages = is_k ? ST_K : ST_V;
            const CUtensorMap *map = is_k ? &tm_k : &tm_v;
            const CUtensorMap *tmap = is_k ? &tm_tk : &tm_tv;
            uint64_t *full = is_k ? ss.k_full : ss.v_full;
            uint64_t *empty = is_k ? ss.k_empty : ss.v_empty;
            uint8_t *ring = sm + (is_k ? OFF_K : OFF_V);
            tc::prefetch_tmap(map);
            if (last) tc::prefetch_tmap(tmap);
            // V stage 1 holds the RoPE angle table until Q is staged
            bool go = is_k || tc::mbar_wait(&ss.q_ready, 0, abort, p.wait_limit);
            const int j0 = is_k ? npre : 0;                  // thread 0 issued K tiles [0, npre) in phase A
            uint32_t issued = is_k ? (1u << npre) - 1u : 0u, last_par = 0;
            if (is_k && p.stall_tile >= 0 && p.stall_tile < npre) issued &= ~(1u << p.stall_tile);
            for (int j = j0; j < n_tiles && go; ++j) {
                const int s = j % stages;
                const uint32_t ph = (uint32_t)(j / stages) & 1u;
                if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort, p.wait_limit)) {
                    flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
                    break;
                }
                uint8_t *dst = ring + s * KV_TILE;
                if (is_k && j == p.stall_tile && j < n_prefix) continue;   // timeout-path test: never loaded
                if (j < n_prefix) {
                    tc::mbar_expect_tx(&full[s], KV_TILE);
                    load_prefix_tile(dst, map, j, &full[s]);
                } else {
                    tc::mbar_expect_tx(&full[s], 2 * BKT * 128);
                    const int y = p.tree_slot_inner ? 0 : b, z = p.tree_slot_inner ? b : 0;
                    tc::tma_load_3d(dst, tmap, g * D, y, z, &full[s]);
                    tc::tma_load_3d(dst + KV_TILE / 2, tmap, g * D + 64, y, z, &full[s]);
                }
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | (ph << s);
            }
            if (!go) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            // no TMA write may be in flight when the CTA exits (bounded)
            for (int s = 0; s < stages; ++s) {
                if (!((issued >> s) & 1u)) continue;
                const long long t0 = clock64();
                while (!tc::mbar_try(&full[s], (last_par >> s) & 1u) && clock64() - t0 < p.wait_limit) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ S = Q K^T issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t IDESC_P = tc::idesc_bf16(MT, BK);
            constexpr uint32_t IDESC_T = tc::idesc_bf16(MT, BKT);
            bool ok = tc::mbar_wait(&ss.q_ready, 0, abort, p.wait_limit);   // Q and the tree tile are staged
            const uint32_t qaddr = smem_u32(sm + OFF_Q);
            for (int j = 0; j < n_tiles && ok; ++j) {
                const bool tree = j == n_prefix;
                if (!tc::mbar_wait(&ss.k_full[j % ST_K], (uint32_t)(j / ST_K) & 1u, abort, p.wait_limit)) {
                    ok = false;
                    break;
                }
                // buffer j % 3 last held P(j - 3): P V(j - 3) must have read it (another thread issues it)
                if (j >= NS && !tc::mbar_wait(&ss.pv_done[j % NS], (uint32_t)((j - NS) / NS) & 1u, abort, p.wait_limit)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t kaddr = smem_u32(k_tile(j));
                const uint32_t kblk = KV_TILE / 2;
                const uint32_t d_s = tmem + TM_S + (uint32_t)((j % NS) * BK);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t blk = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
                    tc::mma_bf16_ss(d_s, tc::desc_sw128(qaddr + blk * (Q_TILE / 2) + kk * 32),
                                    tc::desc_sw128(kaddr + blk * kblk + kk * 32), tree ? IDESC_T : IDESC_P,
                                    k > 0 ? 1u : 0u);
                }
                tc::mma_commit(&ss.s_full[j % NS]);
                tc::mma_commit(&ss.k_empty[j % ST_K]);   // K stage free once S is done
            }
            if (!ok) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            tc::mma_commit(&ss.s_done);
            const long long t0 = clock64();
            while (!tc::mbar_try(&ss.s_done, 0) && clock64() - t0 < p.wait_limit) {
            }
        }
    } else if (warp == 11) {
        // ------------------------------------------------------------------ O += P V issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t IDESC_PV = tc::idesc_bf16_bmn(MT, D);
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const bool tree = j == n_prefix;
                if (!tc::mbar_wait(&ss.v_full[j % ST_V], (uint32_t)(j / ST_V) & 1u, abort, p.wait_limit)) {
                    ok = false;
                    break;
                }
                if (!tc::mbar_wait(&ss.p_full[j % NS], (uint32_t)(j / NS) & 1u, abort, p.wait_limit)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t vaddr = smem_u32(v_tile(j));
                const uint32_t vblk = KV_TILE / 2;
                const uint32_t t_p = tmem + TM_S + (uint32_t)((j % NS) * BK);   // P over S
                const int ksteps = (tree ? BKT : BK) / 16;
                for (int kk = 0; kk < ksteps; ++kk) {
                    tc::mma_bf16_ts(tmem, t_p + (uint32_t)(kk * 8), tc::desc_mn_sw128(vaddr + kk * 2048, vblk, 1024),
                                    IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(&ss.pv_done[j % NS]);
                tc::mma_commit(&ss.v_empty[j % ST_V]);
            }
            if (!ok) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            tc::mma_commit(&ss.pv_mma_done);
            const long long t0 = clock64();
            while (!tc::mbar_try(&ss.pv_mma_done, 0) && clock64() - t0 < p.wait_limit) {
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
                if (bad && split == 0 && g == 0 && half == 0) flag(p.dev_status, EAGLE3_DEV_BAD_TREE);
            }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");   // the eight softmax warps only
        {
            const int c = lane & 7, sub = lane >> 3;
            // RoPE angles of every position in [pos_lo, pos_lo + span), once per CTA, in V stage 1
            // (its first load waits for Q to be staged); others are computed directly
            int pos_lo = 0x7fffffff, pos_hi = -1;
            for (int i = 0; i < nk; ++i) {
                pos_lo = min(pos_lo, ss.pos[i]);
                pos_hi = max(pos_hi, ss.pos[i]);
            }
            const int span = min(pos_hi - pos_lo + 1, ROPE_TABLE_POS);
            float2 *table = reinterpret_cast<float2 *>(sm + OFF_TABLE);
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
            // Q rows of this CTA's slots: warp w8 takes slots s_lo + w8 + 8 t, lane group `sub` the
            // heads sub + 4 h; all of a warp's loads are issued before the first is used
            for (int hh = sub, h4 = 0; h4 * 4 < rep; hh += 4, ++h4) {
                uint4 lo[8], hi[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int sl = w8 + 8 * t;
                    if (s_lo + sl < s_hi && hh < rep) {
                        const __nv_bfloat16 *src = p.q + (size_t)b * p.q_sb + (size_t)(s_lo + sl) * p.q_si +
                                                   ((size_t)g * rep + hh) * D;
                        lo[t] = ld16(src + 8 * c);
                        hi[t] = ld16(src + 64 + 8 * c);
                    }
                }
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int sl = w8 + 8 * t;
                    if (s_lo + sl < s_hi && hh < rep) {
                        float cs[8], sn[8];
                        angles(ss.pos[s_lo + sl], cs, sn);
                        rope_chunks(lo[t], hi[t], cs, sn);
                        const int r = sl * rep + hh;
                        st_chunk(sm + OFF_Q, r, c, Q_TILE / 2, lo[t]);
                        st_chunk(sm + OFF_Q, r, c + 8, Q_TILE / 2, hi[t]);
                    }
                }
            }
            // zero rows of the M tile
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int k = (tid - 64); k < (MT - nrows) * 16; k += 256) {
                const int r = nrows + k / 16, ch = k % 16;
                st_chunk(sm + OFF_Q, r, ch, Q_TILE / 2, z);
            }
            tc::fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor cores
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ss.q_ready);
        }
        // two warps per TMEM lane quarter: quarter = warp % 4 (the lanes this warp may access),
        // hc = which half of the tile's columns (and of O's columns) this warp takes
        const int quarter = warp & 3;
        const int hc = w8 >> 2;
        const int rl = quarter * 32 + lane;              // row within the M tile
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint64_t bits = rl < nrows ? ss.anc[s_lo + rl / rep] : 0ull;
        float m_run = -INFINITY, l_run = 0.0f;
        bool ok = true;
        // every softmax warp runs every iteration (the row-maximum exchange is a barrier of all
        // eight): after a timeout a warp skips its waits and finishes the loop on garbage
        for (int j = 0; j < n_tiles; ++j) {
            const int u = j % NS;
            if (ok && !warp_wait(&ss.s_full[u], (uint32_t)(j / NS) & 1u, abort, p.wait_limit)) ok = false;
            tc::fence_after();
            const bool tree = j == n_prefix;             // the last split's final tile
            const int hw = (tree ? BKT : BK) / 2;        // columns of this warp: 64 (prefix) or 32 (tree)
            const int col0 = hc * hw;                    // first of them within the tile
            float sc[64];
            {
                float a[32];
                tc::tmem_ld32(t_lane + TM_S + (uint32_t)(u * BK + col0), a);
#pragma unroll
                for (int i = 0; i < 32; ++i) sc[i] = a[i];
                if (hw == 64) {
                    tc::tmem_ld32(t_lane + TM_S + (uint32_t)(u * BK + col0 + 32), a);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sc[32 + i] = a[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) sc[32 + i] = -INFINITY;
                }
            }
            const int key0 = k_lo + j * BK + col0;
            const bool full = !tree && key0 + hw <= k_hi;   // every key of this half is visible
            // the maximum is taken over the raw scores (the scale is positive, so it commutes) and
            // the scale is applied inside the exponent's argument
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (full) {
#pragma unroll
                for (int i = 0; i < 64; i += 2) mq[(i >> 1) & 3] = fmax3(mq[(i >> 1) & 3], sc[i], sc[i + 1]);
            } else {
                const uint64_t vm = visible_mask(tree, bits, col0, nk, key0, k_hi, hw);
                const uint32_t vlo = (uint32_t)vm, vhi = (uint32_t)(vm >> 32);
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const bool valid = (((i < 32) ? vlo : vhi) >> (i & 31)) & 1u;
                    sc[i] = valid ? sc[i] : -INFINITY;
                    mq[i & 3] = fmaxf(mq[i & 3], sc[i]);
                }
            }
            // row maximum of the whole tile: exchange with the warp holding the other half
            float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
            ss.mx_x[j & 1][hc][rl] = mx;
            asm volatile("bar.sync 2, 256;" ::: "memory");
            mx = fmaxf(mx, ss.mx_x[j & 1][hc ^ 1][rl]);
            const bool need = (m_run == -INFINITY) ? (mx > -INFINITY) : (mx > m_run + RESCALE_LOG2);
            const bool any_need = __any_sync(0xffffffffu, need);
            if (any_need && j > 0) {
                // O is about to be rescaled: the previous P V must be finished first
                if (ok && !warp_wait(&ss.pv_done[(j - 1) % NS], (uint32_t)((j - 1) / NS) & 1u, abort, p.wait_limit)) ok = false;
                tc::fence_after();
            }
            if (any_need) {
                const float m_new = need ? fmaxf(m_run, mx) : m_run;
                const float corr = need ? (m_run == -INFINITY ? 0.0f : fast_exp2(m_run - m_new)) : 1.0f;
                if (j > 0) {
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {   // this warp's 64 columns of O
                        float o[32];
                        const uint32_t ta = t_lane + (uint32_t)(hc * 64 + cc * 32);
                        tc::tmem_ld32(ta, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= corr;
                        tc::tmem_st32(ta, o);
                    }
                }
                l_run *= corr;
                m_run = m_new;
            }
            const float nmu = m_run == -INFINITY ? 0.0f : -m_run;
            // exponentials and this half's row sum (four chains), packed to bf16 pairs
            // (paired fp32 FMA and add: one instruction per two scores)
            uint32_t pk[32];
            float2 sq[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nmu2 = make_float2(nmu, nmu);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float2 x = __ffma2_rn(make_float2(sc[2 * e], sc[2 * e + 1]), sc2, nmu2);
                const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                sq[e & 3] = __fadd2_rn(sq[e & 3], pe);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(pe.x, pe.y);
                pk[e] = *reinterpret_cast<uint32_t *>(&h2);
            }
            const float2 s01 = __fadd2_rn(__fadd2_rn(sq[0], sq[1]), __fadd2_rn(sq[2], sq[3]));
            l_run += s01.x + s01.y;
            // P of this half over the buffer's first columns: both halves have read their scores
            // (they exchanged maxima after their loads), so the writes cannot overtake a read
            if (hw == 64)
                tc::tmem_st32u(t_lane + TM_S + (uint32_t)(u * BK + hc * 32), pk);
            else
                tc::tmem_st16u(t_lane + TM_S + (uint32_t)(u * BK + hc * 16), pk);   // tree tile: 16 columns
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ss.p_full[u]);
        }
        if (!ok && lane == 0) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
        // ---- epilogue: this warp's 64 columns of O / l
        ss.l_x[hc][rl] = l_run;
        asm volatile("bar.sync 2, 256;" ::: "memory");
        const float l_all = ss.l_x[0][rl] + ss.l_x[1][rl];
        float o[64];
        bool have = false;
        if (ok && n_tiles > 0 &&
            warp_wait(&ss.pv_done[(n_tiles - 1) % NS], (uint32_t)((n_tiles - 1) / NS) & 1u, abort, p.wait_limit)) {
            tc::fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                float t[32];
                tc::tmem_ld32(t_lane + (uint32_t)(hc * 64 + cc * 32), t);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[cc * 32 + i] = t[i];
            }
            have = true;
        }
        float m_fin = m_run, l_fin = l_all;
        if (!have) {
            m_fin = -INFINITY;
            l_fin = 0.0f;
#pragma unroll
            for (int i = 0; i < 64; ++i) o[i] = 0.0f;
        }
        if (rl < nrows) {
            const int qi = s_lo - p.q_lo + rl / rep, h = g * rep + rl % rep;
            const size_t prow_i = ((size_t)b * nq + qi) * p.Hq + h;
            if (p.splits == 1) {
                __nv_bfloat16 *dst =
                    p.out + (size_t)b * p.o_sb + (size_t)qi * p.o_si + (size_t)h * D + (size_t)hc * 64;
                const float inv_l = l_fin > 0.0f ? 1.0f / l_fin : 0.0f;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 hv = __floats2bfloat162_rn(o[cc + 2 * e] * inv_l, o[cc + 2 * e + 1] * inv_l);
                        w[e] = *reinterpret_cast<uint32_t *>(&hv);
                    }
                    *reinterpret_cast<uint4 *>(dst + cc) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                if (p.lse && hc == 0) p.lse[prow_i] = (m_fin + log2f(l_fin)) * 0.6931471805599453f;
            } else {
                const size_t rows_all = (size_t)p.B * nq * p.Hq;
                float *po = p.part_o + ((size_t)split * rows_all + prow_i) * D + (size_t)hc * 64;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 4)
                    *reinterpret_cast<float4 *>(po + cc) = make_float4(o[cc], o[cc + 1], o[cc + 2], o[cc + 3]);
                if (hc == 0) {
                    float *pm = p.part_ml + ((size_t)split * rows_all + prow_i) * 2;
                    pm[0] = m_fin;
                    pm[1] = l_fin;
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

// ------------------------------------------------------------------------------------------------
// Persistent variant for queries and tree keys that arrive rotated (qk_rotated) with a parent
// array: one CTA per SM walks the work items (sequence, KV head, split, half) c, c + grid, ...
// Barriers, TMEM and the TMA descriptors are set up once, and nothing drains between items.
// Warp roles (16 warps):
//   warp 0        TMA: K tiles into the 3-stage ring, running ahead across items
//   warp 1        S = Q K^T into one of three TMEM buffers (S(t) waits for its K tile and for
//                 P V(t - 3), which read the buffer last).  This thread also loads each item's Q:
//                 the next item's Q may only land once the item's last S has read the buffer, and
//                 S waits for it anyway, so the K producer never stalls on it
//   warp 2        TMA: V tiles into the 2-stage ring
//   warp 3        O += P V.  The S and P V MMAs come from two threads: one thread issues a
//                 tcgen05.mma with N = 128 about every 110 cycles, two threads together keep the
//                 tensor pipe at its 64-cycle rate
//   warps 4..11   softmax, two warps per TMEM lane quarter (each half of a row's 128 scores), as
//                 in verify_attn_kernel; at the end of an item they hand the row statistics (m, l)
//                 to the epilogue warps and go straight on to the next item's tiles
//   warps 12..15  epilogue, one warp per lane quarter: the normalised output rows (or the split
//                 partials) read from O as soon as the item's last P V has landed, then the
//                 ancestor bits of the next item's tree tile (from its parent array)
// TMEM: O at columns [0, 128), three S / P buffers at [128, 512).  An item's first P V waits until
// the epilogue has read the previous item's O; the S tiles queued ahead of it keep the pipe busy.
// Every ring position and barrier phase is counted over the whole CTA life (global tile counter,
// item counter n over the CTA's non-empty items), so phases stay consistent across items.
// ------------------------------------------------------------------------------------------------
constexpr int NS_P = 3;                       // S / P buffers of the persistent kernel
constexpr int NWARP_P = 16;
constexpr int NT_P = NWARP_P * 32;
constexpr uint32_t TM_S_P = 128;              // O at columns [0, 128)
static_assert(TM_S_P + NS_P * BK <= 512, "TMEM budget");

struct PersSmem {
    uint64_t k_full[ST_K], k_empty[ST_K], v_full[ST_V], v_empty[ST_V];
    uint64_t s_full[NS_P], p_full[NS_P], pv_done[NS_P];
    uint64_t q_full, q_empty;
    uint64_t o_full, o_free;                  // the item's O complete / read by the epilogue
    uint64_t anc_full[2], anc_empty[2];       // per ancestor-bit buffer (parity of the tree-tile item)
    uint64_t l_full[2], l_empty[2];           // per row-statistics buffer (item parity)
    uint64_t s_done, pv_mma_done;
    uint64_t anc[2][64];                      // [tree-item parity][slot]
    int32_t par[64];
    float mx_x[2][2][MT];                     // [tile parity][column half][row]
    float l_x[2][2][MT];                      // [item parity][column half][row]
    float m_x[2][MT];                         // [item parity][row]
    uint32_t tmem_base;
    int abort_flag;
};

struct ItemGeo {
    int b, g, split, half, L, k_lo, k_hi, n_prefix, n_tiles, s_lo, s_hi, nrows;
    bool last, clamped;
};

E3_DEV ItemGeo item_geo(const Params &p, int it) {
    ItemGeo w;
    w.half = it % p.halves;
    int r = it / p.halves;
    w.split = r % p.splits;
    r /= p.splits;
    w.g = r % p.Hkv;
    w.b = r / p.Hkv;
    w.last = w.split == p.splits - 1;
    int L = __ldg(p.prefix_len + w.b);
    w.clamped = L < 0 || L > p.max_prefix;
    w.L = L = max(0, min(L, p.max_prefix));
    const int t_lo = w.split * p.tiles_per_split;
    w.k_lo = min(L, t_lo * BK);
    w.k_hi = w.last ? L : min(L, (t_lo + p.tiles_per_split) * BK);
    w.n_prefix = (w.k_hi - w.k_lo + BK - 1) / BK;
    w.n_tiles = w.n_prefix + (w.last ? 1 : 0);
    w.s_lo = p.q_lo + (w.half ? p.s_mid : 0);
    w.s_hi = p.halves == 1 ? p.q_hi : (w.half ? p.q_hi : p.q_lo + p.s_mid);
    w.nrows = (w.s_hi - w.s_lo) * p.rep;
    return w;
}

__global__ void __launch_bounds__(NT_P, 1)
    verify_attn_pers_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_tk, const __grid_constant__ CUtensorMap tm_tv,
                            const __grid_constant__ CUtensorMap tm_q, const Params p, const int items) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ PersSmem ss;
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    volatile int *abort = &ss.abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rep = p.rep, nk = p.q_hi;
    if (tid == 0) {
        for (int s = 0; s < ST_K; ++s) {
            tc::mbar_init(&ss.k_full[s], 1);
            tc::mbar_init(&ss.k_empty[s], 1);
        }
        for (int s = 0; s < ST_V; ++s) {
            tc::mbar_init(&ss.v_full[s], 1);
            tc::mbar_init(&ss.v_empty[s], 1);
        }
        for (int u = 0; u < NS_P; ++u) {
            tc::mbar_init(&ss.s_full[u], 1);
            tc::mbar_init(&ss.p_full[u], 8);
            tc::mbar_init(&ss.pv_done[u], 1);
        }
        tc::mbar_init(&ss.o_full, 1);
        tc::mbar_init(&ss.o_free, 4);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&ss.anc_full[b], 4);
            tc::mbar_init(&ss.anc_empty[b], 8);
            tc::mbar_init(&ss.l_full[b], 256);       // every softmax thread, after its own writes
            tc::mbar_init(&ss.l_empty[b], 128);      // every epilogue thread, after its own reads
        }
        tc::mbar_init(&ss.q_full, 1);
        tc::mbar_init(&ss.q_empty, 1);
        tc::mbar_init(&ss.s_done, 1);
        tc::mbar_init(&ss.pv_mma_done, 1);
        ss.abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(&ss.tmem_base, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = ss.tmem_base;
    pdl_wait();   // the previous kernel's outputs (q / tree keys / caches) before any global access
    pdl_trigger();

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------------ TMA producers
        if (lane == 0) {
            const bool is_k = warp == 0;
            const int stages = is_k ? ST_K : ST_V;
            const CUtensorMap *map = is_k ? &tm_k : &tm_v;
            const CUtensorMap *tmap = is_k ? &tm_tk : &tm_tv;
            uint64_t *full = is_k ? ss.k_full : ss.v_full;
            uint64_t *empty = is_k ? ss.k_empty : ss.v_empty;
            uint8_t *ring = sm + (is_k ? OFF_K : OFF_V);
            tc::prefetch_tmap(map);
            tc::prefetch_tmap(tmap);
            uint32_t t = 0;
            bool go = true;
            for (int it = blockIdx.x; it < items && go; it += gridDim.x) {
                const ItemGeo w = item_geo(p, it);
                if (w.n_tiles == 0) continue;
                const int row0 = ((w.b * p.Hkv + w.g) * p.S) + w.k_lo;
                for (int j = 0; j < w.n_tiles; ++j, ++t) {
                    const int s = (int)(t % stages);
                    const uint32_t ph = (t / stages) & 1u;
                    if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort, p.wait_limit)) {
                        go = false;
                        break;
                    }
                    uint8_t *dst = ring + s * KV_TILE;
                    if (is_k && j == p.stall_tile && j < w.n_prefix) continue;   // timeout-path test: never loaded
                    if (j < w.n_prefix) {
                        tc::mbar_expect_tx(&full[s], KV_TILE);
                        if (!p.block_table) {
                            const int y = row0 + j * BK;
                            tc::tma_load_2d(dst, map, 0, y, &full[s]);
                            tc::tma_load_2d(dst + KV_TILE / 2, map, 64, y, &full[s]);
                        } else if (p.pool_box == BK) {   // one page holds the whole tile
                            const int32_t *bt = p.block_table + (size_t)w.b * p.bt_stride;
                            const int pos = w.k_lo + j * BK;
                            int slot = -BK;
                            if (pos < w.L) {
                                const int page = __ldg(bt + pos / p.block_size);
                                if (page >= 0 && page < p.n_pages) slot = page * p.block_size + pos % p.block_size;
                            }
                            tc::tma_load_3d(dst, map, 0, w.g, slot, &full[s]);
                            tc::tma_load_3d(dst + KV_TILE / 2, map, 64, w.g, slot, &full[s]);
                        } else {
                            const int32_t *bt = p.block_table + (size_t)w.b * p.bt_stride;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int pos = w.k_lo + j * BK + 64 * h;
                                int slot = -64;
                                if (pos < w.L) {
                                    const int page = __ldg(bt + pos / p.block_size);
                                    if (page >= 0 && page < p.n_pages) slot = page * p.block_size + pos % p.block_size;
                                }
                                tc::tma_load_3d(dst + h * 8192, map, 0, w.g, slot, &full[s]);
                                tc::tma_load_3d(dst + KV_TILE / 2 + h * 8192, map, 64, w.g, slot, &full[s]);
                            }
                        }
                    } else {
                        tc::mbar_expect_tx(&full[s], 2 * BKT * 128);
                        const int y = p.tree_slot_inner ? 0 : w.b, z = p.tree_slot_inner ? w.b : 0;
                        tc::tma_load_3d(dst, tmap, w.g * D, y, z, &full[s]);
                        tc::tma_load_3d(dst + KV_TILE / 2, tmap, w.g * D + 64, y, z, &full[s]);
                    }
                }
            }
            if (!go) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            // no TMA write may be in flight when the CTA exits: the last load of every stage
            for (uint32_t u = t > (uint32_t)stages ? t - stages : 0; u < t; ++u) {
                const long long t0 = clock64();
                while (!tc::mbar_try(&full[u % stages], (u / stages) & 1u) && clock64() - t0 < p.wait_limit) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ S = Q K^T issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_P = tc::idesc_bf16(MT, BK);
            constexpr uint32_t IDESC_T = tc::idesc_bf16(MT, BKT);
            const uint32_t qaddr = smem_u32(sm + OFF_Q);
            tc::prefetch_tmap(&tm_q);
            // the CTA's next item with tiles after `it`, or items
            auto next_item = [&](int it) {
                for (it += gridDim.x; it < items; it += gridDim.x)
                    if (item_geo(p, it).n_tiles > 0) return it;
                return items;
            };
            // the item's Q: two 64-column boxes (column, first head of the KV group, then slot and
            // sequence in the order of the tensor map's dimensions)
            auto load_q = [&](int it) {
                const ItemGeo w = item_geo(p, it);
                const int c1 = w.g * rep, c2 = p.tree_slot_inner ? w.s_lo : w.b, c3 = p.tree_slot_inner ? w.b : w.s_lo;
                tc::mbar_expect_tx(&ss.q_full, Q_TILE);
                tc::tma_load_4d(sm + OFF_Q, &tm_q, 0, c1, c2, c3, &ss.q_full);
                tc::tma_load_4d(sm + OFF_Q + Q_TILE / 2, &tm_q, 64, c1, c2, c3, &ss.q_full);
            };
            uint32_t kt = 0, n = 0;
            bool ok = true, q_pending = false;
            int it = next_item(blockIdx.x - (int)gridDim.x);
            if (it < items) {
                load_q(it);
                q_pending = true;
            }
            for (; it < items && ok;) {
                const ItemGeo w = item_geo(p, it);
                const int it_next = next_item(it);
                if (!tc::mbar_wait(&ss.q_full, n & 1u, abort, p.wait_limit)) {
                    ok = false;
                    break;
                }
                q_pending = false;
                for (int j = 0; j < w.n_tiles; ++j, ++kt) {
                    const bool tree = j == w.n_prefix;
                    if (!tc::mbar_wait(&ss.k_full[kt % ST_K], (kt / ST_K) & 1u, abort, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    // buffer kt % NS_P last held P(kt - 3): its P V must have read it
                    if (kt >= NS_P &&
                        !tc::mbar_wait(&ss.pv_done[kt % NS_P], ((kt - NS_P) / NS_P) & 1u, abort, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t kaddr = smem_u32(sm + OFF_K + (kt % ST_K) * KV_TILE);
                    const uint32_t d_s = tmem + TM_S_P + (kt % NS_P) * (uint32_t)BK;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t blk = (uint32_t)(k >> 2), kq = (uint32_t)(k & 3);
                        tc::mma_bf16_ss(d_s, tc::desc_sw128(qaddr + blk * (Q_TILE / 2) + kq * 32),
                                        tc::desc_sw128(kaddr + blk * (KV_TILE / 2) + kq * 32), tree ? IDESC_T : IDESC_P,
                                        k > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&ss.s_full[kt % NS_P]);
                    tc::mma_commit(&ss.k_empty[kt % ST_K]);
                }
                if (!ok) break;
                tc::mma_commit(&ss.q_empty);   // the item's S MMAs are done with Q
                if (it_next < items) {
                    // the next item's Q once this item's S MMAs have read the buffer
                    if (!tc::mbar_wait(&ss.q_empty, n & 1u, abort, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    load_q(it_next);
                    q_pending = true;
                }
                ++n;
                it = it_next;
            }
            if (!ok) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            if (q_pending) {   // no TMA write may be in flight when the CTA exits
                const long long t0 = clock64();
                while (!tc::mbar_try(&ss.q_full, n & 1u) && clock64() - t0 < p.wait_limit) {
                }
            }
            tc::mma_commit(&ss.s_done);
            const long long t0 = clock64();
            while (!tc::mbar_try(&ss.s_done, 0) && clock64() - t0 < p.wait_limit) {
            }
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------------ O += P V issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_PV = tc::idesc_bf16_bmn(MT, D);
            uint32_t vt = 0, n = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                const ItemGeo w = item_geo(p, it);
                if (w.n_tiles == 0) continue;
                for (int j = 0; j < w.n_tiles; ++j, ++vt) {
                    const bool tree = j == w.n_prefix;
                    if (!tc::mbar_wait(&ss.v_full[vt % ST_V], (vt / ST_V) & 1u, abort, p.wait_limit) ||
                        !tc::mbar_wait(&ss.p_full[vt % NS_P], (vt / NS_P) & 1u, abort, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    // the item's first P V overwrites O: the epilogue must have read the previous item's
                    if (j == 0 && n >= 1 && !tc::mbar_wait(&ss.o_free, (n - 1) & 1u, abort, p.wait_limit)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t vaddr = smem_u32(sm + OFF_V + (vt % ST_V) * KV_TILE);
                    const uint32_t t_p = tmem + TM_S_P + (vt % NS_P) * (uint32_t)BK;   // P over S
                    const int ksteps = (tree ? BKT : BK) / 16;
                    for (int kk = 0; kk < ksteps; ++kk)
                        tc::mma_bf16_ts(tmem, t_p + (uint32_t)(kk * 8),
                                        tc::desc_mn_sw128(vaddr + kk * 2048, KV_TILE / 2, 1024), IDESC_PV,
                                        (j > 0 || kk > 0) ? 1u : 0u);
                    tc::mma_commit(&ss.pv_done[vt % NS_P]);
                    tc::mma_commit(&ss.v_empty[vt % ST_V]);
                    if (j == w.n_tiles - 1) tc::mma_commit(&ss.o_full);
                }
                ++n;
            }
            if (!ok) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            tc::mma_commit(&ss.pv_mma_done);
            const long long t0 = clock64();
            while (!tc::mbar_try(&ss.pv_mma_done, 0) && clock64() - t0 < p.wait_limit) {
            }
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------------ softmax warps
        const int w8 = warp - 4;
        const int quarter = warp & 3;
        const int hc = w8 >> 2;
        const int rl = quarter * 32 + lane;              // row within the M tile
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t st = 0, n = 0, na = 0;                  // na: items with a tree tile so far
        bool ok = true;
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            const ItemGeo w = item_geo(p, it);
            if (w.n_tiles == 0) continue;
            const int n_tiles = w.n_tiles, n_prefix = w.n_prefix, k_lo = w.k_lo, k_hi = w.k_hi;
            const int anc_slot = rl < w.nrows ? w.s_lo + rl / rep : -1;
            const uint32_t o_acc = t_lane;
            float m_run = -INFINITY, l_run = 0.0f;
            for (int j = 0; j < n_tiles; ++j, ++st) {
                const int u = (int)(st % NS_P);
                if (ok && !warp_wait(&ss.s_full[u], (st / NS_P) & 1u, abort, p.wait_limit)) ok = false;
                tc::fence_after();
                const bool tree = j == n_prefix;
                const int hw = (tree ? BKT : BK) / 2;
                const int col0 = hc * hw;
                const uint32_t t_s = t_lane + TM_S_P + (uint32_t)(u * BK);
                float sc[64];
                {
                    float a[32];
                    tc::tmem_ld32(t_s + (uint32_t)col0, a);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sc[i] = a[i];
                    if (hw == 64) {
                        tc::tmem_ld32(t_s + (uint32_t)(col0 + 32), a);
#pragma unroll
                        for (int i = 0; i < 32; ++i) sc[32 + i] = a[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) sc[32 + i] = -INFINITY;
                    }
                }
                const int key0 = k_lo + j * BK + col0;
                const bool full = !tree && key0 + hw <= k_hi;
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (full) {
#pragma unroll
                    for (int i = 0; i < 64; i += 2) mq[(i >> 1) & 3] = fmax3(mq[(i >> 1) & 3], sc[i], sc[i + 1]);
                } else {
                    uint64_t bits = 0ull;
                    if (tree) {   // the epilogue warps have walked this item's tree
                        if (ok && !warp_wait(&ss.anc_full[na & 1u], (na >> 1) & 1u, abort, p.wait_limit)) ok = false;
                        if (anc_slot >= 0) bits = ss.anc[na & 1u][anc_slot];
                    }
                    const uint64_t vm = visible_mask(tree, bits, col0, nk, key0, k_hi, hw);
                    const uint32_t vlo = (uint32_t)vm, vhi = (uint32_t)(vm >> 32);
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const bool valid = (((i < 32) ? vlo : vhi) >> (i & 31)) & 1u;
                        sc[i] = valid ? sc[i] : -INFINITY;
                        mq[i & 3] = fmaxf(mq[i & 3], sc[i]);
                    }
                }
                // exchange buffers alternate with the CTA-wide tile count, so that consecutive tiles
                // (also across items) never share one
                float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
                ss.mx_x[st & 1][hc][rl] = mx;
                asm volatile("bar.sync 2, 256;" ::: "memory");
                mx = fmaxf(mx, ss.mx_x[st & 1][hc ^ 1][rl]);
                const bool need = (m_run == -INFINITY) ? (mx > -INFINITY) : (mx > m_run + RESCALE_LOG2);
                const bool any_need = __any_sync(0xffffffffu, need);
                float corr = 1.0f;
                if (any_need) {
                    const float m_new = need ? fmaxf(m_run, mx) : m_run;
                    corr = need ? (m_run == -INFINITY ? 0.0f : fast_exp2(m_run - m_new)) : 1.0f;
                    l_run *= corr;
                    m_run = m_new;
                }
                const float nmu = m_run == -INFINITY ? 0.0f : -m_run;
                uint32_t pk[32];
                float2 sq[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nmu2 = make_float2(nmu, nmu);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float2 x = __ffma2_rn(make_float2(sc[2 * e], sc[2 * e + 1]), sc2, nmu2);
                    const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                    sq[e & 3] = __fadd2_rn(sq[e & 3], pe);
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(pe.x, pe.y);
                    pk[e] = *reinterpret_cast<uint32_t *>(&h2);
                }
                const float2 s01 = __fadd2_rn(__fadd2_rn(sq[0], sq[1]), __fadd2_rn(sq[2], sq[3]));
                l_run += s01.x + s01.y;
                if (hw == 64)
                    tc::tmem_st32u(t_s + (uint32_t)(hc * 32), pk);
                else
                    tc::tmem_st16u(t_s + (uint32_t)(hc * 16), pk);
                // O rescaled (the scores are dead by now) once P V of the previous tile has landed in
                // it, and before this tile's P V, which waits for the P arrival below
                if (any_need && j > 0) {
                    if (ok && !warp_wait(&ss.pv_done[(st - 1) % NS_P], ((st - 1) / NS_P) & 1u, abort, p.wait_limit))
                        ok = false;
                    tc::fence_after();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        float o[32];
                        const uint32_t ta = o_acc + (uint32_t)(hc * 64 + cc * 32);
                        tc::tmem_ld32(ta, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= corr;
                        tc::tmem_st32(ta, o);
                    }
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ss.p_full[u]);
            }
            // the item's ancestor bits are no longer read; its row statistics go to the epilogue
            if (w.last) {
                if (lane == 0) tc::mbar_arrive(&ss.anc_empty[na & 1u]);
                ++na;
            }
            if (n >= 2 && ok && !warp_wait(&ss.l_empty[n & 1u], ((n - 2) >> 1) & 1u, abort, p.wait_limit)) ok = false;
            ss.l_x[n & 1u][hc][rl] = l_run;
            if (hc == 0) ss.m_x[n & 1u][rl] = m_run;
            tc::mbar_arrive(&ss.l_full[n & 1u]);
            ++n;
        }
        if (!ok && lane == 0) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
    } else if (warp >= 12) {
        // ------------------------------------------------------------------ epilogue warps
        const int quarter = warp & 3;
        const int rl = quarter * 32 + lane;
        const int te = tid - 12 * 32;                    // 0..127
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const int nq = p.q_hi - p.q_lo;
        const size_t rows_all = (size_t)p.B * nq * p.Hq;
        bool ok = true;
        uint32_t n = 0, na = 0;
        // ancestor-or-self bits of a tree-tile item's tree into ss.anc[m & 1] (m counts those items): slot i
        // walks its own parent chain
        auto prepare_anc = [&](const ItemGeo &w, uint32_t m, int par_val) {
            if (m >= 2 && ok && !warp_wait(&ss.anc_empty[m & 1u], ((m - 2) >> 1) & 1u, abort, p.wait_limit)) ok = false;
            if (te < nk) ss.par[te] = par_val;
            asm volatile("bar.sync 3, 128;" ::: "memory");
            if (te < nk) {
                auto invalid = [&](int j) {
                    const int pj = ss.par[j];
                    return j == 0 ? pj != -1 : (pj < 0 || pj >= j);
                };
                uint64_t bits = 1ull << te;
                int j = te;
                const bool bad = invalid(te);
                while (j > 0 && !invalid(j)) {
                    j = ss.par[j];
                    bits |= 1ull << j;
                }
                ss.anc[m & 1u][te] = bits;
                if (bad && w.g == 0 && w.half == 0) flag(p.dev_status, EAGLE3_DEV_BAD_TREE);
            }
            asm volatile("bar.sync 3, 128;" ::: "memory");   // every walk done before ss.par changes
            if (lane == 0) tc::mbar_arrive(&ss.anc_full[m & 1u]);
        };
        auto epilogue = [&](const ItemGeo &w, uint32_t m) {
            bool have = ok && warp_wait(&ss.l_full[m & 1u], (m >> 1) & 1u, abort, p.wait_limit);
            const float l_all = ss.l_x[m & 1u][0][rl] + ss.l_x[m & 1u][1][rl];
            const float m_row = ss.m_x[m & 1u][rl];
            tc::mbar_arrive(&ss.l_empty[m & 1u]);
            have = have && warp_wait(&ss.o_full, m & 1u, abort, p.wait_limit);
            if (!have) ok = false;
            tc::fence_after();
            const float m_fin = have ? m_row : -INFINITY, l_fin = have ? l_all : 0.0f;
            const bool row_ok = rl < w.nrows;
            const int qi = w.s_lo - p.q_lo + rl / rep, h = w.g * rep + rl % rep;
            const size_t prow_i = ((size_t)w.b * nq + qi) * p.Hq + h;
            const float inv_l = l_fin > 0.0f ? 1.0f / l_fin : 0.0f;
            const uint32_t o_acc = t_lane;
            if (p.splits == 1) {
                __nv_bfloat16 *dst = p.out + (size_t)w.b * p.o_sb + (size_t)qi * p.o_si + (size_t)h * D;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    float t[32];
                    tc::tmem_ld32(o_acc + (uint32_t)(cc * 32), t);   // warp-collective
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        __nv_bfloat162 hv = __floats2bfloat162_rn(have ? t[2 * e] * inv_l : 0.0f,
                                                                  have ? t[2 * e + 1] * inv_l : 0.0f);
                        pk[e] = *reinterpret_cast<uint32_t *>(&hv);
                    }
                    if (row_ok) {
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8)
                            *reinterpret_cast<uint4 *>(dst + cc * 32 + 8 * c8) =
                                make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
                    }
                }
            } else {
                float *po = p.part_o + ((size_t)w.split * rows_all + prow_i) * D;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    float t[32];
                    tc::tmem_ld32(o_acc + (uint32_t)(cc * 32), t);   // warp-collective
                    if (!row_ok) continue;
#pragma unroll
                    for (int c4 = 0; c4 < 32; c4 += 4)
                        *reinterpret_cast<float4 *>(po + cc * 32 + c4) =
                            have ? make_float4(t[c4], t[c4 + 1], t[c4 + 2], t[c4 + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ss.o_free);
            if (row_ok) {
                if (p.splits == 1) {
                    if (p.lse) p.lse[prow_i] = (m_fin + log2f(l_fin)) * 0.6931471805599453f;
                } else {
                    float *pm = p.part_ml + ((size_t)w.split * rows_all + prow_i) * 2;
                    pm[0] = m_fin;
                    pm[1] = l_fin;
                }
            }
        };
        ItemGeo prev;
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            const ItemGeo w = item_geo(p, it);
            const bool first_of_seq = w.split == 0 && w.g == 0 && w.half == 0;
            if (w.clamped && first_of_seq && te == 0) flag(p.dev_status, EAGLE3_DEV_CAPACITY);
            if (w.n_tiles == 0) {
                // an empty split: its partial (m = -inf, l = 0, O = 0) for the merge
                if (p.splits > 1 && rl < w.nrows) {
                    const int qi = w.s_lo - p.q_lo + rl / rep, h = w.g * rep + rl % rep;
                    const size_t prow_i = ((size_t)w.b * nq + qi) * p.Hq + h;
                    float *po = p.part_o + ((size_t)w.split * rows_all + prow_i) * D;
                    for (int cc = 0; cc < D; cc += 4) *reinterpret_cast<float4 *>(po + cc) = make_float4(0.f, 0.f, 0.f, 0.f);
                    float *pm = p.part_ml + ((size_t)w.split * rows_all + prow_i) * 2;
                    pm[0] = -INFINITY;
                    pm[1] = 0.0f;
                }
                continue;
            }
            // the parent values load while the previous item's epilogue waits for its last P V; only
            // an item with the tree tile (the last split) needs the ancestor bits
            const int par_val = (w.last && te < nk) ? __ldg(p.parents + (size_t)w.b * p.n_slots + te) : 0;
            if (n >= 1) epilogue(prev, n - 1);
            if (w.last) prepare_anc(w, na++, par_val);
            prev = w;
            ++n;
        }
        if (n >= 1) epilogue(prev, n - 1);
        if (!ok && lane == 0) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// Rotated tree keys back into tree_k: eight threads per (sequence, query slot, KV head) row, four
// rows per warp, at the slot's position (prefix length + depth from the parent array, or the given
// position), with the same angle arguments and arithmetic the attention kernel uses for Q.
__global__ void tree_rotate_kernel(const Params p) {
    pdl_wait();
    pdl_trigger();
    const int nq = p.q_hi - p.q_lo;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t w = t >> 3;                    // row
    if (w >= (int64_t)p.B * nq * p.Hkv) return;
    const int g = (int)(w % p.Hkv);
    const int i = p.q_lo + (int)((w / p.Hkv) % nq);
    const int b = (int)(w / ((int64_t)p.Hkv * nq));
    int pos;
    if (p.parents) {
        int L = p.prefix_len[b];
        L = max(0, min(L, p.max_prefix));
        const int32_t *par = p.parents + (size_t)b * p.n_slots;
        auto invalid = [&](int j) {
            const int pj = par[j];
            return j == 0 ? pj != -1 : (pj < 0 || pj >= j);
        };
        int d = 0, j = i;
        while (j > 0 && !invalid(j)) {
            j = par[j];
            ++d;
        }
        pos = L + d;
    } else {
        pos = p.pos[(size_t)b * p.pos_sb + i];
    }
    const int c = (int)(t & 7);                  // 16-byte chunks c and c + 8 (dims 8c.. and 64 + 8c..)
    __nv_bfloat16 *kg = p.k + (size_t)b * p.k_sb + (size_t)i * p.k_si + (size_t)g * D;
    uint4 lo = ld16(kg + 8 * c), hi = ld16(kg + 64 + 8 * c);
    float cs[8], sn[8];
    rope_angles((float)pos, p.inv_freq, c, cs, sn);
    rope_chunks(lo, hi, cs, sn);
    *reinterpret_cast<uint4 *>(kg + 8 * c) = lo;
    *reinterpret_cast<uint4 *>(kg + 64 + 8 * c) = hi;
}

// Merge split partials in split order: one warp per (b, query slot, head) row.
__global__ void verify_combine_kernel(const Params p) {
    pdl_wait();
    pdl_trigger();
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
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000)ptr;
        return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    }();
    return fn;
}

// [rows, 128] bf16 cache viewed as a 2-D tensor; 64 x 64 boxes, 128-byte swizzle
// tree K or V of one launch part as a 3-D tensor of the Hkv * D elements of a node, the slots < nk
// and the sequences, the outer two ordered by pitch (slot-major when the slot pitch is the smaller);
// boxes of 64 elements x 64 slots x 1 sequence, 128-byte swizzle: in shared memory a box is 64 slot
// rows of 128 B, laid out like the first 64 keys of a cache tile; slots >= nk read as zeros
bool make_tree_map(CUtensorMap *m, const void *base, int nb, int nk, int64_t kv_width, int64_t sb, int64_t si) {
    auto fn = encode_fn();
    if (!fn) return false;
    const bool slot_inner = si <= sb;
    const cuuint64_t dims[3] = {(cuuint64_t)kv_width, (cuuint64_t)(slot_inner ? nk : nb), (cuuint64_t)(slot_inner ? nb : nk)};
    const cuuint64_t strides[2] = {(cuuint64_t)(slot_inner ? si : sb) * 2, (cuuint64_t)(slot_inner ? sb : si) * 2};
    const cuuint32_t box[3] = {64, slot_inner ? (cuuint32_t)BKT : 1u, slot_inner ? 1u : (cuuint32_t)BKT};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [B, slots, Hq, 128] (slot or batch pitch outermost) as a 4-D tensor whose box is one KV head's
// rep query heads x MT / rep slots x 64 columns: the box lands as rows slot * rep + head, 128-byte
// swizzled like the other tiles
bool make_q_map(CUtensorMap *m, const void *base, int nb, int n_slots, int Hq, int rep, int64_t sb, int64_t si) {
    auto fn = encode_fn();
    if (!fn || rep < 1 || MT % rep || MT / rep > 256 || ((uintptr_t)base & 15) || (sb % 8) || (si % 8)) return false;
    const bool slot_inner = si <= sb;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)(slot_inner ? n_slots : nb),
                                (cuuint64_t)(slot_inner ? nb : n_slots)};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)(slot_inner ? si : sb) * 2,
                                   (cuuint64_t)(slot_inner ? sb : si) * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)rep, slot_inner ? (cuuint32_t)(MT / rep) : 1u,
                               slot_inner ? 1u : (cuuint32_t)(MT / rep)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// paged pool [n_slots, Hkv, 128] as a 3-D tensor (columns, head, slot); boxes of 64 columns x 1
// head x box_slots (64 or 128) slots land like that many rows of a cache tile
bool make_pool_map(CUtensorMap *m, const void *base, int64_t n_slots, int Hkv, int box_slots) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)n_slots};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_slots};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
    const int n = device_sm_count();
    return n > 0 ? n : 1;
}

// Query rows of a (sequence, KV head): one 128-row M tile per CTA; more rows are cut into two
// halves of whole slots.  Returns the CTAs per (sequence, KV head, split) and the first half's
// slot count, or 0 when the rows do not fit (a half would exceed 128 rows).
int plan_halves(int nq, int rep, int *s_mid) {
    if (nq * rep <= MT) {
        *s_mid = nq;
        return 1;
    }
    const int mid = (nq + 1) / 2;
    if (mid * rep > MT || (nq - mid) * rep > MT) return 0;
    *s_mid = mid;
    return 2;
}

// A launch covers sequences [b0, b0 + nb) with `splits` KV splits.  When the (sequence, KV head)
// blocks fill some waves of the GPU and leave a tail smaller than half a wave, the full waves run
// unsplit and the tail sequences are split over the SMs the tail would leave idle.
struct Part {
    int b0, nb, splits;
};

int plan_parts(const AttnLaunch &a, Part parts[2]) {
    const int sms = sm_count_cached();
    int s_mid = 0;
    const int per_b = a.Hkv * max(1, plan_halves(a.q_hi - a.q_lo, a.Hq / a.Hkv, &s_mid));   // CTAs per sequence
    const int items = a.B * per_b;
    if (a.num_splits == 0 && items > sms && items % sms) {
        const int b0 = (items / sms) * sms / per_b;
        const int tail = (a.B - b0) * per_b;
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
    p.halves = plan_halves(nq, p.rep, &p.s_mid);
    if (p.halves == 0) return EAGLE3_ERR_UNSUPPORTED;
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
    const int nk_all = a.q_hi;                       // tree slots visible as keys
    p.tree_slot_inner = a.k_si <= a.k_sb ? 1 : 0;
    if ((a.v_si <= a.v_sb ? 1 : 0) != p.tree_slot_inner) return EAGLE3_ERR_UNSUPPORTED;
    p.block_table = a.block_table ? a.block_table + b0 * a.bt_stride : nullptr;
    p.bt_stride = a.bt_stride;
    p.block_size = a.block_size;
    p.n_pages = a.block_table ? a.pool_slots / a.block_size : 0;
    p.pool_box = a.block_table && a.block_size % BK == 0 ? BK : 64;
    if (a.block_table) {
        if (!make_pool_map(&mk, a.k_cache, a.pool_slots, a.Hkv, p.pool_box) ||
            !make_pool_map(&mv, a.v_cache, a.pool_slots, a.Hkv, p.pool_box))
            return EAGLE3_ERR_CUDA;
    } else {
        const size_t cache_off = b0 * a.Hkv * a.S * D;
        const int64_t cache_rows = (int64_t)pt.nb * a.Hkv * a.S;
        if (!make_cache_map(&mk, a.k_cache + cache_off, cache_rows) ||
            !make_cache_map(&mv, a.v_cache + cache_off, cache_rows))
            return EAGLE3_ERR_CUDA;
    }
    CUtensorMap mtk, mtv;
    if (!make_tree_map(&mtk, p.k, pt.nb, nk_all, (int64_t)a.Hkv * D, a.k_sb, a.k_si) ||
        !make_tree_map(&mtv, p.v, pt.nb, nk_all, (int64_t)a.Hkv * D, a.v_sb, a.v_si))
        return EAGLE3_ERR_CUDA;
    p.qk_rotated = a.qk_rotated ? 1 : 0;
    p.stall_tile = a.stall_tile;
    p.wait_limit = a.wait_limit;
    CUtensorMap mq = mk;   // unused unless Q arrives rotated
    if (p.qk_rotated) {
        if ((a.q_si <= a.q_sb ? 1 : 0) != p.tree_slot_inner) return EAGLE3_ERR_UNSUPPORTED;
        if (!make_q_map(&mq, p.q, pt.nb, a.n_slots, a.Hq, p.rep, a.q_sb, a.q_si)) return EAGLE3_ERR_UNSUPPORTED;
    } else {
        // the query slots' keys rotated in tree_k first; the attention streams them like the prefix
        const int64_t warps = (int64_t)pt.nb * nq * a.Hkv;
        if (launch_pdl(tree_rotate_kernel, dim3((unsigned)((warps + 31) / 32)), dim3(256), 0, stream, p) !=
            cudaSuccess)   // 32 rows per block
            return EAGLE3_ERR_CUDA;
    }
    if (p.qk_rotated) {
        // rotated q (always with a parent array): one persistent CTA per SM walks the work items
        const int items = splits * p.halves * a.Hkv * pt.nb;
        const int grid = std::min(items, sm_count_cached());
        if (launch_pdl(verify_attn_pers_kernel, dim3(grid), dim3(NT_P), SMEM_DYN, stream, mk, mv, mtk, mtv, mq, p,
                       items) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
    } else if (launch_pdl(verify_attn_kernel, dim3(splits * p.halves, a.Hkv, pt.nb), dim3(NT), SMEM_DYN, stream, mk,
                          mv, mtk, mtv, p) != cudaSuccess) {
        return EAGLE3_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (splits > 1) {
        if (launch_pdl(verify_combine_kernel, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, stream, p) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
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
    // rotated q runs on the persistent kernel, which walks a parent array (ancestor masks: in-call RoPE)
    if (a.qk_rotated && !a.parents) return EAGLE3_ERR_UNSUPPORTED;
    const size_t need = tree_attn_workspace(a);
    if (need && (!workspace || ws_bytes < need || ((uintptr_t)workspace & 15))) return EAGLE3_ERR_WORKSPACE;
    // rows of q / tree k / tree v / out are moved 16 bytes at a time
    const int64_t strides[] = {a.q_sb, a.q_si, a.k_sb, a.k_si, a.v_sb, a.v_si, a.o_sb, a.o_si};
    for (int64_t st : strides)
        if (st % 8) return EAGLE3_ERR_INVALID_ARGUMENT;
    const void *row_bases[] = {a.q, a.k, a.v, a.out};
    for (const void *r : row_bases)
        if ((uintptr_t)r & 15) return EAGLE3_ERR_INVALID_ARGUMENT;
    static PerDevice<cudaError_t> attr;
    if (attr.get([] {
            cudaError_t e = cudaFuncSetAttribute(verify_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)SMEM_DYN);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(verify_attn_pers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_DYN);
            return e;
        }) != cudaSuccess)
        return EAGLE3_ERR_CUDA;
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
        (!a->block_table && a->s_max < 1) || a->max_prefix_len < 0 || a->num_splits < 0 || a->q_node_stride < 0 || a->kv_node_stride < 0)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->n_heads % a->n_kv_heads) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->head_dim != D || a->n_nodes > 64) return EAGLE3_ERR_UNSUPPORTED;
    int s_mid = 0;
    if (!plan_halves(a->n_nodes, a->n_heads / a->n_kv_heads, &s_mid)) return EAGLE3_ERR_UNSUPPORTED;
    if (a->block_table) {
        if (a->block_size < 64 || a->block_size % 64 || a->max_blocks < 1 || a->n_slots < a->block_size)
            return EAGLE3_ERR_INVALID_ARGUMENT;
        if ((int64_t)a->max_blocks * a->block_size < a->max_prefix_len) return EAGLE3_ERR_CAPACITY;
    } else if ((int64_t)a->max_prefix_len + a->n_nodes > a->s_max) {
        return EAGLE3_ERR_CAPACITY;
    }
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
    l.qk_rotated = a->qk_rotated ? 1 : 0;
    l.block_table = a->block_table;
    l.bt_stride = a->max_blocks;
    l.block_size = a->block_size;
    l.pool_slots = a->n_slots;
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

extern "C" eagle3_status_t eagle3_test_verify_attn_timeout(const eagle3_verify_attn_args_t *a, void *workspace,
                                                           size_t ws_bytes, int32_t stall_tile,
                                                           int64_t wait_limit_cycles, eagle3_stream_t stream) {
    if (stall_tile < 0 || wait_limit_cycles < 1000 || wait_limit_cycles > WAIT_LIMIT_CYCLES)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    const eagle3_status_t st = verify_validate(a);
    if (st != EAGLE3_OK || a->batch == 0) return st;
    AttnLaunch l = verify_launch(a);
    l.stall_tile = stall_tile;
    l.wait_limit = wait_limit_cycles;
    return tree_attn_launch(l, workspace, ws_bytes, (cudaStream_t)stream);
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

// Host code cannot use the array's name as a device address: look the address up with the device
// current and keep it per device, tagged with the CUDA context it belongs to.  A context that was
// destroyed and recreated (cudaDeviceReset, or the primary context released and retained again)
// loads the module anew, so the address is looked up again when the current context changes.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CUcontext current_context() {
    static const CtxGetCurrentFn fn = [] {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (CtxGetCurrentFn)ptr;
        return (CtxGetCurrentFn) nullptr;
    }();
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

void *noalloc_scratch_address() {
    static std::mutex mu;
    static void *addr[128] = {nullptr};
    static CUcontext owner[128] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(mu);
    if (!ctx || !addr[dev] || owner[dev] != ctx) {
        void *p = nullptr;   // the lookup also makes the device's primary context current
        if (cudaGetSymbolAddress(&p, g_verify_noalloc_scratch) != cudaSuccess) return nullptr;
        ctx = current_context();
        if (!ctx) return nullptr;
        addr[dev] = p;
        owner[dev] = ctx;
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
