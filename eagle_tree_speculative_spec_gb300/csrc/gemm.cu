// Tensor-core linear layer y = x W^T on tcgen05 / TMEM (bf16 in, fp32 accumulate), the
// contraction behind every projection of the draft head and the target layers ("EAGLE-3:
// Engineering Implementation of LLM Inference Acceleration", section VIII and appendix C:
// fc, q/k/v/o, gate/up/down and lm_head are bias-free nn.Linear layers).
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: 128B-swizzled A (x) and B (W) tiles into a STAGES-deep ring
//   warp 1      TMEM owner; lane 0 issues tcgen05.mma (M=128, N=BN, K=16) and commits
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, fused epilogue, stores
// The accumulator is double-buffered in TMEM (2 x BN fp32 columns), so the epilogue of one tile
// overlaps the main loop of the next.  Work units are (m tile, n tile, k split), m fastest, so
// concurrently running CTAs share the same weight tile in L2.  With more than one k split the
// fp32 partials go to a workspace and a second kernel adds them in split order and applies the
// epilogue (deterministic).  A single M tile with at most two waves of N tiles takes the split
// count (up to 8) whose units fill their last wave best: those launches stream weights with few
// rows.  Outputs leave through 128B-swizzled shared memory and TMA stores where the output allows
// it.  The RoPE epilogue (q/k heads of a fused QKV projection, rotated before rounding) is a
// separate instantiation of the kernel.
//
// Stream-K: when the output tiles do not fill whole waves of the GPU, all but the last full wave
// run as above (m fastest, so the CTAs of a wave share weight tiles in L2), and the remaining
// tiles' (tile, k-block) iterations are cut into equal contiguous shares, one per CTA.  A tile cut by a share boundary is
// finished by the CTA that covers its first k-block (it reaches that tile last, at the end of its
// share): the CTAs covering the rest of the tile wrote their fp32 accumulators to a workspace slot
// at the start of their own shares and raised a flag; the owner adds the slots in CTA order
// (deterministic) and applies the epilogue.  Blocks wait on one another here, so this mode is a
// cooperative launch (all CTAs resident), and the waits are bounded like every other wait.
//
// Every mbarrier wait is bounded; on a timeout the kernel records EAGLE3_DEV_TIMEOUT, stops
// issuing work, drains its own TMA loads and frees its TMEM.
#include <algorithm>
#include <cudaTypedefs.h>

#include "../../include/eagle3_linear.h"
#include "tc.cuh"

namespace e3 {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int NTHREADS = 192;

struct GemmParams {
    int M, N, K, epi;
    int tiles_m, tiles_n, splits, kb_total, kb_per_split, units;
    int n_acc;                       // accumulator columns per row of the partial workspace
    void *out;
    int64_t ld_out;
    const __nv_bfloat16 *residual;
    int64_t ld_res;
    float *ws;                       // [splits][M][n_acc] fp32 partials (splits > 1)
    int streamk;                     // stream-K schedule (cooperative launch)
    int dp_tiles;                    // stream-K: tiles [0, dp_tiles) run whole, data-parallel
    long long T;                     // stream-K: (tiles - dp_tiles) * kb_total iterations, shared out
    float4 *sk_part;                 // stream-K: [grid][BN / 4][BM] fp32 accumulator slots (float4 of
                                     // 4 columns, rows fastest: a warp's 32 rows are 512 contiguous bytes)
    int *sk_flag;                    // stream-K: [grid] warps of the slot's CTA that have written it
    int tma_out;                     // outputs leave through shared memory and TMA stores
    int32_t *dev_status;
    // BF16_ROPE: columns [0, rope_cols) rotated per 128-wide head at row position
    // rope_base[row / rope_rows] + rope_depth[row]
    int rope_cols, rope_rows;
    const int32_t *rope_base, *rope_depth;
    float rope_inv[64];              // theta^(-2j/128), computed in double, rounded to float
    uint32_t *row_max;               // F32: [M] atomic max of each row's output order keys, or null
    // split tail: whole waves of tiles run data-parallel (tiles [0, tail_dp)); each tile of the
    // partial last wave is split into tail_splits k-ranges whose fp32 partials go to tail_ws
    // ([unit][BM][n_acc per tile] in unit order) and a second kernel adds them in split order
    int tail_dp, tail_splits;
    float *tail_ws;
    // when set and the word it points to is 0 (read after the previous kernel completed), the
    // launch does nothing: a caller whose row count is known only on the device skips idle launches
    const int32_t *skip_if_zero;
    // folded RMSNorm: row_ssq [tiles_n][M] out (bf16 epilogues, the squares of the stored outputs per
    // row and tile); ssq_in [ssq_blocks][M]: each accumulator row scaled by
    // rsqrt(sum / ssq_dim + ssq_eps) before the epilogue
    float *row_ssq;
    const float *ssq_in;
    int ssq_blocks;
    float ssq_inv_dim, ssq_eps;
};

// the folded RMSNorm's scale of a row (1 without row_ssq_in): the blocks' sums added in block order
E3_DEV float row_norm_scale(const GemmParams &p, int row) {
    if (!p.ssq_in || row >= p.M) return 1.0f;
    float s = 0.0f;
    for (int b = 0; b < p.ssq_blocks; ++b) s += __ldg(p.ssq_in + (size_t)b * p.M + row);
    return rsqrtf(s * p.ssq_inv_dim + p.ssq_eps);
}

// sum of squares of eight bf16 pairs (as stored), added in order
E3_DEV float ssq_bf16x8(const uint4 &u, float acc) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
        acc = fmaf(f.x, f.x, acc);
        acc = fmaf(f.y, f.y, acc);
    }
    return acc;
}

E3_DEV bool skipped(const GemmParams &p) { return p.skip_if_zero && *(volatile const int32_t *)p.skip_if_zero == 0; }

// Order key of each of 32 outputs at columns col0.. (those < N), folded into a running maximum.
E3_DEV uint32_t chunk_max_key(uint32_t run, const float (&v)[32], int col0, int N) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (col0 + i < N) run = max(run, order_key(v[i]));
    return run;
}

// One piece of work of a CTA: k-blocks [kb0, kb1) of output tile (mb, nb).
enum { IT_FULL = 0, IT_SPLITK = 1, IT_CONTRIB = 2, IT_OWNER = 3, IT_TAIL = 4 };
struct Item {
    int mb, nb, sp, kb0, kb1, kind, u;
};

// The same sequence of items for the producer, the MMA issuer and the epilogue of a CTA.
// first k-block iteration (counted from the first stream-K tile) of CTA c's share
E3_DEV long long sk_start(const GemmParams &p, long long c) { return p.T * c / gridDim.x; }

struct WorkIter {
    int unit;
    long long it, it1;
    E3_DEV void init(const GemmParams &p) {
        unit = blockIdx.x;
        if (p.streamk) {
            it = (long long)p.dp_tiles * p.kb_total + sk_start(p, blockIdx.x);
            it1 = (long long)p.dp_tiles * p.kb_total + sk_start(p, blockIdx.x + 1);
        }
    }
    E3_DEV bool next(const GemmParams &p, Item &w) {
        if (p.streamk && unit < p.dp_tiles) {
            w.u = unit;
            w.mb = unit % p.tiles_m;
            w.nb = unit / p.tiles_m;
            w.sp = 0;
            w.kb0 = 0;
            w.kb1 = p.kb_total;
            w.kind = IT_FULL;
            unit += gridDim.x;
            return true;
        }
        if (p.streamk) {
            if (it >= it1) return false;
            w.u = (int)(it / p.kb_total);
            w.kb0 = (int)(it % p.kb_total);
            w.kb1 = (int)min((long long)p.kb_total, (long long)w.kb0 + (it1 - it));
            w.mb = w.u % p.tiles_m;
            w.nb = w.u / p.tiles_m;
            w.sp = 0;
            w.kind = (w.kb0 == 0 && w.kb1 == p.kb_total) ? IT_FULL : (w.kb0 > 0 ? IT_CONTRIB : IT_OWNER);
            it += w.kb1 - w.kb0;
            return true;
        }
        if (unit >= p.units) return false;
        if (p.tail_splits > 1 && unit >= p.tail_dp) {
            // a k-range of a tile of the partial last wave; w.u = its partial slot
            const int v = unit - p.tail_dp, t = p.tail_dp + v / p.tail_splits;
            w.u = v;
            w.mb = t % p.tiles_m;
            w.nb = t / p.tiles_m;
            w.sp = v % p.tail_splits;
            w.kb0 = w.sp * p.kb_per_split;
            w.kb1 = min(p.kb_total, w.kb0 + p.kb_per_split);
            w.kind = IT_TAIL;
            unit += gridDim.x;
            return true;
        }
        w.u = unit;
        w.mb = unit % p.tiles_m;
        const int r = unit / p.tiles_m;
        w.nb = r % p.tiles_n;
        w.sp = r / p.tiles_n;
        w.kb0 = p.tail_splits > 1 ? 0 : w.sp * p.kb_per_split;
        w.kb1 = p.tail_splits > 1 ? p.kb_total : min(p.kb_total, w.kb0 + p.kb_per_split);
        w.kind = p.splits > 1 ? IT_SPLITK : IT_FULL;
        unit += gridDim.x;
        return true;
    }
};

template <int BN>
struct Cfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    // epilogue staging: per epilogue warp two boxes of 32 rows x 128 bytes (128B-swizzled)
    static constexpr int EPI_BOX = 32 * 128;
    static constexpr int EPI_BYTES = 4 * 2 * EPI_BOX;
    static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 1024 /* align */ + 256 /* barriers */;
    static_assert(SMEM <= 232448, "shared memory budget");
};

E3_DEV float silu(float x) { return x / (1.0f + __expf(-x)); }

// sin and cos of an fp32 RoPE angle (|a| < 2^17): Cody-Waite reduction by 2 pi with a three-part
// float split of 2 pi (each product exact inside its fused multiply-add), then the special-function
// unit's sin / cos on the reduced argument in [-pi, pi] (absolute error ~1e-6, below the rounding
// of the fp32 angle itself and of the bf16 output)
constexpr float TWO_PI_A = 0x1.921fb6p+2f, TWO_PI_B = -0x1.777a5cp-23f, TWO_PI_C = -0x1.ee59dap-48f;
constexpr float INV_TWO_PI = 0x1.45f306p-3f;
E3_DEV void rope_sincos(float a, float &s, float &c) {
    const float k = rintf(a * INV_TWO_PI);
    float r = fmaf(-k, TWO_PI_A, a);
    r = fmaf(-k, TWO_PI_B, r);
    r = fmaf(-k, TWO_PI_C, r);
    __sincosf(r, &s, &c);
}

// Residual columns [col0, col0 + 8 n) of one row as n 16-byte vectors (bounds-checked element by
// element at the right edge or for an unaligned row), read through L2 only: each value is read once.
template <int NV>
E3_DEV void load_residual(const GemmParams &p, int row, int col0, uint4 (&r)[NV]) {
    const __nv_bfloat16 *src = p.residual + (size_t)row * p.ld_res + col0;
    if (col0 + 8 * NV <= p.N && ((((uintptr_t)src) & 15) == 0)) {
#pragma unroll
        for (int j = 0; j < NV; ++j) r[j] = __ldcg(reinterpret_cast<const uint4 *>(src) + j);
    } else {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            uint16_t h[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int c = 8 * j + e;
                h[e] = col0 + c < p.N ? reinterpret_cast<const uint16_t *>(src)[c] : (uint16_t)0;
            }
            r[j] = make_uint4(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16),
                              h[4] | ((uint32_t)h[5] << 16), h[6] | ((uint32_t)h[7] << 16));
        }
    }
}

template <int NV>
E3_DEV void add_residual(float *v, const uint4 (&r)[NV]) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const uint32_t w4[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w4[e]);
            const float2 f = __bfloat1622float2(h);
            v[8 * j + 2 * e] += f.x;
            v[8 * j + 2 * e + 1] += f.y;
        }
    }
}

// Epilogue of one 32-column chunk of one row, from fp32 accumulators.
E3_DEV float store_chunk(const GemmParams &p, int row, int col0, const float (&v)[32]) {
    if (row >= p.M) return 0.0f;
    if (p.epi == EAGLE3_EPI_F32) {
        float *o = (float *)p.out + (size_t)row * p.ld_out + col0;
        if (col0 + 32 <= p.N && ((((uintptr_t)o) & 15) == 0)) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4 *>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
            for (int i = 0; i < 32; ++i)
                if (col0 + i < p.N) o[i] = v[i];
        }
        return 0.0f;
    }
    __nv_bfloat16 *o = (__nv_bfloat16 *)p.out + (size_t)row * p.ld_out + col0;
    float w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = v[i];
    if (p.epi == EAGLE3_EPI_BF16_RESIDUAL) {
        uint4 r[4];
        load_residual(p, row, col0, r);
        add_residual(w, r);
    }
    float ssq = 0.0f;
    if (col0 + 32 <= p.N && ((((uintptr_t)o) & 15) == 0)) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            uint4 pk;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(w[i], w[i + 1]), h1 = __floats2bfloat162_rn(w[i + 2], w[i + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(w[i + 4], w[i + 5]), h3 = __floats2bfloat162_rn(w[i + 6], w[i + 7]);
            pk.x = *reinterpret_cast<uint32_t *>(&h0);
            pk.y = *reinterpret_cast<uint32_t *>(&h1);
            pk.z = *reinterpret_cast<uint32_t *>(&h2);
            pk.w = *reinterpret_cast<uint32_t *>(&h3);
            *reinterpret_cast<uint4 *>(o + i) = pk;
            ssq = ssq_bf16x8(pk, ssq);
        }
    } else {
        for (int i = 0; i < 32; ++i)
            if (col0 + i < p.N) {
                const __nv_bfloat16 b = __float2bfloat16_rn(w[i]);
                o[i] = b;
                const float f = __bfloat162float(b);
                ssq = fmaf(f, f, ssq);
            }
    }
    return ssq;
}

// ROPE: the instantiation with the rotary epilogue (kept apart so that the others do not carry its
// registers)
template <int BN, bool ROPE>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_b2, const __grid_constant__ CUtensorMap tm_out,
                   const GemmParams p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sa = smem;                                   // STAGES x A tile
    uint8_t *sb = smem + C::STAGES * C::A_BYTES;          // STAGES x B tile
    uint8_t *epi = smem + C::STAGES * C::STAGE_BYTES;     // 4 warps x 2 output boxes (1024-aligned)
    uint64_t *bars = (uint64_t *)(epi + C::EPI_BYTES);
    uint64_t *full = bars, *empty = bars + C::STAGES, *tfull = bars + 2 * C::STAGES, *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_base_slot = (uint32_t *)(mma_done + 1);
    volatile int *abort = (volatile int *)(tmem_base_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool swiglu = p.epi == EAGLE3_EPI_SWIGLU;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(&tfull[a], 1);
            tc::mbar_init(&tempty[a], 4);
        }
        tc::mbar_init(mma_done, 1);
        *abort = 0;
        tc::fence_barrier_init();
        tc::prefetch_tmap(&tm_a);
        tc::prefetch_tmap(&tm_b);
        if (swiglu) tc::prefetch_tmap(&tm_b2);
    }
    if (warp == 1) tc::tmem_alloc(tmem_base_slot, C::TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_base_slot;
    pdl_wait();   // the previous kernel's outputs (this launch's inputs, or buffers it overwrites)
    pdl_trigger();
    if (skipped(p)) {   // uniform: every thread reads the same word
        tc::fence_before();
        __syncthreads();
        if (warp == 1) {
            __syncwarp();
            tc::fence_after();
            tc::tmem_dealloc(tmem, C::TMEM_COLS);
        }
        return;
    }

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t last_parity = 0, issued_mask = 0;   // parity of the last load issued per stage
            bool ok = true;
            WorkIter wi;
            wi.init(p);
            Item w;
            while (ok && wi.next(p, w)) {
                const int mb = w.mb, nb = w.nb;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!tc::mbar_wait(&empty[stage], phase ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc::mbar_expect_tx(&full[stage], C::STAGE_BYTES);
                    tc::tma_load_2d(sa + stage * C::A_BYTES, &tm_a, kb * BK, mb * BM, &full[stage]);
                    if (!swiglu) {
                        tc::tma_load_2d(sb + stage * C::B_BYTES, &tm_b, kb * BK, nb * BN, &full[stage]);
                    } else {
                        tc::tma_load_2d(sb + stage * C::B_BYTES, &tm_b, kb * BK, nb * (BN / 2), &full[stage]);
                        tc::tma_load_2d(sb + stage * C::B_BYTES + (BN / 2) * BK * 2, &tm_b2, kb * BK, nb * (BN / 2),
                                        &full[stage]);
                    }
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            // no TMA write may still be in flight when the CTA exits: wait (bounded) for the last
            // load issued to every stage; these return at once when the loads were consumed
            for (int st = 0; st < C::STAGES; ++st) {
                if (!((issued_mask >> st) & 1u)) continue;
                const uint32_t par = (last_parity >> st) & 1u;
                const long long t0 = clock64();
                while (!tc::mbar_try(&full[st], par) && clock64() - t0 < WAIT_LIMIT_CYCLES) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = tc::idesc_bf16(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            WorkIter wi;
            wi.init(p);
            Item w;
            while (ok && wi.next(p, w)) {
                const int kb0 = w.kb0, kb1 = w.kb1;
                if (!tc::mbar_wait(&tempty[acc], acc_phase ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!tc::mbar_wait(&full[stage], phase, abort)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t a_addr = smem_u32(sa + stage * C::A_BYTES);
                    const uint32_t b_addr = smem_u32(sb + stage * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = tc::desc_sw128(a_addr + k * 32);
                        const uint64_t bd = tc::desc_sw128(b_addr + k * 32);
                        tc::mma_bf16_ss(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(&empty[stage]);   // frees this smem stage when the MMAs finish
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc::mma_commit(&tfull[acc]);          // accumulator ready for the epilogue
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
            // every MMA this thread issued must retire before TMEM is freed (bounded wait)
            tc::mma_commit(mma_done);
            const long long t0 = clock64();
            while (!tc::mbar_try(mma_done, 0) && clock64() - t0 < WAIT_LIMIT_CYCLES) {
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
        int acc = 0;
        uint32_t acc_phase = 0;
        int sbuf = 0;                                 // output staging buffer of this warp
        WorkIter wi;
        wi.init(p);
        Item w;
        while (wi.next(p, w)) {
            const int mb = w.mb, nb = w.nb, sp = w.sp;
            if (p.epi == EAGLE3_EPI_BF16_RESIDUAL && w.kind != IT_CONTRIB && w.kind != IT_TAIL && p.splits == 1) {
                // pull this tile's residual row into L2 while the main loop runs (one bulk prefetch
                // of the row's whole-16-byte part; the epilogue reads it from there)
                const int prow = mb * BM + quarter * 32 + lane, col0 = nb * BN;
                if (prow < p.M && col0 < p.N) {
                    const __nv_bfloat16 *src = p.residual + (size_t)prow * p.ld_res + col0;
                    const uint32_t bytes = (uint32_t)(min(BN, p.N - col0) * 2) & ~15u;
                    if (bytes && ((((uintptr_t)src) & 15) == 0)) tc::prefetch_l2(src, bytes);
                }
            }
            // warp-uniform wait: lane 0 polls, the outcome is broadcast, so a timeout can never
            // split the warp in front of the warp-collective TMEM loads below
            int ok = 0;
            if (lane == 0) ok = tc::mbar_wait(&tfull[acc], acc_phase, abort) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
                break;
            }
            tc::fence_after();
            const int rl = quarter * 32 + lane;       // row within the tile
            const int row = mb * BM + rl;
            const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            // folded RMSNorm: this row's scale, applied to the accumulators after the stream-K
            // contributions and before the epilogue; the stored outputs' sum of squares goes out
            const float nscale = row_norm_scale(p, row);
            auto nscale32 = [&](float (&v)[32]) {
                if (p.ssq_in) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= nscale;
                }
            };
            float ssq_acc = 0.0f;
            // stream-K owner: the CTAs after this one whose shares start inside this tile hold the
            // rest of its k-blocks; wait (bounded, warp-uniform) until all their warps wrote
            int c_lo = 0, c_hi = 0;
            if (w.kind == IT_OWNER) {
                c_lo = blockIdx.x + 1;
                c_hi = c_lo;
                const long long tile_end = (long long)(w.u + 1 - p.dp_tiles) * p.kb_total;
                while (c_hi < (int)gridDim.x && sk_start(p, c_hi) < tile_end) ++c_hi;
                int fine = 1;
                if (lane == 0) {
                    for (int c = c_lo; c < c_hi && fine; ++c) {
                        const long long t0 = clock64();
                        while (atomicAdd(&p.sk_flag[c], 0) < 4) {
                            if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
                                fine = 0;
                                flag(p.dev_status, EAGLE3_DEV_TIMEOUT);
                                break;
                            }
                        }
                    }
                }
                fine = __shfl_sync(0xffffffffu, fine, 0);
                if (!fine) c_hi = c_lo;
                __threadfence();
            }
            // add the stream-K contributions to a chunk of 32 accumulator columns
            auto add_contrib = [&](float (&v)[32], int col) {
                if (row >= p.M) return;   // rows past M are never stored, so never exchanged
                for (int c = c_lo; c < c_hi; ++c) {
                    const float4 *src = p.sk_part + (size_t)c * (BN / 4) * BM + (size_t)(col / 4) * BM + rl;
                    float4 q[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) q[i] = __ldcg(src + (size_t)i * BM);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        v[4 * i] += q[i].x;
                        v[4 * i + 1] += q[i].y;
                        v[4 * i + 2] += q[i].z;
                        v[4 * i + 3] += q[i].w;
                    }
                }
            };
            if (w.kind == IT_CONTRIB) {
                // this CTA's slot; then count this warp in
                float4 *dst = p.sk_part + (size_t)blockIdx.x * (BN / 4) * BM + rl;
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(t_row + c * 32, v);   // warp-collective: every lane loads
                    if (row < p.M) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            __stcg(dst + (size_t)(c * 8 + i) * BM,
                                   make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
                    }
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(&p.sk_flag[blockIdx.x], 1);
            } else if (w.kind == IT_TAIL) {
                // fp32 partials of a split tail tile: the tile's accumulator layout, unit after unit
                float *wsr = p.tail_ws + ((size_t)w.u * BM + rl) * BN;
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(t_row + c * 32, v);   // warp-collective: every lane loads
                    if (row < p.M) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            __stcg(reinterpret_cast<float4 *>(wsr + c * 32 + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
                    }
                }
            } else if (p.splits > 1) {
                // fp32 partials in accumulator layout.  tcgen05.ld is warp-collective: every lane
                // loads, only lanes that own a row < M store.
                float *wsr = p.ws + ((size_t)sp * p.M + (row < p.M ? row : 0)) * p.n_acc + (size_t)nb * BN;
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(t_row + c * 32, v);
                    if (row < p.M) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(wsr + c * 32 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                }
            } else if (p.tma_out) {
                // 128-byte-wide chunks of this warp's 32 rows: 32 fp32 or 64 bf16 columns
                const int y = mb * BM + quarter * 32;
                const bool f32 = p.epi == EAGLE3_EPI_F32;
                const int chunks = (swiglu ? BN / 2 : BN) / (f32 ? 32 : 64);
                // residual rows one chunk ahead, so that their latency hides behind a chunk's work
                const bool res = p.epi == EAGLE3_EPI_BF16_RESIDUAL && row < p.M;
                uint4 r_cur[8], r_next[8];
                if (res) load_residual(p, row, nb * BN, r_cur);
                // RoPE: this row's position (the chunk pairs of a head are rotated together)
                const bool rope_epi = ROPE && p.epi == EAGLE3_EPI_BF16_ROPE;
                float rope_pos = 0.0f;
                if (rope_epi && row < p.M) rope_pos = (float)(p.rope_base[row / p.rope_rows] + p.rope_depth[row]);
                uint4 u_hi[8];                // the second half of a rotated head, for the next chunk
                uint32_t rmax = 0u;           // F32 with row_max: this row's largest output key in the tile
                for (int sc = 0; sc < chunks; ++sc) {
                    if (res && sc + 1 < chunks) load_residual(p, row, nb * BN + (sc + 1) * 64, r_next);
                    uint4 u[8];
                    const bool rot = rope_epi && nb * BN + sc * 64 < p.rope_cols;   // chunks pair up: BN % 128 == 0
                    if (ROPE && rot && (sc & 1)) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) u[j] = u_hi[j];
                    } else if (ROPE && rot) {
                        // dims 0..63 of the head (this chunk) with dims 64..127 (the next chunk)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float a[32], c[32];
                            tc::tmem_ld32(t_row + sc * 64 + h * 32, a);
                            tc::tmem_ld32(t_row + (sc + 1) * 64 + h * 32, c);
                            nscale32(a);
                            nscale32(c);
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                float lo[2], hi[2];
#pragma unroll
                                for (int q = 0; q < 2; ++q) {
                                    float sn, cs;
                                    rope_sincos(__fmul_rn(rope_pos, p.rope_inv[h * 32 + e + q]), sn, cs);
                                    lo[q] = a[e + q] * cs - c[e + q] * sn;
                                    hi[q] = c[e + q] * cs + a[e + q] * sn;
                                }
                                __nv_bfloat162 l2 = __floats2bfloat162_rn(lo[0], lo[1]);
                                __nv_bfloat162 h2 = __floats2bfloat162_rn(hi[0], hi[1]);
                                const int wi = h * 16 + e / 2;   // packed word of the 64-column chunk
                                reinterpret_cast<uint32_t *>(u)[wi] = *reinterpret_cast<uint32_t *>(&l2);
                                reinterpret_cast<uint32_t *>(u_hi)[wi] = *reinterpret_cast<uint32_t *>(&h2);
                            }
                        }
                    } else if (f32) {
                        float v[32];
                        tc::tmem_ld32(t_row + sc * 32, v);
                        add_contrib(v, sc * 32);
                        nscale32(v);
                        if (p.row_max) rmax = chunk_max_key(rmax, v, nb * BN + sc * 32, p.N);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            u[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                              __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                    } else {
                        float v[64];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float t[32];
                            if (!swiglu) {
                                tc::tmem_ld32(t_row + sc * 64 + h * 32, t);
                                add_contrib(t, sc * 64 + h * 32);
                                nscale32(t);
                            } else {
                                float g[32];
                                const int c = sc * 2 + h;
                                tc::tmem_ld32(t_row + c * 32, g);
                                tc::tmem_ld32(t_row + BN / 2 + c * 32, t);
                                add_contrib(g, c * 32);
                                add_contrib(t, BN / 2 + c * 32);
                                nscale32(g);
                                nscale32(t);
#pragma unroll
                                for (int i = 0; i < 32; ++i) t[i] = silu(g[i]) * t[i];
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[h * 32 + i] = t[i];
                        }
                        if (res) add_residual(v, r_cur);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * j], v[8 * j + 1]);
                            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * j + 2], v[8 * j + 3]);
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * j + 4], v[8 * j + 5]);
                            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * j + 6], v[8 * j + 7]);
                            u[j] = make_uint4(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1),
                                              *reinterpret_cast<uint32_t *>(&h2), *reinterpret_cast<uint32_t *>(&h3));
                            if (p.row_ssq) ssq_acc = ssq_bf16x8(u[j], ssq_acc);
                        }
                    }
                    // the buffer was last stored from two chunks ago: that store must have read it
                    uint8_t *box = epi + (quarter * 2 + sbuf) * C::EPI_BOX;
                    if (lane == 0) tc::bulk_wait_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4 *>(box + lane * 128 + ((j ^ (lane & 7)) << 4)) = u[j];
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    const int x = (swiglu ? nb * (BN / 2) : nb * BN) + sc * (f32 ? 32 : 64);
                    if (lane == 0 && x < p.N && y < p.M) {   // boxes wholly outside the output are skipped
                        tc::tma_store_2d(&tm_out, x, y, box);
                        tc::bulk_commit();
                    }
                    sbuf ^= 1;
                    if (res) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) r_cur[j] = r_next[j];
                    }
                }
                if (p.row_max && row < p.M && rmax) atomicMax(p.row_max + row, rmax);
                if (p.row_ssq && row < p.M) p.row_ssq[(size_t)nb * p.M + row] = ssq_acc;
            } else if (!swiglu) {
                uint32_t rmax = 0u;
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(t_row + c * 32, v);
                    add_contrib(v, c * 32);
                    nscale32(v);
                    if (p.row_max) rmax = chunk_max_key(rmax, v, nb * BN + c * 32, p.N);
                    ssq_acc += store_chunk(p, row, nb * BN + c * 32, v);
                }
                if (p.row_max && row < p.M && rmax) atomicMax(p.row_max + row, rmax);
                if (p.row_ssq && row < p.M) p.row_ssq[(size_t)nb * p.M + row] = ssq_acc;
            } else {
                for (int c = 0; c < BN / 64; ++c) {
                    float g[32], u[32];
                    tc::tmem_ld32(t_row + c * 32, g);
                    tc::tmem_ld32(t_row + BN / 2 + c * 32, u);
                    add_contrib(g, c * 32);
                    add_contrib(u, BN / 2 + c * 32);
                    nscale32(g);
                    nscale32(u);
#pragma unroll
                    for (int i = 0; i < 32; ++i) g[i] = silu(g[i]) * u[i];
                    store_chunk(p, row, nb * (BN / 2) + c * 32, g);
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) tc::bulk_wait<0>();            // every output store has completed
        __syncwarp();
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Row maxima of a warp's 32 consecutive outputs (which may span several rows): one atomic max per
// distinct row, from the lowest lane holding it.  All lanes of the warp call this together.
E3_DEV void warp_row_max(uint32_t *row_max, int row, uint32_t key, bool valid) {
    uint32_t pending = __ballot_sync(0xffffffffu, valid);
    const int lane = threadIdx.x & 31;
    while (pending) {
        const int lead = __ffs(pending) - 1;
        const int r = __shfl_sync(0xffffffffu, row, lead);
        const bool mine = valid && row == r;
        const uint32_t m = __reduce_max_sync(0xffffffffu, mine ? key : 0u);
        if (lane == lead && m) atomicMax(row_max + r, m);
        pending &= ~__ballot_sync(0xffffffffu, mine);
    }
}

// Split-K reduction in split order, then the epilogue.  One thread per output element.
__global__ void gemm_reduce_kernel(const GemmParams p) {
    pdl_wait();
    pdl_trigger();
    if (skipped(p)) return;
    const int n_out = p.N;
    const size_t total = (size_t)p.M * n_out;
    const size_t stride = (size_t)gridDim.x * blockDim.x;   // a multiple of 32: the loop is warp-uniform
    const int lane = threadIdx.x & 31;
    for (size_t base = (size_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < total; base += stride) {
        const size_t idx = base + lane;
        const bool valid = idx < total;
        const int row = valid ? (int)(idx / n_out) : 0, col = valid ? (int)(idx % n_out) : 0;
        uint32_t key = 0u;
        if (valid) {
            float acc, acc2 = 0.0f;
            if (p.epi == EAGLE3_EPI_SWIGLU) {
                // accumulator tile nb holds [gate cols | up cols], BN/2 output columns each
                const int half = p.n_acc / p.tiles_n / 2;
                const int nb = col / half, j = col % half;
                const size_t cg = (size_t)nb * 2 * half + j, cu = cg + half;
                acc = 0.0f;
                for (int s = 0; s < p.splits; ++s) {
                    const float *w = p.ws + ((size_t)s * p.M + row) * p.n_acc;
                    acc += w[cg];
                    acc2 += w[cu];
                }
                acc = silu(acc) * acc2;
            } else {
                acc = 0.0f;
                for (int s = 0; s < p.splits; ++s) acc += p.ws[((size_t)s * p.M + row) * p.n_acc + col];
            }
            if (p.epi == EAGLE3_EPI_F32) {
                ((float *)p.out)[(size_t)row * p.ld_out + col] = acc;
                key = order_key(acc);
            } else {
                if (p.epi == EAGLE3_EPI_BF16_RESIDUAL) acc += __bfloat162float(p.residual[(size_t)row * p.ld_res + col]);
                ((__nv_bfloat16 *)p.out)[(size_t)row * p.ld_out + col] = __float2bfloat16_rn(acc);
            }
        }
        if (p.row_max) warp_row_max(p.row_max, row, key, valid);   // every lane of the warp, one call site
    }
}

// The split tail's tiles: each output of such a tile is the sum of its tail_splits partials in split
// order, then the epilogue.  Block (tile, row group): 4 rows x 64 threads, a thread 4 columns of the
// accumulator tile.
__global__ void __launch_bounds__(256) gemm_tail_reduce_kernel(const GemmParams p) {
    pdl_wait();
    pdl_trigger();
    if (skipped(p)) return;
    constexpr int BNT = 256;   // accumulator columns per tile (the plan's tile width)
    const int t = p.tail_dp + blockIdx.x;
    const int mb = t % p.tiles_m, nb = t / p.tiles_m;
    const int rl = blockIdx.y * 4 + (threadIdx.x >> 6), c4 = (threadIdx.x & 63) * 4;
    const int row = mb * BM + rl;
    const bool swiglu = p.epi == EAGLE3_EPI_SWIGLU;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const size_t slot0 = (size_t)blockIdx.x * p.tail_splits;
    if (row < p.M)
        for (int sp = 0; sp < p.tail_splits; ++sp) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.tail_ws + ((slot0 + sp) * BM + rl) * BNT + c4));
            acc[0] += v.x;
            acc[1] += v.y;
            acc[2] += v.z;
            acc[3] += v.w;
        }
    // SwiGLU tiles hold [gate columns | up columns]: the first half's threads pair with the second's
    float up[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t key = 0u;
    bool any = false;
    float ssq = 0.0f;   // row_ssq: squares of this thread's stored outputs
    if (row < p.M && (!swiglu || c4 < BNT / 2)) {
        if (swiglu) {
            // the up columns of this thread's gate columns live 128 columns further in the same row
            float u4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int sp = 0; sp < p.tail_splits; ++sp) {
                const float4 v =
                    __ldcg(reinterpret_cast<const float4 *>(p.tail_ws + ((slot0 + sp) * BM + rl) * BNT + BNT / 2 + c4));
                u4[0] += v.x;
                u4[1] += v.y;
                u4[2] += v.z;
                u4[3] += v.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) up[e] = u4[e];
        }
        const float ns = row_norm_scale(p, row);   // the folded RMSNorm (1 without it)
        const int col0 = swiglu ? nb * (BNT / 2) + c4 : nb * BNT + c4;
        for (int e = 0; e < 4; ++e) {
            const int col = col0 + e;
            if (col >= p.N) continue;
            float o = p.ssq_in ? acc[e] * ns : acc[e];
            if (swiglu) o = silu(o) * (p.ssq_in ? up[e] * ns : up[e]);
            if (p.epi == EAGLE3_EPI_F32) {
                ((float *)p.out)[(size_t)row * p.ld_out + col] = o;
                const uint32_t k = order_key(o);
                key = any ? max(key, k) : k;
                any = true;
            } else {
                if (p.epi == EAGLE3_EPI_BF16_RESIDUAL) o += __bfloat162float(p.residual[(size_t)row * p.ld_res + col]);
                const __nv_bfloat16 b = __float2bfloat16_rn(o);
                ((__nv_bfloat16 *)p.out)[(size_t)row * p.ld_out + col] = b;
                const float f = __bfloat162float(b);
                ssq = fmaf(f, f, ssq);
            }
        }
    }
    // a warp's 32 threads cover 128 columns of one row: one atomic max per warp
    if (p.row_max) warp_row_max(p.row_max, row, key, any);
    if (p.row_ssq) {
        // the row's sum of squares: each warp's 128 columns by shuffles, then the row's two warps in
        // column order
        __shared__ float part[8];
#pragma unroll
        for (int o = 16; o; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
        if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ssq;
        __syncthreads();
        if ((threadIdx.x & 63) == 0 && row < p.M)
            p.row_ssq[(size_t)nb * p.M + row] = part[(threadIdx.x >> 5)] + part[(threadIdx.x >> 5) + 1];
    }
}

// ---- host side ----------------------------------------------------------------------------------
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

bool make_map(CUtensorMap *m, const void *base, int rows, int cols, int64_t ld_elems, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_elems * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// output [rows, cols] (fp32 or bf16) for TMA stores: 32-row boxes 128 bytes wide, 128B swizzle
bool make_out_map(CUtensorMap *m, void *base, int rows, int cols, int64_t ld_elems, bool f32) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int es = f32 ? 4 : 2;
    if (((uintptr_t)base & 15) || (ld_elems * es) % 16) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_elems * es};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    const int n = device_sm_count();
    return n > 0 ? n : 148;   // no device (workspace sizing on a host without one): a typical count
}

struct Plan {
    int bn, tiles_m, tiles_n, splits, kb_total, kb_per_split, units, n_acc, grid, streamk, dp_tiles;
    int tail_dp = 0, tail_splits = 1;   // split tail (see GemmParams)
    size_t ws_bytes;
};

Plan plan(const eagle3_linear_args_t *a) {
    Plan pl;
    const bool swiglu = a->epilogue == EAGLE3_EPI_SWIGLU;
    pl.bn = 256;
    const int out_per_tile = swiglu ? pl.bn / 2 : pl.bn;
    pl.tiles_m = (a->m + BM - 1) / BM;
    pl.tiles_n = (a->n + out_per_tile - 1) / out_per_tile;
    pl.kb_total = (a->k + BK - 1) / BK;
    const int tiles = pl.tiles_m * pl.tiles_n;
    const int sms = sm_count();
    pl.n_acc = pl.tiles_n * pl.bn;
    // stream-K when whole tiles would leave the last wave less than 97% full and a tile's main loop
    // is long (K >= 12288): the fix-up (a flag reset before the launch, fp32 slots through L2) and
    // the cooperative launch, which cannot start under the previous kernel's last wave, cost about
    // as much as the quantisation they remove when K is 4096
    const int waves = (tiles + sms - 1) / sms;
    pl.dp_tiles = tiles / sms >= 2 ? (tiles / sms - 1) * sms : 0;   // whole waves kept data-parallel
    const long long T = (long long)(tiles - pl.dp_tiles) * pl.kb_total;
    // (or when there is a single M tile: the launch streams weights and every SM should share it)
    // A single M tile with at most two waves of N tiles streams its weights through split-K
    // instead (measured faster than stream-K for these rows-few, weight-bound launches): the split
    // count in 1..8 (at least 4 k-blocks each) whose units fill their last wave best, a larger
    // count only when it fills it by 2% more; the partials are reduced in split order.
    int auto_splits = 1;
    const bool rope = a->epilogue == EAGLE3_EPI_BF16_ROPE;   // rotated in the epilogue: one k pass per tile
    const bool folded = a->row_ssq || a->row_ssq_in;   // per-row epilogue inputs / outputs: no k-split reduce
    if (!rope && !folded && a->splits <= 0 && pl.tiles_m == 1 && tiles <= 2 * sms) {
        double best = 0.0;
        for (int sp = 1; sp <= 8 && pl.kb_total / sp >= 4; ++sp) {
            const int units = tiles * sp, w = (units + sms - 1) / sms;
            const double fill = (double)units / ((double)w * sms);
            if (fill > best + 0.02) {
                best = fill;
                auto_splits = sp;
            }
        }
    }
    // split tail: whole waves data-parallel, and the partial last wave's tiles split along k into as
    // many ranges (2..8, at least 4 k-blocks each) as fill the SMs best, when that fills them at least
    // 10 points better; no CTA waits on another, so the launch stays an ordinary (dependent) one
    int tail_best = 1;
    double tail_fill = 0.0;
    const int tail_dp = (tiles / sms) * sms, tail_tiles = tiles - tail_dp;
    if (!rope && a->splits <= 0 && auto_splits == 1 && tail_dp > 0 && tail_tiles > 0) {
        tail_fill = (double)tail_tiles / sms;
        for (int sp = 2; sp <= 8 && pl.kb_total / sp >= 4; ++sp) {
            const int per = (pl.kb_total + sp - 1) / sp;
            if (tail_tiles * sp > sms || (sp - 1) * per >= pl.kb_total) continue;   // no empty last range
            const double f = (double)tail_tiles * sp / sms;
            if (f > tail_fill + 0.1) {
                tail_best = sp;
                tail_fill = f;
            }
        }
    }
    // stream-K, unless several M tiles run whole waves data-parallel and the split tail fills the
    // last wave at least 75%: then the split tail is faster (an ordinary launch that starts under the
    // previous kernel's last wave, no flags); e.g. 3840 x 4096 x 14336 with the residual epilogue,
    // 0.323 ms stream-K against 0.299 ms with a 6-way split tail
    pl.streamk = !rope && a->splits <= 0 && auto_splits == 1 && (pl.kb_total >= 192 || pl.tiles_m == 1) &&
                 (double)tiles / ((double)waves * sms) < 0.97 && T >= 8LL * sms &&
                 !(pl.tiles_m > 1 && tail_best > 1 && tail_fill >= 0.75);
    if (pl.streamk) {
        pl.splits = 1;
        pl.kb_per_split = pl.kb_total;
        pl.units = tiles;
        pl.grid = sms;
        pl.ws_bytes = (size_t)sms * BM * pl.bn * sizeof(float) + (size_t)sms * sizeof(int);
        return pl;
    }
    if (tail_best > 1) {
        pl.tail_dp = tail_dp;
        pl.tail_splits = tail_best;
        pl.splits = 1;
        pl.kb_per_split = (pl.kb_total + tail_best - 1) / tail_best;
        pl.units = tail_dp + tail_tiles * tail_best;
        pl.grid = sms;
        pl.ws_bytes = (size_t)tail_tiles * tail_best * BM * pl.bn * sizeof(float);
        return pl;
    }
    int splits = rope ? 1 : (a->splits > 0 ? a->splits : auto_splits);
    splits = std::max(1, std::min(splits, pl.kb_total));
    pl.kb_per_split = (pl.kb_total + splits - 1) / splits;
    pl.splits = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
    pl.units = tiles * pl.splits;
    pl.grid = std::min(pl.units, sms);
    pl.ws_bytes = pl.splits > 1 ? (size_t)pl.splits * a->m * pl.n_acc * sizeof(float) : 0;
    return pl;
}

eagle3_status_t validate(const eagle3_linear_args_t *a) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->m < 0 || a->n < 1 || a->k < 1 || a->splits < 0) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue < EAGLE3_EPI_BF16 || a->epilogue > EAGLE3_EPI_BF16_ROPE) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_EPI_BF16_ROPE) {
        if (a->rope_cols < 0 || a->rope_cols > a->n || a->rope_cols % 128 || a->rope_rows_per_seq < 1 ||
            !(a->rope_theta > 0.0f) || a->splits > 1)
            return EAGLE3_ERR_INVALID_ARGUMENT;
        const int64_t ld_o = a->ld_out ? a->ld_out : a->n;
        if (((uintptr_t)a->out & 15) || (ld_o % 8)) return EAGLE3_ERR_UNSUPPORTED;   // TMA-stored output
    }
    if (a->k % 8) return EAGLE3_ERR_UNSUPPORTED;   // 16-byte row pitch for TMA
    if (a->m == 0) return EAGLE3_OK;
    if (!a->x || !a->w || !a->out) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_EPI_BF16_ROPE && a->rope_cols > 0 && (!a->rope_base || !a->rope_depth))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_EPI_SWIGLU && !a->w2) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_EPI_BF16_RESIDUAL && !a->residual) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->row_max && (a->epilogue != EAGLE3_EPI_F32 || ((uintptr_t)a->row_max & 3))) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->row_ssq && ((a->epilogue != EAGLE3_EPI_BF16 && a->epilogue != EAGLE3_EPI_BF16_RESIDUAL) ||
                       ((uintptr_t)a->row_ssq & 3)))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->row_ssq_in && (a->ssq_blocks < 1 || a->ssq_dim < 1 || !(a->ssq_eps >= 0.0f) || ((uintptr_t)a->row_ssq_in & 3)))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if ((a->row_ssq || a->row_ssq_in) && a->splits > 1) return EAGLE3_ERR_UNSUPPORTED;
    const int64_t ld_x = a->ld_x ? a->ld_x : a->k, ld_w = a->ld_w ? a->ld_w : a->k;
    if (ld_x < a->k || ld_w < a->k || (ld_x % 8) || (ld_w % 8)) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)a->x | (uintptr_t)a->w | (uintptr_t)a->w2) & 15) return EAGLE3_ERR_INVALID_ARGUMENT;
    return EAGLE3_OK;
}

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" size_t eagle3_linear_workspace_size(const eagle3_linear_args_t *a) {
    if (validate(a) != EAGLE3_OK || a->m == 0) return 0;
    return plan(a).ws_bytes;
}

namespace e3 {
eagle3_status_t linear_launch(const eagle3_linear_args_t *a, void *workspace, size_t ws_bytes, cudaStream_t stream,
                              const int32_t *skip_if_zero);
}

extern "C" eagle3_status_t eagle3_linear(const eagle3_linear_args_t *a, void *workspace, size_t ws_bytes,
                                         eagle3_stream_t stream) {
    return e3::linear_launch(a, workspace, ws_bytes, (cudaStream_t)stream, nullptr);
}

eagle3_status_t e3::linear_launch(const eagle3_linear_args_t *a, void *workspace, size_t ws_bytes,
                                  cudaStream_t stream, const int32_t *skip_if_zero) {
    const eagle3_status_t st = validate(a);
    if (st != EAGLE3_OK || a->m == 0) return st;
    const Plan pl = plan(a);
    const size_t need = pl.ws_bytes;
    if (need && (!workspace || ws_bytes < need || ((uintptr_t)workspace & 15))) return EAGLE3_ERR_WORKSPACE;
    const bool swiglu = a->epilogue == EAGLE3_EPI_SWIGLU;
    const int64_t ld_x = a->ld_x ? a->ld_x : a->k, ld_w = a->ld_w ? a->ld_w : a->k;

    CUtensorMap ma, mb, mb2;
    const int brows = swiglu ? pl.bn / 2 : pl.bn;
    if (!make_map(&ma, a->x, a->m, a->k, ld_x, BM) || !make_map(&mb, a->w, a->n, a->k, ld_w, brows))
        return EAGLE3_ERR_CUDA;
    if (swiglu) {
        if (!make_map(&mb2, a->w2, a->n, a->k, ld_w, brows)) return EAGLE3_ERR_CUDA;
    } else {
        mb2 = mb;
    }
    GemmParams p;
    p.M = a->m;
    p.N = a->n;
    p.K = a->k;
    p.epi = a->epilogue;
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.splits = pl.splits;
    p.kb_total = pl.kb_total;
    p.kb_per_split = pl.kb_per_split;
    p.units = pl.units;
    p.n_acc = pl.n_acc;
    p.out = a->out;
    p.ld_out = a->ld_out ? a->ld_out : a->n;
    p.residual = (const __nv_bfloat16 *)a->residual;
    p.ld_res = a->ld_res ? a->ld_res : a->n;
    p.ws = (float *)workspace;
    p.streamk = pl.streamk;
    p.dp_tiles = pl.streamk ? pl.dp_tiles : 0;
    p.T = (long long)(pl.tiles_m * pl.tiles_n - p.dp_tiles) * pl.kb_total;
    p.sk_part = pl.streamk ? (float4 *)workspace : nullptr;
    p.sk_flag = pl.streamk ? (int *)((uint8_t *)workspace + (size_t)pl.grid * BM * pl.bn * sizeof(float)) : nullptr;
    p.dev_status = a->dev_status;
    p.rope_cols = a->epilogue == EAGLE3_EPI_BF16_ROPE ? a->rope_cols : 0;
    p.rope_rows = a->rope_rows_per_seq > 0 ? a->rope_rows_per_seq : 1;
    p.rope_base = a->rope_base;
    p.rope_depth = a->rope_depth;
    p.row_max = a->epilogue == EAGLE3_EPI_F32 ? a->row_max : nullptr;
    p.tail_dp = pl.tail_dp;
    p.tail_splits = pl.tail_splits;
    p.tail_ws = pl.tail_splits > 1 ? (float *)workspace : nullptr;
    p.skip_if_zero = skip_if_zero;
    p.row_ssq = a->row_ssq;
    p.ssq_in = a->row_ssq_in;
    p.ssq_blocks = a->row_ssq_in ? a->ssq_blocks : 0;
    p.ssq_inv_dim = a->row_ssq_in ? 1.0f / (float)a->ssq_dim : 0.0f;
    p.ssq_eps = a->ssq_eps;
    for (int j = 0; j < 64; ++j)
        p.rope_inv[j] = p.rope_cols ? (float)std::pow((double)a->rope_theta, -2.0 * j / 128.0) : 0.0f;
    CUtensorMap mo;
    p.tma_out = make_out_map(&mo, a->out, a->m, a->n, p.ld_out, a->epilogue == EAGLE3_EPI_F32) ? 1 : 0;
    if (!p.tma_out) mo = ma;   // unused
    if (p.rope_cols && !p.tma_out) return EAGLE3_ERR_UNSUPPORTED;

    using C = Cfg<256>;
    static PerDevice<cudaError_t> attr;
    if (attr.get([] {
            cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<256, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gemm_tc_kernel<256, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
            return e;
        }) != cudaSuccess)
        return EAGLE3_ERR_CUDA;
    if (pl.streamk) {
        // flags start at zero; blocks wait on one another, so all of them must be resident
        if (cudaMemsetAsync(p.sk_flag, 0, (size_t)pl.grid * sizeof(int), (cudaStream_t)stream) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(pl.grid);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = C::SMEM;
        cfg.stream = (cudaStream_t)stream;
        cudaLaunchAttribute attr_coop[1];
        attr_coop[0].id = cudaLaunchAttributeCooperative;
        attr_coop[0].val.cooperative = 1;
        cfg.attrs = attr_coop;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, gemm_tc_kernel<256, false>, ma, mb, mb2, mo, p) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
    } else if (p.rope_cols) {
        if (launch_pdl(gemm_tc_kernel<256, true>, dim3(pl.grid), dim3(NTHREADS), C::SMEM, (cudaStream_t)stream, ma,
                       mb, mb2, mo, p) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
    } else {
        if (launch_pdl(gemm_tc_kernel<256, false>, dim3(pl.grid), dim3(NTHREADS), C::SMEM, (cudaStream_t)stream, ma,
                       mb, mb2, mo, p) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (pl.tail_splits > 1) {
        const int tail_tiles = pl.tiles_m * pl.tiles_n - pl.tail_dp;
        if (launch_pdl(gemm_tail_reduce_kernel, dim3(tail_tiles, BM / 4), dim3(256), 0, (cudaStream_t)stream, p) !=
            cudaSuccess)
            return EAGLE3_ERR_CUDA;
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    if (pl.splits > 1) {
        const size_t total = (size_t)a->m * a->n;
        const int blocks = (int)std::min<size_t>((total + 255) / 256, (size_t)sm_count() * 8);
        if (launch_pdl(gemm_reduce_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, p) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    return EAGLE3_OK;
}
