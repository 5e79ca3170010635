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
// epilogue (deterministic).  Every mbarrier wait is bounded; on a timeout the kernel records
// EAGLE3_DEV_TIMEOUT, stops issuing work, drains its own TMA loads and frees its TMEM.
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
    int32_t *dev_status;
};

template <int BN>
struct Cfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /* align */ + 256 /* barriers */;
};

E3_DEV float silu(float x) { return x / (1.0f + __expf(-x)); }

// Epilogue of one 32-column chunk of one row, from fp32 accumulators.
E3_DEV void store_chunk(const GemmParams &p, int row, int col0, const float (&v)[32]) {
    if (row >= p.M) return;
    if (p.epi == EAGLE3_EPI_F32) {
        float *o = (float *)p.out + (size_t)row * p.ld_out + col0;
        if (col0 + 32 <= p.N && ((((uintptr_t)o) & 15) == 0)) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4 *>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
            for (int i = 0; i < 32; ++i)
                if (col0 + i < p.N) o[i] = v[i];
        }
        return;
    }
    __nv_bfloat16 *o = (__nv_bfloat16 *)p.out + (size_t)row * p.ld_out + col0;
    float w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = v[i];
    if (p.epi == EAGLE3_EPI_BF16_RESIDUAL) {
        const __nv_bfloat16 *r = p.residual + (size_t)row * p.ld_res + col0;
        for (int i = 0; i < 32; ++i)
            if (col0 + i < p.N) w[i] += __bfloat162float(r[i]);
    }
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
        }
    } else {
        for (int i = 0; i < 32; ++i)
            if (col0 + i < p.N) o[i] = __float2bfloat16_rn(w[i]);
    }
}

template <int BN>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_b2, const GemmParams p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sa = smem;                                   // STAGES x A tile
    uint8_t *sb = smem + C::STAGES * C::A_BYTES;          // STAGES x B tile
    uint64_t *bars = (uint64_t *)(smem + C::STAGES * C::STAGE_BYTES);
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

    auto decode = [&](int unit, int &mb, int &nb, int &sp) {
        mb = unit % p.tiles_m;
        const int r = unit / p.tiles_m;
        nb = r % p.tiles_n;
        sp = r / p.tiles_n;
    };

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t last_parity = 0, issued_mask = 0;   // parity of the last load issued per stage
            bool ok = true;
            for (int unit = blockIdx.x; unit < p.units && ok; unit += gridDim.x) {
                int mb, nb, sp;
                decode(unit, mb, nb, sp);
                const int kb0 = sp * p.kb_per_split, kb1 = min(p.kb_total, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
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
            for (int unit = blockIdx.x; unit < p.units && ok; unit += gridDim.x) {
                int mb, nb, sp;
                decode(unit, mb, nb, sp);
                const int kb0 = sp * p.kb_per_split, kb1 = min(p.kb_total, kb0 + p.kb_per_split);
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
        for (int unit = blockIdx.x; unit < p.units; unit += gridDim.x) {
            int mb, nb, sp;
            decode(unit, mb, nb, sp);
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
            const int row = mb * BM + quarter * 32 + lane;
            const uint32_t t_row = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            if (p.splits > 1) {
                // fp32 partials in accumulator layout.  tcgen05.ld is warp-collective: every lane
                // loads, only lanes that own a row < M store.
                float *w = p.ws + ((size_t)sp * p.M + (row < p.M ? row : 0)) * p.n_acc + (size_t)nb * BN;
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(t_row + c * 32, v);
                    if (row < p.M) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(w + c * 32 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                }
            } else if (!swiglu) {
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(t_row + c * 32, v);
                    store_chunk(p, row, nb * BN + c * 32, v);
                }
            } else {
                for (int c = 0; c < BN / 64; ++c) {
                    float g[32], u[32];
                    tc::tmem_ld32(t_row + c * 32, g);
                    tc::tmem_ld32(t_row + BN / 2 + c * 32, u);
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
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Split-K reduction in split order, then the epilogue.  One thread per output element pair.
__global__ void gemm_reduce_kernel(const GemmParams p) {
    const int n_out = p.N;
    const size_t total = (size_t)p.M * n_out;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
        const int row = (int)(idx / n_out), col = (int)(idx % n_out);
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
        } else {
            if (p.epi == EAGLE3_EPI_BF16_RESIDUAL) acc += __bfloat162float(p.residual[(size_t)row * p.ld_res + col]);
            ((__nv_bfloat16 *)p.out)[(size_t)row * p.ld_out + col] = __float2bfloat16_rn(acc);
        }
    }
}

// ---- host side ----------------------------------------------------------------------------------
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

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

struct Plan {
    int bn, tiles_m, tiles_n, splits, kb_total, kb_per_split, units, n_acc, grid;
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
    int splits = a->splits > 0 ? a->splits : 1;
    if (a->splits <= 0 && tiles < sms) splits = std::max(1, std::min(pl.kb_total / 4, sms / tiles));
    splits = std::max(1, std::min(splits, pl.kb_total));
    pl.kb_per_split = (pl.kb_total + splits - 1) / splits;
    pl.splits = (pl.kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
    pl.units = tiles * pl.splits;
    pl.n_acc = pl.tiles_n * pl.bn;
    pl.grid = std::min(pl.units, sms);
    return pl;
}

eagle3_status_t validate(const eagle3_linear_args_t *a) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->m < 0 || a->n < 1 || a->k < 1 || a->splits < 0) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue < EAGLE3_EPI_BF16 || a->epilogue > EAGLE3_EPI_SWIGLU) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->k % 8) return EAGLE3_ERR_UNSUPPORTED;   // 16-byte row pitch for TMA
    if (a->m == 0) return EAGLE3_OK;
    if (!a->x || !a->w || !a->out) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_EPI_SWIGLU && !a->w2) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_EPI_BF16_RESIDUAL && !a->residual) return EAGLE3_ERR_INVALID_ARGUMENT;
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
    const Plan pl = plan(a);
    return pl.splits > 1 ? (size_t)pl.splits * a->m * pl.n_acc * sizeof(float) : 0;
}

extern "C" eagle3_status_t eagle3_linear(const eagle3_linear_args_t *a, void *workspace, size_t ws_bytes,
                                         eagle3_stream_t stream) {
    const eagle3_status_t st = validate(a);
    if (st != EAGLE3_OK || a->m == 0) return st;
    const Plan pl = plan(a);
    const size_t need = pl.splits > 1 ? (size_t)pl.splits * a->m * pl.n_acc * sizeof(float) : 0;
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
    p.dev_status = a->dev_status;

    using C = Cfg<256>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
            cudaSuccess)
            return EAGLE3_ERR_CUDA;
        attr = true;
    }
    gemm_tc_kernel<256><<<pl.grid, NTHREADS, C::SMEM, (cudaStream_t)stream>>>(ma, mb, mb2, p);
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (pl.splits > 1) {
        const size_t total = (size_t)a->m * a->n;
        const int blocks = (int)std::min<size_t>((total + 255) / 256, (size_t)sm_count() * 8);
        gemm_reduce_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    }
    return EAGLE3_OK;
}
