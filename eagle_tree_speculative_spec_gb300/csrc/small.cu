// fp32 building blocks for small models (the tiny lossless configuration): linear layers with
// fused residual / SwiGLU epilogues, RMSNorm, rotate-half RoPE, embedding gather, argmax, and
// attention over a cache plus the visible new rows.
//
// Sources: "EAGLE-3: Engineering Implementation of LLM Inference Acceleration", appendix C and
// section VIII; "Advanced speculative decoding: tree drafts and EAGLE", section "Implementation".
//
// Every output row depends only on its own inputs and is computed in a fixed order (dot products
// over k in order; row reductions over a fixed lane assignment and shuffle tree; attention over
// the row's keys in sequence order).  A row therefore has the same bits whether it is computed
// alone or inside a batch or tree pass.  Plain SIMT code: these shapes are far too small for the
// tensor cores to matter.
#include <algorithm>
#include <cmath>

#include "../../include/eagle3_f32.h"
#include "common.cuh"

namespace e3 {
namespace {

constexpr int NT = 256;

__global__ void f32_linear_kernel(eagle3_f32_linear_args_t a, int64_t ld_x, int64_t ld_out, int64_t ld_res) {
    const int64_t total = a.m * a.n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / a.n, j = e % a.n;
        const float *x = a.x + i * ld_x;
        const float *w = a.w + j * a.k;
        float acc = 0.0f;
        for (int64_t k = 0; k < a.k; ++k) acc = __fmaf_rn(x[k], w[k], acc);
        float r;
        if (a.epilogue == EAGLE3_F32_EPI_SWIGLU) {
            const float *w2 = a.w2 + j * a.k;
            float acc2 = 0.0f;
            for (int64_t k = 0; k < a.k; ++k) acc2 = __fmaf_rn(x[k], w2[k], acc2);
            r = acc / (1.0f + expf(-acc)) * acc2;
        } else if (a.epilogue == EAGLE3_F32_EPI_RESIDUAL) {
            r = a.residual[i * ld_res + j] + acc;
        } else {
            r = acc;
        }
        a.out[i * ld_out + j] = r;
    }
}

// one warp per row
__global__ void f32_rmsnorm_kernel(int64_t rows, int64_t dim, const float *x, int64_t ld_x, const int32_t *gather,
                                   const float *w, float eps, float *out, int64_t ld_out) {
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float *src = x + (gather ? (int64_t)gather[r] : r) * ld_x;
    float ss = 0.0f;
    for (int64_t c = lane; c < dim; c += 32) ss = __fmaf_rn(src[c], src[c], ss);
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rs = 1.0f / sqrtf(ss / (float)dim + eps);
    for (int64_t c = lane; c < dim; c += 32) out[r * ld_out + c] = w[c] * (src[c] * rs);
}

struct RopeFreq {
    float inv[64];
};

__global__ void f32_rope_kernel(int64_t rows, int heads, int D, float *x, int64_t ld, const int32_t *pos,
                                const RopeFreq f) {
    const int half = D / 2;
    const int64_t total = rows * heads * half;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(e % half);
        const int64_t rh = e / half;
        const int h = (int)(rh % heads);
        const int64_t r = rh / heads;
        float *v = x + r * ld + (int64_t)h * D;
        float sn, cs;
        sincosf(__fmul_rn((float)pos[r], f.inv[j]), &sn, &cs);
        const float x1 = v[j], x2 = v[j + half];
        v[j] = x1 * cs - x2 * sn;
        v[j + half] = x2 * cs + x1 * sn;
    }
}

__global__ void f32_gather_kernel(int64_t rows, int64_t dim, const float *table, const int32_t *idx, float *out,
                                  int64_t ld_out) {
    const int64_t total = rows * dim;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / dim, c = e % dim;
        out[r * ld_out + c] = table[(int64_t)idx[r] * dim + c];
    }
}

// one warp per row
__global__ void f32_argmax_kernel(int64_t rows, int64_t vocab, const float *logits, int32_t *out) {
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    uint64_t best = 0ull;
    for (int64_t v = lane; v < vocab; v += 32) {
        const uint64_t key = pack_argmax(logits[r * vocab + v], (uint32_t)v);
        best = key > best ? key : best;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const uint64_t t = __shfl_xor_sync(0xffffffffu, best, o);
        best = t > best ? t : best;
    }
    if (lane == 0) out[r] = (int32_t)unpack_idx(best);
}

// One warp per (row, query head).  Scores live in shared memory, one per key in sequence order.
__global__ void f32_attn_kernel(const eagle3_f32_attn_args_t a, int64_t ld_q, int64_t ld_kv, float scale) {
    extern __shared__ float sc[];
    __shared__ int sel[64];
    __shared__ int n_sel;
    const int i = blockIdx.x, h = blockIdx.y, lane = threadIdx.x;
    const int D = a.head_dim, g = h / (a.n_heads / a.n_kv_heads);
    if (lane == 0) {
        int n = 0;
        const uint64_t bits = a.visible[i];
        for (int j = 0; j < a.n_rows; ++j)
            if ((bits >> j) & 1ull) sel[n++] = j;
        n_sel = n;
    }
    __syncwarp();
    const int L = a.cache_len, nk = L + n_sel;
    const float *q = a.q + (int64_t)i * ld_q + (int64_t)h * D;
    auto key_row = [&](int kk, const float *cache, const float *fresh) -> const float * {
        return kk < L ? cache + ((int64_t)g * a.s_max + kk) * D : fresh + (int64_t)sel[kk - L] * ld_kv + (int64_t)g * D;
    };
    float mx = -INFINITY;
    for (int kk = lane; kk < nk; kk += 32) {
        const float *k = key_row(kk, a.k_cache, a.k_new);
        float s = 0.0f;
        for (int d = 0; d < D; ++d) s = __fmaf_rn(q[d], k[d], s);
        s = s * scale;
        sc[kk] = s;
        mx = fmaxf(mx, s);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.0f;
    for (int kk = lane; kk < nk; kk += 32) {
        const float e = expf(sc[kk] - mx);
        sc[kk] = e;
        sum += e;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __syncwarp();
    const float inv = 1.0f / sum;
    float *o = a.out + ((int64_t)i * a.n_heads + h) * D;
    for (int d = lane; d < D; d += 32) {
        float acc = 0.0f;
        for (int kk = 0; kk < nk; ++kk) acc = __fmaf_rn(sc[kk], key_row(kk, a.v_cache, a.v_new)[d], acc);
        o[d] = acc * inv;
    }
}

int blocks_for(int64_t n) { return (int)std::min<int64_t>((n + NT - 1) / NT, 4096); }

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" eagle3_status_t eagle3_f32_linear(const eagle3_f32_linear_args_t *a, eagle3_stream_t stream) {
    if (!a || a->m < 0 || a->n < 1 || a->k < 1) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue < EAGLE3_F32_EPI_NONE || a->epilogue > EAGLE3_F32_EPI_SWIGLU) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->m == 0) return EAGLE3_OK;
    if (!a->x || !a->w || !a->out) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_F32_EPI_SWIGLU && !a->w2) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->epilogue == EAGLE3_F32_EPI_RESIDUAL && !a->residual) return EAGLE3_ERR_INVALID_ARGUMENT;
    const int64_t ld_x = a->ld_x ? a->ld_x : a->k, ld_out = a->ld_out ? a->ld_out : a->n;
    const int64_t ld_res = a->ld_res ? a->ld_res : a->n;
    if (ld_x < a->k || ld_out < a->n || ld_res < a->n) return EAGLE3_ERR_INVALID_ARGUMENT;
    f32_linear_kernel<<<blocks_for(a->m * a->n), NT, 0, (cudaStream_t)stream>>>(*a, ld_x, ld_out, ld_res);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}

extern "C" eagle3_status_t eagle3_f32_rmsnorm(int64_t rows, int64_t dim, const float *x, int64_t ld_x,
                                              const int32_t *gather, const float *w, float eps, float *out,
                                              int64_t ld_out, eagle3_stream_t stream) {
    if (rows < 0 || dim < 1 || !(eps >= 0.0f)) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (rows == 0) return EAGLE3_OK;
    if (!x || !w || !out) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (ld_x == 0) ld_x = dim;
    if (ld_out == 0) ld_out = dim;
    if (ld_x < dim || ld_out < dim) return EAGLE3_ERR_INVALID_ARGUMENT;
    const int per = NT / 32;
    f32_rmsnorm_kernel<<<(unsigned)((rows + per - 1) / per), NT, 0, (cudaStream_t)stream>>>(rows, dim, x, ld_x, gather, w,
                                                                                          eps, out, ld_out);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}

extern "C" eagle3_status_t eagle3_f32_rope(int64_t rows, int32_t heads, int32_t head_dim, float *x, int64_t ld,
                                           const int32_t *pos, float theta, eagle3_stream_t stream) {
    if (rows < 0 || heads < 1 || head_dim < 2 || head_dim % 2 || head_dim > 128 || !(theta > 0.0f))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (rows == 0) return EAGLE3_OK;
    if (!x || !pos || ld < (int64_t)heads * head_dim) return EAGLE3_ERR_INVALID_ARGUMENT;
    RopeFreq f;
    for (int j = 0; j < head_dim / 2; ++j) f.inv[j] = (float)std::pow((double)theta, -2.0 * j / head_dim);
    f32_rope_kernel<<<blocks_for(rows * heads * (head_dim / 2)), NT, 0, (cudaStream_t)stream>>>(rows, heads, head_dim,
                                                                                              x, ld, pos, f);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}

extern "C" eagle3_status_t eagle3_f32_gather(int64_t rows, int64_t dim, const float *table, const int32_t *idx,
                                             float *out, int64_t ld_out, eagle3_stream_t stream) {
    if (rows < 0 || dim < 1) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (rows == 0) return EAGLE3_OK;
    if (!table || !idx || !out) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (ld_out == 0) ld_out = dim;
    if (ld_out < dim) return EAGLE3_ERR_INVALID_ARGUMENT;
    f32_gather_kernel<<<blocks_for(rows * dim), NT, 0, (cudaStream_t)stream>>>(rows, dim, table, idx, out, ld_out);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}

extern "C" eagle3_status_t eagle3_f32_argmax(int64_t rows, int64_t vocab, const float *logits, int32_t *out,
                                             eagle3_stream_t stream) {
    if (rows < 0 || vocab < 1 || vocab > 0x7fffffff) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (rows == 0) return EAGLE3_OK;
    if (!logits || !out) return EAGLE3_ERR_INVALID_ARGUMENT;
    const int per = NT / 32;
    f32_argmax_kernel<<<(unsigned)((rows + per - 1) / per), NT, 0, (cudaStream_t)stream>>>(rows, vocab, logits, out);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}

extern "C" eagle3_status_t eagle3_f32_attn(const eagle3_f32_attn_args_t *a, eagle3_stream_t stream) {
    if (!a || a->n_rows < 0 || a->n_rows > 64 || a->n_heads < 1 || a->n_kv_heads < 1 || a->head_dim < 1 ||
        a->head_dim > 128 || a->cache_len < 0 || a->cache_len > a->s_max || a->n_heads % a->n_kv_heads ||
        a->scale < 0.0f)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if ((int64_t)a->cache_len + a->n_rows > 65536) return EAGLE3_ERR_UNSUPPORTED;
    if (a->n_rows == 0) return EAGLE3_OK;
    if (!a->q || !a->k_new || !a->v_new || !a->visible || !a->out || (a->cache_len && (!a->k_cache || !a->v_cache)))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    const int64_t ld_q = a->ld_q ? a->ld_q : (int64_t)a->n_heads * a->head_dim;
    const int64_t ld_kv = a->ld_kv ? a->ld_kv : (int64_t)a->n_kv_heads * a->head_dim;
    const float scale = a->scale > 0.0f ? a->scale : 1.0f / sqrtf((float)a->head_dim);
    const size_t smem = (size_t)(a->cache_len + a->n_rows) * sizeof(float);
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(f32_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return EAGLE3_ERR_CUDA;
    }
    f32_attn_kernel<<<dim3(a->n_rows, a->n_heads), 32, smem, (cudaStream_t)stream>>>(*a, ld_q, ld_kv, scale);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}
