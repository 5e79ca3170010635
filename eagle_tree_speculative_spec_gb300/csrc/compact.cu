// eagle3_compact_kv: copy the accepted path's K/V (and aux rows) into contiguous cache slots.
//
// Sources: "Advanced speculative decoding: tree drafts and EAGLE", section "Implementation" (the
// path's K/V were computed during verification at the right positions: append them without
// recomputation and drop the rest); "EAGLE-3: Engineering Implementation of LLM Inference
// Acceleration", section XI.4 (the cache keeps exactly the committed positions).
//
// Kernel 1 copies, one CTA per (layer, K or V, b, j) item, the Hkv x D row block of tree node
// path[b, j] to cache slot L + j with 16-byte vector moves (aux rows are extra items).  Kernel 2
// then writes slot_map and advances prefix_len; it runs after kernel 1 on the same stream, so no
// copy can read an already-advanced prefix length.
#include "common.cuh"

namespace e3 {
namespace {

constexpr int NT = 128;

struct Params {
    int L_layers, B, N, Hkv, D, E, S, W, A;
    int64_t cache_ls, tree_ls, tree_ns;
    uint8_t *k_cache, *v_cache;
    const uint8_t *tree_k, *tree_v;
    const int32_t *path, *accept_len;
    int32_t *prefix_len, *slot_map, *committed, *dev_status;
    const uint8_t *aux_tree;
    uint8_t *aux_out;
    // paged cache: position p of sequence b is slot block_table[b * bt_stride + p / block_size] *
    // block_size + p % block_size of a pool [n_slots, Hkv, D] per layer; null = contiguous
    const int32_t *block_table;
    int bt_stride, block_size, n_pages;
};

// The slot of position pos of sequence b in a paged cache, or -1 when its page id is outside the pool.
E3_DEV long long paged_slot(const Params &p, int b, int pos) {
    const int page = p.block_table[(size_t)b * p.bt_stride + pos / p.block_size];
    if (page < 0 || page >= p.n_pages) return -1;
    return (long long)page * p.block_size + pos % p.block_size;
}

// Whether sequence b's accepted path fits its cache (and, paged, lands on valid pages).
E3_DEV bool path_fits(const Params &p, int b, int L, int n) {
    if (n < 0 || n >= p.W || L < 0) return false;
    if (!p.block_table) return L + n + 1 <= p.S;
    if ((long long)L + n + 1 > (long long)p.bt_stride * p.block_size) return false;
    for (int j = 0; j <= n; ++j)
        if (paged_slot(p, b, L + j) < 0) return false;
    return true;
}

E3_DEV void copy_bytes(uint8_t *dst, const uint8_t *src, size_t n) {
    // both pointers and n are multiples of 16 when the host allowed the vector path
    if ((((uintptr_t)dst | (uintptr_t)src | n) & 15) == 0) {
        const int4 *s4 = reinterpret_cast<const int4 *>(src);
        int4 *d4 = reinterpret_cast<int4 *>(dst);
        for (size_t i = threadIdx.x; i < n / 16; i += NT) d4[i] = __ldg(s4 + i);
    } else {
        for (size_t i = threadIdx.x; i < n; i += NT) dst[i] = src[i];
    }
}

// Item layout: [layer][kv][b][j] for K/V rows, then [b][j] aux rows.
__global__ void __launch_bounds__(NT) compact_copy_kernel(const Params p) {
    const long long kv_items = (long long)p.L_layers * 2 * p.B * p.W;
    long long item = blockIdx.x;
    int b, j;
    bool aux = false;
    int layer = 0, kv = 0;
    if (item < kv_items) {
        j = (int)(item % p.W);
        item /= p.W;
        b = (int)(item % p.B);
        item /= p.B;
        kv = (int)(item % 2);
        layer = (int)(item / 2);
    } else {
        item -= kv_items;
        j = (int)(item % p.W);
        b = (int)(item / p.W);
        aux = true;
    }
    const int n = p.accept_len[b];
    const int L = p.prefix_len[b];
    if (j > n) return;
    const int src = p.path[(size_t)b * p.W + j];
    if (src < 0 || src >= p.N || !path_fits(p, b, L, n)) {
        if (threadIdx.x == 0 && j == 0 && layer == 0 && kv == 0 && !aux) flag(p.dev_status, EAGLE3_DEV_CAPACITY);
        return;
    }
    if (aux) {
        const size_t row = (size_t)p.A * p.E;
        copy_bytes(p.aux_out + ((size_t)b * p.W + j) * row, p.aux_tree + ((size_t)b * p.N + src) * row, row);
        return;
    }
    const size_t drow = (size_t)p.D * p.E;   // one head's row in bytes
    const uint8_t *tsrc = (kv ? p.tree_v : p.tree_k) + ((size_t)layer * p.tree_ls +
                          ((size_t)b * p.N + src) * (size_t)p.tree_ns) * p.E;
    uint8_t *cdst = (kv ? p.v_cache : p.k_cache) + (size_t)layer * p.cache_ls * p.E;
    if (p.block_table) {   // the slot holds all heads of the position contiguously, like the tree row
        copy_bytes(cdst + (size_t)paged_slot(p, b, L + j) * p.Hkv * drow, tsrc, (size_t)p.Hkv * drow);
        return;
    }
    for (int h = 0; h < p.Hkv; ++h) {
        uint8_t *d = cdst + (((size_t)b * p.Hkv + h) * p.S + (size_t)(L + j)) * drow;
        copy_bytes(d, tsrc + (size_t)h * drow, drow);
    }
}

__global__ void compact_finish_kernel(const Params p) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    const int n = p.accept_len[b];
    const int L = p.prefix_len[b];
    bool ok = path_fits(p, b, L, n);
    for (int j = 0; ok && j <= n; ++j) {
        const int src = p.path[(size_t)b * p.W + j];
        ok = src >= 0 && src < p.N;
    }
    for (int j = 0; j < p.W; ++j) {
        int slot = -1;
        if (ok && j <= n) slot = p.block_table ? (int)paged_slot(p, b, L + j) : L + j;
        p.slot_map[(size_t)b * p.W + j] = slot;
    }
    if (ok) p.prefix_len[b] = L + n + 1;
    if (p.committed) p.committed[b] = ok ? n + 1 : 0;
}

}  // namespace
}  // namespace e3

using namespace e3;

extern "C" eagle3_status_t eagle3_compact_kv(const eagle3_compact_args_t *a, eagle3_stream_t stream) {
    if (!a) return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->n_layers < 1 || a->batch < 0 || a->n_nodes < 1 || a->n_kv_heads < 1 || a->head_dim < 1 ||
        (!a->block_table && a->s_max < 1) || a->max_path < 1 || a->aux_dim < 0)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->block_table && (a->block_size < 1 || a->max_blocks < 1 || a->n_slots < a->block_size))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->elem_bytes != 2 && a->elem_bytes != 4) return EAGLE3_ERR_UNSUPPORTED;
    if (a->n_nodes > 64) return EAGLE3_ERR_UNSUPPORTED;
    if (a->batch == 0) return EAGLE3_OK;
    if (!a->k_cache || !a->v_cache || !a->tree_k || !a->tree_v || !a->path || !a->accept_len ||
        !a->prefix_len || !a->slot_map)
        return EAGLE3_ERR_INVALID_ARGUMENT;
    if (a->aux_dim > 0 && (!a->aux_tree || !a->aux_out)) return EAGLE3_ERR_INVALID_ARGUMENT;
    const int64_t dense_cache = a->block_table ? (int64_t)a->n_slots * a->n_kv_heads * a->head_dim
                                               : (int64_t)a->batch * a->n_kv_heads * a->s_max * a->head_dim;
    if (a->tree_node_stride < 0 || (a->tree_node_stride && a->tree_node_stride < (int64_t)a->n_kv_heads * a->head_dim))
        return EAGLE3_ERR_INVALID_ARGUMENT;
    const int64_t tree_ns = a->tree_node_stride ? a->tree_node_stride : (int64_t)a->n_kv_heads * a->head_dim;
    const int64_t dense_tree = (int64_t)a->batch * a->n_nodes * tree_ns;
    if (a->n_layers > 1 && (a->cache_layer_stride < dense_cache || a->tree_layer_stride < dense_tree))
        return EAGLE3_ERR_INVALID_ARGUMENT;

    Params p;
    p.L_layers = a->n_layers;
    p.B = a->batch;
    p.N = a->n_nodes;
    p.Hkv = a->n_kv_heads;
    p.D = a->head_dim;
    p.E = a->elem_bytes;
    p.S = a->s_max;
    p.W = a->max_path;
    p.A = a->aux_dim;
    p.cache_ls = a->n_layers > 1 ? a->cache_layer_stride : dense_cache;
    p.tree_ls = a->n_layers > 1 ? a->tree_layer_stride : dense_tree;
    p.tree_ns = tree_ns;
    p.k_cache = (uint8_t *)a->k_cache;
    p.v_cache = (uint8_t *)a->v_cache;
    p.tree_k = (const uint8_t *)a->tree_k;
    p.tree_v = (const uint8_t *)a->tree_v;
    p.path = a->path;
    p.accept_len = a->accept_len;
    p.prefix_len = a->prefix_len;
    p.slot_map = a->slot_map;
    p.committed = a->committed;
    p.dev_status = a->dev_status;
    p.aux_tree = (const uint8_t *)a->aux_tree;
    p.aux_out = (uint8_t *)a->aux_out;
    p.block_table = a->block_table;
    p.bt_stride = a->max_blocks;
    p.block_size = a->block_size;
    p.n_pages = a->block_table ? a->n_slots / a->block_size : 0;

    const long long items = (long long)a->n_layers * 2 * a->batch * a->max_path +
                            (a->aux_dim > 0 ? (long long)a->batch * a->max_path : 0);
    if (items > 0x7fffffffLL) return EAGLE3_ERR_UNSUPPORTED;
    compact_copy_kernel<<<(unsigned)items, NT, 0, (cudaStream_t)stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return EAGLE3_ERR_CUDA;
    compact_finish_kernel<<<(a->batch + 127) / 128, 128, 0, (cudaStream_t)stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA;
}
