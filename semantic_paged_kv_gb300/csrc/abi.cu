// C ABI of the IceCache hot path: argument checks, workspace layouts and the
// launch sequence of every entry point declared in ice.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace ice {

size_t select_smem_bytes(const ice_params &p, int k_pages, int n_chunks);

namespace {

thread_local std::string g_last_error;

ice_status fail(ice_status code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

ice_status cuda_status(cudaError_t e, const char *where) {
    if (e == cudaSuccess) return ICE_OK;
    return fail(ICE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Whether p points to device memory (not pinned host memory mapped for the GPU).
bool in_device_memory(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice;
}

}  // namespace

bool fault_armed(const char *what) {
    const char *v = getenv("ICE_FAULT");
    if (!v || !*v) return false;
    const size_t n = strlen(what);
    for (const char *c = v; *c;) {
        const char *e = strchr(c, ',');
        const size_t len = e ? (size_t)(e - c) : strlen(c);
        if (len == n && strncmp(c, what, n) == 0) return true;
        if (!e) break;
        c = e + 1;
    }
    return false;
}

namespace {

ice_status check_params(const ice_params *p) {
    if (!p) return fail(ICE_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->n_kv_heads < 1 || p->n_q_heads < 1)
        return fail(ICE_ERR_INVALID_ARG, "batch, n_q_heads and n_kv_heads must be >= 1");
    if (p->n_q_heads % p->n_kv_heads != 0)
        return fail(ICE_ERR_INVALID_ARG, "n_q_heads (%d) must be a multiple of n_kv_heads (%d)", p->n_q_heads,
                    p->n_kv_heads);
    if (p->n_q_heads / p->n_kv_heads > 16)
        return fail(ICE_ERR_UNSUPPORTED, "at most 16 query heads per KV head are supported");
    if (p->batch >= 4096 || p->n_kv_heads >= 4096)
        return fail(ICE_ERR_INVALID_ARG, "batch and n_kv_heads must be < 4096 (promotion counter layout)");
    if (p->head_dim != kHeadDim) return fail(ICE_ERR_UNSUPPORTED, "head_dim must be %d", kHeadDim);
    if (p->page_size != kPage) return fail(ICE_ERR_UNSUPPORTED, "page_size must be %d", kPage);
    if (p->dtype != ICE_BF16 && p->dtype != ICE_FP32) return fail(ICE_ERR_INVALID_ARG, "dtype must be ICE_BF16 or ICE_FP32");
    if (p->n_levels != 2 && p->n_levels != 3) return fail(ICE_ERR_UNSUPPORTED, "n_levels must be 2 or 3");
    if (p->n_levels == 3 && p->np_cap > kLevel2MaxParents)
        return fail(ICE_ERR_UNSUPPORTED, "three levels need np_cap <= %d", kLevel2MaxParents);
    if (p->promote_thresh > (1ull << 32)) return fail(ICE_ERR_INVALID_ARG, "promote_thresh must be <= 2^32");
    if (p->n_tokens < 0 || p->n_cap < p->n_tokens) return fail(ICE_ERR_INVALID_ARG, "need 0 <= n_tokens <= n_cap");
    if (p->np_cap < 1 || p->page_cap < 1) return fail(ICE_ERR_INVALID_ARG, "np_cap and page_cap must be >= 1");
    if ((long long)p->np_cap * p->n_kv_heads * p->batch > (1ll << 40))
        return fail(ICE_ERR_INVALID_ARG, "capacities too large");
    if (p->n_sink < 0 || p->n_window < 0) return fail(ICE_ERR_INVALID_ARG, "n_sink and n_window must be >= 0");
    return ICE_OK;
}

bool aligned16(const void *x) { return ((uintptr_t)x & 15u) == 0; }

ice_status check_index(const ice_index *x) {
    if (!x) return fail(ICE_ERR_INVALID_ARG, "index is NULL");
    const void *ptrs[] = {x->n_parents, x->n_pages, x->n_indexed, x->m2, x->parent_tok, x->parent_keys,
                          x->parent_e, x->parent_corr, x->parent_first_page, x->parent_last_page,
                          x->parent_n_pages, x->page_parent, x->page_len, x->page_next, x->page_tokens,
                          x->token_parent, x->token_page, x->token_slot, x->pool_k, x->pool_v};
    for (const void *q : ptrs)
        if (!q) return fail(ICE_ERR_INVALID_ARG, "an ice_index array pointer is NULL");
    if (!aligned16(x->parent_keys) || !aligned16(x->pool_k) || !aligned16(x->pool_v))
        return fail(ICE_ERR_INVALID_ARG, "parent_keys, pool_k and pool_v must be 16-byte aligned");
    return ICE_OK;
}

// The level-2 arrays a three-level index needs.
ice_status check_level2(const ice_params *p, const ice_index *x) {
    if (p->n_levels != 3) return ICE_OK;
    if (!x->n_nodes2 || !x->node2 || !x->parent2 || !x->child_start || !x->children)
        return fail(ICE_ERR_INVALID_ARG, "a three-level index needs n_nodes2, node2, parent2, child_start, children");
    return ICE_OK;
}

ice_status check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (need && !ws) return fail(ICE_ERR_INVALID_ARG, "workspace is NULL");
    if (((uintptr_t)ws & 255u) != 0) return fail(ICE_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (ws_bytes < need) return fail(ICE_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    return ICE_OK;
}

int k_pages_of(int budget_tokens) { return (budget_tokens + kPage - 1) / kPage; }

int sm_count();

// The kernels ice_decode_step runs for a shape (see ice_decode_plan).
int decode_plan(const ice_params &p, int k_pages, int max_sel) {
    if (p.n_levels == 3) return ICE_PLAN_DESCENT;
    // one cluster per unit pays off while all clusters fit in one wave; with
    // more units the score / attention kernels keep every SM streaming
    if (units_of(p) * kDecodeCluster <= sm_count()) {
        if (decode_cluster2_supported(p, k_pages, max_sel)) return ICE_PLAN_CLUSTER_BF16;
        if (decode_cluster_supported(p, k_pages, max_sel)) return ICE_PLAN_CLUSTER;
    }
    if (select_tc_supported(p, k_pages))
        return attention_mma_select_supported(p, max_sel) && attention_mma_fits(p, max_sel) ? ICE_PLAN_SCORE_SELECT
                                                                                             : ICE_PLAN_SCORE_TOPK;
    return ICE_PLAN_SIMT;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

BuildWs build_ws_layout(const ice_params &p, void *base) {
    BuildWs w{};
    const size_t U = (size_t)units_of(p);
    const size_t N = (size_t)p.n_tokens;
    const size_t tp = (size_t)ceil_div(p.n_tokens, kLiftTile);
    const size_t tk = (size_t)ceil_div(p.n_tokens, kPackTile);
    char *b = static_cast<char *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *r = b ? b + off : nullptr;
        off += align256(bytes);
        return r;
    };
    w.norm2 = reinterpret_cast<double *>(take(sizeof(double) * U * N));
    w.pcount = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * U * tp));
    w.tile_max = reinterpret_cast<double *>(take(sizeof(double) * U * tp));
    w.tile_min = reinterpret_cast<unsigned long long *>(take(sizeof(unsigned long long) * U * tp));
    w.a_extra = reinterpret_cast<uint4 *>(take(32 * U * N));
    w.b_extra = reinterpret_cast<uint4 *>(take(32 * U * (size_t)p.np_cap));
    w.pack_cnt = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * U * tk * (size_t)p.np_cap));
    w.pack_total = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * U * (size_t)p.np_cap));
    const size_t l2 = (p.n_levels == 3 && p.dtype == ICE_BF16) ? U * (size_t)p.np_cap : 0;
    w.a_extra2 = reinterpret_cast<uint4 *>(take(32 * l2));
    w.keys2 = take(sizeof(uint16_t) * kHeadDim * l2);
    w.b_extra2 = reinterpret_cast<uint4 *>(take(32 * l2));
    w.bytes = off;
    return w;
}

DecodeWs decode_ws_layout(const ice_params &p, int budget_tokens, int max_sel, void *base, bool with_select) {
    DecodeWs w{};
    const size_t U = (size_t)units_of(p);
    const size_t g = (size_t)(p.n_q_heads / p.n_kv_heads);
    w.k_pages = k_pages_of(budget_tokens);
    w.n_chunks = ceil_div(p.np_cap, kSelChunk);
    const size_t kc = (size_t)(w.k_pages < kSelChunk ? w.k_pages : kSelChunk);
    w.n_splits = ceil_div(max_sel > 0 ? max_sel : 1, kAttnPagesPerSplit);
    char *b = static_cast<char *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *r = b ? b + off : nullptr;
        off += align256(bytes);
        return r;
    };
    // the attention alone (with_select false) needs only its ticket and partials
    w.sel_ticket = with_select ? reinterpret_cast<int32_t *>(take(sizeof(int32_t) * U)) : nullptr;
    w.attn_ticket = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * U));
    if (with_select) {
        // (also the per-head page lists [U, g, 32] int32 of the three-level descent)
        const size_t ck = sizeof(unsigned long long) * U * w.n_chunks * g * (kc ? kc : 1);
        w.cand_key = reinterpret_cast<unsigned long long *>(
            take(ck > sizeof(int32_t) * U * g * 32 ? ck : sizeof(int32_t) * U * g * 32));
        w.cand_span = reinterpret_cast<int4 *>(take(sizeof(int4) * U * w.n_chunks * kSelChunk));
    }
    w.part_ml = reinterpret_cast<float *>(take(sizeof(float) * U * w.n_splits * g * 2));
    w.part_o = reinterpret_cast<float *>(take(sizeof(float) * U * w.n_splits * g * kHeadDim));
    w.scores = with_select ? reinterpret_cast<float *>(take(sizeof(float) * U * select_tc_scores(p))) : nullptr;
    w.bytes = off;
    return w;
}

InsertWs insert_ws_layout(const ice_params &p, void *base) {
    InsertWs w{};
    const size_t U = (size_t)units_of(p);
    w.n_chunks = ceil_div(p.np_cap, kSelChunk);
    char *b = static_cast<char *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *r = b ? b + off : nullptr;
        off += align256(bytes);
        return r;
    };
    w.ticket = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * U));
    w.best_s = reinterpret_cast<float *>(take(sizeof(float) * U * w.n_chunks));
    w.best_m = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * U * w.n_chunks));
    w.bytes = off;
    return w;
}

}  // namespace ice

using namespace ice;

extern "C" {

const char *ice_status_string(ice_status s) {
    switch (s) {
    case ICE_OK: return "ok";
    case ICE_ERR_INVALID_ARG: return "invalid argument";
    case ICE_ERR_CUDA: return "CUDA error";
    case ICE_ERR_OOM: return "out of memory";
    case ICE_ERR_CAPACITY: return "capacity exceeded";
    case ICE_ERR_TIMEOUT: return "timeout";
    case ICE_ERR_UNSUPPORTED: return "unsupported";
    default: return "unknown status";
    }
}

const char *ice_last_error(void) { return g_last_error.c_str(); }

const char *ice_version(void) { return "icecache-gb300 0.1 (sm_103a)"; }

int32_t ice_positional_pages(int32_t n_tokens, int32_t n_sink, int32_t n_window, int32_t page_size) {
    if (n_tokens < 0 || n_sink < 0 || n_window < 0 || page_size != kPage) return -1;
    ice_params p{};
    p.n_tokens = n_tokens;
    p.n_sink = n_sink;
    p.n_window = n_window;
    return pos_split(p).n_pos;
}

int32_t ice_page_bound(int32_t n_tokens, int32_t n_parents, int32_t page_size) {
    if (n_tokens < 0 || n_parents < 0 || page_size <= 0) return -1;
    // the page count is an integer, so the floor of the bound holds too
    const long long b = ((long long)n_tokens + (long long)(page_size - 1) * n_parents) / page_size;
    return b > 0x7fffffffll ? 0x7fffffff : (int32_t)b;
}

ice_status ice_default_capacities(ice_params *p) {
    if (!p) return fail(ICE_ERR_INVALID_ARG, "params is NULL");
    if (p->n_tokens < 0) return fail(ICE_ERR_INVALID_ARG, "n_tokens must be >= 0");
    if (p->page_size != kPage) return fail(ICE_ERR_UNSUPPORTED, "page_size must be %d", kPage);
    if (p->promote_thresh > (1ull << 32)) return fail(ICE_ERR_INVALID_ARG, "promote_thresh must be <= 2^32");
    if (p->n_sink < 0 || p->n_window < 0) return fail(ICE_ERR_INVALID_ARG, "n_sink and n_window must be >= 0");
    if (p->n_cap < p->n_tokens) p->n_cap = p->n_tokens > 1 ? p->n_tokens : 1;
    if (p->n_cap < 1) p->n_cap = 1;
    // promoted parents ~ Binomial(n_cap, q): the mean plus 8 standard deviations plus 16
    const double q = (double)p->promote_thresh / 4294967296.0;
    const double mu = (double)p->n_cap * q;
    const double np = floor(mu + 8.0 * sqrt(mu * (1.0 - q) + 1.0) + 16.0);
    p->np_cap = np >= (double)p->n_cap ? p->n_cap : (np < 1.0 ? 1 : (int32_t)np);
    const int32_t bound = ice_page_bound(p->n_cap, p->np_cap, kPage);
    const long long pc = (long long)bound + pos_split(*p).n_pos;
    if (bound < 0 || pc > 0x7fffffffll) return fail(ICE_ERR_INVALID_ARG, "page capacity overflows int32");
    p->page_cap = pc > 0 ? (int32_t)pc : 1;
    return ICE_OK;
}

// One slab holding every array of an index: offsets from the slab's start
// in ice_index field order, each array 256-byte aligned.
static size_t index_layout(const ice_params &p, bool with_pool, char *base, ice_index *out) {
    const size_t U = (size_t)units_of(p), Np = (size_t)p.np_cap, Pc = (size_t)p.page_cap, Nc = (size_t)p.n_cap;
    const size_t S = kPage, d = kHeadDim, esz = p.dtype == ICE_BF16 ? 2 : 4;
    size_t off = 0;
    auto take = [&](size_t bytes) -> void * {
        void *r = base ? base + off : nullptr;
        off += align256(bytes);
        return r;
    };
    ice_index x{};
    x.n_parents = (int32_t *)take(4 * U);
    x.n_pages = (int32_t *)take(4 * U);
    x.n_indexed = (int32_t *)take(4 * U);
    x.m2 = (double *)take(8 * U);
    x.parent_tok = (int32_t *)take(4 * U * Np);
    x.parent_keys = take(esz * U * Np * d);
    x.parent_e = (float *)take(4 * U * Np);
    x.parent_corr = (float *)take(4 * U * Np);
    x.parent_first_page = (int32_t *)take(4 * U * Np);
    x.parent_last_page = (int32_t *)take(4 * U * Np);
    x.parent_n_pages = (int32_t *)take(4 * U * Np);
    x.page_parent = (int32_t *)take(4 * U * Pc);
    x.page_len = (int32_t *)take(4 * U * Pc);
    x.page_next = (int32_t *)take(4 * U * Pc);
    x.page_tokens = (int32_t *)take(4 * U * Pc * S);
    x.token_parent = (int32_t *)take(4 * U * Nc);
    x.token_page = (int32_t *)take(4 * U * Nc);
    x.token_slot = (int32_t *)take(4 * U * Nc);
    if (with_pool) {
        x.pool_k = take(esz * U * Pc * S * d);
        x.pool_v = take(esz * U * Pc * S * d);
    }
    if (p.n_levels == 3) {
        x.n_nodes2 = (int32_t *)take(4 * U);
        x.node2 = (int32_t *)take(4 * U * Np);
        x.parent2 = (int32_t *)take(4 * U * Np);
        x.child_start = (int32_t *)take(4 * U * (Np + 1));
        x.children = (int32_t *)take(4 * U * Np);
    }
    if (out) *out = x;
    return off;
}

ice_status ice_index_bytes(const ice_params *p, int32_t with_pool, size_t *bytes) {
    ice_status st = check_params(p);
    if (st) return st;
    if (!bytes) return fail(ICE_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = index_layout(*p, with_pool != 0, nullptr, nullptr);
    return ICE_OK;
}

ice_status ice_index_layout(const ice_params *p, int32_t with_pool, void *base, ice_index *out) {
    ice_status st = check_params(p);
    if (st) return st;
    if (!base || !out) return fail(ICE_ERR_INVALID_ARG, "base and out must be non-NULL");
    if (((uintptr_t)base & 255u) != 0) return fail(ICE_ERR_INVALID_ARG, "base must be 256-byte aligned");
    index_layout(*p, with_pool != 0, static_cast<char *>(base), out);
    return ICE_OK;
}

ice_status ice_check(int32_t *err_dev, void *stream) {
    if (!err_dev) return fail(ICE_ERR_INVALID_ARG, "err_dev is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    ice_status st = cuda_status(cudaMemcpyAsync(&v, err_dev, sizeof(v), cudaMemcpyDeviceToHost, s), "ice_check copy");
    if (st) return st;
    if ((st = cuda_status(cudaStreamSynchronize(s), "ice_check sync"))) return st;
    if ((st = cuda_status(cudaMemsetAsync(err_dev, 0, sizeof(int32_t), s), "ice_check clear"))) return st;
    if (v != ICE_OK) fail(v, "device reported: %s", ice_status_string(v));
    return v;
}

ice_status ice_build_workspace_bytes(const ice_params *p, size_t *bytes) {
    ice_status st = check_params(p);
    if (st) return st;
    if (!bytes) return fail(ICE_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = build_ws_layout(*p, nullptr).bytes;
    return ICE_OK;
}

static ice_status build_common(const ice_params *p, const void *K, const ice_index *idx, void *ws, size_t ws_bytes,
                               BuildWs *w) {
    ice_status st = check_params(p);
    if (st) return st;
    if ((st = check_index(idx))) return st;
    if ((st = check_level2(p, idx))) return st;
    if (p->n_tokens > 0 && (!K || !aligned16(K))) return fail(ICE_ERR_INVALID_ARG, "K must be a 16-byte aligned device pointer");
    *w = build_ws_layout(*p, ws);
    return check_ws(ws, ws_bytes, w->bytes);
}

// Units with no token: counters zeroed, nothing else to do.
static ice_status build_empty(const ice_params *p, const ice_index *idx, cudaStream_t s) {
    const size_t U = (size_t)units_of(*p);
    cudaMemsetAsync(idx->n_parents, 0, sizeof(int32_t) * U, s);
    cudaMemsetAsync(idx->n_pages, 0, sizeof(int32_t) * U, s);
    cudaMemsetAsync(idx->n_indexed, 0, sizeof(int32_t) * U, s);
    cudaMemsetAsync(idx->m2, 0, sizeof(double) * U, s);
    if (p->n_levels == 3) cudaMemsetAsync(idx->n_nodes2, 0, sizeof(int32_t) * U, s);
    return cuda_status(cudaGetLastError(), "build (empty units)");
}

ice_status ice_build_lift_promote(const ice_params *p, const void *K, const ice_index *idx, void *ws,
                                  size_t ws_bytes, int32_t *err_dev, void *stream) {
    BuildWs w;
    ice_status st = build_common(p, K, idx, ws, ws_bytes, &w);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->n_tokens == 0) return build_empty(p, idx, s);
    return cuda_status(launch_lift_promote(*p, K, *idx, w, err_dev, s), "ice_build_lift_promote");
}

ice_status ice_build_assign(const ice_params *p, const void *K, const ice_index *idx, void *ws, size_t ws_bytes,
                            int32_t *err_dev, void *stream) {
    BuildWs w;
    ice_status st = build_common(p, K, idx, ws, ws_bytes, &w);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->n_tokens == 0)
        return p->n_levels == 3 ? cuda_status(cudaMemsetAsync(idx->n_nodes2, 0, sizeof(int32_t) * units_of(*p), s),
                                              "ice_build_assign")
                                : ICE_OK;
    if ((st = cuda_status(p->dtype == ICE_BF16 ? launch_assign_tc(*p, K, *idx, w, err_dev, s)
                                               : launch_assign_simt(*p, K, *idx, w, err_dev, s),
                          "ice_build_assign")))
        return st;
    if (p->n_levels == 3) return cuda_status(launch_level2(*p, *idx, w, err_dev, s), "ice_build_assign (level 2)");
    return ICE_OK;
}

ice_status ice_build_assign_simt(const ice_params *p, const void *K, const ice_index *idx, void *ws,
                                 size_t ws_bytes, int32_t *err_dev, void *stream) {
    BuildWs w;
    ice_status st = build_common(p, K, idx, ws, ws_bytes, &w);
    if (st) return st;
    if (p->n_tokens == 0) return ICE_OK;
    return cuda_status(launch_assign_simt(*p, K, *idx, w, err_dev, static_cast<cudaStream_t>(stream)),
                       "ice_build_assign_simt");
}

ice_status ice_build_pack(const ice_params *p, const void *K, const void *V, const ice_index *idx, void *ws,
                          size_t ws_bytes, int32_t *err_dev, void *stream) {
    BuildWs w;
    ice_status st = build_common(p, K, idx, ws, ws_bytes, &w);
    if (st) return st;
    if (p->n_tokens > 0 && (!V || !aligned16(V))) return fail(ICE_ERR_INVALID_ARG, "V must be a 16-byte aligned device pointer");
    if (p->n_tokens == 0) return ICE_OK;
    return cuda_status(launch_pack(*p, K, V, *idx, w, err_dev, static_cast<cudaStream_t>(stream)), "ice_build_pack");
}

ice_status ice_build_index(const ice_params *p, const void *K, const void *V, const ice_index *idx, void *ws,
                           size_t ws_bytes, int32_t *err_dev, void *stream) {
    // every argument is checked before the first stage is launched
    BuildWs w;
    ice_status st = build_common(p, K, idx, ws, ws_bytes, &w);
    if (st) return st;
    if (p->n_tokens > 0 && (!V || !aligned16(V))) return fail(ICE_ERR_INVALID_ARG, "V must be a 16-byte aligned device pointer");
    st = ice_build_lift_promote(p, K, idx, ws, ws_bytes, err_dev, stream);
    if (st) return st;
    if ((st = ice_build_assign(p, K, idx, ws, ws_bytes, err_dev, stream))) return st;
    return ice_build_pack(p, K, V, idx, ws, ws_bytes, err_dev, stream);
}

ice_status ice_build_index_reuse(const ice_params *p, const void *K, const void *V, const ice_index *prev,
                                 const ice_index *idx, void *ws, size_t ws_bytes, int32_t *err_dev, void *stream) {
    BuildWs w;
    ice_status st = build_common(p, K, idx, ws, ws_bytes, &w);
    if (st) return st;
    if ((st = check_index(prev)) || (st = check_level2(p, prev))) return st;
    if (p->n_tokens > 0 && (!V || !aligned16(V))) return fail(ICE_ERR_INVALID_ARG, "V must be a 16-byte aligned device pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->n_tokens == 0) return build_empty(p, idx, s);
    return cuda_status(launch_build_reuse(*p, K, V, *prev, *idx, w, err_dev, s), "ice_build_index_reuse");
}

// ------------------------------------------------------------- insert ----
ice_status ice_insert_workspace_bytes(const ice_params *p, size_t *bytes) {
    ice_status st = check_params(p);
    if (st) return st;
    if (!bytes) return fail(ICE_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = insert_ws_layout(*p, nullptr).bytes;
    return ICE_OK;
}

ice_status ice_insert_tokens(const ice_params *p, const ice_index *idx, const void *k_new, const void *v_new,
                             void *ws, size_t ws_bytes, int32_t *err_dev, void *stream) {
    ice_status st = check_params(p);
    if (st) return st;
    if ((st = check_index(idx))) return st;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return fail(ICE_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned device pointers");
    if (p->n_sink > 0 || p->n_window > 0)
        return fail(ICE_ERR_UNSUPPORTED, "incremental insert is not supported with sink or window pages");
    if (p->n_levels != 2) return fail(ICE_ERR_UNSUPPORTED, "incremental insert is supported with two levels");
    const InsertWs w = insert_ws_layout(*p, ws);
    if ((st = check_ws(ws, ws_bytes, w.bytes))) return st;
    return cuda_status(launch_insert(*p, *idx, k_new, v_new, w, err_dev, static_cast<cudaStream_t>(stream)),
                       "ice_insert_tokens");
}

// ------------------------------------------------------------- decode ----
static ice_status decode_common(const ice_params *p, int32_t budget_tokens, int32_t max_sel, void *ws,
                                size_t ws_bytes, DecodeWs *w) {
    ice_status st = check_params(p);
    if (st) return st;
    if (budget_tokens < 0) return fail(ICE_ERR_INVALID_ARG, "budget_tokens must be >= 0");
    if (max_sel < 1) return fail(ICE_ERR_INVALID_ARG, "max_sel must be >= 1");
    *w = decode_ws_layout(*p, budget_tokens, max_sel, ws);
    return check_ws(ws, ws_bytes, w->bytes);
}

ice_status ice_decode_workspace_bytes(const ice_params *p, int32_t budget_tokens, int32_t max_sel, size_t *bytes) {
    ice_status st = check_params(p);
    if (st) return st;
    if (!bytes) return fail(ICE_ERR_INVALID_ARG, "bytes is NULL");
    if (budget_tokens < 0 || max_sel < 1) return fail(ICE_ERR_INVALID_ARG, "need budget_tokens >= 0 and max_sel >= 1");
    *bytes = decode_ws_layout(*p, budget_tokens, max_sel, nullptr).bytes;
    return ICE_OK;
}

static ice_status select_checks(const ice_params *p, const ice_index *idx, const void *Q, int32_t budget_tokens,
                                int32_t *sel_pages, int32_t *sel_count, int32_t max_sel, const DecodeWs &w) {
    ice_status st = check_index(idx);
    if (st) return st;
    if ((st = check_level2(p, idx))) return st;
    if (!Q || !sel_pages || !sel_count) return fail(ICE_ERR_INVALID_ARG, "Q, sel_pages and sel_count must be non-NULL");
    if (!aligned16(Q)) return fail(ICE_ERR_INVALID_ARG, "Q must be 16-byte aligned");
    if (p->n_levels == 3 && k_pages_of(budget_tokens) > 32)
        return fail(ICE_ERR_UNSUPPORTED, "the three-level descent takes at most 32 pages per head");
    const long long g = p->n_q_heads / p->n_kv_heads;
    const long long need = g * (long long)k_pages_of(budget_tokens) + pos_split(*p).n_pos;
    const long long want = need < p->page_cap ? need : p->page_cap;
    if (max_sel < want)
        return fail(ICE_ERR_INVALID_ARG, "max_sel (%d) must be >= min(g * k + positional pages, page_cap) = %lld",
                    max_sel, want);
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const size_t smem = select_smem_bytes(*p, w.k_pages, w.n_chunks);
    if (optin > 0 && smem + 1024 > (size_t)optin)
        return fail(ICE_ERR_UNSUPPORTED, "selection needs %zu bytes of shared memory (budget or page_cap too large)", smem);
    return ICE_OK;
}

ice_status ice_select_pages(const ice_params *p, const ice_index *idx, const void *Q, int32_t budget_tokens,
                            int32_t *sel_pages, int32_t *sel_count, int32_t max_sel, void *ws, size_t ws_bytes,
                            int32_t *err_dev, void *stream) {
    DecodeWs w;
    ice_status st = decode_common(p, budget_tokens, max_sel, ws, ws_bytes, &w);
    if (st) return st;
    if ((st = select_checks(p, idx, Q, budget_tokens, sel_pages, sel_count, max_sel, w))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->n_levels == 3)
        return cuda_status(launch_select3(*p, *idx, Q, w, sel_pages, sel_count, max_sel, err_dev, s),
                           "ice_select_pages");
    return cuda_status(launch_select(*p, *idx, Q, w, sel_pages, sel_count, max_sel, err_dev, s),
                       "ice_select_pages");
}

ice_status ice_gather_pages(const ice_params *p, const ice_index *idx, const int32_t *sel_pages,
                            const int32_t *sel_count, int32_t max_sel, void *kbuf, void *vbuf, int32_t *buf_len,
                            void *stream) {
    ice_status st = check_params(p);
    if (st) return st;
    if ((st = check_index(idx))) return st;
    if (!sel_pages || !sel_count || !kbuf || !vbuf || !buf_len || max_sel < 1)
        return fail(ICE_ERR_INVALID_ARG, "gather needs non-NULL buffers and max_sel >= 1");
    if (!aligned16(kbuf) || !aligned16(vbuf)) return fail(ICE_ERR_INVALID_ARG, "kbuf and vbuf must be 16-byte aligned");
    return cuda_status(launch_gather(*p, *idx, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len,
                                     static_cast<cudaStream_t>(stream)),
                       "ice_gather_pages");
}

ice_status ice_sparse_attn_decode(const ice_params *p, const void *Q, const void *kbuf, const void *vbuf,
                                  const int32_t *buf_len, const int32_t *sel_count, int32_t max_sel, float scale,
                                  float *O, void *ws, size_t ws_bytes, void *stream) {
    DecodeWs w;
    ice_status st = decode_common(p, 0, max_sel, ws, ws_bytes, &w);
    if (st) return st;
    if (!Q || !kbuf || !vbuf || !buf_len || !sel_count || !O)
        return fail(ICE_ERR_INVALID_ARG, "attention needs non-NULL Q, kbuf, vbuf, buf_len, sel_count and O");
    if (!aligned16(kbuf) || !aligned16(vbuf) || !aligned16(Q))
        return fail(ICE_ERR_INVALID_ARG, "Q, kbuf and vbuf must be 16-byte aligned");
    return cuda_status(launch_attention(*p, nullptr, nullptr, Q, const_cast<void *>(kbuf), const_cast<void *>(vbuf),
                                        const_cast<int32_t *>(buf_len), sel_count, max_sel, scale, O, w,
                                        static_cast<cudaStream_t>(stream)),
                       "ice_sparse_attn_decode");
}

ice_status ice_sparse_attn_decode_noalloc(const ice_params *p, const void *Q, const void *kbuf, const void *vbuf,
                                          const int32_t *buf_len, const int32_t *sel_count, int32_t max_sel,
                                          float scale, float *O, void *stream) {
    ice_status st = check_params(p);
    if (st) return st;
    if (max_sel < 1) return fail(ICE_ERR_INVALID_ARG, "max_sel must be >= 1");
    if (!Q || !kbuf || !vbuf || !buf_len || !sel_count || !O)
        return fail(ICE_ERR_INVALID_ARG, "attention needs non-NULL Q, kbuf, vbuf, buf_len, sel_count and O");
    if (!aligned16(kbuf) || !aligned16(vbuf)) return fail(ICE_ERR_INVALID_ARG, "kbuf and vbuf must be 16-byte aligned");
    const size_t need = attention_noalloc_bytes(*p, max_sel);
    if (need > ICE_NOALLOC_SCRATCH_BYTES)
        return fail(ICE_ERR_CAPACITY, "this shape needs %zu bytes of scratch; the allocation-free entry point has %u",
                    need, (unsigned)ICE_NOALLOC_SCRATCH_BYTES);
    return cuda_status(launch_attention_noalloc(*p, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O,
                                                static_cast<cudaStream_t>(stream)),
                       "ice_sparse_attn_decode_noalloc");
}

ice_status ice_decode_step(const ice_params *p, const ice_index *idx, const void *Q, int32_t budget_tokens,
                           int32_t *sel_pages, int32_t *sel_count, int32_t max_sel, void *kbuf, void *vbuf,
                           int32_t *buf_len, float scale, float *O, void *ws, size_t ws_bytes, int32_t *err_dev,
                           void *stream) {
    DecodeWs w;
    ice_status st = decode_common(p, budget_tokens, max_sel, ws, ws_bytes, &w);
    if (st) return st;
    if ((st = select_checks(p, idx, Q, budget_tokens, sel_pages, sel_count, max_sel, w))) return st;
    if (!O) return fail(ICE_ERR_INVALID_ARG, "decode needs a non-NULL O");
    const bool no_buffer = !kbuf && !vbuf && !buf_len;  // pages gathered on chip only
    if (!no_buffer && (!kbuf || !vbuf || !buf_len))
        return fail(ICE_ERR_INVALID_ARG, "kbuf, vbuf and buf_len must be all non-NULL or all NULL");
    if (!aligned16(kbuf) || !aligned16(vbuf)) return fail(ICE_ERR_INVALID_ARG, "kbuf and vbuf must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorNotSupported;
    switch (decode_plan(*p, w.k_pages, max_sel)) {
    case ICE_PLAN_DESCENT:  // descent through level 2, then the pages streamed from the pool
        e = launch_select3(*p, *idx, Q, w, sel_pages, sel_count, max_sel, err_dev, s);
        if (e == cudaSuccess)
            e = launch_attention(*p, idx, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, w, s,
                                 err_dev);
        return cuda_status(e, "ice_decode_step");
    case ICE_PLAN_CLUSTER_BF16:
        e = launch_decode_cluster2(*p, *idx, Q, w.k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale,
                                   O, err_dev, s);
        break;
    case ICE_PLAN_CLUSTER:
        e = launch_decode_cluster(*p, *idx, Q, w.k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale,
                                  O, err_dev, s);
        break;
    case ICE_PLAN_SCORE_SELECT:  // the score table, then attention CTAs that select their unit's pages
        e = launch_score_tc(*p, *idx, Q, w, err_dev, s);
        if (e == cudaSuccess) {
            SelArgs A = select_args(*p, *idx, w, sel_pages, sel_count, max_sel, err_dev);
            if (in_device_memory(idx->pool_k) && in_device_memory(idx->pool_v)) {  // not a host page pool
                A.pf_k = static_cast<const unsigned char *>(idx->pool_k);
                A.pf_v = static_cast<const unsigned char *>(idx->pool_v);
                A.page_bytes = kPage * kHeadDim * 2;  // bf16
            }
            e = launch_attention_mma_select(*p, *idx, A, Q, kbuf, vbuf, buf_len, max_sel, scale, O, w, err_dev, s);
        }
        return cuda_status(e, "ice_decode_step");
    default:
        break;
    }
    if (e != cudaErrorNotSupported) return cuda_status(e, "ice_decode_step");
    // the score table on the tensor cores and the per-unit top-k (bf16), or the SIMT selection;
    // then the fused gather + attention
    if (select_tc_supported(*p, w.k_pages)) {
        e = launch_score_tc(*p, *idx, Q, w, err_dev, s);
        if (e == cudaSuccess) e = launch_topk(*p, select_args(*p, *idx, w, sel_pages, sel_count, max_sel, err_dev), s);
    } else {
        e = launch_select(*p, *idx, Q, w, sel_pages, sel_count, max_sel, err_dev, s);
    }
    if (e == cudaSuccess)
        e = launch_attention(*p, idx, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, w, s, err_dev);
    return cuda_status(e, "ice_decode_step");
}

ice_status ice_decode_plan(const ice_params *p, int32_t budget_tokens, int32_t max_sel, int32_t *step_plan,
                           int32_t *attention_plan) {
    ice_status st = check_params(p);
    if (st) return st;
    if (budget_tokens < 0 || max_sel < 1) return fail(ICE_ERR_INVALID_ARG, "need budget_tokens >= 0 and max_sel >= 1");
    if (step_plan) *step_plan = decode_plan(*p, k_pages_of(budget_tokens), max_sel);
    if (attention_plan) *attention_plan = attention_mma_fits(*p, max_sel) ? ICE_PLAN_ATTN_MMA : ICE_PLAN_ATTN_SIMT;
    return ICE_OK;
}

}  // extern "C"
