// Internal launch interface between the C ABI layer (abi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ice.h"

namespace ice {

// Tokens per tile of the lift/promotion kernels and of the page-packing kernels.
constexpr int kLiftTile = 256;
constexpr int kPackTile = 2048;
// Parents per CTA of the selection scan.
constexpr int kSelChunk = 256;
// Selected pages per CTA of the split attention.
constexpr int kAttnPagesPerSplit = 4;
// Largest parent count whose per-tile histogram fits in shared memory.
constexpr int kPackSmemBins = 12288;

inline int units_of(const ice_params &p) { return p.batch * p.n_kv_heads; }

// Fault injection for tests, on the host: the environment variable ICE_FAULT
// holds a comma-separated list of
//   alloc     ice_host_pool_create fails its first pinned allocation (ICE_ERR_OOM)
//   hostpool  ice_host_pool_create fails after its allocations, at the device
//             mapping (ICE_ERR_CUDA; everything allocated is freed)
//   copy      ice_host_pool_gather_h2d fails its bulk copy (ICE_ERR_CUDA)
//   timeout   the attention kernel's page producer issues no copy, and its
//             bounded waits give up after kFaultWaitNs (ICE_ERR_TIMEOUT)
// Read at every call; unset (the default) nothing changes.
bool fault_armed(const char *what);
constexpr unsigned long long kFaultWaitNs = 20000000ull;  // 20 ms
inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Sink / window split of a build over p.n_tokens tokens: the index covers the
// middle [lo, hi); the sink [0, lo) and the window [hi, N) fill n_pos
// positional pages after the semantic ones.
struct PosSplit {
    int lo, hi, n_pos;
};
inline PosSplit pos_split(const ice_params &p) {
    const int N = p.n_tokens;
    const int lo = p.n_sink < N ? (p.n_sink > 0 ? p.n_sink : 0) : N;
    const int w = p.n_window > 0 ? p.n_window : 0;
    const int hi = N - w > lo ? N - w : lo;
    return PosSplit{lo, hi, (lo + 15) / 16 + (N - hi + 15) / 16};
}

// ------------------------------------------------ workspace layouts -------
struct BuildWs {
    double *norm2;        // [U, N]  |k_j|^2 (double)
    int32_t *pcount;      // [U, Tp] promoted tokens per lift tile
    double *tile_max;     // [U, Tp] largest |k|^2 of each lift tile
    unsigned long long *tile_min;  // [U, Tp] smallest draw << 32 | token of each lift tile
    uint4 *a_extra;       // [U, N, 16] bf16: split lifted coordinate of each token (tensor-core K tail)
    uint4 *b_extra;       // [U, np_cap, 16] bf16: the same for each parent
    int32_t *pack_cnt;    // [U, Tk, np_cap] per-tile parent counts -> offsets
    int32_t *pack_total;  // [U, np_cap] tokens per parent
    // three levels, bf16: the level-2 contraction's operands, gathered dense
    uint4 *a_extra2;      // [U, np_cap, 16] bf16: each parent's split lifted coordinate, row form
    void *keys2;          // [U, np_cap, d] the level-2 nodes' keys
    uint4 *b_extra2;      // [U, np_cap, 16] bf16: each level-2 node's split lifted coordinate, column form
    size_t bytes;
};
BuildWs build_ws_layout(const ice_params &p, void *base);

struct DecodeWs {
    int32_t *sel_ticket;   // [U]  zero between calls
    int32_t *attn_ticket;  // [U]  zero between calls
    unsigned long long *cand_key;  // [U, n_chunks, g, kc] sorted (-score, m) keys
    int4 *cand_span;       // [U, n_chunks, 256] (first page, pages, contiguous, m)
    float *part_ml;        // [U, n_splits, g, 2]  running max, running sum
    float *part_o;         // [U, n_splits, g, d]
    float *scores;         // [U, g, np_cap] parent scores of the tensor-core selection
    int n_chunks, k_pages, n_splits;
    size_t bytes;
};
// What the page selection of a unit reads and writes (score table, group
// maxima, page spans; the ascending page list per unit).
struct SelArgs {
    int g, np_cap, page_cap, k_pages, kc, max_sel;
    int n_pos;  // positional pages at the end of each unit's pages, always in the union
    const int32_t *n_parents, *n_pages;
    const float *scores, *gmax;
    const int32_t *parent_first_page, *parent_last_page, *parent_n_pages, *page_next;
    int32_t *sel_pages, *sel_count, *err;
    // the decode step's page pools (device memory): each query head's first
    // kPrefetchPages pages are prefetched into L2 as soon as they are known
    // (NULL: no prefetch)
    const unsigned char *pf_k, *pf_v;
    int page_bytes;
};

// with_select = false: the attention part only (no selection scratch).
DecodeWs decode_ws_layout(const ice_params &p, int budget_tokens, int max_sel, void *base, bool with_select = true);

struct InsertWs {
    int32_t *ticket;  // [U]  zero between calls
    float *best_s;    // [U, n_chunks]
    int32_t *best_m;  // [U, n_chunks]
    int n_chunks;
    size_t bytes;
};
InsertWs insert_ws_layout(const ice_params &p, void *base);
cudaError_t launch_insert(const ice_params &p, const ice_index &idx, const void *k_new, const void *v_new,
                          const InsertWs &ws, int32_t *err, cudaStream_t s);

// --------------------------------------------------------- launchers ------
// Each returns cudaGetLastError() after enqueueing its kernels.
cudaError_t launch_lift_promote(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                                int32_t *err, cudaStream_t s);
cudaError_t launch_assign_simt(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                               int32_t *err, cudaStream_t s);
cudaError_t launch_assign_tc(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                             int32_t *err, cudaStream_t s);
cudaError_t launch_pack(const ice_params &p, const void *K, const void *V, const ice_index &idx,
                        const BuildWs &ws, int32_t *err, cudaStream_t s);
// Level 2 of a three-level index (promotion, nearest level-2 node, children).
cudaError_t launch_level2(const ice_params &p, const ice_index &idx, const BuildWs &ws, int32_t *err,
                          cudaStream_t s);
// The parents' nearest level-2 node on the tensor cores (bf16): k_assign_tc
// over the parent table against the gathered level-2 table.
cudaError_t launch_assign_level2_tc(const ice_params &p, const ice_index &idx, const BuildWs &ws, int32_t *err,
                                    cudaStream_t s);
// Page selection by descent through level 2 (n_levels = 3).
cudaError_t launch_select3(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                           int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s);
constexpr int kLevel2MaxParents = 50000;  // parent capacity the level-2 counting sort holds in shared memory
// Pieces of the build used by the reuse build: the squared norms and per-tile
// maxima of k_lift_count, and the pool scatter k_pack_copy over idx's pages.
cudaError_t launch_lift_norms(const ice_params &p, const void *K, const BuildWs &ws, cudaStream_t s);
cudaError_t launch_pack_copy(const ice_params &p, const void *K, const void *V, const ice_index &idx,
                             cudaStream_t s);
// Build of a layer on another layer's node structure (parents, assignment,
// pages): lift of this layer's keys, parent keys, table copies, pool.
cudaError_t launch_build_reuse(const ice_params &p, const void *K, const void *V, const ice_index &prev,
                               const ice_index &idx, const BuildWs &ws, int32_t *err, cudaStream_t s);
cudaError_t launch_select(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                          int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s);
// Selection with tensor-core scoring (bf16, g <= 16, k <= 64 pages per head).
bool select_tc_supported(const ice_params &p, int k_pages);
size_t select_tc_scores(const ice_params &p);
cudaError_t launch_select_tc(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                             int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s);
SelArgs select_args(const ice_params &p, const ice_index &idx, const DecodeWs &ws, int32_t *sel_pages,
                    int32_t *sel_count, int max_sel, int32_t *err);
cudaError_t launch_score_tc(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                            int32_t *err, cudaStream_t s);
cudaError_t launch_topk(const ice_params &p, const SelArgs &A, cudaStream_t s);

cudaError_t launch_gather(const ice_params &p, const ice_index &idx, const int32_t *sel_pages,
                          const int32_t *sel_count, int max_sel, void *kbuf, void *vbuf, int32_t *buf_len,
                          cudaStream_t s);
// pool == nullptr: attention over kbuf/vbuf/buf_len (step a10 alone).
// pool != nullptr: each CTA first copies its selected pages from the pool to
// kbuf/vbuf/buf_len (step a9) and attends over that copy (fused a9 + a10).
cudaError_t launch_attention(const ice_params &p, const ice_index *pool, const int32_t *sel_pages,
                             const void *Q, void *kbuf, void *vbuf, int32_t *buf_len, const int32_t *sel_count,
                             int max_sel, float scale, float *O, const DecodeWs &ws, cudaStream_t s,
                             int32_t *err = nullptr);
// The same with the page contractions on warp-level MMAs (bf16, g <= 16).
bool attention_mma_supported(const ice_params &p);
bool attention_mma_fits(const ice_params &p, int max_sel);
// The attention CTAs select their unit's pages first (from the score table).
bool attention_mma_select_supported(const ice_params &p, int max_sel);
cudaError_t launch_attention_mma_select(const ice_params &p, const ice_index &idx, const SelArgs &A, const void *Q,
                                        void *kbuf, void *vbuf, int32_t *buf_len, int max_sel, float scale, float *O,
                                        const DecodeWs &ws, int32_t *err, cudaStream_t s);
cudaError_t launch_attention_mma(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q,
                                 void *kbuf, void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel,
                                 float scale, float *O, const DecodeWs &ws, int32_t *err, cudaStream_t s);

// The whole decode step of a unit in one thread-block cluster (DSMEM
// exchanges, hardware cluster barriers); supported when the unit's parent
// slice and candidate lists fit its shared memory.
constexpr int kDecodeCluster = 8;
bool decode_cluster_supported(const ice_params &p, int k_pages, int max_sel);
cudaError_t launch_decode_cluster(const ice_params &p, const ice_index &idx, const void *Q, int k_pages,
                                  int32_t *sel_pages, int32_t *sel_count, int max_sel, void *kbuf, void *vbuf,
                                  int32_t *buf_len, float scale, float *O, int32_t *err, cudaStream_t s);

// The same for bf16 tables with g <= 8 and k <= 32 pages per head: bulk-copied
// pages, bisection top-k, packed fp32-pair arithmetic.
bool decode_cluster2_supported(const ice_params &p, int k_pages, int max_sel);
cudaError_t launch_decode_cluster2(const ice_params &p, const ice_index &idx, const void *Q, int k_pages,
                                   int32_t *sel_pages, int32_t *sel_count, int max_sel, void *kbuf, void *vbuf,
                                   int32_t *buf_len, float scale, float *O, int32_t *err, cudaStream_t s);

// Allocation-free attention: scratch in the library's static device array.
size_t attention_noalloc_bytes(const ice_params &p, int max_sel);
cudaError_t launch_attention_noalloc(const ice_params &p, const void *Q, const void *kbuf, const void *vbuf,
                                     const int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale,
                                     float *O, cudaStream_t s);

}  // namespace ice
