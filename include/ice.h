/*
 * ice.h -- C ABI of the IceCache hot path for one GB300 (sm_103a).
 *
 * IceCache keeps a long KV cache in pages whose tokens are grouped by key
 * similarity instead of position, and at decode time loads only the pages a
 * query needs.  Sources, by page and section:
 *   [A] "IceCache: Memory-Efficient KV-cache Management for Long-Sequence
 *       LLMs" (papernotes.org ICLR 2026 notes), 方法详解 / 整体框架 and
 *       关键设计 1-4.
 *   [B] IceCache popular-science article (aitangshan.cn/news/751385),
 *       sections 二, 三, 四 and 六.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every function returns an ice_status (ICE_OK = 0).  On a non-zero
 *    return nothing was launched unless the code is ICE_ERR_CUDA, and
 *    ice_last_error() (thread-local) describes the failure.
 *  - Every array argument is a raw pointer owned by the caller: DEVICE memory
 *    unless the argument says "host".  Arrays are dense row-major with the
 *    shapes written next to them.  The library never allocates, frees or
 *    keeps a pointer after the call returns (the host page pool is the one
 *    library-owned object, see ice_host_pool_create).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous: no entry point synchronises unless it says
 *    so.  Scratch memory comes from the caller's workspace `ws` of `ws_bytes`
 *    bytes (256-byte aligned), sized by the matching *_workspace_bytes query.
 *  - K, V, Q, k_new, v_new, kbuf, vbuf and the index's parent_keys, pool_k
 *    and pool_v must be 16-byte aligned (ICE_ERR_INVALID_ARG otherwise).
 *  - A "unit" is one (sequence b, KV head h) pair of one layer; units are
 *    numbered u = b * n_kv_heads + h and are fully independent.
 *  - Conditions only the device can see (a capacity that turns out too
 *    small) are written to the caller's device word `err_dev` (int32, set to
 *    0 by the caller before first use) as an ice_status; the kernels then
 *    clamp every write to the capacities, so memory outside the arrays is
 *    never touched.  ice_check() reads and clears that word.
 *  - Overlap ([A] 关键设计 4, the three-stage pipeline): since every call is
 *    stream-ordered, a caller overlaps layer i + 1's host-to-device copy of
 *    K, V and Q (one stream) with layer i's ice_build_index and
 *    ice_decode_step (another stream), ordering them with events: the copy
 *    of layer i + 1 waits for the last use of the buffers it overwrites, the
 *    build of layer i + 1 for its copy.  Calls that share a workspace stay on
 *    one stream.
 *  - Floating point: keys/values/queries are bf16 or fp32 (ice_params.dtype);
 *    every score and every softmax is accumulated in fp32; outputs O are
 *    fp32.
 */
#ifndef ICE_H_
#define ICE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ice_status;
#define ICE_OK 0
#define ICE_ERR_INVALID_ARG 1
#define ICE_ERR_CUDA 2
#define ICE_ERR_OOM 3
#define ICE_ERR_CAPACITY 4
#define ICE_ERR_TIMEOUT 5
#define ICE_ERR_UNSUPPORTED 6

#define ICE_BF16 0
#define ICE_FP32 1

/* Shapes and knobs of one layer's index.  All fields are plain values. */
typedef struct ice_params {
    int32_t batch;          /* B: sequences */
    int32_t n_q_heads;      /* Hq */
    int32_t n_kv_heads;     /* Hkv; Hq must be a multiple (g = Hq / Hkv) */
    int32_t head_dim;       /* d; 128 is the supported value */
    int32_t n_tokens;       /* N: tokens per unit given to ice_build_index */
    int32_t page_size;      /* S; 16 is the supported value ([B] section 二) */
    int32_t dtype;          /* ICE_BF16 or ICE_FP32 for K, V, Q and the pool */
    int32_t n_levels;       /* index levels: 2 (tokens, parents) or 3 (+ a level above the parents) */
    uint64_t promote_thresh;/* floor(p * 2^32), 0 .. 2^32: promotion probability p */
    uint64_t seed;          /* promotion seed */
    int32_t layer;          /* layer id (enters the promotion draw) */
    int32_t np_cap;         /* parent capacity per unit */
    int32_t page_cap;       /* page capacity per unit */
    int32_t n_cap;          /* token capacity per unit (>= n_tokens; room for inserts) */
    int32_t n_sink;         /* first n_sink tokens kept as positional pages ([B] section 六) */
    int32_t n_window;       /* last n_window tokens of the build kept as positional pages */
} ice_params;

/*
 * Sink and recent-window pages ([B] section 六: the anchor tokens at the start
 * and the window of newest tokens stay resident on the GPU; only the tokens in
 * between are managed by the index).  With n_sink or n_window > 0 a build over
 * N tokens indexes only the middle tokens [sink_end, window_start), where
 * sink_end = min(n_sink, N) and window_start = max(sink_end, N - n_window):
 * M^2, the promotion and the nearest parent are taken over the middle only.
 * After the middle's semantic pages, the sink tokens fill positional pages in
 * token order, S per page, and then the window tokens; these pages have
 * page_parent -1 and their tokens token_parent -2.  Every decode step attends
 * over all positional pages (the last ice_positional_pages(...) pages of the
 * unit) besides the budget's selected pages, so max_sel must cover both, and
 * page_cap must hold the positional pages besides ice_page_bound of the
 * middle.  Incremental insert is not supported with positional pages.
 */
/* The positional page count of a unit: ceil(sink_end / S) +
 * ceil((N - window_start) / S) (0 when n_sink = n_window = 0). */
int32_t ice_positional_pages(int32_t n_tokens, int32_t n_sink, int32_t n_window, int32_t page_size);

/*
 * Device arrays of one layer's index, all caller-owned.  U = B * Hkv units.
 * Sizes: Np = np_cap, Pc = page_cap, Nc = n_cap, S = page_size, d = head_dim.
 *
 *  per unit      n_parents[U], n_pages[U], n_indexed[U] (tokens indexed so
 *                far: N after the build, +1 per insert) int32;
 *                m2[U] double: M^2, the squared largest key norm of the build.
 *  parent level  parent_tok[U,Np] int32 (token of parent m, ascending);
 *                parent_keys[U,Np,d] (dtype, the parent tokens' keys);
 *                parent_e[U,Np] float: lifted extra coordinate
 *                  sqrt(max(0, M^2 - |p|^2));
 *                parent_corr[U,Np] float: (M^2 - max(M^2, |p|^2)) / 2, zero
 *                  for every parent chosen at build time;
 *                parent_first_page[U,Np], parent_last_page[U,Np],
 *                parent_n_pages[U,Np] int32.
 *  pages         page_parent[U,Pc], page_len[U,Pc] (1..S),
 *                page_next[U,Pc] (next page of the same parent, -1 at the
 *                end), page_tokens[U,Pc,S] (token of each slot, -1 pad) int32.
 *  tokens        token_parent[U,Nc], token_page[U,Nc], token_slot[U,Nc] int32.
 *  pool          pool_k[U,Pc,S,d], pool_v[U,Pc,S,d] (dtype): each page's K and
 *                V rows in slot order, pad slots zero ([A] 整体框架: one
 *                node = one physical page).
 * Only the first n_parents / n_pages / n_indexed entries of a unit are
 * defined after a call.
 */
typedef struct ice_index {
    int32_t *n_parents;
    int32_t *n_pages;
    int32_t *n_indexed;
    double *m2;
    int32_t *parent_tok;
    void *parent_keys;
    float *parent_e;
    float *parent_corr;
    int32_t *parent_first_page;
    int32_t *parent_last_page;
    int32_t *parent_n_pages;
    int32_t *page_parent;
    int32_t *page_len;
    int32_t *page_next;
    int32_t *page_tokens;
    int32_t *token_parent;
    int32_t *token_page;
    int32_t *token_slot;
    void *pool_k;
    void *pool_v;
    /* Level 2 (ice_params.n_levels = 3 only; may be NULL with 2 levels):
     * n_nodes2[U]; node2[U,Np] the parent m of level-2 node i (ascending m);
     * parent2[U,Np] the level-2 node of parent m; child_start[U,Np+1] and
     * children[U,Np]: the parents of level-2 node i, ascending, at
     * children[child_start[i] .. child_start[i+1]) (all int32). */
    int32_t *n_nodes2;
    int32_t *node2;
    int32_t *parent2;
    int32_t *child_start;
    int32_t *children;
} ice_index;

/* ---------------------------------------------------------------- misc -- */
const char *ice_status_string(ice_status s);
/* Message for the last failing call on this host thread ("" if none). */
const char *ice_last_error(void);
/* Library version string. */
const char *ice_version(void);
/* Synchronises `stream`, reads the device error word, clears it and returns
 * its value (ICE_OK when no device-side condition was raised). */
ice_status ice_check(int32_t *err_dev, void *stream);
/* Largest page count a unit of N tokens with Np parents can need:
 * sum_m ceil(c_m / S) <= (N + (S - 1) * Np) / S, rounded down (the sum is an
 * integer). */
int32_t ice_page_bound(int32_t n_tokens, int32_t n_parents, int32_t page_size);

/*
 * Capacities.  Fills p->np_cap and p->page_cap (and p->n_cap, raised to
 * max(n_tokens, 1) when smaller) from n_cap, promote_thresh, n_sink and
 * n_window; the other fields are left as they are.
 *   np_cap   = min(n_cap, floor(mu + 8 sqrt(mu (1 - q) + 1) + 16)), at least
 *              1, where q = promote_thresh / 2^32 and mu = n_cap q: the
 *              promoted count is Binomial(n_cap, q), so the 8-sigma margin
 *              is exceeded with negligible probability, and a build that
 *              exceeds it reports ICE_ERR_CAPACITY without writing past it.
 *              np_cap = n_cap is the bound that always holds.
 *   page_cap = ice_page_bound(n_cap, np_cap, S) + the positional pages.
 * ICE_ERR_INVALID_ARG / ICE_ERR_UNSUPPORTED on a bad n_tokens, page_size,
 * promote_thresh, n_sink or n_window.
 */
ice_status ice_default_capacities(ice_params *p);

/*
 * Sizing of an index.  Every array of an ice_index for the shapes and
 * capacities in *p (sizes as listed above ice_index) fits in one slab of
 * *bytes bytes, each array starting on a 256-byte boundary, in ice_index
 * field order.  with_pool = 0 leaves the pool out (a host page pool holds
 * it; see ice_host_pool_create).  The level-2 arrays are counted only when
 * n_levels = 3.
 */
ice_status ice_index_bytes(const ice_params *p, int32_t with_pool, size_t *bytes);
/*
 * Fills *out with pointers into the caller's slab `base` (device memory of
 * ice_index_bytes bytes, 256-byte aligned) at the offsets ice_index_bytes
 * counts.  Nothing is read or written at base: the caller zero-fills the
 * slab if it wants defined contents before the first build.  Pool and
 * level-2 pointers that are not counted are set to NULL.  The caller owns
 * the slab; the library keeps no pointer.
 */
ice_status ice_index_layout(const ice_params *p, int32_t with_pool, void *base, ice_index *out);

/* ------------------------------------------------------ index build ----- */
/* Workspace bytes needed by ice_build_index and its three stages. */
ice_status ice_build_workspace_bytes(const ice_params *p, size_t *bytes);

/*
 * Builds every unit's index from K, V [B, Hkv, N, d] (dtype):
 * ice_build_lift_promote, then ice_build_assign, then ice_build_pack, on one
 * stream.  The three stages are also exported so that they can be timed or
 * overlapped separately; they must run in this order with the same
 * arguments and workspace.  Every argument (params, index arrays, K, V,
 * workspace) is checked before the first stage is launched:
 * ICE_ERR_INVALID_ARG / ICE_ERR_UNSUPPORTED leave the index untouched.
 */
ice_status ice_build_index(const ice_params *p, const void *K, const void *V, const ice_index *idx,
                           void *ws, size_t ws_bytes, int32_t *err_dev, void *stream);

/*
 * Stage a1 + a2: the key lift and the random promotion.
 * Lift ([B] sections 三 and 六; [A] 关键设计 2): with n_j = |k_j|^2 and
 * M^2 = max_j n_j, every key becomes k'_j = [k_j, sqrt(M^2 - n_j)], so all
 * lifted keys have norm M and nearest-neighbour search in lifted space is
 * maximum inner-product search.  n_j and M^2 are computed exactly enough
 * that the fp32 extra coordinate is the correctly rounded value.
 * Promotion ([B] section 三): every token is at level 0; token j is promoted
 * to level 1 iff draw(j) < promote_thresh, where draw is the top 32 bits of
 * a splitmix64 output (Steele, Lea & Flood 2014) at counter
 * (token | 1 << 32 | h << 40 | b << 52) + 1 in the stream keyed by output
 * (layer + 1) of the stream seeded by `seed`.  If no token of a unit is
 * promoted, its token with the smallest draw is (lowest token on equal
 * draws).  Parents m = 0..Np-1 are the promoted tokens in ascending order.
 * Writes m2, n_parents, parent_tok, parent_keys, parent_e, parent_corr (0),
 * token_parent (m for a promoted token, -1 otherwise), n_indexed = N.
 * Requires B, Hkv < 4096.  ICE_ERR_CAPACITY in err_dev if Np > np_cap.
 */
ice_status ice_build_lift_promote(const ice_params *p, const void *K, const ice_index *idx, void *ws,
                                  size_t ws_bytes, int32_t *err_dev, void *stream);

/*
 * Stage a3: nearest parent ([B] section 三: every token takes as parent the
 * most similar point one level up; [A] 关键设计 2).
 *   parent(j) = argmin_m |k'_j - p'_m|^2 = argmax_m (k_j . p_m + e_j e_m)
 * with the dot product of the stored keys accumulated in fp32 (bf16: the
 * sm_103a tensor cores, fp32: CUDA cores) and exact fp32 ties going to the
 * lowest m.  A promoted token keeps itself as parent.  Writes token_parent.
 */
ice_status ice_build_assign(const ice_params *p, const void *K, const ice_index *idx, void *ws,
                            size_t ws_bytes, int32_t *err_dev, void *stream);
/*
 * With n_levels = 3, ice_build_assign (and so ice_build_index) also builds
 * level 2 ([A] 关键设计 2: points are promoted level by level and every
 * point takes its nearest point one level up as parent): parent m is
 * promoted iff the draw of its token at level 2 (the promotion rule above
 * with level 2 in the counter) is below promote_thresh, or, if none is, the
 * parent of smallest such draw (lowest m on ties); node2 lists them in
 * ascending m.  parent2[m] is the level-2 node nearest to parent m in the
 * lifted space, argmax_i (p_m . p_i + e_m e_i) in fp32, exact ties to the
 * lowest i (a level-2 node is its own); children groups the parents by
 * parent2.  Needs np_cap <= 50000.
 */

/*
 * Stage a3 on CUDA cores (fp32 FMA) for either dtype.  Same contract and
 * results as ice_build_assign up to fp32 rounding order; ice_build_assign
 * uses it for ICE_FP32, and for ICE_BF16 it serves as an independent
 * cross-check of the tensor-core kernel.
 */
ice_status ice_build_assign_simt(const ice_params *p, const void *K, const ice_index *idx, void *ws,
                                 size_t ws_bytes, int32_t *err_dev, void *stream);

/*
 * Stage a4 + a5: pages ([B] section 三: the tokens under one parent share a
 * physical page; [A] 关键设计 2: a node larger than a page splits off a new
 * page; [B] section 二: S = 16).  For parents in ascending m, the parent's
 * tokens in ascending token order are cut into consecutive chunks of S, and
 * pages are numbered in that order.  Writes n_pages, page_parent, page_len,
 * page_next, page_tokens, token_page, token_slot, parent_first_page,
 * parent_last_page, parent_n_pages, and copies K/V rows into pool_k/pool_v
 * (pad slots zero).  ICE_ERR_CAPACITY in err_dev if the pages exceed
 * page_cap.
 */
ice_status ice_build_pack(const ice_params *p, const void *K, const void *V, const ice_index *idx,
                          void *ws, size_t ws_bytes, int32_t *err_dev, void *stream);

/*
 * Index build of a layer on another layer's node structure ([B] section 五:
 * "IceCache (reuse)", an inter-layer index reuse that shortens the build; the
 * article does not describe its mechanism).  Rule used here: the promoted
 * tokens, the token -> parent assignment and hence the pages of `prev` are
 * kept; this layer's K gives M^2 (step a1), the parent keys that the
 * selection scores against and their lifted coordinate; this layer's K and V
 * fill the pool (step a5).  The nearest-parent contraction (a3) and the
 * ranking into pages (a4) are skipped.  Results equal those of ice_build_index
 * on this layer's K, V with parent_tok and token_parent taken from prev.
 *  - prev: an index of the same shapes and capacities built over the same N
 *    tokens (ice_build_index or this call; no inserts since).  A unit of prev
 *    whose n_indexed is not N, or whose parent token is outside [0, N), sets
 *    ICE_ERR_INVALID_ARG in err_dev.
 *  - idx may be prev itself (its tables stay and keys, lift values and pool
 *    are overwritten) or share any page or token table array with prev: a
 *    shared array is not copied.  Otherwise prev is only read.
 *  - Workspace: ice_build_workspace_bytes.
 */
ice_status ice_build_index_reuse(const ice_params *p, const void *K, const void *V, const ice_index *prev,
                                 const ice_index *idx, void *ws, size_t ws_bytes, int32_t *err_dev, void *stream);

/* -------------------------------------------------- incremental insert -- */
/* Workspace bytes for ice_insert_tokens (zero-filled once before first use,
 * like a decode workspace). */
ice_status ice_insert_workspace_bytes(const ice_params *p, size_t *bytes);

/*
 * Step a11: appends one new token to every unit's index without a rebuild
 * ([B] section 三: a new token goes through the same random promotion and is
 * attached to the most similar parent one level up; [A] 关键设计 2: a node
 * that outgrows its page opens a new page).  k_new, v_new [B, Hkv, d]
 * (dtype).  The token's position is the unit's n_indexed (then n_indexed
 * grows by one); it is lifted with the build-time M^2 (extra coordinate
 * sqrt(max(0, M^2 - |k|^2))).  If its level-1 draw (the promotion rule of
 * ice_build_lift_promote at that position) is below promote_thresh, it
 * becomes a new parent with a page of its own.  Otherwise its parent is the
 * nearest one in lifted space (exact fp32 ties to the lowest m), and it
 * takes the next slot of that parent's last page, or a new page linked
 * after it (page_next) when that page already holds S tokens.  Existing
 * tokens never move.  Updates every index array and the pool.
 * ICE_ERR_CAPACITY in err_dev (and that unit left unchanged) if n_cap,
 * np_cap or page_cap would be exceeded.  ICE_ERR_UNSUPPORTED (nothing
 * launched) with n_levels = 3 or with sink / window pages.
 */
ice_status ice_insert_tokens(const ice_params *p, const ice_index *idx, const void *k_new, const void *v_new,
                             void *ws, size_t ws_bytes, int32_t *err_dev, void *stream);

/* ------------------------------------------------------- decode step ---- */
/* Workspace bytes for ice_select_pages / ice_sparse_attn_decode /
 * ice_decode_step at this budget and output capacity max_sel.  A decode
 * workspace must be zero-filled once before its first use: it holds one
 * completion counter per unit and kernel, and every call that completes
 * leaves those counters at zero again, so no call has to clear them.  Calls
 * that share a workspace must not overlap on the GPU. */
ice_status ice_decode_workspace_bytes(const ice_params *p, int32_t budget_tokens, int32_t max_sel,
                                      size_t *bytes);

/*
 * Steps a6-a8: page selection and the GQA union ([A] 关键设计 3: each query
 * head chooses its own top-k pages; the query heads of one GQA group share
 * the union of their choices; [B] section 六).
 * Q [B, Hq, d] (dtype); query head hq belongs to KV head hq / g.
 * The lifted query q' = [q, 0] gives |q' - p'|^2 = |q|^2 + M^2 - 2 q.p, so a
 * page scores s = q . (its parent's key), accumulated in fp32.  Each query
 * head takes the first k = ceil(budget_tokens / S) pages in the order
 * (-s, page id); sel_pages[u, 0..sel_count[u]) is the ascending union of the
 * g lists, sel_pages [U, max_sel] int32 (rest -1), sel_count [U] int32.
 * max_sel must be >= min(g * k, page_cap).
 */
/*
 * With n_levels = 3 the selection descends ([A] 关键设计 2: the query finds
 * the k nearest points of the top level, then searches among their
 * children): per query head, the first k level-2 nodes in (-q.p, i) order,
 * then their children (parents) in (-q.p, m) order, whose pages are taken in
 * page-id order until k pages; union and positional pages as above.  Needs
 * k <= 32.  ice_decode_step follows the same rule.
 */
ice_status ice_select_pages(const ice_params *p, const ice_index *idx, const void *Q, int32_t budget_tokens,
                            int32_t *sel_pages, int32_t *sel_count, int32_t max_sel, void *ws,
                            size_t ws_bytes, int32_t *err_dev, void *stream);

/*
 * Step a9: bulk gather ([A] 关键设计 4; [B] section 四): the selected,
 * non-contiguous pages are copied into one contiguous buffer.
 * kbuf, vbuf [U, max_sel, S, d] (dtype): slot u holds page sel_pages[u];
 * buf_len [U, max_sel] int32 its length (0 beyond sel_count).
 */
ice_status ice_gather_pages(const ice_params *p, const ice_index *idx, const int32_t *sel_pages,
                            const int32_t *sel_count, int32_t max_sel, void *kbuf, void *vbuf,
                            int32_t *buf_len, void *stream);

/*
 * Step a10: masked sparse attention ([A] 关键设计 1):
 *   a_ij = s_ij exp(q_i.k_j * scale) / sum_j' s_ij' exp(q_i.k_j' * scale),
 *   o_i  = sum_j a_ij v_j,
 * with s_ij = 1 on the first buf_len[u] slots of each of the sel_count
 * gathered pages of the query head's group and 0 elsewhere; scale is
 * 1/sqrt(d) in the formula (pass it explicitly).  Split over the pages with
 * a log-sum-exp merge; fp32 throughout.  O [B, Hq, d] float; a unit with no
 * selected page gives O = 0.
 */
/* A bounded wait of the attention kernel that gives up (ICE_ERR_TIMEOUT in
 * ice_decode_step's err_dev) leaves NaN in O of the query heads of that unit
 * here, since this call has no error word. */
ice_status ice_sparse_attn_decode(const ice_params *p, const void *Q, const void *kbuf, const void *vbuf,
                                  const int32_t *buf_len, const int32_t *sel_count, int32_t max_sel,
                                  float scale, float *O, void *ws, size_t ws_bytes, void *stream);

/*
 * Allocation-free variant of ice_sparse_attn_decode.  The paper has no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc, such as a plugin inside a serving runtime that owns every byte
 * of device memory through its own pool and forbids raw allocations, or a
 * decode loop that cannot afford the implicit device-wide synchronisation of
 * an allocation.  It takes no workspace: its scratch (one ticket word per
 * unit and the per-split partial results) lives in a device array of
 * ICE_NOALLOC_SCRATCH_BYTES bytes that the library defines statically, which
 * every GPU that loads the library holds until the process exits.
 *  - Same arguments (minus the workspace), layouts and results as
 *    ice_sparse_attn_decode.  The caller still owns Q, kbuf, vbuf, buf_len,
 *    sel_count and O.
 *  - A shape whose scratch exceeds ICE_NOALLOC_SCRATCH_BYTES is rejected
 *    with ICE_ERR_CAPACITY before anything is launched.  The scratch is
 *    r(4 U) + r(8 U n g) + r(512 U n g) bytes with U = B * Hkv units,
 *    g = Hq / Hkv, n = ceil(max_sel / 4) splits and r(x) = x rounded up to
 *    a multiple of 256: about U * n * g * 520 bytes (8 MiB holds, for
 *    instance, 256 units with g = 1 and max_sel = 24, or 128 units with
 *    g = 8 and max_sel = 32).
 *  - A bounded wait that gives up leaves NaN in O for that unit's query
 *    heads (there is no error word).
 *  - The first call on a device looks up the array's device address with
 *    that device current (cudaGetSymbolAddress) and caches it; make that
 *    first call before any stream capture.  The cached address belongs to
 *    the device's primary context: after cudaDeviceReset (or any reset of
 *    that context) the library must not be called again in the process.
 *  - It calls no cudaMalloc, cudaFree or allocating library routine.
 *  - Every call on a device shares the one array, which keeps the last
 *    call's contents; the ticket words are cleared on the stream at the start
 *    of each call.  Calls whose executions overlap on the GPU (different
 *    streams, or different host threads) race on the array: order them.
 */
#define ICE_NOALLOC_SCRATCH_BYTES (8u << 20)
ice_status ice_sparse_attn_decode_noalloc(const ice_params *p, const void *Q, const void *kbuf, const void *vbuf,
                                          const int32_t *buf_len, const int32_t *sel_count, int32_t max_sel,
                                          float scale, float *O, void *stream);

/*
 * The whole decode step a6-a10 (the kernels of ice_decode_plan): every
 * selected page is read once from the pool, written to kbuf/vbuf/buf_len
 * (the contiguous buffer of step a9) and attended (step a10) from the same
 * on-chip copy.  Same outputs as the three separate calls.
 * kbuf, vbuf and buf_len may all be NULL: the selected pages are then
 * gathered into on-chip shared memory only and attended from there, with no
 * contiguous copy in device memory (the pool is still read once); sel_pages,
 * sel_count and O are the same as with the buffer.  Mixing NULL and non-NULL
 * among the three is ICE_ERR_INVALID_ARG.
 */
ice_status ice_decode_step(const ice_params *p, const ice_index *idx, const void *Q, int32_t budget_tokens,
                           int32_t *sel_pages, int32_t *sel_count, int32_t max_sel, void *kbuf, void *vbuf,
                           int32_t *buf_len, float scale, float *O, void *ws, size_t ws_bytes,
                           int32_t *err_dev, void *stream);

/*
 * The kernels ice_decode_step runs for a shape, chosen from the sizes in *p,
 * the budget and max_sel (and the device's SM count):
 *   ICE_PLAN_CLUSTER_BF16  bf16, g <= 8, k <= 32, while every unit's 8-CTA
 *                          cluster fits one wave (U * 8 <= SMs): one kernel,
 *                          the unit's parent slices scored on CUDA cores in
 *                          its 8 CTAs, lists merged over distributed shared
 *                          memory, pages bulk-copied and attended;
 *   ICE_PLAN_CLUSTER       the same cluster kernel for fp32 (or k <= 64,
 *                          g <= 16);
 *   ICE_PLAN_SCORE_SELECT  bf16, g <= 8, k <= 32 with more units: the score
 *                          table of every unit on the tensor cores (TMA +
 *                          tcgen05 over all SMs), then attention CTAs that
 *                          select their unit's pages and attend over them
 *                          (warp-level MMAs on TMA-staged pages);
 *   ICE_PLAN_SCORE_TOPK    other bf16 shapes with g <= 16, k <= 32: the score
 *                          table, a per-unit top-k kernel, then the gather +
 *                          attention kernel;
 *   ICE_PLAN_SIMT          the rest: CUDA-core selection, then the gather +
 *                          attention kernel;
 *   ICE_PLAN_DESCENT       n_levels = 3: the descent kernel, then the gather +
 *                          attention kernel.
 * *attention_plan: the attention kernel of ice_sparse_attn_decode and of the
 * last three plans: ICE_PLAN_ATTN_MMA (bf16, g <= 16, at most 32 pages per
 * warp: warp-level tensor-core MMAs on TMA-staged pages) or
 * ICE_PLAN_ATTN_SIMT.  Either output may be NULL.
 */
#define ICE_PLAN_CLUSTER_BF16 1
#define ICE_PLAN_CLUSTER 2
#define ICE_PLAN_SCORE_SELECT 3
#define ICE_PLAN_SCORE_TOPK 4
#define ICE_PLAN_SIMT 5
#define ICE_PLAN_DESCENT 6
#define ICE_PLAN_ATTN_MMA 1
#define ICE_PLAN_ATTN_SIMT 2
ice_status ice_decode_plan(const ice_params *p, int32_t budget_tokens, int32_t max_sel, int32_t *step_plan,
                           int32_t *attention_plan);

/* ----------------------------------------------------- host page pool --- */
/*
 * Step a12: the page pool in pinned host memory, with the selected pages of
 * a decode step moved to the device in one bulk transfer ([A] 关键设计 4:
 * the non-contiguous selected pages are gathered into one contiguous host
 * buffer and moved in a single transfer instead of many small ones; [B]
 * section 四).  This is the one object the library allocates and owns.
 */
typedef struct ice_host_pool ice_host_pool;

/* Allocates two pinned, device-mapped pools of pool_bytes each (K and V,
 * laid out like ice_index.pool_k / pool_v: [U, page_cap, S, d]), a pinned
 * staging buffer of staging_bytes (see ice_host_pool_staging_bytes) and
 * n_threads host worker threads.  ICE_ERR_OOM if pinned memory runs out. */
ice_status ice_host_pool_create(size_t pool_bytes, size_t staging_bytes, int32_t n_threads, ice_host_pool **out);
/* Waits for the last staged transfer, joins the workers, frees everything. */
ice_status ice_host_pool_destroy(ice_host_pool *hp);
/* Device-visible and host pointers of the two pools (any may be NULL).  Put
 * the device pointers into ice_index.pool_k / pool_v to build into the host
 * pool and to let ice_decode_step / ice_gather_pages read pages straight
 * from host memory over the CPU-GPU link, with no host copy. */
ice_status ice_host_pool_pointers(const ice_host_pool *hp, void **pool_k_dev, void **pool_v_dev, void **pool_k_host,
                                  void **pool_v_host);
/* Staging bytes of one layer's transfer: kbuf | vbuf | buf_len for
 * [U, max_sel] slots (2 * U * max_sel * S * d * elem + 4 * U * max_sel). */
size_t ice_host_pool_staging_bytes(const ice_params *p, int32_t max_sel);
/*
 * Staged gather: host threads copy the selected pages of every unit from the
 * host pool into the staging buffer (slot u * max_sel + x holds page
 * sel_pages_host[u * max_sel + x] for x < sel_count_host[u]; buf_len 0
 * beyond), then ONE cudaMemcpyAsync on `stream` moves the whole staging
 * buffer to dst_dev, laid out as kbuf [U, max_sel, S, d] | vbuf (same) |
 * buf_len [U, max_sel] int32 — ready for ice_sparse_attn_decode.
 * sel_pages_host / sel_count_host are HOST copies of ice_select_pages'
 * outputs (the caller copies them back and synchronises); page_len_host is
 * a HOST copy of ice_index.page_len [U, page_cap].  Returns once the copy is
 * enqueued; the next call first waits for this transfer to have read the
 * staging buffer.  ICE_ERR_CAPACITY if the staging buffer or dst_bytes is
 * too small, ICE_ERR_INVALID_ARG on a page id outside [0, page_cap) or a
 * count outside [0, max_sel] (nothing is transferred then).
 */
ice_status ice_host_pool_gather_h2d(ice_host_pool *hp, const ice_params *p, const int32_t *sel_pages_host,
                                    const int32_t *sel_count_host, const int32_t *page_len_host, int32_t max_sel,
                                    void *dst_dev, size_t dst_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ICE_H_ */
