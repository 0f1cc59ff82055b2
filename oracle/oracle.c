/*
 * IceCache CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct restatement of what the IceCache hot path
 * computes, in IEEE double, one (sequence, layer, KV head) unit at a time.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference leg may load this library.  The product path (the CUDA library)
 * shares no code with it and never calls it.
 *
 * Sources (cited by page and section):
 *   [A] "IceCache: Memory-Efficient KV-cache Management for Long-Sequence
 *       LLMs", papernotes.org ICLR 2026 notes: "方法详解 / 整体框架" and
 *       "关键设计" items 1-4 (item 1 prints the sparse-attention formula).
 *   [B] IceCache popular-science article, aitangshan.cn/news/751385:
 *       section 二 (16-token pages), section 三 (key transform, random
 *       promotion pyramid, nearest parent, parent -> page, incremental insert),
 *       section 四 (bulk loading), section 六 (TK/TQ transform, GQA union).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - lift: k' = [k, sqrt(M^2 - |k|^2)], q' = [q, 0], M = max key norm of the
 *     unit's build set; unscaled.
 *   - promotion draw: splitmix64 (Steele, Lea & Flood 2014), see
 *     orc_promote_draw below.  Two levels: level-1 points are the page parents.
 *   - a promoted token's parent is itself; ties go to the lowest parent index.
 *   - pages: a parent's tokens in ascending token order, cut in chunks of S.
 *   - page score = q . (its parent's key); order (-score, page id); k = ceil(budget/S).
 *   - s_ij = 1 on every slot of the GQA group's union pages, 0 elsewhere.
 *   - insert: build-time M (extra coordinate clamped at 0), no re-parenting,
 *     append to the parent's last page or open a new one when it holds S.
 *
 * Parity-unpinned part: none of these functions reproduces the pages' own
 * approximate P-DCI search; selection here is the exact scan of the parent
 * level (the reading above).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_CAPACITY 4
#define ORC_ERR_NOMEM 3

/* ------------------------------------------------------------------------ */
/* splitmix64, from its published definition: the state advances by the    */
/* golden-ratio increment gamma, and each output is the state passed        */
/* through a fixed 64-bit finaliser (two xor-shift-multiply rounds and a    */
/* final xor-shift).                                                        */
/* ------------------------------------------------------------------------ */
static const uint64_t ORC_GAMMA = 0x9E3779B97F4A7C15ULL;

uint64_t orc_splitmix64_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* n-th output (n >= 1) of the splitmix64 stream whose state starts at s0. */
uint64_t orc_splitmix64_nth(uint64_t s0, uint64_t n)
{
    return orc_splitmix64_mix(s0 + n * ORC_GAMMA);
}

/*
 * Promotion draw for one token at one level ([B] section 三: every token
 * starts at the bottom level; a random subset is promoted one level up, and
 * a random subset of those again).
 *
 *   key = output (layer + 1) of the stream started at `seed`
 *   ctr = token | level << 32 | head << 40 | seq << 52
 *   u   = top 32 bits of output (ctr + 1) of the stream started at `key`
 *
 * token < 2^32, level < 2^8, head < 2^12, seq < 2^12.
 */
uint32_t orc_promote_draw(uint64_t seed, int32_t layer, int32_t seq, int32_t head,
                          int64_t token, int32_t level)
{
    uint64_t key = orc_splitmix64_nth(seed, (uint64_t)(int64_t)layer + 1u);
    uint64_t ctr = (uint64_t)token | ((uint64_t)level << 32) | ((uint64_t)head << 40) |
                   ((uint64_t)seq << 52);
    return (uint32_t)(orc_splitmix64_nth(key, ctr + 1u) >> 32);
}

/* ------------------------------------------------------------------------ */
/* Step a1: the key lift ([B] section 三 and 六; [A] 关键设计 2).            */
/*   n_j = |k_j|^2,  M^2 = max_j n_j,  e_j = sqrt(max(0, M^2 - n_j)).      */
/* so that every lifted key k'_j = [k_j, e_j] has norm M.                    */
/* ------------------------------------------------------------------------ */
int orc_lift(const double *K, int64_t N, int32_t d, double *n_out, double *M2_out, double *e_out)
{
    if (N < 0 || d <= 0) return ORC_ERR_ARG;
    double M2 = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        double s = 0.0;
        for (int32_t i = 0; i < d; ++i) s += K[j * d + i] * K[j * d + i];
        n_out[j] = s;
        if (s > M2) M2 = s;
    }
    for (int64_t j = 0; j < N; ++j) {
        double r = M2 - n_out[j];
        e_out[j] = sqrt(r > 0.0 ? r : 0.0);
    }
    *M2_out = M2;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Step a2: random promotion to level 1 ([B] section 三; [A] 关键设计 2).   */
/* Level-1 members in ascending token order are the parents m = 0..Np-1.    */
/* If no token is promoted (N > 0) the token with the smallest draw is       */
/* promoted (lowest token on equal draws), so that every unit has a parent. */
/* ------------------------------------------------------------------------ */
int orc_promote(uint64_t seed, int32_t layer, int32_t seq, int32_t head, int64_t N,
                uint64_t thresh, int32_t *parent_tok, int32_t *n_parents)
{
    if (N < 0 || thresh > (1ULL << 32)) return ORC_ERR_ARG;
    int32_t np = 0;
    for (int64_t j = 0; j < N; ++j) {
        uint32_t u = orc_promote_draw(seed, layer, seq, head, j, 1);
        if ((uint64_t)u < thresh) parent_tok[np++] = (int32_t)j;
    }
    if (np == 0 && N > 0) {
        int64_t best = 0;
        uint32_t bu = orc_promote_draw(seed, layer, seq, head, 0, 1);
        for (int64_t j = 1; j < N; ++j) {
            uint32_t u = orc_promote_draw(seed, layer, seq, head, j, 1);
            if (u < bu) { bu = u; best = j; }
        }
        parent_tok[np++] = (int32_t)best;
    }
    *n_parents = np;
    return ORC_OK;
}

/* Squared Euclidean distance between lifted points [a, ea] and [b, eb]. */
static double lifted_dist2(const double *a, double ea, const double *b, double eb, int32_t d)
{
    double s = 0.0;
    for (int32_t i = 0; i < d; ++i) {
        double t = a[i] - b[i];
        s += t * t;
    }
    double t = ea - eb;
    return s + t * t;
}

/* ------------------------------------------------------------------------ */
/* Step a3: nearest parent in lifted space ([B] section 三: each token takes */
/* as parent the most similar point of the level above; [A] 关键设计 2).     */
/* parent(j) = argmin_m |k'_j - p'_m|^2, ties -> lowest m; a promoted token  */
/* is its own parent.                                                        */
/* ------------------------------------------------------------------------ */
int orc_assign(const double *K, const double *e, int64_t N, int32_t d,
               const int32_t *parent_tok, int32_t Np, int32_t *token_parent)
{
    if (N < 0 || d <= 0 || Np < 0 || (N > 0 && Np == 0)) return ORC_ERR_ARG;
    for (int64_t j = 0; j < N; ++j) token_parent[j] = -1;
    for (int32_t m = 0; m < Np; ++m) {
        if (parent_tok[m] < 0 || parent_tok[m] >= N) return ORC_ERR_ARG;
        token_parent[parent_tok[m]] = m;
    }
    for (int64_t j = 0; j < N; ++j) {
        if (token_parent[j] >= 0) continue;
        int32_t best = -1;
        double bd = 0.0;
        for (int32_t m = 0; m < Np; ++m) {
            int64_t t = parent_tok[m];
            double D = lifted_dist2(K + j * d, e[j], K + t * d, e[t], d);
            if (best < 0 || D < bd) { bd = D; best = m; }
        }
        token_parent[j] = best;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Step a4: pack the tokens of each parent into pages of at most S tokens   */
/* ([B] section 三: a parent's tokens share a physical page; [A] 关键设计 2: */
/* a node larger than the page splits off a new page; [B] section 二: 16    */
/* tokens per page).  Parents in ascending m, tokens of a parent in         */
/* ascending order, consecutive chunks of S; pages numbered in that order.  */
/* Unused slots of page_tokens are -1.                                       */
/* ------------------------------------------------------------------------ */
int orc_pack(const int32_t *token_parent, int64_t N, int32_t Np, int32_t S, int32_t page_cap,
             int32_t *n_pages, int32_t *page_parent, int32_t *page_len, int32_t *page_tokens,
             int32_t *token_page, int32_t *token_slot)
{
    if (N < 0 || Np < 0 || S <= 0 || page_cap < 0) return ORC_ERR_ARG;
    /* buckets: the tokens of each parent, appended in ascending token order */
    int64_t *count = (int64_t *)calloc((size_t)Np + 1, sizeof(int64_t));
    int64_t *start = (int64_t *)calloc((size_t)Np + 1, sizeof(int64_t));
    int64_t *fill = (int64_t *)calloc((size_t)Np + 1, sizeof(int64_t));
    int32_t *members = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N > 0 ? N : 1));
    int rc = ORC_OK;
    if (!count || !start || !fill || !members) { rc = ORC_ERR_NOMEM; goto done; }
    for (int64_t j = 0; j < N; ++j) {
        int32_t m = token_parent[j];
        if (m < 0 || m >= Np) { rc = ORC_ERR_ARG; goto done; }
        count[m]++;
    }
    for (int32_t m = 1; m <= Np; ++m) start[m] = start[m - 1] + count[m - 1];
    for (int64_t j = 0; j < N; ++j) {
        int32_t m = token_parent[j];
        members[start[m] + fill[m]++] = (int32_t)j;
    }
    int32_t P = 0;
    for (int32_t m = 0; m < Np; ++m) {
        for (int64_t r = 0; r < count[m]; r += S) {
            if (P >= page_cap) { rc = ORC_ERR_CAPACITY; goto done; }
            int32_t len = (int32_t)((count[m] - r) < S ? (count[m] - r) : S);
            page_parent[P] = m;
            page_len[P] = len;
            for (int32_t s = 0; s < S; ++s) {
                if (s < len) {
                    int32_t j = members[start[m] + r + s];
                    page_tokens[(int64_t)P * S + s] = j;
                    token_page[j] = P;
                    token_slot[j] = s;
                } else {
                    page_tokens[(int64_t)P * S + s] = -1;
                }
            }
            ++P;
        }
    }
    *n_pages = P;
done:
    free(count);
    free(start);
    free(fill);
    free(members);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Step a5: the page pool holds each page's K and V rows in slot order;     */
/* unused slots are zero ([A] 方法详解: each node maps to one physical page). */
/* ------------------------------------------------------------------------ */
int orc_scatter(const double *K, const double *V, int64_t N, int32_t d, int32_t S,
                int32_t n_pages, const int32_t *page_tokens, double *pool_k, double *pool_v)
{
    if (N < 0 || d <= 0 || S <= 0 || n_pages < 0) return ORC_ERR_ARG;
    for (int64_t p = 0; p < n_pages; ++p) {
        for (int32_t s = 0; s < S; ++s) {
            int32_t j = page_tokens[p * S + s];
            double *dk = pool_k + (p * S + s) * d;
            double *dv = pool_v + (p * S + s) * d;
            if (j >= 0 && j >= N) return ORC_ERR_ARG;
            for (int32_t i = 0; i < d; ++i) {
                dk[i] = j >= 0 ? K[(int64_t)j * d + i] : 0.0;
                dv[i] = j >= 0 ? V[(int64_t)j * d + i] : 0.0;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Steps a6-a8: page selection per query head and the GQA union.            */
/* [A] 关键设计 3: each query head picks its own top-k pages; the heads of a */
/* GQA group share the union of their picks ([B] section 六).  The lifted   */
/* query q' = [q, 0] makes |q' - p'|^2 = |q|^2 + M^2 - 2 q.p, so ranking by */
/* smallest lifted distance is ranking by largest q.p; a page scores its   */
/* parent's q.p.  Order: (-score, page id).  k = min(k_pages, n_pages).     */
/* ------------------------------------------------------------------------ */
typedef struct { double s; int32_t id; } orc_scored;

static int cmp_scored(const void *a, const void *b)
{
    const orc_scored *x = (const orc_scored *)a, *y = (const orc_scored *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->id > y->id) - (x->id < y->id);
}

int orc_select(const double *q, int32_t g, int32_t d, const double *parent_keys, int32_t Np,
               const int32_t *page_parent, int32_t n_pages, int32_t k_pages,
               int32_t *head_pages /* [g, k_pages] (-1 pad) */,
               int32_t *sel_pages /* [g * k_pages] */, int32_t *sel_count)
{
    if (g <= 0 || d <= 0 || Np < 0 || n_pages < 0 || k_pages < 0) return ORC_ERR_ARG;
    double *score = (double *)malloc(sizeof(double) * (size_t)(Np > 0 ? Np : 1));
    orc_scored *order = (orc_scored *)malloc(sizeof(orc_scored) * (size_t)(n_pages > 0 ? n_pages : 1));
    unsigned char *in_union = (unsigned char *)calloc((size_t)(n_pages > 0 ? n_pages : 1), 1);
    int rc = ORC_OK;
    if (!score || !order || !in_union) { rc = ORC_ERR_NOMEM; goto done; }
    int32_t k = k_pages < n_pages ? k_pages : n_pages;
    for (int32_t h = 0; h < g; ++h) {
        for (int32_t m = 0; m < Np; ++m) {
            double s = 0.0;
            for (int32_t i = 0; i < d; ++i) s += q[(int64_t)h * d + i] * parent_keys[(int64_t)m * d + i];
            score[m] = s;
        }
        for (int32_t p = 0; p < n_pages; ++p) {
            if (page_parent[p] < 0 || page_parent[p] >= Np) { rc = ORC_ERR_ARG; goto done; }
            order[p].s = score[page_parent[p]];
            order[p].id = p;
        }
        qsort(order, (size_t)n_pages, sizeof(orc_scored), cmp_scored);
        for (int32_t r = 0; r < k_pages; ++r) {
            head_pages[(int64_t)h * k_pages + r] = r < k ? order[r].id : -1;
            if (r < k) in_union[order[r].id] = 1;
        }
    }
    {
        int32_t c = 0;
        for (int32_t p = 0; p < n_pages; ++p)
            if (in_union[p]) sel_pages[c++] = p;
        for (int32_t r = c; r < g * k_pages; ++r) sel_pages[r] = -1;
        *sel_count = c;
    }
done:
    free(score);
    free(order);
    free(in_union);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Step a9: bulk gather of the selected pages into one contiguous buffer    */
/* ([A] 关键设计 4; [B] section 四).  Slot u of the buffer holds page         */
/* sel_pages[u]; buf_len[u] its length.                                      */
/* ------------------------------------------------------------------------ */
int orc_gather(const double *pool_k, const double *pool_v, const int32_t *page_len, int32_t n_pages,
               int32_t S, int32_t d, const int32_t *sel_pages, int32_t sel_count,
               double *kbuf, double *vbuf, int32_t *buf_len)
{
    if (S <= 0 || d <= 0 || sel_count < 0) return ORC_ERR_ARG;
    int64_t row = (int64_t)S * d;
    for (int32_t u = 0; u < sel_count; ++u) {
        int32_t p = sel_pages[u];
        if (p < 0 || p >= n_pages) return ORC_ERR_ARG;
        memcpy(kbuf + u * row, pool_k + (int64_t)p * row, sizeof(double) * (size_t)row);
        memcpy(vbuf + u * row, pool_v + (int64_t)p * row, sizeof(double) * (size_t)row);
        buf_len[u] = page_len[p];
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Step a10: masked sparse attention ([A] 关键设计 1 formula):               */
/*   a_ij = s_ij exp(q_i.k_j * scale) / sum_j' s_ij' exp(q_i.k_j' * scale)  */
/*   o_i  = sum_j a_ij v_j,  scale = 1/sqrt(d) in the formula.               */
/* s_ij = 1 on the first buf_len[u] slots of every gathered page u.         */
/* The maximum logit is subtracted before exp (the ratio is unchanged).     */
/* ------------------------------------------------------------------------ */
int orc_attention(const double *q, int32_t g, int32_t d, const double *kbuf, const double *vbuf,
                  const int32_t *buf_len, int32_t count, int32_t S, double scale, double *out)
{
    if (g <= 0 || d <= 0 || S <= 0 || count < 0) return ORC_ERR_ARG;
    int64_t n = (int64_t)count * S;
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!logit) return ORC_ERR_NOMEM;
    for (int32_t h = 0; h < g; ++h) {
        const double *qh = q + (int64_t)h * d;
        double mx = -INFINITY;
        for (int32_t u = 0; u < count; ++u) {
            for (int32_t s = 0; s < S; ++s) {
                int64_t t = (int64_t)u * S + s;
                if (s >= buf_len[u]) { logit[t] = -INFINITY; continue; }
                double dot = 0.0;
                for (int32_t i = 0; i < d; ++i) dot += qh[i] * kbuf[t * d + i];
                logit[t] = dot * scale;
                if (logit[t] > mx) mx = logit[t];
            }
        }
        double den = 0.0;
        for (int64_t t = 0; t < n; ++t)
            if (logit[t] > -INFINITY) den += exp(logit[t] - mx);
        for (int32_t i = 0; i < d; ++i) out[(int64_t)h * d + i] = 0.0;
        if (den > 0.0) {
            for (int64_t t = 0; t < n; ++t) {
                if (!(logit[t] > -INFINITY)) continue;
                double w = exp(logit[t] - mx) / den;
                for (int32_t i = 0; i < d; ++i) out[(int64_t)h * d + i] += w * vbuf[t * d + i];
            }
        }
    }
    free(logit);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Step a11: incremental insert of one new token at position `pos`          */
/* ([B] section 三: a new token goes through the same random promotion and  */
/* attaches to its most similar parent without a rebuild; [A] 关键设计 2: a  */
/* node that outgrows its page opens a new page).                            */
/*                                                                          */
/* The unit's index state is passed as arrays with capacities.  The lift    */
/* keeps the build-time M^2: e_new = sqrt(max(0, M^2 - |k_new|^2)).         */
/* Promoted (draw at level 1 below thresh): new parent m = Np with its own  */
/* new page.  Otherwise parent = argmin_m |k'_new - p'_m|^2 (ties lowest m); */
/* the token goes to that parent's highest-numbered page if it holds fewer  */
/* than S tokens, else to a new page.  Existing tokens never move.          */
/* parent_key_e holds each parent's lifted extra coordinate.                */
/* ------------------------------------------------------------------------ */
int orc_insert(uint64_t seed, int32_t layer, int32_t seq, int32_t head, uint64_t thresh,
               int32_t d, int32_t S, double M2, const double *k_new, const double *v_new,
               int64_t pos, int32_t forced_parent,
               /* parent level */
               int32_t np_cap, int32_t *n_parents, int32_t *parent_tok, double *parent_keys,
               double *parent_key_e,
               /* pages */
               int32_t page_cap, int32_t *n_pages, int32_t *page_parent, int32_t *page_len,
               int32_t *page_tokens, double *pool_k, double *pool_v,
               /* token tables (indexed by position) */
               int64_t n_cap, int32_t *token_parent, int32_t *token_page, int32_t *token_slot)
{
    if (d <= 0 || S <= 0 || pos < 0 || pos >= n_cap) return ORC_ERR_ARG;
    double n = 0.0;
    for (int32_t i = 0; i < d; ++i) n += k_new[i] * k_new[i];
    double r = M2 - n;
    double e = sqrt(r > 0.0 ? r : 0.0);
    int32_t Np = *n_parents, P = *n_pages;
    uint32_t u = orc_promote_draw(seed, layer, seq, head, pos, 1);
    int32_t m;
    int32_t page = -1;
    if ((uint64_t)u < thresh || Np == 0) {
        if (Np >= np_cap) return ORC_ERR_CAPACITY;
        m = Np;
        parent_tok[m] = (int32_t)pos;
        for (int32_t i = 0; i < d; ++i) parent_keys[(int64_t)m * d + i] = k_new[i];
        parent_key_e[m] = e;
        *n_parents = Np + 1;
    } else {
        if (forced_parent >= 0) {
            /* the caller's parent: tests that follow a device's choice at a
             * checked fp32 near-tie of the lifted distance */
            if (forced_parent >= Np) return ORC_ERR_ARG;
            m = forced_parent;
        } else {
            m = -1;
            double bd = 0.0;
            for (int32_t c = 0; c < Np; ++c) {
                double D = lifted_dist2(k_new, e, parent_keys + (int64_t)c * d, parent_key_e[c], d);
                if (m < 0 || D < bd) { bd = D; m = c; }
            }
        }
        for (int32_t p = P - 1; p >= 0; --p)
            if (page_parent[p] == m) { page = p; break; }
        if (page >= 0 && page_len[page] >= S) page = -1;
    }
    if (page < 0) {
        if (P >= page_cap) return ORC_ERR_CAPACITY;
        page = P;
        page_parent[page] = m;
        page_len[page] = 0;
        for (int32_t s = 0; s < S; ++s) {
            page_tokens[(int64_t)page * S + s] = -1;
            for (int32_t i = 0; i < d; ++i) {
                pool_k[((int64_t)page * S + s) * d + i] = 0.0;
                pool_v[((int64_t)page * S + s) * d + i] = 0.0;
            }
        }
        *n_pages = P + 1;
    }
    int32_t slot = page_len[page];
    page_tokens[(int64_t)page * S + slot] = (int32_t)pos;
    for (int32_t i = 0; i < d; ++i) {
        pool_k[((int64_t)page * S + slot) * d + i] = k_new[i];
        pool_v[((int64_t)page * S + slot) * d + i] = v_new[i];
    }
    page_len[page] = slot + 1;
    token_parent[pos] = m;
    token_page[pos] = page;
    token_slot[pos] = slot;
    return ORC_OK;
}
