// Decode steps a6 (score the parent level), a7 (top-k pages per query head)
// and a8 (GQA union) with the scoring on the sm_103a tensor cores.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 3: every attention head picks its own top-k
// pages and the query heads of a GQA group share the union of their picks.
// IceCache popular-science article (aitangshan.cn/news/751385), section 六:
// with the query lifted by a zero coordinate, the nearest lifted parents are
// the parents of largest q.p.  The scores of a unit's g query heads against
// its parent table are the contraction P Q^T (parents x d times d x g), here
// tcgen05.mma with M = 128 parents, N = 16 query rows, K = d = 128, bf16 in,
// fp32 accumulate.  Same selection rule as the SIMT kernel k_select: order
// (-score, m) over parents, pages of a parent in page-id order, k pages per
// head, union as a bitmask.  Used for bf16 tables with g <= 16 query heads
// per KV head and k <= 32 pages per head.
//
// k_score_tc: persistent, one CTA per SM (6 warps), over work items (unit,
// 128-parent tile) in unit-major order, CTA c taking the item range
// [c I / G, (c + 1) I / G):
//   warp 0     TMA producer: at the start of a unit's run the unit's 16 query
//              rows (128-byte swizzle), then the parent tiles (128 x 128
//              bf16) through a 4-stage ring;
//   warp 1     allocates 32 TMEM columns and issues the MMAs (8 K-steps per
//              tile) into one of two 16-column accumulators;
//   warps 2-5  lane = parent: 16 fp32 scores from TMEM; the unit's g are
//              written to the score table [unit][head][parent] (coalesced)
//              and the maximum of each 32-parent group to [unit][head][group].
//   The kernel streams the parent table once; its extra traffic is the score
//   table (g x 4 bytes per 256-byte parent row).
// k_select_topk: one CTA per unit, one warp per query head.  The kc-th
//   largest group maximum T0 is a lower bound of the kc-th best score (kc
//   groups reach it), so the best kc keys (score, -m) all lie in the groups
//   whose maximum is >= T0 (about kc of them): T0 by bisection on the group
//   maxima, then only those groups' scores are read, the keys >= T0 sorted
//   into the ordered best kc (their page spans load during the sort), whose
//   pages (k per head) are ORed into the union bitmask; the block writes the
//   ascending page list.  The kernel is a short chain of dependent loads; it
//   runs after the streaming kernel so that the chain sees an idle memory
//   system (inside the streaming kernel each load waited ~2.5 us).
// Every mbarrier wait gives up after ~2 s and records ICE_ERR_TIMEOUT; the
// roles drain what they issued and TMEM is freed before the CTA returns.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "topk_common.cuh"

namespace ice {
namespace {

using namespace tc;
using namespace topk;

constexpr int BM = 128;    // parents per tile (TMEM lanes)
constexpr int BQ = 16;     // query rows per MMA (N)
constexpr int NS = 4;      // parent-tile ring depth
constexpr int kEpiWarps = 4;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kMaxKc = 32;  // best keys per query head: one per lane of a warp
constexpr int kCand = 256;   // candidate keys a top-k warp collects (more: exact slow path)
constexpr int kGroup = 32;   // parents per group maximum
constexpr uint32_t A_HALF = BM * 128;  // 128 rows x 64 bf16 columns
constexpr uint32_t A_BYTES = 2 * A_HALF;
constexpr uint32_t Q_HALF = BQ * 128;
constexpr uint32_t Q_BYTES = 2 * Q_HALF;
constexpr uint32_t TMEM_COLS = 32;
constexpr uint32_t IDESC = idesc_bf16(BM, BQ);

struct Bars {
    unsigned long long full[NS], empty[NS], qfull[2], qempty[2], tfull[2], tempty[2];
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = 1024 + (size_t)NS * A_BYTES + 2 * Q_BYTES + sizeof(Bars);

// Descending bitonic sort of the warp's 32 E values (E a power of two):
// value i in lane i % 32 of register i / 32.  Strides below 32 pair lanes
// (shuffles), larger strides pair registers of one lane.
template <typename V, int E, int ES>
__device__ __forceinline__ void reg_pass(V (&v)[E], int size, int lane) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if ((e & ES) == 0 && (e | ES) < E) {
            const bool desc = ((e * 32 + lane) & size) == 0;
            const V a = v[e], b = v[e | ES];
            if (desc ? a < b : a > b) {
                v[e] = b;
                v[e | ES] = a;
            }
        }
    }
}
template <typename V, int E>
__device__ __forceinline__ void warp_sort_desc(V (&v)[E]) {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int size = 2; size <= 32 * E; size <<= 1) {
        if (size >= 256) reg_pass<V, E, 4>(v, size, lane);
        if (size >= 128) reg_pass<V, E, 2>(v, size, lane);
        if (size >= 64) reg_pass<V, E, 1>(v, size, lane);
#pragma unroll 1
        for (int stride = min(size >> 1, 16); stride > 0; stride >>= 1) {
            const bool lower = (lane & stride) == 0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const V o = __shfl_xor_sync(0xffffffffu, v[e], stride);
                const bool desc = ((e * 32 + lane) & size) == 0;
                v[e] = (lower == desc) ? (o > v[e] ? o : v[e]) : (o < v[e] ? o : v[e]);
            }
        }
    }
}

struct Seg {
    int u, t0, t1, tv, Np;
};
// The run of the item range starting at `it` (ending before `end`) in one unit.
__device__ __forceinline__ Seg seg_at(long long it, long long end, int T, int np_cap,
                                      const int32_t *__restrict__ n_parents) {
    Seg s;
    s.u = (int)(it / T);
    s.t0 = (int)(it - (long long)s.u * T);
    const long long se = min(end, (long long)(s.u + 1) * T);
    s.t1 = s.t0 + (int)(se - it);
    s.Np = min(n_parents[s.u], np_cap);
    s.tv = max(s.t0, min(s.t1, (s.Np + BM - 1) / BM));
    return s;
}

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Per lane: a[0..GT) values of GT heads; returns the maximum over the warp
// of head *head (set here): recursive halving, each step a lane keeps half of
// its heads and takes its partner's maxima for them (GT - 1 + 5 - log2 GT
// shuffles in all).
template <int GT>
__device__ __forceinline__ float warp_max_heads(float (&a)[GT], int &head) {
    const int lane = threadIdx.x & 31;
    head = 0;
    int o = 16;
#pragma unroll
    for (int n = GT; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? a[i] : a[i + n / 2];
            const float keep = up ? a[i + n / 2] : a[i];
            a[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
        head += up ? n / 2 : 0;
    }
    float v = a[0];
    for (; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// The ordered best kc (<= 32) keys of all Np scores of one head, exactly, by
// kc rounds of a warp-wide maximum below the previous round's (slow; used
// only when very many scores tie with the group-maximum bound).
__device__ unsigned long long best_slow(const float *__restrict__ sh, int Np, int kc) {
    const int lane = threadIdx.x & 31;
    unsigned long long last = ~0ull, mine = 0ull;
    for (int r = 0; r < kc; ++r) {
        unsigned long long best = 0ull;
        for (int m = lane; m < Np; m += 32) {
            const unsigned long long k = sort_key(sh[m], m);
            if (k < last && k > best) best = k;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, off));
        if (lane == r) mine = best;
        last = best;
    }
    return mine;
}

// What the selection of a unit reads and writes.
struct SelArgs {
    int g, np_cap, page_cap, k_pages, kc, max_sel;
    const int32_t *n_parents, *n_pages;
    const float *scores, *gmax;
    const int32_t *parent_first_page, *parent_last_page, *parent_n_pages, *page_next;
    int32_t *sel_pages, *sel_count, *err;
};

// The kc-th largest of the warp's values (8 per lane, order-preserving
// integer form, 0 = none), found bit by bit from the top: the largest c with
// at least kc values >= c.  Stops early once exactly kc values reach the
// prefix: the answer is then their minimum.
__device__ __forceinline__ uint32_t kth_largest_ord(const uint32_t (&v)[8], int kc) {
    uint32_t r = 0u;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t c = r | (1u << bit);
        unsigned cnt = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) cnt += v[e] >= c;
        const int n = (int)__reduce_add_sync(0xffffffffu, cnt);
        if (n >= kc) {
            r = c;
            if (n == kc) {
                uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
                for (int e = 0; e < 8; ++e) mn = v[e] >= c ? min(mn, v[e]) : mn;
                return __reduce_min_sync(0xffffffffu, mn);
            }
        }
    }
    return r;
}

// Selection of unit u by the select group (NSW warps, thread tid of the
// group): warp hh < g takes query head hh, finds its ordered best kc parents
// and ORs their pages (k per head) into the union bitmask; then the group
// writes the ascending page list.  Synchronises the group on barrier 2.
// Parent ids stay below 2^24 (checked by the launcher), so the low key bits
// can carry a candidate's slot while the order is unchanged.
template <int NSW>
__device__ void select_unit(const SelArgs &A, int u, int tid, unsigned *s_mask, unsigned long long *s_cand,
                            int *s_wsum) {
    constexpr int nt = 32 * NSW;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = A.g, np_cap = A.np_cap, kc = A.kc, k_pages = A.k_pages, max_sel = A.max_sel;
    const int Np = min(A.n_parents[u], np_cap);
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * A.page_cap;
    const int P = min(A.n_pages[u], A.page_cap);
    const int words = (P + 31) / 32;
    const int ngc = (np_cap + kGroup - 1) / kGroup, ng = (Np + kGroup - 1) / kGroup;
    for (int x = tid; x < words; x += nt) s_mask[x] = 0u;
    named_bar(2, nt);
    if (k_pages >= P) {
        for (int x = tid; x < words; x += nt) {
            const int rem = P - x * 32;
            s_mask[x] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
        }
    } else if (warp < g) {
        const int hh = warp;
        const float *sh = A.scores + ((size_t)u * g + hh) * np_cap;
        const float *gh = A.gmax + ((size_t)u * g + hh) * ngc;
        unsigned long long *cand = s_cand + (size_t)hh * kCand;
        int *glist = reinterpret_cast<int *>(cand + kCand - 64);  // qualifying groups (tail of the buffer)
        // T0: the kc-th largest group maximum (a lower bound of the kc-th best
        // score: kc groups reach it)
        uint32_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int x = e * 32 + lane;
            v[e] = x < ng ? ord_f32(__ldcg(gh + x)) : 0u;
        }
        float t0 = -INFINITY;
        if (ng >= kc) {
            if (ng <= 8 * 32) {
                t0 = unord_f32(kth_largest_ord(v, kc));
            } else {  // more groups: stretches of 256 with a running bound
                uint32_t res = 0u;
                for (int x0 = 0; x0 < ng; x0 += 8 * 32) {
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int x = x0 + e * 32 + lane;
                        w[e] = x < ng ? ord_f32(__ldcg(gh + x)) : 0u;
                    }
                    const uint32_t prev = res;
                    uint32_t r = 0u;
                    for (int bit = 31; bit >= 0; --bit) {
                        const uint32_t c = r | (1u << bit);
                        unsigned cnt = 0;
#pragma unroll
                        for (int e = 0; e < 8; ++e) cnt += w[e] >= c;
                        // the earlier stretches already hold kc keys >= prev
                        const int n = (int)__reduce_add_sync(0xffffffffu, cnt) + (c <= prev ? kc : 0);
                        if (n >= kc) r = c;
                    }
                    res = r;
                }
                t0 = unord_f32(res);
            }
        }
        // keys with score >= T0, read only from groups whose maximum reaches it
        int cnt = 0;
        for (int x0 = 0; x0 < ng; x0 += 8 * 32) {
            float gm[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int x = x0 + i * 32 + lane;
                if (x0 == 0)
                    gm[i] = x < ng ? unord_f32(v[i]) : -INFINITY;
                else
                    gm[i] = x < ng ? __ldcg(gh + x) : -INFINITY;
            }
            // the qualifying groups of this stretch, in order
            int ngl = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const unsigned b = __ballot_sync(0xffffffffu, gm[i] >= t0);
                if (((b >> lane) & 1u) && ngl + __popc(b & lanemask_lt()) < 128)
                    glist[ngl + __popc(b & lanemask_lt())] = x0 + i * 32 + lane;
                ngl += __popc(b);
            }
            __syncwarp();
            if (ngl > 128) {  // very many ties with T0: exact slow path below
                cnt = kCand + 1;
                break;
            }
            for (int j0 = 0; j0 < ngl; j0 += 16) {  // 16 groups' loads in flight at once
                float sv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = j0 + i < ngl ? glist[j0 + i] * kGroup + lane : Np;
                    sv[i] = m < Np ? __ldcg(sh + m) : -INFINITY;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = j0 + i < ngl ? glist[j0 + i] * kGroup + lane : Np;
                    const bool pass = m < Np && sv[i] >= t0;
                    const unsigned bal = __ballot_sync(0xffffffffu, pass);
                    const int at = cnt + __popc(bal & lanemask_lt());
                    if (pass && at < kCand - 64) cand[at] = sort_key(sv[i], m);
                    cnt += __popc(bal);
                }
            }
            __syncwarp();
        }
        __syncwarp();
        // lane r < kc: the r-th best parent and its pages
        int pm = -1, fp = 0, pc = 0, contig = 1;
        if (cnt <= 64) {
            // the candidates' page spans load while the keys sort; a key's low
            // byte holds its slot in the list
            unsigned long long w[2];
            int4 sp[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = e * 32 + lane;
                const unsigned long long k = i < cnt ? cand[i] : 0ull;
                sp[e] = make_int4(0, 0, 0, 0);
                if (k != 0ull) {
                    const int m = key_id(k);
                    sp[e] = make_int4(A.parent_first_page[up + m], A.parent_n_pages[up + m],
                                      A.parent_last_page[up + m], m);
                }
                w[e] = k == 0ull ? 0ull : ((k & 0xFFFFFFFF00000000ull) | ((k & 0xFFFFFFull) << 8) | (unsigned)i);
            }
            sort64_desc(w);
            __syncwarp();
            int4 *s_span = reinterpret_cast<int4 *>(cand);  // the list is in registers now
            s_span[lane] = sp[0];
            s_span[32 + lane] = sp[1];
            __syncwarp();
            if (lane < kc && w[0] != 0ull) {
                const int4 s = s_span[(int)(w[0] & 0xFFu)];
                pm = s.w;
                fp = s.x;
                pc = s.y;
                contig = s.z - s.x + 1 == s.y;
            }
        } else {
            unsigned long long best;
            if (cnt <= kCand - 64) {
                unsigned long long w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = e * 32 + lane < cnt ? cand[e * 32 + lane] : 0ull;
                warp_sort_desc<unsigned long long, 8>(w);
                best = w[0];
            } else {
                best = best_slow(sh, Np, kc);
            }
            if (lane < kc && best != 0ull) {
                pm = key_id(best);
                fp = A.parent_first_page[up + pm];
                pc = A.parent_n_pages[up + pm];
                contig = A.parent_last_page[up + pm] - fp + 1 == pc;
            }
        }
        // take pages of the ordered parents until k pages
        if (pm < 0) pc = 0;
        int incl = pc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const int tk = max(0, min(pc, k_pages - (incl - pc)));
        int pg = fp;
        for (int i = 0; i < tk; ++i) {
            const int qq = contig ? fp + i : pg;
            if (qq < 0 || qq >= P) break;
            atomicOr(&s_mask[qq >> 5], 1u << (qq & 31));
            if (!contig) pg = A.page_next[ug + qq];
        }
    }
    named_bar(2, nt);
    // ascending list of the union's pages: thread tid owns words
    // [tid * wpt, (tid + 1) * wpt); one block-wide scan of the counts
    const int wpt = (words + nt - 1) / nt;
    const int wb = tid * wpt, we = min(words, wb + wpt);
    int c = 0;
    for (int x = wb; x < we; ++x) c += __popc(s_mask[x]);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_wsum[warp] = incl;
    named_bar(2, nt);
    int pos = incl - c, total = 0;
#pragma unroll
    for (int w = 0; w < NSW; ++w) {
        const int sw = s_wsum[w];
        pos += w < warp ? sw : 0;
        total += sw;
    }
    for (int x = wb; x < we && pos < max_sel; ++x) {
        unsigned bb = s_mask[x];
        while (bb && pos < max_sel) {
            const int bit = __ffs(bb) - 1;
            bb &= bb - 1;
            A.sel_pages[(size_t)u * max_sel + pos++] = x * 32 + bit;
        }
    }
    for (int x = total + tid; x < max_sel; x += nt) A.sel_pages[(size_t)u * max_sel + x] = -1;
    if (tid == 0) {
        if (total > max_sel) set_err(A.err, ICE_ERR_CAPACITY);
        A.sel_count[u] = min(total, max_sel);
    }
}

template <int GT>
__global__ void __launch_bounds__(kThreads, 1)
    k_score_tc(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ, int U, int g,
               int n_q_heads, int n_kv_heads, int np_cap, int T, const int32_t *__restrict__ n_parents,
               float *__restrict__ scores, float *__restrict__ gmax, int32_t *__restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;               // parent-tile ring
    unsigned char *sQ = sA + NS * A_BYTES;  // two query tiles
    Bars *bars = reinterpret_cast<Bars *>(sQ + 2 * Q_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const long long I = (long long)U * T;
    const long long it_begin = (long long)blockIdx.x * I / G, it_end = (long long)(blockIdx.x + 1) * I / G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->qfull[b], 1);
            mbar_init(&bars->qempty[b], 1);
            mbar_init(&bars->tfull[b], 1);
            mbar_init(&bars->tempty[b], kEpiThreads);
        }
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(&bars->tmem_base, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = bars->tmem_base;
    bool ok = true;
    dep_trigger();  // the selection grid may be scheduled now; it waits for this one

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int gt = 0, sv = 0;
            for (long long it = it_begin; ok && it < it_end;) {
                const Seg S = seg_at(it, it_end, T, np_cap, n_parents);
                it += S.t1 - S.t0;
                if (S.tv <= S.t0) continue;
                const int qs = sv & 1;
                if (!mbar_wait(&bars->qempty[qs], ((sv >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                const int b = S.u / n_kv_heads, h = S.u % n_kv_heads;
                const int qrow = b * n_q_heads + h * g;
                mbar_expect_tx(&bars->qfull[qs], Q_BYTES);
                tma_load_2d(sQ + qs * Q_BYTES, &tmQ, &bars->qfull[qs], 0, qrow);
                tma_load_2d(sQ + qs * Q_BYTES + Q_HALF, &tmQ, &bars->qfull[qs], 64, qrow);
                ++sv;
                for (int t = S.t0; t < S.tv; ++t, ++gt) {
                    const int s = gt % NS;
                    if (!mbar_wait(&bars->empty[s], ((gt / NS) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    const int y = S.u * np_cap + t * BM;
                    mbar_expect_tx(&bars->full[s], A_BYTES);
                    tma_load_2d(sA + s * A_BYTES, &tmP, &bars->full[s], 0, y);
                    tma_load_2d(sA + s * A_BYTES + A_HALF, &tmP, &bars->full[s], 64, y);
                }
            }
            // drain: every issued copy has landed before the CTA may exit
            for (int g2 = (gt > NS ? gt - NS : 0); g2 < gt; ++g2) mbar_wait(&bars->full[g2 % NS], (g2 / NS) & 1);
            for (int q2 = (sv > 2 ? sv - 2 : 0); q2 < sv; ++q2) mbar_wait(&bars->qfull[q2 & 1], (q2 >> 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int gt = 0, sv = 0;
            for (long long it = it_begin; ok && it < it_end;) {
                const Seg S = seg_at(it, it_end, T, np_cap, n_parents);
                it += S.t1 - S.t0;
                if (S.tv <= S.t0) continue;
                const int qs = sv & 1;
                if (!mbar_wait(&bars->qfull[qs], (sv >> 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t q0 = su32(sQ + qs * Q_BYTES);
                for (int t = S.t0; t < S.tv; ++t, ++gt) {
                    const int s = gt % NS, b = gt & 1;
                    if (!mbar_wait(&bars->tempty[b], ((gt >> 1) & 1) ^ 1) ||
                        !mbar_wait(&bars->full[s], (gt / NS) & 1)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t a0 = su32(sA + s * A_BYTES);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (k & 3) * 32;  // 16 bf16 columns inside the swizzle atom
                        umma_bf16<IDESC>(tmem + b * BQ, sw128_desc(a0 + (k >> 2) * A_HALF + off),
                                         sw128_desc(q0 + (k >> 2) * Q_HALF + off), k > 0 ? 1u : 0u);
                    }
                    umma_commit(&bars->empty[s]);
                    umma_commit(&bars->tfull[b]);
                }
                if (!ok) break;
                umma_commit(&bars->qempty[qs]);  // the query tile is free once these MMAs finish
                ++sv;
            }
            // drain: the last accumulator is complete before TMEM is freed
            if (gt > 0) mbar_wait(&bars->tfull[(gt - 1) & 1], ((gt - 1) >> 1) & 1);
        }
    } else {
        // ------------------------------------------------------ score writers
        const int q = warp & 3;  // TMEM lane quarter of this warp
        int gt = 0;
        for (long long it = it_begin; it < it_end;) {
            const Seg S = seg_at(it, it_end, T, np_cap, n_parents);
            it += S.t1 - S.t0;
            float *su = scores + (size_t)S.u * g * np_cap;
            const int ngc = (np_cap + kGroup - 1) / kGroup;
            float *gu = gmax + (size_t)S.u * g * ngc;
            for (int t = S.t0; t < S.tv; ++t, ++gt) {
                const int b = gt & 1;
                if (ok) ok = mbar_wait(&bars->tfull[b], (gt >> 1) & 1);
                ok = __all_sync(0xffffffffu, ok);
                fence_after();
                float sc[BQ];
                if (ok) {
                    tmem_ld16_nowait(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BQ), sc);
                    tmem_wait_ld();
                }
                fence_before();
                mbar_arrive(&bars->tempty[b]);
                const int m = t * BM + q * 32 + lane;
                if (ok && t * BM + q * 32 < S.Np) {  // this warp's group holds parents
                    const bool in = m < S.Np;
                    float a[GT];
#pragma unroll
                    for (int hh = 0; hh < GT; ++hh) {
                        if (in && hh < g) __stcg(su + (size_t)hh * np_cap + m, sc[hh]);
                        a[hh] = in ? sc[hh] : -INFINITY;
                    }
                    int head;
                    const float mx = warp_max_heads<GT>(a, head);
                    // lanes holding head h: those whose top log2(GT) bits give h; the lowest writes
                    if ((lane & (32 / GT - 1)) == 0 && head < g)
                        __stcg(gu + (size_t)head * ngc + t * (BM / kGroup) + q, mx);
                }
            }
        }
    }
    if (!ok) set_err(err, ICE_ERR_TIMEOUT);
    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// One CTA per unit, NSW warps (warp hh < g takes query head hh).
template <int NSW>
__global__ void __launch_bounds__(32 * NSW) k_select_topk(const SelArgs A) {
    extern __shared__ unsigned long long s_cand[];  // [NSW][kCand], then the union bitmask
    __shared__ int s_wsum[NSW];
    dep_trigger();  // the attention grid may be scheduled now; it waits for this one
    dep_wait();     // the score table is complete
    select_unit<NSW>(A, blockIdx.x, threadIdx.x, reinterpret_cast<unsigned *>(s_cand + NSW * kCand), s_cand, s_wsum);
}

}  // namespace

static int gt_of(int g) { return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : g <= 8 ? 8 : 16; }
// Warps of the selection CTA: one per query head, at least 4 (the page-list
// scan wants >= 128 threads).
static int nsw_of(int g) { return gt_of(g) < 4 ? 4 : gt_of(g); }
// Shared memory of the selection CTA: candidate keys, then the union bitmask.
static size_t topk_smem(int g, int page_cap) {
    return (size_t)nsw_of(g) * kCand * 8 + sizeof(unsigned) * (size_t)((page_cap + 31) / 32);
}

bool select_tc_supported(const ice_params &p, int k_pages) {
    const int g = p.n_q_heads / p.n_kv_heads;
    return p.dtype == ICE_BF16 && g >= 1 && g <= BQ && k_pages >= 1 && k_pages <= kMaxKc && p.np_cap < (1 << 24) &&
           topk_smem(g, p.page_cap) <= 227 * 1024;
}

// Score-table floats per unit: the scores, then the group maxima.
size_t select_tc_scores(const ice_params &p) {
    return (size_t)(p.n_q_heads / p.n_kv_heads) * ((size_t)p.np_cap + (size_t)ceil_div(p.np_cap, kGroup));
}

// Returns cudaErrorNotSupported (nothing launched) when a tensor map cannot
// be made for these pointers; the caller then uses the SIMT kernel.
cudaError_t launch_select_tc(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                             int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    const int T = ceil_div(p.np_cap, BM);
    CUtensorMap tmP, tmQ;
    if (!make_map_bf16(&tmP, idx.parent_keys, (unsigned long long)U * p.np_cap, kHeadDim, 64, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bf16(&tmQ, Q, (unsigned long long)p.batch * p.n_q_heads, kHeadDim, 64, BQ,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    const int gt = gt_of(g);
    auto kern = gt == 1 ? k_score_tc<1> : gt == 2 ? k_score_tc<2> : gt == 4 ? k_score_tc<4> : gt == 8 ? k_score_tc<8>
                                                                                             : k_score_tc<16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    static int n_sm = 0;
    if (!n_sm) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (n_sm <= 0) n_sm = 1;
    }
    const long long items = (long long)U * T;
    const int grid = items < n_sm ? (int)items : n_sm;
    float *gmax = ws.scores + (size_t)U * g * p.np_cap;
    kern<<<grid, kThreads, kSmemBytes, s>>>(tmP, tmQ, U, g, p.n_q_heads, p.n_kv_heads, p.np_cap, T,
                                                  idx.n_parents, ws.scores, gmax, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    SelArgs A;
    A.g = g;
    A.np_cap = p.np_cap;
    A.page_cap = p.page_cap;
    A.k_pages = ws.k_pages;
    A.kc = ws.k_pages;
    A.max_sel = max_sel;
    A.n_parents = idx.n_parents;
    A.n_pages = idx.n_pages;
    A.scores = ws.scores;
    A.gmax = gmax;
    A.parent_first_page = idx.parent_first_page;
    A.parent_last_page = idx.parent_last_page;
    A.parent_n_pages = idx.parent_n_pages;
    A.page_next = idx.page_next;
    A.sel_pages = sel_pages;
    A.sel_count = sel_count;
    A.err = err;
    const int nsw = nsw_of(g);
    auto topk = nsw == 4 ? k_select_topk<4> : nsw == 8 ? k_select_topk<8> : k_select_topk<16>;
    const size_t smem = topk_smem(g, p.page_cap);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    e = launch_dependent(topk, dim3(U), dim3(32 * nsw), smem, s, A);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ice
