// The page selection of one unit (decode steps a7 and a8) by a group of
// warps of one CTA, from the unit's score table and group maxima.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 3: every attention head picks its own top-k
// pages and the query heads of a GQA group share the union of their picks.
// Order (-score, m) over parents, pages of a parent in page-id order, k pages
// per head, union as a bitmask, then the ascending page list.
//
// Any group maximum T0 that at least kc group maxima reach is a lower bound
// of the kc-th best score (each of those groups holds a score >= T0), so the
// best kc keys (score, -m) all lie in the groups whose maximum is >= T0: T0
// by a radix-4 search on the group maxima that stops once at most kc + 8
// groups reach it, then only those groups' scores are read (16 groups' loads
// in flight), the keys >= T0 are put in order (up to 32 of them by counting
// each key's rank, more by a sorting network; their page spans load
// meanwhile), and the pages of the best kc are ORed into the union bitmask.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ice {
namespace sel {

using namespace topk;

constexpr int kMaxKc = 32;  // best keys per query head: one per lane of a warp
constexpr int kCand = 256;  // candidate keys a warp collects (more: exact slow path)
constexpr int kGroup = 32;  // parents per group maximum
constexpr int kSlack = 8;   // groups allowed above kc at the threshold T0
constexpr int kPrefetchPages = 3;  // first pages of each head prefetched into L2 (decode step)

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }


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

// The ordered best kc (<= 32) keys of all Np scores of one head, exactly, by
// kc rounds of a warp-wide maximum below the previous round's (slow; used
// only when very many scores tie with the group-maximum bound).
static __device__ unsigned long long best_slow(const float *__restrict__ sh, int Np, int kc) {
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

// Selection of unit u by the select group (NSW warps, thread tid of the
// group): warp hh < g takes query head hh, finds its ordered best kc parents
// and ORs their pages (k per head) into the union bitmask; then the group
// writes the ascending page list: to sel_pages / sel_count when write_global,
// and to s_list (shared) when given.  Returns the list's length (all threads).
// Synchronises the group on barrier 2.
// Parent ids stay below 2^24 (checked by the launcher), so the low key bits
// can carry a candidate's slot while the order is unchanged.
template <int NSW>
__device__ int select_unit(const SelArgs &A, int u, int tid, unsigned *s_mask, unsigned long long *s_cand,
                           int *s_wsum, int *s_list = nullptr, bool write_global = true) {
    constexpr int nt = 32 * NSW;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = A.g, np_cap = A.np_cap, kc = A.kc, k_pages = A.k_pages, max_sel = A.max_sel;
    const int Np = min(A.n_parents[u], np_cap);
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * A.page_cap;
    const int P = min(A.n_pages[u], A.page_cap);
    const int Ps = max(0, P - A.n_pos);  // semantic pages; the rest are positional (always in the union)
    const int words = (P + 31) / 32;
    const int ngc = (np_cap + kGroup - 1) / kGroup, ng = (Np + kGroup - 1) / kGroup;
    for (int x = tid; x < words; x += nt) s_mask[x] = 0u;
    named_bar(2, nt);
    if (k_pages >= Ps) {
        for (int x = tid; x < words; x += nt) {
            const int rem = P - x * 32;
            s_mask[x] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
        }
    } else {
        for (int x = Ps + tid; x < P; x += nt) atomicOr(&s_mask[x >> 5], 1u << (x & 31));
    }
    if (k_pages < Ps && warp < g) {
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
                t0 = unord_f32(kth_bound_ord(v, kc, kSlack));
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
            // the qualifying groups of this stretch, in order: the ballots
            // first, then their slots
            unsigned bl[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) bl[i] = __ballot_sync(0xffffffffu, gm[i] >= t0);
            int ngl = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int at = ngl + __popc(bl[i] & lanemask_lt());
                if (((bl[i] >> lane) & 1u) && at < 128) glist[at] = x0 + i * 32 + lane;
                ngl += __popc(bl[i]);
            }
            __syncwarp();
            if (ngl > 128) {  // very many ties with T0: exact slow path below
                cnt = kCand + 1;
                break;
            }
            for (int j0 = 0; j0 < ngl; j0 += 16) {  // 16 groups' loads in flight at once
                float sv[16];
                unsigned pass = 0u;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = j0 + i < ngl ? glist[j0 + i] * kGroup + lane : Np;
                    sv[i] = m < Np ? __ldcg(sh + m) : -INFINITY;
                    pass |= (m < Np ? 1u : 0u) << i;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) pass &= ~((sv[i] >= t0 ? 0u : 1u) << i);
                // this lane's keys >= T0 go to consecutive slots after the
                // lower lanes' (one warp scan of the counts)
                const int c = __popc(pass);
                int incl = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                int at = cnt + incl - c;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if ((pass >> i) & 1u) {
                        if (at < kCand - 64) cand[at] = sort_key(sv[i], glist[j0 + i] * kGroup + lane);
                        ++at;
                    }
                cnt += __shfl_sync(0xffffffffu, incl, 31);
            }
            __syncwarp();
        }
        __syncwarp();
        // lane r < kc: the r-th best parent and its pages
        int pm = -1, fp = 0, pc = 0, contig = 1;
        if (cnt <= 32) {
            // lane i holds candidate i; its rank is the number of larger keys
            // (keys are distinct); the candidates' page spans load meanwhile
            const unsigned long long key = lane < cnt ? cand[lane] : 0ull;
            int4 sp = make_int4(0, 0, 0, 0);
            if (key != 0ull) {
                const int m = key_id(key);
                sp = make_int4(A.parent_first_page[up + m], A.parent_n_pages[up + m], A.parent_last_page[up + m], m);
            }
            int rank = 0;
            for (int j = 0; j < cnt; ++j) rank += cand[j] > key ? 1 : 0;
            int *s_src = glist;  // the group list is spent: lane of the r-th best key
            __syncwarp();
            if (key != 0ull) s_src[rank] = lane;
            __syncwarp();
            const int src = lane < cnt ? s_src[lane] : 0;
            const int4 s = make_int4(__shfl_sync(0xffffffffu, sp.x, src), __shfl_sync(0xffffffffu, sp.y, src),
                                     __shfl_sync(0xffffffffu, sp.z, src), __shfl_sync(0xffffffffu, sp.w, src));
            if (lane < cnt && lane < kc) {
                pm = s.w;
                fp = s.x;
                pc = s.y;
                contig = s.z - s.x + 1 == s.y;
            }
        } else if (cnt <= 64) {
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
        // the head's first pages into L2 while the union and the list are
        // formed: the stream of the decode step starts from there
        if (A.pf_k != nullptr && pm >= 0 && contig && incl - pc < kPrefetchPages && tk > 0 && fp >= 0 &&
            fp + tk <= Ps) {
            const int npf = min(tk, kPrefetchPages - (incl - pc));
            const size_t off = ((size_t)u * A.page_cap + fp) * (size_t)A.page_bytes;
            const unsigned sz = (unsigned)(npf * A.page_bytes);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(A.pf_k + off), "r"(sz) : "memory");
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(A.pf_v + off), "r"(sz) : "memory");
        }
        int pg = fp;
        for (int i = 0; i < tk; ++i) {
            const int qq = contig ? fp + i : pg;
            if (qq < 0 || qq >= Ps) break;
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
            if (write_global) A.sel_pages[(size_t)u * max_sel + pos] = x * 32 + bit;
            if (s_list) s_list[pos] = x * 32 + bit;
            ++pos;
        }
    }
    if (write_global) {
        for (int x = total + tid; x < max_sel; x += nt) A.sel_pages[(size_t)u * max_sel + x] = -1;
        if (tid == 0) {
            if (total > max_sel) set_err(A.err, ICE_ERR_CAPACITY);
            A.sel_count[u] = min(total, max_sel);
        }
    }
    return min(total, max_sel);
}

}  // namespace sel
}  // namespace ice
