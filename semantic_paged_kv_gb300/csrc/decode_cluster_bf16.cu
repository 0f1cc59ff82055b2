// The whole decode step (a6-a10) of a unit in one thread-block cluster, for
// bf16 tables with at most 8 query heads per KV head and k <= 32 pages per
// head.  Same computation as the selection followed by the fused attention
// (papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 1 (sparse attention), 3 (per-head top-k
// pages, GQA union), 4 (bulk gather into a contiguous buffer); IceCache
// popular-science article (aitangshan.cn/news/751385), sections 四 and 六);
// the phases exchange data through distributed shared memory under hardware
// cluster barriers:
//
//   phase 1  CTA r scores its slice of the parent table: 16 lanes per parent
//            row (one 16-byte load each), the lane's q slices of the GT heads
//            in registers (packed fp32-pair FMAs), the 16 partial sums folded
//            by recursive halving.  Per head (one warp each) the slice's best
//            kc keys (score, -m): a bound T on the scores that the best kc
//            reach and at most 64 keys reach (a radix search on their
//            order-preserving integer form that stops as soon as the count is
//            that small), the keys with score >= T collected and sorted by a
//            bitonic network; the page
//            spans of the slice's parents stay in shared memory.
//                                                            -- cluster barrier
//   phase 2  the leader merges the 8 sorted lists of each head pairwise
//            (bitonic merges), takes pages of the ordered parents until k
//            (spans read from the owning CTA), ORs them into a bitmask and
//            writes the ascending union.                    -- cluster barrier
//   phase 3  CTA r bulk-copies its share of the union's pages into shared
//            memory (one mbarrier per page), writes them back to kbuf / vbuf
//            with bulk stores, and attends over them, a page per warp at a
//            time (online softmax per warp), then merges its warps.
//                                                            -- cluster barrier
//   phase 4  CTA r merges head r of all CTAs (log-sum-exp, DSMEM) and writes
//            O.                                              -- barrier, exit
// No CTA waits on a flag; the mbarrier waits are bounded (ICE_ERR_TIMEOUT).
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "topk_common.cuh"

namespace ice {
namespace {

namespace cg = cooperative_groups;
using namespace tc;
using namespace topk;

constexpr int kC = kDecodeCluster;  // CTAs per cluster = per unit
constexpr int kT = 256;
constexpr int kW = kT / 32;
constexpr int kPageElems = kPage * kHeadDim;
constexpr uint32_t kPageBytes = kPageElems * 2;
constexpr int kCand = 64;    // keys a selection warp collects
constexpr int kMaxPPC = 16;  // pages of the union per CTA
constexpr int kSpanPT = 2;   // parent spans per thread loaded with the parent rows


// Shared-memory layout (byte offsets, 128-byte aligned pieces).
struct Lay {
    size_t sc, span, top, cand, mask, uni, kv, p, pp, ml, alpha, pm, pl, po, bars, total;
};
__host__ __device__ inline Lay layout(int gt, int chunk, int page_cap, int max_sel, int ppc) {
    auto al = [](size_t x) { return (x + 127) & ~(size_t)127; };
    Lay L{};
    size_t o = 0;
    L.kv = o;    o += al(ppc * 2 * (size_t)kPageBytes > (size_t)kW * gt * kHeadDim * 4 ? ppc * 2 * (size_t)kPageBytes
                                                                                    : (size_t)kW * gt * kHeadDim * 4);
    L.sc = o;    o += al(sizeof(float) * gt * chunk);
    L.span = o;  o += al(sizeof(int4) * chunk);
    L.top = o;   o += al(sizeof(unsigned long long) * gt * 32);
    L.cand = o;  o += al(sizeof(unsigned long long) * kW * kCand);
    L.mask = o;  o += al(sizeof(unsigned) * ((page_cap + 31) / 32));
    L.uni = o;   o += al(sizeof(int) * (max_sel + 1));
    L.p = o;     o += al(sizeof(float) * kW * kPage * gt);
    L.pp = o;    o += al(sizeof(unsigned long long) * kW * kPage * gt);
    L.ml = o;    o += al(sizeof(float) * kW * gt * 2);
    L.alpha = o; o += al(sizeof(float) * kW * gt);
    L.pm = o;    o += al(sizeof(float) * gt);
    L.pl = o;    o += al(sizeof(float) * gt);
    L.po = o;    o += al(sizeof(float) * gt * kHeadDim);
    L.bars = o;  o += al(sizeof(unsigned long long) * ppc);
    L.total = o;
    return L;
}

template <int GT>
__global__ void __cluster_dims__(kC, 1, 1) __launch_bounds__(kT, 1) k_decode_cluster2(
    const __nv_bfloat16 *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, int np_cap, int page_cap, int k_pages,
    int chunk, int ppc_cap, const int32_t *__restrict__ n_parents, const int32_t *__restrict__ n_pages,
    const __nv_bfloat16 *__restrict__ parent_keys, const int32_t *__restrict__ parent_first_page,
    const int32_t *__restrict__ parent_last_page, const int32_t *__restrict__ parent_n_pages,
    const int32_t *__restrict__ page_next, const int32_t *__restrict__ page_len,
    const __nv_bfloat16 *__restrict__ pool_k, const __nv_bfloat16 *__restrict__ pool_v, int32_t *__restrict__ sel_pages,
    int32_t *__restrict__ sel_count, int max_sel, __nv_bfloat16 *__restrict__ kbuf, __nv_bfloat16 *__restrict__ vbuf,
    int32_t *__restrict__ buf_len, float scale, float *__restrict__ O, int n_pos, int32_t *__restrict__ err) {
    dep_wait();  // the previous kernel of the stream is complete (launched as its dependent)
    cg::cluster_group cluster = cg::this_cluster();
    const int r = (int)cluster.block_rank();
    const int u = blockIdx.y;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kc = k_pages;
    extern __shared__ __align__(128) unsigned char smem[];
    const Lay L = layout(GT, chunk, page_cap, max_sel, ppc_cap);
    float *s_sc = reinterpret_cast<float *>(smem + L.sc);
    int4 *s_span = reinterpret_cast<int4 *>(smem + L.span);
    unsigned long long *s_top = reinterpret_cast<unsigned long long *>(smem + L.top);
    unsigned long long *s_cand = reinterpret_cast<unsigned long long *>(smem + L.cand);
    unsigned *s_mask = reinterpret_cast<unsigned *>(smem + L.mask);
    int *s_uni = reinterpret_cast<int *>(smem + L.uni);
    __nv_bfloat16 *s_kv = reinterpret_cast<__nv_bfloat16 *>(smem + L.kv);
    float *s_p = reinterpret_cast<float *>(smem + L.p);
    unsigned long long *s_pp = reinterpret_cast<unsigned long long *>(smem + L.pp);
    float *s_ml = reinterpret_cast<float *>(smem + L.ml);
    float *s_alpha = reinterpret_cast<float *>(smem + L.alpha);
    float *s_pm = reinterpret_cast<float *>(smem + L.pm);
    float *s_pl = reinterpret_cast<float *>(smem + L.pl);
    float *s_po = reinterpret_cast<float *>(smem + L.po);
    unsigned long long *s_bar = reinterpret_cast<unsigned long long *>(smem + L.bars);
    __shared__ int s_wsum[kW];

    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int Np = min(n_parents[u], np_cap);
    const int m0 = r * chunk;
    const int c = lane & 15, half = lane >> 4;
    if (tid == 0) {
        for (int i = 0; i < ppc_cap; ++i) mbar_init(&s_bar[i], 1);
        mbar_init_fence();
    }

    // q slices: head hh, dims 8c .. 8c + 7 (converted to fp32 pairs once the
    // first parent rows are on their way)
    uint4 qraw[GT];
    {
        const __nv_bfloat16 *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
#pragma unroll
        for (int hh = 0; hh < GT; ++hh)
            qraw[hh] = hh < g ? *reinterpret_cast<const uint4 *>(Qu + (size_t)hh * kHeadDim + 8 * c)
                              : make_uint4(0, 0, 0, 0);
    }
    unsigned long long q[GT][4];

    // ------------------------------------------------------------ phase 1
    // the slice's page spans (read by the leader after the first cluster
    // barrier): their loads go out with the parent rows below
    int4 sp_mine[kSpanPT];
#pragma unroll
    for (int i = 0; i < kSpanPT; ++i) {
        const int loc = tid + i * kT, m = m0 + loc;
        sp_mine[i] = make_int4(0, 0, 0, 0);
        if (loc < chunk && m < Np)
            sp_mine[i] = make_int4(parent_first_page[up + m], parent_n_pages[up + m], parent_last_page[up + m], m);
    }
    {
        constexpr int U4 = 8;  // parent rows per lane in flight
        for (int base = 0; base < chunk; base += kW * 2 * U4) {
            uint4 raw[U4];
#pragma unroll
            for (int i = 0; i < U4; ++i) {
                const int loc = base + (i * kW + warp) * 2 + half;
                const int m = m0 + loc;
                raw[i] = (loc < chunk && m < Np)
                             ? *reinterpret_cast<const uint4 *>(parent_keys + (up + m) * kHeadDim + 8 * c)
                             : make_uint4(0, 0, 0, 0);
            }
            if (base == 0) {
#pragma unroll
                for (int hh = 0; hh < GT; ++hh) {
                    q[hh][0] = bf2_pair(qraw[hh].x);
                    q[hh][1] = bf2_pair(qraw[hh].y);
                    q[hh][2] = bf2_pair(qraw[hh].z);
                    q[hh][3] = bf2_pair(qraw[hh].w);
                }
            }
#pragma unroll
            for (int i = 0; i < U4; ++i) {
                const int loc = base + (i * kW + warp) * 2 + half;
                const int m = m0 + loc;
                const unsigned long long x0 = bf2_pair(raw[i].x), x1 = bf2_pair(raw[i].y), x2 = bf2_pair(raw[i].z),
                                         x3 = bf2_pair(raw[i].w);
                float a[GT];
#pragma unroll
                for (int hh = 0; hh < GT; ++hh) {
                    unsigned long long s2 = fma2(q[hh][0], x0, 0ull);
                    s2 = fma2(q[hh][1], x1, s2);
                    s2 = fma2(q[hh][2], x2, s2);
                    s2 = fma2(q[hh][3], x3, s2);
                    const float2 f = upk2(s2);
                    a[hh] = f.x + f.y;
                }
                int head = 0, off = 8;
#pragma unroll
                for (int nn = GT; nn > 1; nn >>= 1, off >>= 1) {
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int k2 = 0; k2 < nn / 2; ++k2) {
                        const float send = upper ? a[k2] : a[k2 + nn / 2];
                        const float keep = upper ? a[k2 + nn / 2] : a[k2];
                        a[k2] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                    head += upper ? nn / 2 : 0;
                }
                float v = a[0];
                for (; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if ((lane & (16 / GT - 1)) == 0 && head < g && loc < chunk)
                    s_sc[head * chunk + loc] = m < Np ? v : -INFINITY;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kSpanPT; ++i) {
        const int loc = tid + i * kT;
        int4 sp = sp_mine[i];
        sp.z = sp.z - sp.x + 1 == sp.y ? 1 : 0;  // contiguous page run
        if (loc < chunk) s_span[loc] = sp;
    }
    for (int loc = tid + kSpanPT * kT; loc < chunk; loc += kT) {  // slices beyond the register batch
        const int m = m0 + loc;
        int4 sp = make_int4(0, 0, 0, 0);
        if (m < Np) {
            const int fp = parent_first_page[up + m], np = parent_n_pages[up + m], lp = parent_last_page[up + m];
            sp = make_int4(fp, np, lp - fp + 1 == np ? 1 : 0, m);
        }
        s_span[loc] = sp;
    }
    __syncthreads();
    // per head: the slice's best kc keys, sorted (lane = rank), into s_top
    if (warp < g) {
        const int hh = warp;
        const float *sc = s_sc + hh * chunk;
        const int nvalid = max(0, min(chunk, Np - m0));
        uint32_t tbits = 0u;  // order-preserving form of T
        if (nvalid >= kc) {
            uint32_t res = 0u;
            // the lane's values in registers; a bound that the best kc reach and
            // at most kCand keys reach unless ties force more
            if (nvalid <= 8 * 32) {
                uint32_t vo[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) vo[e] = e * 32 + lane < nvalid ? ord_f32(sc[e * 32 + lane]) : 0u;
                res = kth_bound_ord(vo, kc, kCand - kc);
            } else if (nvalid <= 16 * 32) {
                uint32_t vo[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) vo[e] = e * 32 + lane < nvalid ? ord_f32(sc[e * 32 + lane]) : 0u;
                res = kth_bound_ord(vo, kc, kCand - kc);
            } else {
                for (int bit = 31; bit >= 0; --bit) {
                    const uint32_t cnd = res | (1u << bit);
                    unsigned cnt = 0;
                    for (int x = lane; x < nvalid; x += 32) cnt += ord_f32(sc[x]) >= cnd;
                    if ((int)__reduce_add_sync(0xffffffffu, cnt) >= kc) res = cnd;
                }
            }
            tbits = res;
        }
        unsigned long long *cand = s_cand + warp * kCand;
        int cnt = 0;
        for (int x0 = 0; x0 < nvalid; x0 += 32) {
            const int x = x0 + lane;
            const bool pass = x < nvalid && ord_f32(sc[x]) >= tbits;
            const unsigned bal = __ballot_sync(0xffffffffu, pass);
            const int at = cnt + __popc(bal & lanemask_lt());
            if (pass && at < kCand) cand[at] = sort_key(sc[x], m0 + x);
            cnt += __popc(bal);
        }
        __syncwarp();
        unsigned long long best = 0ull;
        if (cnt <= kCand) {
            unsigned long long v[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) v[e] = e * 32 + lane < cnt ? cand[e * 32 + lane] : 0ull;
            sort64_desc(v);
            best = v[0];
        } else {  // very many ties with T: kc rounds of a warp maximum
            unsigned long long last = ~0ull;
            for (int rr = 0; rr < kc; ++rr) {
                unsigned long long bb = 0ull;
                for (int x = lane; x < nvalid; x += 32) {
                    const unsigned long long k = sort_key(sc[x], m0 + x);
                    if (k < last && k > bb) bb = k;
                }
#pragma unroll
                for (int of = 16; of >= 1; of >>= 1) bb = umax64(bb, __shfl_xor_sync(0xffffffffu, bb, of));
                if (lane == rr) best = bb;
                last = bb;
            }
        }
        s_top[hh * 32 + lane] = lane < kc ? best : 0ull;
    }
    const int P = min(n_pages[u], page_cap);
    const int Ps = max(0, P - n_pos);  // semantic pages; the positional rest is always in the union
    const int words = (P + 31) / 32;
    if (r == 0)
        for (int x = tid; x < words; x += kT) s_mask[x] = 0u;
    cluster.sync();

    // ------------------------------------------------------------ phase 2
    if (r == 0) {
        if (k_pages >= Ps) {
            for (int x = tid; x < words; x += kT) {
                const int rem = P - x * 32;
                s_mask[x] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
            }
        } else {
            for (int x = Ps + tid; x < P; x += kT) atomicOr(&s_mask[x >> 5], 1u << (x & 31));
        }
        if (k_pages < Ps && warp < g) {
            const int hh = warp;
            unsigned long long v[kC];
#pragma unroll
            for (int j = 0; j < kC; ++j) v[j] = cluster.map_shared_rank(s_top, j)[hh * 32 + lane];
#pragma unroll
            for (int st = 1; st < kC; st <<= 1)
#pragma unroll
                for (int j = 0; j < kC; j += 2 * st) v[j] = merge32(v[j], v[j + st]);
            const unsigned long long k = lane < kc ? v[0] : 0ull;
            int cnt = 0, fp = 0, contig = 1;
            if (k != 0ull) {
                const int pm = key_id(k);
                const int owner = pm / chunk;
                const int4 sp = cluster.map_shared_rank(s_span, owner)[pm - owner * chunk];
                fp = sp.x;
                cnt = sp.y;
                contig = sp.z;
            }
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            const int tk = max(0, min(cnt, k_pages - (incl - cnt)));
            int pg = fp;
            for (int i = 0; i < tk; ++i) {
                const int qq = contig ? fp + i : pg;
                if (qq < 0 || qq >= Ps) break;
                atomicOr(&s_mask[qq >> 5], 1u << (qq & 31));
                if (!contig) pg = page_next[ug + qq];
            }
        }
        __syncthreads();
        // ascending list of the union's pages: thread tid owns words
        // [tid * wpt, (tid + 1) * wpt); one block-wide scan of the counts
        const int wpt = (words + kT - 1) / kT;
        const int wb = tid * wpt, we = min(words, wb + wpt);
        int cc = 0;
        for (int x = wb; x < we; ++x) cc += __popc(s_mask[x]);
        int incl = cc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int pos = incl - cc, total = 0;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            pos += w < warp ? s_wsum[w] : 0;
            total += s_wsum[w];
        }
        for (int x = wb; x < we && pos < max_sel; ++x) {
            unsigned bb = s_mask[x];
            while (bb && pos < max_sel) {
                const int bit = __ffs(bb) - 1;
                bb &= bb - 1;
                s_uni[1 + pos] = x * 32 + bit;
                sel_pages[(size_t)u * max_sel + pos] = x * 32 + bit;
                ++pos;
            }
        }
        for (int x = total + tid; x < max_sel; x += kT) sel_pages[(size_t)u * max_sel + x] = -1;
        if (tid == 0) {
            if (total > max_sel) set_err(err, ICE_ERR_CAPACITY);
            s_uni[0] = min(total, max_sel);
            sel_count[u] = min(total, max_sel);
        }
    }
    cluster.sync();

    // ------------------------------------------------------------ phase 3
    const int *uni = cluster.map_shared_rank(s_uni, 0);
    const int n = uni[0];
    const int ppc = (n + kC - 1) / kC;
    const int x0 = min(n, r * ppc), x1 = min(n, x0 + ppc);
    const int np = x1 - x0;  // <= ppc_cap (checked on the host from max_sel)
    {
        const int ps = (max_sel + kC - 1) / kC;  // slots past the selection: each CTA a static share
        if (buf_len)  // no buf_len: no contiguous copy
            for (int x = max(n, r * ps) + tid; x < min(max_sel, (r + 1) * ps); x += kT) buf_len[(size_t)u * max_sel + x] = 0;
    }
    if (tid == 0) {
        for (int i = 0; i < np; ++i) {
            const size_t pg = ug + uni[1 + x0 + i];
            mbar_expect_tx(&s_bar[i], 2 * kPageBytes);
            bulk_load(s_kv + (size_t)i * 2 * kPageElems, pool_k + pg * kPageElems, kPageBytes, &s_bar[i]);
            bulk_load(s_kv + (size_t)i * 2 * kPageElems + kPageElems, pool_v + pg * kPageElems, kPageBytes, &s_bar[i]);
        }
    }
    if (lane < GT) {
        s_ml[(warp * GT + lane) * 2 + 0] = -INFINITY;
        s_ml[(warp * GT + lane) * 2 + 1] = 0.f;
    }
    unsigned long long o[GT][2];
#pragma unroll
    for (int hh = 0; hh < GT; ++hh) o[hh][0] = o[hh][1] = 0ull;
    bool ok = true, stored = false;
    float *pw = s_p + warp * kPage * GT;
    unsigned long long *ppw = s_pp + warp * kPage * GT;
    for (int i = warp; i < np; i += kW) {
        const int x = x0 + i;
        const size_t slot = (size_t)u * max_sel + x;
        const int pgid = uni[1 + x];
        const int len = page_len[ug + pgid];
        if (buf_len && lane == 0) buf_len[slot] = len;
        if (ok) ok = mbar_wait(&s_bar[i], 0);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const __nv_bfloat16 *Kp = s_kv + (size_t)i * 2 * kPageElems;
        const __nv_bfloat16 *Vp = Kp + kPageElems;
        if (buf_len && lane == 0) {  // the contiguous buffer, straight from shared memory
            fence_proxy_async();
            bulk_store(kbuf + slot * kPageElems, Kp, kPageBytes);
            bulk_store(vbuf + slot * kPageElems, Vp, kPageBytes);
            bulk_commit();
            stored = true;
        }
        // logits of the page's 16 slots
#pragma unroll 2
        for (int kp = 0; kp < kPage / 2; ++kp) {
            const int j = 2 * kp + half;
            const uint4 raw = *reinterpret_cast<const uint4 *>(Kp + j * kHeadDim + 8 * c);
            const unsigned long long x0p = bf2_pair(raw.x), x1p = bf2_pair(raw.y), x2p = bf2_pair(raw.z),
                                     x3p = bf2_pair(raw.w);
            float a[GT];
#pragma unroll
            for (int hh = 0; hh < GT; ++hh) {
                unsigned long long s2 = fma2(q[hh][0], x0p, 0ull);
                s2 = fma2(q[hh][1], x1p, s2);
                s2 = fma2(q[hh][2], x2p, s2);
                s2 = fma2(q[hh][3], x3p, s2);
                const float2 f = upk2(s2);
                a[hh] = f.x + f.y;
            }
            int head = 0, off = 8;
#pragma unroll
            for (int nn = GT; nn > 1; nn >>= 1, off >>= 1) {
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int k2 = 0; k2 < nn / 2; ++k2) {
                    const float send = upper ? a[k2] : a[k2 + nn / 2];
                    const float keep = upper ? a[k2 + nn / 2] : a[k2];
                    a[k2] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
                head += upper ? nn / 2 : 0;
            }
            float v = a[0];
            for (; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if ((lane & (16 / GT - 1)) == 0 && head < g) pw[j * GT + head] = v;
        }
        __syncwarp();
        // online softmax update per head, 16 lanes per head
#pragma unroll
        for (int e = 0; e < (GT * kPage + 31) / 32; ++e) {
            const int item = e * 32 + lane;
            const int hh = item / kPage, sl = item % kPage;
            const bool on = hh < g && item < GT * kPage;
            const float lg = (on && sl < len) ? pw[sl * GT + hh] * scale : -INFINITY;
            float mx = lg;
#pragma unroll
            for (int of = 8; of >= 1; of >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, of));
            const float m_old = on ? s_ml[(warp * GT + hh) * 2] : -INFINITY;
            const float m_new = fmaxf(m_old, mx);
            const float pr = lg == -INFINITY ? 0.f : expf(lg - m_new);
            float sm = pr;
#pragma unroll
            for (int of = 8; of >= 1; of >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, of);
            if (on) ppw[sl * GT + hh] = pk2(pr, pr);
            __syncwarp();
            if (on && sl == 0) {
                const float alpha = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
                s_alpha[warp * GT + hh] = alpha;
                s_ml[(warp * GT + hh) * 2 + 0] = m_new;
                s_ml[(warp * GT + hh) * 2 + 1] = s_ml[(warp * GT + hh) * 2 + 1] * alpha + sm;
            }
        }
        __syncwarp();
        // o = o * alpha + P V, lane owns dims 4 lane .. 4 lane + 3
#pragma unroll
        for (int hh = 0; hh < GT; ++hh) {
            const float al = hh < g ? s_alpha[warp * GT + hh] : 0.f;
            const unsigned long long aa = pk2(al, al);
            o[hh][0] = fma2(o[hh][0], aa, 0ull);
            o[hh][1] = fma2(o[hh][1], aa, 0ull);
        }
#pragma unroll 4
        for (int sl = 0; sl < kPage; ++sl) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(Vp + sl * kHeadDim + 4 * lane);
            const unsigned long long v01 = bf2_pair(raw.x), v23 = bf2_pair(raw.y);
            const unsigned long long *pps = ppw + sl * GT;
#pragma unroll
            for (int hh = 0; hh < GT; ++hh) {
                const unsigned long long pv = pps[hh];
                o[hh][0] = fma2(pv, v01, o[hh][0]);
                o[hh][1] = fma2(pv, v23, o[hh][1]);
            }
        }
        __syncwarp();
    }
    if (!ok) set_err(err, ICE_ERR_TIMEOUT);
    if (stored) bulk_wait_read_all();  // the page buffers are reused below
    __syncthreads();
    // merge the warps into this CTA's partial (page area reused)
    float *s_ow = reinterpret_cast<float *>(s_kv);  // [kW][GT][128]
#pragma unroll
    for (int hh = 0; hh < GT; ++hh) {
        const float2 a = upk2(o[hh][0]), bq = upk2(o[hh][1]);
        *reinterpret_cast<float4 *>(s_ow + ((size_t)warp * GT + hh) * kHeadDim + 4 * lane) = make_float4(a.x, a.y, bq.x, bq.y);
    }
    __syncthreads();
    if (tid < GT) {
        float M = -INFINITY;
        for (int w = 0; w < kW; ++w) M = fmaxf(M, s_ml[(w * GT + tid) * 2]);
        float Lsum = 0.f;
        for (int w = 0; w < kW; ++w) {
            const float m = s_ml[(w * GT + tid) * 2];
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            s_alpha[w * GT + tid] = wt;  // now the merge weight of warp w
            Lsum = fmaf(s_ml[(w * GT + tid) * 2 + 1], wt, Lsum);
        }
        s_pm[tid] = M;
        s_pl[tid] = Lsum;
    }
    __syncthreads();
    for (int x = tid; x < g * kHeadDim; x += kT) {
        const int hh = x / kHeadDim, d = x % kHeadDim;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kW; ++w) acc = fmaf(s_ow[((size_t)w * GT + hh) * kHeadDim + d], s_alpha[w * GT + hh], acc);
        s_po[hh * kHeadDim + d] = acc;
    }
    cluster.sync();

    // ------------------------------------------------------------ phase 4
    for (int hh = r; hh < g; hh += kC) {
        float ms[kC], ls[kC];
#pragma unroll
        for (int cc = 0; cc < kC; ++cc) {
            ms[cc] = cluster.map_shared_rank(s_pm, cc)[hh];
            ls[cc] = cluster.map_shared_rank(s_pl, cc)[hh];
        }
        float M = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < kC; ++cc) M = fmaxf(M, ms[cc]);
        if (tid < kHeadDim) {
            float os[kC];
#pragma unroll
            for (int cc = 0; cc < kC; ++cc) os[cc] = cluster.map_shared_rank(s_po, cc)[hh * kHeadDim + tid];
            float Ls = 0.f, acc = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int cc = 0; cc < kC; ++cc) {
                    if (ms[cc] == -INFINITY) continue;
                    const float wgt = expf(ms[cc] - M);
                    Ls = fmaf(ls[cc], wgt, Ls);
                    acc = fmaf(os[cc], wgt, acc);
                }
            }
            O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + tid] = Ls > 0.f ? acc / Ls : 0.f;
        }
    }
    cluster.sync();  // every CTA's shared memory stays valid until the remote reads are done
}

struct Shape2 {
    int gt, chunk, ppc;
    size_t smem;
};
Shape2 shape2(const ice_params &p, int max_sel) {
    Shape2 s{};
    const int g = p.n_q_heads / p.n_kv_heads;
    s.gt = g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
    s.chunk = (p.np_cap + kC - 1) / kC;
    if (s.chunk < 1) s.chunk = 1;
    s.ppc = (max_sel + kC - 1) / kC;
    s.smem = layout(s.gt, s.chunk, p.page_cap, max_sel, s.ppc).total;
    return s;
}

template <int GT>
cudaError_t launch_gt(const ice_params &p, const ice_index &idx, const void *Q, int k_pages, int32_t *sel_pages,
                      int32_t *sel_count, int max_sel, void *kbuf, void *vbuf, int32_t *buf_len, float scale,
                      float *O, int32_t *err, cudaStream_t s, const Shape2 &sh) {
    if (sh.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_cluster2<GT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sh.smem);
        if (e != cudaSuccess) return e;
    }
    const int g = p.n_q_heads / p.n_kv_heads;
    {
        const cudaError_t e_ = launch_dependent(k_decode_cluster2<GT>, dim3(kC, units_of(p)), dim3(kT), sh.smem, s,
                                                static_cast<const __nv_bfloat16 *>(Q), g, p.n_q_heads, p.n_kv_heads,
                                                p.np_cap, p.page_cap, k_pages, sh.chunk, sh.ppc, idx.n_parents,
                                                idx.n_pages, static_cast<const __nv_bfloat16 *>(idx.parent_keys),
                                                idx.parent_first_page, idx.parent_last_page, idx.parent_n_pages,
                                                idx.page_next, idx.page_len,
                                                static_cast<const __nv_bfloat16 *>(idx.pool_k),
                                                static_cast<const __nv_bfloat16 *>(idx.pool_v), sel_pages, sel_count,
                                                max_sel, static_cast<__nv_bfloat16 *>(kbuf),
                                                static_cast<__nv_bfloat16 *>(vbuf), buf_len, scale, O,
                                                pos_split(p).n_pos, err);
        if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
}

}  // namespace

bool decode_cluster2_supported(const ice_params &p, int k_pages, int max_sel) {
    const int g = p.n_q_heads / p.n_kv_heads;
    if (p.dtype != ICE_BF16 || g < 1 || g > 8 || k_pages < 1 || k_pages > 32) return false;
    const Shape2 sh = shape2(p, max_sel);
    return sh.ppc <= kMaxPPC && sh.smem <= 200 * 1024;
}

cudaError_t launch_decode_cluster2(const ice_params &p, const ice_index &idx, const void *Q, int k_pages,
                                   int32_t *sel_pages, int32_t *sel_count, int max_sel, void *kbuf, void *vbuf,
                                   int32_t *buf_len, float scale, float *O, int32_t *err, cudaStream_t s) {
    const Shape2 sh = shape2(p, max_sel);
    switch (sh.gt) {
        case 1: return launch_gt<1>(p, idx, Q, k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale, O, err, s, sh);
        case 2: return launch_gt<2>(p, idx, Q, k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale, O, err, s, sh);
        case 4: return launch_gt<4>(p, idx, Q, k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale, O, err, s, sh);
        default: return launch_gt<8>(p, idx, Q, k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale, O, err, s, sh);
    }
}

}  // namespace ice
