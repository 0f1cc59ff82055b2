// The whole decode step (a6-a10) of a unit in one thread-block cluster.
//
// Same computation as k_select followed by the fused k_attn (papernotes.org
// "IceCache: Memory-Efficient KV-cache Management for Long-Sequence LLMs",
// 关键设计 1 (sparse attention), 3 (per-head top-k pages, GQA union), 4 (bulk
// gather into a contiguous buffer); IceCache popular-science article
// (aitangshan.cn/news/751385), sections 四 and 六), but the exchanges between
// the phases go through distributed shared memory under hardware cluster
// barriers instead of global-memory tickets and a second launch:
//
//   phase 1  CTA r of the unit's cluster scores its slice of the parent
//            table against the g query heads (all row loads issued at once,
//            independent of the unit's parent count) and keeps, per head,
//            its best kc parents as packed (score, -m) keys (one warp per
//            head: kc rounds of a warp-wide max below the previous winner;
//            keys are unique, so no marking is needed), plus the page span
//            of each of its parents;                        -- cluster barrier
//   phase 2  the leader CTA reads every CTA's candidates (DSMEM), orders the
//            best k per head the same way, walks the ordered parents (spans
//            read from the owning CTA) taking pages until k, ORs them into a
//            bitmask and writes the ascending union (sel_pages, sel_count);
//                                                            -- cluster barrier
//   phase 3  CTA r takes its share of the union's pages (read from the
//            leader) in batches of up to 8: loads them once from the pool,
//            writes the contiguous buffer (kbuf, vbuf, buf_len), computes all
//            logits of the batch, one online-softmax update per head, and the
//            PV products, keeping (max, sum, o) in its shared memory;
//                                                            -- cluster barrier
//   phase 4  CTA r merges the partials of heads r, r + C, ... of all CTAs
//            (log-sum-exp, DSMEM) and writes O.             -- barrier, exit
// No CTA ever waits on a flag; the four barriers are barrier.cluster.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace cg = cooperative_groups;

namespace ice {
namespace {

using namespace topk;

constexpr int kC = kDecodeCluster;  // CTAs per cluster = per unit
constexpr int kT = 256;             // threads per CTA
constexpr int kWarps = kT / 32;
constexpr int kMaxG = 16;
constexpr int kPB = 8;              // pages per batch in phase 3


// The warp's best kc of keys[0..n) in descending order (0 = no key).  Keys
// are unique, so round r takes the largest key below round r-1's.
__device__ void warp_topk64(const unsigned long long *keys, int n, int kc, unsigned long long *out) {
    const int lane = threadIdx.x & 31;
    unsigned long long last = ~0ull;
    for (int r = 0; r < kc; ++r) {
        unsigned long long best = 0ull;
        if (last != 0ull) {
            for (int x = lane; x < n; x += 32) {
                const unsigned long long k = keys[x];
                if (k < last && k > best) best = k;
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
                best = o > best ? o : best;
            }
        }
        if (lane == 0) out[r] = best;
        last = best;
    }
    __syncwarp();
}

// Shared-memory layout of one CTA (offsets in bytes, 16-byte aligned).
struct Lay {
    size_t q, key, top, cand, ord, span, mask, uni, lg, pm, pl, po, stage, total;
};
__host__ __device__ inline Lay layout(int g, int chunk, int kc, int kt, int page_cap, int max_sel, int esz) {
    auto al = [](size_t x) { return (x + 15) & ~(size_t)15; };
    Lay L{};
    size_t o = 0;
    L.q = o;     o += al(sizeof(float) * g * kHeadDim);
    L.key = o;   o += al(sizeof(unsigned long long) * g * chunk);
    L.top = o;   o += al(sizeof(unsigned long long) * g * kc);
    L.cand = o;  o += al(sizeof(unsigned long long) * g * kC * kc);
    L.ord = o;   o += al(sizeof(unsigned long long) * g * kt);
    L.span = o;  o += al(sizeof(int4) * chunk);
    L.mask = o;  o += al(sizeof(unsigned) * ((page_cap + 31) / 32));
    L.uni = o;   o += al(sizeof(int) * (max_sel + 1));
    L.lg = o;    o += al(sizeof(float) * g * kPB * kPage);
    L.pm = o;    o += al(sizeof(float) * g);
    L.pl = o;    o += al(sizeof(float) * g);
    L.po = o;    o += al(sizeof(float) * 2 * g * kHeadDim);
    L.stage = o; o += al((size_t)2 * kPB * kPage * kHeadDim * esz);
    L.total = o;
    return L;
}

template <typename T>
__global__ void __cluster_dims__(kC, 1, 1) __launch_bounds__(kT) k_decode_cluster(
    const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, int np_cap, int page_cap, int k_pages, int kc,
    int kt, int chunk, const int32_t *__restrict__ n_parents, const int32_t *__restrict__ n_pages,
    const T *__restrict__ parent_keys, const int32_t *__restrict__ parent_first_page,
    const int32_t *__restrict__ parent_last_page, const int32_t *__restrict__ parent_n_pages,
    const int32_t *__restrict__ page_next, const int32_t *__restrict__ page_len, const T *__restrict__ pool_k,
    const T *__restrict__ pool_v, int32_t *__restrict__ sel_pages, int32_t *__restrict__ sel_count, int max_sel,
    T *__restrict__ kbuf, T *__restrict__ vbuf, int32_t *__restrict__ buf_len, float scale, float *__restrict__ O,
    int n_pos, int32_t *__restrict__ err) {
    cg::cluster_group cluster = cg::this_cluster();
    const int r = (int)cluster.block_rank();
    const int u = blockIdx.y;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = threadIdx.x;
    extern __shared__ __align__(16) unsigned char smem[];
    const Lay L = layout(g, chunk, kc, kt, page_cap, max_sel, (int)sizeof(T));
    float *s_q = reinterpret_cast<float *>(smem + L.q);
    unsigned long long *s_key = reinterpret_cast<unsigned long long *>(smem + L.key);
    unsigned long long *s_top = reinterpret_cast<unsigned long long *>(smem + L.top);
    unsigned long long *s_cand = reinterpret_cast<unsigned long long *>(smem + L.cand);
    unsigned long long *s_ord = reinterpret_cast<unsigned long long *>(smem + L.ord);
    int4 *s_span = reinterpret_cast<int4 *>(smem + L.span);
    unsigned *s_mask = reinterpret_cast<unsigned *>(smem + L.mask);
    int *s_uni = reinterpret_cast<int *>(smem + L.uni);  // [0] = count, then the union
    float *s_lg = reinterpret_cast<float *>(smem + L.lg);
    float *s_pm = reinterpret_cast<float *>(smem + L.pm);
    float *s_pl = reinterpret_cast<float *>(smem + L.pl);
    float *s_po = reinterpret_cast<float *>(smem + L.po);
    uint4 *s_stage = reinterpret_cast<uint4 *>(smem + L.stage);
    __shared__ int s_wsum[kWarps];
    __shared__ int s_carry;
    __shared__ float s_alpha[kMaxG];
    __shared__ int s_len[kPB];

    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int m0 = r * chunk;

    // ------------------------------------------------------------ phase 1
    constexpr int RV = row_vecs<T>();
    constexpr int PV = Elem<T>::kPerVec;
    const T *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
    for (int x = t; x < g * kHeadDim; x += kT) s_q[x] = Elem<T>::load(Qu + x);
    const int Np = min(n_parents[u], np_cap);
    __syncthreads();
    for (int loc = t; loc < chunk; loc += kT) {
        const int m = m0 + loc;
        const bool inside = m < np_cap;  // always readable; validity against Np is applied below
        int4 sp = make_int4(0, 0, 0, 0);
        if (inside) {
            const uint4 *row = reinterpret_cast<const uint4 *>(parent_keys + (up + m) * kHeadDim);
            const int fp = parent_first_page[up + m], np = parent_n_pages[up + m], lp = parent_last_page[up + m];
            for (int h0 = 0; h0 < g; h0 += 8) {
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
                for (int v0 = 0; v0 < RV; v0 += 8) {
                    uint4 raw[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) raw[i] = __ldg(row + v0 + i);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float f[PV];
                        Elem<T>::unpack(raw[i], f);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            if (h0 + q < g) {
                                const float4 *qq =
                                    reinterpret_cast<const float4 *>(s_q + (size_t)(h0 + q) * kHeadDim + (v0 + i) * PV);
#pragma unroll
                                for (int e4 = 0; e4 < PV / 4; ++e4) {
                                    const float4 qv = qq[e4];
                                    acc[q] = fmaf(qv.x, f[4 * e4 + 0], acc[q]);
                                    acc[q] = fmaf(qv.y, f[4 * e4 + 1], acc[q]);
                                    acc[q] = fmaf(qv.z, f[4 * e4 + 2], acc[q]);
                                    acc[q] = fmaf(qv.w, f[4 * e4 + 3], acc[q]);
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (h0 + q < g) s_key[(size_t)(h0 + q) * chunk + loc] = m < Np ? sort_key(acc[q], m) : 0ull;
            }
            if (m < Np) sp = make_int4(fp, np, lp - fp + 1 == np ? 1 : 0, m);
        } else {
            for (int hh = 0; hh < g; ++hh) s_key[(size_t)hh * chunk + loc] = 0ull;
        }
        s_span[loc] = sp;
    }
    __syncthreads();
    for (int hh = warp; hh < g; hh += kWarps) warp_topk64(s_key + (size_t)hh * chunk, chunk, kc, s_top + hh * kc);
    cluster.sync();

    // ------------------------------------------------------------ phase 2
    if (r == 0) {
        const int P = min(n_pages[u], page_cap);
        const int Ps = max(0, P - n_pos);  // semantic pages; the positional rest is always in the union
        const int words = (P + 31) / 32;
        for (int x = t; x < words; x += kT) s_mask[x] = 0u;
        if (k_pages >= Ps) {
            __syncthreads();
            for (int x = t; x < words; x += kT) {
                const int rem = P - x * 32;
                s_mask[x] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
            }
        } else {
            const int nc = kC * kc;
            for (int x = t; x < g * nc; x += kT) {
                const int hh = x / nc, i = x % nc;
                s_cand[x] = cluster.map_shared_rank(s_top, i / kc)[hh * kc + i % kc];
            }
            __syncthreads();
            for (int x = Ps + t; x < P; x += kT) atomicOr(&s_mask[x >> 5], 1u << (x & 31));
            for (int hh = warp; hh < g; hh += kWarps) {
                warp_topk64(s_cand + (size_t)hh * nc, nc, kt, s_ord + (size_t)hh * kt);
                int taken = 0;
                for (int t0 = 0; t0 < kt && taken < k_pages; t0 += 32) {
                    int cnt = 0;
                    int4 sp = make_int4(0, 0, 0, 0);
                    if (t0 + lane < kt) {
                        const unsigned long long k = s_ord[(size_t)hh * kt + t0 + lane];
                        if (k != 0ull) {
                            const int pm = key_id(k);
                            const int owner = pm / chunk;
                            sp = cluster.map_shared_rank(s_span, owner)[pm - owner * chunk];
                            cnt = sp.y;
                        }
                    }
                    int incl = cnt;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const int o = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += o;
                    }
                    const int take = max(0, min(cnt, k_pages - (taken + incl - cnt)));
                    int pg = sp.x;
                    for (int i = 0; i < take; ++i) {
                        const int q = sp.z ? pg + i : pg;
                        if (q < 0 || q >= Ps) break;
                        atomicOr(&s_mask[q >> 5], 1u << (q & 31));
                        if (!sp.z) pg = page_next[ug + q];
                    }
                    taken += __shfl_sync(0xffffffffu, incl, 31);
                }
            }
        }
        __syncthreads();
        if (t == 0) s_carry = 0;
        __syncthreads();
        for (int w0 = 0; w0 < words; w0 += kT) {
            const int x = w0 + t;
            const unsigned bits = x < words ? s_mask[x] : 0u;
            const int c = __popc(bits);
            int incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (lane == 31) s_wsum[warp] = incl;
            __syncthreads();
            int pos = s_carry;
            for (int w = 0; w < warp; ++w) pos += s_wsum[w];
            pos += incl - c;
            unsigned bb = bits;
            while (bb) {
                const int bit = __ffs(bb) - 1;
                bb &= bb - 1;
                if (pos < max_sel) {
                    s_uni[1 + pos] = x * 32 + bit;
                    sel_pages[(size_t)u * max_sel + pos] = x * 32 + bit;
                }
                ++pos;
            }
            __syncthreads();
            if (t == kT - 1) s_carry = pos;
            __syncthreads();
        }
        const int total = s_carry;
        for (int x = total + t; x < max_sel; x += kT) sel_pages[(size_t)u * max_sel + x] = -1;
        if (t == 0) {
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
    if (buf_len) {  // no buf_len: no contiguous copy
        for (int x = min(max_sel, r * ppc) + t; x < min(max_sel, (r + 1) * ppc); x += kT)
            if (x >= n) buf_len[(size_t)u * max_sel + x] = 0;
        if (r == kC - 1)  // slots no CTA's share reaches
            for (int x = kC * ppc + t; x < max_sel; x += kT) buf_len[(size_t)u * max_sel + x] = 0;
    }
    if (t < g) {
        s_pm[t] = -INFINITY;
        s_pl[t] = 0.f;
    }
    float o[kMaxG];
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh) o[hh] = 0.f;
    constexpr int PVEC = kPage * RV;          // 16-byte vectors per page
    constexpr int VPT = PVEC / kT > 0 ? PVEC / kT : 1;
    constexpr int CV = 8 / PV;                // vectors per 8-element chunk
    const int c = t & 15, grp = t >> 4;       // logits: 8-element chunk, lane group
    const int dim = t & (kHeadDim - 1), half = t / kHeadDim;
    for (int xb = x0; xb < x1; xb += kPB) {
        const int np = min(kPB, x1 - xb);
        uint4 rk[kPB][VPT], rv[kPB][VPT];
#pragma unroll
        for (int i = 0; i < kPB; ++i) {
            if (i < np) {
                const size_t src = (ug + uni[1 + xb + i]) * PVEC;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    rk[i][v] = reinterpret_cast<const uint4 *>(pool_k)[src + t + v * kT];
                    rv[i][v] = reinterpret_cast<const uint4 *>(pool_v)[src + t + v * kT];
                }
            }
        }
        if (t < np) {
            const int len = page_len[ug + uni[1 + xb + t]];
            s_len[t] = len;
            if (buf_len) buf_len[(size_t)u * max_sel + xb + t] = len;
        }
        __syncthreads();  // the previous batch is consumed
#pragma unroll
        for (int i = 0; i < kPB; ++i) {
            if (i < np) {
                const size_t slot = (size_t)u * max_sel + xb + i;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const int e = t + v * kT;
                    s_stage[(2 * i) * PVEC + e] = rk[i][v];
                    s_stage[(2 * i + 1) * PVEC + e] = rv[i][v];
                    if (buf_len) {
                        reinterpret_cast<uint4 *>(kbuf)[slot * PVEC + e] = rk[i][v];
                        reinterpret_cast<uint4 *>(vbuf)[slot * PVEC + e] = rv[i][v];
                    }
                }
            }
        }
        __syncthreads();
        // logits of every (page, slot pair) of the batch: 16 lanes x 8 elements
        for (int item = grp; item < np * 8; item += kT / 16) {
            const int i = item >> 3, sg = item & 7;
            const uint4 *Kp = s_stage + (2 * i) * PVEC;
            float kf[2][8];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int w = 0; w < CV; ++w) Elem<T>::unpack(Kp[(2 * sg + rr) * RV + c * CV + w], &kf[rr][w * PV]);
            for (int hh = 0; hh < g; ++hh) {
                const float4 q0 = reinterpret_cast<const float4 *>(s_q + (size_t)hh * kHeadDim + 8 * c)[0];
                const float4 q1 = reinterpret_cast<const float4 *>(s_q + (size_t)hh * kHeadDim + 8 * c)[1];
                float a[2];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    float x = q0.x * kf[rr][0];
                    x = fmaf(q0.y, kf[rr][1], x);
                    x = fmaf(q0.z, kf[rr][2], x);
                    x = fmaf(q0.w, kf[rr][3], x);
                    x = fmaf(q1.x, kf[rr][4], x);
                    x = fmaf(q1.y, kf[rr][5], x);
                    x = fmaf(q1.z, kf[rr][6], x);
                    x = fmaf(q1.w, kf[rr][7], x);
                    a[rr] = x;
                }
#pragma unroll
                for (int off = 8; off >= 1; off >>= 1) {
                    a[0] += __shfl_xor_sync(0xffffffffu, a[0], off);
                    a[1] += __shfl_xor_sync(0xffffffffu, a[1], off);
                }
                if (c == 0) {
                    s_lg[(size_t)hh * kPB * kPage + i * kPage + 2 * sg] = a[0];
                    s_lg[(size_t)hh * kPB * kPage + i * kPage + 2 * sg + 1] = a[1];
                }
            }
        }
        __syncthreads();
        // one online-softmax update per head for the whole batch (a warp per head)
        for (int hh = warp; hh < g; hh += kWarps) {
            float *lg = s_lg + (size_t)hh * kPB * kPage;
            float bmax = -INFINITY;
            for (int x = lane; x < np * kPage; x += 32) {
                const float v = (x % kPage) < s_len[x / kPage] ? lg[x] * scale : -INFINITY;
                lg[x] = v;
                bmax = fmaxf(bmax, v);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
            const float m_old = s_pm[hh];
            const float m_new = fmaxf(m_old, bmax);
            float psum = 0.f;
            for (int x = lane; x < np * kPage; x += 32) {
                const float v = lg[x];
                const float pr = (v == -INFINITY) ? 0.f : expf(v - m_new);
                lg[x] = pr;
                psum += pr;
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            if (lane == 0) {
                const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
                s_alpha[hh] = alpha;
                s_pl[hh] = s_pl[hh] * alpha + psum;
                s_pm[hh] = m_new;
            }
        }
        __syncthreads();
        // o[h][dim] += sum over this half's pages of p * v (two halves of the CTA)
#pragma unroll
        for (int hh = 0; hh < kMaxG; ++hh)
            if (hh < g) o[hh] *= s_alpha[hh];
        for (int i = half; i < np; i += kT / kHeadDim) {
            const T *Vp = reinterpret_cast<const T *>(s_stage + (2 * i + 1) * PVEC);
            float vt[kPage];
#pragma unroll
            for (int sl = 0; sl < kPage; ++sl) vt[sl] = Elem<T>::load(Vp + sl * kHeadDim + dim);
#pragma unroll
            for (int hh = 0; hh < kMaxG; ++hh) {
                if (hh < g) {
                    const float *pr = s_lg + (size_t)hh * kPB * kPage + i * kPage;
                    float acc = o[hh];
#pragma unroll
                    for (int sl = 0; sl < kPage; ++sl) acc = fmaf(pr[sl], vt[sl], acc);
                    o[hh] = acc;
                }
            }
        }
    }
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh)
        if (hh < g) s_po[((size_t)half * g + hh) * kHeadDim + dim] = o[hh];
    __syncthreads();
    if (half == 0) {
        for (int hh = 0; hh < g; ++hh) s_po[(size_t)hh * kHeadDim + dim] += s_po[((size_t)g + hh) * kHeadDim + dim];
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
        if (t < kHeadDim) {
            float os[kC];
#pragma unroll
            for (int cc = 0; cc < kC; ++cc) os[cc] = cluster.map_shared_rank(s_po, cc)[(size_t)hh * kHeadDim + t];
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
            O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + t] = Ls > 0.f ? acc / Ls : 0.f;
        }
    }
    cluster.sync();  // every CTA's shared memory stays valid until the remote reads are done
}

struct Shape {
    int chunk, kc, kt;
    size_t smem;
};

Shape shape_of(const ice_params &p, int k_pages, int max_sel) {
    Shape s{};
    const int g = p.n_q_heads / p.n_kv_heads;
    s.chunk = (p.np_cap + kC - 1) / kC;
    if (s.chunk < 1) s.chunk = 1;
    s.kc = k_pages < s.chunk ? k_pages : s.chunk;
    if (s.kc < 1) s.kc = 1;
    s.kt = k_pages < kC * s.kc ? k_pages : kC * s.kc;
    if (s.kt < 1) s.kt = 1;
    s.smem = layout(g, s.chunk, s.kc, s.kt, p.page_cap, max_sel, p.dtype == ICE_BF16 ? 2 : 4).total;
    return s;
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const void *Q, int k_pages, int32_t *sel_pages,
                     int32_t *sel_count, int max_sel, void *kbuf, void *vbuf, int32_t *buf_len, float scale, float *O,
                     int32_t *err, cudaStream_t s) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const Shape sh = shape_of(p, k_pages, max_sel);
    if (sh.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_cluster<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sh.smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(kC, units_of(p));
    k_decode_cluster<T><<<grid, kT, sh.smem, s>>>(
        static_cast<const T *>(Q), g, p.n_q_heads, p.n_kv_heads, p.np_cap, p.page_cap, k_pages, sh.kc, sh.kt,
        sh.chunk, idx.n_parents, idx.n_pages, static_cast<const T *>(idx.parent_keys), idx.parent_first_page,
        idx.parent_last_page, idx.parent_n_pages, idx.page_next, idx.page_len, static_cast<const T *>(idx.pool_k),
        static_cast<const T *>(idx.pool_v), sel_pages, sel_count, max_sel, static_cast<T *>(kbuf),
        static_cast<T *>(vbuf), buf_len, scale, O, pos_split(p).n_pos, err);
    return cudaGetLastError();
}

}  // namespace

bool decode_cluster_supported(const ice_params &p, int k_pages, int max_sel) {
    const Shape sh = shape_of(p, k_pages, max_sel);
    return sh.chunk <= 2048 && sh.kc <= 64 && sh.smem <= 200 * 1024;
}

cudaError_t launch_decode_cluster(const ice_params &p, const ice_index &idx, const void *Q, int k_pages,
                                  int32_t *sel_pages, int32_t *sel_count, int max_sel, void *kbuf, void *vbuf,
                                  int32_t *buf_len, float scale, float *O, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16)
        return launch_t<__nv_bfloat16>(p, idx, Q, k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale,
                                       O, err, s);
    return launch_t<float>(p, idx, Q, k_pages, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, scale, O, err, s);
}

}  // namespace ice
