// Step a11: incremental insert of one new token per unit.
//
// IceCache popular-science article (aitangshan.cn/news/751385), section 三:
// a newly generated token is placed without rebuilding the tree: the same
// random promotion decides its level, and it is attached to the most similar
// parent of the level above.  papernotes.org "IceCache: Memory-Efficient
// KV-cache Management for Long-Sequence LLMs", 关键设计 2: new tokens are
// inserted into a suitable node, and a node that outgrows the page size
// splits off a new page.
//
// Rule (per unit, position pos = n_indexed): lift with the build-time M^2,
// e = sqrt(max(0, M^2 - |k|^2)).  If the level-1 draw of pos is below the
// threshold (or the unit has no parent), the token becomes parent Np with a
// page of its own.  Otherwise its parent is
//   argmin_m |k' - p'_m|^2 = argmax_m (k.p_m + e e_m + c_m),
// c_m = (M^2 - max(M^2, |p_m|^2)) / 2 (zero for build-time parents; it keeps
// the distance exact for parents inserted with |p|^2 > M^2), lowest m on
// exact ties; the token goes to that parent's last page if it holds fewer
// than S tokens, else to a new page linked after it.  Existing tokens never
// move.
//
// One launch, grid (chunks of 256 parents, units): each CTA scores its
// chunk against the new key (fp32 FMA) and writes its best (score, m); the
// unit's last CTA (atomic ticket, reset to zero at the end) takes the argmax
// over the chunks and applies the insert to the index tables and the pool.
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ void block_best(float &s, int &i, float *sh_s, int *sh_i) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, s, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        if (better(os, oi, s, i)) {
            s = os;
            i = oi;
        }
    }
    if (lane == 0) {
        sh_s[warp] = s;
        sh_i[warp] = i;
    }
    __syncthreads();
    s = sh_s[0];
    i = sh_i[0];
    for (int w = 1; w < kWarps; ++w)
        if (better(sh_s[w], sh_i[w], s, i)) {
            s = sh_s[w];
            i = sh_i[w];
        }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_insert(
    const T *__restrict__ k_new, const T *__restrict__ v_new, int n_kv_heads, int np_cap, int page_cap, int n_cap,
    uint64_t thresh, uint64_t key, int n_chunks, int32_t *__restrict__ n_parents, int32_t *__restrict__ n_pages,
    int32_t *__restrict__ n_indexed, const double *__restrict__ m2, int32_t *__restrict__ parent_tok,
    T *__restrict__ parent_keys, float *__restrict__ parent_e, float *__restrict__ parent_corr,
    int32_t *__restrict__ parent_first_page, int32_t *__restrict__ parent_last_page,
    int32_t *__restrict__ parent_n_pages, int32_t *__restrict__ page_parent, int32_t *__restrict__ page_len,
    int32_t *__restrict__ page_next, int32_t *__restrict__ page_tokens, int32_t *__restrict__ token_parent,
    int32_t *__restrict__ token_page, int32_t *__restrict__ token_slot, T *__restrict__ pool_k,
    T *__restrict__ pool_v, float *__restrict__ best_s, int32_t *__restrict__ best_m, int32_t *__restrict__ ticket,
    int32_t *__restrict__ err) {
    __shared__ __align__(16) float s_k[kHeadDim];
    __shared__ float sh_s[kWarps];
    __shared__ int sh_i[kWarps];
    __shared__ double s_n;
    __shared__ int s_last;
    const int u = blockIdx.y, chunk = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T *ku = k_new + (size_t)u * kHeadDim;
    if (threadIdx.x < kHeadDim) s_k[threadIdx.x] = Elem<T>::load(ku + threadIdx.x);
    const int Np = min(n_parents[u], np_cap);
    const double M2 = m2[u];
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap, un = (size_t)u * n_cap;
    __syncthreads();
    if (warp == 0) {  // |k|^2 with double-float accumulation (4 elements per lane)
        float hi = 0.f, lo = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float f = s_k[lane * 4 + i];
            const float t = f * f, te = fmaf(f, f, -t);
            float sum, e;
            two_sum(hi, t, sum, e);
            hi = sum;
            lo += e + te;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ohi = __shfl_xor_sync(0xffffffffu, hi, off);
            const float olo = __shfl_xor_sync(0xffffffffu, lo, off);
            float sum, e;
            two_sum(hi, ohi, sum, e);
            hi = sum;
            lo += olo + e;
        }
        if (lane == 0) s_n = (double)hi + (double)lo;
    }
    __syncthreads();
    const double nk = s_n;
    const double r = M2 - nk;
    const float ek = (float)sqrt(r > 0.0 ? r : 0.0);

    // ---- score this chunk's parents
    const int m = chunk * kSelChunk + threadIdx.x;
    float sc = -INFINITY;
    int mi = 0x7fffffff;
    if (m < Np) {
        const uint4 *row = reinterpret_cast<const uint4 *>(parent_keys + (up + m) * kHeadDim);
        constexpr int RV = row_vecs<T>();
        constexpr int PV = Elem<T>::kPerVec;
        float acc = 0.f;
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
                for (int e = 0; e < PV; ++e) acc = fmaf(s_k[(v0 + i) * PV + e], f[e], acc);
            }
        }
        sc = fmaf(ek, parent_e[up + m], acc) + parent_corr[up + m];
        mi = m;
    }
    block_best(sc, mi, sh_s, sh_i);
    if (threadIdx.x == 0) {
        best_s[(size_t)u * n_chunks + chunk] = sc;
        best_m[(size_t)u * n_chunks + chunk] = mi;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(ticket + u, 1) == n_chunks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- the unit's last CTA: argmax over chunks, then the insert itself
    sc = -INFINITY;
    mi = 0x7fffffff;
    for (int c = threadIdx.x; c < n_chunks; c += kThreads) {
        const float s2 = __ldcg(best_s + (size_t)u * n_chunks + c);
        const int m2i = __ldcg(best_m + (size_t)u * n_chunks + c);
        if (better(s2, m2i, sc, mi)) {
            sc = s2;
            mi = m2i;
        }
    }
    block_best(sc, mi, sh_s, sh_i);
    __shared__ int s_page, s_slot, s_parent, s_ok, s_newpage, s_pos;
    if (threadIdx.x == 0) {
        const int pos = n_indexed[u];
        const int P = min(n_pages[u], page_cap);
        const int seq = u / n_kv_heads, head = u % n_kv_heads;
        int ok = 1, par = -1, page = -1, slot = 0, newpage = 0;
        if (pos >= n_cap) {
            ok = 0;
        } else {
            const bool promote = Np == 0 || (uint64_t)promote_draw(key, seq, head, (uint32_t)pos, 1u) < thresh;
            if (promote) {
                if (Np >= np_cap || P >= page_cap) {
                    ok = 0;
                } else {
                    par = Np;
                    parent_tok[up + par] = pos;
                    parent_e[up + par] = ek;
                    parent_corr[up + par] = (float)(0.5 * (M2 - (nk > M2 ? nk : M2)));
                    parent_first_page[up + par] = P;
                    parent_last_page[up + par] = P;
                    parent_n_pages[up + par] = 1;
                    n_parents[u] = Np + 1;
                    page = P;
                    newpage = 1;
                }
            } else {
                par = mi;
                const int last = parent_last_page[up + par];
                if (page_len[ug + last] < kPage) {
                    page = last;
                    slot = page_len[ug + last];
                    page_len[ug + last] = slot + 1;
                } else if (P >= page_cap) {
                    ok = 0;
                } else {
                    page = P;
                    newpage = 1;
                    page_next[ug + last] = P;
                    parent_last_page[up + par] = P;
                    parent_n_pages[up + par] += 1;
                }
            }
            if (ok && newpage) {
                page_parent[ug + page] = par;
                page_len[ug + page] = 1;
                page_next[ug + page] = -1;
                n_pages[u] = P + 1;
            }
            if (ok) {
                page_tokens[(ug + page) * kPage + slot] = pos;
                token_parent[un + pos] = par;
                token_page[un + pos] = page;
                token_slot[un + pos] = slot;
                n_indexed[u] = pos + 1;
            }
        }
        if (!ok) set_err(err, ICE_ERR_CAPACITY);
        s_ok = ok;
        s_page = page;
        s_slot = slot;
        s_parent = par;
        s_newpage = newpage;
        s_pos = pos;
        ticket[u] = 0;  // ready for the next call
    }
    __syncthreads();
    if (!s_ok) return;
    constexpr int RV = row_vecs<T>();
    const uint4 *k4 = reinterpret_cast<const uint4 *>(ku);
    const uint4 *v4 = reinterpret_cast<const uint4 *>(v_new + (size_t)u * kHeadDim);
    uint4 *pk = reinterpret_cast<uint4 *>(pool_k) + (ug + s_page) * kPage * RV;
    uint4 *pv = reinterpret_cast<uint4 *>(pool_v) + (ug + s_page) * kPage * RV;
    if (s_newpage) {  // a new page: the token in slot 0, zero pad slots
        for (int x = threadIdx.x; x < kPage * RV; x += kThreads) {
            const int sl = x / RV;
            pk[x] = sl == 0 ? k4[x] : make_uint4(0, 0, 0, 0);
            pv[x] = sl == 0 ? v4[x] : make_uint4(0, 0, 0, 0);
        }
        for (int sl = 1 + threadIdx.x; sl < kPage; sl += kThreads) page_tokens[(ug + s_page) * kPage + sl] = -1;
    } else {
        for (int x = threadIdx.x; x < RV; x += kThreads) {
            pk[s_slot * RV + x] = k4[x];
            pv[s_slot * RV + x] = v4[x];
        }
    }
    if (s_parent == Np && s_newpage && s_page >= 0 && Np < np_cap) {  // promoted: its key joins the parent table
        uint4 *dst = reinterpret_cast<uint4 *>(parent_keys + (up + s_parent) * kHeadDim);
        for (int x = threadIdx.x; x < RV; x += kThreads) dst[x] = k4[x];
    }
    (void)s_pos;
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const void *k_new, const void *v_new,
                     const InsertWs &ws, int32_t *err, cudaStream_t s) {
    dim3 grid(ws.n_chunks, units_of(p));
    k_insert<T><<<grid, kThreads, 0, s>>>(
        static_cast<const T *>(k_new), static_cast<const T *>(v_new), p.n_kv_heads, p.np_cap, p.page_cap, p.n_cap,
        p.promote_thresh, promote_key(p.seed, p.layer), ws.n_chunks, idx.n_parents, idx.n_pages, idx.n_indexed,
        idx.m2, idx.parent_tok, static_cast<T *>(idx.parent_keys), idx.parent_e, idx.parent_corr,
        idx.parent_first_page, idx.parent_last_page, idx.parent_n_pages, idx.page_parent, idx.page_len,
        idx.page_next, idx.page_tokens, idx.token_parent, idx.token_page, idx.token_slot,
        static_cast<T *>(idx.pool_k), static_cast<T *>(idx.pool_v), ws.best_s, ws.best_m, ws.ticket, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_insert(const ice_params &p, const ice_index &idx, const void *k_new, const void *v_new,
                          const InsertWs &ws, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, idx, k_new, v_new, ws, err, s);
    return launch_t<float>(p, idx, k_new, v_new, ws, err, s);
}

}  // namespace ice
