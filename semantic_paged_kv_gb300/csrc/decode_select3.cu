// Decode steps a6-a8 with three index levels: page selection by descent.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 2: a query finds the k nearest points of the
// top level and continues the search among their children, level by level;
// 关键设计 3: every head selects its own pages and a GQA group shares the
// union.  With the lifted query q' = [q, 0] the nearest points are those of
// largest q.p.
//
// k_select3: one CTA per unit, one warp per query head (at least 4 warps).
//   1. score every level-2 node (a warp-wide dot product per node, the
//      unit's scores in the decode workspace);
//   2. its best k nodes in (-score, i) order: k rounds of a warp maximum
//      below the previous round's key;
//   3. their children, scored the same way, 32 at a time: each batch sorted
//      (bitonic, one key per lane) and merged into the running best 32;
//   4. the ordered best k parents give their pages (page-id order inside a
//      parent) until k pages, ORed into the union bitmask;
//   5. positional pages ORed in, then the ascending list (block scan).
#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ice {
namespace {

using namespace topk;

// q . row for a 128-dim row, lane holding q's dimensions 4 lane .. 4 lane + 3;
// every lane gets the sum.
template <typename T>
__device__ __forceinline__ float warp_dot(const float (&q)[4], const T *__restrict__ row, int lane) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) a = fmaf(q[i], Elem<T>::load(row + 4 * lane + i), a);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    return a;
}

// Descending bitonic sort of one key per lane.
__device__ __forceinline__ unsigned long long sort32_desc(unsigned long long v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool desc = (lane & size) == 0;
            const bool lower = (lane & stride) == 0;
            v = (lower == desc) ? umax64(v, o) : umin64(v, o);
        }
    }
    return v;
}

template <typename T>
__global__ void k_select3(const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, int np_cap, int page_cap,
                          int k_pages, int n_pos, const int32_t *__restrict__ n_pages,
                          const int32_t *__restrict__ n_nodes2, const int32_t *__restrict__ node2,
                          const int32_t *__restrict__ child_start, const int32_t *__restrict__ children,
                          const T *__restrict__ parent_keys, const int32_t *__restrict__ parent_first_page,
                          const int32_t *__restrict__ parent_last_page, const int32_t *__restrict__ parent_n_pages,
                          const int32_t *__restrict__ page_next, float *__restrict__ scores,
                          int32_t *__restrict__ sel_pages, int32_t *__restrict__ sel_count, int max_sel,
                          int32_t *__restrict__ err) {
    dep_wait();  // the index and Q are complete
    extern __shared__ unsigned s_mask[];  // union bitmask over the unit's pages
    __shared__ int s_wsum[32];
    const int u = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int nt = blockDim.x, nw = nt >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int P = min(n_pages[u], page_cap);
    const int Ps = max(0, P - n_pos);
    const int n2 = min(n_nodes2[u], np_cap);
    const int words = (P + 31) / 32;
    for (int x = threadIdx.x; x < words; x += nt) s_mask[x] = 0u;
    __syncthreads();
    for (int x = Ps + threadIdx.x; x < P; x += nt) atomicOr(&s_mask[x >> 5], 1u << (x & 31));
    const T *Pu = parent_keys + up * kHeadDim;
    for (int hh = warp; hh < g && Ps > 0; hh += nw) {
        float q[4];
        const T *qrow = Q + ((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim;
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = Elem<T>::load(qrow + 4 * lane + i);
        // 1. level-2 scores
        float *s2 = scores + ((size_t)u * g + hh) * np_cap;
        for (int i = 0; i < n2; ++i) {
            const float sc = warp_dot<T>(q, Pu + (size_t)node2[up + i] * kHeadDim, lane);
            if (lane == 0) s2[i] = sc;
        }
        __syncwarp();
        // 2. the best kc level-2 nodes: lane r gets the r-th best key
        const int kc = min(k_pages, n2);
        unsigned long long last = ~0ull, top = 0ull;
        for (int r = 0; r < kc; ++r) {
            unsigned long long best = 0ull;
            for (int i = lane; i < n2; i += 32) {
                const unsigned long long k = sort_key(s2[i], i);
                if (k < last && k > best) best = k;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
            if (lane == r) top = best;
            last = best;
        }
        // 3. their children, 32 at a time, merged into the running best 32
        unsigned long long run = 0ull;  // lane r: r-th best (score, -m) key so far
        unsigned long long batch = 0ull;
        int nb = 0;
        for (int r = 0; r < kc; ++r) {
            const int i = key_id(__shfl_sync(0xffffffffu, top, r));
            const int c0 = child_start[(size_t)u * (np_cap + 1) + i], c1 = child_start[(size_t)u * (np_cap + 1) + i + 1];
            for (int c = c0; c < c1; ++c) {
                const int m = children[up + c];
                const float sc = warp_dot<T>(q, Pu + (size_t)m * kHeadDim, lane);
                if (lane == nb) batch = sort_key(sc, m);
                if (++nb == 32) {
                    run = merge32(run, sort32_desc(batch));
                    batch = 0ull;
                    nb = 0;
                }
            }
        }
        if (nb > 0) run = merge32(run, sort32_desc(lane < nb ? batch : 0ull));
        // 4. pages of the ordered parents until k pages
        int pm = -1, fp = 0, pc = 0, contig = 1;
        if (lane < k_pages && run != 0ull) {
            pm = key_id(run);
            fp = parent_first_page[up + pm];
            pc = parent_n_pages[up + pm];
            contig = parent_last_page[up + pm] - fp + 1 == pc;
        }
        int incl = pc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        const int tk = max(0, min(pc, k_pages - (incl - pc)));
        int pg = fp;
        for (int t = 0; t < tk; ++t) {
            const int qq = contig ? fp + t : pg;
            if (qq < 0 || qq >= Ps) break;
            atomicOr(&s_mask[qq >> 5], 1u << (qq & 31));
            if (!contig) pg = page_next[ug + qq];
        }
    }
    __syncthreads();
    // 5. ascending list of the union's pages: thread t owns words [t wpt, (t + 1) wpt)
    const int wpt = (words + nt - 1) / nt;
    const int wb = threadIdx.x * wpt, we = min(words, wb + wpt);
    int c = 0;
    for (int x = wb; x < we; ++x) c += __popc(s_mask[x]);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int pos = incl - c, total = 0;
    for (int w = 0; w < nw; ++w) {
        pos += w < warp ? s_wsum[w] : 0;
        total += s_wsum[w];
    }
    for (int x = wb; x < we && pos < max_sel; ++x) {
        unsigned bb = s_mask[x];
        while (bb && pos < max_sel) {
            const int bit = __ffs(bb) - 1;
            bb &= bb - 1;
            sel_pages[(size_t)u * max_sel + pos++] = x * 32 + bit;
        }
    }
    for (int x = total + threadIdx.x; x < max_sel; x += nt) sel_pages[(size_t)u * max_sel + x] = -1;
    if (threadIdx.x == 0) {
        if (total > max_sel) set_err(err, ICE_ERR_CAPACITY);
        sel_count[u] = min(total, max_sel);
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws, int32_t *sel_pages,
                     int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const int nw = g < 4 ? 4 : g;
    const size_t smem = sizeof(unsigned) * (size_t)((p.page_cap + 31) / 32);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_select3<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_dependent(
        k_select3<T>, dim3(units_of(p)), dim3(32 * nw), smem, s, static_cast<const T *>(Q), g, p.n_q_heads,
        p.n_kv_heads, p.np_cap, p.page_cap, ws.k_pages, pos_split(p).n_pos, idx.n_pages, idx.n_nodes2, idx.node2,
        idx.child_start, idx.children, static_cast<const T *>(idx.parent_keys), idx.parent_first_page,
        idx.parent_last_page, idx.parent_n_pages, idx.page_next, ws.scores, sel_pages, sel_count, max_sel, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_select3(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                           int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
    return launch_t<float>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
}

}  // namespace ice
