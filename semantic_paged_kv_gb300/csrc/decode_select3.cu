// Decode steps a6-a8 with three index levels: page selection by descent.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 2: a query finds the k nearest points of the
// top level and continues the search among their children, level by level;
// 关键设计 3: every head selects its own pages and a GQA group shares the
// union.  With the lifted query q' = [q, 0] the nearest points are those of
// largest q.p.
//
// k_select3: one CTA per (query head, unit), 4 warps:
//   1. the head's score of every level-2 node (one thread per node row), in
//      shared memory (in the decode workspace for very large level-2 tables);
//   2. warp 0: the best k nodes in (-score, i) order, k rounds of a warp
//      maximum below the previous round's key;
//   3. their children spread over the 4 warps, one child per lane (each lane
//      loads its child's row), batches sorted (bitonic) and merged into each
//      warp's running best 32; the 4 lists merged by warp 0;
//   4. warp 0: the ordered best k parents' pages (page-id order inside a
//      parent) until k pages, written as the head's page list;
//   5. the unit's last CTA (atomic ticket) ORs the g lists and the
//      positional pages into a bitmask and writes the ascending union.
#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ice {
namespace {

using namespace topk;

constexpr size_t kS2Smem = 16 * 1024;  // shared memory for one head's level-2 scores

// q . row for a 128-dim key row and q in shared memory (fp32): the row is
// loaded in two halves, each half's 16-byte loads issued before its
// arithmetic.
template <typename T>
__device__ __forceinline__ float row_dot(const T *__restrict__ row, const float *__restrict__ q) {
    constexpr int PV = Elem<T>::kPerVec;
    constexpr int HV = row_vecs<T>() / 2;  // vectors per half row
    float a = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint4 r[HV];
#pragma unroll
        for (int v = 0; v < HV; ++v) r[v] = __ldg(reinterpret_cast<const uint4 *>(row) + half * HV + v);
#pragma unroll
        for (int v = 0; v < HV; ++v) {
            float f[PV];
            Elem<T>::unpack(r[v], f);
#pragma unroll
            for (int i = 0; i < PV; ++i) a = fmaf(f[i], q[(half * HV + v) * PV + i], a);
        }
    }
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

// 128 threads; bf16 rows leave registers for 5 CTAs per SM, fp32 rows for 3.
template <typename T>
__global__ void __launch_bounds__(128, sizeof(T) == 2 ? 5 : 3)
    k_select3(const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads,
                                                 int np_cap, int page_cap, int k_pages, int n_pos,
                                                 const int32_t *__restrict__ n_pages,
                                                 const int32_t *__restrict__ n_nodes2, const int32_t *__restrict__ node2,
                                                 const int32_t *__restrict__ child_start,
                                                 const int32_t *__restrict__ children,
                                                 const T *__restrict__ parent_keys,
                                                 const int32_t *__restrict__ parent_first_page,
                                                 const int32_t *__restrict__ parent_last_page,
                                                 const int32_t *__restrict__ parent_n_pages,
                                                 const int32_t *__restrict__ page_next, float *__restrict__ scores,
                                                 int32_t *__restrict__ head_pages, int32_t *__restrict__ ticket,
                                                 int32_t *__restrict__ sel_pages, int32_t *__restrict__ sel_count,
                                                 int max_sel, int s2_cap, int32_t *__restrict__ err) {
    dep_wait();  // the index and Q are complete
    constexpr int kW = 4, kT = 32 * kW;
    extern __shared__ float s_s2[];  // [s2_cap] this head's level-2 scores, then the union bitmask (last CTA)
    __shared__ float s_q[kHeadDim];
    __shared__ unsigned long long s_best[kW][32];
    __shared__ int s_g0[32], s_gn[32], s_gend[32], s_wsum[kW];
    __shared__ int s_last;
    const int hh = blockIdx.x, u = blockIdx.y;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int P = min(n_pages[u], page_cap);
    const int Ps = max(0, P - n_pos);
    const int n2 = min(n_nodes2[u], np_cap);
    const T *Pu = parent_keys + up * kHeadDim;
    int32_t *hl = head_pages + ((size_t)u * g + hh) * 32;  // this head's page list (-1 padded)
    for (int x = threadIdx.x; x < kHeadDim; x += kT)
        s_q[x] = Elem<T>::load(Q + ((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + x);
    __syncthreads();
    if (Ps > 0) {
        // 1. level-2 scores
        const bool in_smem = n2 <= s2_cap;
        float *su = in_smem ? s_s2 : scores + ((size_t)u * g + hh) * np_cap;
        for (int i = threadIdx.x; i < n2; i += kT) su[i] = row_dot<T>(Pu + (size_t)node2[up + i] * kHeadDim, s_q);
        __syncthreads();
        // 2. the best kc level-2 nodes and their child ranges
        const int kc = min(k_pages, n2);
        if (warp == 0) {
            unsigned long long last = ~0ull, top = 0ull;
            for (int r = 0; r < kc; ++r) {
                unsigned long long best = 0ull;
                for (int i = lane; i < n2; i += 32) {
                    const unsigned long long k = sort_key(su[i], i);
                    if (k < last && k > best) best = k;
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
                if (lane == r) top = best;
                last = best;
            }
            int g0 = 0, gn = 0;
            if (lane < kc) {
                const int i = key_id(top);
                g0 = child_start[(size_t)u * (np_cap + 1) + i];
                gn = child_start[(size_t)u * (np_cap + 1) + i + 1] - g0;
            }
            int gend = gn;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, gend, o);
                if (lane >= o) gend += x;
            }
            s_g0[lane] = g0;
            s_gn[lane] = gn;
            s_gend[lane] = gend;
        }
        __syncthreads();
        // 3. the children over the 4 warps, one per lane
        const int C = s_gend[31];
        unsigned long long run = 0ull;
        for (int c0 = warp * 32; c0 < C; c0 += kT) {
            const int c = c0 + lane;
            unsigned long long key = 0ull;
            if (c < C) {
                int lo = 0, hi = kc - 1;  // the first group whose inclusive end exceeds c
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (s_gend[mid] <= c) lo = mid + 1;
                    else hi = mid;
                }
                const int grp = lo;
                const int m = children[up + s_g0[grp] + (c - (s_gend[grp] - s_gn[grp]))];
                key = sort_key(row_dot<T>(Pu + (size_t)m * kHeadDim, s_q), m);
            }
            run = merge32(run, sort32_desc(key));
        }
        s_best[warp][lane] = run;
        __syncthreads();
        // 4. warp 0: the best parents of the 4 lists, then their pages
        if (warp == 0) {
            unsigned long long r = s_best[0][lane];
#pragma unroll
            for (int w = 1; w < kW; ++w) r = merge32(r, s_best[w][lane]);
            int fp = 0, pc = 0, contig = 1;
            if (lane < k_pages && r != 0ull) {
                const int pm = key_id(r);
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
            hl[lane] = -1;
            __syncwarp();
            int pg = fp;
            for (int t = 0; t < tk; ++t) {
                const int qq = contig ? fp + t : pg;
                if (qq < 0 || qq >= Ps) break;
                hl[incl - pc + t] = qq;
                if (!contig) pg = page_next[ug + qq];
            }
        }
    } else {
        for (int x = threadIdx.x; x < 32; x += kT) hl[x] = -1;
    }
    // 5. the unit's last CTA forms the union
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket + u, 1) == g - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    unsigned *s_mask = reinterpret_cast<unsigned *>(s_s2);
    const int words = (P + 31) / 32;
    for (int x = threadIdx.x; x < words; x += kT) s_mask[x] = 0u;
    __syncthreads();
    for (int x = Ps + threadIdx.x; x < P; x += kT) atomicOr(&s_mask[x >> 5], 1u << (x & 31));
    const int32_t *ul = head_pages + (size_t)u * g * 32;
    for (int x = threadIdx.x; x < g * 32; x += kT) {
        const int q = __ldcg(ul + x);
        if (q >= 0 && q < Ps) atomicOr(&s_mask[q >> 5], 1u << (q & 31));
    }
    __syncthreads();
    const int wpt = (words + kT - 1) / kT;
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
    for (int w = 0; w < kW; ++w) {
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
    for (int x = total + threadIdx.x; x < max_sel; x += kT) sel_pages[(size_t)u * max_sel + x] = -1;
    if (threadIdx.x == 0) {
        if (total > max_sel) set_err(err, ICE_ERR_CAPACITY);
        sel_count[u] = min(total, max_sel);
        ticket[u] = 0;  // every CTA of the unit has counted: ready for the next call
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws, int32_t *sel_pages,
                     int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const int s2_cap = (int)(kS2Smem / sizeof(float));
    const size_t mask = sizeof(unsigned) * (size_t)((p.page_cap + 31) / 32);
    const size_t smem = sizeof(float) * (size_t)s2_cap > mask ? sizeof(float) * (size_t)s2_cap : mask;
    if (smem > 200 * 1024) return cudaErrorNotSupported;
    {  // static shared memory comes on top: always opt in to the dynamic size
        cudaError_t e = cudaFuncSetAttribute(k_select3<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // the heads' page lists ([U, g, 32] int32) live in the candidate-key area of the workspace
    int32_t *head_pages = reinterpret_cast<int32_t *>(ws.cand_key);
    const cudaError_t e = launch_dependent(
        k_select3<T>, dim3(g, units_of(p)), dim3(128), smem, s, static_cast<const T *>(Q), g, p.n_q_heads,
        p.n_kv_heads, p.np_cap, p.page_cap, ws.k_pages, pos_split(p).n_pos, idx.n_pages, idx.n_nodes2, idx.node2,
        idx.child_start, idx.children, static_cast<const T *>(idx.parent_keys), idx.parent_first_page,
        idx.parent_last_page, idx.parent_n_pages, idx.page_next, ws.scores, head_pages, ws.sel_ticket, sel_pages,
        sel_count, max_sel, s2_cap, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_select3(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                           int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
    return launch_t<float>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
}

}  // namespace ice
