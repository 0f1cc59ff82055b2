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
//   1. every level-2 node scored against all g queries by one thread (its
//      row loaded once, the queries in shared memory), the scores in shared
//      memory (in the decode workspace for very large level-2 tables);
//   2. per head its best k nodes in (-score, i) order: k rounds of a warp
//      maximum below the previous round's key;
//   3. their children: the ids staged in shared memory (all loads in flight),
//      then one per lane (each lane loads its child's row), 32 at a time:
//      each batch sorted (bitonic, one key per lane) and merged into the
//      running best 32;
//   4. the ordered best k parents give their pages (page-id order inside a
//      parent) until k pages, ORed into the union bitmask;
//   5. positional pages ORed in, then the ascending list (block scan).
#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ice {
namespace {

using namespace topk;

constexpr int kCandPerWarp = 256;               // candidate parent ids a warp stages at a time
constexpr int kMaxCand = 16 * kCandPerWarp;     // for up to 16 warps
constexpr size_t kS2Smem = 16 * 1024;           // shared memory for the level-2 scores of all heads

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

template <typename T>
__global__ void __launch_bounds__(512) k_select3(const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, int np_cap, int page_cap,
                          int k_pages, int n_pos, const int32_t *__restrict__ n_pages,
                          const int32_t *__restrict__ n_nodes2, const int32_t *__restrict__ node2,
                          const int32_t *__restrict__ child_start, const int32_t *__restrict__ children,
                          const T *__restrict__ parent_keys, const int32_t *__restrict__ parent_first_page,
                          const int32_t *__restrict__ parent_last_page, const int32_t *__restrict__ parent_n_pages,
                          const int32_t *__restrict__ page_next, float *__restrict__ scores,
                          int32_t *__restrict__ sel_pages, int32_t *__restrict__ sel_count, int max_sel,
                          int s2_cap, int32_t *__restrict__ err) {
    dep_wait();  // the index and Q are complete
    extern __shared__ float s_q[];  // [g][128] the group's queries (fp32), then [g][s2_cap] level-2 scores
    float *s_s2 = s_q + g * kHeadDim;
    unsigned *s_mask = reinterpret_cast<unsigned *>(s_s2 + (size_t)g * s2_cap);  // union bitmask over the unit's pages
    __shared__ int s_cand[kMaxCand];  // [kMaxCand] one head's candidate parents at a time (warp-private slices)
    __shared__ int s_wsum[32];
    __shared__ int s_g0[16][32], s_gn[16][32], s_gend[16][32];  // per warp: the chosen level-2 groups
    const int u = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int nt = blockDim.x, nw = nt >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int P = min(n_pages[u], page_cap);
    const int Ps = max(0, P - n_pos);
    const int n2 = min(n_nodes2[u], np_cap);
    const int words = (P + 31) / 32;
    const T *Pu = parent_keys + up * kHeadDim;
    for (int x = threadIdx.x; x < words; x += nt) s_mask[x] = 0u;
    for (int x = threadIdx.x; x < g * kHeadDim; x += nt)
        s_q[x] = Elem<T>::load(Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim + x);
    __syncthreads();
    for (int x = Ps + threadIdx.x; x < P; x += nt) atomicOr(&s_mask[x >> 5], 1u << (x & 31));
    // 1. level-2 scores of every head: a thread per level-2 node, its row loaded once
    // the scores live in shared memory when the unit's level-2 table fits, else in the workspace
    const bool in_smem = n2 <= s2_cap;
    float *su = in_smem ? s_s2 : scores + (size_t)u * g * np_cap;
    const int ld2 = in_smem ? s2_cap : np_cap;
    for (int i = threadIdx.x; i < n2 && Ps > 0; i += nt) {
        const T *row = Pu + (size_t)node2[up + i] * kHeadDim;
        float acc[16];
#pragma unroll
        for (int hh = 0; hh < 16; ++hh) acc[hh] = 0.f;
        constexpr int PV = Elem<T>::kPerVec;
        constexpr int HV = row_vecs<T>() / 2;
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // each half row loaded once for all heads
            uint4 r[HV];
#pragma unroll
            for (int v = 0; v < HV; ++v) r[v] = __ldg(reinterpret_cast<const uint4 *>(row) + half * HV + v);
#pragma unroll
            for (int v = 0; v < HV; ++v) {
                float f[PV];
                Elem<T>::unpack(r[v], f);
#pragma unroll
                for (int hh = 0; hh < 16; ++hh) {
                    if (hh < g) {
                        const float *qh = s_q + hh * kHeadDim + (half * HV + v) * PV;
#pragma unroll
                        for (int e = 0; e < PV; ++e) acc[hh] = fmaf(f[e], qh[e], acc[hh]);
                    }
                }
            }
        }
#pragma unroll
        for (int hh = 0; hh < 16; ++hh)
            if (hh < g) su[(size_t)hh * ld2 + i] = acc[hh];
    }
    __syncthreads();  // the block's score writes are visible to the whole block
    for (int hh = warp; hh < g && Ps > 0; hh += nw) {
        const float *qh = s_q + hh * kHeadDim;
        const float *s2 = su + (size_t)hh * ld2;
        // 2. the best kc level-2 nodes: lane r gets the r-th best (score, -i) key
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
        // 3. their children: lane r < kc holds group r's range; candidates go
        //    32 at a time, one per lane, each lane loading its child's row
        int g0 = 0, gn = 0;
        if (lane < kc) {
            const int i = key_id(top);
            g0 = child_start[(size_t)u * (np_cap + 1) + i];
            gn = child_start[(size_t)u * (np_cap + 1) + i + 1] - g0;
        }
        int gend = gn;  // inclusive scan of the group sizes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, gend, o);
            if (lane >= o) gend += x;
        }
        const int C = __shfl_sync(0xffffffffu, gend, 31);
        s_g0[warp][lane] = g0;
        s_gn[warp][lane] = gn;
        s_gend[warp][lane] = gend;
        __syncwarp();
        unsigned long long run = 0ull;  // lane r: r-th best (score, -m) parent so far
        int *cand = s_cand + (size_t)warp * kCandPerWarp;
        for (int c0 = 0; c0 < C; c0 += kCandPerWarp) {
            const int cn = min(kCandPerWarp, C - c0);
            // the slice's candidate ids, all loads in flight at once
            for (int x = lane; x < cn; x += 32) {
                const int c = c0 + x;
                int grp = 0;
                for (int j = 0; j < kc; ++j) grp += (j < 32 ? s_gend[warp][j] : 0) <= c;
                cand[x] = children[up + s_g0[warp][grp] + (c - (s_gend[warp][grp] - s_gn[warp][grp]))];
            }
            __syncwarp();
            for (int x0 = 0; x0 < cn; x0 += 32) {
                unsigned long long key = 0ull;
                if (x0 + lane < cn) {
                    const int m = cand[x0 + lane];
                    key = sort_key(row_dot<T>(Pu + (size_t)m * kHeadDim, qh), m);
                }
                run = merge32(run, sort32_desc(key));
            }
            __syncwarp();
        }
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
    const int s2_cap = (int)(kS2Smem / sizeof(float) / g);
    const size_t smem = sizeof(float) * (size_t)g * (kHeadDim + s2_cap) + sizeof(unsigned) * (size_t)((p.page_cap + 31) / 32);
    {  // static shared memory comes on top: always opt in to the dynamic size
        cudaError_t e = cudaFuncSetAttribute(k_select3<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_dependent(
        k_select3<T>, dim3(units_of(p)), dim3(32 * nw), smem, s, static_cast<const T *>(Q), g, p.n_q_heads,
        p.n_kv_heads, p.np_cap, p.page_cap, ws.k_pages, pos_split(p).n_pos, idx.n_pages, idx.n_nodes2, idx.node2,
        idx.child_start, idx.children, static_cast<const T *>(idx.parent_keys), idx.parent_first_page,
        idx.parent_last_page, idx.parent_n_pages, idx.page_next, ws.scores, sel_pages, sel_count, max_sel, s2_cap, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_select3(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                           int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
    return launch_t<float>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
}

}  // namespace ice
