// Decode steps a6-a8 with three index levels: page selection by descent.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 2: a query finds the k nearest points of the
// top level and continues the search among their children, level by level;
// 关键设计 3: every head selects its own pages and a GQA group shares the
// union.  With the lifted query q' = [q, 0] the nearest points are those of
// largest q.p.
//
// k_descent: one CTA per unit, one warp per query head (heads h, h + NW, ...
// when g > NW warps):
//   1. the unit's level-2 rows (their parents' keys) streamed into a
//      three-slot shared-memory ring in 16-byte asynchronous copies spread
//      over the block (R rows a slot, padded so that the rows read without
//      bank conflicts; the row ids loaded beforehand) and scored against
//      every head's query: mma.sync m16n8k16 with the queries as A and 8
//      staged rows as B (bf16), on the CUDA cores for fp32 -> the
//      level-2 scores [g][n2] (shared memory, or the decode workspace);
//   2. warp per head: its best kc = min(k, n2) level-2 nodes in (-q.p, i)
//      order (the kc-th largest score by a radix search, the keys reaching
//      it ranked by counting); the children ranges of those nodes form the
//      head's candidate list;
//   3. every head's candidates (head by head, node by node) through the same
//      ring, each row scored for its head -> the key (q.p, m) of the
//      candidate (shared memory, or the score in the workspace);
//   4. warp per head: the ordered best k parents among its candidates (as in
//      2), their pages (page-id order inside a parent) until k pages, ORed
//      into the union bitmask, where the positional pages already are;
//   5. the block writes the ascending union (one scan).
// Each unit's level-2 table is read once for all heads, each candidate row
// once per head that reaches it.
#include "attn_page.cuh"
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "topk_common.cuh"

namespace ice {
namespace {

using namespace tc;
using namespace topk;

template <typename T> constexpr int stage_rows() { return sizeof(T) == 2 ? 128 : 64; }  // rows per ring slot
template <typename T> constexpr int stage_stride() { return row_bytes<T>() + 16; }       // padded row
constexpr int kSlots = 3;  // ring slots: two batches in flight while one is scored
constexpr int kTopkSlack = 16;  // keys past the k-th that the warp top-k may rank

// The largest index j in [0, n) with a[j] <= x (a non-decreasing, a[0] <= x).
__device__ __forceinline__ int last_le(const int *a, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// 16-byte asynchronous copy global -> shared (the load path, not the copy
// engine: many small rows), and its commit / wait.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Streams the rows of entries 0..n-1 through the kSlots ring slots, R entries
// a batch, kSlots - 1 batches ahead of the one being used; each row is copied
// in 16-byte pieces spread over the block.  row_of(e) gives entry e's row
// address; use(bt, rows, base) consumes batch bt (rows entries from bt * R)
// in shared memory at base (called by every thread).  slot: the ring's next
// slot, carried from call to call.
template <typename T, int NT, typename RowOf, typename Use>
__device__ void stream_rows(int n, unsigned char *ring, int &slot, RowOf row_of, Use use) {
    constexpr int R = stage_rows<T>(), SB = stage_stride<T>(), RV = row_bytes<T>() / 16;
    const int tid = threadIdx.x;
    const int nb = (n + R - 1) / R;
    if (nb == 0) return;
    auto slot_of = [&](int bt) { return (slot + bt) % kSlots; };
    auto issue = [&](int bt) {  // one commit group per batch and thread (empty past the end)
        if (bt < nb) {
            unsigned char *base = ring + (size_t)slot_of(bt) * R * SB;
            const int rows = min(R, n - bt * R);
            for (int i = tid; i < rows * RV; i += NT) {
                const int r = i / RV, c = i - r * RV;
                cp_async16(base + (size_t)r * SB + c * 16, reinterpret_cast<const unsigned char *>(row_of(bt * R + r)) + c * 16);
            }
        }
        cp_async_commit();
    };
    for (int pb = 0; pb < kSlots - 1; ++pb) issue(pb);
    for (int bt = 0; bt < nb; ++bt) {
        issue(bt + kSlots - 1);          // into the slot batch bt - 1 used (released by the barrier below)
        cp_async_wait<kSlots - 1>();     // this thread's pieces of batch bt have landed
        __syncthreads();                 // ... and every other thread's
        use(bt, min(R, n - bt * R), ring + (size_t)slot_of(bt) * R * SB);
        __syncthreads();
    }
    cp_async_wait<0>();  // the empty trailing groups
    slot = slot_of(nb);
}

// Lane r < kc (kc <= 32) receives the r-th largest of the n keys key_of(i),
// i < n (distinct; 0 = none); n <= 32 V.  A bound on the high words (the
// scores) that the best kc reach and at most kc + kTopkSlack keys reach unless
// ties force more (kth_bound_ord: a radix search that stops as soon as the
// count is that small) selects the keys that are ranked by counting (at most
// 64, else k rounds of a warp maximum).  s_tmp: 64 keys of this warp's scratch.
template <int V, typename KeyOf>
__device__ unsigned long long warp_topk(int n, int kc, KeyOf key_of, unsigned long long *s_tmp) {
    const int lane = threadIdx.x & 31;
    unsigned long long k[V];
    uint32_t v[V];
#pragma unroll
    for (int e = 0; e < V; ++e) {
        const int i = e * 32 + lane;
        k[e] = i < n ? key_of(i) : 0ull;
        v[e] = (uint32_t)(k[e] >> 32);
    }
    const uint32_t t = kc < n ? kth_bound_ord<V>(v, kc, kTopkSlack) : 1u;
    unsigned pass = 0u;
#pragma unroll
    for (int e = 0; e < V; ++e) pass |= (k[e] != 0ull && v[e] >= t ? 1u : 0u) << e;
    const int c = __popc(pass);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    unsigned long long top = 0ull;
    if (total <= 64) {
        int at = incl - c;
#pragma unroll
        for (int e = 0; e < V; ++e)
            if ((pass >> e) & 1u) s_tmp[at++] = k[e];
        __syncwarp();
        unsigned long long mine[2] = {lane < total ? s_tmp[lane] : 0ull, lane + 32 < total ? s_tmp[lane + 32] : 0ull};
        int rank[2] = {0, 0};
        for (int j = 0; j < total; ++j) {
            const unsigned long long o = s_tmp[j];
            rank[0] += o > mine[0];
            rank[1] += o > mine[1];
        }
        __syncwarp();
#pragma unroll
        for (int x = 0; x < 2; ++x)
            if (mine[x] != 0ull && rank[x] < 32) s_tmp[rank[x]] = mine[x];
        __syncwarp();
        top = lane < kc && lane < total ? s_tmp[lane] : 0ull;
        __syncwarp();
    } else {  // very many ties at the bound
        unsigned long long last = ~0ull;
        for (int r = 0; r < kc; ++r) {
            unsigned long long best = 0ull;
#pragma unroll
            for (int e = 0; e < V; ++e) best = k[e] < last && k[e] > best ? k[e] : best;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
            if (lane == r) top = best;
            last = best;
        }
    }
    return top;
}

// Lanes of the TPR-thread group of this lane (consecutive lanes share a row).
template <int TPR> __device__ __forceinline__ unsigned group_mask() {
    const unsigned lane = threadIdx.x & 31u;
    return TPR >= 32 ? 0xffffffffu : (((1u << TPR) - 1u) << (lane & ~(unsigned)(TPR - 1)));
}
template <int TPR> __device__ __forceinline__ float group_sum(float v, unsigned mask) {
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) v += __shfl_xor_sync(mask, v, o);
    return v;
}

// The 8 elements at `off` of a staged row, as fp32.
template <typename T>
__device__ __forceinline__ void load_chunk(const unsigned char *row, int off, float (&f)[8]) {
    constexpr int PV = Elem<T>::kPerVec;
#pragma unroll
    for (int v = 0; v < 8 / PV; ++v) {
        float x[PV];
        Elem<T>::unpack(*reinterpret_cast<const uint4 *>(row + (size_t)(off + v * PV) * sizeof(T)), x);
#pragma unroll
        for (int i = 0; i < PV; ++i) f[v * PV + i] = x[i];
    }
}

// The scores of a batch of staged bf16 rows against the group's queries on
// the tensor cores: warp w takes the 8-row tiles w, w + NW, ...; mma.sync
// m16n8k16 with A = the queries (rows = heads; 8 or 16), B = 8 staged rows
// by ldmatrix (the padded rows read without bank conflicts).  out(j, head,
// score) for every row j < rows and head < g.
template <int NW, int HR, typename Out>
__device__ __forceinline__ void score_rows_mma(const uint32_t (&qa)[8][4], const unsigned char *base, int rows, int g,
                                               Out out) {
    constexpr int SB = stage_stride<__nv_bfloat16>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, qr = lane >> 2, qc = lane & 3;
    const uint32_t b0 = su32(base);
    for (int nt = warp; nt * 8 < rows; nt += NW) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
            // matrices: rows 8nt..8nt+7 x 16-byte chunks 2kk .. 2kk + 3
            const uint32_t addr = b0 + (uint32_t)((8 * nt + (lane & 7)) * SB + (2 * kk + (lane >> 3)) * 16);
            uint32_t r0, r1, r2, r3;
            mma::ldsm_x4(addr, r0, r1, r2, r3);
            mma::mma16816(acc, qa[kk], r0, r1);
            mma::mma16816(acc, qa[kk + 1], r2, r3);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int j = 8 * nt + 2 * qc + c;
            if (j < rows) {
                if (qr < g) out(j, qr, acc[c]);
                if (HR > 1 && qr + 8 < g) out(j, qr + 8, acc[2 + c]);
            }
        }
    }
}

// The same on the CUDA cores (fp32 rows): TPR threads share a row; heads(j)
// gives the row's heads [lo, hi).
template <typename T, int NT, typename Heads, typename Out>
__device__ __forceinline__ void score_rows_simt(const float *s_q, const unsigned char *base, int rows, Heads heads,
                                                Out out) {
    constexpr int R = stage_rows<T>(), SB = stage_stride<T>();
    constexpr int TPR = NT / R, DPT = kHeadDim / TPR;
    static_assert(TPR >= 1 && NT % R == 0, "threads per row");
    const int j = threadIdx.x / TPR, d0 = (threadIdx.x % TPR) * DPT;
    if (j >= rows) return;  // uniform over the row's thread group
    const unsigned gm = group_mask<TPR>();
    const unsigned char *row = base + (size_t)j * SB;
    int lo, hi;
    heads(j, lo, hi);
    for (int h0 = lo; h0 < hi; h0 += 8) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = 0.f;
#pragma unroll 1
        for (int off = d0; off < d0 + DPT; off += 8) {
            float f[8];
            load_chunk<T>(row, off, f);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (h0 + i < hi) {
                    const float *q = s_q + (size_t)(h0 + i) * kHeadDim + off;
#pragma unroll
                    for (int x = 0; x < 8; ++x) a[i] = fmaf(f[x], q[x], a[i]);
                }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float v = group_sum<TPR>(a[i], gm);
            if (threadIdx.x % TPR == 0 && h0 + i < hi) out(j, h0 + i, v);
        }
    }
}

// One CTA per unit, NW warps.  HR: query rows of the tensor-core scoring
// (1: g <= 8, 2: g <= 16; bf16), 0: scoring on the CUDA cores (fp32).  cap2 / capc:
// level-2 scores and candidate keys kept in shared memory per head; larger
// tables go through ws_scores.
template <typename T, int NW, int HR>
__global__ void __launch_bounds__(32 * NW, 1)
    k_descent(const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, int np_cap, int page_cap, int k_pages,
              int n_pos, const int32_t *__restrict__ n_pages, const int32_t *__restrict__ n_nodes2,
              const int32_t *__restrict__ node2, const int32_t *__restrict__ child_start,
              const int32_t *__restrict__ children, const T *__restrict__ parent_keys,
              const int32_t *__restrict__ parent_first_page, const int32_t *__restrict__ parent_last_page,
              const int32_t *__restrict__ parent_n_pages, const int32_t *__restrict__ page_next,
              float *__restrict__ ws_scores, int32_t *__restrict__ sel_pages, int32_t *__restrict__ sel_count,
              int max_sel, int cap2, int capc, int32_t *__restrict__ err) {
    constexpr int NT = 32 * NW;
    constexpr int R = stage_rows<T>(), SB = stage_stride<T>();
    constexpr int V = 16;  // keys a lane of the warp top-k (up to 512)
    dep_wait();  // the index and Q are complete
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;                                                     // [kSlots][R][SB] staged rows
    float *s_q = reinterpret_cast<float *>(ring + (size_t)kSlots * R * SB);         // [g][d] the queries
    auto *s_ck = reinterpret_cast<unsigned long long *>(s_q + (size_t)g * kHeadDim);  // [g][capc] candidate keys
    float *s_s2 = reinterpret_cast<float *>(s_ck + (size_t)g * capc);               // [g][cap2] level-2 scores
    int *s_c0 = reinterpret_cast<int *>(s_s2 + (size_t)g * cap2);  // [g][32] children offset of the head's node r
    int *s_cst = s_c0 + g * 32;    // [g][33] first candidate of node r; [32]: the head's candidate count
    int *s_hoff = s_cst + g * 33;  // [g + 1] first entry of each head's candidates
    unsigned *s_mask = reinterpret_cast<unsigned *>(s_hoff + g + 1);  // the union bitmask
    // row ids of the streamed entries, in whichever area is idle: level-2
    // node parents in the candidate keys' area, candidates in the level-2 scores'
    int *ids1 = reinterpret_cast<int *>(s_ck);
    int *ids3 = reinterpret_cast<int *>(s_s2);
    __shared__ unsigned long long s_tmp[NW][64];  // per warp: the top-k's candidates
    __shared__ int s_wsum[NW];

    const int u = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int P = min(n_pages[u], page_cap), Ps = max(0, P - n_pos);
    const int n2 = Ps > 0 ? min(n_nodes2[u], np_cap) : 0;
    const int kc2 = min(k_pages, n2);
    const int words = (P + 31) / 32;
    const T *Pu = parent_keys + up * kHeadDim;
    const T *Qg = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
    float *wsu = ws_scores + (size_t)u * g * np_cap;  // [g][np_cap]: the scores that do not fit shared memory
    const bool s2_in = n2 <= cap2;
    const bool ids1_in = n2 <= 2 * g * capc;

    uint32_t qa[8][4];  // the queries as the A fragment of the tensor-core scoring
    if constexpr (HR > 0) mma::load_q_frag<HR>(reinterpret_cast<const __nv_bfloat16 *>(Qg), g, qa);
    for (int x = tid; x < g * kHeadDim; x += NT) s_q[x] = Elem<T>::load(Qg + x);
    for (int x = tid; x < words; x += NT) s_mask[x] = 0u;
    if (ids1_in)
        for (int e = tid; e < n2; e += NT) ids1[e] = __ldg(node2 + up + e);
    __syncthreads();
    for (int x = Ps + tid; x < P; x += NT) atomicOr(&s_mask[x >> 5], 1u << (x & 31));  // positional pages
    int slot = 0;

    // 1. the level-2 scores of every head
    auto put2 = [&](int e, int hh, float v) {
        if (s2_in) s_s2[(size_t)hh * cap2 + e] = v;
        else wsu[(size_t)hh * np_cap + e] = v;
    };
    stream_rows<T, NT>(
        n2, ring, slot, [&](int e) { return Pu + (size_t)(ids1_in ? ids1[e] : __ldg(node2 + up + e)) * kHeadDim; },
        [&](int bt, int rows, const unsigned char *base) {
            const int e0 = bt * R;
            if constexpr (HR > 0)
                score_rows_mma<NW, HR>(qa, base, rows, g, [&](int j, int hh, float v) { put2(e0 + j, hh, v); });
            else
                score_rows_simt<T, NT>(
                    s_q, base, rows, [&](int, int &lo, int &hi) { lo = 0, hi = g; },
                    [&](int j, int hh, float v) { put2(e0 + j, hh, v); });
        });

    // 2. per head: its best kc2 level-2 nodes, in (-q.p, i) order, and their children ranges
    for (int hh = warp; hh < g; hh += NW) {
        const float *sc = s2_in ? s_s2 + (size_t)hh * cap2 : wsu + (size_t)hh * np_cap;
        unsigned long long top = 0ull;
        if (n2 <= 32 * V) {
            top = warp_topk<V>(n2, kc2, [&](int i) { return sort_key(sc[i], i); }, s_tmp[warp]);
        } else {  // k rounds of a warp maximum
            unsigned long long last = ~0ull;
            for (int r = 0; r < kc2; ++r) {
                unsigned long long best = 0ull;
                for (int i = lane; i < n2; i += 32) {
                    const unsigned long long k = sort_key(sc[i], i);
                    if (k < last && k > best) best = k;
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
                if (lane == r) top = best;
                last = best;
            }
        }
        int c0 = 0, cnt = 0;
        if (lane < kc2) {
            const int i = key_id(top);
            c0 = __ldg(child_start + (size_t)u * (np_cap + 1) + i);
            cnt = __ldg(child_start + (size_t)u * (np_cap + 1) + i + 1) - c0;
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        s_c0[hh * 32 + lane] = c0;
        s_cst[hh * 33 + lane] = incl - cnt;
        if (lane == 31) s_cst[hh * 33 + 32] = incl;
    }
    __syncthreads();
    if (tid == 0) {
        int a = 0;
        for (int hh = 0; hh < g; ++hh) {
            s_hoff[hh] = a;
            a += s_cst[hh * 33 + 32];
        }
        s_hoff[g] = a;
    }
    __syncthreads();
    const int E = s_hoff[g];
    auto head_of = [&](int e) {
        int hh = 0;
        while (hh + 1 < g && s_hoff[hh + 1] <= e) ++hh;
        return hh;
    };
    // the parent (candidate) of entry e
    auto parent_of = [&](int e) {
        const int hh = head_of(e), pos = e - s_hoff[hh];
        const int r = last_le(s_cst + hh * 33, kc2, pos);
        return __ldg(children + up + s_c0[hh * 32 + r] + (pos - s_cst[hh * 33 + r]));
    };
    const bool ids3_in = E <= g * cap2;
    if (ids3_in) {
        constexpr int B = 8;  // loads in flight a thread
        for (int e0 = tid; e0 < E; e0 += B * NT) {
            int m[B];
#pragma unroll
            for (int x = 0; x < B; ++x) m[x] = e0 + x * NT < E ? parent_of(e0 + x * NT) : 0;
#pragma unroll
            for (int x = 0; x < B; ++x)
                if (e0 + x * NT < E) ids3[e0 + x * NT] = m[x];
        }
    }
    __syncthreads();

    // 3. the candidates of every head: the children of its nodes, scored against its query
    auto put3 = [&](int e, int hh, float v) {
        const int pos = e - s_hoff[hh];
        if (s_cst[hh * 33 + 32] <= capc) s_ck[(size_t)hh * capc + pos] = sort_key(v, ids3_in ? ids3[e] : parent_of(e));
        else wsu[(size_t)hh * np_cap + pos] = v;
    };
    stream_rows<T, NT>(
        E, ring, slot, [&](int e) { return Pu + (size_t)(ids3_in ? ids3[e] : parent_of(e)) * kHeadDim; },
        [&](int bt, int rows, const unsigned char *base) {
            const int e0 = bt * R;
            if constexpr (HR > 0)
                score_rows_mma<NW, HR>(qa, base, rows, g, [&](int j, int hh, float v) {
                    if (head_of(e0 + j) == hh) put3(e0 + j, hh, v);
                });
            else
                score_rows_simt<T, NT>(
                    s_q, base, rows,
                    [&](int j, int &lo, int &hi) {
                        lo = head_of(e0 + j);
                        hi = lo + 1;
                    },
                    [&](int j, int hh, float v) { put3(e0 + j, hh, v); });
        });

    // 4. per head: its best parents in (-q.p, m) order, their pages until k pages
    for (int hh = warp; hh < g; hh += NW) {
        const int Ch = s_cst[hh * 33 + 32];
        const int kc = min(k_pages, Ch);  // at most 32 (k <= 32)
        unsigned long long top = 0ull;
        if (Ch <= capc && Ch <= 32 * V) {
            top = warp_topk<V>(Ch, kc, [&](int i) { return s_ck[(size_t)hh * capc + i]; }, s_tmp[warp]);
        } else {  // k rounds of a warp maximum; past capc the scores are in the workspace
            unsigned long long last = ~0ull;
            for (int r = 0; r < kc; ++r) {
                unsigned long long best = 0ull;
                if (Ch <= capc) {
                    for (int i = lane; i < Ch; i += 32) {
                        const unsigned long long k = s_ck[(size_t)hh * capc + i];
                        if (k < last && k > best) best = k;
                    }
                } else {
                    for (int rr = 0; rr < kc2; ++rr) {
                        const int c0 = s_c0[hh * 32 + rr], cs = s_cst[hh * 33 + rr];
                        const int cn = s_cst[hh * 33 + rr + 1] - cs;
                        for (int c = lane; c < cn; c += 32) {
                            const unsigned long long k =
                                sort_key(wsu[(size_t)hh * np_cap + cs + c], __ldg(children + up + c0 + c));
                            if (k < last && k > best) best = k;
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
                if (lane == r) top = best;
                last = best;
            }
        }
        int fp = 0, pc = 0, contig = 1;
        if (lane < kc && top != 0ull) {
            const int pm = key_id(top);
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

    // 5. the ascending union: thread tid owns words [tid * wpt, (tid + 1) * wpt)
    const int wpt = (words + NT - 1) / NT;
    const int wb = tid * wpt, we = min(words, wb + wpt);
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
#pragma unroll
    for (int w = 0; w < NW; ++w) {
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
    for (int x = total + tid; x < max_sel; x += NT) sel_pages[(size_t)u * max_sel + x] = -1;
    if (tid == 0) {
        if (total > max_sel) set_err(err, ICE_ERR_CAPACITY);
        sel_count[u] = min(total, max_sel);
    }
}

// Shared memory of k_descent: the ring, the queries, the per-head arrays and
// the union bitmask, plus cap level-2 scores (4 bytes) and cap candidate keys
// (8 bytes) per head.
template <typename T>
size_t descent_fixed_smem(int g, int page_cap) {
    constexpr int R = stage_rows<T>(), SB = stage_stride<T>();
    return (size_t)kSlots * R * SB + sizeof(float) * (size_t)g * kHeadDim + sizeof(int) * ((size_t)g * 65 + g + 1) +
           sizeof(unsigned) * (size_t)((page_cap + 31) / 32) + 64;
}
// Dynamic shared memory of one CTA; the static part (per warp 64 keys) comes on top.
constexpr size_t kDescentSmem = 216 * 1024;

template <typename T, int NW, int HR>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws, int32_t *sel_pages,
                     int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const size_t fixed = descent_fixed_smem<T>(g, p.page_cap);
    if (fixed + (size_t)g * 12 * 32 > kDescentSmem) return cudaErrorNotSupported;
    int cap = (int)((kDescentSmem - fixed) / ((size_t)g * 12));
    if (cap > p.np_cap) cap = p.np_cap;
    const size_t smem = fixed + (size_t)g * 12 * cap;
    auto kern = k_descent<T, NW, HR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_dependent(kern, dim3(units_of(p)), dim3(32 * NW), smem, s, static_cast<const T *>(Q), g, p.n_q_heads,
                         p.n_kv_heads, p.np_cap, p.page_cap, ws.k_pages, pos_split(p).n_pos, idx.n_pages,
                         idx.n_nodes2, idx.node2, idx.child_start, idx.children,
                         static_cast<const T *>(idx.parent_keys), idx.parent_first_page, idx.parent_last_page,
                         idx.parent_n_pages, idx.page_next, ws.scores, sel_pages, sel_count, max_sel, cap, cap, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_select3(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                           int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const int g = p.n_q_heads / p.n_kv_heads;
    // g <= 16 (ice_params); 16 warps: twice the row copies in flight of 8
    if (p.dtype == ICE_BF16)
        return g <= 8 ? launch_t<__nv_bfloat16, 16, 1>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s)
                      : launch_t<__nv_bfloat16, 16, 2>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
    return launch_t<float, 16, 0>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
}

}  // namespace ice
