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
// k_select_topk: one CTA per unit, one warp per query head (select_unit).  Any
//   group maximum T0 that kc group maxima reach is a lower bound of the kc-th
//   best score, so the best kc keys (score, -m) all lie in the groups whose
//   maximum is >= T0: T0 by a radix search on the group maxima, then only
//   those groups' scores are read, the keys >= T0 put in order (their page
//   spans load meanwhile), whose pages (k per head) are ORed into the union
//   bitmask; the block writes the ascending page list.  The kernel is a short chain of dependent loads; it
//   runs after the streaming kernel so that the chain sees an idle memory
//   system (inside the streaming kernel each load waited ~2.5 us).
// Every mbarrier wait gives up after ~2 s and records ICE_ERR_TIMEOUT; the
// roles drain what they issued and TMEM is freed before the CTA returns.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "select_unit.cuh"
#include "topk_common.cuh"

namespace ice {
namespace {

using namespace tc;
using namespace topk;
using namespace sel;

constexpr int BM = 128;    // parents per tile (TMEM lanes)
constexpr int BQ = 16;     // query rows per MMA (N)
constexpr int NS = 4;      // parent-tile ring depth
constexpr int kEpiWarps = 4;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
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

template <int GT>
__global__ void __launch_bounds__(kThreads, 1)
    k_score_tc(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ, int U, int g,
               int n_q_heads, int n_kv_heads, int np_cap, int T, const int32_t *__restrict__ n_parents,
               float *__restrict__ scores, float *__restrict__ gmax, int32_t *__restrict__ err) {
    dep_wait();  // the previous kernel of the stream is complete (launched as its dependent)
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

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            // the parent rows are read once: evicted first, so the score
            // table stays in L2 for the selection that reads it back
            const uint64_t pol = l2_evict_first();
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
                    tma_load_2d_hint(sA + s * A_BYTES, &tmP, &bars->full[s], 0, y, pol);
                    tma_load_2d_hint(sA + s * A_BYTES + A_HALF, &tmP, &bars->full[s], 64, y, pol);
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
    dep_wait();  // the score table is complete
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

SelArgs select_args(const ice_params &p, const ice_index &idx, const DecodeWs &ws, int32_t *sel_pages,
                    int32_t *sel_count, int max_sel, int32_t *err) {
    const int U = units_of(p);
    SelArgs A;
    A.g = p.n_q_heads / p.n_kv_heads;
    A.np_cap = p.np_cap;
    A.page_cap = p.page_cap;
    A.k_pages = ws.k_pages;
    A.kc = ws.k_pages;
    A.max_sel = max_sel;
    A.n_pos = pos_split(p).n_pos;
    A.n_parents = idx.n_parents;
    A.n_pages = idx.n_pages;
    A.scores = ws.scores;
    A.gmax = ws.scores + (size_t)U * A.g * p.np_cap;
    A.parent_first_page = idx.parent_first_page;
    A.parent_last_page = idx.parent_last_page;
    A.parent_n_pages = idx.parent_n_pages;
    A.page_next = idx.page_next;
    A.sel_pages = sel_pages;
    A.sel_count = sel_count;
    A.err = err;
    A.pf_k = A.pf_v = nullptr;
    A.page_bytes = 0;
    return A;
}

// The score table of every unit (k_score_tc).  Returns cudaErrorNotSupported
// (nothing launched) when a tensor map cannot be made for these pointers.
cudaError_t launch_score_tc(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                            int32_t *err, cudaStream_t s) {
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
    {
        const cudaError_t e_ = launch_dependent(kern, dim3(grid), dim3(kThreads), kSmemBytes, s, tmP, tmQ, U, g,
                                                p.n_q_heads, p.n_kv_heads, p.np_cap, T, idx.n_parents, ws.scores,
                                                gmax, err);
        if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
}

// The page lists from the score table (k_select_topk, one CTA per unit).
cudaError_t launch_topk(const ice_params &p, const SelArgs &A, cudaStream_t s) {
    const int nsw = nsw_of(A.g);
    auto topk = nsw == 4 ? k_select_topk<4> : nsw == 8 ? k_select_topk<8> : k_select_topk<16>;
    const size_t smem = topk_smem(A.g, p.page_cap);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_dependent(topk, dim3(units_of(p)), dim3(32 * nsw), smem, s, A);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Returns cudaErrorNotSupported (nothing launched) when a tensor map cannot
// be made for these pointers; the caller then uses the SIMT kernel.
cudaError_t launch_select_tc(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                             int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const cudaError_t e = launch_score_tc(p, idx, Q, ws, err, s);
    if (e != cudaSuccess) return e;
    return launch_topk(p, select_args(p, idx, ws, sel_pages, sel_count, max_sel, err), s);
}

}  // namespace ice
