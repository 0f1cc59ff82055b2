// Decode steps a9 (bulk gather of the selected pages) and a10 (masked sparse
// attention over them) for bf16 pools with up to 16 query heads per KV head,
// the two contractions of each page on warp-level tensor-core MMAs.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 4: the selected pages are collected into one
// contiguous buffer; 关键设计 1: a_ij = s_ij exp(q_i.k_j/sqrt(d)) /
// sum_j' s_ij' exp(q_i.k_j'/sqrt(d)) over the selected pages only.
//
// k_attn_mma<F, HR>: grid (S, units), 8 warps; CTA s takes its share of the
// unit's union, warp w the share's pages w, w + 8, ... in order, streamed
// through the warp's three shared-memory slots (two pages in flight while
// one is computed) by 2-D TMA loads with a 128-byte swizzle (so the 8-row
// fragment loads below are conflict-free).
// Per page, with the g <= 16 query rows of the group as the M = 16 rows:
//   S = Q K^T     mma.sync m16n8k16 (bf16 in, fp32 accumulate): A = q in
//                 registers (loaded once), B = K rows by ldmatrix; 2 key
//                 tiles x 8 dimension steps;
//   online softmax on the accumulator fragments: a quad of lanes holds a
//                 row's 16 keys (two shuffles per reduction), masked past
//                 the page length;
//   O += P V      P as the A fragment straight from S's accumulators, split
//                 into bf16 hi + lo parts (two MMAs, ~2^-16 relative error
//                 instead of bf16's 2^-9); B = V rows by ldmatrix.trans;
//                 16 dimension tiles.
// With F the page goes back to kbuf / vbuf by 2-D TMA stores from shared
// memory (the slot is reloaded only after its stores have read it) and its
// length to buf_len, unless buf_len is null: then the pages are gathered into
// shared memory only and no contiguous copy is written.  The warps merge in shared memory; with S = 1 the CTA
// writes O, otherwise its partial joins the others through the unit's ticket
// (log-sum-exp, the last CTA writes O).  HR = 2 when g > 8 (rows 8..15 hold
// query heads too).
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "attn_page.cuh"
#include "select_unit.cuh"
#include "tc_common.cuh"

namespace ice {
namespace {

using namespace tc;
using namespace mma;

constexpr int kMW = 8;   // warps per CTA
constexpr int kNS = 3;   // page slots per warp (pages in flight while one is computed)
constexpr int kMT = kMW * 32;
constexpr uint32_t kHalfBytes = kPage * 128;       // 16 rows x 64 bf16 columns (one swizzled box)
constexpr uint32_t kTileBytes = 2 * kHalfBytes;    // K or V of one page: 4 KB
constexpr uint32_t kSlotBytes = 2 * kTileBytes;    // K and V

struct SmemM {
    unsigned char kv[kMW][kNS][kSlotBytes];  // per warp kNS slots: 192 KB, reused by the merge
    float ml[kMW][16][2];                  // per warp and query row: running max, sum
    float wgt[kMW][16];
    float cml[16][2];
    unsigned long long full[kMW][kNS];
    int wsum[kMW];
    int last;
    int bad;  // a bounded wait of some warp gave up: O is NaN for this unit
};

template <bool kFused, int HR, bool kSel>
__global__ void __launch_bounds__(kMT, 1) k_attn_mma(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_vb,
    const __nv_bfloat16 *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, const int32_t *__restrict__ page_len,
    int page_cap, const int32_t *__restrict__ sel_pages, int32_t *__restrict__ buf_len,
    const int32_t *__restrict__ sel_count, int max_sel, float scale, int n_splits, float *__restrict__ part_ml,
    float *__restrict__ part_o, int32_t *__restrict__ ticket, float *__restrict__ O, int32_t *__restrict__ err,
    unsigned long long wait_ns, int fault_skip, const SelArgs SA) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // the swizzled page tiles want 1024-byte alignment
    SmemM &S = *reinterpret_cast<SmemM *>(smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u));
    const int u = blockIdx.y, split = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qr = lane >> 2, qc = lane & 3;  // fragment row (query row) and column pair
    if (tid < kNS * kMW) mbar_init(&S.full[tid / kNS][tid % kNS], 1);
    if (tid == 0) {
        mbar_init_fence();
        S.bad = 0;
    }
    if (lane < 16) {
        S.ml[warp][lane][0] = -INFINITY;
        S.ml[warp][lane][1] = 0.f;
    }
    dep_wait();  // the selected pages, or the score table (kSel), are complete

    // kSel: the CTA selects its unit's pages itself, in the slot area; split 0
    // also writes them out (sel_pages, sel_count)
    int n;
    const int *s_list = nullptr;
    if (kSel) {
        unsigned long long *s_cand = reinterpret_cast<unsigned long long *>(&S.kv[0][0][0]);
        unsigned *s_mask = reinterpret_cast<unsigned *>(s_cand + kMW * sel::kCand);
        int *lst = reinterpret_cast<int *>(s_mask + (page_cap + 31) / 32);
        n = sel::select_unit<kMW>(SA, u, tid, s_mask, s_cand, S.wsum, lst, split == 0);
        s_list = lst;
    } else {
        n = min(sel_count[u], max_sel);
    }
    const int ps = (max_sel + n_splits - 1) / n_splits;
    const int xs = split * ps;
    const int xe = min(n, xs + ps);
    const int np = max(0, xe - xs);
    const size_t ubase = (size_t)u * max_sel;
    const bool store = kFused && buf_len != nullptr;  // write the contiguous buffer
    if (store)
        for (int x = max(xs, n) + tid; x < min(xs + ps, max_sel); x += kMT) buf_len[ubase + x] = 0;
    __syncthreads();

    // this warp's pages: lane k holds page k's id and length
    const int nk = np > warp ? (np - warp + kMW - 1) / kMW : 0;  // <= 32 (checked on the host)
    int my_pid = 0, my_len = 0;
    if (lane < nk) {
        const size_t sl = ubase + xs + warp + lane * kMW;
        if (kFused) {
            my_pid = kSel ? s_list[xs + warp + lane * kMW] : sel_pages[sl];
            my_len = page_len[(size_t)u * page_cap + my_pid];
        } else {
            my_len = buf_len[sl];
        }
    }
    const uint64_t pol = l2_evict_first();  // each selected page is read once per step
    auto issue = [&](int k, int pid) {
        if (fault_skip) return;  // fault injection: the wait below gives up
        const int x = xs + warp + k * kMW;
        const int row = kFused ? (u * page_cap + pid) * kPage : (int)((ubase + x) * kPage);
        unsigned char *slot = S.kv[warp][k % kNS];
        unsigned long long *bar = &S.full[warp][k % kNS];
        mbar_expect_tx(bar, kSlotBytes);
        tma_load_2d_hint(slot, &tm_k, bar, 0, row, pol);
        tma_load_2d_hint(slot + kHalfBytes, &tm_k, bar, 64, row, pol);
        tma_load_2d_hint(slot + kTileBytes, &tm_v, bar, 0, row, pol);
        tma_load_2d_hint(slot + kTileBytes + kHalfBytes, &tm_v, bar, 64, row, pol);
    };
    if (kSel) __syncthreads();  // every warp has its page ids before the slots fill
    {
        int pf[kNS];
#pragma unroll
        for (int k = 0; k < kNS; ++k) pf[k] = __shfl_sync(0xffffffffu, my_pid, k);
        if (lane == 0)
#pragma unroll
            for (int k = 0; k < kNS; ++k)
                if (nk > k) issue(k, pf[k]);
    }

    // A fragments of Q (rows = query rows of the group), 8 steps of 16 dims
    uint32_t qa[8][4];
    load_q_frag<HR>(Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim, g, qa);
    AttnState st;
    st.init();
    bool ok = true;
    for (int k = 0; k < nk; ++k) {
        const int x = xs + warp + k * kMW;
        const size_t slot = ubase + x;
        const int len = __shfl_sync(0xffffffffu, my_len, k);
        const int pid_next = __shfl_sync(0xffffffffu, my_pid, (k + kNS) & 31);
        if (store && lane == 0) buf_len[slot] = len;
        if (ok) ok = mbar_wait(&S.full[warp][k % kNS], (k / kNS) & 1, wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        unsigned char *sp = S.kv[warp][k % kNS];
        if (store && lane == 0) {  // the contiguous buffer, straight from shared memory
            fence_proxy_async();
            const int row = (int)(slot * kPage);
            tma_store_2d(&tm_kb, sp, 0, row);
            tma_store_2d(&tm_kb, sp + kHalfBytes, 64, row);
            tma_store_2d(&tm_vb, sp + kTileBytes, 0, row);
            tma_store_2d(&tm_vb, sp + kTileBytes + kHalfBytes, 64, row);
            bulk_commit();
        }
        attend_page<HR>(qa, su32(sp), su32(sp + kTileBytes), len, scale, st);
        __syncwarp();
        if (lane == 0 && k + kNS < nk) {  // refill this slot once its stores have read it
            if (store) bulk_wait_read_all();
            issue(k + kNS, pid_next);
        }
        __syncwarp();
    }
    if (!ok) {
        set_err(err, ICE_ERR_TIMEOUT);
        if (lane == 0) S.bad = 1;
    }
    if (store && lane == 0) bulk_wait_read_all();  // the slots are reused below
    if (qc == 0) {
        S.ml[warp][qr][0] = st.m[0];
        S.ml[warp][qr][1] = st.l[0];
        if (HR > 1) {
            S.ml[warp][qr + 8][0] = st.m[1];
            S.ml[warp][qr + 8][1] = st.l[1];
        }
    }
    __syncthreads();

    // ---- merge the warps (slot area reused): s_o[w][row][d]
    float *s_o = reinterpret_cast<float *>(&S.kv[0][0][0]);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
        const int d = 8 * nt + 2 * qc;
        *reinterpret_cast<float2 *>(s_o + ((size_t)warp * 16 + qr) * kHeadDim + d) =
            make_float2(st.o[nt][0], st.o[nt][1]);
        if (HR > 1)
            *reinterpret_cast<float2 *>(s_o + ((size_t)warp * 16 + qr + 8) * kHeadDim + d) =
                make_float2(st.o[nt][2], st.o[nt][3]);
    }
    if (tid < g) {
        float M = -INFINITY;
        for (int w = 0; w < kMW; ++w) M = fmaxf(M, S.ml[w][tid][0]);
        float L = 0.f;
        for (int w = 0; w < kMW; ++w) {
            const float m = S.ml[w][tid][0];
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            S.wgt[w][tid] = wt;
            L = fmaf(S.ml[w][tid][1], wt, L);
        }
        if (S.bad) L = __int_as_float(0x7fc00000);  // NaN: carried into O by the merges
        S.cml[tid][0] = M;
        S.cml[tid][1] = L;
        if (n_splits > 1) {
            const size_t pb = ((size_t)u * n_splits + split) * g + tid;
            part_ml[pb * 2 + 0] = M;
            part_ml[pb * 2 + 1] = L;
        }
    }
    __syncthreads();
    for (int xx = tid; xx < g * kHeadDim; xx += kMT) {
        const int hh = xx / kHeadDim, d = xx % kHeadDim;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kMW; ++w) acc = fmaf(s_o[((size_t)w * 16 + hh) * kHeadDim + d], S.wgt[w][hh], acc);
        if (n_splits == 1) {
            const float L = S.cml[hh][1];
            O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + d] = L > 0.f ? acc / L : (L == L ? 0.f : L);
        } else {
            part_o[(((size_t)u * n_splits + split) * g + hh) * kHeadDim + d] = acc;
        }
    }
    if (n_splits == 1) return;
    __threadfence();
    __syncthreads();
    if (tid == 0) S.last = (atomicAdd(ticket + u, 1) == n_splits - 1);
    __syncthreads();
    if (!S.last) return;
    __threadfence();
    float *s_w = s_o;  // [n_splits][g] weights, then [g] totals
    const int nsg = n_splits * g;
    const float *ml = part_ml + (size_t)u * nsg * 2;
    if (tid < g) {
        float M = -INFINITY;
        for (int sp2 = 0; sp2 < n_splits; ++sp2) M = fmaxf(M, __ldcg(ml + 2 * (sp2 * g + tid)));
        float L = 0.f;
        for (int sp2 = 0; sp2 < n_splits; ++sp2) {
            const float m = __ldcg(ml + 2 * (sp2 * g + tid));
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            s_w[sp2 * g + tid] = wt;
            L = fmaf(__ldcg(ml + 2 * (sp2 * g + tid) + 1), wt, L);
        }
        s_w[nsg + tid] = L;
    }
    __syncthreads();
    const float *po = part_o + (size_t)u * nsg * kHeadDim;
    for (int xx = tid; xx < g * kHeadDim; xx += kMT) {
        const int hh = xx / kHeadDim, d = xx % kHeadDim;
        float acc = 0.f;
        for (int sp2 = 0; sp2 < n_splits; ++sp2)
            acc = fmaf(__ldcg(po + ((size_t)sp2 * g + hh) * kHeadDim + d), s_w[sp2 * g + hh], acc);
        const float L = s_w[nsg + hh];
        O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + d] = L > 0.f ? acc / L : (L == L ? 0.f : L);
    }
    if (tid == 0) ticket[u] = 0;
}

int sm_count_cached() {
    static int n_sm = 0;
    if (!n_sm) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (n_sm <= 0) n_sm = 1;
    }
    return n_sm;
}

template <bool F, int HR, bool kSel>
cudaError_t launch_hr(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q, void *kbuf,
                      void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale, float *O,
                      const DecodeWs &ws, int32_t *err, cudaStream_t s, int n_splits, const SelArgs &SA) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    CUtensorMap tk, tv, tkb, tvb;
    const unsigned long long prow = (unsigned long long)U * p.page_cap * kPage;
    const unsigned long long brow = (unsigned long long)U * max_sel * kPage;
    if (brow > 0x7FFFFFFFull || prow > 0x7FFFFFFFull) return cudaErrorNotSupported;
    const bool store = buf_len != nullptr;  // fused without buf_len: no contiguous copy
    if (store && (!make_map_bf16(&tkb, kbuf, brow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B) ||
                  !make_map_bf16(&tvb, vbuf, brow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B)))
        return cudaErrorNotSupported;
    if (!F && !store) return cudaErrorInvalidValue;
    if (F) {
        if (!make_map_bf16(&tk, pool->pool_k, prow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_bf16(&tv, pool->pool_v, prow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorNotSupported;
        if (!store) tkb = tvb = tk;  // unused
    } else {
        tk = tkb;
        tv = tvb;
    }
    const size_t merge = sizeof(float) * (size_t)(n_splits * g + g);
    const size_t need = (sizeof(SmemM) > merge ? sizeof(SmemM) : merge) + 1024;  // + alignment slack
    if (need > 227 * 1024) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k_attn_mma<F, HR, kSel>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need);
    if (e != cudaSuccess) return e;
    const __nv_bfloat16 *Qb = static_cast<const __nv_bfloat16 *>(Q);
    const int32_t *plen = pool ? pool->page_len : nullptr;
    const bool fault = fault_armed("timeout");
    e = launch_dependent(k_attn_mma<F, HR, kSel>, dim3(n_splits, U), dim3(kMT), need, s, tk, tv, tkb, tvb, Qb, g,
                         p.n_q_heads, p.n_kv_heads, plen, p.page_cap, sel_pages, buf_len, sel_count, max_sel, scale,
                         n_splits, ws.part_ml, ws.part_o, ws.attn_ticket, O, err, fault ? kFaultWaitNs : kWaitNs,
                         fault ? 1 : 0, SA);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// The selection runs in the attention CTAs: one warp per query head (g <= 12),
// candidate keys, union bitmask and page list in the 192 KB slot area.
bool attention_mma_select_supported(const ice_params &p, int max_sel) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const size_t need = (size_t)kMW * sel::kCand * 8 + 4 * (size_t)((p.page_cap + 31) / 32) + 4 * (size_t)max_sel;
    return attention_mma_supported(p) && g <= kMW && need <= sizeof(SmemM::kv);
}

cudaError_t launch_attention_mma_select(const ice_params &p, const ice_index &idx, const SelArgs &A, const void *Q,
                                        void *kbuf, void *vbuf, int32_t *buf_len, int max_sel, float scale, float *O,
                                        const DecodeWs &ws, int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    // a unit is split over CTAs only while each keeps its slots full: every
    // split CTA repeats the selection and the last one merges
    int splits = sm_count_cached() / U;
    const int most = (max_sel + kMW * kNS - 1) / (kMW * kNS);
    splits = splits < 1 ? 1 : (splits > most ? most : splits);
    const int per_warp = (ceil_div(max_sel, splits) + kMW - 1) / kMW;
    if (splits > ws.n_splits || per_warp > 32 || ((uintptr_t)Q & 3u) != 0) return cudaErrorNotSupported;
    if (g <= 8)
        return launch_hr<true, 1, true>(p, &idx, A.sel_pages, Q, kbuf, vbuf, buf_len, A.sel_count, max_sel, scale, O,
                                        ws, err, s, splits, A);
    return launch_hr<true, 2, true>(p, &idx, A.sel_pages, Q, kbuf, vbuf, buf_len, A.sel_count, max_sel, scale, O, ws,
                                    err, s, splits, A);
}

bool attention_mma_supported(const ice_params &p) {
    const int g = p.n_q_heads / p.n_kv_heads;
    return p.dtype == ICE_BF16 && g >= 1 && g <= 16;
}

namespace {
// CTAs per unit of the split attention: one per unit while the units fill the
// SMs, else a few per unit.
int attention_splits(const ice_params &p, int max_sel) {
    int splits = sm_count_cached() / units_of(p);
    const int most = (max_sel + kMW - 1) / kMW;
    return splits < 1 ? 1 : (splits > most ? most : splits);
}
}  // namespace

// The shapes the MMA attention takes: bf16, g <= 16, at most 32 pages per
// warp, TMA row coordinates within int32.
bool attention_mma_fits(const ice_params &p, int max_sel) {
    const int splits = attention_splits(p, max_sel);
    const int per_warp = (ceil_div(max_sel, splits) + kMW - 1) / kMW;
    const unsigned long long U = (unsigned long long)units_of(p);
    return attention_mma_supported(p) && per_warp <= 32 && U * p.page_cap * kPage <= 0x7FFFFFFFull &&
           U * max_sel * kPage <= 0x7FFFFFFFull;
}

// One CTA per unit while the units fill the SMs, else a few per unit; each
// warp takes at most 32 pages.  cudaErrorNotSupported: nothing launched.
cudaError_t launch_attention_mma(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q,
                                 void *kbuf, void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel,
                                 float scale, float *O, const DecodeWs &ws, int32_t *err, cudaStream_t s) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const int splits = attention_splits(p, max_sel);
    if (!attention_mma_fits(p, max_sel) || splits > ws.n_splits) return cudaErrorNotSupported;
    if (pool) {
        if (g <= 8) return launch_hr<true, 1, false>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits, SelArgs{});
        return launch_hr<true, 2, false>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits, SelArgs{});
    }
    if (g <= 8) return launch_hr<false, 1, false>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits, SelArgs{});
    return launch_hr<false, 2, false>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits, SelArgs{});
}

}  // namespace ice
