// Decode steps a9 (bulk gather of the selected pages) and a10 (masked sparse
// attention over them) for bf16 pools with at most 8 query heads per KV head.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 4: the selected pages are not contiguous, so
// they are collected into one contiguous buffer and moved in one transfer;
// 关键设计 1: a_ij = s_ij exp(q_i.k_j/sqrt(d)) / sum_j' s_ij' exp(q_i.k_j'/sqrt(d)).
// IceCache popular-science article (aitangshan.cn/news/751385), section 四:
// bulk loading gathers everything needed into one staging area first.
//
// k_attn_stream<F, GT, HS>: grid (splits of 8 / HS selected pages, units),
// 8 warps.  Thread 0 starts one 1-D bulk copy per page for K and for V (4 KB
// each) into shared memory; HS warps share a page, each taking GT / HS of the
// group's heads (HS = 2 for 8 heads, halving the registers so that three CTAs
// fit on an SM):
//   * with F (fused gather) it writes the page back to kbuf / vbuf with 1-D
//     bulk stores straight from shared memory, and the page's length to
//     buf_len; without F the pages come from kbuf / vbuf;
//   * logits: 16 lanes per key, 8 dimensions per lane, the lane's q slices of
//     the group's GT heads in registers; the 16 partial sums of each head are
//     folded by recursive halving (each step a lane keeps half of its heads);
//   * softmax over the page's 16 slots per head (masked past the page length);
//   * P V: lane owns output dimensions 4 lane .. 4 lane + 3 of every head.
// The 8 warps' (max, sum, o) merge in shared memory into one partial per
// split (log-sum-exp rule); the unit's last CTA (atomic ticket, nobody waits)
// merges the splits and writes O.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace ice {
namespace {

using namespace tc;

constexpr int kW = 8;  // warps per CTA
constexpr int kThreads = 32 * kW;
constexpr int kPageElems = kPage * kHeadDim;        // 2048
constexpr uint32_t kPageBytes = kPageElems * 2;     // bf16: 4 KB

// SPP pages per CTA; HS warps share a page, each taking GT / HS of the heads.
template <int SPP>
struct Smem {
    __nv_bfloat16 kv[SPP][2][kPageElems];  // reused by the merges
    float p[SPP][kPage][8];                 // per page: logits [slot][head]
    unsigned long long pp[SPP][kPage][8];   // per page: probabilities, each duplicated into an fp32 pair
    float ml[SPP][8][2];                    // per page and head: max, sum
    float wgt[SPP][8];                      // merge weights
    unsigned long long full[SPP];
    int last;
};


template <bool kFused, int GT, int HS>
__global__ void __launch_bounds__(kThreads, (GT / HS) >= 8 ? 2 : 3) k_attn_stream(
    const __nv_bfloat16 *__restrict__ Q, int g, int n_q_heads, int n_kv_heads,
    const __nv_bfloat16 *__restrict__ pool_k, const __nv_bfloat16 *__restrict__ pool_v,
    const int32_t *__restrict__ page_len, int page_cap, const int32_t *__restrict__ sel_pages,
    __nv_bfloat16 *__restrict__ kbuf, __nv_bfloat16 *__restrict__ vbuf, int32_t *__restrict__ buf_len,
    const int32_t *__restrict__ sel_count, int max_sel, float scale, int n_splits, float *__restrict__ part_ml,
    float *__restrict__ part_o, int32_t *__restrict__ ticket, float *__restrict__ O, int32_t *__restrict__ err) {
    constexpr int SPP = kW / HS;  // pages per CTA
    constexpr int GH = GT / HS;   // heads per warp
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<SPP> &S = *reinterpret_cast<Smem<SPP> *>(smem_raw);
    const int u = blockIdx.y, split = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pw = warp / HS, hbase = (warp % HS) * GH;  // this warp's page and first head
    const int n = min(sel_count[u], max_sel);
    const int x0 = split * SPP;
    const int np = max(0, min(SPP, n - x0));
    const size_t sbase = (size_t)u * max_sel + x0;  // slot of this split's first page

    if (tid == 0) {
        for (int i = 0; i < SPP; ++i) mbar_init(&S.full[i], 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < np; ++i) {
            const __nv_bfloat16 *sk, *sv;
            if (kFused) {
                const size_t pg = (size_t)u * page_cap + sel_pages[sbase + i];
                sk = pool_k + pg * kPageElems;
                sv = pool_v + pg * kPageElems;
            } else {
                sk = kbuf + (sbase + i) * kPageElems;
                sv = vbuf + (sbase + i) * kPageElems;
            }
            mbar_expect_tx(&S.full[i], 2 * kPageBytes);
            bulk_load(S.kv[i][0], sk, kPageBytes, &S.full[i]);
            bulk_load(S.kv[i][1], sv, kPageBytes, &S.full[i]);
        }
    }
    const bool store = kFused && buf_len != nullptr;  // no buf_len: no contiguous copy
    if (store)  // slots of this split past the selection hold no page
        for (int x = max(x0, n) + tid; x < min(x0 + SPP, max_sel); x += kThreads) buf_len[(size_t)u * max_sel + x] = 0;

    // q slices: heads hbase .. hbase + GH - 1, dimensions 8 c .. 8 c + 7 with c = lane % 16
    const int c = lane & 15, half = lane >> 4;
    unsigned long long q[GH][4];  // fp32 pairs of dims 8c + 2i, 8c + 2i + 1
    {
        const __nv_bfloat16 *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (hbase + hh < g) raw = *reinterpret_cast<const uint4 *>(Qu + (size_t)(hbase + hh) * kHeadDim + 8 * c);
            q[hh][0] = bf2_pair(raw.x);
            q[hh][1] = bf2_pair(raw.y);
            q[hh][2] = bf2_pair(raw.z);
            q[hh][3] = bf2_pair(raw.w);
        }
    }
    unsigned long long o[GH][2];  // fp32 pairs of dims 4 lane + {0, 1}, {2, 3}
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) o[hh][0] = o[hh][1] = 0ull;
    bool ok = true;
    bool stored = false;
    if (pw < np) {
        const size_t slot = sbase + pw;
        int len;
        if (kFused) {
            len = page_len[(size_t)u * page_cap + sel_pages[slot]];
            if (store && lane == 0 && hbase == 0) buf_len[slot] = len;
        } else {
            len = buf_len[slot];
        }
        ok = mbar_wait(&S.full[pw], 0);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && store && lane == 0 && hbase == 0) {  // the contiguous buffer, straight from shared memory
            fence_proxy_async();
            bulk_store(kbuf + slot * kPageElems, S.kv[pw][0], kPageBytes);
            bulk_store(vbuf + slot * kPageElems, S.kv[pw][1], kPageBytes);
            bulk_commit();
            stored = true;
        }
        if (ok) {
            const __nv_bfloat16 *Kp = S.kv[pw][0];
            const __nv_bfloat16 *Vp = S.kv[pw][1];
            // ---- logits: keys 2 kp + half, 16 lanes each
#pragma unroll 2
            for (int kp = 0; kp < kPage / 2; ++kp) {
                const int j = 2 * kp + half;
                const uint4 raw = *reinterpret_cast<const uint4 *>(Kp + j * kHeadDim + 8 * c);
                const unsigned long long x0p = bf2_pair(raw.x), x1p = bf2_pair(raw.y), x2p = bf2_pair(raw.z),
                                         x3p = bf2_pair(raw.w);
                float a[GH];
#pragma unroll
                for (int hh = 0; hh < GH; ++hh) {
                    unsigned long long sp = fma2(q[hh][0], x0p, 0ull);
                    sp = fma2(q[hh][1], x1p, sp);
                    sp = fma2(q[hh][2], x2p, sp);
                    sp = fma2(q[hh][3], x3p, sp);
                    const float2 f = upk2(sp);
                    a[hh] = f.x + f.y;
                }
                // fold the 16 lanes of this key: halving over heads, then the rest
                int head = 0, off = 8;
#pragma unroll
                for (int nn = GH; nn > 1; nn >>= 1, off >>= 1) {
                    const bool up = (lane & off) != 0;
#pragma unroll
                    for (int i = 0; i < nn / 2; ++i) {
                        const float send = up ? a[i] : a[i + nn / 2];
                        const float keep = up ? a[i + nn / 2] : a[i];
                        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                    head += up ? nn / 2 : 0;
                }
                float v = a[0];
                for (; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if ((lane & (16 / GH - 1)) == 0 && hbase + head < g) S.p[pw][j][hbase + head] = v;
            }
            __syncwarp();
            // ---- softmax over the page's slots, 16 lanes per head
#pragma unroll
            for (int e = 0; e < (GH * kPage + 31) / 32; ++e) {
                const int item = e * 32 + lane;
                const int hh = hbase + item / kPage, sl = item % kPage;
                const bool on = hh < g && item < GH * kPage;
                const float lg = (on && sl < len) ? S.p[pw][sl][hh] * scale : -INFINITY;
                float mx = lg;
#pragma unroll
                for (int of = 8; of >= 1; of >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, of));
                const float pr = lg == -INFINITY ? 0.f : expf(lg - mx);
                float sm = pr;
#pragma unroll
                for (int of = 8; of >= 1; of >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, of);
                if (on) S.pp[pw][sl][hh] = pk2(pr, pr);
                if (on && sl == 0) {
                    S.ml[pw][hh][0] = mx;
                    S.ml[pw][hh][1] = sm;
                }
            }
            __syncwarp();
            // ---- o[hh][d] = sum_s p[s][hh] v[s][d], d = 4 lane .. 4 lane + 3
#pragma unroll 4
            for (int sl = 0; sl < kPage; ++sl) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(Vp + sl * kHeadDim + 4 * lane);
                const unsigned long long v01 = bf2_pair(raw.x), v23 = bf2_pair(raw.y);
                const unsigned long long *pp = S.pp[pw][sl] + hbase;
#pragma unroll
                for (int hh = 0; hh < GH; ++hh) {
                    const unsigned long long pv = pp[hh];
                    o[hh][0] = fma2(pv, v01, o[hh][0]);
                    o[hh][1] = fma2(pv, v23, o[hh][1]);
                }
            }
        }
    }
    if (!ok) set_err(err, ICE_ERR_TIMEOUT);
    // pages this CTA does not hold contribute nothing
    if (pw >= np || !ok) {
        if (lane < GH) {
            S.ml[pw][hbase + lane][0] = -INFINITY;
            S.ml[pw][hbase + lane][1] = 0.f;
        }
    }
    if (stored) bulk_wait_read_all();  // the page buffers are reused below
    __syncthreads();

    // ---- merge the pages into this split's partial (kv area reused)
    float *s_o = reinterpret_cast<float *>(&S.kv[0][0][0]);  // [SPP][GT][128]
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
        const float2 a = upk2(o[hh][0]), bq = upk2(o[hh][1]);
        *reinterpret_cast<float4 *>(s_o + ((size_t)pw * GT + hbase + hh) * kHeadDim + 4 * lane) =
            make_float4(a.x, a.y, bq.x, bq.y);
    }
    if (tid < g) {
        float M = -INFINITY;
        for (int w = 0; w < SPP; ++w) M = fmaxf(M, S.ml[w][tid][0]);
        float L = 0.f;
        for (int w = 0; w < SPP; ++w) {
            const float m = S.ml[w][tid][0];
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            S.wgt[w][tid] = wt;
            L = fmaf(S.ml[w][tid][1], wt, L);
        }
        const size_t pb = ((size_t)u * n_splits + split) * g + tid;
        part_ml[pb * 2 + 0] = M;
        part_ml[pb * 2 + 1] = L;
    }
    __syncthreads();
    for (int x = tid; x < g * kHeadDim; x += kThreads) {
        const int hh = x / kHeadDim, d = x % kHeadDim;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < SPP; ++w) acc = fmaf(s_o[((size_t)w * GT + hh) * kHeadDim + d], S.wgt[w][hh], acc);
        part_o[(((size_t)u * n_splits + split) * g + hh) * kHeadDim + d] = acc;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) S.last = (atomicAdd(ticket + u, 1) == n_splits - 1);
    __syncthreads();
    if (!S.last) return;
    __threadfence();

    // ---- the unit's last CTA merges the splits (log-sum-exp) and writes O
    float *s_w = s_o;  // [n_splits][g] weights, then [g] totals
    const int nsg = n_splits * g;
    const float *ml = part_ml + (size_t)u * nsg * 2;
    if (tid < g) {
        float M = -INFINITY;
        for (int sp = 0; sp < n_splits; ++sp) M = fmaxf(M, __ldcg(ml + 2 * (sp * g + tid)));
        float L = 0.f;
        for (int sp = 0; sp < n_splits; ++sp) {
            const float m = __ldcg(ml + 2 * (sp * g + tid));
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            s_w[sp * g + tid] = wt;
            L = fmaf(__ldcg(ml + 2 * (sp * g + tid) + 1), wt, L);
        }
        s_w[nsg + tid] = L;
    }
    __syncthreads();
    const float *po = part_o + (size_t)u * nsg * kHeadDim;
    for (int x = tid; x < g * kHeadDim; x += kThreads) {
        const int hh = x / kHeadDim, d = x % kHeadDim;
        float acc = 0.f;
        for (int sp = 0; sp < n_splits; ++sp)
            acc = fmaf(__ldcg(po + ((size_t)sp * g + hh) * kHeadDim + d), s_w[sp * g + hh], acc);
        const float L = s_w[nsg + hh];
        O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + d] = L > 0.f ? acc / L : 0.f;
    }
    if (tid == 0) ticket[u] = 0;
}

template <bool F, int GT, int HS>
cudaError_t launch_gt(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q,
                      void *kbuf, void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale,
                      float *O, const DecodeWs &ws, int32_t *err, cudaStream_t s) {
    constexpr int SPP = kW / HS;
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    const int n_splits = ceil_div(max_sel, SPP);
    if (n_splits > ws.n_splits) return cudaErrorNotSupported;  // the workspace holds fewer partials
    const size_t merge = sizeof(float) * (size_t)(n_splits * g + g);
    const size_t need = sizeof(Smem<SPP>) > merge ? sizeof(Smem<SPP>) : merge;
    if (need > 200 * 1024) return cudaErrorNotSupported;
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_stream<F, GT, HS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need);
    if (e != cudaSuccess) return e;
    const __nv_bfloat16 *pk = pool ? static_cast<const __nv_bfloat16 *>(pool->pool_k) : nullptr;
    const __nv_bfloat16 *pv = pool ? static_cast<const __nv_bfloat16 *>(pool->pool_v) : nullptr;
    const int32_t *pl = pool ? pool->page_len : nullptr;
    k_attn_stream<F, GT, HS><<<dim3(n_splits, U), kThreads, need, s>>>(
        static_cast<const __nv_bfloat16 *>(Q), g, p.n_q_heads, p.n_kv_heads, pk, pv, pl, p.page_cap, sel_pages,
        static_cast<__nv_bfloat16 *>(kbuf), static_cast<__nv_bfloat16 *>(vbuf), buf_len, sel_count, max_sel, scale,
        n_splits, ws.part_ml, ws.part_o, ws.attn_ticket, O, err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// k_attn_unit<F, GT>: grid (S, units), S CTAs per unit (one when the units
// fill the SMs), 12 warps.  CTA s takes the union slots of its share; warp w
// takes the share's pages w, w + 12, ... in order, double-buffering them in
// its own two shared-memory slots (1-D bulk copies, one mbarrier per slot),
// with an online softmax per head across its pages.  With F each page goes
// back to kbuf / vbuf by bulk stores from shared memory (a slot is reloaded
// only after its stores have read it).  The warps merge in shared memory; with
// S = 1 the CTA writes O, otherwise its partial joins the others through the
// unit's ticket (log-sum-exp, the last CTA writes O).
constexpr int kUW = 12;
constexpr int kUT = kUW * 32;

struct SmemU {
    __nv_bfloat16 kv[kUW][2][2][kPageElems];  // per warp two slots of (K, V): 192 KB, reused by the merge
    float p[kUW][kPage][8];                    // per warp: logits [slot][head]
    unsigned long long pp[kUW][kPage][8];      // per warp: probabilities as duplicated fp32 pairs
    float ml[kUW][8][2];                       // per warp and head: running max, sum
    float alpha[kUW][8];                       // per warp and head: rescale of the last update / merge weight
    float cml[8][2];                           // the CTA's merged max, sum
    unsigned long long full[kUW][2];
    int last;
};

template <bool kFused, int GT>
__global__ void __launch_bounds__(kUT, 1) k_attn_unit(
    const __nv_bfloat16 *__restrict__ Q, int g, int n_q_heads, int n_kv_heads,
    const __nv_bfloat16 *__restrict__ pool_k, const __nv_bfloat16 *__restrict__ pool_v,
    const int32_t *__restrict__ page_len, int page_cap, const int32_t *__restrict__ sel_pages,
    __nv_bfloat16 *__restrict__ kbuf, __nv_bfloat16 *__restrict__ vbuf, int32_t *__restrict__ buf_len,
    const int32_t *__restrict__ sel_count, int max_sel, float scale, int n_splits, float *__restrict__ part_ml,
    float *__restrict__ part_o, int32_t *__restrict__ ticket, float *__restrict__ O, int32_t *__restrict__ err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    SmemU &S = *reinterpret_cast<SmemU *>(smem_raw);
    const int u = blockIdx.y, split = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = min(sel_count[u], max_sel);
    const int ps = (max_sel + n_splits - 1) / n_splits;  // union slots per CTA
    const int xs = split * ps;
    const int xe = min(n, xs + ps);                       // this CTA's pages: [xs, xe)
    const int np = max(0, xe - xs);
    const size_t ubase = (size_t)u * max_sel;

    if (tid < 2 * kUW) mbar_init(&S.full[tid >> 1][tid & 1], 1);
    if (tid == 0) mbar_init_fence();
    const bool store = kFused && buf_len != nullptr;  // no buf_len: no contiguous copy
    if (store)  // slots of this share past the selection hold no page
        for (int x = max(xs, n) + tid; x < min(xs + ps, max_sel); x += kUT) buf_len[ubase + x] = 0;
    if (lane < 8) {
        S.ml[warp][lane][0] = -INFINITY;
        S.ml[warp][lane][1] = 0.f;
    }
    __syncthreads();

    // page k of this warp: share index warp + k * kUW, in slot k & 1; lane k
    // holds its page id and length (one round trip for all of them)
    const int nk = np > warp ? (np - warp + kUW - 1) / kUW : 0;  // <= 32 (checked on the host)
    int my_pid = 0, my_len = 0;
    if (lane < nk) {
        const size_t sl = ubase + xs + warp + lane * kUW;
        if (kFused) {
            my_pid = sel_pages[sl];
            my_len = page_len[(size_t)u * page_cap + my_pid];
        } else {
            my_len = buf_len[sl];
        }
    }
    auto issue = [&](int k, int pid) {
        const int x = xs + warp + k * kUW;
        const __nv_bfloat16 *sk, *sv;
        if (kFused) {
            const size_t pg = (size_t)u * page_cap + pid;
            sk = pool_k + pg * kPageElems;
            sv = pool_v + pg * kPageElems;
        } else {
            sk = kbuf + (ubase + x) * kPageElems;
            sv = vbuf + (ubase + x) * kPageElems;
        }
        mbar_expect_tx(&S.full[warp][k & 1], 2 * kPageBytes);
        bulk_load(S.kv[warp][k & 1][0], sk, kPageBytes, &S.full[warp][k & 1]);
        bulk_load(S.kv[warp][k & 1][1], sv, kPageBytes, &S.full[warp][k & 1]);
    };
    {
        const int p0 = __shfl_sync(0xffffffffu, my_pid, 0), p1 = __shfl_sync(0xffffffffu, my_pid, 1);
        if (lane == 0) {
            if (nk > 0) issue(0, p0);
            if (nk > 1) issue(1, p1);
        }
    }

    const int c = lane & 15, half = lane >> 4;
    unsigned long long q[GT][4];
    {
        const __nv_bfloat16 *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
#pragma unroll
        for (int hh = 0; hh < GT; ++hh) {
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (hh < g) raw = *reinterpret_cast<const uint4 *>(Qu + (size_t)hh * kHeadDim + 8 * c);
            q[hh][0] = bf2_pair(raw.x);
            q[hh][1] = bf2_pair(raw.y);
            q[hh][2] = bf2_pair(raw.z);
            q[hh][3] = bf2_pair(raw.w);
        }
    }
    unsigned long long o[GT][2];
#pragma unroll
    for (int hh = 0; hh < GT; ++hh) o[hh][0] = o[hh][1] = 0ull;
    bool ok = true;
    for (int k = 0; k < nk; ++k) {
        const int x = xs + warp + k * kUW;
        const size_t slot = ubase + x;
        const int len = __shfl_sync(0xffffffffu, my_len, k);
        const int pid_next = __shfl_sync(0xffffffffu, my_pid, (k + 2) & 31);
        if (store && lane == 0) buf_len[slot] = len;
        if (ok) ok = mbar_wait(&S.full[warp][k & 1], (k >> 1) & 1);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const __nv_bfloat16 *Kp = S.kv[warp][k & 1][0];
        const __nv_bfloat16 *Vp = S.kv[warp][k & 1][1];
        if (store && lane == 0) {  // the contiguous buffer, straight from shared memory
            fence_proxy_async();
            bulk_store(kbuf + slot * kPageElems, Kp, kPageBytes);
            bulk_store(vbuf + slot * kPageElems, Vp, kPageBytes);
            bulk_commit();
        }
        float *pw = &S.p[warp][0][0];
        unsigned long long *ppw = &S.pp[warp][0][0];
        // ---- logits
#pragma unroll 2
        for (int kp = 0; kp < kPage / 2; ++kp) {
            const int j = 2 * kp + half;
            const uint4 raw = *reinterpret_cast<const uint4 *>(Kp + j * kHeadDim + 8 * c);
            const unsigned long long x0p = bf2_pair(raw.x), x1p = bf2_pair(raw.y), x2p = bf2_pair(raw.z),
                                     x3p = bf2_pair(raw.w);
            float a[GT];
#pragma unroll
            for (int hh = 0; hh < GT; ++hh) {
                unsigned long long sp = fma2(q[hh][0], x0p, 0ull);
                sp = fma2(q[hh][1], x1p, sp);
                sp = fma2(q[hh][2], x2p, sp);
                sp = fma2(q[hh][3], x3p, sp);
                const float2 f = upk2(sp);
                a[hh] = f.x + f.y;
            }
            int head = 0, off = 8;
#pragma unroll
            for (int nn = GT; nn > 1; nn >>= 1, off >>= 1) {
                const bool up = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < nn / 2; ++i) {
                    const float send = up ? a[i] : a[i + nn / 2];
                    const float keep = up ? a[i + nn / 2] : a[i];
                    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
                head += up ? nn / 2 : 0;
            }
            float v = a[0];
            for (; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if ((lane & (16 / GT - 1)) == 0 && head < g) pw[j * 8 + head] = v;
        }
        __syncwarp();
        // ---- online softmax, 16 lanes per head
#pragma unroll
        for (int e = 0; e < (GT * kPage + 31) / 32; ++e) {
            const int item = e * 32 + lane;
            const int hh = item / kPage, sl = item % kPage;
            const bool on = hh < g && item < GT * kPage;
            const float lg = (on && sl < len) ? pw[sl * 8 + hh] * scale : -INFINITY;
            float mx = lg;
#pragma unroll
            for (int of = 8; of >= 1; of >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, of));
            const float m_old = on ? S.ml[warp][hh][0] : -INFINITY;
            const float m_new = fmaxf(m_old, mx);
            const float pr = lg == -INFINITY ? 0.f : expf(lg - m_new);
            float sm = pr;
#pragma unroll
            for (int of = 8; of >= 1; of >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, of);
            if (on) ppw[sl * 8 + hh] = pk2(pr, pr);
            __syncwarp();
            if (on && sl == 0) {
                const float al = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
                S.alpha[warp][hh] = al;
                S.ml[warp][hh][0] = m_new;
                S.ml[warp][hh][1] = S.ml[warp][hh][1] * al + sm;
            }
        }
        __syncwarp();
        // ---- o = o * alpha + P V
#pragma unroll
        for (int hh = 0; hh < GT; ++hh) {
            const float al = hh < g ? S.alpha[warp][hh] : 0.f;
            const unsigned long long aa = pk2(al, al);
            o[hh][0] = fma2(o[hh][0], aa, 0ull);
            o[hh][1] = fma2(o[hh][1], aa, 0ull);
        }
#pragma unroll 4
        for (int sl = 0; sl < kPage; ++sl) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(Vp + sl * kHeadDim + 4 * lane);
            const unsigned long long v01 = bf2_pair(raw.x), v23 = bf2_pair(raw.y);
            const unsigned long long *pp = ppw + sl * 8;
#pragma unroll
            for (int hh = 0; hh < GT; ++hh) {
                const unsigned long long pv = pp[hh];
                o[hh][0] = fma2(pv, v01, o[hh][0]);
                o[hh][1] = fma2(pv, v23, o[hh][1]);
            }
        }
        __syncwarp();
        // refill this slot with page k + 2 once its stores have read it
        if (lane == 0 && k + 2 < nk) {
            if (store) bulk_wait_read_all();
            issue(k + 2, pid_next);
        }
        __syncwarp();
    }
    if (!ok) set_err(err, ICE_ERR_TIMEOUT);
    if (store && lane == 0) bulk_wait_read_all();  // the slots are reused below
    __syncthreads();

    // ---- merge the warps (slot area reused)
    float *s_o = reinterpret_cast<float *>(&S.kv[0][0][0][0]);  // [kUW][GT][128]
#pragma unroll
    for (int hh = 0; hh < GT; ++hh) {
        const float2 a = upk2(o[hh][0]), bq = upk2(o[hh][1]);
        *reinterpret_cast<float4 *>(s_o + ((size_t)warp * GT + hh) * kHeadDim + 4 * lane) =
            make_float4(a.x, a.y, bq.x, bq.y);
    }
    if (tid < g) {
        float M = -INFINITY;
        for (int w = 0; w < kUW; ++w) M = fmaxf(M, S.ml[w][tid][0]);
        float L = 0.f;
        for (int w = 0; w < kUW; ++w) {
            const float m = S.ml[w][tid][0];
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            S.alpha[w][tid] = wt;
            L = fmaf(S.ml[w][tid][1], wt, L);
        }
        S.cml[tid][0] = M;
        S.cml[tid][1] = L;
        if (n_splits > 1) {
            const size_t pb = ((size_t)u * n_splits + split) * g + tid;
            part_ml[pb * 2 + 0] = M;
            part_ml[pb * 2 + 1] = L;
        }
    }
    __syncthreads();
    for (int x = tid; x < g * kHeadDim; x += kUT) {
        const int hh = x / kHeadDim, d = x % kHeadDim;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kUW; ++w) acc = fmaf(s_o[((size_t)w * GT + hh) * kHeadDim + d], S.alpha[w][hh], acc);
        if (n_splits == 1) {
            const float L = S.cml[hh][1];
            O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + d] = L > 0.f ? acc / L : 0.f;
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
        for (int sp = 0; sp < n_splits; ++sp) M = fmaxf(M, __ldcg(ml + 2 * (sp * g + tid)));
        float L = 0.f;
        for (int sp = 0; sp < n_splits; ++sp) {
            const float m = __ldcg(ml + 2 * (sp * g + tid));
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            s_w[sp * g + tid] = wt;
            L = fmaf(__ldcg(ml + 2 * (sp * g + tid) + 1), wt, L);
        }
        s_w[nsg + tid] = L;
    }
    __syncthreads();
    const float *po = part_o + (size_t)u * nsg * kHeadDim;
    for (int x = tid; x < g * kHeadDim; x += kUT) {
        const int hh = x / kHeadDim, d = x % kHeadDim;
        float acc = 0.f;
        for (int sp = 0; sp < n_splits; ++sp)
            acc = fmaf(__ldcg(po + ((size_t)sp * g + hh) * kHeadDim + d), s_w[sp * g + hh], acc);
        const float L = s_w[nsg + hh];
        O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + d] = L > 0.f ? acc / L : 0.f;
    }
    if (tid == 0) ticket[u] = 0;
}

template <bool F, int GT>
cudaError_t launch_unit(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q,
                        void *kbuf, void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale,
                        float *O, const DecodeWs &ws, int32_t *err, cudaStream_t s, int n_splits) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    const size_t merge = sizeof(float) * (size_t)(n_splits * g + g);
    const size_t need = sizeof(SmemU) > merge ? sizeof(SmemU) : merge;
    if (need > 227 * 1024) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k_attn_unit<F, GT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need);
    if (e != cudaSuccess) return e;
    const __nv_bfloat16 *pk = pool ? static_cast<const __nv_bfloat16 *>(pool->pool_k) : nullptr;
    const __nv_bfloat16 *pv = pool ? static_cast<const __nv_bfloat16 *>(pool->pool_v) : nullptr;
    const int32_t *pl = pool ? pool->page_len : nullptr;
    k_attn_unit<F, GT><<<dim3(n_splits, U), kUT, need, s>>>(
        static_cast<const __nv_bfloat16 *>(Q), g, p.n_q_heads, p.n_kv_heads, pk, pv, pl, p.page_cap, sel_pages,
        static_cast<__nv_bfloat16 *>(kbuf), static_cast<__nv_bfloat16 *>(vbuf), buf_len, sel_count, max_sel, scale,
        n_splits, ws.part_ml, ws.part_o, ws.attn_ticket, O, err);
    return cudaGetLastError();
}

template <bool F>
cudaError_t launch_f(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q, void *kbuf,
                     void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale, float *O,
                     const DecodeWs &ws, int32_t *err, cudaStream_t s) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const int U = units_of(p);
    static int n_sm = 0;
    if (!n_sm) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (n_sm <= 0) n_sm = 1;
    }
    // one CTA per unit streams the unit's pages while the units fill the SMs
    // and each unit holds many pages; with few units the unit's pages are
    // shared among several CTAs
    if (max_sel >= 4 * kUW) {
        int splits = n_sm / U;
        const int most = (max_sel + kUW - 1) / kUW;
        splits = splits < 1 ? 1 : (splits > most ? most : splits);
        const int per_warp = (ceil_div(max_sel, splits) + kUW - 1) / kUW;  // pages a warp takes
        if (splits <= ws.n_splits && per_warp <= 32) {
            cudaError_t e = cudaErrorNotSupported;
            if (g <= 1) e = launch_unit<F, 1>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits);
            else if (g <= 2) e = launch_unit<F, 2>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits);
            else if (g <= 4) e = launch_unit<F, 4>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits);
            else e = launch_unit<F, 8>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s, splits);
            if (e != cudaErrorNotSupported) return e;
        }
    }
    if (g <= 1) return launch_gt<F, 1, 1>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s);
    if (g <= 2) return launch_gt<F, 2, 1>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s);
    if (g <= 4) return launch_gt<F, 4, 1>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s);
    return launch_gt<F, 8, 1>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s);
}

}  // namespace

bool attention_stream_supported(const ice_params &p) {
    const int g = p.n_q_heads / p.n_kv_heads;
    return p.dtype == ICE_BF16 && g >= 1 && g <= 8;
}

cudaError_t launch_attention_stream(const ice_params &p, const ice_index *pool, const int32_t *sel_pages,
                                    const void *Q, void *kbuf, void *vbuf, int32_t *buf_len,
                                    const int32_t *sel_count, int max_sel, float scale, float *O, const DecodeWs &ws,
                                    int32_t *err, cudaStream_t s) {
    if (pool)
        return launch_f<true>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s);
    return launch_f<false>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, err, s);
}

}  // namespace ice
