// Decode steps a9 (bulk gather of the selected pages) and a10 (masked sparse
// attention over them).
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 4: the selected pages are not contiguous, so
// they are collected into one contiguous buffer and moved in one transfer;
// 关键设计 1: a_ij = s_ij exp(q_i.k_j/sqrt(d)) / sum_j' s_ij' exp(q_i.k_j'/sqrt(d)).
// IceCache popular-science article (aitangshan.cn/news/751385), section 四:
// bulk loading gathers everything needed into one staging area first.
//
// k_gather     grid (max_sel, units): one CTA copies one selected page's K and
//              V (16 x d) with 16-byte vectors and writes its length.
// k_attn<F>    grid (splits, units), split-KV flash decode: a CTA owns up to
//              kAttnPagesPerSplit consecutive selected pages of a unit and all
//              g query heads of its GQA group.  Per page: K and V are staged
//              in shared memory as fp32, thread (head, slot) computes one
//              logit, thread 0..g-1 fold the page into that head's running
//              max / sum (online softmax), and thread t accumulates output
//              dimension t.  Partials (max, sum, o) go to the workspace; the
//              unit's last CTA (atomic ticket, no waiting) merges them with
//              the log-sum-exp rule and writes O.  With F = true the CTA reads
//              its pages from the pool through sel_pages and also writes them
//              to kbuf / vbuf / buf_len, so steps a9 and a10 read each page
//              from HBM once.
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 128;  // == kHeadDim: thread t owns output dimension t
constexpr int kMaxG = 16;
constexpr int kKStride = kHeadDim + 4;  // fp32 row stride of the staged K page

template <typename T>
__global__ void __launch_bounds__(kThreads) k_gather(const T *__restrict__ pool_k, const T *__restrict__ pool_v,
                                                     const int32_t *__restrict__ page_len, int page_cap,
                                                     const int32_t *__restrict__ sel_pages,
                                                     const int32_t *__restrict__ sel_count, int max_sel,
                                                     T *__restrict__ kbuf, T *__restrict__ vbuf,
                                                     int32_t *__restrict__ buf_len) {
    const int u = blockIdx.y, x = blockIdx.x;
    const int n = sel_count[u];
    const size_t slot = (size_t)u * max_sel + x;
    if (x >= n) {
        if (threadIdx.x == 0) buf_len[slot] = 0;
        return;
    }
    const int pg = sel_pages[slot];
    constexpr int PV = kPage * row_vecs<T>();  // 16-byte vectors per page
    const size_t src = ((size_t)u * page_cap + pg) * PV;
    const uint4 *sk = reinterpret_cast<const uint4 *>(pool_k) + src;
    const uint4 *sv = reinterpret_cast<const uint4 *>(pool_v) + src;
    uint4 *dk = reinterpret_cast<uint4 *>(kbuf) + slot * PV;
    uint4 *dv = reinterpret_cast<uint4 *>(vbuf) + slot * PV;
    for (int i = threadIdx.x; i < PV; i += kThreads) {
        dk[i] = sk[i];
        dv[i] = sv[i];
    }
    if (threadIdx.x == 0) buf_len[slot] = page_len[(size_t)u * page_cap + pg];
}

template <typename T, bool kFused>
__global__ void __launch_bounds__(kThreads) k_attn(
    const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, const T *__restrict__ pool_k,
    const T *__restrict__ pool_v, const int32_t *__restrict__ page_len, int page_cap,
    const int32_t *__restrict__ sel_pages, T *__restrict__ kbuf, T *__restrict__ vbuf,
    int32_t *__restrict__ buf_len, const int32_t *__restrict__ sel_count, int max_sel, float scale,
    int n_splits, float *__restrict__ part_ml, float *__restrict__ part_o, int32_t *__restrict__ ticket,
    float *__restrict__ O) {
    __shared__ __align__(16) float s_q[kMaxG][kHeadDim];
    __shared__ __align__(16) float s_k[kPage][kKStride];
    __shared__ __align__(16) float s_v[kPage][kHeadDim];
    __shared__ float s_p[kMaxG][kPage];
    __shared__ float s_alpha[kMaxG];
    __shared__ float s_m[kMaxG], s_l[kMaxG];
    __shared__ int s_last;
    const int u = blockIdx.y, split = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int t = threadIdx.x;
    const T *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
    for (int x = t; x < g * kHeadDim; x += kThreads) s_q[x / kHeadDim][x % kHeadDim] = Elem<T>::load(Qu + x);
    if (t < g) {
        s_m[t] = -INFINITY;
        s_l[t] = 0.f;
    }
    float o[kMaxG];
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh) o[hh] = 0.f;

    const int n = sel_count[u];
    const int x0 = split * kAttnPagesPerSplit;
    const int x1 = min(n, x0 + kAttnPagesPerSplit);
    constexpr int RV = row_vecs<T>();
    constexpr int PVEC = kPage * RV;
    constexpr int EPV = Elem<T>::kPerVec;
    for (int x = x0; x < x1; ++x) {
        const size_t slot = (size_t)u * max_sel + x;
        const uint4 *sk, *sv;
        int len;
        if (kFused) {
            const int pg = sel_pages[slot];
            const size_t src = ((size_t)u * page_cap + pg) * PVEC;
            sk = reinterpret_cast<const uint4 *>(pool_k) + src;
            sv = reinterpret_cast<const uint4 *>(pool_v) + src;
            len = page_len[(size_t)u * page_cap + pg];
        } else {
            sk = reinterpret_cast<const uint4 *>(kbuf) + slot * PVEC;
            sv = reinterpret_cast<const uint4 *>(vbuf) + slot * PVEC;
            len = buf_len[slot];
        }
        __syncthreads();  // previous page fully consumed
        for (int i = t; i < PVEC; i += kThreads) {
            const uint4 kv = sk[i], vv = sv[i];
            if (kFused) {
                reinterpret_cast<uint4 *>(kbuf)[slot * PVEC + i] = kv;
                reinterpret_cast<uint4 *>(vbuf)[slot * PVEC + i] = vv;
            }
            const int r = i / RV, c = (i % RV) * EPV;
            float f[EPV];
            Elem<T>::unpack(kv, f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) s_k[r][c + e] = f[e];
            Elem<T>::unpack(vv, f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) s_v[r][c + e] = f[e];
        }
        if (kFused && t == 0) buf_len[slot] = len;
        __syncthreads();
        // logits: thread (head, slot)
        for (int hs = t; hs < g * kPage; hs += kThreads) {
            const int hh = hs / kPage, sl = hs % kPage;
            float acc = 0.f;
            const float4 *kr = reinterpret_cast<const float4 *>(&s_k[sl][0]);
            const float4 *qr = reinterpret_cast<const float4 *>(&s_q[hh][0]);
#pragma unroll 8
            for (int i = 0; i < kHeadDim / 4; ++i) {
                const float4 a = kr[i], qq = qr[i];
                acc = fmaf(qq.x, a.x, acc);
                acc = fmaf(qq.y, a.y, acc);
                acc = fmaf(qq.z, a.z, acc);
                acc = fmaf(qq.w, a.w, acc);
            }
            s_p[hh][sl] = sl < len ? acc * scale : -INFINITY;
        }
        __syncthreads();
        // online softmax bookkeeping, one thread per head
        if (t < g) {
            float pmax = -INFINITY;
            for (int sl = 0; sl < kPage; ++sl) pmax = fmaxf(pmax, s_p[t][sl]);
            const float m_old = s_m[t];
            const float m_new = fmaxf(m_old, pmax);
            const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
            float sum = 0.f;
            for (int sl = 0; sl < kPage; ++sl) {
                const float lg = s_p[t][sl];
                const float pr = (lg == -INFINITY) ? 0.f : expf(lg - m_new);
                s_p[t][sl] = pr;
                sum += pr;
            }
            s_alpha[t] = alpha;
            s_l[t] = s_l[t] * alpha + sum;
            s_m[t] = m_new;
        }
        __syncthreads();
#pragma unroll
        for (int hh = 0; hh < kMaxG; ++hh) {
            if (hh < g) {
                float acc = o[hh] * s_alpha[hh];
#pragma unroll
                for (int sl = 0; sl < kPage; ++sl) acc = fmaf(s_p[hh][sl], s_v[sl][t], acc);
                o[hh] = acc;
            }
        }
    }
    if (kFused) {  // slots of this split past the selection hold no page
        for (int x = max(x0, n) + t; x < min(x0 + kAttnPagesPerSplit, max_sel); x += kThreads)
            buf_len[(size_t)u * max_sel + x] = 0;
    }
    __syncthreads();
    // partials of this split
    const size_t pbase = ((size_t)u * n_splits + split) * g;
    if (t < g) {
        part_ml[(pbase + t) * 2 + 0] = s_m[t];
        part_ml[(pbase + t) * 2 + 1] = s_l[t];
    }
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh)
        if (hh < g) part_o[(pbase + hh) * kHeadDim + t] = o[hh];
    __threadfence();
    __syncthreads();
    if (t == 0) s_last = (atomicAdd(ticket + u, 1) == n_splits - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // merge the unit's splits (log-sum-exp)
    for (int hh = 0; hh < g; ++hh) {
        float M = -INFINITY;
        for (int sp = 0; sp < n_splits; ++sp)
            M = fmaxf(M, __ldcg(part_ml + ((((size_t)u * n_splits + sp) * g + hh) * 2)));
        float Lsum = 0.f, acc = 0.f;
        if (M != -INFINITY) {
            for (int sp = 0; sp < n_splits; ++sp) {
                const size_t pb = ((size_t)u * n_splits + sp) * g + hh;
                const float ms = __ldcg(part_ml + pb * 2);
                if (ms == -INFINITY) continue;
                const float w = expf(ms - M);
                Lsum = fmaf(__ldcg(part_ml + pb * 2 + 1), w, Lsum);
                acc = fmaf(__ldcg(part_o + pb * kHeadDim + t), w, acc);
            }
        }
        O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + t] = Lsum > 0.f ? acc / Lsum : 0.f;
    }
    if (t == 0) ticket[u] = 0;
}

template <typename T>
cudaError_t gather_t(const ice_params &p, const ice_index &idx, const int32_t *sel_pages, const int32_t *sel_count,
                     int max_sel, void *kbuf, void *vbuf, int32_t *buf_len, cudaStream_t s) {
    dim3 grid(max_sel, units_of(p));
    k_gather<T><<<grid, kThreads, 0, s>>>(static_cast<const T *>(idx.pool_k), static_cast<const T *>(idx.pool_v),
                                          idx.page_len, p.page_cap, sel_pages, sel_count, max_sel,
                                          static_cast<T *>(kbuf), static_cast<T *>(vbuf), buf_len);
    return cudaGetLastError();
}

template <typename T>
cudaError_t attn_t(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q, void *kbuf,
                   void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale, float *O,
                   const DecodeWs &ws, cudaStream_t s) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    cudaMemsetAsync(ws.attn_ticket, 0, sizeof(int32_t) * U, s);
    dim3 grid(ws.n_splits, U);
    const T *pk = pool ? static_cast<const T *>(pool->pool_k) : nullptr;
    const T *pv = pool ? static_cast<const T *>(pool->pool_v) : nullptr;
    const int32_t *pl = pool ? pool->page_len : nullptr;
    if (pool)
        k_attn<T, true><<<grid, kThreads, 0, s>>>(static_cast<const T *>(Q), g, p.n_q_heads, p.n_kv_heads, pk, pv,
                                                  pl, p.page_cap, sel_pages, static_cast<T *>(kbuf),
                                                  static_cast<T *>(vbuf), buf_len, sel_count, max_sel, scale,
                                                  ws.n_splits, ws.part_ml, ws.part_o, ws.attn_ticket, O);
    else
        k_attn<T, false><<<grid, kThreads, 0, s>>>(static_cast<const T *>(Q), g, p.n_q_heads, p.n_kv_heads, pk, pv,
                                                   pl, p.page_cap, sel_pages, static_cast<T *>(kbuf),
                                                   static_cast<T *>(vbuf), buf_len, sel_count, max_sel, scale,
                                                   ws.n_splits, ws.part_ml, ws.part_o, ws.attn_ticket, O);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const ice_params &p, const ice_index &idx, const int32_t *sel_pages,
                          const int32_t *sel_count, int max_sel, void *kbuf, void *vbuf, int32_t *buf_len,
                          cudaStream_t s) {
    if (p.dtype == ICE_BF16) return gather_t<__nv_bfloat16>(p, idx, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, s);
    return gather_t<float>(p, idx, sel_pages, sel_count, max_sel, kbuf, vbuf, buf_len, s);
}

cudaError_t launch_attention(const ice_params &p, const ice_index *pool, const int32_t *sel_pages, const void *Q,
                             void *kbuf, void *vbuf, int32_t *buf_len, const int32_t *sel_count, int max_sel,
                             float scale, float *O, const DecodeWs &ws, cudaStream_t s) {
    if (p.dtype == ICE_BF16)
        return attn_t<__nv_bfloat16>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, s);
    return attn_t<float>(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel, scale, O, ws, s);
}

}  // namespace ice

// ---------------------------------------------------------------------------
// Allocation-free attention: the same split-KV kernel, with its scratch (one
// ticket word per unit and the per-split partials) in a fixed device array
// that the library owns, so the caller passes no workspace.
// ---------------------------------------------------------------------------
#include <mutex>

namespace ice {
namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ICE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current and cached.
cudaError_t noalloc_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

size_t attention_noalloc_bytes(const ice_params &p, int max_sel) {
    return decode_ws_layout(p, 0, max_sel, nullptr).bytes;
}

cudaError_t launch_attention_noalloc(const ice_params &p, const void *Q, const void *kbuf, const void *vbuf,
                                     const int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale,
                                     float *O, cudaStream_t s) {
    void *base = nullptr;
    cudaError_t e = noalloc_scratch(&base);
    if (e != cudaSuccess) return e;
    const DecodeWs ws = decode_ws_layout(p, 0, max_sel, base);
    if (ws.bytes > ICE_NOALLOC_SCRATCH_BYTES) return cudaErrorInvalidValue;
    return launch_attention(p, nullptr, nullptr, Q, const_cast<void *>(kbuf), const_cast<void *>(vbuf),
                            const_cast<int32_t *>(buf_len), sel_count, max_sel, scale, O, ws, s);
}

}  // namespace ice
