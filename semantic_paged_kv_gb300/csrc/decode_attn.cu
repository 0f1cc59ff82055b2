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
//              g query heads of its GQA group.  All of the split's page loads
//              are issued at once (16-byte vectors into registers), then
//              staged in shared memory in the storage dtype.  Per page: the
//              logits are split over the head dimension (16 lanes x 8
//              elements, two slots per lane group, shuffle reduction), a
//              16-lane group per head folds the page into that head's running
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
    constexpr int PPS = kAttnPagesPerSplit;
    constexpr int RV = row_vecs<T>();        // 16-byte vectors per row
    constexpr int PVEC = kPage * RV;         // 16-byte vectors per page
    constexpr int VPT = PVEC / kThreads;     // vectors per thread per page and tensor
    constexpr int CV = 8 / Elem<T>::kPerVec; // vectors per 8-element chunk (1 bf16, 2 fp32)
    extern __shared__ __align__(16) uint4 s_kv[];  // [PPS][K, V][PVEC], reused by the merge
    __shared__ __align__(16) float s_q[kMaxG][kHeadDim];
    __shared__ float s_p[kMaxG][kPage];
    __shared__ float s_alpha[kMaxG], s_m[kMaxG], s_l[kMaxG];
    __shared__ int s_len[PPS];
    __shared__ int s_last;
    const int u = blockIdx.y, split = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int t = threadIdx.x, lane = t & 31;
    const T *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
    for (int x = t; x < g * kHeadDim; x += kThreads) s_q[x / kHeadDim][x % kHeadDim] = Elem<T>::load(Qu + x);
    if (t < g) {
        s_m[t] = -INFINITY;
        s_l[t] = 0.f;
    }
    const int n = sel_count[u];
    const int x0 = split * PPS;
    const int np = max(0, min(PPS, n - x0));

    // ---- stage the split's pages: all loads in flight at once
    uint4 rk[PPS][VPT], rv[PPS][VPT];
#pragma unroll
    for (int i = 0; i < PPS; ++i) {
        if (i < np) {
            const size_t slot = (size_t)u * max_sel + x0 + i;
            const uint4 *sk, *sv;
            if (kFused) {
                const size_t src = ((size_t)u * page_cap + sel_pages[slot]) * PVEC;
                sk = reinterpret_cast<const uint4 *>(pool_k) + src;
                sv = reinterpret_cast<const uint4 *>(pool_v) + src;
            } else {
                sk = reinterpret_cast<const uint4 *>(kbuf) + slot * PVEC;
                sv = reinterpret_cast<const uint4 *>(vbuf) + slot * PVEC;
            }
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                rk[i][v] = sk[t + v * kThreads];
                rv[i][v] = sv[t + v * kThreads];
            }
        }
    }
    if (t < np) {
        const size_t slot = (size_t)u * max_sel + x0 + t;
        if (kFused) {
            const int len = page_len[(size_t)u * page_cap + sel_pages[slot]];
            s_len[t] = len;
            if (buf_len) buf_len[slot] = len;
        } else {
            s_len[t] = buf_len[slot];
        }
    }
    if (kFused && buf_len) {  // slots of this split past the selection hold no page
        for (int x = max(x0, n) + t; x < min(x0 + PPS, max_sel); x += kThreads) buf_len[(size_t)u * max_sel + x] = 0;
    }
#pragma unroll
    for (int i = 0; i < PPS; ++i) {
        if (i < np) {
            const size_t slot = (size_t)u * max_sel + x0 + i;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                s_kv[(2 * i) * PVEC + t + v * kThreads] = rk[i][v];
                s_kv[(2 * i + 1) * PVEC + t + v * kThreads] = rv[i][v];
                if (kFused && buf_len) {  // no buf_len: no contiguous copy
                    reinterpret_cast<uint4 *>(kbuf)[slot * PVEC + t + v * kThreads] = rk[i][v];
                    reinterpret_cast<uint4 *>(vbuf)[slot * PVEC + t + v * kThreads] = rv[i][v];
                }
            }
        }
    }
    __syncthreads();

    float o[kMaxG];
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh) o[hh] = 0.f;
    const int c = t & 15;      // 8-element chunk of the head dimension
    const int sg = t >> 4;     // slots 2 sg and 2 sg + 1
    for (int i = 0; i < np; ++i) {
        const uint4 *Kp = s_kv + (2 * i) * PVEC;
        const T *Vp = reinterpret_cast<const T *>(s_kv + (2 * i + 1) * PVEC);
        const int len = s_len[i];
        // logits: split-K over 16 lanes, 8 elements each, 2 slots per lane group
        float kf[2][8];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int w = 0; w < CV; ++w) Elem<T>::unpack(Kp[(2 * sg + r) * RV + c * CV + w], &kf[r][w * Elem<T>::kPerVec]);
        }
        for (int hh = 0; hh < g; ++hh) {
            const float4 q0 = reinterpret_cast<const float4 *>(&s_q[hh][8 * c])[0];
            const float4 q1 = reinterpret_cast<const float4 *>(&s_q[hh][8 * c])[1];
            float a[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float x = q0.x * kf[r][0];
                x = fmaf(q0.y, kf[r][1], x);
                x = fmaf(q0.z, kf[r][2], x);
                x = fmaf(q0.w, kf[r][3], x);
                x = fmaf(q1.x, kf[r][4], x);
                x = fmaf(q1.y, kf[r][5], x);
                x = fmaf(q1.z, kf[r][6], x);
                x = fmaf(q1.w, kf[r][7], x);
                a[r] = x;
            }
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) {
                a[0] += __shfl_xor_sync(0xffffffffu, a[0], off);
                a[1] += __shfl_xor_sync(0xffffffffu, a[1], off);
            }
            if (c == 0) {
                s_p[hh][2 * sg] = a[0];
                s_p[hh][2 * sg + 1] = a[1];
            }
        }
        __syncthreads();
        // online softmax: lane group of 16 per head
        for (int hs0 = 0; hs0 < g * kPage; hs0 += kThreads) {
            const int hs = hs0 + t;
            const int hh = hs / kPage, sl = hs % kPage;
            const bool on = hh < g;
            const float lg = (on && sl < len) ? s_p[hh][sl] * scale : -INFINITY;
            float pmax = lg;
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, off));
            const float m_old = on ? s_m[hh] : -INFINITY;
            const float m_new = fmaxf(m_old, pmax);
            const float pr = (lg == -INFINITY) ? 0.f : expf(lg - m_new);
            float psum = pr;
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            if (on) s_p[hh][sl] = pr;
            __syncwarp();
            if (on && sl == 0) {
                const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
                s_alpha[hh] = alpha;
                s_l[hh] = s_l[hh] * alpha + psum;
                s_m[hh] = m_new;
            }
        }
        __syncthreads();
        // o[h][t] += sum_s p[h][s] v[s][t]
        float vt[kPage];
#pragma unroll
        for (int sl = 0; sl < kPage; ++sl) vt[sl] = Elem<T>::load(Vp + sl * kHeadDim + t);
#pragma unroll
        for (int hh = 0; hh < kMaxG; ++hh) {
            if (hh < g) {
                float acc = o[hh] * s_alpha[hh];
#pragma unroll
                for (int sl = 0; sl < kPage; ++sl) acc = fmaf(s_p[hh][sl], vt[sl], acc);
                o[hh] = acc;
            }
        }
        __syncthreads();
    }
    (void)lane;
    // ---- partials of this split
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
    // ---- the unit's last CTA merges the splits (log-sum-exp)
    float *s_w = reinterpret_cast<float *>(s_kv);  // [n_splits * g] weights, then [g] totals
    const int ns_g = n_splits * g;
    const float *ml = part_ml + (size_t)u * ns_g * 2;
    for (int x = t; x < ns_g; x += kThreads) s_w[x] = __ldcg(ml + 2 * x);
    __syncthreads();
    if (t < g) {
        float M = -INFINITY;
        for (int sp = 0; sp < n_splits; ++sp) M = fmaxf(M, s_w[sp * g + t]);
        s_m[t] = M;
    }
    __syncthreads();
    for (int x = t; x < ns_g; x += kThreads) {
        const float ms = s_w[x], M = s_m[x % g];
        s_w[x] = (ms == -INFINITY) ? 0.f : expf(ms - M);
    }
    __syncthreads();
    if (t < g) {
        float L = 0.f;
        for (int sp = 0; sp < n_splits; ++sp) L = fmaf(__ldcg(ml + 2 * (sp * g + t) + 1), s_w[sp * g + t], L);
        s_l[t] = L;
    }
    __syncthreads();
    const float *po = part_o + (size_t)u * ns_g * kHeadDim;
    float acc[kMaxG];
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh) acc[hh] = 0.f;
    for (int sp = 0; sp < n_splits; ++sp) {
#pragma unroll
        for (int hh = 0; hh < kMaxG; ++hh)
            if (hh < g) acc[hh] = fmaf(__ldcg(po + ((size_t)sp * g + hh) * kHeadDim + t), s_w[sp * g + hh], acc[hh]);
    }
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh)
        if (hh < g) {
            const float L = s_l[hh];
            O[((size_t)b * n_q_heads + (size_t)h * g + hh) * kHeadDim + t] = L > 0.f ? acc[hh] / L : 0.f;
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
    dim3 grid(ws.n_splits, U);  // the tickets are zero between calls
    const T *pk = pool ? static_cast<const T *>(pool->pool_k) : nullptr;
    const T *pv = pool ? static_cast<const T *>(pool->pool_v) : nullptr;
    const int32_t *pl = pool ? pool->page_len : nullptr;
    const size_t stage = sizeof(uint4) * 2 * kAttnPagesPerSplit * kPage * row_vecs<T>();
    const size_t merge = sizeof(float) * (size_t)ws.n_splits * g;
    const size_t smem = stage > merge ? stage : merge;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(pool ? (const void *)k_attn<T, true> : (const void *)k_attn<T, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (pool)
        k_attn<T, true><<<grid, kThreads, smem, s>>>(static_cast<const T *>(Q), g, p.n_q_heads, p.n_kv_heads, pk, pv,
                                                  pl, p.page_cap, sel_pages, static_cast<T *>(kbuf),
                                                  static_cast<T *>(vbuf), buf_len, sel_count, max_sel, scale,
                                                  ws.n_splits, ws.part_ml, ws.part_o, ws.attn_ticket, O);
    else
        k_attn<T, false><<<grid, kThreads, smem, s>>>(static_cast<const T *>(Q), g, p.n_q_heads, p.n_kv_heads, pk, pv,
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
                             float scale, float *O, const DecodeWs &ws, cudaStream_t s, int32_t *err) {
    if (attention_mma_fits(p, max_sel)) {
        const cudaError_t e = launch_attention_mma(p, pool, sel_pages, Q, kbuf, vbuf, buf_len, sel_count, max_sel,
                                                   scale, O, ws, err, s);
        if (e != cudaErrorNotSupported) return e;
    }
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
    return decode_ws_layout(p, 0, max_sel, nullptr, false).bytes;
}

cudaError_t launch_attention_noalloc(const ice_params &p, const void *Q, const void *kbuf, const void *vbuf,
                                     const int32_t *buf_len, const int32_t *sel_count, int max_sel, float scale,
                                     float *O, cudaStream_t s) {
    void *base = nullptr;
    cudaError_t e = noalloc_scratch(&base);
    if (e != cudaSuccess) return e;
    const DecodeWs ws = decode_ws_layout(p, 0, max_sel, base, false);
    if (ws.bytes > ICE_NOALLOC_SCRATCH_BYTES) return cudaErrorInvalidValue;
    e = cudaMemsetAsync(ws.attn_ticket, 0, sizeof(int32_t) * units_of(p), s);
    if (e != cudaSuccess) return e;
    return launch_attention(p, nullptr, nullptr, Q, const_cast<void *>(kbuf), const_cast<void *>(vbuf),
                            const_cast<int32_t *>(buf_len), sel_count, max_sel, scale, O, ws, s);
}

}  // namespace ice
