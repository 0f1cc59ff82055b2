// Decode steps a6 (score the parent level), a7 (top-k pages per query head)
// and a8 (GQA union).
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 3: at decode time every attention head picks
// its own top-k pages; for grouped-query attention the query heads of one
// group take the union of their picks and share it.  IceCache popular-
// science article (aitangshan.cn/news/751385), section 六: the union is
// computed over the query heads of a group; the query transform adds a zero
// coordinate, so |q' - p'|^2 = |q|^2 + M^2 - 2 q.p and the nearest lifted
// parents are the parents of largest q.p.
//
// One launch, grid (chunks of 256 parents, units), 256 threads:
//   1. each thread scores one parent against the g query heads (16-byte
//      loads of the parent row, 8 in flight; fp32 FMA in element order);
//   2. per query head the chunk's 256 (score, m) pairs are packed into
//      64-bit keys ordered like (-score, m) and sorted by a block-wide bitonic
//      network in shared memory; the first kc = min(k, 256) go to the
//      workspace together with each parent's page span (first page, page
//      count, contiguity), so the merge needs no further dependent loads;
//   3. the last CTA of the unit to finish (atomic ticket, no waiting; the
//      ticket is back at zero when the kernel ends) sorts each head's
//      n_chunks * kc candidates the same way, walks the ordered parents
//      taking their pages in page-id order until k pages are taken, ORs the
//      pages into a shared-memory bitmask over the unit's pages (the GQA
//      union), and writes the set bits in ascending order.
// Each page inherits its parent's score and the pages of one parent are
// taken in ascending page id, so expanding the top parents in (-score, m)
// order reproduces the (-score, page id) order over pages: page ids ascend
// with m at build time, and pages appended by an insert come after their
// parent's earlier pages through the page_next chain.
#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ice {
namespace {

using namespace topk;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kHeadTile = 8;  // query heads scored per pass over a parent row


// Sorts rows[r][0..n) descending for r < nrows (n a power of two) with every
// thread of the block; ends with a barrier.
__device__ void block_bitonic_desc(unsigned long long *keys, int nrows, int n) {
    const int pairs = nrows * (n / 2);
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int x = threadIdx.x; x < pairs; x += blockDim.x) {
                const int r = x / (n / 2), p = x % (n / 2);
                const int i = 2 * p - (p & (stride - 1));
                const int j = i + stride;
                unsigned long long *row = keys + (size_t)r * n;
                const unsigned long long a = row[i], b = row[j];
                const bool desc = ((i & size) == 0);
                if (desc ? (a < b) : (a > b)) {
                    row[i] = b;
                    row[j] = a;
                }
            }
            __syncthreads();
        }
    }
}

__host__ __device__ inline int pow2_at_least(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

struct SelectSmem {
    size_t q, keys, mask, total;
};
// phase 1-2: q [g][d] f32 + keys [g][256]; phase 3: keys [g][n2] + mask.
__host__ __device__ inline SelectSmem select_smem(int g, int n_chunks, int kc, int page_cap) {
    auto al = [](size_t x) { return (x + 15) & ~(size_t)15; };
    SelectSmem L{};
    L.q = 0;
    L.keys = al(sizeof(float) * (size_t)g * kHeadDim);
    const int n2 = pow2_at_least(n_chunks * kc);
    const size_t kbytes = sizeof(unsigned long long) * (size_t)g * (n2 > kSelChunk ? n2 : kSelChunk);
    L.mask = L.keys + al(kbytes);
    L.total = L.mask + al(sizeof(unsigned) * (size_t)((page_cap + 31) / 32));
    return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_select(
    const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, int np_cap, int page_cap, int k_pages, int kc,
    int n_chunks, const int32_t *__restrict__ n_parents, const int32_t *__restrict__ n_pages,
    const T *__restrict__ parent_keys, const int32_t *__restrict__ parent_first_page,
    const int32_t *__restrict__ parent_last_page, const int32_t *__restrict__ parent_n_pages,
    const int32_t *__restrict__ page_next, unsigned long long *__restrict__ cand_key, int4 *__restrict__ cand_span,
    int32_t *__restrict__ ticket, int32_t *__restrict__ sel_pages, int32_t *__restrict__ sel_count, int max_sel,
    int n_pos, int32_t *__restrict__ err) {
    extern __shared__ __align__(16) unsigned char smem[];
    const SelectSmem L = select_smem(g, n_chunks, kc, page_cap);
    float *s_q = reinterpret_cast<float *>(smem + L.q);
    unsigned long long *s_key = reinterpret_cast<unsigned long long *>(smem + L.keys);
    unsigned *s_mask = reinterpret_cast<unsigned *>(smem + L.mask);
    __shared__ int s_last;
    __shared__ int s_wsum[kWarps];
    __shared__ int s_carry;

    const int u = blockIdx.y, chunk = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;

    // ---- 1. scores of this chunk's parents against the g query heads
    const T *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
    for (int x = threadIdx.x; x < g * kHeadDim; x += kThreads) s_q[x] = Elem<T>::load(Qu + x);
    const int m = chunk * kSelChunk + threadIdx.x;
    const bool valid = m < Np;
    const uint4 *row = reinterpret_cast<const uint4 *>(parent_keys + (up + (valid ? m : 0)) * kHeadDim);
    constexpr int RV = row_vecs<T>();
    constexpr int PV = Elem<T>::kPerVec;
    __syncthreads();
    for (int h0 = 0; h0 < g; h0 += kHeadTile) {
        float acc[kHeadTile];
#pragma unroll
        for (int t = 0; t < kHeadTile; ++t) acc[t] = 0.f;
        if (valid) {
            constexpr int LB = 8;  // 16-byte loads in flight per thread
#pragma unroll
            for (int v0 = 0; v0 < RV; v0 += LB) {
                uint4 raw[LB];
#pragma unroll
                for (int i = 0; i < LB; ++i) raw[i] = __ldg(row + v0 + i);
#pragma unroll
                for (int i = 0; i < LB; ++i) {
                    float f[PV];
                    Elem<T>::unpack(raw[i], f);
#pragma unroll
                    for (int t = 0; t < kHeadTile; ++t) {
                        if (h0 + t < g) {
                            const float4 *qq =
                                reinterpret_cast<const float4 *>(s_q + (size_t)(h0 + t) * kHeadDim + (v0 + i) * PV);
#pragma unroll
                            for (int e4 = 0; e4 < PV / 4; ++e4) {
                                const float4 qv = qq[e4];
                                acc[t] = fmaf(qv.x, f[4 * e4 + 0], acc[t]);
                                acc[t] = fmaf(qv.y, f[4 * e4 + 1], acc[t]);
                                acc[t] = fmaf(qv.z, f[4 * e4 + 2], acc[t]);
                                acc[t] = fmaf(qv.w, f[4 * e4 + 3], acc[t]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kHeadTile; ++t)
            if (h0 + t < g)
                s_key[(size_t)(h0 + t) * kSelChunk + threadIdx.x] = valid ? sort_key(acc[t], m) : 0ull;
    }
    // the page span of this thread's parent rides along with its candidates
    int4 span = make_int4(0, 0, 0, 0);
    if (valid) {
        const int fp = parent_first_page[up + m], np = parent_n_pages[up + m];
        span = make_int4(fp, np, parent_last_page[up + m] - fp + 1 == np ? 1 : 0, m);
    }
    __syncthreads();
    // ---- 2. this chunk's ordered top-kc parents per query head
    block_bitonic_desc(s_key, g, kSelChunk);
    for (int x = threadIdx.x; x < g * kc; x += kThreads) {
        const int hh = x / kc, r = x % kc;
        const size_t o = (((size_t)u * n_chunks + chunk) * g + hh) * kc + r;
        cand_key[o] = s_key[(size_t)hh * kSelChunk + r];
    }
    // spans indexed by (chunk, position of the parent inside the chunk)
    cand_span[((size_t)u * n_chunks + chunk) * kSelChunk + threadIdx.x] = span;

    // ---- 3. the unit's last CTA merges (no CTA waits for another)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(ticket + u, 1) == n_chunks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    const int P = min(n_pages[u], page_cap);
    const int Ps = max(0, P - n_pos);  // semantic pages; the positional rest is always in the union
    const int words = (P + 31) / 32;
    for (int x = threadIdx.x; x < words; x += kThreads) s_mask[x] = 0u;
    if (k_pages >= Ps) {
        __syncthreads();
        for (int x = threadIdx.x; x < words; x += kThreads) {
            const int rem = P - x * 32;
            s_mask[x] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
        }
    } else {
        const int nc = n_chunks * kc;
        const int n2 = pow2_at_least(nc);
        for (int x = threadIdx.x; x < g * n2; x += kThreads) {
            const int hh = x / n2, r = x % n2;
            unsigned long long k = 0ull;
            if (r < nc) {
                const int c = r / kc, t = r % kc;
                k = __ldcg(cand_key + (((size_t)u * n_chunks + c) * g + hh) * kc + t);
            }
            s_key[x] = k;
        }
        __syncthreads();
        for (int x = Ps + threadIdx.x; x < P; x += kThreads) atomicOr(&s_mask[x >> 5], 1u << (x & 31));
        block_bitonic_desc(s_key, g, n2);
        // one warp per head: take pages of the ordered parents until k pages
        const int kt = min(k_pages, nc);
        for (int hh = warp; hh < g; hh += kWarps) {
            int taken = 0;
            for (int r0 = 0; r0 < kt && taken < k_pages; r0 += 32) {
                int cnt = 0;
                int4 sp = make_int4(0, 0, 0, 0);
                if (r0 + lane < kt) {
                    const unsigned long long k = s_key[(size_t)hh * n2 + r0 + lane];
                    if (k != 0ull) {
                        const int pm = key_id(k);
                        sp = __ldcg(cand_span + ((size_t)u * n_chunks + pm / kSelChunk) * kSelChunk + pm % kSelChunk);
                        cnt = sp.y;
                    }
                }
                int incl = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                const int take = max(0, min(cnt, k_pages - (taken + incl - cnt)));
                int pg = sp.x;
                for (int i = 0; i < take; ++i) {
                    const int q = sp.z ? pg + i : pg;
                    if (q < 0 || q >= Ps) break;
                    atomicOr(&s_mask[q >> 5], 1u << (q & 31));
                    if (!sp.z) pg = page_next[ug + q];
                }
                taken += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
    }
    __syncthreads();
    // ascending list of the union's pages
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (int w0 = 0; w0 < words; w0 += kThreads) {
        const int x = w0 + threadIdx.x;
        const unsigned bits = x < words ? s_mask[x] : 0u;
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int pos = s_carry;
        for (int w = 0; w < warp; ++w) pos += s_wsum[w];
        pos += incl - c;
        unsigned bb = bits;
        while (bb) {
            const int bit = __ffs(bb) - 1;
            bb &= bb - 1;
            if (pos < max_sel) sel_pages[(size_t)u * max_sel + pos] = x * 32 + bit;
            ++pos;
        }
        __syncthreads();
        if (threadIdx.x == kThreads - 1) s_carry = pos;
        __syncthreads();
    }
    const int total = s_carry;
    for (int x = total + threadIdx.x; x < max_sel; x += kThreads) sel_pages[(size_t)u * max_sel + x] = -1;
    if (threadIdx.x == 0) {
        if (total > max_sel) set_err(err, ICE_ERR_CAPACITY);
        sel_count[u] = min(total, max_sel);
        ticket[u] = 0;  // ready for the next call
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                     int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    const int kc = ws.k_pages < kSelChunk ? ws.k_pages : kSelChunk;
    const size_t smem = select_smem(g, ws.n_chunks, kc > 0 ? kc : 1, p.page_cap).total;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_select<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(ws.n_chunks, U);
    k_select<T><<<grid, kThreads, smem, s>>>(
        static_cast<const T *>(Q), g, p.n_q_heads, p.n_kv_heads, p.np_cap, p.page_cap, ws.k_pages, kc > 0 ? kc : 1,
        ws.n_chunks, idx.n_parents, idx.n_pages, static_cast<const T *>(idx.parent_keys), idx.parent_first_page,
        idx.parent_last_page, idx.parent_n_pages, idx.page_next, ws.cand_key, ws.cand_span, ws.sel_ticket,
        sel_pages, sel_count, max_sel, pos_split(p).n_pos, err);
    return cudaGetLastError();
}

}  // namespace

size_t select_smem_bytes(const ice_params &p, int k_pages, int n_chunks) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const int kc = k_pages < kSelChunk ? k_pages : kSelChunk;
    return select_smem(g, n_chunks, kc > 0 ? kc : 1, p.page_cap).total;
}

cudaError_t launch_select(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                          int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    if (select_tc_supported(p, ws.k_pages)) {
        const cudaError_t e = launch_select_tc(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
        if (e != cudaErrorNotSupported) return e;
    }
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
    return launch_t<float>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
}

}  // namespace ice
