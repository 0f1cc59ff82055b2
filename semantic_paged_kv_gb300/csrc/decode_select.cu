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
//      loads of the parent row, fp32 FMA);
//   2. warp h keeps the chunk's best kc = min(k, 256) parents of query head
//      h, in the order (-score, m), by kc rounds of a warp argmax, and
//      writes them (sorted) to the workspace;
//   3. the last CTA of the unit to finish (atomic ticket, no waiting) stages
//      each head's sorted chunk lists in shared memory and k-way merges them
//      (one warp per head, lanes own chunk lists) into the head's ordered top
//      parents; it expands those parents into their pages in page-id order
//      until k pages are taken, ORs the pages into a shared-memory bitmask
//      over the unit's pages (the GQA union), and writes the set bits in
//      ascending order.
// Each page inherits its parent's score and the pages of one parent are
// taken in ascending page id, so expanding the top parents in (-score, m)
// order reproduces the (-score, page id) order over pages: page ids ascend
// with m at build time, and pages appended by an insert come after their
// parent's earlier pages through the page_next chain.
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kHeadTile = 8;  // query heads scored per pass over a parent row

__device__ __forceinline__ void warp_best(float &s, int &i) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, s, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        if (better(os, oi, s, i)) {
            s = os;
            i = oi;
        }
    }
}

// kc rounds of a warp argmax over (score[x], id[x]), x < n (shared memory);
// the ordered winners go to out_s / out_i (global).
__device__ void warp_topk(const float *score, const int *id, unsigned char *taken, int n, int kc, float *out_s,
                          int32_t *out_i) {
    const int lane = threadIdx.x & 31;
    for (int x = lane; x < n; x += 32) taken[x] = 0;
    __syncwarp();
    for (int r = 0; r < kc; ++r) {
        float bs = -INFINITY;
        int bi = 0x7fffffff, bx = -1;
        for (int x = lane; x < n; x += 32) {
            if (taken[x]) continue;
            if (bx < 0 || better(score[x], id[x], bs, bi)) {
                bs = score[x];
                bi = id[x];
                bx = x;
            }
        }
        float ws = bs;
        int wi = bi;
        warp_best(ws, wi);
        if (bx >= 0 && bi == wi && bs == ws) taken[bx] = 1;  // ids are unique among valid entries
        if (lane == 0) {
            out_s[r] = ws;
            out_i[r] = wi;
        }
        __syncwarp();
    }
}

struct SelectSmem {
    // phase 1-2
    size_t q, sc, id, taken, front;
    // phase 3
    size_t mask, msc, mid, mptr, mtop, back;
    size_t total;
};

__host__ __device__ inline SelectSmem select_smem(int g, int n_chunks, int kc, int kt, int page_cap) {
    auto al = [](size_t x) { return (x + 15) & ~(size_t)15; };
    SelectSmem L{};
    L.q = 0;
    L.sc = L.q + al(sizeof(float) * (size_t)g * kHeadDim);
    L.id = L.sc + al(sizeof(float) * (size_t)g * kSelChunk);
    L.taken = L.id + al(sizeof(int) * kSelChunk);
    L.front = L.taken + al((size_t)kWarps * kSelChunk);
    L.mask = 0;
    L.msc = L.mask + al(sizeof(unsigned) * (size_t)((page_cap + 31) / 32));
    const size_t per_warp = (size_t)n_chunks * kc;
    L.mid = L.msc + al(sizeof(float) * per_warp * kWarps);
    L.mptr = L.mid + al(sizeof(int) * per_warp * kWarps);
    L.mtop = L.mptr + al(sizeof(int) * (size_t)n_chunks * kWarps);
    L.back = L.mtop + al(sizeof(int) * (size_t)kt * kWarps);
    L.total = L.front > L.back ? L.front : L.back;
    return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_select(
    const T *__restrict__ Q, int g, int n_q_heads, int n_kv_heads, int np_cap, int page_cap, int k_pages, int kc,
    int kt, int n_chunks, const int32_t *__restrict__ n_parents, const int32_t *__restrict__ n_pages,
    const T *__restrict__ parent_keys, const int32_t *__restrict__ parent_first_page,
    const int32_t *__restrict__ parent_last_page, const int32_t *__restrict__ parent_n_pages,
    const int32_t *__restrict__ page_next, float *__restrict__ cand_score, int32_t *__restrict__ cand_id,
    int32_t *__restrict__ ticket, int32_t *__restrict__ sel_pages, int32_t *__restrict__ sel_count, int max_sel,
    int32_t *__restrict__ err) {
    extern __shared__ __align__(16) unsigned char smem[];
    const SelectSmem L = select_smem(g, n_chunks, kc, kt, page_cap);
    __shared__ int s_last;
    __shared__ int s_wsum[kWarps];
    __shared__ int s_carry;

    const int u = blockIdx.y, chunk = blockIdx.x;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);

    // ---- 1. scores of this chunk's parents against the g query heads
    {
        float *s_q = reinterpret_cast<float *>(smem + L.q);
        float *s_sc = reinterpret_cast<float *>(smem + L.sc);
        int *s_id = reinterpret_cast<int *>(smem + L.id);
        unsigned char *s_taken = smem + L.taken;
        const T *Qu = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
        for (int x = threadIdx.x; x < g * kHeadDim; x += kThreads) s_q[x] = Elem<T>::load(Qu + x);
        __syncthreads();
        const int m = chunk * kSelChunk + threadIdx.x;
        const bool valid = m < Np;
        s_id[threadIdx.x] = valid ? m : 0x7fffffff;
        const uint4 *row =
            reinterpret_cast<const uint4 *>(parent_keys + ((size_t)u * np_cap + (valid ? m : 0)) * kHeadDim);
        constexpr int RV = row_vecs<T>();
        constexpr int PV = Elem<T>::kPerVec;
        for (int h0 = 0; h0 < g; h0 += kHeadTile) {
            float acc[kHeadTile];
#pragma unroll
            for (int t = 0; t < kHeadTile; ++t) acc[t] = 0.f;
            if (valid) {
                for (int v = 0; v < RV; ++v) {
                    float f[PV];
                    Elem<T>::unpack(__ldg(row + v), f);
#pragma unroll
                    for (int t = 0; t < kHeadTile; ++t) {
                        if (h0 + t < g) {
                            const float *qq = s_q + (size_t)(h0 + t) * kHeadDim + v * PV;
#pragma unroll
                            for (int e = 0; e < PV; ++e) acc[t] = fmaf(qq[e], f[e], acc[t]);
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kHeadTile; ++t)
                if (h0 + t < g) s_sc[(size_t)(h0 + t) * kSelChunk + threadIdx.x] = valid ? acc[t] : -INFINITY;
        }
        __syncthreads();
        // ---- 2. this chunk's ordered top-kc parents per query head
        for (int hh = warp; hh < g; hh += kWarps) {
            const size_t base = (((size_t)u * n_chunks + chunk) * g + hh) * kc;
            warp_topk(s_sc + (size_t)hh * kSelChunk, s_id, s_taken + warp * kSelChunk, kSelChunk, kc,
                      cand_score + base, cand_id + base);
        }
    }

    // ---- 3. the unit's last CTA merges (no CTA waits for another)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(ticket + u, 1) == n_chunks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    unsigned *s_mask = reinterpret_cast<unsigned *>(smem + L.mask);
    const int P = min(n_pages[u], page_cap);
    const int words = (P + 31) / 32;
    for (int x = threadIdx.x; x < words; x += kThreads) s_mask[x] = 0u;
    __syncthreads();
    const size_t ug = (size_t)u * page_cap, up = (size_t)u * np_cap;
    if (k_pages >= P) {
        for (int x = threadIdx.x; x < words; x += kThreads) {
            const int rem = P - x * 32;
            s_mask[x] = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
        }
    } else {
        const int per_warp = n_chunks * kc;
        float *m_sc = reinterpret_cast<float *>(smem + L.msc) + (size_t)warp * per_warp;
        int *m_id = reinterpret_cast<int *>(smem + L.mid) + (size_t)warp * per_warp;
        int *m_ptr = reinterpret_cast<int *>(smem + L.mptr) + (size_t)warp * n_chunks;
        int *m_top = reinterpret_cast<int *>(smem + L.mtop) + (size_t)warp * kt;
        for (int hh = warp; hh < g; hh += kWarps) {
            for (int x = lane; x < per_warp; x += 32) {
                const int c = x / kc, t = x % kc;
                const size_t o = (((size_t)u * n_chunks + c) * g + hh) * kc + t;
                m_sc[x] = __ldcg(cand_score + o);  // written by other CTAs: read through L2
                m_id[x] = __ldcg(cand_id + o);
            }
            for (int c = lane; c < n_chunks; c += 32) m_ptr[c] = 0;
            __syncwarp();
            // k-way merge of the sorted chunk lists -> ordered top-kt parents
            for (int r = 0; r < kt; ++r) {
                float bs = -INFINITY;
                int bi = 0x7fffffff, bc = -1;
                for (int c = lane; c < n_chunks; c += 32) {
                    const int t = m_ptr[c];
                    if (t >= kc) continue;
                    const float s = m_sc[c * kc + t];
                    const int id = m_id[c * kc + t];
                    if (bc < 0 || better(s, id, bs, bi)) {
                        bs = s;
                        bi = id;
                        bc = c;
                    }
                }
                float ws = bs;
                int wi = bi;
                warp_best(ws, wi);
                if (bc >= 0 && bi == wi && bs == ws) m_ptr[bc] += 1;
                if (lane == 0) m_top[r] = (wi == 0x7fffffff) ? -1 : wi;
                __syncwarp();
            }
            // expand the ordered parents into pages until k pages are taken
            int taken_pages = 0;
            for (int r0 = 0; r0 < kt && taken_pages < k_pages; r0 += 32) {
                const int my_m = (r0 + lane < kt) ? m_top[r0 + lane] : -1;
                const int cnt = (my_m >= 0) ? parent_n_pages[up + my_m] : 0;
                int incl = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                const int before = taken_pages + incl - cnt;
                const int take = max(0, min(cnt, k_pages - before));
                if (take > 0) {
                    int pg = parent_first_page[up + my_m];
                    const bool contiguous = parent_last_page[up + my_m] - pg + 1 == cnt;
                    for (int i = 0; i < take; ++i) {
                        const int q = contiguous ? pg + i : pg;
                        if (q < 0 || q >= P) break;
                        atomicOr(&s_mask[q >> 5], 1u << (q & 31));
                        if (!contiguous) pg = page_next[ug + q];
                    }
                }
                taken_pages += __shfl_sync(0xffffffffu, incl, 31);
            }
            __syncwarp();
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
        ticket[u] = 0;
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                     int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    const int kc = ws.k_pages < kSelChunk ? ws.k_pages : kSelChunk;
    const int kt = ws.k_pages < ws.n_chunks * kc ? ws.k_pages : ws.n_chunks * kc;
    const size_t smem = select_smem(g, ws.n_chunks, kc, kt, p.page_cap).total;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_select<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaMemsetAsync(ws.sel_ticket, 0, sizeof(int32_t) * U, s);
    dim3 grid(ws.n_chunks, U);
    k_select<T><<<grid, kThreads, smem, s>>>(
        static_cast<const T *>(Q), g, p.n_q_heads, p.n_kv_heads, p.np_cap, p.page_cap, ws.k_pages, kc, kt,
        ws.n_chunks, idx.n_parents, idx.n_pages, static_cast<const T *>(idx.parent_keys), idx.parent_first_page,
        idx.parent_last_page, idx.parent_n_pages, idx.page_next, ws.cand_score, ws.cand_id, ws.sel_ticket,
        sel_pages, sel_count, max_sel, err);
    return cudaGetLastError();
}

}  // namespace

size_t select_smem_bytes(const ice_params &p, int k_pages, int n_chunks) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const int kc = k_pages < kSelChunk ? k_pages : kSelChunk;
    const int kt = k_pages < n_chunks * kc ? k_pages : n_chunks * kc;
    return select_smem(g, n_chunks, kc, kt, p.page_cap).total;
}

cudaError_t launch_select(const ice_params &p, const ice_index &idx, const void *Q, const DecodeWs &ws,
                          int32_t *sel_pages, int32_t *sel_count, int max_sel, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
    return launch_t<float>(p, idx, Q, ws, sel_pages, sel_count, max_sel, err, s);
}

}  // namespace ice
