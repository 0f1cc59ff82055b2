// Index build, steps a4 (pack tokens into semantic pages) and a5 (copy K/V
// rows into the page pool).
//
// IceCache popular-science article (aitangshan.cn/news/751385), section 三:
// the clusters formed by shared parents map directly onto physical memory
// pages, the tokens under one parent stored in the same page; section 二:
// a page holds 16 tokens.  papernotes.org "IceCache: Memory-Efficient
// KV-cache Management for Long-Sequence LLMs", 关键设计 2: a node larger
// than the page size splits off a new page.
//
// Layout rule: parents in ascending m; a parent's tokens in ascending token
// order; consecutive chunks of S tokens per page; pages numbered in that
// order.  This is a stable counting sort of the tokens by parent, done
// without library sorts in three kernels:
//   k_pack_count  grid (tiles, units): per 2048-token tile, tokens per parent
//                 (shared-memory histogram, or global atomics when the parent
//                 count is too large for shared memory).
//   k_pack_scan   grid (units): per parent, exclusive scan of its tile counts
//                 (column scan) -> tile offsets and total c_m; exclusive scan
//                 of ceil(c_m / S) over m -> first page; page tables.
//   k_pack_rank_scatter grid (tiles, units): the stable rank of every token
//                 inside its parent = tile offset + rank inside the tile.
//                 Inside a tile, warps take turns (in token order), each
//                 ranking its 32 tokens with __match_any_sync and bumping
//                 per-parent counters; then the CTA copies the K/V rows to
//                 (page, slot) with 16-byte vectors and zeroes pad slots.
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 256;
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kThreads) k_pack_count(const int32_t *__restrict__ token_parent, int N, int n_cap,
                                                         int np_cap, const int32_t *__restrict__ n_parents,
                                                         int32_t *__restrict__ pack_cnt, int n_tiles,
                                                         int smem_path) {
    extern __shared__ int s_hist[];
    const int u = blockIdx.y, tile = blockIdx.x;
    const int Np = min(n_parents[u], np_cap);
    int32_t *row = pack_cnt + ((size_t)u * n_tiles + tile) * np_cap;
    int *hist = smem_path ? s_hist : row;
    if (smem_path) {
        for (int m = threadIdx.x; m < Np; m += kThreads) s_hist[m] = 0;
        __syncthreads();
    }
    const long long t0 = (long long)tile * kPackTile;
    for (int i = threadIdx.x; i < kPackTile; i += kThreads) {
        const long long j = t0 + i;
        if (j >= N) break;
        const int m = token_parent[(size_t)u * n_cap + j];
        if (m >= 0 && m < Np) atomicAdd(&hist[m], 1);
    }
    if (smem_path) {
        __syncthreads();
        for (int m = threadIdx.x; m < Np; m += kThreads) row[m] = s_hist[m];
    }
}

__global__ void __launch_bounds__(kScanThreads) k_pack_scan(int np_cap, int page_cap, int n_tiles,
                                                            const int32_t *__restrict__ n_parents,
                                                            int32_t *__restrict__ pack_cnt,
                                                            int32_t *__restrict__ pack_total,
                                                            int32_t *__restrict__ n_pages,
                                                            int32_t *__restrict__ parent_first_page,
                                                            int32_t *__restrict__ parent_last_page,
                                                            int32_t *__restrict__ parent_n_pages,
                                                            int32_t *__restrict__ page_parent,
                                                            int32_t *__restrict__ page_len,
                                                            int32_t *__restrict__ page_next,
                                                            int32_t *__restrict__ page_tokens,
                                                            int32_t *__restrict__ err) {
    __shared__ int s_warp[kScanThreads / 32];
    __shared__ long long s_carry;
    const int u = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (int m0 = 0; m0 < Np; m0 += kScanThreads) {
        const int m = m0 + threadIdx.x;
        int c = 0;
        if (m < Np) {
            int32_t *col = pack_cnt + (size_t)u * n_tiles * np_cap + m;
            for (int t = 0; t < n_tiles; ++t) {
                const int v = col[(size_t)t * np_cap];
                col[(size_t)t * np_cap] = c;
                c += v;
            }
        }
        const int pages = (c + kPage - 1) / kPage;
        int incl = pages;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        long long woff = 0;
        for (int w = 0; w < warp; ++w) woff += s_warp[w];
        const long long first = s_carry + woff + incl - pages;
        if (m < Np) {
            pack_total[up + m] = c;
            parent_first_page[up + m] = (int32_t)first;
            parent_n_pages[up + m] = pages;
            parent_last_page[up + m] = (int32_t)(first + pages - 1);
            for (int i = 0; i < pages; ++i) {
                const long long pg = first + i;
                if (pg >= page_cap) break;
                page_parent[ug + pg] = m;
                const int len = min(kPage, c - i * kPage);
                page_len[ug + pg] = len;
                page_next[ug + pg] = (i + 1 < pages && pg + 1 < page_cap) ? (int32_t)(pg + 1) : -1;
                for (int sl = len; sl < kPage; ++sl) page_tokens[(ug + pg) * kPage + sl] = -1;
            }
        }
        __syncthreads();
        if (threadIdx.x == kScanThreads - 1) s_carry += woff + incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (s_carry > page_cap) set_err(err, ICE_ERR_CAPACITY);
        n_pages[u] = (int32_t)(s_carry < page_cap ? s_carry : page_cap);
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_pack_rank_scatter(
    const T *__restrict__ K, const T *__restrict__ V, int N, int n_cap, int np_cap, int page_cap, int n_tiles,
    int smem_path, const int32_t *__restrict__ n_parents, const int32_t *__restrict__ token_parent,
    int32_t *__restrict__ pack_cnt, const int32_t *__restrict__ pack_total,
    const int32_t *__restrict__ parent_first_page, int32_t *__restrict__ page_tokens,
    int32_t *__restrict__ token_page, int32_t *__restrict__ token_slot, T *__restrict__ pool_k,
    T *__restrict__ pool_v) {
    extern __shared__ int s_ctr_dyn[];
    __shared__ int s_dst[kThreads];   // page * S + slot, or -1
    __shared__ int s_pad[kThreads];   // first pad slot after this token, or S
    const int u = blockIdx.y, tile = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    int32_t *row = pack_cnt + ((size_t)u * n_tiles + tile) * np_cap;
    int *ctr = smem_path ? s_ctr_dyn : row;
    if (smem_path) {
        for (int m = threadIdx.x; m < Np; m += kThreads) s_ctr_dyn[m] = row[m];
    }
    __syncthreads();
    const size_t un = (size_t)u * n_cap, up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const T *Ku = K + (size_t)u * N * kHeadDim;
    const T *Vu = V + (size_t)u * N * kHeadDim;
    constexpr int RV = row_vecs<T>();
    const long long t0 = (long long)tile * kPackTile;
    for (int r0 = 0; r0 < kPackTile; r0 += kThreads) {
        if (t0 + r0 >= N) break;
        const long long j = t0 + r0 + threadIdx.x;
        const int m = (j < N) ? token_parent[un + j] : -1;
        const bool valid = (m >= 0 && m < Np);
        int rank = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            if (warp == w) {
                const int key = valid ? m : -1 - lane;  // invalid lanes stay alone
                const unsigned peers = __match_any_sync(0xffffffffu, key);
                const int leader = __ffs(peers) - 1;
                int base = 0;
                if (valid && lane == leader) {
                    base = ctr[m];
                    ctr[m] = base + __popc(peers);
                }
                base = __shfl_sync(0xffffffffu, base, leader);
                rank = base + __popc(peers & lanemask_lt());
            }
            __syncthreads();
        }
        int dst = -1, pad = kPage;
        if (valid) {
            const long long pg = (long long)parent_first_page[up + m] + rank / kPage;
            const int slot = rank % kPage;
            if (pg < page_cap) {
                dst = (int)(pg * kPage + slot);
                page_tokens[ug * kPage + dst] = (int32_t)j;
                token_page[un + j] = (int32_t)pg;
                token_slot[un + j] = slot;
                if (rank == pack_total[up + m] - 1) pad = slot + 1;
            }
        }
        s_dst[threadIdx.x] = dst;
        s_pad[threadIdx.x] = pad;
        __syncthreads();
        // K/V rows -> pool, 16-byte vectors
        const uint4 *k4 = reinterpret_cast<const uint4 *>(Ku);
        const uint4 *v4 = reinterpret_cast<const uint4 *>(Vu);
        uint4 *pk4 = reinterpret_cast<uint4 *>(pool_k + ug * kPage * kHeadDim);
        uint4 *pv4 = reinterpret_cast<uint4 *>(pool_v + ug * kPage * kHeadDim);
        for (int x = threadIdx.x; x < kThreads * RV; x += kThreads) {
            const int r = x / RV, v = x % RV;
            const int d = s_dst[r];
            if (d < 0) continue;
            const size_t src = (size_t)(t0 + r0 + r) * RV + v;
            pk4[(size_t)d * RV + v] = k4[src];
            pv4[(size_t)d * RV + v] = v4[src];
        }
        // zero the pad slots after each parent's last token
        for (int r = warp; r < kThreads; r += kThreads / 32) {
            const int pad0 = s_pad[r];
            if (pad0 >= kPage) continue;
            const int d0 = s_dst[r] - (s_dst[r] % kPage);
            for (int x = lane; x < (kPage - pad0) * RV; x += 32) {
                const size_t o = (size_t)(d0 + pad0 + x / RV) * RV + x % RV;
                pk4[o] = make_uint4(0, 0, 0, 0);
                pv4[o] = make_uint4(0, 0, 0, 0);
            }
        }
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const void *K, const void *V, const ice_index &idx, const BuildWs &ws,
                     int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int tiles = ceil_div(p.n_tokens, kPackTile);
    const int smem_path = p.np_cap <= kPackSmemBins;
    const size_t smem = smem_path ? sizeof(int) * (size_t)p.np_cap : 0;
    if (smem > 48 * 1024) {
        cudaFuncSetAttribute(k_pack_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(k_pack_rank_scatter<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    }
    if (!smem_path) cudaMemsetAsync(ws.pack_cnt, 0, sizeof(int32_t) * (size_t)U * tiles * p.np_cap, s);
    dim3 grid(tiles, U);
    k_pack_count<<<grid, kThreads, smem, s>>>(idx.token_parent, p.n_tokens, p.n_cap, p.np_cap, idx.n_parents,
                                              ws.pack_cnt, tiles, smem_path);
    k_pack_scan<<<U, kScanThreads, 0, s>>>(p.np_cap, p.page_cap, tiles, idx.n_parents, ws.pack_cnt, ws.pack_total,
                                           idx.n_pages, idx.parent_first_page, idx.parent_last_page,
                                           idx.parent_n_pages, idx.page_parent, idx.page_len, idx.page_next,
                                           idx.page_tokens, err);
    k_pack_rank_scatter<T><<<grid, kThreads, smem, s>>>(
        static_cast<const T *>(K), static_cast<const T *>(V), p.n_tokens, p.n_cap, p.np_cap, p.page_cap, tiles,
        smem_path, idx.n_parents, idx.token_parent, ws.pack_cnt, ws.pack_total, idx.parent_first_page,
        idx.page_tokens, idx.token_page, idx.token_slot, static_cast<T *>(idx.pool_k),
        static_cast<T *>(idx.pool_v));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(const ice_params &p, const void *K, const void *V, const ice_index &idx,
                        const BuildWs &ws, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, K, V, idx, ws, err, s);
    return launch_t<float>(p, K, V, idx, ws, err, s);
}

}  // namespace ice
