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
// order.  This is a stable counting sort of the tokens by parent, written
// without library sorts, in four kernels:
//   k_pack_count  grid (2048-token tiles, units): tokens per parent in the
//                 tile (shared-memory histogram, or global atomics when the
//                 parent count is too large for shared memory).
//   k_pack_scan   grid (units): per parent, exclusive scan of its tile counts
//                 (column scan, loads batched) -> tile offsets and total c_m;
//                 exclusive scan of ceil(c_m / S) over m -> first page; page
//                 tables.
//   k_pack_rank   grid (tiles, units): stable rank of every token inside its
//                 parent = tile offset + rank inside the tile.  Inside a tile,
//                 warps take turns in token order, each ranking its 32 tokens
//                 with __match_any_sync and bumping per-parent counters; the
//                 token tables and page_tokens get (page, slot).
//   k_pack_copy   grid (pages / 8, units): one warp per page gathers the K
//                 and V rows of the page's tokens (all 16-byte loads issued
//                 before the stores) into the pool and zeroes pad slots.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kTokPerThread = kPackTile / kThreads;  // 8

__global__ void __launch_bounds__(kThreads) k_pack_count(const int32_t *__restrict__ token_parent, int N, int n_cap,
                                                         int np_cap, const int32_t *__restrict__ n_parents,
                                                         int32_t *__restrict__ pack_cnt, int n_tiles,
                                                         int smem_path) {
    extern __shared__ int s_hist[];
    const int u = blockIdx.y, tile = blockIdx.x;
    const int Np = min(n_parents[u], np_cap);
    int32_t *row = pack_cnt + ((size_t)u * n_tiles + tile) * np_cap;
    int *hist = smem_path ? s_hist : row;
    const long long t0 = (long long)tile * kPackTile;
    int m[kTokPerThread];
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {
        const long long j = t0 + i * kThreads + threadIdx.x;
        m[i] = j < N ? token_parent[(size_t)u * n_cap + j] : -1;
    }
    if (smem_path) {
        for (int x = threadIdx.x; x < Np; x += kThreads) s_hist[x] = 0;
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i)
        if (m[i] >= 0 && m[i] < Np) atomicAdd(&hist[m[i]], 1);
    if (smem_path) {
        __syncthreads();
        for (int x = threadIdx.x; x < Np; x += kThreads) row[x] = s_hist[x];
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
    constexpr int kBatch = 16;  // column entries loaded before they are scanned
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
            for (int t0 = 0; t0 < n_tiles; t0 += kBatch) {
                int v[kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; ++i) v[i] = (t0 + i < n_tiles) ? col[(size_t)(t0 + i) * np_cap] : 0;
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    if (t0 + i < n_tiles) col[(size_t)(t0 + i) * np_cap] = c;
                    c += v[i];
                }
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

__global__ void __launch_bounds__(kThreads) k_pack_rank(int N, int n_cap, int np_cap, int page_cap, int n_tiles,
                                                        int smem_path, const int32_t *__restrict__ n_parents,
                                                        const int32_t *__restrict__ token_parent,
                                                        int32_t *__restrict__ pack_cnt,
                                                        const int32_t *__restrict__ parent_first_page,
                                                        int32_t *__restrict__ page_tokens,
                                                        int32_t *__restrict__ token_page,
                                                        int32_t *__restrict__ token_slot) {
    extern __shared__ int s_ctr_dyn[];
    const int u = blockIdx.y, tile = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    int32_t *row = pack_cnt + ((size_t)u * n_tiles + tile) * np_cap;
    int *ctr = smem_path ? s_ctr_dyn : row;
    const size_t un = (size_t)u * n_cap, up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const long long t0 = (long long)tile * kPackTile;
    int m[kTokPerThread], first[kTokPerThread];
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {
        const long long j = t0 + i * kThreads + threadIdx.x;
        m[i] = j < N ? token_parent[un + j] : -1;
    }
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) first[i] = (m[i] >= 0 && m[i] < Np) ? parent_first_page[up + m[i]] : 0;
    if (smem_path) {
        for (int x = threadIdx.x; x < Np; x += kThreads) s_ctr_dyn[x] = row[x];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {
        const long long j = t0 + i * kThreads + threadIdx.x;
        const bool valid = m[i] >= 0 && m[i] < Np;
        int rank = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            if (warp == w) {
                const int key = valid ? m[i] : -1 - lane;  // invalid lanes stay alone
                const unsigned peers = __match_any_sync(0xffffffffu, key);
                const int leader = __ffs(peers) - 1;
                int base = 0;
                if (valid && lane == leader) {
                    base = ctr[m[i]];
                    ctr[m[i]] = base + __popc(peers);
                }
                base = __shfl_sync(0xffffffffu, base, leader);
                rank = base + __popc(peers & lanemask_lt());
            }
            __syncthreads();
        }
        if (valid) {
            const long long pg = (long long)first[i] + rank / kPage;
            const int slot = rank % kPage;
            if (pg < page_cap) {
                page_tokens[(ug + pg) * kPage + slot] = (int32_t)j;
                token_page[un + j] = (int32_t)pg;
                token_slot[un + j] = slot;
            }
        }
    }
}

// k_pack_rank when a warp-private counter per parent fits in shared memory:
// warp w owns tokens [w*256, w*256 + 256) of the tile.  (1) each warp counts
// its segment per parent (match_any groups, the group leader adds; the
// counters are the warp's own, so no atomics); (2) per parent, an exclusive
// scan over the 8 warps turns the counts into warp bases; (3) each warp ranks
// its segment in token order from its bases.  Three block barriers per tile
// instead of one per warp turn.
constexpr int kSegWarps = kThreads / 32;
constexpr int kSeg = kPackTile / kSegWarps;  // 256 tokens per warp

__global__ void __launch_bounds__(kThreads) k_pack_rank_seg(int N, int n_cap, int np_cap, int page_cap, int n_tiles,
                                                            const int32_t *__restrict__ n_parents,
                                                            const int32_t *__restrict__ token_parent,
                                                            const int32_t *__restrict__ pack_cnt,
                                                            const int32_t *__restrict__ parent_first_page,
                                                            int32_t *__restrict__ page_tokens,
                                                            int32_t *__restrict__ token_page,
                                                            int32_t *__restrict__ token_slot) {
    extern __shared__ __align__(16) unsigned char s_raw[];
    const int u = blockIdx.y, tile = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    int32_t *s_off = reinterpret_cast<int32_t *>(s_raw);                       // [Np] tile offsets
    unsigned short *s_ctr = reinterpret_cast<unsigned short *>(s_off + np_cap);  // [8][Np]
    const size_t un = (size_t)u * n_cap, up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int32_t *row = pack_cnt + ((size_t)u * n_tiles + tile) * np_cap;
    const long long j0 = (long long)tile * kPackTile + (long long)warp * kSeg;
    int m[kSeg / 32];
#pragma unroll
    for (int i = 0; i < kSeg / 32; ++i) {
        const long long j = j0 + i * 32 + lane;
        const int v = j < N ? token_parent[un + j] : -1;
        m[i] = (v >= 0 && v < Np) ? v : -1;
    }
    for (int x = threadIdx.x; x < Np; x += kThreads) s_off[x] = row[x];
    for (int x = threadIdx.x; x < kSegWarps * Np; x += kThreads) s_ctr[x] = 0;
    __syncthreads();
    unsigned short *mine = s_ctr + (size_t)warp * Np;
    // (1) counts of this warp's segment
#pragma unroll
    for (int i = 0; i < kSeg / 32; ++i) {
        const int key = m[i] >= 0 ? m[i] : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (m[i] >= 0 && lane == __ffs(peers) - 1) mine[m[i]] += (unsigned short)__popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // (2) per parent: exclusive scan of the warp counts (within-tile bases)
    for (int x = threadIdx.x; x < Np; x += kThreads) {
        unsigned short run = 0;
#pragma unroll
        for (int w = 0; w < kSegWarps; ++w) {
            const unsigned short c = s_ctr[(size_t)w * Np + x];
            s_ctr[(size_t)w * Np + x] = run;
            run = (unsigned short)(run + c);
        }
    }
    __syncthreads();
    // (3) ranks of this warp's segment, in token order
#pragma unroll
    for (int i = 0; i < kSeg / 32; ++i) {
        const int mm = m[i];
        const int key = mm >= 0 ? mm : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int leader = __ffs(peers) - 1;
        int base = 0;
        if (mm >= 0 && lane == leader) {
            base = mine[mm];
            mine[mm] = (unsigned short)(base + __popc(peers));
        }
        base = __shfl_sync(0xffffffffu, base, leader);
        __syncwarp();
        if (mm >= 0) {
            const long long j = j0 + i * 32 + lane;
            const int rank = s_off[mm] + base + __popc(peers & lanemask_lt());
            const long long pg = (long long)parent_first_page[up + mm] + rank / kPage;
            const int slot = rank % kPage;
            if (pg < page_cap) {
                page_tokens[(ug + pg) * kPage + slot] = (int32_t)j;
                token_page[un + j] = (int32_t)pg;
                token_slot[un + j] = slot;
            }
        }
    }
}

// Steps a4 for one unit in one thread-block cluster of kPackCluster CTAs
// (replaces count, scan and rank when the per-warp counters fit in shared
// memory).  CTA r owns tokens [r*Tc, (r+1)*Tc) and parents
// [r*Sc, (r+1)*Sc); warp w of a CTA owns a contiguous run of Tw tokens.
//   A  each warp counts its run per parent (warp-private u16 counters, no
//      atomics); per parent, an exclusive scan over the warps gives warp
//      bases and the CTA's count;                          -- cluster barrier
//   B  per owned parent: c_m = sum of the CTAs' counts (distributed shared
//      memory reads), pages ceil(c_m / S), exclusive scan of pages over the
//      slice; the slice's page total goes to every CTA;     -- cluster barrier
//   C  per owned parent: first page, parent tables, and into every CTA the
//      position base S * first + (tokens of m in the CTAs before it) and the
//      end position S * first + c_m;                        -- cluster barrier
//   D  each warp ranks its run in token order from its bases: position
//      pos -> page pos / S, slot pos % S; the token at a page's slot 0
//      writes the page's parent, length and successor, the parent's last
//      token marks the page's empty slots.
// Positions are global slot indices, so a parent's rank order is token order
// (stable counting sort).
constexpr int kPackCluster = 8;
constexpr int kPCThreads = 256;
constexpr int kPCWarps = kPCThreads / 32;
constexpr size_t kPackClusterSmem = 225 * 1024;  // dynamic shared memory of one cluster CTA, at most

struct PackClusterShape {
    int tc, tw, sc;  // tokens per CTA, tokens per warp, parents per CTA slice
    size_t smem;
};
PackClusterShape pack_cluster_shape(int N, int np_cap) {
    PackClusterShape sh;
    sh.tc = ceil_div(N, kPackCluster);
    sh.tw = ceil_div(sh.tc, kPCWarps);
    sh.sc = ceil_div(np_cap, kPackCluster);
    // s_tok[tc] int32, s_ctr[W][np_cap] u16 (rounded to 4 bytes), s_B, s_E [np_cap], s_F [sc]
    const size_t ctr = ((size_t)kPCWarps * np_cap * 2 + 3) & ~(size_t)3;
    sh.smem = 4 * (size_t)sh.tc + ctr + 8 * (size_t)np_cap + 4 * (size_t)sh.sc;
    return sh;
}

__global__ void __cluster_dims__(kPackCluster, 1, 1) __launch_bounds__(kPCThreads)
    k_pack_cluster(int N, int n_cap, int np_cap, int page_cap, int tc, int tw, int sc,
                   const int32_t *__restrict__ n_parents, const int32_t *__restrict__ token_parent,
                   int32_t *__restrict__ pack_total, int32_t *__restrict__ n_pages,
                   int32_t *__restrict__ parent_first_page, int32_t *__restrict__ parent_last_page,
                   int32_t *__restrict__ parent_n_pages, int32_t *__restrict__ page_parent,
                   int32_t *__restrict__ page_len, int32_t *__restrict__ page_next,
                   int32_t *__restrict__ page_tokens, int32_t *__restrict__ token_page,
                   int32_t *__restrict__ token_slot, int32_t *__restrict__ err) {
    dep_wait();  // the previous kernel of the stream is complete (launched as its dependent)
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char s_raw[];
    __shared__ int s_slice[kPackCluster];
    __shared__ int s_wsum[kPCWarps];
    __shared__ int s_carry;
    const int r = (int)cluster.block_rank();
    const int u = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    int32_t *s_tok = reinterpret_cast<int32_t *>(s_raw);
    unsigned short *s_ctr = reinterpret_cast<unsigned short *>(s_tok + tc);
    int32_t *s_B = reinterpret_cast<int32_t *>(s_raw + 4 * (size_t)tc +
                                               (((size_t)kPCWarps * np_cap * 2 + 3) & ~(size_t)3));
    int32_t *s_E = s_B + np_cap;
    int32_t *s_F = s_E + np_cap;
    const size_t un = (size_t)u * n_cap, up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const long long tok0 = (long long)r * tc;

    // ---- A: load the CTA's token parents, clear the counters, count
    for (int i = threadIdx.x; i < tc; i += kPCThreads) {
        const long long j = tok0 + i;
        const int v = j < N ? token_parent[un + j] : -1;
        s_tok[i] = (v >= 0 && v < Np) ? v : -1;
    }
    for (int x = threadIdx.x; x < kPCWarps * Np; x += kPCThreads) s_ctr[x] = 0;
    __syncthreads();
    unsigned short *mine = s_ctr + (size_t)warp * Np;
    const int w0 = warp * tw;
    for (int i0 = 0; i0 < tw; i0 += 32) {
        const int i = w0 + i0 + lane;
        const int m = (i0 + lane < tw && i < tc) ? s_tok[i] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, m >= 0 ? m : -1 - lane);
        if (m >= 0 && lane == __ffs(peers) - 1) mine[m] += (unsigned short)__popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int x = threadIdx.x; x < Np; x += kPCThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kPCWarps; ++w) {
            const int c = s_ctr[(size_t)w * Np + x];
            s_ctr[(size_t)w * Np + x] = (unsigned short)run;
            run += c;
        }
        s_B[x] = run;  // this CTA's tokens of parent x
    }
    cluster.sync();

    // ---- B: totals and page scan over this CTA's parent slice
    const int lo = min(r * sc, Np), hi = min(lo + sc, Np);
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (int x0 = lo; x0 < hi; x0 += kPCThreads) {
        const int x = x0 + threadIdx.x;
        int c = 0;
        if (x < hi) {
            int v[kPackCluster];
#pragma unroll
            for (int q = 0; q < kPackCluster; ++q) v[q] = cluster.map_shared_rank(s_B, q)[x];
#pragma unroll
            for (int q = 0; q < kPackCluster; ++q) c += v[q];
            s_E[x] = c;  // c_m, kept here until C
        }
        const int pages = (c + kPage - 1) / kPage;
        int incl = pages;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int woff = 0;
        for (int w = 0; w < warp; ++w) woff += s_wsum[w];
        if (x < hi) s_F[x - lo] = s_carry + woff + incl - pages;
        __syncthreads();
        if (threadIdx.x == kPCThreads - 1) s_carry += woff + incl;
        __syncthreads();
    }
    if (threadIdx.x < kPackCluster) cluster.map_shared_rank(s_slice, threadIdx.x)[r] = s_carry;
    cluster.sync();

    // ---- C: first pages, parent tables, position bases in every CTA
    int base = 0, total = 0;
#pragma unroll
    for (int q = 0; q < kPackCluster; ++q) {
        base += q < r ? s_slice[q] : 0;
        total += s_slice[q];
    }
    for (int x = lo + threadIdx.x; x < hi; x += kPCThreads) {
        const int c = s_E[x];
        const int pages = (c + kPage - 1) / kPage;
        const int first = base + s_F[x - lo];
        pack_total[up + x] = c;
        parent_first_page[up + x] = first;
        parent_n_pages[up + x] = pages;
        parent_last_page[up + x] = first + pages - 1;
        int v[kPackCluster];
#pragma unroll
        for (int q = 0; q < kPackCluster; ++q) v[q] = cluster.map_shared_rank(s_B, q)[x];
        int run = first * kPage;
#pragma unroll
        for (int q = 0; q < kPackCluster; ++q) {
            cluster.map_shared_rank(s_B, q)[x] = run;
            cluster.map_shared_rank(s_E, q)[x] = first * kPage + c;
            run += v[q];
        }
    }
    if (r == 0 && threadIdx.x == 0) {
        if (total > page_cap) set_err(err, ICE_ERR_CAPACITY);
        n_pages[u] = total < page_cap ? total : page_cap;
    }
    cluster.sync();  // no distributed shared memory access after this point

    // ---- D: stable ranks of this warp's run
    for (int i0 = 0; i0 < tw; i0 += 32) {
        const int i = w0 + i0 + lane;
        const int m = (i0 + lane < tw && i < tc) ? s_tok[i] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, m >= 0 ? m : -1 - lane);
        const int leader = __ffs(peers) - 1;
        int b = 0;
        if (m >= 0 && lane == leader) {
            b = mine[m];
            mine[m] = (unsigned short)(b + __popc(peers));
        }
        b = __shfl_sync(0xffffffffu, b, leader);
        __syncwarp();
        if (m >= 0) {
            const long long j = tok0 + i;
            const int pos = s_B[m] + b + __popc(peers & lanemask_lt());
            const int end = s_E[m];
            const int pg = pos / kPage, slot = pos % kPage;
            if (pg < page_cap) {
                page_tokens[(ug + pg) * kPage + slot] = (int32_t)j;
                token_page[un + j] = pg;
                token_slot[un + j] = slot;
                if (slot == 0) {
                    page_parent[ug + pg] = m;
                    page_len[ug + pg] = min(kPage, end - pos);
                    page_next[ug + pg] = (pos + kPage < end && pg + 1 < page_cap) ? pg + 1 : -1;
                }
                if (pos == end - 1)
                    for (int sl = slot + 1; sl < kPage; ++sl) page_tokens[(ug + pg) * kPage + sl] = -1;
            }
        }
    }
}

size_t rank_seg_smem(int np_cap) { return (size_t)np_cap * (sizeof(int32_t) + kSegWarps * sizeof(unsigned short)); }

template <typename T>
__global__ void __launch_bounds__(kThreads) k_pack_copy(const T *__restrict__ K, const T *__restrict__ V, int N,
                                                        int page_cap, const int32_t *__restrict__ n_pages,
                                                        const int32_t *__restrict__ page_len,
                                                        const int32_t *__restrict__ page_tokens,
                                                        T *__restrict__ pool_k, T *__restrict__ pool_v) {
    dep_wait();  // the previous kernel of the stream is complete (launched as its dependent)
    constexpr int RV = row_vecs<T>();         // 16-byte vectors per row
    constexpr int PER_LANE = kPage * RV / 32;  // vectors per lane per page (8 bf16, 16 fp32)
    const int u = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pg = blockIdx.x * (kThreads / 32) + warp;
    if (pg >= min(n_pages[u], page_cap)) return;
    const size_t gp = (size_t)u * page_cap + pg;
    const int len = page_len[gp];
    const int tok = lane < kPage ? page_tokens[gp * kPage + lane] : -1;
    const uint4 *k4 = reinterpret_cast<const uint4 *>(K + (size_t)u * N * kHeadDim);
    const uint4 *v4 = reinterpret_cast<const uint4 *>(V + (size_t)u * N * kHeadDim);
    uint4 kv[PER_LANE], vv[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int x = lane + 32 * i, slot = x / RV, vec = x % RV;
        const int j = __shfl_sync(0xffffffffu, tok, slot);
        const bool ok = slot < len && j >= 0 && j < N;
        kv[i] = ok ? __ldg(k4 + (size_t)j * RV + vec) : make_uint4(0, 0, 0, 0);
        vv[i] = ok ? __ldg(v4 + (size_t)j * RV + vec) : make_uint4(0, 0, 0, 0);
    }
    uint4 *pk = reinterpret_cast<uint4 *>(pool_k) + gp * kPage * RV;
    uint4 *pv = reinterpret_cast<uint4 *>(pool_v) + gp * kPage * RV;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        pk[lane + 32 * i] = kv[i];
        pv[lane + 32 * i] = vv[i];
    }
}

// Positional pages after the unit's semantic pages: the sink tokens [0, lo)
// in order, S per page, then the window tokens [hi, N) (IceCache popular-
// science article, section 六: anchor and window tokens stay resident, only
// the middle is indexed).  Page parent -1, page_next -1.
__global__ void __launch_bounds__(kThreads) k_pack_positional(int N, int lo, int hi, int page_cap, int n_cap,
                                                              int32_t *__restrict__ n_pages,
                                                              int32_t *__restrict__ page_parent,
                                                              int32_t *__restrict__ page_len,
                                                              int32_t *__restrict__ page_next,
                                                              int32_t *__restrict__ page_tokens,
                                                              int32_t *__restrict__ token_page,
                                                              int32_t *__restrict__ token_slot,
                                                              int32_t *__restrict__ err) {
    dep_wait();  // the semantic pages are complete
    const int u = blockIdx.x;
    const int ns = (lo + kPage - 1) / kPage, npos = ns + (N - hi + kPage - 1) / kPage;
    const int P_sem = min(n_pages[u], page_cap);
    __syncthreads();  // every thread has the semantic count before it grows
    if (threadIdx.x == 0) {
        if (P_sem + npos > page_cap) set_err(err, ICE_ERR_CAPACITY);
        n_pages[u] = min(P_sem + npos, page_cap);
    }
    for (int x = threadIdx.x; x < npos * kPage; x += kThreads) {
        const int i = x / kPage, sl = x % kPage;
        const int pg = P_sem + i;
        if (pg >= page_cap) break;
        const int a = i < ns ? i * kPage : hi + (i - ns) * kPage;  // first token of the page
        const int e = i < ns ? lo : N;                            // end of its range
        const int tok = a + sl < e ? a + sl : -1;
        const size_t gp = (size_t)u * page_cap + pg;
        page_tokens[gp * kPage + sl] = tok;
        if (sl == 0) {
            page_parent[gp] = -1;
            page_len[gp] = min(kPage, e - a);
            page_next[gp] = -1;
        }
        if (tok >= 0) {
            token_page[(size_t)u * n_cap + tok] = pg;
            token_slot[(size_t)u * n_cap + tok] = sl;
        }
    }
}

void launch_rank_tiles(const ice_params &p, const ice_index &idx, const BuildWs &ws, int32_t *err, cudaStream_t s);

template <typename T>
cudaError_t launch_t(const ice_params &p, const void *K, const void *V, const ice_index &idx, const BuildWs &ws,
                     int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const PackClusterShape pcs = pack_cluster_shape(p.n_tokens, p.np_cap);
    if (pcs.smem <= kPackClusterSmem && pcs.tw <= 65535) {
        if (pcs.smem > 48 * 1024) {
            cudaError_t e =
                cudaFuncSetAttribute(k_pack_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pcs.smem);
            if (e != cudaSuccess) return e;
        }
        {
            const cudaError_t e_ = launch_dependent(k_pack_cluster, dim3(kPackCluster, U), dim3(kPCThreads), pcs.smem,
                                                    s, p.n_tokens, p.n_cap, p.np_cap, p.page_cap, pcs.tc, pcs.tw,
                                                    pcs.sc, idx.n_parents, idx.token_parent, ws.pack_total,
                                                    idx.n_pages, idx.parent_first_page, idx.parent_last_page,
                                                    idx.parent_n_pages, idx.page_parent, idx.page_len, idx.page_next,
                                                    idx.page_tokens, idx.token_page, idx.token_slot, err);
            if (e_ != cudaSuccess) return e_;
        }
    } else {
        launch_rank_tiles(p, idx, ws, err, s);
    }
    const PosSplit ps = pos_split(p);
    if (ps.n_pos > 0) {
        const cudaError_t e_ = launch_dependent(k_pack_positional, dim3(U), dim3(kThreads), 0, s, p.n_tokens, ps.lo,
                                                ps.hi, p.page_cap, p.n_cap, idx.n_pages, idx.page_parent,
                                                idx.page_len, idx.page_next, idx.page_tokens, idx.token_page,
                                                idx.token_slot, err);
        if (e_ != cudaSuccess) return e_;
    }
    dim3 cgrid(ceil_div(p.page_cap, kThreads / 32), U);
    {
        const cudaError_t e_ = launch_dependent(k_pack_copy<T>, dim3(cgrid), dim3(kThreads), 0, s,
                                                static_cast<const T *>(K), static_cast<const T *>(V), p.n_tokens,
                                                p.page_cap, idx.n_pages, idx.page_len, idx.page_tokens,
                                                static_cast<T *>(idx.pool_k), static_cast<T *>(idx.pool_v));
        if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
}

// count, scan and rank as separate kernels over 2048-token tiles
void launch_rank_tiles(const ice_params &p, const ice_index &idx, const BuildWs &ws, int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int tiles = ceil_div(p.n_tokens, kPackTile);
    const int smem_path = p.np_cap <= kPackSmemBins;
    const size_t smem = smem_path ? sizeof(int) * (size_t)p.np_cap : 0;
    if (smem > 48 * 1024) {
        cudaFuncSetAttribute(k_pack_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(k_pack_rank, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    }
    if (!smem_path) cudaMemsetAsync(ws.pack_cnt, 0, sizeof(int32_t) * (size_t)U * tiles * p.np_cap, s);
    dim3 grid(tiles, U);
    k_pack_count<<<grid, kThreads, smem, s>>>(idx.token_parent, p.n_tokens, p.n_cap, p.np_cap, idx.n_parents,
                                              ws.pack_cnt, tiles, smem_path);
    k_pack_scan<<<U, kScanThreads, 0, s>>>(p.np_cap, p.page_cap, tiles, idx.n_parents, ws.pack_cnt, ws.pack_total,
                                           idx.n_pages, idx.parent_first_page, idx.parent_last_page,
                                           idx.parent_n_pages, idx.page_parent, idx.page_len, idx.page_next,
                                           idx.page_tokens, err);
    const size_t seg_smem = rank_seg_smem(p.np_cap);
    if (smem_path && seg_smem <= 200 * 1024) {
        if (seg_smem > 48 * 1024)
            cudaFuncSetAttribute(k_pack_rank_seg, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)seg_smem);
        k_pack_rank_seg<<<grid, kThreads, seg_smem, s>>>(p.n_tokens, p.n_cap, p.np_cap, p.page_cap, tiles,
                                                         idx.n_parents, idx.token_parent, ws.pack_cnt,
                                                         idx.parent_first_page, idx.page_tokens, idx.token_page,
                                                         idx.token_slot);
    } else {
        k_pack_rank<<<grid, kThreads, smem, s>>>(p.n_tokens, p.n_cap, p.np_cap, p.page_cap, tiles, smem_path,
                                                 idx.n_parents, idx.token_parent, ws.pack_cnt,
                                                 idx.parent_first_page, idx.page_tokens, idx.token_page,
                                                 idx.token_slot);
    }
}

template <typename T>
cudaError_t launch_copy_t(const ice_params &p, const void *K, const void *V, const ice_index &idx, cudaStream_t s) {
    const cudaError_t e = launch_dependent(k_pack_copy<T>, dim3(ceil_div(p.page_cap, kThreads / 32), units_of(p)),
                                           dim3(kThreads), 0, s, static_cast<const T *>(K),
                                           static_cast<const T *>(V), p.n_tokens, p.page_cap, idx.n_pages,
                                           idx.page_len, idx.page_tokens, static_cast<T *>(idx.pool_k),
                                           static_cast<T *>(idx.pool_v));
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_copy(const ice_params &p, const void *K, const void *V, const ice_index &idx,
                             cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_copy_t<__nv_bfloat16>(p, K, V, idx, s);
    return launch_copy_t<float>(p, K, V, idx, s);
}

cudaError_t launch_pack(const ice_params &p, const void *K, const void *V, const ice_index &idx,
                        const BuildWs &ws, int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, K, V, idx, ws, err, s);
    return launch_t<float>(p, K, V, idx, ws, err, s);
}

}  // namespace ice
