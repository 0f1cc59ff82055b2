// The whole decode step (a6-a10) of every unit in one kernel, for bf16 tables
// with at most 8 query heads per KV head and k <= 32 pages per head.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 3: every query head scores the parent nodes
// (q' = [q, 0] against the lifted parents, so the score is q.p), picks its
// top-k pages, and the heads of a GQA group share the union of their picks;
// 关键设计 4: the selected pages are gathered; 关键设计 1: masked sparse
// attention over them.  IceCache popular-science article
// (aitangshan.cn/news/751385), section 六: TQ lift and the GQA union.
//
// Grid (C, U): the C CTAs of a thread-block cluster take one unit; C is the
// largest power of two up to 8 with U * C * 2 <= SMs (1 for 128 units, 4 for
// 32, 8 for 8), so that one wave holds every unit.  8 warps per CTA.
//
//   scan    CTA r streams its share of the unit's parent table (32-row tiles,
//           2-D TMA with a 128-byte swizzle, three tiles in flight per warp;
//           warp w takes the CTA's tiles w, w + 8, ...) and scores each tile
//           against the group's queries on mma.sync m16n8k16 (parents as the
//           16 rows, the g <= 8 query heads as the 8 columns, bf16 in, fp32
//           accumulate).  Each warp keeps, per head, its best k keys
//           (score, -m) sorted across lanes (lane i holds the i-th); a score
//           enters only above the head's current k-th score (after the first
//           tiles, rarely), by a ballot-ranked shift.  No score is written to
//           memory.
//   select  the warps' lists are merged per head (bitonic merges of sorted
//           32-lists), then rank 0 merges the CTAs' lists over distributed
//           shared memory; the best k parents of each head give their pages
//           (parent spans, page-id order inside a parent, until k pages),
//           ORed into the union bitmask with the positional pages, and the
//           ascending union list is written (sel_pages / sel_count).
//                                                            -- cluster barrier
//   attend  CTA r takes its share of the union, each warp its pages through
//           three TMA page slots, and runs the MMA attention of every page
//           (attn_page.cuh); with kbuf / vbuf / buf_len the slots also go back
//           out to the contiguous buffer by TMA stores.  Warps merge in
//           shared memory.                                   -- cluster barrier
//   merge   CTA r merges heads r, r + C, ... of all CTAs (log-sum-exp over
//           DSMEM) and writes O.                              -- cluster barrier
// Every mbarrier wait is bounded (ICE_ERR_TIMEOUT, NaN in O); no CTA waits on
// a flag.
#include <cooperative_groups.h>
#include <cuda.h>

#include "attn_page.cuh"
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "topk_common.cuh"

namespace ice {
namespace {

namespace cg = cooperative_groups;
using namespace tc;
using namespace topk;
using namespace mma;

constexpr int kW = 8;                  // warps per CTA
constexpr int kT = kW * 32;
constexpr int kR = 3;                  // slots per warp: tiles or pages in flight
constexpr int kRows = 32;              // parent rows per scan tile
constexpr uint32_t kScanHalf = kRows * 128;  // one 64-column box of a scan tile
constexpr uint32_t kSlot = 8192;       // a scan tile (32 rows x 256 B) or a page (K 4 KB + V 4 KB)
constexpr int kGT = 8;                 // query heads per group
constexpr int kMaxC = 8;  // 16-CTA clusters measured slower (scheduling)
constexpr int kStageRow = 36;          // padded row of 32 scores: the fragment stores hit 32 distinct banks

struct Smem {
    unsigned char slots[kW][kR][kSlot];  // 192 KB: scan tiles; then the warps' lists; pages; the warp merge
    unsigned long long scan_bar[kW][kR];
    unsigned long long page_bar[kW][kR];
    unsigned long long st_full[2];   // a stage buffer holds all warps' scores of its round (8 arrivals)
    unsigned long long st_empty[2];  // the head workers are done with it (g arrivals)
    unsigned long long top[kGT][32];  // this CTA's best keys per head (rank 0 reads them over DSMEM)
    float ml[kW][16][2];
    float wgt[kW][16];
    float cm[kGT], cl[kGT];           // this CTA's (max, sum) per head (read over DSMEM)
    float stage[2][kW][kGT][kStageRow];  // a round's scores (two rounds alternate): warp, head, parent of the tile
    int wsum[kW];
    int n_sel;                        // rank 0: length of the union list
    int bad;                          // a bounded wait gave up
};
// dynamic tail: mask words [ceil(page_cap / 32)], then the union list [max_sel]
inline size_t smem_bytes(int page_cap, int max_sel) {
    return 1024 + sizeof(Smem) + 4 * (size_t)((page_cap + 31) / 32) + 4 * (size_t)max_sel;
}

// Descending bitonic sort of one key per lane.
__device__ __forceinline__ unsigned long long sort32_desc(unsigned long long v, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool desc = (lane & size) == 0, lower = (lane & stride) == 0;
            v = (lower == desc) ? umax64(v, o) : umin64(v, o);
        }
    return v;
}

// Inserts key into the warp's sorted list (lane i holds entry i, i < k,
// descending; lanes >= k hold 0) if it beats the k-th entry.
__device__ __forceinline__ void list_insert(unsigned long long &lst, unsigned long long key, int k, int lane) {
    const unsigned long long kth = __shfl_sync(0xffffffffu, lst, k - 1);
    if (key <= kth) return;  // warp-uniform
    const int pos = __popc(__ballot_sync(0xffffffffu, lane < k && lst > key));
    const unsigned long long up = __shfl_up_sync(0xffffffffu, lst, 1);
    if (lane > pos && lane < k) lst = up;
    if (lane == pos) lst = key;
}

__global__ void __launch_bounds__(kT, 1) k_decode_fused(
    const __grid_constant__ CUtensorMap tm_par, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kb,
    const __grid_constant__ CUtensorMap tm_vb, const __nv_bfloat16 *__restrict__ Q, int g, int n_q_heads,
    int n_kv_heads, int np_cap, int page_cap, int k_pages, int n_pos, const int32_t *__restrict__ n_parents,
    const int32_t *__restrict__ n_pages, const int32_t *__restrict__ parent_first_page,
    const int32_t *__restrict__ parent_last_page, const int32_t *__restrict__ parent_n_pages,
    const int32_t *__restrict__ page_next, const int32_t *__restrict__ page_len, int32_t *__restrict__ sel_pages,
    int32_t *__restrict__ sel_count, int max_sel, int32_t *__restrict__ buf_len, float scale, float *__restrict__ O,
    int32_t *__restrict__ err, unsigned long long wait_ns, int fault_skip) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u));
    const int mask_words = (page_cap + 31) / 32;
    unsigned *s_mask = reinterpret_cast<unsigned *>(&S + 1);
    int *s_list = reinterpret_cast<int *>(s_mask + mask_words);
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)gridDim.x;
    const int r = (int)blockIdx.x, u = (int)blockIdx.y;
    const int b = u / n_kv_heads, h = u % n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qr = lane >> 2, qc = lane & 3;
    if (tid < kW * kR) {
        mbar_init(&S.scan_bar[tid / kR][tid % kR], 1);
        mbar_init(&S.page_bar[tid / kR][tid % kR], 1);
    }
    if (tid < 2) {
        mbar_init(&S.st_full[tid], kW);
        mbar_init(&S.st_empty[tid], g);
    }
    if (tid == 0) {
        mbar_init_fence();
        S.bad = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_par)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
    }
    __syncthreads();
    dep_wait();  // the previous kernel of the stream (an insert or a build) is complete

    const size_t up = (size_t)u * np_cap, ug = (size_t)u * page_cap;
    const int Np = min(n_parents[u], np_cap);
    const int P = min(n_pages[u], page_cap);
    const int Ps = max(0, P - n_pos);  // semantic pages; the last n_pos are positional
    const bool scan = k_pages > 0 && k_pages < Ps && Np > 0;
    const __nv_bfloat16 *Qg = Q + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
    bool ok = true;

    // ------------------------------------------------------------ scan ----
    // Rounds: in round j every warp scores its j-th tile (32 parents x 8 heads) and stages the
    // scores in shared memory; then warp hh < g, the worker of head hh, folds the round's 8 x 32
    // scores of its head into its list: lane i holds the i-th best key (score, -m) of the head
    // so far (i < k), and a score enters only if it reaches the current k-th, one at a time, or,
    // when many do (the first rounds), as a sorted batch merged with the list.
    unsigned long long lst = 0ull;
    if (scan) {
        // B fragments of q^T (k = 16 dims x n = 8 heads) for the 8 dim steps
        uint32_t qb[8][2];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const __nv_bfloat16 *row = Qg + (size_t)qr * kHeadDim + ks * 16 + 2 * qc;
            qb[ks][0] = qr < g ? *reinterpret_cast<const uint32_t *>(row) : 0u;
            qb[ks][1] = qr < g ? *reinterpret_cast<const uint32_t *>(row + 8) : 0u;
        }
        const int T = (Np + kRows - 1) / kRows;
        const int t_lo = (int)((long long)T * r / C), t_hi = (int)((long long)T * (r + 1) / C);
        const int nj = t_hi - t_lo > warp ? (t_hi - t_lo - warp + kW - 1) / kW : 0;
        const int rounds = (t_hi - t_lo + kW - 1) / kW;
        auto issue = [&](int j) {
            if (fault_skip) return;  // fault injection: the waits below give up
            const int row = (int)up + (t_lo + warp + kW * j) * kRows;
            unsigned char *slot = S.slots[warp][j % kR];
            unsigned long long *bar = &S.scan_bar[warp][j % kR];
            mbar_expect_tx(bar, kSlot);
            tma_load_2d(slot, &tm_par, bar, 0, row);
            tma_load_2d(slot + kScanHalf, &tm_par, bar, 64, row);
        };
        if (lane == 0)
            for (int j = 0; j < kR && j < nj; ++j) issue(j);
        float kth_s = -INFINITY;  // worker warps: the k-th score of the head's list (-inf until full)
        int failed = -1;          // the first tile whose wait gave up
        // worker warp `warp` < g folds round jr's scores of its head into its list
        auto head_work = [&](int jr) {
            if (warp >= g) return;
            if (!__all_sync(0xffffffffu, mbar_wait(&S.st_full[jr & 1], (jr >> 1) & 1, wait_ns))) ok = false;
            // lane L takes parent L of each of the round's 8 tiles (NaN: no such parent)
            float v8[kW];
#pragma unroll
            for (int w = 0; w < kW; ++w) {
                const int t = t_lo + w + kW * jr;
                v8[w] = t < t_hi && t * kRows + lane < Np ? S.stage[jr & 1][w][warp][lane] : __int_as_float(0x7fc00000);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.st_empty[jr & 1]);  // the buffer is free: the scores are in registers
            float th = kth_s;
            int npass = 0;
#pragma unroll
            for (int w = 0; w < kW; ++w) npass += __popc(__ballot_sync(0xffffffffu, v8[w] >= th));
            if (npass == 0) return;
            if (npass > 32) {  // many (the first rounds): first raise the bar to the round's own k-th score
                uint32_t o[kW];
#pragma unroll
                for (int w = 0; w < kW; ++w) o[w] = v8[w] == v8[w] ? ord_f32(v8[w]) : 0u;
                const uint32_t T = kth_largest_ord(o, k_pages);
                if (T) th = fmaxf(th, unord_f32(T));
            }
#pragma unroll 1
            for (int w = 0; w < kW; ++w) {
                float v = v8[0];  // v8[w] by selects: the values stay in registers
#pragma unroll
                for (int i = 1; i < kW; ++i) v = w == i ? v8[i] : v;
                const bool pass = v >= th;
                unsigned bal = __ballot_sync(0xffffffffu, pass);
                if (!bal) continue;
                const unsigned long long mine = pass ? sort_key(v, (t_lo + w + kW * jr) * kRows + lane) : 0ull;
                if (__popc(bal) <= 2) {
                    while (bal) {
                        const int src = __ffs(bal) - 1;
                        bal &= bal - 1;
                        list_insert(lst, __shfl_sync(0xffffffffu, mine, src), k_pages, lane);
                    }
                } else {
                    const unsigned long long merged = merge32(lst, sort32_desc(mine, lane));
                    lst = lane < k_pages ? merged : 0ull;
                }
                const unsigned long long kth = __shfl_sync(0xffffffffu, lst, k_pages - 1);
                if (kth) th = fmaxf(th, kth_s = unord_f32((uint32_t)(kth >> 32)));
            }
        };
        // software pipeline without CTA-wide barriers: round j is staged once the workers are
        // done with round j - 2 (its buffer), and a worker folds round j - 1 after staging round j
        for (int j = 0; j < rounds; ++j) {
            bool have = j < nj && ok;
            if (have) {
                ok = __all_sync(0xffffffffu, mbar_wait(&S.scan_bar[warp][j % kR], (j / kR) & 1, wait_ns));
                if (!ok) failed = j;
                have = ok;
            }
            float acc[2][4] = {{-INFINITY, -INFINITY, -INFINITY, -INFINITY}, {-INFINITY, -INFINITY, -INFINITY, -INFINITY}};
            if (have) {
                const uint32_t base = su32(S.slots[warp][j % kR]);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        // matrices: (rows 0-7, dims lo), (rows 8-15, dims lo), (rows 0-7, dims hi), (rows 8-15, dims hi)
                        const int mi = lane >> 3;
                        const uint32_t addr =
                            sw_addr(base, 16 * mt + (mi & 1) * 8 + (lane & 7), 2 * ks + (mi >> 1), kScanHalf);
                        uint32_t a[4];
                        ldsm_x4(addr, a[0], a[1], a[2], a[3]);
                        mma16816(acc[mt], a, qb[ks][0], qb[ks][1]);
                    }
                }
                __syncwarp();
                if (lane == 0 && j + kR < nj) issue(j + kR);  // the slot's rows are in registers now
            }
            if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(&S.st_empty[j & 1], ((j - 2) >> 1) & 1, wait_ns)))
                ok = false;  // (ok stays warp-uniform)
            // acc[mt][e]: parent 16 mt + qr + 8 (e >> 1) of the tile, head 2 qc + (e & 1)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    S.stage[j & 1][warp][2 * qc + (e & 1)][16 * mt + qr + 8 * (e >> 1)] = acc[mt][e];
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.st_full[j & 1]);
            if (j >= 1) head_work(j - 1);
        }
        if (rounds > 0) head_work(rounds - 1);
        ok = __all_sync(0xffffffffu, ok);
        if (failed >= 0 && !fault_skip && lane == 0)  // drain what this warp issued before the slots are reused
            for (int jj = failed; jj < nj && jj < failed + kR; ++jj)
                mbar_wait(&S.scan_bar[warp][jj % kR], (jj / kR) & 1, wait_ns);
    }
    if (!ok) {
        set_err(err, ICE_ERR_TIMEOUT);
        if (lane == 0) S.bad = 1;
    }
    if (scan && warp < g) S.top[warp][lane] = lst;  // this CTA's best k of head `warp`
    __syncthreads();

    // ---------------------------------------------------------- select ----
    if (C > 1) cluster.sync();  // every CTA's lists are in place
    else __syncthreads();
    if (r == 0) {
        // rank 0: the unit's union
        for (int x = tid; x < mask_words; x += kT) {
            unsigned v = 0u;
            if (!scan) {  // every page (the budget covers the semantic pages), or only the positional ones
                const int lo = k_pages > 0 ? 0 : Ps;
                const int a = max(x * 32, lo), e = min(x * 32 + 32, P);
                if (e > a) v = (e - a == 32 ? 0xffffffffu : ((1u << (e - a)) - 1u)) << (a - x * 32);
            } else {
                const int a = max(x * 32, Ps), e = min(x * 32 + 32, P);  // positional pages: always in the union
                if (e > a) v = (e - a == 32 ? 0xffffffffu : ((1u << (e - a)) - 1u)) << (a - x * 32);
            }
            s_mask[x] = v;
        }
        __syncthreads();
        if (scan && warp < g) {
            unsigned long long best = S.top[warp][lane];
            for (int c = 1; c < C; ++c) best = merge32(best, cluster.map_shared_rank(&S.top[warp][0], c)[lane]);
            // lane i < k: the head's i-th best parent and its pages, until k pages
            int pm = -1, fp = 0, pc = 0, contig = 1;
            if (lane < k_pages && best != 0ull) {
                pm = key_id(best);
                fp = parent_first_page[up + pm];
                pc = parent_n_pages[up + pm];
                contig = parent_last_page[up + pm] - fp + 1 == pc;
            }
            int incl = pc;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            const int tk = max(0, min(pc, k_pages - (incl - pc)));
            int pg = fp;
            for (int i = 0; i < tk; ++i) {
                const int qq = contig ? fp + i : pg;
                if (qq < 0 || qq >= Ps) break;
                atomicOr(&s_mask[qq >> 5], 1u << (qq & 31));
                if (!contig) pg = page_next[ug + qq];
            }
        }
        __syncthreads();
        // ascending list of the union: thread tid owns words [tid * wpt, (tid + 1) * wpt)
        const int wpt = (mask_words + kT - 1) / kT;
        const int wb = tid * wpt, we = min(mask_words, wb + wpt);
        int cnt = 0;
        for (int x = wb; x < we; ++x) cnt += __popc(s_mask[x]);
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) S.wsum[warp] = incl;
        __syncthreads();
        int pos = incl - cnt, total = 0;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            pos += w < warp ? S.wsum[w] : 0;
            total += S.wsum[w];
        }
        for (int x = wb; x < we && pos < max_sel; ++x) {
            unsigned bb = s_mask[x];
            while (bb && pos < max_sel) {
                const int bit = __ffs(bb) - 1;
                bb &= bb - 1;
                const int pgid = x * 32 + bit;
                s_list[pos] = pgid;
                sel_pages[(size_t)u * max_sel + pos] = pgid;
                ++pos;
            }
        }
        const int n_sel = min(total, max_sel);
        for (int x = n_sel + tid; x < max_sel; x += kT) {
            sel_pages[(size_t)u * max_sel + x] = -1;
            if (buf_len) buf_len[(size_t)u * max_sel + x] = 0;
        }
        if (tid == 0) {
            if (total > max_sel) set_err(err, ICE_ERR_CAPACITY);
            sel_count[u] = n_sel;
            S.n_sel = n_sel;
        }
    }
    if (C > 1) cluster.sync();  // rank 0's union list is complete
    else __syncthreads();

    // ---------------------------------------------------------- attend ----
    const int *list = r == 0 ? s_list : cluster.map_shared_rank(s_list, 0);
    const int n = r == 0 ? S.n_sel : *cluster.map_shared_rank(&S.n_sel, 0);
    const int ps = (n + C - 1) / C;
    const int xs = r * ps;
    const int np_cta = max(0, min(n, xs + ps) - xs);
    const size_t ubase = (size_t)u * max_sel;
    const bool store = buf_len != nullptr;  // also write the contiguous buffer
    const int nk = np_cta > warp ? (np_cta - warp + kW - 1) / kW : 0;  // <= 32 (checked on the host)
    int my_pid = 0, my_len = 0;
    if (lane < nk) {
        my_pid = list[xs + warp + lane * kW];
        my_len = page_len[ug + my_pid];
    }
    auto issue = [&](int k, int pid) {
        if (fault_skip) return;  // fault injection: the waits below give up
        const int row = (int)((ug + pid) * kPage);
        unsigned char *slot = S.slots[warp][k % kR];
        unsigned long long *bar = &S.page_bar[warp][k % kR];
        mbar_expect_tx(bar, kSlot);
        tma_load_2d(slot, &tm_k, bar, 0, row);
        tma_load_2d(slot + kPageHalf, &tm_k, bar, 64, row);
        tma_load_2d(slot + kPageTile, &tm_v, bar, 0, row);
        tma_load_2d(slot + kPageTile + kPageHalf, &tm_v, bar, 64, row);
    };
    {
        int pf[kR];
#pragma unroll
        for (int k = 0; k < kR; ++k) pf[k] = __shfl_sync(0xffffffffu, my_pid, k);
        if (lane == 0) {
            fence_proxy_async();  // the slots held the warps' lists (generic writes)
#pragma unroll
            for (int k = 0; k < kR; ++k)
                if (nk > k) issue(k, pf[k]);
        }
    }
    uint32_t qa[8][4];
    load_q_frag<1>(Qg, g, qa);
    AttnState st;
    st.init();
    bool pok = true;
    int k = 0;
    for (; k < nk; ++k) {
        const int x = xs + warp + k * kW;
        const int len = __shfl_sync(0xffffffffu, my_len, k);
        const int pid_next = __shfl_sync(0xffffffffu, my_pid, (k + kR) & 31);
        if (store && lane == 0) buf_len[ubase + x] = len;
        if (pok) pok = mbar_wait(&S.page_bar[warp][k % kR], (k / kR) & 1, wait_ns);
        pok = __all_sync(0xffffffffu, pok);
        if (!pok) break;
        unsigned char *sp = S.slots[warp][k % kR];
        if (store && lane == 0) {  // the contiguous buffer, straight from shared memory
            fence_proxy_async();
            const int row = (int)((ubase + x) * kPage);
            tma_store_2d(&tm_kb, sp, 0, row);
            tma_store_2d(&tm_kb, sp + kPageHalf, 64, row);
            tma_store_2d(&tm_vb, sp + kPageTile, 0, row);
            tma_store_2d(&tm_vb, sp + kPageTile + kPageHalf, 64, row);
            bulk_commit();
        }
        attend_page<1>(qa, su32(sp), su32(sp + kPageTile), len, scale, st);
        __syncwarp();
        if (lane == 0 && k + kR < nk) {  // refill this slot once its stores have read it
            if (store) bulk_wait_read_all();
            issue(k + kR, pid_next);
        }
        __syncwarp();
    }
    if (!pok) {
        if (!fault_skip && lane == 0)  // drain what this warp issued before the slots are reused
            for (int kk = k; kk < nk && kk < k + kR; ++kk) mbar_wait(&S.page_bar[warp][kk % kR], (kk / kR) & 1, wait_ns);
        set_err(err, ICE_ERR_TIMEOUT);
        if (lane == 0) S.bad = 1;
    }
    if (store && lane == 0) bulk_wait_read_all();  // the slots are reused below
    if (qc == 0) {
        S.ml[warp][qr][0] = st.m[0];
        S.ml[warp][qr][1] = st.l[0];
    }
    __syncthreads();

    // ----------------------------------------------------------- merge ----
    float *s_o = reinterpret_cast<float *>(&S.slots[0][0][0]);  // [kW][8][d]
    float *s_co = s_o + kW * kGT * kHeadDim;                     // [8][d]: this CTA's output (read over DSMEM)
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2 *>(s_o + ((size_t)warp * kGT + qr) * kHeadDim + 8 * nt + 2 * qc) =
            make_float2(st.o[nt][0], st.o[nt][1]);
    if (tid < g) {
        float M = -INFINITY;
        for (int w = 0; w < kW; ++w) M = fmaxf(M, S.ml[w][tid][0]);
        float L = 0.f;
        for (int w = 0; w < kW; ++w) {
            const float m = S.ml[w][tid][0];
            const float wt = m == -INFINITY ? 0.f : expf(m - M);
            S.wgt[w][tid] = wt;
            L = fmaf(S.ml[w][tid][1], wt, L);
        }
        if (S.bad) L = __int_as_float(0x7fc00000);  // NaN: carried into O
        S.cm[tid] = M;
        S.cl[tid] = L;
    }
    __syncthreads();
    float *Ou = O + ((size_t)b * n_q_heads + (size_t)h * g) * kHeadDim;
    for (int xx = tid; xx < g * kHeadDim; xx += kT) {
        const int hh = xx / kHeadDim, d = xx % kHeadDim;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kW; ++w) acc = fmaf(s_o[((size_t)w * kGT + hh) * kHeadDim + d], S.wgt[w][hh], acc);
        if (C == 1) {
            const float L = S.cl[hh];
            Ou[(size_t)hh * kHeadDim + d] = L > 0.f ? acc / L : (L == L ? 0.f : L);
        } else {
            s_co[hh * kHeadDim + d] = acc;
        }
    }
    if (C > 1) {
        cluster.sync();  // every CTA's partial is in place
        for (int hh = r; hh < g; hh += C) {
            if (tid < kHeadDim) {
                float M = -INFINITY;
                for (int c = 0; c < C; ++c) M = fmaxf(M, *cluster.map_shared_rank(&S.cm[hh], c));
                float L = 0.f, acc = 0.f;
                for (int c = 0; c < C; ++c) {
                    const float m = *cluster.map_shared_rank(&S.cm[hh], c);
                    const float wt = m == -INFINITY ? 0.f : expf(m - M);
                    L = fmaf(*cluster.map_shared_rank(&S.cl[hh], c), wt, L);
                    acc = fmaf(cluster.map_shared_rank(s_co + hh * kHeadDim, c)[tid], wt, acc);
                }
                Ou[(size_t)hh * kHeadDim + tid] = L > 0.f ? acc / L : (L == L ? 0.f : L);
            }
        }
        cluster.sync();  // no CTA leaves while another reads its shared memory
    }
}

}  // namespace

namespace {

int sm_count_here() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// CTAs per unit: the largest power of two up to 8 with U * C * 2 <= SMs.
int cluster_size(int units, int n_sm) {
    int C = 1;
    while (C < kMaxC && (long long)units * C * 2 <= n_sm) C *= 2;
    return C;
}

bool shapes_fit(const ice_params &p, int k_pages, int max_sel, int C) {
    const int g = p.n_q_heads / p.n_kv_heads;
    const long long U = units_of(p);
    return p.dtype == ICE_BF16 && g >= 1 && g <= kGT && k_pages >= 0 && k_pages <= 32 && max_sel <= 256 * C &&
           smem_bytes(p.page_cap, max_sel) <= 227 * 1024 && U * p.np_cap < (1ll << 31) &&
           U * p.page_cap * kPage < (1ll << 31) && U * max_sel * kPage < (1ll << 31);
}

}  // namespace

bool decode_fused_supported(const ice_params &p, int k_pages, int max_sel) {
    return shapes_fit(p, k_pages, max_sel, cluster_size(units_of(p), sm_count_here()));
}

cudaError_t launch_decode_fused(const ice_params &p, const ice_index &idx, const void *Q, int k_pages,
                                int32_t *sel_pages, int32_t *sel_count, int max_sel, void *kbuf, void *vbuf,
                                int32_t *buf_len, float scale, float *O, int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int g = p.n_q_heads / p.n_kv_heads;
    int C = cluster_size(U, sm_count_here());
    if (!shapes_fit(p, k_pages, max_sel, C) || ((uintptr_t)Q & 3u) != 0) return cudaErrorNotSupported;
    CUtensorMap tpar, tk, tv, tkb, tvb;
    const unsigned long long prow = (unsigned long long)U * p.page_cap * kPage;
    if (!make_map_bf16(&tpar, idx.parent_keys, (unsigned long long)U * p.np_cap, kHeadDim, 64, kRows,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bf16(&tk, idx.pool_k, prow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bf16(&tv, idx.pool_v, prow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorNotSupported;
    if (buf_len) {
        const unsigned long long brow = (unsigned long long)U * max_sel * kPage;
        if (!make_map_bf16(&tkb, kbuf, brow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_bf16(&tvb, vbuf, brow, kHeadDim, 64, kPage, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorNotSupported;
    } else {
        tkb = tk;  // unused
        tvb = tv;
    }
    const size_t smem = smem_bytes(p.page_cap, max_sel);
    cudaError_t e = cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
        return e;
    const bool fault = fault_armed("timeout");
    const int n_pos = pos_split(p).n_pos;
    for (;;) {  // the largest cluster the device can schedule
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C, U);
        cfg.blockDim = dim3(kT);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute at[2];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = C;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 2;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, k_decode_fused, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            if (C == 1 || !shapes_fit(p, k_pages, max_sel, C / 2)) return cudaErrorNotSupported;
            C /= 2;
            continue;
        }
        e = cudaLaunchKernelEx(&cfg, k_decode_fused, tpar, tk, tv, tkb, tvb, static_cast<const __nv_bfloat16 *>(Q), g,
                               p.n_q_heads, p.n_kv_heads, p.np_cap, p.page_cap, k_pages, n_pos,
                               (const int32_t *)idx.n_parents, (const int32_t *)idx.n_pages,
                               (const int32_t *)idx.parent_first_page, (const int32_t *)idx.parent_last_page,
                               (const int32_t *)idx.parent_n_pages, (const int32_t *)idx.page_next,
                               (const int32_t *)idx.page_len, sel_pages, sel_count, max_sel, buf_len, scale, O, err,
                               fault ? kFaultWaitNs : kWaitNs, fault ? 1 : 0);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
}

}  // namespace ice
