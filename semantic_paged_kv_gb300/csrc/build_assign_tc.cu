// Index build, step a3 (nearest parent) on the sm_103a tensor cores.
//
// IceCache popular-science article (aitangshan.cn/news/751385), section 三:
// every token is attached to the most similar point of the level above;
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 2: each lower-level point recognises its
// nearest parent one level up.  With every lifted key of norm M,
//   argmin_m |k'_j - p'_m|^2 = argmax_m (k_j . p_m + e_j e_m),
// a dense contraction of the keys with the parent keys followed by a row
// argmax.  The whole score is one contraction here: each key row carries 16
// extra bf16 columns [e1, e1, e2, e1, e2, e3, 0...] and each parent row
// [f1, f2, f1, f3, f2, f1, 0...] (e = e1 + e2 + e3, f likewise, split into
// bf16 parts by the promotion kernel), whose products give e_j e_m to about
// 2^-23 relative; all bf16 products are exact in fp32 and the sum is
// accumulated in fp32.
//
// Persistent kernel, one CTA per SM (18 warps), looping over work items =
// (unit, 128-token tile) in unit-major order, so that the CTAs working at
// the same time share one unit's parent table in L2:
//   warp 0      TMA producer: per item the 128x128 key tile (128-byte
//               swizzle, two 64-column halves) and its 128x16 extra tile
//               (32-byte swizzle) into one of two key buffers, then the
//               unit's parent keys and parent extras in 256-row tiles
//               through a 2-stage ring;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=256, K=16, bf16 -> fp32; 8 K-steps of keys plus
//               one of extras) into one of two TMEM accumulators, committing
//               to the ring's empty barrier, the accumulator's full barrier
//               and, after an item's last tile, the key buffer's empty
//               barrier;
//   warps 2..17 epilogue: warp w reads TMEM lane quarter w % 4 and the 64
//               columns (w - 2) / 4 of each tile in one tcgen05 wait, frees
//               the accumulator at once and then keeps a running argmax with
//               the lowest index on exact ties (the tile maximum by a tree of
//               three-input maxima; a lane whose maximum moved finds its
//               column inside the lowest nine-column group of the tree that
//               holds it when at most 4 lanes of the warp moved, else over
//               all 64); the four column quarters of a
//               row combine through shared memory at the end of the item.
//               The next item's promoted flags are prefetched.
// Every mbarrier wait gives up after ~2 s (globaltimer) and records
// ICE_ERR_TIMEOUT; roles drain what they issued and TMEM is freed before
// the CTA returns.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace ice {
namespace {

using namespace tc;

constexpr int BM = 128;      // tokens per CTA (TMEM lanes)
constexpr int BN = 256;      // parents per MMA tile (TMEM columns per accumulator)
constexpr int NSTAGE = 2;    // parent-tile ring depth
constexpr int kEpiWarps = 16;  // 4 per TMEM lane quarter, 64 columns of each tile apiece
constexpr int kEpiCols = BN / (kEpiWarps / 4);
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kExtra = 16;                  // extra K columns (bf16)
constexpr uint32_t A_HALF = BM * 128;       // 128 rows x 128 bytes (64 bf16 columns)
constexpr uint32_t A_BYTES = 2 * A_HALF;    // d = 128 -> two halves
constexpr uint32_t A2_BYTES = BM * kExtra * 2;
constexpr uint32_t B_HALF = BN * 128;
constexpr uint32_t B_STAGE = 2 * B_HALF;
constexpr uint32_t B2_STAGE = BN * kExtra * 2;
constexpr uint32_t TMEM_COLS = 2 * BN;
// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, N, M.
constexpr uint32_t IDESC = idesc_bf16(BM, BN);

struct Bars {
    unsigned long long full[NSTAGE], empty[NSTAGE], a_full[2], a_empty[2], tfull[2], tempty[2];
    float comb_s[kEpiWarps / 4 - 1][BM];  // column quarters 1..3 of each row
    int comb_i[kEpiWarps / 4 - 1][BM];
    uint32_t tmem_base;
};
static_assert(kEpiCols == 64, "the epilogue's maximum tree is written for 64 columns");

// The lowest index i in [B, B + 9) with v[i] == x (B + 8 if none; the caller
// knows one is there).  The indices are compile-time, so v stays in registers.
template <int B>
__device__ __forceinline__ int lowest9(const float (&v)[64], float x) {
    int f = B + 8;
#pragma unroll
    for (int j = 7; j >= 0; --j) f = v[B + j] == x ? B + j : f;
    return f;
}

// max(a, b, c) in one instruction (no NaN reaches it: scores are finite or -inf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

constexpr size_t kSmemBytes = 1024 /*align slack*/ + 2 * A_BYTES + NSTAGE * B_STAGE + 2 * A2_BYTES +
                              NSTAGE * B2_STAGE + sizeof(Bars);

// Work item -> (unit, first token) and the unit's parent-tile count.
struct Item {
    int u, m0, Np, T;
};
__device__ __forceinline__ Item item_of(int item, int mt_per_unit, const int32_t *n_parents, int np_cap) {
    Item it;
    it.u = item / mt_per_unit;
    it.m0 = (item % mt_per_unit) * BM;
    it.Np = min(n_parents[it.u], np_cap);
    it.T = (it.Np + BN - 1) / BN;
    return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_assign_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmP,
                const __grid_constant__ CUtensorMap tmK2, const __grid_constant__ CUtensorMap tmP2, int N, int np_cap,
                int n_cap, int n_items, int mt_per_unit, const int32_t *__restrict__ n_parents,
                int32_t *__restrict__ token_parent, int32_t *__restrict__ err) {
    dep_wait();  // the previous kernel of the stream is complete (launched as its dependent)
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;                         // two key buffers
    unsigned char *sB = sA + 2 * A_BYTES;             // parent ring
    unsigned char *sA2 = sB + NSTAGE * B_STAGE;       // two key-extra buffers
    unsigned char *sB2 = sA2 + 2 * A2_BYTES;          // parent-extra ring
    Bars *bars = reinterpret_cast<Bars *>(sB2 + NSTAGE * B2_STAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->a_full[b], 1);
            mbar_init(&bars->a_empty[b], 1);
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
            int gt = 0, it = 0;
            int last_a = -1;
            for (int item = blockIdx.x; ok && item < n_items; item += G, ++it) {
                const Item I = item_of(item, mt_per_unit, n_parents, np_cap);
                const int ab = it & 1;
                if (!mbar_wait(&bars->a_empty[ab], ((it >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                unsigned char *a = sA + ab * A_BYTES;
                const int row0 = I.u * N + I.m0;
                mbar_expect_tx(&bars->a_full[ab], A_BYTES + A2_BYTES);
                tma_load_2d(a, &tmK, &bars->a_full[ab], 0, row0);
                tma_load_2d(a + A_HALF, &tmK, &bars->a_full[ab], 64, row0);
                tma_load_2d(sA2 + ab * A2_BYTES, &tmK2, &bars->a_full[ab], 0, row0);
                last_a = it;
                for (int t = 0; t < I.T; ++t, ++gt) {
                    const int s = gt % NSTAGE;
                    if (!mbar_wait(&bars->empty[s], ((gt / NSTAGE) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    unsigned char *dst = sB + s * B_STAGE;
                    const int y = I.u * np_cap + t * BN;
                    mbar_expect_tx(&bars->full[s], B_STAGE + B2_STAGE);
                    tma_load_2d(dst, &tmP, &bars->full[s], 0, y);
                    tma_load_2d(dst + B_HALF, &tmP, &bars->full[s], 64, y);
                    tma_load_2d(sB2 + s * B2_STAGE, &tmP2, &bars->full[s], 0, y);
                }
            }
            // drain: every issued copy has landed before the CTA may exit
            for (int g2 = (gt > NSTAGE ? gt - NSTAGE : 0); g2 < gt; ++g2)
                mbar_wait(&bars->full[g2 % NSTAGE], (g2 / NSTAGE) & 1);
            for (int a2 = (last_a > 0 ? last_a - 1 : 0); a2 <= last_a; ++a2)
                mbar_wait(&bars->a_full[a2 & 1], (a2 >> 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int gt = 0, it = 0;
            for (int item = blockIdx.x; ok && item < n_items; item += G, ++it) {
                const Item I = item_of(item, mt_per_unit, n_parents, np_cap);
                const int ab = it & 1;
                if (!mbar_wait(&bars->a_full[ab], (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t a0 = su32(sA + ab * A_BYTES);
                const uint32_t a2 = su32(sA2 + ab * A2_BYTES);
                for (int t = 0; t < I.T; ++t, ++gt) {
                    const int s = gt % NSTAGE, b = gt & 1;
                    if (!mbar_wait(&bars->tempty[b], ((gt >> 1) & 1) ^ 1) ||
                        !mbar_wait(&bars->full[s], (gt / NSTAGE) & 1)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t b0 = su32(sB + s * B_STAGE);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (k & 3) * 32;  // 16 bf16 columns inside the swizzle atom
                        const uint64_t da = sw128_desc(a0 + (k >> 2) * A_HALF + off);
                        const uint64_t db = sw128_desc(b0 + (k >> 2) * B_HALF + off);
                        umma_bf16<IDESC>(tmem + b * BN, da, db, k > 0 ? 1u : 0u);
                    }
                    umma_bf16<IDESC>(tmem + b * BN, sw32_desc(a2), sw32_desc(su32(sB2 + s * B2_STAGE)), 1u);
                    umma_commit(&bars->empty[s]);
                    umma_commit(&bars->tfull[b]);
                }
                if (!ok) break;
                umma_commit(&bars->a_empty[ab]);  // the key buffer is free once these MMAs finish
            }
            // drain: the last accumulator is complete before TMEM is freed
            if (gt > 0) mbar_wait(&bars->tfull[(gt - 1) & 1], ((gt - 1) >> 1) & 1);
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int ew = warp - 2;  // 0..15
        const int q = warp & 3;   // TMEM lane quarter this warp may access
        const int hf = ew >> 2;   // column quarter of each 256-column tile
        const int row = q * 32 + lane;
        int gt = 0;
        Item I = blockIdx.x < n_items ? item_of(blockIdx.x, mt_per_unit, n_parents, np_cap) : Item{0, 0, 0, 0};
        int r_tp = -1;  // token_parent seed of this row (-1: to assign; >= 0 promoted, -2 sink / window: kept)
        if (blockIdx.x < n_items && (long long)I.m0 + row < N) r_tp = token_parent[(size_t)I.u * n_cap + I.m0 + row];
        for (int item = blockIdx.x; item < n_items; item += G) {
            const long long j = (long long)I.m0 + row;
            const bool keep = r_tp != -1;
            // the next item's row data, loaded while this item runs
            const int nitem = item + G;
            const Item In = nitem < n_items ? item_of(nitem, mt_per_unit, n_parents, np_cap) : Item{0, 0, 0, 0};
            if (nitem < n_items && (long long)In.m0 + row < N) r_tp = token_parent[(size_t)In.u * n_cap + In.m0 + row];
            float best = -INFINITY;
            int bidx = 0x7fffffff;
            for (int t = 0; t < I.T; ++t, ++gt) {
                const int b = gt & 1;
                // a failed wait stops this warp's work
                if (ok) ok = mbar_wait(&bars->tfull[b], (gt >> 1) & 1);
                ok = __all_sync(0xffffffffu, ok);
                fence_after();
                const int c_lo = t * BN + hf * kEpiCols;
                const int valid = ok ? max(0, min(kEpiCols, I.Np - c_lo)) : 0;
                float v[kEpiCols];
                if (valid > 0) {
                    const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + hf * kEpiCols);
#pragma unroll
                    for (int c = 0; c < kEpiCols; c += 32) tmem_ld32_nowait(ta + c, v + c);
                    tmem_wait_ld();
                }
                // the accumulator is free as soon as its values are in registers
                fence_before();
                mbar_arrive(&bars->tempty[b]);
                if (valid > 0) {
                    float cmax = -INFINITY;
                    int gk = -1;  // full tiles: the lowest nine-column group holding cmax (7: column 63)
                    if (valid >= kEpiCols) {
                        // three-input maxima: 64 -> 22 -> 8 -> 3 -> 1
                        float m1[22], m2[8];
#pragma unroll
                        for (int i = 0; i < 21; ++i) m1[i] = fmax3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
                        m1[21] = v[63];
#pragma unroll
                        for (int i = 0; i < 7; ++i) m2[i] = fmax3(m1[3 * i], m1[3 * i + 1], m1[3 * i + 2]);
                        m2[7] = m1[21];
                        cmax = fmax3(fmax3(m2[0], m2[1], m2[2]), fmax3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
                        gk = 7;
#pragma unroll
                        for (int i = 6; i >= 0; --i) gk = m2[i] == cmax ? i : gk;
                    } else {
#pragma unroll
                        for (int i = 0; i < kEpiCols; ++i) {
                            v[i] = i < valid ? v[i] : -INFINITY;
                            cmax = fmaxf(cmax, v[i]);
                        }
                    }
                    // the lanes whose maximum moves search their columns: through the
                    // group that holds cmax when few lanes do (each distinct group
                    // is a branch of the warp), over every column otherwise
                    const bool moved = cmax > best;
                    if (__popc(__ballot_sync(0xffffffffu, moved)) > 4) gk = -1;
                    if (moved) {  // columns ascend, so only a strictly larger score moves the argmax
                        int first = 63;
                        switch (gk) {
                        case 0: first = lowest9<0>(v, cmax); break;
                        case 1: first = lowest9<9>(v, cmax); break;
                        case 2: first = lowest9<18>(v, cmax); break;
                        case 3: first = lowest9<27>(v, cmax); break;
                        case 4: first = lowest9<36>(v, cmax); break;
                        case 5: first = lowest9<45>(v, cmax); break;
                        case 6: first = lowest9<54>(v, cmax); break;
                        case 7: first = 63; break;
                        default:  // many lanes, or a partial tile: every column
#pragma unroll
                            for (int i = kEpiCols - 1; i >= 0; --i)
                                if (v[i] == cmax) first = i;
                        }
                        best = cmax;
                        bidx = c_lo + first;
                    }
                }
            }
            // combine the column quarters of each row
            if (hf > 0) {
                bars->comb_s[hf - 1][row] = best;
                bars->comb_i[hf - 1][row] = bidx;
            }
            asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
            if (hf == 0) {
#pragma unroll
                for (int k = 0; k < kEpiWarps / 4 - 1; ++k) {
                    const float os = bars->comb_s[k][row];
                    const int oi = bars->comb_i[k][row];
                    if (better(os, oi, best, bidx)) {
                        best = os;
                        bidx = oi;
                    }
                }
                // promoted tokens keep themselves as parent, sink / window tokens stay outside the index
                if (ok && j < N && I.Np > 0 && !keep) token_parent[(size_t)I.u * n_cap + j] = bidx;
            }
            asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
            I = In;
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

int sm_count_assign() {
    static int n_sm = 0;
    if (!n_sm) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (n_sm <= 0) n_sm = 1;
    }
    return n_sm;
}

}  // namespace

cudaError_t launch_assign_level2_tc(const ice_params &p, const ice_index &idx, const BuildWs &ws, int32_t *err,
                                    cudaStream_t s) {
    // rows: the parents (their keys and row-form lifted coordinates); columns:
    // the level-2 nodes gathered dense; the output and the keep-seeds: parent2
    const int U = units_of(p);
    CUtensorMap tmK, tmP, tmK2, tmP2;
    const unsigned long long r = (unsigned long long)U * p.np_cap;
    if (r > 0x7FFFFFFFull || !make_map_bf16(&tmK, idx.parent_keys, r, kHeadDim, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bf16(&tmP, ws.keys2, r, kHeadDim, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bf16(&tmK2, ws.a_extra2, r, kExtra, kExtra, BM, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_bf16(&tmP2, ws.b_extra2, r, kExtra, kExtra, BN, CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(k_assign_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int mt = ceil_div(p.np_cap, BM);
    const int items = mt * U;
    const int n_sm = sm_count_assign();
    const int grid = items < n_sm ? items : n_sm;
    e = launch_dependent(k_assign_tc, dim3(grid), dim3(kThreads), kSmemBytes, s, tmK, tmP, tmK2, tmP2, p.np_cap,
                         p.np_cap, p.np_cap, items, mt, idx.n_nodes2, idx.parent2, err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_assign_tc(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                             int32_t *err, cudaStream_t s) {
    if (p.dtype != ICE_BF16) return launch_assign_simt(p, K, idx, ws, err, s);
    const int U = units_of(p);
    CUtensorMap tmK, tmP, tmK2, tmP2;
    const unsigned long long kr = (unsigned long long)U * p.n_tokens, pr = (unsigned long long)U * p.np_cap;
    if (!make_map_bf16(&tmK, K, kr, kHeadDim, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bf16(&tmP, idx.parent_keys, pr, kHeadDim, 64, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bf16(&tmK2, ws.a_extra, kr, kExtra, kExtra, BM, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_bf16(&tmP2, ws.b_extra, pr, kExtra, kExtra, BN, CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_assign_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    static int n_sm = 0;
    if (!n_sm) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (n_sm <= 0) n_sm = 1;
    }
    const int mt = ceil_div(p.n_tokens, BM);
    const int items = mt * U;
    const int grid = items < n_sm ? items : n_sm;
    {
        const cudaError_t e_ = launch_dependent(k_assign_tc, dim3(grid), dim3(kThreads), kSmemBytes, s, tmK, tmP,
                                                tmK2, tmP2, p.n_tokens, p.np_cap, p.n_cap, items, mt, idx.n_parents,
                                                idx.token_parent, err);
        if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
}

}  // namespace ice
