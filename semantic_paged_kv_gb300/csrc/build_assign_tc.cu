// Index build, step a3 (nearest parent) on the sm_103a tensor cores.
//
// IceCache popular-science article (aitangshan.cn/news/751385), section 三:
// every token is attached to the most similar point of the level above;
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 2: each lower-level point recognises its
// nearest parent one level up.  With every lifted key of norm M,
//   argmin_m |k'_j - p'_m|^2 = argmax_m (k_j . p_m + e_j e_m),
// a dense contraction of the keys with the parent keys followed by a row
// argmax.  bf16 products are exact in fp32; the sum is accumulated in fp32.
//
// One CTA per (128-token tile, unit), 6 warps, one CTA per SM:
//   warp 0      TMA producer: the 128x128 key tile once, then the unit's
//               parent keys in 256-row tiles through a 2-stage ring
//               (128-byte swizzled, two 64-column halves per tile);
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=256, K=16, bf16 -> fp32) into one of two TMEM
//               accumulators, committing to the ring's empty barrier and to
//               the accumulator's full barrier;
//   warps 2..5  epilogue: TMEM row = token, 32 columns per tcgen05.ld; score
//               = acc + e_j e_m, running argmax with the lowest index on
//               exact ties; releases the accumulator to the MMA warp.
// Every mbarrier wait gives up after ~2 s (globaltimer), records
// ICE_ERR_TIMEOUT, drains what it issued and frees TMEM before returning.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int BM = 128;      // tokens per CTA (TMEM lanes)
constexpr int BN = 256;      // parents per MMA tile (TMEM columns per accumulator)
constexpr int NSTAGE = 2;    // parent-tile ring depth
constexpr int kThreads = 192;
constexpr uint32_t A_HALF = BM * 128;     // 128 rows x 128 bytes (64 bf16 columns)
constexpr uint32_t A_BYTES = 2 * A_HALF;  // d = 128 -> two halves
constexpr uint32_t B_HALF = BN * 128;
constexpr uint32_t B_STAGE = 2 * B_HALF;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr unsigned long long kWaitNs = 2000000000ull;
// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, N, M.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

struct Bars {
    unsigned long long full[NSTAGE], empty[NSTAGE], a_full, tfull[2], tempty[2];
    uint32_t tmem_base;
};
constexpr size_t kSmemBytes = 1024 /*align slack*/ + A_BYTES + NSTAGE * B_STAGE + 2 * BN * sizeof(float) + sizeof(Bars);

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(unsigned long long *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of the given parity; false after kWaitNs.
__device__ __forceinline__ bool mbar_wait(unsigned long long *b, uint32_t parity) {
    if (mbar_test(b, parity)) return true;
    const unsigned long long t0 = now_ns();
    while (!mbar_test(b, parity))
        if (now_ns() - t0 > kWaitNs) return false;
    return true;
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, unsigned long long *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(su32(bar)), "r"(x), "r"(y)
        : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(IDESC), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(unsigned long long *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_assign_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmP, int N, int np_cap,
                int n_cap, const int32_t *__restrict__ n_parents, const double *__restrict__ m2,
                const double *__restrict__ norm2, const float *__restrict__ parent_e,
                int32_t *__restrict__ token_parent, int32_t *__restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem;
    unsigned char *sB = smem + A_BYTES;
    float *sE = reinterpret_cast<float *>(sB + NSTAGE * B_STAGE);
    Bars *bars = reinterpret_cast<Bars *>(sE + 2 * BN);

    const int u = blockIdx.y;
    const int m0 = blockIdx.x * BM;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    const int T = (Np + BN - 1) / BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->a_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tfull[b], 1);
            mbar_init(&bars->tempty[b], 4 * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&bars->tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    bool ok = true;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0 && T > 0) {
            const int row0 = u * N + m0;
            mbar_expect_tx(&bars->a_full, A_BYTES);
            tma_load_2d(sA, &tmK, &bars->a_full, 0, row0);
            tma_load_2d(sA + A_HALF, &tmK, &bars->a_full, 64, row0);
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int s = t % NSTAGE;
                const uint32_t ph = (t / NSTAGE) & 1;
                if (!mbar_wait(&bars->empty[s], ph ^ 1)) {
                    ok = false;
                    break;
                }
                unsigned char *dst = sB + s * B_STAGE;
                const int y = u * np_cap + t * BN;
                mbar_expect_tx(&bars->full[s], B_STAGE);
                tma_load_2d(dst, &tmP, &bars->full[s], 0, y);
                tma_load_2d(dst + B_HALF, &tmP, &bars->full[s], 64, y);
                issued = t + 1;
            }
            // drain: every issued copy has landed before the CTA may exit
            for (int t = (issued > NSTAGE ? issued - NSTAGE : 0); t < issued; ++t)
                mbar_wait(&bars->full[t % NSTAGE], (t / NSTAGE) & 1);
            mbar_wait(&bars->a_full, 0);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && T > 0) {
            int issued = 0;
            if (!mbar_wait(&bars->a_full, 0)) ok = false;
            const uint32_t a0 = su32(sA);
            for (int t = 0; ok && t < T; ++t) {
                const int s = t % NSTAGE, b = t & 1;
                const uint32_t ph = (t / NSTAGE) & 1, bph = (t >> 1) & 1;
                if (!mbar_wait(&bars->tempty[b], bph ^ 1) || !mbar_wait(&bars->full[s], ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t b0 = su32(sB + s * B_STAGE);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k & 3) * 32;  // 16 bf16 columns inside the swizzle atom
                    const uint64_t da = sw128_desc(a0 + (k >> 2) * A_HALF + off);
                    const uint64_t db = sw128_desc(b0 + (k >> 2) * B_HALF + off);
                    umma_bf16(tmem + b * BN, da, db, k > 0 ? 1u : 0u);
                }
                umma_commit(&bars->empty[s]);
                umma_commit(&bars->tfull[b]);
                issued = t + 1;
            }
            // drain: the last accumulator is complete before TMEM is freed
            if (issued > 0) mbar_wait(&bars->tfull[(issued - 1) & 1], ((issued - 1) >> 1) & 1);
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const long long j = (long long)m0 + row;
        float ej = 0.f;
        if (j < N) {
            const double r = m2[u] - norm2[(size_t)u * N + j];
            ej = (float)sqrt(r > 0.0 ? r : 0.0);
        }
        float best = -INFINITY;
        int bidx = 0x7fffffff;
        const int et = threadIdx.x - 64;  // 0..127 among the epilogue threads
        for (int t = 0; t < T; ++t) {
            const int b = t & 1;
            const uint32_t bph = (t >> 1) & 1;
            float *se = sE + b * BN;
            for (int c = et; c < BN; c += 128) {
                const int m = t * BN + c;
                se[c] = m < Np ? parent_e[(size_t)u * np_cap + m] : 0.f;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            // a failed wait stops this warp's work but not its barrier turns,
            // so the other epilogue warps never wait for it
            if (ok) ok = mbar_wait(&bars->tfull[b], bph);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            const int valid = ok ? min(BN, Np - t * BN) : 0;
            for (int c0 = 0; c0 < valid; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + c0), v);
                float cmax = -INFINITY;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = (c0 + i < valid) ? fmaf(ej, se[c0 + i], v[i]) : -INFINITY;
                    cmax = fmaxf(cmax, v[i]);
                }
                if (cmax > best) {
                    int first = 0;
#pragma unroll
                    for (int i = 31; i >= 0; --i)
                        if (v[i] == cmax) first = i;
                    best = cmax;
                    bidx = t * BN + c0 + first;
                }
            }
            tc_fence_before();
            mbar_arrive(&bars->tempty[b]);
        }
        if (ok && j < N && Np > 0) {
            int32_t *tp = token_parent + (size_t)u * n_cap + j;
            if (*tp < 0) *tp = bidx;  // promoted tokens keep themselves
        }
    }
    if (!ok) set_err(err, ICE_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------------ host --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// 2-D bf16 map over rows of 128 elements (256 bytes), box {64, box_rows}, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, unsigned long long rows, unsigned box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_assign_tc(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                             int32_t *err, cudaStream_t s) {
    if (p.dtype != ICE_BF16) return launch_assign_simt(p, K, idx, ws, err, s);
    const int U = units_of(p);
    CUtensorMap tmK, tmP;
    if (!make_map(&tmK, K, (unsigned long long)U * p.n_tokens, BM) ||
        !make_map(&tmP, idx.parent_keys, (unsigned long long)U * p.np_cap, BN))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_assign_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(ceil_div(p.n_tokens, BM), U);
    k_assign_tc<<<grid, kThreads, kSmemBytes, s>>>(tmK, tmP, p.n_tokens, p.np_cap, p.n_cap, idx.n_parents, idx.m2,
                                                   ws.norm2, idx.parent_e, idx.token_parent, err);
    return cudaGetLastError();
}

}  // namespace ice
