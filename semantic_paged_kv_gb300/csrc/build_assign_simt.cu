// Index build, step a3 (nearest parent) on CUDA cores, fp32 FMA accumulation.
//
// IceCache popular-science article (aitangshan.cn/news/751385), section 三:
// every token is attached to the most similar point of the level above;
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 2: each lower-level point recognises its
// nearest parent in the level above.  With every lifted key of norm M,
//   argmin_m |k'_j - p'_m|^2 = argmax_m (k_j . p_m + e_j e_m).
//
// This variant serves fp32 keys (the tensor cores have no exact fp32 input)
// and any dtype as a cross-check of the tensor-core kernel.  A CTA owns 32
// tokens (8 warps x 4 rows), stages them in shared memory as fp32, and
// streams the unit's parents through shared memory 32 at a time; lane l
// scores parent (chunk + l) against the warp's 4 rows.  Parent rows are
// stored with a 129-float stride so lane l reads bank (l + i) mod 32.
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kRowsPerWarp * (kThreads / 32);  // 32 tokens per CTA
constexpr int kChunk = 32;                             // parents per smem chunk
constexpr int kPad = kHeadDim + 1;

template <typename T>
__global__ void __launch_bounds__(kThreads) k_assign_simt(const T *__restrict__ K, int N, int np_cap, int n_cap,
                                                          const int32_t *__restrict__ n_parents,
                                                          const double *__restrict__ m2,
                                                          const double *__restrict__ norm2,
                                                          const T *__restrict__ parent_keys,
                                                          const float *__restrict__ parent_e,
                                                          int32_t *__restrict__ token_parent) {
    __shared__ float s_k[kRows][kHeadDim];
    __shared__ float s_p[kChunk][kPad];
    __shared__ float s_pe[kChunk];
    const int u = blockIdx.y;
    const long long r0 = (long long)blockIdx.x * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = n_parents[u];
    const T *Ku = K + (size_t)u * N * kHeadDim;
    const T *Pu = parent_keys + (size_t)u * np_cap * kHeadDim;

    for (int x = threadIdx.x; x < kRows * kHeadDim; x += kThreads) {
        const int r = x / kHeadDim, i = x % kHeadDim;
        const long long j = r0 + r;
        s_k[r][i] = j < N ? Elem<T>::load(Ku + (size_t)j * kHeadDim + i) : 0.f;
    }
    const double M2 = m2[u];
    float ej[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const long long j = r0 + warp * kRowsPerWarp + r;
        const double rr = j < N ? M2 - norm2[(size_t)u * N + j] : 0.0;
        ej[r] = (float)sqrt(rr > 0.0 ? rr : 0.0);
    }
    float best[kRowsPerWarp];
    int bidx[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        best[r] = -INFINITY;
        bidx[r] = 0x7fffffff;
    }
    for (int c0 = 0; c0 < Np; c0 += kChunk) {
        __syncthreads();
        for (int x = threadIdx.x; x < kChunk * kHeadDim; x += kThreads) {
            const int c = x / kHeadDim, i = x % kHeadDim;
            s_p[c][i] = (c0 + c < Np) ? Elem<T>::load(Pu + (size_t)(c0 + c) * kHeadDim + i) : 0.f;
        }
        if (threadIdx.x < kChunk)
            s_pe[threadIdx.x] = (c0 + threadIdx.x < Np) ? parent_e[(size_t)u * np_cap + c0 + threadIdx.x] : 0.f;
        __syncthreads();
        float acc[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) acc[r] = 0.f;
#pragma unroll 8
        for (int i = 0; i < kHeadDim; ++i) {
            const float pv = s_p[lane][i];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) acc[r] = fmaf(s_k[warp * kRowsPerWarp + r][i], pv, acc[r]);
        }
        if (c0 + lane < Np) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const float sc = fmaf(ej[r], s_pe[lane], acc[r]);
                if (sc > best[r]) {  // columns of a lane arrive in ascending order
                    best[r] = sc;
                    bidx[r] = c0 + lane;
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        float b = best[r];
        int bi = bidx[r];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, b, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (better(ob, oi, b, bi)) {
                b = ob;
                bi = oi;
            }
        }
        const long long j = r0 + warp * kRowsPerWarp + r;
        if (lane == 0 && j < N && Np > 0) {
            int32_t *tp = token_parent + (size_t)u * n_cap + j;
            if (*tp == -1) *tp = bi;  // promoted tokens keep themselves, sink / window tokens (-2) stay out
        }
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws, cudaStream_t s) {
    const int U = units_of(p);
    dim3 grid(ceil_div(p.n_tokens, kRows), U);
    k_assign_simt<T><<<grid, kThreads, 0, s>>>(static_cast<const T *>(K), p.n_tokens, p.np_cap, p.n_cap,
                                               idx.n_parents, idx.m2, ws.norm2,
                                               static_cast<const T *>(idx.parent_keys), idx.parent_e,
                                               idx.token_parent);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_assign_simt(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                               int32_t *err, cudaStream_t s) {
    (void)err;
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, K, idx, ws, s);
    return launch_t<float>(p, K, idx, ws, s);
}

}  // namespace ice
