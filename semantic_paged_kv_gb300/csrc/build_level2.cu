// Index build with three levels: the level above the parents.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 2: points are promoted at random to higher
// levels and every point of a level takes its nearest point one level up as
// parent; a query finds the k nearest points of the top level and continues
// among their children.  IceCache popular-science article
// (aitangshan.cn/news/751385), section 三: the promotion pyramid.
//
// Level 2 is built from the parents (level 1) after their own build:
//   k_l2_promote   one CTA per unit: parent m is promoted iff the draw of its
//                  token at level 2 is below the threshold (the smallest draw
//                  if none is); ordered compaction into node2 (level-2 node
//                  i -> parent m), parent2 = i for those parents, -1 others
//   k_l2_gather +  bf16: the nearest level-2 node in the lifted space on the
//   k_assign_tc    tensor cores, the parent table against the level-2 nodes
//                  gathered dense (the same contraction and argmax as the
//                  token -> parent step, the split lifted coordinates as
//                  extra K columns)
//   k_l2_assign    fp32 (CUDA cores): 32 parents per CTA, argmax_i
//                  (p_m . p_i + e_m e_i), exact ties to the lowest i (parent
//                  keys staged as fp32 in shared memory, the level-2 nodes
//                  streamed 32 at a time)
//   k_l2_children  one CTA per unit: the parents grouped by parent2,
//                  ascending m inside a group (counting sort: shared-memory
//                  histogram, scan, one warp placing 32 parents at a time)
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kPT = 1024;  // threads of the per-unit kernels
constexpr int kAT = 256;   // threads of the assignment kernel
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kRowsPerWarp * (kAT / 32);  // parents per CTA
constexpr int kChunk = 32;                        // level-2 nodes per shared-memory chunk
constexpr int kPad = kHeadDim + 1;

__global__ void __launch_bounds__(kPT) k_l2_promote(int n_kv_heads, int np_cap, uint64_t thresh, uint64_t key,
                                                    const int32_t *__restrict__ n_parents,
                                                    const int32_t *__restrict__ parent_tok,
                                                    int32_t *__restrict__ n_nodes2, int32_t *__restrict__ node2,
                                                    int32_t *__restrict__ parent2) {
    dep_wait();  // the parents are complete
    const int u = blockIdx.x;
    const int seq = u / n_kv_heads, head = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int s_warp[kPT / 32];
    __shared__ unsigned long long s_min[kPT / 32];
    __shared__ int s_base;
    const int Np = min(n_parents[u], np_cap);
    const size_t up = (size_t)u * np_cap;
    if (threadIdx.x == 0) s_base = 0;
    unsigned long long mn = ~0ull;  // smallest (draw, m) of this thread's parents
    for (int m0 = 0; m0 < Np; m0 += kPT) {
        const int m = m0 + threadIdx.x;
        bool f = false;
        if (m < Np) {
            const uint32_t d = promote_draw(key, seq, head, (uint32_t)parent_tok[up + m], 2u);
            f = (uint64_t)d < thresh;
            const unsigned long long k = ((unsigned long long)d << 32) | (unsigned)m;
            mn = k < mn ? k : mn;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (lane == 0) s_warp[warp] = __popc(bal);
        __syncthreads();
        int off = s_base;
        for (int w = 0; w < warp; ++w) off += s_warp[w];
        const int i = off + __popc(bal & lanemask_lt());
        if (m < Np) {
            parent2[up + m] = f ? i : -1;
            if (f) node2[up + i] = m;
        }
        __syncthreads();
        if (threadIdx.x == 0)
            for (int w = 0; w < kPT / 32; ++w) s_base += s_warp[w];
        __syncthreads();
    }
    // no parent promoted: the one of smallest draw (lowest m on ties) is
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, mn, o);
        mn = x < mn ? x : mn;
    }
    if (lane == 0) s_min[warp] = mn;
    __syncthreads();
    if (threadIdx.x == 0) {
        int total = s_base;
        if (total == 0 && Np > 0) {
            unsigned long long b = ~0ull;
            for (int w = 0; w < kPT / 32; ++w) b = s_min[w] < b ? s_min[w] : b;
            const int m = (int)(b & 0xFFFFFFFFull);
            node2[up] = m;
            parent2[up + m] = 0;
            total = 1;
        }
        n_nodes2[u] = total;
    }
}

template <typename T>
__global__ void __launch_bounds__(kAT) k_l2_assign(int np_cap, const int32_t *__restrict__ n_parents,
                                                   const int32_t *__restrict__ n_nodes2,
                                                   const int32_t *__restrict__ node2,
                                                   const T *__restrict__ parent_keys,
                                                   const float *__restrict__ parent_e,
                                                   int32_t *__restrict__ parent2) {
    dep_wait();  // the level-2 nodes are complete
    __shared__ float s_k[kRows][kHeadDim];
    __shared__ float s_p[kChunk][kPad];
    __shared__ float s_pe[kChunk];
    const int u = blockIdx.y;
    const int r0 = blockIdx.x * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    if (r0 >= Np) return;
    const int n2 = min(n_nodes2[u], np_cap);
    const size_t up = (size_t)u * np_cap;
    const T *Pu = parent_keys + up * kHeadDim;
    for (int x = threadIdx.x; x < kRows * kHeadDim; x += kAT) {
        const int r = x / kHeadDim, i = x % kHeadDim;
        s_k[r][i] = r0 + r < Np ? Elem<T>::load(Pu + (size_t)(r0 + r) * kHeadDim + i) : 0.f;
    }
    float er[kRowsPerWarp], best[kRowsPerWarp];
    int bidx[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int m = r0 + warp * kRowsPerWarp + r;
        er[r] = m < Np ? parent_e[up + m] : 0.f;
        best[r] = -INFINITY;
        bidx[r] = 0x7fffffff;
    }
    for (int c0 = 0; c0 < n2; c0 += kChunk) {
        __syncthreads();
        for (int x = threadIdx.x; x < kChunk * kHeadDim; x += kAT) {
            const int c = x / kHeadDim, i = x % kHeadDim;
            s_p[c][i] = c0 + c < n2 ? Elem<T>::load(Pu + (size_t)node2[up + c0 + c] * kHeadDim + i) : 0.f;
        }
        if (threadIdx.x < kChunk) s_pe[threadIdx.x] = c0 + threadIdx.x < n2 ? parent_e[up + node2[up + c0 + threadIdx.x]] : 0.f;
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
        if (c0 + lane < n2) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const float sc = fmaf(er[r], s_pe[lane], acc[r]);
                if (sc > best[r]) {  // a lane's nodes arrive in ascending order
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
        const int m = r0 + warp * kRowsPerWarp + r;
        if (lane == 0 && m < Np && n2 > 0 && parent2[up + m] < 0) parent2[up + m] = bi;  // level-2 nodes keep themselves
    }
}

__global__ void __launch_bounds__(kPT) k_l2_children(int np_cap, const int32_t *__restrict__ n_parents,
                                                     const int32_t *__restrict__ n_nodes2,
                                                     const int32_t *__restrict__ parent2,
                                                     int32_t *__restrict__ child_start,
                                                     int32_t *__restrict__ children) {
    dep_wait();  // the level-2 parents are complete
    extern __shared__ int s_off[];  // [np_cap + 1]
    const int u = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Np = min(n_parents[u], np_cap);
    const int n2 = min(n_nodes2[u], np_cap);
    const size_t up = (size_t)u * np_cap;
    for (int i = threadIdx.x; i < n2; i += kPT) s_off[i] = 0;
    __syncthreads();
    for (int m = threadIdx.x; m < Np; m += kPT) {
        const int p = parent2[up + m];
        if (p >= 0 && p < n2) atomicAdd(&s_off[p], 1);
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of the group sizes, 32 groups per step
        int carry = 0;
        for (int i0 = 0; i0 < n2; i0 += 32) {
            const int i = i0 + lane;
            const int c = i < n2 ? s_off[i] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += x;
            }
            if (i < n2) {
                s_off[i] = carry + incl - c;
                child_start[(size_t)u * (np_cap + 1) + i] = carry + incl - c;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) child_start[(size_t)u * (np_cap + 1) + n2] = carry;
        __syncwarp();
        // stable placement: 32 parents at a time in ascending m
        for (int m0 = 0; m0 < Np; m0 += 32) {
            const int m = m0 + lane;
            const int p = m < Np ? parent2[up + m] : -1;
            const bool ok = p >= 0 && p < n2;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? p : -1 - lane);
            const int pos = ok ? s_off[p] + __popc(peers & lanemask_lt()) : 0;
            __syncwarp();
            if (ok) {
                children[up + pos] = m;
                if (lane == 31 - __clz(peers)) s_off[p] += __popc(peers);  // the highest peer advances the group
            }
            __syncwarp();
        }
    }
}

// The tensor-core operands of the level-2 contraction (bf16), one warp per
// row: per parent m its token's row-form split lifted coordinate, per
// level-2 node i its key row and column-form split lifted coordinate.
__global__ void __launch_bounds__(kAT) k_l2_gather(int N, int np_cap, const int32_t *__restrict__ n_parents,
                                                   const int32_t *__restrict__ n_nodes2,
                                                   const int32_t *__restrict__ parent_tok,
                                                   const int32_t *__restrict__ node2, const uint4 *__restrict__ keys,
                                                   const uint4 *__restrict__ a_extra, const uint4 *__restrict__ b_extra,
                                                   uint4 *__restrict__ a_extra2, uint4 *__restrict__ keys2,
                                                   uint4 *__restrict__ b_extra2) {
    dep_wait();  // the level-2 nodes are complete
    const int u = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * (kAT / 32) + (threadIdx.x >> 5);
    const size_t up = (size_t)u * np_cap;
    if (r < min(n_parents[u], np_cap) && lane < 2)
        a_extra2[(up + r) * 2 + lane] = a_extra[((size_t)u * N + parent_tok[up + r]) * 2 + lane];
    if (r < min(n_nodes2[u], np_cap)) {
        const int m = node2[up + r];
        if (lane < 16) keys2[(up + r) * 16 + lane] = keys[(up + m) * 16 + lane];  // 16 x 16 B = 128 bf16
        else if (lane < 18) b_extra2[(up + r) * 2 + lane - 16] = b_extra[(up + m) * 2 + lane - 16];
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const ice_index &idx, const BuildWs &ws, int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    cudaError_t e = launch_dependent(k_l2_promote, dim3(U), dim3(kPT), 0, s, p.n_kv_heads, p.np_cap, p.promote_thresh,
                                     promote_key(p.seed, p.layer), idx.n_parents, idx.parent_tok, idx.n_nodes2,
                                     idx.node2, idx.parent2);
    if (e != cudaSuccess) return e;
    bool done = false;
    if (sizeof(T) == 2 && ws.keys2) {  // bf16: the contraction on the tensor cores
        e = launch_dependent(k_l2_gather, dim3(ceil_div(p.np_cap, kAT / 32), U), dim3(kAT), 0, s, p.n_tokens, p.np_cap,
                             idx.n_parents, idx.n_nodes2, idx.parent_tok, idx.node2,
                             static_cast<const uint4 *>(idx.parent_keys), ws.a_extra, ws.b_extra, ws.a_extra2,
                             static_cast<uint4 *>(ws.keys2), ws.b_extra2);
        if (e != cudaSuccess) return e;
        e = launch_assign_level2_tc(p, idx, ws, err, s);
        if (e != cudaSuccess && e != cudaErrorNotSupported) return e;
        done = e == cudaSuccess;
    }
    if (!done) {
        e = launch_dependent(k_l2_assign<T>, dim3(ceil_div(p.np_cap, kRows), U), dim3(kAT), 0, s, p.np_cap,
                             idx.n_parents, idx.n_nodes2, idx.node2, static_cast<const T *>(idx.parent_keys),
                             idx.parent_e, idx.parent2);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(int) * ((size_t)p.np_cap + 1);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(k_l2_children, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    e = launch_dependent(k_l2_children, dim3(U), dim3(kPT), smem, s, p.np_cap, idx.n_parents, idx.n_nodes2,
                         idx.parent2, idx.child_start, idx.children);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_level2(const ice_params &p, const ice_index &idx, const BuildWs &ws, int32_t *err,
                          cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_t<__nv_bfloat16>(p, idx, ws, err, s);
    return launch_t<float>(p, idx, ws, err, s);
}

}  // namespace ice
