// Index build, steps a1 (key lift) and a2 (random promotion to level 1).
//
// IceCache popular-science article (aitangshan.cn/news/751385), section 三:
// keys are transformed so that inner-product similarity becomes Euclidean
// distance, and a random subset of tokens is promoted one level up to form
// the pyramid; section 六: the transform normalises the key and adds one
// coordinate.  papernotes.org "IceCache: Memory-Efficient KV-cache
// Management for Long-Sequence LLMs", 关键设计 2: points are promoted at
// random and each lower point picks its nearest parent one level up.
//
// Two kernels per layer, both over 256-token tiles (one token per thread):
//   k_lift_count    |k_j|^2 for every token with double-float accumulation
//                   (exact enough that sqrt(M^2 - |k|^2) rounds correctly to
//                   fp32): four lanes per token, each loading its 64-byte
//                   quarter of the row for all 8 of its tokens before any
//                   arithmetic (many loads in flight).  Per tile: the largest
//                   |k|^2, the number of promoted tokens and the smallest
//                   (draw, token), written to the workspace (no atomics, no
//                   memset).
//   k_promote_write reduces the unit's tile values (M^2, promoted count,
//                   smallest draw), then order-preserving compaction of the
//                   promoted tokens into the parent table (block scan plus
//                   the counts of the tiles before), parent keys, lifted
//                   extra coordinate of each parent, token_parent seeds.
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = kLiftTile;  // one token per thread
constexpr int kWarps = kThreads / 32;

// Loads of the 32 rows [wt0, wt0 + 32) of a warp (rows >= N read as zero):
// in step s, lane 4t + q holds the 16-byte vectors q, q + 4, ... of row
// wt0 + 8s + t.
template <typename T>
__device__ __forceinline__ void load_rows32(const T *__restrict__ Ku, int N, long long wt0, int lane,
                                            uint4 (&buf)[4][row_vecs<T>() / 4]) {
    constexpr int VPL = row_vecs<T>() / 4;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const long long j = wt0 + s * 8 + lane / 4;
        const uint4 *row = reinterpret_cast<const uint4 *>(Ku + (size_t)(j < N ? j : 0) * kHeadDim);
#pragma unroll
        for (int v = 0; v < VPL; ++v)
            buf[s][v] = (j < N) ? ld_stream16(row + (lane % 4) + 4 * v) : make_uint4(0, 0, 0, 0);
    }
}

// |k|^2 of row wt0 + lane as an unevaluated double-float sum (hi + lo) from
// load_rows32's registers.  bf16: every square is exact in fp32, and the even
// and odd elements run as two double-float sums on packed pairs joined at the
// end; fp32: each square's rounding error is carried too.
template <typename T>
__device__ __forceinline__ void norms32(const uint4 (&buf)[4][row_vecs<T>() / 4], int lane, float &mine_hi,
                                        float &mine_lo) {
    constexpr int VPL = row_vecs<T>() / 4;
    mine_hi = 0.f;
    mine_lo = 0.f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        float hi = 0.f, lo = 0.f;
        if constexpr (sizeof(T) == 2) {
            unsigned long long hi2 = 0ull, lo2 = 0ull;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const uint32_t w[4] = {buf[s][v].x, buf[s][v].y, buf[s][v].z, buf[s][v].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const unsigned long long f2 = bf2_pair(w[i]);
                    unsigned long long s2, e2;
                    two_sum2(hi2, mul2(f2, f2), s2, e2);
                    hi2 = s2;
                    lo2 = add2(lo2, e2);
                }
            }
            const float2 h = upk2(hi2), l = upk2(lo2);
            float err;
            two_sum(h.x, h.y, hi, err);
            lo = (l.x + l.y) + err;
        } else {
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                float f[Elem<T>::kPerVec];
                Elem<T>::unpack(buf[s][v], f);
#pragma unroll
                for (int i = 0; i < Elem<T>::kPerVec; ++i) {
                    const float t = f[i] * f[i];
                    const float te = fmaf(f[i], f[i], -t);  // the square's rounding error
                    float sum, err;
                    two_sum(hi, t, sum, err);
                    hi = sum;
                    lo += err + te;
                }
            }
        }
#pragma unroll
        for (int off = 2; off >= 1; off >>= 1) {
            const float ohi = __shfl_xor_sync(0xffffffffu, hi, off);
            const float olo = __shfl_xor_sync(0xffffffffu, lo, off);
            float sum, err;
            two_sum(hi, ohi, sum, err);
            hi = sum;
            lo += olo + err;
        }
        // token (s*8 + lane/4) of the warp: hand it to lane s*8 + lane/4
        const float ghi = __shfl_sync(0xffffffffu, hi, ((lane - s * 8) & 7) * 4);
        const float glo = __shfl_sync(0xffffffffu, lo, ((lane - s * 8) & 7) * 4);
        if (lane / 8 == s) {
            mine_hi = ghi;
            mine_lo = glo;
        }
    }
}

// e = e1 + e2 + e3 in bf16 parts (each remainder exact in fp32): the extra K
// columns of the tensor-core contraction, [e1, e1, e2, e1, e2, e3] for a
// token and [e1, e2, e1, e3, e2, e1] for a parent, whose dot product holds
// every term e_a f_b with a + b <= 4.
__device__ __forceinline__ void write_lifted(float e, uint4 *tok_row, uint4 *par_row) {
    const __nv_bfloat16 e1 = __float2bfloat16_rn(e);
    const float r1 = e - __bfloat162float(e1);
    const __nv_bfloat16 e2 = __float2bfloat16_rn(r1);
    const __nv_bfloat16 e3 = __float2bfloat16_rn(r1 - __bfloat162float(e2));
    const __nv_bfloat16 z = __float2bfloat16(0.f);
    if (tok_row) {
        const __nv_bfloat16 row[16] = {e1, e1, e2, e1, e2, e3, z, z, z, z, z, z, z, z, z, z};
        const uint4 *w = reinterpret_cast<const uint4 *>(row);
        tok_row[0] = w[0];
        tok_row[1] = w[1];
    }
    if (par_row) {
        const __nv_bfloat16 prow[16] = {e1, e2, e1, e3, e2, e1, z, z, z, z, z, z, z, z, z, z};
        const uint4 *w = reinterpret_cast<const uint4 *>(prow);
        par_row[0] = w[0];
        par_row[1] = w[1];
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 3) k_lift_count(const T *__restrict__ K, int N, int lo, int hi,
                                                         int n_kv_heads, uint64_t thresh, uint64_t key,
                                                         double *__restrict__ norm2, int32_t *__restrict__ pcount,
                                                         double *__restrict__ tile_max,
                                                         unsigned long long *__restrict__ tile_min, int n_tiles) {
    dep_wait();  // the previous kernel of the stream is complete (launched as its dependent)
    const int u = blockIdx.y, tile = blockIdx.x;
    const int seq = u / n_kv_heads, head = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long t0 = (long long)tile * kLiftTile;
    const T *Ku = K + (size_t)u * N * kHeadDim;

    // ---- squared norms: the warp's 32 tokens, 4 lanes per token, 8 tokens per step
    const long long wt0 = t0 + warp * 32;
    uint4 buf[4][row_vecs<T>() / 4];
    load_rows32<T>(Ku, N, wt0, lane, buf);
    float mine_hi, mine_lo;  // lane s*8 + t keeps token s*8 + t's norm
    norms32<T>(buf, lane, mine_hi, mine_lo);
    const long long j = wt0 + lane;
    const bool mid = j >= lo && j < hi;  // indexed tokens (not sink or window)
    double wmax = 0.0;  // one conversion per token: the fp64 units are few
    if (j < N) {
        const double n = (double)mine_hi + (double)mine_lo;
        norm2[(size_t)u * N + j] = n;
        wmax = mid ? n : 0.0;
    }
    // ---- promotion draw of this thread's token
    int cnt = 0;
    unsigned long long best = ~0ull;
    if (mid) {
        const uint32_t d = promote_draw(key, seq, head, (uint32_t)j, 1u);
        cnt = ((uint64_t)d < thresh);
        best = ((unsigned long long)d << 32) | (unsigned long long)j;
    }
    // ---- block reductions
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        wmax = fmax(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o < best ? o : best;
    }
    __shared__ double s_max[kWarps];
    __shared__ int s_cnt[kWarps];
    __shared__ unsigned long long s_best[kWarps];
    if (lane == 0) {
        s_max[warp] = wmax;
        s_cnt[warp] = cnt;
        s_best[warp] = best;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double mx = 0.0;
        int c = 0;
        unsigned long long b = ~0ull;
        for (int w = 0; w < kWarps; ++w) {
            mx = fmax(mx, s_max[w]);
            c += s_cnt[w];
            b = s_best[w] < b ? s_best[w] : b;
        }
        tile_max[(size_t)u * n_tiles + tile] = mx;
        tile_min[(size_t)u * n_tiles + tile] = b;
        pcount[(size_t)u * n_tiles + tile] = c;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_promote_write(
    const T *__restrict__ K, int N, int lo, int hi, int n_kv_heads, uint64_t thresh, uint64_t key, int np_cap,
    int n_cap,
    double *__restrict__ m2, const double *__restrict__ norm2, const int32_t *__restrict__ pcount,
    const double *__restrict__ tile_max, const unsigned long long *__restrict__ tile_min, int n_tiles,
    int32_t *__restrict__ n_parents,
    int32_t *__restrict__ n_indexed, int32_t *__restrict__ parent_tok, T *__restrict__ parent_keys,
    float *__restrict__ parent_e, float *__restrict__ parent_corr, int32_t *__restrict__ token_parent,
    uint4 *__restrict__ a_extra, uint4 *__restrict__ b_extra, int32_t *__restrict__ err) {
    dep_wait();  // the previous kernel of the stream is complete (launched as its dependent)
    const int u = blockIdx.y, tile = blockIdx.x;
    const int seq = u / n_kv_heads, head = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long t0 = (long long)tile * kLiftTile;

    __shared__ int s_part[kWarps][2];
    __shared__ double s_pmax[kWarps];
    __shared__ unsigned long long s_pmin[kWarps];
    __shared__ int s_warp[kWarps];
    __shared__ int s_list_tok[kLiftTile];
    __shared__ int s_list_m[kLiftTile];
    // this thread's token: its squared norm and promotion draw do not depend
    // on the unit's totals, so their loads overlap the reduction below
    const long long j = t0 + threadIdx.x;
    const double n2 = j < N ? norm2[(size_t)u * N + j] : 0.0;
    const bool mid = j >= lo && j < hi;  // indexed tokens (not sink or window)
    const bool drawn = mid && (uint64_t)promote_draw(key, seq, head, (uint32_t)j, 1u) < thresh;
    // the unit's tile values: counts before this tile and in all, M^2, smallest draw
    int before = 0, all = 0;
    double mx = 0.0;
    unsigned long long mn = ~0ull;
    for (int t = threadIdx.x; t < n_tiles; t += kThreads) {
        const size_t o = (size_t)u * n_tiles + t;
        const int c = pcount[o];
        all += c;
        before += (t < tile) ? c : 0;
        mx = fmax(mx, tile_max[o]);
        mn = tile_min[o] < mn ? tile_min[o] : mn;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, off);
        all += __shfl_xor_sync(0xffffffffu, all, off);
        mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, mn, off);
        mn = o < mn ? o : mn;
    }
    if (lane == 0) {
        s_part[warp][0] = before;
        s_part[warp][1] = all;
        s_pmax[warp] = mx;
        s_pmin[warp] = mn;
    }
    __syncthreads();
    int s_base = 0, s_total = 0;
    double M2 = 0.0;
    unsigned long long minpack = ~0ull;
    for (int w = 0; w < kWarps; ++w) {
        s_base += s_part[w][0];
        s_total += s_part[w][1];
        M2 = fmax(M2, s_pmax[w]);
        minpack = s_pmin[w] < minpack ? s_pmin[w] : minpack;
    }
    // No token promoted: the smallest draw (lowest token on ties) is.
    const bool fallback = (s_total == 0 && hi > lo);
    const long long jmin = fallback ? (long long)(minpack & 0xFFFFFFFFull) : -1;
    const int total = fallback ? 1 : s_total;
    const int base = fallback ? 0 : s_base;
    if (tile == 0 && threadIdx.x == 0) {
        if (total > np_cap) set_err(err, ICE_ERR_CAPACITY);
        n_parents[u] = total < np_cap ? total : np_cap;
        n_indexed[u] = N;
        m2[u] = M2;
    }

    const bool f = mid && (fallback ? (j == jmin) : drawn);
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    int woff = 0;
    for (int w = 0; w < warp; ++w) woff += s_warp[w];
    const int local = woff + __popc(bal & lanemask_lt());
    const int m = base + local;
    if (j < N) {
        int32_t tp = mid ? -1 : -2;  // -2: a sink or window token, packed by position
        // M^2 - |k|^2 is exact in fp64 to ~2^-52 M^2; rounded to fp32, its
        // square root is within 1.5 ulp of the exact e (fp32 sqrt: the fp64
        // units are few on this part)
        const double r = M2 - n2;
        const float e = sqrtf(r > 0.0 ? (float)r : 0.f);
        const bool par = f && m < np_cap;
        const size_t up = (size_t)u * np_cap;
        write_lifted(e, a_extra ? a_extra + ((size_t)u * N + j) * 2 : nullptr,
                     (par && b_extra) ? b_extra + (up + m) * 2 : nullptr);
        if (par) {
            tp = m;
            parent_tok[up + m] = (int32_t)j;
            parent_e[up + m] = e;
            parent_corr[up + m] = 0.f;
        }
        token_parent[(size_t)u * n_cap + j] = tp;
        if (f) {
            s_list_tok[local] = (int)j;
            s_list_m[local] = m;
        }
    }
    __syncthreads();
    int nl = 0;
    for (int w = 0; w < kWarps; ++w) nl += s_warp[w];
    // copy the promoted keys into the parent table, one 16-byte vector per thread
    constexpr int RV = row_vecs<T>();
    const uint4 *src = reinterpret_cast<const uint4 *>(K + (size_t)u * N * kHeadDim);
    uint4 *dst = reinterpret_cast<uint4 *>(parent_keys + (size_t)u * np_cap * kHeadDim);
    for (int x = threadIdx.x; x < nl * RV; x += kThreads) {
        const int r = x / RV, v = x % RV;
        if (s_list_m[r] < np_cap) dst[(size_t)s_list_m[r] * RV + v] = src[(size_t)s_list_tok[r] * RV + v];
    }
}

template <typename T>
cudaError_t launch_lift_promote_t(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                                  int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int N = p.n_tokens;
    const int tiles = ceil_div(N, kLiftTile);
    const uint64_t key = promote_key(p.seed, p.layer);
    const PosSplit ps = pos_split(p);
    dim3 grid(tiles, U);
    {
        const cudaError_t e_ = launch_dependent(k_lift_count<T>, dim3(grid), dim3(kThreads), 0, s,
                                                static_cast<const T *>(K), N, ps.lo, ps.hi, p.n_kv_heads,
                                                p.promote_thresh, key,
                                                ws.norm2, ws.pcount, ws.tile_max, ws.tile_min, tiles);
        if (e_ != cudaSuccess) return e_;
    }
    {
        const cudaError_t e_ = launch_dependent(k_promote_write<T>, dim3(grid), dim3(kThreads), 0, s,
                                                static_cast<const T *>(K), N, ps.lo, ps.hi, p.n_kv_heads,
                                                p.promote_thresh, key,
                                                p.np_cap, p.n_cap, idx.m2, ws.norm2, ws.pcount, ws.tile_max,
                                                ws.tile_min, tiles, idx.n_parents, idx.n_indexed, idx.parent_tok,
                                                static_cast<T *>(idx.parent_keys), idx.parent_e, idx.parent_corr,
                                                idx.token_parent, p.dtype == ICE_BF16 ? ws.a_extra : nullptr,
                                                p.dtype == ICE_BF16 ? ws.b_extra : nullptr, err);
        if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_lift_norms_t(const ice_params &p, const void *K, const BuildWs &ws, cudaStream_t s) {
    const int tiles = ceil_div(p.n_tokens, kLiftTile);
    const PosSplit ps = pos_split(p);
    const cudaError_t e = launch_dependent(k_lift_count<T>, dim3(tiles, units_of(p)), dim3(kThreads), 0, s,
                                           static_cast<const T *>(K), p.n_tokens, ps.lo, ps.hi, p.n_kv_heads,
                                           p.promote_thresh,
                                           promote_key(p.seed, p.layer), ws.norm2, ws.pcount, ws.tile_max,
                                           ws.tile_min, tiles);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_lift_norms(const ice_params &p, const void *K, const BuildWs &ws, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_lift_norms_t<__nv_bfloat16>(p, K, ws, s);
    return launch_lift_norms_t<float>(p, K, ws, s);
}

cudaError_t launch_lift_promote(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                                int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_lift_promote_t<__nv_bfloat16>(p, K, idx, ws, err, s);
    return launch_lift_promote_t<float>(p, K, idx, ws, err, s);
}

}  // namespace ice
