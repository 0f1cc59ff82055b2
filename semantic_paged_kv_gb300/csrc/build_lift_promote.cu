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
// Two kernels per layer:
//   k_lift_count    grid (tiles, units): |k_j|^2 for every token (double-float
//                   accumulation, exact enough that sqrt(M^2 - |k|^2) rounds
//                   correctly to fp32), M^2 = max via a 64-bit atomicMax on
//                   the non-negative double's bits, and per tile the number
//                   of promoted tokens plus the unit's smallest draw.
//   k_promote_write grid (tiles, units): order-preserving compaction of the
//                   promoted tokens into the parent table (block scan plus
//                   the counts of the tiles before), parent keys, lifted
//                   extra coordinate of each parent, token_parent seeds.
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPerThread = kLiftTile / kThreads;  // 8

template <typename T>
__global__ void __launch_bounds__(kThreads) k_lift_count(const T *__restrict__ K, int N, int n_kv_heads,
                                                         uint64_t thresh, uint64_t key, double *__restrict__ m2,
                                                         double *__restrict__ norm2, int32_t *__restrict__ pcount,
                                                         unsigned long long *__restrict__ minpack, int n_tiles) {
    const int u = blockIdx.y, tile = blockIdx.x;
    const int seq = u / n_kv_heads, head = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long t0 = (long long)tile * kLiftTile;
    const T *Ku = K + (size_t)u * N * kHeadDim;

    // ---- squared norms: LPT lanes per token, one 16-byte vector per lane
    constexpr int LPT = row_vecs<T>();  // 16 (bf16) or 32 (fp32)
    constexpr int TPS = 32 / LPT;       // tokens per warp step
    double wmax = 0.0;
    const int per_warp = kLiftTile / (kThreads / 32);
    for (int s = 0; s < per_warp; s += TPS) {
        const long long j = t0 + (long long)warp * per_warp + s + lane / LPT;
        float hi = 0.f, lo = 0.f;
        if (j < N) {
            const uint4 v = reinterpret_cast<const uint4 *>(Ku + (size_t)j * kHeadDim)[lane % LPT];
            float f[Elem<T>::kPerVec];
            Elem<T>::unpack(v, f);
#pragma unroll
            for (int i = 0; i < Elem<T>::kPerVec; ++i) {
                const float t = f[i] * f[i];
                const float te = fmaf(f[i], f[i], -t);  // 0 for bf16 inputs
                float sum, err;
                two_sum(hi, t, sum, err);
                hi = sum;
                lo += err + te;
            }
        }
#pragma unroll
        for (int off = LPT / 2; off >= 1; off >>= 1) {
            const float ohi = __shfl_xor_sync(0xffffffffu, hi, off);
            const float olo = __shfl_xor_sync(0xffffffffu, lo, off);
            float sum, err;
            two_sum(hi, ohi, sum, err);
            hi = sum;
            lo += olo + err;
        }
        if (j < N && lane % LPT == 0) {
            const double n = (double)hi + (double)lo;
            norm2[(size_t)u * N + j] = n;
            wmax = fmax(wmax, n);
        }
    }
    // ---- promotion draws: kTokPerThread consecutive tokens per thread
    int cnt = 0;
    unsigned long long best = ~0ull;
    for (int i = 0; i < kTokPerThread; ++i) {
        const long long j = t0 + threadIdx.x * kTokPerThread + i;
        if (j >= N) break;
        const uint32_t d = promote_draw(key, seq, head, (uint32_t)j, 1u);
        cnt += ((uint64_t)d < thresh);
        const unsigned long long pk = ((unsigned long long)d << 32) | (unsigned long long)j;
        best = pk < best ? pk : best;
    }
    // ---- block reductions
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        wmax = fmax(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o < best ? o : best;
    }
    __shared__ double s_max[kThreads / 32];
    __shared__ int s_cnt[kThreads / 32];
    __shared__ unsigned long long s_best[kThreads / 32];
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
        for (int w = 0; w < kThreads / 32; ++w) {
            mx = fmax(mx, s_max[w]);
            c += s_cnt[w];
            b = s_best[w] < b ? s_best[w] : b;
        }
        // non-negative doubles order like their bit patterns
        atomicMax(reinterpret_cast<unsigned long long *>(m2 + u), (unsigned long long)__double_as_longlong(mx));
        atomicMin(minpack + u, b);
        pcount[(size_t)u * n_tiles + tile] = c;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_promote_write(
    const T *__restrict__ K, int N, int n_kv_heads, uint64_t thresh, uint64_t key, int np_cap, int n_cap,
    const double *__restrict__ m2, const double *__restrict__ norm2, const int32_t *__restrict__ pcount,
    const unsigned long long *__restrict__ minpack, int n_tiles, int32_t *__restrict__ n_parents,
    int32_t *__restrict__ n_indexed, int32_t *__restrict__ parent_tok, T *__restrict__ parent_keys,
    float *__restrict__ parent_e, float *__restrict__ parent_corr, int32_t *__restrict__ token_parent,
    int32_t *__restrict__ err) {
    const int u = blockIdx.y, tile = blockIdx.x;
    const int seq = u / n_kv_heads, head = u % n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long t0 = (long long)tile * kLiftTile;

    __shared__ int s_base, s_total;
    __shared__ int s_warp[kThreads / 32];
    __shared__ int s_list_tok[kLiftTile];
    __shared__ int s_list_m[kLiftTile];
    __shared__ int s_nlist;
    if (warp == 0) {
        int before = 0, all = 0;
        for (int t = lane; t < n_tiles; t += 32) {
            const int c = pcount[(size_t)u * n_tiles + t];
            all += c;
            before += (t < tile) ? c : 0;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, off);
            all += __shfl_xor_sync(0xffffffffu, all, off);
        }
        if (lane == 0) {
            s_base = before;
            s_total = all;
            s_nlist = 0;
        }
    }
    __syncthreads();
    // No token promoted: the smallest draw (lowest token on ties) is.
    const bool fallback = (s_total == 0 && N > 0);
    const long long jmin = fallback ? (long long)(minpack[u] & 0xFFFFFFFFull) : -1;
    const int total = fallback ? 1 : s_total;
    const int base = fallback ? 0 : s_base;
    if (tile == 0 && threadIdx.x == 0) {
        if (total > np_cap) set_err(err, ICE_ERR_CAPACITY);
        n_parents[u] = total < np_cap ? total : np_cap;
        n_indexed[u] = N;
    }

    // flags of this thread's tokens, in token order
    unsigned flags = 0;
    for (int i = 0; i < kTokPerThread; ++i) {
        const long long j = t0 + threadIdx.x * kTokPerThread + i;
        if (j >= N) break;
        const bool f = fallback ? (j == jmin)
                                : ((uint64_t)promote_draw(key, seq, head, (uint32_t)j, 1u) < thresh);
        flags |= (unsigned)f << i;
    }
    const int c = __popc(flags);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int woff = 0;
    for (int w = 0; w < warp; ++w) woff += s_warp[w];
    int m = base + woff + incl - c;

    const double M2 = m2[u];
    const size_t ubase_n = (size_t)u * n_cap;
    const size_t ubase_p = (size_t)u * np_cap;
    for (int i = 0; i < kTokPerThread; ++i) {
        const long long j = t0 + threadIdx.x * kTokPerThread + i;
        if (j >= N) break;
        int32_t tp = -1;
        if ((flags >> i) & 1u) {
            if (m < np_cap) {
                tp = m;
                parent_tok[ubase_p + m] = (int32_t)j;
                const double r = M2 - norm2[(size_t)u * N + j];
                parent_e[ubase_p + m] = (float)sqrt(r > 0.0 ? r : 0.0);
                parent_corr[ubase_p + m] = 0.f;
                const int slot = atomicAdd(&s_nlist, 1);
                s_list_tok[slot] = (int)j;
                s_list_m[slot] = m;
            }
            ++m;
        }
        token_parent[ubase_n + j] = tp;
    }
    __syncthreads();
    // copy the promoted keys into the parent table, one 16-byte vector per thread
    constexpr int RV = row_vecs<T>();
    const int nl = s_nlist;
    const uint4 *src = reinterpret_cast<const uint4 *>(K + (size_t)u * N * kHeadDim);
    uint4 *dst = reinterpret_cast<uint4 *>(parent_keys + ubase_p * kHeadDim);
    for (int x = threadIdx.x; x < nl * RV; x += kThreads) {
        const int r = x / RV, v = x % RV;
        dst[(size_t)s_list_m[r] * RV + v] = src[(size_t)s_list_tok[r] * RV + v];
    }
}

template <typename T>
cudaError_t launch_lift_promote_t(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                                  int32_t *err, cudaStream_t s) {
    const int U = units_of(p);
    const int N = p.n_tokens;
    const int tiles = ceil_div(N, kLiftTile);
    cudaMemsetAsync(idx.m2, 0, sizeof(double) * U, s);
    cudaMemsetAsync(ws.minpack, 0xFF, sizeof(unsigned long long) * U, s);
    const uint64_t key = promote_key(p.seed, p.layer);
    dim3 grid(tiles, U);
    k_lift_count<T><<<grid, kThreads, 0, s>>>(static_cast<const T *>(K), N, p.n_kv_heads, p.promote_thresh, key,
                                              idx.m2, ws.norm2, ws.pcount, ws.minpack, tiles);
    k_promote_write<T><<<grid, kThreads, 0, s>>>(
        static_cast<const T *>(K), N, p.n_kv_heads, p.promote_thresh, key, p.np_cap, p.n_cap, idx.m2, ws.norm2,
        ws.pcount, ws.minpack, tiles, idx.n_parents, idx.n_indexed, idx.parent_tok,
        static_cast<T *>(idx.parent_keys), idx.parent_e, idx.parent_corr, idx.token_parent, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lift_promote(const ice_params &p, const void *K, const ice_index &idx, const BuildWs &ws,
                                int32_t *err, cudaStream_t s) {
    if (p.dtype == ICE_BF16) return launch_lift_promote_t<__nv_bfloat16>(p, K, idx, ws, err, s);
    return launch_lift_promote_t<float>(p, K, idx, ws, err, s);
}

}  // namespace ice
