// Index build of one layer on the node structure of another layer.
//
// IceCache popular-science article (aitangshan.cn/news/751385), section 五:
// an inter-layer index reuse ("IceCache (reuse)") shortens the build; the
// article gives its effect on latency but not its mechanism.  The rule taken
// here: the layer keeps the other layer's promoted tokens, its token -> parent
// assignment and therefore its pages; what depends on this layer's keys and
// values is recomputed: M^2 (largest squared key norm, step a1), the parent
// keys that the selection scores against, their lifted coordinate, and the
// pool.  Steps a3 (nearest-parent contraction) and a4 (ranking into pages)
// are skipped.
//
//   k_lift_count (build_lift_promote.cu)  |k|^2 of every token, tile maxima
//   k_reuse_parents                       M^2 = max |k|^2; per parent m: the
//                                         token, its key row and
//                                         e_m = sqrt(M^2 - |p_m|^2)
//   k_copy_tables                         page and token tables, one launch
//                                         (arrays the two indexes share are
//                                         skipped)
//   k_pack_copy (build_pack.cu)           this layer's K / V rows into the pages
#include "common.cuh"
#include "internal.h"

namespace ice {
namespace {

constexpr int kThreads = 256;  // parents per CTA

template <typename T>
__global__ void __launch_bounds__(kThreads) k_reuse_parents(
    const T *__restrict__ K, int N, int np_cap, int n_tiles, const double *__restrict__ norm2,
    const double *__restrict__ tile_max, const int32_t *__restrict__ prev_n_parents,
    const int32_t *__restrict__ prev_n_indexed, const int32_t *__restrict__ prev_parent_tok,
    double *__restrict__ m2, int32_t *__restrict__ n_parents, int32_t *__restrict__ n_indexed,
    int32_t *__restrict__ parent_tok, T *__restrict__ parent_keys, float *__restrict__ parent_e,
    float *__restrict__ parent_corr, int32_t *__restrict__ err) {
    dep_wait();  // the norms are complete
    const int u = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ double s_max[kThreads / 32];
    __shared__ int s_tok[kThreads];
    // this layer's M^2
    double mx = 0.0;
    for (int t = threadIdx.x; t < n_tiles; t += kThreads) mx = fmax(mx, tile_max[(size_t)u * n_tiles + t]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) s_max[warp] = mx;
    const int Np = min(prev_n_parents[u], np_cap);
    const int m0 = blockIdx.x * kThreads, m = m0 + threadIdx.x;
    int tok = -1;
    if (m < Np) {
        tok = prev_parent_tok[(size_t)u * np_cap + m];
        if (tok < 0 || tok >= N) {  // not a token of this build
            set_err(err, ICE_ERR_INVALID_ARG);
            tok = -1;
        }
    }
    s_tok[threadIdx.x] = tok;
    __syncthreads();
    double M2 = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) M2 = fmax(M2, s_max[w]);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (prev_n_indexed[u] != N) set_err(err, ICE_ERR_INVALID_ARG);  // the other index covers other tokens
        n_parents[u] = Np;
        n_indexed[u] = N;
        m2[u] = M2;
    }
    if (m < Np) {
        const size_t pm = (size_t)u * np_cap + m;
        parent_tok[pm] = tok;
        // the same rounding as the full build: fp64 difference, fp32 root
        const double r = tok >= 0 ? M2 - norm2[(size_t)u * N + tok] : 0.0;
        parent_e[pm] = sqrtf(r > 0.0 ? (float)r : 0.f);
        parent_corr[pm] = 0.f;  // every parent is a token of this build: |p| <= M
    }
    // the parents' key rows, one 16-byte vector per thread and step
    constexpr int RV = row_vecs<T>();
    const int nl = max(0, min(kThreads, Np - m0));
    const uint4 *src = reinterpret_cast<const uint4 *>(K + (size_t)u * N * kHeadDim);
    uint4 *dst = reinterpret_cast<uint4 *>(parent_keys + ((size_t)u * np_cap + m0) * kHeadDim);
    for (int x = threadIdx.x; x < nl * RV; x += kThreads) {
        const int r = x / RV, v = x % RV;
        const int t = s_tok[r];
        dst[(size_t)r * RV + v] = t >= 0 ? src[(size_t)t * RV + v] : make_uint4(0, 0, 0, 0);
    }
}

template <typename T>
cudaError_t launch_t(const ice_params &p, const void *K, const ice_index &prev, const ice_index &idx,
                     const BuildWs &ws, int32_t *err, cudaStream_t s) {
    const int tiles = ceil_div(p.n_tokens, kLiftTile);
    return launch_dependent(k_reuse_parents<T>, dim3(ceil_div(p.np_cap, kThreads), units_of(p)), dim3(kThreads), 0,
                            s, static_cast<const T *>(K), p.n_tokens, p.np_cap, tiles, ws.norm2, ws.tile_max,
                            prev.n_parents, prev.n_indexed, prev.parent_tok, idx.m2, idx.n_parents, idx.n_indexed,
                            idx.parent_tok, static_cast<T *>(idx.parent_keys), idx.parent_e, idx.parent_corr, err);
}

// Up to 16 int32 arrays copied by one grid: CTA row y takes array y.
struct CopyList {
    int32_t *dst[16];
    const int32_t *src[16];
    long long n[16];
};

__global__ void __launch_bounds__(kThreads) k_copy_tables(const CopyList L) {
    dep_wait();  // the previous kernel of the stream is complete
    const int a = blockIdx.y;
    const long long n = L.n[a];
    for (long long x = (long long)blockIdx.x * kThreads + threadIdx.x; x < n; x += (long long)gridDim.x * kThreads)
        L.dst[a][x] = L.src[a][x];
}

}  // namespace

cudaError_t launch_build_reuse(const ice_params &p, const void *K, const void *V, const ice_index &prev,
                               const ice_index &idx, const BuildWs &ws, int32_t *err, cudaStream_t s) {
    cudaError_t e = launch_lift_norms(p, K, ws, s);
    if (e != cudaSuccess) return e;
    e = p.dtype == ICE_BF16 ? launch_t<__nv_bfloat16>(p, K, prev, idx, ws, err, s)
                            : launch_t<float>(p, K, prev, idx, ws, err, s);
    if (e != cudaSuccess) return e;
    const long long U = units_of(p);
    const long long np = U * p.np_cap, pc = U * p.page_cap, nc = U * p.n_cap;
    const struct {
        int32_t *d;
        const int32_t *s;
        long long n;
    } tables[] = {{idx.n_pages, prev.n_pages, U},
                  {idx.parent_first_page, prev.parent_first_page, np},
                  {idx.parent_last_page, prev.parent_last_page, np},
                  {idx.parent_n_pages, prev.parent_n_pages, np},
                  {idx.page_parent, prev.page_parent, pc},
                  {idx.page_len, prev.page_len, pc},
                  {idx.page_next, prev.page_next, pc},
                  {idx.page_tokens, prev.page_tokens, pc * kPage},
                  {idx.token_parent, prev.token_parent, nc},
                  {idx.token_page, prev.token_page, nc},
                  {idx.token_slot, prev.token_slot, nc},
                  // level 2 of a three-level index: kept with the rest of the node structure
                  {idx.n_nodes2, prev.n_nodes2, p.n_levels == 3 ? U : 0},
                  {idx.node2, prev.node2, p.n_levels == 3 ? np : 0},
                  {idx.parent2, prev.parent2, p.n_levels == 3 ? np : 0},
                  {idx.child_start, prev.child_start, p.n_levels == 3 ? np + U : 0},
                  {idx.children, prev.children, p.n_levels == 3 ? np : 0}};
    CopyList L{};
    int na = 0;
    long long most = 0;
    for (const auto &t : tables)
        if (t.d != t.s && t.n > 0) {
            L.dst[na] = t.d;
            L.src[na] = t.s;
            L.n[na++] = t.n;
            most = t.n > most ? t.n : most;
        }
    if (na > 0) {
        const int bx = (int)(ceil_div(most, kThreads) < 256 ? ceil_div(most, kThreads) : 256);
        if ((e = launch_dependent(k_copy_tables, dim3(bx, na), dim3(kThreads), 0, s, L)) != cudaSuccess) return e;
    }
    return launch_pack_copy(p, K, V, idx, s);
}

}  // namespace ice
