// One selected page of the masked sparse attention (decode step a10) on
// warp-level tensor-core MMAs, shared by the attention kernels.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 1: a_ij = s_ij exp(q_i.k_j/sqrt(d)) /
// sum_j' s_ij' exp(q_i.k_j'/sqrt(d)) over the selected pages; here s_ij is 1
// on the first `len` slots of the page and 0 on the rest.
//
// A page is a 16-key tile of K and one of V in shared memory, each two
// 64-column halves of 16 rows x 128 bytes written by 2-D TMA with a 128-byte
// swizzle.  With the g <= 16 query rows of a GQA group as M = 16:
//   S = Q K^T   mma.sync m16n8k16 (bf16 in, fp32 accumulate), A = q in
//               registers, B = K rows by ldmatrix: 2 key tiles x 8 dim steps;
//   online softmax on the accumulator fragments (a quad of lanes holds a
//               row's 16 keys), keys past `len` masked;
//   O += P V    P as the A fragment from S's accumulators, split into bf16
//               hi + lo parts (two MMAs, ~2^-16 relative error instead of
//               bf16's 2^-9), B = V rows by ldmatrix.trans: 16 dim tiles.
// HR = 2 when the group has more than 8 query heads (rows 8..15 in use).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_common.cuh"

namespace ice {
namespace mma {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D += A B, m16n8k16, bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16 pair (round to nearest) and the pair of remainders, as packed words.
__device__ __forceinline__ void split_pair(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}
// Shared-memory address of 16-byte chunk `cc` (0..15 across the two
// 64-column halves, each half_bytes long) of row `row` of a tile written by
// TMA with a 128-byte swizzle (1024-byte aligned tile).
__device__ __forceinline__ uint32_t sw_addr(uint32_t tile, int row, int cc, uint32_t half_bytes) {
    return tile + (uint32_t)((cc >> 3) * half_bytes + row * 128 + (((cc & 7) ^ (row & 7)) << 4));
}

constexpr uint32_t kPageHalf = 16 * 128;  // 16 rows x 64 bf16 columns: one swizzled box
constexpr uint32_t kPageTile = 2 * kPageHalf;  // K or V of one page: 4 KB

// A fragments of the group's queries (rows = query heads hh < g), 8 steps of
// 16 dims; Qg points at the group's first query row.
template <int HR>
__device__ __forceinline__ void load_q_frag(const __nv_bfloat16 *Qg, int g, uint32_t (&qa)[8][4]) {
    const int lane = threadIdx.x & 31, qr = lane >> 2, qc = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int c0 = ks * 16 + 2 * qc;
        qa[ks][0] = qr < g ? *reinterpret_cast<const uint32_t *>(Qg + (size_t)qr * kHeadDim + c0) : 0u;
        qa[ks][1] = (HR > 1 && qr + 8 < g) ? *reinterpret_cast<const uint32_t *>(Qg + (size_t)(qr + 8) * kHeadDim + c0)
                                           : 0u;
        qa[ks][2] = qr < g ? *reinterpret_cast<const uint32_t *>(Qg + (size_t)qr * kHeadDim + c0 + 8) : 0u;
        qa[ks][3] = (HR > 1 && qr + 8 < g)
                        ? *reinterpret_cast<const uint32_t *>(Qg + (size_t)(qr + 8) * kHeadDim + c0 + 8)
                        : 0u;
    }
}

// Running state of one warp's online softmax over its pages.
struct AttnState {
    float o[16][4];
    float m[2], l[2];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }
};

// Folds one page (K tile at ks_base, V tile at vs_base, `len` valid keys)
// into the warp's running state.
template <int HR>
__device__ __forceinline__ void attend_page(const uint32_t (&qa)[8][4], uint32_t ks_base, uint32_t vs_base, int len,
                                            float scale, AttnState &st) {
    const int lane = threadIdx.x & 31, qc = lane & 3;
    // ---- S = Q K^T: two 8-key tiles
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
            // matrices: keys 8nt..8nt+7 x 16-byte chunks 2kk .. 2kk + 3
            const int mi = lane >> 3;
            const uint32_t addr = sw_addr(ks_base, 8 * nt + (lane & 7), 2 * kk + mi, kPageHalf);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma16816(s[nt], qa[kk], b0, b1);
            mma16816(s[nt], qa[kk + 1], b2, b3);
        }
    }
    // ---- online softmax of rows qr (and qr + 8): keys 8nt + 2qc + {0, 1}
    float p[2][2][2];  // [row half][tile][pair]
    float alpha[2];
#pragma unroll
    for (int rh = 0; rh < HR; ++rh) {
        float v[2][2];
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = 8 * nt + 2 * qc + e;
                v[nt][e] = key < len ? s[nt][2 * rh + e] * scale : -INFINITY;
                mx = fmaxf(mx, v[nt][e]);
            }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(st.m[rh], mx);
        alpha[rh] = st.m[rh] == -INFINITY ? 0.f : expf(st.m[rh] - m_new);
        float sm = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                p[rh][nt][e] = v[nt][e] == -INFINITY ? 0.f : expf(v[nt][e] - m_new);
                sm += p[rh][nt][e];
            }
        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
        st.l[rh] = st.l[rh] * alpha[rh] + sm;
        st.m[rh] = m_new;
    }
    if (HR == 1) {
        alpha[1] = 0.f;
        p[1][0][0] = p[1][0][1] = p[1][1][0] = p[1][1][1] = 0.f;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
        st.o[nt][0] *= alpha[0];
        st.o[nt][1] *= alpha[0];
        st.o[nt][2] *= alpha[1];
        st.o[nt][3] *= alpha[1];
    }
    // ---- O += P V: A = P (rows x 16 keys) as bf16 hi + lo
    uint32_t ahi[4], alo[4];
    split_pair(p[0][0][0], p[0][0][1], ahi[0], alo[0]);
    split_pair(p[1][0][0], p[1][0][1], ahi[1], alo[1]);
    split_pair(p[0][1][0], p[0][1][1], ahi[2], alo[2]);
    split_pair(p[1][1][0], p[1][1][1], ahi[3], alo[3]);
#pragma unroll
    for (int nt = 0; nt < 16; nt += 2) {
        // matrices: (keys 0-7, chunk nt), (keys 8-15, chunk nt), (keys 0-7, nt+1), (keys 8-15, nt+1)
        const int mi = lane >> 3;
        const uint32_t addr = sw_addr(vs_base, (mi & 1) * 8 + (lane & 7), nt + (mi >> 1), kPageHalf);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma16816(st.o[nt], ahi, b0, b1);
        mma16816(st.o[nt], alo, b0, b1);
        mma16816(st.o[nt + 1], ahi, b2, b3);
        mma16816(st.o[nt + 1], alo, b2, b3);
    }
}

}  // namespace mma
}  // namespace ice
