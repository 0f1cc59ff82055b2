// Keys and warp-level sorting networks shared by the page-selection kernels.
//
// IceCache orders the parents of a head by their score q.p, best first; ties
// go to the smaller parent id.  A 64-bit key carries both: the high word is
// the order-preserving integer form of the fp32 score, the low word the
// complement of the id, so that descending key order is the selection order.
#pragma once

#include <stdint.h>

namespace ice {
namespace topk {

// Order-preserving map of an fp32 value onto uint32, and back.
__device__ __forceinline__ uint32_t ord_f32(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
// 64-bit key whose descending order is (score descending, id ascending).
__device__ __forceinline__ unsigned long long sort_key(float s, int id) {
    return ((unsigned long long)ord_f32(s) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ int key_id(unsigned long long k) { return (int)(0xFFFFFFFFu - (uint32_t)k); }
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }
__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) { return a < b ? a : b; }

// A threshold T (order-preserving form) that at least kc of the warp's values
// (V per lane, 0 = none; kc <= 32 and at least kc values present) reach, and
// at most kc + slack unless ties force more; T is itself one of the values.
// The kc-th largest lies between lo, the smallest of the lanes' maxima (kc or
// more values reach it), and the maximum hi, so the bits above their first
// difference are those of hi; the remaining bits are fixed two at a time from
// the top (three counts per step), and the search stops once at most
// kc + slack values reach the prefix.  T is then the least value at or above
// the prefix.
template <int V>
__device__ __forceinline__ uint32_t kth_bound_ord(const uint32_t (&v)[V], int kc, int slack) {
    uint32_t lm = 0u;
#pragma unroll
    for (int e = 0; e < V; ++e) lm = max(lm, v[e]);
    const uint32_t hi = __reduce_max_sync(0xffffffffu, lm);
    const uint32_t lo = __reduce_min_sync(0xffffffffu, lm != 0u ? lm : 0xFFFFFFFFu);
    int nb = lo >= hi ? 0 : 32 - __clz(lo ^ hi);  // open low bits
    uint32_t r = nb >= 32 ? 0u : (hi >> nb) << nb;
    int nr = 0x7FFFFFFF;  // values >= r (unknown until a step raises r)
    while (nb > 0 && nr > kc + slack) {
        if (nb >= 2) {
            const int b = nb - 2;
            const uint32_t c1 = r | (1u << b), c2 = r | (2u << b), c3 = r | (3u << b);
            unsigned a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
            for (int e = 0; e < V; ++e) {
                a1 += v[e] >= c1;
                a2 += v[e] >= c2;
                a3 += v[e] >= c3;
            }
            const int n1 = (int)__reduce_add_sync(0xffffffffu, a1);
            const int n2 = (int)__reduce_add_sync(0xffffffffu, a2);
            const int n3 = (int)__reduce_add_sync(0xffffffffu, a3);
            if (n3 >= kc) {
                r = c3;
                nr = n3;
            } else if (n2 >= kc) {
                r = c2;
                nr = n2;
            } else if (n1 >= kc) {
                r = c1;
                nr = n1;
            }
            nb = b;
        } else {
            const uint32_t c1 = r | 1u;
            unsigned a1 = 0;
#pragma unroll
            for (int e = 0; e < V; ++e) a1 += v[e] >= c1;
            const int n1 = (int)__reduce_add_sync(0xffffffffu, a1);
            if (n1 >= kc) r = c1;
            nb = 0;
        }
    }
    uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
    for (int e = 0; e < V; ++e) mn = v[e] >= r && v[e] != 0u ? min(mn, v[e]) : mn;
    return __reduce_min_sync(0xffffffffu, mn);
}

// Descending bitonic sort of the warp's 64 keys: key i in lane i % 32 of v[i / 32].
__device__ __forceinline__ void sort64_desc(unsigned long long (&v)[2]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride == 32) {
                const unsigned long long a = v[0], b = v[1];
                v[0] = umax64(a, b);
                v[1] = umin64(a, b);
            } else {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[e], stride);
                    const bool desc = ((e * 32 + lane) & size) == 0;
                    const bool lower = (lane & stride) == 0;
                    v[e] = (lower == desc) ? umax64(v[e], o) : umin64(v[e], o);
                }
            }
        }
    }
}
// The best 32 of two descending lists (one key per lane), descending.
__device__ __forceinline__ unsigned long long merge32(unsigned long long a, unsigned long long b) {
    const int lane = threadIdx.x & 31;
    a = umax64(a, __shfl_sync(0xffffffffu, b, 31 - lane));
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, a, stride);
        a = (lane & stride) == 0 ? umax64(a, o) : umin64(a, o);
    }
    return a;
}

}  // namespace topk
}  // namespace ice
