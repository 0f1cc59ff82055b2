// Internal helpers shared by the sm_103a kernels of the IceCache library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ice.h"

namespace ice {

constexpr int kHeadDim = 128;  // d
constexpr int kPage = 16;      // S

// ---------------------------------------------------------------- errors --
// First device-side condition wins; later ones are dropped.
__device__ __forceinline__ void set_err(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------------ element I/O --
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static float load(const float *p) { return *p; }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
};

// Bytes of one d-element row.
template <typename T> constexpr int row_bytes() { return kHeadDim * (int)sizeof(T); }
// 16-byte vectors per row.
template <typename T> constexpr int row_vecs() { return row_bytes<T>() / 16; }

// 16-byte read-only load issued in program order (volatile asm is not
// reordered with other volatile asm), so a batch of them is in flight before
// the arithmetic that consumes them; no L1 allocation (data read once).
__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------ splitmix64 --
// splitmix64 (Steele, Lea & Flood 2014): state advances by the golden-ratio
// increment; an output is the state run through the 64-bit finaliser.
__host__ __device__ __forceinline__ uint64_t sm64_finalise(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
__host__ __device__ __forceinline__ uint64_t sm64_output(uint64_t state0, uint64_t n) {
    return sm64_finalise(state0 + n * 0x9E3779B97F4A7C15ull);
}
// Stream key of one layer: output (layer + 1) of the stream seeded by seed.
__host__ __device__ __forceinline__ uint64_t promote_key(uint64_t seed, int32_t layer) {
    return sm64_output(seed, (uint64_t)(int64_t)layer + 1ull);
}
// Level-`level` promotion draw of `token` in unit (seq, head).
__device__ __forceinline__ uint32_t promote_draw(uint64_t key, int32_t seq, int32_t head, uint32_t token,
                                                 uint32_t level) {
    const uint64_t ctr = (uint64_t)token | ((uint64_t)level << 32) | ((uint64_t)(uint32_t)head << 40) |
                         ((uint64_t)(uint32_t)seq << 52);
    return (uint32_t)(sm64_output(key, ctr + 1ull) >> 32);
}

// ----------------------------------------------------- packed fp32 pairs --
// Two IEEE fp32 values in one 64-bit register; add / sub / mul / fma.rn.f32x2
// each do two correctly rounded fp32 operations in one instruction.
__device__ __forceinline__ unsigned long long pk2(float x, float y) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 upk2(unsigned long long r) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
    return f;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// bf16 pair in one 32-bit word -> fp32 pair
__device__ __forceinline__ unsigned long long bf2_pair(uint32_t w) {
    return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// ------------------------------------------------- double-float summation --
// Error-free transformation of a + b (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}
// The same on two independent pairs at once.
__device__ __forceinline__ void two_sum2(unsigned long long a, unsigned long long b, unsigned long long &s,
                                         unsigned long long &e) {
    s = add2(a, b);
    const unsigned long long bb = sub2(s, a);
    e = add2(sub2(a, sub2(s, bb)), sub2(b, bb));
}

// ------------------------------------------------------------ warp utils --
__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// (score, index) order used by every argmax / top-k here: larger score first,
// lower index on equal scores.
__device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
    return sa > sb || (sa == sb && ia < ib);
}

// ------------------------------------------- programmatic dependent launch --
// A kernel launched with launch_dependent() is scheduled as the CTAs of the
// previous kernel of the stream exit, without waiting for the whole launch to
// retire; it calls dep_wait() before it touches global memory (returns once
// that grid has completed and its writes are visible; a no-op for a plain
// launch).  No kernel here signals its dependents early: measured on the
// build + decode step, dependents scheduled at the start of their predecessor
// sat on the SMs it was still using and cost ~20 us per step.
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

}  // namespace ice
