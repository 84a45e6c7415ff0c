// common.cuh -- device helpers shared by the RMSNorm kernels: element packs
// moved with one memory instruction, streaming loads/stores, bf16/fp16 <->
// fp32, lane-group reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace rmsk {

typedef __nv_bfloat16 bf16;
typedef __half f16;

// ---------------------------------------------------------------- memory ops
// Row data is touched once per kernel: loads skip L1 allocation so the
// weight (reused by every row) stays resident there. All are volatile asm so
// the compiler keeps their program order (a thread always reads an element
// before it overwrites it, which makes the documented in-place uses safe).

__device__ __forceinline__ uint4 ld_row_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_row_b32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_row_b16(const void *p)
{
    uint16_t v;
    asm volatile("ld.global.L1::no_allocate.b16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_row_v4(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_row_b32(void *p, uint32_t v)
{
    asm volatile("st.global.b32 [%0], %1;" : : "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_row_b16(void *p, uint16_t v)
{
    asm volatile("st.global.b16 [%0], %1;" : : "l"(p), "h"(v) : "memory");
}

// 32-byte accesses (sm_100 family: one instruction moves 8 words per
// thread). RMSK_L2_EVICT_FIRST marks streamed row data as first to leave L2.
#ifndef RMSK_L2_EVICT_FIRST
#define RMSK_L2_EVICT_FIRST 0
#endif
#if RMSK_L2_EVICT_FIRST
#define RMSK_L2_HINT ".L2::evict_first"
#else
#define RMSK_L2_HINT ""
#endif

struct u32x8 {
    uint32_t w[8];
};

__device__ __forceinline__ u32x8 ld_row_v8(const void *p)
{
    u32x8 v;
    asm volatile("ld.global.L1::no_allocate" RMSK_L2_HINT ".v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                   "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_row_v8(void *p, const u32x8 &v)
{
    asm volatile("st.global" RMSK_L2_HINT ".v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :
                 : "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]),
                   "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}

// ------------------------------------------------ 16-bit formats <-> fp32
// Half16<T>: conversions of a 16-bit storage format (bf16 or fp16) to and
// from fp32, on one element or on a 32-bit word holding two (the lower
// address in the low half). Widening is exact in both formats; narrowing
// rounds to nearest even (including fp16 subnormals and overflow to inf).
template <typename T> struct Half16;

template <> struct Half16<bf16> {
    using Tag = void;
    // bf16 is the upper half of an fp32 word, so widening is a shift.
    __device__ __forceinline__ static float2 wide2(uint32_t u)
    {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    }
    __device__ __forceinline__ static float wide1(uint16_t u)
    {
        return __uint_as_float((uint32_t)u << 16);
    }
    __device__ __forceinline__ static uint32_t narrow2(float lo, float hi)
    {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&b);
    }
    __device__ __forceinline__ static uint16_t narrow1(float v)
    {
        __nv_bfloat16 b = __float2bfloat16_rn(v);
        return *reinterpret_cast<uint16_t *>(&b);
    }
};

template <> struct Half16<f16> {
    using Tag = void;
    __device__ __forceinline__ static float2 wide2(uint32_t u)
    {
        __half2 h = *reinterpret_cast<__half2 *>(&u);
        return __half22float2(h);
    }
    __device__ __forceinline__ static float wide1(uint16_t u)
    {
        return __half2float(__ushort_as_half(u));
    }
    __device__ __forceinline__ static uint32_t narrow2(float lo, float hi)
    {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static uint16_t narrow1(float v)
    {
        return __half_as_ushort(__float2half_rn(v));
    }
};

// ------------------------------------------------------- packed fp32 math
// The sm_100 family issues two fp32 operations per FFMA2 / FMUL2 / FADD2
// instruction; pairs of a pack's elements are computed together. Packs of
// one element use plain fp32. The overloads keep the kernels generic.
__device__ __forceinline__ float2 vfma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float vfma(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ float2 vmul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float vmul(float a, float b) { return a * b; }
__device__ __forceinline__ float2 vadd(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float vadd(float a, float b) { return a + b; }
__device__ __forceinline__ float hsum(float2 a) { return a.x + a.y; }
__device__ __forceinline__ float hsum(float a) { return a; }
template <typename F> __device__ __forceinline__ F splat(float s);
template <> __device__ __forceinline__ float2 splat<float2>(float s) { return make_float2(s, s); }
template <> __device__ __forceinline__ float splat<float>(float s) { return s; }

// The E elements of one pack widened to fp32: N lanes of F (float2 pairs
// when E is even, one float otherwise).
template <int E>
struct Vals {
    using F = typename std::conditional<E % 2 == 0, float2, float>::type;
    static constexpr int N = E % 2 == 0 ? E / 2 : 1;
    F v[N];
    __device__ __forceinline__ static Vals zero()
    {
        Vals r;
#pragma unroll
        for (int i = 0; i < N; ++i)
            r.v[i] = splat<F>(0.f);
        return r;
    }
    __device__ __forceinline__ float get(int e) const
    {
        if constexpr (E % 2 == 0)
            return (e & 1) ? v[e >> 1].y : v[e >> 1].x;
        else
            return v[0];
    }
};

// ----------------------------------------------------------------- packs
// Pack<T, E>: E consecutive elements of T moved by one memory instruction
// (E * sizeof(T) == 16 or 32 for the vectorised kernels, E == 1 for the
// scalar ones). idx counts packs from `base`. The 16-bit formats share one
// definition per width (selected through Half16<T>::Tag).
template <typename T, int E, typename Enable = void> struct Pack;

// 16-bit formats (bf16, fp16), 16-byte packs.
template <typename T> struct Pack<T, 8, typename Half16<T>::Tag> {
    using C = Half16<T>;
    uint4 u;
    static constexpr int E = 8;
    __device__ __forceinline__ static Pack zero() { Pack p; p.u = make_uint4(0, 0, 0, 0); return p; }
    __device__ __forceinline__ static Pack load(const void *base, int64_t idx)
    {
        Pack p; p.u = ld_row_v4(static_cast<const uint4 *>(base) + idx); return p;
    }
    __device__ __forceinline__ static Pack load_cached(const void *base, int64_t idx)
    {
        Pack p; p.u = __ldg(static_cast<const uint4 *>(base) + idx); return p;
    }
    __device__ __forceinline__ void store(void *base, int64_t idx) const
    {
        st_row_v4(static_cast<uint4 *>(base) + idx, u);
    }
    __device__ __forceinline__ void to_float(float (&f)[8]) const
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = C::wide2(w[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ __forceinline__ static Pack from_float(const float (&f)[8])
    {
        Pack p;
        p.u.x = C::narrow2(f[0], f[1]); p.u.y = C::narrow2(f[2], f[3]);
        p.u.z = C::narrow2(f[4], f[5]); p.u.w = C::narrow2(f[6], f[7]);
        return p;
    }
    __device__ __forceinline__ void widen(Vals<8> &f) const
    {
        f.v[0] = C::wide2(u.x);
        f.v[1] = C::wide2(u.y);
        f.v[2] = C::wide2(u.z);
        f.v[3] = C::wide2(u.w);
    }
    __device__ __forceinline__ static Pack narrow(const Vals<8> &f)
    {
        Pack p;
        p.u.x = C::narrow2(f.v[0].x, f.v[0].y); p.u.y = C::narrow2(f.v[1].x, f.v[1].y);
        p.u.z = C::narrow2(f.v[2].x, f.v[2].y); p.u.w = C::narrow2(f.v[3].x, f.v[3].y);
        return p;
    }
};

// 16-bit formats, 32-byte packs (one 256-bit access).
template <typename T> struct Pack<T, 16, typename Half16<T>::Tag> {
    using C = Half16<T>;
    u32x8 u;
    static constexpr int E = 16;
    __device__ __forceinline__ static Pack zero()
    {
        Pack p;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p.u.w[i] = 0;
        return p;
    }
    __device__ __forceinline__ static Pack load(const void *base, int64_t idx)
    {
        Pack p; p.u = ld_row_v8(static_cast<const uint4 *>(base) + 2 * idx); return p;
    }
    __device__ __forceinline__ static Pack load_cached(const void *base, int64_t idx)
    {
        Pack p;
        const uint4 *q = static_cast<const uint4 *>(base) + 2 * idx;
        const uint4 a = __ldg(q), b = __ldg(q + 1);
        p.u.w[0] = a.x; p.u.w[1] = a.y; p.u.w[2] = a.z; p.u.w[3] = a.w;
        p.u.w[4] = b.x; p.u.w[5] = b.y; p.u.w[6] = b.z; p.u.w[7] = b.w;
        return p;
    }
    __device__ __forceinline__ void store(void *base, int64_t idx) const
    {
        st_row_v8(static_cast<uint4 *>(base) + 2 * idx, u);
    }
    __device__ __forceinline__ void widen(Vals<16> &f) const
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            f.v[i] = C::wide2(u.w[i]);
    }
    __device__ __forceinline__ static Pack narrow(const Vals<16> &f)
    {
        Pack p;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p.u.w[i] = C::narrow2(f.v[i].x, f.v[i].y);
        return p;
    }
};

template <> struct Pack<float, 8> {
    u32x8 u;
    static constexpr int E = 8;
    __device__ __forceinline__ static Pack zero()
    {
        Pack p;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p.u.w[i] = 0;
        return p;
    }
    __device__ __forceinline__ static Pack load(const void *base, int64_t idx)
    {
        Pack p; p.u = ld_row_v8(static_cast<const uint4 *>(base) + 2 * idx); return p;
    }
    __device__ __forceinline__ static Pack load_cached(const void *base, int64_t idx)
    {
        Pack p;
        const uint4 *q = static_cast<const uint4 *>(base) + 2 * idx;
        const uint4 a = __ldg(q), b = __ldg(q + 1);
        p.u.w[0] = a.x; p.u.w[1] = a.y; p.u.w[2] = a.z; p.u.w[3] = a.w;
        p.u.w[4] = b.x; p.u.w[5] = b.y; p.u.w[6] = b.z; p.u.w[7] = b.w;
        return p;
    }
    __device__ __forceinline__ void store(void *base, int64_t idx) const
    {
        st_row_v8(static_cast<uint4 *>(base) + 2 * idx, u);
    }
    __device__ __forceinline__ void widen(Vals<8> &f) const
    {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f.v[i] = make_float2(__uint_as_float(u.w[2 * i]), __uint_as_float(u.w[2 * i + 1]));
    }
    __device__ __forceinline__ static Pack narrow(const Vals<8> &f)
    {
        Pack p;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            p.u.w[2 * i] = __float_as_uint(f.v[i].x);
            p.u.w[2 * i + 1] = __float_as_uint(f.v[i].y);
        }
        return p;
    }
};

// 16-bit formats, one element per access.
template <typename T> struct Pack<T, 1, typename Half16<T>::Tag> {
    using C = Half16<T>;
    uint16_t u;
    static constexpr int E = 1;
    __device__ __forceinline__ static Pack zero() { Pack p; p.u = 0; return p; }
    __device__ __forceinline__ static Pack load(const void *base, int64_t idx)
    {
        Pack p; p.u = ld_row_b16(static_cast<const uint16_t *>(base) + idx); return p;
    }
    __device__ __forceinline__ static Pack load_cached(const void *base, int64_t idx)
    {
        Pack p; p.u = __ldg(static_cast<const unsigned short *>(base) + idx); return p;
    }
    __device__ __forceinline__ void store(void *base, int64_t idx) const
    {
        st_row_b16(static_cast<uint16_t *>(base) + idx, u);
    }
    __device__ __forceinline__ void to_float(float (&f)[1]) const { f[0] = C::wide1(u); }
    __device__ __forceinline__ static Pack from_float(const float (&f)[1])
    {
        Pack p; p.u = C::narrow1(f[0]); return p;
    }
    __device__ __forceinline__ void widen(Vals<1> &f) const { f.v[0] = C::wide1(u); }
    __device__ __forceinline__ static Pack narrow(const Vals<1> &f)
    {
        Pack p; p.u = C::narrow1(f.v[0]); return p;
    }
};

template <> struct Pack<float, 4> {
    uint4 u;
    static constexpr int E = 4;
    __device__ __forceinline__ static Pack zero() { Pack p; p.u = make_uint4(0, 0, 0, 0); return p; }
    __device__ __forceinline__ static Pack load(const void *base, int64_t idx)
    {
        Pack p; p.u = ld_row_v4(static_cast<const uint4 *>(base) + idx); return p;
    }
    __device__ __forceinline__ static Pack load_cached(const void *base, int64_t idx)
    {
        Pack p; p.u = __ldg(static_cast<const uint4 *>(base) + idx); return p;
    }
    __device__ __forceinline__ void store(void *base, int64_t idx) const
    {
        st_row_v4(static_cast<uint4 *>(base) + idx, u);
    }
    __device__ __forceinline__ void to_float(float (&f)[4]) const
    {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static Pack from_float(const float (&f)[4])
    {
        Pack p;
        p.u = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                         __float_as_uint(f[2]), __float_as_uint(f[3]));
        return p;
    }
    __device__ __forceinline__ void widen(Vals<4> &f) const
    {
        f.v[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        f.v[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
    __device__ __forceinline__ static Pack narrow(const Vals<4> &f)
    {
        Pack p;
        p.u = make_uint4(__float_as_uint(f.v[0].x), __float_as_uint(f.v[0].y),
                         __float_as_uint(f.v[1].x), __float_as_uint(f.v[1].y));
        return p;
    }
};

template <> struct Pack<float, 1> {
    uint32_t u;
    static constexpr int E = 1;
    __device__ __forceinline__ static Pack zero() { Pack p; p.u = 0; return p; }
    __device__ __forceinline__ static Pack load(const void *base, int64_t idx)
    {
        Pack p; p.u = ld_row_b32(static_cast<const uint32_t *>(base) + idx); return p;
    }
    __device__ __forceinline__ static Pack load_cached(const void *base, int64_t idx)
    {
        Pack p; p.u = __ldg(static_cast<const unsigned int *>(base) + idx); return p;
    }
    __device__ __forceinline__ void store(void *base, int64_t idx) const
    {
        st_row_b32(static_cast<uint32_t *>(base) + idx, u);
    }
    __device__ __forceinline__ void to_float(float (&f)[1]) const { f[0] = __uint_as_float(u); }
    __device__ __forceinline__ static Pack from_float(const float (&f)[1])
    {
        Pack p; p.u = __float_as_uint(f[0]); return p;
    }
    __device__ __forceinline__ void widen(Vals<1> &f) const { f.v[0] = __uint_as_float(u); }
    __device__ __forceinline__ static Pack narrow(const Vals<1> &f)
    {
        Pack p; p.u = __float_as_uint(f.v[0]); return p;
    }
};

// ------------------------------------------------------------ reductions
// Butterfly sum over groups of N adjacent lanes (N a power of two <= 32).
// Every lane of a group ends with bit-identical sums: each step adds the
// same two values in either order, and fp32 addition is commutative.
template <int N>
__device__ __forceinline__ float group_allreduce(float v)
{
#pragma unroll
    for (int o = N / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Sum of four values over a warp in six shuffles. Lane l ends with the warp
// total of value number (l >> 3) & 3 (a, b, c, d in that order). The first
// two exchanges halve the work: across 16 lanes each half keeps two of the
// four values and hands the other two to its partner, across 8 lanes one of
// the two; a butterfly over the 8 lanes that now hold the same value
// finishes, so those 8 lanes end bit-identical. Needs all 32 lanes, with
// lane = threadIdx.x % 32 (blocks of whole warps).
__device__ __forceinline__ float warp_sum4_spread(float a, float b, float c, float d)
{
    const unsigned lane = threadIdx.x & 31u;
    const bool h16 = (lane & 16u) != 0, h8 = (lane & 8u) != 0;
    float k0 = h16 ? c : a, k1 = h16 ? d : b;
    const float s0 = h16 ? a : c, s1 = h16 ? b : d;
    k0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 16);
    k1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 16);
    float v = h8 ? k1 : k0;
    const float s = h8 ? k0 : k1;
    v += __shfl_xor_sync(0xFFFFFFFFu, s, 8);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    return v;
}

// ------------------------------------------------------- launch ordering
// Programmatic dependent launch: a kernel launched with the
// programmatic-serialization attribute may start while the previous kernel
// on the stream finishes; griddep_wait() blocks until that kernel has
// completed and its memory is visible. griddep_launch_dependents() lets the
// next such kernel be scheduled early. Both are no-ops without the attribute.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// Bring the line holding p into L2 (L2 is the coherence point, so what a
// later load finds there is never stale). Holds no register.
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

} // namespace rmsk
