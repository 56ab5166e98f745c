// Shared device helpers for the edge-attention kernels: 16-byte row chunks,
// bf16/fp32 conversion, warp reductions, launch bookkeeping.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/sga.h"

#define SGA_FULL_MASK 0xffffffffu

namespace sga {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kWarpsPerBlock = 8;

// ---- element types ---------------------------------------------------------

// One 16-byte chunk of a row holds EL elements of T.
template <typename T> struct Elt;
template <> struct Elt<float> { static constexpr int EL = 4; };
template <> struct Elt<__nv_bfloat16> { static constexpr int EL = 8; };

__device__ __forceinline__ uint4 ldg16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Streaming gather: read-only path, do not keep in L1.
__device__ __forceinline__ uint4 ldg16_stream(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <typename T> __device__ __forceinline__ void unpack(const uint4 &u, float *x);

template <> __device__ __forceinline__ void unpack<float>(const uint4 &u, float *x) {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
}

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
template <> __device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4 &u, float *x) {
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16);
    x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16);
    x[7] = __uint_as_float(u.w & 0xffff0000u);
}

template <typename T> __device__ __forceinline__ uint4 pack(const float *x);

template <> __device__ __forceinline__ uint4 pack<float>(const float *x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t *>(&v);
}

template <> __device__ __forceinline__ uint4 pack<__nv_bfloat16>(const float *x) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Sum over aligned groups of W lanes (W a power of two <= 32); every lane of
// the group receives the group total.
template <int W> __device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(SGA_FULL_MASK, v, o);
    return v;
}

template <int W> __device__ __forceinline__ void group_sum2(float &a, float &b) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) {
        a += __shfl_xor_sync(SGA_FULL_MASK, a, o);
        b += __shfl_xor_sync(SGA_FULL_MASK, b, o);
    }
}

// exp2 that maps -inf to 0 without producing NaN for (-inf) - (-inf).
// Two fp32 fused multiply-adds in one instruction (each lane rounded as fmaf).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
// Two fp32 sums / products in one instruction (each lane rounded as fadd / fmul).
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// sum_x a[x] b[x] over an even count, as two interleaved fma chains
template <int EL> __device__ __forceinline__ float dot2(const float *a, const float *b) {
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int x = 0; x < EL; x += 2) s = ffma2(make_float2(a[x], a[x + 1]), make_float2(b[x], b[x + 1]), s);
    return s.x + s.y;
}
// acc[x] += p x[x]
template <int EL> __device__ __forceinline__ void axpy2(float *acc, float p, const float *x) {
#pragma unroll
    for (int i = 0; i < EL; i += 2) {
        const float2 r = ffma2(make_float2(p, p), make_float2(x[i], x[i + 1]), make_float2(acc[i], acc[i + 1]));
        acc[i] = r.x;
        acc[i + 1] = r.y;
    }
}

// Log2 growth of a row maximum that triggers a rescale of the accumulator
// in the lazily rescaled online softmax.
constexpr float kLazyLog2 = 8.0f;

// 2^x by the MUFU instruction: ex2.approx.ftz (relative error about 2^-22,
// far below the bf16 and fp32 tolerances of the weights it makes; subnormal
// results, weights below 2^-126 of a row's largest, flushed to zero; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^(a - m), zero for a = -inf (also when m = -inf)
__device__ __forceinline__ float exp2_diff(float a, float m) {
    return (a == -INFINITY) ? 0.0f : fast_exp2(a - m);
}

// Device error bits (plan error word).
constexpr int kErrIndexRange = 1;   // a gathered node id was outside [0, N)

}  // namespace sga

// ---- host-side launch bookkeeping (defined in api.cu) -----------------------
namespace sga {
void note_launch(sga_kernel_id which, cudaStream_t s, bool after);

// Let Kernel launch with `smem` bytes of dynamic shared memory: raises the
// kernel's limit whenever a launch needs more than any before it (kernels whose
// size depends on the call's shape would otherwise keep the first call's limit
// and refuse a larger launch).
template <auto Kernel> cudaError_t allow_smem(size_t smem) {
    static std::atomic<size_t> allowed{48 * 1024};
    if (smem <= allowed.load(std::memory_order_relaxed)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    size_t cur = allowed.load(std::memory_order_relaxed);
    while (smem > cur && !allowed.compare_exchange_weak(cur, smem, std::memory_order_relaxed)) {
    }
    return cudaSuccess;
}
}
