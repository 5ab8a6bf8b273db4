// Fused epilogue of the convolution layer, shared by every kernel family:
// bias, activation (ReLU / Mish), conversion to the output type, and the
// int8 requantisation.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace convk {

enum { ACT_NONE = 0, ACT_RELU = 1, ACT_MISH = 2 };

// Mish(v) = v * tanh(ln(1 + e^v)) ("YOLOv4, optimized for Wormhole", section 7).
// With n = e^v, tanh(ln(1 + n)) = ((1+n)^2 - 1) / ((1+n)^2 + 1) = t / (t + 2)
// where t = n (n + 2).  This is the Wormhole kernel's form x - 2x/((1+e^x)^2+1)
// rearranged so that nothing cancels for v << 0 (where t/(t+2) ~ n).  Above
// v = 20, t/(t+2) rounds to 1 in fp32 and n^2 would overflow beyond v ~ 44,
// so the function returns v there.  expf and the division are CUDA's
// IEEE-accurate versions (no fast-math).
__device__ __forceinline__ float mish_f32(float v) {
    if (v > 20.0f) return v;
    float n = expf(v);
    float t = n * (n + 2.0f);
    return v * (t / (t + 2.0f));
}

// The same Mish with the hardware exp2 and reciprocal approximations
// (__expf, __fdividef): relative error ~1e-6, far below the bf16 rounding
// (2^-9) of the outputs it feeds.  t + 2 stays below 2^126 (__fdividef's
// range) because the exponent is clamped at 20.
__device__ __forceinline__ float mish_fast(float v) {
    // Above v = 20, t / (t + 2) rounds to 1: clamping the exponent there
    // gives v exactly, without a branch, and keeps t finite.
    const float n = __expf(fminf(v, 20.0f));
    const float t = n * (n + 2.0f);
    return v * __fdividef(t, t + 2.0f);
}

// Activation for bf16 outputs.
__device__ __forceinline__ float activate_fast(float v, int act) {
    if (act == ACT_RELU) return fmaxf(v, 0.0f);
    if (act == ACT_MISH) return mish_fast(v);
    return v;
}

__device__ __forceinline__ float activate(float v, int act) {
    if (act == ACT_RELU) return fmaxf(v, 0.0f);
    if (act == ACT_MISH) return mish_f32(v);
    return v;
}

// int8 requantisation: q = sat_[-128,127](rne(float(v) * M)), then ReLU as
// max(q, 0).  Each step rounds to nearest-even in IEEE single precision, so
// the result is bit-reproducible on any IEEE machine.
__device__ __forceinline__ int requant_i8(long long v, float M, int act) {
    float f = __ll2float_rn(v);
    float p = __fmul_rn(f, M);
    int q = __float2int_rn(p);
    q = min(max(q, -128), 127);
    if (act == ACT_RELU) q = max(q, 0);
    return q;
}

// Type traits for the three element types.
template <typename T> struct Elem;
template <> struct Elem<float> {
    __device__ static __forceinline__ float to_f(float v) { return v; }
    __device__ static __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ static __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Bounded-wait budget of every spin on an mbarrier, in nanoseconds of
// %globaltimer.  A legitimate wait in these kernels lasts microseconds.
constexpr unsigned long long kWaitBudgetNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace convk
