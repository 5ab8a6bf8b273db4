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

// Packed fp32 pairs (the sm_100 family's f32x2 instructions, through CUDA's
// float2 builtins): each lane of the pair is rounded once, exactly like the
// scalar instruction.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
// Hardware 2^x and 1/x approximations (MUFU), subnormals flushed.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Mish of two values for bf16 outputs, in the Wormhole page's form
// mish(v) = v (1 - 2 / ((1 + e^v)^2 + 1)) (section 9, K1), with e^v =
// 2^(v log2 e).  No clamp is needed: past v ~ 44 the square overflows to
// +inf and the reciprocal to 0, giving v; for v << 0 the bracket is
// 1 - (1 - e^v) (cancellation, absolute error ~|v| 2^-24, far below bf16
// resolution of the result's scale).  Two MUFU operations per value, the
// rest in packed pairs.
__device__ __forceinline__ float2 mish2_fast(float2 v) {
    const float2 e = mul2(v, make_float2(1.4426950408889634f, 1.4426950408889634f));
    const float2 n = make_float2(ex2_approx(e.x), ex2_approx(e.y));
    const float2 w = add2(n, make_float2(1.0f, 1.0f));
    const float2 d = fma2(w, w, make_float2(1.0f, 1.0f));
    const float2 r = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    const float2 s = fma2(r, make_float2(-2.0f, -2.0f), make_float2(1.0f, 1.0f));
    return mul2(v, s);
}

// Activation for bf16 outputs.
__device__ __forceinline__ float activate_fast(float v, int act) {
    if (act == ACT_RELU) return fmaxf(v, 0.0f);
    if (act == ACT_MISH) return mish_fast(v);
    return v;
}

// Two values at a time (packed Mish), for bf16 outputs.
__device__ __forceinline__ float2 activate2_fast(float2 v, int act) {
    if (act == ACT_RELU) return make_float2(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f));
    if (act == ACT_MISH) return mish2_fast(v);
    return v;
}

__device__ __forceinline__ float activate(float v, int act) {
    if (act == ACT_RELU) return fmaxf(v, 0.0f);
    if (act == ACT_MISH) return mish_f32(v);
    return v;
}

// Programmatic dependent launch (see conv_launch): let the next kernel on
// the stream be scheduled, and wait for the previous one to complete (with
// its writes visible) before touching global memory.  Both are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Where a layer's output goes and what is added to it (the conv_output_t
// options): output pixel (n, oh, ow), channel co lands at element
//   base(n, oh, ow) + rep(dy, dx) + co   for dy, dx in [0, up)
// of y, a [N][up*OH][up*OW][Cy] buffer whose channels [c_off, c_off + Cout)
// belong to the layer; res, if not null, is a dense [N][OH][OW][Cout] tensor
// added after the activation.  The plain layer is Cy = Cout, c_off = 0,
// up = 1: base = ((n*OH + oh)*OW + ow)*Cout.
struct OutMap {
    int Cy, c_off, up, OH, OW, Cout;
    const void *res;
    __device__ __forceinline__ long long base(int n, int oh, int ow) const {
        return (((long long)n * OH + oh) * up * ((long long)OW * up) + (long long)ow * up) * Cy + c_off;
    }
    __device__ __forceinline__ long long rep(int dy, int dx) const {
        return ((long long)dy * OW * up + dx) * Cy;
    }
    __device__ __forceinline__ bool plain() const { return up == 1 && c_off == 0 && Cy == Cout; }
};

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
