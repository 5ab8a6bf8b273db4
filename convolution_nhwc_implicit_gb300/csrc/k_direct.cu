// Direct convolution on the CUDA cores: any shape, stride, padding and
// grouping, in fp32 (FFMA, never TF32), bf16 (fp32 accumulation) and int8
// (exact int32 accumulation, dp4a where channels come in fours).
//
// This family serves the layers the tensor-core path does not take: the
// fp32 layers (the MNIST-sized 3x3 conv and the keyword-spotting DS-CNN
// block of the "nanoinfer" page, whose fp32 results must not be silently
// rounded to TF32 -- "nanoinfer", cuDNN comparison, default math mode),
// inputs with too few channels for a 16-byte TMA row (the Cin = 1 stem,
// the Cin = 3 image stem), and grouped layers.
//
// Mapping: one thread owns one output pixel and COT consecutive output
// channels of one group.  Threads of a warp share the output-channel chunk
// (blockIdx.y), so every weight load is a warp-wide broadcast; consecutive
// threads take consecutive pixels.
#include <cuda_bf16.h>
#include <stdint.h>

#include "conv_internal.h"
#include "epilogue.cuh"

using namespace convk;

namespace {

constexpr int kCot = 8;       // output channels per thread
constexpr int kThreads = 128;

struct DirectArgs {
    int N, H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, OH, OW;
    int cin_g, cout_g, chunks_per_group;
    long long npix;
    int act;
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
direct_conv_float(DirectArgs a, const T *__restrict__ x, const T *__restrict__ w,
                  const float *__restrict__ bias, T *__restrict__ y) {
    long long pix = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (pix >= a.npix) return;
    const int g = blockIdx.y / a.chunks_per_group;
    const int cc = blockIdx.y - g * a.chunks_per_group;
    const int co0 = g * a.cout_g + cc * kCot;
    const int nco = min(kCot, a.cout_g - cc * kCot);
    const int ow = (int)(pix % a.OW);
    const long long t = pix / a.OW;
    const int oh = (int)(t % a.OH);
    const int n = (int)(t / a.OH);
    const int g0 = g * a.cin_g;
    const long long K = (long long)a.KH * a.KW * a.cin_g;

    float acc[kCot];
#pragma unroll
    for (int i = 0; i < kCot; ++i) acc[i] = 0.0f;

    for (int r = 0; r < a.KH; ++r) {
        const int ih = oh * a.stride - a.pad_h + r;
        if (ih < 0 || ih >= a.H) continue;  // zero padding
        for (int s = 0; s < a.KW; ++s) {
            const int iw = ow * a.stride - a.pad_w + s;
            if (iw < 0 || iw >= a.W) continue;
            const T *xp = x + (((long long)n * a.H + ih) * a.W + iw) * a.Cin + g0;
            const T *wp = w + (long long)co0 * K + (long long)(r * a.KW + s) * a.cin_g;
            for (int j = 0; j < a.cin_g; ++j) {
                const float xv = Elem<T>::to_f(__ldg(xp + j));
#pragma unroll
                for (int i = 0; i < kCot; ++i)
                    if (i < nco) acc[i] = __fmaf_rn(xv, Elem<T>::to_f(__ldg(wp + i * K + j)), acc[i]);
            }
        }
    }
    T *yp = y + pix * a.Cout + co0;
#pragma unroll
    for (int i = 0; i < kCot; ++i) {
        if (i < nco) {
            float v = acc[i] + (bias ? __ldg(bias + co0 + i) : 0.0f);
            yp[i] = Elem<T>::from_f(activate(v, a.act));
        }
    }
}

// int8: exact int32 accumulation.  With VEC4 the group's channels come in
// fours (cin_g % 4 == 0) and every x / w row start is 4-byte aligned, so four
// products are summed per __dp4a.
template <bool VEC4>
__global__ void __launch_bounds__(kThreads)
direct_conv_i8(DirectArgs a, const int8_t *__restrict__ x, const int8_t *__restrict__ w,
               const int32_t *__restrict__ bias, const float *__restrict__ mult,
               int8_t *__restrict__ y) {
    long long pix = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (pix >= a.npix) return;
    const int g = blockIdx.y / a.chunks_per_group;
    const int cc = blockIdx.y - g * a.chunks_per_group;
    const int co0 = g * a.cout_g + cc * kCot;
    const int nco = min(kCot, a.cout_g - cc * kCot);
    const int ow = (int)(pix % a.OW);
    const long long t = pix / a.OW;
    const int oh = (int)(t % a.OH);
    const int n = (int)(t / a.OH);
    const int g0 = g * a.cin_g;
    const long long K = (long long)a.KH * a.KW * a.cin_g;

    int acc[kCot];
#pragma unroll
    for (int i = 0; i < kCot; ++i) acc[i] = 0;

    for (int r = 0; r < a.KH; ++r) {
        const int ih = oh * a.stride - a.pad_h + r;
        if (ih < 0 || ih >= a.H) continue;
        for (int s = 0; s < a.KW; ++s) {
            const int iw = ow * a.stride - a.pad_w + s;
            if (iw < 0 || iw >= a.W) continue;
            const int8_t *xp = x + (((long long)n * a.H + ih) * a.W + iw) * a.Cin + g0;
            const int8_t *wp = w + (long long)co0 * K + (long long)(r * a.KW + s) * a.cin_g;
            if (VEC4) {
                const int *xp4 = reinterpret_cast<const int *>(xp);
                for (int j = 0; j < a.cin_g / 4; ++j) {
                    const int xv = __ldg(xp4 + j);
#pragma unroll
                    for (int i = 0; i < kCot; ++i)
                        if (i < nco)
                            acc[i] = __dp4a(xv, __ldg(reinterpret_cast<const int *>(wp + i * K) + j), acc[i]);
                }
            } else {
                for (int j = 0; j < a.cin_g; ++j) {
                    const int xv = __ldg(xp + j);
#pragma unroll
                    for (int i = 0; i < kCot; ++i)
                        if (i < nco) acc[i] += xv * (int)__ldg(wp + i * K + j);
                }
            }
        }
    }
    int8_t *yp = y + pix * a.Cout + co0;
#pragma unroll
    for (int i = 0; i < kCot; ++i) {
        if (i < nco) {
            long long v = (long long)acc[i] + (bias ? (long long)__ldg(bias + co0 + i) : 0ll);
            yp[i] = (int8_t)requant_i8(v, __ldg(mult + co0 + i), a.act);
        }
    }
}

DirectArgs make_args(const conv_plan *p) {
    DirectArgs a;
    a.N = p->s.n; a.H = p->s.h; a.W = p->s.w; a.Cin = p->s.c_in; a.Cout = p->s.c_out;
    a.KH = p->s.k_h; a.KW = p->s.k_w; a.stride = p->stride; a.pad_h = p->pad_h; a.pad_w = p->pad_w;
    a.OH = p->oh; a.OW = p->ow;
    a.cin_g = p->s.c_in / p->groups;
    a.cout_g = p->s.c_out / p->groups;
    a.chunks_per_group = (a.cout_g + kCot - 1) / kCot;
    a.npix = (long long)a.N * a.OH * a.OW;
    a.act = (int)p->act;
    return a;
}

}  // namespace

bool direct_supported(const conv_plan *p) {
    const int cout_g = p->s.c_out / p->groups;
    const long long chunks = (long long)p->groups * ((cout_g + kCot - 1) / kCot);
    const long long blocks = ((long long)p->s.n * p->oh * p->ow + kThreads - 1) / kThreads;
    return chunks <= 65535 && blocks <= 0x7fffffffll;
}

cudaError_t launch_direct(const conv_plan *p, const void *x, const void *w, const void *bias,
                          void *y, cudaStream_t st) {
    DirectArgs a = make_args(p);
    dim3 grid((unsigned)((a.npix + kThreads - 1) / kThreads), (unsigned)(p->groups * a.chunks_per_group));
    switch (p->dtype) {
    case CONV_F32:
        direct_conv_float<float><<<grid, kThreads, 0, st>>>(
            a, (const float *)x, (const float *)w, (const float *)bias, (float *)y);
        break;
    case CONV_BF16:
        direct_conv_float<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            a, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w, (const float *)bias,
            (__nv_bfloat16 *)y);
        break;
    case CONV_I8:
        if (a.cin_g % 4 == 0)
            direct_conv_i8<true><<<grid, kThreads, 0, st>>>(
                a, (const int8_t *)x, (const int8_t *)w, (const int32_t *)bias, p->d_mult, (int8_t *)y);
        else
            direct_conv_i8<false><<<grid, kThreads, 0, st>>>(
                a, (const int8_t *)x, (const int8_t *)w, (const int32_t *)bias, p->d_mult, (int8_t *)y);
        break;
    }
    return cudaGetLastError();
}
