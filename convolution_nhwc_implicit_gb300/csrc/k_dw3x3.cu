// Depthwise 3x3 convolution (groups == Cin == Cout), any stride and padding,
// in fp32, bf16 and int8.  No tensor cores: each output channel has its own
// 3x3 filter and there is no reduction across channels, so the layer is a
// bandwidth-bound stencil ("nanoinfer", "What is still slow": depthwise
// convolution is the whole gap, and NHWC lets one vector load cover many
// channels of one pixel).
//
// Mapping: a thread owns one 16-byte channel vector (4 fp32, 8 bf16 or 16
// int8 channels) at one output column, and walks down `th` output rows.  The
// three input rows under its 3x3 window stay in registers; moving down one
// output row at stride 1 loads only the one new input row (three 16-byte
// loads: the columns w-1, w, w+1), at stride 2 two rows.  Consecutive threads
// take consecutive channel vectors and then consecutive columns, so a warp's
// loads and stores cover contiguous bytes of the NHWC rows; the horizontal
// neighbours a thread re-reads are the neighbouring threads' centre columns
// and come from L1.  The 9 taps x 16 bytes of weights and the bias stay in
// registers for the whole walk.  Bias, activation and the int8
// requantisation are applied before the single 16-byte store.
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

#include "conv_internal.h"
#include "epilogue.cuh"

using namespace convk;

namespace {

constexpr int kThreads = 256;

struct DwArgs {
    int N, H, W, C, OH, OW, stride, pad_h, pad_w, th, nstrips, cv;
    long long items;
    int act;
};

__device__ __forceinline__ uint4 ld16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Unpacks a 16-byte vector into V lanes of the accumulation type.
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int V = 4;
    using Acc = float;
    __device__ static __forceinline__ void unpack(const uint4 &u, float (&o)[4]) {
        o[0] = __uint_as_float(u.x); o[1] = __uint_as_float(u.y);
        o[2] = __uint_as_float(u.z); o[3] = __uint_as_float(u.w);
    }
    __device__ static __forceinline__ float wload(const float *w) { return __ldg(w); }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int V = 8;
    using Acc = float;
    __device__ static __forceinline__ void unpack(const uint4 &u, float (&o)[8]) {
        const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = __uint_as_float(wds[i] << 16);
            o[2 * i + 1] = __uint_as_float(wds[i] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ float wload(const __nv_bfloat16 *w) { return __bfloat162float(__ldg(w)); }
};
template <> struct Vec<int8_t> {
    static constexpr int V = 16;
    using Acc = int;
    __device__ static __forceinline__ void unpack(const uint4 &u, int (&o)[16]) {
        const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int b = 0; b < 4; ++b) o[4 * i + b] = (int)(int8_t)(wds[i] >> (8 * b));
    }
    __device__ static __forceinline__ int wload(const int8_t *w) { return (int)__ldg(w); }
};

template <typename T>
__device__ __forceinline__ void load_row(uint4 (&row)[3], const T *xn, const DwArgs &a, int ih,
                                         int iw0, int coff) {
    const bool rok = ih >= 0 && ih < a.H;
#pragma unroll
    for (int s = 0; s < 3; ++s) {
        const int iw = iw0 + s;
        if (rok && iw >= 0 && iw < a.W)
            row[s] = ld16(xn + ((long long)ih * a.W + iw) * a.C + coff);
        else
            row[s] = make_uint4(0u, 0u, 0u, 0u);  // zero padding
    }
}

// S: the stride when known at compile time (1 or 2); 0 = read it from a.stride.
template <typename T, int S>
__global__ void __launch_bounds__(kThreads)
dw3x3_kernel(DwArgs a, const T *__restrict__ x, const T *__restrict__ w,
             const void *__restrict__ bias, const float *__restrict__ mult, T *__restrict__ y) {
    using VT = Vec<T>;
    using Acc = typename VT::Acc;
    constexpr int V = VT::V;
    const long long it = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (it >= a.items) return;
    const int cv = (int)(it % a.cv);
    long long t = it / a.cv;
    const int ow = (int)(t % a.OW);
    t /= a.OW;
    const int strip = (int)(t % a.nstrips);
    const int n = (int)(t / a.nstrips);
    const int c0 = cv * V;
    const int stride = S ? S : a.stride;

    Acc wr[9][V];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int k = 0; k < 9; ++k) wr[k][v] = VT::wload(w + (long long)(c0 + v) * 9 + k);

    const T *xn = x + (long long)n * a.H * a.W * a.C;
    const int oh0 = strip * a.th;
    const int oh1 = min(oh0 + a.th, a.OH);
    const int iw0 = ow * stride - a.pad_w;

    uint4 win[3][3];
    int ih = oh0 * stride - a.pad_h;
    load_row(win[0], xn, a, ih, iw0, c0);
    load_row(win[1], xn, a, ih + 1, iw0, c0);
    load_row(win[2], xn, a, ih + 2, iw0, c0);

    for (int oh = oh0; oh < oh1; ++oh) {
        Acc acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0;
#pragma unroll
        for (int r = 0; r < 3; ++r)
#pragma unroll
            for (int s = 0; s < 3; ++s) {
                Acc xv[V];
                VT::unpack(win[r][s], xv);
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    if constexpr (std::is_same<Acc, float>::value)
                        acc[v] = __fmaf_rn(xv[v], wr[r * 3 + s][v], acc[v]);
                    else
                        acc[v] += xv[v] * wr[r * 3 + s][v];
                }
            }

        uint4 out;
        T *yp = y + (((long long)n * a.OH + oh) * a.OW + ow) * a.C + c0;
        if constexpr (std::is_same<T, int8_t>::value) {
            const int32_t *b = reinterpret_cast<const int32_t *>(bias);
            uint32_t wds[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int v = 0; v < V; ++v) {
                long long val = (long long)acc[v] + (b ? (long long)__ldg(b + c0 + v) : 0ll);
                int q = requant_i8(val, __ldg(mult + c0 + v), a.act);
                wds[v / 4] |= ((uint32_t)(q & 0xff)) << (8 * (v % 4));
            }
            out = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        } else if constexpr (std::is_same<T, float>::value) {
            const float *b = reinterpret_cast<const float *>(bias);
            float o[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) o[v] = activate(acc[v] + (b ? __ldg(b + c0 + v) : 0.0f), a.act);
            out = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                             __float_as_uint(o[3]));
        } else {
            const float *b = reinterpret_cast<const float *>(bias);
            uint32_t wds[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo = activate(acc[2 * i] + (b ? __ldg(b + c0 + 2 * i) : 0.0f), a.act);
                float hi = activate(acc[2 * i + 1] + (b ? __ldg(b + c0 + 2 * i + 1) : 0.0f), a.act);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
                wds[i] = *reinterpret_cast<uint32_t *>(&h2);
            }
            out = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        }
        *reinterpret_cast<uint4 *>(yp) = out;

        if (oh + 1 < oh1) {
            const int nih = (oh + 1) * stride - a.pad_h;
            if (S == 1) {
#pragma unroll
                for (int s = 0; s < 3; ++s) { win[0][s] = win[1][s]; win[1][s] = win[2][s]; }
                load_row(win[2], xn, a, nih + 2, iw0, c0);
            } else if (S == 2) {
#pragma unroll
                for (int s = 0; s < 3; ++s) win[0][s] = win[2][s];
                load_row(win[1], xn, a, nih + 1, iw0, c0);
                load_row(win[2], xn, a, nih + 2, iw0, c0);
            } else {
                load_row(win[0], xn, a, nih, iw0, c0);
                load_row(win[1], xn, a, nih + 1, iw0, c0);
                load_row(win[2], xn, a, nih + 2, iw0, c0);
            }
        }
    }
}

template <typename T>
void launch_t(const DwArgs &a, dim3 grid, const void *x, const void *w, const void *bias,
              const float *mult, void *y, cudaStream_t st) {
    if (a.stride == 1)
        dw3x3_kernel<T, 1><<<grid, kThreads, 0, st>>>(a, (const T *)x, (const T *)w, bias, mult, (T *)y);
    else if (a.stride == 2)
        dw3x3_kernel<T, 2><<<grid, kThreads, 0, st>>>(a, (const T *)x, (const T *)w, bias, mult, (T *)y);
    else
        dw3x3_kernel<T, 0><<<grid, kThreads, 0, st>>>(a, (const T *)x, (const T *)w, bias, mult, (T *)y);
}

}  // namespace

bool dw3x3_supported(const conv_plan *p) {
    const int C = p->s.c_in;
    const int V = 16 / conv_esize(p->dtype);
    return p->groups == C && p->s.c_out == C && p->s.k_h == 3 && p->s.k_w == 3 && C % V == 0;
}

void dw3x3_configure(conv_plan *p) {
    const int V = 16 / conv_esize(p->dtype);
    const long long cols = (long long)p->s.n * p->ow * (p->s.c_in / V);
    // Rows per thread: long walks amortise the weight loads and reuse the
    // register window, but the grid must still fill the GPU several times.
    int th = 16;
    while (th > 1 && cols * ((p->oh + th - 1) / th) < (long long)p->num_sms * kThreads * 4) th /= 2;
    p->dw.th = th;
    p->dw.nstrips = (p->oh + th - 1) / th;
    p->dw.items = cols * p->dw.nstrips;
}

cudaError_t launch_dw3x3(const conv_plan *p, const void *x, const void *w, const void *bias,
                         void *y, cudaStream_t st) {
    DwArgs a;
    a.N = p->s.n; a.H = p->s.h; a.W = p->s.w; a.C = p->s.c_in; a.OH = p->oh; a.OW = p->ow;
    a.stride = p->stride; a.pad_h = p->pad_h; a.pad_w = p->pad_w;
    a.th = p->dw.th; a.nstrips = p->dw.nstrips;
    a.cv = p->s.c_in / (16 / conv_esize(p->dtype));
    a.items = p->dw.items;
    a.act = (int)p->act;
    dim3 grid((unsigned)((a.items + kThreads - 1) / kThreads));
    switch (p->dtype) {
    case CONV_F32: launch_t<float>(a, grid, x, w, bias, p->d_mult, y, st); break;
    case CONV_BF16: launch_t<__nv_bfloat16>(a, grid, x, w, bias, p->d_mult, y, st); break;
    case CONV_I8: launch_t<int8_t>(a, grid, x, w, bias, p->d_mult, y, st); break;
    }
    return cudaGetLastError();
}
