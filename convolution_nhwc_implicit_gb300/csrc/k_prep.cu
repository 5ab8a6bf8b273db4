// Operand preparation for the tensor-core path: widens int8 to bf16 and pads
// the channel axis to a multiple of 16, writing into plan-owned buffers.
//
// Two kinds of layer use it:
//   - int8 layers: tcgen05 on sm_103a has no integer MMA, but an int8 value
//     is exact in bf16 and the product of two is exact in fp32 (|p| < 2^14),
//     so a bf16 MMA with fp32 accumulation reproduces the int32 accumulator
//     exactly while every partial sum stays below 2^24 (guaranteed for
//     K <= 1024 by |sum| <= K * 128 * 127);
//   - bf16 layers whose channel rows are too short for a TMA box (the
//     3-channel image stem: 6-byte pixels), padded with zero channels to 16
//     (32-byte rows).  Zero channels add zero products: the convolution is
//     unchanged.  (This pads the channel axis, like the 16-channel stripes of
//     the BoxDecode tensors on the SiMa page; it does not build im2col.)
// A row is one pixel of x or one (co, r, s) filter row of w: `cin` source
// channels become `cin_p` bf16 channels.  Layers with k_w * Cin <= 16 also
// fold their k_w taps into those 16 channels (see the implicit-GEMM planner).
#include <cuda_bf16.h>
#include <stdint.h>

#include "conv_internal.h"

namespace {

constexpr int kThreads = 256;

// One thread per 8-channel group of a padded row: reads up to 8 source
// values, writes 16 bytes.
// Idx is uint32_t when every index fits (cheaper division), else uint64_t.
template <typename Tin, typename Idx>
__global__ void __launch_bounds__(kThreads)
widen_pad_kernel(const Tin *__restrict__ src, __nv_bfloat16 *__restrict__ dst, Idx rows, int cin, int cin_p) {
    const Idx groups = (Idx)(cin_p >> 3);
    const Idx i = (Idx)blockIdx.x * kThreads + threadIdx.x;
    if (i >= rows * groups) return;
    const Idx row = i / groups;
    const int c0 = (int)(i - row * groups) * 8;
    const Tin *s = src + (long long)row * cin + c0;
    float v[8];
    if (c0 + 8 <= cin && (cin % 8) == 0) {
        if constexpr (sizeof(Tin) == 1) {
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(s));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[e] = (float)(int8_t)(u.x >> (8 * e));
                v[4 + e] = (float)(int8_t)(u.y >> (8 * e));
            }
        } else {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(s));
            const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[2 * e] = __uint_as_float(wds[e] << 16);
                v[2 * e + 1] = __uint_as_float(wds[e] & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (c0 + e < cin) {
                if constexpr (sizeof(Tin) == 1)
                    v[e] = (float)__ldg(s + e);
                else
                    v[e] = __bfloat162float(__ldg(s + e));
            } else {
                v[e] = 0.0f;  // padding channel
            }
        }
    }
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);  // exact for int8 and bf16 inputs
        out[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(dst + (long long)row * cin_p + c0) = make_uint4(out[0], out[1], out[2], out[3]);
}

// Folded x: output pixel (n, h, u) holds, in channel s * cin + ci, the value
// x[n][h][u - pad_w + s][ci] (zero outside the image and past k_w * cin).
// Inside the image those k_w * cin values are one contiguous run of the
// input row, starting at element t0 = (u - pad_w) * cin of the row, so
// channel c is element t0 + c, valid while 0 <= t0 + c < W * cin.
// One thread per 8-channel group of an output pixel.
template <typename Tin, typename Idx>
__global__ void __launch_bounds__(kThreads)
fold_kw_kernel(const Tin *__restrict__ src, __nv_bfloat16 *__restrict__ dst, Idx rows, int W, int Wf,
               int cin, int kw, int pad_w, int cin_p) {
    const Idx groups = (Idx)(cin_p >> 3);
    const Idx i = (Idx)blockIdx.x * kThreads + threadIdx.x;
    if (i >= rows * groups) return;
    const Idx row = i / groups;                 // (n, h, u) of the folded tensor
    const int c0 = (int)(i - row * groups) * 8;
    const Idx nh = row / (Idx)Wf;
    const int u = (int)(row - nh * (Idx)Wf);
    const Tin *xrow = src + (long long)nh * W * cin;  // input row (n, h)
    const int t0 = (u - pad_w) * cin + c0;
    const int tend = W * cin, cend = kw * cin;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int t = t0 + e;
        v[e] = 0.0f;
        if (c0 + e < cend && t >= 0 && t < tend) {
            const Tin q = __ldg(xrow + t);
            if constexpr (sizeof(Tin) == 1)
                v[e] = (float)q;
            else
                v[e] = __bfloat162float(q);
        }
    }
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);  // exact
        out[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(dst + (long long)row * cin_p + c0) = make_uint4(out[0], out[1], out[2], out[3]);
}

template <typename Tin>
cudaError_t fold_kw(const void *src, __nv_bfloat16 *dst, long long rows, int W, int Wf, int cin, int kw,
                    int pad_w, int cin_p, cudaStream_t st) {
    const long long n = rows * (cin_p / 8);
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + kThreads - 1) / kThreads);
    if (n + kThreads < (1ll << 32))
        fold_kw_kernel<Tin, uint32_t><<<blocks, kThreads, 0, st>>>(reinterpret_cast<const Tin *>(src), dst,
                                                                   (uint32_t)rows, W, Wf, cin, kw, pad_w, cin_p);
    else
        fold_kw_kernel<Tin, uint64_t><<<blocks, kThreads, 0, st>>>(reinterpret_cast<const Tin *>(src), dst,
                                                                   (uint64_t)rows, W, Wf, cin, kw, pad_w, cin_p);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t widen(const void *src, __nv_bfloat16 *dst, long long rows, int cin, int cin_p, cudaStream_t st) {
    const long long n = rows * (cin_p / 8);
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + kThreads - 1) / kThreads);
    if (n + kThreads < (1ll << 32))
        widen_pad_kernel<Tin, uint32_t><<<blocks, kThreads, 0, st>>>(reinterpret_cast<const Tin *>(src), dst,
                                                                     (uint32_t)rows, cin, cin_p);
    else
        widen_pad_kernel<Tin, uint64_t><<<blocks, kThreads, 0, st>>>(reinterpret_cast<const Tin *>(src), dst,
                                                                     (uint64_t)rows, cin, cin_p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const conv_plan *p, const void *x, const void *w, cudaStream_t st) {
    const IgemmGeom &g = p->ig;
    const bool i8 = p->dtype == CONV_I8;
    cudaError_t e;
    if (g.fold) {
        // x: (n, h, u) pixels of width g.wx; w: the OHWI rows of one (co, r)
        // already hold (s, ci) contiguously, i.e. the folded channel order.
        const long long xrows = (long long)p->s.n * p->s.h * g.wx;
        const long long wrows = (long long)p->s.c_out * p->s.k_h;
        const int kc = p->s.k_w * p->s.c_in;
        e = i8 ? fold_kw<int8_t>(x, p->d_xprep, xrows, p->s.w, g.wx, p->s.c_in, p->s.k_w, p->pad_w, p->cin_p, st)
               : fold_kw<__nv_bfloat16>(x, p->d_xprep, xrows, p->s.w, g.wx, p->s.c_in, p->s.k_w, p->pad_w,
                                        p->cin_p, st);
        if (e == cudaSuccess)
            e = i8 ? widen<int8_t>(w, p->d_wprep, wrows, kc, p->cin_p, st)
                   : widen<__nv_bfloat16>(w, p->d_wprep, wrows, kc, p->cin_p, st);
        return e;
    }
    const long long xrows = (long long)p->s.n * p->s.h * p->s.w;
    const long long wrows = (long long)p->s.c_out * p->s.k_h * p->s.k_w;
    if (i8) {
        e = widen<int8_t>(x, p->d_xprep, xrows, p->s.c_in, p->cin_p, st);
        if (e == cudaSuccess) e = widen<int8_t>(w, p->d_wprep, wrows, p->s.c_in, p->cin_p, st);
    } else {
        e = widen<__nv_bfloat16>(x, p->d_xprep, xrows, p->s.c_in, p->cin_p, st);
        if (e == cudaSuccess) e = widen<__nv_bfloat16>(w, p->d_wprep, wrows, p->s.c_in, p->cin_p, st);
    }
    return e;
}
