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
#include "epilogue.cuh"

namespace {

constexpr int kThreads = 256;

// One pre-pass job: `rows` output rows of `cin_p` bf16 channels.  widen:
// source row r holds `cin` channels at src + r * cin.  fold (x only): output
// pixel (n, h, u) of width Wf holds x[n][h][u - pad_w + s][ci] in channel
// s * cin + ci (zero outside the image and past kw * cin); inside the image
// those values are the contiguous run of the input row starting at element
// (u - pad_w) * cin, so channel c is element t0 + c, valid while
// 0 <= t0 + c < W * cin.
struct PrepJob {
    const void *src;
    __nv_bfloat16 *dst;
    long long rows;
    int cin, cin_p;
    int fold, W, Wf, kw, pad_w;
};

template <typename Tin>
__device__ __forceinline__ float load_f(const Tin *p) {
    if constexpr (sizeof(Tin) == 1)
        return (float)__ldg(p);
    else
        return __bfloat162float(__ldg(p));
}

// One thread per 8-channel group of an output row: reads up to 8 source
// values, writes 16 bytes.  Idx is uint32_t when every index fits (cheaper
// division), else uint64_t.
template <typename Tin, typename Idx>
__device__ __forceinline__ void prep_one(const PrepJob &j, Idx i) {
    const Idx groups = (Idx)(j.cin_p >> 3);
    const Idx row = i / groups;
    const int c0 = (int)(i - row * groups) * 8;
    const Tin *src = reinterpret_cast<const Tin *>(j.src);
    float v[8];
    if (j.fold) {
        const Idx nh = row / (Idx)j.Wf;
        const int u = (int)(row - nh * (Idx)j.Wf);
        const Tin *xrow = src + (long long)nh * j.W * j.cin;  // input row (n, h)
        const int t0 = (u - j.pad_w) * j.cin + c0;
        const int tend = j.W * j.cin, cend = j.kw * j.cin;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int t = t0 + e;
            v[e] = (c0 + e < cend && t >= 0 && t < tend) ? load_f(xrow + t) : 0.0f;
        }
    } else {
        const Tin *s = src + (long long)row * j.cin + c0;
        if (c0 + 8 <= j.cin && (j.cin % 8) == 0) {
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
            for (int e = 0; e < 8; ++e) v[e] = c0 + e < j.cin ? load_f(s + e) : 0.0f;  // padding channel: 0
        }
    }
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);  // exact for int8 and bf16 inputs
        out[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(j.dst + (long long)row * j.cin_p + c0) = make_uint4(out[0], out[1], out[2], out[3]);
}

// Both operands in one launch: threads [0, nx) prepare x, the rest w.
template <typename Tin, typename Idx>
__global__ void __launch_bounds__(kThreads) prep_kernel(const PrepJob jx, const PrepJob jw, Idx nx, Idx nw) {
    convk::pdl_trigger();
    convk::pdl_wait();
    const Idx i = (Idx)blockIdx.x * kThreads + threadIdx.x;
    if (i < nx)
        prep_one<Tin, Idx>(jx, i);
    else if (i - nx < nw)
        prep_one<Tin, Idx>(jw, i - nx);
}

template <typename Tin>
cudaError_t prep(const PrepJob &jx, const PrepJob &jw, cudaStream_t st) {
    const long long nx = jx.rows * (jx.cin_p / 8), nw = jw.rows * (jw.cin_p / 8);
    const long long n = nx + nw;
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + kThreads - 1) / kThreads);
    PrepJob a = jx, b = jw;
    if (n + kThreads < (1ll << 32)) {
        uint32_t ux = (uint32_t)nx, uw = (uint32_t)nw;
        void *args[] = {&a, &b, &ux, &uw};
        return conv_launch((const void *)&prep_kernel<Tin, uint32_t>, dim3(blocks), dim3(kThreads), args, 0, st);
    }
    uint64_t ux = (uint64_t)nx, uw = (uint64_t)nw;
    void *args[] = {&a, &b, &ux, &uw};
    return conv_launch((const void *)&prep_kernel<Tin, uint64_t>, dim3(blocks), dim3(kThreads), args, 0, st);
}

}  // namespace

cudaError_t launch_prep(const conv_plan *p, const void *x, const void *w, cudaStream_t st) {
    const IgemmGeom &g = p->ig;
    PrepJob jx = {}, jw = {};
    jx.src = x; jx.dst = p->d_xprep; jx.cin_p = p->cin_p;
    jw.src = w; jw.dst = p->d_wprep; jw.cin_p = p->cin_p;
    if (g.fold) {
        // x: (n, h, u) pixels of width g.wx; w: the OHWI rows of one (co, r)
        // already hold (s, ci) contiguously, i.e. the folded channel order.
        jx.rows = (long long)p->s.n * p->s.h * g.wx;
        jx.cin = p->s.c_in; jx.fold = 1; jx.W = p->s.w; jx.Wf = g.wx; jx.kw = p->s.k_w; jx.pad_w = p->pad_w;
        jw.rows = (long long)p->s.c_out * p->s.k_h;
        jw.cin = p->s.k_w * p->s.c_in;
    } else {
        jx.rows = (long long)p->s.n * p->s.h * p->s.w;
        jx.cin = p->s.c_in;
        jw.rows = (long long)p->s.c_out * p->s.k_h * p->s.k_w;
        jw.cin = p->s.c_in;
    }
    return p->dtype == CONV_I8 ? prep<int8_t>(jx, jw, st) : prep<__nv_bfloat16>(jx, jw, st);
}
