// Fused depthwise-separable pair (the DS-CNN block): a depthwise 3x3
// convolution followed by a 1x1 pointwise convolution in one kernel, the
// intermediate kept in shared memory ("nanoinfer", "What is still slow":
// depthwise convolution is the gap, and each extra layer boundary is another
// trip through memory; "YOLOv4, optimized for Wormhole", section 9, K2:
// keep the intermediate on core).
//
//   z[p, c]  = round_T( act_dw( b_dw[c] + sum_{r,s} x[..] * w_dw[c, r, s] ) )
//   y[p, co] = act_pw( b_pw[co] + sum_c z[p, c] * w_pw[co, c] )
//
// round_T rounds z to the layer's type (bf16 round-to-nearest-even; nothing
// for fp32): the pair computes what the two layers run one after the other
// compute, without writing or reading z.
//
// A CTA owns a th x tw tile of output pixels and a chunk of co_chunk output
// channels.  It stages the tile's input halo (all C channels, zeros outside
// the image) in shared memory, computes the depthwise outputs of the tile
// for all C channels into shared memory (rows padded by one float so that
// threads on different pixels read different banks), stages its chunk of
// the pointwise weights transposed to [c][co], and contracts: a thread owns
// one pixel x 4 output channels and walks the C channels with one
// shared-memory broadcast of 4 weights and one z value per step.  fp32
// arithmetic on the CUDA cores (FFMA, never TF32) for both the fp32 and the
// bf16 layer type; the contraction is K = C long and is meant for the
// channel counts of depthwise-separable blocks (C <= 512).
#include <cuda_bf16.h>
#include <stdint.h>

#include "conv_internal.h"
#include "epilogue.cuh"

using namespace convk;

namespace {

constexpr int kThreads = 256;

struct DwpwArgs {
    int N, H, W, C, Cout, OH, OW, stride, pad;
    int th, tw, hin, win, cochunk, tiles_w, tiles_h, zp;  // zp: z row pitch in floats (C + 1)
    int act_dw, act_pw;
};

template <typename T>
__device__ __forceinline__ float act_of(float v, int act) {
    if constexpr (sizeof(T) == 4)
        return activate(v, act);  // fp32 outputs: IEEE expf / division
    else
        return activate_fast(v, act);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) dwpw_kernel(const T *__restrict__ x, const T *__restrict__ wdw,
                                                        const float *__restrict__ bdw, const T *__restrict__ wpw,
                                                        const float *__restrict__ bpw, T *__restrict__ y,
                                                        const DwpwArgs a) {
    pdl_trigger();  // see conv_launch
    pdl_wait();
    extern __shared__ __align__(16) float sm[];
    float *xs = sm;                                   // [hin][win][C]
    float *zs = xs + a.hin * a.win * a.C;             // [th*tw][zp]
    float *ws = zs + ((a.th * a.tw * a.zp + 3) & ~3);  // [C][cochunk], 16-byte aligned
    int t = blockIdx.x;
    const int tw_ = t % a.tiles_w;
    t /= a.tiles_w;
    const int oh0 = (t % a.tiles_h) * a.th;
    const int n = t / a.tiles_h;
    const int ow0 = tw_ * a.tw;
    const int co0 = blockIdx.y * a.cochunk;
    const int ih0 = oh0 * a.stride - a.pad, iw0 = ow0 * a.stride - a.pad;

    // 1. input halo, channels fastest (coalesced), zero outside the image
    for (int e = threadIdx.x; e < a.hin * a.win * a.C; e += kThreads) {
        const int c = e % a.C;
        const int pw_ = (e / a.C) % a.win;
        const int ph = e / (a.C * a.win);
        const int ih = ih0 + ph, iw = iw0 + pw_;
        float v = 0.0f;
        if (ih >= 0 && ih < a.H && iw >= 0 && iw < a.W)
            v = Elem<T>::to_f(__ldg(x + (((long long)n * a.H + ih) * a.W + iw) * a.C + c));
        xs[e] = v;
    }
    // pointwise weight chunk, transposed to [c][co]
    for (int e = threadIdx.x; e < a.C * a.cochunk; e += kThreads) {
        const int j = e % a.cochunk, c = e / a.cochunk;
        ws[e] = co0 + j < a.Cout ? Elem<T>::to_f(__ldg(wpw + (long long)(co0 + j) * a.C + c)) : 0.0f;
    }
    __syncthreads();

    // 2. depthwise outputs of the tile for every channel, rounded to T
    for (int e = threadIdx.x; e < a.th * a.tw * a.C; e += kThreads) {
        const int c = e % a.C;
        const int p = e / a.C;
        const int dh = p / a.tw, dw = p % a.tw;
        const float *xb = xs + ((dh * a.stride) * a.win + dw * a.stride) * a.C + c;
        const T *wc = wdw + (long long)c * 9;
        float acc = bdw ? __ldg(bdw + c) : 0.0f;
#pragma unroll
        for (int r = 0; r < 3; ++r)
#pragma unroll
            for (int s = 0; s < 3; ++s) acc = __fmaf_rn(xb[(r * a.win + s) * a.C], Elem<T>::to_f(__ldg(wc + r * 3 + s)), acc);
        zs[p * a.zp + c] = Elem<T>::to_f(Elem<T>::from_f(act_of<T>(acc, a.act_dw)));
    }
    __syncthreads();

    // 3. pointwise: a thread per (pixel, 4 output channels) of the chunk
    const int groups = a.cochunk / 4;
    for (int e = threadIdx.x; e < a.th * a.tw * groups; e += kThreads) {
        const int g = e % groups;
        const int p = e / groups;
        const int dh = p / a.tw, dw = p % a.tw;
        const int oh = oh0 + dh, ow = ow0 + dw;
        const float *zr = zs + p * a.zp;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < a.C; ++c) {
            const float zv = zr[c];
            const float4 w4 = *reinterpret_cast<const float4 *>(ws + c * a.cochunk + 4 * g);
            acc.x = __fmaf_rn(zv, w4.x, acc.x);
            acc.y = __fmaf_rn(zv, w4.y, acc.y);
            acc.z = __fmaf_rn(zv, w4.z, acc.z);
            acc.w = __fmaf_rn(zv, w4.w, acc.w);
        }
        if (oh >= a.OH || ow >= a.OW) continue;
        const int co = co0 + 4 * g;
        T *yp = y + (((long long)n * a.OH + oh) * a.OW + ow) * a.Cout + co;
        const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (co + j < a.Cout) yp[j] = Elem<T>::from_f(act_of<T>(v[j] + (bpw ? __ldg(bpw + co + j) : 0.0f), a.act_pw));
    }
}

// shared-memory floats of a configuration
long long smem_floats(int C, int th, int tw, int stride, int cochunk) {
    const long long hin = (long long)(th - 1) * stride + 3, win = (long long)(tw - 1) * stride + 3;
    return hin * win * C + (((long long)th * tw * (C + 1) + 3) & ~3ll) + (long long)C * cochunk;
}

}  // namespace

bool dwpw_supported(const conv_plan *p) {
    return (p->dtype == CONV_F32 || p->dtype == CONV_BF16) && p->s.c_in <= 512 && p->stride <= 4;
}

// Tile: the largest th x tw (<= 8 x 8) and co chunk (<= 64, a multiple of 4)
// whose shared memory fits twice per SM, preferring enough CTAs to cover the
// SMs (small layers split the output channels further).
int dwpw_configure(conv_plan *p) {
    DwpwGeom &g = p->dwpw;
    const int C = p->s.c_in, S = p->stride;
    const long long cap = 110 * 1024 / 4;  // floats: two CTAs per SM
    long long best = -1;
    for (int th : {8, 4, 2, 1})
        for (int tw : {8, 4, 2, 1})
            for (int cc : {64, 32, 16, 8, 4}) {
                if (smem_floats(C, th, tw, S, cc) > cap) continue;
                const long long tiles = (long long)((p->oh + th - 1) / th) * ((p->ow + tw - 1) / tw) * p->s.n;
                const long long chunks = (p->s.c_out + cc - 1) / cc;
                const long long ctas = tiles * chunks;
                if (chunks > 65535 || tiles > 0x7fffffffll) continue;
                // work per CTA ~ pixels x (9 C + C x cc) + halo loads; prefer >= 2 CTAs per SM
                const long long per = (long long)th * tw * (9LL * C + (long long)C * cc) +
                                      ((long long)(th - 1) * S + 3) * ((tw - 1) * S + 3) * C;
                const long long waves = (ctas + 2LL * p->num_sms - 1) / (2LL * p->num_sms);
                const long long cost = waves * per + (ctas < p->num_sms ? per * 4 : 0);
                if (best < 0 || cost < best) {
                    best = cost;
                    g.th = th; g.tw = tw; g.cochunk = cc;
                    g.tiles_w = (p->ow + tw - 1) / tw;
                    g.tiles_h = (p->oh + th - 1) / th;
                    g.chunks = (int)chunks;
                }
            }
    if (best < 0) return CONV_ERR_UNSUPPORTED;
    g.hin = (g.th - 1) * S + 3;
    g.win = (g.tw - 1) * S + 3;
    g.smem = (int)(smem_floats(C, g.th, g.tw, S, g.cochunk) * 4);
    const void *k = p->dtype == CONV_F32 ? (const void *)&dwpw_kernel<float> : (const void *)&dwpw_kernel<__nv_bfloat16>;
    return conv_grant_smem(k, p->device, g.smem);
}

cudaError_t launch_dwpw(const conv_plan *p, const void *x, const void *wdw, const void *bdw, const void *wpw,
                        const void *bpw, void *y, cudaStream_t st) {
    const DwpwGeom &g = p->dwpw;
    DwpwArgs a;
    a.N = p->s.n; a.H = p->s.h; a.W = p->s.w; a.C = p->s.c_in; a.Cout = p->s.c_out;
    a.OH = p->oh; a.OW = p->ow; a.stride = p->stride; a.pad = p->pad_h;
    a.th = g.th; a.tw = g.tw; a.hin = g.hin; a.win = g.win; a.cochunk = g.cochunk;
    a.tiles_w = g.tiles_w; a.tiles_h = g.tiles_h; a.zp = p->s.c_in + 1;
    a.act_dw = (int)p->act; a.act_pw = (int)p->act2;
    dim3 grid((unsigned)((long long)g.tiles_w * g.tiles_h * p->s.n), (unsigned)g.chunks);
    void *args[] = {(void *)&x, (void *)&wdw, (void *)&bdw, (void *)&wpw, (void *)&bpw, &y, &a};
    const void *k = p->dtype == CONV_F32 ? (const void *)&dwpw_kernel<float> : (const void *)&dwpw_kernel<__nv_bfloat16>;
    return conv_launch(k, grid, dim3(kThreads), args, (size_t)g.smem, st);
}
