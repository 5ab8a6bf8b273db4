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
    OutMap om;  // output placement and residual
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
direct_conv_float(DirectArgs a, const T *__restrict__ x, const T *__restrict__ w,
                  const float *__restrict__ bias, T *__restrict__ y) {
    pdl_trigger();  // see conv_launch
    pdl_wait();
    const T *res = reinterpret_cast<const T *>(a.om.res);
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
    T *yp = y + a.om.base(n, oh, ow) + co0;
#pragma unroll
    for (int i = 0; i < kCot; ++i) {
        if (i < nco) {
            float v = activate(acc[i] + (bias ? __ldg(bias + co0 + i) : 0.0f), a.act);
            if (res) v += Elem<T>::to_f(__ldg(res + pix * a.Cout + co0 + i));  // residual after the activation
            const T o = Elem<T>::from_f(v);
            for (int dy = 0; dy < a.om.up; ++dy)
                for (int dx = 0; dx < a.om.up; ++dx) yp[a.om.rep(dy, dx) + i] = o;
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
    pdl_trigger();  // see conv_launch
    pdl_wait();
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
    int8_t *yp = y + a.om.base(n, oh, ow) + co0;
#pragma unroll
    for (int i = 0; i < kCot; ++i) {
        if (i < nco) {
            long long v = (long long)acc[i] + (bias ? (long long)__ldg(bias + co0 + i) : 0ll);
            const int8_t q = (int8_t)requant_i8(v, __ldg(mult + co0 + i), a.act);
            for (int dy = 0; dy < a.om.up; ++dy)
                for (int dx = 0; dx < a.om.up; ++dx) yp[a.om.rep(dy, dx) + i] = q;
        }
    }
}

// ---------------------------------------------------------------------------
// Direct convolution with the weights staged in shared memory (fp32 / bf16).
// A CTA owns one chunk of CT output channels of one group and 128 * PT
// output pixels; its weights are staged once as fp32 [K][CT] (K = k_h * k_w
// * Cin/groups).  A thread owns PT pixels x CT channels: per reduction step
// it loads one input value per pixel and reads the CT weights as shared-
// memory broadcasts (every thread of the CTA reads the same row), then issues
// CT FMAs per pixel.  Used for layers the tensor-core path
// does not take: fp32 layers, Cin = 1 or 3 stems, grouped layers.
constexpr int kDThreads = 128;
constexpr int kDMaxSmemFloats = 12288;  // 48 KB of staged weights

template <typename T> struct Out;
template <> struct Out<float> {
    __device__ static __forceinline__ float act(float v, int a) { return activate(v, a); }
};
template <> struct Out<__nv_bfloat16> {
    __device__ static __forceinline__ float act(float v, int a) { return activate_fast(v, a); }
};

template <typename T, int CT, int PT>
__global__ void __launch_bounds__(kDThreads)
direct_conv_smem(DirectArgs a, int chunks_per_group, const T *__restrict__ x, const T *__restrict__ w,
                 const float *__restrict__ bias, T *__restrict__ y) {
    pdl_trigger();  // see conv_launch
    extern __shared__ __align__(16) float wsm[];  // [K][CT]
    const int K = a.KH * a.KW * a.cin_g;
    const int g = blockIdx.y / chunks_per_group;
    const int cc = blockIdx.y - g * chunks_per_group;
    const int co0 = g * a.cout_g + cc * CT;
    const int nco = min(CT, a.cout_g - cc * CT);
    // Before waiting for the previous kernel: this chunk's weight rows (nco
    // rows of K contiguous elements) into L2, 128 bytes a thread-step.  L2 is
    // where global writes land, so this cannot serve stale bytes to the loads
    // after the wait.
    {
        const char *wb = reinterpret_cast<const char *>(w + (long long)co0 * K);
        const long long nbytes = (long long)nco * K * sizeof(T);
        for (long long o = (long long)threadIdx.x * 128; o < nbytes; o += 128LL * kDThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(wb + o));
    }
    pdl_wait();
    // Stage this chunk's weights as [K][CT]: consecutive threads write
    // consecutive channels of one k (no bank conflicts); the strided global
    // reads hit the same few lines of w for all threads of a warp.  Done once
    // the first batch of input loads (below) is in flight, so that the two
    // latencies overlap.
    auto stage_weights = [&]() {
        for (int i = threadIdx.x; i < K * CT; i += kDThreads) {
            const int k = i / CT, j = i - k * CT;
            wsm[i] = j < nco ? Elem<T>::to_f(__ldg(w + (long long)(co0 + j) * K + k)) : 0.0f;
        }
        __syncthreads();
    };

    const int g0 = g * a.cin_g;
    // fp32 rows that start on 16-byte boundaries: vector loads of the channels
    const bool vec4 = sizeof(T) == 4 && (a.Cin % 4) == 0 && (g0 % 4) == 0 && (a.cin_g % 8) == 0;
    long long pix[PT];
    int ihb[PT], iwb[PT], nn[PT];
    bool pv[PT];
#pragma unroll
    for (int i = 0; i < PT; ++i) {
        pix[i] = ((long long)blockIdx.x * PT + i) * kDThreads + threadIdx.x;
        pv[i] = pix[i] < a.npix;
        const long long pp = pv[i] ? pix[i] : 0;
        const int ow = (int)(pp % a.OW);
        const long long t = pp / a.OW;
        const int oh = (int)(t % a.OH);
        nn[i] = (int)(t / a.OH);
        ihb[i] = oh * a.stride - a.pad_h;
        iwb[i] = ow * a.stride - a.pad_w;
    }
    float acc[PT][CT];
#pragma unroll
    for (int i = 0; i < PT; ++i)
#pragma unroll
        for (int j = 0; j < CT; ++j) acc[i][j] = 0.0f;

    auto fma_k = [&](const float (&xv)[PT], const float *wr) {
#pragma unroll
        for (int j = 0; j < CT; j += 4) {
            const float4 w4 = *reinterpret_cast<const float4 *>(wr + j);
#pragma unroll
            for (int i = 0; i < PT; ++i) {
                acc[i][j] = __fmaf_rn(xv[i], w4.x, acc[i][j]);
                acc[i][j + 1] = __fmaf_rn(xv[i], w4.y, acc[i][j + 1]);
                acc[i][j + 2] = __fmaf_rn(xv[i], w4.z, acc[i][j + 2]);
                acc[i][j + 3] = __fmaf_rn(xv[i], w4.w, acc[i][j + 3]);
            }
        }
    };
    // The reduction index k = (r, s, ci) walks K in order (the staged
    // weights' row order) in batches whose input loads are all issued before
    // the batch's FMAs: the loads' latency is paid once per batch, not once
    // per tap.  fp32 rows that start on 16-byte boundaries load 4 channels
    // at a time (NB chunks a batch), others one value at a time (8 a batch).
    // (r, s, ci) advance incrementally: no division per value.
    int r = 0, s = 0, ci = 0;
    auto advance = [&](int step) {
        ci += step;
        if (ci == a.cin_g) {
            ci = 0;
            if (++s == a.KW) { s = 0; ++r; }
        }
    };
    auto src = [&](int i, bool &ok) {
        const int ih = ihb[i] + r, iw = iwb[i] + s;
        ok = pv[i] && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W;  // zero padding
        return x + (((long long)nn[i] * a.H + (ok ? ih : 0)) * a.W + (ok ? iw : 0)) * a.Cin + g0 + ci;
    };
    if (vec4) {
        constexpr int NB = PT == 1 ? 8 : 4;  // 4-channel chunks in flight per pixel
        for (int k0 = 0; k0 < K; k0 += 4 * NB) {
            float4 q[NB][PT];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const bool live = k0 + 4 * b < K;
#pragma unroll
                for (int i = 0; i < PT; ++i) {
                    bool ok = false;
                    const T *xp = live ? src(i, ok) : x;
                    q[b][i] = live && ok ? __ldg(reinterpret_cast<const float4 *>(xp)) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (live) advance(4);
            }
            if (k0 == 0) stage_weights();  // (every thread: K is the same for all)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (k0 + 4 * b >= K) break;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float xv[PT];
#pragma unroll
                    for (int i = 0; i < PT; ++i)
                        xv[i] = e == 0 ? q[b][i].x : (e == 1 ? q[b][i].y : (e == 2 ? q[b][i].z : q[b][i].w));
                    fma_k(xv, wsm + (k0 + 4 * b + e) * CT);
                }
            }
        }
    } else {
        constexpr int NB = 8;  // values in flight per pixel
        for (int k0 = 0; k0 < K; k0 += NB) {
            float v[NB][PT];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const bool live = k0 + b < K;
#pragma unroll
                for (int i = 0; i < PT; ++i) {
                    bool ok = false;
                    const T *xp = live ? src(i, ok) : x;
                    v[b][i] = live && ok ? Elem<T>::to_f(__ldg(xp)) : 0.0f;
                }
                if (live) advance(1);
            }
            if (k0 == 0) stage_weights();  // (every thread: K is the same for all)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (k0 + b >= K) break;
                fma_k(v[b], wsm + (k0 + b) * CT);
            }
        }
    }
    const T *res = reinterpret_cast<const T *>(a.om.res);
#pragma unroll
    for (int i = 0; i < PT; ++i) {
        if (!pv[i]) continue;
        long long yb = pix[i] * a.Cout;
        if (!a.om.plain()) {
            const int ow = (int)(pix[i] % a.OW);
            const long long t = pix[i] / a.OW;
            yb = a.om.base((int)(t / a.OH), (int)(t % a.OH), ow);
        }
        T out[CT];
#pragma unroll
        for (int j = 0; j < CT; ++j) {
            float v = Out<T>::act(acc[i][j] + (bias && j < nco ? __ldg(bias + co0 + j) : 0.0f), a.act);
            if (res && j < nco) v += Elem<T>::to_f(__ldg(res + pix[i] * a.Cout + co0 + j));  // after the activation
            out[j] = Elem<T>::from_f(v);
        }
        for (int dy = 0; dy < a.om.up; ++dy)
            for (int dx = 0; dx < a.om.up; ++dx) {
                T *yp = y + yb + a.om.rep(dy, dx) + co0;
                const bool vec =
                    nco == CT && ((reinterpret_cast<uintptr_t>(yp) & 15) == 0) && (CT * sizeof(T)) % 16 == 0;
                if (vec) {
#pragma unroll
                    for (int j = 0; j < CT; j += 16 / (int)sizeof(T))
                        *reinterpret_cast<uint4 *>(yp + j) = *reinterpret_cast<const uint4 *>(out + j);
                } else {
#pragma unroll
                    for (int j = 0; j < CT; ++j)
                        if (j < nco) yp[j] = out[j];
                }
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
    a.om.Cout = p->s.c_out; a.om.OH = p->oh; a.om.OW = p->ow;
    a.om.Cy = p->up ? p->y_c : p->s.c_out;  // (up == 0: a plan struct without output options)
    a.om.c_off = p->up ? p->y_coff : 0;
    a.om.up = p->up ? p->up : 1;
    a.om.res = nullptr;
    return a;
}

template <typename T, int CT>
void *smem_kernel_pt(int pt) {
    return pt == 2 ? reinterpret_cast<void *>(&direct_conv_smem<T, CT, 2>)
                   : reinterpret_cast<void *>(&direct_conv_smem<T, CT, 1>);
}

template <typename T>
void *smem_kernel(int ct, int pt) {
    switch (ct) {
    case 32: return smem_kernel_pt<T, 32>(pt);
    case 16: return smem_kernel_pt<T, 16>(pt);
    case 8: return smem_kernel_pt<T, 8>(pt);
    default: return smem_kernel_pt<T, 4>(pt);
    }
}

template <typename T>
cudaError_t launch_smem(const conv_plan *p, DirectArgs a, const void *x, const void *w, const void *bias, void *y,
                        cudaStream_t st) {  // a.om carries the residual
    const int ct = p->dct, pt = p->dpt;
    const int chunks = (a.cout_g + ct - 1) / ct;
    const int K = a.KH * a.KW * a.cin_g;
    dim3 grid((unsigned)((a.npix + (long long)kDThreads * pt - 1) / ((long long)kDThreads * pt)),
              (unsigned)(p->groups * chunks));
    void *k = smem_kernel<T>(ct, pt);
    void *args[] = {&a, (void *)&chunks, (void *)&x, (void *)&w, (void *)&bias, &y};
    return conv_launch(k, grid, dim3(kDThreads), args, (size_t)K * ct * sizeof(float), st);
}

}  // namespace

void direct_configure(conv_plan *p) {
    // Shared-memory variant for float layers whose staged weights fit: the
    // widest channel chunk (<= 32, covering the group) whose K x CT floats fit.
    p->dct = 0;
    p->dpt = 1;
    if (p->dtype == CONV_I8) return;
    const int cout_g = p->s.c_out / p->groups;
    const long long K = (long long)p->s.k_h * p->s.k_w * (p->s.c_in / p->groups);
    int ct = 32;
    while (ct > 4 && ct / 2 >= cout_g) ct /= 2;  // no wider than the group needs
    while (ct >= 4 && K * ct > kDMaxSmemFloats) ct /= 2;
    if (ct < 4) return;
    const long long npix = (long long)p->s.n * p->oh * p->ow;
    // Small layers: narrower chunks until the grid has a few CTAs per SM.
    while (ct > 4 && ((npix + kDThreads - 1) / kDThreads) * p->groups * ((cout_g + ct - 1) / ct) <
                         (long long)p->num_sms * 4)
        ct /= 2;
    const long long chunks = (long long)p->groups * ((cout_g + ct - 1) / ct);
    if (chunks > 65535) return;
    p->dct = ct;
    // Two pixels per thread when there are threads to spare: weight rows are
    // then read once for two pixels.
    p->dpt = npix * chunks >= (long long)p->num_sms * kDThreads * 16 ? 2 : 1;
}

bool direct_supported(const conv_plan *p) {
    const int cout_g = p->s.c_out / p->groups;
    const long long chunks = (long long)p->groups * ((cout_g + kCot - 1) / kCot);
    const long long blocks = ((long long)p->s.n * p->oh * p->ow + kThreads - 1) / kThreads;
    return chunks <= 65535 && blocks <= 0x7fffffffll;
}

cudaError_t launch_direct(const conv_plan *p, const void *x, const void *w, const void *bias,
                          const void *res, void *y, cudaStream_t st) {
    DirectArgs a = make_args(p);
    a.om.res = res;
    dim3 grid((unsigned)((a.npix + kThreads - 1) / kThreads), (unsigned)(p->groups * a.chunks_per_group));
    const float *mult = p->d_mult;
    switch (p->dtype) {
    case CONV_F32: {
        if (p->dct > 0) return launch_smem<float>(p, a, x, w, bias, y, st);
        void *args[] = {&a, (void *)&x, (void *)&w, (void *)&bias, &y};
        return conv_launch((const void *)&direct_conv_float<float>, grid, dim3(kThreads), args, 0, st);
    }
    case CONV_BF16: {
        if (p->dct > 0) return launch_smem<__nv_bfloat16>(p, a, x, w, bias, y, st);
        void *args[] = {&a, (void *)&x, (void *)&w, (void *)&bias, &y};
        return conv_launch((const void *)&direct_conv_float<__nv_bfloat16>, grid, dim3(kThreads), args, 0, st);
    }
    default: {
        void *args[] = {&a, (void *)&x, (void *)&w, (void *)&bias, (void *)&mult, &y};
        const void *k = a.cin_g % 4 == 0 ? (const void *)&direct_conv_i8<true> : (const void *)&direct_conv_i8<false>;
        return conv_launch(k, grid, dim3(kThreads), args, 0, st);
    }
    }
}
