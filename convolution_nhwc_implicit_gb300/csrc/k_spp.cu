// SPP block of YOLOv4: max pools of 5x5, 9x9 and 13x13 windows, stride 1,
// output the size of the input, positions outside the image never winning
// the max ("YOLOv4, optimized for Wormhole", section 9, K3: one kernel
// builds the 5, 9 and 13 windows from cascaded smaller windows).
//
// The cascade: a 9x9 max is a 5x5 max of 5x5 maxima and a 13x13 max a 5x5
// max of those (windows of odd sizes a and b compose into a + b - 1), and a
// 5x5 max is a 1x5 max of 5x1 maxima.  So a CTA loads its tile of output
// pixels with a 6-pixel halo once into shared memory (minus infinity outside
// the image) and applies six 1-D 5-wide max passes, each shrinking the region
// by 4 along one axis, writing the 5x5, 9x9 and 13x13 results of its tile as
// they appear.  Each pooled map, and x itself if asked, goes to its own
// channel slice of y, the next layer's concatenated NHWC buffer (K4's
// "write into the next layer's layout").  Max is exact in every type, so the
// result is bit-identical to a direct evaluation of each window.
#include <cuda_bf16.h>
#include <stdint.h>

#include "conv_internal.h"
#include "epilogue.cuh"

using namespace convk;

namespace {

// Elementwise max of two 16-byte vectors, and the vector that never wins.
template <typename T> struct VMax;
template <> struct VMax<float> {
    static constexpr uint32_t kNeg = 0xff800000u;  // -inf
    __device__ static __forceinline__ uint4 max(uint4 a, uint4 b) {
        return make_uint4(__float_as_uint(fmaxf(__uint_as_float(a.x), __uint_as_float(b.x))),
                          __float_as_uint(fmaxf(__uint_as_float(a.y), __uint_as_float(b.y))),
                          __float_as_uint(fmaxf(__uint_as_float(a.z), __uint_as_float(b.z))),
                          __float_as_uint(fmaxf(__uint_as_float(a.w), __uint_as_float(b.w))));
    }
};
template <> struct VMax<__nv_bfloat16> {
    static constexpr uint32_t kNeg = 0xff80ff80u;  // two bf16 -inf
    __device__ static __forceinline__ uint32_t m2(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    __device__ static __forceinline__ uint4 max(uint4 a, uint4 b) {
        return make_uint4(m2(a.x, b.x), m2(a.y, b.y), m2(a.z, b.z), m2(a.w, b.w));
    }
};
template <> struct VMax<int8_t> {
    static constexpr uint32_t kNeg = 0x80808080u;  // four int8 -128
    __device__ static __forceinline__ uint4 max(uint4 a, uint4 b) {
        return make_uint4(__vmaxs4(a.x, b.x), __vmaxs4(a.y, b.y), __vmaxs4(a.z, b.z), __vmaxs4(a.w, b.w));
    }
};

constexpr int kTH = 8, kTW = 8;  // output tile
constexpr int kHalo = 6;         // (13 - 1) / 2
constexpr int kP = kTW + 2 * kHalo;  // row pitch (pixels) of the shared buffers
constexpr int kR = kTH + 2 * kHalo;
constexpr int kThreads = 256;
constexpr int kImgPer = 12;  // whole-image kernel: elements per thread (2 x 12 x 256 x 16 B = 96 KB)

struct SppArgs {
    int N, H, W, CV;       // CV: 16-byte channel vectors per pixel of x
    int cbv;               // channel vectors per CTA
    int tiles_w, tiles_h;
    int Cy;                // 16-byte vectors per pixel of y
    int off[4];            // vector offset in y of mp5, mp9, mp13, x (-1: not written)
};

// One 5-wide max pass along rows (dir 0) or columns (dir 1) over a region of
// rows x cols output pixels: dst[r][c] = max_{d<5} src[r + d*dir][c + d*(1-dir)].
template <typename T>
__device__ __forceinline__ void pass5(const uint4 *src, uint4 *dst, int rows, int cols, int cbv, int dir) {
    const int n = rows * cols * cbv;
    const int step = (dir ? kP : 1) * cbv;
    for (int e = threadIdx.x; e < n; e += kThreads) {
        const int cv = e % cbv;
        const int pc = e / cbv;
        const int r = pc / cols, c = pc % cols;
        const uint4 *s = src + (r * kP + c) * cbv + cv;
        uint4 m = s[0];
#pragma unroll
        for (int d = 1; d < 5; ++d) m = VMax<T>::max(m, s[d * step]);
        dst[(r * kP + c) * cbv + cv] = m;
    }
}

// Writes the tile's part of a pooled region (origin: the buffer position of
// output pixel (h0, w0)) to its slice of y.
__device__ __forceinline__ void store_tile(const uint4 *buf, int org, uint4 *y, const SppArgs &a, int n, int h0, int w0,
                                           int cv0, int slot) {
    if (a.off[slot] < 0) return;
    const int n_el = kTH * kTW * a.cbv;
    for (int e = threadIdx.x; e < n_el; e += kThreads) {
        const int cv = e % a.cbv;
        const int pc = e / a.cbv;
        const int r = pc / kTW, c = pc % kTW;
        const int h = h0 + r, w = w0 + c;
        if (h >= a.H || w >= a.W || cv0 + cv >= a.CV) continue;
        y[(((long long)n * a.H + h) * a.W + w) * a.Cy + a.off[slot] + cv0 + cv] = buf[org + (r * kP + c) * a.cbv + cv];
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) spp_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ y,
                                                       const SppArgs a) {
    pdl_trigger();  // see conv_launch
    pdl_wait();
    extern __shared__ __align__(16) uint4 sm[];
    uint4 *A = sm;
    uint4 *B = sm + kR * kP * a.cbv;
    int t = blockIdx.x;
    const int tw = t % a.tiles_w;
    t /= a.tiles_w;
    const int th = t % a.tiles_h;
    const int n = t / a.tiles_h;
    const int h0 = th * kTH, w0 = tw * kTW;
    const int cv0 = blockIdx.y * a.cbv;
    const uint4 neg = make_uint4(VMax<T>::kNeg, VMax<T>::kNeg, VMax<T>::kNeg, VMax<T>::kNeg);

    // halo of x (kR x kP pixels around the tile), -inf outside the image
    for (int e = threadIdx.x; e < kR * kP * a.cbv; e += kThreads) {
        const int cv = e % a.cbv;
        const int pc = e / a.cbv;
        const int r = pc / kP, c = pc % kP;
        const int h = h0 - kHalo + r, w = w0 - kHalo + c;
        uint4 v = neg;
        if (h >= 0 && h < a.H && w >= 0 && w < a.W && cv0 + cv < a.CV)
            v = __ldg(x + (((long long)n * a.H + h) * a.W + w) * a.CV + cv0 + cv);
        A[e] = v;
    }
    __syncthreads();
    store_tile(A, (kHalo * kP + kHalo) * a.cbv, y, a, n, h0, w0, cv0, 3);  // x itself
    // 5x5: rows kR, cols kP-4 -> rows kR-4, cols kP-4 (origin of the tile: (4, 4))
    pass5<T>(A, B, kR, kP - 4, a.cbv, 0);
    __syncthreads();
    pass5<T>(B, A, kR - 4, kP - 4, a.cbv, 1);
    __syncthreads();
    store_tile(A, (4 * kP + 4) * a.cbv, y, a, n, h0, w0, cv0, 0);
    // 9x9 = 5x5 of the 5x5 maxima: region shrinks to (kR-8) x (kP-8), tile at (2, 2)
    pass5<T>(A, B, kR - 4, kP - 8, a.cbv, 0);
    __syncthreads();
    pass5<T>(B, A, kR - 8, kP - 8, a.cbv, 1);
    __syncthreads();
    store_tile(A, (2 * kP + 2) * a.cbv, y, a, n, h0, w0, cv0, 1);
    // 13x13: region (kR-12) x (kP-12) = the tile itself
    pass5<T>(A, B, kR - 8, kP - 12, a.cbv, 0);
    __syncthreads();
    pass5<T>(B, A, kR - 12, kP - 12, a.cbv, 1);
    __syncthreads();
    store_tile(A, 0, y, a, n, h0, w0, cv0, 2);
}

// Whole-image variant, for images whose (H + 4) x (W + 4) x cbv vectors fit
// in shared memory twice: a CTA owns one image and cbv channel vectors, so
// nothing is loaded or pooled twice (the tiled kernel above re-reads a
// 6-pixel halo around every 8x8 tile).  Both buffers carry a 2-pixel border
// of minus infinity that no pass writes, so every 5-wide max reads its five
// neighbours at fixed offsets: a window clipped at the image's edge is the
// padded window, and a 5-wide max of 5-wide maxima over padded windows is the
// 9-wide max over the padded window, so the cascade is unchanged.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2) spp_image_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ y,
                                                                const SppArgs a) {
    pdl_trigger();  // see conv_launch
    pdl_wait();
    extern __shared__ __align__(16) uint4 sm[];
    const int n = blockIdx.x;
    const int cv0 = blockIdx.y * a.cbv;
    const int np = a.H * a.W;
    const int nel = np * a.cbv;                          // interior elements
    const int pitch = (a.W + 4) * a.cbv;                 // vectors per padded row
    const int npad = (a.H + 4) * pitch;                  // vectors per padded buffer
    uint4 *A = sm;
    uint4 *B = sm + npad;
    const uint4 neg = make_uint4(VMax<T>::kNeg, VMax<T>::kNeg, VMax<T>::kNeg, VMax<T>::kNeg);
    const long long xbase = (long long)n * np;
    // This thread's interior elements e = threadIdx.x + k * kThreads (k <
    // kImgPer; the host keeps nel <= kImgPer * kThreads): their buffer index
    // and their pixel, found once.
    int eb[kImgPer], ep[kImgPer];
#pragma unroll
    for (int k = 0; k < kImgPer; ++k) {
        const int e = threadIdx.x + k * kThreads;
        const int p = e / a.cbv, cv = e - p * a.cbv;
        const int h = p / a.W, w = p - h * a.W;
        ep[k] = p;
        eb[k] = (h + 2) * pitch + (w + 2) * a.cbv + cv;
    }
    // the borders of both buffers: minus infinity
    for (int i = threadIdx.x; i < npad; i += kThreads) {
        const int r = i / pitch, c = i - r * pitch;
        if (r < 2 || r >= a.H + 2 || c < 2 * a.cbv || c >= (a.W + 2) * a.cbv) {
            A[i] = neg;
            B[i] = neg;
        }
    }
    // x -> A (and to its own slice of y, if asked)
#pragma unroll
    for (int k = 0; k < kImgPer; ++k) {
        const int e = threadIdx.x + k * kThreads;
        if (e >= nel) break;
        const int cv = e - ep[k] * a.cbv;
        const long long pix = xbase + ep[k];
        uint4 v = neg;
        if (cv0 + cv < a.CV) {
            v = __ldg(x + pix * a.CV + cv0 + cv);
            if (a.off[3] >= 0) y[pix * a.Cy + a.off[3] + cv0 + cv] = v;
        }
        A[eb[k]] = v;
    }
    __syncthreads();
    for (int level = 0; level < 3; ++level) {  // 5x5, 9x9, 13x13
        // along rows (A -> B), then along columns (B -> A)
#pragma unroll
        for (int k = 0; k < kImgPer; ++k) {
            const int e = threadIdx.x + k * kThreads;
            if (e >= nel) break;
            const uint4 *s = A + eb[k];
            uint4 m = VMax<T>::max(VMax<T>::max(s[-2 * a.cbv], s[-a.cbv]), VMax<T>::max(s[a.cbv], s[2 * a.cbv]));
            B[eb[k]] = VMax<T>::max(m, s[0]);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kImgPer; ++k) {
            const int e = threadIdx.x + k * kThreads;
            if (e >= nel) break;
            const uint4 *s = B + eb[k];
            uint4 m = VMax<T>::max(VMax<T>::max(s[-2 * pitch], s[-pitch]), VMax<T>::max(s[pitch], s[2 * pitch]));
            A[eb[k]] = VMax<T>::max(m, s[0]);
        }
        __syncthreads();
        if (a.off[level] >= 0) {
#pragma unroll
            for (int k = 0; k < kImgPer; ++k) {
                const int e = threadIdx.x + k * kThreads;
                if (e >= nel) break;
                const int cv = e - ep[k] * a.cbv;
                if (cv0 + cv < a.CV) y[(xbase + ep[k]) * a.Cy + a.off[level] + cv0 + cv] = A[eb[k]];
            }
        }
        // (the next level's row pass overwrites B only: A stays readable here)
    }
}

bool overlaps(const void *p, size_t np, const void *q, size_t nq) {
    const uintptr_t a0 = (uintptr_t)p, b0 = (uintptr_t)q;
    return np && nq && a0 < b0 + nq && b0 < a0 + np;
}

}  // namespace

extern "C" int conv_spp_run(int32_t n, int32_t h, int32_t w, int32_t c, conv_dtype_t dtype, const void *x, void *y,
                            int32_t y_channels, int32_t off5, int32_t off9, int32_t off13, int32_t off_x,
                            void *stream) {
    if ((int)dtype < CONV_F32 || (int)dtype > CONV_I8) return CONV_ERR_INVALID_ARG;
    if (n < 0 || h < 1 || w < 1 || c < 1 || y_channels < 1) return CONV_ERR_INVALID_SHAPE;
    const int es = conv_esize(dtype);
    if ((c * es) % 16 != 0 || (y_channels * es) % 16 != 0) return CONV_ERR_MISALIGNED;
    const int offs[4] = {off5, off9, off13, off_x};
    for (int i = 0; i < 4; ++i) {
        if (i < 3 && offs[i] < 0) return CONV_ERR_INVALID_ARG;  // the three pools are always written
        if (offs[i] < 0) continue;
        if ((offs[i] * es) % 16 != 0) return CONV_ERR_MISALIGNED;
        if ((long long)offs[i] + c > y_channels) return CONV_ERR_INVALID_ARG;
        for (int j = 0; j < i; ++j)  // slices must not overlap each other
            if (offs[j] >= 0 && offs[i] < offs[j] + c && offs[j] < offs[i] + c) return CONV_ERR_INVALID_ARG;
    }
    if ((long long)n * h * w >= (1ll << 31) || (long long)n * h * w * y_channels >= (1ll << 40))
        return CONV_ERR_UNSUPPORTED;
    if (n == 0) return CONV_OK;
    if (!x || !y) return CONV_ERR_NULL_ARG;
    if (((uintptr_t)x & 15) || ((uintptr_t)y & 15)) return CONV_ERR_MISALIGNED;
    if (overlaps(x, (size_t)n * h * w * c * es, y, (size_t)n * h * w * y_channels * es)) return CONV_ERR_ALIASING;

    SppArgs a;
    a.N = n; a.H = h; a.W = w; a.CV = c * es / 16;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV_ERR_CUDA;
    int num_sms = 0;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return CONV_ERR_CUDA;
    // Whole images when two padded copies of an image's channel block fit in
    // 96 KB: the fewest channel vectors per CTA that still give every SM two
    // CTAs.
    {
        const long long px = (long long)(h + 4) * (w + 4);
        int cbv = 0;
        for (int v = 1; v <= a.CV && v <= 16; v *= 2) {
            if (a.CV % v != 0 || 2 * px * v * 16 > 96 * 1024) break;
            cbv = v;
            if ((long long)n * (a.CV / v) <= 2LL * num_sms) break;
        }
        if (cbv > 0 && (long long)n * (a.CV / cbv) <= 0x7fffffffll && a.CV / cbv <= 65535) {
            a.cbv = cbv;
            a.tiles_w = a.tiles_h = 1;
            a.Cy = y_channels * es / 16;
            for (int i = 0; i < 4; ++i) a.off[i] = offs[i] < 0 ? -1 : offs[i] * es / 16;
            const size_t smem = (size_t)2 * px * cbv * sizeof(uint4);
            const void *k = dtype == CONV_F32 ? (const void *)&spp_image_kernel<float>
                                              : (dtype == CONV_BF16 ? (const void *)&spp_image_kernel<__nv_bfloat16>
                                                                    : (const void *)&spp_image_kernel<int8_t>);
            const int rc = conv_grant_smem(k, dev, (int)smem);
            if (rc != CONV_OK) return rc;
            const uint4 *xv = static_cast<const uint4 *>(x);
            uint4 *yv = static_cast<uint4 *>(y);
            void *args[] = {(void *)&xv, (void *)&yv, (void *)&a};
            const cudaError_t e = conv_launch(k, dim3((unsigned)n, (unsigned)(a.CV / cbv)), dim3(kThreads), args,
                                              smem, (cudaStream_t)stream);
            return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
        }
    }
    a.cbv = a.CV < 8 ? a.CV : 8;
    a.tiles_w = (w + kTW - 1) / kTW;
    a.tiles_h = (h + kTH - 1) / kTH;
    a.Cy = y_channels * es / 16;
    for (int i = 0; i < 4; ++i) a.off[i] = offs[i] < 0 ? -1 : offs[i] * es / 16;
    const long long tiles = (long long)a.tiles_w * a.tiles_h * n;
    const int cblocks = (a.CV + a.cbv - 1) / a.cbv;
    if (tiles > 0x7fffffffll || cblocks > 65535) return CONV_ERR_UNSUPPORTED;
    const size_t smem = (size_t)2 * kR * kP * a.cbv * sizeof(uint4);  // <= 100 KB
    const void *k = dtype == CONV_F32 ? (const void *)&spp_kernel<float>
                                      : (dtype == CONV_BF16 ? (const void *)&spp_kernel<__nv_bfloat16>
                                                            : (const void *)&spp_kernel<int8_t>);
    const int rc = conv_grant_smem(k, dev, (int)smem);
    if (rc != CONV_OK) return rc;
    const uint4 *xv = static_cast<const uint4 *>(x);
    uint4 *yv = static_cast<uint4 *>(y);
    void *args[] = {(void *)&xv, (void *)&yv, (void *)&a};
    const cudaError_t e = conv_launch(k, dim3((unsigned)tiles, (unsigned)cblocks), dim3(kThreads), args, smem,
                                      (cudaStream_t)stream);
    return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}
