// Depthwise 3x3 convolution (groups == Cin == Cout), any stride and padding,
// in fp32, bf16 and int8.  No tensor cores: each output channel has its own
// 3x3 filter and there is no reduction across channels, so the layer is a
// bandwidth-bound stencil ("nanoinfer", "What is still slow": depthwise
// convolution is the whole gap, and NHWC lets one vector load cover many
// channels of one pixel).
//
// Tiling.  A CTA produces a th x tw block of output pixels for cb channels
// of one image.  Its input halo, ((th-1)S+3) x ((tw-1)S+3) pixels x cb
// channels, arrives in shared memory as ONE TMA box: coordinates outside the
// image read as zeros, which is the zero padding, and the whole halo is in
// flight at once.  A thread owns one channel vector (4 fp32, 4 bf16 or 16
// int8 channels) at one output column and walks down the th rows, keeping
// the three halo rows under its window in registers (one new row of three
// shared-memory loads per output row at stride 1).  Consecutive threads take
// consecutive channel vectors, so shared-memory reads and the global stores
// are contiguous.  The thread's weights (OHWI [C][3][3] keeps a channel's
// taps together) stay in registers; bf16 values are widened to fp32 (exact)
// and products are paired fp32 FMAs, int8 products exact int32.  The bias
// seeds the accumulator; activation and the int8 requantisation run before
// the single vector store.  bf16 stride-1 layers run the rolling-row kernel
// below instead.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>
#include <type_traits>

#include "conv_internal.h"
#include "epilogue.cuh"
#include "tc_ptx.cuh"

using namespace convk;

namespace {

struct DwArgs {
    int H, W, C, OH, OW, stride, pad_h, pad_w;
    int th, tw, cbv;          // tile: output rows, output columns, 16-byte channel vectors
    int hin, win;             // halo rows / columns
    int tiles_w, tiles_h, tiles_c, tiles_total;
    int act;
    const void *bias;
    const float *mult;
    void *y;
    int *status;
};

template <typename T> struct DwT;
// fp32: a thread owns 4 channels (one 16-byte vector).
template <> struct DwT<float> {
    static constexpr int V = 4;
    using Vec = uint4;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    __device__ static __forceinline__ void to_f(const Vec &u, float (&o)[4]) {
        o[0] = __uint_as_float(u.x); o[1] = __uint_as_float(u.y);
        o[2] = __uint_as_float(u.z); o[3] = __uint_as_float(u.w);
    }
};
// bf16: a thread owns 4 channels (one 8-byte vector); widening a bf16 to
// fp32 is a 16-bit shift of its bits, exact.
template <> struct DwT<__nv_bfloat16> {
    static constexpr int V = 4;
    using Vec = uint2;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    __device__ static __forceinline__ void to_f(const Vec &u, float (&o)[4]) {
        o[0] = __uint_as_float(u.x << 16); o[1] = __uint_as_float(u.x & 0xffff0000u);
        o[2] = __uint_as_float(u.y << 16); o[3] = __uint_as_float(u.y & 0xffff0000u);
    }
};
// int8: a thread owns 16 channels (one 16-byte vector), kept packed.
template <> struct DwT<int8_t> {
    static constexpr int V = 16;
    using Vec = uint4;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_UINT8;
};

template <typename T> __host__ __device__ constexpr int V_OF() { return DwT<T>::V; }

// Two fp32 FMAs in one packed instruction (each lane rounded once, like
// two __fmaf_rn): (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1).
// (Inline PTX here: with the float2 builtin the register allocation of the
// general kernel below spills.)
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ uint32_t word(const uint4 &u, int i) {
    return i == 0 ? u.x : (i == 1 ? u.y : (i == 2 ? u.z : u.w));
}

// Output rows a thread walks per tile (the configured th is at most this).
constexpr int kMaxTh = 8;

// Bounded wait for a halo; false if it ran out (status word set).
__device__ __forceinline__ bool wait_halo(uint32_t sbar, uint32_t parity, int *status) {
    if (tc::mbar_try_wait(sbar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (tc::mbar_try_wait(sbar, parity)) return true;
        if ((i & 63u) == 0u && globaltimer_ns() - t0 > kWaitBudgetNs) {
            atomicExch(status, KSTATUS_TIMEOUT_EPILOGUE);
            return false;
        }
    }
}

// Tile t -> (channel block, image, first output row / column); channel
// block fastest.
struct DwTile {
    int tcb, n, oh0, ow0;
};
__device__ __forceinline__ DwTile tile_of(const DwArgs &a, int t) {
    DwTile d;
    d.tcb = t % a.tiles_c; t /= a.tiles_c;
    const int tw_ = t % a.tiles_w; t /= a.tiles_w;
    d.oh0 = (t % a.tiles_h) * a.th;
    d.n = t / a.tiles_h;
    d.ow0 = tw_ * a.tw;
    return d;
}

// Thread 0: start the TMA of tile t's halo into `dst`, completing on `bar`.
template <int V>
__device__ __forceinline__ void issue_halo(const CUtensorMap *tm, const DwArgs &a, uint32_t dst, uint32_t bar,
                                           int t, int stride, uint32_t bytes) {
    const DwTile d = tile_of(a, t);
    // The buffer was last read through ordinary shared-memory loads; order
    // those before the asynchronous-proxy write that reuses it.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::mbar_arrive_expect_tx(bar, bytes);
    tc::tma_load_4d(dst, tm, bar, d.tcb * a.cbv * V, d.ow0 * stride - a.pad_w, d.oh0 * stride - a.pad_h, d.n);
}

// Persistent CTAs: a CTA takes tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// (gridDim.x is a multiple of tiles_c, so they all share one channel block
// and the thread's weights load once).  Two halo buffers: the TMA of the next
// tile runs while the current one is computed.
template <typename T, int S>
__global__ void __launch_bounds__(256, 2)
dw3x3_float_kernel(const __grid_constant__ CUtensorMap tmX, const T *__restrict__ w, const DwArgs a) {
    pdl_trigger();  // see conv_launch
    pdl_wait();
    using Tr = DwT<T>;
    using Vec = typename Tr::Vec;
    constexpr int VB = sizeof(Vec);
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[2];
    const int stride = S ? S : a.stride;
    const uint32_t halo_bytes = (uint32_t)(a.hin * a.win * a.cbv * VB);
    const uint32_t buf_stride = (halo_bytes + 127u) & ~127u;
    const uint32_t sbase = tc::smem_u32(smem);
    const uint32_t sbar0 = tc::smem_u32(&bars[0]);
    if (threadIdx.x == 0) {
        tc::mbar_init(sbar0, 1);
        tc::mbar_init(sbar0 + 8, 1);
        tc::fence_mbar_init();
        if ((int)blockIdx.x < a.tiles_total)
            issue_halo<4>(&tmX, a, sbase, sbar0, blockIdx.x, stride, halo_bytes);
    }
    __syncwarp();
    __syncthreads();

    const int cv = threadIdx.x % a.cbv;
    const int col = threadIdx.x / a.cbv;
    const int tcb = blockIdx.x % a.tiles_c;   // the same for all of this CTA's tiles
    const int c0 = (tcb * a.cbv + cv) * V_OF<T>();
    const bool active = col < a.tw && c0 < a.C;

    // Weights (OHWI [C][3][3]: a channel's nine taps are contiguous, so the
    // thread's 4 x 9 weights are nine vectors) and bias, loaded once.
    float wt[9][4];
    float bv[4] = {0.f, 0.f, 0.f, 0.f};
    if (active) {
        const Vec *wp = reinterpret_cast<const Vec *>(w + (long long)c0 * 9);
        float raw[36];
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            float f[4];
            Tr::to_f(__ldg(wp + k), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) raw[4 * k + e] = f[e];
        }
#pragma unroll
        for (int v = 0; v < 4; ++v)
#pragma unroll
            for (int k = 0; k < 9; ++k) wt[k][v] = raw[v * 9 + k];
        const float *b = reinterpret_cast<const float *>(a.bias);
        if (b) {
            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(b + c0));
            bv[0] = b4.x; bv[1] = b4.y; bv[2] = b4.z; bv[3] = b4.w;
        }
    }
    const int pix_bytes = a.cbv * VB;
    const int cw = col * stride;

    int k = 0;
    for (int t = blockIdx.x; t < a.tiles_total; t += gridDim.x, ++k) {
        const int buf = k & 1;
        if (threadIdx.x == 0 && t + (int)gridDim.x < a.tiles_total)
            issue_halo<4>(&tmX, a, sbase + (buf ^ 1) * buf_stride, sbar0 + 8 * (buf ^ 1), t + gridDim.x, stride,
                          halo_bytes);
        const bool ok = wait_halo(sbar0 + 8 * buf, (uint32_t)(k >> 1) & 1u, a.status);
        if (__syncthreads_or(!ok)) return;  // block-uniform give-up
        const DwTile d = tile_of(a, t);
        const int ow = d.ow0 + col;
        if (active && ow < a.OW) {
            const uint8_t *hp = smem + buf * buf_stride + cv * VB;
            auto load = [&](float (&o)[4], int r, int c) {
                Tr::to_f(*reinterpret_cast<const Vec *>(hp + (r * a.win + c) * pix_bytes), o);
            };
            float win[3][3][4];
#pragma unroll
            for (int r = 0; r < 3; ++r)
#pragma unroll
                for (int s = 0; s < 3; ++s) load(win[r][s], r, cw + s);
            const int rows = min(a.th, a.OH - d.oh0);
            T *yp = reinterpret_cast<T *>(a.y) + (((long long)d.n * a.OH + d.oh0) * a.OW + ow) * a.C + c0;
            const long long ystep = (long long)a.OW * a.C;
            // Fully unrolled walk down the tile (th <= kMaxTh): the window
            // rotation is register renaming, not moves.
#pragma unroll
            for (int i = 0; i < kMaxTh; ++i) {
                if (i >= rows) break;
                float acc[4];
#pragma unroll
                for (int r = 0; r < 3; ++r)
#pragma unroll
                    for (int s = 0; s < 3; ++s) {
                        const int k = r * 3 + s;
                        // the bias seeds the first tap's FMA
                        const float c0_ = k == 0 ? bv[0] : acc[0], c1_ = k == 0 ? bv[1] : acc[1];
                        const float c2_ = k == 0 ? bv[2] : acc[2], c3_ = k == 0 ? bv[3] : acc[3];
                        ffma2(acc[0], acc[1], win[r][s][0], win[r][s][1], wt[k][0], wt[k][1], c0_, c1_);
                        ffma2(acc[2], acc[3], win[r][s][2], win[r][s][3], wt[k][2], wt[k][3], c2_, c3_);
                    }
                if constexpr (std::is_same<T, float>::value) {
                    *reinterpret_cast<uint4 *>(yp) = make_uint4(
                        __float_as_uint(activate(acc[0], a.act)), __float_as_uint(activate(acc[1], a.act)),
                        __float_as_uint(activate(acc[2], a.act)), __float_as_uint(activate(acc[3], a.act)));
                } else {
                    __nv_bfloat162 lo =
                        __floats2bfloat162_rn(activate_fast(acc[0], a.act), activate_fast(acc[1], a.act));
                    __nv_bfloat162 hi =
                        __floats2bfloat162_rn(activate_fast(acc[2], a.act), activate_fast(acc[3], a.act));
                    *reinterpret_cast<uint2 *>(yp) =
                        make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                }
                yp += ystep;
                if (i + 1 < rows) {
                    const int r0 = (i + 1) * stride;  // halo row of the next window's top tap
                    if (S == 1) {
#pragma unroll
                        for (int s = 0; s < 3; ++s)
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                win[0][s][v] = win[1][s][v];
                                win[1][s][v] = win[2][s][v];
                            }
#pragma unroll
                        for (int s = 0; s < 3; ++s) load(win[2][s], r0 + 2, cw + s);
                    } else if (S == 2) {
#pragma unroll
                        for (int s = 0; s < 3; ++s)
#pragma unroll
                            for (int v = 0; v < 4; ++v) win[0][s][v] = win[2][s][v];
#pragma unroll
                        for (int s = 0; s < 3; ++s) {
                            load(win[1][s], r0 + 1, cw + s);
                            load(win[2][s], r0 + 2, cw + s);
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < 3; ++r)
#pragma unroll
                            for (int s = 0; s < 3; ++s) load(win[r][s], r0 + r, cw + s);
                    }
                }
            }
        }
        __syncwarp();
        __syncthreads();  // this buffer is free for the TMA two tiles ahead
    }
}

// bf16, stride 1: rolling row accumulators.  A thread owns 4 channels x 2
// adjacent output columns of the tile and walks down its input halo rows
// once.  Each input row (4 pixels: the two columns' 3-wide windows overlap)
// is loaded and widened once and feeds the three output rows whose windows
// contain it (as their tap row 2, 1 and 0), whose partial sums stay in
// registers; an output row is finished when its tap row 2 has been added:
// activation, bf16, one 8-byte store per column.  Per output value that is
// half a shared-memory load, two widening operations and 4.5 packed FMAs.
// The tile (CBV 4-channel vectors x TW columns x TH rows) is a compile-time
// shape: the walk is fully unrolled, the rolling accumulators are plain
// registers and every shared-memory address is an immediate offset.
template <int CBV, int TW, int TH>
__global__ void __launch_bounds__(CBV * TW / 2, (CBV * TW / 2) <= 128 ? 4 : 2)
dw3x3_bf16_rows_kernel(const __grid_constant__ CUtensorMap tmX, const __nv_bfloat16 *__restrict__ w,
                       const DwArgs a) {
    pdl_trigger();  // see conv_launch
    // Before waiting for the previous kernel: the halos of this CTA's first
    // tiles into L2 (while that kernel's last CTAs run on other SMs)
    if (threadIdx.x == 0) {
        tc::tma_prefetch_desc(&tmX);
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // (the two halo buffers' first tiles)
            const int t = (int)blockIdx.x + j * (int)gridDim.x;
            if (t < a.tiles_total) {
                const DwTile d = tile_of(a, t);
                tc::tma_prefetch_l2_4d(&tmX, d.tcb * CBV * 4, d.ow0 - a.pad_w, d.oh0 - a.pad_h, d.n);
            }
        }
    }
    pdl_wait();
    constexpr int kWin = TW + 2, kHin = TH + 2;
    constexpr uint32_t kPix = CBV * 8;  // bytes of one halo pixel: CBV vectors of 4 bf16
    constexpr uint32_t kHalo = kHin * kWin * kPix;
    constexpr uint32_t kBuf = (kHalo + 127u) & ~127u;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[2];
    const uint32_t sbase = tc::smem_u32(smem);
    const uint32_t sbar0 = tc::smem_u32(&bars[0]);
    if (threadIdx.x == 0) {
        tc::mbar_init(sbar0, 1);
        tc::mbar_init(sbar0 + 8, 1);
        tc::fence_mbar_init();
        if ((int)blockIdx.x < a.tiles_total) issue_halo<4>(&tmX, a, sbase, sbar0, blockIdx.x, 1, kHalo);
    }
    __syncwarp();
    __syncthreads();

    const int cv = threadIdx.x % CBV;
    const int cp = threadIdx.x / CBV;  // column pair (all CBV * TW / 2 threads are active)
    const int tcb = blockIdx.x % a.tiles_c;  // the same for all of this CTA's tiles
    const int c0 = (tcb * CBV + cv) * 4;

    // Weights (OHWI [C][3][3]: the 4 channels' 36 taps are contiguous) as
    // fp32 pairs wt[k][q] = (w[c0 + 2q][k], w[c0 + 2q + 1][k]); bias pairs.
    float2 wt[9][2];
    float2 bv[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    {
        const uint2 *wp = reinterpret_cast<const uint2 *>(w + (long long)c0 * 9);
        float raw[36];
#pragma unroll
        for (int i = 0; i < 9; ++i) {
            const uint2 u = __ldg(wp + i);
            raw[4 * i + 0] = __uint_as_float(u.x << 16);
            raw[4 * i + 1] = __uint_as_float(u.x & 0xffff0000u);
            raw[4 * i + 2] = __uint_as_float(u.y << 16);
            raw[4 * i + 3] = __uint_as_float(u.y & 0xffff0000u);
        }
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            wt[k][0] = make_float2(raw[k], raw[9 + k]);
            wt[k][1] = make_float2(raw[18 + k], raw[27 + k]);
        }
        const float *b = reinterpret_cast<const float *>(a.bias);
        if (b) {
            const float4 b4 = __ldg(reinterpret_cast<const float4 *>(b + c0));
            bv[0] = make_float2(b4.x, b4.y);
            bv[1] = make_float2(b4.z, b4.w);
        }
    }
    const long long ystep = (long long)a.OW * a.C;
    const int act = a.act;
    int k = 0;
    for (int t = blockIdx.x; t < a.tiles_total; t += gridDim.x, ++k) {
        const int buf = k & 1;
        if (threadIdx.x == 0 && t + (int)gridDim.x < a.tiles_total)
            issue_halo<4>(&tmX, a, sbase + (buf ^ 1) * kBuf, sbar0 + 8 * (buf ^ 1), t + gridDim.x, 1, kHalo);
        const bool ok = wait_halo(sbar0 + 8 * buf, (uint32_t)(k >> 1) & 1u, a.status);
        if (__syncthreads_or(!ok)) return;  // block-uniform give-up
        const DwTile d = tile_of(a, t);
        const uint8_t *hp = smem + buf * kBuf + cv * 8 + (2 * cp) * kPix;
        const int ow = d.ow0 + 2 * cp;
        const bool st0 = ow < a.OW, st1 = ow + 1 < a.OW;
        const int rows = a.OH - d.oh0;  // output rows of this tile inside the image (may exceed TH)
        __nv_bfloat16 *yp = reinterpret_cast<__nv_bfloat16 *>(a.y) +
                            (((long long)d.n * a.OH + d.oh0) * a.OW + ow) * a.C + c0;
        float2 acc[3][2][2];  // [output row % 3][column][channel pair]
#pragma unroll
        for (int hr = 0; hr < TH + 2; ++hr) {
            float2 xv[4][2];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint2 u = *reinterpret_cast<const uint2 *>(hp + (hr * kWin + p) * kPix);
                xv[p][0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
                xv[p][1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
            }
            // input row hr is tap row r of output row hr - r; tap s outermost
            // so that consecutive FMAs feed independent accumulators
#pragma unroll
            for (int s = 0; s < 3; ++s)
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    const int o = hr - r;
                    if (o < 0 || o >= TH) continue;
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            acc[o % 3][j][q] = fma2(xv[j + s][q], wt[r * 3 + s][q],
                                                    (r == 0 && s == 0) ? bv[q] : acc[o % 3][j][q]);
                }
            if (hr >= 2) {  // output row hr - 2 has all its taps
                const int o = hr - 2;
                if (o < rows) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float2 v0 = acc[o % 3][j][0], v1 = acc[o % 3][j][1];
                        if (act == ACT_MISH) {
                            v0 = mish2_fast(v0);
                            v1 = mish2_fast(v1);
                        } else if (act == ACT_RELU) {
                            v0 = make_float2(fmaxf(v0.x, 0.f), fmaxf(v0.y, 0.f));
                            v1 = make_float2(fmaxf(v1.x, 0.f), fmaxf(v1.y, 0.f));
                        }
                        __nv_bfloat162 lo = __floats2bfloat162_rn(v0.x, v0.y);
                        __nv_bfloat162 hi = __floats2bfloat162_rn(v1.x, v1.y);
                        if (j == 0 ? st0 : st1)
                            *reinterpret_cast<uint2 *>(yp + j * a.C) =
                                make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                    }
                }
                yp += ystep;
            }
        }
        __syncwarp();
        __syncthreads();  // this buffer is free for the TMA two tiles ahead
    }
}

// Tile shapes of the rolling-row kernel (CBV x TW x TH): whole warps, at most
// 256 threads.
#define DW_ROWS_SHAPES(X) \
    X(32, 8, 8) X(32, 8, 4) X(32, 4, 8) X(32, 4, 4) X(32, 16, 8) X(32, 16, 4) \
    X(16, 8, 8) X(16, 8, 4) X(16, 16, 8) X(16, 16, 4) X(16, 32, 8) X(16, 32, 4) \
    X(8, 8, 8) X(8, 8, 4) X(8, 16, 8) X(8, 16, 4) X(8, 32, 8) X(8, 32, 4) \
    X(4, 16, 8) X(4, 16, 4) X(4, 32, 8) X(4, 32, 4) X(2, 32, 8) X(2, 32, 4)

// int8: 16 channels per thread, packed window and weights, exact int32.
template <int S>
__global__ void __launch_bounds__(256, 2)
dw3x3_i8_kernel(const __grid_constant__ CUtensorMap tmX, const int8_t *__restrict__ w, const DwArgs a) {
    pdl_trigger();  // see conv_launch
    pdl_wait();
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[2];
    const int stride = S ? S : a.stride;
    const uint32_t halo_bytes = (uint32_t)(a.hin * a.win * a.cbv * 16);
    const uint32_t buf_stride = (halo_bytes + 127u) & ~127u;
    const uint32_t sbase = tc::smem_u32(smem);
    const uint32_t sbar0 = tc::smem_u32(&bars[0]);
    if (threadIdx.x == 0) {
        tc::mbar_init(sbar0, 1);
        tc::mbar_init(sbar0 + 8, 1);
        tc::fence_mbar_init();
        if ((int)blockIdx.x < a.tiles_total)
            issue_halo<16>(&tmX, a, sbase, sbar0, blockIdx.x, stride, halo_bytes);
    }
    __syncwarp();
    __syncthreads();
    const int cv = threadIdx.x % a.cbv;
    const int col = threadIdx.x / a.cbv;
    const int c0 = ((int)(blockIdx.x % a.tiles_c) * a.cbv + cv) * 16;
    const bool active = col < a.tw && c0 < a.C;
    uint4 wv[9];
    if (active) {
        const uint4 *wp = reinterpret_cast<const uint4 *>(w + (long long)c0 * 9);
#pragma unroll
        for (int k = 0; k < 9; ++k) wv[k] = __ldg(wp + k);
    }
    const int32_t *b = reinterpret_cast<const int32_t *>(a.bias);
    const int pix_bytes = a.cbv * 16;
    const int cw = col * stride;
    int k = 0;
    for (int t = blockIdx.x; t < a.tiles_total; t += gridDim.x, ++k) {
        const int buf = k & 1;
        if (threadIdx.x == 0 && t + (int)gridDim.x < a.tiles_total)
            issue_halo<16>(&tmX, a, sbase + (buf ^ 1) * buf_stride, sbar0 + 8 * (buf ^ 1), t + gridDim.x, stride,
                           halo_bytes);
        const bool ok = wait_halo(sbar0 + 8 * buf, (uint32_t)(k >> 1) & 1u, a.status);
        if (__syncthreads_or(!ok)) return;
        const DwTile d = tile_of(a, t);
        const int ow = d.ow0 + col;
        if (active && ow < a.OW) {
            const uint8_t *hp = smem + buf * buf_stride + cv * 16;
            auto halo = [&](int r, int c) {
                return *reinterpret_cast<const uint4 *>(hp + (r * a.win + c) * pix_bytes);
            };
            uint4 win[3][3];
#pragma unroll
            for (int r = 0; r < 3; ++r)
#pragma unroll
                for (int s = 0; s < 3; ++s) win[r][s] = halo(r, cw + s);
            const int rows = min(a.th, a.OH - d.oh0);
            for (int i = 0; i < rows; ++i) {
                int acc[16];
#pragma unroll
                for (int v = 0; v < 16; ++v) acc[v] = 0;
#pragma unroll
                for (int r = 0; r < 3; ++r)
#pragma unroll
                    for (int s = 0; s < 3; ++s)
#pragma unroll
                        for (int v = 0; v < 16; ++v) {
                            const int e = v * 9 + r * 3 + s;
                            const int xv = (int)(int8_t)(word(win[r][s], v >> 2) >> (8 * (v & 3)));
                            const int wq = (int)(int8_t)(word(wv[e >> 4], (e >> 2) & 3) >> (8 * (e & 3)));
                            acc[v] += xv * wq;
                        }
                uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    const long long val = (long long)acc[v] + (b ? (long long)__ldg(b + c0 + v) : 0ll);
                    const int q = requant_i8(val, __ldg(a.mult + c0 + v), a.act);
                    wd[v >> 2] |= ((uint32_t)(q & 0xff)) << (8 * (v & 3));
                }
                int8_t *yp = reinterpret_cast<int8_t *>(a.y) +
                             (((long long)d.n * a.OH + d.oh0 + i) * a.OW + ow) * a.C + c0;
                *reinterpret_cast<uint4 *>(yp) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                if (i + 1 < rows) {
                    const int r0 = (i + 1) * stride;
                    if (S == 1) {
#pragma unroll
                        for (int s = 0; s < 3; ++s) {
                            win[0][s] = win[1][s];
                            win[1][s] = win[2][s];
                            win[2][s] = halo(r0 + 2, cw + s);
                        }
                    } else if (S == 2) {
#pragma unroll
                        for (int s = 0; s < 3; ++s) {
                            win[0][s] = win[2][s];
                            win[1][s] = halo(r0 + 1, cw + s);
                            win[2][s] = halo(r0 + 2, cw + s);
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < 3; ++r)
#pragma unroll
                            for (int s = 0; s < 3; ++s) win[r][s] = halo(r0 + r, cw + s);
                    }
                }
            }
        }
        __syncwarp();
        __syncthreads();
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

template <typename T>
void *kernel_for(int stride) {
    if (stride == 1) return reinterpret_cast<void *>(&dw3x3_float_kernel<T, 1>);
    if (stride == 2) return reinterpret_cast<void *>(&dw3x3_float_kernel<T, 2>);
    return reinterpret_cast<void *>(&dw3x3_float_kernel<T, 0>);
}

void *select_rows(int cbv, int tw, int th) {
#define DW_ROWS_CASE(C, W, H) \
    if (cbv == C && tw == W && th == H) return reinterpret_cast<void *>(&dw3x3_bf16_rows_kernel<C, W, H>);
    DW_ROWS_SHAPES(DW_ROWS_CASE)
#undef DW_ROWS_CASE
    return nullptr;
}

void *select(conv_dtype_t dt, int stride) {
    switch (dt) {
    case CONV_F32: return kernel_for<float>(stride);
    case CONV_BF16: return kernel_for<__nv_bfloat16>(stride);
    default:
        if (stride == 1) return reinterpret_cast<void *>(&dw3x3_i8_kernel<1>);
        if (stride == 2) return reinterpret_cast<void *>(&dw3x3_i8_kernel<2>);
        return reinterpret_cast<void *>(&dw3x3_i8_kernel<0>);
    }
}

// Channels a thread owns and bytes of its vector.
int dw_chans(conv_dtype_t dt) { return dt == CONV_I8 ? 16 : 4; }
int dw_vbytes(conv_dtype_t dt) { return dt == CONV_BF16 ? 8 : 16; }

CUtensorMapDataType tma_type(conv_dtype_t dt) {
    return dt == CONV_F32 ? DwT<float>::tma : (dt == CONV_BF16 ? DwT<__nv_bfloat16>::tma : DwT<int8_t>::tma);
}

}  // namespace

bool dw3x3_supported(const conv_plan *p) {
    const int C = p->s.c_in;
    const int V = dw_chans(p->dtype);
    if (!(p->groups == C && p->s.c_out == C && p->s.k_h == 3 && p->s.k_w == 3 && C % V == 0)) return false;
    if (p->stride > 64) return false;                        // halo box sides are at most 256
    if ((long long)p->s.n * p->s.h * p->s.w >= (1ll << 31)) return false;
    return true;  // tile counts fit an int: at most N*H*W tiles
}

// bf16 stride-1 layers: the rolling-row kernel.  Tile = th x tw output
// pixels x 4 cbv channels, a thread per 4 channels x 2 columns.  Among tiles
// of whole warps whose two halo buffers leave room for two CTAs per SM, the
// one with the least estimated work on the busiest SM: tiles per SM x (halo
// bytes + output bytes + a per-row cost of the TMA box + a fixed cost).
static int dw3x3_rows_configure(conv_plan *p) {
    const int C = p->s.c_in;
    DwGeom &g = p->dw;
    long long best = -1;
    for (int cbv : {32, 16, 8, 4, 2}) {
        if ((C / 4) % cbv != 0) continue;
        for (int tw = 2; tw <= 32; tw += 2) {
            const int threads = cbv * tw / 2;
            if (threads > 256) break;
            if (threads % 32 != 0) continue;
            for (int th : {8, 4}) {
                if (!select_rows(cbv, tw, th)) continue;  // shapes with a compiled kernel only
                const int win = tw + 2, hin = th + 2;
                const int halo = hin * win * cbv * 8;
                const int smem = 2 * ((halo + 127) & ~127);
                if (smem > 110 * 1024) continue;
                const long long tiles = (long long)(C / 4 / cbv) * ((p->ow + tw - 1) / tw) *
                                        ((p->oh + th - 1) / th) * p->s.n;
                const long long per_sm = (tiles + p->num_sms - 1) / p->num_sms;
                const long long cost = per_sm * (halo + tw * th * cbv * 8 + hin * win * 64 + 2048);
                if (best < 0 || cost < best || (cost == best && threads > g.threads)) {
                    best = cost;
                    g.cbv = cbv; g.tw = tw; g.th = th; g.threads = threads; g.smem = smem;
                    g.hin = hin; g.win = win;
                }
            }
        }
    }
    if (best < 0) return CONV_ERR_UNSUPPORTED;
    g.kind = 1;
    g.tiles_w = (p->ow + g.tw - 1) / g.tw;
    g.tiles_h = (p->oh + g.th - 1) / g.th;
    g.tiles_c = C / 4 / g.cbv;
    g.tiles = (long long)g.tiles_c * g.tiles_w * g.tiles_h * p->s.n;
    // Persistent grid: the CTAs resident at once (shared memory, threads,
    // 128 registers a thread), a multiple of the channel-block count.
    int res = (227 * 1024) / (g.smem + 1024);
    if (res > 2048 / g.threads) res = 2048 / g.threads;
    if (res > 65536 / (g.threads * 128)) res = 65536 / (g.threads * 128);
    long long grid = (long long)p->num_sms * res;
    if (grid > g.tiles) grid = g.tiles;
    if (grid > g.tiles_c) grid -= grid % g.tiles_c;
    else grid = g.tiles_c;
    g.blocks = grid;
    return conv_grant_smem(select_rows(g.cbv, g.tw, g.th), p->device, g.smem);
}

int dw3x3_configure(conv_plan *p) {
    const int S = p->stride;
    p->dw.kind = 0;
    if (p->dtype == CONV_BF16 && S == 1 && p->s.c_in % 8 == 0) return dw3x3_rows_configure(p);
    const int V = dw_chans(p->dtype);
    const int cvt = p->s.c_in / V;                 // channel vectors in a pixel
    const int maxv = 256 / dw_vbytes(p->dtype);    // at most 256 bytes of channels per tile pixel
    // Channel vectors and output columns per tile: at most 256 threads, the
    // fewest halo columns loaded per output row (ragged tiles load wasted
    // columns too), then the most threads.
    int best_tw = 1, best_cbv = 1;
    long long best_cost = -1;
    // Enough tiles to give every SM two CTAs, if the layer allows.
    const long long rows_tiles = (long long)p->s.n * ((p->oh + kMaxTh - 1) / kMaxTh);
    for (int cbv : {32, 16, 8, 4, 2, 1}) {
        if (cbv > maxv || cbv > cvt || cvt % cbv != 0) continue;
        for (int tw = 1; tw * cbv <= 256 && (tw - 1) * S + 3 <= 256; ++tw) {
            const long long tiles = (p->ow + tw - 1) / tw;
            long long cost = tiles * ((tw - 1) * S + 3) * (cvt / cbv);
            if (tiles * (cvt / cbv) * rows_tiles < (long long)p->num_sms * 2 && tw * cbv > 32)
                cost = cost * 4;  // too few CTAs to keep the GPU busy
            const bool better = best_cost < 0 || cost < best_cost ||
                                (cost == best_cost && tw * cbv > best_tw * best_cbv);
            if (better) { best_cost = cost; best_tw = tw; best_cbv = cbv; }
            if (tw >= p->ow) break;
        }
    }
    const int cbv = best_cbv;
    int th = kMaxTh;
    if (th > p->oh) th = p->oh;
    while ((th - 1) * S + 3 > 256) --th;
    // Small layers: fewer output rows per tile (a shorter serial walk per
    // thread) until there is a tile per SM.
    const long long col_tiles = (long long)((p->ow + best_tw - 1) / best_tw) * ((cvt + cbv - 1) / cbv) * p->s.n;
    while (th > 1 && col_tiles * ((p->oh + th - 1) / th) < (long long)p->num_sms) th = (th + 1) / 2;
    DwGeom &g = p->dw;
    g.tw = best_tw;
    g.th = th;
    g.cbv = cbv;
    g.hin = (th - 1) * S + 3;
    g.win = (best_tw - 1) * S + 3;
    g.tiles_w = (p->ow + best_tw - 1) / best_tw;
    g.tiles_h = (p->oh + th - 1) / th;
    g.tiles_c = (cvt + cbv - 1) / cbv;
    const int halo = g.hin * g.win * cbv * dw_vbytes(p->dtype);
    g.smem = 2 * ((halo + 127) & ~127);  // two halo buffers (double buffering)
    g.threads = ((best_tw * cbv + 31) / 32) * 32;
    g.tiles = (long long)g.tiles_c * g.tiles_w * g.tiles_h * p->s.n;
    // Persistent grid: two CTAs per SM, a multiple of the channel-block count
    // (each CTA then keeps one channel block), at most one CTA per tile.
    long long grid = (long long)p->num_sms * 2;
    if (grid > g.tiles) grid = g.tiles;
    if (grid > g.tiles_c) grid -= grid % g.tiles_c;
    else grid = g.tiles_c;  // one CTA per channel block (tiles is a multiple of tiles_c)
    g.blocks = grid;
    return conv_grant_smem(select(p->dtype, S), p->device, g.smem);
}

cudaError_t launch_dw3x3(const conv_plan *p, const void *x, const void *w, const void *bias, void *y,
                         cudaStream_t st) {
    const DwGeom &g = p->dw;
    PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
    if (!encode) return cudaErrorNotSupported;
    const int es = conv_esize(p->dtype);
    const int V = dw_chans(p->dtype);
    alignas(64) CUtensorMap tm;
    const cuuint64_t dims[4] = {(cuuint64_t)p->s.c_in, (cuuint64_t)p->s.w, (cuuint64_t)p->s.h, (cuuint64_t)p->s.n};
    const cuuint64_t strides[3] = {(cuuint64_t)p->s.c_in * es, (cuuint64_t)p->s.w * p->s.c_in * es,
                                   (cuuint64_t)p->s.h * p->s.w * p->s.c_in * es};
    const cuuint32_t box[4] = {(cuuint32_t)(g.cbv * V), (cuuint32_t)g.win, (cuuint32_t)g.hin, 1};
    const cuuint32_t ones[4] = {1, 1, 1, 1};
    if (encode(&tm, tma_type(p->dtype), 4, const_cast<void *>(x), dims, strides, box, ones,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    DwArgs a;
    a.H = p->s.h; a.W = p->s.w; a.C = p->s.c_in; a.OH = p->oh; a.OW = p->ow;
    a.stride = p->stride; a.pad_h = p->pad_h; a.pad_w = p->pad_w;
    a.th = g.th; a.tw = g.tw; a.cbv = g.cbv; a.hin = g.hin; a.win = g.win;
    a.tiles_w = g.tiles_w; a.tiles_h = g.tiles_h; a.tiles_c = g.tiles_c;
    a.tiles_total = (int)g.tiles;
    a.act = (int)p->act;
    a.bias = bias;
    a.mult = p->d_mult;
    a.y = y;
    a.status = p->d_status;
    void *k = g.kind == 1 ? select_rows(g.cbv, g.tw, g.th) : select(p->dtype, p->stride);
    void *args[] = {&tm, &w, &a};
    return conv_launch(k, dim3((unsigned)g.blocks), dim3(g.threads), args, (size_t)g.smem, st);
}
