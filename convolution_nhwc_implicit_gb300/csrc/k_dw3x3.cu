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
// flight at once.  A thread owns one 16-byte channel vector (4 fp32, 8 bf16
// or 16 int8 channels) at one output column and walks down the th rows,
// keeping the three halo rows under its window in registers (one new row of
// three 16-byte shared-memory loads per output row at stride 1).  Consecutive
// threads take consecutive channel vectors, so shared-memory reads and the
// global stores are contiguous.  The thread's 9 x 16 bytes of weights are
// nine 16-byte loads (OHWI [C][3][3] keeps a channel's taps together) and
// stay in registers, packed: bf16 products use fma.rn.f32.bf16 (bf16
// operands, fp32 accumulation) so nothing is unpacked.  The bias seeds the
// accumulator; activation and the int8 requantisation run before the single
// 16-byte store.
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
    int tiles_w, tiles_h, tiles_c;
    int act;
    const void *bias;
    const float *mult;
    void *y;
    int *status;
};

template <typename T> struct DwT;
template <> struct DwT<float> {
    static constexpr int V = 4;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <> struct DwT<__nv_bfloat16> {
    static constexpr int V = 8;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};
template <> struct DwT<int8_t> {
    static constexpr int V = 16;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_UINT8;
};

// acc += x * w for one 16-byte input vector and the matching 16 bytes of one
// tap's weights (V channels).
__device__ __forceinline__ void fma_vec(float (&acc)[4], const uint4 &x, const float (&w)[4]) {
    acc[0] = __fmaf_rn(__uint_as_float(x.x), w[0], acc[0]);
    acc[1] = __fmaf_rn(__uint_as_float(x.y), w[1], acc[1]);
    acc[2] = __fmaf_rn(__uint_as_float(x.z), w[2], acc[2]);
    acc[3] = __fmaf_rn(__uint_as_float(x.w), w[3], acc[3]);
}

// bf16: both operands are bf16 halves of 32-bit words; fp32 accumulation.
__device__ __forceinline__ float fma_bf16(uint32_t xw, int xh, uint32_t ww, int wh, float c) {
    float d;
    if (xh == 0 && wh == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, %3;\n\t}" : "=f"(d) : "r"(xw), "r"(ww), "f"(c));
    else if (xh == 0 && wh == 1)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, b1, %3;\n\t}" : "=f"(d) : "r"(xw), "r"(ww), "f"(c));
    else if (xh == 1 && wh == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a1, b0, %3;\n\t}" : "=f"(d) : "r"(xw), "r"(ww), "f"(c));
    else
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a1, b1, %3;\n\t}" : "=f"(d) : "r"(xw), "r"(ww), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t word(const uint4 &u, int i) {
    return i == 0 ? u.x : (i == 1 ? u.y : (i == 2 ? u.z : u.w));
}

template <typename T, int S>
__global__ void __launch_bounds__(256, 2)
dw3x3_kernel(const __grid_constant__ CUtensorMap tmX, const T *__restrict__ w, const DwArgs a) {
    constexpr int V = DwT<T>::V;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar;
    const int stride = S ? S : a.stride;

    // tile coordinates: channel block fastest, then columns, rows, image
    int t = blockIdx.x;
    const int tc_ = t % a.tiles_c; t /= a.tiles_c;
    const int tw_ = t % a.tiles_w; t /= a.tiles_w;
    const int th_ = t % a.tiles_h;
    const int n = t / a.tiles_h;
    const int oh0 = th_ * a.th, ow0 = tw_ * a.tw;
    const int cv = threadIdx.x % a.cbv;
    const int col = threadIdx.x / a.cbv;
    const int c0 = (tc_ * a.cbv + cv) * V;  // first channel of this thread's vector
    const int cbytes = a.cbv * 16;           // bytes of one halo pixel

    const uint32_t sbar = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(sbar, 1);
        tc::fence_mbar_init();
        tc::mbar_arrive_expect_tx(sbar, (uint32_t)(a.hin * a.win * cbytes));
        tc::tma_load_4d(tc::smem_u32(smem), &tmX, sbar, tc_ * a.cbv * V, ow0 * stride - a.pad_w,
                        oh0 * stride - a.pad_h, n);
    }

    // Weights and bias while the halo is in flight.
    const bool active = col < a.tw && c0 < a.C;
    uint4 wv[9];
    if (active) {
        const uint4 *wp = reinterpret_cast<const uint4 *>(w + (long long)c0 * 9);
#pragma unroll
        for (int k = 0; k < 9; ++k) wv[k] = __ldg(wp + k);
    }
    __syncthreads();  // barrier initialised before anyone waits on it

    // Bounded wait for the halo (every thread polls the mbarrier).
    bool ok = tc::mbar_try_wait(sbar, 0);
    if (!ok) {
        const unsigned long long t0 = globaltimer_ns();
        for (uint32_t i = 1; !ok; ++i) {
            ok = tc::mbar_try_wait(sbar, 0);
            if (!ok && (i & 63u) == 0u && globaltimer_ns() - t0 > kWaitBudgetNs) {
                if (threadIdx.x == 0) atomicExch(a.status, KSTATUS_TIMEOUT_EPILOGUE);
                break;
            }
        }
    }
    if (!ok || !active) return;
    const int ow = ow0 + col;
    if (ow >= a.OW) return;

    const uint8_t *hp = smem + cv * 16;
    auto halo = [&](int r, int c) {
        return *reinterpret_cast<const uint4 *>(hp + (r * a.win + c) * cbytes);
    };
    const int cw = col * stride;  // halo column of the window's left tap
    uint4 win[3][3];
#pragma unroll
    for (int r = 0; r < 3; ++r)
#pragma unroll
        for (int s = 0; s < 3; ++s) win[r][s] = halo(r, cw + s);

    const int rows = min(a.th, a.OH - oh0);
    for (int i = 0; i < rows; ++i) {
        uint4 out;
        if constexpr (std::is_same<T, float>::value) {
            float acc[4];
            const float *b = reinterpret_cast<const float *>(a.bias);
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[v] = b ? __ldg(b + c0 + v) : 0.0f;
#pragma unroll
            for (int r = 0; r < 3; ++r)
#pragma unroll
                for (int s = 0; s < 3; ++s) {
                    // weights of tap k for channels c0..c0+3: element v*9+k of wv
                    float wt[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int e = v * 9 + r * 3 + s;
                        wt[v] = __uint_as_float(word(wv[e / 4], e % 4));
                    }
                    fma_vec(acc, win[r][s], wt);
                }
            float o[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) o[v] = activate(acc[v], a.act);
            out = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                             __float_as_uint(o[3]));
        } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            float acc[8];
            const float *b = reinterpret_cast<const float *>(a.bias);
            if (b) {
                const float4 b0 = __ldg(reinterpret_cast<const float4 *>(b + c0));
                const float4 b1 = __ldg(reinterpret_cast<const float4 *>(b + c0) + 1);
                acc[0] = b0.x; acc[1] = b0.y; acc[2] = b0.z; acc[3] = b0.w;
                acc[4] = b1.x; acc[5] = b1.y; acc[6] = b1.z; acc[7] = b1.w;
            } else {
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[v] = 0.0f;
            }
#pragma unroll
            for (int r = 0; r < 3; ++r)
#pragma unroll
                for (int s = 0; s < 3; ++s)
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const int e = v * 9 + r * 3 + s;  // weight element (bf16 index)
                        acc[v] = fma_bf16(word(win[r][s], v >> 1), v & 1, word(wv[e >> 3], (e >> 1) & 3), e & 1,
                                          acc[v]);
                    }
            uint32_t wd[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                __nv_bfloat162 h2 =
                    __floats2bfloat162_rn(activate_fast(acc[2 * k], a.act), activate_fast(acc[2 * k + 1], a.act));
                wd[k] = *reinterpret_cast<uint32_t *>(&h2);
            }
            out = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        } else {
            int acc[16];
            const int32_t *b = reinterpret_cast<const int32_t *>(a.bias);
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
                        const int wt = (int)(int8_t)(word(wv[e >> 4], (e >> 2) & 3) >> (8 * (e & 3)));
                        acc[v] += xv * wt;
                    }
            uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int v = 0; v < 16; ++v) {
                const long long val = (long long)acc[v] + (b ? (long long)__ldg(b + c0 + v) : 0ll);
                const int q = requant_i8(val, __ldg(a.mult + c0 + v), a.act);
                wd[v >> 2] |= ((uint32_t)(q & 0xff)) << (8 * (v & 3));
            }
            out = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
        T *yp = reinterpret_cast<T *>(a.y) + (((long long)n * a.OH + oh0 + i) * a.OW + ow) * a.C + c0;
        *reinterpret_cast<uint4 *>(yp) = out;

        if (i + 1 < rows) {
            const int r0 = (i + 1) * stride;  // halo row of the next window's top tap
            if (S == 1) {
#pragma unroll
                for (int s = 0; s < 3; ++s) { win[0][s] = win[1][s]; win[1][s] = win[2][s]; win[2][s] = halo(r0 + 2, cw + s); }
            } else if (S == 2) {
#pragma unroll
                for (int s = 0; s < 3; ++s) {
                    win[0][s] = win[2][s]; win[1][s] = halo(r0 + 1, cw + s); win[2][s] = halo(r0 + 2, cw + s);
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
    if (stride == 1) return reinterpret_cast<void *>(&dw3x3_kernel<T, 1>);
    if (stride == 2) return reinterpret_cast<void *>(&dw3x3_kernel<T, 2>);
    return reinterpret_cast<void *>(&dw3x3_kernel<T, 0>);
}

void *select(conv_dtype_t dt, int stride) {
    switch (dt) {
    case CONV_F32: return kernel_for<float>(stride);
    case CONV_BF16: return kernel_for<__nv_bfloat16>(stride);
    default: return kernel_for<int8_t>(stride);
    }
}

CUtensorMapDataType tma_type(conv_dtype_t dt) {
    return dt == CONV_F32 ? DwT<float>::tma : (dt == CONV_BF16 ? DwT<__nv_bfloat16>::tma : DwT<int8_t>::tma);
}

}  // namespace

bool dw3x3_supported(const conv_plan *p) {
    const int C = p->s.c_in;
    const int V = 16 / conv_esize(p->dtype);
    if (!(p->groups == C && p->s.c_out == C && p->s.k_h == 3 && p->s.k_w == 3 && C % V == 0)) return false;
    if (p->stride > 64) return false;                        // halo box sides are at most 256
    if ((long long)p->s.n * p->s.h * p->s.w >= (1ll << 31)) return false;
    return true;
}

int dw3x3_configure(conv_plan *p) {
    const int S = p->stride;
    const int V = 16 / conv_esize(p->dtype);
    const int cvt = p->s.c_in / V;                 // channel vectors in a pixel
    // Channel vectors and output columns per tile: at most 256 threads, the
    // fewest halo columns loaded per output row (ragged tiles load wasted
    // columns too), then the most threads.
    int best_tw = 1, best_cbv = 1;
    long long best_cost = -1;
    for (int cbv : {16, 8, 4, 2, 1}) {
        if (cbv > cvt || cvt % cbv != 0) continue;
        for (int tw = 1; tw * cbv <= 256 && (tw - 1) * S + 3 <= 256; ++tw) {
            const long long tiles = (p->ow + tw - 1) / tw;
            const long long cost = tiles * ((tw - 1) * S + 3) * (cvt / cbv);
            const bool better = best_cost < 0 || cost < best_cost ||
                                (cost == best_cost && tw * cbv > best_tw * best_cbv);
            if (better) { best_cost = cost; best_tw = tw; best_cbv = cbv; }
            if (tw >= p->ow) break;
        }
    }
    const int cbv = best_cbv;
    int th = 8;
    if (th > p->oh) th = p->oh;
    while ((th - 1) * S + 3 > 256) --th;
    DwGeom &g = p->dw;
    g.tw = best_tw;
    g.th = th;
    g.cbv = cbv;
    g.hin = (th - 1) * S + 3;
    g.win = (best_tw - 1) * S + 3;
    g.tiles_w = (p->ow + best_tw - 1) / best_tw;
    g.tiles_h = (p->oh + th - 1) / th;
    g.tiles_c = (cvt + cbv - 1) / cbv;
    g.smem = g.hin * g.win * cbv * 16;
    g.threads = ((best_tw * cbv + 31) / 32) * 32;
    g.blocks = (long long)g.tiles_c * g.tiles_w * g.tiles_h * p->s.n;
    return conv_grant_smem(select(p->dtype, S), p->device, g.smem);
}

cudaError_t launch_dw3x3(const conv_plan *p, const void *x, const void *w, const void *bias, void *y,
                         cudaStream_t st) {
    const DwGeom &g = p->dw;
    PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
    if (!encode) return cudaErrorNotSupported;
    const int es = conv_esize(p->dtype);
    const int V = 16 / es;
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
    a.act = (int)p->act;
    a.bias = bias;
    a.mult = p->d_mult;
    a.y = y;
    a.status = p->d_status;
    void *k = select(p->dtype, p->stride);
    void *args[] = {&tm, &w, &a};
    return cudaLaunchKernel(k, dim3((unsigned)g.blocks), dim3(g.threads), args, (size_t)g.smem, st);
}
