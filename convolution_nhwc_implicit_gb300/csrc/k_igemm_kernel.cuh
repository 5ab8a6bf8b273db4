#pragma once
// Implicit-GEMM convolution on the 5th-generation tensor cores (tcgen05),
// bf16 operands with fp32 accumulation in TMEM, for dense k x k and 1x1
// layers.  im2col is never materialised ("nanoinfer", "1x1 convolutions are
// already a GEMM": the patch matrix of a 1x1 stride-1 unpadded layer is the
// input itself; for k x k layers each tap's patch rows are fetched straight
// from the NHWC input by TMA).
//
// GEMM view: M = output pixels, N = Cout, K = k_h * k_w * Cin ordered
// (r, s, ci).  NHWC activations and OHWI weights are then both K-contiguous
// ("nanoinfer", cuBLAS layout comparison: both operands K-contiguous is the
// fast layout for tensor cores), so the weight tensor is, as stored, the
// K-major B operand [Cout][K].
//
// Tiles.  An M tile is 128 output pixels.  For a 1x1, stride-1, unpadded
// layer ("flat" mode) it is 128 consecutive pixels of x viewed as
// [N*H*W, Cin].  Otherwise it is a bh x bw rectangle of output pixels of one
// image (bh * bw <= 128; rows past bh * bw are computed from stale shared
// memory and never stored).  For tap (r, s) and channel block cb, the A tile
// is one 4-D TMA box of the NHWC input starting at
// (cb * BK, ow0 * S - pad_w + s, oh0 * S - pad_h + r, n) with element strides
// (1, S, S, 1): TMA fills out-of-image coordinates with zeros, which is the
// zero padding, and the element strides are the convolution stride.  The B
// tile is the [BN x BK] block of the weights at K offset (r, s, cb).
//
// Warp roles (320 or 576 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: fills a ring of `stages` shared-memory stages
//   warp 1      MMA issuer: tcgen05.mma M=128 x N=BN x K=16 per instruction,
//               accumulating a tile in one of two TMEM buffers
//   warps 2..    epilogue: 2 or 4 warpgroups, each draining a slice of the
//               tile's columns (tcgen05.ld, one pixel row per thread), then
//               + bias, ReLU / Mish, round to bf16, 16-byte stores.
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile
// i + 1; an epilogue thread returns its TMEM slice as soon as the values are
// in registers.  Every wait on an mbarrier is bounded; a wait that runs out sets the
// plan's status word and the CTA unwinds (frees its TMEM and returns).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdio.h>

#include <type_traits>

#include "conv_internal.h"
#include "epilogue.cuh"
#include "tc_ptx.cuh"

using namespace convk;

namespace {

constexpr int kBM = 128;     // output pixels per tile (normal mode)
constexpr int kBMSwap = 256; // output pixels per tile (swapped mode)
constexpr int kTP = 272;     // swapped-mode transpose rows: 128 bf16 channels + 16 bytes of padding

// Epilogue warpgroups per CTA: each takes a slice of every tile's columns,
// or (ept: one epilogue per tile) whole tiles in turn.
__host__ __device__ constexpr int epi_groups(int bn, bool swap, bool ept = false) {
    return (swap || ept) ? 4 : (bn >= 128 ? 4 : 2);
}
// Threads per CTA: the TMA warp, the MMA warp and the epilogue warpgroups
// (and, cvt: the converter warpgroup).
__host__ __device__ constexpr int cta_threads(int bn, bool swap, bool ept = false, bool cvt = false) {
    return 64 + 128 * epi_groups(bn, swap, ept) + (cvt ? 128 : 0);
}

struct IgArgs {
    int H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, OH, OW;
    int bw, bh, tiles_w, tiles_h, tiles_n, num_tiles, cblocks, kblocks, stages;
    int wblocks;         // weight K blocks of the layer: KH * KW * cblocks
    int halo;            // 1: halo staging (see the kernel's comment); a ring stage is then
                         //    the K block (s, cb), kblocks = KW * cblocks
    uint32_t a_stage;    // bytes of one activation stage of the ring (a multiple of 1024)
    int tiles_m;         // pixel tiles (pair mode: each CTA of a pair takes one of two)
    long long M;         // flat mode: rows of x viewed as [N*H*W, Cin]
    int flat;
    uint32_t a_bytes;    // bytes TMA writes per A box
    int act;
    const void *bias;    // fp32 [Cout] (bf16 output) or int32 [Cout] (int8 output), or null
    void *y;             // bf16 or int8 NHWC output
    int out_i8;          // 1: int8 output, requantised with mult[co]
    const float *mult;   // int8: requantisation multipliers M[co]
    int out_bufs;        // normal mode: output staging buffers per epilogue group (1 or 2)
    int bias_smem;       // 1: the epilogue warps copy the bias (and the int8 multipliers)
                         //    into shared memory once per CTA and read them from there
    int wres;            // 1: the layer's whole weight tensor (one N block; in pair mode this
                         //    CTA's half of it) is loaded once per CTA and stays in shared
                         //    memory; the ring then holds activations only
    OutMap om;           // output placement (concat slice, 2x upsample) and residual
    int *status;
    // CVT (int8 operands widened in the kernel): the raw int8 activation part
    // of a stage (a_bytes of them written by TMA, box_rows pixel rows of BK
    // bytes), and the raw weights' bytes (loaded once, then widened)
    uint32_t raw_stage;
    int box_rows;
    uint32_t raw_region;  // bytes of the raw region (the raw weights, then the raw ring, share it)
    // CVT == 2 (small-Cin bf16 layers folded in the kernel): the layer's own
    // Cin, k_w and pad_w, the bf16 elements of a raw box row, and the weights
    int fold_cin, fold_kw, fold_padw, raw_inner;
    const __nv_bfloat16 *w_raw;
};

// The output tensor maps of the TMA-store epilogue: one per upsample
// replica (dy, dx) (only the first without upsampling), each a view of y's
// channel slice at that replica's pixels.
struct YMaps {
    CUtensorMap m[4];
};

// Waits for phase `parity` of `bar`, giving up after kWaitBudgetNs or when
// another role of the CTA has given up.  Returns false on give-up.
// CLUSTER: acquire at cluster scope (arrivals may come from the peer CTA).
// The coordinates of a CTA's (or an epilogue group's) tiles tile0, tile0 +
// step, ...: N block nb, M tile mt and, spatial, its tile column tw, tile row
// th and image n, advanced by mixed-radix addition of the step's digits
// (no division per tile).
struct TileWalk {
    int nb, mt, tw, th, n;
    int sn, sm, sw, sh, snn;
    __device__ __forceinline__ void init(const IgArgs &a, int tile0, int step) {
        nb = tile0 % a.tiles_n; mt = tile0 / a.tiles_n;
        tw = mt % a.tiles_w; th = (mt / a.tiles_w) % a.tiles_h; n = mt / (a.tiles_w * a.tiles_h);
        sn = step % a.tiles_n; sm = step / a.tiles_n;
        sw = sm % a.tiles_w; sh = (sm / a.tiles_w) % a.tiles_h; snn = sm / (a.tiles_w * a.tiles_h);
    }
    __device__ __forceinline__ void advance(const IgArgs &a) {
        nb += sn;
        const int c = nb >= a.tiles_n ? 1 : 0;
        nb -= c * a.tiles_n;
        mt += sm + c;
        tw += sw + c;
        const int c2 = tw >= a.tiles_w ? 1 : 0;
        tw -= c2 * a.tiles_w;
        th += sh + c2;
        const int c3 = th >= a.tiles_h ? 1 : 0;
        th -= c3 * a.tiles_h;
        n += snn + c3;
    }
};

template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             int *status, int code) {
    auto poll = [&]() { return CLUSTER ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (poll()) return true;
        if ((i & 63u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitBudgetNs) {
                *abort_flag = 1;
                atomicExch(status, code);
                return false;
            }
        }
    }
}

// Swapped-mode write-out: y element offset (channel 0 of the layer's slice,
// replica (0, 0)) of pixel p of the tile, and whether p is inside the image.
__device__ __forceinline__ void swapped_pixel(const IgArgs &a, long long m0, int n, int oh0, int ow0, int p,
                                              long long &yb, bool &valid) {
    if (a.flat) {  // (no upsampling in flat mode)
        const long long pix = m0 + p;
        valid = pix < a.M;
        yb = pix * a.om.Cy + a.om.c_off;
    } else {
        const int dh = p / a.bw;
        const int oh = oh0 + dh, ow = ow0 + (p - dh * a.bw);
        valid = p < a.bw * a.bh && oh < a.OH && ow < a.OW;
        yb = a.om.base(n, oh, ow);
    }
}

// Pixel index (n, oh, ow flattened) of pixel p of a swapped-mode tile, or -1
// outside the image.
__device__ __forceinline__ long long swapped_pix(const IgArgs &a, long long m0, int n, int oh0, int ow0, int p) {
    if (a.flat) return m0 + p < a.M ? m0 + p : -1;
    const int dh = p / a.bw;
    const int oh = oh0 + dh, ow = ow0 + (p - dh * a.bw);
    if (p >= a.bw * a.bh || oh >= a.OH || ow >= a.OW) return -1;
    return ((long long)n * a.OH + oh) * a.OW + ow;
}

// Epilogue of the swapped mode for one tile.  The accumulator is D[co][px]:
// thread `row` of the group holds output channel co = nb*128 + row and reads
// the group's kCols pixel columns 16 at a time.  Each 16-pixel chunk goes
// through shared memory (rows of 128 channels, padded to kTP bytes) to turn
// channel-per-thread values into pixel rows, which the group then writes
// with 16-byte stores (eight threads cover one pixel's 128 channels).
template <int kCols, bool FUSED>
__device__ __forceinline__ void epilogue_swapped(const IgArgs &a, int tile, uint32_t taddr, uint32_t tempty,
                                                 int row, int grp, int c_base, uint8_t *tbuf, int gt) {
    const int nb = tile % a.tiles_n;
    const int mt = tile / a.tiles_n;
    const int co = nb * 128 + row;
    const bool cov = co < a.Cout;
    const float fbias = (!a.out_i8 && a.bias && cov) ? __ldg(reinterpret_cast<const float *>(a.bias) + co) : 0.0f;
    const long long ibias = (a.out_i8 && a.bias && cov) ? (long long)__ldg(reinterpret_cast<const int32_t *>(a.bias) + co) : 0ll;
    const float mult = (a.out_i8 && cov) ? __ldg(a.mult + co) : 0.0f;
    // Pull the whole slice out of TMEM first and hand the buffer back.
    uint32_t acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; c += 16) tc::tmem_ld_32x16(taddr + (uint32_t)c, *reinterpret_cast<uint32_t(*)[16]>(acc + c));
    tc::tmem_ld_wait();
    tc::fence_before_sync();
    tc::mbar_arrive(tempty);

    int n = 0, oh0 = 0, ow0 = 0;
    long long m0 = 0;
    if (a.flat) {
        m0 = (long long)mt * kBMSwap;
    } else {
        const int tw = mt % a.tiles_w;
        const int t2 = mt / a.tiles_w;
        oh0 = (t2 % a.tiles_h) * a.bh;
        n = t2 / a.tiles_h;
        ow0 = tw * a.bw;
    }
    // this thread's part of the write-out: pixel gt / 8 of the chunk, channels (gt % 8) * 16 .. + 15
    const int wpx = gt >> 3;
    const int wco = nb * 128 + (gt & 7) * 16;
#pragma unroll
    for (int c = 0; c < kCols; c += 16) {
        tc::named_bar_sync(1 + grp, 128);  // the previous chunk's rows have been read
        if (a.out_i8) {
            // exact integer accumulator -> + bias -> requantise (rows of 128 bytes)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const long long v = (long long)__float2int_rn(__uint_as_float(acc[c + i])) + ibias;
                tbuf[i * kTP + row] = (uint8_t)(int8_t)requant_i8(v, mult, a.act);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float2 v = activate2_fast(
                    make_float2(__uint_as_float(acc[c + i]) + fbias, __uint_as_float(acc[c + i + 1]) + fbias), a.act);
                *reinterpret_cast<__nv_bfloat16 *>(tbuf + i * kTP + row * 2) = __float2bfloat16_rn(v.x);
                *reinterpret_cast<__nv_bfloat16 *>(tbuf + (i + 1) * kTP + row * 2) = __float2bfloat16_rn(v.y);
            }
        }
        tc::named_bar_sync(1 + grp, 128);
        const int p = c_base + c + wpx;  // pixel index inside the tile
        long long yb;
        bool valid;
        swapped_pixel(a, m0, n, oh0, ow0, p, yb, valid);
        if (valid && wco < a.Cout) {
            // 16 int8 channels per thread (Cout % 16 == 0 on this path), to
            // every upsample replica of the pixel
            const uint4 v = *reinterpret_cast<const uint4 *>(tbuf + wpx * kTP + (gt & 7) * 16);
            int8_t *dst = reinterpret_cast<int8_t *>(a.y) + yb + wco;
            const int up = FUSED ? a.om.up : 1;
            for (int dy = 0; dy < up; ++dy)
                for (int dx = 0; dx < up; ++dx)
                    *reinterpret_cast<uint4 *>(FUSED ? dst + a.om.rep(dy, dx) : dst) = v;
        }
    }
}

// bf16 output of the swapped mode.  The accumulator slice of this warp
// (lanes = 32 output channels, kCols pixel columns) is read in 16-lane x
// 8-column pieces, so that each thread holds pixel PAIRS of one channel
// (bias + packed Mish) and the pieces are 8x8 fragments: stmatrix.trans
// writes each fragment transposed, i.e. 8 channels (16 bytes) of one pixel
// per row, into the transpose rows, whose 272-byte pitch keeps the eight
// rows of a fragment on distinct banks.  The write-out is the same as the
// general epilogue's.
// FUSED: the layer has a residual or writes upsample replicas (a separate
// instantiation, so that the plain epilogue carries none of that code).
// The bias of the thread's channels (32q + 16h + 8j + lane/4 of the layer's
// single 128-channel block), read once per CTA rather than per tile (a
// global load's latency on every tile's critical path).
__device__ __forceinline__ void swapped_bias(const IgArgs &a, int q, int lane, float (&fb)[2][2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int co = 32 * q + 16 * h + 8 * j + (lane >> 2);
            fb[h][j] = (a.bias && co < a.Cout) ? __ldg(reinterpret_cast<const float *>(a.bias) + co) : 0.0f;
        }
}

template <int kCols, bool FUSED>
__device__ __forceinline__ void epilogue_swapped_bf16(const IgArgs &a, int tile, uint32_t taddr, uint32_t tempty,
                                                      int grp, int c_base, uint8_t *tbuf, int gt, int q, int lane,
                                                      const float (&fb)[2][2]) {
    const int nb = tile % a.tiles_n;
    const int mt = tile / a.tiles_n;
    // the slice in registers, then the TMEM buffer goes back to the MMA warp
    uint32_t acc[2][kCols / 8][4];  // [lane half][8-column group][fragment registers]
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int g = 0; g < kCols / 8; ++g)
            tc::tmem_ld_16x256(taddr + ((uint32_t)(16 * h) << 16) + (uint32_t)(8 * g), acc[h][g]);
    tc::tmem_ld_wait();
    tc::fence_before_sync();
    tc::mbar_arrive(tempty);

    int n = 0, oh0 = 0, ow0 = 0;
    long long m0 = 0;
    if (a.flat) {
        m0 = (long long)mt * kBMSwap;
    } else {
        const int tw = mt % a.tiles_w;
        const int t2 = mt / a.tiles_w;
        oh0 = (t2 % a.tiles_h) * a.bh;
        n = t2 / a.tiles_h;
        ow0 = tw * a.bw;
    }
    const uint32_t tb = tc::smem_u32(tbuf);
    // stmatrix row address of this thread: matrix (lane / 8) = (8-column group
    // g0 + (lane / 16), channels + 8 * ((lane / 8) & 1)), row lane % 8
    const uint32_t srow = tb + (uint32_t)((8 * (lane >> 4) + (lane & 7)) * kTP) +
                          (uint32_t)((32 * q + 8 * ((lane >> 3) & 1)) * 2);
    const int wpx = gt >> 3;
    const int wco = nb * 128 + (gt & 7) * 16;
    const __nv_bfloat16 *res = FUSED ? reinterpret_cast<const __nv_bfloat16 *>(a.om.res) : nullptr;
    // this thread's output pixel of every chunk, located up front (off the
    // chunks' barrier-to-barrier path)
    long long ybs[kCols / 16];
    bool vals[kCols / 16];
#pragma unroll
    for (int i = 0; i < kCols / 16; ++i) swapped_pixel(a, m0, n, oh0, ow0, c_base + 16 * i + wpx, ybs[i], vals[i]);
#pragma unroll
    for (int c = 0; c < kCols; c += 16) {
        // residual rows of this thread's four pixels of the chunk (pixels
        // c_base + c + 8 gg + 2 (lane % 4) + e)
        int rpix[2][2] = {{-1, -1}, {-1, -1}};  // (pixel counts are below 2^31)
        if (FUSED && res) {
#pragma unroll
            for (int gg = 0; gg < 2; ++gg)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    rpix[gg][e] = (int)swapped_pix(a, m0, n, oh0, ow0, c_base + c + 8 * gg + 2 * (lane & 3) + e);
        }
        tc::named_bar_sync(1 + grp, 128);  // the previous chunk's rows have been read
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t fr[4];
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const uint32_t(&r)[4] = acc[h][c / 8 + gg];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float2 v = activate2_fast(
                        make_float2(__uint_as_float(r[2 * j]) + fb[h][j], __uint_as_float(r[2 * j + 1]) + fb[h][j]),
                        a.act);
                    if (FUSED && res) {  // residual after the activation (channel 16 h + 8 j of the thread's rows)
                        const int co = nb * 128 + 32 * q + 16 * h + 8 * j + (lane >> 2);
                        if (co < a.Cout) {
                            if (rpix[gg][0] >= 0) v.x += __bfloat162float(res[(long long)rpix[gg][0] * a.Cout + co]);
                            if (rpix[gg][1] >= 0) v.y += __bfloat162float(res[(long long)rpix[gg][1] * a.Cout + co]);
                        }
                    }
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(v.x, v.y);
                    fr[2 * gg + j] = *reinterpret_cast<uint32_t *>(&b2);
                }
            }
            tc::stmatrix_x4_trans(srow + (uint32_t)(16 * h * 2), fr[0], fr[1], fr[2], fr[3]);
        }
        tc::named_bar_sync(1 + grp, 128);
        if (vals[c / 16]) {
            const uint4 *src = reinterpret_cast<const uint4 *>(tbuf + wpx * kTP + (gt & 7) * 32);
            const uint4 v0 = src[0], v1 = src[1];
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(a.y) + ybs[c / 16] + wco;
            const int up = FUSED ? a.om.up : 1;
            for (int dy = 0; dy < up; ++dy)
                for (int dx = 0; dx < up; ++dx) {
                    __nv_bfloat16 *d = FUSED ? dst + a.om.rep(dy, dx) : dst;
                    if (wco < a.Cout) *reinterpret_cast<uint4 *>(d) = v0;
                    if (wco + 8 < a.Cout) *reinterpret_cast<uint4 *>(d + 8) = v1;
                }
        }
    }
}

// Swapped-mode bf16 epilogue whose write-out is a TMA tensor store (plain
// layers whose tile width is a multiple of 16, or flat tiles: a 16-pixel
// chunk is then one row segment of y).  Each warp owns 32 of the 128
// accumulator rows (channels 32q .. 32q + 31) and writes them out on its own:
// its fragments are transposed by stmatrix as in epilogue_swapped_bf16, but
// into a 64-byte-swizzled [16 pixels][32 channels] box, the layout of the
// store's tensor map (chunk j of row r at chunk j ^ ((r / 2) mod 4): the rows
// of an 8 x 8 fragment on distinct banks), double-buffered per warp; the
// warp's lane 0 then issues the store and the warp goes on to the next chunk
// while the TMA engine reads the buffer.  No barrier couples the warps of a
// group, and the threads' own shared-memory loads, global stores and address
// arithmetic of the write-out disappear.
template <int kCols>
__device__ __forceinline__ void epilogue_swapped_tma(const IgArgs &a, const CUtensorMap *tmY, int mt, uint32_t taddr,
                                                     uint32_t tempty, int c_base, uint32_t wbuf, int q, int lane,
                                                     int &oc, const float (&fb)[2][2]) {
    uint32_t acc[2][kCols / 8][4];  // [lane half][8-column group][fragment registers]
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int g = 0; g < kCols / 8; ++g)
            tc::tmem_ld_16x256(taddr + ((uint32_t)(16 * h) << 16) + (uint32_t)(8 * g), acc[h][g]);
    tc::tmem_ld_wait();
    tc::fence_before_sync();
    tc::mbar_arrive(tempty);

    int n = 0, oh0 = 0, ow0 = 0;
    long long m0 = 0;
    if (a.flat) {
        m0 = (long long)mt * kBMSwap;
    } else {
        const int tw = mt % a.tiles_w;
        const int t2 = mt / a.tiles_w;
        oh0 = (t2 % a.tiles_h) * a.bh;
        n = t2 / a.tiles_h;
        ow0 = tw * a.bw;
    }
    // the chunk's tile row and first column (16-pixel chunks stay in one row)
    int dh = a.flat ? 0 : c_base / a.bw;
    int dw = a.flat ? 0 : c_base - dh * a.bw;
    // stmatrix row address of this thread in a buffer: matrix m = lane / 8
    // (pixels 8 (m / 2) + 0..7, channels 32q + 16h + 8 (m % 2) + 0..7), row
    // lane % 8: pixel r, 16-byte chunk 2h + m % 2 of its 64-byte row,
    // swizzled: chunk (2h + m % 2) ^ ((r / 2) mod 4)
    const int r = 8 * (lane >> 4) + (lane & 7);
    uint32_t coff[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
        coff[h] = (uint32_t)(r * 64) + ((uint32_t)((2 * h + ((lane >> 3) & 1)) ^ ((r >> 1) & 3)) << 4);
    const bool mine = 32 * q < a.Cout;  // (rows past Cout are never stored)
#pragma unroll
    for (int c = 0; c < kCols; c += 16) {
        const uint32_t sb = wbuf + (uint32_t)(oc & 1) * 1024u;
        // the store that last read this buffer (two chunks ago) has read it
        if (lane == 0) tc::bulk_wait_read1();
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t fr[4];
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const uint32_t(&rv)[4] = acc[h][c / 8 + gg];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float2 v = activate2_fast(
                        make_float2(__uint_as_float(rv[2 * j]) + fb[h][j], __uint_as_float(rv[2 * j + 1]) + fb[h][j]),
                        a.act);
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(v.x, v.y);
                    fr[2 * gg + j] = *reinterpret_cast<uint32_t *>(&b2);
                }
            }
            tc::stmatrix_x4_trans(sb + coff[h], fr[0], fr[1], fr[2], fr[3]);
        }
        tc::fence_proxy_async_smem();  // the staged values visible to the TMA engine
        __syncwarp();
        if (lane == 0) {
            if (mine) {
                if (a.flat)
                    tc::tma_store_2d(tmY, sb, 32 * q, (int)(m0 + c_base + c));
                else if (dh < a.bh)  // (rows past the tile belong to the next tile)
                    tc::tma_store_4d(tmY, sb, 32 * q, ow0 + dw, oh0 + dh, n);
            }
            tc::bulk_commit();
        }
        ++oc;
        if (!a.flat) {
            dw += 16;
            if (dw >= a.bw) { dw -= a.bw; ++dh; }
        }
    }
}

// SWAP = false: MMA M = 128 pixels, N = BN output channels (D[pixel][co]).
// SWAP = true (layers with Cout <= 128): the operands trade places, MMA M =
// 128 output channels (weights as A), N = 256 pixels (activations as B),
// D[co][pixel]; every MMA then has N = 256.  Measured on GB300 (one thread
// issuing back to back, M = 128, K = 16): 48 / 64 / 128 cycles for N = 64 /
// 128 / 256.  Up to N = 128 that is the time to read the operands from shared
// memory at 128 bytes a cycle ((128 + N) rows of 32 bytes); at N = 256 it is
// the tensor core's own rate, with a quarter of the shared-memory bandwidth
// left over for the TMA writes and the epilogue.
//
// PAIR (normal layout only): a cluster of two CTAs on two SMs computes a
// 256-pixel x BN tile with tcgen05's CTA-pair MMA (M = 256).  Each CTA stages
// its own 128 pixel rows and HALF of the BN weight rows; the even CTA issues
// the MMAs, which read both CTAs' shared memory and write each CTA's 128
// accumulator rows into its own TMEM.  Per SM this stages (128 + BN/2) rows
// per K block instead of 128 + BN: a third less shared-memory traffic for
// BN = 256, which is what limits the single-CTA layout on large layers.
// Both CTAs' loads complete on the even CTA's full barrier; the even CTA's
// commits arrive on both CTAs' empty / accumulator-full barriers; both CTAs'
// epilogue warps arrive on the even CTA's accumulator-empty barrier.
// FUSED: the layer has a residual or upsample replicas (conv_output_t); a
// separate instantiation, so that plain layers run none of that code.
//
// HALO (stride-1 spatial 3 x k_w layers, tile width bw a multiple of 8):
// taps (r, s) and (r + 1, s) read the same input pixels shifted by one
// output row.  So an activation slot holds, for one column shift s and
// channel block cb, the (bh + 2) x bw input pixels under the tile (one TMA
// box at (cb * BK, ow0 - pad_w + s, oh0 - pad_h, n)), and the MMAs of the
// three taps (r, s) read it from pixel row r * bw on.  An 8-row group of the
// K-major swizzled operand is 8 consecutive pixels of one tile row, so every
// tap's operand starts on a swizzle-atom boundary (r * bw rows) with the
// usual 8-row group stride.  (When bh x bw is below the MMA's 128 or 256
// pixel rows, the slot has room for the rows the last tap reads past the
// box; they are stale and their outputs are never stored.)  Per tile this
// stages k_w * (bh + 2) * bw pixel rows instead of 3 * k_w * bh * bw (480
// instead of 1152 for a 3x3 layer and an 8 x 16 tile).  A stage carries the
// box and, unless they are resident, the three taps' weight blocks: one
// barrier wait per twelve MMAs (measured: splitting the weights into a ring
// of their own, for a deeper ring, was slower).
//
// EPT (normal layout, BN <= 128, single CTAs): one epilogue per tile.  The
// four epilogue warpgroups take whole tiles in turn, each from a TMEM
// accumulator of its own (four buffers instead of two), instead of a slice
// of every tile's columns.  For layers with many short tiles, whose time
// goes to each tile's epilogue latency (TMEM load, activation, staging, TMA
// store), four tiles' epilogues then run at once; and a layer with fewer
// output channels than BN keeps every warpgroup busy.
//
// CVT == 1 (int8 layers, normal layout, single CTAs, resident weights): the
// int8 operands are widened to bf16 in the kernel instead of by a pre-pass
// (no second launch, no bf16 copy in HBM).  TMA brings the raw int8
// activation boxes into a raw ring and, once, the raw int8 weights; a
// converter warpgroup widens each raw stage into the stage's bf16 operand (an
// int8 is exact in bf16), writing it in the swizzled K-major layout the MMA
// reads (the 16-byte chunk index XOR the address bits above the row), then
// fences the writes for the tensor cores and marks the stage full.  The
// widened weights stay resident.
// CVT == 2 (bf16 layers with k_w * Cin <= 16, the image stem; BK = 16): the
// k_w taps are folded into 16 channels in the kernel instead of by a
// pre-pass.  A raw box is a run of each input row's elements (W * Cin per
// row, pixels contiguous) from an 8-element boundary at or before the tile's
// first tap (TMA reads zeros outside the row and the image: the padding);
// the converter writes, for each pixel of the stage, the k_w * Cin values
// starting at its first tap and zeros up to 16, as one 32-byte operand row.
// The raw weights arrive once by a bulk copy into the raw region, and the
// converter writes the folded resident blocks from them (each (co, r) row's
// k_w * Cin values, zero-padded) before the raw ring reuses that memory.
//
// MB == 2 (CVT == 2 with halo staging and an epilogue per tile, BN = 64): a
// tile is two 128-pixel M blocks stacked (its top and bottom bh / 2 rows),
// so the producer, the converter and the ring handshakes run once per 256
// pixels.  Each tap's MMA is issued for both blocks — the second reads the
// box's pixel rows from 128 rows further — into two BN-column accumulators
// side by side, and the epilogue stores them as two boxes of bh / 2 rows.
// The per-tile fixed costs of these roles, not their arithmetic, paced the
// one-block stem.
template <int BN, int BK, bool FLAT, bool SWAP, bool PAIR, bool FUSED, bool HALO = false, bool EPT = false,
          int CVT = 0, int MB = 1>
__global__ void __launch_bounds__(cta_threads(BN, SWAP, EPT, CVT), 1)
igemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ YMaps tmY, const IgArgs a) {
    static_assert(!(PAIR && SWAP), "the CTA-pair mode uses the normal layout");
    static_assert(!(HALO && FLAT), "halo staging is for spatial tiles");
    static_assert(!EPT || (!SWAP && !PAIR && BN <= 128), "one epilogue per tile: normal layout, BN <= 128");
    static_assert(!CVT || (!SWAP && !PAIR && !FUSED), "in-kernel widening: normal layout");
    static_assert(CVT != 2 || (BK == 16 && !FLAT), "in-kernel fold: 16-channel rows of spatial tiles");
    static_assert(MB == 1 || (CVT == 2 && HALO && EPT && MB == 2 && 4 * MB * BN <= 512),
                  "two M blocks a tile: the in-kernel stem fold, halo staging, an epilogue per tile");
    constexpr int kPix = SWAP ? kBMSwap : kBM;  // pixel rows of a tile (per CTA)
    // accumulator columns of a tile (MB = 2: the tile's two 128-pixel M blocks,
    // its top and bottom bh / 2 rows, side by side)
    constexpr int kAcc = SWAP ? kBMSwap : MB * BN;
    constexpr int kBRows = PAIR ? BN / 2 : BN;  // weight rows this CTA stages
    constexpr uint32_t kRowBytes = BK * 2;
    constexpr uint32_t kBStage = kBRows * BK * 2;  // one weight K block (this CTA's part)
    constexpr int kBufs = EPT ? 4 : 2;           // TMEM accumulators
    constexpr uint32_t kTmemCols = kBufs * kAcc;
    constexpr uint32_t kIdesc = SWAP ? tc::idesc_bf16_f32(128, kBMSwap)
                                     : tc::idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN);
    constexpr int kGroups = epi_groups(BN, SWAP, EPT);
    constexpr int kCols = EPT ? kAcc : kAcc / kGroups;  // accumulator columns per epilogue thread
    static_assert(SWAP ? (BN == 128 && kCols % 16 == 0) : (kCols % 32 == 0), "epilogue column slices");
    constexpr uint32_t kOutStage = SWAP ? 16 * kTP : kBM * 64;  // per group: transpose rows / store staging

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
    uint8_t *gbase = smem_raw + (base - raw);
    const int stages = a.stages;
    const bool wres = a.wres != 0;           // resident weights: one B slot per weight K block
    constexpr int kHaloTaps = 3;             // halo staging: k_h (3) taps per activation slot
    // activation (pixel) part of a stage; weight part (none if resident)
    // Shared memory: the ring's activation (pixel) parts, then the weights
    // (the ring's weight parts: one block per stage, three with halo staging;
    // or the resident blocks), the epilogue staging and the barriers.
    const uint32_t aStage = HALO ? a.a_stage : (uint32_t)(kPix * BK * 2);
    const uint32_t sA = base;
    const uint32_t sB = base + stages * aStage;
    const uint32_t sOut = sB + (wres ? (uint32_t)a.wblocks * kBStage : stages * (HALO ? kHaloTaps : 1) * kBStage);
    const uint32_t sBar = sOut + kGroups * a.out_bufs * kOutStage + (CVT ? a.raw_region : 0u);
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    auto empty_bar = [&](int s) { return sBar + 8u * (stages + s); };
    auto tfull_bar = [&](int b) { return sBar + 8u * (2 * stages + b); };       // b < 4
    auto tempty_bar = [&](int b) { return sBar + 8u * (2 * stages + 4 + b); };
    const uint32_t wres_bar = sBar + 8u * (2 * stages + 8);  // the resident weights have landed
    // CVT: the raw region (between the epilogue staging and the barriers),
    // its ring's barriers, and the raw weights' barrier
    const uint32_t sRaw = sOut + kGroups * a.out_bufs * kOutStage;
    auto raw_full_bar = [&](int s) { return sBar + 8u * (2 * stages + 9 + s); };
    auto raw_empty_bar = [&](int s) { return sBar + 8u * (3 * stages + 9 + s); };
    const uint32_t wraw_bar = sBar + 8u * (4 * stages + 9);
    uint8_t *gmisc = gbase + (sBar - base) + 8u * (CVT ? 4 * stages + 10 : 2 * stages + 9);
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(gmisc);
    // the bias copy (fp32 or int32 [Cout]) and, int8, the multipliers [Cout]
    const uint32_t sBias = (sBar + 8u * (CVT ? 4 * stages + 10 : 2 * stages + 9) + 16u + 15u) & ~15u;
    const uint32_t sMult = sBias + (uint32_t)((a.Cout * 4 + 15) & ~15);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gmisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work unit: the CTA, or in pair mode the cluster (CTAs 2u and 2u + 1).
    const uint32_t rank = PAIR ? tc::cluster_ctarank() : 0u;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            // (CVT: filled by the four converter warps, each for its own rows)
            tc::mbar_init(full_bar(s), CVT ? 4 : 1);
            tc::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kBufs; ++b) {
            tc::mbar_init(tfull_bar(b), 1);
            // emptied by every epilogue thread (EPT: of one warpgroup); pair: by each warp
            tc::mbar_init(tempty_bar(b), EPT ? 128 : (PAIR ? 2 * 4 * kGroups : 128 * kGroups));
        }
        tc::mbar_init(wres_bar, 1);
        if constexpr (CVT) {
            for (int s = 0; s < stages; ++s) {
                tc::mbar_init(raw_full_bar(s), 1);
                tc::mbar_init(raw_empty_bar(s), 4);
            }
            tc::mbar_init(wraw_bar, 1);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
        tc::tma_prefetch_desc(&tmY.m[0]);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tc::tmem_alloc_pair(tc::smem_u32((const void *)tmem_holder), kTmemCols);
            tc::tmem_relinquish_pair();
        } else {
            tc::tmem_alloc(tc::smem_u32((const void *)tmem_holder), kTmemCols);
            tc::tmem_relinquish();
        }
    }
    // __syncthreads is an aligned barrier: every warp must reach it converged.
    __syncwarp();
    tc::fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) tc::cluster_sync();  // the peer's barriers are initialised
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    // set-up done: let the next kernel be scheduled, and wait for the
    // previous one's writes before the first global access
    pdl_trigger();
    // Before that wait, the operand boxes of this CTA's first ring stages go
    // into L2 (when the previous kernel's last CTAs still run on other SMs,
    // its tail hides their latency).  L2 is where global writes land, so this
    // cannot serve stale bytes to the loads after the wait.
    if (!CVT && threadIdx.x == 0 && unit < a.num_tiles) {
        const int tile = unit;
        const int nb = tile % a.tiles_n;
        const int mt = PAIR ? (tile / a.tiles_n) * 2 + (int)rank : tile / a.tiles_n;
        int n = 0, oh0 = 0, ow0 = 0;
        if (!FLAT) {
            const int tw = mt % a.tiles_w;
            const int t2 = mt / a.tiles_w;
            oh0 = (t2 % a.tiles_h) * a.bh;
            n = t2 / a.tiles_h;
            ow0 = tw * a.bw;
        }
        const int kpre = a.kblocks < stages ? a.kblocks : stages;
        int r = 0, s = 0, cb = 0;
        for (int kb = 0; kb < kpre; ++kb) {
            if (FLAT) {
                tc::tma_prefetch_l2_2d(&tmA, cb * BK, mt * kPix);
            } else if (HALO) {
                tc::tma_prefetch_l2_4d(&tmA, cb * BK, ow0 - a.pad_w + s, oh0 - a.pad_h, n);
            } else {
                tc::tma_prefetch_l2_4d(&tmA, cb * BK, ow0 * a.stride - a.pad_w + s, oh0 * a.stride - a.pad_h + r, n);
            }
            if (!wres) {
                const int kx = ((HALO ? 0 : r) * a.KW + s) * a.Cin + cb * BK;
                tc::tma_prefetch_l2_2d(&tmB, kx, nb * BN + (PAIR ? (int)rank * kBRows : 0));
            }
            if (++cb == a.cblocks) {
                cb = 0;
                if (++s == a.KW) { s = 0; if (!HALO) ++r; }
            }
        }
    }
    pdl_wait();

    // CVT == 1: int8 -> bf16 (exact) into the swizzled K-major operand, rows
    // [0, rows) of BK bytes at src, items (row, 16-byte chunk) t, t + T, ...:
    // chunk j of row r goes to chunk j ^ ((r * row bytes) >> 7 & (chunks - 1))
    // of the row (the 128-, 64- or 32-byte swizzle of a 1024-aligned slot)
    constexpr int kChunks = BK / 8;  // 16-byte bf16 chunks per row
    auto widen_span = [&](uint32_t src, uint32_t dst, int rows, int t, int T) {
        for (int idx = t; idx < rows * kChunks; idx += T) {
            const int r = idx / kChunks, j = idx % kChunks;
            uint32_t lo, hi;  // 8 int8 values
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(src + (uint32_t)(r * BK + j * 8)));
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t wd = e < 2 ? lo : hi;
                const int sh = (e & 1) * 16;
                const float f0 = (float)(int8_t)(wd >> sh), f1 = (float)(int8_t)(wd >> (sh + 8));
                // bf16 of a small integer is its float's upper half, exactly
                o[e] = (__float_as_uint(f0) >> 16) | (__float_as_uint(f1) & 0xffff0000u);
            }
            const uint32_t sw = (uint32_t)((r * kRowBytes) >> 7) & (uint32_t)(kChunks - 1);
            const uint32_t d = dst + (uint32_t)(r * kRowBytes) + (((uint32_t)j ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d), "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                         : "memory");
        }
    };
    // CVT == 1: the resident weights (every K block, [kBRows x BK] each, the
    // blocks contiguous in the raw region and in sB) are widened once by the
    // converter and the epilogue warps together (the latter idle until the
    // first accumulator), after which the converter marks them resident.
    constexpr int kWidenThreads = 128 * (kGroups + 1);
    auto widen_weights = [&]() {
        const int t = (int)threadIdx.x - 64;  // epilogue warps, then the converter warpgroup
        if (wait_bounded(wraw_bar, 0u, abort_flag, a.status, KSTATUS_TIMEOUT_EPILOGUE)) {
            widen_span(sRaw, sB, a.wblocks * kBRows, t, kWidenThreads);
            tc::fence_proxy_async_smem();  // the widened weights visible to the tensor cores
        }
        tc::named_bar_sync(7, kWidenThreads);  // (reached by every thread: the wait is bounded)
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // pair mode: both CTAs' loads complete on the even CTA's barriers
            const uint32_t full0 = PAIR ? tc::mapa_shared(full_bar(0), 0) : full_bar(0);
            if (CVT == 2 && unit < a.num_tiles) {
                // the raw weights [Cout][k_h][k_w x Cin] into the raw region, as
                // they are (one bulk copy); the converter folds them into the
                // resident blocks, and only then may the raw ring be filled
                const uint32_t wbytes = (uint32_t)(a.Cout * a.KH * a.fold_kw * a.fold_cin * 2);
                tc::mbar_arrive_expect_tx(wraw_bar, wbytes);
                tc::bulk_load(sRaw, a.w_raw, wbytes, wraw_bar);
                ok = wait_bounded(wres_bar, 0u, abort_flag, a.status, KSTATUS_TIMEOUT_PRODUCER);
            } else if (CVT == 1 && unit < a.num_tiles) {
                // the raw int8 weights into the raw region, once; the converter
                // widens them into the resident blocks, and only then may the
                // raw ring (the same memory) be filled
                tc::mbar_arrive_expect_tx(wraw_bar, (uint32_t)a.wblocks * kBRows * BK);
                int r = 0, s = 0, cb = 0;
                for (int kb = 0; kb < a.wblocks; ++kb) {
                    tc::tma_load_2d(sRaw + (uint32_t)kb * kBRows * BK, &tmB, wraw_bar, (r * a.KW + s) * a.Cin + cb * BK, 0);
                    if (++cb == a.cblocks) {
                        cb = 0;
                        if (++s == a.KW) { s = 0; ++r; }
                    }
                }
                ok = wait_bounded(wres_bar, 0u, abort_flag, a.status, KSTATUS_TIMEOUT_PRODUCER);
            } else if (wres && unit < a.num_tiles) {
                // every K block of the (single) N block of weights, once; pair
                // mode: each CTA its half, both completing on the even CTA's barrier
                const uint32_t wbar = PAIR ? tc::mapa_shared(wres_bar, 0) : wres_bar;
                if (rank == 0) tc::mbar_arrive_expect_tx(wres_bar, (PAIR ? 2u : 1u) * (uint32_t)a.wblocks * kBStage);
                int r = 0, s = 0, cb = 0;
                for (int kb = 0; kb < a.wblocks; ++kb) {
                    const int kx = (r * a.KW + s) * a.Cin + cb * BK;
                    if constexpr (PAIR)
                        tc::tma_load_2d_pair(sB + kb * kBStage, &tmB, wbar, kx, (int)rank * kBRows);
                    else
                        tc::tma_load_2d(sB + kb * kBStage, &tmB, wres_bar, kx, 0);
                    if (++cb == a.cblocks) {
                        cb = 0;
                        if (++s == a.KW) { s = 0; ++r; }
                    }
                }
            }
            // (single CTAs: the tiles' coordinates advanced without division,
            // which would sit in this thread's per-tile latency chain)
            TileWalk pwalk;
            if (!PAIR) pwalk.init(a, unit, units);
            for (int tile = unit; tile < a.num_tiles && ok; tile += units) {
                const int nb = PAIR ? tile % a.tiles_n : pwalk.nb;
                // pair mode: this CTA's pixel tile (past tiles_m: an empty
                // half, loaded as zeros from outside the tensor, never stored)
                const int mt = PAIR ? (tile / a.tiles_n) * 2 + (int)rank : pwalk.mt;
                int n = 0, oh0 = 0, ow0 = 0;
                int m0 = 0;
                if (FLAT) {
                    m0 = mt * kPix;
                } else if (PAIR) {
                    const int tw = mt % a.tiles_w;
                    const int t2 = mt / a.tiles_w;
                    oh0 = (t2 % a.tiles_h) * a.bh;
                    n = t2 / a.tiles_h;
                    ow0 = tw * a.bw;
                } else {
                    oh0 = pwalk.th * a.bh;
                    n = pwalk.n;
                    ow0 = pwalk.tw * a.bw;
                }
                if (!PAIR) pwalk.advance(a);
                if constexpr (CVT) {
                    // raw int8 activation boxes into the raw ring (per-tap or halo
                    // boxes, in the K block order of the plain variants)
                    int r = 0, s = 0, cb = 0;
                    for (int kb = 0; kb < a.kblocks; ++kb) {
                        if (!wait_bounded(raw_empty_bar(stage), phase ^ 1u, abort_flag, a.status,
                                          KSTATUS_TIMEOUT_PRODUCER)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dR = sRaw + stage * a.raw_stage;
                        tc::mbar_arrive_expect_tx(raw_full_bar(stage), a.a_bytes);
                        if (CVT == 2) {
                            // the input rows' element runs from the 8-element boundary at
                            // or before the tile's first tap (16-byte aligned start)
                            const int v = (ow0 * a.stride - a.fold_padw) * a.fold_cin;
                            const int x0 = v >= 0 ? (v & ~7) : -((-v + 7) & ~7);
                            const int c2 = HALO ? oh0 - a.pad_h : oh0 * a.stride - a.pad_h + r;
                            tc::tma_load_3d(dR, &tmA, raw_full_bar(stage), x0, c2, n);
                        } else if (FLAT) {
                            tc::tma_load_2d(dR, &tmA, raw_full_bar(stage), cb * BK, m0);
                        } else {
                            const int c1 = ow0 * a.stride - a.pad_w + s, c2 = oh0 * a.stride - a.pad_h + r;
                            tc::tma_load_4d(dR, &tmA, raw_full_bar(stage), cb * BK, c1, c2, n);
                        }
                        if (++stage == stages) { stage = 0; phase ^= 1u; }
                        if (++cb == a.cblocks) {
                            cb = 0;
                            if (++s == a.KW) { s = 0; if (!HALO) ++r; }
                        }
                    }
                    continue;
                }
                if constexpr (HALO) {
                    // K blocks (s, cb), cb fastest: a stage holds the halo box and
                    // (unless resident) the weight blocks of taps r = 0 .. 2
                    int s = 0, cb = 0;
                    for (int kb = 0; kb < a.kblocks; ++kb) {
                        if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.status,
                                          KSTATUS_TIMEOUT_PRODUCER)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dB = sB + stage * (kHaloTaps * kBStage);
                        const uint32_t bytes = a.a_bytes + (wres ? 0u : kHaloTaps * kBStage);
                        const uint32_t fb = PAIR ? full0 + 8u * stage : full_bar(stage);
                        if (!PAIR || rank == 0) tc::mbar_arrive_expect_tx(full_bar(stage), (PAIR ? 2u : 1u) * bytes);
                        const int c1 = ow0 - a.pad_w + s, c2 = oh0 - a.pad_h;
                        if (PAIR) tc::tma_load_4d_pair(sA + stage * aStage, &tmA, fb, cb * BK, c1, c2, n);
                        else tc::tma_load_4d(sA + stage * aStage, &tmA, fb, cb * BK, c1, c2, n);
                        if (!wres) {
#pragma unroll
                            for (int t = 0; t < kHaloTaps; ++t) {
                                const int kx = (t * a.KW + s) * a.Cin + cb * BK;
                                if (PAIR)
                                    tc::tma_load_2d_pair(dB + t * kBStage, &tmB, fb, kx, nb * BN + (int)rank * kBRows);
                                else
                                    tc::tma_load_2d(dB + t * kBStage, &tmB, fb, kx, nb * BN);
                            }
                        }
                        if (++stage == stages) { stage = 0; phase ^= 1u; }
                        if (++cb == a.cblocks) { cb = 0; ++s; }
                    }
                    continue;
                }
                // K block order: (r, s, cb), cb fastest
                int r = 0, s = 0, cb = 0;
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.status,
                                      KSTATUS_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dA = sA + stage * aStage;
                    const uint32_t dB = sB + stage * kBStage;
                    const uint32_t bytes = a.a_bytes + (wres ? 0u : kBStage);
                    const uint32_t fb = PAIR ? full0 + 8u * stage : full_bar(stage);
                    if (!PAIR || rank == 0) tc::mbar_arrive_expect_tx(full_bar(stage), (PAIR ? 2u : 1u) * bytes);
                    if (FLAT) {
                        if (PAIR) tc::tma_load_2d_pair(dA, &tmA, fb, cb * BK, m0);
                        else tc::tma_load_2d(dA, &tmA, fb, cb * BK, m0);
                    } else {
                        const int c1 = ow0 * a.stride - a.pad_w + s, c2 = oh0 * a.stride - a.pad_h + r;
                        if (PAIR) tc::tma_load_4d_pair(dA, &tmA, fb, cb * BK, c1, c2, n);
                        else tc::tma_load_4d(dA, &tmA, fb, cb * BK, c1, c2, n);
                    }
                    if (!wres) {
                        const int kx = (r * a.KW + s) * a.Cin + cb * BK;
                        if (PAIR) tc::tma_load_2d_pair(dB, &tmB, fb, kx, nb * BN + (int)rank * kBRows);
                        else tc::tma_load_2d(dB, &tmB, fb, kx, nb * BN);
                    }
                    if (++stage == stages) { stage = 0; phase ^= 1u; }
                    if (++cb == a.cblocks) {
                        cb = 0;
                        if (++s == a.KW) { s = 0; ++r; }
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (pair mode: even CTA only)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int lt = 0;
            if (wres && unit < a.num_tiles) {  // the resident weights are in shared memory
                ok = wait_bounded(wres_bar, 0u, abort_flag, a.status, KSTATUS_TIMEOUT_MMA);
                tc::fence_after_sync();
            }
            for (int tile = unit; tile < a.num_tiles && ok; tile += units, ++lt) {
                const int buf = lt % kBufs;
                const uint32_t use = (uint32_t)(lt / kBufs);
                if (!wait_bounded<PAIR>(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag, a.status,
                                        KSTATUS_TIMEOUT_MMA))
                    break;
                tc::fence_after_sync();
                const uint32_t d = tmem_base + (uint32_t)(buf * kAcc);
                if constexpr (HALO) {
                    // K blocks (s, cb): tap r reads the halo box from pixel row
                    // r * bw; its weights are the stage's r-th block, or the
                    // resident block (r * KW + s) * cblocks + cb.  The operand
                    // descriptors are formed before the wait: the start address is a
                    // descriptor's low field (address / 16, below 2^14), so the
                    // operand at base + off has descriptor desc(base) + off / 16.
                    int s = 0, cb = 0;
                    const uint64_t p_tap = (uint64_t)(((uint32_t)a.bw * kRowBytes) >> 4);
                    const uint64_t w_tap = wres ? (uint64_t)(a.KW * a.cblocks) * (kBStage >> 4) : (uint64_t)(kBStage >> 4);
                    for (int kb = 0; kb < a.kblocks; ++kb) {
                        const uint64_t pd0 = tc::smem_desc_kmajor(sA + stage * aStage, kRowBytes);  // pixels
                        const uint64_t wd0 = tc::smem_desc_kmajor(                                 // weights
                            wres ? sB + (uint32_t)(s * a.cblocks + cb) * kBStage : sB + stage * (kHaloTaps * kBStage),
                            kRowBytes);
                        if (!wait_bounded(full_bar(stage), phase, abort_flag, a.status, KSTATUS_TIMEOUT_MMA)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
#pragma unroll
                        for (int t = 0; t < kHaloTaps; ++t) {
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k) {
                                const uint64_t pd = pd0 + (uint64_t)t * p_tap + 2u * k;  // +32 bytes per K = 16 step
                                const uint64_t wd = wd0 + (uint64_t)t * w_tap + 2u * k;
                                const uint32_t accum = (kb | t | k) != 0 ? 1u : 0u;
                                if (PAIR)
                                    tc::mma_bf16_pair(d, pd, wd, kIdesc, accum);
                                else if (SWAP)
                                    tc::mma_bf16(d, wd, pd, kIdesc, accum);
                                else {
                                    // (MB = 2: block j's pixel rows start 128 rows further
                                    // into the box, its accumulator BN columns further)
#pragma unroll
                                    for (int j = 0; j < MB; ++j)
                                        tc::mma_bf16(d + (uint32_t)(j * BN), pd + (uint64_t)(j * kBM * kRowBytes / 16), wd,
                                                     kIdesc, accum);
                                }
                            }
                        }
                        if (++cb == a.cblocks) { cb = 0; ++s; }
                        // stage free (in both CTAs of a pair) once these MMAs complete
                        if (PAIR)
                            tc::mma_commit_pair(empty_bar(stage), 0x3);
                        else
                            tc::mma_commit(empty_bar(stage));
                        if (++stage == stages) { stage = 0; phase ^= 1u; }
                    }
                } else {
                    for (int kb = 0; kb < a.kblocks; ++kb) {
                        if (!wait_bounded(full_bar(stage), phase, abort_flag, a.status, KSTATUS_TIMEOUT_MMA)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint32_t aS = sA + stage * aStage;
                        const uint32_t bS = sB + (wres ? kb : stage) * kBStage;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint64_t pd = tc::smem_desc_kmajor(aS + 32u * k, kRowBytes);  // pixels
                            const uint64_t wd = tc::smem_desc_kmajor(bS + 32u * k, kRowBytes);  // weights
                            if (PAIR)
                                tc::mma_bf16_pair(d, pd, wd, kIdesc, (kb | k) != 0 ? 1u : 0u);
                            else if (SWAP)
                                tc::mma_bf16(d, wd, pd, kIdesc, (kb | k) != 0 ? 1u : 0u);
                            else
                                tc::mma_bf16(d, pd, wd, kIdesc, (kb | k) != 0 ? 1u : 0u);
                        }
                        // stage free (in both CTAs of a pair) once these MMAs complete
                        if (PAIR)
                            tc::mma_commit_pair(empty_bar(stage), 0x3);
                        else
                            tc::mma_commit(empty_bar(stage));
                        if (++stage == stages) { stage = 0; phase ^= 1u; }
                    }
                }
                if (ok) {  // accumulator ready
                    if (PAIR)
                        tc::mma_commit_pair(tfull_bar(buf), 0x3);
                    else
                        tc::mma_commit(tfull_bar(buf));
                }
            }
        }
    } else if (CVT && warp >= 2 + 4 * kGroups) {
        // ------------------------------------------------ converter (the last warpgroup)
        const int ct = threadIdx.x - (64 + 128 * kGroups);
        auto widen = [&](uint32_t src, uint32_t dst, int rows) { widen_span(src, dst, rows, ct, 128); };
        // (The folded weights' one-time wait:) one thread does the bounded wait
        // and tells the others through shared memory, so that the warpgroup
        // gives up, if it must, as one (a hardware named barrier has no time
        // limit).
        volatile int *go = reinterpret_cast<volatile int *>(gmisc + 8);
        auto all_ok = [&](bool mine) {
            if (ct == 0) *go = mine ? 1 : 0;
            tc::named_bar_sync(6, 128);
            const bool r = *go != 0;
            tc::named_bar_sync(6, 128);  // everyone has read it before it changes
            return r;
        };
        bool ok = true;
        // CVT == 2: folded operand row m (16 bf16, two 16-byte chunks) from the
        // k_w x Cin consecutive bf16 at element e of the shared buffer `src`,
        // then zeros: nine 32-bit words from the one holding element e (the
        // buffers have 36 bytes of slack after their last row), realigned by
        // a funnel shift, the elements past k_w x Cin masked
        const int kwc = CVT == 2 ? a.fold_kw * a.fold_cin : 0;
        auto fold_load = [&](uint32_t src, int e, uint32_t (&w)[9]) {
            const uint32_t wa = src + (uint32_t)(e & ~1) * 2u;
#pragma unroll
            for (int k = 0; k < 9; ++k)
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[k]) : "r"(wa + 4u * k) : "memory");
        };
        // (output word i keeps its elements 2i, 2i + 1 below k_w x Cin)
        uint32_t keep[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) keep[i] = 2 * i + 1 < kwc ? 0xffffffffu : (2 * i < kwc ? 0xffffu : 0u);
        auto fold_store = [&](const uint32_t (&w)[9], int e, uint32_t dst, int m) {
            const uint32_t sh = (uint32_t)(e & 1) * 16u;  // an odd first element: shift by one
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = __funnelshift_r(w[i], w[i + 1], sh) & keep[i];
            const uint32_t sw = (uint32_t)((m * kRowBytes) >> 7) & (uint32_t)(kChunks - 1);
            const uint32_t d = dst + (uint32_t)(m * kRowBytes);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d + ((0u ^ sw) << 4)), "r"(o[0]), "r"(o[1]),
                         "r"(o[2]), "r"(o[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(d + ((1u ^ sw) << 4)), "r"(o[4]), "r"(o[5]),
                         "r"(o[6]), "r"(o[7])
                         : "memory");
        };
        auto fold_row = [&](uint32_t src, int e, uint32_t dst, int m) {
            uint32_t w[9];
            fold_load(src, e, w);
            fold_store(w, e, dst, m);
        };
        if (CVT == 2 && unit < a.num_tiles) {
            // the folded weights: row co of K block r holds w[co][r][s][ci] at
            // s * Cin + ci (zero past k_w x Cin and for co >= Cout)
            ok = all_ok(ct != 0 || wait_bounded(wraw_bar, 0u, abort_flag, a.status, KSTATUS_TIMEOUT_EPILOGUE));
            if (ok) {
                (void)tc::mbar_try_wait(wraw_bar, 0u);  // (complete: each thread's own acquire of the bytes)
                for (int idx = ct; idx < a.wblocks * kBRows; idx += 128) {
                    const int kb = idx / kBRows, co = idx - kb * kBRows;
                    if (co < a.Cout) {
                        fold_row(sRaw, (co * a.KH + kb) * kwc, sB + (uint32_t)kb * kBStage, co);
                    } else {
                        const uint32_t d = sB + (uint32_t)kb * kBStage + (uint32_t)(co * kRowBytes);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d + 16u), "r"(0u) : "memory");
                    }
                }
                tc::fence_proxy_async_smem();  // the folded weights visible to the tensor cores
                tc::named_bar_sync(6, 128);
                if (ct == 0) tc::mbar_arrive(wres_bar);
            }
        } else if (CVT == 1 && unit < a.num_tiles) {
            widen_weights();
            ok = *abort_flag == 0;  // (a thread that gave up has raised it)
            if (ok && ct == 0) tc::mbar_arrive(wres_bar);
        }
        // CVT == 2: this thread's box rows m = ct + 128 i (at most three: a box
        // has at most 128 + 2 bw <= 384 rows), pixel (m / bw, m % bw), whose taps
        // start at element (m / bw) x raw_inner + (m % bw) x stride x Cin + e0
        // of the raw stage; e0 = (tile column x bw x stride - pad_w) x Cin mod 8
        // (the producer starts the box on the 8-element boundary at or below).
        int roff[3] = {0, 0, 0};
        int nrows = 0;
        int tw = 0, nb = 0, dn = 0, dw = 0;
        const int e_col = CVT == 2 ? a.bw * a.stride * a.fold_cin : 0, e_pad = CVT == 2 ? a.fold_padw * a.fold_cin : 0;
        if constexpr (CVT == 2) {
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const int m = ct + 128 * i;
                if (m < a.box_rows) {
                    roff[i] = (m / a.bw) * a.raw_inner + (m % a.bw) * a.stride * a.fold_cin;
                    nrows = i + 1;
                }
            }
            // the CTA's tiles tile = unit + k units: their N block and tile column,
            // advanced without division
            nb = unit % a.tiles_n;
            tw = (unit / a.tiles_n) % a.tiles_w;
            dn = units % a.tiles_n;
            dw = (units / a.tiles_n) % a.tiles_w;
        }
        // The ring: each converter warp waits for the stage on its own (every
        // lane, bounded), converts its own rows (those of its lanes' thread
        // indices), and hands them on with one arrival per warp on the
        // raw-empty and full barriers (four each), so that the warps run
        // independently of one another.
        const int cl = ct & 31;
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = unit; tile < a.num_tiles && ok; tile += units) {
            const int e0 = (tw * e_col - e_pad) & 7;
            if constexpr (CVT == 2) {
                nb += dn;
                const int carry = nb >= a.tiles_n ? 1 : 0;
                nb -= carry * a.tiles_n;
                tw += dw + carry;
                if (tw >= a.tiles_w) tw -= a.tiles_w;
            }
            for (int kb = 0; kb < a.kblocks; ++kb) {
                // raw stage landed, and its operand slot consumed by the MMAs
                // (each lane's own acquire of the TMA bytes and of the slot)
                const bool got =
                    wait_bounded(raw_full_bar(stage), phase, abort_flag, a.status, KSTATUS_TIMEOUT_EPILOGUE) &&
                    wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.status, KSTATUS_TIMEOUT_EPILOGUE);
                ok = __all_sync(0xffffffffu, got);
                if (!ok) break;
                if constexpr (CVT == 2) {
                    // (every row's loads issued before the first row's stores)
                    const uint32_t rw = sRaw + stage * a.raw_stage, dA = sA + stage * aStage;
                    uint32_t w0[9], w1[9], w2[9];
                    if (nrows > 0) fold_load(rw, roff[0] + e0, w0);
                    if (nrows > 1) fold_load(rw, roff[1] + e0, w1);
                    if (nrows > 2) fold_load(rw, roff[2] + e0, w2);
                    if (nrows > 0) fold_store(w0, roff[0] + e0, dA, ct);
                    if (nrows > 1) fold_store(w1, roff[1] + e0, dA, ct + 128);
                    if (nrows > 2) fold_store(w2, roff[2] + e0, dA, ct + 256);
                } else {
                    widen(sRaw + stage * a.raw_stage, sA + stage * aStage, a.box_rows);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();  // the warp's rows are written
                if (cl == 0) {
                    tc::mbar_arrive(raw_empty_bar(stage));
                    tc::mbar_arrive(full_bar(stage));
                }
                if (++stage == stages) { stage = 0; phase ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2 ..)
        // tcgen05.ld lets warp w reach TMEM lanes 32 * (w % 4) .. + 31, so every
        // run of four consecutive warps covers the 128 accumulator rows; warp
        // group g (warps 2 + 4g .. 5 + 4g) drains columns [g * kCols, (g+1) * kCols)
        // (EPT: all columns of every 4th tile, from accumulator g).
        // The bias (and the int8 multipliers), once per CTA into shared
        // memory: the epilogue of each tile then reads them there instead of
        // waiting on global loads (~0.5 us on a layer of one tile per CTA).
        if (a.bias_smem) {
            const int et = (int)threadIdx.x - 64;
            for (int i = et; i < a.Cout; i += 128 * kGroups) {
                if (a.bias) {
                    const uint32_t bv = __ldg(reinterpret_cast<const uint32_t *>(a.bias) + i);
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(sBias + 4u * (uint32_t)i), "r"(bv) : "memory");
                }
                if (a.out_i8) {
                    const uint32_t mv = __float_as_uint(__ldg(a.mult + i));
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(sMult + 4u * (uint32_t)i), "r"(mv) : "memory");
                }
            }
            tc::named_bar_sync(5, 128 * kGroups);
        }
        const int q = warp & 3;
        const int grp = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const int c_base = EPT ? 0 : grp * kCols;
        const bool issuer = ((warp - 2) & 3) == 0 && lane == 0;  // issues the group's TMA stores
        const uint32_t sStage = sOut + (uint32_t)(grp * a.out_bufs) * kOutStage;  // this group's staging
        int oc = 0;  // TMA stores this group has issued (selects the staging buffer)
        // pair mode: accumulator-empty arrivals go to the even CTA's barrier
        const uint32_t tempty0 = PAIR ? tc::mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
        if (CVT == 1 && unit < a.num_tiles) widen_weights();
        // lt: the CTA's local tile index (EPT: this group's tiles, every 4th)
        const int lt0 = EPT ? grp : 0, lstep = EPT ? kGroups : 1;
        // swapped bf16 layers: this thread's bias values, read once
        float swb[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (SWAP && !a.out_i8) swapped_bias(a, q, lane, swb);
        // (single CTAs: the tiles' coordinates advanced without division)
        TileWalk walk;
        walk.init(a, unit + lt0 * units, lstep * units);
        for (int tile = unit + lt0 * units, lt = lt0; tile < a.num_tiles;
             tile += lstep * units, lt += lstep, walk.advance(a)) {
            const int buf = lt % kBufs;
            const uint32_t use = (uint32_t)(lt / kBufs);
            const bool got = wait_bounded(tfull_bar(buf), use & 1u, abort_flag, a.status,
                                          KSTATUS_TIMEOUT_EPILOGUE);
            __syncwarp();  // tcgen05.ld below is warp-collective (.sync.aligned)
            if (!__all_sync(0xffffffffu, got)) break;
            tc::fence_after_sync();
            if constexpr (SWAP) {
                const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kAcc + c_base);
                uint8_t *tb = gbase + (sOut - base) + grp * a.out_bufs * kOutStage;
                if constexpr (!FUSED) {
                    if (a.out_bufs == 2) {  // plain bf16, 16-pixel chunks in one row: TMA-store write-out
                        epilogue_swapped_tma<kCols>(a, &tmY.m[0], tile, ta, tempty_bar(buf), c_base,
                                                    sOut + (uint32_t)(grp * 2) * 4096u + (uint32_t)q * 2048u, q,
                                                    lane, oc, swb);
                        continue;
                    }
                }
                if (a.out_i8)
                    epilogue_swapped<kCols, FUSED>(a, tile, ta, tempty_bar(buf), row, grp, c_base, tb,
                                                   threadIdx.x - 64 - grp * 128);
                else
                    epilogue_swapped_bf16<kCols, FUSED>(a, tile, ta, tempty_bar(buf), grp, c_base, tb,
                                                        threadIdx.x - 64 - grp * 128, q, lane, swb);
                continue;
            }
            // Plain layers pull this thread's whole accumulator slice out of
            // TMEM and hand the buffer back to the MMA warp at once; FUSED
            // layers (registers for the residual) read it 32 columns at a time
            // and hand it back after the last chunk.
            // (EPT: a whole tile's columns would not fit in registers; the
            // buffer is this group's alone, so it can wait for the last chunk)
            constexpr bool kChunked = FUSED || EPT;
            constexpr int kAccRegs = kChunked ? 32 : kCols;
            uint32_t acc[kAccRegs];
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kAcc + c_base);
            auto release = [&]() {
                tc::fence_before_sync();
                if constexpr (PAIR) {
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive_cluster(tempty0 + 8u * buf);
                } else {
                    tc::mbar_arrive(tempty_bar(buf));
                }
            };
            if constexpr (!kChunked) {
#pragma unroll
                for (int c = 0; c < kCols; c += 32)
                    tc::tmem_ld_32x32(tbase + (uint32_t)c, *reinterpret_cast<uint32_t(*)[32]>(acc + c));
                tc::tmem_ld_wait();
                release();
            }

            // Output slice: bias, activation, bf16, staged in shared memory
            // (64-byte swizzle, matching the store's tensor map) and written by
            // one TMA tensor store per 32 columns.  The box is the tile's
            // bh x bw pixel rectangle (or 128 flat rows): rows past it are
            // never stored and pixels outside the image are clipped by TMA.
            const int nb = PAIR ? tile % a.tiles_n : walk.nb;
            const int mt = PAIR ? (tile / a.tiles_n) * 2 + (int)rank : walk.mt;
            if (PAIR && mt >= a.tiles_m) {  // the empty half of the last pair tile
                if constexpr (kChunked) release();
                continue;
            }
            int n = 0, oh0 = 0, ow0 = 0, m0 = 0;
            if (FLAT) {
                m0 = mt * kPix;
            } else if (PAIR) {
                const int tw = mt % a.tiles_w;
                const int t2 = mt / a.tiles_w;
                oh0 = (t2 % a.tiles_h) * a.bh;
                n = t2 / a.tiles_h;
                ow0 = tw * a.bw;
            } else {
                oh0 = walk.th * a.bh;
                n = walk.n;
                ow0 = walk.tw * a.bw;
            }
            const uint32_t swz = (uint32_t)((row >> 1) & 3);
            // residual pixel of this thread's row (-1: none, or outside the image;
            // pixel counts are below 2^31)
            int rpix = -1;
            if (FUSED && a.om.res) {
                if (FLAT) {
                    if ((long long)m0 + row < a.M) rpix = m0 + row;
                } else if (row < a.bw * a.bh) {
                    const int dh = row / a.bw;
                    const int oh = oh0 + dh, ow = ow0 + (row - dh * a.bw);
                    if (oh < a.OH && ow < a.OW) rpix = (n * a.OH + oh) * a.OW + ow;
                }
            }
#pragma unroll
            for (int c = 0; c < kCols; c += 32) {
                // (MB = 2: columns [j BN, (j + 1) BN) are M block j, rows j bh / 2 ..)
                const int jb = MB == 1 ? 0 : c / BN;
                const int co = nb * BN + c_base + (MB == 1 ? c : c - jb * BN);
                const bool live = co < a.Cout;  // the same for the whole group
                if constexpr (kChunked) {
                    if (live) {
                        tc::tmem_ld_32x32(tbase + (uint32_t)c, *reinterpret_cast<uint32_t(*)[32]>(acc));
                        tc::tmem_ld_wait();
                    }
                    if (c + 32 == kCols) release();
                }
                if (!live) continue;
                const uint32_t *av = acc + (kChunked ? 0 : c);  // this chunk's 32 accumulator columns
                const uint32_t sbuf = sStage + (uint32_t)(oc & (a.out_bufs - 1)) * kOutStage;
                const uint32_t srow = sbuf + (uint32_t)row * 64u;
                // the store that last used this staging buffer has read it
                // (with two buffers that is every store but the latest)
                if (issuer) {
                    if (a.out_bufs == 2)
                        tc::bulk_wait_read1();
                    else
                        tc::bulk_wait_read0();
                }
                tc::named_bar_sync(1 + grp, 128);
                if (a.out_i8) {
                    // int8 output: the accumulator is an exact integer (< 2^24);
                    // + int32 bias, requantise, saturate.  Rows of 32 bytes,
                    // stored unswizzled (the int8 store map has no swizzle).
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int cc = co + e;
                        long long v = (long long)__float2int_rn(__uint_as_float(av[e]));
                        float mlt;
                        if (a.bias_smem) {
                            int32_t bi = 0;
                            if (a.bias)
                                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(bi) : "r"(sBias + 4u * (uint32_t)cc));
                            v += (long long)bi;
                            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(mlt) : "r"(sMult + 4u * (uint32_t)cc));
                        } else {
                            if (a.bias) v += (long long)__ldg(reinterpret_cast<const int32_t *>(a.bias) + cc);
                            mlt = __ldg(a.mult + cc);
                        }
                        const int q = requant_i8(v, mlt, a.act);
                        if ((e & 3) == 0) pk[e >> 2] = 0u;
                        pk[e >> 2] |= ((uint32_t)(q & 0xff)) << (8 * (e & 3));
                    }
                    const uint32_t dst8 = sbuf + (uint32_t)row * 32u;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst8), "r"(pk[0]), "r"(pk[1]),
                                 "r"(pk[2]), "r"(pk[3])
                                 : "memory");
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst8 + 16u), "r"(pk[4]),
                                 "r"(pk[5]), "r"(pk[6]), "r"(pk[7])
                                 : "memory");
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(av[8 * j + e]);
                        if (a.bias && co + 8 * j < a.Cout) {  // Cout % 8 == 0: 8 columns all in or all out
                            float4 b0, b1;
                            if (a.bias_smem) {
                                const uint32_t sb = sBias + 4u * (uint32_t)(co + 8 * j);
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(b0.x), "=f"(b0.y), "=f"(b0.z), "=f"(b0.w) : "r"(sb));
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(b1.x), "=f"(b1.y), "=f"(b1.z), "=f"(b1.w) : "r"(sb + 16u));
                            } else {
                                const float *fb = reinterpret_cast<const float *>(a.bias) + co + 8 * j;
                                b0 = __ldg(reinterpret_cast<const float4 *>(fb));
                                b1 = __ldg(reinterpret_cast<const float4 *>(fb) + 1);
                            }
                            v[0] += b0.x; v[1] += b0.y; v[2] += b0.z; v[3] += b0.w;
                            v[4] += b1.x; v[5] += b1.y; v[6] += b1.z; v[7] += b1.w;
                        }
                        // residual (8 channels, 16 bytes) added after the activation
                        float rv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        if (FUSED && rpix >= 0 && co + 8 * j < a.Cout) {
                            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(
                                reinterpret_cast<const __nv_bfloat16 *>(a.om.res) + (long long)rpix * a.Cout + co + 8 * j));
                            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                rv[2 * e] = __uint_as_float(wd[e] << 16);
                                rv[2 * e + 1] = __uint_as_float(wd[e] & 0xffff0000u);
                            }
                        }
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float2 f = activate2_fast(make_float2(v[2 * e], v[2 * e + 1]), a.act);
                            if constexpr (FUSED) f = add2(f, make_float2(rv[2 * e], rv[2 * e + 1]));
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(f.x, f.y);
                            pk[e] = *reinterpret_cast<uint32_t *>(&h2);
                        }
                        const uint32_t dst = srow + ((((uint32_t)j) ^ swz) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk[0]),
                                     "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                                     : "memory");
                    }
                }
                tc::fence_proxy_async_smem();  // staged values visible to the TMA engine
                tc::named_bar_sync(1 + grp, 128);
                // (MB = 2: a bottom block wholly below the image stores nothing)
                if (issuer && (MB == 1 || oh0 + jb * (a.bh / MB) < a.OH)) {
                    const int reps = FUSED ? a.om.up * a.om.up : 1;
                    for (int rp = 0; rp < reps; ++rp) {  // one store per upsample replica
                        if (FLAT)
                            tc::tma_store_2d(&tmY.m[rp], sbuf, co, m0);
                        else
                            tc::tma_store_4d(&tmY.m[rp], sbuf, co, ow0, oh0 + jb * (a.bh / MB), n);
                    }
                }
                if (issuer) tc::bulk_commit();
                ++oc;
            }
        }
        // The staging buffers must outlive the stores' reads of them; the
        // global writes themselves complete before the grid does.  (The
        // swapped TMA write-out stores from every warp's lane 0.)
        if (issuer || (SWAP && a.out_bufs == 2 && lane == 0)) tc::bulk_wait_read0();
    }

    // Warps 0 and 1 ran their loops on lane 0 only: reconverge each warp
    // before the block barrier, so that the barrier really waits for every
    // role (TMEM is freed only after the epilogue's last tcgen05.ld).
    __syncwarp();
    tc::fence_before_sync();
    __syncthreads();
    // pair mode: neither CTA leaves (or frees TMEM) while the other may still
    // use its shared memory or TMEM
    if constexpr (PAIR) tc::cluster_sync();
    if (warp == 1) {
        tc::fence_after_sync();
        if constexpr (PAIR)
            tc::tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

}  // namespace
