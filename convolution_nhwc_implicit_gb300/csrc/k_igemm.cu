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

#include <mutex>

#include "conv_internal.h"
#include "epilogue.cuh"
#include "tc_ptx.cuh"

using namespace convk;

namespace {

constexpr int kBM = 128;     // output pixels per tile (normal mode)
constexpr int kBMSwap = 256; // output pixels per tile (swapped mode)
constexpr int kTP = 272;     // swapped-mode transpose rows: 128 bf16 channels + 16 bytes of padding

// Epilogue warpgroups per CTA: each takes a slice of every tile's columns.
__host__ __device__ constexpr int epi_groups(int bn, bool swap) { return swap ? 4 : (bn >= 128 ? 4 : 2); }
// Threads per CTA: the TMA warp, the MMA warp and the epilogue warpgroups.
__host__ __device__ constexpr int cta_threads(int bn, bool swap) { return 64 + 128 * epi_groups(bn, swap); }

struct IgArgs {
    int H, W, Cin, Cout, KH, KW, stride, pad_h, pad_w, OH, OW;
    int bw, bh, tiles_w, tiles_h, tiles_n, num_tiles, cblocks, kblocks, stages;
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
    int *status;
};

// Waits for phase `parity` of `bar`, giving up after kWaitBudgetNs or when
// another role of the CTA has given up.  Returns false on give-up.
// CLUSTER: acquire at cluster scope (arrivals may come from the peer CTA).
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

// Epilogue of the swapped mode for one tile.  The accumulator is D[co][px]:
// thread `row` of the group holds output channel co = nb*128 + row and reads
// the group's kCols pixel columns 16 at a time.  Each 16-pixel chunk goes
// through shared memory (rows of 128 channels, padded to kTP bytes) to turn
// channel-per-thread values into pixel rows, which the group then writes
// with 16-byte stores (eight threads cover one pixel's 128 channels).
template <int kCols>
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
        long long pix;
        bool valid;
        if (a.flat) {
            pix = m0 + p;
            valid = pix < a.M;
        } else {
            const int dh = p / a.bw;
            const int oh = oh0 + dh, ow = ow0 + (p - dh * a.bw);
            valid = p < a.bw * a.bh && oh < a.OH && ow < a.OW;
            pix = ((long long)n * a.OH + oh) * a.OW + ow;
        }
        if (valid && a.out_i8) {
            // 16 int8 channels per thread (Cout % 16 == 0 on this path)
            const uint4 *src = reinterpret_cast<const uint4 *>(tbuf + wpx * kTP + (gt & 7) * 16);
            int8_t *dst = reinterpret_cast<int8_t *>(a.y) + pix * a.Cout + wco;
            if (wco < a.Cout) *reinterpret_cast<uint4 *>(dst) = src[0];
        } else if (valid) {
            const uint4 *src = reinterpret_cast<const uint4 *>(tbuf + wpx * kTP + (gt & 7) * 32);
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(a.y) + pix * a.Cout + wco;
            if (wco < a.Cout) *reinterpret_cast<uint4 *>(dst) = src[0];
            if (wco + 8 < a.Cout) *reinterpret_cast<uint4 *>(dst + 8) = src[1];
        }
    }
}

// SWAP = false: MMA M = 128 pixels, N = BN output channels (D[pixel][co]).
// SWAP = true (layers with Cout <= 128): the operands trade places, MMA M =
// 128 output channels (weights as A), N = 256 pixels (activations as B),
// D[co][pixel]; every MMA then has N = 256, the only width at which tcgen05
// reaches its peak rate (the issue cost of an MMA does not shrink with N).
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
template <int BN, int BK, bool FLAT, bool SWAP, bool PAIR>
__global__ void __launch_bounds__(cta_threads(BN, SWAP), 1)
igemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmY, const IgArgs a) {
    static_assert(!(PAIR && SWAP), "the CTA-pair mode uses the normal layout");
    constexpr int kPix = SWAP ? kBMSwap : kBM;  // pixel rows of a tile (per CTA)
    constexpr int kAcc = SWAP ? kBMSwap : BN;   // accumulator columns of a tile
    constexpr int kBRows = PAIR ? BN / 2 : BN;  // weight rows this CTA stages
    constexpr uint32_t kRowBytes = BK * 2;
    constexpr uint32_t kAStage = kPix * BK * 2;  // activation (pixel) tile
    constexpr uint32_t kBStage = kBRows * BK * 2;  // weight tile (this CTA's part)
    constexpr uint32_t kTmemCols = 2 * kAcc;     // two accumulators
    constexpr uint32_t kIdesc = SWAP ? tc::idesc_bf16_f32(128, kBMSwap)
                                     : tc::idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN);
    constexpr int kGroups = epi_groups(BN, SWAP);
    constexpr int kCols = kAcc / kGroups;  // accumulator columns per epilogue thread
    static_assert(SWAP ? (BN == 128 && kCols % 16 == 0) : (kCols % 32 == 0), "epilogue column slices");
    constexpr uint32_t kOutStage = SWAP ? 16 * kTP : kBM * 64;  // per group: transpose rows / store staging

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
    uint8_t *gbase = smem_raw + (base - raw);
    const int stages = a.stages;
    const uint32_t sA = base;
    const uint32_t sB = base + stages * kAStage;
    const uint32_t sOut = sB + stages * kBStage;  // per epilogue group: 128 rows x 64 B output staging
    const uint32_t sBar = sOut + kGroups * a.out_bufs * kOutStage;
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    auto empty_bar = [&](int s) { return sBar + 8u * (stages + s); };
    auto tfull_bar = [&](int b) { return sBar + 8u * (2 * stages + b); };
    auto tempty_bar = [&](int b) { return sBar + 8u * (2 * stages + 2 + b); };
    uint8_t *gmisc = gbase + (sBar - base) + 8u * (2 * stages + 4);
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(gmisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gmisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work unit: the CTA, or in pair mode the cluster (CTAs 2u and 2u + 1).
    const uint32_t rank = PAIR ? tc::cluster_ctarank() : 0u;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            tc::mbar_init(full_bar(s), 1);
            tc::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tfull_bar(b), 1);
            tc::mbar_init(tempty_bar(b), PAIR ? 2 * 4 * kGroups : 128 * kGroups);  // pair: one per warp
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
        tc::tma_prefetch_desc(&tmY);
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

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // pair mode: both CTAs' loads complete on the even CTA's barriers
            const uint32_t full0 = PAIR ? tc::mapa_shared(full_bar(0), 0) : full_bar(0);
            for (int tile = unit; tile < a.num_tiles && ok; tile += units) {
                const int nb = tile % a.tiles_n;
                // pair mode: this CTA's pixel tile (past tiles_m: an empty
                // half, loaded as zeros from outside the tensor, never stored)
                const int mt = PAIR ? (tile / a.tiles_n) * 2 + (int)rank : tile / a.tiles_n;
                int n = 0, oh0 = 0, ow0 = 0;
                int m0 = 0;
                if (FLAT) {
                    m0 = mt * kPix;
                } else {
                    const int tw = mt % a.tiles_w;
                    const int t2 = mt / a.tiles_w;
                    oh0 = (t2 % a.tiles_h) * a.bh;
                    n = t2 / a.tiles_h;
                    ow0 = tw * a.bw;
                }
                int r = 0, s = 0, cb = 0;
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, a.status,
                                      KSTATUS_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dA = sA + stage * kAStage;
                    const uint32_t dB = sB + stage * kBStage;
                    const int kx = (r * a.KW + s) * a.Cin + cb * BK;
                    if constexpr (PAIR) {
                        const uint32_t fb = full0 + 8u * stage;
                        if (rank == 0) tc::mbar_arrive_expect_tx(full_bar(stage), 2u * (a.a_bytes + kBStage));
                        if (FLAT)
                            tc::tma_load_2d_pair(dA, &tmA, fb, cb * BK, m0);
                        else
                            tc::tma_load_4d_pair(dA, &tmA, fb, cb * BK, ow0 * a.stride - a.pad_w + s,
                                                 oh0 * a.stride - a.pad_h + r, n);
                        tc::tma_load_2d_pair(dB, &tmB, fb, kx, nb * BN + (int)rank * kBRows);
                    } else {
                        tc::mbar_arrive_expect_tx(full_bar(stage), a.a_bytes + kBStage);
                        if (FLAT)
                            tc::tma_load_2d(dA, &tmA, full_bar(stage), cb * BK, m0);
                        else
                            tc::tma_load_4d(dA, &tmA, full_bar(stage), cb * BK,
                                            ow0 * a.stride - a.pad_w + s, oh0 * a.stride - a.pad_h + r, n);
                        tc::tma_load_2d(dB, &tmB, full_bar(stage), kx, nb * BN);
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
            for (int tile = unit; tile < a.num_tiles && ok; tile += units, ++lt) {
                const int buf = lt & 1;
                const uint32_t use = (uint32_t)(lt >> 1);
                if (!wait_bounded<PAIR>(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag, a.status,
                                        KSTATUS_TIMEOUT_MMA))
                    break;
                tc::fence_after_sync();
                const uint32_t d = tmem_base + (uint32_t)(buf * kAcc);
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, abort_flag, a.status, KSTATUS_TIMEOUT_MMA)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t aS = sA + stage * kAStage;
                    const uint32_t bS = sB + stage * kBStage;
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
                if (ok) {  // accumulator ready
                    if (PAIR)
                        tc::mma_commit_pair(tfull_bar(buf), 0x3);
                    else
                        tc::mma_commit(tfull_bar(buf));
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2 ..)
        // tcgen05.ld lets warp w reach TMEM lanes 32 * (w % 4) .. + 31, so every
        // run of four consecutive warps covers the 128 accumulator rows; warp
        // group g (warps 2 + 4g .. 5 + 4g) drains columns [g * kCols, (g+1) * kCols).
        const int q = warp & 3;
        const int grp = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const int c_base = grp * kCols;
        const bool issuer = ((warp - 2) & 3) == 0 && lane == 0;  // issues the group's TMA stores
        const uint32_t sStage = sOut + (uint32_t)(grp * a.out_bufs) * kOutStage;  // this group's staging
        int oc = 0;  // TMA stores this group has issued (selects the staging buffer)
        int lt = 0;
        // pair mode: accumulator-empty arrivals go to the even CTA's barrier
        const uint32_t tempty0 = PAIR ? tc::mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
        for (int tile = unit; tile < a.num_tiles; tile += units, ++lt) {
            const int buf = lt & 1;
            const uint32_t use = (uint32_t)(lt >> 1);
            const bool got = wait_bounded(tfull_bar(buf), use & 1u, abort_flag, a.status,
                                          KSTATUS_TIMEOUT_EPILOGUE);
            __syncwarp();  // tcgen05.ld below is warp-collective (.sync.aligned)
            if (!__all_sync(0xffffffffu, got)) break;
            tc::fence_after_sync();
            if constexpr (SWAP) {
                epilogue_swapped<kCols>(a, tile, tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kAcc + c_base),
                                        tempty_bar(buf), row, grp, c_base, gbase + (sOut - base) + grp * a.out_bufs * kOutStage,
                                        threadIdx.x - 64 - grp * 128);
                continue;
            }
            // Move this thread's slice of the accumulator into registers, then
            // hand the TMEM buffer back to the MMA warp before doing the math.
            uint32_t acc[kCols];
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c_base);
#pragma unroll
            for (int c = 0; c < kCols; c += 32)
                tc::tmem_ld_32x32(tbase + (uint32_t)c, *reinterpret_cast<uint32_t(*)[32]>(acc + c));
            tc::tmem_ld_wait();
            tc::fence_before_sync();
            if constexpr (PAIR) {
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_cluster(tempty0 + 8u * buf);
            } else {
                tc::mbar_arrive(tempty_bar(buf));
            }

            // Output slice: bias, activation, bf16, staged in shared memory
            // (64-byte swizzle, matching the store's tensor map) and written by
            // one TMA tensor store per 32 columns.  The box is the tile's
            // bh x bw pixel rectangle (or 128 flat rows): rows past it are
            // never stored and pixels outside the image are clipped by TMA.
            const int nb = tile % a.tiles_n;
            const int mt = PAIR ? (tile / a.tiles_n) * 2 + (int)rank : tile / a.tiles_n;
            if (PAIR && mt >= a.tiles_m) continue;  // the empty half of the last pair tile
            int n = 0, oh0 = 0, ow0 = 0, m0 = 0;
            if (FLAT) {
                m0 = mt * kPix;
            } else {
                const int tw = mt % a.tiles_w;
                const int t2 = mt / a.tiles_w;
                oh0 = (t2 % a.tiles_h) * a.bh;
                n = t2 / a.tiles_h;
                ow0 = tw * a.bw;
            }
            const uint32_t swz = (uint32_t)((row >> 1) & 3);
#pragma unroll
            for (int c = 0; c < kCols; c += 32) {
                const int co = nb * BN + c_base + c;
                if (co >= a.Cout) continue;  // the same for the whole group
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
                        long long v = (long long)__float2int_rn(__uint_as_float(acc[c + e]));
                        if (a.bias) v += (long long)__ldg(reinterpret_cast<const int32_t *>(a.bias) + cc);
                        const int q = requant_i8(v, __ldg(a.mult + cc), a.act);
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
                        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(acc[c + 8 * j + e]);
                        if (a.bias && co + 8 * j < a.Cout) {  // Cout % 8 == 0: 8 columns all in or all out
                            const float *fb = reinterpret_cast<const float *>(a.bias) + co + 8 * j;
                            const float4 b0 = __ldg(reinterpret_cast<const float4 *>(fb));
                            const float4 b1 = __ldg(reinterpret_cast<const float4 *>(fb) + 1);
                            v[0] += b0.x; v[1] += b0.y; v[2] += b0.z; v[3] += b0.w;
                            v[4] += b1.x; v[5] += b1.y; v[6] += b1.z; v[7] += b1.w;
                        }
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = activate2_fast(make_float2(v[2 * e], v[2 * e + 1]), a.act);
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
                if (issuer) {
                    if (FLAT)
                        tc::tma_store_2d(&tmY, sbuf, co, m0);
                    else
                        tc::tma_store_4d(&tmY, sbuf, co, ow0, oh0, n);
                    tc::bulk_commit();
                }
                ++oc;
            }
        }
        // The staging buffers must outlive the stores' reads of them; the
        // global writes themselves complete before the grid does.
        if (issuer) tc::bulk_wait_read0();
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

CUtensorMapSwizzle swizzle_for(int bk) {
    return bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : (bk == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

template <int BN, int BK, bool FLAT, bool SWAP, bool PAIR = false>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, FLAT, SWAP, PAIR>);
}

template <int BN, int BK>
void *kernel_ptr_flat(bool flat) {
    return flat ? kernel_ptr<BN, BK, true, false>() : kernel_ptr<BN, BK, false, false>();
}

template <int BN>
void *kernel_ptr_bk(int bk, bool flat) {
    switch (bk) {
    case 64: return kernel_ptr_flat<BN, 64>(flat);
    case 32: return kernel_ptr_flat<BN, 32>(flat);
    default: return kernel_ptr_flat<BN, 16>(flat);
    }
}

template <int BK>
void *kernel_ptr_swap(bool flat) {
    return flat ? kernel_ptr<128, BK, true, true>() : kernel_ptr<128, BK, false, true>();
}

template <int BK>
void *kernel_ptr_pair(bool flat) {
    return flat ? kernel_ptr<256, BK, true, false, true>() : kernel_ptr<256, BK, false, false, true>();
}

void *select_kernel(int bn, int bk, bool flat, bool swap, bool pair) {
    if (pair) {
        switch (bk) {
        case 64: return kernel_ptr_pair<64>(flat);
        case 32: return kernel_ptr_pair<32>(flat);
        default: return kernel_ptr_pair<16>(flat);
        }
    }
    if (swap) {
        switch (bk) {
        case 64: return kernel_ptr_swap<64>(flat);
        case 32: return kernel_ptr_swap<32>(flat);
        default: return kernel_ptr_swap<16>(flat);
        }
    }
    switch (bn) {
    case 256: return kernel_ptr_bk<256>(bk, flat);
    case 128: return kernel_ptr_bk<128>(bk, flat);
    default: return kernel_ptr_bk<64>(bk, flat);
    }
}

}  // namespace

// Layers whose k_w taps of all input channels fit in 16 channels (the
// 3-channel image stem: 3 x 3 = 9) have those taps folded into the padding:
// the pre-pass writes, for every input row position u, the k_w x Cin values
// x[h][u - pad_w + s][ci] (s-major) as one 16-channel pixel, and the kernel
// runs a k_h x 1 convolution over that tensor.  The padded copy has as many
// bytes as the plain channel-padded one, with k_w times fewer K blocks.
static bool igemm_fold(const conv_plan *p) {
    const bool prep = p->dtype == CONV_I8 || p->s.c_in % 16 != 0;
    return prep && p->s.k_w > 1 && p->s.k_w * p->s.c_in <= 16;
}

// Input channels the tensor-core kernel sees: Cin, or Cin (k_w x Cin when
// folded) rounded up to 16 when the operands go through the widening
// pre-pass (int8 layers, and bf16 layers whose channel rows are not whole
// 32-byte units).
static int igemm_cin(const conv_plan *p) {
    if (igemm_fold(p)) return 16;
    const bool prep = p->dtype == CONV_I8 || p->s.c_in % 16 != 0;
    return prep ? (p->s.c_in + 15) / 16 * 16 : p->s.c_in;
}

bool igemm_supported(const conv_plan *p) {
    if (p->groups != 1 || p->dtype == CONV_F32) return false;  // fp32 stays on FFMA (never TF32)
    if (p->dtype == CONV_BF16 && p->s.c_out % 8 != 0) return false;
    if (p->dtype == CONV_I8) {
        // int8 output rows are stored 16 bytes at a time; exactness of the
        // fp32 accumulation needs K * 128 * 127 < 2^24 (K <= 1024).
        if (p->s.c_out % 16 != 0) return false;
        if ((long long)p->s.k_h * (igemm_fold(p) ? 1 : p->s.k_w) * igemm_cin(p) > 1024) return false;
    }
    if (p->stride > 8) return false;  // TMA element strides are at most 8
    const long long pixels_in = (long long)p->s.n * p->s.h * (p->s.w + 2 * p->pad_w);
    if (pixels_in > 0xFFFFFFFFll) return false;  // TMA dimension limit
    if ((long long)p->s.n * p->oh * p->ow > 0x7FFFFFFFll) return false;
    return true;
}

int igemm_configure(conv_plan *p, int layout) {
    IgemmGeom &g = p->ig;
    const int S = p->stride;
    g.in_i8 = 0;
    const int cin = igemm_cin(p);
    g.prep = (cin != p->s.c_in || p->dtype == CONV_I8) ? 1 : 0;
    g.cin = cin;
    g.fold = igemm_fold(p) ? 1 : 0;
    g.kw = g.fold ? 1 : p->s.k_w;
    g.padw = g.fold ? 0 : p->pad_w;
    g.wx = g.fold ? p->s.w + 2 * p->pad_w - p->s.k_w + 1 : p->s.w;
    g.flat = (p->s.k_h == 1 && g.kw == 1 && S == 1 && p->pad_h == 0 && g.padw == 0) ? 1 : 0;
    g.bk = cin % 64 == 0 ? 64 : (cin % 32 == 0 ? 32 : 16);
    g.cblocks = cin / g.bk;
    if (g.prep) {
        // plan-owned bf16 copies of x and w (channels padded to `cin`)
        const size_t xb = (size_t)p->s.n * p->s.h * g.wx * cin * 2;
        const size_t wb = (size_t)p->s.c_out * p->s.k_h * g.kw * cin * 2;
        p->cin_p = cin;
        if (xb && cudaMalloc(&p->d_xprep, xb) != cudaSuccess) return CONV_ERR_OOM;
        if (cudaMalloc(&p->d_wprep, wb) != cudaSuccess) return CONV_ERR_OOM;
    }
    g.kblocks = p->s.k_h * g.kw * g.cblocks;

    // Candidate layouts: swapped (Cout <= 128) with 256-pixel tiles; normal
    // with 128-pixel tiles and BN in {256, 128, 64}; the CTA pair with
    // 2 x 128-pixel tiles and BN = 256.  Each is scored by an estimate of
    // its time: waves x (per-tile cost + fixed cost), the per-tile cost
    // (per SM) being the largest of
    //   MMA issue   128 cycles per K=16 step whatever N is (so N = 256 is
    //               the only full-rate width),
    //   shared memory  the staged operand bytes are written once by TMA and
    //               read once by the MMAs: 2 * (pixel rows + weight rows
    //               staged) * K * 2 bytes at 128 B/cycle,
    //   epilogue    accumulator lanes x columns (wasted lanes included)
    //               x cycles per value / 128 lanes per cycle per SM,
    // with the epilogue costing ~16 cycles per value with Mish (two MUFU
    // operations), ~10 for an int8 requantisation and ~6 otherwise.
    const long long K = (long long)p->s.k_h * g.kw * cin;
    const long long epi_c = p->dtype == CONV_I8 ? 10 : (p->act == CONV_ACT_MISH ? 16 : 6);
    long long best_cost = -1, best_tiles = 0;
    for (int cand = 0; cand < 5; ++cand) {
        const bool swap = cand == 0;
        const bool pair = cand == 4;
        if (swap && p->s.c_out > 128) continue;
        if (pair && p->num_sms < 2) continue;
        if (layout != 0 && layout != cand + 1) continue;
        const int bn = swap ? 128 : (cand == 1 || pair ? 256 : (cand == 2 ? 128 : 64));
        const int P = swap ? kBMSwap : kBM;
        int bw = P, bh = 1, tw = 1, th = 1;
        long long tiles_m;
        if (g.flat) {
            const long long M = (long long)p->s.n * p->s.h * g.wx;
            tiles_m = (M + P - 1) / P;
        } else {
            // Smallest number of bh x bw rectangles covering the output; among
            // equal counts, the widest (longest contiguous NHWC runs).
            long long best = -1;
            for (int cw = 1; cw <= P && cw <= p->ow * 2; ++cw) {
                if (cw * S > 256) break;
                int ch = P / cw;
                if (ch > p->oh) ch = p->oh;
                while (ch * S > 256) --ch;
                if (ch < 1) continue;
                const long long ctw = (p->ow + cw - 1) / cw, cth = (p->oh + ch - 1) / ch;
                const long long t = ctw * cth * p->s.n;
                if (best < 0 || t < best || (t == best && cw > bw)) {
                    best = t; bw = cw; bh = ch; tw = (int)ctw; th = (int)cth;
                }
                if (cw >= p->ow) break;
            }
            tiles_m = best;
        }
        const long long tiles_n = swap ? 1 : (p->s.c_out + bn - 1) / bn;
        // pair mode: a unit of work is a pair tile on two SMs
        const long long tiles = (pair ? (tiles_m + 1) / 2 : tiles_m) * tiles_n;
        const long long slots = pair ? p->num_sms / 2 : p->num_sms;
        const long long waves = (tiles + slots - 1) / slots;
        const long long t_mma = K / 16 * 128;
        const long long t_smem = (P + (pair ? bn / 2 : bn)) * K / 32;
        const long long t_epi = 128LL * (swap ? P : bn) * epi_c / 128;
        long long t_tile = t_mma > t_smem ? t_mma : t_smem;
        if (t_epi > t_tile) t_tile = t_epi;
        const long long cost = waves * (t_tile + 500);
        // ties: more tiles (more SMs busy), then the narrower N tile
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && tiles > best_tiles) ||
            (cost == best_cost && tiles == best_tiles && bn < g.bn)) {
            best_cost = cost;
            best_tiles = tiles;
            g.swap = swap ? 1 : 0; g.pair = pair ? 1 : 0; g.bn = bn; g.tiles_n = (int)tiles_n;
            g.tiles_m = (int)tiles_m;
            g.bw = bw; g.bh = bh; g.tiles_w = tw; g.tiles_h = th;
        }
    }
    if (best_cost < 0) return CONV_ERR_UNSUPPORTED;  // forced swapped layout with c_out > 128
    const int P = g.swap ? kBMSwap : kBM;  // pixels per tile (per CTA)
    g.num_tiles = g.tiles_n * (g.pair ? (g.tiles_m + 1) / 2 : g.tiles_m);  // work units

    const int stage_bytes = (P + (g.pair ? g.bn / 2 : g.bn)) * g.bk * 2;
    // Epilogue staging: swapped mode, 16 transpose rows per group; normal
    // mode, 128 rows x 64 B per group and buffer.  Two buffers per group let
    // a group fill one while the TMA store of the other is still reading it;
    // they are used when the operand ring keeps at least 4 stages.
    // Short-K layers (few K blocks per tile) are limited by the epilogue and
    // take the second buffer; long-K layers keep the shared memory for
    // operand stages.
    const int one_buf = g.swap ? 4 * 16 * kTP : epi_groups(g.bn, false) * kBM * 64;
    g.out_bufs = 1;
    if (!g.swap && g.kblocks < 16 && (227 * 1024 - 1024 - 256 - 2 * one_buf) / stage_bytes >= 4) g.out_bufs = 2;
    const int out_bytes = one_buf * g.out_bufs;
    const int budget = 227 * 1024 - 1024 - 256 - out_bytes;
    g.stages = budget / stage_bytes;
    if (g.stages > 8) g.stages = 8;
    if (g.stages < 2) return CONV_ERR_UNSUPPORTED;
    g.smem = 1024 + g.stages * stage_bytes + out_bytes + 8 * (2 * g.stages + 4) + 16;
    // Ask for more than half of an SM's shared memory so that no two CTAs of
    // this persistent kernel share an SM: each CTA then owns its TMEM
    // columns (at most 512) without waiting for another to free them.
    if (g.smem < 116 * 1024) g.smem = 116 * 1024;
    if (!tensor_map_encoder()) return CONV_ERR_CUDA;
    void *kern = select_kernel(g.bn, g.bk, g.flat != 0, g.swap != 0, g.pair != 0);
    const int rc = conv_grant_smem(kern, p->device, g.smem);
    if (rc != CONV_OK) return rc;
    if (g.pair) {
        // as many CTA pairs as can be resident at once (a pair occupies two
        // SMs of one GPC), at most one per work unit
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * g.num_tiles);
        cfg.blockDim = dim3(cta_threads(g.bn, false));
        cfg.dynamicSmemBytes = (size_t)g.smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1)
            return CONV_ERR_UNSUPPORTED;
        g.grid = 2 * (g.num_tiles < clusters ? g.num_tiles : clusters);
    } else {
        g.grid = g.num_tiles < p->num_sms ? g.num_tiles : p->num_sms;
    }
    snprintf(p->desc, sizeof(p->desc),
             "igemm_%s_tcgen05 %s%s %s BK=%d tile=%dx%d stages=%d out_bufs=%d tiles=%d grid=%d",
             p->dtype == CONV_I8 ? (g.fold ? "i8-as-bf16-kwfold" : "i8-as-bf16")
                                 : (g.fold ? "bf16-cpad-kwfold" : (g.prep ? "bf16-cpad" : "bf16")),
             g.flat ? "flat" : "spatial",
             g.swap ? " swapped" : (g.pair ? " cta-pair" : ""),
             g.swap ? "M=128co N=256px"
                    : (g.pair ? "M=256px N=256co"
                              : (g.bn == 256 ? "M=128px N=256co" : (g.bn == 128 ? "M=128px N=128co" : "M=128px N=64co"))),
             g.bk, g.bh, g.bw, g.stages, g.out_bufs, g.num_tiles, g.grid);
    return CONV_OK;
}

int launch_igemm(const conv_plan *p, const void *x, const void *w, const void *bias, void *y,
                 cudaStream_t st) {
    const IgemmGeom &g = p->ig;
    if (g.prep) {
        if (launch_prep(p, x, w, st) != cudaSuccess) return CONV_ERR_CUDA;
        x = p->d_xprep;
        w = p->d_wprep;
    }
    const int cin = g.cin;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return CONV_ERR_CUDA;
    const int S = p->stride;
    alignas(64) CUtensorMap tmA, tmB;
    const cuuint32_t ones[4] = {1, 1, 1, 1};
    CUresult rc;
    if (g.flat) {
        const cuuint64_t dims[2] = {(cuuint64_t)cin, (cuuint64_t)p->s.n * p->s.h * g.wx};
        const cuuint64_t strides[1] = {(cuuint64_t)cin * 2};
        const cuuint32_t box[2] = {(cuuint32_t)g.bk, (cuuint32_t)(g.swap ? kBMSwap : kBM)};
        rc = encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, ones,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(g.bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[4] = {(cuuint64_t)cin, (cuuint64_t)g.wx, (cuuint64_t)p->s.h,
                                    (cuuint64_t)p->s.n};
        const cuuint64_t strides[3] = {(cuuint64_t)cin * 2, (cuuint64_t)g.wx * cin * 2,
                                       (cuuint64_t)p->s.h * g.wx * cin * 2};
        const cuuint32_t box[4] = {(cuuint32_t)g.bk, (cuuint32_t)(g.bw * S), (cuuint32_t)(g.bh * S), 1};
        const cuuint32_t estr[4] = {1, (cuuint32_t)S, (cuuint32_t)S, 1};
        rc = encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(x), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(g.bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (rc != CUDA_SUCCESS) return CONV_ERR_CUDA;
    {
        const cuuint64_t K = (cuuint64_t)p->s.k_h * g.kw * cin;
        const cuuint64_t dims[2] = {K, (cuuint64_t)p->s.c_out};
        const cuuint64_t strides[1] = {K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)g.bk, (cuuint32_t)(g.pair ? g.bn / 2 : g.bn)};
        rc = encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w), dims, strides, box, ones,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(g.bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV_ERR_CUDA;
    }

    alignas(64) CUtensorMap tmY;
    {
        // 32 output channels per store box: 64 bytes (bf16, 64-byte swizzle)
        // or 32 bytes (int8, unswizzled)
        const bool i8 = p->dtype == CONV_I8;
        const cuuint64_t es = i8 ? 1 : 2;
        const CUtensorMapDataType dt = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapSwizzle sw = i8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B;
        const cuuint32_t box_n = 32;
        if (g.flat) {
            const cuuint64_t dims[2] = {(cuuint64_t)p->s.c_out, (cuuint64_t)p->s.n * p->oh * p->ow};
            const cuuint64_t strides[1] = {(cuuint64_t)p->s.c_out * es};
            const cuuint32_t box[2] = {box_n, (cuuint32_t)(g.swap ? kBMSwap : kBM)};
            rc = encode(&tmY, dt, 2, y, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            const cuuint64_t dims[4] = {(cuuint64_t)p->s.c_out, (cuuint64_t)p->ow, (cuuint64_t)p->oh,
                                        (cuuint64_t)p->s.n};
            const cuuint64_t strides[3] = {(cuuint64_t)p->s.c_out * es, (cuuint64_t)p->ow * p->s.c_out * es,
                                           (cuuint64_t)p->oh * p->ow * p->s.c_out * es};
            const cuuint32_t box[4] = {box_n, (cuuint32_t)g.bw, (cuuint32_t)g.bh, 1};
            rc = encode(&tmY, dt, 4, y, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (rc != CUDA_SUCCESS) return CONV_ERR_CUDA;
    }

    IgArgs a;
    a.H = p->s.h; a.W = g.wx; a.Cin = cin; a.Cout = p->s.c_out; a.KH = p->s.k_h; a.KW = g.kw;
    a.stride = S; a.pad_h = p->pad_h; a.pad_w = g.padw; a.OH = p->oh; a.OW = p->ow;
    a.bw = g.bw; a.bh = g.bh; a.tiles_w = g.tiles_w; a.tiles_h = g.tiles_h; a.tiles_n = g.tiles_n;
    a.num_tiles = g.num_tiles; a.cblocks = g.cblocks; a.kblocks = g.kblocks; a.stages = g.stages;
    a.tiles_m = g.tiles_m;
    a.M = (long long)p->s.n * p->s.h * g.wx;
    a.a_bytes = (uint32_t)((g.flat ? (g.swap ? kBMSwap : kBM) : g.bw * g.bh) * g.bk * 2);
    a.flat = g.flat;
    a.act = (int)p->act;
    a.bias = bias;
    a.y = y;
    a.out_i8 = p->dtype == CONV_I8 ? 1 : 0;
    a.mult = p->d_mult;
    a.out_bufs = g.out_bufs;
    a.status = p->d_status;

    void *k = select_kernel(g.bn, g.bk, g.flat != 0, g.swap != 0, g.pair != 0);
    void *args[] = {&tmA, &tmB, &tmY, &a};
    cudaError_t e;
    if (g.pair) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(g.grid);
        cfg.blockDim = dim3(cta_threads(g.bn, false));
        cfg.dynamicSmemBytes = (size_t)g.smem;
        cfg.stream = st;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelExC(&cfg, k, args);
    } else {
        e = cudaLaunchKernel(k, dim3(g.grid), dim3(cta_threads(g.bn, g.swap != 0)), args, (size_t)g.smem, st);
    }
    return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}
