// Host side of the tcgen05 implicit-GEMM family: tile-layout planning,
// tensor-map encoding and launch.  The kernel itself (and the description of
// its design) is in k_igemm_kernel.cuh; this translation unit instantiates
// its plain variants, k_igemm_fused.cu the variants with output options.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>

#include "k_igemm_kernel.cuh"

namespace {

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

// The plain (no output options) variant for the tile mode: flat, spatial with
// per-tap boxes, or spatial with halo staging.
template <int BN, int BK, bool SWAP, bool PAIR>
void *kernel_ptr(bool flat, bool halo) {
    if (flat) return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, true, SWAP, PAIR, false, false>);
    if (halo) return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, SWAP, PAIR, false, true>);
    return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, SWAP, PAIR, false, false>);
}

template <int BN, bool SWAP, bool PAIR>
void *kernel_ptr_bk(int bk, bool flat, bool halo) {
    switch (bk) {
    case 64: return kernel_ptr<BN, 64, SWAP, PAIR>(flat, halo);
    case 32: return kernel_ptr<BN, 32, SWAP, PAIR>(flat, halo);
    default: return kernel_ptr<BN, 16, SWAP, PAIR>(flat, halo);
    }
}

void *select_kernel(int bn, int bk, bool flat, bool swap, bool pair, bool fused, bool halo, bool ept, int cvt,
                    int mb) {
    if (fused) return igemm_select_fused(bn, bk, flat, swap, pair, halo);
    if (cvt) return igemm_select_cvt(cvt, bn, bk, flat, halo, ept, mb);
    if (ept) return igemm_select_ept(bn, bk, flat, halo);
    if (pair) return bn == 128 ? kernel_ptr_bk<128, false, true>(bk, flat, halo)
                               : kernel_ptr_bk<256, false, true>(bk, flat, halo);
    if (swap) return kernel_ptr_bk<128, true, false>(bk, flat, halo);
    switch (bn) {
    case 256: return kernel_ptr_bk<256, false, false>(bk, flat, halo);
    case 128: return kernel_ptr_bk<128, false, false>(bk, flat, halo);
    default: return kernel_ptr_bk<64, false, false>(bk, flat, halo);
    }
}

}  // namespace

// A layer with a residual or upsample replicas runs the FUSED kernel variants.
static bool igemm_fused(const conv_plan *p) { return p->has_res || p->up > 1; }

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

// Folded in the kernel: the elements of one input row that a bw-pixel tile
// row reads, ((bw - 1) x stride + k_w) x Cin, plus up to 7 before them (the
// box starts on a 16-byte unit), rounded up to whole 16-byte units.
static int fold_inner(const conv_plan *p, int bw) {
    const long long e = ((long long)(bw - 1) * p->stride + p->s.k_w) * p->s.c_in + 7;
    return (int)((e + 7) / 8 * 8);
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

int igemm_configure(conv_plan *p, int layout, int staging, int epi, int widen) {
    IgemmGeom &g = p->ig;
    const int S = p->stride;
    g.in_i8 = 0;
    const int cin = igemm_cin(p);
    g.cin = cin;
    g.fold = igemm_fold(p) ? 1 : 0;
    g.kw = g.fold ? 1 : p->s.k_w;
    g.padw = g.fold ? 0 : p->pad_w;
    g.wx = g.fold ? p->s.w + 2 * p->pad_w - p->s.k_w + 1 : p->s.w;
    // (a flat tile's pixels have no (oh, ow) structure for the upsample replicas)
    g.flat = (p->s.k_h == 1 && g.kw == 1 && S == 1 && p->pad_h == 0 && g.padw == 0 && p->up == 1) ? 1 : 0;
    // The converter warpgroup (CVT variants) builds the bf16 operand in the
    // kernel: int8 operands widened, where their channel rows are whole
    // 16-byte TMA units and nothing is folded or padded (mode 1); or a bf16
    // k_w-folded stem assembled from the plain NHWC rows, where an image row
    // is a whole number of 16-byte units (mode 2).
    const int cvt_mode =
        igemm_fused(p) ? 0
        : (p->dtype == CONV_I8 && cin == p->s.c_in && !g.fold) ? 1
        : (p->dtype == CONV_BF16 && g.fold && !g.flat && (long long)p->s.w * p->s.c_in * 2 % 16 == 0) ? 2
                                                                                                      : 0;
    const bool cvt_ok = cvt_mode != 0;
    if (widen == 2 && !cvt_ok) return CONV_ERR_UNSUPPORTED;

    // Candidates: the tile layout (swapped, Cout <= 128, with 256-pixel
    // tiles; normal with 128-pixel tiles and BN in {256, 128, 64}; the CTA
    // pair with 2 x 128-pixel tiles and BN in {256, 128}) x the staging
    // (per-tap boxes, or halo staging for stride-1 spatial layers with
    // k_h = 3) x, in spatial mode, the tile's bh x bw shape x the channel
    // block BK: the largest of 64, 32, 16 dividing Cin and half of it (a
    // smaller one only where neither leaves room for two stages).
    // Each candidate is scored by an estimate of its time, waves x (per-tile
    // cost + a fixed cost), the per-tile cost (per SM) being the larger of
    //   the ring  stages per tile x (per-stage time + ~200 cycles of barrier
    //             round trip), a stage taking the longest of
    //               its MMAs     128 cycles per K = 16 step whatever N is (an
    //                            M = 128 MMA alone takes 48 / 64 / 128 cycles for
    //                            N = 64 / 128 / 256, below N = 256 the time to read
    //                            its operands from shared memory at 128 bytes a
    //                            cycle; beside the TMA writes and the epilogue,
    //                            which share that bandwidth, N <= 128 tiles ran no
    //                            faster per output than N = 256 in every layer
    //                            measured, which this flat charge models),
    //               its TMA rows ~1.4 cycles per staged operand row (a pixel's
    //                            or an output channel's BK channels),
    //               the refill   a freed stage is refilled ~2000 cycles later:
    //                            with S stages, 2000 / (S - 1) per stage,
    //   the epilogue  accumulator lanes x columns (wasted lanes included)
    //             x cycles per value / 128 lanes per cycle per SM,
    // with the epilogue costing ~16 cycles per value with Mish (two MUFU
    // operations), ~10 for an int8 requantisation and ~6 otherwise.  The
    // per-stage constants fit the batch-8 sweep's 3x3 layers (measured per
    // stage: 256->256 @80 CTA pair per-tap BK 64, 6 stages, 730-800 cycles;
    // halo BK 64, 2 stages, 2070; halo BK 32, 5 stages, 985 -- the fastest;
    // 512->1024 @40 pair per-tap BK 64 713, halo BK 32 990 a stage, 72
    // against 48 stages a tile: halo the faster by 7 %).
    const long long epi_c = p->dtype == CONV_I8 ? 10 : (p->act == CONV_ACT_MISH ? 16 : 6);
    // The bias (and the int8 multipliers) copied into shared memory once per
    // CTA, where Cout <= 2048, for single-CTA layouts: their epilogue no longer
    // waits on global loads (measured: 3x3 s2 256->512 @80 16.1 -> 15.6 us,
    // 1x1 1024->512 @20 batch 8 10.7 -> 10.4 us); the CTA-pair layers, whose
    // epilogues hide under the next tile's MMAs, measured 0.3-1 % slower with it.
    const int bias_bytes = p->s.c_out <= 2048 ? ((p->s.c_out * 4 + 15) & ~15) * (p->dtype == CONV_I8 ? 2 : 1) : 0;
    const int smem_cap0 = 227 * 1024 - 1024 - 512;  // minus the alignment slack and the barriers
    const bool halo_ok = !g.flat && S == 1 && p->s.k_h == 3;  // (the halo variants' tap count)
    if (staging == 2 && !halo_ok) return CONV_ERR_UNSUPPORTED;
    if (epi == 2 && igemm_fused(p)) return CONV_ERR_UNSUPPORTED;  // (no output options per tile)
    struct Cand {
        int swap, pair, bn, bk, halo, ept, cvt, bw, bh, tw, th, wres, stages, out_bufs, mb;
        long long tiles_m, tiles_n, units, rows;
        uint32_t a_stage, raw_stage, raw_region;
    };
    // two tracks: int8 widened by the pre-pass (or no widening), and widened
    // in the kernel; the second wins wherever it has a candidate (see below)
    Cand bests[2]{};
    long long best_costs[2] = {-1, -1};
    const int bk_max = cin % 64 == 0 ? 64 : (cin % 32 == 0 ? 32 : 16);
    for (int cand = 0; cand < 6; ++cand) {
        const bool swap = cand == 0;
        const bool pair = cand == 4 || cand == 5;
        if (swap && p->s.c_out > 128) continue;
        if (pair && p->num_sms < 2) continue;
        if (layout != 0 && layout != cand + 1) continue;
        const int bn = swap ? 128 : (cand == 1 || cand == 4 ? 256 : (cand == 2 || cand == 5 ? 128 : 64));
        const bool ept_ok = !swap && !pair && bn <= 128 && !igemm_fused(p);
        const int smem_cap = smem_cap0 - (!pair && bias_bytes ? bias_bytes + 32 : 0);  // (and the bias copy)
        if (epi == 2 && !ept_ok) continue;
        const int P = swap ? kBMSwap : kBM;
        const int bnc = swap ? 128 : (pair ? bn / 2 : bn);  // weight rows a CTA stages per K block
        // (the largest channel block and half of it; smaller ones only where
        // neither leaves room for two ring stages of this layout and staging)
        for (int bk = bk_max, fits = 0; bk >= 16 && (2 * bk >= bk_max || !fits); bk /= 2) {
            const long long cblocks = cin / bk;
            const long long wblocks = (long long)p->s.k_h * g.kw * cblocks;
            for (int halo = 0; halo <= (halo_ok ? 1 : 0); ++halo) {
                if ((staging == 1 && halo) || (staging == 2 && !halo)) continue;
                // tile shapes: flat (one); per-tap spatial (the fewest tiles,
                // then the widest); halo (bw a multiple of 8, bh x bw <= P)
                int shapes[40][3] = {};  // bw, bh, M blocks a tile
                int nshapes = 0;
                if (g.flat) {
                    shapes[nshapes][0] = P; shapes[nshapes][1] = 1; shapes[nshapes][2] = 1; ++nshapes;
                } else if (!halo) {
                    // (the fewest tiles, then the widest; and, for the fold built in
                    // the kernel, the same among the widths whose raw box rows fit
                    // TMA's 256 elements)
                    for (int pass = 0; pass < (cvt_mode == 2 ? 2 : 1); ++pass) {
                        long long bt = -1;
                        int bw = P, bh = 1;
                        for (int cw = 1; cw <= P && cw <= p->ow * 2; ++cw) {
                            if (cw * S > 256) break;
                            if (pass == 1 && fold_inner(p, cw) > 256) break;
                            int ch = P / cw;
                            if (ch > p->oh) ch = p->oh;
                            while (ch * S > 256) --ch;
                            if (ch < 1) continue;
                            const long long t = (long long)((p->ow + cw - 1) / cw) * ((p->oh + ch - 1) / ch) * p->s.n;
                            if (bt < 0 || t < bt || (t == bt && cw > bw)) { bt = t; bw = cw; bh = ch; }
                            if (cw >= p->ow) break;
                        }
                        if (bt < 0 || (pass == 1 && bw == shapes[0][0])) continue;
                        shapes[nshapes][0] = bw; shapes[nshapes][1] = bh; shapes[nshapes][2] = 1; ++nshapes;
                    }
                } else {
                    for (int cw = 8; cw <= P && cw <= 256 && nshapes < 40; cw += 8) {
                        int ch = P / cw;
                        if (ch > p->oh) ch = p->oh;
                        if (ch + p->s.k_h - 1 > 256) continue;
                        shapes[nshapes][0] = cw; shapes[nshapes][1] = ch; shapes[nshapes][2] = 1; ++nshapes;
                        if (cw >= p->ow) break;  // wider tiles only waste more columns
                    }
                    // The stem fold built in the kernel (N = 64): also tiles of two
                    // 128-pixel M blocks stacked (bh = 2 x 128 / bw), so that the
                    // roles' fixed costs per tile are paid once per 256 pixels; the
                    // converter reaches at most 384 box rows
                    if (cvt_mode == 2 && !swap && !pair && bn == 64) {
                        for (int i = 0, n1 = nshapes; i < n1 && nshapes < 40; ++i) {
                            const int cw = shapes[i][0], ch = 2 * shapes[i][1];
                            if (shapes[i][1] * cw != kBM || ch > p->oh || ch + p->s.k_h - 1 > 256 ||
                                (ch + p->s.k_h - 1) * cw > 384)
                                continue;
                            shapes[nshapes][0] = cw; shapes[nshapes][1] = ch; shapes[nshapes][2] = 2; ++nshapes;
                        }
                    }
                }
                for (int ci = 0; ci < 2 * nshapes; ++ci) {
                    const int si = ci / 2, cvt = ci % 2;  // cvt: int8 widened in the kernel
                    if (cvt && (!cvt_ok || swap || pair || bn > 128 || widen == 1)) continue;
                    if (!cvt && widen == 2) continue;
                    Cand c{};
                    c.swap = swap; c.pair = pair; c.bn = bn; c.bk = bk; c.halo = halo; c.cvt = cvt;
                    c.bw = shapes[si][0]; c.bh = shapes[si][1]; c.mb = shapes[si][2] == 2 ? 2 : 1;
                    if (c.mb == 2 && !cvt) continue;  // (two M blocks: the in-kernel fold only)
                    if (g.flat) {
                        const long long M = (long long)p->s.n * p->s.h * g.wx;
                        c.tiles_m = (M + P - 1) / P;
                        c.tw = 1; c.th = 1;
                    } else {
                        c.tw = (p->ow + c.bw - 1) / c.bw;
                        c.th = (p->oh + c.bh - 1) / c.bh;
                        c.tiles_m = (long long)c.tw * c.th * p->s.n;
                    }
                    c.tiles_n = swap ? 1 : (p->s.c_out + bn - 1) / bn;
                    c.units = (pair ? (c.tiles_m + 1) / 2 : c.tiles_m) * c.tiles_n;
                    // One epilogue per tile where each CTA gets at least two tiles
                    // (with fewer, slicing every tile's columns over the warpgroups
                    // finishes each tile sooner), or where forced.
                    c.ept = ept_ok && epi != 1 && (epi == 2 || c.units >= 2LL * p->num_sms) ? 1 : 0;
                    if (c.mb == 2 && !c.ept) continue;  // (two M blocks: an epilogue per tile)
                    // Shared memory: ring stages, resident weights, epilogue
                    // staging.  A halo stage holds the box's (bh + k_h - 1) x bw
                    // pixel rows and, when bh x bw < P, the P - bh x bw rows the
                    // last tap's MMAs read past them (stale, never stored).
                    const int hrows = c.bh + p->s.k_h - 1;
                    const int box_rows = halo ? hrows * c.bw : P;  // pixel rows TMA writes per stage
                    const int read_rows = halo ? (p->s.k_h - 1) * c.bw + c.mb * P : P;
                    const int a_rows = box_rows > read_rows ? box_rows : read_rows;
                    c.a_stage = (uint32_t)(((long long)a_rows * bk * 2 + 1023) / 1024 * 1024);
                    const long long ring_kb = halo ? (long long)g.kw * cblocks : wblocks;  // stages per tile
                    const long long wblock = (long long)bnc * bk * 2;
                    // In-kernel widening where each CTA gets at least four tiles,
                    // or where the weights are at most half the bytes of the CTA's
                    // output pixels' input channels (or where forced): every CTA
                    // widens the whole weight tensor before its first MMA, which a
                    // layer of about one tile per CTA pays in full.  Measured
                    // (warm): int8 3x3 64->64 @96, 72 tiles, weights 36 KB against
                    // 8 KB: 14.5 us against 10.5 with the pre-pass; 1x1 32->64
                    // @96, 2 KB against 4 KB: 7.6 against 10.0; 3x3 64->64 @160
                    // batch 8, 1600 tiles: 51.9 against 70.0.
                    if (cvt && cvt_mode == 1 && widen != 2 && c.units < 4LL * p->num_sms) {
                        const long long per_cta = (c.units + p->num_sms - 1) / p->num_sms;
                        if (2 * wblocks * bnc * bk > per_cta * P * cin) continue;
                    }
                    const int one_buf = swap ? 4 * 16 * kTP : epi_groups(bn, false, c.ept != 0) * kBM * 64;
                    // swapped plain bf16 layers whose 16-pixel chunks lie in one row
                    // write out by TMA stores from two staging buffers per warp
                    const bool swap_tma = swap && !igemm_fused(p) && p->dtype == CONV_BF16 && (g.flat || c.bw % 16 == 0);
                    c.out_bufs = swap_tma ? 2 : 1;
                    if (!swap && wblocks < 16 && (smem_cap - 2 * one_buf) / ((long long)c.a_stage + wblock) >= 4)
                        c.out_bufs = 2;
                    const long long out_bytes = (long long)one_buf * c.out_bufs;
                    const long long wall = wblocks * wblock;
                    const int min_stages = halo ? 3 : 4;
                    c.wres = (c.tiles_n == 1 && (smem_cap - out_bytes - wall) / (long long)c.a_stage >= min_stages)
                                 ? 1 : 0;
                    const int taps = halo ? 3 : 1;  // weight blocks a stage carries
                    const long long stage_bytes = c.a_stage + (c.wres ? 0 : taps * wblock);
                    long long st = (smem_cap - out_bytes - (c.wres ? wall : 0)) / stage_bytes;
                    if (st > 8) st = 8;
                    if (cvt) {
                        // resident (widened) weights, and a raw region holding first the
                        // raw int8 weights, then the raw ring of int8 activation boxes;
                        // folded: first the raw bf16 weights (and 36 bytes of slack for the
                        // converter's whole-word reads), then
                        // the raw ring of image-row boxes, each box row the
                        // ((bw - 1) x stride + k_w) x Cin elements under the tile from
                        // the 16-byte unit at or before its first, at most 256
                        if (!c.wres) continue;
                        long long wraw = wblocks * bnc * bk;
                        if (cvt_mode == 2) {
                            const int inner = fold_inner(p, c.bw);
                            if (inner > 256) continue;
                            const int rrows = halo ? hrows : c.bh;
                            // (36 bytes of slack: the converter reads nine whole words per row)
                            c.raw_stage = (uint32_t)(((long long)inner * rrows * 2 + 36 + 127) / 128 * 128);
                            wraw = (long long)p->s.c_out * p->s.k_h * p->s.k_w * p->s.c_in * 2 + 36;
                        } else {
                            c.raw_stage = (uint32_t)(((long long)box_rows * bk + 127) / 128 * 128);
                        }
                        for (; st >= 2; --st) {
                            const long long ring = st * (long long)c.raw_stage;
                            const long long region = ((ring > wraw ? ring : wraw) + 1023) / 1024 * 1024;
                            if (st * c.a_stage + wall + out_bytes + region + 16 * st <= smem_cap) {
                                c.raw_region = (uint32_t)region;
                                break;
                            }
                        }
                    }
                    if (st < 2) continue;
                    c.stages = (int)st;
                    fits = 1;
                    // the estimate
                    const long long slots = pair ? p->num_sms / 2 : p->num_sms;
                    const long long waves = (c.units + slots - 1) / slots;
                    c.rows = ring_kb * box_rows + (c.wres ? 0 : wblocks * bnc);  // staged rows per tile
                    // (the staged swapped write-out -- shared-memory loads, global
                    // stores and their address arithmetic in the epilogue threads --
                    // adds ~650 cycles per 16-pixel chunk, measured; the TMA
                    // write-out moves that to the TMA engine)
                    const long long t_epi = 128LL * (swap ? P : bn) * c.mb * epi_c / 128 + (swap && c.out_bufs == 1 ? 2600 : 0);
                    // a stage: its MMAs, its TMA rows, or the ring's refill latency
                    // spread over the other stages, whichever is longest, plus a
                    // fixed cost of the stage's barrier round trip
                    const long long m_stage = (long long)taps * (bk / 16) * 128 * c.mb;
                    const long long rows_stage = box_rows + (c.wres ? 0 : (long long)taps * bnc);
                    long long per_stage = 2000 / (c.stages - 1);
                    if (per_stage < m_stage) per_stage = m_stage;
                    if (per_stage < 7 * rows_stage / 5) per_stage = 7 * rows_stage / 5;
                    const long long t_ring = ring_kb * (per_stage + 200);
                    const long long t_tile = t_ring > t_epi ? t_ring : t_epi;
                    const long long cost = waves * (t_tile + 500);
                    // ties: the TMA write-out of the swapped layout (measured faster
                    // than the staged one at equal estimates: 64->128 @160 batch 8,
                    // 8x32 tiles 24.7 us warm against 29.8 for 10x24 staged), more
                    // work units (more SMs busy), then fewer staged rows, then the
                    // narrower N tile
                    Cand &best = bests[cvt];
                    long long &best_cost = best_costs[cvt];
                    const int tma_c = swap && c.out_bufs == 2, tma_b = best.swap && best.out_bufs == 2;
                    const bool better =
                        best_cost < 0 || cost < best_cost ||
                        (cost == best_cost &&
                         (tma_c > tma_b ||
                          (tma_c == tma_b &&
                           (c.units > best.units ||
                            (c.units == best.units && (c.rows < best.rows || (c.rows == best.rows && bn < best.bn)))))));
                    if (better) {
                        best_cost = cost;
                        best = c;
                    }
                }
            }
        }
    }
    const int track = best_costs[1] >= 0 ? 1 : 0;
    if (best_costs[track] < 0) return CONV_ERR_UNSUPPORTED;  // e.g. a forced swapped layout with c_out > 128
    const Cand &best = bests[track];
    g.swap = best.swap; g.pair = best.pair; g.bn = best.bn; g.bk = best.bk; g.halo = best.halo; g.ept = best.ept;
    g.cvt = best.cvt;
    g.mb = best.mb;
    g.raw_stage = (int)best.raw_stage;
    g.raw_region = (int)best.raw_region;
    // plan-owned bf16 copies of x and w (channels padded to `cin`), unless the
    // kernel reads the operands as they are (bf16 with whole rows) or widens
    // them itself (CVT)
    g.cvt = g.cvt ? cvt_mode : 0;
    g.prep = !g.cvt && (cin != p->s.c_in || p->dtype == CONV_I8) ? 1 : 0;
    if (g.prep) {
        const size_t xb = (size_t)p->s.n * p->s.h * g.wx * cin * 2;
        const size_t wb = (size_t)p->s.c_out * p->s.k_h * g.kw * cin * 2;
        p->cin_p = cin;
        if (xb && cudaMalloc(&p->d_xprep, xb) != cudaSuccess) return CONV_ERR_OOM;
        if (cudaMalloc(&p->d_wprep, wb) != cudaSuccess) return CONV_ERR_OOM;
    }
    g.cblocks = cin / g.bk;
    const int wblocks = p->s.k_h * g.kw * g.cblocks;
    g.tiles_n = (int)best.tiles_n; g.tiles_m = (int)best.tiles_m;
    g.bw = best.bw; g.bh = best.bh; g.tiles_w = best.tw; g.tiles_h = best.th;
    g.wres = best.wres; g.stages = best.stages; g.out_bufs = best.out_bufs;
    g.a_stage = (int)best.a_stage;
    g.kblocks = g.halo ? g.kw * g.cblocks : wblocks;
    g.num_tiles = (int)best.units;  // work units
    {
        const int bnc = g.swap ? 128 : (g.pair ? g.bn / 2 : g.bn);
        const int wblock = bnc * g.bk * 2;
        const int one_buf = g.swap ? 4 * 16 * kTP : epi_groups(g.bn, false, g.ept != 0) * kBM * 64;
        const int weights = g.wres ? wblocks * wblock : g.stages * (g.halo ? 3 : 1) * wblock;
        g.smem = 1024 + g.stages * g.a_stage + weights + one_buf * g.out_bufs + (g.cvt ? g.raw_region : 0) +
                 8 * (g.cvt ? 4 * g.stages + 10 : 2 * g.stages + 9) + 16;
        g.bias_smem = bias_bytes && !g.pair ? 1 : 0;
        if (g.bias_smem) g.smem += bias_bytes + 16;
    }
    // Ask for more than half of an SM's shared memory so that no two CTAs of
    // this persistent kernel share an SM: each CTA then owns its TMEM
    // columns (at most 512) without waiting for another to free them.
    if (g.smem < 116 * 1024) g.smem = 116 * 1024;
    if (!tensor_map_encoder()) return CONV_ERR_CUDA;
    void *kern = select_kernel(g.bn, g.bk, g.flat != 0, g.swap != 0, g.pair != 0, igemm_fused(p), g.halo != 0, g.ept != 0,
                              g.cvt, g.mb);
    const int rc = conv_grant_smem(kern, p->device, g.smem);
    if (rc != CONV_OK) return rc;
    if (g.pair) {
        // as many CTA pairs as can be resident at once (a pair occupies two
        // SMs of one GPC), at most one per work unit
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * g.num_tiles);
        cfg.blockDim = dim3(cta_threads(g.bn, false, g.ept != 0, g.cvt != 0));
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
             "igemm_%s_tcgen05 %s%s %s BK=%d tile=%dx%d%s%s stages=%d%s out_bufs=%d%s tiles=%d grid=%d",
             p->dtype == CONV_I8 ? (g.fold ? "i8-as-bf16-kwfold" : (g.cvt ? "i8-widened-in-kernel" : "i8-as-bf16"))
                                 : (g.fold ? (g.cvt ? "bf16-kwfold-in-kernel" : "bf16-cpad-kwfold")
                                           : (g.prep ? "bf16-cpad" : "bf16")),
             g.flat ? "flat" : "spatial",
             g.swap ? " swapped" : (g.pair ? " cta-pair" : ""),
             g.swap ? "M=128co N=256px"
                    : (g.pair ? (g.bn == 256 ? "M=256px N=256co" : "M=256px N=128co")
                              : (g.bn == 256 ? "M=128px N=256co" : (g.bn == 128 ? "M=128px N=128co" : "M=128px N=64co"))),
             g.bk, g.bh, g.bw, g.mb == 2 ? " (2 M blocks)" : "", g.halo ? " halo" : "", g.stages,
             g.wres ? " resident-weights" : "", g.out_bufs,
             g.ept ? " epi=tile" : "", g.num_tiles, g.grid);
    return CONV_OK;
}

int launch_igemm(const conv_plan *p, const void *x, const void *w, const void *bias, const void *res, void *y,
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
    // CVT: the operands as they are, int8, unswizzled (the converter
    // warpgroup widens them into the swizzled bf16 layout)
    const cuuint64_t es = g.cvt == 1 ? 1 : 2;
    const CUtensorMapDataType op_type = g.cvt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle op_swz = g.cvt ? CU_TENSOR_MAP_SWIZZLE_NONE : swizzle_for(g.bk);
    const int inner = g.cvt == 2 ? fold_inner(p, g.bw) : 0;
    if (g.cvt == 2) {
        // folded in the kernel: x as [N][H][W x Cin] element rows; a box is
        // `inner` elements of the tile's input rows (every stride-th row per
        // tap, or the bh + k_h - 1 rows of a halo box)
        const cuuint64_t row = (cuuint64_t)p->s.w * p->s.c_in;
        const cuuint64_t dims[3] = {row, (cuuint64_t)p->s.h, (cuuint64_t)p->s.n};
        const cuuint64_t strides[2] = {row * 2, (cuuint64_t)p->s.h * row * 2};
        const cuuint32_t box[3] = {(cuuint32_t)inner,
                                   g.halo ? (cuuint32_t)(g.bh + p->s.k_h - 1) : (cuuint32_t)(g.bh * S), 1};
        const cuuint32_t estr[3] = {1, g.halo ? 1u : (cuuint32_t)S, 1};
        rc = encode(&tmA, op_type, 3, const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    op_swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (g.flat) {
        const cuuint64_t dims[2] = {(cuuint64_t)cin, (cuuint64_t)p->s.n * p->s.h * g.wx};
        const cuuint64_t strides[1] = {(cuuint64_t)cin * es};
        const cuuint32_t box[2] = {(cuuint32_t)g.bk, (cuuint32_t)(g.swap ? kBMSwap : kBM)};
        rc = encode(&tmA, op_type, 2, const_cast<void *>(x), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    op_swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[4] = {(cuuint64_t)cin, (cuuint64_t)g.wx, (cuuint64_t)p->s.h,
                                    (cuuint64_t)p->s.n};
        const cuuint64_t strides[3] = {(cuuint64_t)cin * es, (cuuint64_t)g.wx * cin * es,
                                       (cuuint64_t)p->s.h * g.wx * cin * es};
        // halo staging: the bh + k_h - 1 input rows under the tile (stride 1)
        const cuuint32_t box_h = g.halo ? (cuuint32_t)(g.bh + p->s.k_h - 1) : (cuuint32_t)(g.bh * S);
        const cuuint32_t box[4] = {(cuuint32_t)g.bk, (cuuint32_t)(g.bw * S), box_h, 1};
        const cuuint32_t estr[4] = {1, (cuuint32_t)S, (cuuint32_t)S, 1};
        rc = encode(&tmA, op_type, 4, const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    op_swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (rc != CUDA_SUCCESS) return CONV_ERR_CUDA;
    if (g.cvt == 2) {
        // (the converter reads the weights from global memory; a valid map of
        // x's first 16 bytes stands in for the unused weight map)
        const cuuint64_t dims[2] = {8, 1};
        const cuuint64_t strides[1] = {16};
        const cuuint32_t box[2] = {8, 1};
        rc = encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, ones,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV_ERR_CUDA;
    } else {
        const cuuint64_t K = (cuuint64_t)p->s.k_h * g.kw * cin;
        const cuuint64_t dims[2] = {K, (cuuint64_t)p->s.c_out};
        const cuuint64_t strides[1] = {K * es};
        const cuuint32_t box[2] = {(cuuint32_t)g.bk, (cuuint32_t)(g.pair ? g.bn / 2 : g.bn)};
        rc = encode(&tmB, op_type, 2, const_cast<void *>(w), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    op_swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV_ERR_CUDA;
    }

    // Output maps: y's channel slice [c_off, c_off + Cout) at the pixels of
    // upsample replica (dy, dx); 32 channels per store box (64 bytes of
    // bf16, 64-byte swizzle; or 32 bytes of int8, unswizzled).  Channels past
    // Cout and pixels past the image are clipped by TMA, so neighbouring
    // slices of a concatenated y are never written.
    alignas(64) YMaps tmY;
    {
        const bool i8 = p->dtype == CONV_I8;
        const cuuint64_t es = i8 ? 1 : 2;
        const CUtensorMapDataType dt = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapSwizzle sw = i8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B;
        const cuuint32_t box_n = 32;
        const int up = p->up;
        const cuuint64_t Cy = (cuuint64_t)p->y_c, OWy = (cuuint64_t)p->ow * up, OHy = (cuuint64_t)p->oh * up;
        for (int rp = 0; rp < up * up; ++rp) {
            const int dy = rp / up, dx = rp % up;
            char *base = static_cast<char *>(y) + ((cuuint64_t)p->y_coff + ((cuuint64_t)dy * OWy + dx) * Cy) * es;
            if (g.swap && g.out_bufs == 2) {
                // swapped TMA write-out: [16 pixels][32 channels] boxes, one per
                // warp, 64-byte swizzle
                if (g.flat) {
                    const cuuint64_t dims[2] = {(cuuint64_t)p->s.c_out, (cuuint64_t)p->s.n * p->oh * p->ow};
                    const cuuint64_t strides[1] = {Cy * es};
                    const cuuint32_t box[2] = {32, 16};
                    rc = encode(&tmY.m[rp], dt, 2, base, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                } else {
                    const cuuint64_t dims[4] = {(cuuint64_t)p->s.c_out, (cuuint64_t)p->ow, (cuuint64_t)p->oh,
                                                (cuuint64_t)p->s.n};
                    const cuuint64_t strides[3] = {Cy * es, OWy * Cy * es, OHy * OWy * Cy * es};
                    const cuuint32_t box[4] = {32, 16, 1, 1};
                    rc = encode(&tmY.m[rp], dt, 4, base, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                }
            } else if (g.flat) {  // (up == 1)
                const cuuint64_t dims[2] = {(cuuint64_t)p->s.c_out, (cuuint64_t)p->s.n * p->oh * p->ow};
                const cuuint64_t strides[1] = {Cy * es};
                const cuuint32_t box[2] = {box_n, (cuuint32_t)(g.swap ? kBMSwap : kBM)};
                rc = encode(&tmY.m[rp], dt, 2, base, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            } else {
                const cuuint64_t dims[4] = {(cuuint64_t)p->s.c_out, (cuuint64_t)p->ow, (cuuint64_t)p->oh,
                                            (cuuint64_t)p->s.n};
                const cuuint64_t strides[3] = {up * Cy * es, up * OWy * Cy * es, OHy * OWy * Cy * es};
                // (two M blocks a tile: one store per block, its bh / 2 rows)
                const cuuint32_t box[4] = {box_n, (cuuint32_t)g.bw, (cuuint32_t)(g.bh / g.mb), 1};
                rc = encode(&tmY.m[rp], dt, 4, base, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            }
            if (rc != CUDA_SUCCESS) return CONV_ERR_CUDA;
        }
    }

    IgArgs a;
    a.H = p->s.h; a.W = g.wx; a.Cin = cin; a.Cout = p->s.c_out; a.KH = p->s.k_h; a.KW = g.kw;
    a.stride = S; a.pad_h = p->pad_h; a.pad_w = g.padw; a.OH = p->oh; a.OW = p->ow;
    a.bw = g.bw; a.bh = g.bh; a.tiles_w = g.tiles_w; a.tiles_h = g.tiles_h; a.tiles_n = g.tiles_n;
    a.num_tiles = g.num_tiles; a.cblocks = g.cblocks; a.kblocks = g.kblocks; a.stages = g.stages;
    a.tiles_m = g.tiles_m;
    a.M = (long long)p->s.n * p->s.h * g.wx;
    const int box_rows = g.flat ? (g.swap ? kBMSwap : kBM) : g.bw * (g.halo ? g.bh + p->s.k_h - 1 : g.bh);
    a.a_bytes = g.cvt == 2 ? (uint32_t)(inner * (g.halo ? g.bh + p->s.k_h - 1 : g.bh) * 2)
                           : (uint32_t)(box_rows * g.bk * (int)es);
    a.box_rows = box_rows;
    a.fold_cin = p->s.c_in; a.fold_kw = p->s.k_w; a.fold_padw = p->pad_w; a.raw_inner = inner;
    a.w_raw = static_cast<const __nv_bfloat16 *>(w);
    a.raw_stage = (uint32_t)g.raw_stage;
    a.raw_region = (uint32_t)g.raw_region;
    a.a_stage = (uint32_t)g.a_stage;
    a.halo = g.halo;
    a.wblocks = p->s.k_h * g.kw * g.cblocks;
    a.flat = g.flat;
    a.act = (int)p->act;
    a.bias = bias;
    a.y = y;
    a.out_i8 = p->dtype == CONV_I8 ? 1 : 0;
    a.mult = p->d_mult;
    a.out_bufs = g.out_bufs;
    a.bias_smem = g.bias_smem;
    a.wres = g.wres;
    a.om.Cy = p->y_c; a.om.c_off = p->y_coff; a.om.up = p->up;
    a.om.OH = p->oh; a.om.OW = p->ow; a.om.Cout = p->s.c_out;
    a.om.res = res;
    a.status = p->d_status;

    void *k = select_kernel(g.bn, g.bk, g.flat != 0, g.swap != 0, g.pair != 0, igemm_fused(p), g.halo != 0, g.ept != 0,
                              g.cvt, g.mb);
    void *args[] = {&tmA, &tmB, &tmY, &a};
    const cudaError_t e = conv_launch(k, dim3(g.grid), dim3(cta_threads(g.bn, g.swap != 0, g.ept != 0, g.cvt != 0)), args, (size_t)g.smem, st,
                                      g.pair ? 2 : 1);
    return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}
