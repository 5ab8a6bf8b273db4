// Internal declarations of the fused NHWC convolution library: the plan
// structure and the launchers of the three kernel families.  Not part of the
// public ABI (include/conv_nhwc.h is).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "conv_nhwc.h"

// Status word codes written by kernels (device side) into the plan's status
// word; conv_plan_check_device_status maps any nonzero value to
// CONV_ERR_DEVICE_TIMEOUT.
enum {
    KSTATUS_OK = 0,
    KSTATUS_TIMEOUT_PRODUCER = 1,  // TMA warp gave up waiting for a free stage
    KSTATUS_TIMEOUT_MMA = 2,       // MMA warp gave up waiting for data / TMEM
    KSTATUS_TIMEOUT_EPILOGUE = 3,  // epilogue gave up waiting for an accumulator
};

// Geometry of the tcgen05 implicit-GEMM launch chosen at plan time.
struct IgemmGeom {
    int bn;        // output channels per tile (UMMA N): 64, 128 or 256
    int bk;        // input channels per K block: 64, 32 or 16 (128/64/32-byte rows)
    int flat;      // 1: 1x1 / stride 1 / pad 0, A is x viewed as [N*H*W, Cin]
    int bw, bh;    // spatial mode: an M tile is a bh x bw rectangle of output pixels
    int tiles_w, tiles_h, tiles_m, tiles_n, num_tiles;
    int cblocks;   // Cin / bk
    int kblocks;   // ring stages per tile: k_h * k_w * cblocks, or k_w * cblocks with halo staging
    int halo;      // 1: halo staging (a stage holds the tile's input rows for all k_h taps of one column shift)
    int a_stage;   // bytes of the activation part of a ring stage
    int ept;       // 1: one epilogue per tile (each warpgroup drains whole tiles, four TMEM accumulators)
    int bias_smem; // 1: the bias (and int8 multipliers) copied into shared memory once per CTA
    int cvt;       // 1: int8 operands widened to bf16 in the kernel (converter warpgroup), no pre-pass
    int mb;        // M blocks of 128 pixels a tile (2: the in-kernel stem fold, two blocks stacked)
    int raw_stage; // cvt: bytes of a raw int8 activation stage
    int raw_region;  // cvt: bytes of the raw region (raw weights, then the raw ring)
    int stages;    // shared-memory pipeline depth
    int out_bufs;  // epilogue output staging buffers per group (1 or 2)
    int wres;      // 1: all weights resident in shared memory (one N block, loaded once per CTA)
    int grid;      // persistent CTAs
    int smem;      // dynamic shared memory bytes
    int in_i8;     // operands are int8 (converted to bf16 on chip)
    int swap;      // 1: MMA M = output channels, N = 256 pixels (Cout <= 128)
    int pair;      // 1: CTA-pair MMA, M = 2 x 128 pixels over a cluster of two CTAs, N = 256
    int prep;      // 1: x and w are widened to bf16 / channel-padded first
    int cin;       // input channels the kernel sees (padded when prep)
    int fold;      // 1: the k_w taps are folded into the (padded) channels by the pre-pass
    int kw, wx, padw;  // kernel width, x width and w padding the kernel sees (1, W', 0 when fold)
};

struct DwGeom {
    int kind;      // 0: general kernel; 1: bf16 stride-1 rolling-row kernel
    int th, tw;    // output rows / columns of one CTA tile
    int cbv;       // 16-byte channel vectors per tile
    int hin, win;  // input halo rows / columns (one TMA box)
    int tiles_w, tiles_h, tiles_c;
    int smem;      // dynamic shared memory bytes (the halo)
    int threads;   // threads per CTA
    long long tiles;   // output tiles
    long long blocks;  // persistent CTAs
};

struct DwpwGeom {
    int th, tw;        // output pixels of a CTA tile
    int hin, win;      // its input halo
    int cochunk;       // pointwise output channels per CTA (multiple of 4)
    int chunks;        // ceil(Cout / cochunk)
    int tiles_w, tiles_h;
    int smem;          // dynamic shared memory bytes
};

struct conv_plan {
    conv_shape_t s;
    int stride, pad_h, pad_w, groups;
    conv_dtype_t dtype;
    conv_act_t act;
    int oh, ow;
    int algo;          // conv_algo_t actually used
    int device;
    int num_sms;
    float *d_mult;     // int8: requantisation multipliers M[co] (device)
    int *d_status;     // device status word (bounded-wait timeouts)
    __nv_bfloat16 *d_xprep, *d_wprep;  // bf16 (channel-padded) copies of x and w for the tensor-core path
    int cin_p;         // channels of those copies
    IgemmGeom ig;
    DwGeom dw;
    DwpwGeom dwpw;
    conv_act_t act2;   // fused depthwise -> pointwise plans: the pointwise activation
    int dct, dpt;      // direct kernel: channels / pixels per thread of the smem variant (dct 0: generic)
    // Output options (conv_output_t): y has y_c channels per pixel, the layer
    // writes channels [y_coff, y_coff + c_out) of a (up*OH) x (up*OW) grid,
    // adding the residual tensor when has_res.
    int y_c, y_coff, up, has_res;
    char desc[192];
};

// Element size of a conv_dtype_t.
static inline int conv_esize(conv_dtype_t t) { return t == CONV_F32 ? 4 : (t == CONV_BF16 ? 2 : 1); }

// Every kernel of the library is launched with programmatic stream
// serialisation: it may be scheduled while the previous kernel on the stream
// drains, and waits (griddepcontrol.wait, pdl_wait) until that kernel has
// completed and its writes are visible before its first global access, so
// the launch latency and the kernel's set-up overlap the previous kernel's
// tail.  cluster_x > 1 launches clusters of that many CTAs along x.
cudaError_t conv_launch(const void *kernel, dim3 grid, dim3 block, void **args, size_t smem, cudaStream_t st,
                        int cluster_x = 1);

// Launchers (stream-ordered, no allocation, no synchronisation).
cudaError_t launch_direct(const conv_plan *p, const void *x, const void *w, const void *bias,
                          const void *res, void *y, cudaStream_t st);
cudaError_t launch_dw3x3(const conv_plan *p, const void *x, const void *w, const void *bias,
                         void *y, cudaStream_t st);
// Returns a CONV_* status (tensor-map encoding can fail on the host).
int launch_igemm(const conv_plan *p, const void *x, const void *w, const void *bias, const void *res,
                 void *y, cudaStream_t st);

// Fused depthwise 3x3 -> pointwise pair (conv_plan_create_dwpw).
cudaError_t launch_dwpw(const conv_plan *p, const void *x, const void *wdw, const void *bdw, const void *wpw,
                        const void *bpw, void *y, cudaStream_t st);
bool dwpw_supported(const conv_plan *p);
int dwpw_configure(conv_plan *p);  // CONV_* status

// Widens int8 to bf16 / pads channels into the plan's d_xprep, d_wprep.
cudaError_t launch_prep(const conv_plan *p, const void *x, const void *w, cudaStream_t st);

// Plan-time helpers of each family.
bool direct_supported(const conv_plan *p);
void direct_configure(conv_plan *p);
bool dw3x3_supported(const conv_plan *p);
int dw3x3_configure(conv_plan *p);  // CONV_* status
bool igemm_supported(const conv_plan *p);
// The tcgen05 kernel variant for layers with output options (a residual or
// upsample replicas), compiled in its own translation unit.
void *igemm_select_fused(int bn, int bk, bool flat, bool swap, bool pair, bool halo);
// The variant with one epilogue per tile (normal layout, BN 64 or 128, no
// output options), compiled in its own translation unit.
void *igemm_select_ept(int bn, int bk, bool flat, bool halo);
// The variant that widens int8 operands in the kernel (normal layout,
// resident weights, no output options), compiled in its own translation unit.
void *igemm_select_cvt(int mode, int bn, int bk, bool flat, bool halo, bool ept, int mb);
// Fills p->ig and sets kernel attributes; CONV_* status.  layout 0 picks
// the tile layout by estimated time; 1..6 force swapped, N256, N128, N64,
// CTA pair (N = 256), CTA pair (N = 128).  staging 0 picks per-tap or halo
// staging by estimated time; 1 forces per-tap boxes, 2 halo staging.  epi 0
// picks the epilogue split by the tile count; 1 forces column slices, 2 one
// epilogue per tile.  widen (int8 layers) 0 picks, 1 forces the widening
// pre-pass, 2 the in-kernel converter.
int igemm_configure(conv_plan *p, int layout, int staging, int epi, int widen);

// Host-side argument checks shared by the entry points (api.cu).
int conv_validate_layer(const conv_shape_t *s, int stride, int pad_h, int pad_w, int groups,
                        conv_dtype_t dtype, conv_act_t act, const conv_quant_t *quant, int *oh, int *ow);
int conv_check_run_pointers(conv_dtype_t dtype, const conv_shape_t *s, int groups, int oh, int ow,
                            const void *x, const void *w, const void *bias, const void *y);

// Grants kernel `k` the device's whole opt-in dynamic shared memory (minus its
// static shared memory) and checks that `need` bytes fit.  The attribute is a
// per-kernel permission shared by all plans, so it is never lowered to one
// plan's size.  Returns a CONV_* status.
int conv_grant_smem(const void *k, int device, int need);
