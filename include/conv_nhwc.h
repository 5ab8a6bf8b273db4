/*
 * conv_nhwc.h -- C ABI of the fused NHWC 2-D convolution layer for GB300
 * (sm_103a): y = epilogue(conv(x, w) + bias).
 *
 * The operation.  A 2-D cross-correlation over NHWC activations with OHWI
 * weights, zero padding, one stride for both axes and one pad per axis
 * applied on both sides, followed by a fused epilogue: bias, then ReLU or
 * Mish, then (int8 layers) per-output-channel requantisation.
 *
 *   OH = floor((H + 2*pad_h - k_h) / stride) + 1   (likewise OW)
 *   y[n,oh,ow,co] = act( b[co] + sum_{r<k_h, s<k_w, j<Cin/groups}
 *                        x[n, oh*stride-pad_h+r, ow*stride-pad_w+s, g0+j]
 *                        * w[co, r, s, j] ),    g0 = (co / (Cout/groups)) * (Cin/groups)
 *
 *   - layer types: dense k x k (any k_h, k_w, including asymmetric kernels
 *     such as the 10x4 keyword-spotting stem with padding (5, 1) of the
 *     "nanoinfer" page, section "Asymmetric padding collapsed to one axis"),
 *     1x1 pointwise ("nanoinfer", "1x1 convolutions are already a GEMM"),
 *     depthwise (groups == Cin == Cout) and grouped;
 *   - Mish(v) = v * tanh(ln(1 + e^v)) ("YOLOv4, optimized for Wormhole",
 *     section 7, the Mish / HardMish table), computed in fp32;
 *   - int8 requantisation with symmetric scales and no zero point
 *     ("nanoinfer", post-training quantization: symmetric per-output-channel
 *     weight scales, calibrated activation range):
 *       M[co] = float(double(s_x) * double(s_w[co]) / double(s_y))  (at plan time)
 *       q = saturate_[-128,127]( round_half_even( float(acc + b[co]) * M[co] ) )
 *     every float operation rounded to nearest-even in single precision;
 *     ReLU, if asked for, is max(q, 0).
 *
 * Data types.  x, w and y share one type: CONV_F32 (fp32 arithmetic on FFMA,
 * never TF32), CONV_BF16 (bf16 operands, fp32 accumulation, output rounded to
 * nearest-even bf16) or CONV_I8 (int8 operands, exact int32 accumulation).
 * The bias is float32 for CONV_F32 / CONV_BF16 and int32 for CONV_I8.
 *
 * Layouts (all dense, row-major, no padding between rows):
 *   x    [N][H][W][Cin]                 (NHWC)
 *   w    [Cout][k_h][k_w][Cin/groups]   (OHWI)
 *   bias [Cout]                          (may be NULL: no bias)
 *   y    [N][OH][OW][Cout]              (NHWC)
 *
 * Ownership.  The caller owns x, w, bias, y (device pointers) and the
 * stream.  The plan owns its host structure and the small device buffers it
 * allocates at creation (requantisation multipliers, a status word); they are
 * freed by conv_plan_destroy.  conv_run never allocates and never
 * synchronises: it enqueues kernels on the caller's stream and returns.
 *
 * Errors.  Every entry point returns CONV_OK (0) or a negative CONV_ERR_*
 * code; conv_status_str names it.  Invalid shapes and unsupported
 * combinations are rejected at plan creation, pointer problems at run time.
 * There is no CPU fallback: a plan either runs on the GPU or fails.
 */
#ifndef CONV_NHWC_H
#define CONV_NHWC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CONV_NHWC_ABI_VERSION 2

#if defined(__GNUC__)
#define CONV_API __attribute__((visibility("default")))
#else
#define CONV_API
#endif

typedef struct {
    int32_t n, h, w;      /* batch, input height, input width (n may be 0) */
    int32_t c_in, c_out;  /* input / output channels */
    int32_t k_h, k_w;     /* kernel height, width */
} conv_shape_t;

typedef enum { CONV_F32 = 0, CONV_BF16 = 1, CONV_I8 = 2 } conv_dtype_t;

typedef enum { CONV_ACT_NONE = 0, CONV_ACT_RELU = 1, CONV_ACT_MISH = 2 } conv_act_t;

/* int8 quantisation parameters: activation scale s_x, output scale s_y and
 * c_out per-output-channel weight scales s_w (a HOST array, read and copied
 * during conv_plan_create; the caller may free it afterwards).  All > 0. */
typedef struct {
    float in_scale;
    float out_scale;
    const float *w_scales;
} conv_quant_t;

/* Kernel family a plan runs.  AUTO picks one from the shape; the others force
 * a family (for tests), failing with CONV_ERR_UNSUPPORTED where it cannot
 * run the layer. */
typedef enum {
    CONV_ALGO_AUTO = 0,
    CONV_ALGO_DIRECT = 1,     /* CUDA-core direct convolution, any shape  */
    CONV_ALGO_DEPTHWISE = 2,  /* depthwise 3x3 register/L1 stencil        */
    CONV_ALGO_IGEMM = 3,      /* tcgen05 implicit GEMM (TMA, TMEM)        */
    /* CONV_ALGO_IGEMM with a fixed tile layout instead of the estimated
     * fastest one (conv_plan_algo then reports CONV_ALGO_IGEMM):          */
    CONV_ALGO_IGEMM_SWAPPED = 4, /* MMA M = 128 output channels, N = 256 pixels (c_out <= 128) */
    CONV_ALGO_IGEMM_N256 = 5,    /* MMA M = 128 pixels, N = 256 output channels */
    CONV_ALGO_IGEMM_N128 = 6,    /* MMA M = 128 pixels, N = 128 output channels */
    CONV_ALGO_IGEMM_N64 = 7,     /* MMA M = 128 pixels, N = 64 output channels  */
    CONV_ALGO_IGEMM_PAIR = 8,    /* CTA-pair MMA on two SMs: M = 256 pixels, N = 256 */
    /* (reported by conv_plan_algo for plans of conv_plan_create_dwpw; not a
     * family conv_plan_create_ex can force) */
    CONV_ALGO_DWPW = 9,          /* fused depthwise 3x3 -> pointwise 1x1 pair */
    CONV_ALGO_IGEMM_PAIR128 = 10, /* CTA-pair MMA: M = 256 pixels, N = 128 output channels */
} conv_algo_t;

/* Staging of the tensor-core family's pixel operand, OR-ed into CONV_ALGO_IGEMM
 * or one of its layouts (without either flag the plan's estimate chooses):
 *   TAPS  one TMA box of input pixels per filter tap (r, s) and channel block;
 *   HALO  one box per column shift s and channel block holding the input rows
 *         under the tile for all three row taps, which the MMAs read at row
 *         offsets (stride-1 layers with k_h = 3 only; CONV_ERR_UNSUPPORTED
 *         otherwise).  Both compute the same sums ("nanoinfer", the implicit
 *         GEMM: im2col is never materialised either way). */
#define CONV_ALGO_STAGE_TAPS 0x100
#define CONV_ALGO_STAGE_HALO 0x200
/* Epilogue split of the tensor-core family, OR-ed in the same way (default:
 * one epilogue per tile where each CTA gets at least two tiles):
 *   SLICED    every epilogue warpgroup drains a slice of each tile's columns;
 *   PER_TILE  each warpgroup drains whole tiles in turn from a TMEM
 *             accumulator of its own (normal layouts with N <= 128 and no
 *             conv_output_t options; CONV_ERR_UNSUPPORTED otherwise). */
#define CONV_ALGO_EPI_SLICED 0x400
#define CONV_ALGO_EPI_PER_TILE 0x800
/* How operands that the tensor cores cannot read as they are reach them,
 * OR-ed in the same way (default: in the kernel where it can, else the
 * pre-pass).  These are int8 layers (sm_103a has no integer MMA; an int8
 * value is exact in bf16) and bf16 layers with k_w x c_in <= 16 (the image
 * stem), whose k_w taps are folded into one 16-channel operand row:
 *   PREPASS   a pre-pass kernel writes bf16 copies of x and w (widened,
 *             channel-padded or folded) into plan-owned buffers, which the
 *             tensor-core kernel reads;
 *   INKERNEL  the kernel loads x as it is and a converter warpgroup builds
 *             the bf16 operand in shared memory: int8 widened (c_in % 16 ==
 *             0), or the folded rows assembled from the plain NHWC image rows
 *             (bf16, w x c_in x 2 a multiple of 16 bytes).  Normal layouts
 *             with N <= 128 whose weights stay resident, no conv_output_t
 *             options; CONV_ERR_UNSUPPORTED otherwise. */
#define CONV_ALGO_WIDEN_PREPASS 0x1000
#define CONV_ALGO_WIDEN_INKERNEL 0x2000

enum {
    CONV_OK = 0,
    CONV_ERR_NULL_ARG = -1,        /* a required pointer is NULL            */
    CONV_ERR_INVALID_SHAPE = -2,   /* sizes, stride, pads or groups invalid */
    CONV_ERR_UNSUPPORTED = -3,     /* valid but not implemented (e.g. I8+Mish) */
    CONV_ERR_MISALIGNED = -4,      /* x, w, bias or y not 16-byte aligned   */
    CONV_ERR_ALIASING = -5,        /* y overlaps x, w or bias               */
    CONV_ERR_CUDA = -6,            /* a CUDA runtime/driver call failed     */
    CONV_ERR_DEVICE_TIMEOUT = -7,  /* a kernel gave up waiting on a barrier */
    CONV_ERR_OOM = -8,             /* host or device allocation failed      */
    CONV_ERR_INVALID_ARG = -9,     /* bad enum value or quantisation params */
    CONV_ERR_SCRATCH_LIMIT = -10,  /* layer needs more than a fixed scratch area holds */
};

typedef struct conv_plan conv_plan_t; /* opaque */

/* Validates the layer and builds a plan for the current CUDA device.
 *   shape   : sizes (n >= 0; h, w, c_in, c_out, k_h, k_w >= 1)
 *   stride  : >= 1, both axes
 *   pad_h/w : >= 0, applied on both sides of the axis
 *   groups  : >= 1, dividing c_in and c_out
 *   quant   : required for CONV_I8, must be NULL otherwise
 * CONV_I8 with CONV_ACT_MISH is CONV_ERR_UNSUPPORTED (not bit-reproducible).
 * On success *out_plan receives the plan; on failure it is set to NULL. */
CONV_API int conv_plan_create(const conv_shape_t *shape, int stride, int pad_h, int pad_w,
                     int groups, conv_dtype_t dtype, conv_act_t act,
                     const conv_quant_t *quant, conv_plan_t **out_plan);

/* As conv_plan_create, forcing a kernel family (CONV_ALGO_AUTO = choose). */
CONV_API int conv_plan_create_ex(const conv_shape_t *shape, int stride, int pad_h, int pad_w,
                        int groups, conv_dtype_t dtype, conv_act_t act,
                        const conv_quant_t *quant, conv_algo_t algo,
                        conv_plan_t **out_plan);

/* ---------------------------------------------------------------------------
 * Output placement and residual fusion.
 *
 * Two fused-epilogue options from the "YOLOv4, optimized for Wormhole" page,
 * section 9 (custom Tensix kernels):
 *   - K2, Mish + residual add: the layer adds a skip tensor after its
 *     activation and writes the result once:
 *       y = act(acc + b[co]) + r[n,oh,ow,co]      (then rounded to y's type)
 *   - K4, upsample + concat: the layer writes straight into a channel slice
 *     of the next layer's concatenated NHWC buffer, optionally repeating
 *     every output pixel over the 2x2 block a 2x nearest-neighbour upsample
 *     would give it:
 *       y[n, u*oh+dy, u*ow+dx, y_channel_offset + co] = value(n, oh, ow, co)
 *       for dy, dx in [0, u),  u = upsample.
 * y is then a [N][u*OH][u*OW][y_channels] buffer, of which the layer writes
 * channels [y_channel_offset, y_channel_offset + c_out) and nothing else.
 *
 *   y_channels       channels per pixel of y; 0 means c_out
 *   y_channel_offset first channel of the layer's slice (>= 0,
 *                    y_channel_offset + c_out <= y_channels)
 *   upsample         1 or 2
 *   residual         0, or 1: conv_run_fused takes r, a dense
 *                    [N][OH][OW][c_out] tensor of the layer's dtype
 *                    (CONV_F32 or CONV_BF16; int8 layers return
 *                    CONV_ERR_UNSUPPORTED)
 * y_channels * esize and y_channel_offset * esize must be multiples of 16
 * bytes (CONV_ERR_MISALIGNED).  Other values: CONV_ERR_INVALID_ARG.
 * Depthwise layers with any of these options run on the direct kernel. */
typedef struct {
    int32_t y_channels;
    int32_t y_channel_offset;
    int32_t upsample;
    int32_t residual;
} conv_output_t;

/* As conv_plan_create_ex with output options (`out` NULL: the plain layer,
 * identical to conv_plan_create_ex). */
CONV_API int conv_plan_create_fused(const conv_shape_t *shape, int stride, int pad_h, int pad_w,
                                    int groups, conv_dtype_t dtype, conv_act_t act,
                                    const conv_quant_t *quant, const conv_output_t *out,
                                    conv_algo_t algo, conv_plan_t **out_plan);

/* As conv_run, with the residual r (a device pointer, 16-byte aligned, not
 * overlapping y; required if and only if the plan was created with
 * residual = 1, else CONV_ERR_NULL_ARG / CONV_ERR_INVALID_ARG).  y is the
 * [N][u*OH][u*OW][y_channels] buffer of the plan's output options and must
 * not overlap x, w, bias or r. */
CONV_API int conv_run_fused(const conv_plan_t *plan, const void *x, const void *w, const void *bias,
                            const void *residual, void *y, void *stream);

/* ---------------------------------------------------------------------------
 * SPP block ("YOLOv4, optimized for Wormhole", section 9, K3): the max pools
 * of x over 5x5, 9x9 and 13x13 windows, stride 1, output the size of x,
 * positions outside the image never winning the max:
 *   mpK[n,h,w,c] = max { x[n,i,j,c] : |i-h| <= K/2, |j-w| <= K/2, in the image }
 * each written to its own channel slice of y, a [N][H][W][y_channels]
 * buffer (the next layer's concatenated layout):
 *   y[n,h,w,off5+c] = mp5, y[n,h,w,off9+c] = mp9, y[n,h,w,off13+c] = mp13,
 *   and, when off_x >= 0, y[n,h,w,off_x+c] = x[n,h,w,c].
 * x [N][H][W][C] and y are device pointers of dtype (F32, BF16 or I8), 16-byte
 * aligned, not overlapping.  C * esize, y_channels * esize and every offset *
 * esize must be multiples of 16 bytes (CONV_ERR_MISALIGNED); the slices must
 * lie inside y and not overlap one another (CONV_ERR_INVALID_ARG).  Results
 * are exact (bit-identical to a direct evaluation of each window).
 * Asynchronous on `stream`; allocates nothing. */
CONV_API int conv_spp_run(int32_t n, int32_t h, int32_t w, int32_t c, conv_dtype_t dtype, const void *x,
                          void *y, int32_t y_channels, int32_t off5, int32_t off9, int32_t off13,
                          int32_t off_x, void *stream);

/* ---------------------------------------------------------------------------
 * Fused depthwise-separable pair (the DS-CNN block): a depthwise 3x3
 * convolution, its bias and activation, then a 1x1 pointwise convolution,
 * its bias and activation, in one kernel with the intermediate kept in
 * shared memory ("nanoinfer", "What is still slow": depthwise convolution is
 * the gap and each layer boundary is a trip through memory):
 *   z[n,oh,ow,c]  = round( act_dw( b_dw[c] + sum_{r,s<3}
 *                         x[n, oh*stride-pad+r, ow*stride-pad+s, c] * w_dw[c,r,s,0] ) )
 *   y[n,oh,ow,co] = act_pw( b_pw[co] + sum_{c} z[n,oh,ow,c] * w_pw[co,0,0,c] )
 * where round() rounds z to the layer's type (nearest-even bf16; nothing for
 * fp32), so the pair computes what the two layers run one after the other
 * compute.  shape: n, h, w of x, c_in = channels of x and z (<= 512, a
 * multiple of 4), c_out = channels of y; k_h and k_w must be 3.  dtype F32
 * or BF16 (fp32 arithmetic; I8 is CONV_ERR_UNSUPPORTED).  pad applies to both
 * axes.  Layouts: x NHWC, w_dw [c_in][3][3][1], w_pw [c_out][1][1][c_in],
 * b_dw [c_in] and b_pw [c_out] fp32 or NULL, y NHWC [N][OH][OW][c_out].
 * The plan runs only through conv_run_dwpw (conv_run: CONV_ERR_INVALID_ARG). */
CONV_API int conv_plan_create_dwpw(const conv_shape_t *shape, int stride, int pad, conv_dtype_t dtype,
                                   conv_act_t act_dw, conv_act_t act_pw, conv_plan_t **out_plan);
CONV_API int conv_run_dwpw(const conv_plan_t *plan, const void *x, const void *w_dw, const void *b_dw,
                           const void *w_pw, const void *b_pw, void *y, void *stream);

/* Enqueues the layer on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  x, w, y are device pointers, bias a device pointer or NULL; all
 * 16-byte aligned.  y must not overlap x, w or bias.  Asynchronous: errors
 * of the kernel itself surface through conv_plan_check_device_status. */
CONV_API int conv_run(const conv_plan_t *plan, const void *x, const void *w, const void *bias,
             void *y, void *stream);
/* (conv_run on a plan with output options is conv_run_fused without a
 * residual.) */

/* Frees the plan and its device buffers.  NULL-safe.  The caller must make
 * sure no conv_run of this plan is still executing on the GPU. */
CONV_API void conv_plan_destroy(conv_plan_t *plan);

/* Output height and width of the plan's layer. */
CONV_API int conv_plan_output_shape(const conv_plan_t *plan, int *oh, int *ow);

/* The kernel family (conv_algo_t) the plan runs, or a negative error. */
CONV_API int conv_plan_algo(const conv_plan_t *plan);

/* Number of kernels conv_run enqueues for this plan (the tensor-core path of
 * int8 and small-Cin layers adds its widening pre-pass), or a negative error. */
CONV_API int conv_plan_launches(const conv_plan_t *plan);

/* A short human-readable description of the kernel and tiling chosen. */
CONV_API const char *conv_plan_describe(const conv_plan_t *plan);

/* Synchronises `stream`, reads and clears the plan's device status word.
 * Returns CONV_OK, or CONV_ERR_DEVICE_TIMEOUT if a kernel of this plan gave
 * up on a barrier wait since the last check, or CONV_ERR_CUDA. */
CONV_API int conv_plan_check_device_status(conv_plan_t *plan, void *stream);

/* The name of a status code ("CONV_OK", "CONV_ERR_MISALIGNED", ...). */
CONV_API const char *conv_status_str(int status);

/* CONV_NHWC_ABI_VERSION of the library. */
CONV_API int conv_abi_version(void);

/* ---------------------------------------------------------------------------
 * An int8 layer run that allocates nothing.  (The pages describe no such
 * entry point; it exists for callers of this library, not for the method.)
 *
 * Who needs it: code that may not call cudaMalloc at run time -- an engine
 * that reserves all device memory up front in its own arena, a process
 * working under a fixed memory budget, or a caller holding a lock in which an
 * allocation could block or fail.  conv_plan_create allocates the int8
 * requantisation table on the device; this entry point does not.
 *
 * What it computes: exactly what conv_plan_create(..., CONV_I8, act, quant)
 * followed by conv_run computes (same validation, same bit-exact results),
 * on the CUDA-core direct kernel.  x, w, bias, y and `stream` are as for
 * conv_run.  quant->w_scales is a HOST array of shape->c_out floats.
 *
 * Scratch: the per-channel multipliers M[co] are written into one fixed
 * device array inside the library, CONV_NOALLOC_MAX_COUT floats (16 KiB),
 * which every GPU that loads the library holds until the process exits.
 * Layers with c_out > CONV_NOALLOC_MAX_COUT return CONV_ERR_SCRATCH_LIMIT.
 * Every call rewrites the whole part of the array it uses, before its kernel
 * reads it, in stream order.  All calls share that one array, so two calls
 * that can overlap on the GPU (different streams, or different host
 * threads) race and may read each other's multipliers: serialise them.
 *
 * Set-up: the first call on a device looks up the array's device address on
 * that device (cudaGetSymbolAddress, with that device current) and caches it;
 * make that first call before any stream capture begins.
 *
 * Returns CONV_OK or a CONV_ERR_* code, like conv_plan_create and conv_run
 * together.  Asynchronous: returns once the work is enqueued. */
#define CONV_NOALLOC_MAX_COUT 4096
CONV_API int conv_run_i8_noalloc(const conv_shape_t *shape, int stride, int pad_h, int pad_w,
                                 int groups, conv_act_t act, const conv_quant_t *quant,
                                 const void *x, const void *w, const void *bias, void *y,
                                 void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CONV_NHWC_H */
