// C ABI of the fused NHWC convolution library (declared in conv_nhwc.h):
// argument validation, plan construction, kernel-family selection and the
// stream-ordered run entry point.
//
// Validation happens at plan creation, before any CUDA call, so that an
// invalid or unsupported layer is a named failure at preparation time
// ("nanoinfer", "Pooling read int8 tensors through a float*": unsupported
// op / dtype pairs become a named load failure instead of quiet garbage).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "conv_internal.h"

namespace {

// floor((in + 2 * pad - k) / stride) + 1, or -1 when no output fits.
long long out_dim(long long in, long long k, long long pad, long long stride) {
    const long long span = in + 2 * pad - k;
    if (span < 0) return -1;
    return span / stride + 1;
}

int validate(const conv_shape_t *s, int stride, int pad_h, int pad_w, int groups, conv_dtype_t dtype,
             conv_act_t act, const conv_quant_t *quant, int *oh, int *ow) {
    if (s->n < 0 || s->h < 1 || s->w < 1 || s->c_in < 1 || s->c_out < 1 || s->k_h < 1 || s->k_w < 1)
        return CONV_ERR_INVALID_SHAPE;
    if (stride < 1 || pad_h < 0 || pad_w < 0 || groups < 1) return CONV_ERR_INVALID_SHAPE;
    if (s->c_in % groups != 0 || s->c_out % groups != 0) return CONV_ERR_INVALID_SHAPE;
    if ((int)dtype < CONV_F32 || (int)dtype > CONV_I8) return CONV_ERR_INVALID_ARG;
    if ((int)act < CONV_ACT_NONE || (int)act > CONV_ACT_MISH) return CONV_ERR_INVALID_ARG;
    const long long OH = out_dim(s->h, s->k_h, pad_h, stride);
    const long long OW = out_dim(s->w, s->k_w, pad_w, stride);
    if (OH < 1 || OW < 1) return CONV_ERR_INVALID_SHAPE;
    // Size limits of the kernels' index arithmetic.
    const long long cpg = s->c_in / groups;
    const long long x_elems = (long long)s->n * s->h * s->w * s->c_in;
    const long long y_elems = (long long)s->n * OH * OW * s->c_out;
    const long long w_elems = (long long)s->c_out * s->k_h * s->k_w * cpg;
    const long long lim = 1ll << 40;
    if (x_elems >= lim || y_elems >= lim || w_elems >= lim) return CONV_ERR_UNSUPPORTED;
    if ((long long)s->n * OH * OW >= (1ll << 31) || (long long)s->n * s->h * s->w >= (1ll << 32))
        return CONV_ERR_UNSUPPORTED;
    if (dtype == CONV_I8) {
        if (!quant || !quant->w_scales) return CONV_ERR_NULL_ARG;
        if (!(quant->in_scale > 0.0f) || !(quant->out_scale > 0.0f) || !isfinite(quant->in_scale) ||
            !isfinite(quant->out_scale))
            return CONV_ERR_INVALID_ARG;
        for (int co = 0; co < s->c_out; ++co)
            if (!(quant->w_scales[co] > 0.0f) || !isfinite(quant->w_scales[co])) return CONV_ERR_INVALID_ARG;
        // An int8 MAC is < 2^14 in magnitude: the int32 accumulator of a
        // dot product of length K is exact while K * 2^14 < 2^31.
        if ((long long)s->k_h * s->k_w * cpg >= (1ll << 17)) return CONV_ERR_UNSUPPORTED;
        // Mish of a requantised value is not bit-reproducible across
        // implementations of expf; the int8 path offers NONE and RELU.
        if (act == CONV_ACT_MISH) return CONV_ERR_UNSUPPORTED;
    } else if (quant) {
        return CONV_ERR_INVALID_ARG;
    }
    *oh = (int)OH;
    *ow = (int)OW;
    return CONV_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

// Shared with the other entry points of the library (conv_internal.h).
int conv_validate_layer(const conv_shape_t *s, int stride, int pad_h, int pad_w, int groups,
                        conv_dtype_t dtype, conv_act_t act, const conv_quant_t *quant, int *oh, int *ow) {
    return validate(s, stride, pad_h, pad_w, groups, dtype, act, quant, oh, ow);
}

int conv_check_run_pointers(conv_dtype_t dtype, const conv_shape_t *s, int groups, int oh, int ow,
                            const void *x, const void *w, const void *bias, const void *y) {
    if (!x || !w || !y) return CONV_ERR_NULL_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias))) return CONV_ERR_MISALIGNED;
    const size_t es = (size_t)conv_esize(dtype);
    const size_t xb = (size_t)s->n * s->h * s->w * s->c_in * es;
    const size_t wb = (size_t)s->c_out * s->k_h * s->k_w * (s->c_in / groups) * es;
    const size_t bb = bias ? (size_t)s->c_out * 4 : 0;
    const size_t yb = (size_t)s->n * oh * ow * s->c_out * es;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) || overlaps(y, yb, bias, bb)) return CONV_ERR_ALIASING;
    return CONV_OK;
}

cudaError_t conv_launch(const void *kernel, dim3 grid, dim3 block, void **args, size_t smem, cudaStream_t st,
                        int cluster_x) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (cluster_x > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

int conv_grant_smem(const void *k, int device, int need) {
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, k) != cudaSuccess)
        return CONV_ERR_CUDA;
    const int avail = optin - (int)fa.sharedSizeBytes;
    if (need > avail) return CONV_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, avail) != cudaSuccess)
        return CONV_ERR_CUDA;
    return CONV_OK;
}

extern "C" {

int conv_abi_version(void) { return CONV_NHWC_ABI_VERSION; }

const char *conv_status_str(int status) {
    switch (status) {
    case CONV_OK: return "CONV_OK";
    case CONV_ERR_NULL_ARG: return "CONV_ERR_NULL_ARG";
    case CONV_ERR_INVALID_SHAPE: return "CONV_ERR_INVALID_SHAPE";
    case CONV_ERR_UNSUPPORTED: return "CONV_ERR_UNSUPPORTED";
    case CONV_ERR_MISALIGNED: return "CONV_ERR_MISALIGNED";
    case CONV_ERR_ALIASING: return "CONV_ERR_ALIASING";
    case CONV_ERR_CUDA: return "CONV_ERR_CUDA";
    case CONV_ERR_DEVICE_TIMEOUT: return "CONV_ERR_DEVICE_TIMEOUT";
    case CONV_ERR_OOM: return "CONV_ERR_OOM";
    case CONV_ERR_INVALID_ARG: return "CONV_ERR_INVALID_ARG";
    case CONV_ERR_SCRATCH_LIMIT: return "CONV_ERR_SCRATCH_LIMIT";
    default: return "CONV_ERR_UNKNOWN";
    }
}

int conv_plan_create_fused(const conv_shape_t *shape, int stride, int pad_h, int pad_w, int groups,
                           conv_dtype_t dtype, conv_act_t act, const conv_quant_t *quant,
                           const conv_output_t *out, conv_algo_t algo, conv_plan_t **out_plan) {
    if (!out_plan) return CONV_ERR_NULL_ARG;
    *out_plan = nullptr;
    if (!shape) return CONV_ERR_NULL_ARG;
    // staging and epilogue flags (tensor-core family only), then the family / layout
    const int stage_flags = (int)algo & (CONV_ALGO_STAGE_TAPS | CONV_ALGO_STAGE_HALO);
    const int epi_flags = (int)algo & (CONV_ALGO_EPI_SLICED | CONV_ALGO_EPI_PER_TILE);
    const int widen_flags = (int)algo & (CONV_ALGO_WIDEN_PREPASS | CONV_ALGO_WIDEN_INKERNEL);
    const int unknown_bits = (int)algo & ~(0xFF | CONV_ALGO_STAGE_TAPS | CONV_ALGO_STAGE_HALO | CONV_ALGO_EPI_SLICED |
                                           CONV_ALGO_EPI_PER_TILE | CONV_ALGO_WIDEN_PREPASS | CONV_ALGO_WIDEN_INKERNEL);
    algo = (conv_algo_t)((int)algo & 0xFF);
    if (unknown_bits || (int)algo < CONV_ALGO_AUTO ||
        ((int)algo > CONV_ALGO_IGEMM_PAIR && algo != CONV_ALGO_IGEMM_PAIR128))
        return CONV_ERR_INVALID_ARG;
    if (stage_flags == (CONV_ALGO_STAGE_TAPS | CONV_ALGO_STAGE_HALO) ||
        epi_flags == (CONV_ALGO_EPI_SLICED | CONV_ALGO_EPI_PER_TILE) ||
        widen_flags == (CONV_ALGO_WIDEN_PREPASS | CONV_ALGO_WIDEN_INKERNEL) ||
        ((stage_flags || epi_flags || widen_flags) && (algo < CONV_ALGO_IGEMM || algo == CONV_ALGO_DWPW)))
        return CONV_ERR_INVALID_ARG;
    int oh = 0, ow = 0;
    int rc = validate(shape, stride, pad_h, pad_w, groups, dtype, act, quant, &oh, &ow);
    if (rc != CONV_OK) return rc;
    // Output options (validated before any CUDA call, like the layer).
    conv_output_t o = {shape->c_out, 0, 1, 0};
    if (out) {
        o = *out;
        if (o.y_channels == 0) o.y_channels = shape->c_out;
        if (o.y_channel_offset < 0 || o.y_channels < 1 ||
            (long long)o.y_channel_offset + shape->c_out > (long long)o.y_channels ||
            (o.upsample != 1 && o.upsample != 2) || (o.residual != 0 && o.residual != 1))
            return CONV_ERR_INVALID_ARG;
        if (o.residual && dtype == CONV_I8) return CONV_ERR_UNSUPPORTED;
        const long long es = conv_esize(dtype);
        if ((o.y_channels * es) % 16 != 0 || (o.y_channel_offset * es) % 16 != 0) return CONV_ERR_MISALIGNED;
        if ((long long)shape->n * oh * ow * o.upsample * o.upsample * o.y_channels >= (1ll << 40))
            return CONV_ERR_UNSUPPORTED;
    }
    const bool fused = o.y_channels != shape->c_out || o.y_channel_offset != 0 || o.upsample != 1 || o.residual;

    conv_plan *p = new (std::nothrow) conv_plan();
    if (!p) return CONV_ERR_OOM;
    p->s = *shape;
    p->stride = stride; p->pad_h = pad_h; p->pad_w = pad_w; p->groups = groups;
    p->dtype = dtype; p->act = act; p->oh = oh; p->ow = ow;
    p->y_c = o.y_channels; p->y_coff = o.y_channel_offset; p->up = o.upsample; p->has_res = o.residual;

    // Device properties.  The kernels are built for sm_103a only.
    cudaDeviceProp prop;
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaGetDeviceProperties(&prop, p->device) != cudaSuccess) {
        delete p;
        return CONV_ERR_CUDA;
    }
    if (prop.major != 10 || prop.minor != 3) {
        delete p;
        return CONV_ERR_UNSUPPORTED;
    }
    p->num_sms = prop.multiProcessorCount;

    // Kernel family.
    // (the depthwise kernels have no output options: fused depthwise layers run on the direct kernel)
    const bool can_ig = igemm_supported(p), can_dw = !fused && dw3x3_supported(p),
               can_direct = direct_supported(p);
    int chosen = -1;
    if (algo == CONV_ALGO_AUTO)
        chosen = can_ig ? CONV_ALGO_IGEMM : (can_dw ? CONV_ALGO_DEPTHWISE : (can_direct ? CONV_ALGO_DIRECT : -1));
    else if (algo >= CONV_ALGO_IGEMM && can_ig) chosen = CONV_ALGO_IGEMM;
    else if (algo == CONV_ALGO_DEPTHWISE && can_dw) chosen = CONV_ALGO_DEPTHWISE;
    else if (algo == CONV_ALGO_DIRECT && can_direct) chosen = CONV_ALGO_DIRECT;
    if (chosen < 0) {
        delete p;
        return CONV_ERR_UNSUPPORTED;
    }
    p->algo = chosen;

    // Device-side state: status word and (int8) requantisation multipliers.
    if (cudaMalloc(&p->d_status, sizeof(int)) != cudaSuccess) {
        delete p;
        return CONV_ERR_OOM;
    }
    if (cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) {
        conv_plan_destroy(p);
        return CONV_ERR_CUDA;
    }
    if (dtype == CONV_I8) {
        float *hm = (float *)malloc(sizeof(float) * shape->c_out);
        if (!hm) { conv_plan_destroy(p); return CONV_ERR_OOM; }
        // M[co] = s_x * s_w[co] / s_y, formed in double and rounded once.
        for (int co = 0; co < shape->c_out; ++co)
            hm[co] = (float)((double)quant->in_scale * (double)quant->w_scales[co] / (double)quant->out_scale);
        if (cudaMalloc(&p->d_mult, sizeof(float) * shape->c_out) != cudaSuccess) {
            free(hm);
            conv_plan_destroy(p);
            return CONV_ERR_OOM;
        }
        const cudaError_t e = cudaMemcpy(p->d_mult, hm, sizeof(float) * shape->c_out, cudaMemcpyHostToDevice);
        free(hm);
        if (e != cudaSuccess) { conv_plan_destroy(p); return CONV_ERR_CUDA; }
    }

    if (chosen == CONV_ALGO_IGEMM) {
        // tile layout: 0 = estimated fastest, else swapped / N256 / N128 / N64 / pair / pair N128
        rc = igemm_configure(p,
                             algo == CONV_ALGO_IGEMM_PAIR128
                                 ? 6
                                 : (algo >= CONV_ALGO_IGEMM_SWAPPED ? (int)algo - CONV_ALGO_IGEMM_SWAPPED + 1 : 0),
                             stage_flags == CONV_ALGO_STAGE_TAPS ? 1 : (stage_flags == CONV_ALGO_STAGE_HALO ? 2 : 0),
                             epi_flags == CONV_ALGO_EPI_SLICED ? 1 : (epi_flags == CONV_ALGO_EPI_PER_TILE ? 2 : 0),
                             widen_flags == CONV_ALGO_WIDEN_PREPASS ? 1 : (widen_flags == CONV_ALGO_WIDEN_INKERNEL ? 2 : 0));
        if (rc != CONV_OK) { conv_plan_destroy(p); return rc; }
    } else if (chosen == CONV_ALGO_DEPTHWISE) {
        rc = dw3x3_configure(p);
        if (rc != CONV_OK) { conv_plan_destroy(p); return rc; }
        snprintf(p->desc, sizeof(p->desc), "dw3x3 %s%s tile=%dx%dx%dch halo=%dx%d threads=%d blocks=%lld",
                 dtype == CONV_F32 ? "f32" : (dtype == CONV_BF16 ? "bf16" : "i8"), p->dw.kind == 1 ? " rows" : "",
                 p->dw.th, p->dw.tw,
                 p->dw.cbv * (dtype == CONV_I8 ? 16 : 4), p->dw.hin, p->dw.win, p->dw.threads, p->dw.blocks);
    } else {
        direct_configure(p);
        if (p->dct > 0)
            snprintf(p->desc, sizeof(p->desc), "direct %s smem-weights co/thread=%d px/thread=%d",
                     dtype == CONV_F32 ? "f32-ffma" : "bf16-ffma", p->dct, p->dpt);
        else
            snprintf(p->desc, sizeof(p->desc), "direct %s",
                     dtype == CONV_F32 ? "f32-ffma" : (dtype == CONV_BF16 ? "bf16-ffma" : "i8-dp4a"));
    }
    *out_plan = p;
    return CONV_OK;
}

int conv_plan_create_dwpw(const conv_shape_t *shape, int stride, int pad, conv_dtype_t dtype, conv_act_t act_dw,
                          conv_act_t act_pw, conv_plan_t **out_plan) {
    if (!out_plan) return CONV_ERR_NULL_ARG;
    *out_plan = nullptr;
    if (!shape) return CONV_ERR_NULL_ARG;
    if ((int)act_pw < CONV_ACT_NONE || (int)act_pw > CONV_ACT_MISH) return CONV_ERR_INVALID_ARG;
    if (shape->k_h != 3 || shape->k_w != 3) return CONV_ERR_INVALID_SHAPE;
    if ((int)dtype == CONV_I8) return CONV_ERR_UNSUPPORTED;
    // the depthwise layer validates the input, stride, pad and dtype
    conv_shape_t dws = *shape;
    dws.c_out = shape->c_in;
    int oh = 0, ow = 0;
    int rc = validate(&dws, stride, pad, pad, shape->c_in, dtype, act_dw, nullptr, &oh, &ow);
    if (rc != CONV_OK) return rc;
    if (shape->c_out < 1) return CONV_ERR_INVALID_SHAPE;
    if (shape->c_in % 4 != 0) return CONV_ERR_UNSUPPORTED;
    if ((long long)shape->n * oh * ow * shape->c_out >= (1ll << 40)) return CONV_ERR_UNSUPPORTED;

    conv_plan *p = new (std::nothrow) conv_plan();
    if (!p) return CONV_ERR_OOM;
    p->s = *shape;
    p->stride = stride; p->pad_h = pad; p->pad_w = pad; p->groups = 1;
    p->dtype = dtype; p->act = act_dw; p->act2 = act_pw; p->oh = oh; p->ow = ow;
    p->y_c = shape->c_out; p->y_coff = 0; p->up = 1; p->has_res = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&p->device) != cudaSuccess || cudaGetDeviceProperties(&prop, p->device) != cudaSuccess) {
        delete p;
        return CONV_ERR_CUDA;
    }
    if (prop.major != 10 || prop.minor != 3) {
        delete p;
        return CONV_ERR_UNSUPPORTED;
    }
    p->num_sms = prop.multiProcessorCount;
    if (!dwpw_supported(p)) {
        delete p;
        return CONV_ERR_UNSUPPORTED;
    }
    p->algo = CONV_ALGO_DWPW;
    if (cudaMalloc(&p->d_status, sizeof(int)) != cudaSuccess) {
        delete p;
        return CONV_ERR_OOM;
    }
    if (cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) {
        conv_plan_destroy(p);
        return CONV_ERR_CUDA;
    }
    rc = dwpw_configure(p);
    if (rc != CONV_OK) {
        conv_plan_destroy(p);
        return rc;
    }
    snprintf(p->desc, sizeof(p->desc), "dw3x3+pw1x1 %s fused tile=%dx%d halo=%dx%d co/cta=%d ctas=%lld",
             dtype == CONV_F32 ? "f32" : "bf16", p->dwpw.th, p->dwpw.tw, p->dwpw.hin, p->dwpw.win,
             p->dwpw.cochunk, (long long)p->dwpw.tiles_w * p->dwpw.tiles_h * shape->n * p->dwpw.chunks);
    *out_plan = p;
    return CONV_OK;
}

int conv_run_dwpw(const conv_plan_t *plan, const void *x, const void *w_dw, const void *b_dw, const void *w_pw,
                  const void *b_pw, void *y, void *stream) {
    if (!plan) return CONV_ERR_NULL_ARG;
    const conv_plan *p = plan;
    if (p->algo != CONV_ALGO_DWPW) return CONV_ERR_INVALID_ARG;
    if (p->s.n == 0) return CONV_OK;
    if (!x || !w_dw || !w_pw || !y) return CONV_ERR_NULL_ARG;
    if (!aligned16(x) || !aligned16(w_dw) || !aligned16(w_pw) || !aligned16(y) || (b_dw && !aligned16(b_dw)) ||
        (b_pw && !aligned16(b_pw)))
        return CONV_ERR_MISALIGNED;
    const size_t es = (size_t)conv_esize(p->dtype);
    const size_t C = (size_t)p->s.c_in, Co = (size_t)p->s.c_out;
    const size_t xb = (size_t)p->s.n * p->s.h * p->s.w * C * es;
    const size_t yb = (size_t)p->s.n * p->oh * p->ow * Co * es;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w_dw, C * 9 * es) || overlaps(y, yb, w_pw, Co * C * es) ||
        overlaps(y, yb, b_dw, b_dw ? C * 4 : 0) || overlaps(y, yb, b_pw, b_pw ? Co * 4 : 0))
        return CONV_ERR_ALIASING;
    return launch_dwpw(p, x, w_dw, b_dw, w_pw, b_pw, y, (cudaStream_t)stream) == cudaSuccess ? CONV_OK
                                                                                             : CONV_ERR_CUDA;
}

int conv_plan_create_ex(const conv_shape_t *shape, int stride, int pad_h, int pad_w, int groups,
                        conv_dtype_t dtype, conv_act_t act, const conv_quant_t *quant, conv_algo_t algo,
                        conv_plan_t **out_plan) {
    return conv_plan_create_fused(shape, stride, pad_h, pad_w, groups, dtype, act, quant, nullptr, algo,
                                  out_plan);
}

int conv_plan_create(const conv_shape_t *shape, int stride, int pad_h, int pad_w, int groups,
                     conv_dtype_t dtype, conv_act_t act, const conv_quant_t *quant, conv_plan_t **out_plan) {
    return conv_plan_create_ex(shape, stride, pad_h, pad_w, groups, dtype, act, quant, CONV_ALGO_AUTO,
                               out_plan);
}

void conv_plan_destroy(conv_plan_t *plan) {
    if (!plan) return;
    if (plan->d_status) cudaFree(plan->d_status);
    if (plan->d_mult) cudaFree(plan->d_mult);
    if (plan->d_xprep) cudaFree(plan->d_xprep);
    if (plan->d_wprep) cudaFree(plan->d_wprep);
    delete plan;
}

int conv_plan_output_shape(const conv_plan_t *plan, int *oh, int *ow) {
    if (!plan || !oh || !ow) return CONV_ERR_NULL_ARG;
    *oh = plan->oh;
    *ow = plan->ow;
    return CONV_OK;
}

int conv_plan_algo(const conv_plan_t *plan) {
    if (!plan) return CONV_ERR_NULL_ARG;
    return plan->algo;
}

const char *conv_plan_describe(const conv_plan_t *plan) { return plan ? plan->desc : ""; }

int conv_plan_launches(const conv_plan_t *plan) {
    if (!plan) return CONV_ERR_NULL_ARG;
    if (plan->s.n == 0) return 0;
    return (plan->algo == CONV_ALGO_IGEMM && plan->ig.prep) ? 2 : 1;
}

int conv_run_fused(const conv_plan_t *plan, const void *x, const void *w, const void *bias, const void *residual,
                   void *y, void *stream) {
    if (!plan) return CONV_ERR_NULL_ARG;
    const conv_plan *p = plan;
    if (p->algo == CONV_ALGO_DWPW) return CONV_ERR_INVALID_ARG;  // runs through conv_run_dwpw
    if (p->has_res && !residual) return CONV_ERR_NULL_ARG;
    if (!p->has_res && residual) return CONV_ERR_INVALID_ARG;
    if (p->s.n == 0) return CONV_OK;  // empty batch: nothing to compute
    if (!x || !w || !y) return CONV_ERR_NULL_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
        (residual && !aligned16(residual)))
        return CONV_ERR_MISALIGNED;
    const size_t es = (size_t)conv_esize(p->dtype);
    const size_t xb = (size_t)p->s.n * p->s.h * p->s.w * p->s.c_in * es;
    const size_t wb = (size_t)p->s.c_out * p->s.k_h * p->s.k_w * (p->s.c_in / p->groups) * es;
    const size_t bb = bias ? (size_t)p->s.c_out * 4 : 0;
    const size_t rb = residual ? (size_t)p->s.n * p->oh * p->ow * p->s.c_out * es : 0;
    const size_t yb = (size_t)p->s.n * p->oh * p->up * p->ow * p->up * p->y_c * es;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) || overlaps(y, yb, bias, bb) ||
        overlaps(y, yb, residual, rb))
        return CONV_ERR_ALIASING;

    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    switch (p->algo) {
    case CONV_ALGO_IGEMM: return launch_igemm(p, x, w, bias, residual, y, st);
    case CONV_ALGO_DEPTHWISE: e = launch_dw3x3(p, x, w, bias, y, st); break;
    default: e = launch_direct(p, x, w, bias, residual, y, st); break;
    }
    return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

int conv_run(const conv_plan_t *plan, const void *x, const void *w, const void *bias, void *y, void *stream) {
    return conv_run_fused(plan, x, w, bias, nullptr, y, stream);
}

int conv_plan_check_device_status(conv_plan_t *plan, void *stream) {
    if (!plan) return CONV_ERR_NULL_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int h = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return CONV_ERR_CUDA;
    if (cudaMemcpy(&h, plan->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CONV_ERR_CUDA;
    if (h != 0) {
        if (cudaMemset(plan->d_status, 0, sizeof(int)) != cudaSuccess) return CONV_ERR_CUDA;
        return CONV_ERR_DEVICE_TIMEOUT;
    }
    return CONV_OK;
}

}  // extern "C"
