// conv_run_i8_noalloc: an int8 layer run that performs no device allocation.
//
// The int8 kernels read the per-output-channel requantisation multipliers
// M[co] from device memory.  A plan allocates that table with cudaMalloc at
// creation; some callers cannot allocate at run time (an engine that carves
// every buffer out of its own pre-reserved arena, a process held to a fixed
// device-memory budget, code running where an allocation could block or
// fail).  This entry point keeps the table in one fixed array compiled into
// the library instead, so a call needs nothing but the caller's buffers.
//
// The array, its per-device set-up and the entry point live in this file.
// Host code never uses the array's name as an address (on the host it only
// stands for the symbol): the set-up asks the runtime for the array's device
// address on each device, with that device current, and passes that address
// to the kernel.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "conv_internal.h"

// Requantisation multipliers of the running call.  Every call writes entries
// [0, c_out) before its kernel reads them (stream order); no entry needs to
// start at zero.  All calls share it: calls that may overlap on the GPU race.
static __device__ __align__(256) float g_noalloc_mult[CONV_NOALLOC_MAX_COUT];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kChunk = 1000;  // multipliers per fill launch (kernel parameters stay < 4 KB)

struct MultChunk {
    float m[kChunk];
};

std::mutex g_setup_mu;
float *g_scratch[kMaxDevices];  // device address of g_noalloc_mult per device, or nullptr

// Writes n multipliers (passed by value in the kernel parameters) into the
// fixed array at offset off.
__global__ void fill_multipliers(MultChunk c, int off, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) g_noalloc_mult[off + i] = c.m[i];
}

// Once per device, with `dev` current: check the architecture and look up
// the device address of the fixed array.
int scratch_for_device(int dev, float **out) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch[dev]) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return CONV_ERR_CUDA;
        if (major != 10 || minor != 3) return CONV_ERR_UNSUPPORTED;
        void *addr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_mult);
        if (e != cudaSuccess || addr == nullptr) return CONV_ERR_CUDA;
        g_scratch[dev] = static_cast<float *>(addr);
    }
    *out = g_scratch[dev];
    return CONV_OK;
}

}  // namespace

extern "C" int conv_run_i8_noalloc(const conv_shape_t *shape, int stride, int pad_h, int pad_w, int groups,
                                   conv_act_t act, const conv_quant_t *quant, const void *x, const void *w,
                                   const void *bias, void *y, void *stream) {
    if (!shape) return CONV_ERR_NULL_ARG;
    int oh = 0, ow = 0;
    int rc = conv_validate_layer(shape, stride, pad_h, pad_w, groups, CONV_I8, act, quant, &oh, &ow);
    if (rc != CONV_OK) return rc;
    if (shape->c_out > CONV_NOALLOC_MAX_COUT) return CONV_ERR_SCRATCH_LIMIT;

    // A plan description on the stack, for the existing direct-kernel launcher.
    conv_plan p{};
    p.s = *shape;
    p.stride = stride; p.pad_h = pad_h; p.pad_w = pad_w; p.groups = groups;
    p.dtype = CONV_I8; p.act = act; p.oh = oh; p.ow = ow;
    p.y_c = shape->c_out; p.y_coff = 0; p.up = 1; p.has_res = 0;  // the plain layer output
    p.algo = CONV_ALGO_DIRECT;
    if (!direct_supported(&p)) return CONV_ERR_UNSUPPORTED;
    if (shape->n == 0) return CONV_OK;
    rc = conv_check_run_pointers(CONV_I8, shape, groups, oh, ow, x, w, bias, y);
    if (rc != CONV_OK) return rc;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CONV_ERR_UNSUPPORTED;
    float *scratch = nullptr;
    rc = scratch_for_device(dev, &scratch);
    if (rc != CONV_OK) return rc;
    p.device = dev;
    p.d_mult = scratch;

    // M[co] = s_x * s_w[co] / s_y in double, rounded once to float (the same
    // table conv_plan_create builds), copied in by value through kernel
    // parameters: no host staging buffer, no allocation.
    cudaStream_t st = (cudaStream_t)stream;
    MultChunk chunk;
    for (int off = 0; off < shape->c_out; off += kChunk) {
        const int n = shape->c_out - off < kChunk ? shape->c_out - off : kChunk;
        for (int i = 0; i < n; ++i)
            chunk.m[i] = (float)((double)quant->in_scale * (double)quant->w_scales[off + i] /
                                 (double)quant->out_scale);
        // The launch's own status (not cudaGetLastError, which would also
        // return, and clear, an earlier error of unrelated caller work).
        int o = off, cnt = n;
        void *args[] = {&chunk, &o, &cnt};
        if (cudaLaunchKernel((const void *)fill_multipliers, dim3((n + 255) / 256), dim3(256), args, 0, st) !=
            cudaSuccess)
            return CONV_ERR_CUDA;
    }
    return launch_direct(&p, x, w, bias, nullptr, y, st) == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}
