// noalloc.cu -- softmax_fwd_noalloc: the wide split of k_wide.cu (two
// launches, partial statistics in scratch memory) with its scratch in a fixed
// array that the library owns, so the caller allocates nothing.
//
// Some callers cannot allocate device memory themselves: a plugin run by a
// host engine that owns every device allocation and hands it only inputs and
// outputs, or a latency-critical path where cudaMalloc -- which may
// synchronise the device -- is not allowed.  softmax_fwd_ws needs them to pass
// a workspace; this entry point takes its scratch from g_noalloc_scratch
// instead and calls no allocating routine (no cudaMalloc / cudaFree, no torch).
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its 64 KiB until the process exits.  In host code its name is
// only a host-side stand-in, not a device address; the device address is
// looked up with cudaGetSymbolAddress, with that device current, by the first
// call made on that device, and then passed to the kernels.  Only a lookup
// that succeeded is remembered: if it fails (for instance in a first call made
// while the stream is being captured), the call returns the CUDA error and the
// next call on that device tries again.
#include <cuda_runtime.h>

#include "launch.h"
#include "softmax.h"

#define OSD_API extern "C" __attribute__((visibility("default")))

namespace osd {

// 4096 partial-statistics slots of 16 bytes = 64 KiB: rows x P must fit, with
// P the CTAs per row the wide split uses (about 2 x SMs / rows, at least 1).
constexpr int64_t kNoAllocSlots = 4096;

static __device__ __align__(256) float4 g_noalloc_scratch[kNoAllocSlots];

namespace {

struct Scratch {
    InitOnSuccess init;
    float4 *ptr = nullptr;  // device address of g_noalloc_scratch on this device
};

Scratch g_scratch[64];

int lookup_scratch(Scratch &s)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
        return (int)e;
    s.ptr = static_cast<float4 *>(p);
    return 0;
}

}  // namespace
}  // namespace osd

using namespace osd;

OSD_API int softmax_fwd_noalloc(const void *x, void *y, int64_t rows, int64_t cols, int dtype,
                                softmax_stream_t stream)
{
    int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    softmax_device_info dev;
    rc = softmax_device_query(&dev);
    if (rc != SOFTMAX_OK)
        return rc;
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess)
        return record_cuda_error((int)e);
    if (d < 0 || d >= 64)
        return SOFTMAX_ERR_INVALID_ARG;
    Scratch &s = g_scratch[d];
    const int le0 = s.init.run([&] { return lookup_scratch(s); });  // device d is current here
    if (le0 != 0)
        return record_cuda_error(le0);
    softmax_launch_plan plan;
    rc = softmax_plan(&dev, x, y, rows, cols, dtype, SOFTMAX_VARIANT_SPLITK_WIDE, &plan);
    if (rc != SOFTMAX_OK)
        return rc;
    if (plan.grid_x * plan.grid_y > kNoAllocSlots)
        return SOFTMAX_ERR_UNSUPPORTED_SHAPE;  // more partials than the fixed array holds
    rc = validate_plan(dev, x, y, rows, cols, dtype, plan);
    if (rc != SOFTMAX_OK)
        return rc;
    Launch l{x, y, rows, cols, dtype, plan, stream, nullptr};
    const int le = launch_wide(l, s.ptr);
    return le == 0 ? SOFTMAX_OK : record_cuda_error(le);
}
