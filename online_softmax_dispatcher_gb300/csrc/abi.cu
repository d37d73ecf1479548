// abi.cu -- the extern "C" entry points of libosd_softmax.so (declared and
// documented in include/softmax.h): argument checks, the per-device attribute
// cache, the dispatcher call and the single kernel launch.  No allocation, no
// host<->device copy and no synchronisation on the launch path.
#include <cuda_runtime.h>

#include <functional>
#include <mutex>

#include "launch.h"
#include "softmax.h"
#include "tma.cuh"

#define OSD_API extern "C" __attribute__((visibility("default")))

namespace osd {

// Device-side error word: kernels with bounded waits OR a code in here when a
// wait gives up.  Its device address is looked up once per device and passed
// to the kernels (separate translation units cannot name it directly).
__device__ unsigned int g_device_error;

// Self-test of the bounded-wait machinery: one thread waits on an mbarrier
// that nothing arrives on, gives up after `limit_ns`, records kErrFullWait in
// the error word and returns (the same path a kernel takes when a bulk copy
// never lands).
__global__ void k_selftest_wait(unsigned *err, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, &abort_flag, true, limit_ns))
        atomicOr(err, kErrFullWait);
}

namespace {

thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;

struct DeviceCache {
    InitOnSuccess init;
    softmax_device_info info = {};
    unsigned int *error_word = nullptr;
};

DeviceCache g_devices[kMaxDevices];

int cuda_fail(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    return SOFTMAX_ERR_CUDA;
}

// Fills c for device dev (current); SOFTMAX_OK or the failing call's status.
int init_device(DeviceCache &c, int dev)
{
    int v = 0;
    cudaError_t e;
#define OSD_ATTR(field, attr)                                 \
    e = cudaDeviceGetAttribute(&v, attr, dev);                \
    if (e != cudaSuccess)                                     \
        return cuda_fail(e);                                  \
    c.info.field = v;
    OSD_ATTR(sm_count, cudaDevAttrMultiProcessorCount)
    OSD_ATTR(max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin)
    OSD_ATTR(cluster_launch, cudaDevAttrClusterLaunch)
    OSD_ATTR(l2_bytes, cudaDevAttrL2CacheSize)
    OSD_ATTR(cc_major, cudaDevAttrComputeCapabilityMajor)
    OSD_ATTR(cc_minor, cudaDevAttrComputeCapabilityMinor)
#undef OSD_ATTR
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess)
        return cuda_fail(e);
    c.error_word = static_cast<unsigned int *>(p);
    return SOFTMAX_OK;
}

int current_device(DeviceCache **out)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices)
        return SOFTMAX_ERR_INVALID_ARG;
    DeviceCache &c = g_devices[dev];
    const int rc = c.init.run([&] { return init_device(c, dev); });  // device dev is current here
    if (rc != SOFTMAX_OK)
        return rc;
    *out = &c;
    return SOFTMAX_OK;
}

int launch(const DeviceCache &dc, const void *x, void *y, int64_t rows, int64_t cols, int dtype,
           const softmax_launch_plan &plan, softmax_stream_t stream, void *workspace = nullptr,
           uint64_t workspace_bytes = 0)
{
    // every plan, the dispatcher's own included, is checked before it runs
    const int rc = validate_plan(dc.info, x, y, rows, cols, dtype, plan);
    if (rc != SOFTMAX_OK)
        return rc;
    Launch l{x, y, rows, cols, dtype, plan, stream, dc.error_word};
    int e;
    if (plan.variant == SOFTMAX_VARIANT_SPLITK_GRID && grid_capturing(stream)) {
        // the grid split's scratch slots are ordered by CUDA events, which a
        // graph capture cannot take: capture the cluster split (or the stream
        // kernel) instead
        softmax_launch_plan alt;
        if (softmax_plan(&dc.info, x, y, rows, cols, dtype, SOFTMAX_VARIANT_SPLITK, &alt) != SOFTMAX_OK &&
            softmax_plan(&dc.info, x, y, rows, cols, dtype, SOFTMAX_VARIANT_STREAM, &alt) != SOFTMAX_OK)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        return launch(dc, x, y, rows, cols, dtype, alt, stream);
    }
    switch (plan.variant) {
    case SOFTMAX_VARIANT_SPLITK_GRID:
        e = launch_grid(l);
        break;
    case SOFTMAX_VARIANT_SPLITK_WIDE:
        // needs the workspace only softmax_fwd_ws supplies
        if (!workspace || workspace_bytes < wide_workspace_bytes(plan))
            return SOFTMAX_ERR_INVALID_ARG;
        e = launch_wide(l, workspace);
        break;
    case SOFTMAX_VARIANT_ROWGROUP:
        e = launch_rowgroup(l);
        break;
    case SOFTMAX_VARIANT_BLOCK:
        e = launch_block(l);
        break;
    case SOFTMAX_VARIANT_BLOCK_TMA:
        e = launch_block_tma(l);
        break;
    case SOFTMAX_VARIANT_STREAM:
        e = launch_stream(l);
        break;
    case SOFTMAX_VARIANT_SPLITK:
        e = launch_splitk(l);
        break;
    default:
        return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
    }
    if (e != 0)
        return cuda_fail((cudaError_t)e);
    return SOFTMAX_OK;
}

}  // namespace

int record_cuda_error(int cuda_error) { return cuda_fail((cudaError_t)cuda_error); }

}  // namespace osd

using namespace osd;

OSD_API int softmax_fwd_variant(const void *x, void *y, int64_t rows, int64_t cols, int dtype, int variant,
                                softmax_stream_t stream)
{
    int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    softmax_launch_plan plan;
    rc = softmax_plan(&dc->info, x, y, rows, cols, dtype, variant, &plan);
    if (rc != SOFTMAX_OK)
        return rc;
    return launch(*dc, x, y, rows, cols, dtype, plan, stream);
}

OSD_API int softmax_fwd_masked_variant(const void *x, void *y, int64_t rows, int64_t cols, int dtype, float scale,
                                      const void *mask, int64_t mask_rows, int64_t causal_q, int variant,
                                      softmax_stream_t stream)
{
    int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (causal_q < 0 || variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    if (mask) {
        const int64_t S = dtype_bytes(dtype);
        if (mask_rows < 1 || reinterpret_cast<uintptr_t>(mask) % S || cols > INT64_MAX / S ||
            mask_rows > INT64_MAX / (cols * S > 0 ? cols * S : 1))
            return SOFTMAX_ERR_INVALID_ARG;
        const uint64_t mbytes = (uint64_t)(mask_rows * cols * S), ybytes = (uint64_t)(rows * cols * S);
        const uintptr_t ma = reinterpret_cast<uintptr_t>(mask), ya = reinterpret_cast<uintptr_t>(y);
        if (ma < ya + ybytes && ya < ma + mbytes)
            return SOFTMAX_ERR_ALIAS;
    }
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    MaskedLaunch l{x, y, rows, cols, dtype, {}, stream, scale, mask, mask_rows, causal_q};
    rc = plan_masked(dc->info, x, y, rows, cols, dtype, variant, &l.plan);
    if (rc != SOFTMAX_OK)
        return rc;
    const int e = launch_masked(l);
    return e == 0 ? SOFTMAX_OK : cuda_fail((cudaError_t)e);
}

OSD_API int softmax_fwd_masked(const void *x, void *y, int64_t rows, int64_t cols, int dtype, float scale,
                               const void *mask, int64_t mask_rows, int64_t causal_q, softmax_stream_t stream)
{
    return softmax_fwd_masked_variant(x, y, rows, cols, dtype, scale, mask, mask_rows, causal_q,
                                      SOFTMAX_VARIANT_AUTO, stream);
}

OSD_API int norm_fwd_variant(int kind, const void *x, void *y, int64_t rows, int64_t cols, int dtype,
                             const void *gamma, const void *beta, float eps, float *mean, float *rstd, int variant,
                             softmax_stream_t stream)
{
    int rc = validate_norm_args(kind, x, y, rows, cols, dtype, gamma, beta, eps, mean, rstd);
    if (rc != SOFTMAX_OK)
        return rc;
    if (variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    NormLaunch l{x, y, rows, cols, dtype, {}, stream, kind, 0, gamma, kind == kNormLayer ? beta : nullptr, eps,
                 kind == kNormLayer ? mean : nullptr, rstd};
    rc = plan_norm(dc->info, kind, x, y, rows, cols, dtype, gamma, l.beta, variant, &l.plan, &l.mode);
    if (rc != SOFTMAX_OK)
        return rc;
    const int e = launch_norm(l);
    return e == 0 ? SOFTMAX_OK : cuda_fail((cudaError_t)e);
}

OSD_API int layernorm_fwd(const void *x, void *y, int64_t rows, int64_t cols, int dtype, const void *gamma,
                          const void *beta, float eps, float *mean, float *rstd, softmax_stream_t stream)
{
    return norm_fwd_variant(kNormLayer, x, y, rows, cols, dtype, gamma, beta, eps, mean, rstd,
                            SOFTMAX_VARIANT_AUTO, stream);
}

OSD_API int rmsnorm_fwd(const void *x, void *y, int64_t rows, int64_t cols, int dtype, const void *gamma,
                        float eps, float *rstd, softmax_stream_t stream)
{
    return norm_fwd_variant(kNormRms, x, y, rows, cols, dtype, gamma, nullptr, eps, nullptr, rstd,
                            SOFTMAX_VARIANT_AUTO, stream);
}

OSD_API int softmax_bwd_variant(const void *y, const void *dy, void *dx, int64_t rows, int64_t cols, int dtype,
                                int variant, softmax_stream_t stream)
{
    int rc = validate_bwd_args(y, dy, dx, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    BwdLaunch l{y, dy, dx, rows, cols, dtype, {}, stream, 0, 0};
    rc = plan_bwd(dc->info, y, dy, dx, rows, cols, dtype, variant, &l.plan, &l.dy_vec, &l.dx_vec);
    if (rc != SOFTMAX_OK)
        return rc;
    const int e = launch_bwd(l);
    return e == 0 ? SOFTMAX_OK : cuda_fail((cudaError_t)e);
}

OSD_API int softmax_bwd(const void *y, const void *dy, void *dx, int64_t rows, int64_t cols, int dtype,
                        softmax_stream_t stream)
{
    return softmax_bwd_variant(y, dy, dx, rows, cols, dtype, SOFTMAX_VARIANT_AUTO, stream);
}

OSD_API int softmax_fwd(const void *x, void *y, int64_t rows, int64_t cols, int dtype, softmax_stream_t stream)
{
    return softmax_fwd_variant(x, y, rows, cols, dtype, SOFTMAX_VARIANT_AUTO, stream);
}

OSD_API int softmax_fwd_plan(const void *x, void *y, int64_t rows, int64_t cols, int dtype,
                             const softmax_launch_plan *plan, softmax_stream_t stream)
{
    int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (!plan)
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    return launch(*dc, x, y, rows, cols, dtype, *plan, stream);
}

namespace {

// The plan softmax_fwd_ws launches: the dispatcher's choice, with the two-launch
// SPLITK_WIDE (partials in the caller's workspace) in place of the cluster or
// grid split of few, very long rows (fewer rows than SMs; many long rows keep
// the cluster split's one CTA per row, which needs no workspace).
int plan_ws(const DeviceCache &dc, const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
            softmax_launch_plan *plan)
{
    int rc = softmax_plan(&dc.info, x, y, rows, cols, dtype, SOFTMAX_VARIANT_AUTO, plan);
    if (rc != SOFTMAX_OK)
        return rc;
    if ((plan->variant == SOFTMAX_VARIANT_SPLITK && rows < dc.info.sm_count) ||
        plan->variant == SOFTMAX_VARIANT_SPLITK_GRID) {
        softmax_launch_plan wide;
        if (softmax_plan(&dc.info, x, y, rows, cols, dtype, SOFTMAX_VARIANT_SPLITK_WIDE, &wide) == SOFTMAX_OK)
            *plan = wide;
    }
    return SOFTMAX_OK;
}

bool ranges_overlap(const void *a, uint64_t na, const void *b, uint64_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace

OSD_API int softmax_workspace_size(const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
                                   uint64_t *bytes)
{
    if (!bytes)
        return SOFTMAX_ERR_INVALID_ARG;
    int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    *bytes = 0;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    softmax_launch_plan plan;
    rc = plan_ws(*dc, x, y, rows, cols, dtype, &plan);
    if (rc != SOFTMAX_OK)
        return rc;
    *bytes = wide_workspace_bytes(plan);
    return SOFTMAX_OK;
}

OSD_API int softmax_fwd_ws(const void *x, void *y, int64_t rows, int64_t cols, int dtype, void *workspace,
                           uint64_t workspace_bytes, softmax_stream_t stream)
{
    int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if ((!workspace && workspace_bytes) || reinterpret_cast<uintptr_t>(workspace) % 16)
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    const uint64_t nbytes = (uint64_t)(rows * cols * dtype_bytes(dtype));
    if (workspace && workspace_bytes &&
        (ranges_overlap(workspace, workspace_bytes, x, nbytes) || ranges_overlap(workspace, workspace_bytes, y, nbytes)))
        return SOFTMAX_ERR_ALIAS;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    softmax_launch_plan plan;
    rc = plan_ws(*dc, x, y, rows, cols, dtype, &plan);
    if (rc != SOFTMAX_OK)
        return rc;
    if (plan.variant == SOFTMAX_VARIANT_SPLITK_WIDE && (!workspace || workspace_bytes < wide_workspace_bytes(plan))) {
        rc = softmax_plan(&dc->info, x, y, rows, cols, dtype, SOFTMAX_VARIANT_AUTO, &plan);
        if (rc != SOFTMAX_OK)
            return rc;
    }
    return launch(*dc, x, y, rows, cols, dtype, plan, stream, workspace, workspace_bytes);
}

OSD_API int softmax_query_variant(const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
                                  int *variant)
{
    if (!variant)
        return SOFTMAX_ERR_INVALID_ARG;
    int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    DeviceCache *dc = nullptr;
    rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    softmax_launch_plan plan;
    rc = softmax_plan(&dc->info, x, y, rows, cols, dtype, SOFTMAX_VARIANT_AUTO, &plan);
    if (rc != SOFTMAX_OK)
        return rc;
    *variant = plan.variant;
    return SOFTMAX_OK;
}

OSD_API int softmax_device_query(softmax_device_info *dev)
{
    if (!dev)
        return SOFTMAX_ERR_INVALID_ARG;
    DeviceCache *dc = nullptr;
    const int rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    *dev = dc->info;
    return SOFTMAX_OK;
}

OSD_API int softmax_get_device_error(softmax_stream_t stream, unsigned int *code)
{
    if (!code)
        return SOFTMAX_ERR_INVALID_ARG;
    DeviceCache *dc = nullptr;
    const int rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, dc->error_word, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(dc->error_word, 0, sizeof v, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e);
    *code = v;
    if (v) {
        // a wait gave up: the grid split's barrier counts may be left mid-way
        const int re = reset_grid_scratch();
        if (re != 0)
            return record_cuda_error(re);
    }
    return v ? SOFTMAX_ERR_DEVICE_TIMEOUT : SOFTMAX_OK;
}

OSD_API int softmax_selftest_bounded_wait(softmax_stream_t stream, unsigned int limit_us)
{
    if (limit_us == 0 || limit_us > 1000000)
        return SOFTMAX_ERR_INVALID_ARG;
    DeviceCache *dc = nullptr;
    const int rc = current_device(&dc);
    if (rc != SOFTMAX_OK)
        return rc;
    k_selftest_wait<<<1, 32, 0, (cudaStream_t)stream>>>(dc->error_word, (uint64_t)limit_us * 1000u);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SOFTMAX_OK : cuda_fail(e);
}

OSD_API int softmax_last_cuda_error(void) { return t_last_cuda_error; }

OSD_API const char *softmax_strerror(int status)
{
    switch (status) {
    case SOFTMAX_OK:
        return "ok";
    case SOFTMAX_ERR_INVALID_ARG:
        return "invalid argument";
    case SOFTMAX_ERR_UNSUPPORTED_DTYPE:
        return "unsupported dtype";
    case SOFTMAX_ERR_ALIAS:
        return "buffers overlap (other than exactly, in place)";
    case SOFTMAX_ERR_CUDA:
        return "CUDA runtime error (see softmax_last_cuda_error)";
    case SOFTMAX_ERR_UNSUPPORTED_SHAPE:
        return "variant cannot serve this shape on this device";
    case SOFTMAX_ERR_DEVICE_TIMEOUT:
        return "a bounded device-side wait gave up";
    default:
        return "unknown status";
    }
}

OSD_API const char *softmax_variant_name(int variant)
{
    switch (variant) {
    case SOFTMAX_VARIANT_AUTO:
        return "auto";
    case SOFTMAX_VARIANT_ROWGROUP:
        return "rowgroup";
    case SOFTMAX_VARIANT_BLOCK:
        return "block";
    case SOFTMAX_VARIANT_BLOCK_TMA:
        return "block_tma";
    case SOFTMAX_VARIANT_STREAM:
        return "stream";
    case SOFTMAX_VARIANT_SPLITK:
        return "splitk";
    case SOFTMAX_VARIANT_SPLITK_WIDE:
        return "splitk_wide";
    case SOFTMAX_VARIANT_SPLITK_GRID:
        return "splitk_grid";
    default:
        return "unknown";
    }
}

OSD_API int softmax_abi_version(void) { return 1; }
