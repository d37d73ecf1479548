// launch.h -- host-side interface between the C ABI (abi.cu), the dispatcher
// (plan.cpp) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <stdint.h>

#include <atomic>
#include <mutex>

#include "softmax.h"

struct CUstream_st;

namespace osd {

// Chunk counts and limits the dispatcher and the kernels agree on.
constexpr int kRowgroupThreads = 256;   // largest CTA of the lanes-per-row kernel (the default)
constexpr int kRowgroupMaxFloats = 32;  // V * E cached per lane (registers)
constexpr int kBlockMaxChunks = 16;     // V of the block-per-row kernel
constexpr int kStreamThreads = 512;     // CTA size of the streaming kernel
constexpr int kStreamUnroll = 8;        // 16-byte loads in flight per thread per step
constexpr int kWideStep = 4;            // the same for the wide split: 64 registers at two 512-thread CTAs per SM
constexpr int kGridThreads = 512;       // SPLITK_GRID: CTA size (ring and streaming forms)
constexpr int kGridSlots = 16;          // SPLITK_GRID: scratch slots (launches in flight at once)
constexpr int kGridMaxRows = 128;       // SPLITK_GRID: rows a slot serves
constexpr int kGridMaxPartials = 4096;  // SPLITK_GRID: rows x CTAs per row a slot serves
constexpr int kGridMaxRing = 8;         // SPLITK_GRID ring form: shared-memory buffers
constexpr int kGridStaticSmem = 2048;   // SPLITK_GRID ring form: static shared memory, upper bound
constexpr int kGridPipeFold = 256;      // SPLITK_GRID pipelined form: threads of the fold team
constexpr int kGridPipeMaxCtas = 256;   // SPLITK_GRID pipelined form: CTAs whose partials one warp merges
constexpr int kMaxCluster = 16;         // non-portable cluster size limit
constexpr int kSplitStages = 6;         // SPLITK: shared-memory ring depth
constexpr int kSplitStageBytes = 32768; // SPLITK: bytes per stage (one bulk copy)
constexpr int kSplitConsumerWarps = 16; // SPLITK: consumer warps per CTA
constexpr int kSplitThreads = 32 * (1 + kSplitConsumerWarps);  // + one producer warp
constexpr int kTmaConsumerWarps = 16;   // BLOCK_TMA: consumer warps per CTA
constexpr int kTmaThreads = 32 * (1 + kTmaConsumerWarps);  // + one producer warp
constexpr int kTmaMaxStagesHost = 8;    // BLOCK_TMA ring depth limit
constexpr int kTmaStaticSmem = 4096;    // BLOCK_TMA static shared memory (barriers, slots), upper bound

// Largest CTA size the block kernel is compiled for at a given V.  V >= 8 is
// compiled for two resident CTAs per SM, so that one CTA's loads overlap the
// other's reductions; the register file then bounds threads x registers.
constexpr int block_max_threads_ct(int v) { return v >= 8 ? 512 : 1024; }
inline int block_max_threads(int v) { return block_max_threads_ct(v); }

// A per-device initialisation that is remembered only once it has succeeded.
// run(f) calls f (which returns 0 on success, else an error code) until one
// call succeeds; later calls return 0 without calling it.  A failed attempt --
// say, a first call made while the stream is being captured into a graph --
// leaves nothing behind, so the next call retries it rather than failing for
// the life of the process.  Thread-safe.
class InitOnSuccess {
public:
    template <class F>
    int run(F &&f)
    {
        if (done_.load(std::memory_order_acquire))
            return 0;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_.load(std::memory_order_relaxed))
            return 0;
        const int rc = f();
        if (rc == 0)
            done_.store(true, std::memory_order_release);
        return rc;
    }

private:
    std::mutex mu_;
    std::atomic<bool> done_{false};
};

struct Launch {
    const void *x;
    void *y;
    int64_t rows;
    int64_t cols;
    int dtype;
    softmax_launch_plan plan;
    CUstream_st *stream;
    unsigned int *dev_err;  // device address of the library's error word
};

// Backward launch: dx = y * (dy - sum dy*y).  plan.aligned: y, dy and dx rows
// all 16-byte aligned and whole chunks; dy_vec / dx_vec: that tensor's rows
// share y's 16-byte phase.
struct BwdLaunch {
    const void *y;
    const void *dy;
    void *dx;
    int64_t rows;
    int64_t cols;
    int dtype;
    softmax_launch_plan plan;
    CUstream_st *stream;
    int dy_vec;
    int dx_vec;
};

int launch_bwd(const BwdLaunch &l);

// Scaled, masked forward: y = softmax(scale * x + mask[r % mask_rows]) with an
// optional causal cut; plan.variant ROWGROUP or BLOCK.
struct MaskedLaunch {
    const void *x;
    void *y;
    int64_t rows;
    int64_t cols;
    int dtype;
    softmax_launch_plan plan;
    CUstream_st *stream;
    float scale;
    const void *mask;
    int64_t mask_rows;
    int64_t causal_q;
};

int launch_masked(const MaskedLaunch &l);
int plan_masked(const softmax_device_info &dev, const void *x, const void *y, int64_t rows, int64_t cols,
                int dtype, int variant, softmax_launch_plan *plan);

// LayerNorm / RMSNorm (k_norm.cuh): kind 0 / 1; `mode` says how rows, y and the
// gain / bias vectors sit on the 16-byte grid (kNormFast: rows, y, gamma and
// beta all on it -- vector gain / bias loads; kNormSame: y on x's phase;
// kNormOther: y on another phase).
constexpr int kNormLayer = 0;
constexpr int kNormRms = 1;
constexpr int kNormFast = 0;
constexpr int kNormSame = 1;
constexpr int kNormOther = 2;
constexpr int kNormMaxV = 4;  // chunks per thread (registers)

struct NormLaunch {
    const void *x;
    void *y;
    int64_t rows;
    int64_t cols;
    int dtype;
    softmax_launch_plan plan;
    CUstream_st *stream;
    int kind;
    int mode;
    const void *gamma;
    const void *beta;
    float eps;
    float *mean;
    float *rstd;
};

int launch_norm_f32(const NormLaunch &l);
int launch_norm_f16(const NormLaunch &l);
int launch_norm_bf16(const NormLaunch &l);
inline int launch_norm(const NormLaunch &l)
{
    return l.dtype == SOFTMAX_F32 ? launch_norm_f32(l)
                                  : (l.dtype == SOFTMAX_F16 ? launch_norm_f16(l) : launch_norm_bf16(l));
}
int validate_norm_args(int kind, const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
                       const void *gamma, const void *beta, float eps, const float *mean, const float *rstd);
int plan_norm(const softmax_device_info &dev, int kind, const void *x, const void *y, int64_t rows, int64_t cols,
              int dtype, const void *gamma, const void *beta, int variant, softmax_launch_plan *plan, int *mode);

// Remember a failing cudaError_t for softmax_last_cuda_error (this thread) and
// return SOFTMAX_ERR_CUDA.
int record_cuda_error(int cuda_error);

// SPLITK_GRID: one cooperative launch over every SM (k_grid.cu); scratch in the
// library's slot pool.  grid_capturing: the stream is being captured into a
// graph (the slot pool's event waits cannot be captured: callers plan
// another variant then).  reset_grid_scratch: clear the pool's barrier state
// after a reported device time-out.
int launch_grid(const Launch &l);
int grid_capturing(void *stream);
int reset_grid_scratch();

// SPLITK_WIDE: two launches, partials in `workspace` (rows * grid_x float4).
int launch_wide(const Launch &l, void *workspace);
uint64_t wide_workspace_bytes(const softmax_launch_plan &p);

// Backward dispatcher and validation (plan.cpp).
int plan_bwd(const softmax_device_info &dev, const void *y, const void *dy, const void *dx, int64_t rows,
             int64_t cols, int dtype, int variant, softmax_launch_plan *plan, int *dy_vec, int *dx_vec);
int validate_bwd_args(const void *y, const void *dy, const void *dx, int64_t rows, int64_t cols, int dtype);

// Each returns the cudaError_t of its launch (0 = success).
int launch_rowgroup_f32(const Launch &l);
int launch_rowgroup_f16(const Launch &l);
int launch_rowgroup_bf16(const Launch &l);
inline int launch_rowgroup(const Launch &l)
{
    return l.dtype == SOFTMAX_F32 ? launch_rowgroup_f32(l)
                                  : (l.dtype == SOFTMAX_F16 ? launch_rowgroup_f16(l) : launch_rowgroup_bf16(l));
}
int launch_block(const Launch &l);
int launch_block_tma(const Launch &l);
int launch_stream(const Launch &l);
int launch_splitk(const Launch &l);

// Validation shared by every entry point (no CUDA calls).
int validate_args(const void *x, const void *y, int64_t rows, int64_t cols, int dtype);

// Checks that a plan can serve this shape without any out-of-bounds access.
int validate_plan(const softmax_device_info &dev, const void *x, const void *y, int64_t rows,
                  int64_t cols, int dtype, const softmax_launch_plan &p);

inline int dtype_bytes(int dtype) { return dtype == SOFTMAX_F32 ? 4 : 2; }

}  // namespace osd
