// k_tma.cu -- persistent CTAs that stage row tiles in shared memory with 1-D
// bulk async copies (the TMA engine), one HBM read and one HBM write per
// element, for rows up to ~110 KB.
//
// Prior art: the register + shared-memory one-pass kernels of "[CUDA] safe
// online softmax", section 2.2 (medium / extreme: part of the row cached in
// 32-96 KB of shared memory filled by ordinary loads, one block per row), and
// the tiling ("Softmax on DCU", section 4.6: linearise many short rows into
// fixed-size tiles handed to blocks).  Here:
//
// * A tile is R consecutive rows -- one contiguous byte range of x -- copied
//   by ONE cp.async.bulk into a ring of shared-memory stages.  Warp 0 is the
//   producer (one elected lane); it keeps up to `stages` tiles in flight, so an
//   SM always has tens of KB of HBM reads outstanding while its 16 consumer
//   warps work on landed tiles.  Each stage has a "full" mbarrier (bulk-copy
//   bytes landed) and an "empty" mbarrier (all 16 consumer warps are done with
//   it).
// * The grid is one CTA per SM; CTA b takes tiles b, b + grid, ...
// * Consumers: W warps (W = 1..16) share a row; the 16 / W row groups take the
//   tile's rows in turn.  Per row: a max pass, an exp-sum pass and a write pass
//   over the row's 16-byte chunks in shared memory; group reductions are warp
//   butterflies plus, for W > 1, a named barrier and one shared slot per warp.
//   Outputs go straight from registers to global memory as 16-byte stores.
// * Unaligned rows: the bulk copy moves the 16-byte-aligned interior of the
//   tile; the (at most two) partial chunks at the tile's ends are read with
//   scalar loads; elements of a chunk that belong to a neighbouring row are
//   masked to -inf.
// * Every mbarrier wait is bounded (tma.cuh).  A consumer group agrees on a
//   give-up with a barrier-AND before it enters any named barrier, so no warp
//   is left waiting for one that left.
#include <atomic>

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace osd {

constexpr int kTmaMaxStages = kTmaMaxStagesHost;

struct TmaParams {
    const char *x;
    char *y;
    int64_t rows;
    int64_t cols;
    int R;            // rows per tile
    int W;            // warps per row group
    int stages;       // ring depth
    int stage_bytes;  // bytes per stage, multiple of 128
    int y_vec;        // y rows share x rows' 16-byte phase
    unsigned *err;    // device error word
};

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kTmaThreads, 1) k_tma(const TmaParams p)
{
    pdl_enter();
    using M = Math<DT>;
    using Acc = typename M::Acc;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ __align__(8) uint64_t full_bar[kTmaMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kTmaMaxStages];
    __shared__ float red_max[kTmaConsumerWarps][kTmaConsumerWarps];
    __shared__ Acc red_sum[kTmaConsumerWarps][kTmaConsumerWarps];
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row_bytes = p.cols * S;
    const int64_t ntiles = (p.rows + p.R - 1) / p.R;
    const uint32_t stage0 = smem_u32(stage_mem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), kTmaConsumerWarps);
        }
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0)
            return;
        uint32_t pending = 0, pend_parity = 0;
        uint32_t i = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
            const uint32_t s = i % p.stages, u = i / p.stages;
            const uint32_t fb = smem_u32(&full_bar[s]), eb = smem_u32(&empty_bar[s]);
            if (u > 0 && !mbar_wait(eb, (u - 1) & 1, &abort_flag)) {
                atomicOr(p.err, kErrEmptyWait);
                abort_flag = 1;
                break;
            }
            const int64_t r0 = tile * p.R;
            const int64_t nr = p.rows - r0 < p.R ? p.rows - r0 : p.R;
            const char *ts = p.x + r0 * row_bytes;
            const int lead = (int)(reinterpret_cast<uintptr_t>(ts) & 15);
            const int64_t c_lo = (lead + 15) >> 4;
            const int64_t c_hi = (lead + nr * row_bytes) >> 4;
            if (c_hi > c_lo) {
                const uint32_t bytes = (uint32_t)(16 * (c_hi - c_lo));
                mbar_arrive_expect_tx(fb, bytes);
                bulk_g2s(stage0 + s * p.stage_bytes + 16 * (uint32_t)c_lo, ts - lead + 16 * c_lo, bytes, fb);
            } else {
                mbar_arrive(fb);
            }
            pending |= 1u << s;
            pend_parity = (pend_parity & ~(1u << s)) | ((u & 1) << s);
        }
        // the CTA must not retire with copies in flight: wait (bounded) for the
        // last copy issued into each stage.
        for (int s = 0; s < p.stages; s++)
            if (pending & (1u << s))
                (void)mbar_wait(smem_u32(&full_bar[s]), (pend_parity >> s) & 1, &abort_flag, false);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int W = p.W, NG = kTmaConsumerWarps / W;
    const int group = cw / W, wig = cw % W;
    const int gt = wig * 32 + lane, GT = W * 32;
    const uint32_t bar_id = 1 + group, bar_threads = GT;

    uint32_t i = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
        const uint32_t s = i % p.stages, u = i / p.stages;
        bool ok = mbar_wait(smem_u32(&full_bar[s]), u & 1, &abort_flag);
        ok = W > 1 ? named_and(bar_id, bar_threads, ok) : (__all_sync(0xFFFFFFFFu, ok) != 0);
        if (!ok) {
            if (gt == 0) {
                atomicOr(p.err, kErrFullWait);
                abort_flag = 1;
            }
            break;
        }
        const uint32_t sbase = stage0 + s * p.stage_bytes;
        const int64_t r0 = tile * p.R;
        const int64_t nr = p.rows - r0 < p.R ? p.rows - r0 : p.R;
        const char *ts = p.x + r0 * row_bytes;
        char *ys = p.y + r0 * row_bytes;
        const int lead = (int)(reinterpret_cast<uintptr_t>(ts) & 15);
        const int h0 = lead / S;
        const int64_t c_lo = (lead + 15) >> 4;
        const int64_t c_hi = (lead + nr * row_bytes) >> 4;
        const int64_t tile_elems = nr * p.cols;

        for (int64_t j = group; j < nr; j += NG) {
            const int64_t e_lo = j * p.cols, e_hi = e_lo + p.cols;  // row j's tile elements
            const int64_t cf = (e_lo + h0) / E, cl = (e_hi - 1 + h0) / E;

            // chunk c of the tile, slots outside row j set to -inf
            auto read_raw = [&](int64_t c) -> uint4 {
                if (ALIGNED)
                    return lds_chunk(sbase + 16 * (uint32_t)c);
                const uint4 raw = (c >= c_lo && c < c_hi) ? lds_chunk(sbase + 16 * (uint32_t)c)
                                                          : ld_partial<DT>(ts, c * E - h0, tile_elems);
                const int64_t t0 = c * E - h0;
                return (t0 >= e_lo && t0 + E <= e_hi) ? raw : mask_chunk<DT>(raw, t0, e_lo, e_hi);
            };

            float m = -INFINITY;
            for (int64_t c = cf + gt; c <= cl; c += GT)
                m = fmaxf(m, chunk_max<DT>(read_raw(c)));
            m = warp_max_redux(m);
            if (W > 1) {
                if (lane == 0)
                    red_max[group][wig] = m;
                named_sync(bar_id, bar_threads);
                m = warp_max_redux(lane < W ? red_max[group][lane] : -INFINITY);
            }

            Acc acc = M::zero();
            for (int64_t c = cf + gt; c <= cl; c += GT) {
                float f[E];
                chunk_exp<DT>(read_raw(c), m, f);
#pragma unroll
                for (int e = 0; e < E; e++)
                    M::add(acc, f[e]);
            }
            acc = group_sum<DT, 32>(acc);
            if (W > 1) {
                if (lane == 0)
                    red_sum[group][wig] = acc;
                named_sync(bar_id, bar_threads);
                acc = group_sum<DT, 32>(lane < W ? red_sum[group][lane] : M::zero());
            }
            const float inv = 1.0f / M::value(acc);

            for (int64_t c = cf + gt; c <= cl; c += GT) {
                float f[E];
                chunk_exp<DT>(read_raw(c), m, f);
#pragma unroll
                for (int e = 0; e < E; e++)
                    f[e] *= inv;
                const uint4 o = pack<DT>(f);
                const int64_t t0 = c * E - h0;
                if (ALIGNED || (p.y_vec && t0 >= e_lo && t0 + E <= e_hi)) {
                    st_chunk(ys - lead + 16 * c, o);
                } else {
                    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                    for (int e = 0; e < E; e++) {
                        const int64_t t = t0 + e;
                        if (t >= e_lo && t < e_hi) {
                            if constexpr (S == 4)
                                st_u32(ys + 4 * t, w[e]);
                            else
                                st_u16(ys + 2 * t, (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
                        }
                    }
                }
            }
        }
        // this warp is done reading stage s
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&empty_bar[s]));
    }
}

namespace {

// Opt the kernel in to `bytes` of dynamic shared memory on the current device
// (static shared memory counts against the same 48 KB default, so every launch
// checks); the largest value set so far is cached per device.
template <int DT, bool A>
int ensure_dynamic_smem(int bytes)
{
    static std::atomic<int> granted[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return (int)e;
    if (dev < 0 || dev >= 64)
        return (int)cudaErrorInvalidDevice;
    if (granted[dev].load(std::memory_order_relaxed) >= bytes)
        return 0;
    e = cudaFuncSetAttribute(&k_tma<DT, A>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return (int)e;
    int cur = granted[dev].load();
    while (cur < bytes && !granted[dev].compare_exchange_weak(cur, bytes)) {
    }
    return 0;
}

template <int DT, bool A>
int launch_one(const Launch &l)
{
    auto *kern = &k_tma<DT, A>;
    const softmax_launch_plan &pl = l.plan;
    const int e = ensure_dynamic_smem<DT, A>(pl.smem_bytes);
    if (e != 0)
        return e;
    TmaParams p;
    p.x = (const char *)l.x;
    p.y = (char *)l.y;
    p.rows = l.rows;
    p.cols = l.cols;
    p.R = pl.rows_per_tile;
    p.W = pl.lanes_per_row / 32;
    p.stages = pl.stages;
    p.stage_bytes = pl.smem_bytes / pl.stages;
    p.y_vec = pl.y_vector;
    p.err = l.dev_err;
    return launch_pdl(kern, dim3((unsigned)pl.grid_x), dim3(kTmaThreads), (size_t)pl.smem_bytes,
                      (cudaStream_t)l.stream, no_attr(), p);
}

template <int DT>
int launch_a(const Launch &l)
{
    return l.plan.aligned ? launch_one<DT, true>(l) : launch_one<DT, false>(l);
}

}  // namespace

int launch_block_tma(const Launch &l)
{
    switch (l.dtype) {
    case kF32:
        return launch_a<kF32>(l);
    case kF16:
        return launch_a<kF16>(l);
    case kBF16:
        return launch_a<kBF16>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace osd
