// k_block.cu -- one CTA per row, the row cached in registers: one HBM read and
// one HBM write per element for rows of up to 512 threads x 16 chunks x 16 B
// = 128 KiB (past 256 threads at 16 chunks one CTA fills an SM: the grid is
// then one CTA per SM looping over rows, each prefetching its next row into L2).
//
// A row off the 16-byte grid is read as its interior chunks (16-byte vectors,
// interior chunk q to thread q mod T) plus at most 2E - 2 edge elements, one
// per thread of the first few, outside the unrolled chunk loops.
//
// Prior art: the one-pass kernels of "[CUDA] safe online softmax", section 2
// (fp16x8 register cache, 2.1; register + shared-memory cache, 2.2), written
// for a 48 KB-per-block, 64K-register sm_120 part, and the block-per-row kernel
// of the HIP softmax tutorial, section 3.  Differences here: any dtype and any
// alignment (16-byte chunks with peeled partial edges), the CTA size is a
// launch parameter (a multiple of 32 chosen by the dispatcher so that
// threads x V just covers the row), the max is reduced before any exp so that
// exp runs once per element (twice only when V * 8 > 32 floats would not fit
// next to the cached chunks), and the reductions are shuffle butterflies with
// one shared slot per warp ("Softmax on DCU", section 5.2: shuffles instead of
// a shared-memory tree).
#include "common.cuh"
#include "launch.h"

namespace osd {

// LOOP: 16 chunks at more than 256 threads (one CTA per SM, looping over
// rows); the other instances keep two CTAs per SM at 16 chunks.
template <int DT, int V, int PH, bool LOOP>
__global__ void __launch_bounds__(V >= 16 ? (LOOP ? 512 : 256) : block_max_threads_ct(V),
                                  V >= 16 ? (LOOP ? 1 : 2) : (V >= 8 ? 2 : 1))
    k_block(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols)
{
    pdl_enter();
    using M = Math<DT>;
    using Acc = typename M::Acc;
    constexpr int E = Fmt<DT>::kPerChunk;
    // keep e = exp(x - m) in registers when it fits next to the cached chunks,
    // else recompute it
    constexpr bool kKeepE = V * E <= 32 && V <= 4;
    constexpr bool kEdges = PH != kPhAligned;  // a CTA has >= 32 threads: one edge element each at most
    __shared__ float smax[32];
    __shared__ Acc ssum[32];
    const int T = blockDim.x;
    const int t = threadIdx.x;

    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        // LOOP: one CTA per SM (up to 512 threads x 16 chunks, rows of up to
        // 128 KiB) looping over rows: ask L2 for the CTA's next row, so HBM
        // keeps streaming while this row is reduced and written.  (A separate
        // instance: the check alone, in the other kernels, cost up to 6 points.)
        if constexpr (LOOP) {
            if (threadIdx.x == 0 && r + gridDim.x < rows)
                prefetch_row_l2(x + (r + gridDim.x) * cols * Fmt<DT>::kBytes, cols * Fmt<DT>::kBytes);
        }
        const ShortRow g = short_row<DT, PH == kPhAligned>(x, y, r, (int)cols);
        // Thread t takes interior chunks q = t + i * T - sh: the shift sh puts
        // every 8th slot on a 128-byte line, so a warp's 32 chunks span 4
        // lines, not 5 (taken when the CTA has sh slots to spare).
        int sh = (int)(((reinterpret_cast<uintptr_t>(g.x0) >> 4) + g.kf) & 7);
        if (sh > T * V - g.span)
            sh = 0;
        const int t0 = t - sh;
        uint4 raw[V];
#pragma unroll
        for (int i = 0; i < V; i++)
            raw[i] = load_interior<DT>(g, t0 + i * T);
        int je = -1;
        float xe = -INFINITY;
        if (kEdges && t < g.ne) {
            je = edge_col(g, t);
            xe = ld_elem<DT>(g.xr, je);
        }

        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < V; i++)
            m = fmaxf(m, chunk_max<DT>(raw[i]));
        if (kEdges)
            m = fmaxf(m, xe);
        m = block_max(m, smax);
        if (kEdges)
            xe = je >= 0 ? M::exp_shift(xe, m) : 0.f;

        if constexpr (kKeepE) {
            float v[V][E];
            Acc acc = M::zero();
#pragma unroll
            for (int i = 0; i < V; i++) {
                chunk_exp<DT>(raw[i], m, v[i]);
#pragma unroll
                for (int e = 0; e < E; e++)
                    M::add(acc, v[i][e]);
            }
            if (kEdges)
                M::add(acc, xe);
            acc = block_sum<DT>(acc, ssum);
            const float inv = 1.0f / M::value(acc);
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int q = t0 + i * T;
                if ((unsigned)q < (unsigned)g.span) {
                    float o[E];
#pragma unroll
                    for (int e = 0; e < E; e++)
                        o[e] = v[i][e] * inv;
                    store_interior<DT, PH>(g, q, pack<DT>(o));
                }
            }
            if (kEdges && je >= 0)
                st_elem<DT>(g.yr, je, xe * inv);
        } else {
#pragma unroll
            for (int i = 0; i < V; i++)
                opaque(raw[i]);
            Acc acc = M::zero();
#pragma unroll
            for (int i = 0; i < V; i++) {
                float f[E];
                chunk_exp<DT>(raw[i], m, f);
#pragma unroll
                for (int e = 0; e < E; e++)
                    M::add(acc, f[e]);
            }
            if (kEdges)
                M::add(acc, xe);
            acc = block_sum<DT>(acc, ssum);
            const float inv = 1.0f / M::value(acc);
#pragma unroll
            for (int i = 0; i < V; i++)
                opaque(raw[i]);
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int q = t0 + i * T;
                if ((unsigned)q < (unsigned)g.span) {
                    float f[E];
                    chunk_exp<DT>(raw[i], m, f);
#pragma unroll
                    for (int e = 0; e < E; e++)
                        f[e] *= inv;
                    store_interior<DT, PH>(g, q, pack<DT>(f));
                }
            }
            if (kEdges && je >= 0)
                st_elem<DT>(g.yr, je, xe * inv);
        }
    }
}

namespace {

template <int DT, int V, int PH>
int launch_one(const Launch &l)
{
    if constexpr (V >= 16) {
        if (l.plan.block_threads > 256)
            return launch_pdl(k_block<DT, V, PH, true>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads),
                              0, (cudaStream_t)l.stream, no_attr(), (const char *)l.x, (char *)l.y, l.rows, l.cols);
    }
    return launch_pdl(k_block<DT, V, PH, false>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), (const char *)l.x, (char *)l.y, l.rows, l.cols);
}

template <int DT, int V>
int launch_a(const Launch &l)
{
    if (l.plan.aligned)
        return launch_one<DT, V, kPhAligned>(l);
    return l.plan.y_vector ? launch_one<DT, V, kPhSame>(l) : launch_one<DT, V, kPhOther>(l);
}

template <int DT>
int launch_v(const Launch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 1:
        return launch_a<DT, 1>(l);
    case 2:
        return launch_a<DT, 2>(l);
    case 4:
        return launch_a<DT, 4>(l);
    case 8:
        return launch_a<DT, 8>(l);
    case 16:
        return launch_a<DT, 16>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace

int launch_block(const Launch &l)
{
    switch (l.dtype) {
    case kF32:
        return launch_v<kF32>(l);
    case kF16:
        return launch_v<kF16>(l);
    case kBF16:
        return launch_v<kBF16>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace osd
