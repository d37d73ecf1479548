// k_rowgroup.cuh -- G lanes per row (G = 1, 2, ..., 32), the row cached in
// registers, one HBM read and one HBM write per element.  Instantiated once
// per dtype (k_rowgroup_f32.cu, k_rowgroup_f16.cu, k_rowgroup_bf16.cu) so the
// instances compile in parallel.
//
// Prior art: the wavefront-per-row kernel of "Softmax on DCU", section 4.1
// (one 64-lane wavefront per row, shuffle-reduced max), and the block-per-row
// register-cached fp16x8 kernel of "[CUDA] safe online softmax", section 2.1.
// On this GPU a row of up to 32 lanes x 32 floats is served by a group of
// lanes of one 32-lane warp instead: short rows get G < 32 lanes (the HIP
// softmax tutorial, section 5, likewise sizes its block to the next power of
// two >= cols) so that a warp holds 32 / G rows and no lane idles; long rows
// get a whole warp.
//
// Per row: the group's lanes load their 16-byte interior chunks (interior
// chunk q goes to lane q mod G) and, for a row off the 16-byte grid, its at
// most 2E - 2 edge elements one by one (edge element p to lane p mod G), take
// the max with a G-lane xor butterfly, compute e = exp(x - m) once per element
// and keep it in registers, butterfly-sum e, then write e * (1 / d): 16-byte
// stores for interior chunks, element stores for the edges.  The edge work
// sits outside the unrolled chunk loops, which stay as short as for aligned
// rows.  The grid normally covers every
// row once (many small CTAs: HBM latency is hidden by occupancy, and the tail
// of the launch is one short CTA); a smaller grid walks the rows with a
// stride.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace osd {

template <int DT, int G, int V, int PH>
__global__ void __launch_bounds__(kRowgroupThreads)
    k_rowgroup(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols)
{
    pdl_enter();
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int NE = PH == kPhAligned ? 0 : edge_slots<DT, G>();
    const int groups = blockDim.x / G;  // rows per CTA per step
    const int gl = threadIdx.x & (G - 1);
    const int64_t stride = (int64_t)gridDim.x * groups;
    // every thread of a CTA runs the same number of iterations (the loop bound
    // is the CTA's first row), so the butterflies see converged warps.
    for (int64_t base = (int64_t)blockIdx.x * groups; base < rows; base += stride) {
        const int64_t r = base + threadIdx.x / G;
        const bool valid = r < rows;
        const ShortRow g = short_row<DT, PH == kPhAligned>(x, y, valid ? r : 0, (int)cols);

        uint4 raw[V];
#pragma unroll
        for (int i = 0; i < V; i++)
            raw[i] = valid ? load_interior<DT>(g, gl + i * G) : neg_inf_chunk<DT>();
        // this lane's edge elements (unaligned rows): column je, value xe
        int je[NE > 0 ? NE : 1];
        float xe[NE > 0 ? NE : 1];
#pragma unroll
        for (int u = 0; u < NE; u++) {
            const int p = gl + u * G;
            je[u] = (valid && p < g.ne) ? edge_col(g, p) : -1;
            xe[u] = je[u] >= 0 ? ld_elem<DT>(g.xr, je[u]) : -INFINITY;
        }

        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < V; i++)
            m = fmaxf(m, chunk_max<DT>(raw[i]));
#pragma unroll
        for (int u = 0; u < NE; u++)
            m = fmaxf(m, xe[u]);
        m = G == 32 ? warp_max_redux(m) : group_max<G>(m);

        float v[V][E];
        typename M::Acc acc = M::zero();
#pragma unroll
        for (int i = 0; i < V; i++) {
            chunk_exp<DT>(raw[i], m, v[i]);
#pragma unroll
            for (int e = 0; e < E; e++)
                M::add(acc, v[i][e]);
        }
#pragma unroll
        for (int u = 0; u < NE; u++) {
            xe[u] = je[u] >= 0 ? M::exp_shift(xe[u], m) : 0.f;
            M::add(acc, xe[u]);
        }
        acc = group_sum<DT, G>(acc);
        const float inv = 1.0f / M::value(acc);

        if (valid) {
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int q = gl + i * G;
                if (q < g.span) {
                    float o[E];
#pragma unroll
                    for (int e = 0; e < E; e++)
                        o[e] = v[i][e] * inv;
                    store_interior<DT, PH>(g, q, pack<DT>(o));
                }
            }
#pragma unroll
            for (int u = 0; u < NE; u++)
                if (je[u] >= 0)
                    st_elem<DT>(g.yr, je[u], xe[u] * inv);
        }
    }
}

template <int DT, int G, int V, int PH>
int rowgroup_launch_one(const Launch &l)
{
    return launch_pdl(k_rowgroup<DT, G, V, PH>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), (const char *)l.x, (char *)l.y, l.rows, l.cols);
}

template <int DT, int G, int V>
int rowgroup_launch_a(const Launch &l)
{
    if (l.plan.aligned)
        return rowgroup_launch_one<DT, G, V, kPhAligned>(l);
    return l.plan.y_vector ? rowgroup_launch_one<DT, G, V, kPhSame>(l) : rowgroup_launch_one<DT, G, V, kPhOther>(l);
}

// V chunks per lane, V * E <= 32 floats: V in {1, 2, 4} (and 8 for fp32).
template <int DT, int G>
int rowgroup_launch_v(const Launch &l)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    switch (l.plan.chunks_per_thread) {
    case 1:
        return rowgroup_launch_a<DT, G, 1>(l);
    case 2:
        return rowgroup_launch_a<DT, G, 2>(l);
    case 4:
        return rowgroup_launch_a<DT, G, 4>(l);
    case 8:
        if constexpr (8 * E <= kRowgroupMaxFloats)
            return rowgroup_launch_a<DT, G, 8>(l);
        return (int)cudaErrorInvalidValue;
    default:
        return (int)cudaErrorInvalidValue;
    }
}

// A single lane per row only serves rows of one chunk.
template <int DT>
int rowgroup_launch_dt(const Launch &l)
{
    switch (l.plan.lanes_per_row) {
    case 1:
        return l.plan.chunks_per_thread == 1 ? rowgroup_launch_a<DT, 1, 1>(l) : (int)cudaErrorInvalidValue;
    case 2:
        return rowgroup_launch_v<DT, 2>(l);
    case 4:
        return rowgroup_launch_v<DT, 4>(l);
    case 8:
        return rowgroup_launch_v<DT, 8>(l);
    case 16:
        return rowgroup_launch_v<DT, 16>(l);
    case 32:
        return rowgroup_launch_v<DT, 32>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace osd
