// k_wide.cu -- few rows, huge cols, on every SM: SPLITK_WIDE.
//
// A thread-block cluster holds at most 16 CTAs, so the cluster split (k_splitk)
// puts at most 16 SMs on a row: 4 rows use 64 of 152 SMs.  This path splits
// each row over P CTAs (about two per SM over all rows) and merges the partial
// statistics through a small workspace in global memory, in two launches on
// the caller's stream -- the split of "[CUDA] safe online softmax", section
// 3.2 (pass 1 writes per-block partials, pass 2 merges them and writes), with
// the partials merged by every CTA of the row in the same fixed order instead
// of redundantly re-reduced per block:
//
// * k_wide_stats: CTA (p, r) reduces chunks [p * per, (p + 1) * per) of row r
//   to one partial: fp16 / bf16 the online pair (m_p, d_p); fp32 its max m_p
//   and then the compensated sum of exp(x - m_p) (a second pass over the
//   segment, served by L2 on these shapes), so each partial is rescaled once
//   in the merge and no rescale errors pile up.
// * k_wide_write: every CTA of row r merges the P partials (lane i takes
//   partials i, i + 32, ...; a fixed butterfly finishes), giving bit-identical
//   (m, d) in all of them, then re-reads its segment and writes exp(x - m) / d.
//
// Workspace: rows * P slots of 16 bytes (float4: m, d or s, c, unused),
// written by the first launch and read by the second; the caller provides it
// (softmax_fwd_ws).
#include "common.cuh"
#include "launch.h"
#include "stream_passes.cuh"

namespace osd {

// kWideStep (4) chunks in flight per thread per step keeps both kernels within
// the 64 registers that two 512-thread CTAs per SM leave; x re-reads in
// k_wide_write are L2 hits, every row segment having been read by k_wide_stats
// just before.
template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kStreamThreads, 2)
    k_wide_stats(const char *__restrict__ x, int64_t rows, int64_t cols, int P, float4 *__restrict__ ws)
{
    pdl_enter();
    using M = Math<DT>;
    __shared__ float smax[32];
    __shared__ typename M::Acc ssum[32];
    __shared__ MD smd[32];
    const int64_t r = blockIdx.y;
    const int p = blockIdx.x;
    const RowGeom g = row_geom<DT, ALIGNED>(x, const_cast<char *>(x), r, cols);
    const int64_t per = (g.nch + P - 1) / P;
    const int64_t kb = per * p < g.nch ? per * p : g.nch;
    const int64_t ke = kb + per < g.nch ? kb + per : g.nch;
    float4 out;
    if constexpr (DT == kF32) {
        const float m = block_max(pass_max<DT, ALIGNED, kWideStep>(g, kb, ke, cols), smax);
        CSum acc{0.f, 0.f};
        if (m != -INFINITY)
            acc = pass_sum<DT, ALIGNED, kWideStep>(g, kb, ke, cols, m);
        acc = block_sum<DT>(acc, ssum);
        out = make_float4(m, acc.s, acc.c, 0.f);
    } else {
        const MD md = block_md<DT>(pass_online<DT, ALIGNED, kWideStep>(g, kb, ke, cols), smd);
        out = make_float4(md.m, md.d, 0.f, 0.f);
    }
    if (threadIdx.x == 0)
        ws[r * P + p] = out;
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kStreamThreads, 2)
    k_wide_write(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols, int P,
                 const float4 *__restrict__ ws, int y_vec)
{
    pdl_enter();
    const int64_t r = blockIdx.y;
    const int p = blockIdx.x;
    const RowGeom g = row_geom<DT, ALIGNED>(x, y, r, cols);
    const int64_t per = (g.nch + P - 1) / P;
    const int64_t kb = per * p < g.nch ? per * p : g.nch;
    const int64_t ke = kb + per < g.nch ? kb + per : g.nch;
    float m, inv;
    merge_partials<DT>(ws, r, P, m, inv);
    pass_write<DT, ALIGNED, kWideStep>(g, kb, ke, cols, m, inv, y_vec != 0);
}

namespace {

template <int DT, bool A>
int wide_one(const Launch &l, float4 *ws)
{
    const dim3 grid((unsigned)l.plan.grid_x, (unsigned)l.plan.grid_y, 1);
    const int P = (int)l.plan.grid_x;
    const dim3 block(l.plan.block_threads);
    const int e = launch_pdl(k_wide_stats<DT, A>, grid, block, 0, (cudaStream_t)l.stream, no_attr(),
                             (const char *)l.x, l.rows, l.cols, P, ws);
    if (e != 0)
        return e;
    return launch_pdl(k_wide_write<DT, A>, grid, block, 0, (cudaStream_t)l.stream, no_attr(), (const char *)l.x,
                      (char *)l.y, l.rows, l.cols, P, (const float4 *)ws, (int)l.plan.y_vector);
}

template <int DT>
int wide_dt(const Launch &l, float4 *ws)
{
    return l.plan.aligned ? wide_one<DT, true>(l, ws) : wide_one<DT, false>(l, ws);
}

}  // namespace

int launch_wide(const Launch &l, void *workspace)
{
    float4 *ws = static_cast<float4 *>(workspace);
    switch (l.dtype) {
    case kF32:
        return wide_dt<kF32>(l, ws);
    case kF16:
        return wide_dt<kF16>(l, ws);
    case kBF16:
        return wide_dt<kBF16>(l, ws);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace osd
