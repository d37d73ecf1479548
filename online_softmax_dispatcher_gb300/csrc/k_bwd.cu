// k_bwd.cu -- softmax backward, dx = y * (dy - s), s = sum_k dy_k y_k, per row.
//
// The derivative of the definition (dy_i/dx_j = y_i (delta_ij - y_j)); the pages
// name the backward pass as separate work ("Softmax on DCU", section 5.4).  The
// same read-reduce-write skeleton as the forward kernels, with two inputs:
//
// * ROWGROUP: G lanes per row, V 16-byte chunks of y and of dy per lane held in
//   registers, one HBM read of each and one HBM write of dx per element.
// * BLOCK: one CTA per row, V <= 4 chunks of each per thread in registers.
// * STREAM: one CTA per row of any length; a sum pass, then a pass that
//   re-reads y and dy (from L2 when the rows fit there) and writes dx.
//
// s is a compensated (TwoSum) fp32 sum for every dtype: dx_j nearly cancels
// when dy_j ~ s, and the error of s is what is left of dx_j then.  The chunk
// grid is y's; dy and dx use vector accesses when their rows share y's 16-byte
// phase and per-element accesses when they do not.
#include "common.cuh"
#include "launch.h"

namespace osd {

namespace {

struct BwdArgs {
    const char *y;
    const char *dy;
    char *dx;
    int64_t rows;
    int64_t cols;
    int dy_vec;  // dy rows share y rows' 16-byte phase
    int dx_vec;  // dx rows share y rows' 16-byte phase
};

// chunk k (of y's grid) of another tensor's row starting at `row`: vector load
// when that row shares y's phase, else element by element (-inf padding is
// irrelevant here: the caller masks by y's slots).
template <int DT, bool ALIGNED>
__device__ __forceinline__ uint4 load_other(const RowGeom &g, const char *row, bool same_phase, int64_t k,
                                            int64_t cols)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    if (k >= g.nch)
        return make_uint4(0, 0, 0, 0);
    if (ALIGNED)
        return ld_chunk(row + 16 * k);
    const int64_t j0 = k * E - g.head;
    if (same_phase && j0 >= 0 && j0 + E <= cols)
        return ld_chunk(row - g.head * S + 16 * k);
    return ld_partial<DT>(row, j0, cols);
}

template <int DT, bool ALIGNED>
__device__ __forceinline__ void store_other(const RowGeom &g, char *row, bool same_phase, int64_t k, int64_t cols,
                                            const uint4 &p)
{
    RowGeom o = g;
    o.yr = row;
    o.y0 = row - g.head * Fmt<DT>::kBytes;
    store_chunk<DT, ALIGNED>(o, k, cols, p, same_phase);
}

// dy * y summed into a compensated accumulator; slots outside the row read as
// y = -inf (y's padding), which would give NaN: they are skipped by index.
template <int DT, bool ALIGNED>
__device__ __forceinline__ void dot_chunk(const uint4 &yc, const uint4 &dc, const RowGeom &g, int64_t k,
                                          int64_t cols, CSum &acc)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    float fy[E], fd[E];
    unpack<DT>(yc, fy);
    unpack<DT>(dc, fd);
    const int64_t j0 = k * E - g.head;
#pragma unroll
    for (int e = 0; e < E; e++) {
        const bool in_row = ALIGNED || (j0 + e >= 0 && j0 + e < cols);
        if (in_row && k < g.nch)
            Math<kF32>::add(acc, fd[e] * fy[e]);
    }
}

template <int DT>
__device__ __forceinline__ uint4 grad_chunk(const uint4 &yc, const uint4 &dc, float s)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    float fy[E], fd[E];
    unpack<DT>(yc, fy);
    unpack<DT>(dc, fd);
#pragma unroll
    for (int e = 0; e < E; e++)
        fy[e] = fy[e] * (fd[e] - s);
    return pack<DT>(fy);
}

template <int G>
__device__ __forceinline__ CSum group_csum(CSum a)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1)
        a = Math<kF32>::merge(a, Math<kF32>::shfl_xor(a, o));
    return a;
}

}  // namespace

template <int DT, int G, int V, bool ALIGNED>
__global__ void __launch_bounds__(kRowgroupThreads) k_bwd_rowgroup(const BwdArgs a)
{
    pdl_enter();
    const int groups = blockDim.x / G;
    const int gl = threadIdx.x & (G - 1);
    const int64_t stride = (int64_t)gridDim.x * groups;
    for (int64_t base = (int64_t)blockIdx.x * groups; base < a.rows; base += stride) {
        const int64_t r = base + threadIdx.x / G;
        const bool valid = r < a.rows;
        const int64_t rr = valid ? r : 0;
        const RowGeom g = row_geom<DT, ALIGNED>(a.y, a.dx, rr, a.cols);
        const int64_t off = rr * a.cols * Fmt<DT>::kBytes;
        uint4 yc[V], dc[V];
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int64_t k = gl + i * G;
            yc[i] = valid ? load_chunk<DT, ALIGNED>(g, k, a.cols) : make_uint4(0, 0, 0, 0);
            dc[i] = valid ? load_other<DT, ALIGNED>(g, a.dy + off, a.dy_vec != 0, k, a.cols) : make_uint4(0, 0, 0, 0);
        }
        CSum acc{0.f, 0.f};
        if (valid) {
#pragma unroll
            for (int i = 0; i < V; i++)
                dot_chunk<DT, ALIGNED>(yc[i], dc[i], g, gl + i * G, a.cols, acc);
        }
        acc = group_csum<G>(acc);
        const float s = acc.s + acc.c;
#pragma unroll
        for (int i = 0; i < V; i++) {
            opaque(yc[i]);
            opaque(dc[i]);
        }
        if (valid) {
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int64_t k = gl + i * G;
                if (k < g.nch)
                    store_other<DT, ALIGNED>(g, a.dx + off, a.dx_vec != 0, k, a.cols, grad_chunk<DT>(yc[i], dc[i], s));
            }
        }
    }
}

template <int DT, int V, bool ALIGNED>
__global__ void __launch_bounds__(512) k_bwd_block(const BwdArgs a)
{
    pdl_enter();
    __shared__ CSum slots[32];
    const int T = blockDim.x, t = threadIdx.x;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const RowGeom g = row_geom<DT, ALIGNED>(a.y, a.dx, r, a.cols);
        const int64_t off = r * a.cols * Fmt<DT>::kBytes;
        uint4 yc[V], dc[V];
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int64_t k = t + (int64_t)i * T;
            yc[i] = load_chunk<DT, ALIGNED>(g, k, a.cols);
            dc[i] = load_other<DT, ALIGNED>(g, a.dy + off, a.dy_vec != 0, k, a.cols);
        }
        CSum acc{0.f, 0.f};
#pragma unroll
        for (int i = 0; i < V; i++)
            dot_chunk<DT, ALIGNED>(yc[i], dc[i], g, t + (int64_t)i * T, a.cols, acc);
        acc = block_sum<kF32>(acc, slots);
        const float s = acc.s + acc.c;
#pragma unroll
        for (int i = 0; i < V; i++) {
            opaque(yc[i]);
            opaque(dc[i]);
        }
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int64_t k = t + (int64_t)i * T;
            if (k < g.nch)
                store_other<DT, ALIGNED>(g, a.dx + off, a.dx_vec != 0, k, a.cols, grad_chunk<DT>(yc[i], dc[i], s));
        }
    }
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kStreamThreads) k_bwd_stream(const BwdArgs a)
{
    pdl_enter();
    constexpr int U = 4;
    __shared__ CSum slots[32];
    const int64_t T = blockDim.x;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const RowGeom g = row_geom<DT, ALIGNED>(a.y, a.dx, r, a.cols);
        const int64_t off = r * a.cols * Fmt<DT>::kBytes;
        CSum acc{0.f, 0.f};
        for (int64_t k0 = threadIdx.x; k0 < g.nch; k0 += T * U) {
            uint4 yc[U], dc[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t k = k0 + u * T;
                yc[u] = load_chunk<DT, ALIGNED>(g, k, a.cols);
                dc[u] = load_other<DT, ALIGNED>(g, a.dy + off, a.dy_vec != 0, k, a.cols);
            }
#pragma unroll
            for (int u = 0; u < U; u++)
                dot_chunk<DT, ALIGNED>(yc[u], dc[u], g, k0 + u * T, a.cols, acc);
        }
        acc = block_sum<kF32>(acc, slots);
        const float s = acc.s + acc.c;
        for (int64_t k0 = threadIdx.x; k0 < g.nch; k0 += T * U) {
            uint4 yc[U], dc[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t k = k0 + u * T;
                yc[u] = load_chunk<DT, ALIGNED>(g, k, a.cols);
                dc[u] = load_other<DT, ALIGNED>(g, a.dy + off, a.dy_vec != 0, k, a.cols);
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t k = k0 + u * T;
                if (k < g.nch)
                    store_other<DT, ALIGNED>(g, a.dx + off, a.dx_vec != 0, k, a.cols, grad_chunk<DT>(yc[u], dc[u], s));
            }
        }
    }
}

namespace {

BwdArgs args_of(const BwdLaunch &l)
{
    return BwdArgs{(const char *)l.y, (const char *)l.dy, (char *)l.dx, l.rows, l.cols, l.dy_vec, l.dx_vec};
}

template <int DT, int G, int V, bool A>
int bwd_rowgroup_one(const BwdLaunch &l)
{
    return launch_pdl(k_bwd_rowgroup<DT, G, V, A>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT, int G, int V>
int bwd_rowgroup_a(const BwdLaunch &l)
{
    return l.plan.aligned ? bwd_rowgroup_one<DT, G, V, true>(l) : bwd_rowgroup_one<DT, G, V, false>(l);
}

template <int DT, int G>
int bwd_rowgroup_v(const BwdLaunch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 1:
        return bwd_rowgroup_a<DT, G, 1>(l);
    case 2:
        return bwd_rowgroup_a<DT, G, 2>(l);
    case 4:
        return bwd_rowgroup_a<DT, G, 4>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT>
int bwd_rowgroup_dt(const BwdLaunch &l)
{
    switch (l.plan.lanes_per_row) {
    case 1:
        return l.plan.chunks_per_thread == 1 ? bwd_rowgroup_a<DT, 1, 1>(l) : (int)cudaErrorInvalidValue;
    case 2:
        return bwd_rowgroup_v<DT, 2>(l);
    case 4:
        return bwd_rowgroup_v<DT, 4>(l);
    case 8:
        return bwd_rowgroup_v<DT, 8>(l);
    case 16:
        return bwd_rowgroup_v<DT, 16>(l);
    case 32:
        return bwd_rowgroup_v<DT, 32>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT, int V, bool A>
int bwd_block_one(const BwdLaunch &l)
{
    return launch_pdl(k_bwd_block<DT, V, A>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT>
int bwd_block_dt(const BwdLaunch &l)
{
    const bool A = l.plan.aligned != 0;
    switch (l.plan.chunks_per_thread) {
    case 2:
        return A ? bwd_block_one<DT, 2, true>(l) : bwd_block_one<DT, 2, false>(l);
    case 4:
        return A ? bwd_block_one<DT, 4, true>(l) : bwd_block_one<DT, 4, false>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT>
int bwd_stream_dt(const BwdLaunch &l)
{
    const dim3 grid((unsigned)l.plan.grid_x), block(l.plan.block_threads);
    if (l.plan.aligned)
        return launch_pdl(k_bwd_stream<DT, true>, grid, block, 0, (cudaStream_t)l.stream, no_attr(), args_of(l));
    return launch_pdl(k_bwd_stream<DT, false>, grid, block, 0, (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT>
int bwd_dt(const BwdLaunch &l)
{
    switch (l.plan.variant) {
    case SOFTMAX_VARIANT_ROWGROUP:
        return bwd_rowgroup_dt<DT>(l);
    case SOFTMAX_VARIANT_BLOCK:
        return bwd_block_dt<DT>(l);
    case SOFTMAX_VARIANT_STREAM:
        return bwd_stream_dt<DT>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace

int launch_bwd(const BwdLaunch &l)
{
    switch (l.dtype) {
    case kF32:
        return bwd_dt<kF32>(l);
    case kF16:
        return bwd_dt<kF16>(l);
    case kBF16:
        return bwd_dt<kBF16>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace osd
