// k_norm.cuh -- LayerNorm and RMSNorm along the last dimension on the
// softmax's skeleton: the row is read once into registers, reduced, normalised
// and written once.  Instantiated per dtype (k_norm_f32.cu, k_norm_f16.cu,
// k_norm_bf16.cu) so the instances compile in parallel.
//
// "Softmax on DCU", section 9, carries the softmax techniques (shuffle
// reductions, packed 16-bit access) over to LayerNorm and RMSNorm, which read,
// reduce, normalise and write the same way; the Pangu-Weather profile,
// section 3, runs fixed-width fp16 LayerNorm with one 64-lane wavefront per
// row and fp32 mean / variance.  Here a row is served either by a group of G
// lanes of one warp (G = 1 .. 32, V <= 4 chunks of 16 bytes per lane) or by a
// whole CTA (V <= 4 chunks per thread, up to 1024 threads), as the softmax
// kernels do, with the same interior-chunk / edge-element split for rows off
// the 16-byte grid.
//
// Per row: mu = (1/n) sum x (LayerNorm only), then var = (1/n) sum (x - mu)^2
// from the registers (two passes over the cached row, none over HBM),
// rstd = rsqrt(var + eps) on the SFU (about 2 ulp of fp32), and
// y = (x * rstd - mu * rstd) * g + b as two FMAs (the rounding of mu * rstd
// shifts every output of the row alike, by at most 2^-24 |mu| rstd), rounded
// to nearest even.  Sums are fp32, compensated (TwoSum) for fp32 input.  The
// lanes-per-row kernel keeps the row as floats after one unpack; the
// CTA-per-row kernel keeps it packed and unpacks per pass.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace osd {

struct NormArgs {
    const char *x;
    char *y;
    int64_t rows;
    int cols;
    const char *gamma;  // [cols] or null
    const char *beta;   // [cols] or null (always null for RMSNorm)
    float eps;
    float *mean;  // [rows] or null
    float *rstd;  // [rows] or null
};

// 16 bytes of gain / bias, L1-cached (every row reads the same vector).
__device__ __forceinline__ uint4 ld_chunk_shared(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The gain or bias values of interior chunk q: one vector load when rows and
// vector share the 16-byte grid (MODE kNormFast), else element loads.
template <int DT, int MODE>
__device__ __forceinline__ void vec_chunk(const char *v, const ShortRow &g, int q, float (&f)[Fmt<DT>::kPerChunk])
{
    constexpr int E = Fmt<DT>::kPerChunk;
    if constexpr (MODE == kNormFast) {
        unpack<DT>(ld_chunk_shared(v + ((int64_t)(g.kf + q) << 4)), f);
    } else {
        const int j0 = (g.kf + q) * E - g.head;
#pragma unroll
        for (int e = 0; e < E; e++)
            f[e] = ld_elem<DT>(v, j0 + e);
    }
}

template <int DT, int G>
struct GroupSum {
    __device__ __forceinline__ typename Math<DT>::Acc operator()(typename Math<DT>::Acc a) const
    {
        return group_sum<DT, G>(a);
    }
};

template <int DT>
struct CtaSum {
    typename Math<DT>::Acc *slots;
    __device__ __forceinline__ typename Math<DT>::Acc operator()(typename Math<DT>::Acc a) const
    {
        return block_sum<DT>(a, slots);
    }
};

// The row's chunk i as floats: from the floats kept after the first unpack
// (KEEP) or unpacked again from the packed chunk.
template <int DT, int V, bool KEEP>
struct RowCache {
    static constexpr int E = Fmt<DT>::kPerChunk;
    uint4 raw[V];
    float f[KEEP ? V : 1][KEEP ? E : 1];
    __device__ __forceinline__ void get(int i, float (&out)[E]) const
    {
        if constexpr (KEEP) {
#pragma unroll
            for (int e = 0; e < E; e++)
                out[e] = f[i][e];
        } else {
            unpack<DT>(raw[i], out);
        }
    }
};

// One row for a team of L threads (lane = this thread's index in the team).
// NE edge elements per thread; `valid` false for a lane group past the last
// row (it still takes part in the team's reductions).
// AFF false: no gain and no bias (the caller knows), so the output loop
// carries no test of the vectors at all.
template <int DT, int KIND, int V, int MODE, int NE, bool KEEP, bool AFF, class Red>
__device__ __forceinline__ void norm_row(const NormArgs &a, int64_t r, bool valid, int lane, int L, float inv_n,
                                         Red red)
{
    using M = Math<DT>;
    using Acc = typename M::Acc;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int PH = MODE == kNormFast ? kPhAligned : (MODE == kNormSame ? kPhSame : kPhOther);
    const ShortRow g = short_row<DT, MODE == kNormFast>(a.x, a.y, valid ? r : 0, a.cols);

    RowCache<DT, V, KEEP> c;
    // interior chunk lane + i * L of this row exists
    // which interior chunks lane + i * L exist, decided once before the loads
    // (measured: deciding it again in each pass slows the CTA-per-row kernel
    // by a quarter)
    const int span = valid ? g.span : 0;
    unsigned okm = 0;  // bit i: chunk lane + i * L exists
#pragma unroll
    for (int i = 0; i < V; i++)
        okm |= (unsigned)(lane + i * L < span) << i;
    const auto has = [okm](int i) { return ((okm >> i) & 1u) != 0; };
#pragma unroll
    for (int i = 0; i < V; i++) {
        const int q = lane + i * L;
        c.raw[i] = has(i) ? ld_chunk(g.x0 + ((int64_t)(g.kf + q) << 4)) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (KEEP) {
#pragma unroll
        for (int i = 0; i < V; i++)
            unpack<DT>(c.raw[i], c.f[i]);
    }
    int je[NE > 0 ? NE : 1];
    float xe[NE > 0 ? NE : 1];
#pragma unroll
    for (int u = 0; u < NE; u++) {
        const int p = lane + u * L;
        je[u] = (valid && p < g.ne) ? edge_col(g, p) : -1;
        xe[u] = je[u] >= 0 ? ld_elem<DT>(g.xr, je[u]) : 0.f;
    }

    // mean (LayerNorm): slots past the row hold +0 and add nothing
    float mu = 0.f;
    if constexpr (KIND == kNormLayer) {
        Acc s = M::zero();
#pragma unroll
        for (int i = 0; i < V; i++) {
            float f[E];
            c.get(i, f);
#pragma unroll
            for (int e = 0; e < E; e++)
                M::add(s, f[e]);
        }
#pragma unroll
        for (int u = 0; u < NE; u++)
            M::add(s, xe[u]);
        mu = M::value(red(s)) * inv_n;
    }

    // variance about mu (RMSNorm: mean square), from the registers
    Acc q2 = M::zero();
#pragma unroll
    for (int i = 0; i < V; i++) {
        if (has(i)) {
            float f[E];
            c.get(i, f);
#pragma unroll
            for (int e = 0; e < E; e++) {
                const float d = f[e] - mu;
                M::add(q2, d * d);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NE; u++) {
        if (je[u] >= 0) {
            const float d = xe[u] - mu;
            M::add(q2, d * d);
        }
    }
    const float var = M::value(red(q2)) * inv_n;
    const float rs = rsqrtf(var + a.eps);
    const float nmr = -mu * rs;  // y = x * rs + nmr, before the gain and bias
    if (valid && lane == 0) {
        if (KIND == kNormLayer && a.mean)
            a.mean[r] = mu;
        if (a.rstd)
            a.rstd[r] = rs;
    }

    // y = (x - mu) * rstd * g + b
    if (!valid)
        return;
#pragma unroll
    for (int i = 0; i < V; i++) {
        if (has(i)) {
            const int q = lane + i * L;
            float f[E];
            c.get(i, f);
            if constexpr (AFF) {
                float gv[E], bv[E];
                if (a.gamma)
                    vec_chunk<DT, MODE>(a.gamma, g, q, gv);
                if (KIND == kNormLayer && a.beta)
                    vec_chunk<DT, MODE>(a.beta, g, q, bv);
#pragma unroll
                for (int e = 0; e < E; e++) {
                    const float z = fmaf(f[e], rs, nmr);
                    if (a.gamma || (KIND == kNormLayer && a.beta)) {
                        const float gg = a.gamma ? gv[e] : 1.0f;
                        const float bb = (KIND == kNormLayer && a.beta) ? bv[e] : 0.0f;
                        f[e] = fmaf(z, gg, bb);
                    } else {
                        f[e] = z;
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; e++)
                    f[e] = fmaf(f[e], rs, nmr);
            }
            store_interior<DT, PH>(g, q, pack<DT>(f));
        }
    }
#pragma unroll
    for (int u = 0; u < NE; u++) {
        if (je[u] >= 0) {
            const float z = fmaf(xe[u], rs, nmr);
            if constexpr (AFF) {
                const float gg = a.gamma ? ld_elem<DT>(a.gamma, je[u]) : 1.0f;
                const float bb = (KIND == kNormLayer && a.beta) ? ld_elem<DT>(a.beta, je[u]) : 0.0f;
                st_elem<DT>(g.yr, je[u], fmaf(z, gg, bb));
            } else {
                st_elem<DT>(g.yr, je[u], z);
            }
        }
    }
}

// G lanes per row, 256 / G rows per CTA per step.
template <int DT, int KIND, int G, int V, int MODE, bool AFF>
__global__ void __launch_bounds__(kRowgroupThreads) k_norm_rowgroup(const NormArgs a)
{
    pdl_enter();
    constexpr int NE = MODE == kNormFast ? 0 : edge_slots<DT, G>();
    const int groups = blockDim.x / G;
    const int gl = threadIdx.x & (G - 1);
    const int64_t stride = (int64_t)gridDim.x * groups;
    const float inv_n = 1.0f / (float)a.cols;
    // every thread of a CTA runs the same number of iterations, so the
    // butterflies see converged warps
    for (int64_t base = (int64_t)blockIdx.x * groups; base < a.rows; base += stride) {
        const int64_t r = base + threadIdx.x / G;
        norm_row<DT, KIND, V, MODE, NE, true, AFF>(a, r, r < a.rows, gl, G, inv_n, GroupSum<DT, G>{});
    }
}

// One CTA per row.
template <int DT, int KIND, int V, int MODE>
__global__ void __launch_bounds__(1024) k_norm_block(const NormArgs a)
{
    pdl_enter();
    __shared__ typename Math<DT>::Acc slots[32];
    constexpr int NE = MODE == kNormFast ? 0 : 1;  // >= 32 threads: one edge element each at most
    const float inv_n = 1.0f / (float)a.cols;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        norm_row<DT, KIND, V, MODE, NE, false, true>(a, r, true, threadIdx.x, blockDim.x, inv_n, CtaSum<DT>{slots});
}

namespace norm_detail {

inline NormArgs args_of(const NormLaunch &l)
{
    return NormArgs{(const char *)l.x, (char *)l.y, l.rows, (int)l.cols, (const char *)l.gamma,
                    l.kind == kNormLayer ? (const char *)l.beta : nullptr, l.eps,
                    l.kind == kNormLayer ? l.mean : nullptr, l.rstd};
}

template <int DT, int KIND, int G, int V, int MODE>
int rg_one(const NormLaunch &l)
{
    const NormArgs a = args_of(l);
    if (a.gamma || a.beta)
        return launch_pdl(k_norm_rowgroup<DT, KIND, G, V, MODE, true>, dim3((unsigned)l.plan.grid_x),
                          dim3(l.plan.block_threads), 0, (cudaStream_t)l.stream, no_attr(), a);
    return launch_pdl(k_norm_rowgroup<DT, KIND, G, V, MODE, false>, dim3((unsigned)l.plan.grid_x),
                      dim3(l.plan.block_threads), 0, (cudaStream_t)l.stream, no_attr(), a);
}

template <int DT, int KIND, int V, int MODE>
int blk_one(const NormLaunch &l)
{
    return launch_pdl(k_norm_block<DT, KIND, V, MODE>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads),
                      0, (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT, int KIND, int G, int V>
int rg_mode(const NormLaunch &l)
{
    switch (l.mode) {
    case kNormFast:
        return rg_one<DT, KIND, G, V, kNormFast>(l);
    case kNormSame:
        return rg_one<DT, KIND, G, V, kNormSame>(l);
    default:
        return rg_one<DT, KIND, G, V, kNormOther>(l);
    }
}

template <int DT, int KIND, int G>
int rg_v(const NormLaunch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 1:
        return rg_mode<DT, KIND, G, 1>(l);
    case 2:
        if constexpr (G > 1)
            return rg_mode<DT, KIND, G, 2>(l);
        break;
    case 3:
        if constexpr (G > 1)
            return rg_mode<DT, KIND, G, 3>(l);
        break;
    case 4:
        if constexpr (G > 1)
            return rg_mode<DT, KIND, G, 4>(l);
        break;
    default:
        break;
    }
    return (int)cudaErrorInvalidValue;
}

template <int DT, int KIND>
int rg_g(const NormLaunch &l)
{
    switch (l.plan.lanes_per_row) {
    case 1:
        return rg_v<DT, KIND, 1>(l);
    case 2:
        return rg_v<DT, KIND, 2>(l);
    case 4:
        return rg_v<DT, KIND, 4>(l);
    case 8:
        return rg_v<DT, KIND, 8>(l);
    case 16:
        return rg_v<DT, KIND, 16>(l);
    case 32:
        return rg_v<DT, KIND, 32>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT, int KIND, int V>
int blk_mode(const NormLaunch &l)
{
    switch (l.mode) {
    case kNormFast:
        return blk_one<DT, KIND, V, kNormFast>(l);
    case kNormSame:
        return blk_one<DT, KIND, V, kNormSame>(l);
    default:
        return blk_one<DT, KIND, V, kNormOther>(l);
    }
}

template <int DT, int KIND>
int blk_v(const NormLaunch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 1:
        return blk_mode<DT, KIND, 1>(l);
    case 2:
        return blk_mode<DT, KIND, 2>(l);
    case 4:
        return blk_mode<DT, KIND, 4>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT, int KIND>
int launch_kind(const NormLaunch &l)
{
    if (l.plan.variant == SOFTMAX_VARIANT_ROWGROUP)
        return rg_g<DT, KIND>(l);
    if (l.plan.variant == SOFTMAX_VARIANT_BLOCK)
        return blk_v<DT, KIND>(l);
    return (int)cudaErrorInvalidValue;
}

template <int DT>
int launch_dt(const NormLaunch &l)
{
    return l.kind == kNormLayer ? launch_kind<DT, kNormLayer>(l) : launch_kind<DT, kNormRms>(l);
}

}  // namespace norm_detail
}  // namespace osd
