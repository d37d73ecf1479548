// stream_passes.cuh -- per-thread passes over a chunk range [kb, ke) of one
// row, kStreamUnroll 16-byte loads in flight per thread per step, shared by the
// streaming kernel and the wide split kernels (which pass a shorter STEP to
// stay within 64 registers at two CTAs per SM).  Each returns this thread's
// share; the caller reduces over the CTA.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace osd {
constexpr int kStep = kStreamUnroll;  // chunks per thread per step

// L2 policy of a pass's loads on rows on the 16-byte grid: 0 none, 1
// evict-last (the row is read again later in the launch), 2 evict-first (its
// last read).  Taken by the streaming kernel when the rows in flight outgrow
// L2 (its backward walk), where it keeps more of each row there for the
// re-read; where the rows fit L2 the plain loads measured faster.
template <int POL>
__device__ __forceinline__ uint4 ld_chunk_pol(const void *p)
{
    if constexpr (POL == 0) {
        return ld_chunk(p);
    } else {
        uint64_t pol;
        if constexpr (POL == 1)
            asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
        else
            asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        uint4 v;
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p), "l"(pol));
        return v;
    }
}

template <int DT, bool ALIGNED, int STEP, int POL = 0>
__device__ __forceinline__ void load_step(const RowGeom &g, int64_t k0, int64_t ke, int64_t cols,
                                          uint4 (&raw)[STEP])
{
    const int64_t T = blockDim.x;
#pragma unroll
    for (int u = 0; u < STEP; u++) {
        const int64_t k = k0 + u * T;
        if constexpr (ALIGNED && POL != 0)
            raw[u] = k < ke ? ld_chunk_pol<POL>(g.x0 + 16 * k) : neg_inf_chunk<DT>();
        else
            raw[u] = k < ke ? load_chunk<DT, ALIGNED>(g, k, cols) : neg_inf_chunk<DT>();
    }
}

// online (m, d) over chunks [kb, ke) of a row, this thread's share.
template <int DT, bool ALIGNED, int STEP = kStep, int POL = 0>
__device__ MD pass_online(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    MD md{-INFINITY, 0.f};
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP, POL>(g, k0, ke, cols, raw);
        float mt = -INFINITY;
#pragma unroll
        for (int u = 0; u < STEP; u++)
            mt = fmaxf(mt, chunk_max<DT>(raw[u]));
        // a step of all -inf (genuine -inf inputs) leaves (m, d) unchanged
        if (mt == -INFINITY)
            continue;
        if (mt > md.m) {
            md.d = md.m == -INFINITY ? 0.f : md.d * M::exp_of(md.m - mt);
            md.m = mt;
        }
#pragma unroll
        for (int u = 0; u < STEP; u++)
            opaque(raw[u]);
        float s = 0.f;
#pragma unroll
        for (int u = 0; u < STEP; u++) {
            float f[E];
            chunk_exp<DT>(raw[u], md.m, f);
#pragma unroll
            for (int e = 0; e < E; e++)
                s += f[e];
        }
        md.d += s;
    }
    return md;
}

template <int DT, bool ALIGNED, int STEP = kStep, int POL = 0>
__device__ float pass_max(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols)
{
    float m = -INFINITY;
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP, POL>(g, k0, ke, cols, raw);
#pragma unroll
        for (int u = 0; u < STEP; u++)
            m = fmaxf(m, chunk_max<DT>(raw[u]));
    }
    return m;
}

template <int DT, bool ALIGNED, int STEP = kStep, int POL = 0>
__device__ typename Math<DT>::Acc pass_sum(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols, float m)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    typename M::Acc acc = M::zero();
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP, POL>(g, k0, ke, cols, raw);
#pragma unroll
        for (int u = 0; u < STEP; u++) {
            float f[E];
            chunk_exp<DT>(raw[u], m, f);
#pragma unroll
            for (int e = 0; e < E; e++)
                M::add(acc, f[e]);
        }
    }
    return acc;
}

template <int DT, bool ALIGNED, int STEP = kStep, int POL = 0>
__device__ void pass_write(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols, float m, float inv,
                           bool y_vec)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP, POL>(g, k0, ke, cols, raw);
#pragma unroll
        for (int u = 0; u < STEP; u++) {
            const int64_t k = k0 + u * T;
            if (k < ke) {
                float f[E];
                chunk_exp<DT>(raw[u], m, f);
#pragma unroll
                for (int e = 0; e < E; e++)
                    f[e] *= inv;
                store_chunk<DT, ALIGNED>(g, k, cols, pack<DT>(f), y_vec);
            }
        }
    }
}

// Merge the P partial statistics of row r (float4 slots: fp32 (m, s, c), the
// local max and compensated sum of exp(x - m); 16-bit (m, d)); every warp does
// it, identically, so every CTA of the row holds bit-identical (m, 1/d).  The
// slots are read through L2 (another CTA, or the previous launch, wrote them).
template <int DT>
__device__ __forceinline__ void merge_partials(const float4 *ws, int64_t r, int P, float &m, float &inv)
{
    const int lane = threadIdx.x & 31;
    if constexpr (DT == kF32) {
        float mloc = -INFINITY;
        for (int i = lane; i < P; i += 32)
            mloc = fmaxf(mloc, __ldcg(&ws[r * P + i]).x);
        m = warp_max_redux(mloc);
        CSum acc{0.f, 0.f};
        for (int i = lane; i < P; i += 32) {
            const float4 q = __ldcg(&ws[r * P + i]);
            if (q.x != -INFINITY) {
                // one rescale per partial: (s + c) * exp(m_p - m), exp_shift keeps
                // m_p - m exact
                const float f = Math<kF32>::exp_shift(q.x, m);
                Math<kF32>::add(acc, q.y * f);
                Math<kF32>::add(acc, q.z * f);
            }
        }
        acc = group_sum<kF32, 32>(acc);
        inv = 1.0f / (acc.s + acc.c);
    } else {
        MD md{-INFINITY, 0.f};
        for (int i = lane; i < P; i += 32) {
            const float4 q = __ldcg(&ws[r * P + i]);
            md = md_merge<DT>(md, MD{q.x, q.y});
        }
        md = warp_md<DT>(md);
        m = md.m;
        inv = 1.0f / md.d;
    }
}

}  // namespace osd
