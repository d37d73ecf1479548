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

template <int DT, bool ALIGNED, int STEP>
__device__ __forceinline__ void load_step(const RowGeom &g, int64_t k0, int64_t ke, int64_t cols,
                                          uint4 (&raw)[STEP])
{
    const int64_t T = blockDim.x;
#pragma unroll
    for (int u = 0; u < STEP; u++) {
        const int64_t k = k0 + u * T;
        raw[u] = k < ke ? load_chunk<DT, ALIGNED>(g, k, cols) : neg_inf_chunk<DT>();
    }
}

// online (m, d) over chunks [kb, ke) of a row, this thread's share.
template <int DT, bool ALIGNED, int STEP = kStep>
__device__ MD pass_online(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    MD md{-INFINITY, 0.f};
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP>(g, k0, ke, cols, raw);
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

template <int DT, bool ALIGNED, int STEP = kStep>
__device__ float pass_max(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols)
{
    float m = -INFINITY;
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP>(g, k0, ke, cols, raw);
#pragma unroll
        for (int u = 0; u < STEP; u++)
            m = fmaxf(m, chunk_max<DT>(raw[u]));
    }
    return m;
}

template <int DT, bool ALIGNED, int STEP = kStep>
__device__ typename Math<DT>::Acc pass_sum(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols, float m)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    typename M::Acc acc = M::zero();
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP>(g, k0, ke, cols, raw);
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

template <int DT, bool ALIGNED, int STEP = kStep>
__device__ void pass_write(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols, float m, float inv,
                           bool y_vec)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * STEP) {
        uint4 raw[STEP];
        load_step<DT, ALIGNED, STEP>(g, k0, ke, cols, raw);
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

}  // namespace osd
