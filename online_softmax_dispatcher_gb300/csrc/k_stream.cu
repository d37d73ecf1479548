// k_stream.cu -- rows too long to cache on chip.
//
// STREAM: one CTA per row.  For fp16 / bf16 a first pass keeps a per-thread
// online pair (m, d) -- per step of 8 chunks: m' = max(m, max(step)),
// d = d e^(m - m') + sum e^(x - m') -- which a block merge of (m, d) pairs
// finishes; a second pass re-reads x (from L2 when the row set fits there) and
// writes exp(x - m) / d.  This is the two-pass "vanilla" kernel of "[CUDA]
// safe online softmax", section 3.1, with the chunked update of its section 1
// (safe_online_softmax) and the per-element update of "Softmax on DCU",
// section 4.3.  For fp32 the rescaling is dropped: a max pass, then a sum pass
// with that fixed max (compensated), then the write pass -- each rescale of a
// partial sum costs up to an ulp, and a row whose max keeps growing would pile
// those up past the fp32 error budget.
//
// SPLITK: a thread-block cluster of C CTAs per row (grid = C x rows), each CTA
// streaming a contiguous 1/C of the row.  The CTAs publish their partial
// statistics in shared memory and read their peers' over distributed shared
// memory after a hardware cluster barrier, merge them in rank order (so all C
// CTAs hold bit-identical m and d), and write their slice.  The split-k
// kernel of "[CUDA] safe online softmax", section 3.2, needs two launches and a
// global workspace for the partial (m, d) pairs, and section 3.2 rejects a
// grid-wide sync or atomics-and-polling in one kernel; the cluster barrier is
// the hardware-scheduled alternative it did not have, with no workspace and no
// spin loop.
#include "common.cuh"
#include "launch.h"

namespace osd {

namespace {

constexpr int U = kStreamUnroll;

template <int DT, bool ALIGNED>
__device__ __forceinline__ void load_step(const RowGeom &g, int64_t k0, int64_t ke, int64_t cols,
                                          uint4 (&raw)[U])
{
    const int64_t T = blockDim.x;
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int64_t k = k0 + u * T;
        raw[u] = k < ke ? load_chunk<DT, ALIGNED>(g, k, cols) : neg_inf_chunk<DT>();
    }
}

// online (m, d) over chunks [kb, ke) of a row, this thread's share.
template <int DT, bool ALIGNED>
__device__ MD pass_online(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    MD md{-INFINITY, 0.f};
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * U) {
        uint4 raw[U];
        load_step<DT, ALIGNED>(g, k0, ke, cols, raw);
        float mt = -INFINITY;
#pragma unroll
        for (int u = 0; u < U; u++)
            mt = fmaxf(mt, chunk_max<DT>(raw[u]));
        if (mt > md.m) {
            md.d = md.m == -INFINITY ? 0.f : md.d * M::exp_of(md.m - mt);
            md.m = mt;
        }
#pragma unroll
        for (int u = 0; u < U; u++)
            opaque(raw[u]);
        float s = 0.f;
#pragma unroll
        for (int u = 0; u < U; u++) {
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

template <int DT, bool ALIGNED>
__device__ float pass_max(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols)
{
    float m = -INFINITY;
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * U) {
        uint4 raw[U];
        load_step<DT, ALIGNED>(g, k0, ke, cols, raw);
#pragma unroll
        for (int u = 0; u < U; u++)
            m = fmaxf(m, chunk_max<DT>(raw[u]));
    }
    return m;
}

template <int DT, bool ALIGNED>
__device__ typename Math<DT>::Acc pass_sum(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols, float m)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    typename M::Acc acc = M::zero();
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * U) {
        uint4 raw[U];
        load_step<DT, ALIGNED>(g, k0, ke, cols, raw);
#pragma unroll
        for (int u = 0; u < U; u++) {
            float f[E];
            chunk_exp<DT>(raw[u], m, f);
#pragma unroll
            for (int e = 0; e < E; e++)
                M::add(acc, f[e]);
        }
    }
    return acc;
}

template <int DT, bool ALIGNED>
__device__ void pass_write(const RowGeom &g, int64_t kb, int64_t ke, int64_t cols, float m, float inv,
                           bool y_vec)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    const int64_t T = blockDim.x;
    for (int64_t k0 = kb + threadIdx.x; k0 < ke; k0 += T * U) {
        uint4 raw[U];
        load_step<DT, ALIGNED>(g, k0, ke, cols, raw);
#pragma unroll
        for (int u = 0; u < U; u++) {
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

// ---------------------------------------------------------------- cluster helpers

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float that CTA `rank` of this cluster keeps at the same shared-memory
// offset as `local` (distributed shared memory).
__device__ __forceinline__ float ld_peer(const float *local, uint32_t rank)
{
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

}  // namespace

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kStreamThreads)
    k_stream(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols, int y_vec)
{
    using M = Math<DT>;
    __shared__ float smax[32];
    __shared__ typename M::Acc ssum[32];
    __shared__ MD smd[32];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const RowGeom g = row_geom<DT, ALIGNED>(x, y, r, cols);
        float m, inv;
        if constexpr (DT == kF32) {
            m = block_max(pass_max<DT, ALIGNED>(g, 0, g.nch, cols), smax);
            const auto acc = block_sum<DT>(pass_sum<DT, ALIGNED>(g, 0, g.nch, cols, m), ssum);
            inv = 1.0f / M::value(acc);
        } else {
            const MD md = block_md<DT>(pass_online<DT, ALIGNED>(g, 0, g.nch, cols), smd);
            m = md.m;
            inv = 1.0f / md.d;
        }
        pass_write<DT, ALIGNED>(g, 0, g.nch, cols, m, inv, y_vec != 0);
    }
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kStreamThreads)
    k_splitk(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols, int y_vec)
{
    using M = Math<DT>;
    __shared__ float smax[32];
    __shared__ typename M::Acc ssum[32];
    __shared__ MD smd[32];
    __shared__ float pub[3];  // this CTA's partial statistics, read by its peers
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int lane = threadIdx.x & 31;
    const int64_t r = blockIdx.y;  // grid.y == rows (at most 65535)

    const RowGeom g = row_geom<DT, ALIGNED>(x, y, r, cols);
    const int64_t per = (g.nch + C - 1) / C;
    const int64_t kb = per * rank < g.nch ? per * rank : g.nch;
    const int64_t ke = kb + per < g.nch ? kb + per : g.nch;

    float m, inv;
    if constexpr (DT == kF32) {
        const float m_loc = block_max(pass_max<DT, ALIGNED>(g, kb, ke, cols), smax);
        if (threadIdx.x == 0)
            pub[0] = m_loc;
        cluster_arrive();
        cluster_wait();
        // every warp merges the C partial maxima itself (lane i reads CTA i)
        m = group_max<32>(lane < (int)C ? ld_peer(&pub[0], lane) : -INFINITY);
        const auto acc_loc = block_sum<DT>(pass_sum<DT, ALIGNED>(g, kb, ke, cols, m), ssum);
        if (threadIdx.x == 0) {
            pub[1] = acc_loc.s;
            pub[2] = acc_loc.c;
        }
        cluster_arrive();
        cluster_wait();
        CSum part = M::zero();
        if (lane < (int)C)
            part = CSum{ld_peer(&pub[1], lane), ld_peer(&pub[2], lane)};
        inv = 1.0f / M::value(group_sum<DT, 32>(part));
    } else {
        const MD md_loc = block_md<DT>(pass_online<DT, ALIGNED>(g, kb, ke, cols), smd);
        if (threadIdx.x == 0) {
            pub[0] = md_loc.m;
            pub[1] = md_loc.d;
        }
        cluster_arrive();
        cluster_wait();
        MD part{-INFINITY, 0.f};
        if (lane < (int)C)
            part = MD{ld_peer(&pub[0], lane), ld_peer(&pub[1], lane)};
        const MD md = warp_md<DT>(part);
        m = md.m;
        inv = 1.0f / md.d;
    }
    // peers may still be reading `pub`: arrive now, and wait before leaving
    cluster_arrive();
    pass_write<DT, ALIGNED>(g, kb, ke, cols, m, inv, y_vec != 0);
    cluster_wait();
}

namespace {

template <int DT, bool A>
int launch_stream_one(const Launch &l)
{
    k_stream<DT, A><<<(unsigned)l.plan.grid_x, l.plan.block_threads, 0, (cudaStream_t)l.stream>>>(
        (const char *)l.x, (char *)l.y, l.rows, l.cols, l.plan.y_vector);
    return (int)cudaGetLastError();
}

template <int DT, bool A>
int launch_splitk_one(const Launch &l)
{
    auto *kern = &k_splitk<DT, A>;
    const int C = l.plan.cluster_x;
    if (C > 8) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess)
            return (int)e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)l.plan.grid_x, (unsigned)l.plan.grid_y, 1);
    cfg.blockDim = dim3((unsigned)l.plan.block_threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)l.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, (const char *)l.x, (char *)l.y, l.rows, l.cols,
                                             (int)l.plan.y_vector);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    return (int)cudaGetLastError();
}

template <int DT>
int stream_dt(const Launch &l)
{
    return l.plan.aligned ? launch_stream_one<DT, true>(l) : launch_stream_one<DT, false>(l);
}

template <int DT>
int splitk_dt(const Launch &l)
{
    return l.plan.aligned ? launch_splitk_one<DT, true>(l) : launch_splitk_one<DT, false>(l);
}

}  // namespace

int launch_stream(const Launch &l)
{
    switch (l.dtype) {
    case kF32:
        return stream_dt<kF32>(l);
    case kF16:
        return stream_dt<kF16>(l);
    case kBF16:
        return stream_dt<kBF16>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

int launch_splitk(const Launch &l)
{
    switch (l.dtype) {
    case kF32:
        return splitk_dt<kF32>(l);
    case kF16:
        return splitk_dt<kF16>(l);
    case kBF16:
        return splitk_dt<kBF16>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace osd
