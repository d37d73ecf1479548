// k_masked.cu -- softmax(scale * x + mask) with an optional causal mask, for
// attention scores: the scale, the additive mask and the causal cut are applied
// to each element as it is loaded, so the logits never go to memory.
//
// "Softmax on DCU", section 9, lists fusing the scale and the mask into the
// softmax as the next step for attention; the Pangu-Weather profile, section 6,
// tried a bias + mask + softmax fusion on its own shapes.  Here:
//
// * z_j = scale * x_j + mask[r % mask_rows, j]; with causal_q > 0 every key
//   j > i + (cols - causal_q), i = r % causal_q, is cut (z_j = -inf).
// * fp16 / bf16: z is one fp32 FMA (its rounding, 2^-24 |z|, is far below
//   half an ulp of the output for logits of moderate size); fp32: z is kept as
//   an unevaluated pair zh + zl (the product split exactly by an FMA, the mask
//   added with TwoSum), and exp(z - m) = expf(th) (1 + tl + zl) with
//   th + tl = zh - m exactly, so fp32 keeps its 2e-6 bound.
// * ROWGROUP form (G lanes per row, the logits kept in registers) for rows of
//   up to 32 lanes x 32 floats; BLOCK form (one CTA per row, x kept packed in
//   registers, the mask chunk re-read through L1 and the logits recomputed in
//   each of the three passes) up to 2048 chunks (4 per thread x 512 threads;
//   more spills registers).
#include "common.cuh"
#include "launch.h"

namespace osd {

namespace {

struct MaskedArgs {
    const char *x;
    char *y;
    int64_t rows;
    int64_t cols;
    int y_vec;
    float scale;
    const char *mask;  // NULL: no additive mask
    int64_t mask_rows;
    int64_t causal_q;  // 0: no causal cut
};

// Visible keys of row r: j < limit.
__device__ __forceinline__ int64_t visible_limit(const MaskedArgs &a, int64_t r)
{
    return a.causal_q > 0 ? r % a.causal_q + (a.cols - a.causal_q) + 1 : a.cols;
}

// Chunk k (on x's chunk grid for this row) of the mask row `mrow`: vector load
// when the mask row sits on x's 16-byte phase and the chunk is whole, else
// element by element.
// A mask row is typically shared by many rows, so its reads may allocate in L1.
__device__ __forceinline__ uint4 ld_chunk_cached(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int DT, bool ALIGNED>
__device__ __forceinline__ uint4 load_mask_chunk(const RowGeom &g, const char *mrow, bool same_phase, int64_t k,
                                                 int64_t cols)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    if (k >= g.nch)
        return make_uint4(0, 0, 0, 0);
    const int64_t j0 = k * E - g.head;
    if (ALIGNED || (same_phase && j0 >= 0 && j0 + E <= cols))
        return ld_chunk_cached(mrow - g.head * S + 16 * k);
    return ld_partial<DT>(mrow, j0, cols);
}

// Logits of chunk k: zh (and, for fp32, the low part zl); cut slots -> -inf.
template <int DT, bool ALIGNED>
__device__ __forceinline__ void chunk_logits(const MaskedArgs &a, const RowGeom &g, int64_t k, int64_t limit,
                                             const uint4 &xc, const uint4 &mc, bool has_mask,
                                             float (&zh)[Fmt<DT>::kPerChunk], float (&zl)[Fmt<DT>::kPerChunk])
{
    constexpr int E = Fmt<DT>::kPerChunk;
    float xf[E], mf[E];
    unpack<DT>(xc, xf);
    if (has_mask)
        unpack<DT>(mc, mf);
    // row-local indices fit 32 bits: these kernels serve rows of at most 64 KiB
    const int j0 = (int)k * E - g.head;
    const int lim = (int)(k < g.nch ? limit : 0);
#pragma unroll
    for (int e = 0; e < E; e++) {
        const float mv = has_mask ? mf[e] : 0.f;
        if constexpr (DT == kF32) {
            const float ph = a.scale * xf[e];
            const float pl = fmaf(a.scale, xf[e], -ph);
            float s, err;
            two_sum(ph, mv, s, err);
            zh[e] = s;
            zl[e] = err + pl;
        } else {
            zh[e] = fmaf(a.scale, xf[e], mv);
            zl[e] = 0.f;
        }
        const int j = j0 + e;
        if (j < 0 || j >= lim) {
            zh[e] = -INFINITY;
            zl[e] = 0.f;
        }
    }
}

// exp(z - m) for a logit z = zh + zl (scaled as Math<DT>::exp_shift scales).
template <int DT>
__device__ __forceinline__ float exp_logit(float zh, float zl, float m)
{
    if constexpr (DT == kF32) {
        float th, tl;
        two_sum(zh, -m, th, tl);
        const float e = expf(th);
        const float r = tl + zl;
        return (fabsf(r) < INFINITY) ? fmaf(e, r, e) : e;
    } else {
        return Math<DT>::exp_shift(zh, m);
    }
}

}  // namespace

template <int DT, int G, int V, bool ALIGNED>
__global__ void __launch_bounds__(kRowgroupThreads) k_masked_rowgroup(const MaskedArgs a)
{
    pdl_enter();
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    const int groups = blockDim.x / G;
    const int gl = threadIdx.x & (G - 1);
    const int64_t stride = (int64_t)gridDim.x * groups;
    const bool has_mask = a.mask != nullptr;
    for (int64_t base = (int64_t)blockIdx.x * groups; base < a.rows; base += stride) {
        const int64_t r = base + threadIdx.x / G;
        const bool valid = r < a.rows;
        const int64_t rr = valid ? r : 0;
        const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, rr, a.cols);
        const char *mrow = has_mask ? a.mask + (rr % a.mask_rows) * a.cols * S : nullptr;
        const bool m_same = has_mask && ((reinterpret_cast<uintptr_t>(mrow) - reinterpret_cast<uintptr_t>(g.xr)) & 15) == 0;
        const int64_t limit = visible_limit(a, rr);

        // chunks wholly past the causal limit are neither read nor exponentiated
        float zh[V][E], zl[V][E];
        bool live[V];
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int64_t k = gl + i * G;
            live[i] = valid && k < g.nch && k * E - g.head < limit;
            const uint4 xc = live[i] ? load_chunk<DT, ALIGNED>(g, k, a.cols) : neg_inf_chunk<DT>();
            const uint4 mc = (live[i] && has_mask) ? load_mask_chunk<DT, ALIGNED>(g, mrow, m_same, k, a.cols)
                                                   : make_uint4(0, 0, 0, 0);
            chunk_logits<DT, ALIGNED>(a, g, k, limit, xc, mc, has_mask, zh[i], zl[i]);
        }
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < V; i++)
#pragma unroll
            for (int e = 0; e < E; e++)
                m = fmaxf(m, zh[i][e]);
        m = G == 32 ? warp_max_redux(m) : group_max<G>(m);
        typename M::Acc acc = M::zero();
#pragma unroll
        for (int i = 0; i < V; i++) {
            if (live[i]) {
#pragma unroll
                for (int e = 0; e < E; e++) {
                    zh[i][e] = exp_logit<DT>(zh[i][e], zl[i][e], m);
                    M::add(acc, zh[i][e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; e++)
                    zh[i][e] = 0.f;
            }
        }
        acc = group_sum<DT, G>(acc);
        const float inv = 1.0f / M::value(acc);
        if (valid) {
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int64_t k = gl + i * G;
                if (k < g.nch) {
                    float o[E];
#pragma unroll
                    for (int e = 0; e < E; e++)
                        o[e] = zh[i][e] * inv;
                    store_chunk<DT, ALIGNED>(g, k, a.cols, pack<DT>(o), a.y_vec != 0);
                }
            }
        }
    }
}

template <int DT, int V, bool ALIGNED>
__global__ void __launch_bounds__(512) k_masked_block(const MaskedArgs a)
{
    pdl_enter();
    using M = Math<DT>;
    using Acc = typename M::Acc;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    __shared__ float smax[32];
    __shared__ Acc ssum[32];
    const int T = blockDim.x, t = threadIdx.x;
    const bool has_mask = a.mask != nullptr;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, r, a.cols);
        const char *mrow = has_mask ? a.mask + (r % a.mask_rows) * a.cols * S : nullptr;
        const bool m_same = has_mask && ((reinterpret_cast<uintptr_t>(mrow) - reinterpret_cast<uintptr_t>(g.xr)) & 15) == 0;
        const int64_t limit = visible_limit(a, r);
        // x stays packed in registers; the mask chunk is re-read each pass
        // chunks wholly past the causal limit are not read (their logits are all
        // -inf; exp gives the zeros the write pass stores)
        const int lim32 = (int)limit;  // row-local: rows here are at most 32 KiB
        auto live = [&](int64_t k) { return k < g.nch && (int)k * E - g.head < lim32; };
        auto logits = [&](const uint4 &xc, int64_t k, float(&zh)[E], float(&zl)[E]) {
            const uint4 mc = (has_mask && live(k)) ? load_mask_chunk<DT, ALIGNED>(g, mrow, m_same, k, a.cols)
                                                   : make_uint4(0, 0, 0, 0);
            chunk_logits<DT, ALIGNED>(a, g, k, limit, xc, mc, has_mask, zh, zl);
        };
        uint4 xc[V];
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int64_t k = t + (int64_t)i * T;
            xc[i] = live(k) ? load_chunk<DT, ALIGNED>(g, k, a.cols) : neg_inf_chunk<DT>();
        }
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < V; i++) {
            float zh[E], zl[E];
            logits(xc[i], t + (int64_t)i * T, zh, zl);
#pragma unroll
            for (int e = 0; e < E; e++)
                m = fmaxf(m, zh[e]);
        }
        m = block_max(m, smax);
#pragma unroll
        for (int i = 0; i < V; i++)
            opaque(xc[i]);
        Acc acc = M::zero();
#pragma unroll
        for (int i = 0; i < V; i++) {
            float zh[E], zl[E];
            logits(xc[i], t + (int64_t)i * T, zh, zl);
#pragma unroll
            for (int e = 0; e < E; e++)
                M::add(acc, exp_logit<DT>(zh[e], zl[e], m));
        }
        acc = block_sum<DT>(acc, ssum);
        const float inv = 1.0f / M::value(acc);
#pragma unroll
        for (int i = 0; i < V; i++)
            opaque(xc[i]);
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int64_t k = t + (int64_t)i * T;
            if (k < g.nch) {
                float zh[E], zl[E];
                logits(xc[i], k, zh, zl);
#pragma unroll
                for (int e = 0; e < E; e++)
                    zh[e] = exp_logit<DT>(zh[e], zl[e], m) * inv;
                store_chunk<DT, ALIGNED>(g, k, a.cols, pack<DT>(zh), a.y_vec != 0);
            }
        }
    }
}

namespace {

MaskedArgs args_of(const MaskedLaunch &l)
{
    return MaskedArgs{(const char *)l.x, (char *)l.y, l.rows, l.cols, l.plan.y_vector, l.scale,
                      (const char *)l.mask, l.mask_rows, l.causal_q};
}

template <int DT, int G, int V, bool A>
int mrg_one(const MaskedLaunch &l)
{
    return launch_pdl(k_masked_rowgroup<DT, G, V, A>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT, int G, int V>
int mrg_a(const MaskedLaunch &l)
{
    return l.plan.aligned ? mrg_one<DT, G, V, true>(l) : mrg_one<DT, G, V, false>(l);
}

// V chunks per lane with the logits (fp32: two floats each) in at most 32
// registers: V <= 4 for 16-bit, V <= 4 for fp32 (4 x 4 x 2).
template <int DT, int G>
int mrg_v(const MaskedLaunch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 1:
        return mrg_a<DT, G, 1>(l);
    case 2:
        return mrg_a<DT, G, 2>(l);
    case 4:
        return mrg_a<DT, G, 4>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT>
int mrg_dt(const MaskedLaunch &l)
{
    switch (l.plan.lanes_per_row) {
    case 1:
        return l.plan.chunks_per_thread == 1 ? mrg_a<DT, 1, 1>(l) : (int)cudaErrorInvalidValue;
    case 2:
        return mrg_v<DT, 2>(l);
    case 4:
        return mrg_v<DT, 4>(l);
    case 8:
        return mrg_v<DT, 8>(l);
    case 16:
        return mrg_v<DT, 16>(l);
    case 32:
        return mrg_v<DT, 32>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT, int V, bool A>
int mblk_one(const MaskedLaunch &l)
{
    return launch_pdl(k_masked_block<DT, V, A>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT>
int mblk_dt(const MaskedLaunch &l)
{
    const bool A = l.plan.aligned != 0;
    switch (l.plan.chunks_per_thread) {
    case 2:
        return A ? mblk_one<DT, 2, true>(l) : mblk_one<DT, 2, false>(l);
    case 4:
        return A ? mblk_one<DT, 4, true>(l) : mblk_one<DT, 4, false>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT>
int masked_dt(const MaskedLaunch &l)
{
    return l.plan.variant == SOFTMAX_VARIANT_ROWGROUP ? mrg_dt<DT>(l) : mblk_dt<DT>(l);
}

}  // namespace

int launch_masked(const MaskedLaunch &l)
{
    switch (l.dtype) {
    case kF32:
        return masked_dt<kF32>(l);
    case kF16:
        return masked_dt<kF16>(l);
    case kBF16:
        return masked_dt<kBF16>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace osd
