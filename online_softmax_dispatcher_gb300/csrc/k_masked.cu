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
// * fp32: z is kept as an unevaluated pair zh + zl (the product split exactly
//   by an FMA, the mask added with TwoSum), and exp(z - m) = expf(th)
//   (1 + tl + zl) with th + tl = zh - m exactly, so fp32 keeps its 2e-6 bound.
// * fp16 / bf16: the max pass takes z as one fp32 FMA (any shift m works:
//   softmax does not depend on it).  Its rounding moves exp(z_j - m) by up to
//   2^-24 (|z_j| + |m|) relative; an output that is not below the 16-bit range
//   has z_j >= m - 100, so while |m| < kPairFreeMax = 512 that stays under
//   2^-24 * 1124 = 6.7e-5, well inside half an fp16 ulp (2^-12 at least), and
//   the exps are taken from those logits.  Otherwise the shifted logit
//   t = z - m is formed directly from x: fma(scale, x, -m) rounds the exact
//   product minus m once (with a mask, (mask - m) is first split exactly by
//   TwoSum), so t carries an error of about 2^-24 |t|, not 2^-24 |z|, and the
//   16-bit outputs keep the bound of the plain softmax however large the
//   logits are.  The CTA-per-row form always does this (it forms the logits
//   again in each pass anyway); the lanes-per-row form sends a warp with such
//   a row down a separate, rare path (masked_row_shifted) so that the common
//   path keeps its registers.
// * ROWGROUP form (G lanes per row, the logits kept in registers) for rows of
//   up to 32 lanes x 32 floats; BLOCK form (one CTA per row, x kept packed in
//   registers, the mask chunk re-read through L1 and the logits recomputed in
//   each of the three passes) up to 2048 chunks (4 per thread x 512 threads;
//   more spills registers).
// * A row is its interior 16-byte chunks plus at most 2E - 2 edge elements
//   taken one by one; per interior chunk the number of visible values is
//   computed once: chunks wholly past the causal limit are not read, only the
//   one the limit falls in cuts values one by one.  The mask's presence and
//   the rows' 16-byte phases are template parameters.
// * Lean form (k_masked_lean): the lanes-per-row case of 16-bit rows on the
//   16-byte grid with no additive mask and a positive scale -- causal
//   attention scores -- with the max taken on packed x and no per-row 64-bit
//   division (its own account is above the kernel).
#include <type_traits>

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
    // rows, causal_q and mask_rows all below 2^31: r mod causal_q and r mod
    // mask_rows by a multiply-high with these host-made constants (the lean
    // form's account below), not by a 64-bit division
    int div32;
    uint32_t q_magic, q_shift, m_magic, m_shift;
};

// r mod d for 0 <= r < 2^31 and 1 <= d < 2^31 by the round-up multiply-high.
__device__ __forceinline__ uint32_t mod_u31(uint32_t r, uint32_t d, uint32_t magic, uint32_t shift)
{
    return r - ((__umulhi(r, magic) + r) >> shift) * d;
}

// Visible keys of row r: j < limit.
__device__ __forceinline__ int64_t visible_limit(const MaskedArgs &a, int64_t r)
{
    if (a.causal_q <= 0)
        return a.cols;
    const int64_t i = a.div32 ? (int64_t)mod_u31((uint32_t)r, (uint32_t)a.causal_q, a.q_magic, a.q_shift)
                              : r % a.causal_q;
    return i + (a.cols - a.causal_q) + 1;
}

// The mask row of row r.
__device__ __forceinline__ int64_t mask_row_of(const MaskedArgs &a, int64_t r)
{
    return a.div32 ? (int64_t)mod_u31((uint32_t)r, (uint32_t)a.mask_rows, a.m_magic, a.m_shift) : r % a.mask_rows;
}

// A mask row is typically shared by many rows, so its reads may allocate in L1.
__device__ __forceinline__ uint4 ld_chunk_cached(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Row phases: x, y and mask rows all on the 16-byte grid (kMFast); y on x's
// phase (kMSame); y on another phase (kMOther).  Off the grid, a mask row on x's
// phase is read in vectors, one on another phase element by element (decided
// per row).
constexpr int kMFast = 0;
constexpr int kMSame = 1;
constexpr int kMOther = 2;

// 16-bit rows of the lanes-per-row form whose max logit is smaller than this
// in magnitude take their exps from the single-float logits (the header's
// bound).
constexpr float kPairFreeMax = 512.f;

// exp(z - m) for an fp32 logit z = zh + zl.
__device__ __forceinline__ float exp_logit32(float zh, float zl, float m)
{
    float th, tl;
    two_sum(zh, -m, th, tl);
    const float e = expf(th);
    const float r = tl + zl;
    return (fabsf(r) < INFINITY) ? fmaf(e, r, e) : e;
}

// t = scale * x + mv - m for a 16-bit value, rounded about once relative to
// t itself (the header's account).  A -inf mask or a NaN leaves t -inf or
// NaN, as the definition does.
template <bool HAS_MASK>
__device__ __forceinline__ float shifted_logit16(float scale, float xv, float mv, float m)
{
    if constexpr (HAS_MASK) {
        float uh, ul;
        two_sum(mv, -m, uh, ul);
        const float t = fmaf(scale, xv, uh);
        return fabsf(ul) < INFINITY ? t + ul : t;
    } else {
        (void)mv;
        return fmaf(scale, xv, -m);
    }
}

// The (scaled) 16-bit exp of a shifted logit: 2^(t log2e + bias), the bias of
// Math<DT> (bf16 keeps its subnormal outputs; it cancels in y).
template <int DT>
__device__ __forceinline__ float exp_shifted16(float t)
{
    return ex2_ftz(fmaf(t, kLog2e, DT == kBF16 ? Math<kBF16>::kExpBias : 0.f));
}

// The logit of one value: zh (and the fp32 low part zl) of scale * x + mv.
template <int DT>
__device__ __forceinline__ void logit(float scale, float xv, float mv, float &zh, float &zl)
{
    if constexpr (DT == kF32) {
        const float ph = scale * xv;
        const float pl = fmaf(scale, xv, -ph);
        float s, err;
        two_sum(ph, mv, s, err);
        zh = s;
        zl = err + pl;
    } else {
        zh = fmaf(scale, xv, mv);
        zl = 0.f;
    }
}

// The mask values of interior chunk q: one vector load where the mask row
// shares x's 16-byte phase, else element by element.
template <int DT, int MODE, bool HAS_MASK>
__device__ __forceinline__ void chunk_mask(const ShortRow &g, const char *mrow, bool m_vec, int q,
                                           float (&mf)[Fmt<DT>::kPerChunk])
{
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    if constexpr (HAS_MASK) {
        if (MODE == kMFast || m_vec) {
            unpack<DT>(ld_chunk_cached(mrow - g.head * S + ((int64_t)(g.kf + q) << 4)), mf);
        } else {
            const int j0 = (g.kf + q) * E - g.head;
#pragma unroll
            for (int e = 0; e < E; e++)
                mf[e] = ld_elem<DT>(mrow, j0 + e);
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; e++)
            mf[e] = 0.f;
    }
}

// Logits of interior chunk q holding nv visible values (0 < nv <= E); slots
// past nv are cut to -inf.
template <int DT, int MODE, bool HAS_MASK>
__device__ __forceinline__ void chunk_logits(const MaskedArgs &a, const ShortRow &g, const char *mrow, bool m_vec,
                                             int q, int nv, const uint4 &xc, float (&zh)[Fmt<DT>::kPerChunk],
                                             float (&zl)[Fmt<DT>::kPerChunk])
{
    constexpr int E = Fmt<DT>::kPerChunk;
    float xf[E], mf[E];
    unpack<DT>(xc, xf);
    chunk_mask<DT, MODE, HAS_MASK>(g, mrow, m_vec, q, mf);
#pragma unroll
    for (int e = 0; e < E; e++)
        logit<DT>(a.scale, xf[e], mf[e], zh[e], zl[e]);
    if (nv < E) {
#pragma unroll
        for (int e = 0; e < E; e++)
            if (e >= nv) {
                zh[e] = -INFINITY;
                zl[e] = 0.f;
            }
    }
}

// The exps exp(z - m) of interior chunk q (0 for the slots past nv), formed
// from x: fp32 through the logit pairs, 16-bit through the shifted logits.
template <int DT, int MODE, bool HAS_MASK>
__device__ __forceinline__ void chunk_exps(const MaskedArgs &a, const ShortRow &g, const char *mrow, bool m_vec,
                                           int q, int nv, const uint4 &xc, float m,
                                           float (&ev)[Fmt<DT>::kPerChunk])
{
    constexpr int E = Fmt<DT>::kPerChunk;
    if constexpr (DT == kF32) {
        float h[E], l[E];
        chunk_logits<DT, MODE, HAS_MASK>(a, g, mrow, m_vec, q, nv, xc, h, l);
#pragma unroll
        for (int e = 0; e < E; e++)
            ev[e] = exp_logit32(h[e], l[e], m);
    } else {
        float xf[E], mf[E];
        unpack<DT>(xc, xf);
        chunk_mask<DT, MODE, HAS_MASK>(g, mrow, m_vec, q, mf);
#pragma unroll
        for (int e = 0; e < E; e++)
            ev[e] = e < nv ? exp_shifted16<DT>(shifted_logit16<HAS_MASK>(a.scale, xf[e], mf[e], m)) : 0.f;
    }
}

template <int G>
struct MaxGroup {
    __device__ __forceinline__ float operator()(float v) const { return G == 32 ? warp_max_redux(v) : group_max<G>(v); }
};

template <int DT, int G>
struct SumGroup {
    __device__ __forceinline__ typename Math<DT>::Acc operator()(typename Math<DT>::Acc a) const
    {
        return group_sum<DT, G>(a);
    }
};

template <int DT>
struct MaxSumCta {
    float *smax;
    typename Math<DT>::Acc *ssum;
    __device__ __forceinline__ float max(float v) const { return block_max(v, smax); }
    __device__ __forceinline__ typename Math<DT>::Acc sum(typename Math<DT>::Acc a) const
    {
        return block_sum<DT>(a, ssum);
    }
};

template <int DT, int G>
struct MaxSumGroup {
    __device__ __forceinline__ float max(float v) const { return MaxGroup<G>{}(v); }
    __device__ __forceinline__ typename Math<DT>::Acc sum(typename Math<DT>::Acc a) const
    {
        return SumGroup<DT, G>{}(a);
    }
};

// The rest of a 16-bit row for the lanes-per-row form once its max m is known
// and at least kPairFreeMax in magnitude: every visible value again, from x
// read element by element (from L2: the row was just loaded, and none of its
// output is stored yet, so an in-place call still reads x), its exp taken
// from the shifted logit -- once for the sum, once for the output.  Out of
// line and with only values as arguments, so that this rare path adds no
// registers or local memory to the common one.  Lane `lane` of a team of L
// takes elements lane, lane + L, ...  Called by whole warps.
template <int DT, bool HAS_MASK, class Red>
__device__ __noinline__ void masked_row_shifted(const char *xr, char *yr, const char *mrow, int cols, int lim,
                                                float scale, float m, int lane, int L, bool valid, Red red)
{
    float acc = 0.f;
    for (int j = lane; j < lim; j += L)
        acc += exp_shifted16<DT>(
            shifted_logit16<HAS_MASK>(scale, ld_elem<DT>(xr, j), HAS_MASK ? ld_elem<DT>(mrow, j) : 0.f, m));
    acc = red.sum(acc);
    const float inv = 1.0f / acc;
    if (!valid)
        return;
    for (int j = lane; j < cols; j += L) {
        const float e = j < lim ? exp_shifted16<DT>(shifted_logit16<HAS_MASK>(
                                      scale, ld_elem<DT>(xr, j), HAS_MASK ? ld_elem<DT>(mrow, j) : 0.f, m))
                                : 0.f;
        st_elem<DT>(yr, j, e * inv);
    }
}

// One row for a team of L threads.  KEEP: the logits, then their exps, stay
// in registers (lanes per row); else x stays packed and the exps are formed
// again for the output (CTA per row, with the 128-byte-line chunk map).  Interior chunks wholly past the causal limit are neither read nor
// exponentiated; only the chunk the limit falls in tests its values one by
// one.
template <int DT, int V, int MODE, bool HAS_MASK, int NE, bool KEEP, class Red>
__device__ __forceinline__ void masked_row(const MaskedArgs &a, int64_t r, bool valid, int lane, int L, Red red)
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    constexpr int PH = MODE == kMFast ? kPhAligned : (MODE == kMSame ? kPhSame : kPhOther);
    constexpr bool KEEP_Z = KEEP && DT == kF32;  // fp32 logit pairs kept from the max pass
    const int64_t rr = valid ? r : 0;
    const ShortRow g = short_row<DT, MODE == kMFast>(a.x, a.y, rr, (int)a.cols);
    const char *mrow = HAS_MASK ? a.mask + mask_row_of(a, rr) * a.cols * S : nullptr;
    const bool m_vec = HAS_MASK && ((reinterpret_cast<uintptr_t>(mrow) - reinterpret_cast<uintptr_t>(g.xr)) & 15) == 0;
    // row-local indices fit 32 bits: these kernels serve rows of at most 64 KiB
    const int lim = valid ? (int)visible_limit(a, rr) : 0;
    const int span = valid ? g.span : 0;
    int sh = 0;
    if constexpr (!KEEP) {
        sh = (int)(((reinterpret_cast<uintptr_t>(g.x0) >> 4) + g.kf) & 7);
        if (sh > L * V - span)
            sh = 0;
    }
    const int q0 = lane - sh;
    // visible values of interior chunk i (0: absent or wholly cut)
    int nv[V];
    uint4 xc[V];
#pragma unroll
    for (int i = 0; i < V; i++) {
        const int q = q0 + i * L;
        const int j0 = (g.kf + q) * E - g.head;
        const int left = lim - j0;
        nv[i] = (unsigned)q < (unsigned)span ? (left < 0 ? 0 : (left > E ? E : left)) : 0;
        xc[i] = nv[i] > 0 ? ld_chunk(g.x0 + ((int64_t)(g.kf + q) << 4)) : make_uint4(0, 0, 0, 0);
    }
    // edge elements: fp32 keeps the logit pair (eh, el), 16-bit the value and
    // its mask value; ev the exp once m is known
    int je[NE > 0 ? NE : 1];
    float eh[NE > 0 ? NE : 1], el[NE > 0 ? NE : 1];
    float m = -INFINITY;
#pragma unroll
    for (int u = 0; u < NE; u++) {
        const int p = lane + u * L;
        je[u] = (valid && p < g.ne) ? edge_col(g, p) : -1;
        eh[u] = -INFINITY;
        el[u] = 0.f;
        if (je[u] >= 0 && je[u] < lim) {
            const float xv = ld_elem<DT>(g.xr, je[u]), mv = HAS_MASK ? ld_elem<DT>(mrow, je[u]) : 0.f;
            if constexpr (DT == kF32) {
                logit<DT>(a.scale, xv, mv, eh[u], el[u]);
                m = fmaxf(m, eh[u]);
            } else {
                eh[u] = xv;
                el[u] = mv;
                float zh, zl;
                logit<DT>(a.scale, xv, mv, zh, zl);
                m = fmaxf(m, zh);
            }
        }
    }

    float zh[KEEP ? V : 1][E], zl[KEEP_Z ? V : 1][E];
#pragma unroll
    for (int i = 0; i < V; i++) {
        if (nv[i] > 0) {
            float h[E], l[E];
            chunk_logits<DT, MODE, HAS_MASK>(a, g, mrow, m_vec, q0 + i * L, nv[i], xc[i], h, l);
#pragma unroll
            for (int e = 0; e < E; e++) {
                m = fmaxf(m, h[e]);
                if constexpr (KEEP)
                    zh[i][e] = h[e];
                if constexpr (KEEP_Z)
                    zl[i][e] = l[e];
            }
        }
    }
    m = red.max(m);
    if constexpr (KEEP && DT != kF32) {
        // warp-uniform, so that the reductions inside stay converged
        if (__any_sync(0xffffffffu, !(fabsf(m) < kPairFreeMax))) {
            masked_row_shifted<DT, HAS_MASK>(g.xr, g.yr, mrow, (int)a.cols, lim, a.scale, m, lane, L, valid, red);
            return;
        }
    }
    // 16-bit rows of the lanes-per-row form: exp(zh - m) = 2^(zh log2e + c)
    // with c = bias - m log2e formed once (its rounding scales the whole row's
    // exps by one factor, which the normalisation cancels)
    const float c16 = DT == kBF16 ? Math<kBF16>::kExpBias - m * kLog2e : -m * kLog2e;

    typename M::Acc acc = M::zero();
#pragma unroll
    for (int i = 0; i < V; i++) {
        if (nv[i] > 0) {
            float ev[E];
            if constexpr (KEEP_Z) {
#pragma unroll
                for (int e = 0; e < E; e++)
                    ev[e] = exp_logit32(zh[i][e], zl[i][e], m);
            } else if constexpr (KEEP) {
#pragma unroll
                for (int e = 0; e < E; e++)
                    ev[e] = ex2_ftz(fmaf(zh[i][e], kLog2e, c16));
            } else {
                opaque(xc[i]);
                chunk_exps<DT, MODE, HAS_MASK>(a, g, mrow, m_vec, q0 + i * L, nv[i], xc[i], m, ev);
            }
#pragma unroll
            for (int e = 0; e < E; e++) {
                M::add(acc, ev[e]);
                if constexpr (KEEP)
                    zh[i][e] = ev[e];
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NE; u++) {
        if constexpr (DT == kF32)
            eh[u] = je[u] >= 0 ? exp_logit32(eh[u], el[u], m) : 0.f;
        else
            eh[u] = (je[u] >= 0 && je[u] < lim) ? exp_shifted16<DT>(shifted_logit16<HAS_MASK>(a.scale, eh[u], el[u], m))
                                                : 0.f;
        M::add(acc, eh[u]);
    }
    acc = red.sum(acc);
    const float inv = 1.0f / M::value(acc);
    if (!valid)
        return;
#pragma unroll
    for (int i = 0; i < V; i++) {
        const int q = q0 + i * L;
        if ((unsigned)q < (unsigned)span) {
            float o[E];
            if (nv[i] > 0) {
                if constexpr (KEEP) {
#pragma unroll
                    for (int e = 0; e < E; e++)
                        o[e] = zh[i][e] * inv;
                } else {
                    opaque(xc[i]);
                    chunk_exps<DT, MODE, HAS_MASK>(a, g, mrow, m_vec, q, nv[i], xc[i], m, o);
#pragma unroll
                    for (int e = 0; e < E; e++)
                        o[e] *= inv;
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; e++)
                    o[e] = 0.f * inv;  // a cut chunk: exp(-inf) = 0 (NaN for a row with no visible key)
            }
            store_interior<DT, PH>(g, q, pack<DT>(o));
        }
    }
#pragma unroll
    for (int u = 0; u < NE; u++)
        if (je[u] >= 0)
            st_elem<DT>(g.yr, je[u], eh[u] * inv);
}

}  // namespace

template <int DT, int G, int V, int MODE, bool HAS_MASK>
__global__ void __launch_bounds__(kRowgroupThreads) k_masked_rowgroup(const MaskedArgs a)
{
    pdl_enter();
    constexpr int NE = MODE == kMFast ? 0 : edge_slots<DT, G>();
    const int groups = blockDim.x / G;
    const int gl = threadIdx.x & (G - 1);
    const int64_t stride = (int64_t)gridDim.x * groups;
    // every thread of a CTA runs the same number of iterations, so the
    // butterflies see converged warps
    for (int64_t base = (int64_t)blockIdx.x * groups; base < a.rows; base += stride) {
        const int64_t r = base + threadIdx.x / G;
        masked_row<DT, V, MODE, HAS_MASK, NE, true>(a, r, r < a.rows, gl, G, MaxSumGroup<DT, G>{});
    }
}

template <int DT, int V, int MODE, bool HAS_MASK>
__global__ void __launch_bounds__(512) k_masked_block(const MaskedArgs a)
{
    pdl_enter();
    __shared__ float smax[32];
    __shared__ typename Math<DT>::Acc ssum[32];
    constexpr int NE = MODE == kMFast ? 0 : 1;  // >= 32 threads: one edge element each at most
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        masked_row<DT, V, MODE, HAS_MASK, NE, false>(a, r, true, threadIdx.x, blockDim.x,
                                                     MaxSumCta<DT>{smax, ssum});
}

// ---------------------------------------------------------------- lean form
//
// The common attention case with its own, smaller instruction budget: 16-bit
// rows on the 16-byte grid, no additive mask, 0 < scale < inf, fewer than
// 2^31 rows.  The general kernel above spends ~19 instructions per element
// there and is bound by instruction issue, not by HBM.  Here:
// * scale > 0 makes fl(scale * x) non-decreasing in x, so the row's max
//   logit is fl(scale * max_j x_j): the max is taken on the packed 16-bit
//   pairs (one instruction per two values), the cut values of the chunk the
//   causal limit falls in first set to -inf in the packed words.  This is the
//   same m the general kernel finds.
// * exp(z_j - m) = 2^(x_j * fl(scale log2e) + c), c = bias - fl(m log2e)
//   formed once per row: c's rounding is common to the row (the
//   normalisation cancels it), and per element the exponent carries about
//   2^-24 (|z_j| log2e + |t_j|) -- with |m| < kPairFreeMax and z_j >= m - 100
//   for any output above the 16-bit range, below 2^-24 * 1030 = 6.2e-5
//   (4.3e-5 relative in the exp), the same class as the general kernel's
//   bound.  Rows with |m| >= kPairFreeMax go down masked_row_shifted.
// * r mod causal_q by a multiply-high with a host-made constant: the
//   round-up method of Granlund and Montgomery, "Division by invariant
//   integers using multiplication" (PLDI 1994), for dividends below 2^31:
//   with l = ceil(log2 q) and M = floor(2^32 (2^l - q) / q) + 1,
//   floor(r / q) = (umulhi(M, r) + r) >> l.
struct LeanArgs {
    const char *x;
    char *y;
    uint32_t rows;
    int cols;
    float scale;
    int causal_q;  // 0: no causal cut
    uint32_t q_magic;
    uint32_t q_shift;
};

// Slots nv.. of a chunk set to -inf (0 < nv < E), on the packed words.
template <int DT>
__device__ __forceinline__ uint4 cut_chunk(const uint4 &c, int nv)
{
    constexpr uint32_t ni = Fmt<DT>::kNegInf;
    uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        if (2 * k + 1 >= nv)
            w[k] = 2 * k < nv ? ((w[k] & 0xFFFFu) | (ni << 16)) : (ni | (ni << 16));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Max of the V chunks' slots as a float: packed pairwise maxima, one
// conversion at the end (the max of representable values is exact).
template <int DT, int V>
__device__ __forceinline__ float packed_max(const uint4 (&xc)[V])
{
    using H2 = typename std::conditional<DT == kF16, __half2, __nv_bfloat162>::type;
    H2 h[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint32_t w = k == 0 ? xc[0].x : k == 1 ? xc[0].y : k == 2 ? xc[0].z : xc[0].w;
        *reinterpret_cast<uint32_t *>(&h[k]) = w;
    }
#pragma unroll
    for (int i = 1; i < V; i++) {
        const uint32_t w[4] = {xc[i].x, xc[i].y, xc[i].z, xc[i].w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            H2 t;
            *reinterpret_cast<uint32_t *>(&t) = w[k];
            h[k] = __hmax2(h[k], t);
        }
    }
    const H2 r = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return fmaxf(__low2float(r), __high2float(r));
}

template <int DT, int G, int V>
__global__ void __launch_bounds__(kRowgroupThreads) k_masked_lean(const LeanArgs a)
{
    pdl_enter();
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    const int groups = blockDim.x / G;
    const int lane = threadIdx.x & (G - 1);
    const float sl2e = a.scale * kLog2e;
    const int span = a.cols / E;  // rows on the 16-byte grid: every chunk is interior
    const int64_t stride = (int64_t)gridDim.x * groups;
    // every thread of a CTA runs the same number of iterations, so the
    // butterflies see converged warps
    for (int64_t base = (int64_t)blockIdx.x * groups; base < a.rows; base += stride) {
        const int64_t r64 = base + threadIdx.x / G;
        const bool valid = r64 < a.rows;
        const uint32_t r = valid ? (uint32_t)r64 : 0u;
        int lim = 0;
        if (valid) {
            lim = a.cols;
            if (a.causal_q > 0) {
                const uint32_t quo = (__umulhi(r, a.q_magic) + r) >> a.q_shift;
                lim = (int)(r - quo * (uint32_t)a.causal_q) + (a.cols - a.causal_q) + 1;
            }
        }
        const char *xr = a.x + (int64_t)r * a.cols * S;
        char *yr = a.y + (int64_t)r * a.cols * S;
        uint4 xc[V];
        int nv[V];
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int q = lane + i * G;
            const int left = lim - q * E;
            nv[i] = q < span ? (left < 0 ? 0 : (left > E ? E : left)) : 0;
            xc[i] = nv[i] > 0 ? ld_chunk(xr + ((int64_t)q << 4)) : neg_inf_chunk<DT>();
            if (nv[i] > 0 && nv[i] < E)
                xc[i] = cut_chunk<DT>(xc[i], nv[i]);
        }
        const float mz = a.scale * MaxGroup<G>{}(packed_max<DT, V>(xc));
        // warp-uniform, so that the reductions inside stay converged
        if (__any_sync(0xffffffffu, valid && !(fabsf(mz) < kPairFreeMax))) {
            masked_row_shifted<DT, false>(xr, yr, nullptr, a.cols, lim, a.scale, mz, lane, G, valid,
                                          MaxSumGroup<DT, G>{});
            continue;
        }
        const float c = Math<DT>::kExpBias - mz * kLog2e;
        float ev[V][E];
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < V; i++) {
            if (nv[i] > 0) {
                float xf[E];
                unpack<DT>(xc[i], xf);
#pragma unroll
                for (int e = 0; e < E; e++) {
                    ev[i][e] = ex2_ftz(fmaf(xf[e], sl2e, c));  // a cut slot: 2^-inf = 0
                    acc += ev[i][e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; e++)
                    ev[i][e] = 0.f;
            }
        }
        acc = SumGroup<DT, G>{}(acc);
        const float inv = 1.0f / acc;
        if (valid) {
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int q = lane + i * G;
                if (q < span) {
                    float o[E];
#pragma unroll
                    for (int e = 0; e < E; e++)
                        o[e] = ev[i][e] * inv;
                    st_chunk_stream(yr + ((int64_t)q << 4), pack<DT>(o));
                }
            }
        }
    }
}

namespace {

// The multiply-high constants of the round-up method for a divisor 1 <= d <
// 2^31 (shift = ceil(log2 d), magic = floor(2^32 (2^shift - d) / d) + 1; d = 1:
// magic 1, shift 0, which gives r).
void magic_u31(int64_t d, uint32_t &magic, uint32_t &shift)
{
    magic = 1u;
    shift = 0u;
    if (d <= 1)
        return;
    const uint64_t q = (uint64_t)d;
    uint32_t lg = 0;
    while ((1ull << lg) < q)
        lg++;
    shift = lg;
    magic = (uint32_t)((((1ull << lg) - q) << 32) / q + 1);
}

MaskedArgs args_of(const MaskedLaunch &l)
{
    MaskedArgs a{(const char *)l.x, (char *)l.y, l.rows, l.cols, l.plan.y_vector, l.scale,
                 (const char *)l.mask, l.mask_rows, l.causal_q, 0, 1u, 0u, 1u, 0u};
    a.div32 = l.rows <= INT32_MAX && l.causal_q <= INT32_MAX && (l.mask == nullptr || l.mask_rows <= INT32_MAX);
    if (a.div32) {
        magic_u31(l.causal_q, a.q_magic, a.q_shift);
        if (l.mask)
            magic_u31(l.mask_rows, a.m_magic, a.m_shift);
    }
    return a;
}

int mode_of(const MaskedLaunch &l)
{
    if (l.plan.aligned)
        return kMFast;
    return l.plan.y_vector ? kMSame : kMOther;
}

template <int DT, int G, int V, int MODE, bool HM>
int mrg_one(const MaskedLaunch &l)
{
    return launch_pdl(k_masked_rowgroup<DT, G, V, MODE, HM>, dim3((unsigned)l.plan.grid_x),
                      dim3(l.plan.block_threads), 0, (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT, int G, int V, int MODE>
int mrg_m(const MaskedLaunch &l)
{
    return l.mask ? mrg_one<DT, G, V, MODE, true>(l) : mrg_one<DT, G, V, MODE, false>(l);
}

template <int DT, int G, int V>
int mrg_a(const MaskedLaunch &l)
{
    switch (mode_of(l)) {
    case kMFast:
        return mrg_m<DT, G, V, kMFast>(l);
    case kMSame:
        return mrg_m<DT, G, V, kMSame>(l);
    default:
        return mrg_m<DT, G, V, kMOther>(l);
    }
}

// V chunks per lane with the logits (fp32: two floats each) in at most 32
// registers: V <= 4.
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

template <int DT, int V, int MODE, bool HM>
int mblk_one(const MaskedLaunch &l)
{
    return launch_pdl(k_masked_block<DT, V, MODE, HM>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads),
                      0, (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT, int V, int MODE>
int mblk_m(const MaskedLaunch &l)
{
    return l.mask ? mblk_one<DT, V, MODE, true>(l) : mblk_one<DT, V, MODE, false>(l);
}

template <int DT, int V>
int mblk_a(const MaskedLaunch &l)
{
    switch (mode_of(l)) {
    case kMFast:
        return mblk_m<DT, V, kMFast>(l);
    case kMSame:
        return mblk_m<DT, V, kMSame>(l);
    default:
        return mblk_m<DT, V, kMOther>(l);
    }
}

template <int DT>
int mblk_dt(const MaskedLaunch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 2:
        return mblk_a<DT, 2>(l);
    case 4:
        return mblk_a<DT, 4>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

// The lean form's conditions: a lanes-per-row plan for 16-bit rows on the
// 16-byte grid, no additive mask, a positive finite scale, and row indices and
// causal_q below 2^31 (32-bit division by the host's constant).
bool lean_fits(const MaskedLaunch &l)
{
    return l.dtype != kF32 && l.plan.variant == SOFTMAX_VARIANT_ROWGROUP && l.plan.aligned && l.mask == nullptr &&
           l.scale > 0.f && l.scale <= 3.4028234663852886e38f && l.rows <= INT32_MAX && l.causal_q <= INT32_MAX &&
           l.cols <= INT32_MAX;
}

LeanArgs lean_args_of(const MaskedLaunch &l)
{
    LeanArgs a{(const char *)l.x, (char *)l.y, (uint32_t)l.rows, (int)l.cols, l.scale, (int)l.causal_q, 1u, 0u};
    magic_u31(l.causal_q, a.q_magic, a.q_shift);
    return a;
}

template <int DT, int G, int V>
int lean_one(const MaskedLaunch &l)
{
    return launch_pdl(k_masked_lean<DT, G, V>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), lean_args_of(l));
}

template <int DT, int G>
int lean_v(const MaskedLaunch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 1:
        return lean_one<DT, G, 1>(l);
    case 2:
        return lean_one<DT, G, 2>(l);
    case 4:
        return lean_one<DT, G, 4>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT>
int lean_dt(const MaskedLaunch &l)
{
    switch (l.plan.lanes_per_row) {
    case 1:
        return l.plan.chunks_per_thread == 1 ? lean_one<DT, 1, 1>(l) : (int)cudaErrorInvalidValue;
    case 2:
        return lean_v<DT, 2>(l);
    case 4:
        return lean_v<DT, 4>(l);
    case 8:
        return lean_v<DT, 8>(l);
    case 16:
        return lean_v<DT, 16>(l);
    case 32:
        return lean_v<DT, 32>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT>
int masked_dt(const MaskedLaunch &l)
{
    if constexpr (DT != kF32) {
        if (lean_fits(l))
            return lean_dt<DT>(l);
    }
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
