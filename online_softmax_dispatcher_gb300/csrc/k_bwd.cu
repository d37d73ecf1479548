// k_bwd.cu -- softmax backward, dx = y * (dy - s), s = sum_k dy_k y_k, per row.
//
// The derivative of the definition (dy_i/dx_j = y_i (delta_ij - y_j)); the pages
// name the backward pass as separate work ("Softmax on DCU", section 5.4).  The
// same read-reduce-write skeleton as the forward kernels, with two inputs:
//
// * ROWGROUP: G lanes per row, V 16-byte chunks of y and of dy per lane held in
//   registers, one HBM read of each and one HBM write of dx per element.
// * BLOCK: one CTA per row, V <= 8 chunks of each per thread in registers
//   (rows of up to 512 threads x 8 chunks = 64 KiB), the chunk-to-thread map
//   shifted per row so that warp accesses start on 128-byte lines.
// * STREAM: one CTA per row of any length; a sum pass, then a pass that
//   re-reads y and dy (from L2 when the rows fit there) and writes dx.
//
// s is a compensated (TwoSum) fp32 sum for every dtype: dx_j nearly cancels
// when dy_j ~ s, and the error of s is what is left of dx_j then.  The chunk
// grid is y's.  ROWGROUP and BLOCK split a row into interior chunks (vector
// accesses of all three tensors when dy and dx share y's 16-byte phase, else
// element accesses of dy / dx) and at most 2E - 2 edge elements handled one by
// one outside the unrolled loops; STREAM peels partial edge chunks.
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

// Row phases for the short-row kernels: all rows of y, dy and dx on the 16-byte
// grid (kBwdFast); dy and dx on y's phase (kBwdSame); otherwise (kBwdOther:
// dy read and dx written element by element in the interior).
constexpr int kBwdFast = 0;
constexpr int kBwdSame = 1;
constexpr int kBwdOther = 2;

// Interior chunk q of the dy row (dyr = its start), on y's chunk grid.
template <int DT, int MODE>
__device__ __forceinline__ uint4 dy_interior(const ShortRow &g, const char *dyr, int q)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    if constexpr (MODE != kBwdOther) {
        return ld_chunk(dyr - g.head * S + ((int64_t)(g.kf + q) << 4));
    } else {
        const int j0 = (g.kf + q) * E - g.head;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            if constexpr (S == 4)
                w[i] = ld_u32(dyr + 4 * (int64_t)(j0 + i));
            else
                w[i] = ld_u16(dyr + 2 * (int64_t)(j0 + 2 * i)) | (ld_u16(dyr + 2 * (int64_t)(j0 + 2 * i + 1)) << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// dy * y products of the two 16-bit values in each word: one mixed-precision
// FMA per product (the product of two 16-bit values is exact in fp32, the
// added +0 leaves it so), without unpacking either operand.
template <int DT>
__device__ __forceinline__ void mul_pair(uint32_t yw, uint32_t dw, float &p0, float &p1)
{
    if constexpr (DT == kF16) {
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
            "fma.rn.f32.f16 %0, a0, b0, 0f00000000;\n\tfma.rn.f32.f16 %1, a1, b1, 0f00000000;\n\t}"
            : "=f"(p0), "=f"(p1)
            : "r"(yw), "r"(dw));
    } else {
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, 0f00000000;\n\tfma.rn.f32.bf16 %1, a1, b1, 0f00000000;\n\t}"
            : "=f"(p0), "=f"(p1)
            : "r"(yw), "r"(dw));
    }
}

// acc += sum of dy * y over the slots of one chunk (compensated additions;
// products of 16-bit values are exact in fp32 either way).  MIXED: one
// mixed-precision FMA per product, else unpack both and multiply; measured,
// the first is faster in the CTA-per-row kernel (unaligned [8192, 5003] fp16:
// 95 % vs 80 % of HBM bandwidth), the second in the lanes-per-row kernel
// ([65536, 512] fp16: 97 % vs 91 %).
template <int DT, bool MIXED>
__device__ __forceinline__ void dot_add(const uint4 &yc, const uint4 &dc, CSum &acc)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    if constexpr (MIXED && DT != kF32) {
        const uint32_t yw[4] = {yc.x, yc.y, yc.z, yc.w}, dw[4] = {dc.x, dc.y, dc.z, dc.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float p0, p1;
            mul_pair<DT>(yw[i], dw[i], p0, p1);
            Math<kF32>::add(acc, p0);
            Math<kF32>::add(acc, p1);
        }
    } else {
        float fy[E], fd[E];
        unpack<DT>(yc, fy);
        unpack<DT>(dc, fd);
#pragma unroll
        for (int e = 0; e < E; e++)
            Math<kF32>::add(acc, fd[e] * fy[e]);
    }
}

// dx = y * (dy - s) for one chunk: dy - s by one mixed-precision FMA per
// value for 16-bit data (the correctly rounded difference, dy unpacked by the
// FMA itself; unpacking both tensors here spills registers in the CTA-per-row
// kernel).
template <int DT>
__device__ __forceinline__ uint4 grad_chunk_fast(const uint4 &yc, const uint4 &dc, float s)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    if constexpr (DT == kF32) {
        return grad_chunk<DT>(yc, dc, s);
    } else {
        float fy[E], t[E];
        unpack<DT>(yc, fy);
        const uint32_t dw[4] = {dc.x, dc.y, dc.z, dc.w};
#pragma unroll
        for (int i = 0; i < 4; i++)
            sub_pair<DT>(dw[i], -s, t[2 * i], t[2 * i + 1]);
#pragma unroll
        for (int e = 0; e < E; e++)
            fy[e] *= t[e];
        return pack<DT>(fy);
    }
}

template <int G>
struct CsumGroup {
    __device__ __forceinline__ CSum operator()(CSum a) const { return group_csum<G>(a); }
};

struct CsumCta {
    CSum *slots;
    __device__ __forceinline__ CSum operator()(CSum a) const { return block_sum<kF32>(a, slots); }
};

// One row for a team of L threads (lane = this thread's index in it); SHIFT
// (the CTA-per-row kernel) moves the chunk map so that every 8th slot starts a
// 128-byte line, and takes the products by mixed-precision FMAs.
template <int DT, int V, int MODE, int NE, bool SHIFT, class Red>
__device__ __forceinline__ void bwd_row(const BwdArgs &a, int64_t r, bool valid, int lane, int L, Red red)
{
    constexpr int S = Fmt<DT>::kBytes;
    constexpr int PH = MODE == kBwdFast ? kPhAligned : (MODE == kBwdSame ? kPhSame : kPhOther);
    const int64_t rr = valid ? r : 0;
    const ShortRow g = short_row<DT, MODE == kBwdFast>(a.y, a.dx, rr, (int)a.cols);
    const char *dyr = a.dy + rr * a.cols * S;
    const int span = valid ? g.span : 0;
    int sh = 0;
    if constexpr (SHIFT) {
        sh = (int)(((reinterpret_cast<uintptr_t>(g.x0) >> 4) + g.kf) & 7);
        if (sh > L * V - span)
            sh = 0;
    }
    const int q0 = lane - sh;
    unsigned okm = 0;  // bit i: interior chunk q0 + i * L exists
#pragma unroll
    for (int i = 0; i < V; i++)
        okm |= (unsigned)((unsigned)(q0 + i * L) < (unsigned)span) << i;
    uint4 yc[V], dc[V];
#pragma unroll
    for (int i = 0; i < V; i++) {
        const bool ok = (okm >> i) & 1u;
        const int q = q0 + i * L;
        yc[i] = ok ? ld_chunk(g.x0 + ((int64_t)(g.kf + q) << 4)) : make_uint4(0, 0, 0, 0);
        dc[i] = ok ? dy_interior<DT, MODE>(g, dyr, q) : make_uint4(0, 0, 0, 0);
    }
    int je[NE > 0 ? NE : 1];
    float ye[NE > 0 ? NE : 1], de[NE > 0 ? NE : 1];
#pragma unroll
    for (int u = 0; u < NE; u++) {
        const int p = lane + u * L;
        je[u] = (valid && p < g.ne) ? edge_col(g, p) : -1;
        ye[u] = je[u] >= 0 ? ld_elem<DT>(g.xr, je[u]) : 0.f;
        de[u] = je[u] >= 0 ? ld_elem<DT>(dyr, je[u]) : 0.f;
    }

    // s = sum dy * y: slots past the row hold +0 on both sides and add 0
    CSum acc{0.f, 0.f};
#pragma unroll
    for (int i = 0; i < V; i++)
        dot_add<DT, SHIFT>(yc[i], dc[i], acc);
#pragma unroll
    for (int u = 0; u < NE; u++)
        Math<kF32>::add(acc, de[u] * ye[u]);
    acc = red(acc);
    const float sum = acc.s + acc.c;
#pragma unroll
    for (int i = 0; i < V; i++) {
        opaque(yc[i]);
        opaque(dc[i]);
    }
    if (!valid)
        return;
#pragma unroll
    for (int i = 0; i < V; i++)
        if ((okm >> i) & 1u)
            store_interior<DT, PH>(g, q0 + i * L, grad_chunk_fast<DT>(yc[i], dc[i], sum));
#pragma unroll
    for (int u = 0; u < NE; u++)
        if (je[u] >= 0)
            st_elem<DT>(g.yr, je[u], ye[u] * (de[u] - sum));
}

template <int DT, int G, int V, int MODE>
__global__ void __launch_bounds__(kRowgroupThreads) k_bwd_rowgroup(const BwdArgs a)
{
    pdl_enter();
    constexpr int NE = MODE == kBwdFast ? 0 : edge_slots<DT, G>();
    const int groups = blockDim.x / G;
    const int gl = threadIdx.x & (G - 1);
    const int64_t stride = (int64_t)gridDim.x * groups;
    // every thread of a CTA runs the same number of iterations, so the
    // butterflies see converged warps
    for (int64_t base = (int64_t)blockIdx.x * groups; base < a.rows; base += stride) {
        const int64_t r = base + threadIdx.x / G;
        bwd_row<DT, V, MODE, NE, false>(a, r, r < a.rows, gl, G, CsumGroup<G>{});
    }
}

// V = 8 (rows past 512 x 4 chunks, 128 registers a thread): one 512-thread CTA
// per SM, whose loads stop while it reduces and writes; the grid is one CTA
// per SM looping over rows, and each row starts by asking L2 for y and dy of
// the CTA's next row, so HBM keeps streaming through those gaps and the next
// row's loads hit L2.
template <int DT, int V, int MODE>
__global__ void __launch_bounds__(512, V >= 8 ? 1 : 2) k_bwd_block(const BwdArgs a)
{
    pdl_enter();
    __shared__ CSum slots[32];
    constexpr int NE = MODE == kBwdFast ? 0 : 1;  // >= 32 threads: one edge element each at most
    const int64_t row_bytes = a.cols * Fmt<DT>::kBytes;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        if constexpr (V >= 8) {
            const int64_t nx = r + gridDim.x;
            if (threadIdx.x == 0 && nx < a.rows) {
                prefetch_row_l2(a.y + nx * row_bytes, row_bytes);
                prefetch_row_l2(a.dy + nx * row_bytes, row_bytes);
            }
        }
        bwd_row<DT, V, MODE, NE, true>(a, r, true, threadIdx.x, blockDim.x, CsumCta{slots});
    }
}

// A 16-byte load of y or dy with an L2 policy: 1 evict-last (read again in
// this launch), 2 evict-first (its last read).
template <int POL>
__device__ __forceinline__ uint4 ld_chunk_l2(const void *p)
{
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

// Chunk k of y and of dy for a pass with L2 policy POL (0: plain loads; the
// policies apply to rows on the 16-byte grid).
template <int DT, bool ALIGNED, int POL>
__device__ __forceinline__ void load_y_dy(const RowGeom &g, const char *dyrow, bool dy_vec, int64_t k, int64_t cols,
                                          uint4 &yc, uint4 &dc)
{
    if constexpr (ALIGNED && POL != 0) {
        if (k < g.nch) {
            yc = ld_chunk_l2<POL>(g.x0 + 16 * k);
            dc = ld_chunk_l2<POL>(dyrow + 16 * k);
        } else {
            yc = neg_inf_chunk<DT>();
            dc = make_uint4(0, 0, 0, 0);
        }
    } else {
        yc = load_chunk<DT, ALIGNED>(g, k, cols);
        dc = load_other<DT, ALIGNED>(g, dyrow, dy_vec, k, cols);
    }
}

// BACK: the write pass walks the row from its end, step by step, so that it
// starts on the y and dy chunks the sum pass read last (still in L2 when the
// rows in flight outgrow it), and (rows on the 16-byte grid) the sum pass's
// loads mark their lines evict-last in L2, the write pass's evict-first; it
// changes no output bit.
template <int DT, bool ALIGNED, bool BACK>
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
            for (int u = 0; u < U; u++)
                load_y_dy<DT, ALIGNED, BACK ? 1 : 0>(g, a.dy + off, a.dy_vec != 0, k0 + u * T, a.cols, yc[u], dc[u]);
#pragma unroll
            for (int u = 0; u < U; u++)
                dot_chunk<DT, ALIGNED>(yc[u], dc[u], g, k0 + u * T, a.cols, acc);
        }
        acc = block_sum<kF32>(acc, slots);
        const float s = acc.s + acc.c;
        const int64_t span = T * U;
        const int64_t nst = (g.nch + span - 1) / span;
        for (int64_t st = 0; st < nst; st++) {
            // k >= nch loads give neutral chunks and are not stored
            const int64_t k0 = threadIdx.x + (BACK ? nst - 1 - st : st) * span;
            uint4 yc[U], dc[U];
#pragma unroll
            for (int u = 0; u < U; u++)
                load_y_dy<DT, ALIGNED, BACK ? 2 : 0>(g, a.dy + off, a.dy_vec != 0, k0 + u * T, a.cols, yc[u], dc[u]);
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

int bwd_mode(const BwdLaunch &l)
{
    if (l.plan.aligned)
        return kBwdFast;
    return (l.dy_vec && l.dx_vec) ? kBwdSame : kBwdOther;
}

template <int DT, int G, int V, int MODE>
int bwd_rowgroup_one(const BwdLaunch &l)
{
    return launch_pdl(k_bwd_rowgroup<DT, G, V, MODE>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads),
                      0, (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT, int G, int V>
int bwd_rowgroup_a(const BwdLaunch &l)
{
    switch (bwd_mode(l)) {
    case kBwdFast:
        return bwd_rowgroup_one<DT, G, V, kBwdFast>(l);
    case kBwdSame:
        return bwd_rowgroup_one<DT, G, V, kBwdSame>(l);
    default:
        return bwd_rowgroup_one<DT, G, V, kBwdOther>(l);
    }
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

template <int DT, int V, int MODE>
int bwd_block_one(const BwdLaunch &l)
{
    return launch_pdl(k_bwd_block<DT, V, MODE>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), args_of(l));
}

template <int DT, int V>
int bwd_block_mode(const BwdLaunch &l)
{
    switch (bwd_mode(l)) {
    case kBwdFast:
        return bwd_block_one<DT, V, kBwdFast>(l);
    case kBwdSame:
        return bwd_block_one<DT, V, kBwdSame>(l);
    default:
        return bwd_block_one<DT, V, kBwdOther>(l);
    }
}

template <int DT>
int bwd_block_dt(const BwdLaunch &l)
{
    switch (l.plan.chunks_per_thread) {
    case 2:
        return bwd_block_mode<DT, 2>(l);
    case 4:
        return bwd_block_mode<DT, 4>(l);
    case 8:
        return bwd_block_mode<DT, 8>(l);
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <int DT>
int bwd_stream_dt(const BwdLaunch &l)
{
    const dim3 grid((unsigned)l.plan.grid_x), block(l.plan.block_threads);
    if (l.plan.aligned)
        return l.plan.back_passes == 1
                   ? launch_pdl(k_bwd_stream<DT, true, true>, grid, block, 0, (cudaStream_t)l.stream, no_attr(),
                                args_of(l))
                   : launch_pdl(k_bwd_stream<DT, true, false>, grid, block, 0, (cudaStream_t)l.stream, no_attr(),
                                args_of(l));
    return l.plan.back_passes == 1
               ? launch_pdl(k_bwd_stream<DT, false, true>, grid, block, 0, (cudaStream_t)l.stream, no_attr(),
                            args_of(l))
               : launch_pdl(k_bwd_stream<DT, false, false>, grid, block, 0, (cudaStream_t)l.stream, no_attr(),
                            args_of(l));
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
