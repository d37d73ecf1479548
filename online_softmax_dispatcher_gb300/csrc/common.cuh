// common.cuh -- device primitives shared by the softmax kernels (sm_103a).
//
// * 16-byte chunk I/O: every kernel moves a row as 16-byte chunks laid on the
//   16-byte address grid.  A row whose start or end is not on that grid has a
//   partial first / last chunk; those slots are read with scalar loads and the
//   out-of-row slots are filled with -inf, which contributes exp(-inf) = 0
//   (the vector-plus-scalar-edge technique of the InfiniTrain BF16 kernel PR,
//   "AlignedVector" with an alignment check and a scalar tail, rebuilt as a
//   per-row head/tail peel so that unaligned rows keep the vector body).
// * dtype decode / RNE encode: fp32, fp16 (IEEE binary16), bf16.  Output
//   rounding is round-to-nearest-even, as the half kernels of "[CUDA] safe
//   online softmax" (section 2.1) and "Softmax on DCU" (section 4.5) do.
// * exp: for fp16 / bf16 outputs exp(x - m) = 2^((x - m) * log2 e) on the SFU
//   (ex2.approx.ftz: results below 2^-126 flush to zero); its ~2^-22 relative
//   error is far below half an ulp of either 16-bit format.  bf16 reaches
//   subnormal outputs, so its exps are taken pre-scaled by 2^64 (the argument
//   is (x - m) log2 e + 64; the scale cancels in y) and only terms below
//   2^-190, which bf16 rounds to 0 anyway, flush (Math<DT> below).  fp16
//   outputs are 0 below 2^-25 and need no scale.  For fp32 outputs the shift
//   t = x - m is split exactly into t + r (Knuth's TwoSum) and
//   exp(x - m) = expf(t) * (1 + r), which keeps the result within a few fp32
//   ulps even when |x - m| is in the hundreds.
// * sums: fp32 accumulation everywhere ("Softmax on DCU", section 4.5); for
//   fp32 outputs the sum is a compensated (s, c) pair merged with TwoSum so a
//   row of 2^22 terms stays within ~2 ulps.
// * reductions: xor-butterfly warp shuffles ("[CUDA] safe online softmax",
//   section 2.1.1) -- every lane ends with the identical value because each
//   merge is commutative -- then one shared-memory slot per warp.
// * (m, d) merge for the online form: m = max(m1, m2),
//   d = d1 e^(m1 - m) + d2 e^(m2 - m) ("[CUDA] safe online softmax", section 1,
//   safe_online_softmax, and its warp reduce in section 2.1).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace osd {

enum : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

template <int DT>
struct Fmt;
template <>
struct Fmt<kF32> {
    static constexpr int kBytes = 4;  // element size
    static constexpr int kPerChunk = 4;  // elements per 16-byte chunk
};
template <>
struct Fmt<kF16> {
    static constexpr int kBytes = 2;
    static constexpr int kPerChunk = 8;
    static constexpr uint32_t kNegInf = 0xFC00u;
};
template <>
struct Fmt<kBF16> {
    static constexpr int kBytes = 2;
    static constexpr int kPerChunk = 8;
    static constexpr uint32_t kNegInf = 0xFF80u;
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kNegInfF32 = 0xFF800000u;

// ---------------------------------------------------------------- global memory

// 16-byte load, no L1 allocation (x is read once per pass).  Coherent, not
// the read-only path: an in-place call (y == x) writes the tensor it reads,
// which the read-only path does not allow within one kernel (measured: the
// same speed).
__device__ __forceinline__ uint4 ld_chunk(const void *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_chunk(void *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// An L2 access policy that marks lines evict-first.
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// A whole chunk of output that nothing reads again in this launch: stored with
// the evict-first policy, so the line leaves L2 (and reaches HBM) early rather
// than crowding lines still being read.  Only for rows on the 16-byte grid: a
// chunk of a row off the grid shares its sector with element stores of the
// next row, and evicting it half written costs a partial write (measured:
// [65536, 512] fp16 93.8 -> 95.6 %, its backward 96.8 -> 99.0 %; rows off the
// grid, [8192, 5003] fp16, 86.4 -> 85.1 % when they used it too).
__device__ __forceinline__ void st_chunk_stream(void *p, const uint4 &v)
{
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(l2_evict_first())
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_u16(const void *p)
{
    unsigned short v;
    asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_u32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_u16(void *p, uint32_t v)
{
    asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"((unsigned short)v) : "memory");
}

__device__ __forceinline__ void st_u32(void *p, uint32_t v)
{
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- launch

// Programmatic dependent launch.  Every kernel of the library starts with
// pdl_enter(): it lets the next kernel in the stream be scheduled once every
// CTA of this grid has started (the next grid then fills this one's tail
// instead of waiting for it to drain), and waits until the previous kernel in
// the stream has completed and its writes are visible, before this kernel's
// first global memory access.  Without a programmatic predecessor the wait
// returns at once.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kernel` on `stream` with programmatic stream serialisation allowed
// (see pdl_enter); `extra` adds one more launch attribute (a cluster shape)
// when its id is not cudaLaunchAttributeIgnore.  Returns the launch status and
// leaves no pending launch error behind.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      cudaLaunchAttribute extra, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (extra.id != cudaLaunchAttributeIgnore)
        attr[cfg.numAttrs++] = extra;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess)
        (void)cudaGetLastError();
    return (int)e;
}

inline cudaLaunchAttribute no_attr()
{
    cudaLaunchAttribute a = {};
    a.id = cudaLaunchAttributeIgnore;
    return a;
}

// ---------------------------------------------------------------- decode / encode

template <int DT>
__device__ __forceinline__ void unpack(const uint4 &c, float (&f)[Fmt<DT>::kPerChunk])
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    if constexpr (DT == kF32) {
#pragma unroll
        for (int i = 0; i < 4; i++)
            f[i] = __uint_as_float(w[i]);
    } else if constexpr (DT == kF16) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            __half2 h;
            *reinterpret_cast<uint32_t *>(&h) = w[i];
            const float2 p = __half22float2(h);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    } else {
        // bf16 is the top half of an fp32 pattern: exact by shifting.
#pragma unroll
        for (int i = 0; i < 4; i++) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

template <int DT>
__device__ __forceinline__ uint4 pack(const float (&f)[Fmt<DT>::kPerChunk])
{
    uint32_t w[4];
    if constexpr (DT == kF32) {
#pragma unroll
        for (int i = 0; i < 4; i++)
            w[i] = __float_as_uint(f[i]);
    } else if constexpr (DT == kF16) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// A chunk whose every slot is -inf in the dtype.
template <int DT>
__device__ __forceinline__ uint4 neg_inf_chunk()
{
    if constexpr (DT == kF32) {
        return make_uint4(kNegInfF32, kNegInfF32, kNegInfF32, kNegInfF32);
    } else {
        const uint32_t w = Fmt<DT>::kNegInf | (Fmt<DT>::kNegInf << 16);
        return make_uint4(w, w, w, w);
    }
}

// ---------------------------------------------------------------- row geometry

// Where a row sits on the 16-byte grid.  Chunk k of the row covers element
// indices [k * E - head, k * E - head + E); chunk 0 starts at `x0`.
struct RowGeom {
    const char *x0;   // 16-byte aligned address of chunk 0 of the x row
    char *y0;         // same for y (meaningful when y rows share x rows' phase)
    const char *xr;   // x row start
    char *yr;         // y row start
    int head;         // elements of chunk 0 that precede the row (0 when aligned)
    int64_t nch;      // chunks covering the row
    int64_t kf, kl;   // chunks [kf, kl) lie wholly inside the row
};

template <int DT, bool ALIGNED>
__device__ __forceinline__ RowGeom row_geom(const char *x, char *y, int64_t r, int64_t cols)
{
    constexpr int S = Fmt<DT>::kBytes;
    const int64_t row_bytes = cols * S;
    RowGeom g;
    g.xr = x + r * row_bytes;
    g.yr = y + r * row_bytes;
    if constexpr (ALIGNED) {
        g.x0 = g.xr;
        g.y0 = g.yr;
        g.head = 0;
        g.nch = row_bytes >> 4;
        g.kf = 0;
        g.kl = g.nch;
    } else {
        const uintptr_t a = reinterpret_cast<uintptr_t>(g.xr);
        const int lead = (int)(a & 15);
        g.x0 = g.xr - lead;
        g.y0 = g.yr - lead;
        g.head = lead / S;
        g.nch = (lead + row_bytes + 15) >> 4;
        g.kf = lead ? 1 : 0;
        g.kl = ((lead + row_bytes) & 15) ? g.nch - 1 : g.nch;
    }
    return g;
}

// A row of fewer than 2^31 bytes split into interior chunks and edge
// elements, in 32-bit arithmetic (the lanes-per-row and CTA-per-row kernels,
// which set this up once per row in every thread).  The interior chunks
// kf .. kf + span - 1 (chunk k at x0 + 16 k) lie wholly inside the row and are
// read and written as 16-byte vectors; the at most 2E - 2 edge elements
// [0, enh) and [et0, cols) are read and written one by one.  Aligned rows are
// all interior.
struct ShortRow {
    const char *x0;  // 16-byte aligned address of chunk 0 of the x row
    char *y0;        // same for y (meaningful when y rows share x rows' phase)
    const char *xr;  // x row start
    char *yr;        // y row start
    int head;        // elements of chunk 0 that precede the row
    int kf, span;    // first interior chunk, interior chunks
    int enh, et0, ne;  // edge elements: head count, tail start, total
};

template <int DT, bool ALIGNED>
__device__ __forceinline__ ShortRow short_row(const char *x, char *y, int64_t r, int cols)
{
    constexpr int S = Fmt<DT>::kBytes;
    constexpr int E = Fmt<DT>::kPerChunk;
    const int rb = cols * S;
    ShortRow g;
    g.xr = x + r * rb;
    g.yr = y + r * rb;
    if constexpr (ALIGNED) {
        g.x0 = g.xr;
        g.y0 = g.yr;
        g.head = 0;
        g.kf = 0;
        g.span = rb >> 4;
        g.enh = 0;
        g.et0 = cols;
        g.ne = 0;
    } else {
        const int lead = (int)(reinterpret_cast<uintptr_t>(g.xr) & 15);
        g.x0 = g.xr - lead;
        g.y0 = g.yr - lead;
        g.head = lead / S;
        g.kf = lead != 0;
        const int kl = (lead + rb) >> 4;  // chunks before kl end inside the row
        // a row inside one chunk with both edges partial has kl < kf: no interior
        g.span = kl > g.kf ? kl - g.kf : 0;
        g.enh = g.kf ? (E - g.head < cols ? E - g.head : cols) : 0;
        const int t0 = kl * E - g.head;
        g.et0 = t0 > g.enh ? t0 : g.enh;
        g.ne = g.enh + (cols - g.et0);
    }
    return g;
}

// Scalar read of the in-row slots of a partial chunk; other slots are -inf.
template <int DT>
__device__ __forceinline__ uint4 ld_partial(const char *xr, int64_t j0, int64_t cols)
{
    uint32_t w[4];
    if constexpr (DT == kF32) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int64_t j = j0 + e;
            w[e] = (j >= 0 && j < cols) ? ld_u32(xr + 4 * j) : kNegInfF32;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int64_t j = j0 + 2 * i;
            const uint32_t lo = (j >= 0 && j < cols) ? ld_u16(xr + 2 * j) : Fmt<DT>::kNegInf;
            const uint32_t hi = (j + 1 >= 0 && j + 1 < cols) ? ld_u16(xr + 2 * (j + 1)) : Fmt<DT>::kNegInf;
            w[i] = lo | (hi << 16);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT>
__device__ __forceinline__ uint4 mask_chunk(const uint4 &c, int64_t t0, int64_t lo, int64_t hi);

// Load chunk k of a row (k may be >= nch: then an all -inf chunk).  Every
// chunk k < nch is one aligned 16-byte load, the two edge chunks of an
// unaligned row included: such a chunk holds at least one byte of the row,
// and an aligned 16-byte granule never crosses a page, so the granule is
// mapped wherever that byte is.  Its slots outside the row (bytes of the
// neighbouring rows, or just past either end of x) are replaced by -inf in
// registers and never used.
template <int DT, bool ALIGNED>
__device__ __forceinline__ uint4 load_chunk(const RowGeom &g, int64_t k, int64_t cols)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    if (k >= g.nch)
        return neg_inf_chunk<DT>();
    const uint4 c = ld_chunk(g.x0 + 16 * k);
    if constexpr (ALIGNED) {
        return c;
    } else {
        if (k >= g.kf && k < g.kl)
            return c;
        return mask_chunk<DT>(c, k * E - g.head, 0, cols);
    }
}

// Store chunk k (k < nch) of a row.  `y_vec` says that y rows sit on the same
// 16-byte phase as x rows, so whole chunks go out as one 16-byte store; when
// they do not, every element is stored on its own.
template <int DT, bool ALIGNED>
__device__ __forceinline__ void store_chunk(const RowGeom &g, int64_t k, int64_t cols, const uint4 &p,
                                            bool y_vec)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    if constexpr (ALIGNED) {
        st_chunk_stream(g.y0 + 16 * k, p);
    } else {
        if (y_vec && k >= g.kf && k < g.kl) {
            st_chunk(g.y0 + 16 * k, p);
            return;
        }
        const int64_t j0 = k * E - g.head;
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int64_t j = j0 + e;
            if (j >= 0 && j < cols) {
                if constexpr (S == 4)
                    st_u32(g.yr + 4 * j, w[e]);
                else
                    st_u16(g.yr + 2 * j, (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
            }
        }
    }
}

// ---------------------------------------------------------------- interior chunks, edge elements

// Where y rows sit relative to x rows, for the kernels built on the
// interior / edge split: kPhAligned -- every row on the 16-byte grid and whole
// chunks long; kPhSame -- unaligned rows, y on the same 16-byte phase as x (an
// interior chunk of x is one of y); kPhOther -- y on another phase, so
// interior results are stored element by element.
constexpr int kPhAligned = 0;
constexpr int kPhSame = 1;
constexpr int kPhOther = 2;

// Interior chunk q of a row; q outside [0, span) gives -inf.
template <int DT>
__device__ __forceinline__ uint4 load_interior(const ShortRow &g, int q)
{
    return (unsigned)q < (unsigned)g.span ? ld_chunk(g.x0 + ((int64_t)(g.kf + q) << 4)) : neg_inf_chunk<DT>();
}

// Store interior chunk q (0 <= q < span) of a row.
template <int DT, int PH>
__device__ __forceinline__ void store_interior(const ShortRow &g, int q, const uint4 &p)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int S = Fmt<DT>::kBytes;
    if constexpr (PH == kPhAligned) {
        st_chunk_stream(g.y0 + ((int64_t)(g.kf + q) << 4), p);
    } else if constexpr (PH == kPhSame) {
        st_chunk(g.y0 + ((int64_t)(g.kf + q) << 4), p);
    } else {
        const int j0 = (g.kf + q) * E - g.head;
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int e = 0; e < E; e++) {
            if constexpr (S == 4)
                st_u32(g.yr + 4 * (int64_t)(j0 + e), w[e]);
            else
                st_u16(g.yr + 2 * (int64_t)(j0 + e), (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
        }
    }
}

// Column of edge element p (0 <= p < ne).
__device__ __forceinline__ int edge_col(const ShortRow &g, int p) { return p < g.enh ? p : g.et0 + (p - g.enh); }

// One element of a row as a float, and one float stored rounded to nearest
// even in the dtype (the rounding pack() applies).
template <int DT>
__device__ __forceinline__ float ld_elem(const char *row, int j)
{
    if constexpr (DT == kF32) {
        return __uint_as_float(ld_u32(row + 4 * (int64_t)j));
    } else if constexpr (DT == kF16) {
        return __half2float(__ushort_as_half((unsigned short)ld_u16(row + 2 * (int64_t)j)));
    } else {
        return __uint_as_float(ld_u16(row + 2 * (int64_t)j) << 16);
    }
}

template <int DT>
__device__ __forceinline__ void st_elem(char *row, int j, float v)
{
    if constexpr (DT == kF32)
        st_u32(row + 4 * (int64_t)j, __float_as_uint(v));
    else if constexpr (DT == kF16)
        st_u16(row + 2 * (int64_t)j, __half_as_ushort(__float2half_rn(v)));
    else
        st_u16(row + 2 * (int64_t)j, __bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

// Edge elements a lane of an L-lane team holds: a row has at most 2E - 2.
template <int DT, int L>
__host__ __device__ constexpr int edge_slots() { return (2 * Fmt<DT>::kPerChunk - 2 + L - 1) / L; }

// Make the compiler treat a cached chunk as freshly defined, so that values
// unpacked from it before this point are not kept alive in registers to be
// reused after it (the chunk is cheaper to hold than its unpacked floats).
__device__ __forceinline__ void opaque(uint4 &c)
{
    asm volatile("" : "+r"(c.x), "+r"(c.y), "+r"(c.z), "+r"(c.w));
}

// Replace the slots of a chunk whose element index (t0 + slot) falls outside
// [lo, hi) with -inf.
template <int DT>
__device__ __forceinline__ uint4 mask_chunk(const uint4 &c, int64_t t0, int64_t lo, int64_t hi)
{
    uint32_t w[4] = {c.x, c.y, c.z, c.w};
    if constexpr (DT == kF32) {
#pragma unroll
        for (int e = 0; e < 4; e++)
            if (t0 + e < lo || t0 + e >= hi)
                w[e] = kNegInfF32;
    } else {
#pragma unroll
        for (int e = 0; e < 8; e++)
            if (t0 + e < lo || t0 + e >= hi) {
                const int sh = 16 * (e & 1);
                w[e >> 1] = (w[e >> 1] & ~(0xFFFFu << sh)) | (Fmt<DT>::kNegInf << sh);
            }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// L2 prefetch (one bulk request) of the 16-byte granules holding bytes
// [p, p + n) of a row (n < 4 GiB): every granule holds a byte of the row, so
// all are mapped.
__device__ __forceinline__ void prefetch_row_l2(const char *p, int64_t n)
{
    const uintptr_t b = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15);
    const uintptr_t e = (reinterpret_cast<uintptr_t>(p) + (uintptr_t)n + 15u) & ~uintptr_t(15);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(b), "r"((uint32_t)(e - b)) : "memory");
}

// ---------------------------------------------------------------- exp and sums

// 2^v on the SFU, subnormal results flushed to zero (one instruction).
__device__ __forceinline__ float ex2_ftz(float v)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Knuth's TwoSum: s + e == a + b exactly (no ordering requirement, symmetric in
// a and b).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// Compensated sum: the value is s + c.
struct CSum {
    float s, c;
};

// Per-dtype arithmetic policy.  Acc is the running sum type.
//
// fp16 / bf16: exp_shift(v, m) = 2^(kExpBias) * exp(v - m), with the SFU's
// flush-to-zero 2^x.  Every consumer divides by a sum of the same scaled terms,
// so the scale cancels in y; it exists for bf16, whose outputs reach subnormals
// (down to 2^-133): without it exp(v - m) would flush below 2^-126 and lose
// them, with it only terms below 2^-190 flush, which bf16 rounds to 0 anyway.
// fp16 outputs underflow to 0 below 2^-25, so fp16 needs no scale.
// v - m is computed first (exact for inputs on a common dyadic grid), so a
// shifted input gives bit-identical results.
template <int DT>
struct Math {
    using Acc = float;
    static constexpr float kExpBias = DT == kBF16 ? 64.f : 0.f;
    // the scaled exp of an already shifted value t = v - m
    static __device__ __forceinline__ float exp_t(float t)
    {
        if constexpr (DT == kBF16)
            return ex2_ftz(fmaf(t, kLog2e, kExpBias));
        else
            return ex2_ftz(t * kLog2e);
    }
    static __device__ __forceinline__ float exp_shift(float v, float m) { return exp_t(v - m); }
    // exp(a) for a <= 0, the ratio used to rescale partial sums (unscaled).
    static __device__ __forceinline__ float exp_of(float a) { return ex2_ftz(a * kLog2e); }
    static __device__ __forceinline__ Acc zero() { return 0.f; }
    static __device__ __forceinline__ void add(Acc &a, float v) { a += v; }
    static __device__ __forceinline__ Acc merge(const Acc &a, const Acc &b) { return a + b; }
    static __device__ __forceinline__ Acc scale(const Acc &a, float f) { return a * f; }
    static __device__ __forceinline__ float value(const Acc &a) { return a; }
    static __device__ __forceinline__ Acc shfl_xor(const Acc &a, int o)
    {
        return __shfl_xor_sync(0xFFFFFFFFu, a, o);
    }
};

template <>
struct Math<kF32> {
    using Acc = CSum;
    static __device__ __forceinline__ float exp_shift(float v, float m)
    {
        // t + r == v - m exactly; exp(v - m) = exp(t) * exp(r), exp(r) ~ 1 + r.
        float t, r;
        two_sum(v, -m, t, r);
        const float e = expf(t);
        return (fabsf(r) < INFINITY) ? fmaf(e, r, e) : e;
    }
    static __device__ __forceinline__ float exp_of(float a) { return expf(a); }
    static __device__ __forceinline__ Acc zero() { return CSum{0.f, 0.f}; }
    static __device__ __forceinline__ void add(Acc &a, float v)
    {
        float s, e;
        two_sum(a.s, v, s, e);
        a.s = s;
        a.c += e;
    }
    static __device__ __forceinline__ Acc merge(const Acc &a, const Acc &b)
    {
        float s, e;
        two_sum(a.s, b.s, s, e);
        return CSum{s, (a.c + b.c) + e};
    }
    static __device__ __forceinline__ Acc scale(const Acc &a, float f) { return CSum{a.s * f, a.c * f}; }
    static __device__ __forceinline__ float value(const Acc &a) { return a.s + a.c; }
    static __device__ __forceinline__ Acc shfl_xor(const Acc &a, int o)
    {
        return CSum{__shfl_xor_sync(0xFFFFFFFFu, a.s, o), __shfl_xor_sync(0xFFFFFFFFu, a.c, o)};
    }
};

// x - m in fp32 for the two 16-bit values packed in w (low half first): one
// mixed-precision FMA each (16-bit x times 1, plus the fp32 -m), which is the
// correctly rounded x - m -- the same value as converting x and subtracting.
template <int DT>
__device__ __forceinline__ void sub_pair(uint32_t w, float neg_m, float &t0, float &t1)
{
    if constexpr (DT == kF16) {
        const unsigned short one = 0x3C00u;
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "fma.rn.f32.f16 %0, lo, %3, %4;\n\tfma.rn.f32.f16 %1, hi, %3, %4;\n\t}"
            : "=f"(t0), "=f"(t1)
            : "r"(w), "h"(one), "f"(neg_m));
    } else {
        const unsigned short one = 0x3F80u;
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "fma.rn.f32.bf16 %0, lo, %3, %4;\n\tfma.rn.f32.bf16 %1, hi, %3, %4;\n\t}"
            : "=f"(t0), "=f"(t1)
            : "r"(w), "h"(one), "f"(neg_m));
    }
}

// Max over the slots of a chunk.  16-bit formats compare packed pairs (the max
// of two representable values is exact in any format).
template <int DT>
__device__ __forceinline__ float chunk_max(const uint4 &c)
{
    if constexpr (DT == kF32) {
        return fmaxf(fmaxf(__uint_as_float(c.x), __uint_as_float(c.y)),
                     fmaxf(__uint_as_float(c.z), __uint_as_float(c.w)));
    } else if constexpr (DT == kF16) {
        __half2 a, b, cc, d;
        *reinterpret_cast<uint32_t *>(&a) = c.x;
        *reinterpret_cast<uint32_t *>(&b) = c.y;
        *reinterpret_cast<uint32_t *>(&cc) = c.z;
        *reinterpret_cast<uint32_t *>(&d) = c.w;
        const __half2 h = __hmax2(__hmax2(a, b), __hmax2(cc, d));
        return fmaxf(__low2float(h), __high2float(h));
    } else {
        __nv_bfloat162 a, b, cc, d;
        *reinterpret_cast<uint32_t *>(&a) = c.x;
        *reinterpret_cast<uint32_t *>(&b) = c.y;
        *reinterpret_cast<uint32_t *>(&cc) = c.z;
        *reinterpret_cast<uint32_t *>(&d) = c.w;
        const __nv_bfloat162 h = __hmax2(__hmax2(a, b), __hmax2(cc, d));
        return fmaxf(__low2float(h), __high2float(h));
    }
}

// f[e] = exp_shift(slot e of chunk c, m) for every slot.  16-bit formats go
// straight from the packed words (sub_pair), skipping the separate convert.
template <int DT>
__device__ __forceinline__ void chunk_exp(const uint4 &c, float m, float (&f)[Fmt<DT>::kPerChunk])
{
    if constexpr (DT == kF32) {
        unpack<DT>(c, f);
#pragma unroll
        for (int e = 0; e < 4; e++)
            f[e] = Math<DT>::exp_shift(f[e], m);
    } else {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        const float nm = -m;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float t0, t1;
            sub_pair<DT>(w[i], nm, t0, t1);
            f[2 * i] = Math<DT>::exp_t(t0);
            f[2 * i + 1] = Math<DT>::exp_t(t1);
        }
    }
}

// ---------------------------------------------------------------- warp / block reductions

// Max over the full warp in one instruction (sm_100-family redux on f32; a
// NaN input is ignored, as fmaxf ignores it).
__device__ __forceinline__ float warp_max_redux(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// Max over aligned groups of G lanes (xor butterfly; all 32 lanes must call).
template <int G>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

template <int DT, int G>
__device__ __forceinline__ typename Math<DT>::Acc group_sum(typename Math<DT>::Acc a)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1)
        a = Math<DT>::merge(a, Math<DT>::shfl_xor(a, o));
    return a;
}

// Online (m, d) pair and its merge.  An empty side (m = -inf) contributes 0.
struct MD {
    float m, d;
};

template <int DT>
__device__ __forceinline__ MD md_merge(const MD &a, const MD &b)
{
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY)
        return MD{m, 0.f};
    const float da = (a.m == -INFINITY) ? 0.f : a.d * Math<DT>::exp_of(a.m - m);
    const float db = (b.m == -INFINITY) ? 0.f : b.d * Math<DT>::exp_of(b.m - m);
    return MD{m, da + db};
}

template <int DT>
__device__ __forceinline__ MD warp_md(MD v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MD w{__shfl_xor_sync(0xFFFFFFFFu, v.m, o), __shfl_xor_sync(0xFFFFFFFFu, v.d, o)};
        v = md_merge<DT>(v, w);
    }
    return v;
}

// Block-wide max; every thread gets the result.  `slots` holds >= 32 floats and
// may be reused by the next reduction call (the leading barrier protects it).
__device__ __forceinline__ float block_max(float v, float *slots)
{
    v = warp_max_redux(v);  // one instruction per warp stage, not a 5-step butterfly
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0)
        slots[warp] = v;
    __syncthreads();
    v = lane < nw ? slots[lane] : -INFINITY;
    return warp_max_redux(v);
}

template <int DT>
__device__ __forceinline__ typename Math<DT>::Acc block_sum(typename Math<DT>::Acc a,
                                                            typename Math<DT>::Acc *slots)
{
    a = group_sum<DT, 32>(a);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0)
        slots[warp] = a;
    __syncthreads();
    a = lane < nw ? slots[lane] : Math<DT>::zero();
    return group_sum<DT, 32>(a);
}

template <int DT>
__device__ __forceinline__ MD block_md(MD v, MD *slots)
{
    v = warp_md<DT>(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0)
        slots[warp] = v;
    __syncthreads();
    v = lane < nw ? slots[lane] : MD{-INFINITY, 0.f};
    return warp_md<DT>(v);
}

}  // namespace osd
