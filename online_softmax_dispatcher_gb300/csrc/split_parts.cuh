// split_parts.cuh -- pieces shared by the kernels that split a row over several
// CTAs and hold each CTA's share in shared memory (the grid split's ring and
// pipelined forms, the cluster split's held form): the share geometry, the
// bulk copies that fill a share, the online fold of landed chunks and a
// warp's (m, d) reduction.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace osd {

// Bulk copies per share in the pipelined forms.  Their shares are small (a
// quarter to a half of the ring form's), and a fold thread must find several
// chunks per piece to keep independent work in flight: with 8 pieces it found
// one or two, and the fold became a chain of dependent steps (0.35 us a piece).
constexpr int kPipePieces = 2;

// The whole chunks [fb, fe) of CTA p's share [kb, ke) of row g (a partial
// first or last chunk of the row is left to load_chunk).
struct Share {
    int64_t kb, ke, fb, fe;
    int64_t edge_k;  // the row's partial edge chunk this thread holds, or -1
};

template <int DT, bool ALIGNED>
__device__ __forceinline__ Share share_of(const RowGeom &g, int64_t cols, int P, int p, int tid)
{
    constexpr int E = Fmt<DT>::kPerChunk;
    Share s;
    const int64_t per = (g.nch + P - 1) / P;
    s.kb = per * p < g.nch ? per * p : g.nch;
    s.ke = s.kb + per < g.nch ? s.kb + per : g.nch;
    const int64_t first_whole = ALIGNED || g.head == 0 ? 0 : 1;
    const int64_t end_whole = ALIGNED || (g.head + cols) % E == 0 ? g.nch : g.nch - 1;
    s.fb = s.kb > first_whole ? s.kb : first_whole;
    s.fe = s.ke < end_whole ? s.ke : end_whole;
    if (s.fe < s.fb)
        s.fe = s.fb;
    // threads 0 and 1 take the row's partial first and last chunk
    s.edge_k = -1;
    if (tid == 0 && first_whole == 1 && 0 >= s.kb && 0 < s.ke)
        s.edge_k = 0;
    if (tid == 1 && end_whole == g.nch - 1 && g.nch - 1 >= s.kb && g.nch - 1 < s.ke &&
        !(g.nch == 1 && first_whole == 1))
        s.edge_k = g.nch - 1;
    return s;
}

// Fold K chunks into the online pair (m, d); all -inf chunks leave it as it is.
template <int DT, int K>
__device__ __forceinline__ void md_absorb(MD &md, const uint4 (&raw)[K])
{
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    float mt = -INFINITY;
#pragma unroll
    for (int u = 0; u < K; u++)
        mt = fmaxf(mt, chunk_max<DT>(raw[u]));
    if (mt == -INFINITY)
        return;
    if (mt > md.m) {
        md.d = md.m == -INFINITY ? 0.f : md.d * M::exp_of(md.m - mt);
        md.m = mt;
    }
    // four partial sums: a dependency chain of K * E / 4 additions, not K * E
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < K; u++) {
        float f[E];
        chunk_exp<DT>(raw[u], md.m, f);
#pragma unroll
        for (int e = 0; e < E; e++)
            s[e & 3] += f[e];
    }
    md.d += (s[0] + s[1]) + (s[2] + s[3]);
}

// Load CTA p's share of row r (its whole chunks, n of them) into shared
// memory at `dst` as PIECES bulk copies, one mbarrier each (bar0, bar0 + 8,
// ...).  One thread.
template <int DT, bool ALIGNED, int PIECES>
__device__ __forceinline__ void issue_share(const char *x, char *y, int64_t cols, int64_t r, int P, int p,
                                            uint32_t dst, uint32_t bar0)
{
    const RowGeom g = row_geom<DT, ALIGNED>(x, y, r, cols);
    const Share sh = share_of<DT, ALIGNED>(g, cols, P, p, 0);
    const int n = (int)(sh.fe - sh.fb);
    const int piece = (n + PIECES - 1) / PIECES;
    // the buffer's previous contents were read through the generic proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int i = 0; i < PIECES; i++) {
        const int c0 = i * piece, cnt = n - c0 < piece ? n - c0 : piece;
        if (cnt <= 0)
            break;
        mbar_arrive_expect_tx(bar0 + 8u * i, (uint32_t)(16 * cnt));
        bulk_g2s(dst + 16u * (uint32_t)c0, g.x0 + 16 * (sh.fb + c0), (uint32_t)(16 * cnt), bar0 + 8u * i);
    }
}

// (m, d) over a warp: the max in one instruction, each lane's sum rescaled to
// it once, then an xor butterfly of plain additions (both partners of a step
// add the same two numbers, so every lane ends with the same value).
template <int DT>
__device__ __forceinline__ MD warp_md_max_first(MD v)
{
    const float m = warp_max_redux(v.m);
    float d = (v.m == -INFINITY) ? 0.f : v.d * Math<DT>::exp_of(v.m - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
    return MD{m, d};
}

}  // namespace osd
