// k_grid.cu -- few rows, huge cols, on every SM in one launch: SPLITK_GRID.
//
// A thread-block cluster holds at most 16 CTAs, so the cluster split (k_splitk)
// puts at most 16 SMs on a row.  Here a cooperative launch of P CTAs per row --
// all of them resident at once, which the cooperative launch guarantees -- splits
// each row over every SM; the CTAs of a row publish their partial statistics
// to global memory and meet at a per-row barrier before they write.  It is the
// split of "[CUDA] safe online softmax", section 3.2 (per-block partials, then
// a merge) in one kernel, with the grid synchronisation that page set aside
// made safe here by the cooperative launch (co-residency) and a bounded wait.
//
// * Ring form (a CTA's share of a row fits a shared-memory buffer; one CTA
//   per SM): G groups of P CTAs; a group takes every G-th row in turn, each
//   CTA holding share p of the row.  Shares pass through a ring of Q buffers
//   filled by bulk copies (x is read from HBM once); the statistics of one
//   row, the output of the row before it and the loads of the rows after it
//   overlap.  The dispatcher takes as few rows per group as the buffers allow
//   (one, when a share of 1/G of the SMs fits), since each row costs a CTA
//   a fixed few microseconds in turn.
// * Streaming form (shares too long for shared memory; two CTAs per SM, P
//   per row): the passes of the two-launch split (stream_passes.cuh) around
//   the barrier; the write pass re-reads x, from L2 when the rows fit there.
// * Barrier: each row has two arrival counters used by alternate launches of a
//   slot (the launch's generation number picks one); a CTA stores its
//   partial, adds one to the launch's counter with release semantics and
//   waits -- for at most kWaitLimitNs of %globaltimer time -- until an acquire
//   load of it reads P.  The first CTA zeroes the other parity's counters of
//   every row the slot serves, ready for the slot's next launch whatever its
//   row count (the previous launch that used them has finished), so a launch
//   that gave up leaves nothing stale behind.  A wait
//   that gives up records kErrGridWait in the library's device error word and
//   the CTA returns without writing.
// * Every CTA of a row merges the P partials in the same fixed order, so all
//   hold bit-identical (m, 1/d).
//
// Scratch: the partials, counts and flags live in a small pool of slots of
// library-owned device memory (kGridSlots slots); a call takes the next slot,
// its stream first waits for the CUDA event recorded after the slot's
// previous launch, so launches that share a slot never overlap on the GPU
// whatever streams they run on.
#include <cuda_runtime.h>

#include <atomic>
#include <functional>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "stream_passes.cuh"
#include "tma.cuh"

namespace osd {

constexpr unsigned kErrGridWait = 4u;  // waiting at a row's grid barrier
constexpr int kGridPieces = 8;         // bulk copies per share in the ring form, consumed as they land

struct GridArgs {
    const char *x;
    char *y;
    int64_t rows;
    int64_t cols;
    int P;    // CTAs per row
    int Q;    // ring form: shared-memory buffers (0: streaming form)
    int buf;  // ring form: bytes per buffer
    int y_vec;
    float4 *part;      // [rows * P] partial statistics
    unsigned *arrive;  // [rows][2] arrival counters, one per launch parity
    unsigned gen;      // this launch's number in its slot (its parity picks the counter)
    unsigned *err;
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned *p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Publish this CTA's partial and wait (bounded) until every CTA of row r has
// published its own.  Called by one thread per CTA; false on time-out.
__device__ __forceinline__ bool grid_row_barrier(const GridArgs &a, int64_t r, int p, float4 partial)
{
    a.part[r * a.P + p] = partial;
    unsigned *cnt = &a.arrive[2 * r + (a.gen & 1u)];
    // release: the partial is visible to whoever acquires the count after it
    red_add_release_gpu(cnt, 1u);
    // poll without sleeping (the wait is short and one thread per CTA polls)
    const uint64_t t0 = global_ns();
    while (ld_acquire_gpu(cnt) < (unsigned)a.P)
        if (global_ns() - t0 > kWaitLimitNs)
            return false;
    return true;
}

// Zero the slot's counters of the other parity, for every row a slot serves
// (not only this launch's rows: the slot's next launch may have more), so
// that the next launch starts from zero.  The first CTA does it.
__device__ __forceinline__ void grid_prepare_next(const GridArgs &a)
{
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < kGridMaxRows; i += blockDim.x)
            a.arrive[2 * i + ((a.gen + 1u) & 1u)] = 0u;
}

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

// merge_partials spread over the CTA: thread i loads partial i (all P in one
// round trip through L2 rather than P / 32 dependent ones per warp), then the
// block reductions combine them in a fixed order, so every CTA of the row holds
// bit-identical (m, 1/d).  All threads call it.
template <int DT>
__device__ __forceinline__ void merge_partials_cta(const float4 *ws, int64_t r, int P, float &m, float &inv,
                                                   float *smax, typename Math<DT>::Acc *ssum, MD *smd)
{
    const int T = blockDim.x;
    if constexpr (DT == kF32) {
        float4 q[2];
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int i = threadIdx.x + j * T;
            q[j] = i < P ? __ldcg(&ws[r * P + i]) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        }
        float mloc = fmaxf(q[0].x, q[1].x);
        for (int i = threadIdx.x + 2 * T; i < P; i += T)
            mloc = fmaxf(mloc, __ldcg(&ws[r * P + i]).x);
        m = block_max(mloc, smax);
        CSum acc{0.f, 0.f};
        auto add = [&](const float4 &v) {
            if (v.x != -INFINITY) {
                const float f = Math<kF32>::exp_shift(v.x, m);
                Math<kF32>::add(acc, v.y * f);
                Math<kF32>::add(acc, v.z * f);
            }
        };
        add(q[0]);
        add(q[1]);
        for (int i = threadIdx.x + 2 * T; i < P; i += T)
            add(__ldcg(&ws[r * P + i]));
        acc = block_sum<kF32>(acc, ssum);
        inv = 1.0f / (acc.s + acc.c);
    } else {
        MD md{-INFINITY, 0.f};
        for (int i = threadIdx.x; i < P; i += T) {
            const float4 v = __ldcg(&ws[r * P + i]);
            md = md_merge<DT>(md, MD{v.x, v.y});
        }
        md = block_md<DT>(md, smd);
        m = md.m;
        inv = 1.0f / md.d;
    }
}

// Load CTA p's share of row r (its whole chunks, n of them) into ring buffer
// `dst` as kGridPieces bulk copies, one mbarrier each.  One thread.
template <int DT, bool ALIGNED>
__device__ __forceinline__ void grid_issue(const GridArgs &a, int64_t r, int p, uint32_t dst, uint32_t bar0)
{
    const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, r, a.cols);
    const Share sh = share_of<DT, ALIGNED>(g, a.cols, a.P, p, 0);
    const int n = (int)(sh.fe - sh.fb);
    const int piece = (n + kGridPieces - 1) / kGridPieces;
    // the buffer's previous contents were read through the generic proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int i = 0; i < kGridPieces; i++) {
        const int c0 = i * piece, cnt = n - c0 < piece ? n - c0 : piece;
        if (cnt <= 0)
            break;
        mbar_arrive_expect_tx(bar0 + 8u * i, (uint32_t)(16 * cnt));
        bulk_g2s(dst + 16u * (uint32_t)c0, g.x0 + 16 * (sh.fb + c0), (uint32_t)(16 * cnt), bar0 + 8u * i);
    }
}

// Store this CTA's partial of row r and count it in (release); one thread.
__device__ __forceinline__ void grid_publish(const GridArgs &a, int64_t r, int p, float4 partial)
{
    a.part[r * a.P + p] = partial;
    red_add_release_gpu(&a.arrive[2 * r + (a.gen & 1u)], 1u);
}

// Wait (bounded) until every CTA that shares row r has counted its partial in.
__device__ __forceinline__ bool grid_wait_row(const GridArgs &a, int64_t r)
{
    const unsigned *cnt = &a.arrive[2 * r + (a.gen & 1u)];
    const uint64_t t0 = global_ns();
    while (ld_acquire_gpu(cnt) < (unsigned)a.P)
        if (global_ns() - t0 > kWaitLimitNs)
            return false;
    return true;
}

// Ring form: the grid is G groups (blockIdx.y) of P CTAs (blockIdx.x), one CTA
// per SM; group gy takes rows gy, gy + G, gy + 2G, ... and CTA p of the group
// holds share p of each of them.  The shares pass through a ring of Q
// shared-memory buffers filled by bulk copies, so x is read from HBM once.
// Row k of the group: wait for its pieces, fold them into this CTA's partial
// statistics and count it in at the row's barrier without waiting; then
// (lagging one row behind when Q >= 2) wait at the previous row's barrier,
// merge its P partials, write it from its buffer and refill that buffer with
// the row Q places further on.  The loads of later rows, the statistics of
// this one and the output of the one before overlap, and a row's barrier is
// normally complete by the time a CTA asks for it.
template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kGridThreads, 1) k_grid_ring(const GridArgs a)
{
    pdl_enter();
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int K = 4;  // chunks per thread per step
    extern __shared__ __align__(128) unsigned char seg[];
    __shared__ __align__(8) uint64_t bars[kGridMaxRing * kGridPieces];
    __shared__ int pending[kGridMaxRing];  // group row whose copies into a buffer are unawaited, or -1
    __shared__ float smax[32];
    __shared__ typename M::Acc ssum[32];
    __shared__ MD smd[32];
    __shared__ volatile int abort_flag;
    const int p = blockIdx.x, gy = blockIdx.y, G = gridDim.y;
    const int tid = threadIdx.x, T = blockDim.x;
    const int Q = a.Q;
    const int nr = a.rows > gy ? (int)((a.rows - gy + G - 1) / G) : 0;
    const uint32_t seg0 = smem_u32(seg), bar0 = smem_u32(bars);
    const int lag = Q >= 2 ? 1 : 0;  // rows a CTA's output trails its statistics

    grid_prepare_next(a);
    if (tid == 0) {
        for (int i = 0; i < Q * kGridPieces; i++)
            mbar_init(bar0 + 8u * i, 1);
        abort_flag = 0;
        mbar_init_fence();
        for (int b = 0; b < Q; b++) {
            pending[b] = b < nr ? b : -1;
            if (b < nr)
                grid_issue<DT, ALIGNED>(a, gy + (int64_t)b * G, p, seg0 + (uint32_t)b * a.buf,
                                        bar0 + 8u * kGridPieces * b);
        }
    }
    __syncthreads();

    for (int k = 0; k < nr + lag; k++) {
        if (k < nr) {
            // ---- statistics of row k
            const int64_t r = gy + (int64_t)k * G;
            const int b = k % Q;
            const uint32_t par = (uint32_t)(k / Q) & 1u, buf = seg0 + (uint32_t)b * a.buf;
            const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, r, a.cols);
            const Share sh = share_of<DT, ALIGNED>(g, a.cols, a.P, p, tid);
            const int n = (int)(sh.fe - sh.fb);
            const int piece = (n + kGridPieces - 1) / kGridPieces;
            const uint4 edge = sh.edge_k >= 0 ? load_chunk<DT, ALIGNED>(g, sh.edge_k, a.cols) : neg_inf_chunk<DT>();
            float4 partial;
            if constexpr (DT == kF32) {
                // fp32: the share's max, then the compensated sum of exp(x - max)
                bool ok = true;
                for (int i = 0; i < kGridPieces && i * piece < n && ok; i++)
                    ok = mbar_wait(bar0 + 8u * (kGridPieces * b + i), par, &abort_flag);
                if (!ok) {
                    if (!abort_flag)
                        atomicOr(a.err, kErrFullWait);
                    abort_flag = 1;
                }
                float mx = chunk_max<DT>(edge);
                if (!abort_flag) {
                    float mx2 = -INFINITY;
                    int c = tid;
                    for (; c + T < n; c += 2 * T) {
                        mx = fmaxf(mx, chunk_max<DT>(lds_chunk(buf + 16u * (uint32_t)c)));
                        mx2 = fmaxf(mx2, chunk_max<DT>(lds_chunk(buf + 16u * (uint32_t)(c + T))));
                    }
                    if (c < n)
                        mx = fmaxf(mx, chunk_max<DT>(lds_chunk(buf + 16u * (uint32_t)c)));
                    mx = fmaxf(mx, mx2);
                }
                mx = block_max(mx, smax);
                // one compensated accumulator per slot of a chunk: E independent
                // dependency chains, merged in a fixed order
                CSum acc[E];
#pragma unroll
                for (int e = 0; e < E; e++)
                    acc[e] = M::zero();
                if (!abort_flag && mx != -INFINITY) {
                    float f[E];
                    chunk_exp<DT>(edge, mx, f);
#pragma unroll
                    for (int e = 0; e < E; e++)
                        M::add(acc[e], f[e]);
#pragma unroll 2
                    for (int c = tid; c < n; c += T) {
                        chunk_exp<DT>(lds_chunk(buf + 16u * (uint32_t)c), mx, f);
#pragma unroll
                        for (int e = 0; e < E; e++)
                            M::add(acc[e], f[e]);
                    }
                }
                CSum tot = M::merge(M::merge(acc[0], acc[1]), M::merge(acc[2], acc[3]));
                tot = block_sum<DT>(tot, ssum);
                partial = make_float4(mx, tot.s, tot.c, 0.f);
            } else {
                // 16-bit: one online (m, d) pass, each piece as it lands
                MD md{-INFINITY, 0.f};
                {
                    uint4 one[1] = {edge};
                    md_absorb<DT, 1>(md, one);
                }
                for (int i = 0; i < kGridPieces && i * piece < n; i++) {
                    if (!mbar_wait(bar0 + 8u * (kGridPieces * b + i), par, &abort_flag)) {
                        if (!abort_flag)
                            atomicOr(a.err, kErrFullWait);
                        abort_flag = 1;
                        break;
                    }
                    const int c0 = i * piece, c1 = n - c0 < piece ? n : c0 + piece;
                    for (int c = c0 + tid; c < c1; c += T * K) {
                        uint4 raw[K];
#pragma unroll
                        for (int u = 0; u < K; u++) {
                            const int cc = c + u * T;
                            raw[u] = cc < c1 ? lds_chunk(buf + 16u * (uint32_t)cc) : neg_inf_chunk<DT>();
                        }
                        md_absorb<DT, K>(md, raw);
                    }
                }
                md = block_md<DT>(md, smd);
                partial = make_float4(md.m, md.d, 0.f, 0.f);
            }
            // (the block reduction's barriers make a time-out seen by any thread seen by all)
            if (abort_flag)
                break;
            if (tid == 0) {
                pending[b] = -1;
                grid_publish(a, r, p, partial);
            }
        }
        if (k >= lag) {
            // ---- output of row j = k - lag
            const int j = k - lag;
            const int64_t r = gy + (int64_t)j * G;
            const int b = j % Q;
            const uint32_t buf = seg0 + (uint32_t)b * a.buf;
            if (tid == 0 && !grid_wait_row(a, r)) {
                atomicOr(a.err, kErrGridWait);
                abort_flag = 1;
            }
            __syncthreads();
            if (abort_flag)
                break;
            // (thread 0's acquire and the barrier order the partials' loads)
            float m, inv;
            merge_partials_cta<DT>(a.part, r, a.P, m, inv, smax, ssum, smd);
            const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, r, a.cols);
            const Share sh = share_of<DT, ALIGNED>(g, a.cols, a.P, p, tid);
            const int n = (int)(sh.fe - sh.fb);
            if (sh.edge_k >= 0) {
                float f[E];
                chunk_exp<DT>(load_chunk<DT, ALIGNED>(g, sh.edge_k, a.cols), m, f);
#pragma unroll
                for (int e = 0; e < E; e++)
                    f[e] *= inv;
                store_chunk<DT, ALIGNED>(g, sh.edge_k, a.cols, pack<DT>(f), a.y_vec != 0);
            }
#pragma unroll 4
            for (int c = tid; c < n; c += T) {
                float f[E];
                chunk_exp<DT>(lds_chunk(buf + 16u * (uint32_t)c), m, f);
#pragma unroll
                for (int e = 0; e < E; e++)
                    f[e] *= inv;
                store_chunk<DT, ALIGNED>(g, sh.fb + c, a.cols, pack<DT>(f), a.y_vec != 0);
            }
            __syncthreads();  // buffer b is free
            if (tid == 0 && j + Q < nr) {
                pending[b] = j + Q;
                grid_issue<DT, ALIGNED>(a, gy + (int64_t)(j + Q) * G, p, buf, bar0 + 8u * kGridPieces * b);
            }
        }
    }
    if (abort_flag) {
        if (tid == 0) {
            // no copy may still be landing in shared memory when the CTA leaves
            for (int b = 0; b < Q; b++)
                if (pending[b] >= 0)
                    for (int i = 0; i < kGridPieces; i++)
                        (void)mbar_wait(bar0 + 8u * (kGridPieces * b + i), (uint32_t)(pending[b] / Q) & 1u,
                                        &abort_flag, false);
        }
        __syncthreads();
    }
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kStreamThreads, 2) k_grid_stream(const GridArgs a)
{
    pdl_enter();
    using M = Math<DT>;
    __shared__ float smax[32];
    __shared__ typename M::Acc ssum[32];
    __shared__ MD smd[32];
    __shared__ volatile int abort_flag;
    const int64_t r = blockIdx.y;
    const int p = blockIdx.x;
    const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, r, a.cols);
    const int64_t per = (g.nch + a.P - 1) / a.P;
    const int64_t kb = per * p < g.nch ? per * p : g.nch;
    const int64_t ke = kb + per < g.nch ? kb + per : g.nch;
    grid_prepare_next(a);
    float4 out;
    if constexpr (DT == kF32) {
        const float m = block_max(pass_max<DT, ALIGNED, kWideStep>(g, kb, ke, a.cols), smax);
        CSum acc{0.f, 0.f};
        if (m != -INFINITY)
            acc = pass_sum<DT, ALIGNED, kWideStep>(g, kb, ke, a.cols, m);
        acc = block_sum<DT>(acc, ssum);
        out = make_float4(m, acc.s, acc.c, 0.f);
    } else {
        const MD md = block_md<DT>(pass_online<DT, ALIGNED, kWideStep>(g, kb, ke, a.cols), smd);
        out = make_float4(md.m, md.d, 0.f, 0.f);
    }
    if (threadIdx.x == 0) {
        abort_flag = 0;
        if (!grid_row_barrier(a, r, p, out)) {
            atomicOr(a.err, kErrGridWait);
            abort_flag = 1;
        }
    }
    __syncthreads();
    if (abort_flag)
        return;
    __threadfence();
    float m, inv;
    merge_partials<DT>(a.part, r, a.P, m, inv);
    pass_write<DT, ALIGNED, kWideStep>(g, kb, ke, a.cols, m, inv, a.y_vec != 0);
}

// ---------------------------------------------------------------- host side

namespace {

// kGridSlots slots; a slot serves rows * P <= kGridMaxPartials and rows <= kGridMaxRows
static __device__ __align__(256) float4 g_grid_part[kGridSlots][kGridMaxPartials];
static __device__ unsigned g_grid_arrive[kGridSlots][2 * kGridMaxRows];

struct GridPool {
    InitOnSuccess init;
    float4 *part = nullptr;
    unsigned *arrive = nullptr;
    cudaEvent_t ev[kGridSlots] = {};
    bool used[kGridSlots] = {};
    cudaStream_t last[kGridSlots] = {};  // stream of the slot's previous launch
    unsigned gen[kGridSlots] = {};
    std::mutex mu[kGridSlots];
    std::atomic<unsigned> next{0};
};

GridPool g_pools[64];

// The device addresses of the scratch arrays and the slots' events, for the
// current device.  Safe to call again after a failure: events made by an
// earlier attempt are kept.
int pool_init(GridPool &pl)
{
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_grid_part);
    if (e != cudaSuccess)
        return (int)e;
    pl.part = static_cast<float4 *>(p);
    e = cudaGetSymbolAddress(&p, g_grid_arrive);
    if (e != cudaSuccess)
        return (int)e;
    pl.arrive = static_cast<unsigned *>(p);
    for (int i = 0; i < kGridSlots; i++)
        if (pl.ev[i] == nullptr && (e = cudaEventCreateWithFlags(&pl.ev[i], cudaEventDisableTiming)) != cudaSuccess) {
            pl.ev[i] = nullptr;
            return (int)e;
        }
    return 0;
}

template <int DT, bool A, bool RES>
int grid_launch_one(const Launch &l, const GridArgs &args)
{
    auto kern = RES ? &k_grid_ring<DT, A> : &k_grid_stream<DT, A>;
    if (RES) {
        // opt in once per device to the largest segment the planner gives this
        // kernel (the device's opt-in limit less the static shared memory)
        static std::atomic<int> opted[64];
        int d = 0;
        cudaError_t e = cudaGetDevice(&d);
        if (e != cudaSuccess)
            return (int)e;
        if (d < 0 || d >= 64)
            return (int)cudaErrorInvalidDevice;
        if (!opted[d].load(std::memory_order_acquire)) {
            int optin = 0;
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         optin - kGridStaticSmem);
            if (e != cudaSuccess)
                return (int)e;
            opted[d].store(1, std::memory_order_release);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)l.plan.grid_x, (unsigned)l.plan.grid_y, 1);
    cfg.blockDim = dim3((unsigned)l.plan.block_threads, 1, 1);
    cfg.dynamicSmemBytes = RES ? (size_t)l.plan.smem_bytes : 0;
    cfg.stream = (cudaStream_t)l.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess)
        (void)cudaGetLastError();
    return (int)e;
}

template <int DT>
int grid_dt(const Launch &l, const GridArgs &args)
{
    const bool res = l.plan.stages >= 1;
    if (l.plan.aligned)
        return res ? grid_launch_one<DT, true, true>(l, args) : grid_launch_one<DT, true, false>(l, args);
    return res ? grid_launch_one<DT, false, true>(l, args) : grid_launch_one<DT, false, false>(l, args);
}

}  // namespace

int grid_capturing(void *stream)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &st);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return st != cudaStreamCaptureStatusNone;
}

int launch_grid(const Launch &l)
{
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess)
        return (int)e;
    if (d < 0 || d >= 64)
        return (int)cudaErrorInvalidDevice;
    GridPool &pl = g_pools[d];
    const int pe = pl.init.run([&] { return pool_init(pl); });  // device d is current here
    if (pe != 0)
        return pe;
    if (l.rows > kGridMaxRows || l.plan.grid_x * l.rows > kGridMaxPartials || l.plan.stages > kGridMaxRing)
        return (int)cudaErrorInvalidValue;
    const unsigned s = pl.next.fetch_add(1, std::memory_order_relaxed) % kGridSlots;
    std::lock_guard<std::mutex> lock(pl.mu[s]);
    cudaStream_t st = (cudaStream_t)l.stream;
    // the slot's previous launch has finished before this one starts: stream
    // order on the same stream, its event on another
    if (pl.used[s] && pl.last[s] != st && (e = cudaStreamWaitEvent(st, pl.ev[s], 0)) != cudaSuccess)
        return (int)e;
    const unsigned gen = pl.gen[s] + 1u;
    const int Q = l.plan.stages;
    GridArgs args{(const char *)l.x, (char *)l.y, l.rows, l.cols, (int)l.plan.grid_x, Q,
                  Q > 0 ? l.plan.smem_bytes / Q : 0, l.plan.y_vector,
                  pl.part + (size_t)s * kGridMaxPartials, pl.arrive + (size_t)s * 2 * kGridMaxRows, gen,
                  l.dev_err};
    int rc;
    switch (l.dtype) {
    case kF32:
        rc = grid_dt<kF32>(l, args);
        break;
    case kF16:
        rc = grid_dt<kF16>(l, args);
        break;
    case kBF16:
        rc = grid_dt<kBF16>(l, args);
        break;
    default:
        rc = (int)cudaErrorInvalidValue;
    }
    if (rc != 0)
        return rc;
    pl.gen[s] = gen;
    pl.used[s] = true;
    pl.last[s] = st;
    return (int)cudaEventRecord(pl.ev[s], st);
}

int reset_grid_scratch()
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64)
        return 0;
    GridPool &pl = g_pools[d];
    if (!pl.arrive)
        return 0;
    for (int s = 0; s < kGridSlots; s++)
        pl.mu[s].lock();
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemset(pl.arrive, 0, sizeof(unsigned) * kGridSlots * 2 * kGridMaxRows);
    for (int s = 0; s < kGridSlots; s++)
        pl.mu[s].unlock();
    return (int)e;
}

}  // namespace osd
