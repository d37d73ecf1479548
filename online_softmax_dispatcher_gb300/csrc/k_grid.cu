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
#include "split_parts.cuh"
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
    int nf;            // pipelined form: threads that fold (the rest write); 0 in the other forms
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

// ---------------------------------------------------------------- team reductions

constexpr int kPipeMaxPerLane = kGridPipeMaxCtas / 32;  // partials each lane of the merging warp holds


// The P partials of row r merged by one warp: lane i loads partials i, i + 32,
// ... (one round trip through L2), the max in one instruction, then the
// rescaled sums -- each lane in a fixed order, then an xor butterfly -- so
// every CTA of the row computes bit-identical (m, 1/d).  Called by a whole
// warp after an acquire of the row's count that the warp has synchronised on.
template <int DT>
__device__ __forceinline__ void merge_partials_warp(const float4 *part, int64_t r, int P, float &m_out,
                                                    float &inv_out)
{
    const int lane = threadIdx.x & 31;
    float pm[kPipeMaxPerLane], ps[kPipeMaxPerLane], pc[kPipeMaxPerLane];
    float mloc = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPipeMaxPerLane; j++) {
        const int i = lane + 32 * j;
        const float4 v = i < P ? __ldcg(&part[r * P + i]) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        pm[j] = v.x;
        ps[j] = v.y;
        pc[j] = v.z;
        mloc = fmaxf(mloc, v.x);
    }
    const float m = warp_max_redux(mloc);
    if constexpr (DT == kF32) {
        CSum acc{0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kPipeMaxPerLane; j++) {
            if (pm[j] != -INFINITY) {
                const float f = Math<kF32>::exp_shift(pm[j], m);
                Math<kF32>::add(acc, ps[j] * f);
                Math<kF32>::add(acc, pc[j] * f);
            }
        }
        acc = group_sum<kF32, 32>(acc);
        inv_out = 1.0f / (acc.s + acc.c);
    } else {
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < kPipeMaxPerLane; j++)
            if (pm[j] != -INFINITY)
                d += ps[j] * Math<DT>::exp_of(pm[j] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
        inv_out = 1.0f / d;
    }
    m_out = m;
}

// Load CTA p's share of row r into ring buffer `dst` as PIECES bulk copies.
// One thread.
template <int DT, bool ALIGNED, int PIECES = kGridPieces>
__device__ __forceinline__ void grid_issue(const GridArgs &a, int64_t r, int p, uint32_t dst, uint32_t bar0)
{
    issue_share<DT, ALIGNED, PIECES>(a.x, a.y, a.cols, r, a.P, p, dst, bar0);
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
    __shared__ float2 mi;  // (m, 1/d) of the row being written
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
                // warps' sums into slots, merged by warp 0 (only thread 0 publishes)
                tot = group_sum<DT, 32>(tot);
                __syncthreads();
                if ((tid & 31) == 0)
                    ssum[tid >> 5] = tot;
                __syncthreads();
                if (tid < 32) {
                    tot = group_sum<DT, 32>((tid << 5) < T ? ssum[tid] : M::zero());
                    partial = make_float4(mx, tot.s, tot.c, 0.f);
                }
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
                // the CTA's (m, d): warps' pairs (max first) into slots, merged by
                // warp 0 -- only thread 0 needs it, to publish it
                md = warp_md_max_first<DT>(md);
                __syncthreads();  // the slots' previous readers are done
                if ((tid & 31) == 0)
                    smd[tid >> 5] = md;
                __syncthreads();
                if (tid < 32) {
                    md = warp_md_max_first<DT>((tid << 5) < T ? smd[tid] : MD{-INFINITY, 0.f});
                    partial = make_float4(md.m, md.d, 0.f, 0.f);
                }
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
            if (tid < 32) {
                float mm, ii;
                merge_partials_warp<DT>(a.part, r, a.P, mm, ii);
                if (tid == 0)
                    mi = make_float2(mm, ii);
            }
            __syncthreads();
            const float m = mi.x, inv = mi.y;
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

// Pipelined form: one CTA per SM, all P of them on every row; CTA p holds share
// p of each row, the rows passing in order through a ring of Q shared-memory
// buffers filled by bulk copies (x read from HBM once).  The CTA's warps split
// into two teams that work on different rows at once:
// * fold team (the first nf threads): for each row in turn, waits for its
//   share's pieces and folds them as they land, reduces over the team only
//   (warp max in one instruction, team slots behind a named barrier) and
//   publishes the CTA's partial at the row's grid barrier -- then goes on to
//   the next row without waiting for the barrier;
// * write team (the rest): for each row in turn, waits at its grid barrier
//   (one thread polls), merges the P partials in one warp, writes the share
//   from shared memory, and refills the buffer with the row Q places further
//   on.
// So the loads and fold of row k + 1 overlap the barrier, merge and output of
// row k, and the rows' barriers are normally complete by the time the write
// team asks.  The teams share only the buffers (mbarriers of the bulk copies)
// and the abort flag.  Every wait is bounded; on a time-out every thread still
// walks its team's barrier sequence, skipping the work, and the CTA waits
// (bounded) for its copies in flight before it leaves.
template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kGridThreads, 1) k_grid_pipe(const GridArgs a)
{
    pdl_enter();
    using M = Math<DT>;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int K = 4;  // chunks per fold thread per step
    constexpr int kFoldWarpsMax = kGridThreads / 32;
    extern __shared__ __align__(128) unsigned char seg[];
    __shared__ __align__(8) uint64_t bars[kGridMaxRing * kPipePieces];
    __shared__ int pending[kGridMaxRing];           // row whose copies into a buffer are unawaited, or -1
    __shared__ float4 fslot[2][kFoldWarpsMax];      // fold warps' partials, by row parity
    __shared__ float2 mrow[2];                      // (m, 1/d) of the row the write team writes, by parity
    __shared__ volatile int abort_flag;
    const int p = blockIdx.x, P = a.P, Q = a.Q, NF = a.nf;
    const int R = (int)a.rows;
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t seg0 = smem_u32(seg), bar0 = smem_u32(bars);

    grid_prepare_next(a);
    if (tid == 0) {
        for (int i = 0; i < Q * kPipePieces; i++)
            mbar_init(bar0 + 8u * i, 1);
        abort_flag = 0;
        mbar_init_fence();
        for (int b = 0; b < Q; b++) {
            pending[b] = b < R ? b : -1;
            if (b < R)
                grid_issue<DT, ALIGNED, kPipePieces>(a, b, p, seg0 + (uint32_t)b * a.buf, bar0 + 8u * kPipePieces * b);
        }
    }
    __syncthreads();

    if (tid < NF) {
        // ---------------- fold team
        const int tf = tid, wf = tf >> 5, nwf = NF >> 5;
        for (int k = 0; k < R; k++) {
            const int b = k % Q;
            const uint32_t par = (uint32_t)(k / Q) & 1u, buf = seg0 + (uint32_t)b * a.buf;
            const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, k, a.cols);
            const Share sh = share_of<DT, ALIGNED>(g, a.cols, P, p, tf);
            const int n = (int)(sh.fe - sh.fb);
            const int piece = (n + kPipePieces - 1) / kPipePieces;
            const uint4 edge = sh.edge_k >= 0 ? load_chunk<DT, ALIGNED>(g, sh.edge_k, a.cols) : neg_inf_chunk<DT>();
            float4 partial = make_float4(-INFINITY, 0.f, 0.f, 0.f);
            if constexpr (DT == kF32) {
                // fp32: the share's max, then the compensated sum of exp(x - max)
                bool ok = true;
                for (int i = 0; i < kPipePieces && i * piece < n && ok; i++)
                    ok = mbar_wait(bar0 + 8u * (kPipePieces * b + i), par, &abort_flag);
                if (!ok) {
                    if (!abort_flag)
                        atomicOr(a.err, kErrFullWait);
                    abort_flag = 1;
                }
                float mx = chunk_max<DT>(edge);
                if (!abort_flag) {
                    float mx2 = -INFINITY;
                    int c = tf;
                    for (; c + NF < n; c += 2 * NF) {
                        mx = fmaxf(mx, chunk_max<DT>(lds_chunk(buf + 16u * (uint32_t)c)));
                        mx2 = fmaxf(mx2, chunk_max<DT>(lds_chunk(buf + 16u * (uint32_t)(c + NF))));
                    }
                    if (c < n)
                        mx = fmaxf(mx, chunk_max<DT>(lds_chunk(buf + 16u * (uint32_t)c)));
                    mx = fmaxf(mx, mx2);
                }
                mx = warp_max_redux(mx);
                if (lane == 0)
                    fslot[k & 1][wf].x = mx;
                named_sync(1, NF);
                mx = -INFINITY;
                for (int w = 0; w < nwf; w++)
                    mx = fmaxf(mx, fslot[k & 1][w].x);
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
                    for (int c = tf; c < n; c += NF) {
                        chunk_exp<DT>(lds_chunk(buf + 16u * (uint32_t)c), mx, f);
#pragma unroll
                        for (int e = 0; e < E; e++)
                            M::add(acc[e], f[e]);
                    }
                }
                CSum tot = M::merge(M::merge(acc[0], acc[1]), M::merge(acc[2], acc[3]));
                tot = group_sum<DT, 32>(tot);
                if (lane == 0) {
                    fslot[k & 1][wf].y = tot.s;
                    fslot[k & 1][wf].z = tot.c;
                }
                named_sync(1, NF);
                if (tf == 0) {
                    CSum all = M::zero();
                    for (int w = 0; w < nwf; w++)
                        all = M::merge(all, CSum{fslot[k & 1][w].y, fslot[k & 1][w].z});
                    partial = make_float4(mx, all.s, all.c, 0.f);
                }
            } else {
                // 16-bit: one online (m, d) pass, each piece as it lands
                MD md{-INFINITY, 0.f};
                {
                    uint4 one[1] = {edge};
                    md_absorb<DT, 1>(md, one);
                }
                for (int i = 0; i < kPipePieces && i * piece < n; i++) {
                    if (!mbar_wait(bar0 + 8u * (kPipePieces * b + i), par, &abort_flag)) {
                        if (!abort_flag)
                            atomicOr(a.err, kErrFullWait);
                        abort_flag = 1;
                    }
                    if (abort_flag)
                        break;
                    const int c0 = i * piece, c1 = n - c0 < piece ? n : c0 + piece;
                    // K chunks a step while a thread has K, then one at a time:
                    // no exps spent on padding
                    int c = c0 + tf;
                    for (; c + (K - 1) * NF < c1; c += NF * K) {
                        uint4 raw[K];
#pragma unroll
                        for (int u = 0; u < K; u++)
                            raw[u] = lds_chunk(buf + 16u * (uint32_t)(c + u * NF));
                        md_absorb<DT, K>(md, raw);
                    }
                    for (; c < c1; c += NF) {
                        uint4 one[1] = {lds_chunk(buf + 16u * (uint32_t)c)};
                        md_absorb<DT, 1>(md, one);
                    }
                }
                md = warp_md_max_first<DT>(md);
                if (lane == 0)
                    fslot[k & 1][wf] = make_float4(md.m, md.d, 0.f, 0.f);
                named_sync(1, NF);
                if (tf == 0) {
                    MD all{-INFINITY, 0.f};
                    for (int w = 0; w < nwf; w++)
                        all = md_merge<DT>(all, MD{fslot[k & 1][w].x, fslot[k & 1][w].y});
                    partial = make_float4(all.m, all.d, 0.f, 0.f);
                }
            }
            if (tf == 0 && !abort_flag) {
                pending[b] = -1;
                grid_publish(a, k, p, partial);
            }
        }
    } else {
        // ---------------- write team
        const int to = tid - NF, wo = to >> 5, NO = blockDim.x - NF;
        for (int k = 0; k < R; k++) {
            const int b = k % Q;
            const uint32_t buf = seg0 + (uint32_t)b * a.buf;
            if (wo == 0) {
                int ok = 1;
                if (lane == 0 && !abort_flag)
                    ok = grid_wait_row(a, k) ? 1 : 0;
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);  // (also orders lane 0's acquire before the loads)
                if (!ok && lane == 0) {
                    atomicOr(a.err, kErrGridWait);
                    abort_flag = 1;
                }
                __syncwarp();
                if (!abort_flag) {
                    float m, inv;
                    merge_partials_warp<DT>(a.part, k, P, m, inv);
                    if (lane == 0)
                        mrow[k & 1] = make_float2(m, inv);
                }
            }
            named_sync(2, NO);
            if (!abort_flag) {
                const float m = mrow[k & 1].x, inv = mrow[k & 1].y;
                const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, k, a.cols);
                const Share sh = share_of<DT, ALIGNED>(g, a.cols, P, p, to);
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
                for (int c = to; c < n; c += NO) {
                    float f[E];
                    chunk_exp<DT>(lds_chunk(buf + 16u * (uint32_t)c), m, f);
#pragma unroll
                    for (int e = 0; e < E; e++)
                        f[e] *= inv;
                    store_chunk<DT, ALIGNED>(g, sh.fb + c, a.cols, pack<DT>(f), a.y_vec != 0);
                }
            }
            named_sync(2, NO);  // buffer b is consumed
            if (to == 0 && !abort_flag && k + Q < R) {
                pending[b] = k + Q;
                grid_issue<DT, ALIGNED, kPipePieces>(a, k + Q, p, buf, bar0 + 8u * kPipePieces * b);
            }
        }
    }
    __syncthreads();
    if (abort_flag) {
        if (tid == 0) {
            // no copy may still be landing in shared memory when the CTA leaves
            for (int b = 0; b < Q; b++) {
                if (pending[b] < 0)
                    continue;
                const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, pending[b], a.cols);
                const Share sh = share_of<DT, ALIGNED>(g, a.cols, P, p, 0);
                const int n = (int)(sh.fe - sh.fb), piece = (n + kPipePieces - 1) / kPipePieces;
                for (int i = 0; i < kPipePieces && i * piece < n; i++)
                    (void)mbar_wait(bar0 + 8u * (kPipePieces * b + i), (uint32_t)(pending[b] / Q) & 1u, &abort_flag,
                                    false);
            }
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

// FORM: 0 streaming, 1 ring, 2 pipelined
template <int DT, bool A, int FORM>
int grid_launch_one(const Launch &l, const GridArgs &args)
{
    constexpr bool RES = FORM >= 1;  // shares held in shared memory
    auto kern = FORM == 2 ? &k_grid_pipe<DT, A> : (FORM == 1 ? &k_grid_ring<DT, A> : &k_grid_stream<DT, A>);
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
    const int form = l.plan.stages < 1 ? 0 : (l.plan.lanes_per_row > 0 ? 2 : 1);
    if (l.plan.aligned)
        return form == 2 ? grid_launch_one<DT, true, 2>(l, args)
                         : (form == 1 ? grid_launch_one<DT, true, 1>(l, args) : grid_launch_one<DT, true, 0>(l, args));
    return form == 2 ? grid_launch_one<DT, false, 2>(l, args)
                     : (form == 1 ? grid_launch_one<DT, false, 1>(l, args) : grid_launch_one<DT, false, 0>(l, args));
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
                  l.dev_err, Q > 0 ? l.plan.lanes_per_row : 0};
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
