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
// * Resident form (fp16 / bf16 rows whose share fits shared memory, one CTA
//   per SM): the CTA's segment is copied into shared memory by bulk copies in
//   kGridPieces pieces, the online (m, d) pass starts on each piece as it
//   lands, and after the barrier the output is computed from shared memory:
//   x is read from HBM once.
// * Streaming form (fp32, or longer shares; two CTAs per SM): the passes of
//   the two-launch split (stream_passes.cuh) around the barrier; the write pass
//   re-reads x, from L2 when the rows fit there.
// * Barrier: each row has two arrival counters used by alternate launches of a
//   slot (the launch's generation number picks one); a CTA stores its
//   partial, adds one to the launch's counter with release semantics and
//   waits -- for at most kWaitLimitNs of %globaltimer time -- until an acquire
//   load of it reads P.  The first CTA of each row zeroes the other counter,
//   ready for the slot's next launch (the previous launch that used it has
//   finished), so a launch that gave up leaves nothing stale behind.  A wait
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
constexpr int kGridPieces = 8;         // bulk copies per resident segment, consumed as they land

struct GridArgs {
    const char *x;
    char *y;
    int64_t rows;
    int64_t cols;
    int P;  // CTAs per row
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

// Zero the row's counter of the slot's next launch (first CTA of the row).
__device__ __forceinline__ void grid_prepare_next(const GridArgs &a, int64_t r, int p)
{
    if (p == 0 && threadIdx.x == 0)
        a.arrive[2 * r + ((a.gen + 1u) & 1u)] = 0u;
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
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < K; u++) {
        float f[E];
        chunk_exp<DT>(raw[u], md.m, f);
#pragma unroll
        for (int e = 0; e < E; e++)
            s += f[e];
    }
    md.d += s;
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kGridThreads, 1) k_grid_resident(const GridArgs a)
{
    pdl_enter();
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int K = 4;  // chunks per thread per step
    extern __shared__ __align__(128) unsigned char seg[];
    __shared__ __align__(8) uint64_t bars[kGridPieces];
    __shared__ MD smd[32];
    __shared__ volatile int abort_flag;
    const int64_t r = blockIdx.y;
    const int p = blockIdx.x;
    const int tid = threadIdx.x, T = blockDim.x;
    const RowGeom g = row_geom<DT, ALIGNED>(a.x, a.y, r, a.cols);
    const Share sh = share_of<DT, ALIGNED>(g, a.cols, a.P, p, tid);
    grid_prepare_next(a, r, p);
    const int n = (int)(sh.fe - sh.fb);  // whole chunks held in shared memory
    const int piece = (n + kGridPieces - 1) / kGridPieces;
    const uint32_t seg0 = smem_u32(seg);

    if (tid == 0) {
        for (int i = 0; i < kGridPieces; i++)
            mbar_init(smem_u32(&bars[i]), 1);
        abort_flag = 0;
        mbar_init_fence();
        for (int i = 0; i < kGridPieces; i++) {
            const int c0 = i * piece, cnt = n - c0 < piece ? n - c0 : piece;
            if (cnt <= 0)
                break;
            mbar_arrive_expect_tx(smem_u32(&bars[i]), (uint32_t)(16 * cnt));
            bulk_g2s(seg0 + 16u * (uint32_t)c0, g.x0 + 16 * (sh.fb + c0), (uint32_t)(16 * cnt), smem_u32(&bars[i]));
        }
    }
    __syncthreads();

    const uint4 edge = sh.edge_k >= 0 ? load_chunk<DT, ALIGNED>(g, sh.edge_k, a.cols) : neg_inf_chunk<DT>();
    MD md{-INFINITY, 0.f};
    {
        uint4 one[1] = {edge};
        md_absorb<DT, 1>(md, one);
    }
    for (int i = 0; i < kGridPieces; i++) {
        const int c0 = i * piece, cnt = n - c0 < piece ? n - c0 : piece;
        if (cnt <= 0)
            break;
        if (!mbar_wait(smem_u32(&bars[i]), 0, &abort_flag)) {
            if (tid == 0 && !abort_flag) {
                atomicOr(a.err, kErrFullWait);
                abort_flag = 1;
            }
            break;
        }
        for (int c = c0 + tid; c < c0 + cnt; c += T * K) {
            uint4 raw[K];
#pragma unroll
            for (int u = 0; u < K; u++) {
                const int cc = c + u * T;
                raw[u] = cc < c0 + cnt ? lds_chunk(seg0 + 16u * (uint32_t)cc) : neg_inf_chunk<DT>();
            }
            md_absorb<DT, K>(md, raw);
        }
    }
    md = block_md<DT>(md, smd);
    if (tid == 0 && !abort_flag && !grid_row_barrier(a, r, p, make_float4(md.m, md.d, 0.f, 0.f))) {
        atomicOr(a.err, kErrGridWait);
        abort_flag = 1;
    }
    __syncthreads();
    if (abort_flag) {
        // no copy may still be landing in shared memory when the CTA leaves
        if (tid == 0)
            for (int i = 0; i < kGridPieces && i * piece < n; i++)
                (void)mbar_wait(smem_u32(&bars[i]), 0, &abort_flag, false);
        __syncthreads();
        return;
    }
    __threadfence();
    float m, inv;
    merge_partials<DT>(a.part, r, a.P, m, inv);

    if (sh.edge_k >= 0) {
        float f[E];
        chunk_exp<DT>(edge, m, f);
#pragma unroll
        for (int e = 0; e < E; e++)
            f[e] *= inv;
        store_chunk<DT, ALIGNED>(g, sh.edge_k, a.cols, pack<DT>(f), a.y_vec != 0);
    }
    for (int c = tid; c < n; c += T) {
        float f[E];
        chunk_exp<DT>(lds_chunk(seg0 + 16u * (uint32_t)c), m, f);
#pragma unroll
        for (int e = 0; e < E; e++)
            f[e] *= inv;
        store_chunk<DT, ALIGNED>(g, sh.fb + c, a.cols, pack<DT>(f), a.y_vec != 0);
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
    grid_prepare_next(a, r, p);
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
    std::once_flag once;
    cudaError_t status = cudaSuccess;
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

void pool_init(GridPool &pl)
{
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_grid_part);
    pl.part = static_cast<float4 *>(p);
    if (e == cudaSuccess)
        e = cudaGetSymbolAddress(&p, g_grid_arrive);
    pl.arrive = static_cast<unsigned *>(p);
    for (int i = 0; i < kGridSlots && e == cudaSuccess; i++)
        e = cudaEventCreateWithFlags(&pl.ev[i], cudaEventDisableTiming);
    pl.status = e;
}

template <int DT, bool A, bool RES>
int grid_launch_one(const Launch &l, const GridArgs &args)
{
    auto kern = RES ? &k_grid_resident<DT, A> : &k_grid_stream<DT, A>;
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
    const bool res = l.plan.stages == 1;
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
    std::call_once(pl.once, pool_init, std::ref(pl));  // device d is current here
    if (pl.status != cudaSuccess)
        return (int)pl.status;
    if (l.plan.grid_y > kGridMaxRows || l.plan.grid_x * l.plan.grid_y > kGridMaxPartials)
        return (int)cudaErrorInvalidValue;
    const unsigned s = pl.next.fetch_add(1, std::memory_order_relaxed) % kGridSlots;
    std::lock_guard<std::mutex> lock(pl.mu[s]);
    cudaStream_t st = (cudaStream_t)l.stream;
    // the slot's previous launch has finished before this one starts: stream
    // order on the same stream, its event on another
    if (pl.used[s] && pl.last[s] != st && (e = cudaStreamWaitEvent(st, pl.ev[s], 0)) != cudaSuccess)
        return (int)e;
    const unsigned gen = pl.gen[s] + 1u;
    GridArgs args{(const char *)l.x, (char *)l.y, l.rows, l.cols, (int)l.plan.grid_x, l.plan.y_vector,
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
    if (!pl.arrive || pl.status != cudaSuccess)
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
