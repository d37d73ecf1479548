// k_splitk.cu -- few rows, huge cols: a thread-block cluster of C CTAs per row
// (grid = C x rows), each CTA streaming a contiguous 1/C of its row through a
// ring of shared-memory stages filled by 1-D bulk async copies.
//
// Prior art: the split-k kernels of "[CUDA] safe online softmax", section 3.2
// (pass 1 writes per-block (m, d) partials to a global workspace, pass 2 --
// a second launch -- merges them and writes; the single-kernel alternatives,
// a cooperative grid sync or atomics plus polling, are rejected there), and
// the multi-block large-cols pipeline of the HIP softmax tutorial, section 6
// (five kernels).  Here one launch does it, with no workspace:
//
// * Warp 0 (one lane) is the producer: it copies the CTA's segment, 32 KB per
//   cp.async.bulk, into 6 stages -- 192 KB of HBM reads in flight per SM --
//   once per pass; 16 consumer warps process each landed stage and release it.
// * Passes: fp16 / bf16 take one online pass (per thread (m, d), rescaled by
//   e^(m - m') when the max grows, "[CUDA] safe online softmax", section 1)
//   and one write pass; fp32 takes a max pass, a sum pass with that fixed max
//   (compensated) and a write pass, because each rescale of a partial sum
//   would cost up to an fp32 ulp.  Later passes re-read the segment, from L2
//   when the rows fit there; the producer starts a pass's copies while the
//   consumers are still merging the previous pass's statistics.  With one
//   CTA per row (many long rows), the copies of every pass but the last mark
//   their lines evict-last in L2 and the last pass's evict-first, so that
//   more of a row is still in L2 when it is read again (measured: [2048,
//   262144] fp16 424.5 -> 404.2 us, [608, 262144] fp16 137.2 -> 131.0, fp32
//   [1024, 262144] 714 -> 702; [3072, 196608] fp16 445.7 -> 448.5, within
//   noise; with clusters of 4 - 16 on few rows, no change, so they keep
//   plain copies).
// * Merge: each CTA's consumer leader stores its partial statistics into
//   every cluster peer's shared memory (distributed shared memory) and
//   arrives on the peer's mbarrier; every CTA waits for its C arrivals and
//   merges the C partials in rank order, so all C CTAs of a row hold
//   bit-identical statistics.
// * Every wait is bounded (tma.cuh).  A wait that gives up sets the CTA's
//   abort flag; the remaining waits then fail at once, so every warp still
//   walks the same sequence of barriers and the kernel returns.
#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

#include <atomic>

namespace osd {

constexpr int kSplitChunksPerStage = kSplitStageBytes / 16;

// An L2 access policy that marks lines evict-last.
__device__ __forceinline__ uint64_t l2_evict_last()
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy for the lines it reads.
__device__ __forceinline__ void bulk_g2s_policy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                                uint64_t pol)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
                 "[%3], %4;" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar), "l"(pol)
                 : "memory");
}
constexpr int kSplitConsumers = 32 * kSplitConsumerWarps;

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kSplitThreads, 1)
    k_splitk(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols, int y_vec,
             unsigned *err)
{
    pdl_enter();
    using M = Math<DT>;
    using Acc = typename M::Acc;
    constexpr int E = Fmt<DT>::kPerChunk;
    constexpr int P = DT == kF32 ? 3 : 2;  // passes over the segment
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full_bar[kSplitStages];
    __shared__ __align__(8) uint64_t empty_bar[kSplitStages];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ __align__(8) float2 slots[2][kMaxCluster];
    __shared__ float red_a[kSplitConsumerWarps];
    __shared__ float red_b[kSplitConsumerWarps];
    __shared__ volatile int abort_flag;

    const uint32_t C = cluster_nctarank(), rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = blockIdx.y;  // grid.y == rows
    const RowGeom g = row_geom<DT, ALIGNED>(x, y, r, cols);
    const int64_t per = (g.nch + C - 1) / C;
    const int64_t kb = per * rank < g.nch ? per * rank : g.nch;
    const int64_t ke = kb + per < g.nch ? kb + per : g.nch;
    // chunks lying wholly inside the row go through the ring; a partial first
    // or last chunk of the row is read with scalar loads
    const int64_t first_whole = ALIGNED || g.head == 0 ? 0 : 1;
    const int64_t end_whole = ALIGNED || (g.head + cols) % E == 0 ? g.nch : g.nch - 1;
    const int64_t fb = kb > first_whole ? kb : first_whole;
    int64_t fe = ke < end_whole ? ke : end_whole;
    if (fe < fb)
        fe = fb;
    const uint32_t npieces = (uint32_t)((fe - fb + kSplitChunksPerStage - 1) / kSplitChunksPerStage);
    const uint32_t ring0 = smem_u32(ring);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSplitStages; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), kSplitConsumerWarps);
        }
        mbar_init(smem_u32(&xbar[0]), C);
        mbar_init(smem_u32(&xbar[1]), C);
        abort_flag = 0;
        mbar_init_fence();
    }
    // peers arrive on xbar: every CTA's barriers must exist before any arrival
    cluster_sync_all();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            uint32_t pending = 0, pend_parity = 0;
            for (uint32_t i = 0; i < P * npieces; i++) {
                const uint32_t s = i % kSplitStages, u = i / kSplitStages;
                if (u > 0 && !mbar_wait(smem_u32(&empty_bar[s]), (u - 1) & 1, &abort_flag)) {
                    atomicOr(err, kErrEmptyWait);
                    abort_flag = 1;
                    break;
                }
                const int64_t c0 = fb + (int64_t)(i % npieces) * kSplitChunksPerStage;
                const int64_t n = fe - c0 < kSplitChunksPerStage ? fe - c0 : kSplitChunksPerStage;
                const uint32_t fbar = smem_u32(&full_bar[s]);
                mbar_arrive_expect_tx(fbar, (uint32_t)(16 * n));
                if (C == 1)
                    bulk_g2s_policy(ring0 + s * kSplitStageBytes, g.x0 + 16 * c0, (uint32_t)(16 * n), fbar,
                                    i / npieces + 1 < (uint32_t)P ? l2_evict_last() : l2_evict_first());
                else
                    bulk_g2s(ring0 + s * kSplitStageBytes, g.x0 + 16 * c0, (uint32_t)(16 * n), fbar);
                pending |= 1u << s;
                pend_parity = (pend_parity & ~(1u << s)) | ((u & 1) << s);
            }
            // retire no copy in flight: wait (bounded) for the last one per stage
            for (int s = 0; s < kSplitStages; s++)
                if (pending & (1u << s))
                    (void)mbar_wait(smem_u32(&full_bar[s]), (pend_parity >> s) & 1, &abort_flag, false);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- consumers
        const int tid = threadIdx.x - 32;
        const int cw = warp - 1;
        uint32_t item = 0;

        // Wait for stage `item`; a give-up marks the CTA aborted (later waits
        // then fail at once) and the stage is treated as empty.
        auto acquire = [&](uint32_t it) -> bool {
            const uint32_t s = it % kSplitStages;
            if (mbar_wait(smem_u32(&full_bar[s]), (it / kSplitStages) & 1, &abort_flag))
                return true;
            if (lane == 0 && !abort_flag) {
                atomicOr(err, kErrFullWait);
                abort_flag = 1;
            }
            return false;
        };
        auto release = [&](uint32_t it) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&empty_bar[it % kSplitStages]));
        };
        auto piece_bounds = [&](uint32_t it, int64_t &c0, int64_t &n) {
            c0 = fb + (int64_t)(it % npieces) * kSplitChunksPerStage;
            n = fe - c0 < kSplitChunksPerStage ? fe - c0 : kSplitChunksPerStage;
        };
        // the partial first / last chunk of the row, if it is this CTA's:
        // handled by consumer threads 0 and 1
        const int64_t edge_k = tid == 0 ? 0 : g.nch - 1;
        const bool has_edge = tid < 2 && (tid == 0 ? first_whole == 1 : end_whole == g.nch - 1) &&
                              edge_k >= kb && edge_k < ke && !(tid == 1 && g.nch == 1 && first_whole == 1);

        // publish (a, b) in slot `rank` of every cluster CTA's slots[q], then
        // wait until all C CTAs have published theirs into ours
        auto exchange = [&](int q, float a, float b) {
            if (tid == 0) {
                const uint32_t sa = smem_u32(&slots[q][rank]), xa = smem_u32(&xbar[q]);
                for (uint32_t j = 0; j < C; j++) {
                    st_cluster_f32x2(mapa(sa, j), a, b);
                    mbar_arrive_cluster(mapa(xa, j));
                }
            }
            if (!mbar_wait_cluster(smem_u32(&xbar[q]), 0, &abort_flag) && tid == 0) {
                atomicOr(err, kErrPeerWait);
                abort_flag = 1;
            }
        };

        float m, inv;
        if constexpr (DT == kF32) {
            // pass 0: max
            float mt = -INFINITY;
            if (has_edge)
                mt = chunk_max<DT>(load_chunk<DT, ALIGNED>(g, edge_k, cols));
            for (uint32_t p = 0; p < npieces; p++, item++) {
                if (acquire(item)) {
                    int64_t c0, n;
                    piece_bounds(item, c0, n);
                    const uint32_t sb = ring0 + (item % kSplitStages) * kSplitStageBytes;
                    for (int64_t c = tid; c < n; c += kSplitConsumers)
                        mt = fmaxf(mt, chunk_max<DT>(lds_chunk(sb + 16 * (uint32_t)c)));
                }
                release(item);
            }
            mt = warp_max_redux(mt);
            if (lane == 0)
                red_a[cw] = mt;
            named_sync(1, kSplitConsumers);
            mt = warp_max_redux(lane < kSplitConsumerWarps ? red_a[lane] : -INFINITY);
            named_sync(1, kSplitConsumers);
            exchange(0, mt, 0.f);
            m = -INFINITY;
            for (uint32_t j = 0; j < C; j++)
                m = fmaxf(m, slots[0][j].x);

            // pass 1: compensated sum of exp(x - m)
            Acc acc = M::zero();
            if (has_edge) {
                float f[E];
                chunk_exp<DT>(load_chunk<DT, ALIGNED>(g, edge_k, cols), m, f);
#pragma unroll
                for (int e = 0; e < E; e++)
                    M::add(acc, f[e]);
            }
            for (uint32_t p = 0; p < npieces; p++, item++) {
                if (acquire(item)) {
                    int64_t c0, n;
                    piece_bounds(item, c0, n);
                    const uint32_t sb = ring0 + (item % kSplitStages) * kSplitStageBytes;
                    for (int64_t c = tid; c < n; c += kSplitConsumers) {
                        float f[E];
                        chunk_exp<DT>(lds_chunk(sb + 16 * (uint32_t)c), m, f);
#pragma unroll
                        for (int e = 0; e < E; e++)
                            M::add(acc, f[e]);
                    }
                }
                release(item);
            }
            acc = group_sum<DT, 32>(acc);
            if (lane == 0) {
                red_a[cw] = acc.s;
                red_b[cw] = acc.c;
            }
            named_sync(1, kSplitConsumers);
            acc = group_sum<DT, 32>(lane < kSplitConsumerWarps ? CSum{red_a[lane], red_b[lane]} : M::zero());
            named_sync(1, kSplitConsumers);
            exchange(1, acc.s, acc.c);
            Acc tot = M::zero();
            for (uint32_t j = 0; j < C; j++)
                tot = M::merge(tot, CSum{slots[1][j].x, slots[1][j].y});
            inv = 1.0f / M::value(tot);
        } else {
            // pass 0: online (m, d)
            constexpr int kPer = kSplitChunksPerStage / kSplitConsumers;  // chunks per thread per stage
            MD md{-INFINITY, 0.f};
            // fold K chunks into (m, d); all -inf chunks (slots outside the
            // segment, or genuine -inf inputs) leave it unchanged
            auto absorb = [&](const uint4(&raw)[kPer], int K) {
                float mt = -INFINITY;
#pragma unroll
                for (int u = 0; u < kPer; u++)
                    if (u < K)
                        mt = fmaxf(mt, chunk_max<DT>(raw[u]));
                if (mt == -INFINITY)
                    return;
                if (mt > md.m) {
                    md.d = md.m == -INFINITY ? 0.f : md.d * M::exp_of(md.m - mt);
                    md.m = mt;
                }
                float s = 0.f;
#pragma unroll
                for (int u = 0; u < kPer; u++) {
                    if (u < K) {
                        float f[E];
                        chunk_exp<DT>(raw[u], md.m, f);
#pragma unroll
                        for (int e = 0; e < E; e++)
                            s += f[e];
                    }
                }
                md.d += s;
            };
            if (has_edge) {
                uint4 raw[kPer];
                raw[0] = load_chunk<DT, ALIGNED>(g, edge_k, cols);
                absorb(raw, 1);
            }
            for (uint32_t p = 0; p < npieces; p++, item++) {
                if (acquire(item)) {
                    int64_t c0, n;
                    piece_bounds(item, c0, n);
                    const uint32_t sb = ring0 + (item % kSplitStages) * kSplitStageBytes;
                    uint4 raw[kPer];
#pragma unroll
                    for (int u = 0; u < kPer; u++) {
                        const int64_t c = tid + (int64_t)u * kSplitConsumers;
                        raw[u] = c < n ? lds_chunk(sb + 16 * (uint32_t)c) : neg_inf_chunk<DT>();
                    }
                    absorb(raw, kPer);
                }
                release(item);
            }
            md = warp_md<DT>(md);
            if (lane == 0) {
                red_a[cw] = md.m;
                red_b[cw] = md.d;
            }
            named_sync(1, kSplitConsumers);
            md = warp_md<DT>(lane < kSplitConsumerWarps ? MD{red_a[lane], red_b[lane]} : MD{-INFINITY, 0.f});
            named_sync(1, kSplitConsumers);
            exchange(0, md.m, md.d);
            MD tot{-INFINITY, 0.f};
            for (uint32_t j = 0; j < C; j++)
                tot = md_merge<DT>(tot, MD{slots[0][j].x, slots[0][j].y});
            m = tot.m;
            inv = 1.0f / tot.d;
        }

        // last pass: write exp(x - m) / d
        if (has_edge) {
            float f[E];
            chunk_exp<DT>(load_chunk<DT, ALIGNED>(g, edge_k, cols), m, f);
#pragma unroll
            for (int e = 0; e < E; e++)
                f[e] *= inv;
            store_chunk<DT, ALIGNED>(g, edge_k, cols, pack<DT>(f), y_vec != 0);
        }
        for (uint32_t p = 0; p < npieces; p++, item++) {
            if (acquire(item)) {
                int64_t c0, n;
                piece_bounds(item, c0, n);
                const uint32_t sb = ring0 + (item % kSplitStages) * kSplitStageBytes;
                for (int64_t c = tid; c < n; c += kSplitConsumers) {
                    float f[E];
                    chunk_exp<DT>(lds_chunk(sb + 16 * (uint32_t)c), m, f);
#pragma unroll
                    for (int e = 0; e < E; e++)
                        f[e] *= inv;
                    store_chunk<DT, ALIGNED>(g, c0 + c, cols, pack<DT>(f), y_vec != 0);
                }
            }
            release(item);
        }
    }
    // no CTA leaves while a peer may still touch its shared memory
    __syncwarp();
    cluster_sync_all();
}

namespace {

template <int DT, bool A>
int splitk_prepare(int cluster)
{
    // opt in once per device: dynamic shared memory above 48 KB, and clusters
    // above the portable 8
    static std::atomic<int> done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return (int)e;
    if (dev < 0 || dev >= 64)
        return (int)cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire))
        return 0;
    auto *kern = &k_splitk<DT, A>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitStages * kSplitStageBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
        return (int)e;
    (void)cluster;
    done[dev].store(1, std::memory_order_release);
    return 0;
}

template <int DT, bool A>
int splitk_launch_one(const Launch &l)
{
    const int C = l.plan.cluster_x;
    int rc = splitk_prepare<DT, A>(C);
    if (rc != 0)
        return rc;
    cudaLaunchAttribute cluster = {};
    cluster.id = cudaLaunchAttributeClusterDimension;
    cluster.val.clusterDim.x = (unsigned)C;
    cluster.val.clusterDim.y = 1;
    cluster.val.clusterDim.z = 1;
    return launch_pdl(k_splitk<DT, A>, dim3((unsigned)l.plan.grid_x, (unsigned)l.plan.grid_y, 1), dim3(kSplitThreads),
                      (size_t)(kSplitStages * kSplitStageBytes), (cudaStream_t)l.stream, cluster, (const char *)l.x,
                      (char *)l.y, l.rows, l.cols, (int)l.plan.y_vector, l.dev_err);
}

template <int DT>
int splitk_dt(const Launch &l)
{
    return l.plan.aligned ? splitk_launch_one<DT, true>(l) : splitk_launch_one<DT, false>(l);
}

}  // namespace

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
