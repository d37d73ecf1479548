// k_stream.cu -- STREAM: rows too long to cache on chip, many of them.
//
// One CTA per row.  For fp16 / bf16 a first pass keeps a per-thread
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
// Where the rows in flight outgrow L2, the re-read of a row misses if every
// pass walks it forward: each chunk is read again a whole pass after its first
// read.  The plan then asks (back_passes = 1) for each pass after the first
// to walk the row from the other end, so that it starts on the chunks read
// last, still in L2, and only the chunks read longest ago come from HBM again
// (16-bit: forward, then backward; fp32: forward, backward, forward).  Those
// launches also mark the lines of every pass but the last evict-last in L2
// and the last pass's evict-first (rows on the 16-byte grid), which keeps
// still more of a row for its re-read (measured: [4096, 131072] bf16 409.0 ->
// 370.5 us, [2048, 131072] bf16 206.3 -> 191.6, [2048, 262144] fp16 441.4 ->
// 415.6; fp32 within 1.5 %); forward launches keep plain loads (with the
// policies, [4096, 65600] fp16 was 4 % slower).
//
#include "common.cuh"
#include "launch.h"
#include "stream_passes.cuh"

namespace osd {

// A pass over chunks [0, nch) of a row taken step by step from the last
// step: step s covers chunks [s span, (s + 1) span), span = blockDim x kStep,
// and is handed to the pass function as a range of its own (one step each).
template <int DT, bool ALIGNED>
__device__ __forceinline__ typename Math<DT>::Acc sum_backward(const RowGeom &g, int64_t cols, float m)
{
    using M = Math<DT>;
    const int64_t span = (int64_t)blockDim.x * kStep;
    typename M::Acc acc = M::zero();
    for (int64_t lo = g.nch > 0 ? (g.nch - 1) / span * span : -1; lo >= 0; lo -= span)
        acc = M::merge(acc, pass_sum<DT, ALIGNED, kStep, 1>(g, lo, lo + span < g.nch ? lo + span : g.nch, cols, m));
    return acc;
}

template <int DT, bool ALIGNED>
__device__ __forceinline__ void write_backward(const RowGeom &g, int64_t cols, float m, float inv, bool y_vec)
{
    const int64_t span = (int64_t)blockDim.x * kStep;
    for (int64_t lo = g.nch > 0 ? (g.nch - 1) / span * span : -1; lo >= 0; lo -= span)
        pass_write<DT, ALIGNED, kStep, 2>(g, lo, lo + span < g.nch ? lo + span : g.nch, cols, m, inv, y_vec);
}

// BACK: the passes after the first alternate direction (see above).  Two
// CTAs per SM for every instance: rows off the 16-byte grid (98 - 116
// registers unbounded, one CTA per SM) then spill 8 - 24 bytes but keep twice
// the loads in flight (measured: [4096, 65599] fp16 330.8 -> 261.0 us,
// [2048, 131071] fp16 288.7 -> 254.3, [1024, 262143] fp32 801.1 -> 714.6,
// [512, 1048575] fp16 594.4 -> 546.7).
template <int DT, bool ALIGNED, bool BACK>
__global__ void __launch_bounds__(kStreamThreads, 2)
    k_stream(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols, int y_vec)
{
    pdl_enter();
    using M = Math<DT>;
    __shared__ float smax[32];
    __shared__ typename M::Acc ssum[32];
    __shared__ MD smd[32];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const RowGeom g = row_geom<DT, ALIGNED>(x, y, r, cols);
        // L2 policies of the passes' loads (with the backward walk only):
        // evict-last, then evict-first for the last pass
        constexpr int KEEP = BACK ? 1 : 0, LAST = BACK ? 2 : 0;
        if constexpr (DT == kF32) {
            const float m = block_max(pass_max<DT, ALIGNED, kStep, KEEP>(g, 0, g.nch, cols), smax);
            typename M::Acc acc;
            if constexpr (BACK)
                acc = sum_backward<DT, ALIGNED>(g, cols, m);
            else
                acc = pass_sum<DT, ALIGNED>(g, 0, g.nch, cols, m);
            const float inv = 1.0f / M::value(block_sum<DT>(acc, ssum));
            pass_write<DT, ALIGNED, kStep, LAST>(g, 0, g.nch, cols, m, inv, y_vec != 0);
        } else {
            const MD md = block_md<DT>(pass_online<DT, ALIGNED, kStep, KEEP>(g, 0, g.nch, cols), smd);
            const float inv = 1.0f / md.d;
            if constexpr (BACK)
                write_backward<DT, ALIGNED>(g, cols, md.m, inv, y_vec != 0);
            else
                pass_write<DT, ALIGNED>(g, 0, g.nch, cols, md.m, inv, y_vec != 0);
        }
    }
}

namespace {

template <int DT, bool A, bool BACK>
int launch_stream_one(const Launch &l)
{
    return launch_pdl(k_stream<DT, A, BACK>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), (const char *)l.x, (char *)l.y, l.rows, l.cols,
                      (int)l.plan.y_vector);
}

template <int DT>
int stream_dt(const Launch &l)
{
    if (l.plan.back_passes == 1)
        return l.plan.aligned ? launch_stream_one<DT, true, true>(l) : launch_stream_one<DT, false, true>(l);
    return l.plan.aligned ? launch_stream_one<DT, true, false>(l) : launch_stream_one<DT, false, false>(l);
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

}  // namespace osd
