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
#include "common.cuh"
#include "launch.h"
#include "stream_passes.cuh"

namespace osd {

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kStreamThreads)
    k_stream(const char *__restrict__ x, char *__restrict__ y, int64_t rows, int64_t cols, int y_vec)
{
    pdl_enter();
    using M = Math<DT>;
    __shared__ float smax[32];
    __shared__ typename M::Acc ssum[32];
    __shared__ MD smd[32];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const RowGeom g = row_geom<DT, ALIGNED>(x, y, r, cols);
        float m, inv;
        if constexpr (DT == kF32) {
            m = block_max(pass_max<DT, ALIGNED>(g, 0, g.nch, cols), smax);
            const auto acc = block_sum<DT>(pass_sum<DT, ALIGNED>(g, 0, g.nch, cols, m), ssum);
            inv = 1.0f / M::value(acc);
        } else {
            const MD md = block_md<DT>(pass_online<DT, ALIGNED>(g, 0, g.nch, cols), smd);
            m = md.m;
            inv = 1.0f / md.d;
        }
        pass_write<DT, ALIGNED>(g, 0, g.nch, cols, m, inv, y_vec != 0);
    }
}

namespace {

template <int DT, bool A>
int launch_stream_one(const Launch &l)
{
    return launch_pdl(k_stream<DT, A>, dim3((unsigned)l.plan.grid_x), dim3(l.plan.block_threads), 0,
                      (cudaStream_t)l.stream, no_attr(), (const char *)l.x, (char *)l.y, l.rows, l.cols,
                      (int)l.plan.y_vector);
}

template <int DT>
int stream_dt(const Launch &l)
{
    return l.plan.aligned ? launch_stream_one<DT, true>(l) : launch_stream_one<DT, false>(l);
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
