// plan.cpp -- argument validation and the cols-based dispatcher, as pure host
// code (no CUDA calls), so that it runs and is tested on a machine without a
// GPU.
//
// The HIP softmax tutorial (forum.sourcefind.cn), section 7, switches on cols
// alone (cols <= 4096: one block per row, else a multi-block pipeline), and
// section 5 sizes the block from cols; "[CUDA] safe online softmax", sections
// 4.2-4.3, measures that no single kernel wins everywhere and leaves the
// choice open.  Here the choice is made on the 16-byte chunks a row spans
// (cols * sizeof(dtype)), the row count against the SM count, and alignment:
//
//   row fits 32 lanes' registers      -> ROWGROUP   (G lanes per row, G = 1..32)
//   few rows, long rows, clusters     -> SPLITK     (cluster of CTAs per row)
//   row fits one CTA's registers      -> BLOCK      (one CTA per row)
//   two tiles of one row fit in smem  -> BLOCK_TMA  (bulk-copy staged row tiles)
//   otherwise                         -> SPLITK if rows < SMs, else STREAM
#include <stdint.h>

#include <initializer_list>

#include "launch.h"

namespace osd {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t next_pow2(int64_t v)
{
    int64_t p = 1;
    while (p < v)
        p <<= 1;
    return p;
}

int64_t pow2_floor(int64_t v)
{
    int64_t p = 1;
    while (p * 2 <= v)
        p <<= 1;
    return p;
}

struct Geometry {
    int S;            // element bytes
    int E;            // elements per 16-byte chunk
    int64_t row_bytes;
    bool aligned;     // every x and y row starts on the 16-byte grid and spans whole chunks
    bool y_vec;       // y rows have the same 16-byte phase as x rows
    int64_t nch_max;  // most 16-byte chunks any row spans
    int64_t nint;     // most whole 16-byte chunks inside any row (the interior
                      // chunks of the lanes-per-row and CTA-per-row kernels,
                      // which take the partial edges element by element)
};

Geometry geometry(const void *x, const void *y, int64_t cols, int dtype)
{
    Geometry g;
    g.S = dtype_bytes(dtype);
    g.E = 16 / g.S;
    g.row_bytes = cols * g.S;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
    g.aligned = (xa % 16 == 0) && (ya % 16 == 0) && (g.row_bytes % 16 == 0);
    g.y_vec = ((ya - xa) % 16) == 0;
    // an unaligned row starts up to 16 - S bytes into its first chunk
    g.nch_max = g.aligned ? g.row_bytes / 16 : ceil_div(g.row_bytes + 16 - g.S, 16);
    g.nint = g.row_bytes / 16;
    return g;
}

bool rowgroup_fits(const Geometry &g) { return g.nint <= 32 * (kRowgroupMaxFloats / g.E); }

bool block_fits(const Geometry &g) { return g.nint <= int64_t(block_max_threads(kBlockMaxChunks)) * kBlockMaxChunks; }

// G lanes per row with V chunks each: aim for 32 cached floats per lane (4
// chunks of fp16 / bf16, 8 of fp32) so that the per-row shuffles and the
// reciprocal are spread over many elements; rows of up to 4 chunks get one
// chunk per lane.  One row per lane group: a grid-stride walk over rows with a
// smaller, persistent grid measured slower on the [65536, 512] fp16 rows.
void plan_rowgroup(const Geometry &g, int64_t rows, const softmax_device_info &dev, softmax_launch_plan &p)
{
    int64_t G, V;
    const int64_t n = g.nint > 1 ? g.nint : 1;
    if (n <= 4) {
        G = next_pow2(n);
        V = 1;
    } else {
        // chunks per lane: up to 32 floats' worth (8 fp32 / 4 16-bit chunks),
        // but 2 for 16-bit rows of 17 - 64 chunks: twice the lanes on a row
        // measured faster there ([65536, 512] fp16: 32 x 2 at 94.7 %, 16 x 4
        // at 93.4 %; 256 columns +0.8 points; 128 columns -0.6 points, so
        // those stay at 4)
        const int64_t vt = (g.E == 8 && n > 16) ? 2 : kRowgroupMaxFloats / g.E;
        G = next_pow2(ceil_div(n, vt));
        if (G < 2)
            G = 2;
        if (G > 32)
            G = 32;
        V = next_pow2(ceil_div(n, G));
    }
    // 128-thread CTAs (measured 0.3 - 0.6 points above 256 on 128 - 1024
    // column rows), halved (down to one warp) while that leaves SMs idle: few
    // rows then spread over more SMs ([128, 1000] fp32: 16 CTAs of 8 rows each
    // ran at 284 - 301 GB/s, one 64-thread CTA a row at 344 GB/s)
    int64_t T = kRowgroupThreads / 2;
    while (T / 2 >= (G > 32 ? G : 32) && ceil_div(rows, T / G) < dev.sm_count)
        T /= 2;
    p.variant = SOFTMAX_VARIANT_ROWGROUP;
    p.lanes_per_row = (int)G;
    p.chunks_per_thread = (int)V;
    p.block_threads = (int)T;
    const int64_t ctas = ceil_div(rows, T / G);
    p.grid_x = ctas < INT32_MAX ? ctas : INT32_MAX;
}

void plan_block(const Geometry &g, int64_t rows, const softmax_device_info &dev, softmax_launch_plan &p)
{
    // V chunks per thread: 8 when that still leaves two warps per row (more
    // loads in flight per thread, fewer reduction rounds per element), else 4;
    // raised to 16 when the CTA would pass 256 threads, so that several CTAs --
    // several rows -- stay resident per SM and one's loads overlap another's
    // reductions.  Back to 4 when 8 leaves more than a tenth of the CTA's
    // chunk slots idle and 4 leaves fewer (16-bit rows then also keep
    // exp(x - m) instead of computing it twice).  Measured: [8192, 5003] fp16
    // (625 interior chunks) at V = 4 x 160 threads 86.3 %, at 8 x 96 84.0 %;
    // [8192, 6000] (750) at 8 x 96 94.8 %, at 4 x 192 91.7 %; [32768, 32000]
    // bf16 at V = 16 x 256 (V = 8 x 512 is slower).
    const auto slots = [&](int v) { return ceil_div(ceil_div(g.nint, v), 32) * 32 * v; };
    int V = ceil_div(g.nint, 8) >= 64 ? 8 : 4;
    while (V < kBlockMaxChunks && ceil_div(g.nint, V) > 256)
        V *= 2;
    if (V == 8 && (slots(8) - g.nint) * 10 > slots(8) && slots(4) < slots(8))
        V = 4;
    int64_t threads = ceil_div(ceil_div(g.nint, V), 32) * 32;
    if (threads < 64)
        threads = 64;
    p.variant = SOFTMAX_VARIANT_BLOCK;
    p.chunks_per_thread = V;
    p.block_threads = (int)threads;
    p.grid_x = rows < INT32_MAX ? rows : INT32_MAX;
    // past 256 threads at 16 chunks (rows of 64 - 128 KiB) one CTA fills an
    // SM: one CTA per SM, looping over rows with a next-row L2 prefetch
    if (V >= 16 && threads > 256 && p.grid_x > dev.sm_count)
        p.grid_x = dev.sm_count;
}

// Bytes of shared memory one BLOCK_TMA tile of R rows needs: the 16-byte
// chunks it spans from the aligned address below its start, rounded to 128.
int64_t tma_stage_bytes(const Geometry &g, int64_t R)
{
    const int64_t lead_max = g.aligned ? 0 : 16 - g.S;
    const int64_t chunks = ceil_div(lead_max + R * g.row_bytes, 16);
    return ceil_div(chunks * 16, 128) * 128;
}

int tma_budget(const softmax_device_info &dev) { return dev.max_smem_optin - kTmaStaticSmem; }

// BLOCK_TMA shape: about 32 KB per tile; rows of 32 KB and more get a tile of
// their own and all 16 consumer warps; shorter rows share a tile, and the
// consumer warps split into row groups (one warp per row below 2 KB).
bool plan_tma(const Geometry &g, int64_t rows, const softmax_device_info &dev, softmax_launch_plan &p)
{
    const int64_t target = 32 * 1024;
    int64_t R = 1, W = kTmaConsumerWarps;
    if (g.row_bytes < target) {
        R = pow2_floor(target / g.row_bytes);
        if (R > 256)
            R = 256;
        W = kTmaConsumerWarps / (R < kTmaConsumerWarps ? R : kTmaConsumerWarps);
    }
    if (R > rows)
        R = next_pow2(rows);
    int64_t stage = tma_stage_bytes(g, R);
    int64_t stages = tma_budget(dev) / stage;
    if (stages > kTmaMaxStagesHost)
        stages = kTmaMaxStagesHost;
    if (stages < 2)
        return false;
    const int64_t tiles = ceil_div(rows, R);
    p.variant = SOFTMAX_VARIANT_BLOCK_TMA;
    p.lanes_per_row = (int)(32 * W);
    p.rows_per_tile = (int)R;
    p.stages = (int)stages;
    p.smem_bytes = (int)(stages * stage);
    p.block_threads = kTmaThreads;
    p.grid_x = tiles < dev.sm_count ? tiles : dev.sm_count;
    return true;
}

bool tma_fits(const Geometry &g, const softmax_device_info &dev)
{
    return tma_stage_bytes(g, 1) * 2 <= tma_budget(dev);
}

// STREAM: one CTA per row.  back_passes = 1 (the passes after the first walk each
// row from the other end, their loads with L2 policies) where the rows in
// flight hold more than 5/12 of L2 (55 MB of GB300's; measured between the
// forward walk's last win, 50 MB, and the backward walk's first, 60 MB),
// so that a re-read starts on the chunks read last; the rows in flight are the
// resident CTAs, 2 per SM (every instance fits 64 registers at 512 threads).  Measured on GB300 (rows in
// flight x row bytes; forward against backward with the policies, us):
// [4096, 65600] fp16 (40 MB) 181.5 against 190.1; [8192, 81920] fp16 (50 MB)
// 451.7 against 456.3; [6144, 98304] fp16 (60 MB) 461.3 against 389.0;
// [2048, 65536] fp32 (80 MB) 312.6 against 274.4; [4096, 131072] bf16 (80 MB)
// 409.0 against 370.5.
void plan_stream(const Geometry &g, int64_t rows, const softmax_device_info &dev, softmax_launch_plan &p)
{
    p.variant = SOFTMAX_VARIANT_STREAM;
    p.chunks_per_thread = kStreamUnroll;
    p.block_threads = kStreamThreads;
    p.grid_x = rows < INT32_MAX ? rows : INT32_MAX;
    const int64_t resident = int64_t(dev.sm_count > 0 ? dev.sm_count : 1) * 2;
    const int64_t in_flight = rows < resident ? rows : resident;
    p.back_passes = dev.l2_bytes > 0 && in_flight * g.row_bytes * 12 > int64_t(dev.l2_bytes) * 5 ? 1 : 0;
}

// Cluster size (power of two, <= 16): about two CTAs per SM over all rows,
// and at least two full shared-memory stages of work per CTA.
int splitk_cluster(const Geometry &g, int64_t rows, const softmax_device_info &dev)
{
    if (rows >= dev.sm_count)
        return 1;  // as many rows as SMs: one CTA per row
    int64_t c = next_pow2(ceil_div(2 * int64_t(dev.sm_count > 0 ? dev.sm_count : 1), rows > 0 ? rows : 1));
    const int64_t by_work = pow2_floor(g.nch_max / (2 * int64_t(kSplitStageBytes / 16)));
    if (c > by_work)
        c = by_work;
    if (c > kMaxCluster)
        c = kMaxCluster;
    if (c < 1)
        c = 1;
    return (int)c;
}

void plan_splitk(const Geometry &g, int64_t rows, const softmax_device_info &dev, softmax_launch_plan &p)
{
    const int c = splitk_cluster(g, rows, dev);
    p.variant = SOFTMAX_VARIANT_SPLITK;
    p.stages = kSplitStages;
    p.smem_bytes = kSplitStages * kSplitStageBytes;
    p.block_threads = kSplitThreads;
    p.cluster_x = c;
    p.grid_x = c;
    p.grid_y = rows;
}

// SPLITK_WIDE: P CTAs per row, about two per SM over all rows, each with at
// least one full streaming step per thread.
void plan_wide(const Geometry &g, int64_t rows, const softmax_device_info &dev, softmax_launch_plan &p)
{
    int64_t P = ceil_div(2 * int64_t(dev.sm_count > 0 ? dev.sm_count : 1), rows > 0 ? rows : 1);
    const int64_t by_work = g.nch_max / (int64_t(kStreamThreads) * kWideStep);
    if (P > by_work)
        P = by_work;
    if (P > 1024)
        P = 1024;
    if (P < 1)
        P = 1;
    p.variant = SOFTMAX_VARIANT_SPLITK_WIDE;
    p.chunks_per_thread = kWideStep;
    p.block_threads = kStreamThreads;
    p.grid_x = P;
    p.grid_y = rows;
}

// SPLITK_GRID: P CTAs per row, all resident (cooperative launch).  Rows whose
// CTA share fits a shared-memory buffer at one CTA per SM take the ring form
// (each share read from HBM once, into shared memory); the rest take the
// streaming form at two CTAs per SM.
bool grid_possible(int64_t rows, const softmax_device_info &dev)
{
    return dev.cc_major >= 9 && rows >= 1 && rows * 2 <= dev.sm_count && rows <= kGridMaxRows;
}

void plan_grid(const Geometry &g, int64_t rows, const softmax_device_info &dev, softmax_launch_plan &p)
{
    const int64_t budget = int64_t(dev.max_smem_optin) - kGridStaticSmem;
    p.variant = SOFTMAX_VARIANT_SPLITK_GRID;
    p.chunks_per_thread = kWideStep;
    p.block_threads = kGridThreads;
    // Ring form: G groups of P = SMs / G CTAs, one CTA per SM.  Each row a CTA
    // takes in turn costs it a fixed few microseconds (its fold, the block
    // reductions, the release, the merge's round trip), so the plan takes the
    // fewest rows per group (npg) for which a CTA's share of a row fits one
    // buffer and the partials fit a scratch slot, and for that count the
    // fewest groups (the most CTAs on a row: the smallest shares, the deepest
    // ring).
    int64_t P = 0, G = 0, buf = 0, npg_found = 0;
    for (int64_t npg = 1; npg <= rows; npg++) {
        const int64_t gg = ceil_div(rows, npg);
        if (npg > 1 && ceil_div(rows, gg) != npg)
            continue;  // the same group count as a smaller npg
        const int64_t pp = int64_t(dev.sm_count) / gg;
        if (pp < 1 || pp * rows > kGridMaxPartials)
            continue;
        const int64_t bb = ceil_div(ceil_div(g.nch_max, pp) * 16, 128) * 128;
        if (bb > budget)
            continue;
        P = pp;
        G = gg;
        buf = bb;
        npg_found = npg;
        break;
    }
    // Pipelined form, where the ring would give a group several rows in turn:
    // every SM on every row, the rows in turn through Q >= 2 buffers, a fold
    // team working on one row while the write team waits at the grid barrier
    // of the row before and writes it, so that those rows' fixed costs overlap
    // each other and the loads.  Measured on [4, 4194304]: fp32 (ring: 2
    // groups of 76 CTAs, two rows each) 44.4 us pipelined against 47.2 us;
    // fp16 (ring: one row per group of 38 CTAs) 24.7 us pipelined against
    // 20.5 us, so one row per group stays with the ring.
    if (npg_found != 1 && rows >= 2 && dev.sm_count <= kGridPipeMaxCtas &&
        int64_t(dev.sm_count) * rows <= kGridMaxPartials) {
        const int64_t PP = dev.sm_count;
        const int64_t bb = ceil_div(ceil_div(g.nch_max, PP) * 16, 128) * 128;
        int64_t Q = budget / bb;
        if (Q > rows)
            Q = rows;
        if (Q > kGridMaxRing)
            Q = kGridMaxRing;
        if (Q >= 2) {
            p.lanes_per_row = kGridPipeFold;
            p.stages = (int)Q;
            p.smem_bytes = (int)(Q * bb);
            p.grid_x = PP;
            p.grid_y = 1;
            return;
        }
    }
    if (P > 0) {
        int64_t Q = ceil_div(rows, G);
        if (Q > budget / buf)
            Q = budget / buf;
        if (Q > kGridMaxRing)
            Q = kGridMaxRing;
        p.stages = (int)Q;
        p.smem_bytes = (int)(Q * buf);
        p.grid_x = P;
        p.grid_y = G;
        return;
    }
    // Streaming form: two CTAs per SM, P per row, no shared-memory copy
    P = 2 * int64_t(dev.sm_count) / rows;
    const int64_t by_work = g.nch_max / (int64_t(kGridThreads) * kWideStep);
    if (P > by_work)
        P = by_work;
    if (P * rows > kGridMaxPartials)
        P = kGridMaxPartials / rows;
    if (P < 1)
        P = 1;
    p.stages = 0;
    p.smem_bytes = 0;
    p.grid_x = P;
    p.grid_y = rows;
}

bool splitk_possible(int64_t rows, const softmax_device_info &dev)
{
    return dev.cluster_launch && rows >= 1 && rows <= 65535 &&
           dev.max_smem_optin >= kSplitStages * kSplitStageBytes + 1024;
}

// Many 16-bit rows on the 16-byte grid of more than 256 KiB and less than 2
// MiB: the cluster split with one CTA per row, whose bulk copies keep 192 KB
// in flight per SM and whose one row per SM in flight leaves more of a row in
// L2 for its re-read, beats the streaming kernel (both with their L2 policies;
// measured on GB300, us: [2048, 262144] fp16 404.5 against 416.5, [2048,
// 393216] bf16 613.6 against 647.8, [1024, 524288] fp16 447.0 against 460.8;
// level at 384 KiB, [3072, 196608] fp16 448.7 against 449.7).  At 256 KiB and
// at 2 MiB the streaming kernel is as fast or faster ([4096, 131072] bf16
// 370.7 against 437.9; [512, 1048576] fp16 474.2 against 482.3), and fp32
// rows and shorter rows stay with it ([1024, 262144] fp32 714 against 622 -
// 657 before the policies, [4096, 65600] fp16 278 against 185).
bool splitk_long_rows(const Geometry &g, int64_t rows, const softmax_device_info &dev)
{
    return g.S == 2 && g.aligned && rows >= dev.sm_count && rows <= 65535 && splitk_possible(rows, dev) &&
           g.row_bytes > (int64_t(1) << 18) && g.row_bytes < (int64_t(1) << 21);
}

}  // namespace

int validate_args(const void *x, const void *y, int64_t rows, int64_t cols, int dtype)
{
    if (dtype < SOFTMAX_F32 || dtype > SOFTMAX_BF16)
        return SOFTMAX_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || cols < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    if (!x || !y)
        return SOFTMAX_ERR_INVALID_ARG;
    const int64_t S = dtype_bytes(dtype);
    if (cols > INT64_MAX / S || rows > INT64_MAX / (cols * S))
        return SOFTMAX_ERR_INVALID_ARG;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
    if (xa % S || ya % S)
        return SOFTMAX_ERR_INVALID_ARG;
    const uint64_t bytes = (uint64_t)(rows * cols * S);
    const uint64_t gap = xa <= ya ? (uint64_t)(ya - xa) : (uint64_t)(xa - ya);
    // x == y is in place (every kernel reads each element before the thread
    // that owns it writes it, and nothing reads it afterwards); any other
    // overlap would let a row be read after another row's write
    if (gap != 0 && gap < bytes)
        return SOFTMAX_ERR_ALIAS;
    return SOFTMAX_OK;
}

int validate_plan(const softmax_device_info &dev, const void *x, const void *y, int64_t rows,
                  int64_t cols, int dtype, const softmax_launch_plan &p)
{
    const Geometry g = geometry(x, y, cols, dtype);
    if ((p.aligned != 0) != g.aligned || (p.y_vector != 0) != g.y_vec)
        return SOFTMAX_ERR_INVALID_ARG;
    if (p.block_threads < 32 || p.block_threads % 32 || p.block_threads > 1024)
        return SOFTMAX_ERR_INVALID_ARG;
    if (p.grid_x < 1 || p.grid_x > INT32_MAX || p.smem_bytes < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    // the walk direction of the streaming kernel's re-read passes
    if (p.back_passes != 0 && (p.back_passes != 1 || p.variant != SOFTMAX_VARIANT_STREAM))
        return SOFTMAX_ERR_INVALID_ARG;
    const int V = p.chunks_per_thread;
    switch (p.variant) {
    case SOFTMAX_VARIANT_ROWGROUP: {
        const int G = p.lanes_per_row;
        if (G < 1 || G > 32 || (G & (G - 1)) || V < 1 || V > 8 || (V & (V - 1)))
            return SOFTMAX_ERR_INVALID_ARG;
        if (V * g.E > kRowgroupMaxFloats || int64_t(G) * V < g.nint || (G == 1 && V != 1))
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.block_threads > kRowgroupThreads || p.grid_y != 1 || p.cluster_x != 1)
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    }
    case SOFTMAX_VARIANT_BLOCK:
        if (V < 1 || V > kBlockMaxChunks || (V & (V - 1)))
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.block_threads > block_max_threads(V) || int64_t(p.block_threads) * V < g.nint)
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.grid_y != 1 || p.cluster_x != 1)
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    case SOFTMAX_VARIANT_BLOCK_TMA: {
        const int W = p.lanes_per_row / 32;
        if (p.lanes_per_row % 32 || W < 1 || W > kTmaConsumerWarps || (W & (W - 1)))
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.block_threads != kTmaThreads || p.grid_y != 1 || p.cluster_x != 1)
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.rows_per_tile < 1 || p.stages < 2 || p.stages > kTmaMaxStagesHost)
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.smem_bytes % p.stages || (p.smem_bytes / p.stages) % 128 || p.smem_bytes > tma_budget(dev))
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.smem_bytes / p.stages < tma_stage_bytes(g, p.rows_per_tile))
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    }
    case SOFTMAX_VARIANT_STREAM:
        if (V != kStreamUnroll || p.block_threads > kStreamThreads || p.grid_y != 1 || p.cluster_x != 1 ||
            p.stages != 0)
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    case SOFTMAX_VARIANT_SPLITK_WIDE:
        if (V != kWideStep || p.block_threads > kStreamThreads || p.cluster_x != 1)
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.grid_y != rows || rows > 65535 || p.grid_x > 65535)
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    case SOFTMAX_VARIANT_SPLITK_GRID: {
        if (p.block_threads != kGridThreads || p.cluster_x != 1 || !grid_possible(rows, dev))
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.grid_x < 1 || p.grid_x * rows > kGridMaxPartials || V != kWideStep)
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.lanes_per_row != 0) {
            // pipelined form: one group of P CTAs (one per SM) on every row, Q
            // buffers, a fold team of lanes_per_row threads and a write team
            if (p.stages < 1 || p.stages > kGridMaxRing || p.grid_y != 1 || p.grid_x > dev.sm_count ||
                p.grid_x > kGridPipeMaxCtas || p.lanes_per_row < 32 || p.lanes_per_row % 32 != 0 ||
                p.lanes_per_row >= p.block_threads || p.smem_bytes % p.stages != 0)
                return SOFTMAX_ERR_INVALID_ARG;
            const int64_t buf = p.smem_bytes / p.stages;
            if (buf % 16 != 0 || buf < ceil_div(g.nch_max, p.grid_x) * 16 ||
                p.smem_bytes > dev.max_smem_optin - kGridStaticSmem)
                return SOFTMAX_ERR_INVALID_ARG;
        } else if (p.stages >= 1) {
            // ring form: G groups of P CTAs, one CTA per SM, Q buffers that each
            // hold a CTA's share of a row
            if (p.stages > kGridMaxRing || p.grid_y < 1 || p.grid_y > rows ||
                p.grid_x * p.grid_y > dev.sm_count || p.smem_bytes % p.stages != 0)
                return SOFTMAX_ERR_INVALID_ARG;
            const int64_t buf = p.smem_bytes / p.stages;
            if (buf % 16 != 0 || buf < ceil_div(g.nch_max, p.grid_x) * 16 ||
                p.smem_bytes > dev.max_smem_optin - kGridStaticSmem)
                return SOFTMAX_ERR_INVALID_ARG;
        } else if (p.stages != 0 || p.smem_bytes != 0 || p.grid_y != rows ||
                   p.grid_x * p.grid_y > 2 * int64_t(dev.sm_count)) {
            return SOFTMAX_ERR_INVALID_ARG;
        }
        return SOFTMAX_OK;
    }
    case SOFTMAX_VARIANT_SPLITK:
        if (p.block_threads != kSplitThreads || p.stages != kSplitStages ||
            p.smem_bytes != kSplitStages * kSplitStageBytes)
            return SOFTMAX_ERR_INVALID_ARG;
        if (p.cluster_x < 1 || p.cluster_x > kMaxCluster || p.grid_x != p.cluster_x || p.grid_y != rows)
            return SOFTMAX_ERR_INVALID_ARG;
        if (rows > 65535 || !splitk_possible(rows, dev))
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    default:
        return SOFTMAX_ERR_INVALID_ARG;
    }
}

uint64_t wide_workspace_bytes(const softmax_launch_plan &p)
{
    return p.variant == SOFTMAX_VARIANT_SPLITK_WIDE ? (uint64_t)p.grid_x * (uint64_t)p.grid_y * 16u : 0u;
}

// ---------------------------------------------------------------- masked forward

// Lanes per row while the logits fit 32 registers per lane (4 chunks for every
// dtype: fp32 keeps two floats per logit), else one CTA per row with x held
// packed (up to 4 chunks per thread, 512 threads: 2048 chunks, 32 KiB rows).
int plan_masked(const softmax_device_info &dev, const void *x, const void *y, int64_t rows, int64_t cols,
                int dtype, int variant, softmax_launch_plan *plan)
{
    (void)dev;
    const Geometry g = geometry(x, y, cols, dtype);
    softmax_launch_plan p = {};
    p.grid_y = 1;
    p.cluster_x = 1;
    p.aligned = g.aligned;
    p.y_vector = g.y_vec;
    // sized by a row's whole interior chunks (its partial edges go element by
    // element)
    const int64_t n = g.nint > 1 ? g.nint : 1;
    const bool rg_fits = n <= 32 * 4;
    const bool blk_fits = n <= 512 * 4;
    int v = variant;
    if (v == SOFTMAX_VARIANT_AUTO)
        v = rg_fits ? SOFTMAX_VARIANT_ROWGROUP : SOFTMAX_VARIANT_BLOCK;
    if (v == SOFTMAX_VARIANT_ROWGROUP) {
        if (!rg_fits)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        // as the forward: 2 chunks a lane for 16-bit rows of 17 - 64 chunks,
        // 128-thread CTAs (measured on the attention workload with scale 1/8
        // and a causal cut: 93.6 % against 86.0 % at 16 lanes x 4 chunks in
        // 256-thread CTAs)
        int64_t G = n <= 4 ? next_pow2(n) : next_pow2(ceil_div(n, (g.E == 8 && n > 16) ? 2 : 4));
        if (G > 32)
            G = 32;
        p.variant = v;
        p.lanes_per_row = (int)G;
        p.chunks_per_thread = (int)next_pow2(ceil_div(n, G));
        p.block_threads = kRowgroupThreads / 2;
        const int64_t ctas = ceil_div(rows, kRowgroupThreads / 2 / G);
        p.grid_x = ctas < INT32_MAX ? ctas : INT32_MAX;
    } else if (v == SOFTMAX_VARIANT_BLOCK) {
        if (!blk_fits)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        const int V = ceil_div(n, 4) >= 32 ? 4 : 2;
        p.variant = v;
        p.chunks_per_thread = V;
        p.block_threads = (int)(ceil_div(ceil_div(n, V), 32) * 32);
        p.grid_x = rows < INT32_MAX ? rows : INT32_MAX;
    } else {
        return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
    }
    *plan = p;
    return SOFTMAX_OK;
}

// ---------------------------------------------------------------- LayerNorm / RMSNorm

namespace {

bool ranges_meet(uintptr_t a, uint64_t na, uintptr_t b, uint64_t nb) { return a < b + nb && b < a + na; }

}  // namespace

int validate_norm_args(int kind, const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
                       const void *gamma, const void *beta, float eps, const float *mean, const float *rstd)
{
    if (kind != kNormLayer && kind != kNormRms)
        return SOFTMAX_ERR_INVALID_ARG;
    int rc = validate_args(x, y, rows, cols, dtype);  // dtype, sizes, alignment, x / y overlap
    if (rc != SOFTMAX_OK)
        return rc;
    if (!(eps >= 0.0f) || !(eps <= 3.4e38f))
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    const int64_t S = dtype_bytes(dtype);
    const uint64_t ybytes = (uint64_t)(rows * cols * S), vbytes = (uint64_t)(cols * S);
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
    // gain and bias are read by every row while y is written
    for (const void *v : {gamma, kind == kNormLayer ? beta : nullptr}) {
        if (!v)
            continue;
        const uintptr_t va = reinterpret_cast<uintptr_t>(v);
        if (va % S)
            return SOFTMAX_ERR_INVALID_ARG;
        if (ranges_meet(va, vbytes, ya, ybytes))
            return SOFTMAX_ERR_ALIAS;
    }
    // the statistics are written: they may overlap nothing else
    const float *stats[2] = {kind == kNormLayer ? mean : nullptr, rstd};
    for (int i = 0; i < 2; i++) {
        if (!stats[i])
            continue;
        const uintptr_t sa = reinterpret_cast<uintptr_t>(stats[i]);
        const uint64_t sb = (uint64_t)rows * 4u;
        if (sa % 4 || (uint64_t)rows > UINT64_MAX / 4u)
            return SOFTMAX_ERR_INVALID_ARG;
        if (ranges_meet(sa, sb, xa, ybytes) || ranges_meet(sa, sb, ya, ybytes) ||
            (gamma && ranges_meet(sa, sb, reinterpret_cast<uintptr_t>(gamma), vbytes)) ||
            (beta && kind == kNormLayer && ranges_meet(sa, sb, reinterpret_cast<uintptr_t>(beta), vbytes)))
            return SOFTMAX_ERR_ALIAS;
        if (i == 1 && stats[0] && ranges_meet(sa, sb, reinterpret_cast<uintptr_t>(stats[0]), sb))
            return SOFTMAX_ERR_ALIAS;
    }
    return SOFTMAX_OK;
}

// Lanes per row while a row fits 32 lanes x 4 chunks (V = 1..4, V = 3 included
// so that rows of 24 or 48 chunks -- 192 / 384 fp16 features -- fill every
// slot), else one CTA per row of up to 1024 threads x 4 chunks.  Sized by the
// row's whole 16-byte chunks; partial edges go element by element.
int plan_norm(const softmax_device_info &dev, int kind, const void *x, const void *y, int64_t rows, int64_t cols,
              int dtype, const void *gamma, const void *beta, int variant, softmax_launch_plan *plan, int *mode)
{
    (void)dev;
    const Geometry g = geometry(x, y, cols, dtype);
    softmax_launch_plan p = {};
    p.grid_y = 1;
    p.cluster_x = 1;
    p.aligned = g.aligned;
    p.y_vector = g.y_vec;
    bool vec_ok = g.aligned;
    for (const void *v : {gamma, kind == kNormLayer ? beta : nullptr})
        if (v && reinterpret_cast<uintptr_t>(v) % 16)
            vec_ok = false;
    *mode = vec_ok ? kNormFast : (g.y_vec ? kNormSame : kNormOther);
    const int64_t n = g.nint > 1 ? g.nint : 1;
    const bool rg_fits = n <= 32 * kNormMaxV;
    const bool blk_fits = n <= 1024 * kNormMaxV;
    int v = variant;
    if (v == SOFTMAX_VARIANT_AUTO)
        v = rg_fits ? SOFTMAX_VARIANT_ROWGROUP : SOFTMAX_VARIANT_BLOCK;
    if (v == SOFTMAX_VARIANT_ROWGROUP) {
        if (!rg_fits)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        int64_t G, V;
        if (n <= 4) {
            G = next_pow2(n);
            V = 1;
        } else {
            G = next_pow2(ceil_div(n, kNormMaxV));
            if (G < 2)
                G = 2;
            if (G > 32)
                G = 32;
            V = ceil_div(n, G);
        }
        p.variant = v;
        p.lanes_per_row = (int)G;
        p.chunks_per_thread = (int)V;
        // 128-thread CTAs ([32760, 384] fp16 LayerNorm: 71.6 % against 69.3 %
        // in 256-thread CTAs)
        p.block_threads = kRowgroupThreads / 2;
        const int64_t ctas = ceil_div(rows, kRowgroupThreads / 2 / G);
        p.grid_x = ctas < INT32_MAX ? ctas : INT32_MAX;
    } else if (v == SOFTMAX_VARIANT_BLOCK) {
        if (!blk_fits)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        const int V = ceil_div(n, 4) >= 64 ? 4 : 2;
        int64_t threads = ceil_div(ceil_div(n, V), 32) * 32;
        p.variant = v;
        p.chunks_per_thread = V;
        p.block_threads = (int)threads;
        p.grid_x = rows < INT32_MAX ? rows : INT32_MAX;
    } else {
        return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
    }
    *plan = p;
    return SOFTMAX_OK;
}

// ---------------------------------------------------------------- backward

namespace {

bool overlaps(const void *a, const void *b, uint64_t bytes)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    const uint64_t gap = x <= y ? (uint64_t)(y - x) : (uint64_t)(x - y);
    return gap < bytes;
}

}  // namespace

int validate_bwd_args(const void *y, const void *dy, const void *dx, int64_t rows, int64_t cols, int dtype)
{
    if (dtype < SOFTMAX_F32 || dtype > SOFTMAX_BF16)
        return SOFTMAX_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || cols < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    if (!y || !dy || !dx)
        return SOFTMAX_ERR_INVALID_ARG;
    const int64_t S = dtype_bytes(dtype);
    if (cols > INT64_MAX / S || rows > INT64_MAX / (cols * S))
        return SOFTMAX_ERR_INVALID_ARG;
    for (const void *p : {y, dy, (const void *)dx})
        if (reinterpret_cast<uintptr_t>(p) % S)
            return SOFTMAX_ERR_INVALID_ARG;
    const uint64_t bytes = (uint64_t)(rows * cols * S);
    // y and dy are only read and may overlap each other; dx may be exactly y
    // or exactly dy (in place), but overlap neither otherwise
    if ((dx != y && overlaps(dx, y, bytes)) || (dx != dy && overlaps(dx, dy, bytes)))
        return SOFTMAX_ERR_ALIAS;
    return SOFTMAX_OK;
}

// Backward dispatcher: lanes per row while y and dy fit 4 chunks per lane,
// one CTA per row up to 4096 chunks (64 KiB rows: 512 threads x 8 chunks of
// each), then the two-pass streaming kernel.
int plan_bwd(const softmax_device_info &dev, const void *y, const void *dy, const void *dx, int64_t rows,
             int64_t cols, int dtype, int variant, softmax_launch_plan *plan, int *dy_vec, int *dx_vec)
{
    const Geometry g = geometry(y, dx, cols, dtype);
    const uintptr_t ya = reinterpret_cast<uintptr_t>(y), da = reinterpret_cast<uintptr_t>(dy);
    const bool aligned = g.aligned && da % 16 == 0;
    const int64_t nch = aligned ? g.row_bytes / 16 : ceil_div(g.row_bytes + 16 - g.S, 16);
    softmax_launch_plan p = {};
    p.grid_y = 1;
    p.cluster_x = 1;
    p.aligned = aligned;
    p.y_vector = g.y_vec;
    *dy_vec = ((da - ya) % 16) == 0;
    *dx_vec = g.y_vec;
    // the lanes-per-row and CTA-per-row kernels hold a row's whole interior
    // chunks (its partial edges go element by element); the stream kernel
    // walks all of its chunks
    const int64_t n = g.nint > 1 ? g.nint : 1;
    const bool rg_fits = n <= 32 * 4;
    const bool blk_fits = n <= 512 * 8;
    (void)nch;
    int v = variant;
    if (v == SOFTMAX_VARIANT_AUTO)
        v = rg_fits ? SOFTMAX_VARIANT_ROWGROUP : (blk_fits ? SOFTMAX_VARIANT_BLOCK : SOFTMAX_VARIANT_STREAM);
    if (v == SOFTMAX_VARIANT_ROWGROUP) {
        if (!rg_fits)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        // as the forward: 2 chunks a lane for 16-bit rows of 17 - 64 chunks,
        // 128-thread CTAs ([65536, 512] fp16: 99.6 % against 99.3 % at 16
        // lanes x 4 chunks in 256-thread CTAs)
        int64_t G = n <= 4 ? next_pow2(n) : next_pow2(ceil_div(n, (g.S == 2 && n > 16) ? 2 : 4));
        if (G > 32)
            G = 32;
        const int64_t V = next_pow2(ceil_div(n, G));
        p.variant = v;
        p.lanes_per_row = (int)G;
        p.chunks_per_thread = (int)V;
        p.block_threads = kRowgroupThreads / 2;
        const int64_t ctas = ceil_div(rows, kRowgroupThreads / 2 / G);
        p.grid_x = ctas < INT32_MAX ? ctas : INT32_MAX;
    } else if (v == SOFTMAX_VARIANT_BLOCK) {
        if (!blk_fits)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        // 8 chunks of each tensor per thread only past 512 x 4 (registers)
        const int V = n > 512 * 4 ? 8 : (ceil_div(n, 4) >= 32 ? 4 : 2);
        int64_t T = ceil_div(ceil_div(n, V), 32) * 32;
        p.variant = v;
        p.chunks_per_thread = V;
        p.block_threads = (int)T;
        p.grid_x = rows < INT32_MAX ? rows : INT32_MAX;
        if (V == 8 && p.grid_x > dev.sm_count)
            p.grid_x = dev.sm_count;  // one CTA per SM, looping (and prefetching) over rows
    } else if (v == SOFTMAX_VARIANT_STREAM) {
        p.variant = v;
        p.chunks_per_thread = 4;
        p.block_threads = kStreamThreads;
        p.grid_x = rows < INT32_MAX ? rows : INT32_MAX;
        // the write pass walks each row from its end (back_passes = 1) where the
        // rows in flight (2 CTAs per SM on the 16-byte grid, else 1) hold
        // more than half of L2 in y and dy (the forward streaming kernel's own
        // line, 5/12, was measured on its shapes; this one on the backward's)
        const int64_t resident = int64_t(dev.sm_count > 0 ? dev.sm_count : 1) * (aligned ? 2 : 1);
        const int64_t in_flight = rows < resident ? rows : resident;
        p.back_passes = dev.l2_bytes > 0 && in_flight * 2 * g.row_bytes > int64_t(dev.l2_bytes) / 2 ? 1 : 0;
    } else {
        return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
    }
    *plan = p;
    return SOFTMAX_OK;
}

}  // namespace osd

using namespace osd;

extern "C" __attribute__((visibility("default"))) int softmax_plan(
    const softmax_device_info *dev, const void *x, const void *y, int64_t rows, int64_t cols,
    int dtype, int variant, softmax_launch_plan *plan)
{
    if (!dev || !plan)
        return SOFTMAX_ERR_INVALID_ARG;
    const int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    softmax_launch_plan p = {};
    p.grid_x = 1;
    p.grid_y = 1;
    p.cluster_x = 1;
    if (rows == 0 || cols == 0) {
        p.variant = variant == SOFTMAX_VARIANT_AUTO ? SOFTMAX_VARIANT_ROWGROUP : variant;
        p.grid_x = 0;
        *plan = p;
        return SOFTMAX_OK;
    }
    const Geometry g = geometry(x, y, cols, dtype);
    p.aligned = g.aligned;
    p.y_vector = g.y_vec;

    int v = variant;
    if (v == SOFTMAX_VARIANT_AUTO) {
        const bool few_rows = rows * 2 <= dev->sm_count;
        const bool long_rows = g.nch_max >= int64_t(8) * (kSplitStageBytes / 16);
        // (a launch-bound 1 MB call such as [128, 1000] fp32 measured within
        // run-to-run noise either way: lanes per row 2.97 - 3.14 us, one CTA
        // per row 3.02 - 3.10 us over two builds and boxes)
        if (rowgroup_fits(g))
            v = SOFTMAX_VARIANT_ROWGROUP;
        else if (few_rows && long_rows && grid_possible(rows, *dev))
            v = SOFTMAX_VARIANT_SPLITK_GRID;
        else if (few_rows && long_rows && splitk_possible(rows, *dev))
            v = SOFTMAX_VARIANT_SPLITK;
        // rows of 64 - 128 KiB: the bulk-copy tiles when the rows are on the
        // 16-byte grid (measured [16384, 40000] fp16 97.2 % against 92.9 % for
        // one looping 320-thread CTA per SM), else the block kernel ([16384,
        // 50257] bf16: 87.8 % against 58.3 %)
        else if (block_fits(g) && !(g.nint > 4096 && g.aligned && tma_fits(g, *dev)))
            v = SOFTMAX_VARIANT_BLOCK;
        else if (tma_fits(g, *dev))
            v = SOFTMAX_VARIANT_BLOCK_TMA;
        else if (rows < dev->sm_count && splitk_possible(rows, *dev))
            v = SOFTMAX_VARIANT_SPLITK;
        else if (splitk_long_rows(g, rows, *dev))
            v = SOFTMAX_VARIANT_SPLITK;
        else
            v = SOFTMAX_VARIANT_STREAM;
    }
    switch (v) {
    case SOFTMAX_VARIANT_ROWGROUP:
        if (!rowgroup_fits(g))
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        plan_rowgroup(g, rows, *dev, p);
        break;
    case SOFTMAX_VARIANT_BLOCK:
        if (!block_fits(g))
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        plan_block(g, rows, *dev, p);
        break;
    case SOFTMAX_VARIANT_BLOCK_TMA:
        if (!tma_fits(g, *dev) || !plan_tma(g, rows, *dev, p))
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        break;
    case SOFTMAX_VARIANT_STREAM:
        plan_stream(g, rows, *dev, p);
        break;
    case SOFTMAX_VARIANT_SPLITK:
        if (!splitk_possible(rows, *dev))
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        plan_splitk(g, rows, *dev, p);
        break;
    case SOFTMAX_VARIANT_SPLITK_WIDE:
        if (rows > 65535)
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        plan_wide(g, rows, *dev, p);
        break;
    case SOFTMAX_VARIANT_SPLITK_GRID:
        if (!grid_possible(rows, *dev))
            return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
        plan_grid(g, rows, *dev, p);
        break;
    default:
        return SOFTMAX_ERR_UNSUPPORTED_SHAPE;
    }
    *plan = p;
    return SOFTMAX_OK;
}

// The dispatchers of the other operations as pure host functions (no CUDA
// call): the plan softmax_bwd_variant / softmax_fwd_masked_variant /
// norm_fwd_variant would launch on a device described by *dev.
extern "C" __attribute__((visibility("default"))) int softmax_bwd_plan(
    const softmax_device_info *dev, const void *y, const void *dy, const void *dx, int64_t rows, int64_t cols,
    int dtype, int variant, softmax_launch_plan *plan)
{
    if (!dev || !plan)
        return SOFTMAX_ERR_INVALID_ARG;
    int rc = validate_bwd_args(y, dy, dx, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    *plan = softmax_launch_plan{};
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    int dy_vec = 0, dx_vec = 0;
    return plan_bwd(*dev, y, dy, dx, rows, cols, dtype, variant, plan, &dy_vec, &dx_vec);
}

extern "C" __attribute__((visibility("default"))) int softmax_masked_plan(
    const softmax_device_info *dev, const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
    int variant, softmax_launch_plan *plan)
{
    if (!dev || !plan)
        return SOFTMAX_ERR_INVALID_ARG;
    const int rc = validate_args(x, y, rows, cols, dtype);
    if (rc != SOFTMAX_OK)
        return rc;
    if (variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    *plan = softmax_launch_plan{};
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    return plan_masked(*dev, x, y, rows, cols, dtype, variant, plan);
}

extern "C" __attribute__((visibility("default"))) int norm_plan(
    const softmax_device_info *dev, int kind, const void *x, const void *y, int64_t rows, int64_t cols, int dtype,
    const void *gamma, const void *beta, int variant, softmax_launch_plan *plan)
{
    if (!dev || !plan)
        return SOFTMAX_ERR_INVALID_ARG;
    const int rc = validate_norm_args(kind, x, y, rows, cols, dtype, gamma, beta, 1e-5f, nullptr, nullptr);
    if (rc != SOFTMAX_OK)
        return rc;
    if (variant < SOFTMAX_VARIANT_AUTO || variant >= SOFTMAX_VARIANT_COUNT)
        return SOFTMAX_ERR_INVALID_ARG;
    *plan = softmax_launch_plan{};
    if (rows == 0 || cols == 0)
        return SOFTMAX_OK;
    int mode = 0;
    return plan_norm(*dev, kind, x, y, rows, cols, dtype, gamma, beta, variant, plan, &mode);
}
