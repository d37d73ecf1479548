"""GPU parity: the CUDA path, called through the C ABI, against the fp64
oracle, element by element, at the tolerances of include/softmax.h.

Sizes: every workload's first rows (several tiles and a ragged tail) under
every variant that accepts the shape; the full-size workloads in the launch
configuration the benchmark times (the dispatcher's choice); edge shapes
(empty, cols = 1, every small cols, chunk and tile boundaries, the largest row
each variant caches), unaligned pointers, a y on a different 16-byte phase
than x, special values and bitwise shift invariance.  Output buffers sit
between canary guard bands, checked after each kernel."""
import math

import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import ELEM, NUMPY, TORCH, check, np_to_torch, run, torch_to_np, variants_for

pytestmark = pytest.mark.gpu

NAMES = {v: k for k, v in osd.VARIANTS.items()}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()
    rc, dev = osd.softmax_device_query()
    assert rc == 0 and dev.sm_count > 0


def test_worked_example_every_variant():
    x = np.array([[1, 2, 3], [1, 1, 1]], dtype=np.float32)
    want = np.array([[0.0900, 0.2447, 0.6652], [0.3333, 0.3333, 0.3333]])
    for v in variants_for(2, 3, 0):
        rc, y = run(x, 0, variant=v)
        assert rc == 0, NAMES[v]
        assert np.array_equal(np.round(y.astype(np.float64), 4), want), (NAMES[v], y)
        check(x, y, 0)


PREFIX = {
    "fp32_128x1000": 128,
    "attn_fp16_65536x512": 3000,
    "awkward_fp16_8192x5003": 700,
    "vocab_bf16_32768x32000": 300,
    "splitk_fp32_4x4194304": 4,
    "splitk_fp16_4x4194304": 4,
}


@pytest.mark.parametrize("name", list(PREFIX))
def test_workload_prefix_every_variant(name):
    w = W.WORKLOADS[name]
    rows = PREFIX[name]
    x = W.generate(w, rows=rows)
    vs = variants_for(rows, w.cols, w.dtype_code)
    assert 0 in vs
    for v in vs:
        rc, y = run(x, w.dtype_code, variant=v)
        assert rc == 0, (NAMES[v], rc)
        check(x, y, w.dtype_code)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_workload_full_size_dispatcher(name):
    """Full size, the kernel and launch shape the benchmark times."""
    w = W.WORKLOADS[name]
    x = W.generate(w)
    xt = np_to_torch(x, w.dtype_code).cuda()
    yt = osd.softmax(xt)
    torch.cuda.synchronize()
    y = torch_to_np(yt, w.dtype_code)
    del xt, yt
    check(x, y, w.dtype_code)


SMALL_COLS = list(range(1, 41)) + [63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1000,
                                     1023, 1024, 1025, 2047, 2048, 2049, 4093, 5003, 8192, 16381,
                                     32000, 32768, 32771]


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_edge_shapes_every_variant(dt):
    rng = np.random.default_rng(100 + dt)
    for cols in SMALL_COLS:
        for rows in (1, 3, 37):
            x64 = rng.normal(0, 6, (rows, cols))
            x = x64.astype(NUMPY[dt]) if dt != 2 else W._round_to(x64, "bf16")
            offs = [(0, 0), (1, 1)] if cols < 4096 else [(0, 0)]
            for xo, yo in offs:
                for v in variants_for(rows, cols, dt, xo, yo):
                    rc, y = run(x, dt, variant=v, x_off=xo, y_off=yo)
                    assert rc == 0, (cols, rows, NAMES[v], xo, yo)
                    check(x, y, dt)


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_y_on_another_phase(dt):
    rng = np.random.default_rng(7)
    for cols in (7, 100, 1000, 5003, 20000):
        x64 = rng.normal(0, 3, (9, cols))
        x = x64.astype(NUMPY[dt]) if dt != 2 else W._round_to(x64, "bf16")
        for xo, yo in ((0, 1), (3, 0), (2, 5)):
            vs = variants_for(9, cols, dt, xo, yo)
            assert 0 in vs
            for v in vs:
                rc, y = run(x, dt, variant=v, x_off=xo, y_off=yo)
                assert rc == 0, (cols, NAMES[v])
                check(x, y, dt)


def _largest_cols(v, dt, x_off, step):
    """Largest cols (a multiple of `step`) the dispatcher accepts for variant v."""
    lo, hi = 1, 1 << 22
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if v in variants_for(3, mid * step, dt, x_off, x_off):
            lo = mid
        else:
            hi = mid - 1
    return lo * step


def test_largest_rows_each_variant_caches():
    for dt in (0, 1, 2):
        e = ELEM[dt]
        for v in (osd.VARIANTS["rowgroup"], osd.VARIANTS["block"], osd.VARIANTS["block_tma"]):
            for x_off, step in ((0, 16 // e), (1, 1)):
                cols = _largest_cols(v, dt, x_off, step)
                assert cols >= 64
                assert v not in variants_for(3, cols + step, dt, x_off, x_off)
                x = np.random.default_rng(cols).normal(0, 2, (3, cols))
                x = x.astype(NUMPY[dt]) if dt != 2 else W._round_to(x, "bf16")
                rc, y = run(x, dt, variant=v, x_off=x_off, y_off=x_off)
                assert rc == 0, (NAMES[v], dt, cols)
                check(x, y, dt)


def test_empty_and_degenerate_shapes():
    for dt in (0, 1, 2):
        for shape in ((0, 5), (5, 0), (0, 0)):
            x = torch.empty(shape, dtype=TORCH[dt], device="cuda")
            y = osd.softmax(x)
            assert y.shape == shape
        x = torch.randn(17, 1, device="cuda").to(TORCH[dt])
        assert torch.equal(osd.softmax(x), torch.ones_like(x))


def test_special_values():
    inf, nan = np.inf, np.nan
    rows = [
        [0.0, -inf, 1.0, -inf],      # -inf entries -> exact zeros
        [-inf, -inf, -inf, -inf],    # all -inf -> NaN row
        [0.0, nan, 1.0, 2.0],        # NaN -> NaN row
        [0.0, inf, 1.0, 2.0],        # +inf -> NaN row
        [5.0, 5.0, 5.0, 5.0],        # constant -> 1/4
        [1.0, 2.0, 3.0, 4.0],
    ]
    for dt in (0, 1, 2):
        x = np.array(rows)
        x = x.astype(NUMPY[dt]) if dt != 2 else W._round_to(x, "bf16")
        xw = np.repeat(x, 3, axis=1)  # also longer rows
        for arr in (x, xw):
            for v in variants_for(arr.shape[0], arr.shape[1], dt):
                rc, y = run(arr, dt, variant=v)
                assert rc == 0
                check(arr, y, dt, finite_expected=False)
                yd = oracle.decode(y, dt)
                xd = oracle.decode(arr, dt)
                assert np.isnan(yd[1:4]).all(), NAMES[v]
                assert (yd[0][xd[0] == -np.inf] == 0).all(), NAMES[v]
                assert np.isfinite(yd[[0, 4, 5]]).all()


def test_long_runs_of_minus_inf():
    """Whole thread / CTA shares of -inf next to finite values: the online
    (m, d) passes must treat an all -inf share as empty, not as NaN."""
    rng = np.random.default_rng(21)
    for dt in (0, 1, 2):
        for cols in (3000, 70000, 300000):
            x = rng.normal(0, 3, (3, cols))
            x[0, : cols // 2] = -np.inf       # first half
            x[1, cols // 3:] = -np.inf        # last two thirds
            x[2, ::2] = -np.inf               # every other element
            x = x.astype(NUMPY[dt]) if dt != 2 else W._round_to(x, "bf16")
            for v in variants_for(3, cols, dt):
                rc, y = run(x, dt, variant=v)
                assert rc == 0
                check(x, y, dt)
                yd = oracle.decode(y, dt)
                assert (yd[oracle.decode(x, dt) == -np.inf] == 0).all(), NAMES[v]


def test_extreme_magnitudes():
    for dt, big in ((0, 3.0e38), (1, 65504.0), (2, 3.0e38)):
        x = np.array([[big, -big, 0.0, big / 2], [-big, -big, -big, -big / 2], [1.0, -big, 2.0, 3.0]])
        x = x.astype(NUMPY[dt]) if dt != 2 else W._round_to(x, "bf16")
        for v in variants_for(3, 4, dt):
            rc, y = run(x, dt, variant=v)
            assert rc == 0
            check(x, y, dt)


def test_bf16_subnormal_outputs():
    # y = e^-90 / (1 + e^-90) ~ 8.2e-40: a bf16 subnormal, which a flush-to-zero
    # exp would lose
    x = np.array([[0.0, -90.0], [0.0, -88.0], [0.0, -92.5], [-91.0, 0.0]])
    xb = W._round_to(x, "bf16")
    for v in variants_for(4, 2, 2):
        rc, y = run(xb, 2, variant=v)
        assert rc == 0
        check(xb, y, 2)
        assert (y[:, :] != 0).sum() >= 6


def test_ramp_rows():
    # the HIP softmax tutorial's large-cols shape (4 x 32768) on a ramp
    # x_j = j / 32 (its printed outputs grow by e^(1/32) per column): every
    # variant that accepts the shape, against the oracle, and the ratio of
    # neighbouring outputs within the fp32 tolerance
    n = 32768
    j = np.arange(n, dtype=np.float64)
    x = np.stack([j / 32.0, j / 32.0 - 100.0, j / 32.0 + 7.25, (n - 1 - j) / 32.0]).astype(np.float32)
    for v in variants_for(4, n, 0):
        rc, y = run(x, 0, variant=v)
        assert rc == 0, v
        check(x, y, 0)
        big = y[0, :-1] > 1e-30
        r = y[0, 1:][big].astype(np.float64) / y[0, :-1][big]
        assert np.allclose(r, math.exp(1.0 / 32.0), rtol=5e-6), v


def test_looping_block_rows():
    # rows of 64 - 128 KiB: 16 chunks a thread past 256 threads, one CTA per SM
    # looping over more rows than SMs, each prefetching its next row into L2;
    # off the 16-byte grid (the dispatcher's choice) and forced on the grid
    rng = np.random.default_rng(41)
    block = osd.VARIANTS["block"]
    for rows, cols, dt, off, v in ((400, 50257, 2, 0, 0), (300, 50003, 1, 1, 0), (200, 30000, 0, 0, block),
                                   (170, 65536, 2, 0, 0)):
        x = rng.normal(0, 3, (rows, cols))
        x[:, ::1009] += 25.0
        x = x.astype(NUMPY[dt]) if dt != 2 else W._round_to(x, "bf16")
        rc, y = run(x, dt, variant=v, x_off=off, y_off=off)
        assert rc == 0, (rows, cols, dt)
        check(x, y, dt)


def test_shift_invariance_bitwise():
    rng = np.random.default_rng(9)
    for cols in (300, 5003, 40000):
        grid = rng.integers(-511, 512, size=(6, cols)) / 16.0
        x = grid.astype(np.float16)
        xs = (grid + 16.0).astype(np.float16)
        for v in variants_for(6, cols, 1):
            _, y1 = run(x, 1, variant=v)
            _, y2 = run(xs, 1, variant=v)
            assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16)), NAMES[v]


def test_custom_plans_persistence_and_tiles():
    w = W.WORKLOADS["attn_fp16_65536x512"]
    x = W.generate(w, rows=5000)
    xt = np_to_torch(x, 1).cuda()
    yt = torch.empty_like(xt)
    base = osd.plan_for(xt, yt)
    for grid in (1, 7, 152, 1000, base.grid_x):
        p = osd.LaunchPlan(**{**base.as_dict(), "grid_x": grid})
        osd.softmax(xt, out=yt.fill_(0), plan=p)
        check(x, torch_to_np(yt, 1), 1)
    tp = osd.plan_for(xt, yt, "block_tma")
    for R, Wp, stages in ((1, 16, 2), (4, 4, 3), (16, 1, 8), (64, 1, 3), (32, 2, 2)):
        stage = -(-(R * 1024) // 128) * 128
        p = osd.LaunchPlan(**{**tp.as_dict(), "rows_per_tile": R, "lanes_per_row": 32 * Wp,
                             "stages": stages, "smem_bytes": stage * stages, "grid_x": 100})
        osd.softmax(xt, out=yt.fill_(0), plan=p)
        check(x, torch_to_np(yt, 1), 1)


def test_stream_walks_both_ways():
    # the streaming kernel with every pass forward (back_passes 0) and with
    # the passes after the first walking back from the row's end (1): rows
    # of several full steps (512 threads x 8 chunks), a partial last step, a
    # row shorter than one step, rows off the 16-byte grid, special rows
    rng = np.random.default_rng(17)
    rc, dev = osd.softmax_device_query()
    assert rc == 0
    names = ("fp32", "fp16", "bf16")
    ninf = {0: np.float32(-np.inf), 1: np.float16(-np.inf), 2: np.uint16(0xFF80)}
    pinf = {0: np.float32(np.inf), 1: np.float16(np.inf), 2: np.uint16(0x7F80)}
    for dt in (0, 1, 2):
        e = ELEM[dt]
        E = 16 // e
        for cols, off in ((2 * 4096 * E, 0), (2 * 4096 * E + 3 * E, 0), (1000, 0), (4096 * E + 5, 1)):
            x = W._round_to(rng.normal(0, 4, (5, cols)), names[dt])
            x[3, : cols // 3] = ninf[dt]
            x[4, cols // 2] = pinf[dt]
            # the plan for run()'s buffers: a 256-byte aligned base shifted by off elements
            rc, base = osd.softmax_plan(dev, (1 << 40) + off * e, (1 << 40) + (1 << 38) + off * e, 5, cols, dt,
                                        osd.VARIANTS["stream"])
            assert rc == 0 and base.aligned == (off == 0 and cols * e % 16 == 0)
            outs = []
            for back in (0, 1):
                p = osd.LaunchPlan(**{**base.as_dict(), "back_passes": back})
                rc, y = run(x, dt, plan=p, x_off=off, y_off=off)
                assert rc == 0, (dt, cols, back)
                check(x[:4], y[:4], dt)
                assert np.isnan(oracle.decode(y[4:], dt)).all()  # +inf in the row: inf - inf
                outs.append(y)
            if dt:
                # the write pass goes element by element: its order changes no bit
                assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16)), (dt, cols)
    xd = torch.randn(4, 3 * 4096 * 8, device="cuda", dtype=torch.float16)
    yd = torch.empty_like(xd)
    for field, value in (("back_passes", 2), ("stages", 1)):
        bad = osd.LaunchPlan(**{**osd.plan_for(xd, yd, "stream").as_dict(), field: value})
        with pytest.raises(osd.SoftmaxError):
            osd.softmax(xd, out=yd, plan=bad)
    # only the streaming kernel takes back_passes
    xs = torch.randn(64, 512, device="cuda", dtype=torch.float16)
    ys = torch.empty_like(xs)
    bad = osd.LaunchPlan(**{**osd.plan_for(xs, ys).as_dict(), "back_passes": 1})
    with pytest.raises(osd.SoftmaxError):
        osd.softmax(xs, out=ys, plan=bad)


def test_many_long_rows_cluster_split():
    # 16-bit rows of 384 KiB, more of them than SMs: the dispatcher's cluster
    # split with one CTA per row, against the oracle; the workspace entry point
    # keeps that plan (it needs no workspace) and gives the same bits
    rc, dev = osd.softmax_device_query()
    assert rc == 0
    rng = np.random.default_rng(23)
    rows, cols = dev.sm_count + 9, 196608
    for dt in (1, 2):
        x = W._round_to(rng.normal(0, 3, (rows, cols)), ("fp32", "fp16", "bf16")[dt])
        x[5, : cols // 2] = (np.float16(-np.inf) if dt == 1 else np.uint16(0xFF80))
        xd = np_to_torch(x, dt).cuda()
        yd = torch.empty_like(xd)
        p = osd.plan_for(xd, yd)
        assert p.variant == osd.VARIANTS["splitk"] and p.cluster_x == 1 and p.grid_y == rows
        s = torch.cuda.current_stream().cuda_stream
        assert osd.softmax_fwd(xd.data_ptr(), yd.data_ptr(), rows, cols, dt, s) == 0
        rc, need = osd.softmax_workspace_size(xd.data_ptr(), yd.data_ptr(), rows, cols, dt)
        assert rc == 0 and need == 0
        yw = torch.empty_like(xd)
        ws = torch.empty(16, dtype=torch.uint8, device="cuda")
        assert osd.softmax_fwd_ws(xd.data_ptr(), yw.data_ptr(), rows, cols, dt, ws.data_ptr(), 16, s) == 0
        torch.cuda.synchronize()
        assert torch.equal(yd.view(torch.int16), yw.view(torch.int16))
        check(x, torch_to_np(yd, dt), dt)


def test_bad_custom_plan_is_refused():
    x = torch.randn(64, 512, device="cuda", dtype=torch.float16)
    y = torch.empty_like(x)
    p = osd.plan_for(x, y)
    bad = osd.LaunchPlan(**{**p.as_dict(), "chunks_per_thread": 1})  # 32 lanes x 1 chunk < 64 chunks
    with pytest.raises(osd.SoftmaxError):
        osd.softmax(x, out=y, plan=bad)
    bad = osd.LaunchPlan(**{**p.as_dict(), "aligned": 0})
    with pytest.raises(osd.SoftmaxError):
        osd.softmax(x, out=y, plan=bad)


def test_side_stream_and_overlap_refusal():
    x = torch.randn(300, 777, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = osd.softmax(x)
    s.synchronize()
    check(x.cpu().numpy(), y.cpu().numpy(), 0)
    # in place is accepted; a partial overlap is refused
    buf = torch.randn(301 * 777, device="cuda")
    with pytest.raises(osd.SoftmaxError) as e:
        osd.softmax(buf[: 300 * 777].view(300, 777), out=buf[777:].view(300, 777))
    assert e.value.status == -3


def test_device_error_word_is_clear():
    x = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    osd.softmax(x, variant="block_tma")
    rc, code = osd.softmax_get_device_error(torch.cuda.current_stream().cuda_stream)
    assert rc == 0 and code == 0


def test_bounded_wait_gives_up_and_reports():
    """A wait that nothing satisfies gives up after its limit, the error word
    reports it, and the context stays usable."""
    s = torch.cuda.current_stream().cuda_stream
    rc, code = osd.softmax_get_device_error(s)
    assert rc == 0 and code == 0
    assert osd.softmax_selftest_bounded_wait(s, 20000) == 0
    rc, code = osd.softmax_get_device_error(s)
    assert rc == -6 and code == 1
    rc, code = osd.softmax_get_device_error(s)  # read-and-clear
    assert rc == 0 and code == 0
    x = torch.randn(64, 1000, device="cuda")
    check(x.cpu().numpy(), osd.softmax(x).cpu().numpy(), 0)
    assert osd.softmax_selftest_bounded_wait(s, 0) == -1


def test_query_variant_matches_plan():
    x = torch.randn(65536, 512, device="cuda", dtype=torch.float16)
    y = torch.empty_like(x)
    rc, v = osd.softmax_query_variant(x.data_ptr(), y.data_ptr(), 65536, 512, 1)
    assert rc == 0 and v == osd.plan_for(x, y).variant
