"""GPU parity of SPLITK_GRID (few very long rows over every SM in one
cooperative launch, partials exchanged at a bounded per-row grid barrier
through the library's scratch slots) against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import check, np_to_torch, run, torch_to_np

pytestmark = pytest.mark.gpu
GRID = osd.VARIANTS["splitk_grid"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _quant(a64, dt):
    return {0: a64.astype(np.float32), 1: a64.astype(np.float16)}.get(dt) if dt != 2 else W._round_to(a64, "bf16")


def _no_device_error():
    rc, code = osd.softmax_get_device_error(torch.cuda.current_stream().cuda_stream)
    assert rc == 0 and code == 0, code


@pytest.mark.parametrize("name", ["splitk_fp32_4x4194304", "splitk_fp16_4x4194304"])
def test_grid_full_size_workloads(name):
    w = W.WORKLOADS[name]
    x = W.generate(w)
    xt = np_to_torch(x, w.dtype_code).cuda()
    assert osd.plan_for(xt, torch.empty_like(xt)).variant == GRID
    y = osd.softmax(xt)
    torch.cuda.synchronize()
    check(x, torch_to_np(y, w.dtype_code), w.dtype_code)
    _no_device_error()


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_grid_shapes_and_offsets(dt):
    rng = np.random.default_rng(300 + dt)
    # pipelined (every CTA on every row), ring (shares that fit shared
    # memory) and streamed forms, ragged rows, few and many CTAs per row, more
    # rows than buffers
    for rows, cols in ((1, 300001), (3, 1 << 20), (4, (1 << 21) + 5), (7, 150003), (2, 1 << 23), (76, 20000),
                       (11, (1 << 19) + 1), (26, 1 << 18), (5, 3 << 20)):
        x = rng.normal(0, 4, (rows, cols))
        x[:, ::97] += 60.0
        x = _quant(x, dt)
        for xo, yo in ((0, 0), (1, 1), (0, 3)):
            rc, y = run(x, dt, variant=GRID, x_off=xo, y_off=yo)
            assert rc == 0, (rows, cols, xo, yo)
            check(x, y, dt)
    _no_device_error()


def test_grid_special_rows_and_in_place():
    for dt in (0, 1, 2):
        cols = 600000
        x = np.random.default_rng(3).normal(0, 2, (4, cols))
        x[0, : cols // 2] = -np.inf
        x[1, 7] = np.nan
        x[2, :] = -np.inf
        x = _quant(x, dt)
        rc, y = run(x, dt, variant=GRID)
        assert rc == 0
        check(x, y, dt, finite_expected=False)
        yd = oracle.decode(y, dt)
        assert np.isnan(yd[1]).all() and np.isnan(yd[2]).all() and np.isfinite(yd[[0, 3]]).all()
    # in place, through the dispatcher
    xt = torch.randn(4, 3_000_001, device="cuda", dtype=torch.bfloat16) * 5
    ref = torch_to_np(xt, 2).copy()
    osd.softmax_(xt)
    torch.cuda.synchronize()
    check(ref, torch_to_np(xt, 2), 2)
    _no_device_error()


def test_grid_slots_across_streams_and_repeats():
    # more launches than slots, alternating between two streams and a chain on
    # one stream: launches sharing a slot are ordered by the slot's event
    torch.manual_seed(4)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    xs = [torch.randn(4, 1 << 20, device="cuda", dtype=torch.float16) * 6 for _ in range(6)]
    torch.cuda.synchronize()
    outs = []
    for i in range(40):
        st = s1 if i % 2 == 0 else s2
        with torch.cuda.stream(st):
            outs.append(osd.softmax(xs[i % 6]))
    chain = [xs[0]]
    with torch.cuda.stream(s1):
        for _ in range(20):
            chain.append(osd.softmax(chain[-1]))
    torch.cuda.synchronize()
    ref = {}
    for i, o in enumerate(outs):
        k = i % 6
        if k not in ref:
            check(torch_to_np(xs[k], 1), torch_to_np(o, 1), 1)
            ref[k] = o
        else:
            assert torch.equal(o.view(torch.int16), ref[k].view(torch.int16))  # bit-identical runs
    for a, b in zip(chain[:-1], chain[1:]):
        check(torch_to_np(a, 1), torch_to_np(b, 1), 1)
    _no_device_error()


def test_grid_under_graph_capture_falls_back():
    # a capture cannot take the slot events: the call captures the cluster split
    x = torch.randn(4, 1 << 21, device="cuda", dtype=torch.float16) * 3
    y = torch.empty_like(x)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        osd.softmax(x, out=y)  # warm (eager: the grid split)
        torch.cuda.synchronize()
        y.zero_()
        with torch.cuda.graph(g, stream=s):
            osd.softmax(x, out=y)
    g.replay()
    torch.cuda.synchronize()
    check(torch_to_np(x, 1), torch_to_np(y, 1), 1)
    _no_device_error()


def _grid_plan(rows, cols, dt, x_off=0, y_off=0):
    rc, dev = osd.softmax_device_query()
    assert rc == 0
    e = {0: 4, 1: 2, 2: 2}[dt]
    base = 1 << 40
    rc, p = osd.softmax_plan(dev, base + x_off * e, base + (1 << 38) + y_off * e, rows, cols, dt, GRID)
    assert rc == 0
    return dev, p


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_grid_ring_groups_and_depths(dt):
    # hand-made plans: the ring form with every CTA on every row (G = 1) and a
    # ring of 1 to 4 buffers, two groups, one group per row; the pipelined form
    # with 1 to 4 buffers and fold teams of 128, 256 and 384 threads; and plans
    # the checks refuse
    rng = np.random.default_rng(310 + dt)
    rows, cols = 4, (1 << 20) + 3
    x = rng.normal(0, 3, (rows, cols))
    x[:, ::89] += 55.0
    x = _quant(x, dt)
    dev, p = _grid_plan(rows, cols, dt, 1, 1)
    assert p.stages >= 1
    S = dev.sm_count
    budget = dev.max_smem_optin - 2048

    def buf_for(P):
        nch = (cols * {0: 4, 1: 2, 2: 2}[dt]) // 16 + 2
        return -(-(-(-nch // P) * 16) // 128) * 128

    good = []
    for G, Q in ((1, 1), (1, 2), (1, 4), (2, 1), (2, 2), (4, 1)):
        P = S // G
        if Q * buf_for(P) <= budget:
            good.append(dict(grid_x=P, grid_y=G, stages=Q, smem_bytes=Q * buf_for(P), lanes_per_row=0))
    for Q, NF in ((1, 256), (2, 128), (3, 384), (4, 256)):
        if Q * buf_for(S) <= budget:
            good.append(dict(grid_x=S, grid_y=1, stages=Q, smem_bytes=Q * buf_for(S), lanes_per_row=NF))
    assert len(good) >= 8
    for ch in good:
        q = osd.LaunchPlan(**{**p.as_dict(), **ch})
        rc, y = run(x, dt, plan=q, x_off=1, y_off=1)
        assert rc == 0, ch
        check(x, y, dt)
    ring = dict(lanes_per_row=0)
    pipe = dict(grid_x=S, grid_y=1, stages=2, smem_bytes=2 * buf_for(S), lanes_per_row=256)
    bad = [dict(ring, grid_y=rows + 1), dict(ring, grid_x=S + 1, grid_y=1), dict(ring, stages=9, smem_bytes=9 * 128),
           dict(smem_bytes=(p.smem_bytes // p.stages // 32 * 16) * p.stages), dict(smem_bytes=p.smem_bytes + 8),
           dict(pipe, grid_y=2), dict(pipe, grid_x=S + 1), dict(pipe, lanes_per_row=48),
           dict(pipe, lanes_per_row=512), dict(pipe, lanes_per_row=16), dict(pipe, stages=0, smem_bytes=0),
           dict(pipe, smem_bytes=2 * (buf_for(S) - 128))]
    for ch in bad:
        q = osd.LaunchPlan(**{**p.as_dict(), **ch})
        rc, _ = run(x, dt, plan=q, x_off=1, y_off=1)
        assert rc == osd.ERR_INVALID_ARG, ch
    _no_device_error()


def test_grid_slot_reuse_with_changing_row_counts():
    # blocks of 16 launches (one per scratch slot) with 7, then 3, then 7 rows:
    # every slot's third launch finds counters its second launch had no rows for
    torch.manual_seed(5)
    xa = torch.randn(7, 1 << 20, device="cuda", dtype=torch.float16) * 5
    xb = torch.randn(3, 1 << 20, device="cuda", dtype=torch.float16) * 5
    assert osd.plan_for(xa, torch.empty_like(xa)).variant == GRID
    assert osd.plan_for(xb, torch.empty_like(xb)).variant == GRID
    outs = []
    for i in range(64):
        outs.append(osd.softmax(xb if (i // 16) % 2 else xa))
    torch.cuda.synchronize()
    check(torch_to_np(xa, 1), torch_to_np(outs[0], 1), 1)
    check(torch_to_np(xb, 1), torch_to_np(outs[16], 1), 1)
    for i, o in enumerate(outs):
        ref = outs[16] if (i // 16) % 2 else outs[0]
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), i
    _no_device_error()
