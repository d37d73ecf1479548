"""GPU parity of softmax_fwd_ws (few, very long rows split over every SM, with
the partial statistics in a caller-provided workspace) against the oracle,
through the C ABI; y and the workspace sit between canary guard bands."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import ELEM, GUARD, NUMPY, check, np_to_torch, torch_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _quant(a64, dt):
    return a64.astype(NUMPY[dt]) if dt != 2 else W._round_to(a64, "bf16")


def run_ws(x, dt, x_off=0, y_off=0, ws_bytes=None):
    """softmax_fwd_ws on device copies of x; returns (status, y, workspace bytes used)."""
    rows, cols = x.shape
    e = ELEM[dt]
    n = rows * cols
    dev = torch.device("cuda")
    xb = torch.empty(n * e + 64 + x_off * e, dtype=torch.uint8, device=dev)
    xb[x_off * e: x_off * e + n * e].copy_(torch.from_numpy(np.ascontiguousarray(x).view(np.uint8).reshape(-1)).to(dev))
    yb = torch.full((2 * GUARD + n * e + y_off * e,), 0xA5, dtype=torch.uint8, device=dev)
    xp, yp = xb.data_ptr() + x_off * e, yb.data_ptr() + GUARD + y_off * e
    rc, need = osd.softmax_workspace_size(xp, yp, rows, cols, dt)
    assert rc == 0
    size = need if ws_bytes is None else ws_bytes
    wb = torch.full((2 * GUARD + size,), 0x3C, dtype=torch.uint8, device=dev)
    wp = wb.data_ptr() + GUARD
    rc = osd.softmax_fwd_ws(xp, yp, rows, cols, dt, wp if size else 0, size, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = yb.cpu().numpy()
    assert (host[: GUARD + y_off * e] == 0xA5).all() and (host[GUARD + y_off * e + n * e:] == 0xA5).all()
    wh = wb.cpu().numpy()
    assert (wh[:GUARD] == 0x3C).all() and (wh[GUARD + size:] == 0x3C).all(), "write outside the workspace"
    y = host[GUARD + y_off * e: GUARD + y_off * e + n * e].view(NUMPY[dt]).reshape(rows, cols).copy()
    return rc, y, need


@pytest.mark.parametrize("name", ["splitk_fp32_4x4194304", "splitk_fp16_4x4194304"])
def test_wide_full_size_workloads(name):
    w = W.WORKLOADS[name]
    x = W.generate(w)
    xt = np_to_torch(x, w.dtype_code).cuda()
    y = torch.empty_like(xt)
    rc, need = osd.softmax_workspace_size(xt.data_ptr(), y.data_ptr(), w.rows, w.cols, w.dtype_code)
    assert rc == 0 and need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    osd.softmax(xt, out=y, workspace=ws)
    torch.cuda.synchronize()
    check(x, torch_to_np(y, w.dtype_code), w.dtype_code)
    # two calls in a row on the same workspace give the same bits
    y2 = osd.softmax(xt, workspace=ws)
    assert torch.equal(y.view(torch.uint8), y2.view(torch.uint8))


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_wide_shapes_and_offsets(dt):
    rng = np.random.default_rng(40 + dt)
    for rows, cols in ((1, 300001), (3, 1 << 20), (7, 150003), (2, (1 << 21) + 5)):
        x = rng.normal(0, 4, (rows, cols))
        x[:, ::97] += 60.0
        x = _quant(x, dt)
        for xo, yo in ((0, 0), (1, 1), (0, 3)):
            rc, y, need = run_ws(x, dt, xo, yo)
            assert rc == 0 and need > 0
            check(x, y, dt)


def test_wide_special_rows():
    for dt in (0, 1, 2):
        cols = 400000
        x = np.random.default_rng(3).normal(0, 2, (4, cols))
        x[0, : cols // 2] = -np.inf
        x[1, 7] = np.nan
        x[2, :] = -np.inf
        x = _quant(x, dt)
        rc, y, _ = run_ws(x, dt)
        assert rc == 0
        check(x, y, dt, finite_expected=False)
        yd = oracle.decode(y, dt)
        assert np.isnan(yd[1]).all() and np.isnan(yd[2]).all() and np.isfinite(yd[[0, 3]]).all()


def test_wide_fallbacks_and_errors():
    x = _quant(np.random.default_rng(5).normal(0, 1, (4, 1 << 20)), 1)
    # too small a workspace: the cluster split runs instead, still correct
    rc, y, need = run_ws(x, 1, ws_bytes=16)
    assert rc == 0 and need > 16
    check(x, y, 1)
    # shapes that need no workspace report 0 and run the ordinary dispatcher
    xs = _quant(np.random.default_rng(6).normal(0, 1, (4096, 512)), 1)
    rc, y, need = run_ws(xs, 1)
    assert rc == 0 and need == 0
    check(xs, y, 1)
    xt = torch.randn(4, 1 << 20, device="cuda")
    yt = torch.empty_like(xt)
    s = torch.cuda.current_stream().cuda_stream
    # the variant cannot run without a workspace
    assert osd.softmax_fwd_variant(xt.data_ptr(), yt.data_ptr(), 4, 1 << 20, 0, 6, s) == -1
    # a workspace inside y is refused; null with a size is refused
    assert osd.softmax_fwd_ws(xt.data_ptr(), yt.data_ptr(), 4, 1 << 20, 0, yt.data_ptr() + 4096, 4096, s) == -3
    assert osd.softmax_fwd_ws(xt.data_ptr(), yt.data_ptr(), 4, 1 << 20, 0, 0, 4096, s) == -1
