"""In-place calls (y == x for the forward, dx == dy or dx == y for the
backward) against the oracle, through the C ABI, for every variant that serves
the shape, on aligned rows and on rows one element off the 16-byte grid; a
guard band around the buffer shows that nothing outside it is written.
Partial overlaps are refused."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import ELEM, GUARD, NUMPY, check, variants_for

pytestmark = pytest.mark.gpu

NAMES = {v: k for k, v in osd.VARIANTS.items()}
# the tolerances of the masked and backward parity tests
TOLM = {
    0: dict(rel_tol=2e-6, abs_floor=2.0**-126, rowsum_a=2e-6, rowsum_b=2.0**-126, zrel=0.0),
    1: dict(max_ulp=1, rowsum_a=2.0**-10, rowsum_b=2.0**-24, zrel=2.0**-22),
    2: dict(max_ulp=1, rowsum_a=2.0**-7, rowsum_b=2.0**-133, zrel=2.0**-22),
}
TOLB = {0: dict(rel_tol=2e-6, max_ulp=0, k_eps=8.0), 1: dict(max_ulp=1, k_eps=8.0), 2: dict(max_ulp=1, k_eps=8.0)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _quant(a64, dt):
    return a64.astype(NUMPY[dt]) if dt != 2 else W._round_to(a64, "bf16")


def _guarded(a, off, dt):
    """a copied into a device byte buffer at element offset `off` inside canary
    bands; returns (buffer, pointer)."""
    e = ELEM[dt]
    n = a.size
    b = torch.full((2 * GUARD + (n + off) * e,), 0xA5, dtype=torch.uint8, device="cuda")
    raw = torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).cuda()
    b[GUARD + off * e: GUARD + off * e + n * e].copy_(raw)
    return b, b.data_ptr() + GUARD + off * e


def _read_back(b, off, n, dt, shape):
    e = ELEM[dt]
    host = b.cpu().numpy()
    assert (host[: GUARD + off * e] == 0xA5).all() and (host[GUARD + off * e + n * e:] == 0xA5).all(), \
        "write outside the buffer"
    return host[GUARD + off * e: GUARD + off * e + n * e].view(NUMPY[dt]).reshape(shape).copy()


SHAPES = [(37, 3), (300, 511), (1000, 1000), (64, 5003), (9, 20011), (3, 70001), (2, 1 << 20)]


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_forward_in_place_every_variant(dt):
    rng = np.random.default_rng(70 + dt)
    s = torch.cuda.current_stream().cuda_stream
    for rows, cols in SHAPES:
        x = _quant(rng.normal(0, 6, (rows, cols)), dt)
        for off in (0, 1):
            for v in variants_for(rows, cols, dt, off, off):
                b, p = _guarded(x, off, dt)
                rc = osd.softmax_fwd_variant(p, p, rows, cols, dt, v, s)
                torch.cuda.synchronize()
                assert rc == 0, (rows, cols, off, NAMES[v])
                check(x, _read_back(b, off, x.size, dt, x.shape), dt)


@pytest.mark.parametrize("dt", [0, 1])
def test_forward_in_place_with_workspace_and_noalloc(dt):
    rows, cols = 4, (1 << 21) + 3
    x = _quant(np.random.default_rng(80 + dt).normal(0, 3, (rows, cols)), dt)
    s = torch.cuda.current_stream().cuda_stream
    for off in (0, 1):
        b, p = _guarded(x, off, dt)
        rc, need = osd.softmax_workspace_size(p, p, rows, cols, dt)
        assert rc == 0 and need > 0
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        assert osd.softmax_fwd_ws(p, p, rows, cols, dt, ws.data_ptr(), need, s) == 0
        torch.cuda.synchronize()
        check(x, _read_back(b, off, x.size, dt, x.shape), dt)
        b, p = _guarded(x, off, dt)
        assert osd.softmax_fwd_noalloc(p, p, rows, cols, dt, s) == 0
        torch.cuda.synchronize()
        check(x, _read_back(b, off, x.size, dt, x.shape), dt)


def test_forward_in_place_torch_api_and_partial_overlap():
    x = torch.randn(4, 32, 128, 512, device="cuda", dtype=torch.float16) * 20
    ref = x.cpu().numpy().reshape(-1, 512).copy()
    y = osd.softmax_(x)
    assert y.data_ptr() == x.data_ptr()
    check(ref, x.cpu().numpy().reshape(-1, 512), 1)
    buf = torch.randn(301 * 64, device="cuda")
    a, b = buf[: 300 * 64].view(300, 64), buf[64:].view(300, 64)  # b is a shifted by one row
    with pytest.raises(osd.SoftmaxError) as e:
        osd.softmax(a, out=b)
    assert e.value.status == -3
    s = torch.cuda.current_stream().cuda_stream
    assert osd.softmax_fwd(buf.data_ptr(), buf.data_ptr() + 4, 300, 64, 0, s) == -3


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_masked_in_place(dt):
    rng = np.random.default_rng(90 + dt)
    for rows, cols in ((512, 512), (300, 777), (64, 5003)):
        x = _quant(rng.normal(0, 4, (rows, cols)), dt)
        mask = _quant(rng.normal(0, 1, (1, cols)), dt)
        mb, mp = _guarded(mask, 0, dt)
        for off in (0, 1):
            for v in (osd.VARIANTS["rowgroup"], osd.VARIANTS["block"]):
                b, p = _guarded(x, off, dt)
                rc = osd.softmax_fwd_masked_variant(p, p, rows, cols, dt, 0.5, mp, 1, rows, v,
                                                    torch.cuda.current_stream().cuda_stream)
                torch.cuda.synchronize()
                if rc == -5:
                    continue
                assert rc == 0, (rows, cols, off, NAMES[v])
                y = _read_back(b, off, x.size, dt, x.shape)
                res = oracle.check_masked(x, y, dt, 0.5, mask, rows, **TOLM[dt])
                assert res["violations"] == 0 and res["rowsum_violations"] == 0, res


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_backward_in_place(dt):
    rng = np.random.default_rng(100 + dt)
    s = torch.cuda.current_stream().cuda_stream
    for rows, cols in ((300, 511), (64, 5003), (3, 70001)):
        y64 = rng.normal(0, 2, (rows, cols))
        y64 = np.exp(y64 - y64.max(1, keepdims=True))
        y = _quant(y64 / y64.sum(1, keepdims=True), dt)
        dy = _quant(rng.normal(0, 1, (rows, cols)), dt)
        for into in ("dy", "y"):
            for off in (0, 1):
                yb, yp = _guarded(y, off, dt)
                db, dp = _guarded(dy, off, dt)
                dxp = dp if into == "dy" else yp
                rc = osd.softmax_bwd(yp, dp, dxp, rows, cols, dt, s)
                torch.cuda.synchronize()
                assert rc == 0, (rows, cols, into, off)
                dx = _read_back(db if into == "dy" else yb, off, y.size, dt, y.shape)
                res = oracle.check_bwd(y, dy, dx, dt, **TOLB[dt])
                assert res["nonfinite"] == 0, res
                assert res["violations"] == 0, (rows, cols, into, off, res)
