"""GPU parity of LayerNorm and RMSNorm (layernorm_fwd / rmsnorm_fwd /
norm_fwd_variant) against the oracle, through the C ABI, y between canary
guard bands.  Tolerance (include/softmax.h): 1 ulp of the dtype (fp16 / bf16)
plus 64 * 2^-24 * (|g| (|z| + a rstd) + |b|); the per-row mean and rstd within
64 * 2^-24 of a and of rstd."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import ELEM, GUARD, NUMPY, np_to_torch

pytestmark = pytest.mark.gpu

NAMES = {v: k for k, v in osd.VARIANTS.items()}
KEPS = 64.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _quant(a64, dt):
    return a64.astype(NUMPY[dt]) if dt != 2 else W._round_to(a64, "bf16")


def _dev(a, off, dt):
    e = ELEM[dt]
    b = torch.empty(a.size * e + 64 + off * e, dtype=torch.uint8, device="cuda")
    b[off * e: off * e + a.size * e].copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).cuda())
    return b, b.data_ptr() + off * e


def run_norm(kind, x, dt, g=None, b=None, eps=1e-5, variant=0, offs=(0, 0, 0), stats=True):
    """offs: element offsets of x, y and the gain / bias vectors."""
    rows, cols = x.shape
    e = ELEM[dt]
    n = rows * cols
    xb, xp = _dev(x, offs[0], dt)
    gb, gp = _dev(g, offs[2], dt) if g is not None else (None, 0)
    bb, bp = _dev(b, offs[2], dt) if b is not None else (None, 0)
    yb = torch.full((2 * GUARD + n * e + offs[1] * e,), 0xA5, dtype=torch.uint8, device="cuda")
    yp = yb.data_ptr() + GUARD + offs[1] * e
    mean = torch.full((rows + 2,), 7.0, device="cuda") if stats else None
    rstd = torch.full((rows + 2,), 7.0, device="cuda") if stats else None
    rc = osd.norm_fwd_variant(kind, xp, yp, rows, cols, dt, gp, bp, eps,
                              mean.data_ptr() + 4 if stats else 0, rstd.data_ptr() + 4 if stats else 0, variant,
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = yb.cpu().numpy()
    assert (host[: GUARD + offs[1] * e] == 0xA5).all() and (host[GUARD + offs[1] * e + n * e:] == 0xA5).all()
    y = host[GUARD + offs[1] * e: GUARD + offs[1] * e + n * e].view(NUMPY[dt]).reshape(rows, cols).copy()
    m = r = None
    if stats:
        mh, rh = mean.cpu().numpy(), rstd.cpu().numpy()
        assert rh[0] == 7.0 and rh[-1] == 7.0 and mh[0] == 7.0 and mh[-1] == 7.0, "write outside mean / rstd"
        m, r = mh[1:-1], rh[1:-1]
        if kind == osd.RMSNORM:
            assert (mh == 7.0).all(), "RMSNorm writes no mean"
            m = None
    return rc, y, m, r


def check_norm(kind, x, y, dt, g=None, b=None, eps=1e-5, mean=None, rstd=None, finite_expected=True):
    tol = dict(max_ulp=0 if dt == 0 else 1, k_eps=KEPS)
    res = oracle.check_norm(kind, x, y, dt, g, b if kind == 0 else None, eps, mean, rstd, **tol)
    assert res["violations"] == 0, res
    assert res["rowsum_violations"] == 0, res
    if finite_expected:
        assert res["nonfinite"] == 0, res
    return res


def _variants(cols, dt):
    nint = cols * ELEM[dt] // 16
    out = [0, osd.VARIANTS["block"]]
    if max(nint, 1) <= 128:
        out.append(osd.VARIANTS["rowgroup"])
    return out


@pytest.mark.parametrize("dt", [0, 1, 2])
@pytest.mark.parametrize("kind", [0, 1])
def test_norm_shapes_offsets_affine(kind, dt):
    rng = np.random.default_rng(200 + 10 * kind + dt)
    cols_list = list(range(1, 41)) + [63, 64, 65, 127, 128, 129, 192, 384, 511, 512, 1000, 1024, 4093, 4096, 8200]
    for cols in cols_list:
        rows = 5 if cols > 1000 else 11
        x = _quant(rng.normal(rng.uniform(-3, 3), rng.uniform(0.5, 5), (rows, cols)), dt)
        g = _quant(rng.normal(1, 0.3, cols), dt)
        b = _quant(rng.normal(0, 0.5, cols), dt)
        for offs in ((0, 0, 0), (1, 1, 0), (0, 0, 1), (1, 2, 3)):
            for v in _variants(cols, dt):
                for affine in (False, True):
                    gg, bb = (g, b) if affine else (None, None)
                    rc, y, m, r = run_norm(kind, x, dt, gg, bb, 1e-5, v, offs)
                    assert rc == 0, (cols, offs, NAMES[v], affine)
                    check_norm(kind, x, y, dt, gg, bb, 1e-5, m, r)


@pytest.mark.parametrize("name", list(W.NORM_WORKLOADS))
def test_norm_workloads_full_size(name):
    w = W.NORM_WORKLOADS[name]
    x = W.generate(w)
    g, b = W.norm_params(w)
    xt = np_to_torch(x, w.dtype_code).cuda()
    gt = np_to_torch(g, w.dtype_code).cuda() if g is not None else None
    bt = np_to_torch(b, w.dtype_code).cuda() if b is not None else None
    mean = torch.empty(w.rows, device="cuda")
    rstd = torch.empty(w.rows, device="cuda")
    if w.kind == 0:
        y = osd.layer_norm(xt, gt, bt, eps=w.eps, mean=mean, rstd=rstd)
    else:
        y = osd.rms_norm(xt, gt, eps=w.eps, rstd=rstd)
    torch.cuda.synchronize()
    from tests.gpu_helpers import torch_to_np
    check_norm(w.kind, x, torch_to_np(y, w.dtype_code), w.dtype_code, g, b, w.eps,
               mean.cpu().numpy() if w.kind == 0 else None, rstd.cpu().numpy())


def test_norm_special_rows():
    for dt in (0, 1, 2):
        cols = 300
        x = np.random.default_rng(5).normal(0, 1, (6, cols))
        x[0] = 0.75          # constant row: y = beta (eps > 0)
        x[1, :] = 1e3        # large common level
        x[1, ::2] += 1.0
        x[2, 5] = np.nan     # NaN propagates to the row
        x[3] = 0.0           # all zero
        x = _quant(x, dt)
        b = _quant(np.linspace(-1, 1, cols), dt)
        for kind in (0, 1):
            rc, y, m, r = run_norm(kind, x, dt, None, b if kind == 0 else None, 1e-5)
            assert rc == 0
            check_norm(kind, x, y, dt, None, b if kind == 0 else None, 1e-5, m, r, finite_expected=False)
            yd = oracle.decode(y, dt)
            assert np.isnan(yd[2]).all() and np.isfinite(yd[[0, 1, 3, 4, 5]]).all()
        # eps = 0 and a constant row: 0 * inf = NaN, as the definition gives
        rc, y, _, _ = run_norm(0, x[:1], dt, None, None, 0.0)
        assert rc == 0 and np.isnan(oracle.decode(y, dt)).all()


def test_norm_in_place_and_torch_api():
    x = torch.randn(4096, 384, device="cuda", dtype=torch.float16) * 3 + 1
    ref = x.cpu().numpy().copy()
    w = torch.randn(384, device="cuda", dtype=torch.float16)
    bias = torch.randn(384, device="cuda", dtype=torch.float16)
    y = osd.layer_norm(x, w, bias, out=x)
    assert y.data_ptr() == x.data_ptr()
    check_norm(0, ref, x.cpu().numpy(), 1, w.cpu().numpy(), bias.cpu().numpy(), 1e-5)
    # against torch's own layer norm: within the same budget
    x2 = torch.randn(64, 1000, device="cuda")
    yt = torch.nn.functional.layer_norm(x2, (1000,), eps=1e-5)
    assert (osd.layer_norm(x2) - yt).abs().max().item() < 1e-5
    yr = torch.nn.functional.rms_norm(x2, (1000,), eps=1e-6)
    assert (osd.rms_norm(x2) - yr).abs().max().item() < 1e-5


def test_norm_errors():
    s = torch.cuda.current_stream().cuda_stream
    x = torch.randn(8, 64, device="cuda")
    y = torch.empty_like(x)
    g = torch.ones(64, device="cuda")
    # gain overlapping y is refused; eps must be >= 0 and finite
    assert osd.layernorm_fwd(x.data_ptr(), y.data_ptr(), 8, 64, 0, y.data_ptr(), 0, 1e-5, 0, 0, s) == -3
    assert osd.layernorm_fwd(x.data_ptr(), y.data_ptr(), 8, 64, 0, g.data_ptr(), 0, -1.0, 0, 0, s) == -1
    assert osd.layernorm_fwd(x.data_ptr(), y.data_ptr(), 8, 64, 0, g.data_ptr(), 0, float("nan"), 0, 0, s) == -1
    # rows of more than 64 KiB are not served
    big = torch.randn(2, 20000, device="cuda")
    assert osd.rmsnorm_fwd(big.data_ptr(), torch.empty_like(big).data_ptr(), 2, 20000, 0, 0, 1e-6, 0, s) == -5
    # the rowgroup variant serves rows of up to 128 chunks only
    mid = torch.randn(2, 600, device="cuda")
    assert osd.norm_fwd_variant(0, mid.data_ptr(), torch.empty_like(mid).data_ptr(), 2, 600, 0, 0, 0, 1e-5, 0, 0,
                                osd.VARIANTS["rowgroup"], s) == -5
