"""GPU parity of the softmax backward (dx = y * (dy - sum dy*y)) against the
fp64 oracle, through the C ABI, dx between canary guard bands.  y is the
oracle's forward output rounded to the dtype (independent of the GPU forward
path); dy is seeded N(0, 1).  Tolerance (include/softmax.h): 1 ulp of the
dtype (fp32: 2e-6 relative) plus 8 * 2^-24 * y_j * (|dy_j| + sum_k |dy_k y_k|)."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import ELEM, GUARD, NUMPY

pytestmark = pytest.mark.gpu

NAMES = {v: k for k, v in osd.VARIANTS.items()}
TOL = {0: dict(rel_tol=2e-6, max_ulp=0, k_eps=8.0), 1: dict(max_ulp=1, k_eps=8.0), 2: dict(max_ulp=1, k_eps=8.0)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _quant(a64, dt):
    return a64.astype(NUMPY[dt]) if dt != 2 else W._round_to(a64, "bf16")


def make_case(rows, cols, dt, seed, scale=3.0):
    rng = np.random.default_rng(seed)
    x = _quant(rng.normal(0, scale, (rows, cols)), dt)
    y = oracle.softmax_rounded(x, dt)
    if dt == 0:
        y = y.astype(np.float32)
    dy = _quant(rng.normal(0, 1, (rows, cols)), dt)
    return y, dy


def run_bwd(y, dy, dt, variant=0, offs=(0, 0, 0)):
    rows, cols = y.shape
    e = ELEM[dt]
    n = rows * cols
    dev = torch.device("cuda")
    bufs = []
    for a, o in ((y, offs[0]), (dy, offs[1])):
        b = torch.empty(n * e + 64 + o * e, dtype=torch.uint8, device=dev)
        b[o * e: o * e + n * e].copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).to(dev))
        bufs.append((b, b.data_ptr() + o * e))
    xb = torch.full((2 * GUARD + n * e + offs[2] * e,), 0x5A, dtype=torch.uint8, device=dev)
    dxp = xb.data_ptr() + GUARD + offs[2] * e
    rc = osd.softmax_bwd_variant(bufs[0][1], bufs[1][1], dxp, rows, cols, dt, variant,
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = xb.cpu().numpy()
    lo, hi = host[: GUARD + offs[2] * e], host[GUARD + offs[2] * e + n * e:]
    assert (lo == 0x5A).all() and (hi == 0x5A).all(), "write outside dx"
    dx = host[GUARD + offs[2] * e: GUARD + offs[2] * e + n * e].view(NUMPY[dt]).reshape(rows, cols).copy()
    return rc, dx


def check_bwd(y, dy, dx, dt):
    res = oracle.check_bwd(y, dy, dx, dt, **TOL[dt])
    assert res["violations"] == 0, res
    assert res["nonfinite"] == 0, res
    return res


def bwd_variants():
    return [0, osd.VARIANTS["rowgroup"], osd.VARIANTS["block"], osd.VARIANTS["stream"]]


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_bwd_shapes_and_variants(dt):
    # (2049 .. 4096 chunks: the cluster-pair kernel for BLOCK)
    for cols in list(range(1, 34)) + [63, 64, 65, 255, 256, 512, 513, 1000, 2047, 2048, 2049, 5003, 8193, 16384,
                                      20000, 24577, 32000, 40001]:
        for rows in (1, 7):
            y, dy = make_case(rows, cols, dt, seed=cols * 10 + rows)
            for v in bwd_variants():
                for offs in ((0, 0, 0), (1, 1, 1), (0, 1, 2)):
                    rc, dx = run_bwd(y, dy, dt, v, offs)
                    if rc == -5:  # variant cannot serve this row length
                        assert v in (osd.VARIANTS["rowgroup"], osd.VARIANTS["block"])
                        continue
                    assert rc == 0, (cols, rows, NAMES[v], offs, rc)
                    check_bwd(y, dy, dx, dt)


@pytest.mark.parametrize("name", ["attn_fp16_65536x512", "awkward_fp16_8192x5003", "vocab_bf16_32768x32000",
                                  "fp32_128x1000", "splitk_fp16_4x4194304"])
def test_bwd_workload_shapes(name):
    w = W.WORKLOADS[name]
    rows = {"attn_fp16_65536x512": 65536, "awkward_fp16_8192x5003": 8192, "vocab_bf16_32768x32000": 2048,
            "fp32_128x1000": 128, "splitk_fp16_4x4194304": 4}[name]
    x = W.generate(w, rows=rows)
    y = oracle.softmax_rounded(x, w.dtype_code)
    if w.dtype_code == 0:
        y = y.astype(np.float32)
    dy = _quant(np.random.default_rng(5).normal(0, 1, x.shape), w.dtype_code)
    rc, dx = run_bwd(y, dy, w.dtype_code)
    assert rc == 0
    check_bwd(y, dy, dx, w.dtype_code)


def test_bwd_closed_cases():
    # dy constant -> dx ~ 0; y one-hot -> dx = 0 everywhere
    for dt in (0, 1, 2):
        y, _ = make_case(5, 300, dt, seed=3)
        dy = _quant(np.full(y.shape, 2.5), dt)
        rc, dx = run_bwd(y, dy, dt)
        assert rc == 0
        check_bwd(y, dy, dx, dt)
        onehot = np.zeros((3, 70))
        onehot[np.arange(3), [0, 33, 69]] = 1.0
        yo = _quant(onehot, dt)
        dyo = _quant(np.random.default_rng(1).normal(0, 1, (3, 70)), dt)
        rc, dx = run_bwd(yo, dyo, dt)
        assert rc == 0 and (oracle.decode(dx, dt) == 0).all()


def test_bwd_torch_api_and_alias():
    y = torch.softmax(torch.randn(300, 777, device="cuda"), -1)
    dy = torch.randn_like(y)
    dx = osd.softmax_backward(y, dy)
    check_bwd(y.cpu().numpy(), dy.cpu().numpy(), dx.cpu().numpy(), 0)
    # dx may be dy itself (in place); a partial overlap is refused
    buf = torch.randn(301 * 777, device="cuda")
    with pytest.raises(osd.SoftmaxError) as e:
        osd.softmax_backward(y, buf[: 300 * 777].view(300, 777), out=buf[777:].view(300, 777))
    assert e.value.status == -3
    # y and dy may be the same buffer (both are only read)
    dx2 = osd.softmax_backward(y, y)
    check_bwd(y.cpu().numpy(), y.cpu().numpy(), dx2.cpu().numpy(), 0)


def test_bwd_stream_walks_back_on_long_rows():
    # the streaming backward kernel's write pass walks each row from its end
    # where the rows in flight hold more than half of L2 in y and dy: parity
    # on shapes on both sides of that line, on and off the 16-byte grid
    rc, dev = osd.softmax_device_query()
    assert rc == 0
    for dt, rows, cols, off in ((1, 400, 65600, 0), (2, 400, 65600, 0), (0, 320, 65536, 0), (1, 400, 131073, 1),
                                (1, 400, 65601, 1), (0, 40, 65536, 0)):
        e = ELEM[dt]
        b = 1 << 40
        rc, p = osd.softmax_bwd_plan(dev, b + off * e, b + (1 << 38) + off * e, b + (2 << 38) + off * e, rows, cols,
                                     dt, 0)
        assert rc == 0 and p.variant == osd.VARIANTS["stream"]
        resident = dev.sm_count * (2 if p.aligned else 1)
        assert p.back_passes == int(min(rows, resident) * 2 * cols * e > dev.l2_bytes // 2), (dt, rows, cols)
        y, dy = make_case(rows, cols, dt, seed=rows + cols)
        rc, dx = run_bwd(y, dy, dt, 0, (off, off, off))
        assert rc == 0
        check_bwd(y, dy, dx, dt)
