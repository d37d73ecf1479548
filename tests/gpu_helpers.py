"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
device buffers with guard bands, and compare with the oracle at the tolerances
the library promises (include/softmax.h):

    fp32        |y - y*| <= 2e-6 y* + 2^-126
    fp16, bf16  |bits(y) - bits(RNE(y*))| <= 1
    row sums    fp32 |sum - 1| <= 2e-6 + cols 2^-126
                fp16 2^-10 + cols 2^-24,  bf16 2^-7 + cols 2^-133
"""
import numpy as np
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle

TOL = {
    0: dict(rel_tol=2e-6, abs_floor=2.0**-126, rowsum_a=2e-6, rowsum_b=2.0**-126),
    1: dict(max_ulp=1, rowsum_a=2.0**-10, rowsum_b=2.0**-24),
    2: dict(max_ulp=1, rowsum_a=2.0**-7, rowsum_b=2.0**-133),
}
TORCH = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}
NUMPY = {0: np.float32, 1: np.float16, 2: np.uint16}
ELEM = {0: 4, 1: 2, 2: 2}
GUARD = 4096  # bytes of canary on each side of y


def np_to_torch(a: np.ndarray, dt: int) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dt == 2:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t


def torch_to_np(t: torch.Tensor, dt: int) -> np.ndarray:
    t = t.cpu()
    if dt == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run(x: np.ndarray, dt: int, variant=0, plan=None, x_off: int = 0, y_off: int = 0, stream=None):
    """softmax of x on the GPU via the C ABI.  x_off / y_off shift x and y by
    that many ELEMENTS from a 256-byte aligned base.  y lies inside canary
    guard bands that are checked after the kernel.  Returns (status, y)."""
    rows, cols = x.shape
    e = ELEM[dt]
    n = rows * cols
    dev = torch.device("cuda")
    xb = torch.empty(n * e + 64 + x_off * e, dtype=torch.uint8, device=dev)
    xb[x_off * e: x_off * e + n * e].copy_(torch.from_numpy(np.ascontiguousarray(x).view(np.uint8).reshape(-1)).to(dev))
    yb = torch.full((2 * GUARD + n * e + y_off * e,), 0xA5, dtype=torch.uint8, device=dev)
    xp = xb.data_ptr() + x_off * e
    yp = yb.data_ptr() + GUARD + y_off * e
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    if plan is not None:
        rc = osd.softmax_fwd_plan(xp, yp, rows, cols, dt, plan, s)
    else:
        rc = osd.softmax_fwd_variant(xp, yp, rows, cols, dt, variant, s)
    torch.cuda.synchronize()
    host = yb.cpu().numpy()
    lo, hi = host[: GUARD + y_off * e], host[GUARD + y_off * e + n * e:]
    assert (lo == 0xA5).all() and (hi == 0xA5).all(), "write outside y"
    y = host[GUARD + y_off * e: GUARD + y_off * e + n * e].view(NUMPY[dt]).reshape(rows, cols).copy()
    return rc, y


def check(x: np.ndarray, y: np.ndarray, dt: int, finite_expected: bool = True, rows_sel=None):
    res = oracle.check(x, y, dt, rows_sel=rows_sel, **TOL[dt])
    assert res["violations"] == 0, res
    assert res["rowsum_violations"] == 0, res
    if finite_expected:
        assert res["nonfinite"] == 0, res
    return res


def variants_for(rows: int, cols: int, dt: int, x_off: int = 0, y_off: int = 0):
    """Variants the dispatcher accepts for this shape on the current device."""
    rc, dev = osd.softmax_device_query()
    assert rc == 0
    e = ELEM[dt]
    base = 1 << 40
    x, y = base + x_off * e, base + (1 << 38) + y_off * e
    out = []
    for v in range(osd.VARIANTS["splitk"] + 1):
        rc, _ = osd.softmax_plan(dev, x, y, rows, cols, dt, v)
        if rc == 0:
            out.append(v)
    return out
