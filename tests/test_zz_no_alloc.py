"""softmax_fwd_noalloc: the wide split with its scratch in the library's fixed
array, for callers that may not allocate device memory (a plugin whose host
engine owns every allocation, a latency-critical path where cudaMalloc may
synchronise the device).  Called through the C ABI, its output must match the
existing workspace entry point (softmax_fwd_ws, workspace allocated here) on
two calls in a row, within the tolerances the parity tests use.  This file is
collected last on purpose."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
from online_softmax_dispatcher_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _within(a: torch.Tensor, b: torch.Tensor, dt: int) -> bool:
    if dt == 0:
        a64, b64 = a.double(), b.double()
        return bool(((a64 - b64).abs() <= 2e-6 * b64.abs() + 2.0**-126).all())
    ai = a.view(torch.int16).to(torch.int32) & 0xFFFF
    bi = b.view(torch.int16).to(torch.int32) & 0xFFFF
    return bool(((ai - bi).abs() <= 1).all())


@pytest.mark.parametrize("name,rows", [("splitk_fp32_4x4194304", 4), ("splitk_fp16_4x4194304", 4),
                                       ("vocab_bf16_32768x32000", 3)])
def test_noalloc_matches_workspace_entry_point(name, rows):
    w = W.WORKLOADS[name]
    x = W.as_torch(W.generate(w, rows=rows), w.dtype).cuda()
    s = torch.cuda.current_stream().cuda_stream
    ref = torch.empty_like(x)
    rc, need = osd.softmax_workspace_size(x.data_ptr(), ref.data_ptr(), rows, w.cols, w.dtype_code)
    assert rc == 0
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    assert osd.softmax_fwd_ws(x.data_ptr(), ref.data_ptr(), rows, w.cols, w.dtype_code, ws.data_ptr(),
                              ws.numel(), s) == 0
    for _ in range(2):
        y = torch.full_like(x, float("nan"))
        assert osd.softmax_fwd_noalloc(x.data_ptr(), y.data_ptr(), rows, w.cols, w.dtype_code, s) == 0
        torch.cuda.synchronize()
        assert _within(y, ref, w.dtype_code)


def test_noalloc_refuses_more_partials_than_it_holds():
    x = torch.randn(5000, 64, device="cuda")
    y = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert osd.softmax_fwd_noalloc(x.data_ptr(), y.data_ptr(), 5000, 64, 0, s) == -5
    # argument checks come first, as for every entry point: y one element past
    # x overlaps it without being an in-place call
    assert osd.softmax_fwd_noalloc(x.data_ptr(), x.data_ptr() + 4, 5000, 64, 0, s) == -3
