"""softmax_fwd_noalloc: the wide split with its scratch in the library's fixed
array, for callers that may not allocate device memory (a plugin whose host
engine owns every allocation, a latency-critical path where cudaMalloc may
synchronise the device).  Called through the C ABI, its output must be
bit-identical to the existing workspace entry point's (softmax_fwd_ws, with a
workspace allocated here) on two calls in a row -- both run the same kernels
with the same plan and merge the partials in the same fixed order, so any
difference would mean a stale or shared scratch read -- and within the
library's tolerances of the oracle.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import check, torch_to_np

pytestmark = pytest.mark.gpu

SLOTS = 4096  # partial-statistics slots of the fixed array (rows x CTAs per row)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


@pytest.mark.parametrize("name,rows", [("splitk_fp32_4x4194304", 4), ("splitk_fp16_4x4194304", 4),
                                       ("vocab_bf16_32768x32000", 3)])
def test_noalloc_matches_workspace_entry_point(name, rows):
    w = W.WORKLOADS[name]
    x_np = W.generate(w, rows=rows)
    x = W.as_torch(x_np, w.dtype).cuda()
    s = torch.cuda.current_stream().cuda_stream
    ref = torch.empty_like(x)
    rc, need = osd.softmax_workspace_size(x.data_ptr(), ref.data_ptr(), rows, w.cols, w.dtype_code)
    assert rc == 0
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    assert osd.softmax_fwd_ws(x.data_ptr(), ref.data_ptr(), rows, w.cols, w.dtype_code, ws.data_ptr(),
                              ws.numel(), s) == 0
    for call in range(2):
        y = torch.full_like(x, float("nan"))
        assert osd.softmax_fwd_noalloc(x.data_ptr(), y.data_ptr(), rows, w.cols, w.dtype_code, s) == 0
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.uint8), ref.view(torch.uint8)), f"call {call}: differs from softmax_fwd_ws"
        check(x_np, torch_to_np(y, w.dtype_code), w.dtype_code)


def test_noalloc_largest_accepted_and_first_refused_shape():
    rc, dev = osd.softmax_device_query()
    assert rc == 0
    s = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(11)
    # rows x P == the array's slots exactly (P = 1 CTA per row at this many rows)
    rows, cols = SLOTS, 3001
    x_np = rng.normal(0, 3, (rows, cols)).astype(np.float16)
    x = torch.from_numpy(x_np).cuda()
    rc, plan = osd.softmax_plan(dev, x.data_ptr(), x.data_ptr() + (1 << 36), rows, cols, 1,
                                osd.VARIANTS["splitk_wide"])
    assert rc == 0 and plan.grid_x * plan.grid_y == SLOTS
    for _ in range(2):
        y = torch.full_like(x, float("nan"))
        assert osd.softmax_fwd_noalloc(x.data_ptr(), y.data_ptr(), rows, cols, 1, s) == 0
        torch.cuda.synchronize()
        check(x_np, y.cpu().numpy(), 1)
    # one partial more than the array holds is refused, and nothing is written
    xr = torch.randn(SLOTS + 1, 64, device="cuda")
    yr = torch.full_like(xr, 7.0)
    assert osd.softmax_fwd_noalloc(xr.data_ptr(), yr.data_ptr(), SLOTS + 1, 64, 0, s) == -5
    torch.cuda.synchronize()
    assert bool((yr == 7.0).all())


def test_noalloc_refuses_more_partials_than_it_holds():
    x = torch.randn(5000, 64, device="cuda")
    y = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert osd.softmax_fwd_noalloc(x.data_ptr(), y.data_ptr(), 5000, 64, 0, s) == -5
    # argument checks come first, as for every entry point: y one element past
    # x overlaps it without being an in-place call
    assert osd.softmax_fwd_noalloc(x.data_ptr(), x.data_ptr() + 4, 5000, 64, 0, s) == -3
