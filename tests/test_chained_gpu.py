"""Dependent launches back to back on one stream, with no host synchronisation
between them: every kernel of the library starts with programmatic dependent
launch, so each one may begin while its predecessor drains, and must see the
predecessor's writes before it reads.  Each chain is checked against the
oracle applied to the same chain on the host."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from tests.gpu_helpers import check, torch_to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _enc(v64, dt):
    return oracle.encode(v64, dt) if dt else v64.astype(np.float32)


@pytest.mark.parametrize("shape", [(65536, 512), (8192, 5003), (64, 40000), (4, 1 << 21)])
def test_softmax_of_softmax_chain(shape):
    # y_{k+1} = softmax(y_k), each launch reading what the previous one wrote
    torch.manual_seed(0)
    x = torch.randn(*shape, device="cuda", dtype=torch.float16) * 8
    bufs = [x] + [torch.empty_like(x) for _ in range(3)]
    for k in range(3):
        osd.softmax(bufs[k], out=bufs[k + 1])
    torch.cuda.synchronize()
    for k in range(3):
        check(torch_to_np(bufs[k], 1), torch_to_np(bufs[k + 1], 1), 1)


def test_in_place_chain_and_mixed_ops():
    torch.manual_seed(1)
    x = torch.randn(4096, 1000, device="cuda", dtype=torch.bfloat16) * 4
    x0 = torch_to_np(x, 2).copy()
    # in place twice, then the backward on the result with dy = the result
    osd.softmax_(x)
    y1 = x.clone()  # a copy kernel in between (torch's own, plain stream order)
    osd.softmax_(x)
    dx = osd.softmax_backward(x, y1)
    ln = osd.layer_norm(dx, eps=1e-5)
    y3 = osd.softmax(ln)
    torch.cuda.synchronize()
    a1 = torch_to_np(y1, 2)
    check(x0, a1, 2)
    a2 = torch_to_np(x, 2)
    check(a1, a2, 2)
    res = oracle.check_bwd(a2, a1, torch_to_np(dx, 2), 2, max_ulp=1, k_eps=8.0)
    assert res["violations"] == 0, res
    d = torch_to_np(dx, 2)
    res = oracle.check_norm(0, d, torch_to_np(ln, 2), 2, None, None, 1e-5, max_ulp=1, k_eps=64.0)
    assert res["violations"] == 0, res
    check(torch_to_np(ln, 2), torch_to_np(y3, 2), 2)


def test_wide_split_chain():
    # the two-launch split (statistics, then write) twice in a row on the
    # same workspace: the second call's first kernel must not overwrite the
    # partials the first call's second kernel is still reading
    torch.manual_seed(2)
    x = torch.randn(4, 3_000_001, device="cuda") * 3
    y1, y2 = torch.empty_like(x), torch.empty_like(x)
    rc, need = osd.softmax_workspace_size(x.data_ptr(), y1.data_ptr(), 4, 3_000_001, 0)
    assert rc == 0 and need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    osd.softmax(x, out=y1, workspace=ws)
    osd.softmax(y1, out=y2, workspace=ws)
    torch.cuda.synchronize()
    check(x.cpu().numpy(), y1.cpu().numpy(), 0)
    check(y1.cpu().numpy(), y2.cpu().numpy(), 0)
