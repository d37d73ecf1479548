"""GPU parity of the scaled, masked softmax (softmax(scale * x + mask) with an
optional causal cut) against the oracle, through the C ABI, y between canary
guard bands.  Tolerances: those of softmax_fwd (fp32 2e-6 relative, fp16 /
bf16 1 ulp of the correctly rounded result), whatever the size of the logits.

The C ABI takes `scale` as a C float, so the call computes with fl32(scale):
the oracle is given that same value (scale * x is then exact in binary64),
which makes it the definition of the call as made."""
import numpy as np
import pytest
import torch

import online_softmax_dispatcher_gb300 as osd
import oracle
from online_softmax_dispatcher_gb300 import workloads as W
from tests.gpu_helpers import ELEM, GUARD, NUMPY

pytestmark = pytest.mark.gpu

NAMES = {v: k for k, v in osd.VARIANTS.items()}
TOLM = {
    0: dict(rel_tol=2e-6, abs_floor=2.0**-126, rowsum_a=2e-6, rowsum_b=2.0**-126),
    1: dict(max_ulp=1, rowsum_a=2.0**-10, rowsum_b=2.0**-24),
    2: dict(max_ulp=1, rowsum_a=2.0**-7, rowsum_b=2.0**-133),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _quant(a64, dt):
    return a64.astype(NUMPY[dt]) if dt != 2 else W._round_to(a64, "bf16")


def _dev(a, off, dt):
    e = ELEM[dt]
    n = a.size
    b = torch.empty(n * e + 64 + off * e, dtype=torch.uint8, device="cuda")
    b[off * e: off * e + n * e].copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).cuda())
    return b, b.data_ptr() + off * e


def run_masked(x, dt, scale, mask=None, causal_q=0, variant=0, offs=(0, 0, 0)):
    rows, cols = x.shape
    e = ELEM[dt]
    n = rows * cols
    xb, xp = _dev(x, offs[0], dt)
    mb, mp, mrows = None, 0, 0
    if mask is not None:
        mb, mp = _dev(mask, offs[1], dt)
        mrows = mask.shape[0]
    yb = torch.full((2 * GUARD + n * e + offs[2] * e,), 0xA5, dtype=torch.uint8, device="cuda")
    yp = yb.data_ptr() + GUARD + offs[2] * e
    rc = osd.softmax_fwd_masked_variant(xp, yp, rows, cols, dt, scale, mp, mrows, causal_q, variant,
                                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = yb.cpu().numpy()
    assert (host[: GUARD + offs[2] * e] == 0xA5).all() and (host[GUARD + offs[2] * e + n * e:] == 0xA5).all()
    y = host[GUARD + offs[2] * e: GUARD + offs[2] * e + n * e].view(NUMPY[dt]).reshape(rows, cols).copy()
    return rc, y


def as_call_scale(scale):
    """The scale the kernel computes with: the C ABI's float argument."""
    return float(np.float32(scale))


def check_masked(x, y, dt, scale, mask=None, causal_q=0, finite_expected=True):
    res = oracle.check_masked(x, y, dt, as_call_scale(scale), mask, causal_q, **TOLM[dt])
    assert res["violations"] == 0, res
    assert res["rowsum_violations"] == 0, res
    if finite_expected:
        assert res["nonfinite"] == 0, res
    return res


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_attention_scores_causal_and_masks(dt):
    # [B=2, H=4, Sq, Sk] scores from the attention workload's distribution
    w = W.WORKLOADS["attn_fp16_65536x512"]
    for sq, sk in ((512, 512), (64, 512), (100, 300)):
        rows = 8 * sq
        x64 = W.generate(w, rows=rows).astype(np.float64)[:, :sk]
        x = _quant(x64, dt)
        rng = np.random.default_rng(sq + sk)
        pad = np.zeros((1, sk))
        pad[0, sk - 37:] = -np.inf
        alibi = _quant(-0.05 * np.abs(np.arange(sk)[None, :] - np.arange(sq)[:, None]), dt)
        for mask, causal in ((None, sq), (_quant(pad, dt), 0), (alibi, sq), (_quant(rng.normal(0, 1, (rows, sk)), dt), 0)):
            for v in (0, osd.VARIANTS["rowgroup"], osd.VARIANTS["block"]):
                rc, y = run_masked(x, dt, 0.125, mask, causal, v)
                if rc == -5:
                    assert v == osd.VARIANTS["rowgroup"]
                    continue
                assert rc == 0, (sq, sk, NAMES[v])
                check_masked(x, y, dt, 0.125, mask, causal)


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_masked_shapes_and_offsets(dt):
    rng = np.random.default_rng(60 + dt)
    for cols in list(range(1, 37)) + [127, 128, 129, 511, 512, 1000, 1023, 1025, 4093, 8192, 16000]:
        rows = 9
        x = _quant(rng.normal(0, 5, (rows, cols)), dt)
        mask = _quant(rng.normal(0, 2, (3, cols)), dt)
        for scale, causal in ((0.7, 0), (80 ** -0.5, 0), (1.0, 3), (-1.5, 0), (2.0, 9), (80 ** -0.5, 5)):
            for offs in ((0, 0, 0), (1, 2, 3)):
                for v in (osd.VARIANTS["rowgroup"], osd.VARIANTS["block"]):
                    rc, y = run_masked(x, dt, scale, mask, causal, v, offs)
                    if rc == -5:
                        continue
                    assert rc == 0, (cols, NAMES[v], offs)
                    check_masked(x, y, dt, scale, mask, causal)


def test_rows_with_no_visible_key_and_specials():
    for dt in (0, 1, 2):
        x = _quant(np.random.default_rng(1).normal(0, 1, (8, 3)), dt)
        rc, y = run_masked(x, dt, 1.0, None, causal_q=4)  # queries 0, 1 of each block see no key
        assert rc == 0
        check_masked(x, y, dt, 1.0, None, 4, finite_expected=False)
        yd = oracle.decode(y, dt)
        assert np.isnan(yd[[0, 4]]).all() and np.isfinite(yd[[2, 3, 6, 7]]).all()


def test_large_logits_keep_one_ulp():
    # |z| up to ~4e4, where one fp32 rounding of z (2^-24 |z| ~ 2e-3) alone
    # would move the 16-bit outputs by several ulps: the logits are carried as
    # an unevaluated pair, so the bound of softmax_fwd still holds
    rng = np.random.default_rng(2)
    for dt in (0, 1, 2):
        x = _quant(rng.normal(0, 200, (64, 700)), dt)
        mask = _quant(rng.normal(0, 300, (5, 700)), dt)
        for scale, m in ((40.0, None), (40.0 + 2.0**-9, None), (80 ** -0.5 * 300, mask), (0.7, mask)):
            for v in (osd.VARIANTS["rowgroup"], osd.VARIANTS["block"]):
                rc, y = run_masked(x, dt, scale, m, 0, v)
                if rc == -5:
                    continue
                assert rc == 0
                check_masked(x, y, dt, scale, m)


def test_max_logit_around_the_pair_threshold():
    # 16-bit rows keep single-float logits while their max logit is below 512
    # in magnitude and form pairs beyond it: rows on both sides of that line,
    # with logits spread over ~100 below the max (every output in range)
    rng = np.random.default_rng(4)
    for dt in (0, 1, 2):
        for centre in (440.0, 506.0, 520.0, -420.0, -506.0, -530.0):
            x64 = rng.uniform(centre - 100.0, centre, (48, 900)) / 0.7
            x = _quant(x64, dt)
            mask = _quant(rng.normal(0, 3, (7, 900)), dt)
            for m in (None, mask):
                for v in (osd.VARIANTS["rowgroup"], osd.VARIANTS["block"]):
                    rc, y = run_masked(x, dt, 0.7, m, 0, v)
                    if rc == -5:
                        continue
                    assert rc == 0
                    check_masked(x, y, dt, 0.7, m)


def test_reduces_to_plain_softmax():
    rng = np.random.default_rng(3)
    for dt in (0, 1, 2):
        x = _quant(rng.normal(0, 4, (33, 777)), dt)
        rc, y = run_masked(x, dt, 1.0)
        assert rc == 0
        ref = oracle.softmax_rounded(x, dt) if dt else None
        if dt:
            assert np.abs(y.view(np.uint16).astype(np.int32) - ref.astype(np.int32)).max() <= 1


def test_torch_api_and_errors():
    x = torch.randn(2, 4, 128, 256, device="cuda", dtype=torch.float16)
    mask = torch.zeros(1, 256, device="cuda", dtype=torch.float16)
    mask[0, -5:] = float("-inf")
    y = osd.softmax_masked(x, scale=0.125, mask=mask, causal=True)
    xn = x.cpu().numpy().reshape(-1, 256)
    check_masked(xn, y.cpu().numpy().reshape(-1, 256), 1, 0.125, mask.cpu().numpy(), 128)
    s = torch.cuda.current_stream().cuda_stream
    xx = torch.randn(4, 64, device="cuda")
    yy = torch.empty_like(xx)
    # a mask that overlaps y is refused; one that overlaps x is fine (both are read only)
    assert osd.softmax_fwd_masked(xx.data_ptr(), yy.data_ptr(), 4, 64, 0, 1.0, yy.data_ptr(), 1, 0, s) == -3
    assert osd.softmax_fwd_masked(xx.data_ptr(), yy.data_ptr(), 4, 64, 0, 1.0, xx.data_ptr(), 4, 0, s) == 0
    assert osd.softmax_fwd_masked(xx.data_ptr(), yy.data_ptr(), 4, 64, 0, 1.0, xx.data_ptr(), 0, 0, s) == -1
    assert osd.softmax_fwd_masked(xx.data_ptr(), yy.data_ptr(), 4, 64, 0, 1.0, 0, 0, -1, s) == -1
    big = torch.randn(2, 20000, device="cuda")
    assert osd.softmax_fwd_masked(big.data_ptr(), torch.empty_like(big).data_ptr(), 2, 20000, 0, 1.0, 0, 0, 0,
                                  s) == -5


# The lean form: 16-bit rows on the 16-byte grid, no additive mask, scale > 0
# (the kernel takes the max on packed x and r mod causal_q by a multiply-high).
LEAN_COLS = (8, 16, 24, 32, 40, 64, 120, 128, 136, 256, 264, 512, 520, 1000, 1024)


@pytest.mark.parametrize("dt", [1, 2])
def test_lean_form_shapes_scales_and_causal_cuts(dt):
    rng = np.random.default_rng(70 + dt)
    for cols in LEAN_COLS:
        rows = 37  # not a multiple of the rows a CTA takes
        x = _quant(rng.normal(0, 5, (rows, cols)), dt)
        for scale in (0.125, 80 ** -0.5, 1.0, 3.0):
            for causal in (0, 1, 3, 7, cols, cols + 5):
                rc, y = run_masked(x, dt, scale, None, causal)
                assert rc == 0, (cols, scale, causal)
                # causal_q > cols leaves the first queries of a block without a key
                check_masked(x, y, dt, scale, None, causal, finite_expected=causal <= cols)
        # the general kernel takes the other scales
        for scale in (-0.5, 0.0):
            rc, y = run_masked(x, dt, scale, None, 3)
            assert rc == 0
            check_masked(x, y, dt, scale, None, 3)


@pytest.mark.parametrize("dt", [1, 2])
def test_lean_form_large_logits_and_the_pair_threshold(dt):
    rng = np.random.default_rng(80 + dt)
    x = _quant(rng.normal(0, 200, (64, 704)), dt)
    for scale in (40.0, 40.0 + 2.0**-9, 80 ** -0.5 * 300):
        rc, y = run_masked(x, dt, scale, None, 64)
        assert rc == 0
        check_masked(x, y, dt, scale, None, 64)
    for centre in (440.0, 506.0, 520.0, -420.0, -506.0, -530.0):
        xc = _quant(rng.uniform(centre - 100.0, centre, (48, 896)) / 0.7, dt)
        for causal in (0, 48):
            rc, y = run_masked(xc, dt, 0.7, None, causal)
            assert rc == 0
            check_masked(xc, y, dt, 0.7, None, causal)


def test_lean_form_in_place_matches_out_of_place():
    for dt, tdt in ((1, torch.float16), (2, torch.bfloat16)):
        x = (torch.randn(4 * 512, 512, device="cuda") * 3).to(tdt)
        y = torch.empty_like(x)
        s = torch.cuda.current_stream().cuda_stream
        assert osd.softmax_fwd_masked(x.data_ptr(), y.data_ptr(), 2048, 512, dt, 0.125, 0, 0, 512, s) == 0
        xi = x.clone()
        assert osd.softmax_fwd_masked(xi.data_ptr(), xi.data_ptr(), 2048, 512, dt, 0.125, 0, 0, 512, s) == 0
        torch.cuda.synchronize()
        assert torch.equal(xi.view(torch.int16), y.view(torch.int16))


def test_lean_form_large_row_indices():
    # 2^21 + 5 rows: the causal cut of rows far from 0 (r mod causal_q by the
    # multiply-high) checked on blocks that start at multiples of causal_q, so
    # that the oracle sees the same query index i = r mod causal_q
    rows, cols, q = (1 << 21) + 5, 64, 1000
    g = torch.Generator(device="cuda").manual_seed(5)
    x = (torch.randn(rows, cols, device="cuda", generator=g) * 4).half()
    y = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert osd.softmax_fwd_masked(x.data_ptr(), y.data_ptr(), rows, cols, 1, 0.125, 0, 0, q, s) == 0
    torch.cuda.synchronize()
    for start in (0, 1000 * q, 2096 * q):
        n = min(2 * q, rows - start)
        xs = x[start:start + n].cpu().numpy()
        ys = y[start:start + n].cpu().numpy()
        check_masked(xs, ys, 1, 0.125, None, q)
