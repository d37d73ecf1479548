"""Pins that tie the fp64 oracle to something other than itself.

Each pin is a function of an ``oracle.Oracle`` so that the same pins also run
against deliberately broken builds of the oracle source (``test_mutants_fail``):
every plausible slip there (a flipped sign, a dropped term, a wrong bias, a
tie rounded the wrong way, a swapped row) must trip at least one pin.

What pins what:
* the worked example of the HIP softmax tutorial, section 1, and its printed
  run output, section 8 (tests/golden, values as printed on the page);
* closed forms: cols = 1, constant rows (1/n), the two-element case
  (scipy.special.expit), a single planted peak, and a sum whose small terms
  vanish without compensation;
* invariants: unit row sums, bitwise shift invariance on dyadic grids;
* the chunked online form equals the direct definition;
* scipy.special.softmax on random and brute-force enumerated rows;
* dtype decode against numpy (fp16) and torch (bf16) on all 65536 patterns;
* dtype encode against numpy (fp16, fp32) and against ties built at every
  midpoint between consecutive fp16 / bf16 values;
* the comparison helper against planted errors.
"""
import math
import os
import re
import shutil
import tempfile

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import BF16, F16, F32
from tests.conftest import load_golden

# ----------------------------------------------------------------------------- helpers


def _bf16_bits_from_f32(vals):
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _all_positive_finite(dtype):
    """All positive finite bit patterns of a 16-bit dtype, ascending by value."""
    if dtype == F16:
        return np.arange(0x0000, 0x7C00, dtype=np.uint16)
    return np.arange(0x0000, 0x7F80, dtype=np.uint16)


# ----------------------------------------------------------------------------- pins


def pin_worked_example(o):
    g = load_golden("worked_example.txt")
    d = int(g["decimals"])
    x = np.array(g["x"], dtype=np.float64)
    want = np.array(g["y"])
    for y in (o.softmax_f64(x), o.softmax(x.astype(np.float32)), o.softmax(x.astype(np.float16))):
        assert np.array_equal(np.round(y, d), want), y


def pin_printed_output(o):
    g = load_golden("printed_run_output.txt")
    sig = int(g["significant"])
    y = o.softmax_f64(np.array(g["x"]))
    for got_row, want_row in zip(y, g["y"]):
        for got, want in zip(got_row, want_row):
            assert float(f"{got:.{sig}g}") == want, (got, want)


def pin_cols_one(o):
    x = np.array([[-200.0], [0.0], [3.5], [1e30]])
    assert np.array_equal(o.softmax_f64(x), np.ones_like(x))
    for dt, arr in ((F16, np.array([[7.0]], np.float16)), (F32, np.array([[-3.0]], np.float32))):
        assert o.softmax(arr, dt)[0, 0] == 1.0


def pin_constant_rows(o):
    for n in (1, 2, 3, 7, 1000, 4096):
        for c in (-200.0, 0.0, 1.0, 200.0):
            y = o.softmax_f64(np.full((1, n), c))
            assert np.allclose(y, 1.0 / n, rtol=1e-15, atol=0)


def pin_two_element_logistic(o):
    rng = np.random.default_rng(11)
    a = rng.normal(0, 10, 200)
    b = rng.normal(0, 10, 200)
    y = o.softmax_f64(np.stack([a, b], axis=1))
    assert np.allclose(y[:, 0], scipy.special.expit(a - b), rtol=1e-14, atol=1e-300)
    assert np.allclose(y[:, 1], scipy.special.expit(b - a), rtol=1e-14, atol=1e-300)


def pin_planted_peak(o):
    # zeros everywhere except one entry of +30: y_peak = 1 / (1 + (n - 1) e^-30)
    for n, pos in ((5, 0), (1000, 517), (32000, 31999)):
        x = np.zeros((1, n))
        x[0, pos] = 30.0
        y = o.softmax_f64(x)
        peak = 1.0 / (1.0 + (n - 1) * math.exp(-30.0))
        rest = math.exp(-30.0) * peak
        assert abs(y[0, pos] - peak) <= 1e-15 * peak
        others = np.delete(y[0], pos)
        assert np.allclose(others, rest, rtol=1e-14, atol=0)


def pin_ramp_geometric(o):
    # the HIP softmax tutorial's large-cols run (4 rows of 32768; its printed
    # outputs grow by e^(1/32) from one column to the next, as a ramp
    # x_j = j / 32 gives; input not printed): softmax of an arithmetic ramp is
    # a normalised geometric sequence, y_j = q^(n-1-j) (1 - q) / (1 - q^n),
    # q = e^(-1/32)
    n = 32768
    j = np.arange(n, dtype=np.float64)
    x = np.stack([j / 32.0, j / 32.0 - 100.0, j / 32.0 + 7.25, (n - 1 - j) / 32.0])
    y = o.softmax_f64(x)
    q = math.exp(-1.0 / 32.0)
    want = np.exp((j - (n - 1)) / 32.0) * (1.0 - q) / (1.0 - q ** n)
    # (the first ~9000 columns lie below double's normal range: exact up to
    # the absolute floor there)
    for r in range(3):
        assert np.allclose(y[r], want, rtol=1e-12, atol=1e-300)
    assert np.allclose(y[3], want[::-1], rtol=1e-12, atol=1e-300)
    big = y[0, :-1] > 1e-290
    assert big.sum() > 20000
    ratio = y[0, 1:][big] / y[0, :-1][big]
    assert np.allclose(ratio, math.exp(1.0 / 32.0), rtol=1e-13, atol=0)


def pin_compensated_sum(o):
    # one 0 and N entries of -40: y_0 = 1 / (1 + N e^-40).  N e^-40 ~ 4e-13 is made
    # of terms far below half an ulp of 1, so only a compensated sum keeps it.
    n = 100_000
    x = np.full((1, n + 1), -40.0)
    x[0, 0] = 0.0
    y = o.softmax_f64(x)
    want = 1.0 / (1.0 + n * math.exp(-40.0))
    assert abs(y[0, 0] - want) <= 2e-16, (y[0, 0], want)


def pin_row_sums(o):
    rng = np.random.default_rng(12)
    for dt, arr in ((F32, rng.normal(0, 5, (16, 999)).astype(np.float32)),
                    (F16, rng.normal(0, 20, (16, 512)).astype(np.float16)),
                    (BF16, _bf16_bits_from_f32(rng.normal(0, 4, (16, 3000))))):
        y = o.softmax(arr, dt)
        for row in y:
            assert abs(math.fsum(row) - 1.0) <= 1e-14


def pin_shift_invariance(o):
    # fp16 multiples of 2^-4 with |x| < 32; x + 16 stays exact, so x - max is
    # the same number and y must be bitwise identical.
    rng = np.random.default_rng(13)
    grid = rng.integers(-511, 512, size=(8, 300)) / 16.0
    x = grid.astype(np.float16)
    xs = (grid + 16.0).astype(np.float16)
    assert np.array_equal(xs.astype(np.float64) - 16.0, grid)
    assert np.array_equal(o.softmax(x, F16), o.softmax(xs, F16))
    g32 = rng.integers(-2**20, 2**20, size=(4, 777)) / 1024.0
    assert np.array_equal(o.softmax(g32.astype(np.float32), F32),
                          o.softmax((g32 + 64.0).astype(np.float32), F32))


def pin_online_equals_direct(o):
    rng = np.random.default_rng(14)
    x = rng.normal(0, 30, (5, 1000))
    x[:, 13] = 250.0
    direct = o.softmax_f64(x)
    for chunk in (1, 7, 256, 1000):
        online = o.online_softmax_f64(x, chunk)
        assert np.allclose(online, direct, rtol=1e-14, atol=1e-300), chunk


def pin_scipy_random(o):
    rng = np.random.default_rng(15)
    for scale, cols in ((1.0, 17), (20.0, 512), (200.0, 64), (1000.0, 9)):
        x = rng.normal(0, scale, (32, cols))
        want = scipy.special.softmax(x, axis=1)
        got = o.softmax_f64(x)
        assert np.allclose(got, want, rtol=1e-13, atol=1e-300)


def pin_brute_force_tiny(o):
    # every row of length 1..4 over a fixed value set, in each dtype
    vals = [-200.0, -3.0, -1.0, 0.0, 0.5, 2.0, 3.0, 200.0]
    for n in range(1, 5):
        rows = np.array(np.meshgrid(*([vals] * n), indexing="ij")).reshape(n, -1).T
        want = scipy.special.softmax(rows, axis=1)
        for dt, arr in ((F32, rows.astype(np.float32)), (F16, rows.astype(np.float16)),
                        (BF16, _bf16_bits_from_f32(rows))):
            got = o.softmax(arr, dt)
            assert np.allclose(got, want, rtol=1e-13, atol=1e-300)
        assert np.array_equal(o.encode(want, F16), want.astype(np.float16).view(np.uint16))


def pin_decode_f16_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = o.decode(bits, F16)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def pin_decode_bf16_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = o.decode(bits, BF16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_encode_f16_numpy(o):
    rng = np.random.default_rng(16)
    y = np.concatenate([rng.uniform(0, 1, 20000), rng.uniform(0, 7e4, 2000),
                        np.exp(rng.uniform(-40, 0, 20000)), -rng.uniform(0, 1, 100),
                        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, np.inf, -np.inf]])
    got = o.encode(y, F16)
    with np.errstate(over="ignore"):
        want = y.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def pin_encode_f32_numpy(o):
    rng = np.random.default_rng(17)
    y = np.concatenate([rng.uniform(0, 1, 5000), np.exp(rng.uniform(-110, 0, 5000)),
                        [1e-45, 7e-46, 1.5e-45, 3.4028235677973366e38, 1e39]])
    with np.errstate(over="ignore"):
        want = y.astype(np.float32)
    assert np.array_equal(o.encode(y, F32), want)


def _encode_midpoints(o, dtype):
    pos = _all_positive_finite(dtype)
    v = o.decode(pos, dtype)
    a, b = v[:-1], v[1:]
    abits, bbits = pos[:-1], pos[1:]
    mid = (a + b) / 2.0  # exact in binary64
    even = np.where(abits % 2 == 0, abits, bbits)
    lo = np.nextafter(mid, -np.inf)
    hi = np.nextafter(mid, np.inf)
    assert np.array_equal(o.encode(mid, dtype), even)
    assert np.array_equal(o.encode(lo, dtype), abits)
    assert np.array_equal(o.encode(hi, dtype), bbits)
    assert np.array_equal(o.encode(a, dtype), abits)
    # negatives mirror the positives with the sign bit set
    assert np.array_equal(o.encode(-mid[1:], dtype), even[1:] | 0x8000)
    # top of the range: the midpoint above the largest finite value rounds to inf
    top = v[-1]
    step = top - v[-2]
    inf_bits = 0x7C00 if dtype == F16 else 0x7F80
    assert o.encode(np.array([top + step / 2]), dtype)[0] == inf_bits
    assert o.encode(np.array([np.nextafter(top + step / 2, 0)]), dtype)[0] == pos[-1]


def pin_encode_f16_midpoints(o):
    _encode_midpoints(o, F16)


def pin_encode_bf16_midpoints(o):
    _encode_midpoints(o, BF16)


def pin_nonfinite(o):
    x = np.array([[0.0, np.nan, 1.0], [0.0, np.inf, 1.0], [-np.inf, -np.inf, -np.inf],
                  [-np.inf, 0.0, 0.0]])
    y = o.softmax_f64(x)
    assert np.isnan(y[0]).all() and np.isnan(y[1]).all() and np.isnan(y[2]).all()
    assert np.array_equal(y[3], [0.0, 0.5, 0.5])


def pin_check_helper(o):
    rng = np.random.default_rng(18)
    x = rng.normal(0, 3, (6, 40)).astype(np.float16)
    ref = o.softmax_rounded(x, F16)
    res = o.check(x, ref, F16, max_ulp=0, rowsum_a=2**-10, rowsum_b=2**-24)
    assert res["violations"] == 0 and res["checked"] == x.size and res["rowsum_violations"] == 0
    bad = ref.copy()
    bad[3, 7] += 1
    assert o.check(x, bad, F16, max_ulp=1)["violations"] == 0
    r0 = o.check(x, bad, F16, max_ulp=0)
    assert r0["violations"] == 1 and r0["first_bad"] == 3 * 40 + 7 and r0["max_ulp"] == 1
    bad[1, 2] += 2
    assert o.check(x, bad, F16, max_ulp=1)["first_bad"] == 1 * 40 + 2
    x32 = rng.normal(0, 3, (3, 50)).astype(np.float32)
    y32 = o.softmax(x32, F32).astype(np.float32)
    assert o.check(x32, y32, F32, rel_tol=2e-6, abs_floor=2**-126)["violations"] == 0
    y32[2, 5] *= 1 + 1e-5
    r = o.check(x32, y32, F32, rel_tol=2e-6, abs_floor=2**-126)
    assert r["violations"] == 1 and r["first_bad"] == 2 * 50 + 5
    sel = o.check(x32, y32, F32, rel_tol=2e-6, abs_floor=2**-126, rows_sel=np.array([0, 1]))
    assert sel["violations"] == 0 and sel["checked"] == 100


def pin_bwd_finite_difference(o):
    # dx_i = d/dx_i sum_j softmax(x)_j dy_j, by central differences of the
    # (separately pinned) forward definition
    rng = np.random.default_rng(19)
    x = rng.normal(0, 2, (3, 9))
    dy = rng.normal(0, 1, (3, 9))
    dx = o.softmax_bwd_f64(o.softmax_f64(x), dy)
    h = 1e-6
    for r in range(3):
        for i in range(9):
            xp, xm = x[r].copy(), x[r].copy()
            xp[i] += h
            xm[i] -= h
            fd = (o.softmax_f64(xp[None]) @ dy[r] - o.softmax_f64(xm[None]) @ dy[r]) / (2 * h)
            assert abs(fd[0] - dx[r, i]) <= 1e-8, (r, i, fd, dx[r, i])


def pin_bwd_closed_forms(o):
    rng = np.random.default_rng(20)
    x = rng.normal(0, 3, (50, 2))
    dy = rng.normal(0, 1, (50, 2))
    y = o.softmax_f64(x)
    dx = o.softmax_bwd_f64(y, dy)
    want0 = y[:, 0] * y[:, 1] * (dy[:, 0] - dy[:, 1])
    # dy_0 - s cancels when y_1 is small: the error budget is absolute in y |dy|
    tol = 8 * 2.0**-52 * y[:, 0] * (np.abs(dy).sum(axis=1))
    assert (np.abs(dx[:, 0] - want0) <= tol).all()
    assert (np.abs(dx[:, 1] + want0) <= 8 * 2.0**-52 * y[:, 1] * np.abs(dy).sum(axis=1)).all()
    # a constant upstream gradient has zero gradient; every row of dx sums to 0
    y = o.softmax_f64(rng.normal(0, 5, (8, 300)))
    assert np.abs(o.softmax_bwd_f64(y, np.full_like(y, 3.5))).max() <= 1e-14
    dx = o.softmax_bwd_f64(y, rng.normal(0, 1, y.shape))
    assert np.abs(dx.sum(axis=1)).max() <= 1e-14


def pin_bwd_compensated_sum(o):
    # one dominant entry and 1e5 entries of e^-40 relative to it, dy = 1: the
    # exact gradient is 0, and s = sum dy*y = 1 only if the tiny terms are kept
    n = 100_000
    x = np.full((1, n + 1), -40.0)
    x[0, 0] = 0.0
    y = o.softmax_f64(x)
    dx = o.softmax_bwd_f64(y, np.ones_like(y))
    assert np.abs(dx).max() <= 1e-15, np.abs(dx).max()


def pin_bwd_check_helper(o):
    rng = np.random.default_rng(22)
    y16 = o.softmax_rounded(rng.normal(0, 2, (4, 64)).astype(np.float16), F16)
    dy16 = rng.normal(0, 1, (4, 64)).astype(np.float16).view(np.uint16)
    want = o.softmax_bwd_f64(o.decode(y16, F16), o.decode(dy16, F16))
    dx16 = o.encode(want, F16)
    assert o.check_bwd(y16, dy16, dx16, F16, max_ulp=1, k_eps=4)["violations"] == 0
    bad = dx16.copy()
    j = int(np.argmax(np.abs(want[2])))
    bad[2, j] ^= 0x0004  # 4 ulp away at the largest |dx|
    r = o.check_bwd(y16, dy16, bad, F16, max_ulp=1, k_eps=4)
    assert r["violations"] == 1 and r["first_bad"] == 2 * 64 + j


def pin_masked_reduces_to_plain(o):
    rng = np.random.default_rng(30)
    for dt, x in ((F32, rng.normal(0, 3, (6, 77)).astype(np.float32)),
                  (F16, rng.normal(0, 3, (6, 77)).astype(np.float16)),
                  (BF16, _bf16_bits_from_f32(rng.normal(0, 3, (6, 77))))):
        assert np.array_equal(o.softmax_masked(x, dt, 1.0), o.softmax(x, dt))


def pin_masked_scale_and_mask(o):
    # scale by a power of two and an additive mask are exact in binary64, so the
    # masked form must equal the plain definition on the transformed rows
    rng = np.random.default_rng(31)
    x = rng.normal(0, 10, (7, 50)).astype(np.float16)
    mask = rng.normal(0, 4, (3, 50)).astype(np.float16)
    got = o.softmax_masked(x, F16, 0.125, mask)
    z = 0.125 * x.astype(np.float64) + mask.astype(np.float64)[np.arange(7) % 3]
    assert np.allclose(got, scipy.special.softmax(z, axis=1), rtol=1e-14, atol=1e-300)
    assert np.array_equal(got, o.softmax_f64(z))


def pin_masked_causal_closed_form(o):
    # zero logits: row i of a causal block sees i + 1 + (cols - q) keys, each 1/(that)
    for q, cols in ((8, 8), (5, 12)):
        x = np.zeros((2 * q, cols), dtype=np.float32)
        y = o.softmax_masked(x, F32, 1.0, causal_q=q)
        for r in range(2 * q):
            vis = r % q + 1 + (cols - q)
            assert np.allclose(y[r, :vis], 1.0 / vis, rtol=1e-15, atol=0)
            assert (y[r, vis:] == 0).all()
    # more queries than keys: the first rows see nothing -> NaN (definition of an all -inf row)
    y = o.softmax_masked(np.zeros((4, 2), dtype=np.float32), F32, 1.0, causal_q=4)
    assert np.isnan(y[:2]).all() and np.allclose(y[2], [1.0, 0.0]) and np.allclose(y[3], [0.5, 0.5])


def pin_masked_check_helper(o):
    rng = np.random.default_rng(32)
    x = rng.normal(0, 8, (6, 40)).astype(np.float16)
    mask = rng.normal(0, 2, (1, 40)).astype(np.float16)
    want = o.encode(o.softmax_masked(x, F16, 0.25, mask, causal_q=3), F16)
    kw = dict(max_ulp=1, rowsum_a=2**-10, rowsum_b=2**-24)
    assert o.check_masked(x, want, F16, 0.25, mask, 3, **kw)["violations"] == 0
    bad = want.copy()
    bad[4, 1] += 3
    r = o.check_masked(x, bad, F16, 0.25, mask, 3, **kw)
    assert r["violations"] == 1 and r["first_bad"] == 4 * 40 + 1
    # the logit allowance admits a relative error up to zrel * max|z|
    bad = want.copy()
    bad[0, 0] += 3
    exact = o.softmax_masked(x, F16, 0.25, mask, causal_q=3)[0, 0]
    rel = abs(o.decode(bad, F16)[0, 0] / exact - 1)
    zmax = np.abs(0.25 * x[0].astype(np.float64) + mask[0].astype(np.float64))[:1 + 40 - 3].max()
    assert o.check_masked(x, bad, F16, 0.25, mask, 3, zrel=1.01 * rel / zmax, **kw)["violations"] == 0


# ----------------------------------------------------------------------------- LayerNorm / RMSNorm


def _norm_inputs(rng, rows, cols, dt, loc=0.0, scale=1.0):
    v = rng.normal(loc, scale, (rows, cols))
    if dt == F32:
        return v.astype(np.float32)
    if dt == F16:
        return v.astype(np.float16)
    return _bf16_bits_from_f32(v.astype(np.float32)).reshape(rows, cols)


def pin_norm_torch_layer_norm(o):
    # torch's float64 layer_norm (its own implementation) on the decoded values
    rng = np.random.default_rng(30)
    for dt in (F32, F16, BF16):
        for eps in (1e-5, 1e-2):
            x = _norm_inputs(rng, 7, 33, dt, loc=3.0, scale=2.0)
            g = _norm_inputs(rng, 1, 33, dt, loc=1.0, scale=0.5)[0]
            b = _norm_inputs(rng, 1, 33, dt)[0]
            y, mean, rstd = o.norm_f64(oracle.LAYERNORM, x, dt, g, b, eps)
            xd, gd, bd = (torch.from_numpy(o.decode(v, dt)) for v in (x, g, b))
            ref = torch.nn.functional.layer_norm(xd, (33,), gd, bd, eps).numpy()
            assert np.abs(y - ref).max() <= 1e-12, (dt, eps)
            var, mu = torch.var_mean(xd, dim=1, unbiased=False)
            assert np.abs(mean - mu.numpy()).max() <= 1e-13
            assert np.abs(rstd - 1 / np.sqrt(var.numpy() + eps)).max() <= 1e-12 * rstd.max()


def pin_norm_torch_rms_norm(o):
    rng = np.random.default_rng(31)
    for dt in (F32, F16, BF16):
        x = _norm_inputs(rng, 5, 40, dt, loc=0.5, scale=3.0)
        g = _norm_inputs(rng, 1, 40, dt, loc=1.0, scale=0.5)[0]
        y, _, rstd = o.norm_f64(oracle.RMSNORM, x, dt, g, None, 1e-6)
        xd, gd = torch.from_numpy(o.decode(x, dt)), torch.from_numpy(o.decode(g, dt))
        ref = torch.nn.functional.rms_norm(xd, (40,), gd, 1e-6).numpy()
        assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max(), dt
        assert np.abs(rstd - 1 / np.sqrt((xd.numpy() ** 2).mean(1) + 1e-6)).max() <= 1e-12 * rstd.max()
        # a bias is ignored by RMSNorm
        y2, _, _ = o.norm_f64(oracle.RMSNORM, x, dt, g, g, 1e-6)
        assert (y2 == y).all()


def pin_norm_two_elements(o):
    # x = [a, b]: mu = (a + b) / 2, var = d^2 with d = (a - b) / 2, so
    # y = (d, -d) / sqrt(d^2 + eps)
    rng = np.random.default_rng(32)
    ab = rng.normal(0, 4, (64, 2)).astype(np.float32)
    for eps in (0.0, 0.25):
        y, _, _ = o.norm_f64(oracle.LAYERNORM, ab, F32, None, None, eps)
        a, b = ab[:, 0].astype(np.float64), ab[:, 1].astype(np.float64)
        d = (a - b) / 2
        want = d / np.sqrt(d * d + eps)
        assert np.abs(y[:, 0] - want).max() <= 1e-15 and np.abs(y[:, 1] + want).max() <= 1e-15


def pin_norm_brute_force_tiny(o):
    # every row of length 1..3 over a small value set against exact rational
    # statistics (fractions), rounded once at the square root
    from fractions import Fraction
    vals = [-3.0, -0.5, 0.0, 0.25, 1.0, 6.0]
    eps = Fraction(1, 64)
    for n in (1, 2, 3):
        rows = np.array(np.meshgrid(*([vals] * n), indexing="ij")).reshape(n, -1).T.astype(np.float32)
        for kind in (oracle.LAYERNORM, oracle.RMSNORM):
            y, _, _ = o.norm_f64(kind, rows, F32, None, None, float(eps))
            for r, row in enumerate(rows):
                fr = [Fraction(float(v)) for v in row]
                mu = sum(fr) / n if kind == oracle.LAYERNORM else Fraction(0)
                var = sum((v - mu) ** 2 for v in fr) / n
                rs = 1 / math.sqrt(var + eps)
                want = [float(v - mu) * rs for v in fr]
                assert np.abs(y[r] - want).max() <= 1e-15 * (1 + np.abs(want).max()), (kind, row)


def pin_norm_dyadic_invariances(o):
    # on dyadic grids with a power-of-two row length (the mean is then exact)
    # these hold bit for bit: LayerNorm(x + c) == LayerNorm(x), and
    # norm(2^k x, 4^k eps) == norm(x, eps) for both kinds
    rng = np.random.default_rng(33)
    x = (np.round(rng.normal(0, 8, (6, 128)) * 16) / 16).astype(np.float32)
    y0, _, _ = o.norm_f64(oracle.LAYERNORM, x, F32, None, None, 0.5)
    y1, _, _ = o.norm_f64(oracle.LAYERNORM, (x + 32).astype(np.float32), F32, None, None, 0.5)
    assert (y0 == y1).all()
    for kind in (oracle.LAYERNORM, oracle.RMSNORM):
        a, _, ra = o.norm_f64(kind, x, F32, None, None, 0.5)
        b, _, rb = o.norm_f64(kind, (x * 8).astype(np.float32), F32, None, None, 0.5 * 64)
        assert (a == b).all() and (ra == rb * 8).all()


def pin_norm_moments(o):
    # the standardised row has mean 0 and mean square var / (var + eps);
    # RMSNorm's has mean square ms / (ms + eps) (moments by math.fsum)
    rng = np.random.default_rng(34)
    x = rng.normal(5, 3, (4, 1000)).astype(np.float32)
    xd = x.astype(np.float64)
    for kind in (oracle.LAYERNORM, oracle.RMSNORM):
        y, mean, rstd = o.norm_f64(kind, x, F32, None, None, 1e-3)
        for r in range(4):
            mu = math.fsum(xd[r]) / 1000 if kind == oracle.LAYERNORM else 0.0
            var = math.fsum((xd[r] - mu) ** 2) / 1000
            rs = 1 / math.sqrt(var + 1e-3)
            want_mean = 0.0 if kind == oracle.LAYERNORM else math.fsum(xd[r]) / 1000 * rs
            assert abs(math.fsum(y[r]) / 1000 - want_mean) <= 1e-12
            assert abs(math.fsum(y[r] ** 2) / 1000 - var / (var + 1e-3)) <= 1e-12
            assert abs(mean[r] - mu) <= 1e-12 and abs(rstd[r] - 1 / math.sqrt(var + 1e-3)) <= 1e-12


def pin_norm_affine_columns(o):
    # gain and bias act per column: y(g, b)_j == z_j * g_j + b_j
    rng = np.random.default_rng(35)
    x = rng.normal(0, 2, (3, 17)).astype(np.float32)
    g = np.linspace(-2, 3, 17).astype(np.float32)
    b = np.arange(17, dtype=np.float32) * 0.25
    z, _, _ = o.norm_f64(oracle.LAYERNORM, x, F32, None, None, 1e-5)
    y, _, _ = o.norm_f64(oracle.LAYERNORM, x, F32, g, b, 1e-5)
    assert (y == z * g.astype(np.float64) + b.astype(np.float64)).all()
    zr, _, _ = o.norm_f64(oracle.RMSNORM, x, F32, None, None, 1e-5)
    yr, _, _ = o.norm_f64(oracle.RMSNORM, x, F32, g, None, 1e-5)
    assert (yr == zr * g.astype(np.float64)).all()


def pin_norm_check_helper(o):
    # the checker's budget: an element at x_j == mu (z = 0) may be off by
    # about k 2^-24 a rstd (the fp32 error of the mean), not by twice that
    x = np.array([[-3.0, 0.0, 3.0, -1.0, 1.0]], dtype=np.float32)
    y, mean, rstd = o.norm_f64(oracle.LAYERNORM, x, F32, None, None, 0.0)
    a = np.abs(x.astype(np.float64)).mean()
    bound = 64 * 2.0**-24 * a * rstd[0]
    for f, want in ((0.5, 0), (2.0, 1)):
        cand = y.astype(np.float32)
        cand[0, 1] = np.float32(f * bound)
        r = o.check_norm(oracle.LAYERNORM, x, cand, F32, eps=0.0, k_eps=64)
        assert r["violations"] == want and (want == 0 or r["first_bad"] == 1), (f, r)
    # fp16 outputs: one ulp passes, two fail, at the right element
    x16 = np.random.default_rng(36).normal(0, 1, (2, 50)).astype(np.float16)
    want16 = o.encode(o.norm_f64(oracle.RMSNORM, x16, F16)[0], F16)
    for d, nbad in ((1, 0), (2, 1)):
        cand = want16.copy()
        cand[1, 7] = cand[1, 7] + d if cand[1, 7] & 0x7FFF else cand[1, 7]
        r = o.check_norm(oracle.RMSNORM, x16, cand.view(np.float16), F16, max_ulp=1)
        assert r["violations"] == nbad and (nbad == 0 or r["first_bad"] == 57), (d, r)
    # statistics: planted errors in mean and rstd are counted per row
    _, m, s = o.norm_f64(oracle.LAYERNORM, x16, F16)
    mf, sf = m.astype(np.float32), s.astype(np.float32)
    assert o.check_norm(oracle.LAYERNORM, x16, o.encode(o.norm_f64(oracle.LAYERNORM, x16, F16)[0], F16).view(np.float16),
                        F16, mean=mf, rstd=sf, max_ulp=1, k_eps=64)["rowsum_violations"] == 0
    sf[1] *= 1.001
    assert o.check_norm(oracle.LAYERNORM, x16, o.encode(o.norm_f64(oracle.LAYERNORM, x16, F16)[0], F16).view(np.float16),
                        F16, mean=mf, rstd=sf, max_ulp=1, k_eps=64)["rowsum_violations"] == 1


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


# ----------------------------------------------------------------------------- mutants

# (name, text in softmax_oracle.c, replacement).  Each is a plausible slip.
MUTANTS = [
    ("exp_sign_flipped", "yr[j] = exp(xr[j] - m) / s;", "yr[j] = exp(m - xr[j]) / s;"),
    ("sum_drops_last_term", "static double row_expsum(const double *xr, int64_t cols, double m)\n{\n"
     "    double s = 0.0, c = 0.0;\n    for (int64_t j = 0; j < cols; j++)",
     "static double row_expsum(const double *xr, int64_t cols, double m)\n{\n"
     "    double s = 0.0, c = 0.0;\n    for (int64_t j = 0; j < cols - 1; j++)"),
    ("max_skips_first", "    double m = -INFINITY;\n    for (int64_t j = 0; j < cols; j++) {\n"
     "        if (isnan(xr[j]))", "    double m = -INFINITY;\n    for (int64_t j = 1; j < cols; j++) {\n"
     "        if (isnan(xr[j]))"),
    ("compensation_sign", "        double t = exp(xr[j] - m);\n        double u = s + t;\n        if (fabs(s) >= fabs(t))\n"
     "            c += (s - u) + t;", "        double t = exp(xr[j] - m);\n        double u = s + t;\n"
     "        if (fabs(s) >= fabs(t))\n            c -= (s - u) + t;"),
    ("no_compensation", "    return s + c;\n}\n\n/* One row", "    return s;\n}\n\n/* One row"),
    ("ties_away", "(frac == 0.5 && fmod(r, 2.0) != 0.0)", "(frac == 0.5)"),
    ("f16_bias", "e - 25); /* (1 + f/1024)", "e - 24); /* (1 + f/1024)"),
    ("bf16_shift", "((uint32_t)b) << 16;", "((uint32_t)b) << 15;"),
    ("online_no_rescale", "d = d * scale + d_local;", "d = d + d_local;"),
    ("overflow_threshold", "if (isinf(a) || a >= ovf)", "if (isinf(a) || a > maxf)"),
    ("row_swapped", "softmax_row(x + r * cols, cols, y + r * cols);",
     "softmax_row(x + r * cols, cols, y + (rows - 1 - r) * cols);"),
    ("check_off_by_one", "bad = dist > t->max_ulp && ", "bad = dist > t->max_ulp + 1 && "),
    ("subnormal_quantum", "q = ldexp(1.0, min_exp - fbits); /* subnormal quantum */",
     "q = ldexp(1.0, min_exp - fbits + 1); /* subnormal quantum */"),
    ("bwd_sign", "dxr[j] = yr[j] * (dyr[j] - s);", "dxr[j] = yr[j] * (dyr[j] + s);"),
    ("causal_off_by_one", "limit = r % causal_q + (cols - causal_q) + 1;", "limit = r % causal_q + (cols - causal_q);"),
    ("mask_row_index", "v += decode_at(mask, dtype, (r % mask_rows) * cols + j);",
     "v += decode_at(mask, dtype, (r % mask_rows) * cols + (cols - 1 - j));"),
    ("scale_ignored", "double v = scale * decode_at(x, dtype, r * cols + j);",
     "double v = decode_at(x, dtype, r * cols + j);"),
    ("bwd_missing_y", "double t = dyr[j] * yr[j];", "double t = dyr[j];"),
    ("norm_unbiased_variance", "const double var = (q + cq) / (double)n;",
     "const double var = (q + cq) / (double)(n > 1 ? n - 1 : 1);"),
    ("norm_eps_outside_sqrt", "const double rstd = 1.0 / sqrt(var + eps);", "const double rstd = 1.0 / (sqrt(var) + eps);"),
    ("norm_no_sqrt", "const double rstd = 1.0 / sqrt(var + eps);", "const double rstd = 1.0 / (var + eps);"),
    ("norm_bias_dropped", "            v += b[j];", "            v += 0.0 * b[j];"),
    ("norm_gain_column", "            v *= g[j];", "            v *= g[n - 1 - j];"),
    ("norm_rms_centred", "const double mu = kind == ORACLE_LAYERNORM ? (s + c) / (double)n : 0.0;",
     "const double mu = (s + c) / (double)n;"),
    ("norm_mean_count", "const double mu = kind == ORACLE_LAYERNORM ? (s + c) / (double)n : 0.0;",
     "const double mu = kind == ORACLE_LAYERNORM ? (s + c) / (double)(n + 1) : 0.0;"),
    ("norm_check_drops_mean_error", "u * (gj * (fabs(z) + shift) + bj);", "u * (gj * fabs(z) + bj);"),
    ("norm_check_ignores_rstd", "sbad |= !(fabs((double)rstd[r] - rs) <= u * rs);", "sbad |= 0;"),
    ("bwd_drops_compensation", "    s += c;\n    for (int64_t j = 0; j < cols; j++)\n        dxr[j]",
     "    for (int64_t j = 0; j < cols; j++)\n        dxr[j]"),
]


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutants_fail(mutant_dir, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique / missing"
    path = os.path.join(mutant_dir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.build(force=True, src=path, out=os.path.join(mutant_dir, f"lib{name}.so"))
    o = oracle.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


def test_mutation_anchors_are_code():
    # keep the anchors honest: none of them may sit inside a comment
    src = open(oracle.SOURCE).read()
    no_comments = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for name, old, _ in MUTANTS:
        first = old.splitlines()[0].split("/*")[0].strip()
        assert first in no_comments, name
