"""The seeded input generators: determinism, the prefix property, and the
distribution each workload promises (they hold no softmax arithmetic)."""
import numpy as np
import pytest

from online_softmax_dispatcher_gb300 import workloads as W


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_deterministic_and_prefix_stable(name):
    w = W.WORKLOADS[name]
    rows = min(w.rows, 40)
    a = W.generate(w, rows=rows)
    b = W.generate(w, rows=rows, threads=1)
    assert a.dtype == W.storage_dtype(w.dtype) and a.shape == (rows, w.cols)
    assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    c = W.generate(w, rows=min(w.rows, 3))
    assert np.array_equal(a[: c.shape[0]].view(np.uint8), c.view(np.uint8))


def _f64(a, dtype):
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def test_attention_spikes():
    w = W.WORKLOADS["attn_fp16_65536x512"]
    x = _f64(W.generate(w, rows=4096), w.dtype)
    frac = np.mean(np.abs(x) == 200.0)
    assert 0.009 < frac < 0.011
    assert abs(np.mean(x[x == 200.0]) - 200) < 1e-9 and 0.45 < np.mean(x[np.abs(x) == 200] > 0) < 0.55
    rest = x[np.abs(x) != 200.0]
    assert abs(rest.std() - 20.0) < 0.2 and abs(rest.mean()) < 0.1


def test_vocab_peak_per_row():
    w = W.WORKLOADS["vocab_bf16_32768x32000"]
    x = _f64(W.generate(w, rows=64), w.dtype)
    assert (x.max(axis=1) == 30.0).all()
    assert abs(x[x != 30.0].std() - 4.0) < 0.05


def test_splitk_large_entries():
    w = W.WORKLOADS["splitk_fp32_4x4194304"]
    x = _f64(W.generate(w, rows=1), w.dtype)
    big = x >= 50.0
    assert 0.049 < big.mean() < 0.051 and x[big].max() <= 100.0


def test_uniform_and_awkward_rows():
    w = W.WORKLOADS["awkward_fp16_8192x5003"]
    x = _f64(W.generate(w, rows=200), w.dtype)
    assert x.min() >= -10 and x.max() <= 10 and abs(x.mean()) < 0.05
    assert (w.cols * w.elem_bytes) % 16 != 0


def test_bytes_moved():
    w = W.WORKLOADS["attn_fp16_65536x512"]
    assert w.bytes_moved() == 65536 * 512 * 4
    assert W.WORKLOADS["splitk_fp32_4x4194304"].bytes_moved(2) == 2 * 4194304 * 8
