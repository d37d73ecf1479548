"""Host logic of bench.py for the masked softmax, on CPU: the bytes the method
must move (visible part of x, all of y, the --mask bias once), the bias's
definition, and that the oracle legs count what the GPU line counts."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from online_softmax_dispatcher_gb300 import workloads as W  # noqa: E402


def test_visible_elements_closed_forms():
    # one block of q queries over q keys: row i sees i + 1 keys
    for q in (1, 2, 7, 512):
        assert bench.masked_visible_elems(q, q, q) == q * (q + 1) // 2
        # whole blocks add up, a partial block adds its first rows
        assert bench.masked_visible_elems(3 * q, q, q) == 3 * q * (q + 1) // 2
        assert bench.masked_visible_elems(q + 1, q, q) == q * (q + 1) // 2 + 1
    # keys before the block: row i sees (cols - q) + i + 1
    assert bench.masked_visible_elems(4, 10, 4) == sum(6 + i + 1 for i in range(4))
    # more queries than keys: the first rows see none
    assert bench.masked_visible_elems(5, 3, 5) == sum(max(0, i - 2 + 1) for i in range(5))
    # no causal cut: every element
    assert bench.masked_visible_elems(7, 9, 0) == 63


def test_alibi_mask_definition():
    m = bench.alibi_mask(4, 10)
    assert m.shape == (4, 10)
    for i in range(4):
        pos = 10 - 4 + i  # the query's own key
        assert m[i, pos] == 0.0
        assert m[i, 0] == pytest.approx(-0.05 * pos)
        assert np.all(m[i] <= 0.0)


@pytest.mark.parametrize("mask", [False, True])
def test_oracle_leg_counts_the_gpu_lines_bytes(mask):
    w = W.WORKLOADS["attn_fp16_65536x512"]
    rows = 1024
    _, nbytes, _ = bench.oracle_pass(w, "masked", rows, mask)
    q = min(512, w.rows)
    want = (bench.masked_visible_elems(rows, w.cols, q) + rows * w.cols) * 2
    if mask:
        want += q * w.cols * 2
    assert nbytes == want


def test_mask_needs_the_masked_op():
    p = subprocess.run([sys.executable, "bench.py", "--op", "forward", "--mask"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert p.returncode == 2 and "--mask applies to --op masked" in p.stderr


def test_reference_arm_masked_with_mask():
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--op", "masked", "--mask", "--steps",
                        "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"]["op"] == "masked"
    assert line["config"]["mask"].startswith("ALiBi-style")
    assert line["value"] > 0
