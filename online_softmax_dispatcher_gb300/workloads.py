"""Seeded synthetic inputs shaped like the workloads the softmax pages discuss.

This module draws numbers and rounds them to the storage dtype; it holds no
softmax arithmetic.  Tests, the oracle checks and the benchmark all take their
inputs from here, so both sides of every comparison see the same values.

Recipe (every workload): values are drawn as binary64 by numpy's PCG64, in
blocks of consecutive rows (about 2^22 elements per block); block b of a
workload with seed s uses ``PCG64(SeedSequence([s, b]))``, so the first R rows
of a workload do not depend on how many rows are generated, and blocks can be
drawn in parallel.  The binary64 values are then rounded to the dtype:
fp32 and fp16 with numpy's round-to-nearest-even casts, bf16 by rounding to
fp32 (RNE) and then to bf16 (RNE on the fp32 bit pattern).

Workloads (rows x cols, dtype, distribution):

* fp32_128x1000         fp32, N(0, 1); seed 1.  Small rows, launch-bound.
* attn_fp16_65536x512   fp16, N(0, 20^2), then each entry independently with
                        probability 1% replaced by +200 or -200 (sign a fair
                        coin); seed 2.  The attention-score softmax of
                        [4, 32, 512, 512] ("Softmax on DCU"), flattened.
* awkward_fp16_8192x5003 fp16, U[-10, 10]; seed 3.  Rows of 10006 bytes: every
                        row start but the first is off the 16-byte grid.
* vocab_bf16_32768x32000 bf16, N(0, 4^2), then one entry per row at a column
                        drawn uniformly from [0, cols) set to +30; seed 4.
* splitk_fp32_4x4194304 fp32, N(0, 1), then each entry independently with
                        probability 5% replaced by U[50, 100]; seed 5.
* splitk_fp16_4x4194304 fp16, as above; seed 6.

Normalisation workloads (NORM_WORKLOADS; LayerNorm / RMSNorm of each row):

* ln_fp16_131040x192    fp16, row r drawn N(mu_r, s_r^2) with mu_r ~ U[-2, 2] and
                        s_r ~ U[0.5, 4] per row (activations whose level and
                        spread vary by token); seed 7.  LayerNorm without gain
                        or bias: the [1, 131040, 192] shape of the
                        Pangu-Weather profile, section 3.
* ln_fp16_32760x384     fp16, as above; seed 8.  Its [1, 32760, 384] shape.
* rms_bf16_16384x4096   bf16, as above; seed 9.  RMSNorm with a gain vector
                        drawn N(1, 0.1^2) (seed 109): a transformer-sized
                        hidden dimension (not a shape from the pages).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass

import numpy as np

DTYPE_CODES = {"fp32": 0, "fp16": 1, "bf16": 2}
ELEM_BYTES = {"fp32": 4, "fp16": 2, "bf16": 2}
BLOCK_ELEMS = 1 << 22


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    cols: int
    dtype: str
    dist: str
    seed: int
    about: str

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    def bytes_moved(self, rows: int | None = None) -> int:
        """Algorithmic bytes of one softmax pass: every element read once and written once."""
        r = self.rows if rows is None else rows
        return 2 * r * self.cols * self.elem_bytes


WORKLOADS = {w.name: w for w in [
    Workload("fp32_128x1000", 128, 1000, "fp32", "normal1", 1,
             "fp32 [128, 1000], N(0, 1)"),
    Workload("attn_fp16_65536x512", 65536, 512, "fp16", "attn", 2,
             "attention scores [4, 32, 512, 512] as [65536, 512] fp16, N(0, 20^2) + 1% at +-200"),
    Workload("awkward_fp16_8192x5003", 8192, 5003, "fp16", "uniform10", 3,
             "fp16 [8192, 5003], U[-10, 10], rows off the 16-byte grid"),
    Workload("vocab_bf16_32768x32000", 32768, 32000, "bf16", "vocab", 4,
             "vocabulary-sized bf16 [32768, 32000], N(0, 4^2) + one +30 peak per row"),
    Workload("splitk_fp32_4x4194304", 4, 4194304, "fp32", "splitk", 5,
             "few huge rows fp32 [4, 4194304], N(0, 1) + 5% in U[50, 100]"),
    Workload("splitk_fp16_4x4194304", 4, 4194304, "fp16", "splitk", 6,
             "few huge rows fp16 [4, 4194304], N(0, 1) + 5% in U[50, 100]"),
]}


@dataclass(frozen=True)
class NormWorkload(Workload):
    kind: int = 0        # 0 LayerNorm, 1 RMSNorm
    affine: bool = False  # gain (and, for LayerNorm, bias) vectors
    eps: float = 1e-5


NORM_WORKLOADS = {w.name: w for w in [
    NormWorkload("ln_fp16_131040x192", 131040, 192, "fp16", "resid", 7,
                 "LayerNorm fp16 [131040, 192] (no gain / bias), rows N(U[-2, 2], U[0.5, 4]^2)", 0, False, 1e-5),
    NormWorkload("ln_fp16_32760x384", 32760, 384, "fp16", "resid", 8,
                 "LayerNorm fp16 [32760, 384] (no gain / bias), rows N(U[-2, 2], U[0.5, 4]^2)", 0, False, 1e-5),
    NormWorkload("rms_bf16_16384x4096", 16384, 4096, "bf16", "resid", 9,
                 "RMSNorm bf16 [16384, 4096] with gain N(1, 0.1^2), rows N(U[-2, 2], U[0.5, 4]^2)", 1, True, 1e-6),
]}


def norm_params(w: NormWorkload):
    """(gain, bias) vectors of a normalisation workload in storage dtype, or
    None where it has none."""
    if not w.affine:
        return None, None
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed + 100])))
    g = _round_to(rng.normal(1.0, 0.1, w.cols), w.dtype)
    b = _round_to(rng.normal(0.0, 0.1, w.cols), w.dtype) if w.kind == 0 else None
    return g, b


def rows_per_block(cols: int) -> int:
    return max(1, BLOCK_ELEMS // max(1, cols))


def _draw_block(dist: str, rng: np.random.Generator, nrows: int, cols: int) -> np.ndarray:
    n = nrows * cols
    if dist == "normal1":
        return rng.standard_normal(n).reshape(nrows, cols)
    if dist == "attn":
        v = rng.standard_normal(n) * 20.0
        hit = rng.random(n) < 0.01
        sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
        v[hit] = 200.0 * sign[hit]
        return v.reshape(nrows, cols)
    if dist == "uniform10":
        return rng.uniform(-10.0, 10.0, n).reshape(nrows, cols)
    if dist == "vocab":
        v = (rng.standard_normal(n) * 4.0).reshape(nrows, cols)
        peak = rng.integers(0, cols, size=nrows)
        v[np.arange(nrows), peak] = 30.0
        return v
    if dist == "resid":
        mu = rng.uniform(-2.0, 2.0, (nrows, 1))
        sd = rng.uniform(0.5, 4.0, (nrows, 1))
        return mu + sd * rng.standard_normal(n).reshape(nrows, cols)
    if dist == "splitk":
        v = rng.standard_normal(n)
        hit = rng.random(n) < 0.05
        v[hit] = rng.uniform(50.0, 100.0, int(hit.sum()))
        return v.reshape(nrows, cols)
    raise ValueError(f"unknown distribution {dist}")


def _round_to(v: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "fp32":
        return v.astype(np.float32)
    if dtype == "fp16":
        return v.astype(np.float16)
    if dtype == "bf16":
        u = v.astype(np.float32).view(np.uint32)
        # round-to-nearest-even on the low 16 bits (inputs here are finite)
        u = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
        return u.astype(np.uint16)
    raise ValueError(dtype)


def storage_dtype(dtype: str):
    return {"fp32": np.float32, "fp16": np.float16, "bf16": np.uint16}[dtype]


def generate(w: Workload | str, rows: int | None = None, threads: int | None = None) -> np.ndarray:
    """The first `rows` rows (default: all) of workload `w`, in storage dtype
    (numpy float32 / float16; bf16 as uint16 bit patterns)."""
    if isinstance(w, str):
        w = WORKLOADS[w] if w in WORKLOADS else NORM_WORKLOADS[w]
    rows = w.rows if rows is None else rows
    out = np.empty((rows, w.cols), dtype=storage_dtype(w.dtype))
    rpb = rows_per_block(w.cols)
    blocks = [(b, b * rpb, min(rows, (b + 1) * rpb)) for b in range((rows + rpb - 1) // rpb)]

    def work(item):
        b, r0, r1 = item
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, b])))
        # a block is always drawn whole, so a prefix matches the full workload
        full = _draw_block(w.dist, rng, rpb, w.cols)
        out[r0:r1] = _round_to(full[: r1 - r0], w.dtype)

    n = threads or min(len(blocks), os.cpu_count() or 1)
    if n <= 1:
        for item in blocks:
            work(item)
    else:
        with cf.ThreadPoolExecutor(max_workers=n) as ex:
            list(ex.map(work, blocks))
    return out


def as_torch(a: np.ndarray, dtype: str):
    """A CPU torch tensor over the same storage (bf16 bit patterns viewed as bfloat16)."""
    import torch

    t = torch.from_numpy(a)
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t


def from_torch(t) -> np.ndarray:
    """Storage of a CPU torch tensor as numpy (bf16 as uint16 bit patterns)."""
    import torch

    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
