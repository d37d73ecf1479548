"""fp64 CPU oracle for row-wise safe softmax -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
path (``online_softmax_dispatcher_gb300``) never imports it and fails loudly
when its CUDA library is missing.

The arithmetic lives in ``softmax_oracle.c`` (plain C, binary64, compiled with
``-ffp-contract=off`` so that x86 and Arm hosts round identically).  This
module only builds that file and marshals numpy arrays into it:

* ``softmax(x)``            -- the definition y = exp(x - max) / sum exp(x - max)
                               in binary64 for fp32/fp16/bf16 input arrays
                               ("[CUDA] safe online softmax", section 1,
                               safe_softmax; HIP softmax tutorial, section 1).
* ``softmax_f64(x)``        -- the same definition on a float64 array.
* ``online_softmax_f64``    -- the chunked (m, d) form of "[CUDA] safe online
                               softmax", section 1, safe_online_softmax.
* ``decode`` / ``encode``   -- exact dtype -> binary64, and binary64 -> dtype
                               with round-to-nearest-even from binary64.
* ``check``                 -- streaming comparison of a candidate output with
                               the definition, row by row, over OpenMP threads.
* ``softmax_bwd_f64``       -- the backward pass dx = y * (dy - sum dy*y), the
                               derivative of the definition.
* ``check_bwd``             -- streaming comparison of a candidate dx.
* ``softmax_masked``        -- softmax(scale * x + mask) with an optional causal
                               mask (attention scores).
* ``check_masked``          -- streaming comparison against the masked form.
* ``norm_f64``              -- LayerNorm / RMSNorm along the last dimension
                               (optional gain and bias), with the per-row mean
                               and 1/sqrt(var + eps).
* ``check_norm``            -- streaming comparison of a candidate norm output
                               (and its fp32 statistics).

bf16 arrays travel as ``numpy.uint16`` bit patterns (numpy has no bfloat16);
fp16 arrays may be ``numpy.float16`` or ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, F16, BF16 = 0, 1, 2
LAYERNORM, RMSNORM = 0, 1
DTYPE_NAMES = {F32: "fp32", F16: "fp16", BF16: "bf16"}

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "softmax_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = SOURCE, out: str = _LIB_PATH) -> str:
    """Compile an oracle C source (by default softmax_oracle.c) into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class CheckResult(ctypes.Structure):
    _fields_ = [
        ("checked", ctypes.c_int64),
        ("violations", ctypes.c_int64),
        ("nonfinite", ctypes.c_int64),
        ("first_bad", ctypes.c_int64),
        ("max_rel", ctypes.c_double),
        ("max_ulp", ctypes.c_int64),
        ("max_rowsum_dev", ctypes.c_double),
        ("rowsum_violations", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Contiguous storage of x in the oracle's layout for `dtype`."""
    if dtype == F32:
        if x.dtype != np.float32:
            raise TypeError(f"fp32 input must be numpy.float32, got {x.dtype}")
        return np.ascontiguousarray(x)
    if x.dtype not in (np.uint16, np.float16):
        raise TypeError(f"{DTYPE_NAMES[dtype]} input must be 16-bit, got {x.dtype}")
    return np.ascontiguousarray(x).view(np.uint16)


def dtype_of(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.float16:
        return F16
    raise TypeError("pass dtype= explicitly for uint16 (bf16 or fp16 bit patterns)")


def _rows_cols(x: np.ndarray) -> tuple[int, int]:
    if x.ndim == 1:
        return 1, x.shape[0]
    if x.ndim != 2:
        raise ValueError("oracle works on [rows, cols] arrays")
    return x.shape[0], x.shape[1]


class Oracle:
    """Marshalling around one build of the oracle C source."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f64.restype = ctypes.c_double
        L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f64.restype = ctypes.c_double
        L.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        L.oracle_f64_to_f16.restype = ctypes.c_uint16
        L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        L.oracle_f64_to_bf16.restype = ctypes.c_uint16
        L.oracle_decode.argtypes = [vp, i32, i64, vp]
        L.oracle_encode.argtypes = [vp, i32, i64, vp]
        L.oracle_softmax_f64.argtypes = [vp, i64, i64, vp]
        L.oracle_softmax.argtypes = [vp, i32, i64, i64, vp]
        L.oracle_online_softmax_f64.argtypes = [vp, i64, i64, i64, vp]
        L.oracle_check.argtypes = [vp, vp, i32, i64, i64, vp, i64, ctypes.c_double,
                                   ctypes.c_double, i64, ctypes.c_double, ctypes.c_double,
                                   ctypes.POINTER(CheckResult)]
        L.oracle_num_threads.argtypes = []
        L.oracle_set_num_threads.argtypes = [i32]
        L.oracle_softmax_bwd_f64.argtypes = [vp, vp, i64, i64, vp]
        L.oracle_softmax_masked.argtypes = [vp, i32, i64, i64, ctypes.c_double, vp, i64, i64, vp]
        L.oracle_check_masked.argtypes = [vp, vp, i32, i64, i64, ctypes.c_double, vp, i64, i64, ctypes.c_double,
                                          ctypes.c_double, i64, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_double, ctypes.POINTER(CheckResult)]
        L.oracle_check_bwd.argtypes = [vp, vp, vp, i32, i64, i64, ctypes.c_double, i64, ctypes.c_double,
                                       ctypes.POINTER(CheckResult)]
        L.oracle_norm_f64.argtypes = [i32, vp, i32, i64, i64, vp, vp, ctypes.c_double, vp, vp, vp]
        L.oracle_check_norm.argtypes = [i32, vp, vp, i32, i64, i64, vp, vp, ctypes.c_double, vp, vp,
                                        ctypes.c_double, i64, ctypes.c_double, ctypes.POINTER(CheckResult)]
        for name in ("oracle_decode", "oracle_encode", "oracle_softmax_f64", "oracle_softmax",
                     "oracle_online_softmax_f64", "oracle_check", "oracle_num_threads", "oracle_set_num_threads",
                     "oracle_softmax_bwd_f64", "oracle_check_bwd", "oracle_softmax_masked",
                     "oracle_check_masked", "oracle_norm_f64", "oracle_check_norm"):
            getattr(L, name).restype = ctypes.c_int
        self.lib = L
        self.path = path

    def decode(self, x: np.ndarray, dtype: int | None = None) -> np.ndarray:
        """Exact dtype -> binary64."""
        dtype = dtype_of(x) if dtype is None else dtype
        bits = _as_bits(x, dtype)
        out = np.empty(bits.shape, dtype=np.float64)
        rc = self.lib.oracle_decode(_ptr(bits), dtype, bits.size, _ptr(out))
        assert rc == 0
        return out

    def encode(self, y: np.ndarray, dtype: int) -> np.ndarray:
        """binary64 -> dtype (RNE from binary64).  fp16/bf16 come back as uint16 bits."""
        y = np.ascontiguousarray(y, dtype=np.float64)
        out = np.empty(y.shape, dtype=np.float32 if dtype == F32 else np.uint16)
        rc = self.lib.oracle_encode(_ptr(y), dtype, y.size, _ptr(out))
        assert rc == 0
        return out

    def softmax_f64(self, x: np.ndarray) -> np.ndarray:
        """The definition on a float64 [rows, cols] array."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        rows, cols = _rows_cols(x)
        y = np.empty_like(x)
        rc = self.lib.oracle_softmax_f64(_ptr(x), rows, cols, _ptr(y))
        assert rc == 0
        return y

    def softmax(self, x: np.ndarray, dtype: int | None = None) -> np.ndarray:
        """The definition in binary64 on a dtype-typed [rows, cols] array."""
        dtype = dtype_of(x) if dtype is None else dtype
        bits = _as_bits(x, dtype)
        rows, cols = _rows_cols(bits)
        y = np.empty(bits.shape, dtype=np.float64)
        rc = self.lib.oracle_softmax(_ptr(bits), dtype, rows, cols, _ptr(y))
        assert rc == 0
        return y

    def softmax_rounded(self, x: np.ndarray, dtype: int | None = None) -> np.ndarray:
        """The definition rounded once (RNE from binary64) to the input dtype."""
        dtype = dtype_of(x) if dtype is None else dtype
        return self.encode(self.softmax(x, dtype), dtype)

    def online_softmax_f64(self, x: np.ndarray, chunk: int) -> np.ndarray:
        """The chunked (m, d) form on a float64 [rows, cols] array."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        rows, cols = _rows_cols(x)
        y = np.empty_like(x)
        rc = self.lib.oracle_online_softmax_f64(_ptr(x), rows, cols, int(chunk), _ptr(y))
        assert rc == 0
        return y

    def check(self, x: np.ndarray, y: np.ndarray, dtype: int, *, rel_tol: float = 0.0,
              abs_floor: float = 0.0, max_ulp: int = 0, rowsum_a: float = 0.0,
              rowsum_b: float = 0.0, rows_sel: np.ndarray | None = None) -> dict:
        """Compare a candidate output y with the definition applied to x, row by row."""
        xb = _as_bits(x, dtype)
        yb = _as_bits(y, dtype)
        if xb.shape != yb.shape:
            raise ValueError(f"shape mismatch {xb.shape} vs {yb.shape}")
        rows, cols = _rows_cols(xb)
        res = CheckResult()
        sel_ptr, n_sel = None, 0
        if rows_sel is not None:
            rows_sel = np.ascontiguousarray(rows_sel, dtype=np.int64)
            sel_ptr, n_sel = _ptr(rows_sel), rows_sel.size
        rc = self.lib.oracle_check(_ptr(xb), _ptr(yb), dtype, rows, cols, sel_ptr, n_sel,
                                   float(rel_tol), float(abs_floor), int(max_ulp),
                                   float(rowsum_a), float(rowsum_b), ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_check rejected its arguments")
        return res.as_dict()

    def softmax_bwd_f64(self, y: np.ndarray, dy: np.ndarray) -> np.ndarray:
        """dx = y * (dy - sum(dy * y)) per row, binary64."""
        y = np.ascontiguousarray(y, dtype=np.float64)
        dy = np.ascontiguousarray(dy, dtype=np.float64)
        if y.shape != dy.shape:
            raise ValueError("y and dy shapes differ")
        rows, cols = _rows_cols(y)
        dx = np.empty_like(y)
        rc = self.lib.oracle_softmax_bwd_f64(_ptr(y), _ptr(dy), rows, cols, _ptr(dx))
        assert rc == 0
        return dx

    def check_bwd(self, y: np.ndarray, dy: np.ndarray, dx: np.ndarray, dtype: int, *, rel_tol: float = 0.0,
                  max_ulp: int = 0, k_eps: float = 0.0) -> dict:
        """Compare a candidate dx with the backward definition on the decoded y, dy."""
        yb, dyb, dxb = _as_bits(y, dtype), _as_bits(dy, dtype), _as_bits(dx, dtype)
        if not (yb.shape == dyb.shape == dxb.shape):
            raise ValueError("shape mismatch")
        rows, cols = _rows_cols(yb)
        res = CheckResult()
        rc = self.lib.oracle_check_bwd(_ptr(yb), _ptr(dyb), _ptr(dxb), dtype, rows, cols, float(rel_tol),
                                       int(max_ulp), float(k_eps), ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_check_bwd rejected its arguments")
        return res.as_dict()

    def softmax_masked(self, x: np.ndarray, dtype: int, scale: float, mask: np.ndarray | None = None,
                       causal_q: int = 0) -> np.ndarray:
        """softmax(scale * x + mask) with an optional causal mask, binary64.
        mask: [mask_rows, cols] in x's dtype; row r uses mask row r % mask_rows."""
        xb = _as_bits(x, dtype)
        rows, cols = _rows_cols(xb)
        mb, mrows = None, 0
        if mask is not None:
            mb = _as_bits(mask, dtype)
            mrows = _rows_cols(mb)[0]
        y = np.empty((rows, cols), dtype=np.float64)
        rc = self.lib.oracle_softmax_masked(_ptr(xb), dtype, rows, cols, float(scale),
                                            _ptr(mb) if mb is not None else None, mrows, int(causal_q), _ptr(y))
        assert rc == 0
        return y

    def check_masked(self, x, y, dtype, scale, mask=None, causal_q=0, *, rel_tol=0.0, abs_floor=0.0, max_ulp=0,
                     rowsum_a=0.0, rowsum_b=0.0, zrel=0.0) -> dict:
        """Compare a candidate with softmax(scale * x + mask) (+ causal mask)."""
        xb, yb = _as_bits(x, dtype), _as_bits(y, dtype)
        rows, cols = _rows_cols(xb)
        mb, mrows = None, 0
        if mask is not None:
            mb = _as_bits(mask, dtype)
            mrows = _rows_cols(mb)[0]
        res = CheckResult()
        rc = self.lib.oracle_check_masked(_ptr(xb), _ptr(yb), dtype, rows, cols, float(scale),
                                          _ptr(mb) if mb is not None else None, mrows, int(causal_q),
                                          float(rel_tol), float(abs_floor), int(max_ulp), float(rowsum_a),
                                          float(rowsum_b), float(zrel), ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_check_masked rejected its arguments")
        return res.as_dict()

    def norm_f64(self, kind: int, x: np.ndarray, dtype: int, gamma: np.ndarray | None = None,
                 beta: np.ndarray | None = None, eps: float = 1e-5):
        """LayerNorm (kind 0) or RMSNorm (kind 1) of a dtype-typed [rows, cols]
        array in binary64; gamma / beta: [cols] in the same dtype or None.
        Returns (y, mean, rstd) as float64 arrays."""
        xb = _as_bits(x, dtype)
        rows, cols = _rows_cols(xb)
        gb = _as_bits(gamma, dtype) if gamma is not None else None
        bb = _as_bits(beta, dtype) if beta is not None else None
        for v in (gb, bb):
            if v is not None and v.size != cols:
                raise ValueError("gamma / beta must hold cols values")
        y = np.empty((rows, cols), dtype=np.float64)
        mean = np.empty(rows, dtype=np.float64)
        rstd = np.empty(rows, dtype=np.float64)
        rc = self.lib.oracle_norm_f64(int(kind), _ptr(xb), dtype, rows, cols,
                                      _ptr(gb) if gb is not None else None,
                                      _ptr(bb) if bb is not None else None, float(eps), _ptr(y), _ptr(mean),
                                      _ptr(rstd))
        if rc != 0:
            raise ValueError("oracle_norm_f64 rejected its arguments")
        return y, mean, rstd

    def check_norm(self, kind: int, x: np.ndarray, y: np.ndarray, dtype: int, gamma=None, beta=None,
                   eps: float = 1e-5, mean=None, rstd=None, *, rel_tol: float = 0.0, max_ulp: int = 0,
                   k_eps: float = 0.0) -> dict:
        """Compare a candidate norm output (and optional fp32 mean / rstd per
        row) with the definition; statistic violations count as
        rowsum_violations."""
        xb, yb = _as_bits(x, dtype), _as_bits(y, dtype)
        if xb.shape != yb.shape:
            raise ValueError("shape mismatch")
        rows, cols = _rows_cols(xb)
        gb = _as_bits(gamma, dtype) if gamma is not None else None
        bb = _as_bits(beta, dtype) if beta is not None else None
        mp = np.ascontiguousarray(mean, dtype=np.float32) if mean is not None else None
        rp = np.ascontiguousarray(rstd, dtype=np.float32) if rstd is not None else None
        for v in (mp, rp):
            if v is not None and v.size != rows:
                raise ValueError("mean / rstd must hold rows values")
        res = CheckResult()
        rc = self.lib.oracle_check_norm(int(kind), _ptr(xb), _ptr(yb), dtype, rows, cols,
                                        _ptr(gb) if gb is not None else None,
                                        _ptr(bb) if bb is not None else None, float(eps),
                                        _ptr(mp) if mp is not None else None,
                                        _ptr(rp) if rp is not None else None, float(rel_tol), int(max_ulp),
                                        float(k_eps), ctypes.byref(res))
        if rc != 0:
            raise ValueError("oracle_check_norm rejected its arguments")
        return res.as_dict()

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> int:
        """OpenMP threads for later oracle calls from this host thread; returns the number in force."""
        return int(self.lib.oracle_set_num_threads(int(n)))


def default() -> Oracle:
    """The oracle built from softmax_oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def decode(x, dtype=None):
    return default().decode(x, dtype)


def encode(y, dtype):
    return default().encode(y, dtype)


def softmax_f64(x):
    return default().softmax_f64(x)


def softmax(x, dtype=None):
    return default().softmax(x, dtype)


def softmax_rounded(x, dtype=None):
    return default().softmax_rounded(x, dtype)


def online_softmax_f64(x, chunk):
    return default().online_softmax_f64(x, chunk)


def check(x, y, dtype, **kw):
    return default().check(x, y, dtype, **kw)


def num_threads():
    return default().num_threads()


def softmax_masked(x, dtype, scale, mask=None, causal_q=0):
    return default().softmax_masked(x, dtype, scale, mask, causal_q)


def check_masked(x, y, dtype, scale, mask=None, causal_q=0, **kw):
    return default().check_masked(x, y, dtype, scale, mask, causal_q, **kw)


def softmax_bwd_f64(y, dy):
    return default().softmax_bwd_f64(y, dy)


def check_bwd(y, dy, dx, dtype, **kw):
    return default().check_bwd(y, dy, dx, dtype, **kw)


def norm_f64(kind, x, dtype, gamma=None, beta=None, eps=1e-5):
    return default().norm_f64(kind, x, dtype, gamma, beta, eps)


def check_norm(kind, x, y, dtype, gamma=None, beta=None, eps=1e-5, mean=None, rstd=None, **kw):
    return default().check_norm(kind, x, y, dtype, gamma, beta, eps, mean, rstd, **kw)
