"""Host-only checks of the C ABI: the library loads, exports exactly what
include/softmax.h declares, rejects bad arguments before touching CUDA, and
its dispatcher (softmax_plan, pure host code) picks launch shapes that cover
every row.  No call here reaches a CUDA runtime function."""
import ctypes
import os
import re

import pytest

from online_softmax_dispatcher_gb300 import _binding as B
from online_softmax_dispatcher_gb300 import build as build_mod
from online_softmax_dispatcher_gb300 import workloads as W
from online_softmax_dispatcher_gb300.workloads import WORKLOADS

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "softmax.h")

# A GB300 as the dispatcher sees it (152 SMs, 227 KB opt-in shared memory).
GB300 = B.DeviceInfo(sm_count=152, max_smem_optin=232448, cluster_launch=1, l2_bytes=132644864,
                     cc_major=10, cc_minor=3)


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b((?:softmax|layernorm|rmsnorm|norm)_\w+)\s*\(", text))


def exported_symbols(path):
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    prefixes = ("softmax_", "layernorm_", "rmsnorm_", "norm_")
    return {line.split()[-1] for line in out.splitlines() if " T " in line and line.split()[-1].startswith(prefixes)}


def test_exports_match_header(lib):
    declared = declared_functions()
    assert declared == set(B.EXPORTS)
    assert exported_symbols(B.LIB_PATH) == declared
    for name in declared:
        assert hasattr(lib, name)


def test_strings_and_version(lib):
    assert B.softmax_abi_version() == 1
    assert B.softmax_strerror(0) == "ok"
    assert "overlap" in B.softmax_strerror(B.ERR_ALIAS)
    assert B.softmax_strerror(12345) == "unknown status"
    names = [B.softmax_variant_name(v) for v in range(B.VARIANT_COUNT)]
    assert names == list(B.VARIANTS)


BASE = 1 << 40  # fake, 256-byte aligned "device" addresses: validation only looks at them


@pytest.mark.parametrize("args,want", [
    ((BASE, BASE + 4096, 2, 3, 7), B.ERR_UNSUPPORTED_DTYPE),
    ((BASE, BASE + 4096, -1, 3, 0), B.ERR_INVALID_ARG),
    ((BASE, BASE + 4096, 2, -3, 0), B.ERR_INVALID_ARG),
    ((0, BASE, 2, 3, 0), B.ERR_INVALID_ARG),
    ((BASE, 0, 2, 3, 0), B.ERR_INVALID_ARG),
    ((BASE + 2, BASE + 4096, 2, 3, 0), B.ERR_INVALID_ARG),       # fp32 needs 4-byte alignment
    ((BASE + 1, BASE + 4097, 2, 3, 1), B.ERR_INVALID_ARG),       # fp16 needs 2-byte alignment
    ((BASE, BASE + 20, 2, 3, 0), B.ERR_ALIAS),                   # 24 bytes of x overlap y
    ((BASE + 20, BASE, 2, 3, 0), B.ERR_ALIAS),                   # y overlaps the start of x
    ((BASE, BASE + 4, 2, 3, 0), B.ERR_ALIAS),                    # y one element past x
    ((BASE, BASE + 64, 2**40, 2**40, 0), B.ERR_INVALID_ARG),     # rows*cols*4 overflows int64
    ((0, 0, 0, 5, 0), B.OK),                                     # empty: no launch, no device
    ((0, 0, 5, 0, 2), B.OK),
])
def test_argument_validation(lib, args, want):
    x, y, rows, cols, dt = args
    assert B.softmax_fwd(x, y, rows, cols, dt, 0) == want
    assert B.softmax_fwd_variant(x, y, rows, cols, dt, 0, 0) == want
    rc, _ = B.softmax_plan(GB300, x, y, rows, cols, dt)
    assert rc == want


def test_in_place_is_accepted(lib):
    # y == x exactly is an in-place call; every variant's plan accepts it
    for rows, cols, dt in ((2, 3, 0), (8192, 5003, 1), (32768, 32000, 2), (4, 4194304, 0)):
        rc, p = B.softmax_plan(GB300, BASE, BASE, rows, cols, dt)
        assert rc == B.OK
        for v in range(1, B.VARIANT_COUNT):
            rc, _ = B.softmax_plan(GB300, BASE, BASE, rows, cols, dt, v)
            assert rc in (B.OK, B.ERR_UNSUPPORTED_SHAPE, B.ERR_INVALID_ARG), (rows, cols, v, rc)
            assert rc != B.ERR_ALIAS


def test_adjacent_buffers_are_not_aliases(lib):
    # x = [BASE, BASE+24), y starts right after: no overlap
    rc, p = B.softmax_plan(GB300, BASE, BASE + 24, 2, 3, 0)
    assert rc == B.OK


def test_bad_variant_and_null_out(lib):
    assert B.softmax_fwd_variant(BASE, BASE + 4096, 2, 3, 0, 99, 0) == B.ERR_INVALID_ARG
    assert B.softmax_fwd_variant(BASE, BASE + 4096, 2, 3, 0, -1, 0) == B.ERR_INVALID_ARG
    assert lib.softmax_query_variant(BASE, BASE + 4096, 2, 3, 0, None) == B.ERR_INVALID_ARG
    assert lib.softmax_plan(None, BASE, BASE + 4096, 2, 3, 0, 0, None) == B.ERR_INVALID_ARG
    assert lib.softmax_device_query(None) == B.ERR_INVALID_ARG
    assert lib.softmax_get_device_error(None, None) == B.ERR_INVALID_ARG
    assert lib.softmax_fwd_plan(BASE, BASE + 4096, 2, 3, 0, None, None) == B.ERR_INVALID_ARG


def _nch_max(cols, elem, aligned):
    rb = cols * elem
    return rb // 16 if aligned else -(-(rb + 16 - elem) // 16)


def _covers(p, rows, cols, elem, aligned):
    """The plan's threads cover every 16-byte chunk of a row: for the
    lanes-per-row and CTA-per-row kernels, every whole chunk inside a row (they
    take the partial edge chunks element by element)."""
    n = _nch_max(cols, elem, aligned)
    n_int = cols * elem // 16
    if p.variant == B.VARIANT_ROWGROUP:
        return p.lanes_per_row * p.chunks_per_thread >= n_int and (p.lanes_per_row > 1 or p.chunks_per_thread == 1)
    if p.variant == B.VARIANT_BLOCK:
        return p.block_threads * p.chunks_per_thread >= n_int
    if p.variant == B.VARIANT_BLOCK_TMA:
        stage = p.smem_bytes // p.stages
        lead = 0 if aligned else 16 - elem
        return stage * 1 >= -(-(lead + p.rows_per_tile * cols * elem) // 16) * 16
    return p.variant in (B.VARIANT_STREAM, B.VARIANT_SPLITK, B.VARIANT_SPLITK_WIDE, B.VARIANT_SPLITK_GRID)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_dispatch_of_workloads(lib, name):
    w = WORKLOADS[name]
    x = BASE
    y = BASE + (1 << 36)
    rc, p = B.softmax_plan(GB300, x, y, w.rows, w.cols, w.dtype_code)
    assert rc == B.OK
    aligned = (w.cols * w.elem_bytes) % 16 == 0
    assert p.aligned == int(aligned) and p.y_vector == 1
    assert _covers(p, w.rows, w.cols, w.elem_bytes, aligned)
    expect = {
        "fp32_128x1000": B.VARIANT_ROWGROUP,
        "attn_fp16_65536x512": B.VARIANT_ROWGROUP,
        "awkward_fp16_8192x5003": B.VARIANT_BLOCK,
        "vocab_bf16_32768x32000": B.VARIANT_BLOCK,
        "splitk_fp32_4x4194304": B.VARIANT_SPLITK_GRID,
        "splitk_fp16_4x4194304": B.VARIANT_SPLITK_GRID,
    }[name]
    assert p.variant == expect, B.softmax_variant_name(p.variant)
    if p.variant == B.VARIANT_SPLITK_GRID:
        assert p.block_threads == 512 and p.cluster_x == 1
        if w.dtype == "fp16":
            # ring form, one row per group: 4 groups of 38 CTAs, a 220 KB share each
            assert (p.grid_x, p.grid_y, p.stages, p.lanes_per_row) == (38, 4, 1, 0)
            buf = -(-(-(-(w.cols * w.elem_bytes // 16) // 38) * 16) // 128) * 128
            assert p.smem_bytes == buf <= 232448 - 2048
        else:
            # the ring would give each group two rows in turn: the pipelined
            # form, every CTA on every row, two 110 KB buffers the rows pass
            # through two at a time, a 256-thread fold team
            assert (p.grid_x, p.grid_y, p.stages, p.lanes_per_row) == (152, 1, 2, 256)
            buf = -(-(-(-(w.cols * w.elem_bytes // 16) // 152) * 16) // 128) * 128
            assert p.smem_bytes == 2 * buf <= 232448 - 2048


@pytest.mark.parametrize("dt,elem", [(0, 4), (1, 2), (2, 2)])
def test_dispatch_sweep_covers_rows(lib, dt, elem):
    for cols in list(range(1, 70)) + [127, 128, 129, 255, 256, 257, 511, 512, 513, 1000, 1023, 1024, 1025,
                                      2047, 2048, 4096, 5003, 8191, 8192, 16384, 32000, 50000, 65536,
                                      100000, 131072, 1 << 20, (1 << 22) + 3]:
        for rows in (1, 3, 77, 4096):
            for xoff, yoff in ((0, 0), (elem, elem), (0, elem), (2 * elem, 6 * elem)):
                x, y = BASE + xoff, BASE + (1 << 38) + yoff
                for v in range(B.VARIANT_COUNT):
                    rc, p = B.softmax_plan(GB300, x, y, rows, cols, dt, v)
                    if rc == B.ERR_UNSUPPORTED_SHAPE:
                        assert v != B.VARIANT_AUTO and v != B.VARIANT_STREAM
                        continue
                    assert rc == B.OK, (cols, rows, v)
                    aligned = x % 16 == 0 and y % 16 == 0 and (cols * elem) % 16 == 0
                    assert p.aligned == int(aligned)
                    assert p.y_vector == int((y - x) % 16 == 0)
                    assert _covers(p, rows, cols, elem, aligned), (cols, rows, v, p.as_dict())
                    if v != B.VARIANT_AUTO:
                        assert p.variant == v
                    assert p.grid_x >= 1


def test_splitk_needs_clusters(lib):
    no_clusters = B.DeviceInfo(sm_count=152, max_smem_optin=232448, cluster_launch=0,
                               l2_bytes=1 << 27, cc_major=10, cc_minor=3)
    rc, p = B.softmax_plan(no_clusters, BASE, BASE + (1 << 36), 4, 1 << 22, 0)
    assert rc == B.OK and p.variant == B.VARIANT_SPLITK_GRID  # the grid split needs no cluster
    rc, _ = B.softmax_plan(no_clusters, BASE, BASE + (1 << 36), 4, 1 << 22, 0, B.VARIANT_SPLITK)
    assert rc == B.ERR_UNSUPPORTED_SHAPE
    # a GPU without cooperative launch of this kind: the stream kernel
    old = B.DeviceInfo(sm_count=152, max_smem_optin=232448, cluster_launch=0, l2_bytes=1 << 27,
                       cc_major=8, cc_minor=0)
    rc, p = B.softmax_plan(old, BASE, BASE + (1 << 36), 4, 1 << 22, 0)
    assert rc == B.OK and p.variant == B.VARIANT_STREAM


def test_grid_split_limits(lib):
    # few rows only (rows * 2 <= SMs); the ring form while a CTA's share of a
    # row fits a buffer and rows x CTAs per row fit a scratch slot (4096)
    rc, _ = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 77, 1 << 20, 1, B.VARIANT_SPLITK_GRID)
    assert rc == B.ERR_UNSUPPORTED_SHAPE
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 76, 1 << 20, 1, B.VARIANT_SPLITK_GRID)
    # 76 rows of 2 MiB: shares fit a buffer from 10 CTAs a row on, so 6 rows per
    # group at least, and with 6, 13 groups of 11 CTAs
    assert rc == B.OK and (p.grid_x, p.grid_y) == (11, 13) and p.stages == 1
    assert p.smem_bytes == -(-(-(-(1 << 17) // 11) * 16) // 128) * 128
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 1, 1 << 24, 1, B.VARIANT_SPLITK_GRID)
    assert rc == B.OK and p.stages == 1 and p.grid_x == 152 and p.grid_y == 1   # 32 MiB over 152 SMs
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 1, 1 << 25, 1, B.VARIANT_SPLITK_GRID)
    assert rc == B.OK and p.stages == 0 and p.grid_x == 304 and p.grid_y == 1   # 64 MiB: streamed
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 2, 1 << 24, 1, B.VARIANT_SPLITK_GRID)
    assert rc == B.OK and p.stages == 1 and (p.grid_x, p.grid_y) == (152, 1)     # two rows, one buffer
    assert p.lanes_per_row == 0                                                   # ring form
    # one row per group when the shares fit: the ring form
    rc, p = B.softmax_plan(GB300, BASE + 2, BASE + (1 << 36) + 2, 3, (1 << 21) + 7, 2, B.VARIANT_SPLITK_GRID)
    assert rc == B.OK and p.aligned == 0 and (p.grid_x, p.grid_y, p.stages, p.lanes_per_row) == (50, 3, 1, 0)
    # where the ring would give a group several rows in turn: the pipelined form
    # (every CTA on every row, a 256-thread fold team), as many buffers as fit,
    # at most one per row and at most 8.  16 rows of 2 MiB: the ring would take
    # 8 groups of 19 CTAs, two rows each
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 16, 1 << 20, 1, B.VARIANT_SPLITK_GRID)
    assert rc == B.OK and (p.grid_x, p.grid_y, p.stages, p.lanes_per_row) == (152, 1, 8, 256)
    assert p.smem_bytes == 8 * (-(-(-(-(1 << 17) // 152) * 16) // 128) * 128)
    # the pipelined form's partials (rows x 152) must fit a scratch slot (4096)
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 26, 1 << 20, 1, B.VARIANT_SPLITK_GRID)
    assert rc == B.OK and p.lanes_per_row == 256 and p.grid_y == 1
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 27, 1 << 20, 1, B.VARIANT_SPLITK_GRID)
    assert rc == B.OK and p.lanes_per_row == 0 and p.grid_y > 1



def test_forced_variants_reject_rows_too_long(lib):
    rc, _ = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 8, 1 << 20, 1, B.VARIANT_ROWGROUP)
    assert rc == B.ERR_UNSUPPORTED_SHAPE
    rc, _ = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 8, 1 << 20, 1, B.VARIANT_BLOCK)
    assert rc == B.ERR_UNSUPPORTED_SHAPE
    rc, _ = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 8, 1 << 20, 1, B.VARIANT_BLOCK_TMA)
    assert rc == B.ERR_UNSUPPORTED_SHAPE
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 8, 1 << 20, 1, B.VARIANT_STREAM)
    assert rc == B.OK and p.variant == B.VARIANT_STREAM


def test_library_refuses_to_load_when_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(B.SoftmaxLibraryMissing):
        B.lib()


def test_plan_struct_layout():
    # the ctypes mirror must match the C struct (ints, then int64 grid dims)
    assert ctypes.sizeof(B.LaunchPlan) == 64
    assert B.LaunchPlan.grid_x.offset == 24 and B.LaunchPlan.cluster_x.offset == 40
    assert B.LaunchPlan.back_passes.offset == 56
    assert ctypes.sizeof(B.DeviceInfo) == 24


def test_norm_argument_validation(lib):
    # argument checks run before any device query, so they work without a GPU
    x, y = BASE, BASE + (1 << 30)
    g = BASE + (1 << 31)
    m, r = BASE + (1 << 32), BASE + (1 << 32) + 4096
    f = B.norm_fwd_variant
    assert f(2, x, y, 8, 64, 0, 0, 0, 1e-5, 0, 0, 0, 0) == B.ERR_INVALID_ARG          # bad kind
    assert f(0, x, y, 8, 64, 0, 0, 0, -1e-5, 0, 0, 0, 0) == B.ERR_INVALID_ARG         # eps < 0
    assert f(0, x, y, 8, 64, 0, 0, 0, float("inf"), 0, 0, 0, 0) == B.ERR_INVALID_ARG  # eps not finite
    assert f(0, x, y, 8, 64, 0, g + 2, 0, 1e-5, 0, 0, 0, 0) == B.ERR_INVALID_ARG      # gain misaligned
    assert f(0, x, y, 8, 64, 1, g + 1, 0, 1e-5, 0, 0, 0, 0) == B.ERR_INVALID_ARG
    assert f(0, x, y, 8, 64, 0, y + 64, 0, 1e-5, 0, 0, 0, 0) == B.ERR_ALIAS           # gain inside y
    assert f(0, x, y, 8, 64, 0, 0, y, 1e-5, 0, 0, 0, 0) == B.ERR_ALIAS                # bias inside y
    assert f(1, x, y, 8, 64, 0, 0, y, 1e-5, 0, 0, 0, 0) != B.ERR_ALIAS                # RMSNorm ignores the bias
    assert f(0, x, y, 8, 64, 0, 0, 0, 1e-5, m + 2, 0, 0, 0) == B.ERR_INVALID_ARG      # mean misaligned
    assert f(0, x, y, 8, 64, 0, 0, 0, 1e-5, y + 16, 0, 0, 0) == B.ERR_ALIAS           # mean inside y
    assert f(0, x, y, 8, 64, 0, 0, 0, 1e-5, x, 0, 0, 0) == B.ERR_ALIAS                # mean inside x
    assert f(0, x, y, 8, 64, 0, 0, 0, 1e-5, m, m + 16, 0, 0) == B.ERR_ALIAS           # mean and rstd overlap
    assert f(0, x, y, 8, 64, 0, g, 0, 1e-5, 0, g + 8, 0, 0) == B.ERR_ALIAS            # rstd inside the gain
    assert f(0, x, x + 4, 8, 64, 0, 0, 0, 1e-5, 0, 0, 0, 0) == B.ERR_ALIAS            # partial x / y overlap
    assert f(0, x, y, 0, 64, 0, 0, 0, 1e-5, 0, 0, 0, 0) == B.OK                       # empty: no launch
    assert B.layernorm_fwd(x, y, 8, 64, 7, 0, 0, 1e-5, 0, 0, 0) == B.ERR_UNSUPPORTED_DTYPE
    assert B.rmsnorm_fwd(x, y, 8, 64, 0, g + 2, 1e-5, 0, 0) == B.ERR_INVALID_ARG


def test_other_operations_dispatch(lib):
    # the backward, masked and normalisation dispatchers as host functions
    y, dy, dx = BASE, BASE + (1 << 36), BASE + (2 << 36)
    expect_bwd = {"attn_fp16_65536x512": (B.VARIANT_ROWGROUP, None), "awkward_fp16_8192x5003": (B.VARIANT_BLOCK, 4),
                  "vocab_bf16_32768x32000": (B.VARIANT_BLOCK, 8)}
    for name, (v, V) in expect_bwd.items():
        w = W.WORKLOADS[name]
        rc, p = B.softmax_bwd_plan(GB300, y, dy, dx, w.rows, w.cols, w.dtype_code)
        assert rc == B.OK and p.variant == v, name
        if V is not None:
            assert p.chunks_per_thread == V
            assert p.block_threads * V >= -(-w.cols * w.elem_bytes // 16)
        if V == 8:
            # one 512-thread CTA per SM: the grid is one CTA per SM, looping over rows
            assert p.grid_x == 152 and p.block_threads == 512
    rc, p = B.softmax_masked_plan(GB300, BASE, BASE + (1 << 36), 65536, 512, 1)
    # 2 chunks a lane for 16-bit rows of 17 - 64 chunks, 128-thread CTAs
    assert rc == B.OK and p.variant == B.VARIANT_ROWGROUP
    assert (p.lanes_per_row, p.chunks_per_thread, p.block_threads) == (32, 2, 128)
    rc, p = B.softmax_bwd_plan(GB300, y, dy, dx, 65536, 512, 1)
    assert rc == B.OK and (p.lanes_per_row, p.chunks_per_thread, p.block_threads) == (32, 2, 128)
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 65536, 512, 1)
    assert rc == B.OK and (p.lanes_per_row, p.chunks_per_thread, p.block_threads, p.grid_x) == (32, 2, 128, 16384)
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 36), 262144, 128, 1)    # 16 chunks: 4 a lane
    assert rc == B.OK and (p.lanes_per_row, p.chunks_per_thread) == (4, 4)
    for name, (v, G, V) in {"ln_fp16_131040x192": (B.VARIANT_ROWGROUP, 8, 3),
                            "ln_fp16_32760x384": (B.VARIANT_ROWGROUP, 16, 3),
                            "rms_bf16_16384x4096": (B.VARIANT_BLOCK, 0, 4)}.items():
        w = W.NORM_WORKLOADS[name]
        rc, p = B.norm_plan(GB300, w.kind, BASE, BASE + (1 << 36), w.rows, w.cols, w.dtype_code)
        assert rc == B.OK and p.variant == v and p.chunks_per_thread == V, (name, p.as_dict())
        if G:
            assert p.lanes_per_row == G and p.block_threads == 128
    # arguments are checked as the launching calls check them
    assert lib.softmax_bwd_plan(None, y, dy, dx, 2, 3, 0, 0, None) == B.ERR_INVALID_ARG
    rc, _ = B.softmax_bwd_plan(GB300, y, dy, dx, 2, 3, 7)
    assert rc == B.ERR_UNSUPPORTED_DTYPE
    rc, _ = B.softmax_masked_plan(GB300, BASE, BASE + 4, 2, 3, 0)
    assert rc == B.ERR_ALIAS
    rc, _ = B.norm_plan(GB300, 5, BASE, BASE + (1 << 36), 2, 3, 0)
    assert rc == B.ERR_INVALID_ARG
    rc, p = B.norm_plan(GB300, 0, BASE, BASE + (1 << 36), 0, 3, 0)
    assert rc == B.OK and p.grid_x == 0


def test_long_block_rows_dispatch(lib):
    # rows of 64 - 128 KiB: off the 16-byte grid the block kernel at 16 chunks
    # and up to 512 threads, one CTA per SM looping over rows; on the grid the
    # bulk-copy tiles; past 8192 chunks neither holds the row in registers
    y = BASE + (1 << 36)
    rc, p = B.softmax_plan(GB300, BASE, y, 16384, 50257, 2)
    assert rc == B.OK and p.variant == B.VARIANT_BLOCK
    assert p.chunks_per_thread == 16 and 256 < p.block_threads <= 512 and p.grid_x == 152
    assert p.block_threads * 16 >= 50257 * 2 // 16
    rc, p = B.softmax_plan(GB300, BASE, y, 100, 50257, 2)
    assert rc == B.OK and p.variant == B.VARIANT_BLOCK and p.grid_x == 100     # fewer rows than SMs
    rc, p = B.softmax_plan(GB300, BASE, y, 16384, 40000, 1)                      # on the grid: 5000 chunks
    assert rc == B.OK and p.variant == B.VARIANT_BLOCK_TMA
    rc, p = B.softmax_plan(GB300, BASE, y, 16384, 40000, 1, B.VARIANT_BLOCK)    # still allowed when forced
    assert rc == B.OK and p.chunks_per_thread == 16 and p.grid_x == 152
    rc, p = B.softmax_plan(GB300, BASE, y, 8192, 65536, 2)                       # 8192 chunks exactly
    assert rc == B.OK and p.variant == B.VARIANT_BLOCK and p.block_threads == 512
    rc, _ = B.softmax_plan(GB300, BASE, y, 8192, 65544, 2, B.VARIANT_BLOCK)      # 8193 chunks
    assert rc == B.ERR_UNSUPPORTED_SHAPE
    # up to 64 KiB rows keep one CTA per row
    rc, p = B.softmax_plan(GB300, BASE, y, 32768, 32000, 2)
    assert rc == B.OK and p.variant == B.VARIANT_BLOCK and p.block_threads == 256 and p.grid_x == 32768


def test_stream_walk_direction(lib):
    # back_passes = 1 (re-read passes walk each row from the other end) once the
    # rows in flight (2 CTAs per SM) hold more than 5/12 of L2
    line = GB300.l2_bytes * 5 / 12
    for rows, cols, dt, x_off, want in (
            (4096, 65600, 1, 0, 0),      # 304 rows x 131 KB = 40 MB
            (2048, 131072, 2, 0, 1),     # 304 x 262 KB = 80 MB
            (2048, 262144, 1, 0, 1),
            (1024, 262144, 0, 0, 1),
            (8, 1 << 20, 1, 0, 0),       # few rows: 8 x 2 MB
            (2048, 131071, 1, 1, 1),     # off the grid: 304 rows x 262 KB = 80 MB
            (4096, 65599, 1, 1, 0),      # off the grid: 40 MB
            (2048, 262143, 1, 1, 1),     # off the grid: 80 MB
            (6144, 98304, 1, 0, 1),      # 60 MB
            (8192, 81920, 1, 0, 0)):     # 50 MB
        e = (4, 2, 2)[dt]
        rc, p = B.softmax_plan(GB300, BASE + x_off * e, BASE + (1 << 36) + x_off * e, rows, cols, dt,
                               B.VARIANT_STREAM)
        assert rc == B.OK and p.variant == B.VARIANT_STREAM, (rows, cols)
        assert (min(rows, 304) * cols * e > line) == bool(want)
        assert p.back_passes == want and p.stages == 0, (rows, cols, dt, p.back_passes)
    # a device that reports no L2 size: forward
    dev = B.DeviceInfo(**{**{f: getattr(GB300, f) for f, _ in GB300._fields_}, "l2_bytes": 0})
    rc, p = B.softmax_plan(dev, BASE, BASE + (1 << 36), 2048, 262144, 1, B.VARIANT_STREAM)
    assert rc == B.OK and p.back_passes == 0


def test_bwd_stream_walk_direction(lib):
    half = GB300.l2_bytes // 2
    for rows, cols, dt, off, want in ((400, 65600, 1, 0, 1), (4096, 40000, 1, 0, 0), (4096, 128256, 2, 0, 1),
                                      (512, 262144, 0, 0, 1), (400, 65601, 1, 1, 0), (40, 65536, 0, 0, 0)):
        e = (4, 2, 2)[dt]
        rc, p = B.softmax_bwd_plan(GB300, BASE + off * e, BASE + (1 << 36) + off * e, BASE + (2 << 36) + off * e,
                                   rows, cols, dt, 0)
        assert rc == B.OK and p.variant == B.VARIANT_STREAM, (rows, cols)
        resident = 152 * (2 if p.aligned else 1)
        assert (min(rows, resident) * 2 * cols * e > half) == bool(want)
        assert p.back_passes == want, (rows, cols, dt)


def test_many_long_16bit_rows_take_the_cluster_split(lib):
    # 16-bit rows on the 16-byte grid of more than 256 KiB and less than 2 MiB,
    # at least as many as SMs: the cluster split with one CTA per row
    for rows, cols, dt, off, want in ((2048, 262144, 1, 0, B.VARIANT_SPLITK), (3072, 196608, 1, 0, B.VARIANT_SPLITK),
                                      (152, 262144, 2, 0, B.VARIANT_SPLITK), (1024, 524288, 1, 0, B.VARIANT_SPLITK),
                                      (4096, 131072, 2, 0, B.VARIANT_STREAM),   # 256 KiB
                                      (512, 1 << 20, 1, 0, B.VARIANT_STREAM),   # 2 MiB
                                      (1024, 262144, 0, 0, B.VARIANT_STREAM),   # fp32
                                      (2048, 262143, 1, 1, B.VARIANT_STREAM),   # off the grid
                                      (70000, 131080, 1, 0, B.VARIANT_STREAM)):  # more rows than a grid's y
        e = (4, 2, 2)[dt]
        rc, p = B.softmax_plan(GB300, BASE + off * e, BASE + (1 << 38) + off * e, rows, cols, dt)
        assert rc == B.OK and p.variant == want, (rows, cols, dt, p.variant)
        if want == B.VARIANT_SPLITK:
            assert (p.cluster_x, p.grid_x, p.grid_y, p.back_passes) == (1, 1, rows, 0)
    # a forced cluster split on at least as many rows as SMs: one CTA per row
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 38), 200, 1 << 20, 1, B.VARIANT_SPLITK)
    assert rc == B.OK and p.cluster_x == 1 and p.grid_y == 200
    rc, p = B.softmax_plan(GB300, BASE, BASE + (1 << 38), 100, 1 << 20, 1, B.VARIANT_SPLITK)
    assert rc == B.OK and p.cluster_x == 4
