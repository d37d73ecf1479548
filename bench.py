"""Benchmark: row-wise softmax GB/s on one GB300 (and N replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one softmax pass over the whole workload batch (the default is the
attention-score softmax [4, 32, 512, 512] fp16 = [65536, 512]).  The timed
region is K steps bracketed by a barrier and torch.cuda.synchronize(),
measured with CUDA events on the launching stream; consecutive steps rotate
over input/output buffer sets that total more than twice the L2 size, so every
step reads x from and writes y to HBM.  value = algorithmic bytes
(rows * cols * (in + out dtype bytes)) / time, summed over ranks.

Extra keys: `e2e` (the same metric through the public API with pinned host
buffers, host->device copy of x and device->host copy of y inside the timed
region), `roofline` (the dominant kernel's achieved bandwidth against the
measured HBM copy peak, and against the rated one), `latency_us` (median
single-launch time, cold L2), `clocks` (nvidia-smi samples during the timed
region), `per_config` (the forward softmax of every softmax workload, each
timed the same way in the same process), `cpu_baseline` (the fp64 oracle on
all the host's cores and on one core over a bounded sample, rank 0 only).

--impl reference times the oracle itself on the host cores (the pages'
method has no runnable reference implementation here) on the same config.
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "softmax GB/s (read+write) and % of GB300 HBM peak; latency at [4,32,512,512] fp16"
DEFAULT_WORKLOAD = "attn_fp16_65536x512"
FALLBACK_HBM_GBS = 6800.0
# NVIDIA's rated HBM3e bandwidth of one GB300 GPU (8 TB/s); the memory clock
# nvidia-smi reports (3996 MHz, double data rate) on the 8192-bit bus gives
# 8184 GB/s.  A copy kernel reaches about 6.8 TB/s of it.
RATED_HBM_GBS = 8000.0
RATED_SOURCE = "NVIDIA's rated GB300 HBM3e bandwidth, 8 TB/s"


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


# ----------------------------------------------------------------------------- distributed


def dist_setup(n_gpus: int):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as dist

    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, ws, local


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    """Largest v over all ranks (every rank gets it)."""
    if ws <= 1:
        return v
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, ws: int) -> float:
    if ws <= 1:
        return v
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, with host timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.gpu_id = gpu_id
        self.t_start = time.time()

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd[1:1] = ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self) -> list[dict]:
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for rec in csv.reader(io.StringIO(out)):
            if len(rec) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(rec[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + rec[0].strip().split(".")[1]) if "." in rec[0] else 0.0
                active = [v.strip() == "Active" for v in rec[5:9]]
                rows.append({"t": ts + frac, "sm": float(rec[1]), "sm_max": float(rec[2]),
                             "power": float(rec[3]) if rec[3].strip() not in ("[N/A]", "") else None,
                             "hw_slowdown": active[0], "hw_thermal": active[1],
                             "sw_thermal": active[2], "sw_power_cap": active[3]})
            except (ValueError, IndexError):
                continue
        return rows


def summarize_clocks(samples: list[dict], t0: float, t1: float) -> dict:
    inside = [s for s in samples if t0 - 0.15 <= s["t"] <= t1 + 0.15]
    if not inside and samples:
        inside = [min(samples, key=lambda s: abs(s["t"] - (t0 + t1) / 2))]
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
    reasons = sorted({k for s in inside for k in ("hw_slowdown", "hw_thermal", "sw_thermal", "sw_power_cap") if s[k]})
    return {"sm_mhz": statistics.median(s["sm"] for s in inside), "sm_max_mhz": max(s["sm_max"] for s in inside),
            "reasons": reasons, "samples": len(inside)}


def gpu_id_for_nvsmi() -> str | None:
    import torch

    try:
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", None)
        dev = getattr(props, "pci_device_id", None)
        if bus is not None and dom is not None and dev is not None:
            return f"{dom:08X}:{bus:02X}:{dev:02X}.0"
    except Exception:  # noqa: BLE001 - best effort; fall back to the visible index
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    return vis.split(",")[torch.cuda.current_device()] if vis else None


# ----------------------------------------------------------------------------- traffic record


def kernel_fingerprint(variant: str) -> str:
    """Hash of the sources the dominant kernel is built from (invalidates stale ncu traffic)."""
    csrc = os.path.join(ROOT, "online_softmax_dispatcher_gb300", "csrc")
    files = {"rowgroup": ("k_rowgroup.cuh",), "block": ("k_block.cu",), "block_tma": ("k_tma.cu",),
             "stream": ("k_stream.cu", "stream_passes.cuh"), "splitk": ("k_splitk.cu",),
             "splitk_grid": ("k_grid.cu", "split_parts.cuh", "stream_passes.cuh"),
             "splitk_wide": ("k_wide.cu", "stream_passes.cuh"),
             "layernorm": ("k_norm.cuh",), "rmsnorm": ("k_norm.cuh",), "backward": ("k_bwd.cu",),
             "masked": ("k_masked.cu",)}
    h = hashlib.sha256()
    for name in files.get(variant, ()) + ("common.cuh", "tma.cuh", "launch.h"):
        p = os.path.join(csrc, name)
        if name and os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, variant: str, plan: dict) -> tuple[float | None, str]:
    """dram bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source with the same launch plan.  `workload` is the record's
    key: the workload's name for its default forward softmax, name:op for the
    other operations (name:ws for the forward with a workspace)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None, "no ncu record"
    if not rec or rec.get("variant") != variant:
        return None, "no ncu record for this kernel"
    if rec.get("fingerprint") != kernel_fingerprint(variant) or rec.get("plan") != plan:
        return None, "kernel or launch plan changed since the ncu capture"
    return float(rec["dram_bytes_per_launch"]), rec.get("source", "")


# ----------------------------------------------------------------------------- CPU oracle timing


def alibi_mask(causal_q: int, cols: int):
    """The --mask bias as float64: -0.05 x |query position - key| for the
    causal_q queries of a block (query i sits at key cols - causal_q + i)."""
    import numpy as np

    qi = np.arange(causal_q, dtype=np.float64)[:, None] + (cols - causal_q)
    kj = np.arange(cols, dtype=np.float64)[None, :]
    return -0.05 * np.abs(qi - kj)


def oracle_pass(w, op: str, rows: int, mask: bool = False):
    """(one oracle pass of `op` over the first `rows` rows of w, bytes it
    stands for, oracle).  Inputs are prepared outside the pass.  The bytes are
    those the GPU line counts for the same op (masked: the visible part of x,
    all of y, and the --mask bias once)."""
    import numpy as np

    import oracle
    from online_softmax_dispatcher_gb300 import workloads as W

    o = oracle.default()
    x = W.generate(w, rows=rows)
    dt = w.dtype_code
    nbytes = w.bytes_moved(rows)
    if op == "backward":
        y = o.softmax(x, dt)
        dy = np.random.default_rng(0).standard_normal(y.shape)
        return (lambda: o.softmax_bwd_f64(y, dy)), nbytes // 2 * 3, o
    if op == "masked":
        q = min(512, w.rows)
        esz = nbytes // (2 * rows * w.cols)
        nbytes = (masked_visible_elems(rows, w.cols, q) + rows * w.cols) * esz
        m = None
        if mask:
            m = W._round_to(alibi_mask(q, w.cols), w.dtype)
            nbytes += m.size * esz
        return (lambda: o.softmax_masked(x, dt, 0.125, m, q)), nbytes, o
    if op == "norm":
        g, b = W.norm_params(w)
        return (lambda: o.norm_f64(w.kind, x, dt, g, b, w.eps)), nbytes, o
    return (lambda: o.softmax(x, dt)), nbytes, o


def time_oracle(w, op: str, sample_rows: int, reps: int, budget_s: float, mask: bool = False) -> dict:
    """The oracle (fp64, OpenMP over rows) on the first sample_rows rows."""
    one, nbytes, o = oracle_pass(w, op, sample_rows, mask)
    one()  # warm
    times = []
    t_all = time.perf_counter()
    for _ in range(reps):
        t = time.perf_counter()
        one()
        times.append(time.perf_counter() - t)
        if time.perf_counter() - t_all > budget_s:
            break
    per = statistics.median(times)
    return {"value": nbytes / per / 1e9, "unit": "GB/s", "cores": o.num_threads(),
            "kind": "oracle", "sample": f"{op} on the first {sample_rows} of {w.rows} rows, "
                                        f"median of {len(times)} passes",
            "seconds_per_pass": per, "passes": len(times)}


def oracle_sample_rows(w, target_elems: int = 1 << 25) -> int:
    return max(1, min(w.rows, target_elems // w.cols))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline_leg(w, op: str, mask: bool = False) -> dict:
    """The oracle on all host cores (the sample of oracle_sample_rows), then on
    one core over a smaller sample; both as GB/s of the same algorithmic bytes."""
    import oracle

    res = time_oracle(w, op, oracle_sample_rows(w), reps=5, budget_s=20.0, mask=mask)
    o = oracle.default()
    all_cores = o.num_threads()
    o.set_num_threads(1)
    try:
        one = time_oracle(w, op, oracle_sample_rows(w, 1 << 22), reps=3, budget_s=15.0, mask=mask)
    finally:
        o.set_num_threads(all_cores)
    res["one_core"] = {"value": one["value"], "unit": "GB/s", "cores": 1, "sample": one["sample"],
                       "seconds_per_pass": one["seconds_per_pass"]}
    res["host_cpu"] = {"model": cpu_model(), "os_cpu_count": os.cpu_count()}
    return res


def masked_visible_elems(rows: int, cols: int, causal_q: int) -> int:
    """Elements of x the causal masked softmax must read: row r sees keys
    j <= r % causal_q + (cols - causal_q)."""
    if causal_q <= 0:
        return rows * cols
    per_q = [min(cols, max(0, i + (cols - causal_q) + 1)) for i in range(causal_q)]
    full, rest = divmod(rows, causal_q)
    return full * sum(per_q) + sum(per_q[:rest])


# ----------------------------------------------------------------------------- GPU arm


def find_workload(W, args):
    """The workload named by --workload (softmax or normalisation workloads);
    --op norm defaults to the first normalisation workload."""
    if args.shape:
        rows, cols, dt = args.shape.split(",")
        if dt not in W.DTYPE_CODES:
            raise SystemExit(f"--shape dtype must be one of {list(W.DTYPE_CODES)}")
        return W.Workload(f"shape_{dt}_{int(rows)}x{int(cols)}", int(rows), int(cols), dt, "normal1", 99,
                          f"{dt} [{int(rows)}, {int(cols)}], N(0, 1) (an ad-hoc shape)")
    name = args.workload
    if args.op == "norm":
        if name == DEFAULT_WORKLOAD:
            name = next(iter(W.NORM_WORKLOADS))
        if name not in W.NORM_WORKLOADS:
            raise SystemExit(f"--op norm needs one of {list(W.NORM_WORKLOADS)}")
        return W.NORM_WORKLOADS[name]
    if name not in W.WORKLOADS:
        raise SystemExit(f"unknown workload {name}; softmax workloads: {list(W.WORKLOADS)}")
    return W.WORKLOADS[name]


def run_ours(args, rank: int, ws: int) -> dict | None:
    import torch

    import online_softmax_dispatcher_gb300 as osd
    from online_softmax_dispatcher_gb300 import workloads as W

    w = find_workload(W, args)
    if args.rows is not None:
        w = dataclasses.replace(w, rows=min(args.rows, w.rows))
    dev = torch.device("cuda")
    x_np = W.generate(w)
    x_host = W.as_torch(x_np, w.dtype).pin_memory()
    set_bytes = w.bytes_moved()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nbuf = max(2, -(-int(2.5 * l2) // set_bytes) + 1)
    xs = [x_host.to(dev) for _ in range(nbuf)]
    ys = [torch.empty_like(xs[0]) for _ in range(nbuf)]
    plan = osd.plan_for(xs[0], ys[0])
    variant = osd.softmax_variant_name(plan.variant)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    rows, cols, dt = w.rows, w.cols, w.dtype_code
    ptrs = [(a.data_ptr(), b.data_ptr()) for a, b in zip(xs, ys)]
    fwd = osd.lib().softmax_fwd
    # the same step through the public Python API, for the e2e figure:
    # (host inputs copied in each step, api(device inputs, device output))
    api_inputs = [x_host]

    def api(dev_in, out, i=0):
        osd.softmax(dev_in[0], out=out)

    if args.op == "norm":
        g_np, b_np = W.norm_params(w)
        gt = W.as_torch(g_np, w.dtype).to(dev) if g_np is not None else None
        bt = W.as_torch(b_np, w.dtype).to(dev) if b_np is not None else None
        gp = gt.data_ptr() if gt is not None else 0
        bp = bt.data_ptr() if bt is not None else 0
        variant = "layernorm" if w.kind == 0 else "rmsnorm"
        rc, plan = osd.norm_plan(osd.softmax_device_query()[1], w.kind, ptrs[0][0], ptrs[0][1], rows, cols, dt,
                                 gp, bp)
        if rc != 0:
            raise osd.SoftmaxError(rc)
        ln, rms = osd.lib().layernorm_fwd, osd.lib().rmsnorm_fwd

        def step(i):
            xp, yp = ptrs[i % nbuf]
            if w.kind == 0:
                rc = ln(xp, yp, rows, cols, dt, gp or None, bp or None, w.eps, None, None, s)
            else:
                rc = rms(xp, yp, rows, cols, dt, gp or None, w.eps, None, s)
            if rc != 0:
                raise osd.SoftmaxError(rc)

        def api(dev_in, out, i=0):
            if w.kind == 0:
                osd.layer_norm(dev_in[0], gt, bt, eps=w.eps, out=out)
            else:
                osd.rms_norm(dev_in[0], gt, eps=w.eps, out=out)
    elif args.op == "backward":
        # y = softmax(x) (our forward), dy ~ N(0, 1); each step writes dx
        for a, b in zip(xs, ys):
            osd.softmax(a, out=b)
        dys = [torch.randn(xs[0].shape, device=dev).to(xs[0].dtype) for _ in range(nbuf)]
        dxs = [torch.empty_like(xs[0]) for _ in range(nbuf)]
        ptrs3 = [(b.data_ptr(), d.data_ptr(), o.data_ptr()) for b, d, o in zip(ys, dys, dxs)]
        set_bytes = set_bytes // 2 * 3
        bwd = osd.lib().softmax_bwd
        variant = "backward"
        rc, plan = osd.softmax_bwd_plan(osd.softmax_device_query()[1], *ptrs3[0], rows, cols, dt)
        if rc != 0:
            raise osd.SoftmaxError(rc)
        api_inputs = [ys[0].cpu().pin_memory(), dys[0].cpu().pin_memory()]

        def api(dev_in, out, i=0):
            osd.softmax_backward(dev_in[0], dev_in[1], out=out)

        def step(i):
            yp, dyp, dxp = ptrs3[i % nbuf]
            rc = bwd(yp, dyp, dxp, rows, cols, dt, s)
            if rc != 0:
                raise osd.SoftmaxError(rc)
    elif args.op == "masked":
        masked = osd.lib().softmax_fwd_masked
        causal_q = min(512, rows)
        variant = "masked"
        # the bytes the method must move: the visible part of x (keys past the
        # causal limit are never read), all of y
        esz = set_bytes // (2 * rows * cols)
        set_bytes = masked_visible_elems(rows, cols, causal_q) * esz + rows * cols * esz
        mask_t, mp, mrows = None, None, 0
        if args.mask:
            # an ALiBi-style additive bias, -0.05 x the query-key distance, one
            # row per query of the block (read by every block: counted once)
            mask_t = W.as_torch(W._round_to(alibi_mask(causal_q, cols), w.dtype), w.dtype).to(dev).contiguous()
            mp, mrows = mask_t.data_ptr(), causal_q
            set_bytes += mask_t.numel() * mask_t.element_size()
        rc, plan = osd.softmax_masked_plan(osd.softmax_device_query()[1], ptrs[0][0], ptrs[0][1], rows, cols, dt)
        if rc != 0:
            raise osd.SoftmaxError(rc)

        def api(dev_in, out, i=0):
            osd.softmax_masked(dev_in[0].view(-1, causal_q, cols), scale=0.125, mask=mask_t, causal=True,
                               out=out.view(-1, causal_q, cols))

        def step(i):
            xp, yp = ptrs[i % nbuf]
            rc = masked(xp, yp, rows, cols, dt, 0.125, mp, mrows, causal_q, s)
            if rc != 0:
                raise osd.SoftmaxError(rc)
    elif args.workspace:
        rc, need = osd.softmax_workspace_size(ptrs[0][0], ptrs[0][1], rows, cols, dt)
        if rc != 0:
            raise osd.SoftmaxError(rc)
        wss = [torch.empty(max(need, 16), dtype=torch.uint8, device=dev) for _ in range(nbuf)]
        wptrs = [(a, b, t.data_ptr()) for (a, b), t in zip(ptrs, wss)]
        fwd_ws = osd.lib().softmax_fwd_ws
        if need:
            variant = "splitk_wide"
            plan = osd.plan_for(xs[0], ys[0], "splitk_wide")

        def api(dev_in, out, i=0):
            osd.softmax(dev_in[0], out=out, workspace=wss[i])  # one workspace per step in flight

        def step(i):
            xp, yp, wp = wptrs[i % nbuf]
            rc = fwd_ws(xp, yp, rows, cols, dt, wp, need, s)
            if rc != 0:
                raise osd.SoftmaxError(rc)
    elif args.variant is not None:
        vcode = osd.VARIANTS[args.variant]
        rc, plan = osd.softmax_plan(osd.softmax_device_query()[1], ptrs[0][0], ptrs[0][1], rows, cols, dt, vcode)
        if rc != 0:
            return {"metric": METRIC, "impl": "ours", "unsupported": f"variant {args.variant}: "
                    f"{osd.softmax_strerror(rc)}", "config": {"workload": w.name, "variant": args.variant}}
        variant = args.variant
        fwd_v = osd.lib().softmax_fwd_variant

        def api(dev_in, out, i=0):
            osd.softmax(dev_in[0], out=out, variant=args.variant)

        def step(i):
            xp, yp = ptrs[i % nbuf]
            rc = fwd_v(xp, yp, rows, cols, dt, vcode, s)
            if rc != 0:
                raise osd.SoftmaxError(rc)
    else:
        def step(i):
            xp, yp = ptrs[i % nbuf]
            rc = fwd(xp, yp, rows, cols, dt, s)
            if rc != 0:
                raise osd.SoftmaxError(rc)

    # the clock sampler starts (and settles) before the warm-up steps, so
    # that the timed region follows the warm-up with no idle gap: an idle
    # GPU takes its first launch back at 1.5 - 3x the time of the next ones
    sampler = ClockSampler(gpu_id_for_nvsmi()).start() if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # ---- timed region: K steps
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(ws)
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, ws)
    samples = sampler.stop() if sampler is not None else []
    clocks = summarize_clocks(samples, t_host0, t_host1)

    # ---- single-launch latency (cold: each launch on the next buffer set)
    lat = []
    for i in range(min(200, max(20, args.steps))):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(i)
        b.record(stream)
        b.synchronize()
        lat.append(a.elapsed_time(b) * 1e3)
    latency_us = statistics.median(lat)

    # ---- e2e through the public API: every step copies its inputs from pinned
    # host memory to the device, runs the op and copies its output back to
    # pinned host memory.  Two steps are in flight on two streams with their
    # own buffers (a step's device->host copy overlaps the next step's
    # host->device copy: the two directions of the host link run at once).
    e2e_streams = [torch.cuda.Stream() for _ in range(2)]
    dev_ins = [[t.to(dev) for t in api_inputs] for _ in range(2)]
    out_devs = [torch.empty_like(xs[0]) for _ in range(2)]
    y_hosts = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    ke = max(4, min(args.steps, 30))

    def e2e_step(k):
        i = k % 2
        with torch.cuda.stream(e2e_streams[i]):
            for d, h in zip(dev_ins[i], api_inputs):
                d.copy_(h, non_blocking=True)
            api(dev_ins[i], out_devs[i], i)
            y_hosts[i].copy_(out_devs[i], non_blocking=True)

    for k in range(4):
        e2e_step(k)
    torch.cuda.synchronize()
    barrier(ws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for st in e2e_streams:
        st.wait_event(a)
    for k in range(ke):
        e2e_step(k)
    for st in e2e_streams:
        stream.wait_stream(st)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / ke, ws)
    y_host = y_hosts[0]

    total_bytes = sum_over_ranks(float(set_bytes) * args.steps, ws)
    value = total_bytes / (ms_max / 1e3) / 1e9
    peaks = load_peaks()
    per_launch_ms = ms / args.steps
    achieved = set_bytes / (per_launch_ms / 1e3) / 1e9
    rec_key = f"{w.name}:ws" if args.workspace else (w.name if args.op == "forward" else f"{w.name}:{args.op}")
    if args.op == "masked" and args.mask:
        rec_key += "+mask"
    traffic, tsrc = recorded_traffic(rec_key, variant, plan.as_dict())
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "rows": w.rows, "cols": w.cols, "about": w.about, "op": args.op,
                   "entry": {"norm": "layernorm_fwd" if getattr(w, "kind", 0) == 0 else "rmsnorm_fwd",
                             "backward": "softmax_bwd", "masked": "softmax_fwd_masked"}.get(
                                 args.op, "softmax_fwd_ws" if args.workspace else "softmax_fwd"),
                   "variant": variant, "plan": plan.as_dict(),
                   "l2": f"rotating {nbuf} buffer sets, {nbuf * set_bytes / 2**20:.0f} MiB > 2x L2 "
                         f"({l2 / 2**20:.0f} MiB)",
                   "pct_of_peak": round(100 * value / ws / RATED_HBM_GBS, 2),
                   "pct_of_peak_source": RATED_SOURCE,
                   "pct_of_measured_peak": round(100 * value / ws / peaks["hbm_gbs"], 2),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "latency_us": round(latency_us, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": f"{peaks['source']} hbm_gbs (copy of 1 Gi bf16)",
                     "frac_of_rated": round(achieved / RATED_HBM_GBS, 4), "rated_source": RATED_SOURCE,
                     "algorithmic_bytes_per_launch": set_bytes,
                     "traffic": traffic, "traffic_source": tsrc},
        "e2e": {"value": round(set_bytes / (e2e_ms / 1e3) / 1e9 * ws, 2), "unit": "GB/s",
                "pipeline": "2 steps in flight on 2 streams",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in api_inputs),
                "d2h_bytes_per_step": y_host.numel() * y_host.element_size(), "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": args.steps * (2 if variant == "splitk_wide" else 1),
        "clocks": clocks,
    }
    if args.op == "masked":
        res["roofline"]["algorithmic_bytes_note"] = (
            "visible x (keys past the causal limit are never read) + all of y"
            + (" + the additive mask once" if args.mask else ""))
        res["config"]["mask"] = "ALiBi-style [512, cols], -0.05 x distance" if args.mask else None
    if per_config_wanted(args):
        # free the headline's buffers first: the vocabulary workload needs ~8 GB
        del xs, ys, dev_ins, out_devs
        torch.cuda.empty_cache()
        res["per_config"] = run_per_config(args, ws)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_leg(w, args.op, args.op == "masked" and args.mask)
    return res if rank == 0 else None


def per_config_wanted(args) -> bool:
    return (args.op == "forward" and not args.workspace and args.variant is None and args.rows is None
            and args.shape is None and not args.no_per_config)


def time_forward(w, args, ws: int) -> dict:
    """softmax_fwd on workload w, timed like the headline: W warm-up steps, then
    K steps between barrier + synchronize, CUDA events on the launching stream,
    consecutive steps on rotating buffer sets totalling > 2x L2."""
    import torch

    import online_softmax_dispatcher_gb300 as osd
    from online_softmax_dispatcher_gb300 import workloads as W

    dev = torch.device("cuda")
    x_dev = W.as_torch(W.generate(w), w.dtype).to(dev)
    set_bytes = w.bytes_moved()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nbuf = max(2, -(-int(2.5 * l2) // set_bytes) + 1)
    xs = [x_dev] + [x_dev.clone() for _ in range(nbuf - 1)]
    ys = [torch.empty_like(x_dev) for _ in range(nbuf)]
    plan = osd.plan_for(xs[0], ys[0])
    variant = osd.softmax_variant_name(plan.variant)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    fwd = osd.lib().softmax_fwd
    ptrs = [(a.data_ptr(), b.data_ptr()) for a, b in zip(xs, ys)]

    def step(i):
        xp, yp = ptrs[i % nbuf]
        rc = fwd(xp, yp, w.rows, w.cols, w.dtype_code, s)
        if rc != 0:
            raise osd.SoftmaxError(rc)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms = max_over_ranks(e0.elapsed_time(e1), ws)
    peaks = load_peaks()
    gbs = set_bytes * args.steps * ws / (ms / 1e3) / 1e9
    traffic, tsrc = recorded_traffic(w.name, variant, plan.as_dict())
    out = {"workload": w.name, "rows": w.rows, "cols": w.cols, "dtype": w.dtype, "variant": variant,
           "plan": plan.as_dict(), "ms_per_step": round(ms / args.steps, 5), "value": round(gbs, 2),
           "unit": "GB/s", "frac": round(gbs / ws / peaks["hbm_gbs"], 4),
           "frac_of_rated": round(gbs / ws / RATED_HBM_GBS, 4), "algorithmic_bytes_per_launch": set_bytes,
           "traffic_ratio": round(traffic / set_bytes, 4) if traffic else None, "traffic_source": tsrc,
           "l2": f"rotating {nbuf} buffer sets, {nbuf * set_bytes / 2**20:.0f} MiB"}
    del xs, ys, x_dev
    torch.cuda.empty_cache()
    return out


def run_per_config(args, ws: int) -> dict:
    """Every softmax workload but the headline's, through softmax_fwd, timed
    with the same --steps / --warmup; clocks sampled over the whole set."""
    from online_softmax_dispatcher_gb300 import workloads as W

    rank = int(os.environ.get("RANK", "0"))
    sampler = ClockSampler(gpu_id_for_nvsmi()).start() if rank == 0 else None
    t0 = time.time()
    lines = [time_forward(w, args, ws) for name, w in W.WORKLOADS.items() if name != args.workload]
    t1 = time.time()
    samples = sampler.stop() if sampler is not None else []
    return {"timing": "same --steps/--warmup as the headline, CUDA events, rotating buffers > 2x L2",
            "peak": load_peaks()["hbm_gbs"], "rated_peak": RATED_HBM_GBS, "lines": lines,
            "clocks": summarize_clocks(samples, t0, t1)}


def run_reference(args, rank: int, ws: int) -> dict | None:
    if rank != 0:
        return None
    from online_softmax_dispatcher_gb300 import workloads as W

    w = find_workload(W, args)
    rows = oracle_sample_rows(w, target_elems=1 << 23)
    one, nbytes, o = oracle_pass(w, args.op, rows, args.op == "masked" and args.mask)
    for _ in range(max(0, min(args.warmup, 3))):
        one()
    t = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt_s = (time.perf_counter() - t) / max(1, args.steps)
    value = nbytes / dt_s / 1e9
    sample = f"each step: {args.op} on the first {rows} of {w.rows} rows of {w.name}"
    config = {"workload": w.name, "rows": w.rows, "cols": w.cols, "about": w.about, "op": args.op,
              "reference": "fp64 CPU oracle (OpenMP over rows) standing in for the pages' method"}
    if args.op == "masked":
        config["mask"] = "ALiBi-style [512, cols], -0.05 x distance" if args.mask else None
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt_s * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--shape", default=None, metavar="ROWS,COLS,DTYPE",
                    help="an ad-hoc softmax shape instead of --workload: N(0, 1) inputs of that shape and dtype "
                         "(fp32, fp16, bf16), for sweeps and per-kernel profiles")
    ap.add_argument("--rows", type=int, default=None,
                    help="time only the first ROWS rows of the workload (for small profiling captures)")
    ap.add_argument("--op", choices=("forward", "backward", "masked", "norm"), default="forward",
                    help="backward times softmax_bwd (dx = y*(dy - sum dy*y)) on the workload's shape, "
                         "bytes = rows*cols*(2 reads + 1 write); masked times softmax_fwd_masked with scale 1/8 "
                         "and a causal cut over query blocks of 512 rows (attention scores [B, H, 512, cols]); "
                         "norm times layernorm_fwd / rmsnorm_fwd on a normalisation workload "
                         "(ln_fp16_131040x192, ln_fp16_32760x384, rms_bf16_16384x4096)")
    ap.add_argument("--mask", action="store_true",
                    help="with --op masked: add an additive ALiBi-style bias (-0.05 x query-key distance, one "
                         "row per query of a 512-row block), which the general masked kernel serves")
    ap.add_argument("--workspace", action="store_true",
                    help="forward through softmax_fwd_ws with a workspace the bench allocates (lets few, very "
                         "long rows use every SM)")
    ap.add_argument("--variant", default=None,
                    help="forward only: force this kernel (rowgroup, block, block_tma, stream, splitk, "
                         "splitk_grid) through softmax_fwd_variant instead of the dispatcher's choice; a variant "
                         "that cannot serve the shape prints an 'unsupported' line and exits 0")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config lines (the forward softmax of every other softmax workload)")
    args = ap.parse_args()
    if args.shape is not None and args.op == "norm":
        ap.error("--shape is for the softmax operations (norm workloads are named by --workload)")
    if args.mask and args.op != "masked":
        ap.error("--mask applies to --op masked")
    if args.variant is not None and (args.op != "forward" or args.workspace):
        ap.error("--variant applies to the forward softmax without --workspace")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, ws, _ = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, rank, ws)
    else:
        import __graft_entry__

        if rank == 0 or ws == 1:
            __graft_entry__.build()
        barrier(ws)
        res = run_ours(args, rank, ws)
    if res is not None:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
