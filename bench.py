"""Benchmark of the B300 selective-scan library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--all] [--no-others] [--no-cpu]

Prints ONE JSON line.  A step is one call of the library over one batch of the
workload (inputs resident in HBM).  The headline workload is the largest one
that fits one GPU: the long-sequence scan (batch 1, 5120 channels, L = 131072,
N = 16, bf16 I/O, fp32 state, z gate, D skip, last_state; the chunked path).
The Mamba-130M layer scan, the Vision Mamba bidirectional scan and the VMamba
SS2D scan are measured the same way and reported under "workloads", each with
its own roofline, end-to-end and CPU-oracle figures.  --all adds the other
measured paths (fused Conv1D, windowed orders, decode, DWConv, backward passes)
under "more"; --workload NAME prints one workload's line alone.

Timing: W untimed warm-up steps, then K steps between a barrier and a device
synchronisation on each side, timed with CUDA events on the launching stream;
each call is also bracketed by its own events to give the kernels' average
duration for the roofline.  Inputs rotate over several copies whose total size
exceeds the 126 MB L2, so every step reads cold data.  SM clocks and throttle
reasons are sampled through NVML during the timed region.

Multi-GPU: the scan shards over batch and channels with no exchange, so each
rank runs an independent replica (weak scaling); value = all ranks' elements /
the slowest rank's time.

--impl reference times the float64 CPU oracle (the only other arm: the pages
ship no code) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import re
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from selective_state_space_120_b300 import workloads as wk  # noqa: E402

METRIC = "selective-scan Gelem/s (B·D·L) and achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "Gelem/s"
L2_BYTES = 126 * 2 ** 20
FALLBACK_HBM_GBS = 6400.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "ncu_traffic.json")
CSRC = os.path.join(ROOT, "selective_state_space_120_b300", "csrc")

WORKLOADS = {w.name: w for w in wk.ALL + (wk.MAMBA_LAYER_CONV, wk.MAMBA_LAYER_UNALIGNED,
                                           wk.VMAMBA_SS2D_14, wk.LOCAL_WIN, wk.LONG_SEQ_PROFILE)}
HEADLINE = wk.LONG_SEQ
# the other workloads of the target set, one compact record each
TARGETS = (wk.MAMBA_LAYER, wk.VIM_BIDIR, wk.VMAMBA_SS2D)
# further measured paths (--all)
EXTRA = (wk.MAMBA_LAYER_CONV, wk.MAMBA_LAYER_UNALIGNED, wk.VMAMBA_SS2D_14, wk.LOCAL_WIN)


# ------------------------------------------------------------------ accounting
def algorithmic_bytes(wl: wk.Workload) -> int:
    """Bytes a step must move at least: every input element read once, the
    output written once (and last_state if returned).  B/C are shared by the
    channels of a group, so they count once per (batch, direction, group)."""
    es = 2 if wl.io == "bf16" else 4
    per_chan = wl.batch * wl.dim * wl.L * es
    n = per_chan * (1 + wl.K)                     # u, Delta per direction
    if wl.with_z:
        n += per_chan                             # z
    n += per_chan                                 # out
    n += 2 * wl.batch * wl.K * wl.G * wl.N * wl.L * es   # B, C
    n += wl.K * wl.dim * (wl.N + 2) * 4           # A, D, delta_bias
    if wl.last_state:
        n += wl.batch * wl.K * wl.dim * wl.N * 4
    return n


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code, comments removed and whitespace runs
    collapsed: it keys the committed ncu traffic figures, which a change of code
    (not of a comment or of layout) invalidates."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            code = " ".join(_COMMENT.sub(" ", fh.read()).split())
        h.update(f.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def ncu_traffic(wl: wk.Workload):
    """DRAM bytes per launch of the workload's dominant kernel from the committed
    ncu summary, or None if absent or taken on different kernel sources."""
    return ncu_traffic_named(wl.name)


def ncu_traffic_named(name: str):
    try:
        with open(PROFILE_TRAFFIC) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    ent = rec.get("workloads", {}).get(name)
    return None if ent is None else ent.get("dram_bytes_per_launch")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks
_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class _Nvml:
    """Minimal NVML reader through ctypes (libnvidia-ml ships with the driver):
    SM clock, its maximum, and the active clock-event (throttle) reasons."""

    def __init__(self, index: int):
        import ctypes.util
        lib = None
        for name in ("libnvidia-ml.so.1", ctypes.util.find_library("nvidia-ml")):
            if not name:
                continue
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise OSError("libnvidia-ml not found")
        self.lib = lib
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("nvmlDeviceGetHandleByIndex failed")
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons_fn = fn or lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self) -> int:
        v = ctypes.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(v)) != 0:  # NVML_CLOCK_SM
            raise OSError("nvmlDeviceGetClockInfo failed")
        return int(v.value)

    def sm_max_mhz(self) -> int:
        v = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(v)) != 0:
            raise OSError("nvmlDeviceGetMaxClockInfo failed")
        return int(v.value)

    def reasons(self) -> int:
        v = ctypes.c_ulonglong()
        if self._reasons_fn(self.h, ctypes.byref(v)) != 0:
            raise OSError("clock event reasons query failed")
        return int(v.value)


class ClockSampler:
    """Samples the SM clock and the clock-event reasons through NVML in a thread
    while the timed region runs (reading only; no GPU setting is changed)."""

    def __init__(self, index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._thr = None
        try:
            self._nv = _Nvml(index)
            self.max_mhz = self._nv.sm_max_mhz()
        except Exception as e:  # noqa: BLE001 -- clocks are reported as unavailable
            self._nv = None
            self.error = f"{type(e).__name__}: {e}"

    def _sample(self):
        self.samples.append(self._nv.sm_mhz())
        self.reasons |= self._nv.reasons()

    def _run(self):
        while True:
            try:
                self._sample()
            except Exception as e:  # noqa: BLE001
                self.error = f"{type(e).__name__}: {e}"
            if self._stop.wait(self.period):
                break

    def __enter__(self):
        if self._nv is not None:
            self._thr = threading.Thread(target=self._run, daemon=True)
            self._thr.start()
        return self

    def __exit__(self, *exc):
        if self._thr is not None:
            self._stop.set()
            self._thr.join()

    def summary(self):
        if self._nv is None or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"],
                    "samples": 0, "error": self.error}
        names = [n for bit, n in _REASONS.items() if self.reasons & bit]
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(self.samples)}


# ------------------------------------------------------------------ GPU arm
class Runner:
    """Holds device inputs of one workload (several rotating copies) and issues
    one library call per step through the C ABI with prebuilt arguments."""

    def __init__(self, wl: wk.Workload, device, seed: int = 0):
        import torch
        import selective_state_space_120_b300 as ss
        from selective_state_space_120_b300 import _binding as b
        self.wl, self.dev = wl, device
        self.lib = b.load()
        inp = wk.make_inputs(wl, seed=seed)
        self.host = inp
        t = {n: self._to_dev(getattr(inp, n)) for n in
             ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "conv_w", "conv_b")}
        set_bytes = algorithmic_bytes(wl)
        self.copies = max(2, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
        self.copies = min(self.copies, 8)
        self.sets = []
        for i in range(self.copies):
            s = {k: (None if v is None else (v if i == 0 else v.clone())) for k, v in t.items()}
            s["out"] = torch.empty_like(s["u"])
            s["last"] = (torch.empty(wl.batch, wl.K, wl.dim, wl.N, dtype=torch.float32,
                                     device=device) if wl.last_state else None)
            self.sets.append(s)
        self.stream = torch.cuda.current_stream(device)
        self.ws = None
        conv_w, conv_b = self.sets[0]["conv_w"], self.sets[0]["conv_b"]
        self.opts = b.options(0, b.SS_SCAN_CONV_SILU if wl.conv else 0, None,
                              None if conv_w is None else conv_w.data_ptr(),
                              None if conv_b is None else conv_b.data_ptr())
        if wl.orders:
            wsb = int(self.lib.ss_multi_scan_workspace_bytes(wl.batch, wl.dim, wl.H, wl.W, wl.K))
            self.ords = (ctypes.c_int * wl.K)(*wl.orders)
        else:
            kind = {1: b.SS_KIND_SCAN, 2: b.SS_KIND_BIDIR, 4: b.SS_KIND_CROSS2D}[wl.K]
            wsb = int(self.lib.ss_workspace_bytes_opts(kind, wl.batch, wl.dim, wl.L, wl.N,
                                                       ctypes.byref(self.opts)))
        if wsb:
            self.ws = torch.empty(wsb, dtype=torch.uint8, device=device)
        self.args = [self._args(s) for s in self.sets]
        self.launches_per_step = self._launches()
        self._ss = ss

    @staticmethod
    def _to_dev(a):
        import torch
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def _args(self, s):
        wl = self.wl
        p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        io = 1 if wl.io == "bf16" else 0
        st = ctypes.c_void_p(self.stream.cuda_stream)
        ws = p(self.ws)
        wsb = 0 if self.ws is None else self.ws.numel()
        if wl.orders:
            return (self.lib.ss_multi_scan_fwd,
                    (wl.batch, wl.dim, wl.H, wl.W, wl.K, self.ords, wl.win, wl.N, wl.G, io,
                     p(s["u"]), p(s["delta"]), p(s["A"]), p(s["B"]), p(s["C"]), p(s["D"]),
                     p(s["delta_bias"]), 1, p(s["z"]), p(s["out"]), p(s["last"]), ws, wsb, st))
        if wl.K == 1:
            return (self.lib.ss_selective_scan_fwd_opts,
                    (wl.batch, wl.dim, wl.L, wl.N, wl.G, io, p(s["u"]), p(s["delta"]), p(s["A"]),
                     p(s["B"]), p(s["C"]), p(s["D"]), p(s["z"]), p(s["delta_bias"]), 1,
                     p(s["out"]), p(s["last"]), ws, wsb, ctypes.byref(self.opts), st))
        if wl.K == 2:
            return (self.lib.ss_bidir_scan_fwd,
                    (wl.batch, wl.dim, wl.L, wl.N, wl.G, io, p(s["u"]), p(s["delta"]), p(s["A"]),
                     p(s["B"]), p(s["C"]), p(s["D"]), p(s["z"]), p(s["delta_bias"]), 1,
                     p(s["out"]), p(s["last"]), ws, wsb, st))
        return (self.lib.ss_cross_scan2d_fwd,
                (wl.batch, wl.dim, wl.H, wl.W, wl.N, wl.G, io, p(s["u"]), p(s["delta"]),
                 p(s["A"]), p(s["B"]), p(s["C"]), p(s["D"]), p(s["delta_bias"]), 1, p(s["z"]),
                 p(s["out"]), p(s["last"]), ws, wsb, st))

    def _launches(self):
        """Kernels one step launches: 1 on the direct path; 3 on the chunked
        long-sequence path (two passes and the carry); 2 for a bidirectional call
        through its workspace (the two directions over one accumulator, or the
        direction pair and its merge over rows read through a view); 3 for SS2D
        (the transposed copy, the four directions, the merge); for an any-order
        call, one permuted copy of u per base traversal other than the row order,
        one launch per two directions and the merge."""
        if self.wl.orders:
            bases = {0 if o in (0, 2) else 1 if o in (1, 3) else 2 if o in (4, 6) else 3
                     for o in self.wl.orders}
            return len(bases - {0}) + (self.wl.K + 1) // 2 + 1
        if self.ws is None:
            return 1
        return {1: 3, 2: 2, 4: 3}[self.wl.K]

    def step(self, i: int):
        fn, args = self.args[i % self.copies]
        st = fn(*args)
        if st != 0:
            from selective_state_space_120_b300 import _binding as b
            b.check(st)

    def timed(self, steps: int, warmup: int, barrier=None):
        import torch
        for i in range(warmup):
            self.step(i)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if barrier:
            barrier()
        torch.cuda.synchronize()
        with ClockSampler(torch.cuda.current_device()) as clk:
            t0.record(self.stream)
            for i in range(steps):
                ev[i][0].record(self.stream)
                self.step(warmup + i)
                ev[i][1].record(self.stream)
            t1.record(self.stream)
            torch.cuda.synchronize()
        if barrier:
            barrier()
        self._ss.device_status()
        total_ms = t0.elapsed_time(t1)
        kern_ms = [a.elapsed_time(b) for a, b in ev]
        return total_ms, float(np.mean(kern_ms)), clk.summary()

    def e2e(self, steps: int, warmup: int):
        """Same metric through the public call with the step's inputs copied from
        pinned host memory and the output read back, every step.  The steps are
        pipelined over two device buffer sets and three streams: the host->device
        copies of step i+1 and the read-back of step i-1 overlap the call of step
        i (PCIe carries both directions at once); every step still moves all its
        inputs in and its output out."""
        import torch
        nb = 2
        sets = self.sets[:nb]
        names = [n for n in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
                 if sets[0][n] is not None]
        host = {n: sets[0][n].cpu().pin_memory() for n in names}
        outs_h = [torch.empty(sets[0]["out"].shape, dtype=sets[0]["out"].dtype).pin_memory()
                  for _ in range(nb)]
        has_last = sets[0]["last"] is not None
        lasts_h = [torch.empty(sets[0]["last"].shape, dtype=torch.float32).pin_memory()
                   for _ in range(nb)] if has_last else None
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = outs_h[0].numel() * outs_h[0].element_size()
        if has_last:
            d2h += lasts_h[0].numel() * 4
        s_in = torch.cuda.Stream(self.dev)
        s_out = torch.cuda.Stream(self.dev)
        s_cmp = self.stream
        ev_in = [torch.cuda.Event() for _ in range(nb)]
        ev_cmp = [torch.cuda.Event() for _ in range(nb)]
        ev_out = [torch.cuda.Event() for _ in range(nb)]

        def run(n, t0=None, t1=None):
            for i in range(n):
                b = i % nb
                with torch.cuda.stream(s_in):
                    if i == 0 and t0 is not None:
                        t0.record(s_in)
                    if i >= nb:
                        s_in.wait_event(ev_cmp[b])   # the call that last read buffer b is done
                    for name in names:
                        sets[b][name].copy_(host[name], non_blocking=True)
                    ev_in[b].record(s_in)
                s_cmp.wait_event(ev_in[b])
                if i >= nb:
                    s_cmp.wait_event(ev_out[b])      # buffer b's last output has been read back
                self.step(b)
                ev_cmp[b].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[b])
                    outs_h[b].copy_(sets[b]["out"], non_blocking=True)
                    if has_last:
                        lasts_h[b].copy_(sets[b]["last"], non_blocking=True)
                    ev_out[b].record(s_out)
                    if i == n - 1 and t1 is not None:
                        t1.record(s_out)

        run(max(warmup, nb))
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        run(steps, t0, t1)
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        return {"value": self.wl.elems / (ms * 1e-3) / 1e9, "unit": UNIT,
                "ms_per_step": ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "3 streams, 2 buffer sets"}


# ------------------------------------------------------------------ CPU oracle arm
_OS: dict = {}  # the oracle sample's inputs, in the process that computes rows


def _oracle_sample_workload(wl: wk.Workload) -> wk.Workload:
    """A reduced copy of the workload: one batch entry and as many channels as
    keep the host arrays near 4 M elements, with the same per-row shape and
    recipe."""
    dim = min(wl.dim, max(wl.G, ((1 << 22) // wl.L) // wl.G * wl.G))
    return wk.scaled(wl, wl.name + "_oracle_sample", batch=1, dim=dim)


def _oracle_sample_init(wl: wk.Workload):
    """Builds the sample's inputs (seeded, so every process holds the same)."""
    import oracle
    small = _oracle_sample_workload(wl)
    inp = wk.make_inputs(small, seed=0)
    if wl.orders:
        # the library's SS_DIR_* codes in the oracle's numbering
        lib_to_oracle = {0: oracle.ORDER_FWD, 1: oracle.ORDER_COL, 2: oracle.ORDER_REV,
                         3: oracle.ORDER_COL_REV, 4: oracle.ORDER_WIN, 5: oracle.ORDER_WIN_COL,
                         6: oracle.ORDER_WIN_REV, 7: oracle.ORDER_WIN_COL_REV}
        orders = tuple(lib_to_oracle[o] for o in wl.orders)
    else:
        orders = {1: (oracle.ORDER_FWD,), 2: (oracle.ORDER_FWD, oracle.ORDER_REV),
                  4: oracle.SS2D_ORDERS}[wl.K]
    _OS.clear()
    _OS.update(wl=wl, small=small, orders=orders,
               HW=(wl.H, wl.W) if (wl.K == 4 or wl.orders) else (1, wl.L),
               **{n: inp.as_f64(n) for n in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")})


def _oracle_sample_ready(_):
    return bool(_OS)


def _oracle_sample_rows(rows) -> int:
    """Runs the oracle on whole (batch, channel) rows of the sample."""
    import oracle
    S = _OS
    wl, small = S["wl"], S["small"]
    K, dpg = wl.K, small.dim // wl.G
    H, W = S["HW"]
    u, dl, A, B, C, D, z, bias = (S[n] for n in ("u", "delta", "A", "B", "C", "D", "z",
                                                 "delta_bias"))
    for b, d in rows:
        g = d // dpg
        sel = [k * small.dim + d for k in range(K)]
        oracle.scan(u[b:b + 1, d:d + 1], dl[b:b + 1, :, d:d + 1], A[sel],
                    B[b:b + 1, :, g:g + 1], C[b:b + 1, :, g:g + 1],
                    None if D is None else D[sel], None if z is None else z[b:b + 1, d:d + 1],
                    bias[sel], True, S["orders"], H=H, W=W, win=wl.win)
    return len(rows)


class OracleSampler:
    """Times the float64 oracle, as it stands, on whole (batch, channel) rows of a
    workload: in this process (processes = 1), or over a pool of spawned worker
    processes, each with its own copy of the sample's inputs (threads would
    serialise on the Python work around each row's call into the C oracle).
    Only the rows' computation is timed, not the workers' start."""

    def __init__(self, wl: wk.Workload, processes: int | None = None):
        import oracle
        oracle.build()
        self.wl = wl
        self.n = processes or os.cpu_count() or 1
        small = _oracle_sample_workload(wl)
        self.rows = [(0, d) for d in range(small.dim)]
        self.pool = None
        if self.n == 1:
            _oracle_sample_init(wl)
        else:
            import multiprocessing as mp
            self.pool = mp.get_context("spawn").Pool(self.n, _oracle_sample_init, (wl,))
            self.pool.map(_oracle_sample_ready, range(4 * self.n), chunksize=1)

    def run(self, budget_s: float):
        """Rows until about `budget_s` of wall time: (Gelem/s, rows, processes, s)."""
        done = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            batch = [self.rows[(done + i) % len(self.rows)] for i in range(4 * self.n)]
            if self.pool is None:
                done += _oracle_sample_rows(batch)
            else:
                chunks = [batch[i:i + 4] for i in range(0, len(batch), 4)]
                done += sum(self.pool.map(_oracle_sample_rows, chunks, chunksize=1))
        dt = time.perf_counter() - t0
        return done * self.wl.L / dt / 1e9, done, self.n, dt

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
            self.pool = None


def oracle_sample(wl: wk.Workload, budget_s: float = 12.0, processes: int | None = None):
    """One timed sample of the oracle (see OracleSampler)."""
    sampler = OracleSampler(wl, processes)
    try:
        return sampler.run(budget_s)
    finally:
        sampler.close()


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------------ replicas
def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank runs its own replica of the workload
    (the scan shards over batch and channels with no exchange), so the job is
    as fast as its slowest rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(elems_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job throughput in Gelem/s: all ranks' elements over the slowest time."""
    return world * elems_per_rank / (max_ms * 1e-3) / 1e9


# ------------------------------------------------------------------ main
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def config_of(wl: wk.Workload, n_gpus: int, copies: int | None = None):
    c = {"workload": wl.name, "batch": wl.batch, "dim": wl.dim, "seq_len": wl.L,
         "d_state": wl.N, "groups": wl.G, "directions": wl.K, "io_dtype": wl.io,
         "state_dtype": "f32", "z_gate": wl.with_z, "d_skip": wl.with_D,
         "last_state": wl.last_state, "delta_softplus": True,
         "parallelism": f"replicas{n_gpus}" if n_gpus > 1 else "single"}
    if wl.K == 4 or wl.orders:
        c["H"], c["W"] = wl.H, wl.W
    if wl.orders:
        c["orders"] = list(wl.orders)
        c["window"] = wl.win
    if copies:
        c["l2"] = (f"inputs rotate over {copies} copies "
                   f"({copies * algorithmic_bytes(wl) / 1e6:.0f} MB > 126 MB L2)")
    return c


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    wl = WORKLOADS.get(args.workload, HEADLINE)
    steps, warmup = args.steps, args.warmup
    budget = max(1.0, min(20.0, 60.0 / max(1, steps + warmup)))
    vals = []
    info = None
    sampler = OracleSampler(wl)
    try:
        for i in range(warmup + steps):
            v, rows, thr, dt = sampler.run(budget)
            if i >= warmup:
                vals.append(v)
                info = (rows, thr, dt)
    finally:
        sampler.close()
    v = float(np.median(vals))
    rows, thr, dt = info
    sample = (f"whole (batch, channel) rows of the workload (L={wl.L}, N={wl.N}, K={wl.K}), "
              f"{rows} rows in {dt:.1f} s per step, parallel over rows on {thr} processes; "
              f"host CPU {cpu_model()}")
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": wl.elems / (v * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded NumPy PCG64; recipe of the workload)",
            "config": config_of(wl, 1), "impl": "reference",
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def measure_gpu(wl, steps, warmup, barrier=None):
    r = Runner(wl, "cuda")
    total_ms, kern_ms, clocks = r.timed(steps, warmup, barrier)
    return r, total_ms / steps, kern_ms, clocks


DECODE_NAME = "decode_step_b8_d1536_n16"


def measure_decode(steps: int):
    """Token-by-token inference on the Mamba-130M layer shape: one state-update
    call per step (batch 8, dim 1536, N 16, bf16 I/O, fp32 state updated in
    place), over `steps` consecutive tokens with inputs resident in HBM."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = wk.Workload(DECODE_NAME, 8, 1536, steps, N=16)
    inp = wk.make_inputs(wl, 0)
    dev = lambda a: None if a is None else Runner._to_dev(a)  # noqa: E731
    u, dl, A = dev(inp.u), dev(inp.delta[:, 0]), dev(inp.A)
    B, C = dev(inp.B[:, 0]), dev(inp.C[:, 0])
    D, z, bias = dev(inp.D), dev(inp.z), dev(inp.delta_bias)
    # one token per step: per-token slices laid out contiguously
    xs = u.permute(2, 0, 1).contiguous()
    ds = dl.permute(2, 0, 1).contiguous()
    zs = z.permute(2, 0, 1).contiguous()
    Bs = B.permute(3, 0, 1, 2).contiguous()
    Cs = C.permute(3, 0, 1, 2).contiguous()
    state = torch.zeros(wl.batch, wl.dim, wl.N, device="cuda")
    out = torch.empty(wl.batch, wl.dim, dtype=u.dtype, device="cuda")
    def step(k):
        ss.selective_state_update(xs[k], ds[k], A, Bs[k], Cs[k], state, D, zs[k], bias, True,
                                  out=out)
    for k in range(min(3, steps)):
        step(k)
    torch.cuda.synchronize()
    # the steps are captured in a CUDA graph so that the host's per-call cost
    # (argument checks, ctypes) is not what gets timed
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for k in range(steps):
                step(k)
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * steps)
    rows = wl.batch * wl.dim
    # per channel and token: state read + write, A row, x, delta, z, out; B/C per batch
    nbytes = rows * (2 * wl.N * 4 + wl.N * 4 + 4 * 2) + wl.batch * 2 * wl.N * 2
    return {"value": rows / (ms * 1e-3) / 1e9, "unit": "Gelem/s (channel-tokens)",
            "ms_per_step": ms, "kernel_launches_per_step": 1, "bytes_per_step": nbytes,
            "note": "launch-latency bound: the state of a layer (786 KB) stays in L2",
            "config": {"workload": DECODE_NAME, "batch": wl.batch, "dim": wl.dim,
                       "d_state": wl.N, "io_dtype": "bf16", "tokens": steps}}


BWD_NAME = "mamba130m_layer_bwd_b8_d1536_l2048_n16"
# Algorithmic fp32 lane operations of the backward pass (an FMA counts once):
# per element and state, the state recompute (Delta'*A, x*B, the state FMA, the
# readout FMA: 4) and the reverse recurrence (dh FMA, carry, two products for
# the Abar term, dDelta', dA and sum_n dh*B FMAs, dB and dC products and their
# sums over channels: 11); per element about 20 more (softplus, sigmoid, SiLU
# and its derivative, the du, ddelta and dz epilogue).
BWD_OPS_PER_STATE = 15
BWD_OPS_PER_ELEM = 20
FP32_LANES_PER_SM = 128


def bwd_algorithmic_bytes(wl: wk.Workload) -> int:
    """u, delta, z, dout read and du, ddelta, dz written once; B, C read and dB,
    dC (fp32) written once per group; A, D, bias read and their gradients written."""
    es = 2 if wl.io == "bf16" else 4
    per_chan = wl.batch * wl.dim * wl.L * es
    bc = wl.batch * wl.G * wl.N * wl.L
    return 7 * per_chan + 2 * bc * es + 2 * bc * 4 + 2 * wl.dim * (wl.N + 2) * 4


def measure_bwd(steps: int, warmup: int, peak_gbs: float, peak_kind: str):
    """Backward pass of the Mamba-130M layer shape (8 x 1536 x 2048, N = 16,
    bf16 I/O): one ss_selective_scan_bwd call per step on resident inputs,
    rotating over two input sets (each larger than L2)."""
    import torch
    from selective_state_space_120_b300 import _binding as b
    wl = wk.MAMBA_LAYER
    lib = b.load()
    inp = wk.make_inputs(wl, 0)
    dout = wk.make_dout(wl, 0)
    dev = lambda a: None if a is None else Runner._to_dev(a)  # noqa: E731
    base = {"u": dev(inp.u), "delta": dev(inp.delta[:, 0]), "A": dev(inp.A),
            "B": dev(inp.B[:, 0]), "C": dev(inp.C[:, 0]), "D": dev(inp.D), "z": dev(inp.z),
            "bias": dev(inp.delta_bias), "dout": dev(dout)}
    f32 = dict(dtype=torch.float32, device="cuda")
    sets = []
    for i in range(2):
        s = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
        s.update(du=torch.empty_like(s["u"]), ddelta=torch.empty_like(s["u"]),
                 dz=torch.empty_like(s["u"]), dA=torch.empty(wl.dim, wl.N, **f32),
                 dB=torch.empty(wl.batch, wl.G, wl.N, wl.L, **f32),
                 dC=torch.empty(wl.batch, wl.G, wl.N, wl.L, **f32),
                 dD=torch.empty(wl.dim, **f32), dbias=torch.empty(wl.dim, **f32))
        sets.append(s)
    wsb = int(lib.ss_workspace_bytes(b.SS_KIND_SCAN_BWD, wl.batch, wl.dim, wl.L, wl.N))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    st = ctypes.c_void_p(stream.cuda_stream)
    p = lambda t: t.data_ptr()  # noqa: E731
    calls = [(wl.batch, wl.dim, wl.L, wl.N, wl.G, 1, p(s["u"]), p(s["delta"]), p(s["A"]),
              p(s["B"]), p(s["C"]), p(s["D"]), p(s["z"]), p(s["bias"]), 1, p(s["dout"]),
              p(s["du"]), p(s["ddelta"]), p(s["dA"]), p(s["dB"]), p(s["dC"]), p(s["dD"]),
              p(s["dz"]), p(s["dbias"]), p(ws), wsb, st) for s in sets]

    def step(i):
        b.check(lib.ss_selective_scan_bwd(*calls[i % 2]))

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    import selective_state_space_120_b300 as ss
    ss.device_status()
    ms = float(np.mean([a.elapsed_time(c) for a, c in ev]))
    props = torch.cuda.get_device_properties(0)
    max_mhz = 2032
    try:
        max_mhz = _Nvml(torch.cuda.current_device()).sm_max_mhz() or max_mhz
    except Exception:  # noqa: BLE001 -- NVML missing: the B300's maximum SM clock
        pass
    peak_tops = props.multi_processor_count * FP32_LANES_PER_SM * max_mhz * 1e6 / 1e12
    ops = wl.elems * (wl.N * BWD_OPS_PER_STATE + BWD_OPS_PER_ELEM)
    ach = ops / (ms * 1e-3) / 1e12
    alg = bwd_algorithmic_bytes(wl)
    return {"value": wl.elems / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms,
            "kernel_launches_per_step": 1, "memsets_per_step": 5,
            "roofline": {"bound": "alu", "achieved": ach, "peak": peak_tops, "unit": "TFLOP/s",
                         "frac": ach / peak_tops,
                         "peak_source": f"fp32 lane ops: {props.multi_processor_count} SMs x "
                                        f"{FP32_LANES_PER_SM} lanes x {max_mhz} MHz",
                         "ops_per_launch": ops,
                         "hbm_achieved_gbs": alg / (ms * 1e-3) / 1e9,
                         "hbm_frac": alg / (ms * 1e-3) / 1e9 / peak_gbs,
                         "hbm_peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": alg, "traffic": ncu_traffic_named(BWD_NAME)},
            "config": {"workload": BWD_NAME, "batch": wl.batch, "dim": wl.dim,
                       "seq_len": wl.L, "d_state": wl.N, "groups": wl.G, "io_dtype": "bf16",
                       "z_gate": True, "d_skip": True, "delta_softplus": True,
                       "l2": "inputs rotate over 2 copies (201 MB of inputs each > 126 MB L2)"}}


SS2D_BWD_NAME = "vmamba_t_ss2d_bwd_b32_d192_56x56_n16"
WIN_BWD_NAME = "localmamba_win7_bwd_b32_d192_56x56_n16"


def measure_ss2d_bwd(steps: int, warmup: int, peak_gbs: float, peak_kind: str,
                     wl: wk.Workload = wk.VMAMBA_SS2D, name: str = SS2D_BWD_NAME):
    """Backward pass of a four-direction map workload through ss_multi_scan_bwd,
    on resident inputs rotating over two copies: SS2D (32 x 192 x 56 x 56, N = 16,
    bf16, row/column orders and their reverses, no gate), or the same shape with
    LocalMamba's four windowed orders (7 x 7 windows)."""
    import torch
    from selective_state_space_120_b300 import _binding as b
    lib = b.load()
    inp = wk.make_inputs(wl, 0)
    dout = wk.make_dout(wl, 0)
    dev = lambda a: None if a is None else Runner._to_dev(a)  # noqa: E731
    base = {"u": dev(inp.u), "delta": dev(inp.delta), "A": dev(inp.A), "B": dev(inp.B),
            "C": dev(inp.C), "D": dev(inp.D), "bias": dev(inp.delta_bias), "dout": dev(dout)}
    K = wl.K
    f32 = dict(dtype=torch.float32, device="cuda")
    sets = []
    for i in range(2):
        s = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
        s.update(du=torch.empty_like(s["u"]), ddelta=torch.empty_like(s["delta"]),
                 dA=torch.empty(K * wl.dim, wl.N, **f32),
                 dB=torch.empty(wl.batch, K, wl.G, wl.N, wl.L, **f32),
                 dC=torch.empty(wl.batch, K, wl.G, wl.N, wl.L, **f32),
                 dD=torch.empty(K * wl.dim, **f32), dbias=torch.empty(K * wl.dim, **f32))
        sets.append(s)
    wsb = int(lib.ss_multi_scan_bwd_workspace_bytes(wl.batch, wl.dim, wl.H, wl.W, wl.N, K))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    order_list = list(wl.orders) if wl.orders else [0, 1, 2, 3]
    ords = (ctypes.c_int * K)(*order_list)
    window = int(wl.win or 0)
    stream = torch.cuda.current_stream()
    st = ctypes.c_void_p(stream.cuda_stream)
    p = lambda t: t.data_ptr()  # noqa: E731
    calls = [(wl.batch, wl.dim, wl.H, wl.W, K, ords, window, wl.N, wl.G, 1, p(s["u"]), p(s["delta"]),
              p(s["A"]), p(s["B"]), p(s["C"]), p(s["D"]), p(s["bias"]), 1, None, p(s["dout"]),
              p(s["du"]), p(s["ddelta"]), p(s["dA"]), p(s["dB"]), p(s["dC"]), p(s["dD"]), None,
              p(s["dbias"]), p(ws), wsb, st) for s in sets]
    for i in range(warmup):
        b.check(lib.ss_multi_scan_bwd(*calls[i % 2]))
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        b.check(lib.ss_multi_scan_bwd(*calls[i % 2]))
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    import selective_state_space_120_b300 as ss
    ss.device_status()
    ms = float(np.mean([a.elapsed_time(c) for a, c in ev]))
    props = torch.cuda.get_device_properties(0)
    peak_tops = props.multi_processor_count * FP32_LANES_PER_SM * 2032 * 1e6 / 1e12
    ops = wl.elems * K * (wl.N * BWD_OPS_PER_STATE + BWD_OPS_PER_ELEM)
    ach = ops / (ms * 1e-3) / 1e12
    return {"value": wl.elems / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms,
            "kernel_launches_per_step": K + 1, "memsets_per_step": 5,
            "roofline": {"bound": "alu", "achieved": ach, "peak": peak_tops, "unit": "TFLOP/s",
                         "frac": ach / peak_tops,
                         "peak_source": f"fp32 lane ops: {props.multi_processor_count} SMs x "
                                        f"{FP32_LANES_PER_SM} lanes x 2032 MHz",
                         "ops_per_launch": ops, "traffic": ncu_traffic_named(name)},
            "config": {"workload": name, "batch": wl.batch, "dim": wl.dim, "H": wl.H,
                       "W": wl.W, "d_state": wl.N, "directions": K, "io_dtype": "bf16",
                       "z_gate": False, "orders": order_list, "window": window}}


DWCONV_NAME = "vmamba_t_dwconv3x3_b32_d192_56x56"


def measure_dwconv(steps: int, warmup: int, peak_gbs: float, peak_kind: str):
    """The SS2D block's input branch (DWConv 3x3 + SiLU) on the VMamba-T stage-1
    map, 32 x 192 x 56 x 56, bf16: one call per step, rotating over input/output
    copies larger than L2."""
    import torch
    from selective_state_space_120_b300 import _binding as b
    lib = b.load()
    wl = wk.Workload(DWCONV_NAME, 32, 192, 56 * 56, K=4, with_z=False, H=56, W=56, conv2d=True)
    inp = wk.make_inputs(wl, 0)
    x0 = Runner._to_dev(inp.u)
    w = Runner._to_dev(inp.conv2d_w)
    bias = Runner._to_dev(inp.conv2d_b)
    es = 2
    alg = 2 * wl.elems * es + wl.dim * 10 * 4
    copies = max(2, int(np.ceil(3 * L2_BYTES / alg)) + 1)
    xs = [x0 if i == 0 else x0.clone() for i in range(copies)]
    us = [torch.empty_like(x0) for _ in range(copies)]
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    calls = [(wl.batch, wl.dim, wl.H, wl.W, 1, xs[i].data_ptr(), w.data_ptr(), bias.data_ptr(),
              us[i].data_ptr(), st) for i in range(copies)]
    for i in range(warmup):
        b.check(lib.ss_dwconv3x3_silu_fwd(*calls[i % copies]))
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    stream = torch.cuda.current_stream()
    for i in range(steps):
        ev[i][0].record(stream)
        b.check(lib.ss_dwconv3x3_silu_fwd(*calls[(warmup + i) % copies]))
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(c) for a, c in ev]))
    ach = alg / (ms * 1e-3) / 1e9
    return {"value": wl.elems / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms,
            "kernel_launches_per_step": 1,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak_gbs, "unit": "GB/s",
                         "frac": ach / peak_gbs, "peak_source": f"{peak_kind} (copy bandwidth)",
                         "algorithmic_bytes_per_launch": alg, "traffic": ncu_traffic_named(DWCONV_NAME)},
            "config": {"workload": DWCONV_NAME, "batch": wl.batch, "dim": wl.dim, "H": wl.H,
                       "W": wl.W, "io_dtype": "bf16",
                       "l2": f"inputs rotate over {copies} copies ({copies * alg / 1e6:.0f} MB > 126 MB L2)"}}


# Algorithmic work of the forward scan (fp32 lane operations, an FMA counts once;
# SFU operations counted apart): per element, state and direction Delta'*A, x*B,
# the state FMA and the readout FMA (4) and one exponential; per element and
# direction about 10 more (the softplus, Delta'*u, the skip term, the sum over
# directions) and 2 SFU operations (the softplus's exponential and logarithm);
# per element, once, the gate: about 4 lane operations and 2 SFU operations
# (SiLU's exponential and reciprocal).
FWD_OPS_PER_STATE, FWD_OPS_PER_ELEM_DIR, FWD_OPS_GATE = 4, 10, 4
FWD_SFU_PER_STATE, FWD_SFU_PER_ELEM_DIR, FWD_SFU_GATE = 1, 2, 2
# ex2 results per SM and clock: 30 measured on the B300 by a probe of
# independent ex2.approx streams over all 148 SMs (32 nominal).
SFU_LANES_PER_SM = 30


def alu_peaks(max_mhz: int = 2032, sms: int = 148):
    """fp32 lane operations and SFU operations per second at the maximum SM clock."""
    return (sms * FP32_LANES_PER_SM * max_mhz * 1e6 / 1e12, sms * SFU_LANES_PER_SM * max_mhz * 1e6 / 1e12)


def roofline(wl, kern_ms, peak, peak_kind):
    """The forward scan's roofline.  Of its three floors the SFU one binds at
    N = 16 (20 SFU operations per element of a gated single direction at 30 per
    SM and clock, against 78 fp32 lane operations at 128, and 8-13 bytes per
    element of HBM traffic), so `frac` is the SFU fraction; the fp32 and HBM
    fractions sit beside it."""
    alg = algorithmic_bytes(wl)
    ach_gbs = alg / (kern_ms * 1e-3) / 1e9
    elem_dirs = wl.elems * wl.K
    gated = wl.elems if wl.with_z else 0
    ops = elem_dirs * (wl.N * FWD_OPS_PER_STATE + FWD_OPS_PER_ELEM_DIR) + gated * FWD_OPS_GATE
    sfu = elem_dirs * (wl.N * FWD_SFU_PER_STATE + FWD_SFU_PER_ELEM_DIR) + gated * FWD_SFU_GATE
    fp32_peak, sfu_peak = alu_peaks()
    ach_sfu = sfu / (kern_ms * 1e-3) / 1e12
    return {"bound": "alu", "achieved": round(ach_sfu, 3), "peak": round(sfu_peak, 3),
            "unit": "Tops/s", "frac": round(ach_sfu / sfu_peak, 4),
            "peak_source": f"SFU: 148 SMs x {SFU_LANES_PER_SM}/clk x 2032 MHz",
            "fp32_frac": round(ops / (kern_ms * 1e-3) / 1e12 / fp32_peak, 4),
            "hbm_gbs": round(ach_gbs, 1), "hbm_peak": peak,
            "hbm_frac": round(ach_gbs / peak, 4), "traffic": ncu_traffic(wl)}


def cpu_sample(wl, budget_s):
    """The oracle on whole rows of the workload, over worker processes on all cores."""
    v, rows, thr, dt = oracle_sample(wl, budget_s=budget_s)
    return {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"{rows} whole rows (L={wl.L}, K={wl.K}) in {dt:.1f} s"}


def measure_record(wl, steps, warmup, peak, peak_kind, e2e_steps, cpu_s, barrier=None):
    """One workload's compact record: device-resident throughput, the kernels'
    roofline, the end-to-end figure and (cpu_s > 0) the oracle's."""
    import torch
    r, ms, kern_ms, _ = measure_gpu(wl, steps, warmup, barrier)
    e2e = r.e2e(e2e_steps, 3)
    rf = roofline(wl, kern_ms, peak, peak_kind)
    rec = {"value": round(wl.elems / (ms * 1e-3) / 1e9, 3), "ms_per_step": round(ms, 5),
           "kernel_ms": round(kern_ms, 5), "launches_per_step": r.launches_per_step,
           "roofline": {k: rf[k] for k in ("bound", "frac", "fp32_frac", "hbm_frac", "hbm_gbs",
                                          "traffic")},
           "e2e": {"value": round(e2e["value"], 3), "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                   "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]}}
    del r
    torch.cuda.empty_cache()
    if cpu_s > 0:
        c = cpu_sample(wl, cpu_s)
        rec["cpu_baseline"] = {"value": round(c["value"], 5), "cores": c["cores"],
                               "sample": c["sample"]}
    return rec


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=HEADLINE.name,
                    choices=sorted(WORKLOADS) + [BWD_NAME, SS2D_BWD_NAME, WIN_BWD_NAME, DWCONV_NAME],
                    help="workload to time (a non-default one prints its own line only)")
    ap.add_argument("--all", action="store_true",
                    help="also the fused Conv1D, windowed, decode, DWConv and backward lines")
    ap.add_argument("--no-others", action="store_true", help="skip the other target workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--e2e-steps", type=int, default=10)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = dist.barrier
    import selective_state_space_120_b300 as ss
    ss.load_library()

    peak, peak_kind = measured_peaks()
    if args.workload in (DWCONV_NAME, BWD_NAME, SS2D_BWD_NAME, WIN_BWD_NAME):
        # one of the further paths alone, on one GPU per rank (replicas), device-resident inputs
        if args.workload == DWCONV_NAME:
            r = measure_dwconv(args.steps, args.warmup, peak, peak_kind)
            metric, elems = "DWConv3x3+SiLU Gelem/s (B·D·H·W)", 32 * 192 * 56 * 56
        elif args.workload == BWD_NAME:
            r = measure_bwd(args.steps, args.warmup, peak, peak_kind)
            metric, elems = "selective-scan backward Gelem/s (B·D·L)", wk.MAMBA_LAYER.elems
        else:
            bwl = wk.VMAMBA_SS2D if args.workload == SS2D_BWD_NAME else wk.LOCAL_WIN
            r = measure_ss2d_bwd(args.steps, args.warmup, peak, peak_kind, bwl, args.workload)
            metric, elems = "selective-scan backward Gelem/s (B·D·L)", bwl.elems
        ms = max_over_ranks(r["ms_per_step"], world, "cuda")
        if rank == 0:
            line = {"metric": metric, "value": job_value(elems, world, ms), "unit": UNIT,
                    "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded NumPy PCG64)",
                    "config": r["config"], "roofline": r["roofline"],
                    "gpu_launches": args.steps * r["kernel_launches_per_step"]}
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    wl = WORKLOADS[args.workload]
    r, ms, kern_ms, clocks = measure_gpu(wl, args.steps, args.warmup, barrier)
    ms = max_over_ranks(ms, world, "cuda")
    value = job_value(wl.elems, world, ms)
    e2e = r.e2e(args.e2e_steps, 3)
    e2e["value"] *= world
    e2e.pop("ms_per_step", None)
    copies = r.copies
    launches = r.launches_per_step * args.steps
    del r
    torch.cuda.empty_cache()

    default = args.workload == HEADLINE.name
    cpu_s = 0.0 if (args.no_cpu or rank != 0) else 8.0
    others = {}
    if default and not args.no_others:
        for owl in TARGETS:
            try:
                others[owl.name] = measure_record(owl, max(3, min(args.steps, 50)),
                                                  max(3, min(args.warmup, 5)), peak, peak_kind,
                                                  max(3, min(args.e2e_steps, 10)), cpu_s, barrier)
            except Exception as e:  # noqa: BLE001 -- reported, not hidden
                others[owl.name] = {"error": f"{type(e).__name__}: {e}"}
    more = {}
    if default and args.all:
        for owl in EXTRA:
            try:
                r2, oms, okern, _ = measure_gpu(owl, max(3, min(args.steps, 50)), 3, barrier)
                more[owl.name] = {"value": owl.elems / (oms * 1e-3) / 1e9, "ms_per_step": oms,
                                  "launches_per_step": r2.launches_per_step,
                                  "roofline": roofline(owl, okern, peak, peak_kind)}
                del r2
                torch.cuda.empty_cache()
            except Exception as e:  # noqa: BLE001 -- reported, not hidden
                more[owl.name] = {"error": f"{type(e).__name__}: {e}"}
        for name, fn in ((DECODE_NAME, lambda: measure_decode(256)),
                         (DWCONV_NAME, lambda: measure_dwconv(50, 5, peak, peak_kind)),
                         (SS2D_BWD_NAME, lambda: measure_ss2d_bwd(20, 3, peak, peak_kind)),
                         (WIN_BWD_NAME, lambda: measure_ss2d_bwd(20, 3, peak, peak_kind,
                                                                 wk.LOCAL_WIN, WIN_BWD_NAME)),
                         (BWD_NAME, lambda: measure_bwd(30, 3, peak, peak_kind))):
            try:
                more[name] = fn()
                torch.cuda.empty_cache()
            except Exception as e:  # noqa: BLE001 -- reported, not hidden
                more[name] = {"error": f"{type(e).__name__}: {e}"}

    cpu = None
    if cpu_s > 0:
        cpu = cpu_sample(wl, 12.0)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic (seeded NumPy PCG64; recipe of the workload)",
                "config": config_of(wl, world, copies),
                "roofline": roofline(wl, kern_ms, peak, peak_kind),
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
                "kernel_ms": kern_ms}
        if others:
            line["workloads"] = others
        if more:
            line["more"] = more
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
