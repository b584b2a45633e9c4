"""Throughput benchmark of the chunkwise (Gated) DeltaNet path on GB300.

One step = one pass of the hot path over one batch of synthetic input resident in
HBM: the Gated DeltaNet forward (L2 norm, gate cumsum, Gram + UT solve, W/U, state
scan, output, final state) on the workload B4 H16 T8192 d128 bf16 with an initial
state, chunk 64 — or, with --workload, another workload of
chunkwise_delta_rule_02_gb300.workloads (the forward+backward one runs the
forward and the backward per step; two forward workloads take chunk 32, one of
them head dim 256).

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own replica of
the workload on its own GPU (the path shards over sequences and heads with no
exchange), so the value is the tokens of all ranks / the slowest rank's time.

--impl reference times the fp64 CPU oracle (token-by-token recurrence) on the
host cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "delta-rule chunk fwd(+bwd) tokens/s on 1 GB300; % of roofline (tensor/HBM)"
DEFAULT_WORKLOAD = "gdn_fwd_bf16_b4h16t8192d128_h0"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129e6


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def chunk_lengths(w, x):
    """Lengths of every chunk of one head: the chunks of each sequence, the last one
    possibly partial (chunks never cross a sequence)."""
    C = w.chunk
    if x["cu_seqlens"] is not None:
        cu = [int(t) for t in x["cu_seqlens"].tolist()]
        lens = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    else:
        lens = [x["q"].shape[2]] * x["q"].shape[0]
    out = []
    for L in lens:
        out += [C] * (L // C) + ([L % C] if L % C else [])
    return out


def chunk_flops_fwd(c: int, dk: int, dv: int) -> int:
    """Counted FLOPs of the forward's dense contractions on one chunk of c rows, as
    dense rectangles: K K^T, Q K^T, T (diag(Gamma) K) (2 c^2 dk each), T V, P Unew
    (2 c^2 dv each), W S, Q S, K~^T Unew (2 c dk dv each), plus the unit-lower-
    triangular inverse (about c^3 / 3 multiply-adds)."""
    return 2 * (3 * c * c * dk + 2 * c * c * dv + 3 * c * dk * dv) + (2 * c ** 3) // 3


def chunk_flops_bwd(c: int, dk: int, dv: int) -> int:
    """Counted FLOPs of the backward's dense contractions on one chunk, as the
    backward kernels run them (recompute included):
      recompute   K K^T, Q K^T, T (Gamma K)  [c^2 dk];  T V  [c^2 dv];  W S, K~^T Unew  [c dk dv];
                  the inverse (c^3 / 3 multiply-adds)
      dS scan     P^T dO  [c^2 dv];  K~ dS, (Gamma Q)^T dO, W^T dUnew  [c dk dv]
      states      dO S_in^T, dUnew S_in^T, Unew dS_out^T  [c dk dv]
      c x c part  K K^T, dW (Gamma K)^T  [c^2 dk];  dUnew V^T, dO Unew^T  [c^2 dv];
                  the inverse's adjoint, two c x c x c products
      c x d part  (dP o D) K, (dP o D)^T Q, T^T dW, (dKK + dKK^T) K  [c^2 dk];  T^T dUnew  [c^2 dv]"""
    return 2 * (9 * c * c * dk + 5 * c * c * dv + 8 * c * dk * dv + 2 * c ** 3) + (2 * c ** 3) // 3


def algorithmic_flops(w, x, backward=False) -> int:
    """Counted FLOPs of one forward (or backward) call over every (sequence, head)."""
    dk, dv = x["q"].shape[-1], x["v"].shape[-1]
    f = chunk_flops_bwd if backward else chunk_flops_fwd
    return x["q"].shape[1] * sum(f(c, dk, dv) for c in chunk_lengths(w, x))


def roofline(abytes: int, flops: int, ms: float, pk: dict, src: str, sustained: bool) -> dict:
    """The slower of the two bounds (compulsory bytes at the measured HBM copy rate,
    counted FLOPs at the measured dense bf16 rate) and the fraction of it reached:
    frac = roofline time / measured time = achieved / peak of the binding bound."""
    tf_key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    tflops = pk.get(tf_key) or FALLBACK_PEAKS[tf_key]
    t_hbm = abytes / (pk["hbm_gbs"] * 1e9)
    t_flop = flops / (tflops * 1e12)
    secs = ms / 1000.0
    if t_hbm >= t_flop:
        r = {"bound": "hbm", "achieved": abytes / secs / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": flops / secs / 1e12, "peak": tflops, "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r.update({"hbm_time_us": t_hbm * 1e6, "tensor_time_us": t_flop * 1e6,
              "hbm_frac": t_hbm / secs, "tensor_frac": t_flop / secs,
              "algorithmic_bytes_per_launch": int(abytes), "flops_per_launch": int(flops),
              "peak_source": src + (" (HBM copy; bf16 %s)" % ("sustained" if sustained else "burst"))})
    return r


def algorithmic_bytes(w, x) -> int:
    """Compulsory HBM bytes of one forward: read q, k, v, beta (input dtype), g (fp32),
    h0 (fp32 state); write o (input dtype) and the final state (fp32)."""
    es = 2 if w.dtype == "bf16" else 4
    tokheads = x["q"].shape[0] * x["q"].shape[1] * x["q"].shape[2]
    d = w.d
    n = tokheads * (3 * d * es + es + d * es)
    if x["g"] is not None:
        n += tokheads * 4
    nstate = x["h0"].numel() * 4 if x["h0"] is not None else 0
    n += nstate                                        # h0 read
    n += (len(x["lengths"]) if x["lengths"] else x["q"].shape[0]) * x["q"].shape[1] * d * d * 4  # hT
    return int(n)


def algorithmic_bytes_bwd(w, x) -> int:
    """Compulsory bytes of one backward: read q, k, v, beta, g, h0, dO, dhT; write
    dq, dk, dv, dbeta, dg, dh0."""
    es = 2 if w.dtype == "bf16" else 4
    tokheads = x["q"].shape[0] * x["q"].shape[1] * x["q"].shape[2]
    d = w.d
    per = (4 * d * es + es) + (3 * d * es + es) + (8 if x["g"] is not None else 0)
    nstate = x["h0"].numel() * 4 if x["h0"] is not None else 0
    return int(tokheads * per + 3 * nstate)


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, read-only
    queries) every millisecond on a host thread, each sample time-stamped, so that
    even a timed region of a few milliseconds holds samples."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.ok = False
        self._stop = False
        self._thread = None
        try:
            import ctypes
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            self.get_reasons = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = (float(mx.value) if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0
                            else None)
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        import ctypes
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            a = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
            b = self.get_reasons(self.h, ctypes.byref(rs))
            if a == 0:
                self.samples.append((time.perf_counter(), float(mhz.value), int(rs.value) if b == 0 else 0))
            time.sleep(0.001)

    def start(self):
        if self.ok:
            import threading
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop = True
            self._thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        """Median SM clock and the reasons seen in the samples taken in [t0, t1]."""
        sel = [s for s in self.samples if t0 <= s[0] <= t1]
        if not sel:
            return None
        reasons = sorted({n for _, _, r in sel for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for _, m, _ in sel), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sel)}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clk", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


SOAK_SECONDS = 0.6   # untimed steps after the timed region, so nvidia-smi's 200 ms samples see load


def run_timed(step, steps: int, stream, barrier, index: int):
    """Time exactly `steps` calls of step() with CUDA events on `stream`, bracketed by
    barrier() (a synchronize) on both sides.  NVML samples the SM clock every
    millisecond from just before to just after the timed region; afterwards untimed
    steps keep the GPU loaded for SOAK_SECONDS while nvidia-smi samples too.
    Returns (per-step milliseconds, clocks record)."""
    import torch
    nv = NvmlSampler(index)
    smi = ClockSampler(index)
    nv.start()
    smi.start()
    time.sleep(0.02)
    barrier()
    t0 = time.perf_counter()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    barrier()
    t1 = time.perf_counter()
    soak_end = t1 + SOAK_SECONDS
    n_soak = 0
    while time.perf_counter() < soak_end:
        step()
        n_soak += 1
        if n_soak % 8 == 0:
            torch.cuda.synchronize()
    barrier()
    t2 = time.perf_counter()
    nv.stop()
    under_load = smi.stop()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    timed = nv.summary(t0, t1)
    clocks = dict(timed) if timed else (dict(under_load) if under_load else {})
    clocks["source"] = "nvml, 1 ms, timed region" if timed else "nvidia-smi, 200 ms"
    clocks["timed_region_s"] = t1 - t0
    clocks["soak"] = {"steps": n_soak, "seconds": t2 - t1,
                      "nvml": nv.summary(t1, t2), "nvidia_smi": under_load}
    return per, clocks


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, pg, device) -> float:
    """The slowest rank's time (every rank runs its own replica; no data exchange)."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_rank: int, world: int, ms: float) -> float:
    """Tokens of all ranks per second of the slowest rank."""
    return tokens_per_rank * world / (ms / 1000.0)


# the translation unit and headers each profiled kernel is built from
KERNEL_SOURCES = {
    "k_coop_fwd": ["coop.cu", "fast.h", "prep_math.cuh", "sm100.cuh", "common.cuh"],
}


def kernel_source_sha(kernel: str) -> str:
    """Hash of the sources `kernel` is compiled from (all of csrc for an unlisted one)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunkwise_delta_rule_02_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(csrc))
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode())
            h.update(f.read())
    with open(os.path.join(ROOT, "include", "gdn.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def record_traffic(csv_path: str, kernel: str, workload: str, capture: str, out: str = None) -> dict:
    """Write profiles/traffic.json's entry for (kernel, workload) from the CSV of an ncu
    capture of one launch (dram__bytes_read.sum, dram__bytes_write.sum), stamped with
    the hash of the kernel's current sources.  Runs on any host (no GPU needed)."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    hdr = next(r for r in rows if "Metric Name" in r)
    start = rows.index(hdr) + 1
    ki, mi, vi = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    got = {}
    for r in rows[start:]:
        if len(r) > vi and kernel in r[ki]:
            got.setdefault(r[mi], float(r[vi].replace(",", "")))
    if "dram__bytes_read.sum" not in got or "dram__bytes_write.sum" not in got:
        raise SystemExit("no dram byte counters for %s in %s" % (kernel, csv_path))
    rd, wr = int(got["dram__bytes_read.sum"]), int(got["dram__bytes_write.sum"])
    p = out or os.path.join(ROOT, "profiles", "traffic.json")
    d = json.load(open(p)) if os.path.exists(p) else {}
    d[kernel + "@" + workload] = {
        "dram_bytes_per_launch": rd + wr, "dram_read": rd, "dram_write": wr,
        "source_sha": kernel_source_sha(kernel),
        "sources": ", ".join(["csrc/" + f for f in KERNEL_SOURCES.get(kernel, [])] + ["include/gdn.h"]),
        "capture": capture}
    with open(p, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")
    return d[kernel + "@" + workload]


STEP_KERNELS = ("k_coop_fwd", "k_bscan_tc", "k_bwd_tc")   # one step of the training path


def record_step_traffic(csv_path: str, workload: str, capture: str, out: str = None) -> dict:
    """Write profiles/traffic.json's entry for one whole forward+backward step: the read +
    write DRAM bytes of one launch of each of STEP_KERNELS in an ncu CSV (exactly one each),
    stamped with the hash of every kernel source ("step@workload")."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    hdr = next(r for r in rows if "Metric Name" in r)
    start = rows.index(hdr) + 1
    ii, ki, mi, vi = hdr.index("ID"), hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    launches = {}   # launch id -> (step kernel, {metric: value})
    for r in rows[start:]:
        if len(r) <= vi:
            continue
        name = next((k for k in STEP_KERNELS if k in r[ki]), None)
        if name is None:
            continue
        launches.setdefault(r[ii], (name, {}))[1][r[mi]] = float(r[vi].replace(",", ""))
    names = sorted(n for n, _ in launches.values())
    if names != sorted(STEP_KERNELS):
        raise SystemExit("need exactly one launch of each of %s in %s, found %s" % (STEP_KERNELS, csv_path, names))
    rd = wr = 0
    for _, m in launches.values():
        if "dram__bytes_read.sum" not in m or "dram__bytes_write.sum" not in m:
            raise SystemExit("no dram byte counters in %s" % csv_path)
        rd += int(m["dram__bytes_read.sum"])
        wr += int(m["dram__bytes_write.sum"])
    p = out or os.path.join(ROOT, "profiles", "traffic.json")
    d = json.load(open(p)) if os.path.exists(p) else {}
    d["step@" + workload] = {
        "dram_bytes_per_launch": rd + wr, "dram_read": rd, "dram_write": wr,
        "source_sha": kernel_source_sha("step"), "sources": "csrc/*, include/gdn.h",
        "kernels": ", ".join(STEP_KERNELS), "capture": capture}
    with open(p, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")
    return d["step@" + workload]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture of this exact kernel source
    (profiles/traffic.json), scaled to the workload; None if absent or stale."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel + "@" + workload)
    if not e or e.get("source_sha") != kernel_source_sha(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def oracle_sample_fwd(x, w, items, nthreads, backward=False):
    """Run the fp64 oracle forward (with backward=True: its backward, which runs the
    forward too) on `items` (sequence, head) pairs of x in one call, the items side by
    side so that every host thread has work; returns (seconds, tokens) where tokens
    counts whole tokens (all heads of a position).  Only the oracle call is timed, not
    the gathering of the items."""
    import numpy as np
    import torch
    import oracle
    H = x["q"].shape[1]
    f = lambda t: None if t is None else t.double().numpy()
    if x["cu_seqlens"] is not None:
        # one packed row, one head, one sequence per item
        cu = x["cu_seqlens"].numpy().astype(np.int64)
        spans = [(int(cu[s]), int(cu[s + 1]), h) for s, h in items]
        cat = lambda t: None if t is None else torch.cat([t[0, h, a:b] for a, b, h in spans])[None, None]
        offs = np.concatenate([[0], np.cumsum([b - a for a, b, _ in spans])]).astype(np.int64)
        h0 = None if x["h0"] is None else torch.stack([x["h0"][s, h] for s, h in items])[:, None]
        args = [f(cat(x[n])) for n in ("q", "k", "v", "beta", "g")]
        t0 = time.perf_counter()
        if backward:
            dhT = None if x.get("dhT") is None else torch.stack([x["dhT"][s, h] for s, h in items])[:, None]
            oracle.bwd(*args, f(h0), f(cat(x["do"])), f(dhT), cu_seqlens=offs, nthreads=nthreads)
        else:
            oracle.fwd(*args, f(h0), cu_seqlens=offs, nthreads=nthreads)
        secs = time.perf_counter() - t0
        return secs, float(offs[-1]) / H
    st = lambda t: None if t is None else torch.stack([t[b, h] for b, h in items])[None]
    args = [f(st(x[n])) for n in ("q", "k", "v", "beta", "g", "h0")]
    t0 = time.perf_counter()
    if backward:
        oracle.bwd(*args, f(st(x["do"])), f(st(x["dhT"])), nthreads=nthreads)
    else:
        oracle.fwd(*args, nthreads=nthreads)
    secs = time.perf_counter() - t0
    return secs, float(x["q"].shape[2]) * len(items) / H


def sample_items(x, n_items):
    if x["cu_seqlens"] is not None:
        N = x["cu_seqlens"].numel() - 1
        H = x["q"].shape[1]
        allitems = [(s, h) for s in range(N) for h in range(H)]
    else:
        allitems = [(b, h) for b in range(x["q"].shape[0]) for h in range(x["q"].shape[1])]
    step = max(1, len(allitems) // n_items)
    return allitems[::step][:n_items]


CPU_BASELINE_MIN_CPU_SECONDS = 10.0   # host threads x wall seconds
CPU_BASELINE_MAX_PASSES = 8
SINGLE_CORE_MIN_SECONDS = 2.0


def host_cpu() -> dict:
    """Architecture and model name of the host CPU (lscpu, else /proc/cpuinfo)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    return {"arch": platform.machine(), "model": model, "logical_cpus": os.cpu_count()}


def cpu_baseline(x, w, budget_items=256):
    """The oracle, as it stands (its backward, which includes the forward, on a
    forward+backward workload), on up to `budget_items` (sequence, head) items of the
    workload (all of them for the bench workloads), repeated until the passes add up to
    about 10 s of host-thread time; plus the same oracle on one host thread, on one
    item, repeated for about 2 s."""
    nthreads = os.cpu_count() or 1
    items = sample_items(x, budget_items)
    secs, tok, passes = 0.0, 0.0, 0
    while passes < CPU_BASELINE_MAX_PASSES and (passes == 0 or
                                                secs * min(nthreads, len(items)) < CPU_BASELINE_MIN_CPU_SECONDS):
        s, t = oracle_sample_fwd(x, w, items, nthreads, backward=w.backward)
        secs += s
        tok += t
        passes += 1
    cores = min(nthreads, len(items))
    s1, t1, p1 = 0.0, 0.0, 0
    while p1 == 0 or s1 < SINGLE_CORE_MIN_SECONDS:
        s, t = oracle_sample_fwd(x, w, items[:1], 1, backward=w.backward)
        s1 += s
        t1 += t
        p1 += 1
    what = "backward (with its forward)" if w.backward else "forward"
    return {"value": tok / secs, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": "fp64 oracle %s on %d of the workload's %d (sequence, head) items, whole "
                      "sequences, in one call over %d host threads, %d pass(es); tokens counted as "
                      "whole tokens (items / heads)" % (what, len(items), len(sample_items(x, 1 << 30)),
                                                        cores, passes),
            "seconds": secs,
            "single_core": {"value": t1 / s1, "unit": "tokens/s", "cores": 1, "seconds": s1,
                            "sample": "the same oracle %s on 1 (sequence, head) item, %d pass(es)"
                                      % (what, p1)},
            "host": host_cpu()}


def run_reference(args, w, x):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    nthreads = os.cpu_count() or 1
    items = sample_items(x, max(nthreads, 8))
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample_fwd(x, w, items[:1], nthreads)
    times, toks = [], 0.0
    for _ in range(args.steps):
        s, t = oracle_sample_fwd(x, w, items, nthreads)
        times.append(s)
        toks = t
    ms = 1000.0 * sum(times) / len(times)
    value = toks / (ms / 1000.0)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "chunk": w.chunk,
                       "pass": "forward", "sample_items": len(items)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(nthreads, len(items)),
                             "kind": "oracle",
                             "sample": "per step: fp64 oracle forward on %d (sequence, head) items "
                                       "of the workload, whole sequences" % len(items)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DECODE_WORKLOAD = "gdn_decode_bf16_n256h16d128"
DECODE_SHAPE = (256, 16, 128)   # sequences, heads, head dim


def decode_inputs():
    """The decode workload's seeded inputs on the host: q, k, v [N,H,d] bf16, beta [N,H]
    bf16, log-gate g [N,H] fp32 and the fp32 state [N,H,d,d]."""
    import torch
    N, H, d = DECODE_SHAPE
    gen = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(N, H, d, generator=gen).to(torch.bfloat16) for _ in range(3))
    beta = torch.sigmoid(torch.randn(N, H, generator=gen)).to(torch.bfloat16)
    g = -torch.nn.functional.softplus(torch.randn(N, H, generator=gen)) / 16
    S = 0.02 * torch.randn(N, H, d, d, generator=gen)
    return q, k, v, beta, g, S


def oracle_decode_step(inputs, nthreads):
    """One decode step of every (sequence, head) by the fp64 oracle (its token loop on
    sequences of length 1, from the given state); returns the seconds it took."""
    import oracle
    f = lambda t: t.double().numpy()
    q, k, v, beta, g, S = (f(t) for t in inputs)
    args = (q[:, :, None], k[:, :, None], v[:, :, None], beta[:, :, None], g[:, :, None], S)
    t0 = time.perf_counter()
    oracle.fwd(*args, nthreads=nthreads)
    return time.perf_counter() - t0


def decode_cpu_baseline(inputs):
    """The oracle's decode step on all of the workload's items, repeated until the
    passes add up to about 10 s of host-thread time."""
    nthreads = os.cpu_count() or 1
    N, H, _ = DECODE_SHAPE
    secs, passes = 0.0, 0
    while passes < 64 and (passes == 0 or secs * nthreads < CPU_BASELINE_MIN_CPU_SECONDS):
        secs += oracle_decode_step(inputs, nthreads)
        passes += 1
    return {"value": N * passes / secs, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": "fp64 oracle decode step of all %d sequences x %d heads over %d host threads, "
                      "%d pass(es)" % (N, H, nthreads, passes),
            "seconds": secs}


def run_reference_decode(args):
    """The reference arm on the decode workload: the oracle's decode step on the host,
    rank 0 only."""
    rank, _, _ = dist_env()
    if rank != 0:
        return
    inputs = decode_inputs()
    nthreads = os.cpu_count() or 1
    N, H, d = DECODE_SHAPE
    for _ in range(min(max(args.warmup, 0), 1)):
        oracle_decode_step(inputs, nthreads)
    times = [oracle_decode_step(inputs, nthreads) for _ in range(args.steps)]
    ms = 1000.0 * sum(times) / len(times)
    value = N / (ms / 1000.0)
    line = {"metric": "recurrent decode step tokens/s on 1 GB300; % of HBM roofline",
            "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": DECODE_WORKLOAD, "N": N, "H": H, "d": d},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                             "sample": "per step: fp64 oracle decode step of all %d sequences x %d heads"
                                       % (N, H)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_decode(args):
    """Recurrent decode step (one token for each of 256 sequences x 16 heads, d = 128,
    bf16, gated, state updated in place): tokens/s and the HBM roofline of its
    compulsory bytes (the fp32 state read and written, q, k, v, beta, g in, o out)."""
    import torch
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    rank, world, local = dist_env()
    N, H, d = DECODE_SHAPE
    host_inputs = decode_inputs()
    q, k, v, beta, g, S = (t.clone() for t in host_inputs)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    qd, kd, vd, bd, gd, Sd = (t.to(dev) for t in (q, k, v, beta, g, S))
    o = torch.empty(N, H, d, dtype=torch.bfloat16, device=dev)
    shape = binding.make_shape(qd.view(N, H, 1, d), vd.view(N, H, 1, d))
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.gdn_decode_step(shape, qd, kd, vd, bd, gd, Sd, Sd, o, stream)

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        step()
    barrier()
    per, clocks = run_timed(step, args.steps, stream, barrier, local)
    ms = max_over_ranks(sum(per) / len(per), pg, dev)
    if rank == 0:
        pk, src = peaks()
        nbytes = N * H * (2 * d * d * 4 + 4 * d * 2 + 2 + 4)
        achieved = nbytes / (ms / 1000.0) / 1e9
        line = {"metric": "recurrent decode step tokens/s on 1 GB300; % of HBM roofline",
                "value": N * world / (ms / 1000.0), "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": DECODE_WORKLOAD, "N": N, "H": H, "d": d,
                           "l2": "no flush: the 268 MB state read and written per step > 129 MB L2"},
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                             "frac": achieved / pk["hbm_gbs"], "traffic": None, "kernel": "k_decode",
                             "algorithmic_bytes_per_launch": nbytes, "peak_source": src},
                "clocks": clocks, "e2e": None, "gpu_launches": args.steps}
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = decode_cpu_baseline(host_inputs)
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="write profiles/traffic.json's entry for --workload from this ncu CSV and exit")
    ap.add_argument("--capture", default="", help="with --record-traffic: the ncu command that made the CSV")
    args = ap.parse_args()

    if args.record_traffic:
        from chunkwise_delta_rule_02_gb300 import workloads
        if workloads.WORKLOADS[args.workload].backward:
            print(json.dumps(record_step_traffic(args.record_traffic, args.workload, args.capture)))
        else:
            print(json.dumps(record_traffic(args.record_traffic, "k_coop_fwd", args.workload, args.capture)))
        return

    if args.workload == DECODE_WORKLOAD:
        if args.impl == "ours":
            run_decode(args)
        else:
            run_reference_decode(args)
        return
    import torch
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]
    x = workloads.generate(w)
    rank, world, local = dist_env()

    if args.impl == "reference":
        run_reference(args, w, x)
        return

    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    shape = gdn.make_shape(d["q"], d["v"], w.chunk, d["cu_seqlens"])
    # fwd+bwd: the training step keeps the forward's per-chunk operands for the backward
    # (gdn_chunk_fwd_save / gdn_chunk_bwd_saved) where the library has that path
    saved = None
    if w.backward and binding.dn_saved_size(shape) > 0:
        saved = torch.empty(binding.dn_saved_size(shape), dtype=torch.uint8, device=dev)
    ws = binding.alloc_workspace(shape, w.backward, dev)
    wsb = binding.alloc_workspace(shape, 2, dev) if saved is not None else None
    o = torch.empty_like(d["v"])
    N = shape.num_seqs if d["cu_seqlens"] is not None else w.B
    hT = torch.empty((N, w.H, w.d, w.d), dtype=torch.float32, device=dev)
    if w.backward:
        grads = dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]), dv=torch.empty_like(d["v"]),
                     dbeta=torch.empty_like(d["beta"]), dg=torch.empty_like(d["g"]),
                     dh0=torch.empty_like(d["h0"]))
    stream = torch.cuda.current_stream(dev)
    fast = binding.dn_uses_fast_path(shape, False) == 1

    def step():
        if saved is not None:
            binding.gdn_chunk_fwd_save(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], o, hT, saved,
                                       ws, stream)
            binding.gdn_chunk_bwd_saved(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["do"], d["dhT"],
                                        saved, grads["dq"], grads["dk"], grads["dv"], grads["dbeta"],
                                        grads["dg"], grads["dh0"], wsb, stream)
            return
        if d["g"] is None:
            binding.dn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["h0"], o, hT, ws, stream)
        else:
            binding.gdn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], o, hT, ws,
                                  stream)
        if w.backward:
            binding.gdn_chunk_bwd(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["do"],
                                  d["dhT"], grads["dq"], grads["dk"], grads["dv"], grads["dbeta"],
                                  grads["dg"], grads["dh0"], ws, stream)

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        step()
    barrier()
    if binding.dn_device_status(ws, stream) != binding.DN_OK or (
            wsb is not None and binding.dn_device_status(wsb, stream) != binding.DN_OK):
        raise RuntimeError("device status error after warm-up")

    per, clocks = run_timed(step, args.steps, stream, barrier, local)
    ms = max_over_ranks(sum(per) / len(per), pg, dev)
    tokens = w.tokens
    value = whole_job_value(tokens, world, ms)

    # end to end through the host-buffer entry point (forward workloads)
    e2e = None
    if not w.backward:
        hx = {k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("q", "k", "v", "beta", "g", "h0")
                  else v) for k, v in x.items()}
        ho = torch.empty(x["v"].shape, dtype=x["v"].dtype).pin_memory()
        hhT = torch.empty((N, w.H, w.d, w.d), dtype=torch.float32).pin_memory()
        arena = torch.empty(binding.dn_host_arena_size(shape, hx["g"] is not None, hx["h0"] is not None),
                            dtype=torch.uint8, device=dev)

        def e2e_step():
            binding.gdn_chunk_fwd_host(shape, hx["q"], hx["k"], hx["v"], hx["beta"], hx["g"], hx["h0"], ho,
                                       hhT, arena, ws, stream)
        for _ in range(2):
            e2e_step()
        barrier()
        n_e2e = max(3, min(args.steps, 10))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        t1.record(stream)
        barrier()
        ms_e2e = t0.elapsed_time(t1) / n_e2e
        h2d = sum(hx[k].numel() * hx[k].element_size() for k in ("q", "k", "v", "beta", "g", "h0")
                  if hx[k] is not None)
        d2h = ho.numel() * ho.element_size() + hhT.numel() * hhT.element_size()
        e2e = {"value": tokens * world / (ms_e2e / 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e}
    elif saved is not None:
        # the training step end to end: its inputs (q, k, v, beta, g, h0, dO, dhT) from
        # pinned host buffers, the forward and backward through the public calls, o, h_T
        # and every gradient back to pinned host buffers, inside the timed region
        names_in = ("q", "k", "v", "beta", "g", "h0", "do", "dhT")
        hx = {k: x[k].pin_memory() for k in names_in}
        outs_d = [o, hT] + [grads[k] for k in ("dq", "dk", "dv", "dbeta", "dg", "dh0")]
        outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs_d]

        def e2e_step():
            for k in names_in:
                d[k].copy_(hx[k], non_blocking=True)
            step()
            for hd, dd in zip(outs_h, outs_d):
                hd.copy_(dd, non_blocking=True)
        for _ in range(2):
            e2e_step()
        barrier()
        n_e2e = max(3, min(args.steps, 10))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        t1.record(stream)
        barrier()
        ms_e2e = t0.elapsed_time(t1) / n_e2e
        h2d = sum(hx[k].numel() * hx[k].element_size() for k in names_in)
        d2h = sum(t.numel() * t.element_size() for t in outs_h)
        e2e = {"value": tokens * world / (ms_e2e / 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e}

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return

    pk, src = peaks()
    abytes = algorithmic_bytes(w, x) + (algorithmic_bytes_bwd(w, x) if w.backward else 0)
    flops = algorithmic_flops(w, x) + (algorithmic_flops(w, x, backward=True) if w.backward else 0)
    path, launches_per_step = binding.dn_plan(shape, False)
    kname = {binding.DN_PATH_COOP: "k_coop_fwd", binding.DN_PATH_FUSED: "k_fast_fwd"}.get(path, "general_fwd")
    bwd_desc = ""
    if w.backward and saved is not None:
        launches_per_step += binding.dn_plan(shape, 2)[1]
        bwd_desc = ("; the forward keeps every chunk's operands and states (gdn_chunk_fwd_save, %.2f GB);"
                    " backward from them (gdn_chunk_bwd_saved): the reverse scan, tcgen05 per-chunk gradients"
                    % (saved.numel() / 1e9))
    elif w.backward:
        nb = binding.dn_plan(shape, True)[1]
        launches_per_step += nb
        coop_bwd = nb == 3 + (2 if d["cu_seqlens"] is not None else 0)
        bwd_desc = ("; backward: the cooperative forward re-run writing every chunk's operands and"
                    " states, the reverse scan over them, tcgen05 per-chunk gradients" if coop_bwd else
                    "; backward: recompute, reverse scan and per-chunk kernels")
    if w.backward:
        # the timed region is the whole step: the forward plus the backward's kernels
        kdesc = "whole forward+backward step (%d kernels)" % launches_per_step
    else:
        kdesc = kname if fast else "whole step (general kernels)"
    # a single forward kernel is timed back to back on its own (burst tensor peak); the
    # forward+backward step is a sequence of kernels (sustained tensor peak)
    roof = roofline(abytes, flops, ms, pk, src, sustained=w.backward)
    roof["traffic"] = recorded_traffic("step", w.name) if w.backward else recorded_traffic(kname, w.name)
    roof["kernel"] = kdesc
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "chunk": w.chunk,
                       "pass": "forward+backward" if w.backward else "forward",
                       "path": {binding.DN_PATH_COOP: "cooperative tcgen05 kernel",
                                binding.DN_PATH_FUSED: "fused tcgen05 kernel per (sequence, head)"}.get(
                                    path, "general fp32 kernels")
                               + bwd_desc,
                       "l2": "no flush: inputs %.2f GB per step > 129 MB L2" % (abytes / 1e9),
                       "parallelism": "replicas over ranks" if world > 1 else "single GPU"},
            "roofline": roof, "clocks": clocks, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x, w)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
