"""Benchmark of the GB300 fused Compressor (forward + backward step).

One step = csa_compress_fwd + csa_compress_bwd (forward kernel, backward
kernel, dape reduce) over the 256k-token headline workload: ratio 4, coff 2,
head_dim 512, 262144 tokens in 64 segments, capacity = true rows + 1024.
Inputs are seeded synthetic data (workloads.config("headline")) resident in
HBM; kv + score alone are 1 GiB, far above the 129 MB L2, so no flush is
needed between steps.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on
the host cores instead (the reference arm of this repository).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
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
sys.path.insert(0, ROOT)

METRIC = "Compressor fwd/bwd tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
WORKLOAD = ("headline: ratio=4 coff=2 head_dim=512, 262144 tokens in 64 segments "
            "(lengths U{1..8191} renormalised), capacity = true rows + 1024 padding rows")
FALLBACK_HBM_GBS = 6800.0
# GB300's nominal HBM3e bandwidth (about 8 TB/s): the 70% target for the
# forward and the backward is stated against this figure
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 2**20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=262144,
                    help="scale the headline recipe to this many tokens (profiling runs)")
    ap.add_argument("--workload", default="headline",
                    help="another seeded workload instead of the headline: r4d512, r2d128rag, "
                         "r128c1, or a pack `pack-r{ratio}c{coff}d{head_dim}-{n}x{len}`")
    ap.add_argument("--graph", action="store_true",
                    help="also time one forward + backward step captured in a CUDA graph and replayed")
    ap.add_argument("--exact", action="store_true",
                    help="time the exact mode (csa_compress_fwd_exact / csa_compress_bwd_exact; "
                         "windows of at most 8 slots)")
    ap.add_argument("--l2", choices=["auto", "flush", "clean", "warm"], default="auto",
                    help="flush L2 before every call (auto: when kv + score fit in twice the L2); "
                         "clean: the flush write followed by a read of a second buffer twice the L2, "
                         "so the call does not also write back the flush's dirty lines")
    args = ap.parse_args()
    if args.workload not in ("headline", "r4d512", "r2d128rag", "r128c1") and \
            not args.workload.startswith("pack-"):
        ap.error(f"unknown workload {args.workload}")
    return args


def pick_case(args, seed: int, fill: bool = True):
    import workloads
    if args.workload == "headline":
        return headline_case(args.tokens, seed=seed, fill=fill)
    return workloads.config(args.workload, seed=seed, fill=fill)


def headline_case(tokens: int, seed: int, fill: bool = True):
    """The headline workload, or the same recipe scaled to `tokens` tokens."""
    import workloads
    if tokens == 262144:
        return workloads.config("headline", seed=seed, fill=fill)
    nseg = max(1, round(64 * tokens / 262144))
    lens = workloads.headline_seqlens(seed, total=tokens, nseg=nseg)
    return workloads.make_case(f"headline@{tokens}", lens, 4, 2, 512,
                               pad_rows=max(1, round(1024 * tokens / 262144)), seed=seed, fill=fill)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------------ bytes


def algorithmic_bytes(case):
    """Compulsory HBM bytes of one forward and one backward call, per the
    scope table's per-token accounting: every (token, column) element of kv
    and score read once; out written for every capacity row; the backward
    also reads grad_out of the true rows and writes dkv / dscore in full;
    ape read (and dape written) once."""
    T, d, r, coff, C = case.total_tokens, case.head_dim, case.ratio, case.coff, case.capacity
    R = case.true_rows
    ape = r * coff * d * 4
    fwd = T * coff * d * 2 * 2 + C * d * 2 + ape
    bwd = 2 * T * coff * d * 2 * 2 + R * d * 2 + 2 * ape
    return fwd, bwd


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_softmax_kv_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str, units: float) -> dict:
    """Bytes per launch of `kernel_key` from the committed ncu record, scaled to
    this launch's units: {"traffic": DRAM reads + bytes stored into L2, and
    where the record has them "traffic_read" / "traffic_write" /
    "traffic_dram_write_counter"}; {"traffic": None} when the kernel sources
    changed since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel_key]
        if rec["source_hash"] != source_hash(rec["sources"]):
            return {"traffic": None}
        out = {"traffic": rec["dram_bytes_per_unit"] * units}
        if "dram_read_bytes_per_unit" in rec:
            out["traffic_read"] = rec["dram_read_bytes_per_unit"] * units
            out["traffic_write"] = rec["l2_write_bytes_per_unit"] * units
            out["traffic_dram_write_counter"] = rec["dram_write_bytes_per_unit"] * units
        return out
    except Exception:
        return {"traffic": None}


# ------------------------------------------------------------------ clocks


# NVML clock-event reason bits and the names the bench line reports
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes): SM
    clock, maximum SM clock, active clock-event reasons and power draw of one
    device. Nothing here changes a setting of the GPU."""

    CLOCK_SM = 1

    def __init__(self, pci_bus_id=None, index=0):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        h = ctypes.c_void_p()
        rc = -1
        if pci_bus_id:
            rc = lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
        if rc != 0:
            raise RuntimeError("no NVML handle for the device")
        self.h = h
        self._u = ctypes.c_uint()
        self._ull = ctypes.c_ulonglong()
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self):
        return self._uint(self.lib.nvmlDeviceGetClockInfo, self.CLOCK_SM)

    def sm_max_mhz(self):
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.CLOCK_SM)

    def power_w(self):
        if self.lib.nvmlDeviceGetPowerUsage(self.h, self.ct.byref(self._u)) != 0:
            return None
        return self._u.value / 1000.0

    def reasons(self):
        if self._reasons(self.h, self.ct.byref(self._ull)) != 0:
            return None
        return int(self._ull.value)

    def _uint(self, fn, arg):
        if fn(self.h, self.ct.c_int(arg), self.ct.byref(self._u)) != 0:
            return None
        return int(self._u.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock, clock-event reasons and power sampled from a host thread every
    `period_s` (read-only NVML queries) from start() to stop(); mark() and
    unmark() bracket the timed loop, whose samples give the reported median.
    Falls back to `nvidia-smi -lms 50` when NVML cannot be loaded."""

    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, pci_bus_id=None, period_s: float = 0.0005):
        self.index, self.pci, self.period = index, pci_bus_id, period_s
        self.samples = []   # (t, sm_mhz, reasons_mask, power_w)
        self.window = None
        self.nvml = None
        self.thread = None
        self.proc = None
        self.path = None
        self.max_mhz = None

    def start(self):
        import threading
        try:
            self.nvml = _Nvml(self.pci, self.index)
            self.max_mhz = self.nvml.sm_max_mhz()
        except Exception:
            self.nvml = None
        if self.nvml is None:
            self._start_smi()
            return
        self.stop_flag = threading.Event()

        def loop():
            n = 0
            while not self.stop_flag.is_set():
                t = time.perf_counter()
                pw = self.nvml.power_w() if n % 20 == 0 else None
                self.samples.append((t, self.nvml.sm_mhz(), self.nvml.reasons(), pw))
                n += 1
                time.sleep(self.period)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()

    def mark(self):
        self.window = [time.perf_counter(), None]

    def unmark(self):
        if self.window is not None:
            self.window[1] = time.perf_counter()

    def stop(self):
        if self.nvml is None:
            return self._stop_smi()
        self.stop_flag.set()
        self.thread.join(timeout=5)
        self.nvml.close()
        rows = self.samples
        timed = rows
        if self.window is not None and self.window[1] is not None:
            timed = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
        use = timed or rows
        sm = [r[1] for r in use if r[1] is not None]
        reasons = set()
        for r in use:
            if r[2]:
                reasons.update(n for bit, n in NVML_REASONS.items() if r[2] & bit)
        power = [r[3] for r in rows if r[3] is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(rows), "samples_timed": len(timed),
                "sm_mhz_min_timed": min(sm) if sm else None,
                "period_ms": self.period * 1e3, "source": "NVML (read-only queries, host thread)",
                "power_w_max": max(power) if power else None}

    def _start_smi(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.SMI_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def _stop_smi(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "source": "nvidia-smi -lms 50",
                "power_w_max": max(power) if power else None}


def pci_bus_id(dev_index: int):
    """NVML-style PCI bus id of a CUDA device (domain:bus:device.0), or None."""
    try:
        import torch
        pr = torch.cuda.get_device_properties(dev_index)
        return "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle


def oracle_rate(case, budget_s: float = 12.0, min_tokens: int = 16384):
    """Tokens/s of the CPU oracle (fp32 fwd + bwd, all host cores) on a prefix
    of the workload's segments sized from a short calibration run, and the
    single-thread rate on the calibration prefix."""
    import numpy as np
    import oracle
    import workloads

    oracle.build()
    cores = os.cpu_count() or 1

    def sub_case(tokens):
        lens, acc = [], 0
        for L in case.seqlens:
            take = int(min(L, tokens - acc))
            if take <= 0:
                break
            lens.append(take)
            acc += take
        pad = max(0, round(1024 * acc / case.total_tokens))
        return workloads.make_case("sample", lens, case.ratio, case.coff, case.head_dim,
                                   pad_rows=pad, seed=1)

    def run(c, nthreads=cores):
        p = oracle.Problem(c.cu_seqlens, c.cu_seqlens_comp, c.total_tokens, c.capacity,
                           c.ratio, c.coff, c.head_dim)
        t0 = time.perf_counter()
        oracle.fwd32(p, c.kv, c.score, c.ape, nthreads=nthreads)
        oracle.bwd32(p, c.kv, c.score, c.ape, c.grad_out, nthreads=nthreads)
        return time.perf_counter() - t0

    cal = sub_case(min_tokens)
    t_cal = run(cal)
    per_token = t_cal / cal.total_tokens
    tokens = int(min(case.total_tokens, max(min_tokens, budget_s / per_token)))
    sample = sub_case(tokens)
    # when the whole workload takes less than the budget, repeat it until
    # about that much CPU time has been measured
    t = run(sample)
    passes = 1
    while t < 0.8 * budget_s and passes < 64:
        t += run(sample)
        passes += 1
    # the calibration prefix once more on a single thread, beside its all-cores time
    t1 = run(cal, nthreads=1)
    single = {"value_1thread": cal.total_tokens / t1,
              "sample_1thread": f"first {len(cal.seqlens)} segments ({cal.total_tokens} tokens), "
                                f"O32 fwd + bwd: one thread {t1:.2f} s, all {cores} cores {t_cal:.2f} s"}
    return passes * sample.total_tokens / t, cores, (
        f"first {len(sample.seqlens)} segments of the workload ({sample.total_tokens} tokens, "
        f"{sample.capacity} rows incl. proportional padding), O32 fwd + bwd, "
        f"{passes} pass{'es' if passes > 1 else ''}, {t:.1f} s"), single


# ------------------------------------------------------------------ arms


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return 0
    import oracle
    import workloads

    case = headline_case(args.tokens, seed=0, fill=False)
    steps, warm = args.steps, args.warmup
    oracle.build()
    cores = os.cpu_count() or 1
    # one calibration, then a per-step sample sized so that the whole run ends in ~2 minutes
    cal = workloads.make_case("cal", case.seqlens[:1], 4, 2, 512, seed=2)
    p = oracle.Problem(cal.cu_seqlens, cal.cu_seqlens_comp, cal.total_tokens, cal.capacity, 4, 2, 512)
    t0 = time.perf_counter()
    oracle.fwd32(p, cal.kv, cal.score, cal.ape)
    oracle.bwd32(p, cal.kv, cal.score, cal.ape, cal.grad_out)
    per_token = (time.perf_counter() - t0) / cal.total_tokens
    per_step_s = max(0.02, 120.0 / max(1, steps + warm))
    tokens = int(max(64, min(case.total_tokens, per_step_s / per_token)))
    lens, acc = [], 0
    for L in case.seqlens:
        take = int(min(L, tokens - acc))
        if take <= 0:
            break
        lens.append(take)
        acc += take
    sample = workloads.make_case("ref", lens, 4, 2, 512, pad_rows=max(0, round(1024 * acc / case.total_tokens)),
                                 seed=3)
    sp = oracle.Problem(sample.cu_seqlens, sample.cu_seqlens_comp, sample.total_tokens, sample.capacity,
                        4, 2, 512)

    def step():
        oracle.fwd32(sp, sample.kv, sample.score, sample.ape)
        oracle.bwd32(sp, sample.kv, sample.score, sample.ape, sample.grad_out)

    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    value = sample.total_tokens * steps / el
    desc = (f"per step: first {len(lens)} segments of the headline workload ({sample.total_tokens} tokens), "
            f"O32 fwd + bwd on all {cores} host cores")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": desc},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class Ranks:
    """Ranks of a torchrun job (one process per GPU, replicas of the workload):
    a barrier and the max of a value over ranks through a process group when
    WORLD_SIZE > 1, no-ops for a single process."""

    def __init__(self, rank: int, world: int, backend: str = "nccl", device=None):
        self.rank, self.world, self.backend, self.device = rank, world, backend, device
        self.dist = None
        if world > 1:
            import torch.distributed as dist
            if not dist.is_initialized():
                kw = {"device_id": device} if backend == "nccl" and device is not None else {}
                dist.init_process_group(backend, **kw)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        where = self.device if self.backend == "nccl" else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=where)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def run_e2e(args, case, dev, stream, ranks):
    """Pipelined end-to-end loop through the C ABI (see the call site)."""
    import numpy as np
    import torch

    import gated_softmax_kv_gb300 as gsk

    T, C, r, coff, d = case.total_tokens, case.capacity, case.ratio, case.coff, case.head_dim

    def pinned(a, dtype):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype == torch.bfloat16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.pin_memory()

    h_in = [pinned(case.kv, torch.bfloat16), pinned(case.score, torch.bfloat16),
            pinned(case.grad_out, torch.bfloat16), pinned(case.ape, torch.float32),
            pinned(case.cu_seqlens, torch.int32), pinned(case.cu_seqlens_comp, torch.int32)]
    d_in = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in h_in] for _ in range(2)]
    out_shapes = [((C, d), torch.bfloat16), ((T, coff * d), torch.bfloat16),
                  ((T, coff * d), torch.bfloat16), ((r, coff * d), torch.float32)]
    d_out = [[torch.empty(sh, dtype=dt, device=dev) for sh, dt in out_shapes] for _ in range(2)]
    h_out = [[torch.empty(sh, dtype=dt, pin_memory=True) for sh, dt in out_shapes] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sh = int(stream.cuda_stream)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    used = [False, False]

    def step(i):
        s = i % 2
        kv, score, go, ape, cu, cuc = d_in[s]
        out, dkv, dscore, dape = d_out[s]
        with torch.cuda.stream(s_h2d):
            if used[s]:
                s_h2d.wait_event(ev["comp"][s])   # step i-2 finished reading this set
            for dt, ht in zip(d_in[s], h_in):
                dt.copy_(ht, non_blocking=True)
            ev["in"][s].record(s_h2d)
        stream.wait_event(ev["in"][s])
        if used[s]:
            stream.wait_event(ev["out"][s])       # step i-2's results have left this set
        gsk.csa_compress_fwd_ptr(kv.data_ptr(), score.data_ptr(), ape.data_ptr(), cu.data_ptr(),
                                 cuc.data_ptr(), case.num_seqs, T, C, r, coff, d, out.data_ptr(), sh,
                                 args.exact)
        gsk.csa_compress_bwd_ptr(kv.data_ptr(), score.data_ptr(), ape.data_ptr(), cu.data_ptr(),
                                 cuc.data_ptr(), case.num_seqs, T, C, r, coff, d, go.data_ptr(),
                                 dkv.data_ptr(), dscore.data_ptr(), dape.data_ptr(), sh, args.exact)
        ev["comp"][s].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["comp"][s])
            for dt, ht in zip(d_out[s], h_out[s]):
                ht.copy_(dt, non_blocking=True)
            ev["out"][s].record(s_d2h)
        used[s] = True

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    KE = max(1, args.e2e_steps)
    ranks.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(KE):
        step(i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    el = ranks.max(el)
    return el, h2d, d2h, KE


def run_graph(args, fwd_g, bwd_g, l2, stream):
    """One forward + backward step captured in a CUDA graph, replayed K times;
    each replay timed with events on the replay stream (the L2 treatment of
    the eager loop applies between replays)."""
    import torch

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fwd_g(int(side.cuda_stream))
        bwd_g(int(side.cuda_stream))
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        h = int(torch.cuda.current_stream().cuda_stream)
        fwd_g(h)
        bwd_g(h)
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for _ in range(args.warmup):
        l2()
        g.replay()
    torch.cuda.synchronize()
    for i in range(K):
        l2()
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    return {"step_us": statistics.mean(ms) * 1e3, "step_us_median": statistics.median(ms) * 1e3,
            "replays": K, "what": "fwd + bwd captured once in a CUDA graph, replay timed by events"}


def run_gpu(args, rank, world, local):
    import numpy as np
    import torch

    import gated_softmax_kv_gb300 as gsk
    import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks(rank, world, "nccl", dev)

    gsk.build()
    lib = gsk.load()  # noqa: F841  (fails loudly if the library is missing)
    case = pick_case(args, seed=rank)
    T, C, r, coff, d = case.total_tokens, case.capacity, case.ratio, case.coff, case.head_dim

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    kv, score, grad_out = up(case.kv), up(case.score), up(case.grad_out)
    ape = torch.from_numpy(case.ape).to(dev)
    cu = torch.from_numpy(case.cu_seqlens).to(dev)
    cuc = torch.from_numpy(case.cu_seqlens_comp).to(dev)
    out = torch.empty((C, d), dtype=torch.bfloat16, device=dev)
    dkv = torch.empty_like(kv)
    dscore = torch.empty_like(score)
    dape = torch.empty_like(ape)
    stream = torch.cuda.current_stream(dev)
    sh = int(stream.cuda_stream)
    nseq = case.num_seqs

    def fwd_g(h):
        gsk.csa_compress_fwd_ptr(kv.data_ptr(), score.data_ptr(), ape.data_ptr(), cu.data_ptr(),
                                 cuc.data_ptr(), nseq, T, C, r, coff, d, out.data_ptr(), h, args.exact)

    def bwd_g(h):
        gsk.csa_compress_bwd_ptr(kv.data_ptr(), score.data_ptr(), ape.data_ptr(), cu.data_ptr(),
                                 cuc.data_ptr(), nseq, T, C, r, coff, d, grad_out.data_ptr(),
                                 dkv.data_ptr(), dscore.data_ptr(), dape.data_ptr(), h, args.exact)

    def fwd():
        fwd_g(sh)

    def bwd():
        bwd_g(sh)

    barrier = ranks.barrier
    # Small workloads would stay in the 129 MB L2 from one call to the next:
    # then every call is preceded by a write of a buffer twice the L2 size
    # (outside the per-call events) and the step rate is taken from the calls.
    in_bytes = kv.numel() * 2 + score.numel() * 2
    flush = args.l2 in ("flush", "clean") or (args.l2 == "auto" and in_bytes < 2 * L2_BYTES)
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if flush else None
    clean = torch.ones(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if args.l2 == "clean" else None
    sink = torch.empty((), dtype=torch.int64, device=dev) if clean is not None else None

    def l2():
        if scrub is not None:
            scrub.fill_(0x5A5A5A5A)
        if clean is not None:
            torch.sum(clean, dim=0, dtype=torch.int64, out=sink)

    clocks = ClockSampler(local, pci_bus_id(local))
    clocks.start()
    for _ in range(args.warmup):
        l2()
        fwd()
        l2()
        bwd()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.mark()
    start.record(stream)
    for i in range(K):
        l2()
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        l2()
        ev[i][2].record(stream)
        bwd()
        ev[i][3].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    clocks.unmark()
    barrier()
    elapsed = start.elapsed_time(end) / 1e3
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    bwd_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K)]
    if flush:  # the scrubbing writes are not part of a step
        elapsed = (sum(fwd_ms) + sum(bwd_ms)) / 1e3
    elapsed = ranks.max(elapsed)

    graph = run_graph(args, fwd_g, bwd_g, l2, stream) if args.graph else None

    # End to end through the same C ABI with host buffers. Every step copies its
    # inputs from pinned host memory to HBM, runs both calls and copies every
    # result back. Consecutive steps overlap: two device buffer sets, H2D and D2H
    # on their own streams, ordered against the compute stream by events (the
    # H2D of step i+1 and the D2H of step i-1 run while step i computes).
    e2e_s, h2d, d2h, KE = run_e2e(args, case, dev, stream, ranks)
    clk = clocks.stop()

    if rank != 0:
        ranks.close()
        return 0

    fwd_bytes, bwd_bytes = algorithmic_bytes(case)
    peak, peak_src = measured_peak()
    fwd_avg = statistics.mean(fwd_ms) / 1e3
    bwd_avg = statistics.mean(bwd_ms) / 1e3
    fwd_gbs = fwd_bytes / fwd_avg / 1e9
    bwd_gbs = bwd_bytes / bwd_avg / 1e9
    value = T * K * world / elapsed
    dominant = "bwd" if bwd_avg >= fwd_avg else "fwd"
    dom_bytes, dom_gbs = (bwd_bytes, bwd_gbs) if dominant == "bwd" else (fwd_bytes, fwd_gbs)
    # the recorded DRAM counters were taken on the default mode's kernels
    traffic = {"traffic": None} if args.exact else \
        ncu_traffic("csa_compress_bwd" if dominant == "bwd" else "csa_compress_fwd", T)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, cores, desc, single = oracle_rate(case)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc,
               **single}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": elapsed / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic (seeded SplitMix64/Box-Muller, the page's gate distribution)",
        "config": {"workload": (WORKLOAD if T == 262144 else f"headline recipe scaled to {T} tokens")
                   if args.workload == "headline" else args.workload, "tokens": T, "true_rows": case.true_rows, "capacity": C,
                   "ratio": r, "coff": coff, "head_dim": d, "segments": case.num_seqs,
                   "l2": (f"L2 flushed before every call ({2 * L2_BYTES >> 20} MiB write"
                          + (f", then a {2 * L2_BYTES >> 20} MiB read that leaves it clean" if clean is not None else "")
                          + ", outside the per-call events); value from the summed call times") if flush else
                         (f"inputs larger than L2 (kv+score {in_bytes / 2**20:.0f} MiB per step), no flush"
                          if in_bytes >= 2 * L2_BYTES else "L2 warm between calls (--l2 warm)"),
                   "step": ("csa_compress_fwd_exact + csa_compress_bwd_exact (3 kernels)" if args.exact
                            else "csa_compress_fwd + csa_compress_bwd (3 kernels)")},
        "roofline": {"bound": "hbm", "kernel": "csa_compress_" + dominant + (" (bwd kernel + dape reduce)" if dominant == "bwd" else ""),
                     "achieved": dom_gbs, "peak": peak, "unit": "GB/s", "frac": dom_gbs / peak,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": dom_gbs / NOMINAL_HBM_GBS,
                     "fractions": ("frac: of the measured copy bandwidth; frac_of_nominal: of the "
                                   "~8 TB/s nominal HBM3e peak, the figure the >= 70% target is "
                                   "stated in"),
                     **traffic, "algorithmic_bytes": dom_bytes, "peak_source": peak_src,
                     **({"note": "the exact mode is bound by instruction issue (the fast "
                                 "arithmetic plus its error enclosures, and the exact pass over "
                                 "undecided outputs), not by HBM; the HBM fraction is shown for "
                                 "comparison with the default mode"} if args.exact else {})},
        "fwd": {"ms": fwd_avg * 1e3, "tokens_per_s": T / fwd_avg, "GBps": fwd_gbs, "frac": fwd_gbs / peak,
                "frac_of_nominal": fwd_gbs / NOMINAL_HBM_GBS, "algorithmic_bytes": fwd_bytes},
        "bwd": {"ms": bwd_avg * 1e3, "tokens_per_s": T / bwd_avg, "GBps": bwd_gbs, "frac": bwd_gbs / peak,
                "frac_of_nominal": bwd_gbs / NOMINAL_HBM_GBS, "algorithmic_bytes": bwd_bytes},
        "e2e": {"value": T * KE * world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": KE},
        "gpu_launches": 3 * K,
        **({"graph": graph} if graph is not None else {}),
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    ranks.close()
    return 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_gpu(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
