"""ncu harness: the profiling commands behind profiles/ and their summaries.

Run on a machine with the GPU (every command first runs the same bench.py
line without ncu and profiles only if that exits 0; ncu always gets
--clock-control none, so it never locks the GPU's clocks):

  python -m gated_softmax_kv_gb300.ncu_harness launches [bench args...]
      every launch of a short bench run with its device time (one ncu pass,
      gpu__time_duration.sum); prints kernel, launches, total and per-launch
      time and share as a markdown table. Times under ncu are cold-cache and
      serialised: compare shares, not absolute times.

  python -m gated_softmax_kv_gb300.ncu_harness capture --kernel NAME [--skip N] [--count N]
          [--out NAME] [bench args...]
      a --set full capture (plus the L2 read / write sector counts) of one to
      three launches of ONE kernel (a plain function name such as
      bwd_small_kernel, no alternation) on a small case (defaults: the
      headline recipe at 65536 tokens, above the L2 size but a few GB on the
      device), then a table of the DRAM bytes, stored bytes, throughput,
      occupancy, issue and pipe figures per captured launch.

  python -m gated_softmax_kv_gb300.ncu_harness traffic --fwd REPORT --bwd REPORT
          --reduce REPORT --tokens N
      the per-token bytes of the forward call (its kernel's capture) and of
      the backward call (the backward kernel's capture plus the dape reduce's)
      on the headline recipe at N tokens: DRAM reads, DRAM writes, and the
      bytes the kernels' global stores wrote (l1tex global store sectors x
      32: every one of them is written back to DRAM, also when it is still
      dirty in L2 at the kernel's end; local-memory spill stores and the L2's
      own traffic between GB300's two dies are not in that count), written to
      profiles/dram_traffic.json with a hash of the kernels' sources, which
      bench.py uses for roofline.traffic while the sources are unchanged.

The parsing functions take ncu's CSV text and need no GPU.
"""
from __future__ import annotations

import argparse
import collections
import csv
import json
import os
import re
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TRAFFIC = os.path.join(ROOT, "profiles", "dram_traffic.json")

# the figures a capture table shows: (metric, label)
CAPTURE_METRICS = [
    ("gpu__time_duration.sum", "duration"),
    ("dram__bytes_read.sum", "DRAM read"),
    ("dram__bytes_write.sum", "DRAM write"),
    ("l1tex__t_sectors_pipe_lsu_mem_global_op_st.sum", "global store sectors"),
    ("l1tex__t_requests_pipe_lsu_mem_local_op_st.sum", "local (spill) store requests"),
    ("lts__t_sectors_srcunit_tex_op_read.sum", "L2 read sectors from the SMs"),
    ("lts__t_sectors_srcunit_ltcfabric.sum", "L2 sectors between the two dies"),
    ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "DRAM throughput (% of peak)"),
    ("launch__registers_per_thread", "registers / thread"),
    ("launch__occupancy_limit_registers", "blocks / SM (register limit)"),
    ("sm__warps_active.avg.pct_of_peak_sustained_active", "warps active (% of peak)"),
    ("smsp__inst_executed.sum", "instructions (warp)"),
    ("smsp__issue_active.avg.pct_of_peak_sustained_active", "issue active (%)"),
    ("smsp__average_warps_issue_stalled_long_scoreboard_per_issue_active.ratio",
     "stall long scoreboard / issue"),
    ("smsp__average_warps_issue_stalled_barrier_per_issue_active.ratio", "stall barrier / issue"),
    ("sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active", "FMA pipe (% active)"),
    ("sm__pipe_alu_cycles_active.avg.pct_of_peak_sustained_active", "ALU pipe (% active)"),
    ("sm__inst_executed_pipe_xu.avg.pct_of_peak_sustained_active", "XU pipe (% of peak)"),
]

# counters a capture asks for by name on top of --set full: global store
# sectors (the store audit) and the SM-originated L2 traffic
EXTRA_METRICS = ("l1tex__t_sectors_pipe_lsu_mem_global_op_st.sum,"
                 "lts__t_sectors_srcunit_tex_op_read.sum,lts__t_sectors_srcunit_tex_op_write.sum")
SECTOR_BYTES = 32

# the calls whose traffic the record holds: the reports (one kernel each) that
# make them up and the csrc/ sources of those kernels
TRAFFIC_KERNELS = {
    "csa_compress_fwd": dict(reports=["fwd"], kernel="fwd_small_kernel<4,2,512>",
                             sources=["csa_fwd.cu", "csa_device.cuh", "csa_internal.h"]),
    "csa_compress_bwd": dict(reports=["bwd", "reduce"],
                             kernel="bwd_small_kernel<4,2,512> + dape_reduce_kernel",
                             sources=["csa_bwd.cu", "csa_bwd_common.cuh", "csa_device.cuh",
                                      "csa_internal.h"]),
}

_KERNEL_NAME = re.compile(r"[A-Za-z_][A-Za-z0-9_]*")

_TIME_SCALE = {"nsecond": 1e-3, "ns": 1e-3, "usecond": 1.0, "us": 1.0, "msecond": 1e3, "ms": 1e3,
               "second": 1e6, "s": 1e6}
_BYTE_SCALE = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6,
               "GB": 1e9}


def _num(text: str) -> float:
    return float(text.replace(",", ""))


def short_name(kernel: str) -> str:
    """`void (anonymous namespace)::fwd_small_kernel<4, 2, 512>(FwdParams)` ->
    `fwd_small_kernel<4, 2, 512>`."""
    name = re.sub(r"\(.*$", "", kernel.strip())
    name = re.sub(r"^void\s+", "", name)
    return name.split("::")[-1]


def parse_launches(text: str):
    """Rows of an ncu --csv --metrics gpu__time_duration.sum log -> per kernel
    (launches, total us, grid, block), in order of first appearance."""
    lines = [ln for ln in text.splitlines() if ln.startswith('"')]
    rows = list(csv.reader(lines))
    if not rows:
        return collections.OrderedDict()
    hdr = rows[0]
    ki, vi, ui = hdr.index("Kernel Name"), hdr.index("Metric Value"), hdr.index("Metric Unit")
    mi = hdr.index("Metric Name")
    gi = hdr.index("Grid Size") if "Grid Size" in hdr else None
    bi = hdr.index("Block Size") if "Block Size" in hdr else None
    out = collections.OrderedDict()
    for r in rows[1:]:
        if len(r) <= vi or r[mi] != "gpu__time_duration.sum":
            continue
        us = _num(r[vi]) * _TIME_SCALE.get(r[ui], 1.0)
        k = short_name(r[ki])
        e = out.setdefault(k, dict(launches=0, total_us=0.0, grid=r[gi] if gi is not None else "",
                                   block=r[bi] if bi is not None else ""))
        e["launches"] += 1
        e["total_us"] += us
    return out


def launches_table(summary) -> str:
    total = sum(e["total_us"] for e in summary.values()) or 1.0
    out = ["| kernel | launches | total µs | µs / launch | share | grid | block |",
           "|---|---|---|---|---|---|---|"]
    for k, e in sorted(summary.items(), key=lambda kv: -kv[1]["total_us"]):
        out.append("| `%s` | %d | %.1f | %.1f | %.1f%% | %s | %s |" % (
            k, e["launches"], e["total_us"], e["total_us"] / e["launches"],
            100.0 * e["total_us"] / total, e["grid"], e["block"]))
    return "\n".join(out)


def parse_raw(text: str):
    """ncu -i REPORT --page raw --csv -> list of (kernel, {metric: (value, unit)})."""
    lines = [ln for ln in text.splitlines() if ln.startswith('"')]
    rows = list(csv.reader(lines))
    if len(rows) < 3:
        return []
    hdr, units = rows[0], rows[1]
    ki = hdr.index("Kernel Name")
    out = []
    for r in rows[2:]:
        vals = {}
        for i, h in enumerate(hdr):
            if i < len(r):
                vals[h] = (r[i], units[i] if i < len(units) else "")
        out.append((short_name(r[ki]), vals))
    return out


def metric_value(vals, name: str):
    """A metric of a parse_raw row as a float (bytes in bytes, times in us), or None."""
    if name not in vals:
        return None
    text, unit = vals[name]
    try:
        v = _num(text)
    except ValueError:
        return None
    if unit in _BYTE_SCALE:
        return v * _BYTE_SCALE[unit]
    if unit in _TIME_SCALE:
        return v * _TIME_SCALE[unit]
    return v


def capture_table(kernels) -> str:
    names = [k for k, _ in kernels]
    out = ["| metric | " + " | ".join("`%s`" % n for n in names) + " |",
           "|---|" + "---|" * len(names)]
    for metric, label in CAPTURE_METRICS:
        cells = []
        for _, vals in kernels:
            v = metric_value(vals, metric)
            if v is None:
                cells.append("—")
            elif metric.startswith("dram__bytes"):
                cells.append("%.2f MB" % (v / 1e6))
            elif metric == "gpu__time_duration.sum":
                cells.append("%.1f µs" % v)
            elif metric == "smsp__inst_executed.sum":
                cells.append("%.2f M" % (v / 1e6))
            else:
                cells.append("%.4g" % v)
        out.append("| %s | %s |" % (label, " | ".join(cells)))
    return "\n".join(out)


def single_kernel_name(name: str) -> str:
    """The --kernel argument of a capture: one plain function name (a full
    capture of several kernels at once is not allowed)."""
    if not _KERNEL_NAME.fullmatch(name or ""):
        raise ValueError(f"--kernel takes one kernel's function name, not {name!r}")
    return name


def launch_bytes(vals) -> dict:
    """DRAM reads, DRAM writes and bytes of global stores of one captured launch."""
    rd = metric_value(vals, "dram__bytes_read.sum")
    wr = metric_value(vals, "dram__bytes_write.sum")
    st = metric_value(vals, "l1tex__t_sectors_pipe_lsu_mem_global_op_st.sum")
    if rd is None or wr is None or st is None:
        raise ValueError("the capture lacks dram__bytes_read/write.sum or "
                         "l1tex__t_sectors_pipe_lsu_mem_global_op_st.sum")
    return {"read": rd, "dram_write": wr, "l2_write": st * SECTOR_BYTES}


def traffic_record(reports, tokens: int, command: str) -> dict:
    """Per-token bytes of the forward and backward calls from single-kernel
    captures: `reports` maps "fwd", "bwd" and "reduce" to parse_raw rows of
    one kernel each (the first launch of each is used; the backward call is
    its kernel plus the dape reduce). The traffic of a call is its DRAM reads
    plus the bytes of its global stores (all of which reach DRAM)."""
    import bench  # the source hash bench.py checks the record against
    rec = {"note": ("per-token bytes of one launch per kernel from ncu --set full "
                    "on the headline recipe scaled to %d tokens, "
                    "one capture per kernel; bench.py scales them to the measured launch (traffic "
                    "grows with the tokens: every token's kv and score are read once). traffic = "
                    "DRAM reads + bytes of global stores (l1tex global store sectors x 32; every "
                    "stored byte is written back, while the DRAM write counter misses lines still "
                    "dirty in L2 when the kernel ends). Valid while the listed sources hash to "
                    "source_hash. Command: %s" % (tokens, command))}
    for key, spec in TRAFFIC_KERNELS.items():
        tot = {"read": 0.0, "dram_write": 0.0, "l2_write": 0.0}
        names = []
        for part in spec["reports"]:
            rows = reports.get(part)
            if not rows:
                raise ValueError(f"no capture for the {part} kernel")
            kernels = {k for k, _ in rows}
            if len(kernels) != 1:
                raise ValueError(f"the {part} capture holds {sorted(kernels)}: one kernel per capture")
            names.append(rows[0][0])
            for k, v in launch_bytes(rows[0][1]).items():
                tot[k] += v
        rec[key] = dict(kernel=" + ".join(names), unit="token",
                        dram_read_bytes_per_unit=tot["read"] / tokens,
                        dram_write_bytes_per_unit=tot["dram_write"] / tokens,
                        l2_write_bytes_per_unit=tot["l2_write"] / tokens,
                        dram_bytes_per_unit=(tot["read"] + tot["l2_write"]) / tokens,
                        sources=spec["sources"], source_hash=bench.source_hash(spec["sources"]))
    return rec


# ---------------------------------------------------------------- commands


def _ncu() -> str:
    path = shutil.which("ncu") or "/usr/local/cuda/bin/ncu"
    if not os.path.exists(path):
        raise SystemExit("ncu not found")
    return path


def _plain_then(cmd, ncu_args):
    """Run cmd without ncu; only if it exits 0, run it again under ncu."""
    r = subprocess.run(cmd, cwd=ROOT)
    if r.returncode != 0:
        raise SystemExit(f"the plain run exited {r.returncode}: not profiled")
    r = subprocess.run([_ncu(), "--clock-control", "none", *ncu_args, *cmd], cwd=ROOT)
    if r.returncode != 0:
        raise SystemExit(f"ncu exited {r.returncode}")


def _bench(args):
    return [sys.executable, os.path.join(ROOT, "bench.py"), *args]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(prog="python -m gated_softmax_kv_gb300.ncu_harness")
    sub = ap.add_subparsers(dest="cmd", required=True)
    a = sub.add_parser("launches")
    a.add_argument("--out", default="ncu_out/launches.csv")
    a.add_argument("--count", type=int, default=60)
    c = sub.add_parser("capture")
    c.add_argument("--kernel", required=True,
                   help="one kernel's function name, e.g. bwd_small_kernel")
    c.add_argument("--skip", type=int, default=3)
    c.add_argument("--count", type=int, default=1, choices=[1, 2, 3])
    c.add_argument("--out", default="ncu_out/prof")
    t = sub.add_parser("traffic")
    t.add_argument("--fwd", required=True)
    t.add_argument("--bwd", required=True)
    t.add_argument("--reduce", required=True)
    t.add_argument("--tokens", type=int, required=True)
    t.add_argument("--command", default="")
    args, rest = ap.parse_known_args(argv)

    if args.cmd == "launches":
        bench_args = rest or ["--steps", "5", "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "1"]
        os.makedirs(os.path.dirname(os.path.join(ROOT, args.out)), exist_ok=True)
        _plain_then(_bench(bench_args), ["--metrics", "gpu__time_duration.sum", "-c", str(args.count),
                                         "--csv", "--log-file", os.path.join(ROOT, args.out)])
        with open(os.path.join(ROOT, args.out)) as f:
            print(launches_table(parse_launches(f.read())))
    elif args.cmd == "capture":
        bench_args = rest or ["--tokens", "65536", "--steps", "2", "--warmup", "1", "--no-cpu-baseline",
                              "--e2e-steps", "1"]
        os.makedirs(os.path.dirname(os.path.join(ROOT, args.out)), exist_ok=True)
        kernel = single_kernel_name(args.kernel)
        _plain_then(_bench(bench_args), ["--set", "full", "--metrics", EXTRA_METRICS,
                                         "-k", "regex:" + kernel,
                                         "-s", str(args.skip), "-c", str(args.count),
                                         "-o", os.path.join(ROOT, args.out)])
        raw = subprocess.run([_ncu(), "-i", os.path.join(ROOT, args.out) + ".ncu-rep", "--page", "raw",
                              "--csv"], capture_output=True, text=True, check=True).stdout
        print(capture_table(parse_raw(raw)))
    else:
        reports = {}
        for part in ("fwd", "bwd", "reduce"):
            raw = subprocess.run([_ncu(), "-i", getattr(args, part), "--page", "raw", "--csv"],
                                 capture_output=True, text=True, check=True).stdout
            reports[part] = parse_raw(raw)
        rec = traffic_record(reports, args.tokens, args.command)
        with open(TRAFFIC, "w") as f:
            json.dump(rec, f, indent=1)
            f.write("\n")
        print(json.dumps({k: v["dram_bytes_per_unit"] for k, v in rec.items() if k != "note"}))
    return 0


if __name__ == "__main__":
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    sys.exit(main())
