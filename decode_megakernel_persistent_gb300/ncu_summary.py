"""Summaries of Nsight Compute output for the profiles/ notes.

  python -m decode_megakernel_persistent_gb300.ncu_summary launches LAUNCHES.csv
      per kernel: launches, total device time, share (from a
      `--metrics gpu__time_duration.sum --csv --log-file` run)
  python -m decode_megakernel_persistent_gb300.ncu_summary raw RAW.csv
      selected counters of one captured launch (from `ncu -i REP --page raw --csv`)
  python -m decode_megakernel_persistent_gb300.ncu_summary metrics METRICS.csv
      every launch of a `--metrics a,b,... --csv --log-file` run, one row per
      launch, one column per metric
"""
from __future__ import annotations

import collections
import csv
import sys

RAW_KEYS = (
    "gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
    "dram__throughput.avg.pct_of_peak_sustained_elapsed", "sm__throughput.avg.pct_of_peak_sustained_elapsed",
    "smsp__issue_active.avg.pct_of_peak_sustained_active", "smsp__inst_executed.sum",
    "sm__warps_active.avg.pct_of_peak_sustained_active", "launch__registers_per_thread",
    "sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active",
    "sm__pipe_alu_cycles_active.avg.pct_of_peak_sustained_active",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active",
    "sm__inst_executed_pipe_lsu.avg.pct_of_peak_sustained_active", "lts__t_sector_hit_rate.pct",
    "l1tex__data_bank_conflicts_pipe_lsu_mem_shared.sum",
    "smsp__average_warps_issue_stalled_barrier_per_issue_active.ratio",
    "smsp__average_warps_issue_stalled_long_scoreboard_per_issue_active.ratio",
    "smsp__average_warps_issue_stalled_short_scoreboard_per_issue_active.ratio",
    "smsp__average_warps_issue_stalled_wait_per_issue_active.ratio",
    "smsp__average_warps_issue_stalled_math_pipe_throttle_per_issue_active.ratio",
    "smsp__average_warps_issue_stalled_mio_throttle_per_issue_active.ratio",
)


def _rows(path):
    with open(path, newline="") as f:
        lines = [ln for ln in f if not ln.startswith("==")]
    return list(csv.reader(lines))


def launches(path: str) -> str:
    rows = _rows(path)
    hdr = rows[0]
    ki, mi, vi = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    ui = hdr.index("Metric Unit")
    per = collections.defaultdict(lambda: [0, 0.0])
    for r in rows[1:]:
        if len(r) <= vi or r[mi] != "gpu__time_duration.sum":
            continue
        scale = {"ns": 1e-3, "us": 1.0, "usecond": 1.0, "nsecond": 1e-3, "ms": 1e3, "msecond": 1e3}.get(r[ui], 1.0)
        v = float(r[vi].replace(",", "")) * scale
        name = r[ki].split("(")[0]
        per[name][0] += 1
        per[name][1] += v
    total = sum(t for _, t in per.values())
    out = ["| kernel | launches | total us | mean us | share |", "|---|---|---|---|---|"]
    for name, (n, t) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        out.append(f"| {name} | {n} | {t:.1f} | {t / n:.1f} | {t / total:.1%} |")
    return "\n".join(out)


def metrics(path: str) -> str:
    rows = _rows(path)
    hdr = rows[0]
    ii, ki, mi, vi = hdr.index("ID"), hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value")
    ui = hdr.index("Metric Unit")
    per = collections.OrderedDict()
    names = []
    for r in rows[1:]:
        if len(r) <= vi:
            continue
        key = (r[ii], r[ki].split("(")[0])
        per.setdefault(key, {})[r[mi]] = f"{r[vi]} {r[ui]}".strip()
        if r[mi] not in names:
            names.append(r[mi])
    out = ["| launch | kernel | " + " | ".join(names) + " |", "|---" * (len(names) + 2) + "|"]
    for (i, k), d in per.items():
        out.append(f"| {i} | {k} | " + " | ".join(d.get(n, "") for n in names) + " |")
    return "\n".join(out)


def raw(path: str) -> str:
    rows = _rows(path)
    hdr, units, vals = rows[0], rows[1], rows[2]
    d = dict(zip(hdr, vals))
    u = dict(zip(hdr, units))
    out = ["| counter | value | unit |", "|---|---|---|"]
    for k in RAW_KEYS:
        if k in d:
            out.append(f"| {k} | {d[k]} | {u.get(k, '')} |")
    return "\n".join(out)


if __name__ == "__main__":
    kind, path = sys.argv[1], sys.argv[2]
    print({"launches": launches, "raw": raw, "metrics": metrics}[kind](path))
