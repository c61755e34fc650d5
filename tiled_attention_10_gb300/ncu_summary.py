"""Summarise ncu output for the profiles/ folder.

    python -m tiled_attention_10_gb300.ncu_summary launches <launches.csv> <out.md> "<command>"
    python -m tiled_attention_10_gb300.ncu_summary kernel <report.ncu-rep> <workload> <out.md> "<command>"

`launches` turns a `--metrics gpu__time_duration.sum --csv` launch list into a
per-kernel table (launches, total time, share).  `kernel` reads one
`--set full` capture (via `ncu -i --page raw --csv`) and writes the figures
the roofline uses, plus a JSON record (DRAM bytes per launch and the hash of
the kernel sources it was taken on) that bench.py reads.
"""
from __future__ import annotations

import collections
import csv
import io
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEY_METRICS = [
    ("gpu__time_duration.sum", "kernel duration"),
    ("sm__cycles_elapsed.avg.per_second", "SM clock"),
    ("dram__bytes_read.sum", "DRAM read"),
    ("dram__bytes_write.sum", "DRAM write"),
    ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "DRAM throughput % of peak"),
    ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed", "tensor pipe active % (elapsed)"),
    ("sm__throughput.avg.pct_of_peak_sustained_elapsed", "SM throughput %"),
    ("lts__t_sector_hit_rate.pct", "L2 hit rate"),
    ("l1tex__m_xbar2l1tex_read_bytes.sum.per_second", "L2 -> SM read bandwidth"),
    ("sm__warps_active.avg.pct_of_peak_sustained_active", "warps active %"),
    ("launch__registers_per_thread", "registers / thread"),
    ("launch__grid_size", "grid"),
    ("launch__block_size", "block"),
    ("l1tex__data_bank_conflicts_pipe_lsu_mem_shared.sum", "smem bank conflicts (LSU)"),
    ("l1tex__data_pipe_tc_wavefronts_mem_shared.sum.pct_of_peak_sustained_elapsed",
     "shared memory read by the tensor cores, % of peak"),
]


def _scale(value: str, unit: str) -> float:
    v = float(value.replace(",", ""))
    mult = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}
    return v * mult.get(unit, 1)


def launches(csv_path: str, out_md: str, command: str) -> None:
    text = open(csv_path).read()
    start = text.find('"ID"')
    rows = list(csv.DictReader(io.StringIO(text[start:])))
    per = collections.OrderedDict()
    for r in rows:
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        name = r["Kernel Name"].split("(")[0]
        t = float(r["Metric Value"].replace(",", ""))
        unit = r.get("Metric Unit", "ns")
        t_ns = t * {"ns": 1, "usecond": 1e3, "us": 1e3, "msecond": 1e6, "ms": 1e6}.get(unit, 1)
        c, tot = per.get(name, (0, 0.0))
        per[name] = (c + 1, tot + t_ns)
    total = sum(v[1] for v in per.values()) or 1.0
    lines = [f"# Launch list: `{os.path.basename(csv_path)}`", "",
             f"Command: `{command}`", "",
             "Per-launch times under ncu are cold-cache and serialised: compare shares, not absolutes.",
             "", "| kernel | launches | total (us) | share |", "|---|---|---|---|"]
    for name, (c, tot) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        lines.append(f"| `{name}` | {c} | {tot / 1e3:.1f} | {100 * tot / total:.1f} % |")
    open(out_md, "w").write("\n".join(lines) + "\n")


def kernel(rep: str, workload: str, out_md: str, command: str, kname: str = "fa_fwd") -> None:
    raw = subprocess.run(["ncu", "-i", rep, "--page", "raw", "--csv"], capture_output=True,
                         text=True, check=True).stdout
    rows = list(csv.reader(io.StringIO(raw)))
    hdr, units, vals = rows[0], rows[1], rows[2]
    col = {h: i for i, h in enumerate(hdr)}
    lines = [f"# ncu `--set full`: {kname}_kernel on {workload}", "",
             f"Command: `{command}`", "", "| metric | value | unit |", "|---|---|---|"]
    for key, label in KEY_METRICS:
        if key in col:
            lines.append(f"| {label} (`{key}`) | {vals[col[key]]} | {units[col[key]]} |")
    stalls = [(h, vals[i]) for h, i in col.items()
              if h.startswith("smsp__average_warps_issue_stalled_") and h.endswith("_per_issue_active.ratio")]
    stalls = sorted(((h, float(v or 0)) for h, v in stalls), key=lambda x: -x[1])[:6]
    lines += ["", "Top warp stall reasons (warps stalled per issue):", ""]
    lines += [f"- `{h.replace('smsp__average_warps_issue_stalled_', '').replace('_per_issue_active.ratio', '')}`: {v:.2f}"
              for h, v in stalls]
    rd = _scale(vals[col["dram__bytes_read.sum"]], units[col["dram__bytes_read.sum"]])
    wr = _scale(vals[col["dram__bytes_write.sum"]], units[col["dram__bytes_write.sum"]])
    open(out_md, "w").write("\n".join(lines) + "\n")
    sys.path.insert(0, ROOT)
    import bench
    rec = {"workload": workload, "dram_bytes_per_launch": rd + wr, "dram_read": rd,
           "dram_write": wr, "kernel_sha": bench.kernel_source_sha(), "command": command}
    with open(os.path.join(os.path.dirname(out_md), f"{kname}_{workload}.ncu.json"), "w") as f:
        json.dump(rec, f, indent=1)


if __name__ == "__main__":
    if sys.argv[1] == "launches":
        launches(sys.argv[2], sys.argv[3], sys.argv[4])
    else:
        kernel(sys.argv[2], sys.argv[3], sys.argv[4], sys.argv[5], *sys.argv[6:7])
