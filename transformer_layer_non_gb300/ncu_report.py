"""Summaries of Nsight Compute output for the layer-step benchmark.

Four reports, each written as a short markdown file (and one JSON file that
bench.py reads):

  launches  ncu CSV of `--metrics gpu__time_duration.sum` over whole layer
            steps -> per kernel and per operator: launches, device time, share,
            next to the share the benchmark measured without the profiler.
  traffic   ncu CSV of dram__bytes_{read,write}.sum over `bench.py
            --profile-op all` -> DRAM bytes per operator launch against the
            operator's algorithmic bytes; also written as JSON keyed by the
            hash of the kernel sources, so that a later change of any kernel
            voids the figures.
  full      an `ncu --set full` report (.ncu-rep) -> the counters that say
            what bounds the kernel (DRAM, issue, pipes, stalls, occupancy).
  range     ncu CSVs of range replay (`--replay-mode range`) over `bench.py
            --profile-op OP --profile-sets K --profile-flush-mb M`: K launches
            of one operator on K buffer sets, then a read of a clean M MB buffer
            that evicts their dirty lines from L2, so that reads AND write-backs
            are counted -> DRAM bytes per launch (the flush read subtracted)
            against the algorithmic bytes; also written to the JSON.

Per-launch times under ncu are serialised and cold-cache (ncu flushes the
caches before every profiled launch): compare shares, not absolutes.  DRAM
write bytes undercount the stores of a kernel whose output still fits in L2
when it ends, since L2 writes back later.

    python -m transformer_layer_non_gb300.ncu_report launches --csv L.csv \
        --bench-log plain.log --command "..." --out profiles/X.md
    python -m transformer_layer_non_gb300.ncu_report traffic --csv T.csv \
        --profile-log all.log --workload bert-base --command "..." \
        --out profiles/Y.md --json profiles/ncu_traffic.json
    python -m transformer_layer_non_gb300.ncu_report full --rep R.ncu-rep \
        --command "..." --out profiles/Z.md
    python -m transformer_layer_non_gb300.ncu_report range \
        --case bert-base:softmax_bwd=R.csv,plain.log ... --command "..." \
        --out profiles/W.md --json profiles/ncu_traffic.json
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import re
import subprocess
from collections import OrderedDict

PKG = os.path.dirname(os.path.abspath(__file__))


def kernels_sha() -> str:
    """Hash of every kernel source file (names and contents)."""
    h = hashlib.sha256()
    csrc = os.path.join(PKG, "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(f.encode())
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_ncu_csv(path):
    """Rows of an ncu --csv log (the lines ncu itself prints are skipped)."""
    with open(path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    return list(csv.DictReader(lines))


def short_name(kernel: str) -> str:
    """The kernel's name and template arguments: the return type, the leading
    namespaces (ncu writes the anonymous one as `unnamed>::`) and the trailing
    argument list dropped."""
    name = kernel.strip()
    if name.endswith(")"):  # the argument list: back to its matching parenthesis
        depth = 0
        for i in range(len(name) - 1, -1, -1):
            if name[i] == ")":
                depth += 1
            elif name[i] == "(":
                depth -= 1
                if depth == 0:
                    name = name[:i]
                    break
    name = re.sub(r"^void\s+", "", name)
    return re.sub(r"^(\w+>::|<\w+>::|\(anonymous namespace\)::|\w+::)+", "", name)


def value(row) -> float:
    v = float(row["Metric Value"].replace(",", ""))
    scale = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "msecond": 1e3,
             "byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    return v * scale.get(row["Metric Unit"], 1.0)


def launches_by_id(rows, metrics):
    """[(kernel, grid, block, {metric: value})] in launch order."""
    out = OrderedDict()
    for r in rows:
        if r["Metric Name"] not in metrics:
            continue
        k = out.setdefault(r["ID"], (r["Kernel Name"], r["Grid Size"], r["Block Size"], {}))
        k[3][r["Metric Name"]] = value(r)
    return list(out.values())


def last_json_line(path):
    with open(path) as f:
        lines = [ln for ln in f if ln.startswith("{")]
    return json.loads(lines[-1])


def report_launches(a):
    launches = launches_by_id(read_ncu_csv(a.csv), {"gpu__time_duration.sum"})
    bench = last_json_line(a.bench_log)
    per_op = bench["per_op"]
    order = [(n, v["launches"]) for n, v in per_op.items()]
    per_step = sum(c for _, c in order)
    if len(launches) % per_step:
        raise SystemExit(f"{len(launches)} launches is not a whole number of "
                         f"{per_step}-launch steps")
    slots = [n for n, c in order for _ in range(c)]
    total = sum(k[3]["gpu__time_duration.sum"] for k in launches)
    kern = OrderedDict()
    ops = OrderedDict((n, 0.0) for n, _ in order)
    for i, (name, grid, block, m) in enumerate(launches):
        t = m["gpu__time_duration.sum"]
        e = kern.setdefault((short_name(name), grid, block), [0, 0.0, []])
        e[0] += 1
        e[1] += t
        op = slots[i % per_step]
        if op not in e[2]:
            e[2].append(op)
        ops[op] += t
    steps = len(launches) // per_step
    alone = {n: v.get("us", v.get("alone_us")) for n, v in per_op.items()}
    alone_sum = sum(alone.values())
    out = [f"# Kernel launch list: {bench['config']['workload']} layer step "
           "(every fused operator, forward and backward)", "",
           "Command (one GB300; one-pass metric, so every launch is serialised and "
           "cold-cache: compare the SHARES, not the absolute times):", ""]
    out += ["    " + ln for ln in a.command.splitlines()]
    out += ["", f"{len(launches)} launches = {steps} graph replays of the step "
            f"({per_step} launches per step).  Step time without the profiler: "
            f"{bench['ms_per_step'] * 1e3:.1f} us.", "",
            "| kernel | grid | block | launches | total us | us / launch | share | operators |",
            "|---|---|---|---|---|---|---|---|"]
    for (name, grid, block), (n, t, who) in sorted(kern.items(), key=lambda kv: -kv[1][1]):
        out.append(f"| `{name}` | {grid} | {block} | {n} | {t:.1f} | {t / n:.2f} | "
                   f"{100 * t / total:.1f}% | {', '.join(who)} |")
    out += ["", "Per operator (main kernel plus its column reduction, if any): share of "
            "the profiled device time against the share of the operator's own time "
            "measured by bench.py without the profiler (operator alone, CUDA events, "
            "L2-cold buffer sets).", "",
            "| operator | ncu us / launch | ncu share | bench us | bench share |",
            "|---|---|---|---|---|"]
    for n, t in ops.items():
        out.append(f"| {n} | {t / steps:.2f} | {100 * t / total:.1f}% | {alone[n]:.2f} | "
                   f"{100 * alone[n] / alone_sum:.1f}% |")
    if a.note:
        out += ["", a.note]
    with open(a.out, "w") as f:
        f.write("\n".join(out) + "\n")


def report_traffic(a):
    mets = {"dram__bytes_read.sum", "dram__bytes_write.sum", "gpu__time_duration.sum"}
    launches = launches_by_id(read_ncu_csv(a.csv), mets)
    prof = last_json_line(a.profile_log)
    order = prof["launch_order"]
    if len(order) != len(launches):
        raise SystemExit(f"{len(launches)} profiled launches, {len(order)} expected")
    per_op = OrderedDict()
    for op, (name, _, _, m) in zip(order, launches):
        e = per_op.setdefault(op, {"read": 0.0, "write": 0.0, "us": 0.0, "kernels": []})
        e["read"] += m["dram__bytes_read.sum"]
        e["write"] += m["dram__bytes_write.sum"]
        e["us"] += m["gpu__time_duration.sum"]
        if short_name(name) not in e["kernels"]:
            e["kernels"].append(short_name(name))
    reps = prof["launches_per_op"]
    sha = a.sha or kernels_sha()
    out = [f"# DRAM traffic per operator launch: {a.workload} layer", "",
           "Command (one GB300; ncu flushes the caches before each profiled launch):", ""]
    out += ["    " + ln for ln in a.command.splitlines()]
    out += ["", f"Kernel sources hash: `{sha}`.  {reps} launches per operator; figures "
            "are per operator launch (main kernel plus its column reduction, if any).  "
            "Algorithmic bytes: every input the operator needs read once, every output "
            "written once.", "",
            "| operator | kernels | algorithmic MB | DRAM read MB | DRAM write MB | "
            "read+write / algorithmic |", "|---|---|---|---|---|---|"]
    js = {}
    for op, e in per_op.items():
        alg = prof["algorithmic_bytes"][op]
        rd, wr = e["read"] / reps, e["write"] / reps
        out.append(f"| {op} | {', '.join('`%s`' % k for k in e['kernels'])} | {alg / 1e6:.2f} | "
                   f"{rd / 1e6:.2f} | {wr / 1e6:.2f} | {(rd + wr) / alg:.2f} |")
        js[op] = {"dram_bytes_per_launch": int(rd + wr), "dram_read_bytes": int(rd),
                  "dram_write_bytes": int(wr), "algorithmic_bytes": int(alg)}
    if a.note:
        out += ["", a.note]
    with open(a.out, "w") as f:
        f.write("\n".join(out) + "\n")
    if a.json:
        d = {}
        if os.path.exists(a.json):
            with open(a.json) as f:
                d = json.load(f)
            if d.get("kernels_sha") != sha:
                d = {}
        d["kernels_sha"] = sha
        d["note"] = ("DRAM bytes per operator launch from ncu (dram__bytes_read.sum + "
                     "dram__bytes_write.sum); valid only for the kernel sources of this hash")
        d.setdefault("ops", {})[a.workload] = js
        with open(a.json, "w") as f:
            json.dump(d, f, indent=1)
            f.write("\n")


def range_case(csv_path, log_path):
    """(workload, op, launches, read, write, algorithmic, flush) of one range
    capture: per-launch DRAM read bytes (the flush read subtracted) and write
    bytes."""
    rows = read_ncu_csv(csv_path)
    m = {r["Metric Name"]: value(r) for r in rows}
    prof = last_json_line(log_path)
    (op, alg), = prof["algorithmic_bytes"].items()
    n = prof["buffer_sets"] * prof["launches_per_op"]
    flush = prof.get("flush_read_bytes", 0)
    rd = (m["dram__bytes_read.sum"] - flush) / n
    wr = m["dram__bytes_write.sum"] / n
    return prof["workload"], op, n, rd, wr, float(alg), flush, prof.get("kernels_sha")


def report_range(a):
    cases = []
    for spec in a.case:
        csv_path, log_path = spec.split("=", 1)[1].split(",")
        cases.append(range_case(csv_path, log_path))
    shas = {c[7] for c in cases}
    sha = a.sha or (shas.pop() if len(shas) == 1 else kernels_sha())
    out = ["# DRAM traffic per operator launch, reads and write-backs (ncu range replay)", "",
           "Command per case (one GB300; OP, WORKLOAD, K as in the table):", ""]
    out += ["    " + ln for ln in a.command.splitlines()]
    out += ["", f"Kernel sources hash: `{sha}`.  Each range holds K launches of the operator "
            "on K distinct buffer sets, then a read of a clean buffer larger than L2 that "
            "evicts their dirty lines, so the write-backs land inside the range; the "
            "flush's own reads are subtracted.  Figures are per operator launch (main "
            "kernel plus its column reduction, if any).", "",
            "| workload | operator | K | algorithmic MB | DRAM read MB | DRAM write MB | "
            "read+write / algorithmic |", "|---|---|---|---|---|---|---|"]
    js = {}
    for wl, op, n, rd, wr, alg, _, _ in cases:
        out.append(f"| {wl} | {op} | {n} | {alg / 1e6:.2f} | {rd / 1e6:.2f} | {wr / 1e6:.2f} | "
                   f"{(rd + wr) / alg:.3f} |")
        js.setdefault(wl, {})[op] = {"dram_bytes_per_launch": int(rd + wr),
                                     "dram_read_bytes": int(rd), "dram_write_bytes": int(wr),
                                     "algorithmic_bytes": int(alg),
                                     "method": "range replay, L2 flushed by a read"}
    if a.note:
        out += ["", a.note]
    with open(a.out, "w") as f:
        f.write("\n".join(out) + "\n")
    if a.json:
        d = {}
        if os.path.exists(a.json):
            with open(a.json) as f:
                d = json.load(f)
            if d.get("kernels_sha") != sha:
                d = {}
        d["kernels_sha"] = sha
        d["note"] = ("DRAM bytes per operator launch from ncu (dram__bytes_read.sum + "
                     "dram__bytes_write.sum); valid only for the kernel sources of this hash")
        for wl, ops in js.items():
            d.setdefault("ops", {}).setdefault(wl, {}).update(ops)
        with open(a.json, "w") as f:
            json.dump(d, f, indent=1)
            f.write("\n")


FULL_METRICS = [
    ("gpu__time_duration.sum", "duration"),
    ("launch__grid_size", "grid"),
    ("launch__block_size", "block"),
    ("launch__registers_per_thread", "registers / thread"),
    ("launch__shared_mem_per_block_dynamic", "dynamic shared memory / block"),
    ("launch__occupancy_limit_registers", "CTAs / SM allowed by registers"),
    ("launch__occupancy_limit_shared_mem", "CTAs / SM allowed by shared memory"),
    ("sm__warps_active.avg.pct_of_peak_sustained_active", "warps active (% of max)"),
    ("dram__bytes_read.sum", "DRAM read"),
    ("dram__bytes_write.sum", "DRAM write"),
    ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "DRAM throughput (% of peak)"),
    ("lts__t_sector_hit_rate.pct", "L2 hit rate"),
    ("sm__throughput.avg.pct_of_peak_sustained_elapsed", "SM throughput (% of peak)"),
    ("smsp__issue_active.avg.pct_of_peak_sustained_active", "issue slots busy"),
    ("smsp__inst_executed.sum", "warp instructions"),
    ("sm__inst_executed_pipe_alu.avg.pct_of_peak_sustained_active", "ALU pipe"),
    ("sm__inst_executed_pipe_fma.avg.pct_of_peak_sustained_active", "FMA pipe"),
    ("sm__inst_executed_pipe_lsu.avg.pct_of_peak_sustained_active", "LSU pipe"),
    ("sm__inst_executed_pipe_adu.avg.pct_of_peak_sustained_active", "ADU pipe"),
    ("sm__inst_executed_pipe_xu.avg.pct_of_peak_sustained_active", "XU pipe"),
    ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", "tensor pipe"),
]


def report_full(a):
    raw = subprocess.run(["ncu", "-i", a.rep, "--page", "raw", "--csv"], check=True,
                         capture_output=True, text=True).stdout
    rows = list(csv.reader([ln for ln in raw.splitlines() if ln.startswith('"')]))
    head, units = rows[0], rows[1]
    out = [f"# ncu --set full: {a.title}", "", "Command (one GB300):", ""]
    out += ["    " + ln for ln in a.command.splitlines()]
    for vals in rows[2:]:
        col = dict(zip(head, vals))
        unit = dict(zip(head, units))
        out += ["", f"Kernel: `{short_name(col.get('Kernel Name', '?'))}`", "",
                "| counter | value | unit | metric |", "|---|---|---|---|"]
        for m, label in FULL_METRICS:
            if m in col:
                out.append(f"| {label} | {col[m]} | {unit[m]} | `{m}` |")
        stalls = []
        for m in head:
            g = re.match(r"smsp__average_warps_issue_stalled_(\w+)_per_issue_active\.ratio$", m)
            if g and g.group(1) not in ("selected",):
                try:
                    stalls.append((float(col[m].replace(",", "")), g.group(1)))
                except ValueError:
                    pass
        stalls.sort(reverse=True)
        out += ["", "Top warp stall reasons (cycles per issued instruction): " +
                ", ".join(f"{n} {v:.2f}" for v, n in stalls[:6]) + "."]
    if a.note:
        out += ["", a.note]
    with open(a.out, "w") as f:
        f.write("\n".join(out) + "\n")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    sub = ap.add_subparsers(dest="mode", required=True)
    p = sub.add_parser("launches")
    p.add_argument("--csv", required=True)
    p.add_argument("--bench-log", required=True, help="output of the same bench.py command "
                   "run without ncu (its last JSON line)")
    p.add_argument("--command", required=True)
    p.add_argument("--out", required=True)
    p.add_argument("--note", default="")
    p = sub.add_parser("traffic")
    p.add_argument("--csv", required=True)
    p.add_argument("--profile-log", required=True, help="stdout of the profiled "
                   "bench.py --profile-op command (its last JSON line)")
    p.add_argument("--workload", required=True)
    p.add_argument("--command", required=True)
    p.add_argument("--out", required=True)
    p.add_argument("--json", default=None)
    p.add_argument("--sha", default=None, help="kernel sources hash the capture ran on "
                   "(default: the current sources)")
    p.add_argument("--note", default="")
    p = sub.add_parser("range")
    p.add_argument("--case", action="append", required=True,
                   help="LABEL=CSV,LOG: one range capture and the stdout of its bench.py "
                        "--profile-op command (repeatable)")
    p.add_argument("--command", required=True)
    p.add_argument("--out", required=True)
    p.add_argument("--json", default=None)
    p.add_argument("--sha", default=None)
    p.add_argument("--note", default="")
    p = sub.add_parser("full")
    p.add_argument("--rep", required=True)
    p.add_argument("--title", required=True)
    p.add_argument("--command", required=True)
    p.add_argument("--out", required=True)
    p.add_argument("--note", default="")
    a = ap.parse_args(argv)
    {"launches": report_launches, "traffic": report_traffic, "full": report_full,
     "range": report_range}[a.mode](a)


if __name__ == "__main__":
    main()
