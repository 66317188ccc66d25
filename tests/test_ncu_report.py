"""The ncu summary tooling (transformer_layer_non_gb300/ncu_report.py) on
synthetic ncu CSV output, without a GPU: unit scaling, per-launch averages,
the per-operator grouping of the launch list, the hash-keyed traffic JSON
(replaced when the kernel sources change) and the benchmark's lookup of it."""
import json
import os

import pytest

import bench
from transformer_layer_non_gb300 import ncu_report

HEADER = '"ID","Kernel Name","Grid Size","Block Size","Metric Name","Metric Unit","Metric Value"\n'


def _csv(path, rows):
    with open(path, "w") as f:
        f.write("==PROF== a line ncu prints, skipped\n")
        f.write(HEADER)
        for r in rows:
            f.write(",".join(f'"{v}"' for v in r) + "\n")


def _json_line(path, obj):
    with open(path, "w") as f:
        f.write("some output\n" + json.dumps(obj) + "\n")


def test_kernels_sha_is_stable_hex():
    a, b = ncu_report.kernels_sha(), ncu_report.kernels_sha()
    assert a == b and len(a) == 16
    int(a, 16)


def test_value_scales_units():
    v = lambda x, u: ncu_report.value({"Metric Value": x, "Metric Unit": u})  # noqa: E731
    assert v("1,500", "ns") == pytest.approx(1.5)      # to microseconds
    assert v("2", "usecond") == pytest.approx(2.0)
    assert v("3", "Mbyte") == pytest.approx(3e6)       # to bytes
    assert v("4", "Kbyte") == pytest.approx(4e3)


@pytest.mark.parametrize("raw", [
    # as ncu writes names from an anonymous namespace
    "void unnamed>::softmax_group_kernel<__half, 32, 2, 1, 0>(T1 *, const T1 *, long, "
    "unnamed>::RowMask, unnamed>::DropArgs)",
    "void ls::(anonymous namespace)::softmax_group_kernel<__half, 32, 2, 1, 0>(T1 *, int)",
    "void ls::<unnamed>::softmax_group_kernel<__half, 32, 2, 1, 0>(T1 *, int)",
    "softmax_group_kernel<__half, 32, 2, 1, 0>",
])
def test_short_name_drops_namespaces_and_arguments(raw):
    assert ncu_report.short_name(raw) == "softmax_group_kernel<__half, 32, 2, 1, 0>"


def test_traffic_report_averages_and_hash_keyed_json(tmp_path):
    csv_p, log_p = tmp_path / "t.csv", tmp_path / "p.log"
    out_p, js_p = tmp_path / "t.md", tmp_path / "t.json"
    rows = []
    # two operators, two launches each; op "b" is a main kernel plus a reduction
    launches = [("a", "kern_a", 100, 10), ("a", "kern_a", 300, 30),
                ("b", "kern_b", 50, 0), ("b", "colreduce", 10, 0),
                ("b", "kern_b", 70, 0), ("b", "colreduce", 10, 0)]
    for i, (_, k, rd, wr) in enumerate(launches):
        rows.append((i, f"void {k}(int)", "(1, 1, 1)", "(32, 1, 1)", "dram__bytes_read.sum",
                     "byte", rd))
        rows.append((i, f"void {k}(int)", "(1, 1, 1)", "(32, 1, 1)", "dram__bytes_write.sum",
                     "byte", wr))
        rows.append((i, f"void {k}(int)", "(1, 1, 1)", "(32, 1, 1)", "gpu__time_duration.sum",
                     "ns", 1000))
    _csv(csv_p, rows)
    _json_line(log_p, {"launch_order": ["a", "a", "b", "b", "b", "b"], "launches_per_op": 2,
                       "algorithmic_bytes": {"a": 200, "b": 100}})
    # a stale file (another hash) is replaced, not merged
    js_p.write_text(json.dumps({"kernels_sha": "0" * 16, "ops": {"old": {}}}))
    ncu_report.main(["traffic", "--csv", str(csv_p), "--profile-log", str(log_p),
                     "--workload", "w", "--command", "cmd", "--out", str(out_p),
                     "--json", str(js_p), "--sha", "f" * 16])
    d = json.loads(js_p.read_text())
    assert d["kernels_sha"] == "f" * 16 and list(d["ops"]) == ["w"]
    a, b = d["ops"]["w"]["a"], d["ops"]["w"]["b"]
    assert a["dram_read_bytes"] == 200 and a["dram_write_bytes"] == 20   # per launch
    assert a["dram_bytes_per_launch"] == 220
    assert b["dram_read_bytes"] == 70 and b["dram_write_bytes"] == 0     # (50+10+70+10)/2
    md = out_p.read_text()
    assert "`kern_b`, `colreduce`" in md and "| a |" in md and "1.10 |" in md  # 220/200
    # the same hash merges a second workload in
    ncu_report.main(["traffic", "--csv", str(csv_p), "--profile-log", str(log_p),
                     "--workload", "w2", "--command", "cmd", "--out", str(out_p),
                     "--json", str(js_p), "--sha", "f" * 16])
    assert sorted(json.loads(js_p.read_text())["ops"]) == ["w", "w2"]


def test_traffic_report_rejects_a_launch_count_mismatch(tmp_path):
    csv_p, log_p = tmp_path / "t.csv", tmp_path / "p.log"
    _csv(csv_p, [(0, "void k(int)", "(1, 1, 1)", "(32, 1, 1)", "dram__bytes_read.sum",
                  "byte", 1)])
    _json_line(log_p, {"launch_order": ["a", "a"], "launches_per_op": 2,
                       "algorithmic_bytes": {"a": 1}})
    with pytest.raises(SystemExit):
        ncu_report.main(["traffic", "--csv", str(csv_p), "--profile-log", str(log_p),
                         "--workload", "w", "--command", "c", "--out", str(tmp_path / "o.md")])


def test_launch_list_groups_by_position_in_the_step(tmp_path):
    csv_p, log_p, out_p = tmp_path / "l.csv", tmp_path / "b.log", tmp_path / "l.md"
    # a step of 3 launches: op x (1 launch), op y (main + reduction); 2 steps
    seq = [("kx", 2000), ("ky", 1000), ("colreduce", 1000)] * 2
    _csv(csv_p, [(i, f"void {k}(int)", "(8, 1, 1)", "(256, 1, 1)", "gpu__time_duration.sum",
                  "ns", t) for i, (k, t) in enumerate(seq)])
    _json_line(log_p, {"per_op": {"x": {"launches": 1, "us": 2.0},
                                  "y": {"launches": 2, "us": 2.0}},
                       "ms_per_step": 0.004, "config": {"workload": "w"}})
    ncu_report.main(["launches", "--csv", str(csv_p), "--bench-log", str(log_p),
                     "--command", "c", "--out", str(out_p)])
    md = out_p.read_text()
    assert "6 launches = 2 graph replays of the step (3 launches per step)" in md
    assert "| x | 2.00 | 50.0% | 2.00 | 50.0% |" in md   # per step, share
    assert "| y | 2.00 | 50.0% | 2.00 | 50.0% |" in md
    with pytest.raises(SystemExit):                   # not a whole number of steps
        _csv(csv_p, [(0, "void kx(int)", "(8, 1, 1)", "(256, 1, 1)",
                      "gpu__time_duration.sum", "ns", 1)])
        ncu_report.main(["launches", "--csv", str(csv_p), "--bench-log", str(log_p),
                         "--command", "c", "--out", str(out_p)])


def test_bench_reads_traffic_only_for_the_current_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("softmax_bwd", "bert-base") is None       # no file
    entry = {"softmax_bwd": {"dram_bytes_per_launch": 123}}
    (prof / "ncu_traffic.json").write_text(json.dumps(
        {"kernels_sha": ncu_report.kernels_sha(), "ops": {"bert-base": entry}}))
    assert bench.ncu_traffic("softmax_bwd", "bert-base") == 123
    assert bench.ncu_traffic("softmax_bwd", "gpt2-large") is None      # other workload
    (prof / "ncu_traffic.json").write_text(json.dumps(
        {"kernels_sha": "0" * 16, "ops": {"bert-base": entry}}))
    assert bench.ncu_traffic("softmax_bwd", "bert-base") is None       # stale sources
    assert os.path.isdir(prof)


def test_range_report_subtracts_the_flush_and_divides_by_launches(tmp_path):
    # Two range captures: 4 launches each, a 512 MB flush read in the range.
    flush = 512 << 20
    for tag, op, rd, wr, alg in [("a", "softmax_bwd", 4 * 64e6 + flush, 4 * 51e6, 111e6),
                                 ("b", "ln2_bwd", 8 * 12.6e6 + flush, 8 * 6.9e6, 18.9e6)]:
        n = 4 if tag == "a" else 8
        _csv(tmp_path / f"{tag}.csv", [
            ("0", "range", "", "", "dram__bytes_read.sum", "byte", f"{rd:.0f}"),
            ("0", "range", "", "", "dram__bytes_write.sum", "byte", f"{wr:.0f}"),
            ("0", "range", "", "", "gpu__time_duration.sum", "ns", "1000")])
        _json_line(tmp_path / f"{tag}.log", {
            "profile_op": op, "workload": "bert-base", "kernels_sha": "abc", "buffer_sets": n,
            "launches_per_op": 1, "flush_read_bytes": flush, "launch_order": [op] * n,
            "algorithmic_bytes": {op: alg}})
    out, js = tmp_path / "r.md", tmp_path / "t.json"
    ncu_report.main(["range", "--case", f"x={tmp_path / 'a.csv'},{tmp_path / 'a.log'}",
                     "--case", f"y={tmp_path / 'b.csv'},{tmp_path / 'b.log'}",
                     "--command", "cmd", "--out", str(out), "--json", str(js)])
    d = json.load(open(js))
    assert d["kernels_sha"] == "abc"
    e = d["ops"]["bert-base"]["softmax_bwd"]
    assert e["dram_read_bytes"] == 64000000 and e["dram_write_bytes"] == 51000000
    e = d["ops"]["bert-base"]["ln2_bwd"]
    assert e["dram_read_bytes"] == 12600000 and e["dram_write_bytes"] == 6900000
    assert "| bert-base | softmax_bwd | 4 |" in open(out).read()
