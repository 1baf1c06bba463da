"""Host side of the measurement: the DRAM-traffic record of the persistent
step kernel (written from an ncu CSV by ``ncu_record``) and its use by
``bench.py``, which reports a launch's traffic only while the record was taken
on the current kernel source.  No GPU: the CSV is a small synthetic one in
ncu's ``--csv --print-units base`` layout."""
import json
import subprocess
import sys

import pytest

import bench
from autoregressive_decode_step_gb300 import configs as C
from autoregressive_decode_step_gb300 import ncu_record

HEADER = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",' \
         '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'


def csv_line(launch_id, kernel, metric, value, unit="byte"):
    return ('"%d","1","python","h","%s","1","7","(288, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler '
            'metrics","%s","%s","%s"\n' % (launch_id, kernel, metric, unit, value))


def write_csv(path, rows):
    with open(path, "w") as f:
        f.write("==PROF== a line ncu prints before the table\n")
        f.write(HEADER)
        for r in rows:
            f.write(csv_line(*r))


def test_read_metrics_takes_the_first_step_kernel_launch(tmp_path):
    p = tmp_path / "t.csv"
    write_csv(p, [(0, "void ds::other_kernel(int)", "dram__bytes_read.sum", "5"),
                  (1, "void ds::step_kernel<bf16, bf16, 4>(ds::StepParams)", "dram__bytes_read.sum", "1,000"),
                  (1, "void ds::step_kernel<bf16, bf16, 4>(ds::StepParams)", "dram__bytes_write.sum", "24"),
                  (2, "void ds::step_kernel<bf16, bf16, 4>(ds::StepParams)", "dram__bytes_read.sum", "7")])
    assert ncu_record.read_metrics(str(p)) == {"dram__bytes_read.sum": 1000.0, "dram__bytes_write.sum": 24.0}


def test_read_metrics_refuses_scaled_units(tmp_path):
    p = tmp_path / "t.csv"
    write_csv(p, [(1, "void ds::step_kernel<bf16, bf16, 4>(ds::StepParams)", "dram__bytes_read.sum", "2.8",
                   "Gbyte")])
    with pytest.raises(ValueError):
        ncu_record.read_metrics(str(p))


def test_record_round_trip_and_source_check(tmp_path, monkeypatch):
    """The written record holds DRAM bytes / algorithmic bytes of the captured
    model (every weight byte once + the K/V of the attended positions), and
    bench.py returns that ratio for the current source's digest only."""
    layers, n_ctx = 4, 1027
    alg = C.step_bytes(dict(C.LLAMA3_8B, n_layer=layers), n_ctx)
    read, write = int(alg * 1.002), 7_000_000
    p = tmp_path / "t.csv"
    write_csv(p, [(3, "void ds::step_kernel<bf16, bf16, 4>(ds::StepParams)", "dram__bytes_read.sum", str(read)),
                  (3, "void ds::step_kernel<bf16, bf16, 4>(ds::StepParams)", "dram__bytes_write.sum", str(write))])
    out = tmp_path / "rec.json"
    subprocess.run([sys.executable, "-m", "autoregressive_decode_step_gb300.ncu_record", str(p), "--layers",
                    str(layers), "--n-ctx", str(n_ctx), "--command", "ncu ...", "--out", str(out)],
                   check=True, capture_output=True)
    rec = json.loads(out.read_text())
    assert rec["algorithmic_bytes"] == alg
    assert rec["dram_bytes"] == read + write
    assert rec["ratio"] == pytest.approx((read + write) / alg)
    assert rec["kernel_source_sha256"] == ncu_record.kernel_source_sha()
    monkeypatch.setattr(bench, "STEP_TRAFFIC", str(out))
    assert bench.traffic_ratio(bench.kernel_source_sha()) == pytest.approx((read + write) / alg)
    assert bench.traffic_ratio("0" * 64) is None
    monkeypatch.setattr(bench, "STEP_TRAFFIC", str(tmp_path / "missing.json"))
    assert bench.traffic_ratio(bench.kernel_source_sha()) is None


def test_committed_record_is_consistent():
    """The committed record's ratio is its DRAM bytes over its algorithmic
    bytes, and those are the captured workload's (4 layers, 1,027 positions)."""
    with open(bench.STEP_TRAFFIC) as f:
        rec = json.load(f)
    assert rec["dram_bytes"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert rec["ratio"] == pytest.approx(rec["dram_bytes"] / rec["algorithmic_bytes"])
    assert rec["algorithmic_bytes"] == C.step_bytes(dict(C.LLAMA3_8B, n_layer=4), 1027)
    assert 1.0 <= rec["ratio"] < 1.05
