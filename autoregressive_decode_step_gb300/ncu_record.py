"""Write the machine-readable DRAM-traffic record of the persistent step kernel
that bench.py reads (``profiles/step_kernel_llama3_8b.json``).

Input: the CSV of one ncu capture of a step-kernel launch with the metrics
dram__bytes_read.sum and dram__bytes_write.sum, taken with ``--csv
--print-units base`` on a small case of bench.py, e.g.

    ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none \\
        --print-units base --csv -k regex:step_kernel -s 2 -c 1 --log-file traffic.csv \\
        python bench.py --layers 4 --steps 3 --warmup 3 --kv-fill synthetic \\
        --no-cpu-baseline --no-batched --no-ops --no-legs --chunk 1

(the third launch: warm-up step 3, attending ctx + 3 positions).  The record
holds the measured bytes, the launch's algorithmic bytes (every weight byte of
the captured model once plus the K/V of every attended position), their
ratio, the command, and the sha256 of the kernel's sources, so that bench.py
uses the ratio only while the kernel is unchanged.

    python -m autoregressive_decode_step_gb300.ncu_record traffic.csv --layers 4 --n-ctx 1027 \\
        --command "<the ncu command>" --out profiles/step_kernel_llama3_8b.json
"""
import argparse
import csv
import hashlib
import json
import os

from . import configs as C

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ("step.cu", "common.cuh", "internal.h")


def kernel_source_sha():
    """sha256 over the step kernel's sources (the same digest bench.py takes)."""
    h = hashlib.sha256()
    for name in SOURCES:
        with open(os.path.join(HERE, "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def read_metrics(path, kernel="step_kernel"):
    """{metric name: value} of the first launch of `kernel` in an ncu CSV."""
    with open(path, newline="") as f:
        lines = [l for l in f if l.startswith('"')]
    rows = list(csv.DictReader(lines))
    out = {}
    first_id = None
    for r in rows:
        if kernel not in r.get("Kernel Name", ""):
            continue
        if first_id is None:
            first_id = r.get("ID")
        if r.get("ID") != first_id:
            continue
        unit = r.get("Metric Unit", "")
        if unit not in ("byte", "bytes", ""):
            raise ValueError("expected bytes (ncu --print-units base), got %r" % unit)
        out[r["Metric Name"]] = float(r["Metric Value"].replace(",", ""))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("csv")
    ap.add_argument("--layers", type=int, required=True)
    ap.add_argument("--n-ctx", type=int, required=True, help="positions the captured launch attends")
    ap.add_argument("--command", required=True)
    ap.add_argument("--out", required=True)
    a = ap.parse_args()
    m = read_metrics(a.csv)
    dram = m["dram__bytes_read.sum"] + m["dram__bytes_write.sum"]
    cfg = dict(C.LLAMA3_8B, n_layer=a.layers)
    alg = C.step_bytes(cfg, a.n_ctx)
    rec = {"kernel": "ds::step_kernel (persistent batch-1 decode step)", "workload": "llama3-8b shape, %d layers, "
           "one step attending %d positions" % (a.layers, a.n_ctx),
           "kernel_source_sha256": kernel_source_sha(), "kernel_sources": list(SOURCES),
           "dram_bytes_read": m["dram__bytes_read.sum"], "dram_bytes_write": m["dram__bytes_write.sum"],
           "dram_bytes": dram, "algorithmic_bytes": alg, "ratio": dram / alg, "command": a.command}
    with open(a.out, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec))


if __name__ == "__main__":
    main()
