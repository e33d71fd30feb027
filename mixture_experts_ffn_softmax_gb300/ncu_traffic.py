"""Writes the DRAM-traffic record that bench.py reports beside a kernel's
roofline, from an Nsight Compute CSV export.

    python -m mixture_experts_ffn_softmax_gb300.ncu_traffic CSV \
        --kernel gemm1_swiglu --workload mixtral_prefill \
        --ncu-kernel-regex 'grouped_gemm' --launch 0 \
        --source mixture_experts_ffn_softmax_gb300/csrc/gemm.cu \
        --command '<the ncu command that wrote CSV>' > profiles/traffic_<kernel>_<workload>.json

CSV is the output of ``ncu --csv --print-units base --metrics
dram__bytes_read.sum,dram__bytes_write.sum ... --log-file CSV`` (one row per
launch and metric), or of ``ncu -i REP --page raw --csv --print-units base``
(one row per launch, one column per metric).  The record holds the kernel's
name in the bench line, the workload, the ncu kernel name and launch index it
was taken from, the read and write bytes of that launch, their sum, and the
first 16 hex digits of the SHA-256 of the kernel's source file: bench.py
reports the traffic only while that source is unchanged.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import re
import sys

_UNIT = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
         "kibyte": 1024, "mibyte": 1024 ** 2, "gibyte": 1024 ** 3}
READ, WRITE = "dram__bytes_read.sum", "dram__bytes_write.sum"


def source_hash(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _to_bytes(value: str, unit: str) -> float:
    v = float(value.replace(",", ""))
    return v * _UNIT.get(unit.strip().lower() or "byte", 1)


def _rows(text: str):
    """CSV rows of the export, from its header line on (ncu prints its own
    log lines, prefixed '==', before the table)."""
    lines = [ln for ln in text.splitlines() if ln.strip() and not ln.startswith("==")]
    return list(csv.reader(io.StringIO("\n".join(lines))))


def launches(text: str, kernel_regex: str):
    """[(kernel name, read bytes, write bytes)] per matching launch, in order."""
    rows = _rows(text)
    if not rows:
        return []
    head = rows[0]
    pat = re.compile(kernel_regex)
    out = []
    if "Metric Name" in head:
        # long form: one row per (launch, metric)
        i_id, i_name = head.index("ID"), head.index("Kernel Name")
        i_metric, i_unit, i_val = (head.index("Metric Name"), head.index("Metric Unit"),
                                   head.index("Metric Value"))
        per = {}
        order = []
        for r in rows[1:]:
            if len(r) <= i_val or not pat.search(r[i_name]):
                continue
            key = r[i_id]
            if key not in per:
                per[key] = [r[i_name], None, None]
                order.append(key)
            if r[i_metric] == READ:
                per[key][1] = _to_bytes(r[i_val], r[i_unit])
            elif r[i_metric] == WRITE:
                per[key][2] = _to_bytes(r[i_val], r[i_unit])
        out = [tuple(per[k]) for k in order]
    else:
        # raw page: header row, then a units row, then one row per launch
        i_name = head.index("Kernel Name")
        i_r, i_w = head.index(READ), head.index(WRITE)
        units = rows[1]
        for r in rows[2:]:
            if len(r) <= max(i_r, i_w) or not pat.search(r[i_name]):
                continue
            out.append((r[i_name], _to_bytes(r[i_r], units[i_r]), _to_bytes(r[i_w], units[i_w])))
    return [t for t in out if t[1] is not None and t[2] is not None]


def record(text: str, kernel: str, workload: str, kernel_regex: str, launch: int,
           source: str, command: str) -> dict:
    found = launches(text, kernel_regex)
    if not found or launch >= len(found):
        raise SystemExit(f"no launch {launch} of a kernel matching {kernel_regex!r} "
                         f"with {READ} and {WRITE} ({len(found)} found)")
    name, rd, wr = found[launch]
    return {"kernel": kernel, "workload": workload, "ncu_kernel": name, "launch": launch,
            "dram_bytes_read": int(rd), "dram_bytes_write": int(wr),
            "traffic_bytes_per_launch": int(rd + wr), "source": source,
            "source_sha256_16": source_hash(source), "command": command}


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("csv")
    ap.add_argument("--kernel", required=True)
    ap.add_argument("--workload", required=True)
    ap.add_argument("--ncu-kernel-regex", required=True)
    ap.add_argument("--launch", type=int, default=0)
    ap.add_argument("--source", required=True)
    ap.add_argument("--command", required=True)
    a = ap.parse_args(argv)
    with open(a.csv) as f:
        text = f.read()
    rec = record(text, a.kernel, a.workload, a.ncu_kernel_regex, a.launch, a.source, a.command)
    json.dump(rec, sys.stdout, indent=1)
    sys.stdout.write("\n")


if __name__ == "__main__":
    main()
