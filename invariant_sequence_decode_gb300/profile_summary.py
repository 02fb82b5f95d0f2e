"""Summaries of ncu CSV output (``ncu --csv --log-file ...``), written as
short text or JSON for the repository's profile notes.

  python -m invariant_sequence_decode_gb300.profile_summary launches CSV
      per kernel: launches, total device time, share (from
      gpu__time_duration.sum; serialised, cold-cache: compare shares)
  python -m invariant_sequence_decode_gb300.profile_summary traffic CSV OUT.json [--kernels REGEX] [--per N]
      DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the last N
      matching launches (one layer's projections launched back to back), per
      launch and summed, with the SHA-256 prefix of the matvec sources they
      were taken with; bench.py reports the figure only while that hash matches.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import re
import statistics
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
MATVEC_SOURCES = ("matvec.cu", "matvec_tma.cu", "matvec_mma.cu", "ring.cuh", "common.cuh")
_UNIT = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "B": 1, "KB": 1e3, "MB": 1e6, "GB": 1e9,
         "ns": 1e-3, "us": 1.0, "ms": 1e3, "nsecond": 1e-3, "usecond": 1.0, "msecond": 1e3,
         "second": 1e6}


def matvec_sources_hash() -> str:
    """First 16 hex digits of the SHA-256 over the matvec kernels' sources."""
    h = hashlib.sha256()
    for f in MATVEC_SOURCES:
        h.update(open(os.path.join(PKG, "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def read_rows(path: str):
    """(kernel name, launch id, metric name, value in bytes or microseconds) per CSV row."""
    text = open(path).read()
    start = text.find('"ID"')
    rows = list(csv.reader(text[start:].splitlines()))
    hdr = rows[0]
    ix = {k: hdr.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value")}
    for r in rows[1:]:
        if len(r) < len(hdr):
            continue
        v = float(r[ix["Metric Value"]].replace(",", ""))
        yield r[ix["Kernel Name"]], int(r[ix["ID"]]), r[ix["Metric Name"]], v * _UNIT.get(r[ix["Metric Unit"]], 1.0)


def short(name: str) -> str:
    return re.sub(r"\(.*", "", name).replace("void ", "")


def launches(path: str) -> str:
    per = {}
    for name, _id, metric, us in read_rows(path):
        if metric == "gpu__time_duration.sum":
            per.setdefault(short(name), []).append(us)
    total = sum(sum(v) for v in per.values())
    lines = [f"{'kernel':70s} {'launches':>8s} {'total us':>10s} {'mean us':>9s} {'share':>7s}"]
    for k, v in sorted(per.items(), key=lambda kv: -sum(kv[1])):
        lines.append(f"{k[:70]:70s} {len(v):8d} {sum(v):10.2f} {statistics.mean(v):9.2f} {sum(v) / total:7.1%}")
    lines.append(f"{'all':70s} {sum(len(v) for v in per.values()):8d} {total:10.2f}")
    return "\n".join(lines)


def traffic(path: str, regex: str, per: int) -> dict:
    by_id = {}
    for name, i, metric, b in read_rows(path):
        if re.search(regex, name) and metric in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            by_id.setdefault(i, {"kernel": short(name)})[metric] = b
    last = sorted(by_id)[-per:]
    b = [int(by_id[i].get("dram__bytes_read.sum", 0) + by_id[i].get("dram__bytes_write.sum", 0)) for i in last]
    return {"matvec_src_sha256_16": matvec_sources_hash(), "kernels": [by_id[i]["kernel"] for i in last],
            "launches_per_group": per, "traffic_bytes_per_group": sum(b), "traffic_bytes_per_launch": b}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("what", choices=["launches", "traffic"])
    ap.add_argument("csv")
    ap.add_argument("out", nargs="?")
    ap.add_argument("--kernels", default="q8_matvec")
    ap.add_argument("--per", type=int, default=4)
    a = ap.parse_args(argv)
    if a.what == "launches":
        print(launches(a.csv))
    else:
        d = traffic(a.csv, a.kernels, a.per)
        text = json.dumps(d, indent=1)
        if a.out:
            open(a.out, "w").write(text + "\n")
        print(text)


if __name__ == "__main__":
    sys.exit(main())
