"""Bookkeeping for measured DRAM traffic of the decode-attention launches.

``profiles/decode_attention_traffic.json`` holds, per workload, the DRAM bytes (read +
written) of one decode-attention call as ncu counted them, together with a digest of the
kernel sources they were counted on.  ``bench.py`` reports the figure only while the digest
still matches the sources; once a kernel changes, the figure is stale and it reports null.

    python -m kv_cache_quantization_gb300.profiling <ncu csv> <workload> [<workload> ...]

reads an ncu ``--csv --page raw`` export with the metrics ``dram__bytes_read.sum`` and
``dram__bytes_write.sum``, sums every launch of each decode call (the query-operand kernel
and the split kernel, or the asymmetric split kernel and its merge) and records it under the
given workload names, one call per name, in the order they were captured.
"""
from __future__ import annotations

import csv
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_attention_traffic.json")
# the sources whose code decides a decode call's DRAM traffic
SOURCES = ["decode_tc.cu", "tile_mma.h", "tc_ptx.h", "decode_args.h", "decode_asym.cu",
           "attention.cu"]


def kernel_sources_digest() -> str:
    h = hashlib.sha256()
    for name in SOURCES:
        with open(os.path.join(HERE, "csrc", name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """(bytes, note): the DRAM bytes of one decode call of `workload`, or None with the
    reason when there is no figure for the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None, "no traffic record"
    if not isinstance(rec, dict):
        return None, "no traffic record for this workload"
    if rec.get("sources") != kernel_sources_digest():
        return None, "kernel sources changed since the counters were taken"
    return int(rec["bytes"]), (f"ncu dram__bytes_read.sum + dram__bytes_write.sum, "
                               f"{rec.get('how', 'one capture')}")


def _launch_bytes(path):
    """[(kernel name, dram bytes)] of every launch in an ncu raw-page CSV export."""
    with open(path, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    head = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    cols = rows[head]
    name_i = cols.index("Kernel Name")
    rd, wr = cols.index("dram__bytes_read.sum"), cols.index("dram__bytes_write.sum")
    units = rows[head + 1] if not rows[head + 1][0].strip().isdigit() else None
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6,
             "GB": 1e9, "B": 1}
    out = []
    for r in rows[head + (2 if units else 1):]:
        def val(i):
            s = float(r[i].replace(",", ""))
            return s * (scale.get(units[i], 1) if units else 1)
        out.append((r[name_i], val(rd) + val(wr)))
    return out


def record(csv_path, workloads, how):
    launches = _launch_bytes(csv_path)
    calls, cur = [], 0.0
    for name, b in launches:
        cur += b
        # a call ends with its split kernel (symmetric) or the merge (asymmetric)
        if "decode_tc_kernel" in name or "merge_kernel" in name:
            calls.append(cur)
            cur = 0.0
    if len(calls) < len(workloads):
        raise SystemExit(f"{len(calls)} decode calls in {csv_path}, {len(workloads)} names given")
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    digest = kernel_sources_digest()
    for w, b in zip(workloads, calls):
        data[w] = {"bytes": int(round(b)), "sources": digest, "how": how}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    if len(sys.argv) < 3:
        raise SystemExit(__doc__)
    record(sys.argv[1], sys.argv[2:], "one capture of each call")
