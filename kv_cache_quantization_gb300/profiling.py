"""Bookkeeping for measured DRAM traffic of the decode-attention launches.

``profiles/decode_attention_traffic.json`` holds, per workload, the DRAM bytes (read +
written) of one decode-attention call as ncu counted them, together with a digest of the
kernel sources they were counted on.  ``bench.py`` reports the figure only while the digest
still matches the sources; once a kernel changes, the figure is stale and it reports null.

    python -m kv_cache_quantization_gb300.profiling <ncu csv> <workload>

reads an ncu ``--csv`` export with the metrics ``dram__bytes_read.sum`` and
``dram__bytes_write.sum`` of one captured launch of the workload's split kernel (the dominant
kernel of a decode call) and records its bytes under the workload's name.
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
    """[(kernel name, dram bytes read + written)] of every launch in an ncu ``--csv`` export
    (one row per launch and metric)."""
    with open(path, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    head = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    cols = rows[head]
    ci, cn, cm, cu, cv = (cols.index(x) for x in ("ID", "Kernel Name", "Metric Name",
                                                  "Metric Unit", "Metric Value"))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    launches = {}
    for r in rows[head + 1:]:
        if len(r) <= cv or r[cm] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        name, total = launches.get(r[ci], (r[cn], 0.0))
        launches[r[ci]] = (name, total + float(r[cv].replace(",", "")) * scale.get(r[cu], 1))
    return [launches[k] for k in sorted(launches, key=int)]


def record(csv_path, workload, how):
    """Stores the DRAM bytes of the last launch in an ncu CSV export (one capture of the
    workload's split kernel) under `workload`, with the current sources' digest."""
    launches = _launch_bytes(csv_path)
    if not launches:
        raise SystemExit(f"no launch in {csv_path}")
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    name, nbytes = launches[-1]
    data[workload] = {"bytes": int(round(nbytes)), "sources": kernel_sources_digest(),
                      "kernel": name.split("(")[0][:80], "how": how}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    if len(sys.argv) != 3:
        raise SystemExit(__doc__)
    record(sys.argv[1], sys.argv[2], "one ncu capture of the split kernel")
