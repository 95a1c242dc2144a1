"""Per-rank model-state memory of the ZeRO stages: a report built on zero_memory_bytes.

Mixed-precision Adam keeps 16 bytes per parameter: a 2-byte fp16 weight, a 2-byte fp16
gradient and 12 bytes of fp32 optimizer state (master weight, momentum, variance) (ZeRO
explainer, "The 16 Bytes per Parameter Audit"). Plain data parallelism replicates all of
it on every rank; ZeRO-1 partitions the optimizer state, ZeRO-2 the gradients as well,
ZeRO-3 the parameters too, which takes the per-rank footprint down by about 4x, about 8x
and by Nd (Chapter 02 "What each stage shards"; the stage table after Chapter 05). This
module asks the library (zero_memory_bytes, host only: no GPU is needed) for the per-rank
bytes of stages 0 to 3 of a flat buffer and prints them with the reduction against
stage 0.

    python -m sharded_emulated_reduce_gb300.accounting                  # the named workloads
    python -m sharded_emulated_reduce_gb300.accounting --n 7e9 --nd 64  # one model
"""
from __future__ import annotations

import argparse
import json
import sys

from . import zero_memory_bytes

STAGES = (0, 1, 2, 3)
STAGE_NAMES = {0: "DP (replicated)", 1: "ZeRO-1 P_os", 2: "ZeRO-2 P_os+g", 3: "ZeRO-3 P_os+g+p"}


def stage_report(n_params: int, nd: int, align: int = 1) -> dict:
    """Per-rank bytes of each stage and its reduction against stage 0 (replication)."""
    per_rank = {st: zero_memory_bytes(n_params, nd, align, st) for st in STAGES}
    return {"n_params": n_params, "nd": nd, "align": align,
            "bytes_per_rank": per_rank,
            "reduction": {st: per_rank[0] / per_rank[st] for st in STAGES}}


def workload_reports() -> list[dict]:
    """The report for every named synthetic workload, at its own Nd and alignment."""
    from synth import workloads as wl
    out = []
    for w in wl.WORKLOADS.values():
        r = stage_report(w.n, w.nd, w.align)
        r["workload"] = w.name
        out.append(r)
    return out


def _gb(x: int) -> str:
    return f"{x / 1e9:,.3f}"


def format_table(reports: list[dict]) -> str:
    head = (f"{'workload':<24} {'N':>15} {'Nd':>4}  "
            + "  ".join(f"{STAGE_NAMES[st] + ' GB':>22}" for st in STAGES))
    lines = [head, "-" * len(head)]
    for r in reports:
        cells = []
        for st in STAGES:
            b = r["bytes_per_rank"][st]
            cells.append(f"{_gb(b):>13} ({r['reduction'][st]:6.2f}x)")
        lines.append(f"{r.get('workload', '-'):<24} {r['n_params']:>15,} {r['nd']:>4}  "
                     + "  ".join(f"{c:>22}" for c in cells))
    return "\n".join(lines)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--n", type=float, help="parameters (default: every named workload)")
    ap.add_argument("--nd", type=int, default=64, help="data-parallel ranks")
    ap.add_argument("--align", type=int, default=1, help="shard alignment in elements")
    ap.add_argument("--json", action="store_true", help="print JSON instead of a table")
    a = ap.parse_args(argv)
    reports = ([stage_report(int(a.n), a.nd, a.align)] if a.n is not None
               else workload_reports())
    if a.json:
        print(json.dumps(reports))
    else:
        print(format_table(reports))
    return 0


if __name__ == "__main__":
    sys.exit(main())
