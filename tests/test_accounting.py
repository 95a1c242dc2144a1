"""The stage-accounting report (sharded_emulated_reduce_gb300.accounting) on the CPU.

Its figures come from the library's zero_memory_bytes; here they must equal the oracle's
accounting for every named workload and stage, reproduce the pages' printed totals (a 7B
model's replicated state is about 112 GB, a 100B model's about 1.6 TB: ZeRO explainer,
"The 16 Bytes per Parameter Audit" and Chapter 01 "The Replication Trap"), and show the
stage ladder's reductions (about 4x, about 8x, and Nd: Chapter 02 "What each stage
shards" and the stage table after Chapter 05).
"""
import contextlib
import io
import json
import os

import oracle
from sharded_emulated_reduce_gb300 import accounting
from synth import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "accounting.json")


def test_every_workload_matches_the_oracle():
    reports = accounting.workload_reports()
    assert [r["workload"] for r in reports] == list(wl.WORKLOADS)
    for r in reports:
        for st in accounting.STAGES:
            assert r["bytes_per_rank"][st] == oracle.memory_bytes(r["n_params"], r["nd"],
                                                                  r["align"], st), (r, st)


def test_printed_totals_of_the_pages():
    with open(GOLDEN) as f:
        g = json.load(f)
    for key in ("model_7B", "model_100B"):
        case = g[key]
        r = accounting.stage_report(case["params"], 64)
        assert r["bytes_per_rank"][0] == case["bytes"]
        assert r["bytes_per_rank"][0] == g["bytes_per_param_replicated"]["value"] * case["params"]


def test_stage_ladder_reductions():
    # at Nd = 64 with the shards dividing the model: 16 / (4 + 12/64), 16 / (2 + 14/64), 64
    r = accounting.stage_report(13_000_000_000, 64)
    red = r["reduction"]
    assert red[0] == 1.0 and red[3] == 64.0
    assert abs(red[1] - 16 / (4 + 12 / 64)) < 1e-12 and abs(red[2] - 16 / (2 + 14 / 64)) < 1e-12
    # the printed limits as Nd grows
    big = accounting.stage_report(2 ** 40, 2 ** 16)["reduction"]
    assert 3.99 < big[1] < 4.0 and 7.99 < big[2] < 8.0 and big[3] == 2 ** 16
    # padding: a rank holds its whole padded shard
    padded = accounting.stage_report(1001, 8, align=128)
    assert padded["bytes_per_rank"][3] == 16 * 128


def test_command_line_table_and_json():
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert accounting.main([]) == 0
    text = out.getvalue()
    for name in wl.WORKLOADS:
        assert name in text
    assert "ZeRO-3" in text and "64.00x" in text
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert accounting.main(["--n", "7e9", "--nd", "8", "--json"]) == 0
    (r,) = json.loads(out.getvalue())
    assert r["bytes_per_rank"]["0"] == 112_000_000_000 and r["bytes_per_rank"]["3"] == 14_000_000_000
