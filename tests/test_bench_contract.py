"""The bench's one-line JSON output: the keys and types every line must carry.

The reference arm (the oracle on the host cores) runs here on the CPU; the GPU lines (the
shard step with its end-to-end, roofline, CPU-baseline and clock objects, and the
gather) run with a few steps on a GPU."""
import contextlib
import io
import json

import pytest

import bench

COMMON = {"metric": str, "value": float, "unit": str, "n_gpus": int, "steps": int,
          "warmup": int, "ms_per_step": float, "higher_is_better": bool, "scaling": str,
          "dtype": str, "data": str, "config": dict}


def run(argv):
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        rc = bench.main(argv)
    assert rc == 0
    lines = [l for l in out.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def check_common(d):
    for k, t in COMMON.items():
        assert isinstance(d[k], t), k
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["vs_baseline"] is None
    assert isinstance(d["config"]["workload"], str)


def check_cpu_baseline(c):
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1
    assert isinstance(c["unit"], str) and isinstance(c["sample"], str)


def check_roofline(r):
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert abs(r["frac_of_nominal"] - r["achieved"] / bench.NOMINAL_HBM_GBS) < 1e-9


def test_default_workload_is_the_largest_single_gpu_config():
    assert bench.DEFAULT_WORKLOAD == "zero3_13b_rank0_nd64"


def test_reference_arm_line(tmp_path):
    log = tmp_path / "results.jsonl"
    d = run(["--impl", "reference", "--workload", "zero2_tiny_1m_nd4", "--steps", "2",
             "--warmup", "3", "--cpu-seconds", "0.5", "--results", str(log)])
    recs = [json.loads(l) for l in log.read_text().splitlines()]
    assert len(recs) == 1 and recs[0]["impl"] == "reference"
    assert recs[0]["kernel"] == "whole step"
    assert recs[0]["params_per_s"] == d["value"] and recs[0]["oracle_cores"] >= 1
    check_common(d)
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    check_cpu_baseline(d["cpu_baseline"])
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    check_cpu_baseline(d["gather"]["cpu_baseline"])
    # the oracle arm names the workload exactly as the GPU arm does
    from synth import workloads as wl
    assert d["config"] == bench.config_of(wl.WORKLOADS["zero2_tiny_1m_nd4"], 1)
    assert d["scaling"] == "strong"


def test_process_spans():
    from synth import workloads as wl
    w5 = wl.WORKLOADS["zero3_13b_rank0_nd64"]
    spans = [bench.process_span(w5, 4, g) for g in range(4)]
    assert [(w.r0, w.r1, k) for w, k in spans] == [(g, g + 1, "weak") for g in range(4)]
    assert bench.job_params(w5, 4) == 4 * w5.span()[2]
    w2 = wl.WORKLOADS["gpt2_small_flat_nd8"]
    spans = [bench.process_span(w2, 2, g) for g in range(2)]
    assert [(w.r0, w.r1, k) for w, k in spans] == [(0, 4, "strong"), (4, 8, "strong")]
    assert bench.job_params(w2, 2) == w2.n


@pytest.mark.gpu
def test_step_line(tmp_path):
    log = tmp_path / "results.jsonl"
    d = run(["--workload", "zero2_tiny_1m_nd4", "--steps", "20", "--warmup", "3",
             "--cpu-seconds", "1", "--results", str(log)])
    # the results log: one record per kernel that ran (the one-launch step here), the
    # whole step and the gather
    recs = {r["kernel"]: r for r in map(json.loads, log.read_text().splitlines())}
    assert set(recs) == {"whole step", "gather", d["roofline"]["kernel"]}
    assert recs["whole step"]["params_per_s"] == d["value"]
    assert recs["whole step"]["oracle_s_per_step"] > 0
    assert abs(recs[d["roofline"]["kernel"]]["frac_of_peak"] - d["roofline"]["frac"]) < 1e-9
    assert recs["gather"]["params_per_s"] == d["gather"]["value"]
    check_common(d)
    assert d["unit"] == "params/s" and d["higher_is_better"] is True
    # the 1M workload is timed with an L2 flush before every step, each step between its
    # own events: the median step is reported beside the mean
    assert 0 < d["ms_per_step_median"] <= 2 * d["ms_per_step"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 4 * 2 * 1048576
    assert e["d2h_bytes_per_step"] > 0 and set(e["by_mode"]) == {"copy", "copy_overlap",
                                                                  "zero_copy"}
    assert e["value"] == max(e["by_mode"].values())
    p = e["with_params_to_host"]
    assert p["value"] > 0 and p["d2h_bytes_per_step"] == e["d2h_bytes_per_step"] + 2 * 1048576
    assert d["gpu_launches"] >= 20  # one launch per step for this small span, else two or three
    check_roofline(d["roofline"])
    check_cpu_baseline(d["cpu_baseline"])
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
    assert d["last_step"]["skipped"] == 0
    # the gather of the step's output (one full-buffer layer here) in the same line
    g = d["gather"]
    assert g["value"] > 0 and g["layers"] == 1 and g["params_per_call"] == 1048576
    assert g["gpu_launches"] == 20
    check_roofline(g["roofline"])
    check_cpu_baseline(g["cpu_baseline"])
    assert d["hot_path"]["ms_per_pass"] > 0
    # both arms name the workload identically
    ref = run(["--impl", "reference", "--workload", "zero2_tiny_1m_nd4", "--steps", "2",
               "--warmup", "3", "--cpu-seconds", "0"])
    assert ref["config"] == d["config"] and ref["scaling"] == d["scaling"]


@pytest.mark.gpu
def test_gather_line():
    d = run(["--op", "gather", "--workload", "zero3_1p3b_rank0_nd64", "--steps", "3",
             "--warmup", "3", "--cpu-seconds", "0.5"])
    check_common(d)
    assert d["gpu_launches"] == 3 and d["roofline"]["kernel"] == "gather"
    check_cpu_baseline(d["cpu_baseline"])


@pytest.mark.gpu
def test_full_buffer_gather_line():
    # a workload without a layer table: the ZeRO-1/2 all-gather into one flat buffer
    d = run(["--op", "gather", "--workload", "flat_32m_nd8", "--steps", "3", "--warmup", "3",
             "--cpu-seconds", "0"])
    check_common(d)
    assert d["config"]["layers"] == 1 and d["gpu_launches"] == 3


@pytest.mark.gpu
def test_gather_prefetch_line():
    d = run(["--op", "gather", "--workload", "zero3_1p3b_rank0_nd64", "--steps", "3",
             "--warmup", "3", "--cpu-seconds", "0", "--prefetch"])
    check_common(d)
    layers = d["config"]["layers"]
    assert d["gpu_launches"] == 3 * layers
    ready = d["prefetch"]["layer_ready_ms"]
    # consecutive layers run on two streams, so their events need not complete in order
    assert len(ready) == layers and min(ready) > 0 and ready[0] < max(ready)
