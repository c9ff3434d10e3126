"""Host-side parts of bench.py (no GPU): the reference arm's JSON line, the
peak each dtype is measured against, and the rule that a stored DRAM traffic
figure is reported only for the kernel sources it was captured on."""

import argparse
import io
import json
import os
from contextlib import redirect_stdout

import pytest

import bench
from tiled_attention_fa2_gb300 import inputs


def test_reference_arm_prints_one_complete_line():
    args = argparse.Namespace(steps=1, warmup=0, workload="tiny_f32", impl="reference", cpu_budget=1.0,
                              no_cpu_baseline=False, pass_="fwd", gpus=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference_arm(args, inputs.WORKLOADS["tiny_f32"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference" and line["gpu_launches"] == 0
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny_f32"
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["value"] > 0


def test_reference_arm_is_silent_off_rank_zero(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(steps=1, warmup=0, workload="tiny_f32", impl="reference", cpu_budget=1.0,
                              no_cpu_baseline=False, pass_="fwd", gpus=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference_arm(args, inputs.WORKLOADS["tiny_f32"])
    assert buf.getvalue() == ""


def test_each_dtype_takes_the_peak_of_its_own_contraction():
    peaks = {"bf16_tflops": 1000.0, "bf16_tflops_sustained": 900.0, "hbm_gbs": 5000.0}
    assert bench.dtype_peak("bf16", peaks)[0] == 1000.0
    assert bench.dtype_peak("e4m3", peaks)[0] == 2000.0  # nominal fp8 : bf16 dense ratio


def test_stored_traffic_is_reported_only_for_its_own_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"w": {"kernel_source_hash": bench.kernel_source_hash(), "dram_bytes_per_launch": 123}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "tiled_attention_fa2_gb300" / "csrc"
    csrc.mkdir(parents=True)
    real = os.path.join(os.path.dirname(bench.__file__), "tiled_attention_fa2_gb300", "csrc")
    for f in bench.FWD_SOURCES:
        (csrc / f).write_bytes(open(os.path.join(real, f), "rb").read())
    assert bench.profile_traffic("w") == 123
    assert bench.profile_traffic("other") is None
    # any change to the forward's sources hides the figure
    (csrc / "attn_tc_sm103.cuh").write_bytes(b"// changed\n" + (csrc / "attn_tc_sm103.cuh").read_bytes())
    assert bench.profile_traffic("w") is None


def test_committed_traffic_records_are_well_formed():
    # Each record names a workload and a sources hash; bench.py reports it only
    # while that hash matches the current forward sources.
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert rec, "no traffic records"
    for name, e in rec.items():
        assert name in inputs.WORKLOADS
        assert len(e["kernel_source_hash"]) == 16
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"]


@pytest.mark.parametrize("world,steps,ms,expect", [(1, 10, 20.0, 1000.0), (4, 10, 20.0, 4000.0)])
def test_job_throughput_counts_every_rank(world, steps, ms, expect):
    assert bench.job_throughput(2e12, world, steps, ms) == pytest.approx(expect)


def test_gpu_count_must_match_the_launch():
    # --gpus N is one process per GPU under torchrun; a single process asking for
    # two GPUs is refused instead of silently timing one.
    import subprocess
    import sys

    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"), "--gpus", "2",
                        "--impl", "reference"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 2 and "WORLD_SIZE=1" in r.stderr


def test_datasheet_fraction_beside_the_measured_one():
    assert bench.datasheet_fraction("bf16", 1125.0) == {"datasheet_peak": 2250.0, "frac_of_datasheet": 0.5}
    assert bench.datasheet_fraction("e4m3", 2250.0) == {"datasheet_peak": 4500.0, "frac_of_datasheet": 0.5}
    assert bench.datasheet_fraction("f32", 1.0) == {}


def test_grouped_query_workloads_read_their_own_kv_heads():
    w = inputs.WORKLOADS["prefill_gqa_bf16"]
    assert bench.kv_heads(w) == 8 and w["H"] % bench.kv_heads(w) == 0
    assert bench.kv_heads(inputs.WORKLOADS["dit_e4m3"]) == 56


def test_oracle_head_inputs_follow_the_head_map():
    # query head h of batch b reads K/V head b * H_kv + h // (H / H_kv)
    import numpy as np
    import oracle

    w = dict(B=2, H=4, Hkv=2, N=8, d=4, dtype="f32", causal=False, q_mult=1.0)
    host, ds = bench.make_host_inputs(w)
    assert tuple(host[1].shape) == (2, 2, 8, 4)
    for h in range(8):
        q, k, v = bench._oracle_head_inputs(w, host, ds, h)
        b, hq = divmod(h, 4)
        g = oracle.kv_head_of(hq, 4, 2)
        assert np.array_equal(q, host[0][b, hq].double().numpy())
        assert np.array_equal(k, host[1][b, g].double().numpy())
        assert np.array_equal(v, host[2][b, g].double().numpy())


def test_backward_pass_refuses_grouped_query_workloads():
    import subprocess
    import sys

    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"), "--pass", "bwd",
                        "--workload", "prefill_gqa_bf16"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 2 and "multi-head attention only" in r.stderr
