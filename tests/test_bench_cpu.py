"""Host-only checks of bench.py's bookkeeping: the gate on the recorded GEMM traffic (a hash of
the kernel sources that ignores comments) and the `config` both arms report."""
import os
import shutil

import bench


def _copy_sources(tmp_path):
    for rel in bench.GEMM_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)


def test_gemm_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.gemm_source_sha256()
    gemm = tmp_path / bench.GEMM_SOURCES[0]
    text = gemm.read_text()

    # a new whole-line comment, a trailing comment and blank lines leave the hash alone
    gemm.write_text("// a note\n\n" + text.replace("namespace adahop {", "namespace adahop {  // here", 1) + "\n\n")
    assert bench.gemm_source_sha256() == base

    # any change to the code changes it
    gemm.write_text(text.replace("constexpr int kThreads = 320;", "constexpr int kThreads = 352;", 1))
    assert "kThreads = 352" in gemm.read_text()
    assert bench.gemm_source_sha256() != base


def test_gemm_traffic_is_null_for_other_sources(tmp_path, monkeypatch):
    _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    gemm = tmp_path / bench.GEMM_SOURCES[0]
    gemm.write_text(gemm.read_text().replace("constexpr int kEpiWarps = 8;", "constexpr int kEpiWarps = 4;", 1))
    assert bench.gemm_traffic() is None


def test_reference_arm_reports_the_gpu_arms_config():
    import oracle as O
    plan = O.plan_from_patterns(O.PAT_COL, O.PAT_NONE, O.PAT_ROW, 64)
    ref = bench.run_config(bench.oracle_strategies(plan), plan["oe_rank"])
    # what the GPU arm reports for the calibrated Llama3.1-8B block (binding names)
    gpu = bench.run_config({"patterns": {"X": "Column-wise", "W": "None", "G_Y": "Row-wise"},
                            "fwd": "IHT", "dgrad": "OE-Left", "wgrad": "OE-Left",
                            "uniform_over_linears": True}, 64)
    assert ref == gpu
    assert gpu["flops_per_step"] == 42880953483264            # 6 M N K over the seven linears


def test_reference_arm_line_carries_the_contract_keys(capsys):
    """One oracle step of the reference arm on rank 0: the line has every key the driver reads,
    the GPU arm's metric, unit and config, and a zero-copy e2e of its own value."""
    import json
    import types
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=1)
    bench.run_reference(args, 1, 0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"].startswith("llama3.1-8b linear block")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_roofline_peak_is_the_burst_bf16_figure_times_the_nominal_ratio():
    """The fused GEMM is timed alone, so its peak is MEASURED_PEAKS' burst BF16 figure x 6 (not the
    sustained one), and every fraction recomputes from the line's own fields."""
    peaks = {"bf16_tflops": 1920.8, "bf16_tflops_sustained": 1730.4, "hbm_gbs": 6793.1}
    pipe = {"flop_per_clk_per_sm": 32768.0, "sms": 152, "sm_mhz": 1957.0, "tflops": 9746.0}
    r = bench.roofline_fields(7265.0, peaks, "measured", pipe, 1850.0)
    assert r["peak"] == 1920.8 * 6
    assert abs(r["frac"] - 7265.0 / (1920.8 * 6)) < 1e-12
    assert abs(r["pipe_probe"]["frac"] - round(7265.0 / 9746.0, 4)) < 1e-12
    assert abs(r["clock_normalised"]["frac"] - round(7265e12 / 1850e6 / (32768 * 152), 4)) < 1e-12
    assert r["nominal"]["peak"] == 13500.0
    assert bench.roofline_fields(7265.0, peaks, "measured", pipe, None)["clock_normalised"]["frac"] is None


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
