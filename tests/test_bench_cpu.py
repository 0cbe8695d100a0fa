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
