"""bench.py's reference arm on the CPU: the CPU oracle timed on a bounded
sample of the dense sweep workload, printed as one JSON line with the same
metric, unit and direction as the GPU arm.  Under torchrun only rank 0 runs
it; the other ranks exit 0 without work or output."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *args):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1"}, "--impl", "reference", "--steps", "1",
             "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["unit"] == "TFLOP/s" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "sample" in cb
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["gpu_launches"] == 0


def test_reference_arm_other_ranks_do_nothing():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"}, "--impl", "reference", "--steps", "1",
             "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    """The committed DRAM-traffic profile is tied to the kernels' code: a
    comment edit keeps its hash, a code edit changes it."""
    import shutil

    sys.path.insert(0, ROOT)
    import bench

    csrc = tmp_path / "block_scaled_fp8_quant_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for rel in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(ROOT, rel), tmp_path / rel)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    g = csrc / "gemm_kernels.cu"
    g.write_text(g.read_text() + "\n// a comment\n/* another\n   comment */\n\n")
    assert bench.kernel_source_hash() == h0
    g.write_text(g.read_text() + "static const int kUnusedForTheTest = 1;\n")
    assert bench.kernel_source_hash() != h0
