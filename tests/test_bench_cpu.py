"""bench.py's host logic on the CPU: the algorithmic FLOP counts behind the
roofline, the lookup of committed ncu traffic by kernel, workload, mode and
source digest, the bounded oracle baseline, and the reference arm's JSON
line (the oracle timed on the host: no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from onnx_recurrent_gb300.synth import workload  # noqa: E402


def test_algorithmic_flops_of_the_lstm_workload():
    c = workload("lstm_fwd_s64_b32_i256_h512")
    rec, proj, proj_bytes = bench.algorithmic(c)
    assert rec == 2.0 * 64 * 32 * 4 * 512 * 512           # 2 S N G H^2: every row runs every step
    assert proj == 2.0 * 64 * 32 * 4 * 512 * 256          # 2 S N G H I
    assert proj_bytes == 4.0 * (64 * 32 * 256 + 4 * 512 * 256 + 64 * 32 * 4 * 512)


def test_algorithmic_flops_count_valid_steps_only():
    c = workload("gru_bidi_s128_b64_i512_h1024")
    rec, _, _ = bench.algorithmic(c)
    valid = int(c.sequence_lens.sum()) * 2
    assert rec == 2.0 * valid * 3 * 1024 * 1024
    assert valid < c.cell_steps()


def test_traffic_lookup_follows_the_source_digest(tmp_path, monkeypatch):
    d = bench.source_digest("recurrence")
    assert len(d) == 16 and d != bench.source_digest("cell")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "x.md").write_text(f"summary\n\ntraffic_key: recurrence wl exact {d} 1234\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("recurrence", "wl", "exact", d) == 1234
    assert bench.profiled_traffic("recurrence", "wl", "fast", d) is None       # another mode
    assert bench.profiled_traffic("recurrence", "wl", "exact", "0" * 16) is None  # sources changed


def test_committed_profiles_parse():
    keys = []
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        with open(os.path.join(ROOT, "profiles", name)) as f:
            for line in f:
                if line.startswith("traffic_key:"):
                    kernel, wl, mode, digest, nbytes = line.split()[1:]
                    assert kernel in bench.KERNEL_SOURCES and int(nbytes) > 0 and len(digest) == 16
                    keys.append((kernel, wl, mode))
    assert ("recurrence", "lstm_fwd_s64_b32_i256_h512", "exact") in keys


def test_cpu_baseline_is_bounded():
    out = bench.cpu_baseline(workload("rnn_fwd_s8_b1_i16_h128"), budget_s=0.3)
    assert out["kind"] == "oracle" and out["cores"] == 1 and out["value"] > 0
    assert "cell-steps" in out["sample"]


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "rnn_fwd_s8_b1_i16_h128", "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == bench.UNIT and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["value"] == pytest.approx(d["e2e"]["value"])
