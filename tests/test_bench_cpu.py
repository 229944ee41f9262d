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
    d = bench.source_digest("rnn_recurrent_kernel")
    assert len(d) == 16 and d != bench.source_digest("rnn_cell_kernel")
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
                    kind, wl, mode, digest, nbytes = line.split()[1:]
                    assert kind in ("recurrence", "projection", "cell") and int(nbytes) > 0 and len(digest) == 16
                    # the summary's kernel (its file name) is one the digests know
                    assert any(name.startswith(k + "_") for k in bench.KERNEL_SOURCES)
                    keys.append((kind, wl, mode))
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


def test_live_rows_follow_the_lengths():
    c = workload("lstm_bidi_s512_b128_i1024_h1024")
    live = bench.live_rows_per_step(c)
    assert len(live) == int(c.sequence_lens.max())
    assert live[0] == c.batch and live[-1] >= 1
    assert sum(live) == int(c.sequence_lens.sum())          # sum over steps = sum of lengths
    assert all(a >= b for a, b in zip(live, live[1:]))


def test_step_roofline_terms():
    # LSTM forward, fast mode: 2 * 32 * 4 * 512^2 FLOP per step against
    # 152 SMs x 128 lanes x 2 FLOP x 2070 MHz; R (4 MiB) fits in shared memory
    c = workload("lstm_fwd_s64_b32_i256_h512")
    sr = bench.step_roofline(c, "fast", 1.0, 152, 2070.0, 20000.0, 232448)
    alu_us = 2.0 * 32 * 4 * 512 * 512 / (152 * 128 * 2 * 2070e6) * 1e6
    smem_us = 4.0 * 4 * 512 * 512 / (152 * 128 * 2070e6) * 1e6
    assert sr["terms_us_per_step"]["alu"] == pytest.approx(alu_us, rel=1e-3)
    assert sr["terms_us_per_step"]["smem"] == pytest.approx(smem_us, rel=1e-3)
    assert sr["terms_us_per_step"]["l2"] == 0.0 and sr["r_streamed_bytes_per_step"] == 0.0
    # 512 dependent fused multiply-adds per output and step (0.99 us) bind
    # before the fused ALU peak (0.83 us) in fast mode
    chain_us = 512 * bench.FP32_CHAIN_CYCLES / 2070e6 * 1e6
    assert sr["terms_us_per_step"]["chain"] == pytest.approx(chain_us, rel=1e-3)
    assert sr["binding"] == "chain"
    assert sr["roof_ms"] == pytest.approx(64 * max(alu_us, smem_us, chain_us) / 1e3, rel=1e-3)
    assert sr["frac"] == pytest.approx(sr["roof_ms"] / 1.0, rel=1e-3)
    # exact mode halves the ALU peak (no fused multiply-add): the ALU binds
    ex = bench.step_roofline(c, "exact", 1.0, 152, 2070.0, 20000.0, 232448)
    assert ex["terms_us_per_step"]["alu"] == pytest.approx(2 * alu_us, rel=1e-3)
    assert ex["binding"] == "alu"


def test_step_roofline_streams_what_does_not_fit():
    # GRU reverse, hidden 2048: R is 3 * 2048^2 * 4 bytes = 48 MiB, more than
    # 152 SMs x 227 KiB of shared memory; the rest streams from L2 every step
    c = workload("gru_rev_s4096_b4_i256_h2048")
    sr = bench.step_roofline(c, "fast", 10.0, 152, 2070.0, 10000.0, 232448)
    r = 4.0 * 3 * 2048 * 2048
    assert sr["r_bytes_per_step"] == r
    assert sr["r_streamed_bytes_per_step"] == r - 152 * 232448
    assert sr["terms_us_per_step"]["l2"] == pytest.approx((r - 152 * 232448) / 10000e9 * 1e6, rel=1e-3)
    assert sr["steps"] == 4096
    # every output's 2048 dependent adds a step: 2048 * 4 cycles at 2070 MHz
    chain_us = 2048 * bench.FP32_CHAIN_CYCLES / 2070e6 * 1e6
    assert sr["terms_us_per_step"]["chain"] == pytest.approx(chain_us, rel=1e-3)
    assert sr["binding"] == "chain"
    assert sr["roof_ms"] == pytest.approx(4096 * chain_us / 1e3, rel=1e-3)


def test_step_roofline_chain_doubles_for_two_gru_products():
    from onnx_recurrent_gb300.synth import make_case
    a = make_case("GRU", "forward", 3, 2, 4, 256, linear_before_reset=0)
    b = make_case("GRU", "forward", 3, 2, 4, 256, linear_before_reset=1)
    ca = bench.step_roofline(a, "exact", 1.0, 152, 2070.0, 10000.0, 232448)["terms_us_per_step"]["chain"]
    cb = bench.step_roofline(b, "exact", 1.0, 152, 2070.0, 10000.0, 232448)["terms_us_per_step"]["chain"]
    assert ca == pytest.approx(2 * cb, rel=1e-3)


def test_traffic_lookup_reads_every_key_of_a_summary(tmp_path, monkeypatch):
    # a summary captured on a shorter sequence carries a key for that case
    # and a scaled one for the bench workload
    d = bench.source_digest("rnn_recurrent_kernel")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "x.md").write_text(f"traffic_key: recurrence short fast {d} 10\\n"
                                                f"traffic_key: recurrence long fast {d} 80\\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("recurrence", "short", "fast", d) == 10
    assert bench.profiled_traffic("recurrence", "long", "fast", d) == 80



def test_source_digest_is_per_kernel():
    # a change to one kernel's code leaves the digests of kernels built from
    # other sources (and so their committed traffic figures) as they are
    csrc = os.path.join(ROOT, "onnx_recurrent_gb300", "csrc")

    def read(changed):
        def r(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                t = f.read()
            return t + "\nint changed_here;\n" if name == changed else t
        return r

    for k, srcs in bench.KERNEL_SOURCES.items():
        assert all(os.path.exists(os.path.join(csrc, n)) for n in srcs)
    tc = read("k_recur_tc.cu")
    assert bench.source_digest("rnn_tc_kernel", tc) != bench.source_digest("rnn_tc_kernel")
    for k in ("rnn_recurrent_kernel", "rnn_dataflow_kernel", "rnn_wavefront_kernel", "proj_tc_kernel"):
        assert bench.source_digest(k, tc) == bench.source_digest(k)
    # a header every recurrent kernel is built from changes them all
    shared = read("k_recur.cuh")
    for k in ("rnn_recurrent_kernel", "rnn_dataflow_kernel", "rnn_wavefront_kernel", "rnn_tc_kernel"):
        assert bench.source_digest(k, shared) != bench.source_digest(k)
    # every translation unit of the library is some kernel's source, or host code
    from onnx_recurrent_gb300 import _build
    covered = set().union(*bench.KERNEL_SOURCES.values())
    assert set(_build.SOURCES) - covered == {"rnn_api.cpp", "k_misc.cu", "rnn_static.cu"}


def test_kernel_sources_cover_their_includes():
    # every header a kernel's translation units include (transitively) is in
    # its digest, except the dataflow header in the staged kernel's units
    import re
    csrc = os.path.join(ROOT, "onnx_recurrent_gb300", "csrc")

    def closure(name, seen):
        if name in seen:
            return seen
        seen.add(name)
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            for m in re.finditer(r'#include\s+"([^"]+)"', f.read()):
                if os.path.exists(os.path.join(csrc, m.group(1))):
                    closure(m.group(1), seen)
        return seen

    allowed = {"rnn_recurrent_kernel": {"k_recur2.cuh"}}
    for k, srcs in bench.KERNEL_SOURCES.items():
        inc = set()
        for tu in (s for s in srcs if s.endswith(".cu")):
            inc |= closure(tu, set())
        assert inc - set(srcs) <= allowed.get(k, set()), k


def test_source_digest_ignores_comments_and_blank_space():
    a = 'int f(int x) {  // one\n  return x + 1; /* two */ }\nconst char* s = "a // not a comment";\n'
    b = 'int f(int x) {\n\n    return x + 1;   }\nconst char* s = "a // not a comment";'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "a // not a comment";'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert "not a comment" in bench.code_only(a)


def test_h_bytes_per_step_and_its_term():
    # LSTM bidirectional, batch 128, hidden 1024 on the staged kernel with 74
    # CTAs per direction: every CTA copies all 128 rows of h (fp32) each step
    c = workload("lstm_bidi_s512_b128_i1024_h1024")
    geo = {"kernel": 1, "unit_groups": 74, "row_groups": 1}
    hb = bench.h_bytes_per_step(geo, c)
    assert hb == 2 * 74 * 128 * 1024 * 4
    # the tensor-core kernel copies them in fp16; the in-cluster exchange none
    assert bench.h_bytes_per_step({"kernel": 3, "unit_groups": 74}, c) == hb / 2
    assert bench.h_bytes_per_step({"kernel": 5, "unit_groups": 16}, c) == 0.0
    # dataflow, batch 32 in 4 row groups of 8: each CTA its group's rows
    c2 = workload("lstm_fwd_s64_b32_i256_h512")
    assert bench.h_bytes_per_step({"kernel": 2, "unit_groups": 37, "row_groups": 4}, c2) == 37 * 4 * 8 * 512 * 4
    sr = bench.step_roofline(c, "fast", 10.0, 152, 2070.0, 7000.0, 232448, hb)
    # counted for the live rows only: on average the live fraction of the batch
    live = bench.live_rows_per_step(c)
    mean_live = sum(live) / len(live) / 128
    assert sr["terms_us_per_step"]["h"] == pytest.approx(hb / 7000e9 * 1e6 * mean_live, rel=1e-3)
    assert sr["h_bytes_per_step"] == hb
    # on the tensor cores (the measured bf16 burst) the h term binds
    st = bench.step_roofline(c, "tf32", 10.0, 152, 2070.0, 7000.0, 232448, hb / 2, tensor_tflops=1874.7)
    assert st["binding"] == "h" and st["terms_us_per_step"]["chain"] == 0.0
