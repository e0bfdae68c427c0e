"""bench.py pieces that run on the CPU: the reference arm (the oracle timed
on the host) prints one contract-shaped JSON line, and the parity summary of
the bench line measures what it claims to."""
import json
import os
import subprocess
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["config"]["workload"].startswith("tiny")


def test_parity_summary_measures_the_stated_errors():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((8, 32))
    exact = bench.parity_summary(torch.tensor(ref, dtype=torch.float32), ref)
    assert exact["pass"] and exact["rel_fro"] < 1e-6 and exact["tokens"] == 8
    off = ref.copy()
    off[3, 5] += 0.1 * np.sqrt(np.mean(ref ** 2))          # one element 0.1 RMS off
    s = bench.parity_summary(torch.tensor(off, dtype=torch.float32), ref)
    assert not s["pass"] and abs(s["max_abs_over_rms"] - 0.1) < 1e-3
    nan = bench.parity_summary(torch.full((8, 32), float("nan")), ref)
    assert not nan["pass"]


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    """The key of the committed ncu traffic figures changes with the code,
    not with its comments."""
    d = tmp_path / "lora_mixture_experts_gb300" / "csrc"
    d.mkdir(parents=True)
    for n in ("gemm_tc.cu", "gemm_tc.cuh", "common.cuh", "merge.cu", "merge.cuh"):
        (d / n).write_text("int f() { return 1; }  // one\n/* two */\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash()
    (d / "gemm_tc.cu").write_text("// a new comment\nint f() {   return 1; }\n")
    assert bench.source_hash() == h0
    (d / "gemm_tc.cu").write_text("int f() { return 2; }\n")
    assert bench.source_hash() != h0
