"""bench.py's output contract and its refusal to run the product path without a GPU (CPU only)."""
import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def run_bench(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    """The reference arm (the fp64 CPU oracle on a bounded sample per step) runs without a GPU and
    prints the same keys as the product arm, with its own cpu_baseline and a zero-copy e2e."""
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["dtype"] == "f64"
    assert d["config"] == bench.workload_config(bench.WORKLOADS[bench.DEFAULT_WORKLOAD], 1)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_product_arm_refuses_to_run_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = run_bench("--steps", "3", "--warmup", "3", "--no-cpu-baseline", timeout=300)
    assert r.returncode != 0
    assert "needs a CUDA device" in (r.stdout + r.stderr)
    assert not any(ln.startswith("{") for ln in r.stdout.splitlines())


def test_warmup_below_three_is_rejected():
    r = run_bench("--warmup", "2", timeout=120)
    assert r.returncode != 0 and "--warmup must be at least 3" in r.stderr


def test_committed_profiles_carry_traffic_for_the_current_sources():
    """Every bench workload's ncu summary was taken on the kernel sources as they are (the
    line's roofline.traffic is null otherwise)."""
    for workload, kernel, family in (("b4h16n4096d128", "attn_fwd_sm103", "fwd"),
                                     ("b1h16n16384d128_causal_q4", "attn_fwd_sm103", "fwd"),
                                     ("b16h32n512d64_causal", "attn_fwd_short_sm103", "fwd"),
                                     ("b2h8n1024d64", "attn_fwd_sm103", "fwd"),
                                     ("b8h16nq512nk8192d128_causal", "attn_fwd_sm103", "fwd"),
                                     ("based_b16h16n4096f16d64", "based_fwd_sm103", "based"),
                                     ("b4h16n4096d128", "attn_bwd", "bwd")):
        traffic = bench.ncu_traffic(workload, kernel, family)
        assert traffic is not None and traffic > 0, (workload, kernel)


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    src = tmp_path / "k.cuh"
    src.write_text("int a = 1;  // one\n/* block */\nint b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "t", ["k.cuh"])
    h1 = bench.kernel_source_hash("t")
    src.write_text("int a = 1;  // changed comment\n\nint b = 2;\n")
    assert bench.kernel_source_hash("t") == h1
    src.write_text("int a = 3;\nint b = 2;\n")
    assert bench.kernel_source_hash("t") != h1
