"""The bench's JSON contract for the reference arm, which runs on the host
(the fp64 oracle): one line, the same metric and config as the GPU arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "1", "--workload", "ring2-s4k-h4-d64-bf16"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    import bench
    assert d["metric"] == bench.METRIC
    assert d["config"]["workload"] == "ring2-s4k-h4-d64-bf16" and d["config"]["seq_len"] == 4096
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["value"] > 0


@pytest.mark.gpu
def test_gpu_arm_prints_one_contract_line():
    """The GPU arm on the 32K workload: one line with the contract's keys, the
    roofline and end-to-end objects, and an end-to-end figure that moves the
    step's inputs and outputs through host memory."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "2", "--warmup", "3",
                          "--workload", "ring4-s32k-h32kv8-d128-causal-contiguous", "--no-cpu-baseline",
                          "--no-backward", "--no-extra"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and 0 < r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    e = d["e2e"]
    # q, k, v in (bf16) and out (bf16) + lse (fp32) back, every step
    S, H, Hkv, dh = 32768, 32, 8, 128
    assert e["h2d_bytes_per_step"] == 2 * S * dh * (H + 2 * Hkv)
    assert e["d2h_bytes_per_step"] == 2 * S * dh * H + 4 * S * H
    assert 0 < e["value"] and e["ms_per_step"] > 0 and e["serial_ms_per_step"] > 0
    # the copies are inside the timed region: the end-to-end step cannot beat the device-resident one
    assert e["ms_per_step"] >= 0.98 * d["ms_per_step"]
    assert d["gpu_launches"] >= d["steps"]


def test_gpus_other_than_one_are_refused():
    """The bench measures on one GPU; a multi-GPU request is refused before
    any work, with a message and exit status 2."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 2
    assert out.stdout.strip() == ""
    assert "one GPU" in out.stderr
