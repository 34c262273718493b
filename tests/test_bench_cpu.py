"""The benchmark's CPU legs without a GPU: the reference arm (the fp64 oracle
timed on the host cores) prints the contract's JSON line for the attention,
decode and FFN workloads, and the argument checks hold."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(*args, timeout=240):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=timeout, cwd=ROOT)
    return out


@pytest.mark.parametrize("extra,unit", [
    (["--config", "tiny"], "TFLOP/s"),
    (["--config", "gqa_decode", "--n", "4096"], "GB/s"),
    (["--config", "ffn"], "TFLOP/s"),
])
def test_reference_arm_prints_one_contract_line(extra, unit):
    out = run("--impl", "reference", "--steps", "3", "--warmup", "3", "--ref-seconds", "3", *extra)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == unit and d["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config"):
        assert key in d, key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_refused():
    out = run("--impl", "reference", "--warmup", "2")
    assert out.returncode != 0 and "warmup" in (out.stderr + out.stdout)


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the multi-GPU bench is (one process per rank), only rank 0
    runs the reference arm and prints; the other rank exits 0 without work."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--config",
           "tiny", "--steps", "3", "--warmup", "3", "--ref-seconds", "2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=240, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
