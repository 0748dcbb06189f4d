"""The benchmark's output contract and the absence of a CPU fallback, on CPU.

bench.py --impl reference times the CPU oracle and must print one JSON line
with the fields the measurement contract fixes.  Without a GPU the product
path must fail loudly: the library refuses to create a context, and the
benchmark's own arm exits non-zero instead of measuring anything else.
"""
import json
import os
import subprocess
import sys

import pytest

from text_embedding_encoder_gb300 import binding, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def _run_bench(*args, timeout=600):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="2", OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_the_contract_line():
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_reference_arm_under_torchrun_prints_once():
    # two ranks: rank 0 alone runs the oracle and prints; the other exits 0 without work
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["impl"] == "reference"


@pytest.mark.skipif(_cuda_available(), reason="checks the behaviour without a GPU")
def test_library_refuses_to_run_without_a_gpu():
    try:
        lib = binding.load()
    except RuntimeError:
        pytest.skip("library not built")
    assert lib is not None
    with pytest.raises(binding.TeeError) as e:
        binding.Encoder(synth.TINY, "fp32", max_tokens=64, max_texts=4)
    assert e.value.code in (binding.TEE_ECUDA, binding.TEE_ENOMEM, binding.TEE_EINVAL)


@pytest.mark.skipif(_cuda_available(), reason="checks the behaviour without a GPU")
def test_bench_gpu_arm_fails_without_a_gpu():
    r = _run_bench("--steps", "1", "--warmup", "3", "--no-cpu-baseline", timeout=300)
    assert r.returncode != 0
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{") and '"value"' in ln]
