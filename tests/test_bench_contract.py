"""The bench's JSON contract on the host: the reference arm (the CPU oracle) prints one
line with the keys a bench line needs, and the GPU arm refuses to report anything
without a GPU (there is no CPU fallback of the library)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT)


def test_reference_arm_line():
    res = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.5")
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, "exactly one JSON line on stdout"
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "batched_decode_64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_speculative_verify():
    """The speculative-verification workload's reference arm: the oracle's scan over the
    same 4 tokens, scaled to a token's v-heads."""
    res = run_bench("--impl", "reference", "--workload", "spec_verify_64x4", "--steps", "1",
                    "--warmup", "3")
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["config"]["workload"] == "spec_verify_64x4"
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]


def test_gpu_arm_fails_loudly_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    res = run_bench("--steps", "1", "--warmup", "3", timeout=300)
    assert res.returncode != 0
    assert not any(ln.lstrip().startswith("{") for ln in res.stdout.splitlines())


def test_gpus_flag_without_a_launcher_fails_loudly():
    """--gpus 2 in a single process (no torchrun, WORLD_SIZE unset) must not run as one
    rank and report n_gpus 1."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT, env=env)
    assert res.returncode != 0
    assert "WORLD_SIZE" in res.stderr
    assert not any(ln.lstrip().startswith("{") for ln in res.stdout.splitlines())


def test_cpu_baseline_names_the_host_and_the_oracle_build():
    res = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert res.returncode == 0, res.stderr[-2000:]
    cb = json.loads(res.stdout.strip().splitlines()[-1])["cpu_baseline"]
    assert cb["nproc"] == os.cpu_count() and cb["cores"] == 1
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    assert "-ffp-contract=off" in cb["oracle_build"]


def test_ncu_traffic_comes_from_the_json_record(monkeypatch):
    """roofline.traffic is read from profiles/ncu_traffic.json, and only while the
    kernel's source hash is the one recorded beside the counters."""
    sys.path.insert(0, ROOT)
    import bench
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)
    assert rec
    for key, entry in rec.items():
        assert os.path.exists(os.path.join(ROOT, "profiles", entry["summary"])), key
        kernel = next(k for k in bench.KERNEL_SOURCES if key.startswith(k + "_"))
        workload = key[len(kernel) + 1:]
        monkeypatch.setattr(bench, "source_sha", lambda files, h=entry["source_sha256_16"]: h)
        assert bench.ncu_traffic(kernel, workload) == float(entry["dram_bytes_per_launch"])
        monkeypatch.setattr(bench, "source_sha", lambda files: "0" * 16)
        assert bench.ncu_traffic(kernel, workload) is None


def test_reference_arm_under_a_launcher_prints_one_line():
    """Launched as two ranks (torchrun, as for N > 1), rank 0 alone runs the oracle and
    prints the line; the other rank exits 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    res = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                          "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                          "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
                          "--cpu-budget", "0.5"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.lstrip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
