"""The reference arm of bench.py (the CPU oracle on host cores) keeps the JSON-line
contract: one line with the metric, the per-step timing and a cpu_baseline that
states the sample and the core count. Runs on the CPU with a small budget."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, LQ_REFERENCE_BUDGET_S="2")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "1", "--steps", "2",
                          "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [line for line in out.stdout.splitlines() if line.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    for key in ("metric", "value", "unit", "n_gpus", "ms_per_step", "higher_is_better", "scaling", "dtype", "data",
                "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "gdn-tiny-1x2"


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the driver launches N > 1 (torch.distributed.run, two ranks on
    127.0.0.1): rank 0 alone runs the oracle and prints the line; rank 1 exits 0."""
    env = dict(os.environ, LQ_REFERENCE_BUDGET_S="2")
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", "29517", "bench.py", "--impl", "reference",
                          "--gpus", "2", "--workload", "1", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [line for line in out.stdout.splitlines() if line.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 1 and d["value"] > 0
