"""The bench's JSON contract, checked on the CPU through its reference arm (the fp64
oracle timed on host cores): one line with the keys the driver reads, rank 0 alone
printing under a two-rank torchrun (gloo)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(cmd, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.update(env_extra or {})
    env.setdefault("OMP_NUM_THREADS", "1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def _check(line, gpus, steps, warmup):
    d = json.loads(line)
    assert KEYS <= set(d)
    assert d["impl"] == "reference"
    assert d["metric"] == "kda_prefill_tokens_per_s" and d["unit"] == "tokens/s"
    assert d["n_gpus"] == gpus and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert "workload" in d["config"] and d["config"]["seq_len"] == 8192
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_contract_line():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert len(lines) == 1
    _check(lines[0], 1, 1, 0)


def test_reference_arm_under_two_gloo_ranks_prints_once():
    pytest.importorskip("torch.distributed.run")
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                  "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
                  "--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert len(lines) == 1
    _check(lines[0], 2, 1, 0)
