"""The benchmark's reference arm: the fp64 oracle timed on the host cores.

`bench.py --impl reference` needs no GPU.  Rank 0 prints one JSON line in the
same metric and unit as the kernel arm, with the oracle described as the CPU
baseline and an end-to-end figure that moves no bytes; the other ranks of a
multi-process launch exit without work.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "0",
        "--cpu-seconds", "1", "--workload", "llama7b_s32k"]


def run(env_extra):
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env.update(env_extra)
    return subprocess.run(ARGS, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_line_keeps_the_contract():
    r = run({})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"].startswith("causal attn fwd+bwd TFLOP/s") and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "llama7b_s32k" and d["config"]["S"] == 32768
    # the same config object as the GPU arm prints for this workload, so the two lines compare
    sys.path.insert(0, ROOT)
    import bench
    from long_context_causal_gb300.inputs import WORKLOADS
    assert d["config"] == bench.config_of(WORKLOADS["llama7b_s32k"], "balanced")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
