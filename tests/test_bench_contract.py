"""bench.py's output contract, checked on the CPU through its reference arm
(the oracle timed on a bounded sample; no GPU needed): one JSON line with
the keys the benchmark contract requires, and the rank handling under a
two-rank launch (rank 0 prints, the other exits without work)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "3",
       "--ref-feats", "128", "--ref-rows", "4"]


def run(env_extra=None, extra_args=()):
    env = dict(os.environ)
    env.update(env_extra or {})
    out = subprocess.run(CMD + list(extra_args), capture_output=True, text=True, timeout=240, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    return [line for line in out.stdout.splitlines() if line.strip()]


def test_reference_arm_prints_one_contract_line():
    lines = run()
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "decoder_layer_32768"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_non_zero_rank_exits_without_output():
    assert run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, ["--gpus", "2"]) == []


def test_gpus_flag_launches_the_ranks_itself():
    """`--gpus 2` without torchrun's environment starts two ranks of the same
    command; rank 0 alone prints, with n_gpus = 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "LOCAL_WORLD_SIZE")}
    out = subprocess.run(CMD + ["--gpus", "2"], capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    assert "[bench] rank 0/2 (reference arm)" in out.stderr and "[bench] rank 1/2 (reference arm)" in out.stderr
    lines = [line for line in out.stdout.splitlines() if line.strip().startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["n_gpus"] == 2


def test_gpus_flag_must_match_the_rank_environment():
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    out = subprocess.run(CMD + ["--gpus", "4"], capture_output=True, text=True, timeout=240, env=env, cwd=ROOT)
    assert out.returncode != 0 and "does not match WORLD_SIZE" in out.stderr


def test_gpu_arm_refuses_more_gpus_than_visible():
    """The GPU arm fails loudly instead of timing fewer GPUs than asked."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"], capture_output=True,
                         text=True, timeout=240, env=env, cwd=ROOT)
    assert out.returncode != 0 and "needs 2 visible CUDA devices" in out.stderr
