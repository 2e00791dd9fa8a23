"""bench.py's output contract on CPU: the reference arm (the fp64 oracle timed on the host)
prints exactly one JSON line with the keys the benchmark contract names."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "5", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env=dict(os.environ, WORLD_SIZE="1", RANK="0"))
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 5 and d["warmup"] == 3
    assert d["config"]["calls_per_step"] == 32
    assert d["config"]["workload"] == "decode_distinct"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["value"] > 0 and d["unit"] == "GB/s"


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "5", "--warmup", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode != 0


def test_gpus_flag_relaunches_n_ranks():
    """--gpus 2 without an external launcher runs the script as two local ranks (here the
    reference arm, on CPU): rank 0 alone prints, and the line reports n_gpus = 2."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env={k: v for k, v in os.environ.items()
                              if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    assert json.loads(lines[0])["n_gpus"] == 2


def test_gpus_flag_must_match_world_size():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT,
                         env=dict(os.environ, WORLD_SIZE="1", RANK="0"))
    assert out.returncode != 0 and "disagrees" in out.stderr
