"""bench.py's reference arm on the host cores: one JSON line with the keys the
benchmark contract names (the GPU arm's line is checked on the GPU runs)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = dict(os.environ, SSD_BENCH_ORACLE_ROWS="8")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in out, k
    assert out["value"] > 0 and out["unit"] == "tokens/s" and out["steps"] == 1
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["e2e"]["value"] == out["value"]
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["d2h_bytes_per_step"] == 0
    assert out["config"]["seq_len"] == 8


def test_link_bound_of_a_step():
    """The least step time the host link allows: the shorter direction's bytes
    at the both-ways rate, beside as many of the longer one's, then the rest of
    the longer direction alone (hand-computed cases)."""
    sys.path.insert(0, ROOT)
    import bench
    link = {"h2d_gbs": 200.0, "d2h_gbs": 100.0, "both_ways_gbs_per_direction": 50.0}
    # 4 GB in, 1 GB out: 1 GB each way at 50 GB/s (20 ms), then 3 GB in at 200 (15 ms)
    assert abs(bench.link_bound_ms(4_000_000_000, 1_000_000_000, link) - 35.0) < 1e-9
    # 1 GB in, 3 GB out: 1 GB each way (20 ms), then 2 GB out at 100 (20 ms)
    assert abs(bench.link_bound_ms(1_000_000_000, 3_000_000_000, link) - 40.0) < 1e-9
    # one direction only: its own rate
    assert abs(bench.link_bound_ms(2_000_000_000, 0, link) - 10.0) < 1e-9
    assert abs(bench.link_bound_ms(0, 0, link)) < 1e-12
