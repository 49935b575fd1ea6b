"""bench.py on the CPU: the reference arm (the oracle, timed on the host)
prints one complete JSON line; the vocabulary cuts of --shards and the
option checks."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                        "--ref-requests", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]


def test_shard_cuts_cover_the_vocabulary_in_8_entry_steps():
    sys.path.insert(0, ROOT)
    import bench

    for V, S in ((128256, 2), (152064, 3), (1000, 3), (41, 2), (129280, 4)):
        cuts = bench.shard_cuts(V, S)
        assert cuts[0] == 0 and cuts[-1] == V and len(cuts) == S + 1
        assert all(a < b for a, b in zip(cuts, cuts[1:]))
        assert all(c % 8 == 0 for c in cuts[1:-1])


def test_shards_option_rejects_other_layouts():
    sys.path.insert(0, ROOT)
    import pytest

    import bench

    for argv in (["--shards", "2", "--packed"], ["--shards", "2", "--early-exit"], ["--shards", "2", "--config", "3"],
                 ["--shards", "0"]):
        with pytest.raises(SystemExit):
            bench.main(argv)
