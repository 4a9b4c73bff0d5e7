"""bench.py's reference arm (the CPU oracle on the host cores) keeps the JSON
contract, on the small workload so that it runs in a second or two; under a
multi-rank launch only rank 0 works and prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env, *args):
    env = dict(os.environ, **extra_env)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "single_128x256x512", *args],
                          capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)


def test_reference_line_keys():
    r = _run({}, "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "single_128x256x512"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}, "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_warmup_below_three_is_refused():
    r = _run({}, "--steps", "2", "--warmup", "2")
    assert r.returncode != 0


def test_traffic_lookup(tmp_path, monkeypatch):
    """roofline.traffic comes from profiles/traffic.txt: bytes for a listed
    workload, None for one that is not listed or marked none."""
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# comment line\nworkload_a 12345\nworkload_b none\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("workload_a") == 12345
    assert bench.load_traffic("workload_b") is None
    assert bench.load_traffic("workload_c") is None
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "missing"))
    assert bench.load_traffic("workload_a") is None
