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
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}, "--steps", "2", "--warmup", "3",
             "--gpus", "2")
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


def test_gpus_n_relaunches_n_ranks():
    """--gpus 2 started without torchrun re-launches itself as two ranks
    (gloo-free here: the reference arm needs no process group); rank 0 prints
    the one JSON line and the other rank exits quietly."""
    r = _run({}, "--steps", "2", "--warmup", "3", "--gpus", "2")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert json.loads(lines[0])["impl"] == "reference"
    assert "launching 2 ranks" in r.stderr


def test_gpus_mismatching_world_size_fails():
    r = _run({"RANK": "0", "LOCAL_RANK": "0", "WORLD_SIZE": "2"}, "--steps", "2", "--warmup", "3",
             "--gpus", "1")
    assert r.returncode != 0
    assert "does not match" in r.stderr


def test_gpu_arm_without_a_gpu_fails_loudly():
    """The measured arm never falls back to the CPU: with no CUDA device it
    exits non-zero, also when asked for two ranks."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for extra in ([], ["--gpus", "2"]):
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "single_128x256x512",
                            "--steps", "2", "--warmup", "3", "--no-clocks", "--no-cpu-baseline", *extra],
                           capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
        assert r.returncode != 0, (extra, r.stdout)
        assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_parity_rows_cover_group_edges():
    """The rows bench.py compares per shape include every group's first and
    last row (contiguous) and every live group's first and last valid row
    (masked)."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    p = wl.make_contiguous([128, 256, 384], 256, 256, seed=1)
    [(g, rows)] = bench.parity_rows(p)
    assert g is None
    for first, last in ((0, 127), (128, 383), (384, 767)):
        assert first in rows and last in rows
    q = wl.make_masked([0, 5, 200, 256], 256, 256, 256, seed=2)
    got = {g: set(r.tolist()) for g, r in bench.parity_rows(q)}
    assert set(got) == {1, 2, 3}
    assert {0, 4} <= got[1] and {0, 127, 128, 199} <= got[2] and {0, 255} <= got[3]
    assert all(max(r) < int(q.masked_m[g]) for g, r in got.items())
