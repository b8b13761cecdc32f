"""bench.py's command-line contract on the CPU: the reference arm (the oracle
timed on the host cores) prints one JSON line with the contract's keys, and
the library arm refuses to run without a GPU instead of falling back to the
CPU.  No GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                          capture_output=True, text=True, timeout=600, env=env)


def test_reference_arm_prints_one_contract_line():
    r = _run(["--impl", "reference", "--config", "0", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] >= 3
    assert d["vs_baseline"] is None
    assert d["config"]["workload"] == "swiglu_f32_L512_d64_h128_E8_K2"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_library_arm_needs_a_gpu():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = _run(["--config", "0", "--steps", "1"], env=env)
    assert r.returncode != 0
    assert not any(ln.startswith("{") for ln in r.stdout.splitlines())


def _tree(tmp_path, source, profile):
    (tmp_path / "profiles").mkdir(parents=True)
    (tmp_path / "k.cu").write_text(source)
    (tmp_path / "profiles" / "p.md").write_text(profile)
    return tmp_path


def test_code_hash_ignores_comments_and_whitespace(tmp_path):
    import bench
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text("int f(int x) {  // doubles\n  return 2 * x;\n}\n")
    b.write_text("/* a note */ int f(int x)\n{\n    return 2 * x;   // same code\n}\n")
    assert bench.code_sha256(str(a)) == bench.code_sha256(str(b))
    b.write_text("int f(int x) { return 3 * x; }\n")
    assert bench.code_sha256(str(a)) != bench.code_sha256(str(b))


def test_traffic_lookup_follows_the_code(tmp_path, monkeypatch):
    """The roofline's DRAM traffic comes from a committed ncu summary only
    while the kernel source still hashes to the value recorded with it."""
    import bench
    src = "__global__ void k() {}\n"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text(src)
    sha = bench.code_sha256(str(tmp_path / "k.cu"))
    _tree(tmp_path / "t", src, f"notes\n\ntraffic-per-launch workload=w file=k.cu code-sha256={sha}\nup 123\ndown 456\n\nmore\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "t"))
    assert bench.traffic_per_launch("w", "up", "k.cu") == 123
    assert bench.traffic_per_launch("w", "down", "k.cu") == 456
    assert bench.traffic_per_launch("w", "dx", "k.cu") is None
    assert bench.traffic_per_launch("other", "up", "k.cu") is None
    # a change of comments keeps the figures, a change of code drops them
    (tmp_path / "t" / "k.cu").write_text("// the kernel\n" + src)
    assert bench.traffic_per_launch("w", "up", "k.cu") == 123
    (tmp_path / "t" / "k.cu").write_text("__global__ void k() { return; }\n")
    assert bench.traffic_per_launch("w", "up", "k.cu") is None


def test_committed_traffic_figures_match_the_sources():
    """Each committed traffic block names a source whose current code hash it
    was captured on (a stale block would silently give null traffic)."""
    import bench
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        for ln in open(os.path.join(ROOT, "profiles", name)).read().splitlines():
            g = ln.split()
            if g and g[0] == "traffic-per-launch":
                fields = dict(x.split("=", 1) for x in g[1:])
                assert bench.code_sha256(os.path.join(ROOT, fields["file"])) == fields["code-sha256"], \
                    f"{name}: the kernel changed since this capture; recapture it or drop the block ({ln})"
