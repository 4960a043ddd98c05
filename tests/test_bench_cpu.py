"""The reference arm of bench.py (the CPU oracle) on the smallest workload:
one JSON line with the keys a benchmark consumer reads, the oracle's own
arithmetic type, no host/device copies, and a positive throughput.  No GPU
is touched."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "c1", "--steps", "2",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["warmup"] == 3
    assert abs(d["ms_per_step"] - 16.0 / d["value"] * 1e3) < 1e-6 * d["ms_per_step"]   # batch 1 x K = 16
    assert d["config"]["workload"] == "c1_tiny_f32" and d["config"]["weights"] == "f32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_roofline_traffic_only_with_a_matching_capture(tmp_path, monkeypatch):
    """The bench reports a kernel class's measured DRAM traffic only from a
    capture taken on the current GEMM sources: a record whose fingerprint
    no longer matches (the kernel changed since) gives null, and so does a
    workload without a record."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    cfg = synth.get_config("c5")
    fname, sources = bench.TRAFFIC_PROFILES[cfg.name]
    text = open(os.path.join(ROOT, "profiles", fname)).read()
    fields = dict(l.split(":", 1) for l in text.splitlines()
                  if l.split(":")[0] in ("traffic_per_launch_bytes", "source_fingerprint"))
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the same sources under the temporary root
    csrc = tmp_path / "block_diffusion_speculative_hidden_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in sources:
        src = open(os.path.join(ROOT, "block_diffusion_speculative_hidden_gb300", "csrc", f)).read()
        (csrc / f).write_text(src)
    (tmp_path / "profiles" / fname).write_text(text)
    got = bench.gemm_traffic(cfg)
    # a record matching the sources is read back as recorded; one that does not gives null
    if got is not None:
        assert got == float(fields["traffic_per_launch_bytes"].strip())
    first = open(os.path.join(ROOT, "block_diffusion_speculative_hidden_gb300", "csrc", sources[0])).read()
    (csrc / sources[0]).write_text(first + "\nint an_edit_of_the_kernel;\n")
    assert bench.gemm_traffic(cfg) is None
    # a comment-only edit keeps the record valid
    (csrc / sources[0]).write_text(first + "\n// a note\n")
    assert bench.gemm_traffic(cfg) == got
    assert bench.gemm_traffic(synth.get_config("c1")) is None
