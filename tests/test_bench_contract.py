"""bench.py's output contract on CPU: the reference arm (the oracle on the
host cores, no GPU) prints one JSON line with the contract's keys, and the
DRAM traffic it reports for a kernel is the committed figure only while the
kernel's sources are the ones the figure was measured on."""
import importlib.util
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def test_reference_arm_prints_the_contract_line():
    # the small fp32 workload: the same line as the headline's, in seconds
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_fp32", "--steps", "1", "--warmup", "0",
                          "--ref-rows", "4"],
                         cwd=ROOT, check=True, capture_output=True, text=True, timeout=600).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["data"] == "synthetic"
    assert d["config"]["workload"].startswith("tiny_fp32")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_profiled_traffic_is_keyed_to_the_kernel_sources():
    bench = _bench()
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        data = json.load(f)
    for kernel, sources in (("k_gemm_tc", bench.GEMM_SOURCES), ("k_jsd_rows", bench.ROWS_SOURCES)):
        entry = data[kernel]["headline"]
        got = bench._profiled_traffic(kernel, sources, "headline")
        if entry["source_sha256_16"] == bench.sources_hash(sources):
            assert got == entry["traffic_bytes_per_launch"] and got > 0
        else:
            assert got is None
        assert bench._profiled_traffic(kernel, sources, "no_such_workload") is None
    # the figure of one kernel is never reported for another kernel's sources
    assert bench._profiled_traffic("k_gemm_tc", bench.ROWS_SOURCES, "headline") is None
