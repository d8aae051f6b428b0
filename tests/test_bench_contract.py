"""The bench's host-side contract, on CPU (no GPU).

`bench.py --impl reference` times the fp64 oracle's cached decode step on the host cores:
it needs no device, so its JSON line is checked here end to end (a short run). Also
checked: the warm-up floor, the attention kernel's source key and the committed DRAM-traffic
records that the roofline's `traffic` is looked up in.
"""
import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run(args, timeout=600):
    env = dict(os.environ, OMP_NUM_THREADS="4", CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["name"] == bench.DEFAULT_CONFIG and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] == 4 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_refused():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "2"], timeout=120)
    assert r.returncode == 2 and "warmup" in r.stderr
    assert not r.stdout.strip()


def test_build_key_is_printed_and_matches_the_sources():
    r = _run(["--build-key"], timeout=120)
    assert r.returncode == 0
    key = r.stdout.strip()
    assert re.fullmatch(r"[0-9a-f]{16}", key)
    assert key == bench.kernel_build_key("attn_tc5")


def test_traffic_records_parse_and_are_keyed(tmp_path, monkeypatch):
    recs = []
    for line in open(bench.TRAFFIC_FILE):
        if line.startswith("#") or not line.strip():
            continue
        kernel, key, workload, nbytes = line.split()[:4]
        assert kernel in bench.KERNEL_SOURCES and re.fullmatch(r"[0-9a-f]{16}", key) and workload
        assert float(nbytes) > 0
        recs.append((kernel, key, workload, float(nbytes)))
    assert recs
    # a record is used only while the kernel's sources still have its key
    kernel, key, workload, nbytes = recs[0]
    want = nbytes if key == bench.kernel_build_key(kernel) else None
    assert bench.dram_traffic(kernel, workload) == want
    stale = tmp_path / "traffic.txt"
    stale.write_text(f"{kernel} {'0' * 16} {workload} {int(nbytes)} a capture of other sources\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(stale))
    assert bench.dram_traffic(kernel, workload) is None
