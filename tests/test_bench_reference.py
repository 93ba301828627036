"""CPU tests of bench.py's oracle legs (the fp64 oracle timed on all host
cores): the split of the sample over the cores, and the reference arm's JSON
line.  No GPU is used."""

import importlib.util
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_balance_gives_every_unit_to_exactly_one_core_and_evens_the_load():
    b = _bench()
    weights = [16384] * 37 + [5, 7000, 1]
    shares = b.balance(weights, 8)
    assert len(shares) == 8
    assert sorted(u for s in shares for u in s) == list(range(len(weights)))
    loads = [sum(weights[u] for u in s) for s in shares]
    # longest-processing-time-first: no core ends more than one unit above another
    assert max(loads) - min(loads) <= max(weights)
    # more cores than units: the extra cores get nothing
    assert [len(s) for s in b.balance([3, 2], 4)] == [1, 1, 0, 0]


def test_reference_line_uses_all_host_cores():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "llama31_8b_rag", "--steps", "3", "--warmup", "3", "--ref-seconds", "12"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == "stitched KV GB/s" and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["steps"] == 3 and line["warmup"] == 3 and line["higher_is_better"] is True
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"]
    # the Llama workload has 32 (request, layer) units: enough for every core here
    assert cpu["cores"] == min(_bench().host_cores(), 32)
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_covers_the_stitch_only():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--mode", "attend",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line
