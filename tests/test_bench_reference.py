"""CPU tests of bench.py's reference arm (the fp64 oracle timed on the host):
its bounded sample and the JSON line it prints.  No GPU is used."""

import importlib.util
import json
import os
import subprocess
import sys

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_prefix_sample_cuts_every_request_to_the_same_fraction():
    b = _bench()
    for name in ("llama31_8b_rag", "deepseek_v3_mla", "qwen3_8b_batch"):
        wl = W.WORKLOADS[name]()
        sub = b.prefix_sample(wl, 0.25)
        assert len(sub.requests) == len(wl.requests)
        for full, cut in zip(wl.requests, sub.requests):
            n_full, n_cut = sum(t for _, t in full), sum(t for _, t in cut)
            assert n_cut == max(1, round(0.25 * n_full))
            # a prefix: the same chunks in the same order, whole but for the last
            assert [c for c, _ in cut] == [c for c, _ in full[:len(cut)]]
            assert all(t == tf for (_, t), (_, tf) in zip(cut[:-1], full))
            assert 0 < cut[-1][1] <= full[len(cut) - 1][1]
        assert sub.chunk_lens == wl.chunk_lens and sub.model == wl.model


def test_reference_line_on_the_default_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == "stitched KV GB/s" and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["steps"] == 3 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_covers_the_stitch_only():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--mode", "attend",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "unavailable" in line
