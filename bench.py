#!/usr/bin/env python
"""Benchmark of position-independent KV stitching on GB300.

One step = one pass of the whole path over one batch: compose the request(s)
and build the block table (host, C ABI), upload the table, and one pic_stitch
launch (gather + delta-RoPE + paged scatter + recompute list).  Inputs are
resident in HBM when the timed region starts; the pool and the cache are
both larger than L2 (no flush needed).  Prints ONE JSON line on rank 0.

--impl reference times the fp64 CPU oracle (the reference arm of this
build) on the same workload, on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

WORKLOAD_TEXT = {
    "llama31_8b_rag": "Llama-3.1-8B shapes: 32 layers, 8 KV heads x 128, bf16, RoPE theta 5e5 + llama3 "
                      "scaling (neox); 128-token system prompt + 10 x 1024-token chunks in seeded "
                      "permutation; paged block 16; batch 1; recompute first 4 tokens of non-leading chunks",
    "tiny_gqa": "1 layer, 8 KV heads x 128, theta 1e4 neox, 32-token prefix + 4 x 256 chunks, block 16",
    "qwen3_8b_batch": "Qwen3-8B shapes: 36 layers, 8 KV heads x 128, theta 1e6; 8 requests x 32,768 tokens "
                      "from a 64-chunk pool (lengths U[128,4096]), per-request random order; block 16",
    "deepseek_v3_mla": "DeepSeek-V3 MLA shapes: 61 layers, 512 latent + 64 rope (interleaved), theta 1e4; "
                       "65,536 tokens of 16-128-token chunks behind a 32-token leading chunk; block 16",
    "serving_stress": "Llama-3.1-8B shapes; 64 requests x 16,384 tokens, Zipf(1.1) reuse of a 256-chunk "
                      "pool with log-uniform lengths 64-8192; block 16",
}
FALLBACK_HBM_GBS = 6800.0


def bytes_per_token_layer(model, mode):
    row = model.num_kv_heads * model.head_dim * 2
    if mode == "inplace":
        return 2 * row                       # K read + K write
    return 4 * row if model.kind == "gqa" else 2 * row   # pool read + cache write (K and V)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ("pic_kernels.cu", "pic_kernels_tma.cu", "pic_device.cuh", "pic_host.cpp#stitch-schedule",
                  "pic_internal.h#stitch-schedule")


def source_text(name):
    """A source file's bytes, or with "file#region" only the lines between
    its "region <name>" and "end region <name>" comments."""
    fname, _, region = name.partition("#")
    with open(os.path.join(ROOT, "position_independent_kv_stitch_gb300", "csrc", fname), "rb") as f:
        data = f.read()
    if not region:
        return data
    begin = data.index(f"// region {region}:".encode())
    end = data.index(f"// end region {region}".encode(), begin)
    return data[begin:end]


def kernel_source_hash(names=KERNEL_SOURCES):
    """Hash of the kernel and launch-schedule sources a traffic record was taken on."""
    h = hashlib.sha256()
    for name in names:
        h.update(source_text(name))
    return h.hexdigest()[:16]


def recorded_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the sources (the record's own list) as they are now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(key)
        if e and e.get("kernel_source_sha256_16") == kernel_source_hash(tuple(e.get("sources", KERNEL_SOURCES))):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons; only samples whose timestamps
    fall inside the timed region are kept."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index, period_ms=20):
        self.index, self.period_ms = index, period_ms
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader",
                 "-lms", str(self.period_ms)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            deadline = time.time() + 5.0
            while time.time() < deadline and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(2 * self.period_ms / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        import datetime
        inside, all_rows = [], []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    row = (ts, float(parts[2].split()[0]), float(parts[3].split()[0]), parts[6:10])
                except ValueError:
                    continue
                all_rows.append(row)
                if self.t0 is not None and self.t0 <= ts <= self.t1 + self.period_ms / 1000.0:
                    inside.append(row)
        os.unlink(self.path)
        rows = inside
        note = None
        if not rows and all_rows and self.t0 is not None:
            rows = [min(all_rows, key=lambda r: abs(r[0] - self.t0))]
            note = "timed region shorter than the sampling period: nearest sample reported"
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for n, v in zip(self.REASONS, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
               "reasons": sorted(reasons), "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ------------------------------------------------------------------ oracle
#
# The oracle runs as it stands, on every host core: one spawned process per
# core (spawned, not forked: a child forked after the first CUDA call can
# hang), each running whole units of the sample it is handed.  A unit is one
# request x one layer (stitch, attention) or one document (chunking).  The
# pool layer the units read is drawn once and shared through a file every
# process maps read-only.  Time is the wall clock from handing out a sample
# until the last core has finished its share.

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_oracle_sample(wl, pool_k_bits, pool_v_bits, layers):
    """The oracle as it stands, on the given pool layers of every request."""
    import oracle
    m = wl.model
    theta = oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)
    pairing = oracle.NEOX_HALF if m.pairing == "neox" else oracle.INTERLEAVED
    chunks = [oracle.Chunk(off, n, 0) for off, n in zip(wl.pool_offsets, wl.chunk_lens)]
    nb = sum(-(-t // m.block_size) for t in wl.request_tokens)
    pool = oracle.BlockPool(nb)
    plans, tables = [], []
    for req in wl.requests:
        segs = oracle.compose(chunks, [c for c, _ in req], take=[t for _, t in req])
        total = segs[-1].dst_pos + segs[-1].length
        tables.append(pool.allocate(oracle.blocks_needed(total, m.block_size)))
        plans.append(segs)
        oracle.recompute_positions(segs, wl.k_nonleading, wl.k_leading)
    oracle.stitch_paged(pool_k_bits, pool_v_bits, plans, tables, nb, m.block_size, theta, pairing,
                        m.rope_offset, m.rope_dim, layers=layers)


def run_oracle_attend(wl, r, kb, vb, hq, rng):
    """The oracle's decode attention for request r over one layer: chunk keys
    rotated in fp64 from the pool (the fused path's definition), the sink
    bias on the recompute positions, then attention_decode."""
    import oracle
    m = wl.model
    theta = oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)
    pairing = oracle.NEOX_HALF if m.pairing == "neox" else oracle.INTERLEAVED
    chunks = [oracle.Chunk(off, n, 0) for off, n in zip(wl.pool_offsets, wl.chunk_lens)]
    mla = m.kind == "mla"
    vdim = m.head_dim - m.rope_dim if mla else m.head_dim
    scale = 1.0 / (192 ** 0.5) if mla else 1.0 / (m.head_dim ** 0.5)
    req = wl.requests[r]
    segs = oracle.compose(chunks, [c for c, _ in req], take=[t for _, t in req])
    T = segs[-1].dst_pos + segs[-1].length
    keys = np.empty((T, m.num_kv_heads, m.head_dim))
    vals = np.empty((T, m.num_kv_heads, vdim))
    for sg in segs:
        src = oracle.bf16_bits_to_f64(kb[sg.src_tok:sg.src_tok + sg.length]).reshape(sg.length, -1, m.head_dim)
        keys[sg.dst_pos:sg.dst_pos + sg.length] = oracle.rotate_rows(src, sg.delta, theta, pairing,
                                                                    m.rope_offset, m.rope_dim)
        if mla:
            vals[sg.dst_pos:sg.dst_pos + sg.length] = src[..., :vdim]
        else:
            vals[sg.dst_pos:sg.dst_pos + sg.length] = oracle.bf16_bits_to_f64(
                vb[sg.src_tok:sg.src_tok + sg.length]).reshape(sg.length, -1, vdim)
    bias = oracle.sink_bias(segs, T, wl.k_nonleading, -15.0)
    oracle.attention_decode(rng.standard_normal((hq, m.head_dim)), keys, vals, scale, bias)


def _oracle_worker(conn, job):
    """One host core: maps the shared inputs, then runs each share it is sent
    (a list of unit ids) and answers with its busy seconds."""
    import traceback
    try:
        import oracle
        kind = job["kind"]
        if kind == "cdc":
            tokens = np.load(job["tokens"], mmap_mode="r")
            offsets = np.load(job["offsets"])
            gear = np.load(job["gear"])
        else:
            wl = job["wl"]
            kb = np.load(job["k"], mmap_mode="r")[0]
            vb = np.load(job["v"], mmap_mode="r")[0] if job["v"] else None
            rng = np.random.default_rng(0)
        conn.send(("ready", None))
        while True:
            share = conn.recv()
            if share is None:
                break
            t0 = time.perf_counter()
            produced = 0
            for u in share:
                if kind == "stitch":
                    sub = W.Workload(wl.name, wl.model, wl.chunk_lens, [wl.requests[u]], wl.k_nonleading,
                                     wl.k_leading)
                    run_oracle_sample(sub, kb[None], None if vb is None else vb[None], [0])
                elif kind == "attend":
                    run_oracle_attend(wl, u, kb, vb, job["hq"], rng)
                else:
                    doc = tokens[offsets[u]:offsets[u + 1]]
                    ends, _ = oracle.chunk_document(list(doc), gear, job["thr"], job["min_len"], job["max_len"])
                    produced += len(ends)
            conn.send(("done", (time.perf_counter() - t0, produced)))
    except Exception:
        conn.send(("error", traceback.format_exc()))


def balance(weights, n):
    """Split unit ids 0..len(weights)-1 over n cores: heaviest first, each to
    the least loaded core (ties to the lowest core).  Returns n lists."""
    shares = [[] for _ in range(n)]
    load = [0] * n
    for u in sorted(range(len(weights)), key=lambda u: (-weights[u], u)):
        c = min(range(n), key=lambda i: (load[i], i))
        shares[c].append(u)
        load[c] += weights[u]
    return shares


class OracleCores:
    """One spawned oracle process per host core."""

    def __init__(self, job, n=None):
        import multiprocessing as mp
        self.n = n or host_cores()
        ctx = mp.get_context("spawn")
        saved = {k: os.environ.get(k) for k in _THREAD_VARS}
        for k in _THREAD_VARS:       # one thread per process: the cores are the parallelism
            os.environ[k] = "1"
        self.procs, self.conns = [], []
        try:
            for _ in range(self.n):
                a, b = ctx.Pipe()
                p = ctx.Process(target=_oracle_worker, args=(b, job), daemon=True)
                p.start()
                self.procs.append(p)
                self.conns.append(a)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for c in self.conns:
            self._answer(c)

    @staticmethod
    def _answer(conn):
        tag, val = conn.recv()
        if tag == "error":
            raise RuntimeError("oracle process failed:\n" + val)
        return val

    def run(self, units, weights):
        """Runs the given units (ids) spread over the cores; returns (wall
        seconds, cores that got work, what the units produced in all: chunks
        for chunking, else 0)."""
        shares = balance([weights[u] for u in units], self.n)
        shares = [[units[i] for i in s] for s in shares]
        t0 = time.perf_counter()
        for c, s in zip(self.conns, shares):
            c.send(s)
        produced = sum(self._answer(c)[1] for c in self.conns)
        return time.perf_counter() - t0, sum(1 for s in shares if s), produced

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except Exception:
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()


def host_pool_bits(wl, which):
    """bf16 bits of pool layer 0, drawn on the host (the oracle's own inputs)."""
    import torch
    t = W.make_pool(W.Workload(wl.name, W.Model(**{**wl.model.__dict__, "num_layers": 1}),
                               wl.chunk_lens, wl.requests, wl.k_nonleading, wl.k_leading), which, "cpu")
    return t.view(torch.int16).numpy().view(np.uint16)


class OracleRun:
    """The oracle's stitch (kind "stitch") or decode attention ("attend") of a
    workload on all host cores.  Every unit reads pool layer 0: the oracle's
    cost per unit does not depend on the layer's values."""

    def __init__(self, wl, kind, hq=0, n=None):
        self.wl, self.kind = wl, kind
        self.dir = tempfile.mkdtemp(prefix="pic_oracle_")
        paths = {"k": os.path.join(self.dir, "k.npy"), "v": None}
        np.save(paths["k"], host_pool_bits(wl, "k"))
        if wl.model.kind == "gqa":
            paths["v"] = os.path.join(self.dir, "v.npy")
            np.save(paths["v"], host_pool_bits(wl, "v"))
        self.cores = OracleCores({"kind": kind, "wl": wl, "hq": hq, **paths}, n)
        # units, layer-major: every request of layer 0, then of layer 1, ...
        R = len(wl.requests)
        self.units = [r for _ in range(wl.model.num_layers) for r in range(R)]
        self.weights = {r: t for r, t in enumerate(wl.request_tokens)}

    def sample(self, wall_s):
        """The first units (layer-major) that keep every core busy for about
        wall_s seconds: a whole number of units per core, at least one,
        sized by two runs of one unit per core (the first warms the cores up)
        and at most the whole workload.  Returns the number of units."""
        n = self.cores.n
        first = self.units[:n]
        for _ in range(2):
            el, _, _ = self.cores.run(first, self.weights)
        rate = sum(self.weights[u] for u in first) / max(el, 1e-6)   # token-layers/s, all cores
        want = rate * wall_s
        k, acc = 0, 0
        while k < len(self.units) and (k < n or acc < want):
            acc += self.weights[self.units[k]]
            k += 1
        return min(len(self.units), -(-k // n) * n)

    def run(self, k):
        """Runs the first k units; returns (wall seconds, token-layers, cores used)."""
        units = self.units[:k]
        el, used, _ = self.cores.run(units, self.weights)
        return el, sum(self.weights[u] for u in units), used

    def describe(self, k):
        wl = self.wl
        R, L = len(wl.requests), wl.model.num_layers
        if k == R * L:
            return f"the whole workload ({R} request(s) x {L} layers)"
        return (f"{k} of the workload's {R * L} (request, layer) units, layer-major "
                f"({k // R} whole layer(s) of every request" + (f" + {k % R} request(s)" if k % R else "") + ")")

    def close(self):
        self.cores.close()
        import shutil
        shutil.rmtree(self.dir, ignore_errors=True)


def cpu_baseline(wl, mode="stitch", hq=0, cpu_seconds=24.0):
    """Oracle rate on a bounded sample spread over all host cores: about
    cpu_seconds of CPU work in all (whole units, layer-major)."""
    run = OracleRun(wl, mode, hq)
    try:
        k = run.sample(cpu_seconds / run.cores.n)
        el, tl, used = run.run(k)
    finally:
        run.close()
    m = wl.model
    if mode == "attend":
        row = m.num_kv_heads * m.head_dim * 2
        bpt = row * (1 if m.kind == "mla" else 2)
    else:
        bpt = bytes_per_token_layer(m, "stitch")
    what = f"{hq} query heads, " if mode == "attend" else ""
    return {"value": tl * bpt / el / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": f"{run.describe(k)}: {tl} token-layers, {what}{el:.2f} s wall on {used} host cores "
                      f"(fp64 numpy, one process per core)",
            "tokens_layers_per_s": tl / el}


def run_reference(args, wl, budget_s=None):
    """Reference arm: the fp64 oracle timed on all host cores.  A step is the
    whole workload when K + W of them fit in about budget_s seconds, else the
    first (request, layer) units, layer-major, that do; the bytes counted are
    the sample's."""
    budget_s = args.ref_seconds if budget_s is None else budget_s
    run = OracleRun(wl, "stitch")
    try:
        k = run.sample(budget_s / (args.steps + args.warmup))
        for _ in range(args.warmup):
            run.run(k)
        times, used = [], 0
        for _ in range(args.steps):
            el, tl, used = run.run(k)
            times.append(el)
    finally:
        run.close()
    el = sum(times)
    tl_all = tl * args.steps
    gbs = tl_all * bytes_per_token_layer(wl.model, "stitch") / el / 1e9
    sample = run.describe(k)
    line = {
        "impl": "reference", "metric": "stitched KV GB/s", "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {WORKLOAD_TEXT.get(wl.name, '')}",
                   "step": f"{sample} ({tl} token-layers), bounded sample"},
        "tokens_layers_per_s": tl_all / el,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": f"{sample} per step, on {used} host cores (fp64 numpy, one process per core)"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU arm

class Rig:
    """Everything one rank needs to run steps of a workload through the C ABI."""

    def __init__(self, wl, device, mode, q_heads=0):
        import torch
        from position_independent_kv_stitch_gb300 import pic
        self.torch, self.pic = torch, pic
        self.wl, self.m, self.dev, self.mode = wl, wl.model, device, mode
        m = wl.model
        self.bs = m.block_size
        self.nb = sum(-(-t // self.bs) for t in wl.request_tokens)
        self.max_blocks = max(-(-t // self.bs) for t in wl.request_tokens)
        self.ctx = pic.create_from_spec(pic.model_spec_from(m), self.nb)
        self.ids = [pic.pic_register_chunk(self.ctx, W.chunk_key(wl.name, c), off, n)[0]
                    for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens))]
        self.k_pool = W.make_pool(wl, "k", device=device)
        self.v_pool = W.make_pool(wl, "v", device=device) if m.kind == "gqa" else None
        self.chunk_blocks = None
        if mode == "mapped":
            # chunks resident in cache blocks (after the requests' own blocks)
            pic.pic_destroy(self.ctx)
            nblk = [-(-n // self.bs) for n in wl.chunk_lens]
            first = self.nb
            self.nb += sum(nblk)
            self.ctx = pic.create_from_spec(pic.model_spec_from(m), self.nb)
            self.chunk_blocks = []
            b = first
            for n in nblk:
                self.chunk_blocks.append(list(range(b, b + n)))
                b += n
        shape = (m.num_layers, self.nb, self.bs) + tuple(m.row_shape)
        self.k_cache = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.v_cache = torch.empty(shape, dtype=torch.bfloat16, device=device) if m.kind == "gqa" else None
        self.orders = None
        if mode == "mapped":
            self._load_chunks_into_blocks()
        self.ws_bytes = 0
        for _ in range(2 if self.orders is not None else 1):   # both orders of the mapped mode
            plans, bt = self.plan()
            self.n_rec = sum(pic.pic_plan_info(p)["num_recompute"] for p in plans)
            self.ws_bytes = max(self.ws_bytes, pic.pic_workspace_bytes(self.ctx, plans))
            self.free(plans)
        self.ridx = torch.empty(max(1, self.n_rec), dtype=torch.int32, device=device)
        self.indptr = torch.empty(len(wl.requests) + 1, dtype=torch.int32, device=device)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.d_bt = torch.empty((len(wl.requests), self.max_blocks), dtype=torch.int32, device=device)
        self.bt_pinned = [torch.empty_like(self.d_bt, device="cpu").pin_memory() for _ in range(2)]
        self.bt_events = [None, None]
        self.slot = 0
        self.moved = 0
        self.shift_segs = None
        self.attn = None
        if mode in ("attend", "attend_cache"):
            # GQA: 4 query heads per KV head (Llama-3.1-8B: 32 over 8); MLA: 16
            # query heads over the latent (DeepSeek-V3's 128 split over 8 GPUs)
            hq = q_heads or (16 if m.kind == "mla" else 4 * m.num_kv_heads)
            vdim = m.head_dim - m.rope_dim if m.kind == "mla" else m.head_dim
            g = torch.Generator(device=device)
            g.manual_seed(11)
            q = torch.empty((m.num_layers, len(wl.requests), hq, m.head_dim), dtype=torch.bfloat16, device=device)
            q.normal_(0.0, 1.0, generator=g)
            # A decode loop attends to the same composed requests every step:
            # the plans and block tables are built once and kept.
            plans, bt = self.plan()
            self.attn_plans = plans
            self.d_bt.copy_(torch.from_numpy(bt))
            aws = pic.pic_attend_workspace_bytes(self.ctx, plans, hq, m.num_layers)
            self.attn = {
                "q": q, "hq": hq,
                "scale": 1.0 / (192 ** 0.5) if m.kind == "mla" else 1.0 / (m.head_dim ** 0.5),
                "out": torch.empty((m.num_layers, len(wl.requests), hq, vdim), dtype=torch.float32, device=device),
                "lse": torch.empty((m.num_layers, len(wl.requests), hq), dtype=torch.float32, device=device),
                "ws": torch.empty(aws, dtype=torch.uint8, device=device),
            }
        if mode == "inplace":
            self.shift_segs = self._shift_segments()
            self.ws_shift = torch.empty(pic.pic_rerotate_workspace_bytes(self.ctx, self.shift_segs),
                                        dtype=torch.uint8, device=device)

    def _load_chunks_into_blocks(self):
        """Writes every pool chunk into its cache blocks (rows 0.. of each) and
        registers it as block-resident at position 0; requests then alternate
        between their own chunk order and a second seeded order, so mapped
        chunks really move every step."""
        torch, pic, wl = self.torch, self.pic, self.wl
        bs = self.bs
        self.ids = []
        for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens)):
            blks = self.chunk_blocks[c]
            for j, b in enumerate(blks):
                t0, t1 = j * bs, min(n, (j + 1) * bs)
                self.k_cache[:, b, :t1 - t0] = self.k_pool[:, off + t0:off + t1]
                if self.v_cache is not None:
                    self.v_cache[:, b, :t1 - t0] = self.v_pool[:, off + t0:off + t1]
            self.ids.append(pic.pic_register_chunk_blocks(self.ctx, W.chunk_key(wl.name, c), blks, n, 0)[0])
        alt = []
        for r, req in enumerate(wl.requests):
            head, rest = req[:1], list(req[1:])
            perm = W.Stream(1, f"mapped/order/{r}").permutation(len(rest))
            alt.append(head + [rest[i] for i in perm])
        self.orders = [wl.requests, alt]
        self.step_no = 0

    def _shift_segments(self):
        plans, bt = self.plan()
        segs = []
        for r, plan in enumerate(plans):
            for j in range(self.pic.pic_plan_info(plan)["num_segments"]):
                s = self.pic.pic_plan_segment(plan, j)
                new = self.wl.new_pos[r][j] if self.wl.new_pos else s["dst_pos"] + 100003
                segs.append((r, s["dst_pos"], s["num_tokens"], new - s["dst_pos"]))
        self.d_bt.copy_(self.torch.from_numpy(bt))
        self._kept_plans = plans
        # fill the cache with stitched keys once, so the shift runs on real data
        self.pic.pic_stitch(self.ctx, plans, self.k_pool, self.v_pool, self.k_cache, self.v_cache, self.d_bt,
                            self.ridx, self.indptr, self.ws)
        return segs

    def plan(self):
        pic, wl = self.pic, self.wl
        plans, tables = [], []
        reqs = wl.requests
        if self.orders is not None:
            reqs = self.orders[self.step_no % 2]
            self.step_no += 1
        for req in reqs:
            plan, bt = pic.pic_build_block_table(self.ctx, [self.ids[c] for c, _ in req], self.max_blocks,
                                                 take_tokens=[t for _, t in req],
                                                 k_nonleading=wl.k_nonleading, k_leading=wl.k_leading,
                                                 alias=self.orders is not None)
            plans.append(plan)
            tables.append(bt)
        return plans, np.stack(tables)

    def moved_bytes(self, plans):
        """Bytes a stitch of these plans must move: copied rows read + written
        (K and V), mapped keys read + written when they move, nothing else."""
        pic = self.pic
        row = self.m.num_kv_heads * self.m.head_dim * 2
        tensors = 2 if self.m.kind == "gqa" else 1
        total = 0
        for plan in plans:
            for j in range(pic.pic_plan_info(plan)["num_segments"]):
                sg = pic.pic_plan_segment(plan, j)
                mode = pic.pic_plan_segment_mode(plan, j)
                if mode == pic.PIC_SEG_MAPPED:
                    total += 0 if sg["delta"] == 0 else 2 * row * sg["num_tokens"]
                else:
                    total += 2 * tensors * row * sg["num_tokens"]
        return total * self.m.num_layers

    def free(self, plans):
        for p in plans:
            self.pic.pic_free_request(self.ctx, p)

    def upload_tables(self, bt):
        s = self.slot
        if self.bt_events[s] is not None:
            self.bt_events[s].synchronize()
        self.bt_pinned[s].numpy()[...] = bt
        self.d_bt.copy_(self.bt_pinned[s], non_blocking=True)
        ev = self.torch.cuda.Event()
        ev.record()
        self.bt_events[s] = ev
        self.slot ^= 1

    def step(self, kernel_events=None):
        """One step: plan + table upload + one launch (in place: one shift
        launch; attend modes: one decode step over the plans built at set-up,
        stitched first for attend_cache); returns nothing."""
        if self.mode == "inplace":
            if kernel_events:
                kernel_events[0].record()
            self.pic.pic_rerotate_inplace(self.ctx, self.k_cache, self.d_bt, self.shift_segs, self.ws_shift)
            if kernel_events:
                kernel_events[1].record()
            return
        if self.attn is not None:
            # one decode step over the kept plans (attend_cache: stitched first)
            plans, a = self.attn_plans, self.attn
            if kernel_events:
                kernel_events[0].record()
            if self.mode == "attend_cache":
                self.pic.pic_stitch(self.ctx, plans, self.k_pool, self.v_pool, self.k_cache, self.v_cache,
                                    self.d_bt, self.ridx, self.indptr, self.ws)
            src = self.pic.PIC_ATTEND_FUSED if self.mode == "attend" else self.pic.PIC_ATTEND_CACHE
            self.pic.pic_attend_decode(self.ctx, plans, src, a["q"], a["scale"], self.k_pool, self.v_pool,
                                       self.k_cache, self.v_cache, a["out"], a["lse"], a["ws"], sink_bias=-15.0)
            if kernel_events:
                kernel_events[1].record()
            return
        plans, bt = self.plan()
        if self.orders is not None:
            self.moved += self.moved_bytes(plans)
        self.upload_tables(bt)
        if kernel_events:
            kernel_events[0].record()
        self.pic.pic_stitch(self.ctx, plans, self.k_pool, self.v_pool, self.k_cache, self.v_cache, self.d_bt,
                            self.ridx, self.indptr, self.ws)
        if kernel_events:
            kernel_events[1].record()
        self.free(plans)

    def check_status(self):
        ws = self.ws_shift if self.mode == "inplace" else self.ws
        self.pic.pic_query_device_status(self.ctx, ws)
        if self.attn is not None:
            self.pic.pic_query_device_status(self.ctx, self.attn["ws"])


E2E_GROUPS = 32  # request groups of the staged end-to-end leg (measured: 4, 8, 16, 32 groups took 202.6, 197.7, 195.4, 194.3 ms on serving stress)


def run_e2e(rig, steps, warmup, cache_on_host=False, stage=False):
    """Same metric end to end through the public API with the chunk pool in
    HOST memory: the pool lives in pinned host memory (a host-side chunk
    store), so the pool's bytes cross host->device inside the timed region
    every step.  Streamed (stage False): the stitch kernel reads the pool
    over the host link directly (on GB300, NVLink-C2C to Grace memory), a row
    as often as the batch places it.  Staged: pic_stitch_staged copies every
    pool row the batch reads, once, into the device pool buffers (cleared
    before the first step, so only this leg's copies feed the stitch), in
    groups of requests, each stitched from HBM while the next is copied.  The
    paged cache is in HBM,
    where decode attention reads it (cache_on_host: in pinned host memory
    too, so the stitched bytes also cross device->host).  Each step also
    plans, uploads the block table and reads the recompute list back to the
    host."""
    torch = rig.torch
    pic = rig.pic
    def pinned_copy(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    hk = pinned_copy(rig.k_pool)
    hv = pinned_copy(rig.v_pool) if rig.v_pool is not None else None
    if cache_on_host:
        hkc = torch.empty(rig.k_cache.shape, dtype=rig.k_cache.dtype).pin_memory()
        hvc = torch.empty(rig.v_cache.shape, dtype=rig.v_cache.dtype).pin_memory() if rig.v_cache is not None else None
    else:
        hkc, hvc = rig.k_cache, rig.v_cache
    oi = torch.empty_like(rig.ridx, device="cpu").pin_memory()
    op = torch.empty_like(rig.indptr, device="cpu").pin_memory()

    staged = [0]
    if stage:
        rig.k_pool.zero_()
        if rig.v_pool is not None:
            rig.v_pool.zero_()
        plans0, _ = rig.plan()
        ws_staged = torch.empty(pic.pic_stitch_staged_workspace_bytes(rig.ctx, plans0, E2E_GROUPS), dtype=torch.uint8,
                                device=rig.d_bt.device)
        rig.free(plans0)

    def one():
        plans, bt = rig.plan()
        rig.upload_tables(bt)
        if stage:
            # request groups staged on the library's copy stream while the
            # earlier groups stitch, into the device pool buffers
            staged[0] = pic.pic_stitch_staged(rig.ctx, plans, hk, hv, rig.k_pool, rig.v_pool, hkc, hvc, rig.d_bt,
                                              rig.ridx, rig.indptr, ws_staged, n_groups=E2E_GROUPS)
        else:
            pic.pic_stitch(rig.ctx, plans, hk, hv, hkc, hvc, rig.d_bt, rig.ridx, rig.indptr, rig.ws)
        oi.copy_(rig.ridx, non_blocking=True)
        op.copy_(rig.indptr, non_blocking=True)
        rig.free(plans)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    pic.pic_query_device_status(rig.ctx, ws_staged if stage else rig.ws)
    ms = e0.elapsed_time(e1) / steps
    wl = rig.wl
    rows = wl.token_layers * rig.m.num_kv_heads * rig.m.head_dim * 2   # bytes of K rows moved
    tensors = 2 if hv is not None else 1
    pool = staged[0] if stage else rows * tensors
    h2d = pool + rig.d_bt.numel() * 4 + (ws_staged.numel() if stage else rig.ws_bytes)
    d2h = (rows * tensors if cache_on_host else 0) + oi.numel() * 4 + op.numel() * 4
    return ms, h2d, d2h


# ------------------------------------------------- content-defined chunking

CDC_TEXT = ("rag_corpus: 8,192 documents of log-uniform 512-16,384 tokens (37.6M int32 token ids, uniform over a "
            "128,256-id vocabulary), Gear hash over 64-token windows, xxHash64 fingerprints")


def cdc_oracle_sample(corpus, thr, min_len, max_len, cpu_seconds=24.0):
    """The oracle as it stands, on all host cores: whole documents in corpus
    order, about cpu_seconds of CPU work in all (sized by a run of one
    document per core).  Returns (documents, tokens, chunks, wall s, cores)."""
    d = tempfile.mkdtemp(prefix="pic_cdc_oracle_")
    paths = {k: os.path.join(d, k + ".npy") for k in ("tokens", "offsets", "gear")}
    np.save(paths["tokens"], corpus.tokens)
    np.save(paths["offsets"], corpus.offsets)
    np.save(paths["gear"], corpus.gear)
    cores = OracleCores({"kind": "cdc", "thr": thr, "min_len": min_len, "max_len": max_len, **paths})
    try:
        lens = np.diff(corpus.offsets).tolist()
        first = list(range(min(cores.n, corpus.n_docs)))
        el, _, _ = cores.run(first, lens)
        want = sum(lens[u] for u in first) / max(el, 1e-6) * cpu_seconds / cores.n
        k, acc = 0, 0
        while k < corpus.n_docs and (k == 0 or acc < want):
            acc += lens[k]
            k += 1
        el, used, n_chunks = cores.run(list(range(k)), lens)
    finally:
        cores.close()
        import shutil
        shutil.rmtree(d, ignore_errors=True)
    return k, int(sum(lens[:k])), n_chunks, el, used


def run_cdc(args):
    """One step = content-defined chunking of the whole corpus: every kernel
    of pic_cdc_chunk (offset checks, Gear hash + cut bits, [length rules],
    counts, scan, chunk ends, fingerprints)."""
    import torch
    import torch.distributed as dist
    import oracle
    from position_independent_kv_stitch_gb300 import pic
    from position_independent_kv_stitch_gb300.sharding import max_over_ranks
    pic.load()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    corpus = W.rag_corpus()
    thr = oracle.threshold_for_mean(args.cdc_mean) if args.cdc_mean > 0 else 0
    n_tok, n_docs = len(corpus.tokens), corpus.n_docs
    tokens = torch.from_numpy(corpus.tokens).to(dev)
    offsets = torch.from_numpy(corpus.offsets).to(dev)
    gear = torch.from_numpy(corpus.gear.view(np.int64)).to(dev)
    cap = n_tok // 4 + n_docs   # room for chunks of 4 tokens on average
    indptr = torch.empty(n_docs + 1, dtype=torch.int64, device=dev)
    ends = torch.empty(cap, dtype=torch.int64, device=dev)
    fps = torch.empty(cap, dtype=torch.int64, device=dev)
    ws = torch.empty(pic.pic_cdc_workspace_bytes(n_tok), dtype=torch.uint8, device=dev)

    def step(toks=tokens):
        pic.pic_cdc_chunk(toks, offsets, gear, thr, indptr, ends, fps, args.cdc_min, args.cdc_max, 0, workspace=ws)

    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == args.warmup - 1:
            w0.record()
        step()
    w1.record()
    torch.cuda.synchronize()
    if args.steps is None:
        args.steps = auto_steps(w0.elapsed_time(w1), dev)
    if pic.pic_query_device_status(None, ws) != 0:
        raise RuntimeError("chunking reported a device error")
    n_chunks = int(indptr[-1].item())
    if n_chunks > cap:
        raise RuntimeError("chunk capacity too small")

    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    t0.record()
    for i in range(args.steps):
        evs[i][0].record()
        step()
        evs[i][1].record()
    t1.record()
    torch.cuda.synchronize()
    clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    pic.pic_query_device_status(None, ws)
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, dev)
    kms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    dev_props = torch.cuda.get_device_properties(dev)
    gather_mhz = (clk or {}).get("sm_mhz") or 2070.0  # the GB300's maximum SM clock when unsampled

    # algorithmic bytes: token ids read once, offsets read, CSR offsets + ends + fingerprints written
    algo = 4 * n_tok + 8 * (n_docs + 1) * 2 + 16 * n_chunks
    peak, peak_kind = measured_peak()
    value = world * algo / (ms * 1e-3) / 1e9

    # end to end: token ids from pinned host memory, chunk ends and
    # fingerprints back, pipelined over document groups: group g + 1's ids
    # are copied on a copy stream while group g is chunked (documents are
    # independent, so each group is one pic_cdc_chunk call over its own
    # documents; its token view starts at a 16-byte boundary, up to 3 ids
    # before its first document, and its offsets are rebased to that view)
    htok = torch.from_numpy(corpus.tokens).pin_memory()
    dtok = torch.empty_like(tokens)
    G = min(8, n_docs)
    db = [n_docs * g // G for g in range(G + 1)]
    ind_all = indptr.cpu().numpy()
    copy_stream = torch.cuda.Stream(dev)
    grp = []
    for g in range(G):
        d0, d1 = db[g], db[g + 1]
        lo, hi = int(corpus.offsets[d0]), int(corpus.offsets[d1])
        base = lo & ~3
        n_ch = int(ind_all[d1] - ind_all[d0])
        grp.append(dict(lo=lo, hi=hi, base=base, n_ch=n_ch,
                        offs=torch.from_numpy(corpus.offsets[d0:d1 + 1] - base).to(dev),
                        indptr=torch.empty(d1 - d0 + 1, dtype=torch.int64, device=dev),
                        ends=torch.empty(n_ch + 16, dtype=torch.int64, device=dev),
                        fps=torch.empty(n_ch + 16, dtype=torch.int64, device=dev),
                        hind=torch.empty(d1 - d0 + 1, dtype=torch.int64).pin_memory(),
                        hends=torch.empty(n_ch + 16, dtype=torch.int64).pin_memory(),
                        hfps=torch.empty(n_ch + 16, dtype=torch.int64).pin_memory(),
                        ws=torch.empty(pic.pic_cdc_workspace_bytes(hi - base), dtype=torch.uint8, device=dev)))

    def e2e_step():
        cur = torch.cuda.current_stream(dev)
        # this step's copies start once the last step's chunking is done
        copy_stream.wait_stream(cur)
        for x in grp:
            with torch.cuda.stream(copy_stream):
                dtok[x["lo"]:x["hi"]].copy_(htok[x["lo"]:x["hi"]], non_blocking=True)
            cur.wait_stream(copy_stream)
            pic.pic_cdc_chunk(dtok[x["base"]:x["hi"]], x["offs"], gear, thr, x["indptr"], x["ends"], x["fps"],
                              args.cdc_min, args.cdc_max, 0, workspace=x["ws"])
            x["hind"].copy_(x["indptr"], non_blocking=True)
            x["hends"][:x["n_ch"]].copy_(x["ends"][:x["n_ch"]], non_blocking=True)
            x["hfps"][:x["n_ch"]].copy_(x["fps"][:x["n_ch"]], non_blocking=True)

    e2e = None
    if not args.no_e2e:
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        k = max(3, min(args.steps, 20))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(k):
            e2e_step()
        b.record()
        torch.cuda.synchronize()
        ems = max_over_ranks(a.elapsed_time(b) / k, dev)
        for x in grp:
            if pic.pic_query_device_status(None, x["ws"]) != 0:
                raise RuntimeError("chunking reported a device error")
        got = sum(int(x["hind"][-1]) for x in grp)
        if got != n_chunks:
            raise RuntimeError(f"document groups gave {got} chunks, the whole corpus {n_chunks}")
        e2e = {"value": world * algo / (ems * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ems,
               "h2d_bytes_per_step": 4 * (n_tok - int(corpus.offsets[0])),
               "d2h_bytes_per_step": 8 * (n_docs + G) + 16 * n_chunks,
               "how": f"token ids copied from pinned host memory, chunk offsets, ends and fingerprints copied back; "
                      f"{G} document groups, group g + 1's ids copied on a copy stream while group g is chunked"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        d, ntk, nch, el, used = cdc_oracle_sample(corpus, thr, args.cdc_min, args.cdc_max)
        cpu_algo = 4 * ntk + 16 * nch + 16 * (d + 1)
        cpu = {"value": cpu_algo / el / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": f"first {d} documents ({ntk} tokens, {nch} chunks), {el:.2f} s wall on {used} host "
                         f"cores (Python, one process per core)",
               "tokens_per_s": ntk / el}

    line = {
        "metric": "CDC token GB/s", "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u64", "data": "synthetic",
        "config": {"workload": CDC_TEXT, "mode": "cdc", "threshold_mean_len": args.cdc_mean,
                   "min_len": args.cdc_min, "max_len": args.cdc_max, "tokens_per_step_per_gpu": n_tok,
                   "documents": n_docs, "chunks": n_chunks, "algorithmic_bytes_per_step_per_gpu": algo,
                   "l2": "no flush: the 150 MB of token ids exceed the 129 MB L2",
                   "parallelism": f"replicas x{world} (independent corpora per GPU, no collective)"},
        "tokens_per_s": world * n_tok / (ms * 1e-3),
        "pct_hbm_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "hbm", "kernel": "pic_cdc_chunk (all launches; k_cdc_hash dominant)",
                     "achieved": algo / (kms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": algo / (kms * 1e-3) / 1e9 / peak, "peak_source": peak_kind,
                     "traffic": recorded_traffic("rag_corpus/cdc" if not (args.cdc_min or args.cdc_max) else "-"),
                     "algorithmic_bytes_per_launch": algo, "launch_ms": kms},
        # The bound that binds here is not HBM: every token costs one random
        # 8-byte Gear load, one L1TEX request of its own (a warp's 32 loads
        # are 32 requests), and an SM takes about one request per cycle.
        "roofline_gather": {"bound": "l1tex requests", "kernel": "pic_cdc_chunk (all launches)",
                            "achieved": n_tok / (kms * 1e-3), "unit": "requests/s",
                            "peak": dev_props.multi_processor_count * gather_mhz * 1e6,
                            "frac": n_tok / (kms * 1e-3) / (dev_props.multi_processor_count * gather_mhz * 1e6),
                            "peak_source": f"one request per SM per cycle at {gather_mhz:.0f} MHz "
                                           f"(the median SM clock of the timed region)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (7 if (args.cdc_min > 1 or args.cdc_max > 0) else 5),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def auto_steps(step_ms, dev):
    """Timed steps when --steps is not given: about 10 s of steps, 20 to 1000,
    the same on every rank (sized by the slowest rank's last warm-up step)."""
    from position_independent_kv_stitch_gb300.sharding import max_over_ranks
    ms = max_over_ranks(step_ms, dev)
    return int(min(1000, max(20, 10000.0 / max(ms, 1e-3))))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 10 s of GPU steps, 20 to 1000; 20 for the reference arm)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pic", choices=["pic", "reference"])
    ap.add_argument("--workload", default="serving_stress", choices=sorted(W.WORKLOADS))
    ap.add_argument("--mode", default="stitch",
                    choices=["stitch", "inplace", "mapped", "attend", "attend_cache", "cdc"])
    ap.add_argument("--cdc-mean", type=int, default=64, help="cdc mode: mean chunk length the threshold aims at")
    ap.add_argument("--cdc-min", type=int, default=0, help="cdc mode: minimum chunk length (0: none)")
    ap.add_argument("--cdc-max", type=int, default=0, help="cdc mode: maximum chunk length (0: none)")
    ap.add_argument("--q-heads", type=int, default=0, help="query heads for the attend modes (default 4 per KV head)")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling captures only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-cache-on-host", action="store_true",
                    help="end-to-end leg: keep the paged cache in pinned host memory too")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: about how long all its steps (warm-up and timed) may take")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = W.WORKLOADS[args.workload]()
    if args.layers:
        wl = W.Workload(wl.name, W.Model(**{**wl.model.__dict__, "num_layers": args.layers}), wl.chunk_lens,
                        wl.requests, wl.k_nonleading, wl.k_leading, wl.new_pos)

    if args.impl == "reference":
        if rank != 0:
            return
        if args.steps is None:
            args.steps = 20
        if args.mode != "stitch":
            # only the stitch has a reference arm; every mode's own line
            # carries an oracle timing in its cpu_baseline field
            print(json.dumps({"impl": "reference", "unavailable": f"only --mode stitch has a reference arm (the oracle's "
                              f"stitch); the --mode {args.mode} line carries an oracle timing in cpu_baseline"}),
                  flush=True)
            return
        run_reference(args, wl)
        return
    if args.mode == "cdc":
        run_cdc(args)
        return

    import torch
    import torch.distributed as dist
    from position_independent_kv_stitch_gb300 import pic
    from position_independent_kv_stitch_gb300.sharding import max_over_ranks
    pic.load()  # fails loudly when libpic is not built
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    rig = Rig(wl, dev, args.mode, args.q_heads)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == args.warmup - 1:
            w0.record()
        rig.step()
    w1.record()
    torch.cuda.synchronize()
    rig.check_status()
    if args.steps is None:
        args.steps = auto_steps(w0.elapsed_time(w1), dev)

    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rig.moved = 0
    clocks.mark_start()
    t0.record()
    for i in range(args.steps):
        rig.step(kev[i])
    t1.record()
    torch.cuda.synchronize()
    clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    rig.check_status()
    ms = t0.elapsed_time(t1) / args.steps
    kms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    ms = max_over_ranks(ms, dev)

    tl = wl.token_layers
    if args.mode == "mapped":
        algo_bytes = rig.moved / args.steps           # bytes actually moved per step
        bpt = algo_bytes / tl
    elif args.mode in ("attend", "attend_cache"):
        # attention reads every context K and V row once (MLA: the one latent
        # row serves as both); the cache path also stitches first (pool read +
        # cache write)
        row = wl.model.num_kv_heads * wl.model.head_dim * 2
        tensors = 1 if wl.model.kind == "mla" else 2
        bpt = tensors * row + (2 * tensors * row if args.mode == "attend_cache" else 0)
        algo_bytes = tl * bpt
    else:
        bpt = bytes_per_token_layer(wl.model, args.mode)
        algo_bytes = tl * bpt
    peak, peak_kind = measured_peak()
    value = world * algo_bytes / (ms * 1e-3) / 1e9
    achieved = algo_bytes / (kms * 1e-3) / 1e9
    # the recorded DRAM bytes are for the workload at full size, default heads
    traffic = recorded_traffic(f"{wl.name}/{args.mode}") if not (args.layers or args.q_heads) else None

    e2e = None
    if not args.no_e2e and args.mode == "stitch":
        # Stage the pool rows in HBM when the batch reads rows more than once
        # (the rule a caller applies: each distinct row then crosses the host
        # link once instead of once per placement); else stream them.
        plans, _ = rig.plan()
        distinct, read = pic.pic_pool_read_rows(rig.ctx, plans)
        rig.free(plans)
        stage = not args.e2e_cache_on_host and distinct * 10 < read * 9
        e_steps = max(3, min(args.steps, 10))
        legs = [("streamed", False)] + ([("staged", True)] if stage else [])
        res = {}
        for name, st in legs:
            ems, h2d, d2h = run_e2e(rig, e_steps, 3, args.e2e_cache_on_host, stage=st)
            res[name] = (max_over_ranks(ems, dev), h2d, d2h)
        ems, h2d, d2h = res["staged" if stage else "streamed"]
        where = "pool and cache" if args.e2e_cache_on_host else "pool"
        how = (f"{where} in pinned host memory; each step pic_stitch_staged copies the pool rows the batch reads, "
               f"each once ({distinct} of the {read} rows read per layer), into the device pool buffers, and "
               f"stitches from HBM: {E2E_GROUPS} request groups, group g + 1 staged on the library's copy stream while "
               f"group g is stitched" if stage else
               f"{where} in pinned host memory, streamed by the kernel over NVLink-C2C")
        e2e = {"value": world * algo_bytes / (ems * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ems,
               "how": how + ("" if args.e2e_cache_on_host else ", cache written to HBM")
                      + "; block table up, recompute list down"}
        if stage:
            sms, sh2d, _ = res["streamed"]
            e2e["streamed"] = {"value": world * algo_bytes / (sms * 1e-3) / 1e9, "ms_per_step": sms,
                               "h2d_bytes_per_step": int(sh2d),
                               "how": "the same pool streamed by the stitch kernel over NVLink-C2C, a row per placement"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(wl, "attend", rig.attn["hq"]) if args.mode == "attend" else cpu_baseline(wl)

    bulk = pic.pic_kernel_variant(rig.ctx, 1 if args.mode == "inplace" else 0) == pic.PIC_VARIANT_BULK_PIPELINE
    if bulk and args.mode not in ("attend", "attend_cache"):
        kname = "k_tma_pipeline<" + ("stitch K+V" if wl.model.kind == "gqa" else "stitch MLA rows") \
            + ">" if args.mode != "inplace" else "k_tma_pipeline<in place>"
    else:
        tc = pic.pic_kernel_variant(rig.ctx, 2) == pic.PIC_VARIANT_TENSOR_CORE_TMEM
        kname = {"stitch": "k_stitch_mla" if wl.model.kind == "mla" else "k_rotate_rows<stitch>",
                 "mapped": "k_rotate_rows<stitch, mapped chunks in place>",
                 "attend": ("k_attend_mla_tc (tcgen05, TMEM, TMA tensor loads)" if tc
                            else "k_attend_mla" if wl.model.kind == "mla" else "k_attend")
                 + " + k_attend_merge (fused delta-rotation)",
                 "attend_cache": "stitch, then decode attention over the cache",
                 "inplace": "k_rotate_rows<in place>"}[args.mode]
    line = {
        "metric": "stitched KV GB/s", "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {WORKLOAD_TEXT.get(wl.name, '')}"
                   + (f" [layers overridden to {args.layers}]" if args.layers else ""), "mode": args.mode,
                   "token_layers_per_step_per_gpu": tl, "algorithmic_bytes_per_step_per_gpu": algo_bytes,
                   "bytes_per_token_layer": bpt, "requests_per_gpu": len(wl.requests),
                   "l2": "no flush: pool and cache are each larger than the 129 MB L2",
                   "parallelism": f"replicas x{world} (independent requests per GPU, no collective)"},
        "tokens_layers_per_s": world * tl / (ms * 1e-3),
        "pct_hbm_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": traffic, "algorithmic_bytes_per_launch": algo_bytes,
                     "launch_ms": kms},
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per step: the stitch or shift kernel; attention adds its merge kernel
        "gpu_launches": args.steps * {"stitch": 1, "mapped": 1, "inplace": 1, "attend": 2, "attend_cache": 3}[args.mode],
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    pic.pic_destroy(rig.ctx)


if __name__ == "__main__":
    main()
