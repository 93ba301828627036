"""Helpers for the GPU parity tests: buffer set-up and comparisons.

The tolerance for rotated keys is the contract's: per element
|gpu - oracle| <= 2^-7 |oracle| + 1e-3.  Copies (values, MLA latent, block
tables, indices) must be bit-exact."""

import numpy as np
import torch

import oracle
import workloads as W
from position_independent_kv_stitch_gb300 import pic

REL, ABS = 2.0 ** -7, 1e-3
SENTINEL = -1  # int16 view of the bf16 NaN pattern 0xFFFF


def bits(t) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns (on the host)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t) -> np.ndarray:
    return t.float().cpu().double().numpy()


def sentinel_like(shape, device):
    return torch.full(shape, SENTINEL, dtype=torch.int16, device=device).view(torch.bfloat16)


def assert_k_close(got, want, what=""):
    """Element-wise contract tolerance; NaN in `want` marks rows nothing may write."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    written = ~np.isnan(want)
    err = np.abs(got[written] - want[written])
    bound = REL * np.abs(want[written]) + ABS
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, worst {err.max():.3e}"
    return err


def rel_l2(got, want):
    m = ~np.isnan(want)
    return float(np.linalg.norm(got[m] - want[m]) / np.linalg.norm(want[m]))


class Stitched:
    """One stitch of a workload through the C ABI, with its inputs kept for checks."""

    def __init__(self, wl: W.Workload, device="cuda", pool_device=None, spare_blocks=0,
                 k_pool=None, v_pool=None):
        self.wl = wl
        m = wl.model
        self.m = m
        self.bs = m.block_size
        self.nb = sum(-(-t // self.bs) for t in wl.request_tokens) + spare_blocks
        self.max_blocks = max(-(-t // self.bs) for t in wl.request_tokens)
        self.ctx = pic.create_from_spec(pic.model_spec_from(m), self.nb)
        ids = [pic.pic_register_chunk(self.ctx, W.chunk_key(wl.name, c), off, n)[0]
               for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens))]
        self.plans, tables = [], []
        for req in wl.requests:
            plan, bt = pic.pic_build_block_table(self.ctx, [ids[c] for c, _ in req], self.max_blocks,
                                                 take_tokens=[t for _, t in req],
                                                 k_nonleading=wl.k_nonleading, k_leading=wl.k_leading)
            self.plans.append(plan)
            tables.append(bt)
        self.tables = np.stack(tables)
        pool_device = pool_device or device
        self.k_pool = k_pool if k_pool is not None else W.make_pool(wl, "k", device=pool_device)
        if pool_device != device:
            self.k_pool = self.k_pool.to(device)
        self.v_pool = None
        if m.kind == "gqa":
            self.v_pool = v_pool if v_pool is not None else W.make_pool(wl, "v", device=pool_device)
            if pool_device != device:
                self.v_pool = self.v_pool.to(device)
        shape = (m.num_layers, self.nb, self.bs) + tuple(m.row_shape)
        self.k_cache = sentinel_like(shape, device)
        self.v_cache = sentinel_like(shape, device) if m.kind == "gqa" else None
        self.d_bt = torch.from_numpy(self.tables).to(device)
        _, h_idx = pic.pic_recompute_indices(self.plans)
        self.n_rec = len(h_idx)
        self.ridx = torch.full((max(1, self.n_rec),), -7, dtype=torch.int32, device=device)
        self.indptr = torch.full((len(self.plans) + 1,), -7, dtype=torch.int32, device=device)
        self.ws = torch.empty(pic.pic_workspace_bytes(self.ctx, self.plans), dtype=torch.uint8, device=device)

    def run(self):
        pic.pic_stitch(self.ctx, self.plans, self.k_pool, self.v_pool, self.k_cache, self.v_cache,
                       self.d_bt, self.ridx, self.indptr, self.ws)
        assert pic.pic_query_device_status(self.ctx, self.ws) == 0
        return self

    def close(self):
        pic.pic_destroy(self.ctx)


def oracle_side(wl: W.Workload, num_blocks: int):
    """The oracle's own plan: segments, block tables, recompute lists."""
    chunks = [oracle.Chunk(off, n, 0) for off, n in zip(wl.pool_offsets, wl.chunk_lens)]
    pool = oracle.BlockPool(num_blocks)
    segs, tables, rec = [], [], []
    for req in wl.requests:
        s = oracle.compose(chunks, [c for c, _ in req], take=[t for _, t in req])
        total = s[-1].dst_pos + s[-1].length if s else 0
        tables.append(pool.allocate(oracle.blocks_needed(total, wl.model.block_size)))
        segs.append(s)
        rec.append(oracle.recompute_positions(s, wl.k_nonleading, wl.k_leading))
    return segs, tables, rec


def theta_of(m):
    return oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)


def pairing_of(m):
    return oracle.NEOX_HALF if m.pairing == "neox" else oracle.INTERLEAVED


def random_attend_layout(rng, bs, max_chunk=300, max_req_tokens=2500):
    """A seeded random decode context, as plain numbers: 2-10 pool chunks of
    1..max_chunk tokens, maybe one block-resident chunk (1-79 tokens, cached
    at a random base position), and 1-4 requests of 1-8 chunk occurrences
    (repeats, some truncated, some to nothing), inline tokens before, between
    and after them, and a pseudo-sink width k of 0-6.  `nb` is the cache
    blocks the requests and the block-resident chunk need, plus two."""
    lens = [int(x) for x in rng.integers(1, max_chunk + 1, size=int(rng.integers(2, 11)))]
    offs = [0]
    for n in lens[:-1]:
        offs.append(offs[-1] + n)
    block_chunk = (int(rng.integers(1, 80)), int(rng.integers(0, 5000))) if rng.random() < 0.5 else None
    kinds = len(lens) + (1 if block_chunk else 0)
    reqs = []
    for _ in range(int(rng.integers(1, 5))):
        start = int(rng.integers(0, 21)) if rng.random() < 0.5 else 0
        chunks, takes, pos, p = [], [], [], start
        for _ in range(int(rng.integers(1, 9))):
            c = int(rng.integers(kinds))
            full = lens[c] if c < len(lens) else block_chunk[0]
            take = full if rng.random() < 0.8 else int(rng.integers(0, full + 1))
            gap = int(rng.integers(1, 31)) if rng.random() < 0.3 else 0
            if p + gap + take > max_req_tokens:
                break
            p += gap
            chunks.append(c)
            takes.append(take)
            pos.append(p)
            p += take
        tail = int(rng.integers(0, 41)) if rng.random() < 0.5 else 0
        reqs.append(dict(chunks=chunks, takes=takes, pos=pos, start=start, total=max(1, p + tail)))
    nb = sum(-(-r["total"] // bs) for r in reqs) + (-(-block_chunk[0] // bs) if block_chunk else 0) + 2
    return dict(lens=lens, offs=offs, P=sum(lens), block_chunk=block_chunk, reqs=reqs, nb=nb,
                k=int(rng.integers(0, 7)))


def register_attend_layout(ctx, layout, tag, bs):
    """Registers the layout's chunks with ctx (the block-resident one in the
    cache's last blocks) and builds its requests.  Returns (plans, block
    tables, sources), sources mapping a chunk id to ("pool", first token) or
    ("blocks", block ids)."""
    ids, sources = [], {}
    for c, (o, n) in enumerate(zip(layout["offs"], layout["lens"])):
        cid = pic.pic_register_chunk(ctx, W.chunk_key(tag, c), o, n)[0]
        ids.append(cid)
        sources[cid] = ("pool", o)
    if layout["block_chunk"]:
        n_b, base = layout["block_chunk"]
        nblk = -(-n_b // bs)
        blocks = list(range(layout["nb"] - nblk, layout["nb"]))
        cid = pic.pic_register_chunk_blocks(ctx, W.chunk_key(tag, 99), blocks, n_b, base)[0]
        ids.append(cid)
        sources[cid] = ("blocks", blocks)
    plans, tables = [], []
    for r in layout["reqs"]:
        plan, bt = pic.pic_build_block_table(ctx, [ids[c] for c in r["chunks"]], -(-r["total"] // bs),
                                             take_tokens=r["takes"], dst_pos=r["pos"], start_pos=r["start"],
                                             total_tokens=r["total"], k_nonleading=layout["k"])
        plans.append(plan)
        tables.append(bt)
    return plans, tables, sources
