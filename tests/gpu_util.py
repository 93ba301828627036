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
