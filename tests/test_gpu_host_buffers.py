"""Pools and caches in pinned host memory: the kernels stream them over the
host link directly.  Results must equal the device-memory path bit for bit
and match the oracle; pageable host memory is refused before any launch."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import Stitched, assert_k_close, bits, f64, oracle_side, pairing_of, theta_of
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pic.load(build_if_missing=True)


def _pinned_like(t):
    return torch.empty(t.shape, dtype=t.dtype).pin_memory()


@pytest.mark.parametrize("name", ["tiny_gqa", "mla_small"])
def test_host_pool_and_cache_match_device_path_and_oracle(name):
    if name == "tiny_gqa":
        wl = W.tiny_gqa()
    else:
        base = W.deepseek_v3_mla(context_tokens=1500, num_layers=2)
        wl = W.Workload("mla-host", base.model, base.chunk_lens, base.requests, 0, 32)
    dev = Stitched(wl, pool_device="cpu").run()
    try:
        hk = dev.k_pool.cpu().pin_memory()
        hv = dev.v_pool.cpu().pin_memory() if dev.v_pool is not None else None
        hkc = _pinned_like(dev.k_cache)
        hkc.view(torch.int16).fill_(-1)
        hvc = None
        if dev.v_cache is not None:
            hvc = _pinned_like(dev.v_cache)
            hvc.view(torch.int16).fill_(-1)
        ws = torch.empty_like(dev.ws)
        ridx = torch.empty_like(dev.ridx)
        indptr = torch.empty_like(dev.indptr)
        pic.pic_stitch(dev.ctx, dev.plans, hk, hv, hkc, hvc, dev.d_bt, ridx, indptr, ws)
        assert pic.pic_query_device_status(dev.ctx, ws) == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(hkc), bits(dev.k_cache))
        if hvc is not None:
            assert np.array_equal(bits(hvc), bits(dev.v_cache))
        assert torch.equal(ridx, dev.ridx) and torch.equal(indptr, dev.indptr)
        segs, tables, _ = oracle_side(wl, dev.nb)
        m = wl.model
        want_k, _ = oracle.stitch_paged(bits(hk), None, segs, tables, dev.nb, dev.bs, theta_of(m),
                                        pairing_of(m), m.rope_offset, m.rope_dim)
        assert_k_close(f64(hkc), want_k, "host K")
    finally:
        dev.close()


def test_host_cache_in_place_shift():
    m = W.Model("ip-host", "gqa", 2, 2, 128, 128, 0, "neox", 1e4, 16)
    ctx = pic.create_from_spec(pic.model_spec_from(m), 8)
    try:
        cache = torch.empty((2, 8, 16, 2, 128), dtype=torch.bfloat16)
        W.fill_random_bf16(cache, 9, "host-inplace")
        host = cache.pin_memory()
        devc = cache.to(DEV)
        tables = [[3, 1, 6, 0]]
        bt = torch.tensor(tables, dtype=torch.int32, device=DEV)
        segs = [(0, 2, 30, 4097), (0, 40, 9, -3)]
        ws = torch.empty(pic.pic_rerotate_workspace_bytes(ctx, segs), dtype=torch.uint8, device=DEV)
        pic.pic_rerotate_inplace(ctx, host, bt, segs, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        pic.pic_rerotate_inplace(ctx, devc, bt, segs, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        assert np.array_equal(bits(host), bits(devc))
        want = oracle.rerotate_inplace(bits(cache), tables, segs, 16, oracle.rope_inv_freq(128, 1e4),
                                       oracle.NEOX_HALF, 0, 128)
        assert_k_close(f64(host), want, "host in place")
    finally:
        pic.pic_destroy(ctx)


def test_pageable_host_memory_is_refused_before_launch():
    m = W.Model("pageable", "gqa", 1, 1, 64, 64, 0, "neox", 1e4, 16)
    ctx = pic.create_from_spec(pic.model_spec_from(m), 2)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("p", 0), 0, 10)
        plan, bt = pic.pic_build_block_table(ctx, [0], 1)
        pageable = np.zeros((1, 16, 1, 64), dtype=np.uint16)   # plain numpy memory, not pinned
        dcache = torch.empty((1, 2, 16, 1, 64), dtype=torch.bfloat16, device=DEV)
        d_bt = torch.from_numpy(bt).to(DEV).view(1, -1)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, [plan]), dtype=torch.uint8, device=DEV)
        arr = pic._plan_array([plan])
        p = ctypes.c_void_p(pageable.ctypes.data)
        L = pic.load()
        st = L.pic_stitch(ctx, arr, 1, p, p, 16 * 64 * 2, ctypes.c_void_p(dcache.data_ptr()),
                          ctypes.c_void_p(dcache.data_ptr()), dcache.stride(0) * 2, ctypes.c_void_p(d_bt.data_ptr()),
                          1, None, None, 0, ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
        assert "pageable" in pic.pic_last_error(ctx)
    finally:
        pic.pic_destroy(ctx)
