"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The bulk-copy pipeline and the tcgen05 MLA attention wait on mbarriers for
their own copies and products, and every wait is bounded.
pic_debug_stall_next_launch makes one tile of the first CTA never arrive, so
the waits for it run out: the launch must raise PIC_DEV_TIMEOUT in the
workspace status word, return, and leave the context usable -- the next
launch must give the clean result bit for bit."""

import time

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import Stitched, bits, sentinel_like
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu


def _stitch(st, cache):
    pic.pic_stitch(st.ctx, st.plans, st.k_pool, st.v_pool, cache, None, st.d_bt, st.ridx, st.indptr, st.ws)
    t0 = time.perf_counter()
    status = pic.pic_query_device_status(st.ctx, st.ws, raise_on_device_error=False)
    return status, time.perf_counter() - t0


def test_bulk_pipeline_wait_runs_out_and_context_recovers():
    wl = W.deepseek_v3_mla(context_tokens=4096, num_layers=4)
    st = Stitched(wl)
    try:
        assert pic.pic_kernel_variant(st.ctx, 0) == pic.PIC_VARIANT_BULK_PIPELINE
        clean = sentinel_like(st.k_cache.shape, "cuda")
        status, _ = _stitch(st, clean)
        assert status == 0
        want = bits(clean)

        for spins in (1_000, 10_000):
            stalled = sentinel_like(st.k_cache.shape, "cuda")
            pic.pic_debug_stall_next_launch(st.ctx, 2, spins)
            status, waited = _stitch(st, stalled)
            assert status & pic.PIC_DEV_TIMEOUT, status
            assert waited < 30.0
            got = bits(stalled)
            # the other CTAs finished their tiles; the stalled CTA stopped early
            assert 0 < np.count_nonzero(got == want) < got.size
            print(f"stalled launch with {spins} tries per wait: {waited * 1e3:.1f} ms")

        again = sentinel_like(st.k_cache.shape, "cuda")
        status, _ = _stitch(st, again)   # the hook applied to one launch only
        assert status == 0
        np.testing.assert_array_equal(bits(again), want)
        torch.cuda.synchronize()
    finally:
        st.close()


def test_stall_hook_is_consumed_by_the_next_stitch_and_clearable():
    wl = W.deepseek_v3_mla(context_tokens=2048, num_layers=2)
    st = Stitched(wl)
    try:
        pic.pic_debug_stall_next_launch(st.ctx, 1, 1000)
        pic.pic_debug_stall_next_launch(st.ctx, -1)     # cleared before any launch
        status, _ = _stitch(st, sentinel_like(st.k_cache.shape, "cuda"))
        assert status == 0
    finally:
        st.close()


def test_tcgen05_attention_wait_runs_out_and_context_recovers():
    """The tcgen05 MLA attention has many roles per CTA (producers, query
    warp, score and value issuers, softmax warps).  A tile whose rows are
    never requested must end all of them through bounded waits and the CTA's
    abort flag, free the CTA's TMEM, and leave the next launch (on the same
    SMs, which must allocate TMEM again) exact."""
    wl = W.deepseek_v3_mla(context_tokens=4096, num_layers=2)
    st = Stitched(wl)
    try:
        assert pic.pic_kernel_variant(st.ctx, 2) == pic.PIC_VARIANT_TENSOR_CORE_TMEM
        H, L, row = 16, wl.model.num_layers, wl.model.head_dim
        g = torch.Generator(device="cuda")
        g.manual_seed(12)
        q = torch.empty((L, 1, H, row), dtype=torch.bfloat16, device="cuda").normal_(0.0, 1.0, generator=g)
        ws = torch.empty(pic.pic_attend_workspace_bytes(st.ctx, st.plans, H, L), dtype=torch.uint8, device="cuda")

        def attend():
            out = torch.empty((L, 1, H, 512), dtype=torch.float32, device="cuda")
            lse = torch.empty((L, 1, H), dtype=torch.float32, device="cuda")
            pic.pic_attend_decode(st.ctx, st.plans, pic.PIC_ATTEND_FUSED, q, 0.07, st.k_pool, None, st.k_cache,
                                  None, out, lse, ws)
            t0 = time.perf_counter()
            status = pic.pic_query_device_status(st.ctx, ws, raise_on_device_error=False)
            return status, time.perf_counter() - t0, bits(out), bits(lse)

        status, _, want_o, want_l = attend()
        assert status == 0
        for spins in (1_000, 10_000):
            pic.pic_debug_stall_next_launch(st.ctx, 0, spins)  # CTA 0 holds one or two tiles here
            status, waited, _, _ = attend()
            assert status & pic.PIC_DEV_TIMEOUT, status
            assert waited < 30.0
            print(f"stalled attention with {spins} tries per wait: {waited * 1e3:.1f} ms")
        status, _, got_o, got_l = attend()  # the hook applied to one launch only
        assert status == 0
        np.testing.assert_array_equal(got_o, want_o)
        np.testing.assert_array_equal(got_l, want_l)
        torch.cuda.synchronize()
    finally:
        st.close()
