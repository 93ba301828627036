"""CPU tests of the chunking entry points' host side (Irminsul 2.2, "Content-Hash
Keying with CDC"; "Hybrid Strategies (S1/S2)"): the S1 windows against the
oracle, workspace sizes, and argument checks that fail before anything is
enqueued (the pointers below are fake and never reach a kernel)."""

import ctypes

import pytest

import oracle
from harness import lib
from position_independent_kv_stitch_gb300 import pic


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


@pytest.mark.parametrize("b,e,w", [(0, 0, 128), (0, 1, 128), (5, 133, 128), (0, 256, 128), (10, 1000, 128),
                                   (7, 8, 1), (3, 50, 7), (100, 100 + 128 * 9, 128)])
def test_s1_windows_match_oracle(b, e, w):
    starts, ends = pic.pic_s1_windows(b, e, w)
    assert list(zip(starts, ends)) == oracle.s1_windows(b, e, w)


def test_s1_windows_rejects_bad_arguments():
    L = pic.load()
    n = ctypes.c_int64()
    assert pic.STATUS_NAMES[L.pic_s1_windows(5, 4, 128, None, None, 0, ctypes.byref(n))] == "PIC_ERR_INVALID_ARG"
    assert pic.STATUS_NAMES[L.pic_s1_windows(0, 4, 0, None, None, 0, ctypes.byref(n))] == "PIC_ERR_INVALID_ARG"
    a = (ctypes.c_int64 * 1)()
    st = L.pic_s1_windows(0, 300, 128, a, a, 1, ctypes.byref(n))
    assert pic.STATUS_NAMES[st] == "PIC_ERR_CAPACITY" and n.value == 3


def test_workspace_covers_one_cut_bit_per_token():
    assert pic.pic_cdc_workspace_bytes(0) >= 256
    prev = 0
    for n in (1, 8191, 8192, 8193, 1 << 20, 37_000_000):
        ws = pic.pic_cdc_workspace_bytes(n)
        assert ws % 256 == 0 and ws >= 256 + n // 8 and ws >= prev
        prev = ws


def test_chunk_argument_checks_need_no_gpu():
    L = pic.load()
    good = ctypes.c_void_p(0x10000)
    odd4 = ctypes.c_void_p(0x10004)
    ws = pic.pic_cdc_workspace_bytes(1000)

    def call(tokens=good, n_tokens=1000, offsets=good, n_docs=2, gear=good, vocab=100, min_len=0, max_len=0,
             indptr=good, ends=good, fps=good, cap=10, workspace=good, ws_bytes=ws):
        st = L.pic_cdc_chunk(tokens, n_tokens, offsets, n_docs, gear, vocab, 1 << 58, min_len, max_len, 0,
                             indptr, ends, fps, cap, workspace, ws_bytes, None)
        return pic.STATUS_NAMES[st]

    assert call(offsets=None) == "PIC_ERR_INVALID_ARG"
    assert call(indptr=None) == "PIC_ERR_INVALID_ARG"
    assert call(workspace=None) == "PIC_ERR_INVALID_ARG"
    assert call(gear=None) == "PIC_ERR_INVALID_ARG"
    assert call(vocab=0) == "PIC_ERR_INVALID_ARG"
    assert call(n_tokens=-1) == "PIC_ERR_INVALID_ARG"
    assert call(n_docs=-1) == "PIC_ERR_INVALID_ARG"
    assert call(min_len=-1) == "PIC_ERR_INVALID_ARG"
    assert call(max_len=-2) == "PIC_ERR_INVALID_ARG"
    assert call(cap=-1) == "PIC_ERR_INVALID_ARG"
    assert call(ends=None) == "PIC_ERR_INVALID_ARG"
    assert call(tokens=odd4) == "PIC_ERR_ALIGNMENT"
    assert call(offsets=odd4) == "PIC_ERR_ALIGNMENT"
    assert call(ends=odd4) == "PIC_ERR_ALIGNMENT"
    assert call(ws_bytes=ws - 1) == "PIC_ERR_CAPACITY"
    assert "workspace" in pic.load().pic_last_error(None).decode()


def test_fingerprint_argument_checks_need_no_gpu():
    L = pic.load()
    good = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)

    def call(tokens=good, n_tokens=100, starts=good, ends=good, n=3, out=good, status=good):
        return pic.STATUS_NAMES[L.pic_fingerprint_spans(tokens, n_tokens, starts, ends, n, 0, out, status, None)]

    assert call(starts=None) == "PIC_ERR_INVALID_ARG"
    assert call(out=None) == "PIC_ERR_INVALID_ARG"
    assert call(status=None) == "PIC_ERR_INVALID_ARG"
    assert call(n=-1) == "PIC_ERR_INVALID_ARG"
    assert call(tokens=None) == "PIC_ERR_INVALID_ARG"
    assert call(starts=odd) == "PIC_ERR_ALIGNMENT"
    assert call(out=odd) == "PIC_ERR_ALIGNMENT"
