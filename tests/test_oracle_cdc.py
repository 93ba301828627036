"""Pins of the oracle's content-defined chunking (Irminsul 2.2, "Content-Hash
Keying with CDC"; "Hybrid Strategies (S1/S2)"): the Gear hash's 64-token
window, the threshold cut rule, boundaries that follow content, xxHash64
against the system library, and the S1 windows."""

import ctypes
import ctypes.util
import random

import numpy as np
import pytest

import oracle
import workloads as W

MASK64 = (1 << 64) - 1


def _gear(vocab=1000, seed=1):
    return W.gear_table(seed, vocab)


def test_rolling_hash_equals_the_64_token_window_sum():
    gear = _gear()
    toks = W.random_tokens(2, "pin/gear", 700, 1000)
    rolling = oracle.gear_hashes(toks, gear)
    window = oracle.gear_hashes_window(toks, gear)
    assert [int(x) for x in window] == rolling


def test_hash_forgets_tokens_older_than_64_positions():
    """h_i depends on t_{i-63..i} only: a change 64 back leaves h_i alone;
    a change 63 back moves h_i by (delta gear) * 2^63, i.e. flips only the top
    bit and only when the two gear values differ in parity."""
    gear = _gear()
    toks = list(W.random_tokens(3, "pin/win", 200, 1000))
    base = oracle.gear_hashes(toks, gear)
    i = 150
    t64 = toks.copy()
    t64[i - 64] = (t64[i - 64] + 1) % 1000
    assert oracle.gear_hashes(t64, gear)[i] == base[i]
    t63 = toks.copy()
    old, new = t63[i - 63], (t63[i - 63] + 7) % 1000
    t63[i - 63] = new
    want = (base[i] + ((int(gear[new]) - int(gear[old])) << 63)) & MASK64
    assert oracle.gear_hashes(t63, gear)[i] == want
    assert (want ^ base[i]) in (0, 1 << 63)


def test_constant_stream_closed_form():
    """t_i = c for all i: h_i = g (2^(i+1) - 1) mod 2^64, so -g from i = 63 on."""
    gear = _gear()
    g = int(gear[5])
    h = oracle.gear_hashes([5] * 100, gear)
    for i, x in enumerate(h):
        assert x == (g * ((1 << (i + 1)) - 1)) & MASK64
    assert h[63] == h[99] == (-g) & MASK64


def test_cuts_exactly_where_the_hash_is_below_threshold():
    gear = _gear()
    toks = W.random_tokens(4, "pin/cut", 5000, 1000)
    h = oracle.gear_hashes(toks, gear)
    thr = oracle.threshold_for_mean(64)
    ends = oracle.cdc_chunk_ends(h, thr)
    want = [i + 1 for i, x in enumerate(h) if x < thr]
    if not want or want[-1] != len(toks):
        want.append(len(toks))
    assert ends == want
    # about one cut per 64 tokens
    assert 40 < len(toks) / len(ends) < 100


def test_boundaries_follow_content_under_a_shifting_prefix():
    """Prefixing a document moves its cut points by the prefix length once the
    64-token window lies inside the original document (content-aligned
    boundaries, the point of CDC)."""
    gear = _gear()
    doc = list(W.random_tokens(5, "pin/doc", 4000, 1000))
    pre = list(W.random_tokens(6, "pin/pre", 37, 1000))
    thr = oracle.threshold_for_mean(128)
    a = oracle.cdc_chunk_ends(oracle.gear_hashes(doc, gear), thr)
    b = oracle.cdc_chunk_ends(oracle.gear_hashes(pre + doc, gear), thr)
    a_tail = [e for e in a if e - 1 >= 63]
    b_tail = [e - len(pre) for e in b if e - 1 - len(pre) >= 63]
    assert a_tail == b_tail and len(a_tail) > 10
    # and the chunks between those cuts have equal fingerprints
    fa = {oracle.fingerprint(doc[s:e]) for s, e in zip(a_tail, a_tail[1:])}
    fb = {oracle.fingerprint((pre + doc)[s + len(pre):e + len(pre)]) for s, e in zip(b_tail, b_tail[1:])}
    assert fa == fb


@pytest.mark.parametrize("min_len,max_len", [(16, 0), (0, 100), (32, 256), (64, 64)])
def test_min_and_max_length_rules(min_len, max_len):
    gear = _gear()
    toks = W.random_tokens(7, "pin/minmax", 6000, 1000)
    h = oracle.gear_hashes(toks, gear)
    thr = oracle.threshold_for_mean(48)
    ends = oracle.cdc_chunk_ends(h, thr, min_len, max_len)
    starts = [0] + ends[:-1]
    lens = [e - s for s, e in zip(starts, ends)]
    assert ends[-1] == len(toks) and all(x > 0 for x in lens)
    if max_len:
        assert max(lens) <= max_len
    if min_len:
        assert min(lens[:-1]) >= min_len
    for s, e in zip(starts[:-1], ends[:-1]):
        cut_by_hash = h[e - 1] < thr and e - s >= max(min_len, 1)
        assert cut_by_hash or (max_len and e - s == max_len)
        # no earlier position in the chunk could have ended it
        for i in range(s, e - 1):
            assert not (h[i] < thr and i - s + 1 >= max(min_len, 1))


def _libxxhash():
    name = ctypes.util.find_library("xxhash")
    if not name:
        return None
    lib = ctypes.CDLL(name)
    lib.XXH64.restype = ctypes.c_uint64
    lib.XXH64.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64]
    return lib


def test_xxh64_matches_the_system_library():
    lib = _libxxhash()
    if lib is None:
        pytest.skip("libxxhash not installed")
    rng = random.Random(11)
    for n in list(range(0, 80)) + [127, 128, 129, 255, 256, 1000, 4096, 4100]:
        data = bytes(rng.getrandbits(8) for _ in range(n))
        for seed in (0, 1, 0x9E3779B97F4A7C15, MASK64):
            buf = ctypes.create_string_buffer(data, max(n, 1))
            assert oracle.xxh64(data, seed) == lib.XXH64(buf, n, seed), (n, seed)


def test_xxh64_of_empty_input():
    """The well-known digest of the empty input at seed 0."""
    assert oracle.xxh64(b"", 0) == 0xEF46DB3751D8E999


def test_fingerprint_is_xxh64_of_little_endian_int32():
    toks = [1, 2, 0x01020304, -1]
    raw = b"".join(int(t & 0xFFFFFFFF).to_bytes(4, "little") for t in toks)
    assert oracle.fingerprint(toks) == oracle.xxh64(raw)
    key = oracle.registry_key(oracle.fingerprint(toks))
    assert len(key) == 32 and key[8:] == bytes(24)


@pytest.mark.parametrize("b,e", [(0, 0), (0, 1), (5, 133), (0, 256), (10, 1000)])
def test_s1_windows(b, e):
    w = oracle.s1_windows(b, e)
    covered = [p for lo, hi in w for p in range(lo, hi)]
    assert covered == list(range(b, e))
    assert all(hi - lo == 128 for lo, hi in w[:-1])
    assert all(lo == b + 128 * k for k, (lo, _) in enumerate(w))


def test_chunk_document_extreme_thresholds():
    """Threshold 0 never cuts: one chunk, the document's own XXH64 (checked
    against the system library when it is installed).  Threshold 2^64 - 1
    cuts after every token whose hash is below it (all but a 2^-64 chance):
    one-token chunks.  An empty document has no chunks."""
    gear = _gear()
    doc = [int(t) for t in W.random_tokens(7, "pin/doc-ext", 300, 1000)]
    ends, fps = oracle.chunk_document(doc, gear, 0)
    assert ends == [len(doc)] and fps == [oracle.fingerprint(doc)]
    lib = _libxxhash()
    if lib is not None:
        raw = np.asarray(doc, dtype="<i4").tobytes()
        assert fps[0] == lib.XXH64(raw, len(raw), 0)
    ends, fps = oracle.chunk_document(doc, gear, MASK64, seed=9)
    assert ends == list(range(1, len(doc) + 1))
    assert fps == [oracle.fingerprint([t], 9) for t in doc]
    assert oracle.chunk_document([], gear, 1 << 60) == ([], [])


def test_chunk_document_tiles_the_document():
    gear = _gear()
    doc = [int(t) for t in W.random_tokens(8, "pin/doc-tile", 3000, 1000)]
    for lo, hi in ((0, 0), (16, 128), (50, 50)):
        ends, fps = oracle.chunk_document(doc, gear, oracle.threshold_for_mean(64), lo, hi)
        starts = [0] + ends[:-1]
        assert ends[-1] == len(doc) and all(b > a for a, b in zip(starts, ends))
        assert sum((doc[s:e] for s, e in zip(starts, ends)), []) == doc
        assert len(fps) == len(ends)
