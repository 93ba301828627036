"""Content-defined chunking and chunk fingerprints, restated plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Irminsul: MLA-Native Position-Independent Caching for Agentic LLM Serving,
2.2 "Content-Hash Keying with CDC": chunk boundaries come from a rolling
Gear hash over 64-token windows, a chunk ends where the hash falls below a
threshold, and every chunk is fingerprinted with xxHash64; "Hybrid Strategies
(S1/S2)", S1: a chunk that misses the registry is subdivided into fixed
128-token windows.

Readings taken where the page is silent:
* Gear over tokens: h_i = 2 h_{i-1} + gear[t_i] (mod 2^64), h = 0 before a
  document starts, gear a table of random 64-bit values indexed by token id
  (byte Gear generalised to the token alphabet).  A 64-bit h forgets inputs
  older than 64 steps, which is the 64-token window.
* A chunk ends after token i when h_i < threshold; optional min_len (a cut
  needs at least min_len tokens in the chunk) and max_len (a chunk of
  max_len tokens is cut regardless); the tail of a document is a chunk.
* A fingerprint is XXH64 (seed 0 unless given) of the chunk's token ids as
  little-endian int32 bytes; a registry key is that 64-bit value
  little-endian, zero-padded to 32 bytes.
* S1 windows of a missed chunk [b, e): [b + 128k, min(b + 128(k + 1), e)).

xxHash64 follows its published specification (Y. Collet, "xxHash fast
digest algorithm", XXH64): four lanes over 32-byte stripes, a lane merge,
the length, 8-, 4- and 1-byte tails, and the final avalanche.
"""

from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GEAR_WINDOW = 64
S1_WINDOW = 128


# ---------------------------------------------------------------------------
# Gear hash
# ---------------------------------------------------------------------------

def gear_hashes(tokens, gear) -> list:
    """The rolling Gear hash at every position of one document (Python ints)."""
    h = 0
    out = []
    for t in tokens:
        h = ((h << 1) + int(gear[int(t)])) & MASK64
        out.append(h)
    return out


def gear_hashes_window(tokens, gear) -> np.ndarray:
    """The same hashes as the explicit window sum
    h_i = sum_{k=0}^{63} gear[t_{i-k}] * 2^k (mod 2^64), vectorised (uint64)."""
    g = np.asarray(gear, dtype=np.uint64)[np.asarray(tokens, dtype=np.int64)]
    n = len(g)
    h = np.zeros(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for k in range(min(GEAR_WINDOW, n)):
            h[k:] += g[:n - k] << np.uint64(k)
    return h


def cdc_chunk_ends(hashes, threshold: int, min_len: int = 0, max_len: int = 0) -> list:
    """End positions (exclusive) of the chunks of one document."""
    ends = []
    start = 0
    n = len(hashes)
    for i in range(n):
        length = i - start + 1
        cut = False
        if max_len and length >= max_len:
            cut = True
        elif int(hashes[i]) < threshold and length >= max(min_len, 1):
            cut = True
        if cut:
            ends.append(i + 1)
            start = i + 1
    if start < n:
        ends.append(n)
    return ends


def threshold_for_mean(mean_len: int) -> int:
    """The threshold at which a uniform 64-bit hash cuts once per mean_len tokens."""
    return (1 << 64) // mean_len


# ---------------------------------------------------------------------------
# xxHash64
# ---------------------------------------------------------------------------

_P1 = 0x9E3779B185EBCA87
_P2 = 0xC2B2AE3D27D4EB4F
_P3 = 0x165667B19E3779F9
_P4 = 0x85EBCA77C2B2AE63
_P5 = 0x27D4EB2F165667C5


def _rotl(x: int, r: int) -> int:
    return ((x << r) | (x >> (64 - r))) & MASK64


def _round(acc: int, lane: int) -> int:
    acc = (acc + lane * _P2) & MASK64
    acc = _rotl(acc, 31)
    return (acc * _P1) & MASK64


def _merge(acc: int, lane: int) -> int:
    acc ^= _round(0, lane)
    return (acc * _P1 + _P4) & MASK64


def xxh64(data: bytes, seed: int = 0) -> int:
    n = len(data)
    pos = 0
    if n >= 32:
        v1 = (seed + _P1 + _P2) & MASK64
        v2 = (seed + _P2) & MASK64
        v3 = seed & MASK64
        v4 = (seed - _P1) & MASK64
        while pos + 32 <= n:
            v1 = _round(v1, int.from_bytes(data[pos:pos + 8], "little"))
            v2 = _round(v2, int.from_bytes(data[pos + 8:pos + 16], "little"))
            v3 = _round(v3, int.from_bytes(data[pos + 16:pos + 24], "little"))
            v4 = _round(v4, int.from_bytes(data[pos + 24:pos + 32], "little"))
            pos += 32
        acc = (_rotl(v1, 1) + _rotl(v2, 7) + _rotl(v3, 12) + _rotl(v4, 18)) & MASK64
        for v in (v1, v2, v3, v4):
            acc = _merge(acc, v)
    else:
        acc = (seed + _P5) & MASK64
    acc = (acc + n) & MASK64
    while pos + 8 <= n:
        acc ^= _round(0, int.from_bytes(data[pos:pos + 8], "little"))
        acc = (_rotl(acc, 27) * _P1 + _P4) & MASK64
        pos += 8
    if pos + 4 <= n:
        acc ^= (int.from_bytes(data[pos:pos + 4], "little") * _P1) & MASK64
        acc = (_rotl(acc, 23) * _P2 + _P3) & MASK64
        pos += 4
    while pos < n:
        acc ^= (data[pos] * _P5) & MASK64
        acc = (_rotl(acc, 11) * _P1) & MASK64
        pos += 1
    acc ^= acc >> 33
    acc = (acc * _P2) & MASK64
    acc ^= acc >> 29
    acc = (acc * _P3) & MASK64
    acc ^= acc >> 32
    return acc


def fingerprint(tokens, seed: int = 0) -> int:
    """XXH64 of token ids as little-endian int32 bytes."""
    return xxh64(np.asarray(tokens, dtype="<i4").tobytes(), seed)


def registry_key(fp: int) -> bytes:
    """A 32-byte registry key: the fingerprint little-endian, zero-padded."""
    return fp.to_bytes(8, "little") + bytes(24)


def s1_windows(begin: int, end: int, window: int = S1_WINDOW) -> list:
    """Fixed windows [b + w k, min(b + w (k + 1), e)) covering [begin, end)."""
    return [(b, min(b + window, end)) for b in range(begin, end, window)]


def chunk_document(tokens, gear, threshold: int, min_len: int = 0, max_len: int = 0, seed: int = 0):
    """(end positions, fingerprints) of one document's CDC chunks."""
    ends = cdc_chunk_ends(gear_hashes(tokens, gear), threshold, min_len, max_len)
    fps = []
    start = 0
    for e in ends:
        fps.append(fingerprint(tokens[start:e], seed))
        start = e
    return ends, fps
