"""Plain float64 restatement of position-independent KV stitching.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every function is the
definition written out, slow and obvious; no blocking, no fusion, no reuse of
anything in the CUDA library.

Notation follows the pages: ``theta_i`` the RoPE frequencies, ``R_m`` the
block-diagonal rotation at position m, ``delta`` (EPIC: dp) the position
shift of a cached chunk, ``base_pos`` the position a chunk was computed at.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

NEOX_HALF = 0      # pair (i, i + d/2)
INTERLEAVED = 1    # pair (2i, 2i + 1)
BF16_SENTINEL = 0xFFFF  # a NaN bit pattern the tests pre-fill destinations with


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16 / int16) -> exact float64 values.

    A bfloat16 is the upper half of an IEEE binary32, so widening the bits by
    16 zero bits gives the binary32 with the same value, which float64 holds
    exactly.
    """
    u = np.asarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# RoPE frequencies
# ---------------------------------------------------------------------------

def rope_inv_freq(rope_dim: int, base: float) -> np.ndarray:
    """theta_i = b^(-2i/d) for i = 0 .. d/2 - 1.

    EPIC Guide: Position-Independent Caching for LLM Serving, "Mathematical
    Foundations: RoPE In-Place Key Transformation", 1. RoPE Mathematical
    Structure (definition of theta_i under the R_m^(i) matrix).  For an MLA
    row, d is the width of the decoupled rope key (64), not of the row.
    """
    if rope_dim <= 0 or rope_dim % 2:
        raise ValueError("rope_dim must be a positive even number")
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * i / rope_dim)


def llama3_inv_freq(theta: np.ndarray, factor: float, low_freq_factor: float,
                    high_freq_factor: float, orig_max_pos: int) -> np.ndarray:
    """Llama-3.1 long-context rescaling of the RoPE frequencies.

    This rule is not on the pages; it is the public Llama-3.1 rule, stated
    as math, and pinned by values derived from it by hand (wavelengths placed
    so that the blend weight below is exactly 1/4, 1/2 or 3/4, the regime
    edges, factor 1, and Llama-3.1-8B's own table), not by a second
    transcription.  With wavelength lambda_i = 2 pi / theta_i:
    lambda_i < orig/high keeps theta_i; lambda_i > orig/low uses
    theta_i/factor; in between the two are blended linearly in
    s = (orig/lambda_i - low) / (high - low):
    theta_i' = (1 - s) theta_i / factor + s theta_i.
    """
    theta = np.asarray(theta, dtype=np.float64)
    out = np.empty_like(theta)
    low_wavelen = orig_max_pos / low_freq_factor
    high_wavelen = orig_max_pos / high_freq_factor
    for i, t in enumerate(theta):
        wavelen = 2.0 * math.pi / t
        if wavelen < high_wavelen:
            out[i] = t
        elif wavelen > low_wavelen:
            out[i] = t / factor
        else:
            s = (orig_max_pos / wavelen - low_freq_factor) / (high_freq_factor - low_freq_factor)
            out[i] = (1.0 - s) * t / factor + s * t
    return out


def model_inv_freq(rope_dim: int, base: float, scaling: dict | None = None) -> np.ndarray:
    """The frequency table of a model: plain theta_i, optionally llama3-scaled."""
    theta = rope_inv_freq(rope_dim, base)
    if scaling:
        theta = llama3_inv_freq(theta, scaling["factor"], scaling["low_freq_factor"],
                                scaling["high_freq_factor"], scaling["orig_max_pos"])
    return theta


# ---------------------------------------------------------------------------
# the rotation
# ---------------------------------------------------------------------------

def rope_pairs(rope_dim: int, pairing: int):
    """Index arrays (a, b): pair i rotates coordinates (a[i], b[i]) by angle m*theta_i.

    INTERLEAVED is the layout the EPIC guide prints ("for each 2D coordinate
    (2i, 2i+1)", and the listing's even/odd slices).  NEOX_HALF pairs
    coordinate i with i + d/2, the half-split layout of GPT-NeoX / Llama
    checkpoints; the pages do not print it.
    """
    half = rope_dim // 2
    i = np.arange(half)
    if pairing == INTERLEAVED:
        return 2 * i, 2 * i + 1
    if pairing == NEOX_HALF:
        return i, i + half
    raise ValueError(f"unknown pairing {pairing}")


def rotate(x, delta: int, theta: np.ndarray, pairing: int) -> np.ndarray:
    """R_delta x over the last axis, in float64.

    EPIC Guide, "Mathematical Foundations", 1. RoPE Mathematical Structure:
    each plane i is rotated by [[cos, -sin], [sin, cos]] of angle m*theta_i;
    2. The In-Place Shift Transformation: k_target = R_dp k_cached, with one
    dp for the whole chunk (R_{n+dp} = R_dp R_n).  Irminsul, 2.2 System
    Design, "delta-Rotation Rule": R(delta) applied to the stored key,
    delta = p_target - p_source (negative delta is a rotation backwards).
    """
    x = np.asarray(x, dtype=np.float64)
    a, b = rope_pairs(x.shape[-1], pairing)
    phi = np.float64(delta) * np.asarray(theta, dtype=np.float64)
    c = np.cos(phi)
    s = np.sin(phi)
    xa = x[..., a]
    xb = x[..., b]
    out = np.empty_like(x)
    out[..., a] = xa * c - xb * s
    out[..., b] = xa * s + xb * c
    return out


def rotate_rows(rows, delta: int, theta: np.ndarray, pairing: int,
                rope_offset: int, rope_dim: int) -> np.ndarray:
    """Rotate only the rope slice [rope_offset, rope_offset + rope_dim) of each row.

    For a GQA key the slice is the whole head (EPIC: the full key is
    re-rotated).  For an MLA row it is the 64-d decoupled rope key after the
    512-d latent, and the latent is passed through unchanged (Irminsul,
    2.1 Structural Insight: MLA Decomposition).
    """
    rows = np.asarray(rows, dtype=np.float64)
    out = rows.copy()
    sl = slice(rope_offset, rope_offset + rope_dim)
    out[..., sl] = rotate(rows[..., sl], delta, theta, pairing)
    return out


# ---------------------------------------------------------------------------
# registry entries, the prompt composer
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Chunk:
    """A registry entry: where the chunk's rows sit in the pool, its length,
    and the position it was computed at (0 = cached at virtual offset 0)."""
    pool_offset: int
    num_tokens: int
    base_pos: int = 0


@dataclass(frozen=True)
class Segment:
    chunk: int
    src_tok: int      # first pool token row read
    length: int       # tokens taken from the chunk
    dst_pos: int      # absolute position of the first token in the prompt
    delta: int        # dst_pos - base_pos


def compose(chunks, chunk_ids, take=None, dst_pos=None, start_pos: int = 0):
    """Place the chunks of one prompt and give each its shift.

    EPIC Guide, "Algorithmic Architecture: The EPIC Serving Runtime",
    2. Modular Prompt Composer: every hit chunk gets its absolute offset dp;
    chunks follow one another, so without explicit positions chunk j starts
    where chunk j-1 ended (the figure "Prefix Caching vs. Position-Independent
    Caching" stitches a 128-token block A, then B at 128, then C at 8,320).
    Irminsul "delta-Rotation Rule": delta = p_target - p_source, here
    dst_pos - base_pos.  ``take`` keeps only the first take[j] tokens of a
    chunk; ``dst_pos`` gives explicit positions (each at or after the end of
    the previous chunk, as in the guide's client request with "offset").
    """
    segs = []
    pos = start_pos
    prev_end = None
    for j, cid in enumerate(chunk_ids):
        c = chunks[cid]
        n = c.num_tokens if take is None else int(take[j])
        if n < 0 or n > c.num_tokens:
            raise ValueError("take exceeds the chunk")
        p = pos if dst_pos is None else int(dst_pos[j])
        if p < 0 or (prev_end is not None and p < prev_end):
            raise ValueError("chunks overlap or go backwards")
        segs.append(Segment(cid, c.pool_offset, n, p, p - c.base_pos))
        pos = p + n
        prev_end = pos
    return segs


def blocks_needed(total_tokens: int, block_size: int) -> int:
    return -(-total_tokens // block_size)


class BlockPool:
    """Physical paged-cache blocks; hands out the lowest-numbered free ids.

    The pages reuse PagedAttention's block pool without fixing an allocation
    order; lowest-free-first gives one deterministic table, so tables can be
    compared exactly.
    """

    def __init__(self, num_blocks: int):
        self.free = [True] * num_blocks

    def allocate(self, n: int):
        got = []
        for b in range(len(self.free)):
            if len(got) == n:
                break
            if self.free[b]:
                got.append(b)
        if len(got) < n:
            raise MemoryError("out of cache blocks")
        for b in got:
            self.free[b] = False
        return got

    def release(self, ids):
        for b in ids:
            if self.free[b]:
                raise ValueError("double free")
            self.free[b] = True


# ---------------------------------------------------------------------------
# selective-recompute token list
# ---------------------------------------------------------------------------

def recompute_positions(segs, k_nonleading: int, k_leading: int):
    """Ascending positions whose KV is recomputed after stitching.

    EPIC Guide, LegoLink "1. Identifying and Neutralizing Pseudo-Sinks": the
    first tokens of each chunk (sink_tokens = 4 in the listing's EPICConfig
    and the --pic-legolink-sink-tokens 4 flag) are the boundary tokens to fix,
    and the chunk at global position 0 is left alone ("Protect global token
    0").  Irminsul "First-Chunk Carve-Out": the first 32 tokens of a chunk that
    starts at absolute position 0 are prefilled normally and later chunks need
    nothing.  So a segment at position 0 contributes its first k_leading
    tokens, every other segment its first k_nonleading tokens, each clamped
    to the segment's own length.
    """
    out = []
    for s in segs:
        k = k_leading if s.dst_pos == 0 else k_nonleading
        out.extend(range(s.dst_pos, s.dst_pos + min(k, s.length)))
    return out


def recompute_csr(per_request):
    """Batch the per-request lists as CSR: (indptr[n_req + 1], idx)."""
    indptr = [0]
    idx = []
    for lst in per_request:
        idx.extend(lst)
        indptr.append(len(idx))
    return np.asarray(indptr, dtype=np.int64), np.asarray(idx, dtype=np.int64)


# ---------------------------------------------------------------------------
# the stitch and the in-place shift, token by token
# ---------------------------------------------------------------------------

def stitch_paged(k_pool_bits, v_pool_bits, plans, block_tables, num_blocks: int,
                 block_size: int, theta, pairing: int, rope_offset: int, rope_dim: int,
                 layers=None):
    """Expected paged caches after stitching ``plans`` (one list of Segments per request).

    For every layer l, segment, token t < length:
        slot  = block_tables[req][p // block_size], row p % block_size, p = dst_pos + t
        K[l][slot][row] = R(delta) K_pool[l][src_tok + t]     (rope slice only)
        V[l][slot][row] = V_pool[l][src_tok + t]              (bit copy)
    EPIC Guide, "Mathematical Foundations" 2: keys rotated, "Values (V) are
    completely untouched"; runtime figure: the prompt's chunks land in
    PagedAttention blocks.  Irminsul: the latent (rope_offset > 0) is copied
    verbatim.

    k_pool_bits: uint16 [L][P][*row]; v_pool_bits same or None.
    Returns (K float64 [L'][num_blocks][block_size][*row] with NaN where
    nothing was written, V uint16 same shape filled with BF16_SENTINEL
    elsewhere, or None).  ``layers`` restricts to a subset of layers (in
    that order).
    """
    k_pool_bits = np.asarray(k_pool_bits).view(np.uint16)
    L = k_pool_bits.shape[0]
    layers = list(range(L)) if layers is None else list(layers)
    row_shape = k_pool_bits.shape[2:]
    k_out = np.full((len(layers), num_blocks, block_size) + row_shape, np.nan)
    v_out = None
    if v_pool_bits is not None:
        v_pool_bits = np.asarray(v_pool_bits).view(np.uint16)
        v_out = np.full((len(layers), num_blocks, block_size) + row_shape,
                        BF16_SENTINEL, dtype=np.uint16)
    for li, l in enumerate(layers):
        for req, segs in enumerate(plans):
            bt = block_tables[req]
            for s in segs:
                for t in range(s.length):
                    p = s.dst_pos + t
                    slot = bt[p // block_size]
                    row = p % block_size
                    src = bf16_bits_to_f64(k_pool_bits[l, s.src_tok + t])
                    k_out[li, slot, row] = rotate_rows(src, s.delta, theta, pairing,
                                                       rope_offset, rope_dim)
                    if v_out is not None:
                        v_out[li, slot, row] = v_pool_bits[l, s.src_tok + t]
    return k_out, v_out


def rerotate_inplace(k_cache_bits, block_tables, segs, block_size: int, theta,
                     pairing: int, rope_offset: int, rope_dim: int):
    """Expected cache after rotating listed token ranges in place.

    EPIC Guide, runtime figure step 2 "Fast In-Place RoPE Key Rotation:
    Shifter applies delta_p to keys in HBM"; "Mathematical Foundations" 2.
    ``segs`` are (req, start_pos, length, delta); each listed key row
    becomes R(delta) of itself (rope slice only); nothing else changes.
    Returns float64 [L][num_blocks][block_size][*row] (unlisted rows are the
    input values; listed rows are unrounded).
    """
    bits = np.asarray(k_cache_bits).view(np.uint16)
    out = bf16_bits_to_f64(bits)
    for (req, start, length, delta) in segs:
        for t in range(length):
            p = start + t
            slot = block_tables[req][p // block_size]
            row = p % block_size
            out[:, slot, row] = rotate_rows(out[:, slot, row], delta, theta, pairing,
                                            rope_offset, rope_dim)
    return out


def expected_row(k_pool_row_bits, delta: int, theta, pairing: int, rope_offset: int,
                 rope_dim: int) -> np.ndarray:
    """One stitched key row from its pool row: R(delta) on the rope slice."""
    return rotate_rows(bf16_bits_to_f64(k_pool_row_bits), delta, theta, pairing,
                       rope_offset, rope_dim)


# ---------------------------------------------------------------------------
# virtual block mapping (chunks resident in paged blocks)
# ---------------------------------------------------------------------------

@dataclass
class BlockChunk:
    """A chunk whose KV sits in physical blocks of the paged cache: blocks[j]
    holds its tokens [j*bs, (j+1)*bs) (the last block partly).  cur_pos is the
    position its keys are currently rotated to (its base position when
    registered); refs counts live requests that use it, mapped_by the one
    request that has its blocks mapped (or None)."""
    blocks: tuple
    num_tokens: int
    cur_pos: int = 0
    refs: int = 0
    mapped_by: object = None


@dataclass(frozen=True)
class MappedSegment:
    """One chunk occurrence.  mode 'alias': the chunk's own blocks serve these
    positions and its keys rotate in place by delta.  mode 'copy': tokens are
    read from src_rows (pool token rows when src_kind == 'pool', absolute
    cache rows block*bs + row when 'cache') and written rotated by delta."""
    chunk: int
    mode: str
    src_kind: str
    length: int
    dst_pos: int
    delta: int
    src_rows: tuple


class BusyError(Exception):
    """A chunk is mapped by a live request and cannot be used by another."""


def map_request(chunks, chunk_ids, block_size, pool: BlockPool, req_id, start_pos=0,
                total_tokens=0, alias=True):
    """Compose a request whose chunks may sit in paged blocks.

    EPIC Guide, runtime figure: step 1 "Virtual Block Mapping" (the request
    reuses the chunk's physical blocks) and step 2 (the keys are rotated in
    place by dp; values untouched).  The figure states no conditions; the
    rules taken here: a block-resident chunk is mapped when aliasing is on, it starts on a
    block boundary, it occurs once in the request and no other live request
    uses it; otherwise it is copied out of its blocks.  A chunk mapped by a
    live request may not be used by any other (BusyError).  delta is always
    dst_pos - cur_pos.  Logical blocks not served by a mapped chunk get fresh
    blocks, lowest id first.  On success the registry state changes: refs of
    used block chunks +1, mapped chunks record the request and move cur_pos to
    their new position.  Returns (segments, table, fresh blocks, undo list).
    """
    bs = block_size
    counts = {}
    for cid in chunk_ids:
        counts[cid] = counts.get(cid, 0) + 1
    segs, mapped, pos = [], {}, start_pos
    for cid in chunk_ids:
        c = chunks[cid]
        n = c.num_tokens
        if isinstance(c, BlockChunk):
            if c.mapped_by is not None:
                raise BusyError(cid)
            delta = pos - c.cur_pos
            if alias and pos % bs == 0 and counts[cid] == 1 and c.refs == 0:
                for j, b in enumerate(c.blocks):
                    mapped[pos // bs + j] = b
                segs.append(MappedSegment(cid, "alias", "", n, pos, delta, ()))
            else:
                rows = tuple(c.blocks[t // bs] * bs + t % bs for t in range(n))
                segs.append(MappedSegment(cid, "copy", "cache", n, pos, delta, rows))
        else:
            rows = tuple(range(c.pool_offset, c.pool_offset + n))
            segs.append(MappedSegment(cid, "copy", "pool", n, pos, pos - c.base_pos, rows))
        pos += n
    total = max(pos, total_tokens)
    n_logical = blocks_needed(total, bs)
    need = [j for j in range(n_logical) if j not in mapped]
    fresh = pool.allocate(len(need))
    table = [0] * n_logical
    for j, b in mapped.items():
        table[j] = b
    for j, b in zip(need, fresh):
        table[j] = b
    undo = []
    for s in segs:
        c = chunks[s.chunk]
        if isinstance(c, BlockChunk):
            c.refs += 1
            if s.mode == "alias":
                undo.append((s.chunk, c.cur_pos))
                c.mapped_by = req_id
                c.cur_pos = s.dst_pos
    return segs, table, fresh, undo


def release_request(chunks, segs, fresh, undo, pool: BlockPool, applied: bool):
    """Free a mapped request: fresh blocks go back, block chunks lose a
    reference, mapped chunks are released (and, if the request's in-place
    rotations never ran, return to their old position)."""
    pool.release(fresh)
    for s in segs:
        c = chunks[s.chunk]
        if isinstance(c, BlockChunk):
            c.refs -= 1
            if s.mode == "alias":
                c.mapped_by = None
    if not applied:
        for cid, old in undo:
            chunks[cid].cur_pos = old


def apply_mapped(k_cache_bits, v_cache_bits, k_pool_bits, v_pool_bits, segs, table, block_size,
                 theta, pairing, rope_offset, rope_dim):
    """Expected caches after one mapped request runs: K float64 (NaN-free: the
    whole input cache, updated), V bits.  Every read sees the cache as it was
    before the request (the rules above keep reads and in-place writes of one
    launch on different rows).  k_cache_bits: uint16 [L][blocks][bs][*row]."""
    bs = block_size
    kc = np.asarray(k_cache_bits).view(np.uint16)
    k_before = bf16_bits_to_f64(kc)
    k_out = k_before.copy()
    L = kc.shape[0]
    flat_k = k_before.reshape((L, -1) + kc.shape[3:])
    v_out = flat_v = None
    if v_cache_bits is not None:
        vc = np.asarray(v_cache_bits).view(np.uint16)
        v_out = vc.copy()
        flat_v = vc.reshape((L, -1) + vc.shape[3:])
    for s in segs:
        for t in range(s.length):
            p = s.dst_pos + t
            slot, row = table[p // bs], p % bs
            if s.mode == "alias":
                src = k_before[:, slot, row]
            elif s.src_kind == "cache":
                src = flat_k[:, s.src_rows[t]]
                if v_out is not None:
                    v_out[:, slot, row] = flat_v[:, s.src_rows[t]]
            else:
                src = bf16_bits_to_f64(np.asarray(k_pool_bits).view(np.uint16)[:, s.src_rows[t]])
                if v_out is not None:
                    v_out[:, slot, row] = np.asarray(v_pool_bits).view(np.uint16)[:, s.src_rows[t]]
            k_out[:, slot, row] = rotate_rows(src, s.delta, theta, pairing, rope_offset, rope_dim)
    return k_out, v_out


# ---------------------------------------------------------------------------
# decode attention over a stitched context
# ---------------------------------------------------------------------------

def attention_decode(q, keys, values, scale: float, bias=None):
    """One decode step of grouped-query attention, in float64.

    q: [Hq][D] (already rotated to the query's position); keys, values:
    [T][Hkv][D] (keys rotated to their positions); query head g reads KV head
    g // (Hq / Hkv).  scores = scale * q.k + bias (bias: [T] or None),
    p = softmax over the T positions, out = sum_t p_t v_t.  Returns
    (out [Hq][D], log-sum-exp of the scaled scores [Hq]).  The definition of
    attention the pages rely on (EPIC Guide's listing computes the same
    softmax(q k^T / sqrt(d)) v in its LegoLink repair).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    hq = q.shape[0]
    hkv = keys.shape[1]
    group = hq // hkv
    out = np.empty((hq, values.shape[2]))
    lse = np.empty(hq)
    for g in range(hq):
        h = g // group
        s = scale * (keys[:, h, :] @ q[g])
        if bias is not None:
            s = s + bias
        m = s.max()
        e = np.exp(s - m)
        out[g] = (e[:, None] * values[:, h, :]).sum(axis=0) / e.sum()
        lse[g] = m + np.log(e.sum())
    return out, lse


def sink_bias(segs, total_tokens: int, k_nonleading: int, bias_value: float):
    """Per-position logit bias of LegoLink's pseudo-sink suppression: the
    first k tokens of every chunk not at global position 0 get bias_value
    (EPIC Guide, LegoLink "1. Identifying and Neutralizing Pseudo-Sinks";
    the listing subtracts 15 from those logits and leaves boundary 0 alone)."""
    b = np.zeros(total_tokens)
    for s in segs:
        if s.dst_pos == 0:
            continue
        b[s.dst_pos:s.dst_pos + min(k_nonleading, s.length)] = bias_value
    return b
