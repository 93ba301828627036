"""Seeded synthetic inputs for position-independent KV stitching.

This module serves both the fp64 oracle's tests and the CUDA library's tests
and benchmark.  It holds no arithmetic of the method: no RoPE, no positions,
no shifts, no block tables, no recompute lists.  It only draws

* the chunk pool: how many chunks, their lengths, where their rows sit in the
  pool tensor (chunks stored back to back, in pool order);
* each request's chunk sequence (which chunk ids, in what order, how many
  tokens taken from the last one);
* the new positions of the in-place shift workload;
* the bfloat16 K / V / latent values (N(0, 1));
* token-id documents and the Gear table (one 64-bit random value per
  vocabulary id) for content-defined chunking.

Random structure comes from splitmix64 (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014), one stream per
purpose, so the same workload is drawn on every machine.  Tensor values come
from torch's seeded generator on the device that holds them (values differ
between CPU and CUDA generators; a check always reads the values actually
generated).

Value distribution: a cached key at local position n is R_n k_raw.  With
k_raw ~ N(0, I), R_n k_raw ~ N(0, I) again (a rotation of an isotropic
Gaussian), so i.i.d. N(0, 1) bfloat16 values have exactly the distribution
of offset-0 cached keys; values and MLA latents are drawn the same way.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from itertools import accumulate

import numpy as np

MASK64 = (1 << 64) - 1


def _fnv1a64(text: str) -> int:
    h = 0xCBF29CE484222325
    for ch in text.encode():
        h ^= ch
        h = (h * 0x100000001B3) & MASK64
    return h


def _splitmix64_next(state: int):
    state = (state + 0x9E3779B97F4A7C15) & MASK64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return state, z ^ (z >> 31)


class Stream:
    """One splitmix64 stream, keyed by (seed, purpose)."""

    def __init__(self, seed: int, purpose: str):
        self.state = (seed * 0x9E3779B97F4A7C15 ^ _fnv1a64(purpose)) & MASK64

    def u64(self) -> int:
        self.state, z = _splitmix64_next(self.state)
        return z

    def uniform(self) -> float:
        """Uniform in [0, 1) with 53 random bits."""
        return (self.u64() >> 11) * (1.0 / (1 << 53))

    def integers(self, lo: int, hi: int) -> int:
        """Uniform integer in [lo, hi] (inclusive), by rejection (no bias)."""
        span = hi - lo + 1
        if span <= 0:
            raise ValueError("empty range")
        limit = (1 << 64) - ((1 << 64) % span)
        while True:
            z = self.u64()
            if z < limit:
                return lo + z % span

    def permutation(self, n: int):
        """Fisher-Yates shuffle of range(n)."""
        p = list(range(n))
        for i in range(n - 1, 0, -1):
            j = self.integers(0, i)
            p[i], p[j] = p[j], p[i]
        return p

    def zipf_rank(self, n: int, s: float) -> int:
        """0-based rank r in [0, n) with P(r) proportional to (r + 1)^-s (inverse CDF)."""
        weights = [(r + 1) ** (-s) for r in range(n)]
        total = sum(weights)
        u = self.uniform() * total
        acc = 0.0
        for r, w in enumerate(weights):
            acc += w
            if u < acc:
                return r
        return n - 1

    def log_uniform_int(self, lo: int, hi: int) -> int:
        """round(exp(U[ln lo, ln hi]))."""
        x = math.log(lo) + self.uniform() * (math.log(hi) - math.log(lo))
        return int(round(math.exp(x)))


# ---------------------------------------------------------------------------
# model geometries and workloads
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Model:
    """KV geometry and RoPE settings of a model family (plain data)."""
    name: str
    kind: str                 # "gqa" | "mla"
    num_layers: int
    num_kv_heads: int         # GQA: KV heads per token row; MLA: 1
    head_dim: int             # GQA: dims per head; MLA: row width (latent + rope)
    rope_dim: int             # GQA: == head_dim; MLA: 64
    rope_offset: int          # GQA: 0; MLA: latent width
    pairing: str              # "neox" | "interleaved"
    rope_theta: float
    block_size: int = 16
    llama3: dict | None = None   # {"factor", "low_freq_factor", "high_freq_factor", "orig_max_pos"}

    @property
    def row_elems(self) -> int:
        return self.num_kv_heads * self.head_dim

    @property
    def row_shape(self):
        return (self.num_kv_heads, self.head_dim) if self.kind == "gqa" else (self.head_dim,)


LLAMA3_SCALING = {"factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
                  "orig_max_pos": 8192}


@dataclass
class Workload:
    """A chunk pool plus the requests composed from it.

    ``requests[r]`` is a list of (chunk_id, take_tokens).  ``k_nonleading`` /
    ``k_leading`` are the recompute settings.  ``new_pos[r][j]`` (optional)
    is the position chunk j of request r is moved to by the in-place shift
    workload.
    """
    name: str
    model: Model
    chunk_lens: list
    requests: list
    k_nonleading: int
    k_leading: int
    new_pos: list = field(default_factory=list)

    @property
    def pool_offsets(self):
        return [0] + list(accumulate(self.chunk_lens))[:-1]

    @property
    def pool_tokens(self) -> int:
        return sum(self.chunk_lens)

    @property
    def request_tokens(self):
        return [sum(t for _, t in r) for r in self.requests]

    @property
    def token_layers(self) -> int:
        return sum(self.request_tokens) * self.model.num_layers


def _fill_to(order, lens, target):
    """Take chunks from ``order`` until ``target`` tokens; truncate the last one."""
    out, total = [], 0
    for cid in order:
        if total >= target:
            break
        take = min(lens[cid], target - total)
        out.append((cid, take))
        total += take
    if total != target:
        raise ValueError("pool too small for the request length")
    return out


def tiny_gqa(seed: int = 0) -> Workload:
    """1 layer, 8 KV heads x 128, theta 1e4 neox; a 32-token prefix chunk
    then 4 chunks x 256 in seeded order; block 16; k = 4."""
    m = Model("tiny-gqa", "gqa", 1, 8, 128, 128, 0, "neox", 1.0e4)
    lens = [32, 256, 256, 256, 256]
    order = Stream(seed, "tiny/order").permutation(4)
    req = [(0, 32)] + [(1 + c, 256) for c in order]
    return Workload("tiny_gqa", m, lens, [req], 4, 0)


def llama31_8b_rag(seed: int = 0) -> Workload:
    """Llama-3.1-8B shapes: 32 layers, 8 KV heads x 128, theta 5e5 with llama3
    scaling; a 128-token system prompt then a permutation of 10 x 1024
    chunks; batch 1; k = 4."""
    m = Model("llama-3.1-8b", "gqa", 32, 8, 128, 128, 0, "neox", 5.0e5, 16, LLAMA3_SCALING)
    lens = [128] + [1024] * 10
    order = Stream(seed, "llama/order").permutation(10)
    req = [(0, 128)] + [(1 + c, 1024) for c in order]
    return Workload("llama31_8b_rag", m, lens, [req], 4, 0)


def qwen3_8b_batch(seed: int = 0, n_requests: int = 8, request_tokens: int = 32768) -> Workload:
    """Qwen3-8B shapes: 36 layers, 8 KV heads x 128, theta 1e6; a 64-chunk pool
    with lengths U[128, 4096]; 8 requests of 32,768 tokens, each a random
    order of the pool truncated to the length; k = 4."""
    m = Model("qwen3-8b", "gqa", 36, 8, 128, 128, 0, "neox", 1.0e6)
    ls = Stream(seed, "qwen/lengths")
    lens = [ls.integers(128, 4096) for _ in range(64)]
    reqs = []
    for r in range(n_requests):
        order = Stream(seed, f"qwen/order/{r}").permutation(64)
        reqs.append(_fill_to(order, lens, request_tokens))
    return Workload("qwen3_8b_batch", m, lens, reqs, 4, 0)


def deepseek_v3_mla(seed: int = 0, context_tokens: int = 65536, num_layers: int = 61) -> Workload:
    """DeepSeek-V3 MLA shapes: 61 layers, rows of a 512-d latent + 64-d rope key,
    theta 1e4 (interleaved pairs); a 32-token leading chunk then chunks of
    U[16, 128] tokens up to 65,536 tokens; the leading 32 tokens recomputed,
    nothing else."""
    m = Model("deepseek-v3", "mla", num_layers, 1, 576, 64, 512, "interleaved", 1.0e4)
    ls = Stream(seed, "mla/lengths")
    lens = [32]
    total = 32
    while total < context_tokens:
        n = ls.integers(16, 128)
        lens.append(n)
        total += n
    req = [(c, n) for c, n in enumerate(lens)]
    over = total - context_tokens
    if over:
        c, n = req[-1]
        req[-1] = (c, n - over)
    return Workload("deepseek_v3_mla", m, lens, [req], 0, 32)


def serving_stress(seed: int = 0, n_requests: int = 64, request_tokens: int = 16384,
                   pool_chunks: int = 256) -> Workload:
    """Llama-3.1-8B shapes; a 256-chunk pool with log-uniform lengths in
    [64, 8192]; 64 requests of 16,384 tokens whose chunks are Zipf(1.1) draws
    over pool rank (no repeats inside a request); for the in-place mode each
    chunk gets a new position uniform in [0, 131072 - length]; k = 4."""
    m = Model("llama-3.1-8b", "gqa", 32, 8, 128, 128, 0, "neox", 5.0e5, 16, LLAMA3_SCALING)
    ls = Stream(seed, "serve/lengths")
    lens = [ls.log_uniform_int(64, 8192) for _ in range(pool_chunks)]
    reqs, new_pos = [], []
    for r in range(n_requests):
        zs = Stream(seed, f"serve/zipf/{r}")
        seen, order = set(), []
        total = 0
        while total < request_tokens:
            cid = zs.zipf_rank(pool_chunks, 1.1)
            if cid in seen:
                continue
            seen.add(cid)
            order.append(cid)
            total += lens[cid]
        req = _fill_to(order, lens, request_tokens)
        reqs.append(req)
        ps = Stream(seed, f"serve/newpos/{r}")
        new_pos.append([ps.integers(0, 131072 - take) for _, take in req])
    return Workload("serving_stress", m, lens, reqs, 4, 0, new_pos)


WORKLOADS = {
    "tiny_gqa": tiny_gqa,
    "llama31_8b_rag": llama31_8b_rag,
    "qwen3_8b_batch": qwen3_8b_batch,
    "deepseek_v3_mla": deepseek_v3_mla,
    "serving_stress": serving_stress,
}


def chunk_key(workload_name: str, chunk_id: int) -> bytes:
    """A 32-byte registry key for a pool chunk (stands in for a content hash)."""
    raw = f"{workload_name}/chunk/{chunk_id}".encode()
    out = bytearray(32)
    h = _fnv1a64(raw.decode())
    for i in range(4):
        h, z = _splitmix64_next(h)
        out[8 * i:8 * i + 8] = z.to_bytes(8, "little")
    return bytes(out)


# ---------------------------------------------------------------------------
# tensor values (torch only here; no arithmetic of the method)
# ---------------------------------------------------------------------------

def make_pool(workload: Workload, which: str, device="cpu", seed: int = 0, generator=None):
    """bf16 pool tensor [L][pool_tokens][*row] with N(0, 1) values.

    ``which`` in {"k", "v"} (MLA rows use "k").  Filled layer by layer so no
    float32 temporary of the whole pool is ever made.
    """
    import torch

    m = workload.model
    shape = (m.num_layers, workload.pool_tokens) + tuple(m.row_shape)
    t = torch.empty(shape, dtype=torch.bfloat16, device=device)
    g = generator
    if g is None:
        g = torch.Generator(device=device)
        g.manual_seed((seed * 1000003 + _fnv1a64(workload.name + "/" + which)) & 0x7FFFFFFFFFFFFFFF)
    for layer in range(m.num_layers):
        t[layer].normal_(0.0, 1.0, generator=g)
    return t


def fill_random_bf16(t, seed: int, purpose: str):
    """Fill an existing bf16 tensor with N(0, 1) values from a seeded generator."""
    import torch

    g = torch.Generator(device=t.device)
    g.manual_seed((seed * 1000003 + _fnv1a64(purpose)) & 0x7FFFFFFFFFFFFFFF)
    flat = t.view(t.shape[0], -1) if t.dim() > 1 else t.view(1, -1)
    for i in range(flat.shape[0]):
        flat[i].normal_(0.0, 1.0, generator=g)
    return t


# ---------------------------------------------------------------------------
# token documents for content-defined chunking
# ---------------------------------------------------------------------------

_GOLDEN_GAMMA = 0x9E3779B97F4A7C15


def u64_array(seed: int, purpose: str, n: int) -> np.ndarray:
    """The first n outputs of Stream(seed, purpose), vectorised (uint64).

    splitmix64 is counter-based: output i is mix(state0 + (i + 1) * gamma),
    so a whole array is drawn at once and equals the sequential stream."""
    s0 = np.uint64(Stream(seed, purpose).state)
    with np.errstate(over="ignore"):
        z = s0 + np.uint64(_GOLDEN_GAMMA) * np.arange(1, n + 1, dtype=np.uint64)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


@dataclass
class Corpus:
    """Token-id documents stored back to back (int32), with the Gear table."""
    name: str
    vocab: int
    tokens: np.ndarray        # int32 [n_tokens]
    offsets: np.ndarray       # int64 [n_docs + 1]
    gear: np.ndarray          # uint64 [vocab]

    @property
    def n_docs(self) -> int:
        return len(self.offsets) - 1

    def doc(self, i: int) -> np.ndarray:
        return self.tokens[self.offsets[i]:self.offsets[i + 1]]


def gear_table(seed: int, vocab: int) -> np.ndarray:
    """One random 64-bit value per vocabulary id."""
    return u64_array(seed, "cdc/gear", vocab)


def random_tokens(seed: int, purpose: str, n: int, vocab: int) -> np.ndarray:
    """n token ids, uniform over [0, vocab) (modulo of 64 random bits)."""
    return (u64_array(seed, purpose, n) % np.uint64(vocab)).astype(np.int32)


def corpus_from_lengths(name: str, seed: int, lengths, vocab: int) -> Corpus:
    offsets = np.zeros(len(lengths) + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    tokens = random_tokens(seed, name + "/tokens", int(offsets[-1]), vocab)
    return Corpus(name, vocab, tokens, offsets, gear_table(seed, vocab))


def rag_corpus(seed: int = 0, n_docs: int = 8192, lo: int = 512, hi: int = 16384, vocab: int = 128256) -> Corpus:
    """Multi-document RAG corpus: n_docs documents of round(exp(U[ln lo, ln
    hi])) tokens (mean ~4k), token ids uniform over a Llama-3-sized vocabulary."""
    st = Stream(seed, "cdc/lengths")
    lengths = [st.log_uniform_int(lo, hi) for _ in range(n_docs)]
    return corpus_from_lengths("rag_corpus", seed, lengths, vocab)
