"""The seeded generators draw the workloads' stated structure, deterministically."""

import math

import workloads as W


def test_splitmix64_reference_values():
    # splitmix64 from state 0: the first outputs of the published generator.
    st, z = W._splitmix64_next(0)
    assert z == 0xE220A8397B1DCDAF
    st, z = W._splitmix64_next(st)
    assert z == 0x6E789E6AA1B965F4


def test_determinism():
    a, b = W.serving_stress(), W.serving_stress()
    assert a.requests == b.requests and a.chunk_lens == b.chunk_lens and a.new_pos == b.new_pos
    assert W.qwen3_8b_batch(seed=1).requests != W.qwen3_8b_batch(seed=0).requests


def test_tiny_and_llama_structure():
    t = W.tiny_gqa()
    assert t.request_tokens == [1056] and t.token_layers == 1056
    assert t.requests[0][0] == (0, 32) and sorted(c for c, _ in t.requests[0][1:]) == [1, 2, 3, 4]
    l = W.llama31_8b_rag()
    assert l.request_tokens == [10368] and l.token_layers == 331776
    assert l.model.llama3 == W.LLAMA3_SCALING and l.model.rope_theta == 5e5


def test_qwen_batch_structure():
    w = W.qwen3_8b_batch()
    assert len(w.chunk_lens) == 64 and all(128 <= n <= 4096 for n in w.chunk_lens)
    assert w.request_tokens == [32768] * 8
    for r in w.requests:
        ids = [c for c, _ in r]
        assert len(ids) == len(set(ids))
        assert all(t == w.chunk_lens[c] for c, t in r[:-1]) and 0 < r[-1][1] <= w.chunk_lens[r[-1][0]]
    assert w.token_layers == 9437184


def test_mla_structure():
    w = W.deepseek_v3_mla()
    assert w.model.kind == "mla" and w.model.head_dim == 576 and w.model.rope_offset == 512
    assert w.request_tokens == [65536] and w.chunk_lens[0] == 32
    assert all(16 <= n <= 128 for n in w.chunk_lens[1:])
    assert (w.k_leading, w.k_nonleading) == (32, 0)
    assert w.token_layers == 65536 * 61


def test_serving_structure():
    w = W.serving_stress()
    assert len(w.chunk_lens) == 256 and all(64 <= n <= 8192 for n in w.chunk_lens)
    assert w.request_tokens == [16384] * 64
    for r, np_ in zip(w.requests, w.new_pos):
        ids = [c for c, _ in r]
        assert len(ids) == len(set(ids))
        assert len(np_) == len(r)
        assert all(0 <= p <= 131072 - t for p, (_, t) in zip(np_, r))
    # Zipf(1.1): rank 0 is drawn far more often than a late rank
    counts = [0] * 256
    for r in w.requests:
        for c, _ in r:
            counts[c] += 1
    assert counts[0] >= 50 and counts[0] > 4 * max(1, counts[200])


def test_stream_ranges():
    s = W.Stream(0, "t")
    xs = [s.integers(3, 7) for _ in range(2000)]
    assert min(xs) == 3 and max(xs) == 7
    p = s.permutation(50)
    assert sorted(p) == list(range(50))
    ls = [s.log_uniform_int(64, 8192) for _ in range(2000)]
    assert min(ls) >= 64 and max(ls) <= 8192
    # log-uniform: the median sits near the geometric mean sqrt(64 * 8192) = 724
    ls.sort()
    assert abs(math.log(ls[1000]) - math.log(724)) < 0.2


def test_chunk_keys_distinct_32_bytes():
    keys = {W.chunk_key("w", i) for i in range(1000)}
    assert len(keys) == 1000 and all(len(k) == 32 for k in keys)
