"""GPU parity of content-defined chunking and fingerprints (Irminsul 2.2,
"Content-Hash Keying with CDC"; "Hybrid Strategies (S1/S2)") against the
oracle, through the C ABI.  Chunk boundaries, CSR offsets and fingerprints are
integers: they must match bit for bit."""

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

MASK64 = (1 << 64) - 1


@pytest.fixture(scope="module")
def pic():
    from position_independent_kv_stitch_gb300 import pic as p
    p.load()
    return p


def _corpus(lengths, vocab=1000, seed=3, lead=0, trail=0):
    """Documents of the given lengths stored back to back after `lead` tokens
    that belong to no document, followed by `trail` such tokens."""
    n = lead + sum(lengths) + trail
    tokens = W.random_tokens(seed, "test/cdc", n, vocab)
    offsets = np.zeros(len(lengths) + 1, dtype=np.int64)
    offsets[0] = lead
    offsets[1:] = lead + np.cumsum(np.asarray(lengths, dtype=np.int64))
    return tokens, offsets, W.gear_table(seed, vocab)


def _oracle(tokens, offsets, gear, thr, min_len=0, max_len=0, seed=0, docs=None):
    """indptr, ends (global), fingerprints of the given documents (all by default)."""
    docs = range(len(offsets) - 1) if docs is None else docs
    indptr, ends, fps = [0], [], []
    for d in docs:
        s, e = int(offsets[d]), int(offsets[d + 1])
        if e > s:
            le, lf = oracle.chunk_document(list(tokens[s:e]), gear, thr, min_len, max_len, seed)
            ends += [s + x for x in le]
            fps += lf
        indptr.append(len(ends))
    return np.asarray(indptr, dtype=np.int64), np.asarray(ends, dtype=np.int64), np.asarray(fps, dtype=np.uint64)


def _gpu(pic, tokens, offsets, gear, thr, min_len=0, max_len=0, seed=0, cap=None, fingerprints=True, ws=None):
    import torch
    dev = torch.device("cuda", 0)
    t = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).to(dev)
    o = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int64)).to(dev)
    g = torch.from_numpy(np.ascontiguousarray(gear, dtype=np.uint64).view(np.int64)).to(dev)
    n_docs = len(offsets) - 1
    if cap is None:
        cap = len(tokens) + 1
    indptr = torch.full((n_docs + 1,), -7, dtype=torch.int64, device=dev)
    ends = torch.full((max(cap, 1),), -7, dtype=torch.int64, device=dev)[:cap]
    fps = torch.full((max(cap, 1),), -7, dtype=torch.int64, device=dev)[:cap] if fingerprints else None
    ws = pic.pic_cdc_chunk(t, o, g, thr, indptr, ends, fps, min_len, max_len, seed, workspace=ws)
    status = pic.pic_query_device_status(None, ws, raise_on_device_error=False)
    out_f = fps.cpu().numpy().view(np.uint64) if fps is not None else None
    return indptr.cpu().numpy(), ends.cpu().numpy(), out_f, status, ws


def _assert_same(got, want, cap=None):
    gi, ge, gf, st, _ = got
    wi, we, wf = want
    assert gi.tolist() == wi.tolist()
    n = len(we) if cap is None else min(cap, len(we))
    assert ge[:n].tolist() == we[:n].tolist()
    if gf is not None:
        assert gf[:n].tolist() == wf[:n].tolist()


EDGE_LENGTHS = [0, 1, 31, 32, 33, 63, 64, 65, 0, 0, 127, 8191, 2, 8192, 8193, 20000, 1, 300, 0, 5000]


@pytest.mark.parametrize("mean", [16, 24, 32, 64, 256])
def test_edge_lengths_match_oracle(pic, mean):
    """Empty, tiny and tile-straddling documents (tiles are 8192 tokens),
    from about 512 chunks a tile (mean 16) down to about 32 (mean 256)."""
    tokens, offsets, gear = _corpus(EDGE_LENGTHS)
    thr = oracle.threshold_for_mean(mean)
    got = _gpu(pic, tokens, offsets, gear, thr)
    assert got[3] == 0
    _assert_same(got, _oracle(tokens, offsets, gear, thr))


@pytest.mark.parametrize("min_len,max_len", [(16, 0), (0, 100), (32, 256), (64, 64), (16, 128), (1, 1),
                                             (5000, 0), (200, 50)])
def test_length_rules_match_oracle(pic, min_len, max_len):
    tokens, offsets, gear = _corpus(EDGE_LENGTHS, seed=4)
    thr = oracle.threshold_for_mean(48)
    got = _gpu(pic, tokens, offsets, gear, thr, min_len, max_len)
    assert got[3] == 0
    _assert_same(got, _oracle(tokens, offsets, gear, thr, min_len, max_len))


def test_tokens_outside_documents_and_seeded_fingerprints(pic):
    """Offsets need not start at 0 nor end at the last token; a seed changes
    every fingerprint but no boundary."""
    tokens, offsets, gear = _corpus([700, 9000, 13], lead=37, trail=1000, seed=5)
    thr = oracle.threshold_for_mean(64)
    seed = 0x9E3779B97F4A7C15
    got = _gpu(pic, tokens, offsets, gear, thr, seed=seed)
    assert got[3] == 0
    _assert_same(got, _oracle(tokens, offsets, gear, thr, seed=seed))


@pytest.mark.parametrize("thr", [0, 1, MASK64])
def test_extreme_thresholds(pic, thr):
    """threshold 0: no hash cut (one chunk per document); 2^64 - 1: a cut at
    nearly every token."""
    tokens, offsets, gear = _corpus([100, 0, 3000, 64], seed=6)
    got = _gpu(pic, tokens, offsets, gear, thr)
    _assert_same(got, _oracle(tokens, offsets, gear, thr))
    if thr == 0:
        assert got[0].tolist() == [0, 1, 1, 2, 3]


def test_without_fingerprints_and_reused_workspace(pic):
    tokens, offsets, gear = _corpus([5000, 17, 9000], seed=7)
    thr = oracle.threshold_for_mean(32)
    want = _oracle(tokens, offsets, gear, thr)
    first = _gpu(pic, tokens, offsets, gear, thr, fingerprints=False)
    _assert_same(first, want)
    again = _gpu(pic, tokens, offsets, gear, thr, ws=first[4])
    _assert_same(again, want)
    assert again[3] == 0


def test_capacity_overflow_writes_a_prefix(pic):
    tokens, offsets, gear = _corpus([3000, 3000], seed=8)
    thr = oracle.threshold_for_mean(32)
    want = _oracle(tokens, offsets, gear, thr)
    cap = len(want[1]) // 3
    got = _gpu(pic, tokens, offsets, gear, thr, cap=cap)
    assert got[3] & pic.PIC_DEV_CAPACITY
    _assert_same(got, want, cap=cap)
    assert got[0][-1] == len(want[1])   # the total is reported even past capacity


def test_out_of_vocabulary_token_counts_as_zero(pic):
    tokens, offsets, gear = _corpus([400, 400], vocab=500, seed=9)
    tokens = tokens.copy()
    tokens[150] = 500
    tokens[600] = -5
    got = _gpu(pic, tokens, offsets, gear, oracle.threshold_for_mean(16))
    assert got[3] & pic.PIC_DEV_BAD_TOKEN
    # boundaries: the same as a Gear table whose extra entry (the bad ids'
    # stand-in) is 0; fingerprints: of the token ids as they are
    g2 = np.concatenate([gear, np.zeros(1, dtype=np.uint64)])
    t2 = tokens.copy()
    t2[[150, 600]] = 500
    wi, we, _ = _oracle(t2, offsets, g2, oracle.threshold_for_mean(16))
    starts = [int(offsets[0])] + we[:-1].tolist()
    for d in range(len(offsets) - 1):
        starts[wi[d]] = int(offsets[d])
    wf = np.asarray([oracle.fingerprint(tokens[s:e]) for s, e in zip(starts, we)], dtype=np.uint64)
    _assert_same(got, (wi, we, wf))


@pytest.mark.parametrize("bad", [[0, 50, 40, 100], [0, 50, 101], [-1, 50, 100]])
def test_bad_offsets_are_caught_on_the_device(pic, bad):
    tokens, _, gear = _corpus([100])
    got = _gpu(pic, tokens, np.asarray(bad, dtype=np.int64), gear, oracle.threshold_for_mean(16))
    assert got[3] & pic.PIC_DEV_BAD_DOCS
    assert got[0].tolist() == [0] * len(bad)


def test_no_documents_and_no_tokens(pic):
    gear = W.gear_table(1, 10)
    got = _gpu(pic, np.zeros(0, dtype=np.int32), np.zeros(1, dtype=np.int64), gear, 1 << 60)
    assert got[0].tolist() == [0] and got[3] == 0
    got = _gpu(pic, np.zeros(0, dtype=np.int32), np.zeros(4, dtype=np.int64), gear, 1 << 60)
    assert got[0].tolist() == [0, 0, 0, 0] and got[3] == 0


def test_fingerprint_spans_s1_windows(pic):
    """S1: a chunk that missed the registry is cut into 128-token windows, each
    fingerprinted; spans outside the tokens are flagged and hashed as 0."""
    import torch
    dev = torch.device("cuda", 0)
    tokens, offsets, gear = _corpus([3000], seed=10)
    spans = oracle.s1_windows(17, 1000) + [(5, 5), (0, 3000), (2999, 3000), (10, 7)]
    t = torch.from_numpy(tokens).to(dev)
    s = torch.tensor([a for a, _ in spans], dtype=torch.int64, device=dev)
    e = torch.tensor([b for _, b in spans], dtype=torch.int64, device=dev)
    out = torch.empty(len(spans), dtype=torch.int64, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    seed = 12345
    pic.pic_fingerprint_spans(t, s, e, out, status, seed=seed)
    got = out.cpu().numpy().view(np.uint64).tolist()
    want = [oracle.fingerprint(tokens[a:b], seed) for a, b in spans[:-1]] + [0]
    assert got == want
    assert int(status.item()) == pic.PIC_DEV_BAD_SPAN


def test_full_rag_corpus_sampled(pic):
    """The benchmark's corpus (8,192 documents, log-uniform 512-16,384 tokens,
    Llama-3 vocabulary) in the benchmark's launch configuration: sampled
    documents are compared with the oracle in full, and at every document the
    CSR offsets and the last chunk end are checked."""
    corpus = W.rag_corpus()
    thr = oracle.threshold_for_mean(64)
    got = _gpu(pic, corpus.tokens, corpus.offsets, corpus.gear, thr, cap=len(corpus.tokens) // 8)
    indptr, ends, fps, status, _ = got
    assert status == 0
    counts = np.diff(indptr)
    assert np.all(counts >= 1)
    assert np.array_equal(ends[indptr[1:] - 1], corpus.offsets[1:])     # every document's tail is a chunk
    assert np.all(np.diff(ends[:indptr[-1]]) > 0)
    n_docs = corpus.n_docs
    lens = np.diff(corpus.offsets)
    sample = sorted({0, 1, n_docs - 1, int(np.argmax(lens)), int(np.argmin(lens))}
                    | set(int(x) for x in np.random.default_rng(0).choice(n_docs, 24, replace=False)))
    for d in sample:
        wi, we, wf = _oracle(corpus.tokens, corpus.offsets, corpus.gear, thr, docs=[d])
        a, b = indptr[d], indptr[d + 1]
        assert b - a == wi[-1], d
        assert ends[a:b].tolist() == we.tolist(), d
        assert fps[a:b].tolist() == wf.tolist(), d
