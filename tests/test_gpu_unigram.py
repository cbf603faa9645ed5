"""GPU parity of Unigram (Viterbi) encoding against the CPU oracle, bit for bit.

Small cases run the oracle live; the batch workload and the 64 MiB document
are compared with the oracle's recorded results (tests/golden/workloads.json)
by SHA-256.  All calls go through the C ABI (unigram_create/encode).
"""
import hashlib
import json
import os
import random

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ALPHA = [b"a", b"b", b"c", b" ", "ı".encode(), "ş".encode(), "€".encode()]


def sha(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


@pytest.fixture(scope="module")
def ctx():
    import bpe_trie_encode_gb300 as bt
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    c = bt.Context(0)
    yield c
    c.close()


@pytest.fixture(scope="module")
def golden():
    with open(os.path.join(GOLDEN, "workloads.json")) as f:
        return json.load(f)


def vocab_arrays(tokens):
    vb = b"".join(tokens)
    off = np.cumsum([0] + [len(t) for t in tokens]).astype(np.uint64)
    return np.frombuffer(vb, dtype=np.uint8).copy(), off


def dev_u8(a):
    a = np.frombuffer(a, dtype=np.uint8) if isinstance(a, (bytes, bytearray)) else a
    if a.size == 0:
        return torch.empty(0, dtype=torch.uint8, device="cuda")
    return torch.from_numpy(np.ascontiguousarray(a).copy()).cuda()


def f32(x):
    return float(np.float32(x))


def check_unigram(ctx, vb, off, scores, unk_id, unk_score, docs, chunk=0):
    import bpe_trie_encode_gb300 as bt
    data = b"".join(docs)
    doc_off = np.cumsum([0] + [len(d) for d in docs]).astype(np.int64)
    trie = ctx.trie_build(vb, off)
    model = ctx.unigram(trie, scores, unk_id, unk_score)
    ctx.set_option(bt.BPE_OPT_UNI_CHUNK, chunk)
    try:
        ids, id_off = ctx.unigram_encode(model, dev_u8(data), torch.from_numpy(doc_off).cuda())
    finally:
        ctx.set_option(bt.BPE_OPT_UNI_CHUNK, 0)
    wids, woff = oracle.Trie(vb, off).unigram_encode(data, scores, unk_id, unk_score, doc_off.astype(np.uint64))
    got = ids.cpu().numpy()
    assert got.size == wids.size
    if not np.array_equal(got, wids):
        i = int(np.nonzero(got != wids)[0][0])
        raise AssertionError(f"first difference at id {i}: {got[i - 3:i + 3]} vs {wids[i - 3:i + 3]}")
    assert np.array_equal(id_off.cpu().numpy().astype(np.uint64), woff)
    return got


def test_hand_worked(ctx):
    vb, off = vocab_arrays([b"a", b"b", b"ab"])
    assert check_unigram(ctx, vb, off, [-1.0, -1.0, -1.5], 9, -50.0, [b"ab"]).tolist() == [2]
    assert check_unigram(ctx, vb, off, [-1.0, -1.0, -2.5], 9, -50.0, [b"ab"]).tolist() == [0, 1]
    assert check_unigram(ctx, vb, off, [-1.0, -1.0, -2.0], 9, -50.0, [b"ab"]).tolist() == [2]
    assert check_unigram(ctx, vb, off, [-1.0, -1.0, -1.5], 9, -50.0, [b"abcab"]).tolist() == [2, 9, 2]
    vb, off = vocab_arrays([b"a", b"\xc4", b"a\xc4", b"\xb1"])
    sc = [-1.0, -0.125, -0.125, -0.125]
    assert check_unigram(ctx, vb, off, sc, 7, -20.0, ["aı".encode()]).tolist() == [0, 7]
    assert check_unigram(ctx, vb, off, sc, 7, -20.0, ["a€a".encode()]).tolist() == [0, 7, 0]


def random_model(rng, n_tok, max_tok=6, partial=0.1):
    toks = []
    while len(toks) < n_tok:
        t = b"".join(rng.choice(ALPHA) for _ in range(rng.randint(1, max_tok)))
        if rng.random() < partial:
            t = t[: rng.randint(1, len(t))]
        toks.append(t)
    scores = [f32(-rng.uniform(1.0, 12.0)) for _ in toks]
    return toks, scores


@pytest.mark.parametrize("seed", range(10))
def test_random_vocab_ragged_docs(ctx, seed):
    rng = random.Random(seed)
    toks, scores = random_model(rng, rng.choice([5, 40, 400, 3000]))
    if seed % 2:   # integer scores: many ties
        scores = [float(-rng.randint(1, 5)) for _ in toks]
    vb, off = vocab_arrays(toks)
    docs = [b"".join(rng.choice(ALPHA) for _ in range(rng.choice([0, 1, 5, 100, 300, 1000, 3000])))
            for _ in range(rng.randint(1, 30))]
    check_unigram(ctx, vb, off, scores, len(toks), -30.0, docs, chunk=256)


@pytest.mark.parametrize("chunk", [256, 320, 512, 1024, 4096])
def test_chunk_sizes_agree(ctx, chunk):
    rng = random.Random(5)
    toks, scores = random_model(rng, 2000, max_tok=10)
    vb, off = vocab_arrays(toks)
    docs = [b"".join(rng.choice(ALPHA) for _ in range(n)) for n in (20000, 7, 4095, 4096, 4097, 0, 12345)]
    check_unigram(ctx, vb, off, scores, len(toks), -30.0, docs, chunk=chunk)


def test_repairs_parity_runs(ctx):
    """'a' * n under {a: -1, aa: -1.5}: the best path's parity is set by the
    document start, so every speculative chunk is wrong and both repair
    passes re-run every chunk."""
    vb, off = vocab_arrays([b"a", b"aa"])
    docs = [b"a" * n for n in (1, 2, 255, 256, 257, 5000, 40001)]
    check_unigram(ctx, vb, off, [-1.0, -1.5], 2, -30.0, docs, chunk=256)
    assert ctx.stats()["unigram_fix"]["bytes"] > 0


def test_repairs_many_flagged(ctx):
    """The same parity runs over about 1,200 chunks of 256 bytes, more flagged
    chunks than the cooperative repair has CTAs: the warp-per-chunk repair
    takes them."""
    vb, off = vocab_arrays([b"a", b"aa"])
    check_unigram(ctx, vb, off, [-1.0, -1.5], 2, -30.0, [b"a" * 200001, b"a" * 100000, b"a" * 3], chunk=256)


def test_repairs_mixed(ctx):
    """Runs of 'a' between ordinary text: repairs start and stop inside documents."""
    rng = random.Random(3)
    toks, scores = random_model(rng, 500)
    toks += [b"a", b"aa"]
    scores += [-1.0, -1.5]
    vb, off = vocab_arrays(toks)
    docs = []
    for _ in range(8):
        parts = []
        for _ in range(rng.randint(1, 12)):
            if rng.random() < 0.4:
                parts.append(b"a" * rng.randint(1, 3000))
            else:
                parts.append(b"".join(rng.choice(ALPHA[1:]) for _ in range(rng.randint(1, 2000))))
        docs.append(b"".join(parts))
    check_unigram(ctx, vb, off, scores, len(toks), -30.0, docs, chunk=256)


def test_many_edges_per_position(ctx):
    """Tokens a, aa, ..., a^20: every position of a run of 'a' has 20 edges,
    more than a warp lists, so those runs are redone with a private ring."""
    rng = random.Random(4)
    toks = [b"a" * n for n in range(1, 21)] + [b"b", b"ba", b"ab"]
    scores = [f32(-rng.uniform(1.0, 30.0)) for _ in toks]
    vb, off = vocab_arrays(toks)
    docs = [b"a" * 3000, b"b" + b"a" * 700 + b"b" * 300 + b"a" * 1500, b"ab" * 900, b"a" * 33]
    check_unigram(ctx, vb, off, scores, len(toks), -40.0, docs, chunk=256)


@pytest.mark.parametrize("seed", range(3))
def test_wide_scores_thread_path(ctx, seed):
    """Scores beyond 32-bit units take the per-thread kernels (same answers)."""
    rng = random.Random(100 + seed)
    toks, _ = random_model(rng, 300)
    scores = [float(-rng.randint(1, 3) * 1_000_000_007) for _ in toks]   # integers above 2^31
    vb, off = vocab_arrays(toks)
    docs = [b"".join(rng.choice(ALPHA) for _ in range(rng.choice([1, 700, 2000]))) for _ in range(6)]
    check_unigram(ctx, vb, off, scores, len(toks), -9e9, docs, chunk=256)


def test_spread_beyond_32_bits(ctx):
    """Scores near 2^28 units and runs of unknown characters push a window's
    values more than 2^30 apart: those runs are redone in 64 bits."""
    vb, off = vocab_arrays([b"a", b"b", b"ab", b"ba"])
    sc = [-1.0, float(-(1 << 28)), -3.0, float(-(1 << 28) + 5)]
    rng = random.Random(8)
    docs = []
    for _ in range(6):
        parts = [rng.choice([b"a" * rng.randint(1, 400), b"z" * rng.randint(1, 300), b"ab" * rng.randint(1, 200),
                             "ş".encode() * rng.randint(1, 100)]) for _ in range(rng.randint(2, 10))]
        docs.append(b"".join(parts))
    check_unigram(ctx, vb, off, sc, 4, float(-(1 << 28) - 7), docs, chunk=256)


def test_long_tokens_wide_ring(ctx):
    """Tokens of up to 200 bytes take the 255-byte span (256-entry ring)."""
    rng = random.Random(9)
    toks, scores = random_model(rng, 300)
    base = b"".join(rng.choice(ALPHA[:4]) for _ in range(5000))
    for _ in range(200):
        s = rng.randrange(0, 4700)
        toks.append(base[s:s + rng.randint(64, 200)])
        scores.append(f32(-rng.uniform(5.0, 9.0)))
    vb, off = vocab_arrays(toks)
    docs = [base, base[::-1], base[17:3000] + base[100:900]]
    check_unigram(ctx, vb, off, scores, len(toks), -30.0, docs)


def test_unknown_characters(ctx):
    vb, off = vocab_arrays([b"a", b"b", b"ab", "ı".encode()])
    sc = [-1.0, -1.0, -1.5, -2.0]
    docs = ["aı€xbış€€aab".encode() * 50, "€".encode(), b"", "zzz".encode()]
    got = check_unigram(ctx, vb, off, sc, 4, -25.0, docs, chunk=256)
    assert (got == 4).sum() > 0


def test_many_small_documents(ctx):
    """20,000 documents of 0..60 bytes: the per-document index, repair and
    offset kernels over many documents, most of them one chunk or empty."""
    rng = random.Random(31)
    toks, scores = random_model(rng, 500)
    vb, off = vocab_arrays(toks)
    docs = [b"".join(rng.choice(ALPHA) for _ in range(rng.choice([0, 0, 1, 2, 7, 20, 60])))
            for _ in range(20_000)]
    check_unigram(ctx, vb, off, scores, len(toks), -30.0, docs, chunk=256)


def test_degenerate_inputs(ctx):
    vb, off = vocab_arrays([b"a", b"b"])
    check_unigram(ctx, vb, off, [-1.0, -1.0], 2, -9.0, [b""])
    check_unigram(ctx, vb, off, [-1.0, -1.0], 2, -9.0, [b"", b"", b"a", b""])
    trie = ctx.trie_build(vb, off)
    model = ctx.unigram(trie, [-1.0, -1.0], 2, -9.0)
    ids, id_off = ctx.unigram_encode(model, dev_u8(b"ab"), torch.zeros(1, dtype=torch.int64, device="cuda"))
    assert ids.numel() == 0 and id_off.cpu().tolist() == [0]


def test_errors(ctx):
    import bpe_trie_encode_gb300 as bt
    vb, off = vocab_arrays([b"a", b"b"])
    trie = ctx.trie_build(vb, off)
    with pytest.raises(bt.BpeError):
        ctx.unigram(trie, [-1.0, float("nan")], 2, -9.0)
    with pytest.raises(bt.BpeError):
        ctx.unigram(trie, [-1.0, 1e-300], 2, -9.0)    # needs more than 62 fraction bits
    with pytest.raises(bt.BpeError):
        ctx.unigram(trie, [-1.0], 2, -9.0)            # one score per token
    model = ctx.unigram(trie, [-1.0, -1.0], 2, -9.0)
    with pytest.raises(bt.BpeError) as e:              # 70 continuation bytes: no edge spans them
        ctx.unigram_encode(model, dev_u8(b"a" + b"\x80" * 70 + b"b"))
    assert e.value.name == "INVALID_ARG"
    with pytest.raises(bt.BpeError) as e:              # no token can start a document
        ctx.unigram_encode(model, dev_u8(b"\x80ab"))
    assert e.value.name == "INVALID_ARG"
    with pytest.raises(oracle.OracleError):             # (the recurrence reaches nothing either)
        oracle.Trie(vb, off).unigram_encode(b"\x80ab", [-1.0, -1.0], 2, -9.0)
    with pytest.raises(bt.BpeError) as e:
        ctx.unigram_encode(model, dev_u8(b"abab"), capacity=2)
    assert e.value.name == "CAPACITY"
    fine = ctx.unigram(trie, [-0.1, -1.0], 2, -0.5)    # 55 fraction bits: documents under 128 bytes
    assert ctx.unigram_encode(fine, dev_u8(b"ab" * 30))[0].numel() == 60
    with pytest.raises(bt.BpeError):
        ctx.unigram_encode(fine, dev_u8(b"ab" * 100))
    # 'a' ends inside a character: a 41-byte <unk>, then 'b'
    check_unigram(ctx, vb, off, [-1.0, -1.0], 2, -9.0, [b"a" + b"\x80" * 40 + b"b"])


def test_bounded_wait_times_out(ctx):
    """A scan tile that never publishes: the tiles after it give up their
    bounded wait, the call returns TIMEOUT, and the context keeps working."""
    import bpe_trie_encode_gb300 as bt
    from bpe_trie_encode_gb300 import _capi
    rng = random.Random(12)
    toks, scores = random_model(rng, 300)
    vb, off = vocab_arrays(toks)
    data = b"".join(rng.choice(ALPHA) for _ in range(400_000))   # about 2,000 chunks: 8 scan tiles
    trie = ctx.trie_build(vb, off)
    model = ctx.unigram(trie, scores, len(toks), -30.0)
    ctx.set_option(_capi.BPE_OPT_TEST_STALL_TILE, 1)
    try:
        with pytest.raises(bt.BpeError) as e:
            ctx.unigram_encode(model, dev_u8(data))
        assert e.value.name == "TIMEOUT"
    finally:
        ctx.set_option(_capi.BPE_OPT_TEST_STALL_TILE, -1)
    check_unigram(ctx, vb, off, scores, len(toks), -30.0, [data[:50_000]])


def unigram_workload(ctx, golden, name, data, doc_off, vb, off):
    g = golden[name]
    assert sha(data) == g["text_sha256"]
    scores = synth.unigram_scores(off.size - 1)
    assert sha(scores) == g["scores_sha256"]
    trie = ctx.trie_build(vb, off)
    model = ctx.unigram(trie, scores, g["unk_id"], g["unk_score"])
    ids, id_off = ctx.unigram_encode(model, dev_u8(data), torch.from_numpy(doc_off.astype(np.int64)).cuda())
    assert ids.numel() == g["n_ids"]
    assert ids[:16].cpu().tolist() == g["ids_head"]
    assert sha(ids.cpu().numpy()) == g["ids_sha256"]
    assert sha(id_off.cpu().numpy().astype(np.uint64)) == g["id_off_sha256"]


@pytest.fixture(scope="module")
def batch_vocab():
    big = synth.corpus("large")
    vb, off = synth.substring_vocab(big)
    return vb, off


def test_batch_workload(ctx, golden, batch_vocab):
    """512 documents of >= 64 KiB, 250,000-token vocabulary, synthetic scores."""
    data, doc_off = synth.batch_documents()
    unigram_workload(ctx, golden, "unigram", data, doc_off, *batch_vocab)


def test_long_document(ctx, golden, batch_vocab):
    """One 64 MiB document: every chunk but the first few runs speculatively."""
    data = synth.corpus("enc", 64 << 20)
    unigram_workload(ctx, golden, "unigram_doc", data, np.array([0, data.size], dtype=np.uint64), *batch_vocab)


def test_wide_windows(ctx):
    """Scores of a fine unit with many short tokens: a 63-byte window's values
    lie more than 2^30 units apart, so the forward runs (and the repairs of
    the parity runs) take 64-bit windows; the result is still exact."""
    # unit 2^-23 (from b's score); every score within the warp kernels' 2^29 units
    sc = [float(np.float32(x)) for x in (-20.0, -30.5, -1.0000001)]
    assert sc[2] != -1.0
    vb, off = vocab_arrays([b"a", b"aa", b"b"])
    docs = [b"a" * 5000, b"ab" * 3000, b"b" * 700, b"a" * 40001, b""]
    check_unigram(ctx, vb, off, sc, 3, -40.0, docs, chunk=256)
    assert ctx.stats()["unigram_wide"]["launches"] > 0
    # the smoke's model: the tiny corpus's 64 merges, Zipf scores over 320 tokens
    merges, _ = oracle.train_words(oracle.pretokenize(synth.corpus("tiny", 32 * 1024)), 64)
    vb, off = oracle.vocab_from_merges(merges)
    n_tok = off.size - 1
    scores = synth.unigram_scores(n_tok)
    unk = synth.unigram_unk_score(scores)
    lex = synth.lexicon("tiny")
    docs = [lex.corpus(7, 16 * 1024).tobytes()] + [lex.corpus(20 + d, 3000 + 997 * d).tobytes() for d in range(6)]
    check_unigram(ctx, vb, off, scores, n_tok, unk, docs)
    assert ctx.stats()["unigram_wide"]["launches"] > 0
