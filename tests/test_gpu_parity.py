"""GPU parity: the CUDA path against the CPU oracle, bit for bit.

Small cases are compared element by element with the oracle run live; the
five workloads are compared with the oracle's recorded results
(tests/golden/workloads.json, written by tests/golden/make_golden.py), by
SHA-256 of the full outputs.  All calls go through the C ABI.
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

WS = 0x10000
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def sha(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


@pytest.fixture(scope="module")
def golden():
    with open(os.path.join(GOLDEN, "workloads.json")) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def ctx():
    import bpe_trie_encode_gb300 as bt
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    c = bt.Context(0)
    yield c
    c.close()


def dev_u8(a) -> "torch.Tensor":
    a = np.frombuffer(a, dtype=np.uint8) if isinstance(a, (bytes, bytearray)) else a
    return torch.from_numpy(np.ascontiguousarray(a).copy()).cuda()


def dev_sym(a) -> "torch.Tensor":
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32).copy()).cuda()


def host_u32(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def rand_bytes(rng, n, alphabet):
    return bytes(rng.choice(alphabet) for _ in range(n))


# ------------------------------------------------------------- pretokenize --
@pytest.mark.parametrize("n", [0, 1, 2, 15, 16, 17, 31, 33, 1000, (1 << 20) + 7])
def test_pretokenize_sizes(ctx, n):
    rng = np.random.default_rng(n)
    data = rng.integers(0, 256, n, dtype=np.uint8)
    data[rng.random(n) < 0.3] = ord("a")   # runs of one class
    got = host_u32(ctx.pretokenize(dev_u8(data)))
    assert np.array_equal(got, oracle.pretokenize(data))


def test_pretokenize_unaligned_and_all_bytes(ctx):
    data = np.arange(256 * 40, dtype=np.uint32).astype(np.uint8)
    d = dev_u8(np.concatenate([np.array([7], dtype=np.uint8), data]))
    got = host_u32(ctx.pretokenize(d[1:]))            # 1-byte offset: scalar path
    assert np.array_equal(got, oracle.pretokenize(data))


def test_pretokenize_corpus(ctx, golden):
    text = synth.corpus("med")
    assert sha(text) == golden["med"]["corpus_sha256"], "generator output differs on this machine"
    got = host_u32(ctx.pretokenize(dev_u8(text)))
    assert sha(got) == golden["med"]["symbols_sha256"]


# ------------------------------------------------------------------- train --
def check_train(ctx, sym, n_merges, **kw):
    m, f = ctx.train(dev_sym(sym), n_merges)
    wm, wf = oracle.train_stream(sym, n_merges)
    assert np.array_equal(m, wm), (m[:5], wm[:5])
    assert np.array_equal(host_u32(f), wf)
    return m


def test_train_worked_examples(ctx):
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        ex = json.load(f)
    for e in ex["train"]:
        sym = oracle.pretokenize(e["text"].encode())
        m, fin = ctx.train(dev_sym(sym), e["n_merges"])
        assert m.tolist() == e["merges"], e["name"]
        assert [[x & 0xFFFF, x >> 16] for x in host_u32(fin).tolist()] == e["final"], e["name"]


@pytest.mark.parametrize("seed", range(16))
def test_train_random_small(ctx, seed):
    rng = random.Random(seed)
    alphabets = [b"ab", b"aab ", b"abc a.\n1", b"a", b"ab1 ", bytes(range(97, 123)) + b" ."]
    n = rng.choice([2, 3, 5, 100, 2047, 2048, 2049, 4096 + 3, 9000])
    text = rand_bytes(rng, n, alphabets[seed % len(alphabets)])
    check_train(ctx, oracle.pretokenize(text), 60)


@pytest.mark.parametrize("n", [4096 * 3 - 1, 4096 * 3, 4096 * 3 + 1, 1_000_001, 5_000_001])
def test_train_identical_runs_cross_tiles(ctx, n):
    # one run of identical letters spans many 4096-symbol tiles (at 5M, several
    # tiles per CTA range): leftmost-first pairing must carry its parity across
    # every tile and range boundary
    text = b"a" * n + b" " + b"a" * (n // 3) + b".bb" + b"b" * 4097
    check_train(ctx, oracle.pretokenize(text), 12)


@pytest.mark.parametrize("mode", ["two_pass", "lookback", "tiles", "persistent"])
@pytest.mark.parametrize("case", ["runs", "random", "tiny", "med"])
def test_train_merge_variants_agree(ctx, golden, case, mode):
    # the full-stream loops -- two-pass merge, single-pass merge (decoupled
    # look-back), gapped tiles, persistent two-pass -- give the same merges
    # and stream as the default occurrence-list loop
    import bpe_trie_encode_gb300 as bt
    ctx.set_option(bt.BPE_OPT_MERGE, {"lookback": bt.BPE_MERGE_LOOKBACK, "tiles": bt.BPE_MERGE_TILES,
                                      "persistent": bt.BPE_MERGE_TWO_PASS, "two_pass": bt.BPE_MERGE_TWO_PASS}[mode])
    ctx.set_option(bt.BPE_OPT_PERSISTENT, 1 if mode == "persistent" else 0)
    try:
        if case == "runs":
            text = b"a" * 1_000_001 + b" " + b"a" * 4097 + b".bb" + b"b" * 4097
            check_train(ctx, oracle.pretokenize(text), 12)
        elif case == "random":
            for seed in range(4):
                rng = random.Random(100 + seed)
                check_train(ctx, oracle.pretokenize(rand_bytes(rng, 9000 + 4096 * seed, b"aab c.")), 60)
        elif case == "tiny":
            m, f = ctx.train(dev_sym(oracle.pretokenize(synth.corpus("tiny"))), 256)
            assert sha(m.astype(np.uint32)) == golden["tiny"]["merges_sha256"]
            assert sha(host_u32(f)) == golden["tiny"]["final_sha256"]
        else:   # the medium workload with checkpoints: streams after 1, 100 and 1,000 merges
            g = golden["med"]
            sym = ctx.pretokenize(dev_u8(synth.corpus("med")))
            m, f = ctx.train(sym, g["n_merges"])
            assert sha(m.astype(np.uint32)) == g["merges_sha256"] and sha(host_u32(f)) == g["final_sha256"]
            for k in (1, 100, 1000):
                _, fk = ctx.train(sym, k)
                assert sha(host_u32(fk)) == g["checkpoints"][str(k)]["sha256"], k
    finally:
        ctx.set_option(bt.BPE_OPT_MERGE, bt.BPE_MERGE_LISTS)
        ctx.set_option(bt.BPE_OPT_PERSISTENT, 0)


@pytest.mark.parametrize("mode", ["auto", "auto-eager", "always", "always-eager"])
@pytest.mark.parametrize("case", ["runs", "random", "alternating", "tiny", "med"])
def test_train_sparse_modes_agree(ctx, golden, case, mode):
    # the two-pass loop's occurrence-driven merges (tombstones, exact
    # deltas, compaction) after the automatic switch and from merge 0, with
    # graphs and with host launches, give the oracle's merges and final
    # stream; the automatic switch comes at the first poll (merge 96), so
    # only the longer cases exercise it, while merge 0 on puts million-symbol
    # runs through the l == r walk.  Where the mode must have engaged, the
    # call's statistics show its scan kernel.
    import bpe_trie_encode_gb300 as bt
    ctx.set_option(bt.BPE_OPT_MERGE, bt.BPE_MERGE_TWO_PASS)
    ctx.set_option(bt.BPE_OPT_SPARSE_MERGE, 2 if mode.startswith("always") else 1)
    ctx.set_option(bt.BPE_OPT_GRAPH, 0 if mode.endswith("eager") else 1)

    def engaged():
        st = ctx.stats()
        return st.get("merge_scan", {}).get("launches", 0) > 0

    try:
        if case == "runs":
            text = b" ".join(b"a" * n for n in list(range(1, 40)) + [1001, 4097, 64, 65]) + b"aaaa bbbb abab" * 3
            check_train(ctx, oracle.pretokenize(text), 60)
            check_train(ctx, oracle.pretokenize(b"a" * 1_000_001 + b" " + b"a" * 4097 + b".bb" + b"b" * 4097), 12)
        elif case == "random":
            for seed in range(4):
                rng = random.Random(200 + seed)
                alphabet = [b"ab", b"aab ", b"aab c.", b"abc a.\n1"][seed]
                check_train(ctx, oracle.pretokenize(rand_bytes(rng, 9000 + 4096 * seed, alphabet)), 150)
            if mode.startswith("always"):
                assert engaged()
        elif case == "alternating":
            check_train(ctx, oracle.pretokenize(b"ab" * 50000 + b" " + b"ba" * 777), 40)
            if mode.startswith("always"):
                assert engaged()
        elif case == "tiny":
            m, f = ctx.train(dev_sym(oracle.pretokenize(synth.corpus("tiny"))), 256)
            assert sha(m.astype(np.uint32)) == golden["tiny"]["merges_sha256"]
            assert sha(host_u32(f)) == golden["tiny"]["final_sha256"]
            assert engaged()   # the best count falls below 1/64 of the input within the first windows
        else:
            g = golden["med"]
            sym = ctx.pretokenize(dev_u8(synth.corpus("med")))
            m, f = ctx.train(sym, g["n_merges"])
            assert engaged()
            assert sha(m.astype(np.uint32)) == g["merges_sha256"] and sha(host_u32(f)) == g["final_sha256"]
            for k in (1, 100, 1000):
                _, fk = ctx.train(sym, k)
                assert sha(host_u32(fk)) == g["checkpoints"][str(k)]["sha256"], k
    finally:
        ctx.set_option(bt.BPE_OPT_SPARSE_MERGE, 0)
        ctx.set_option(bt.BPE_OPT_GRAPH, 1)
        ctx.set_option(bt.BPE_OPT_MERGE, bt.BPE_MERGE_LISTS)


@pytest.mark.parametrize("fcap", [1, 2, 7, 64])
def test_train_lists_small_frontier(ctx, golden, fcap):
    # the occurrence-list loop with a tiny argmax frontier: it overflows and
    # is rescanned over and over, and still gives the oracle's merges
    import bpe_trie_encode_gb300 as bt
    ctx.set_option(bt.BPE_OPT_LIST_FRONTIER, fcap)
    try:
        rng = random.Random(fcap)
        check_train(ctx, oracle.pretokenize(rand_bytes(rng, 20000, b"abcde fgh.")), 300)
        m, f = ctx.train(dev_sym(oracle.pretokenize(synth.corpus("tiny"))), 256)
        assert sha(m.astype(np.uint32)) == golden["tiny"]["merges_sha256"]
        assert sha(host_u32(f)) == golden["tiny"]["final_sha256"]
    finally:
        ctx.set_option(bt.BPE_OPT_LIST_FRONTIER, 0)


@pytest.mark.parametrize("tail", [0, 1, 64, -1])
def test_train_lists_tail_modes(ctx, golden, tail):
    # merges on all SMs only (0), a single-CTA tail that takes only lists of
    # one or 64 entries (mixing the two paths merge by merge), and the default
    import bpe_trie_encode_gb300 as bt
    ctx.set_option(bt.BPE_OPT_LIST_TAIL, tail)
    try:
        rng = random.Random(300 + tail)
        check_train(ctx, oracle.pretokenize(rand_bytes(rng, 30000, b"aab c.")), 200)
        # late merges of this text have short lists: the default tail takes some, none when off
        tail_merges = ctx.stats()["merge_tail"]["launches"]
        if tail == 0:
            assert tail_merges == 0
        elif tail == -1:
            assert tail_merges > 0
        check_train(ctx, oracle.pretokenize(b"a" * 5001 + b" " + b"ab" * 3000 + b" " + b"a" * 7), 30)
        g = golden["med"]
        sym = ctx.pretokenize(dev_u8(synth.corpus("med")))
        m, f = ctx.train(sym, g["n_merges"])
        assert sha(m.astype(np.uint32)) == g["merges_sha256"] and sha(host_u32(f)) == g["final_sha256"]
    finally:
        ctx.set_option(bt.BPE_OPT_LIST_TAIL, -1)


def test_train_lists_unaligned_and_wide_ids(ctx):
    # an input that starts 4 bytes into an allocation (the count's scalar
    # path), an input without WORD_START at position 0, and ids past one byte
    # (handed to the two-pass loop) all match the oracle
    sym = oracle.pretokenize(synth.corpus("tiny", 30000))
    d = dev_sym(np.concatenate([np.array([7], dtype=np.uint32), sym]))
    m, f = ctx.train(d[1:], 100)
    wm, wf = oracle.train_stream(sym, 100)
    assert np.array_equal(m, wm) and np.array_equal(host_u32(f), wf)
    s2 = sym.copy()
    s2[0] &= ~np.uint32(WS)
    check_train(ctx, s2, 80)
    wide = sym.copy()
    wide[::7] = (wide[::7] & np.uint32(WS)) | np.uint32(65000)   # no merge of these 50 makes id 65000
    check_train(ctx, wide, 50)


def test_train_lists_long_runs(ctx):
    # runs of one symbol (l == r merges walk each run once from its first
    # valid start) next to runs of a merged token, odd and even lengths
    parts = [b"a" * n for n in (1, 2, 3, 4, 5, 31, 32, 33, 1000, 1001, 65537)]
    text = b" ".join(parts) + b" " + b"ab" * 3001 + b"." + b"aab" * 999 + b" " + b"abab" * 777
    check_train(ctx, oracle.pretokenize(text), 40)


def test_train_alternating_and_ties(ctx):
    check_train(ctx, oracle.pretokenize(b"ab" * 50000 + b" " + b"ba" * 777), 20)
    check_train(ctx, oracle.pretokenize(b"ab cd ef gh ba dc fe hg"), 10)


def test_train_degenerate(ctx):
    m, f = ctx.train(dev_sym(oracle.pretokenize(b"a")), 5)
    assert m.shape == (0, 4) and host_u32(f).tolist() == [97 | WS]
    m, f = ctx.train(dev_sym(oracle.pretokenize(b"abc")), 0)
    assert m.shape == (0, 4) and host_u32(f).size == 3
    m, f = ctx.train(dev_sym(oracle.pretokenize(b"a1 .\n")), 5)   # no countable pair
    assert m.shape == (0, 4)


def test_train_rejects_too_many_merges(ctx):
    import bpe_trie_encode_gb300 as bt
    with pytest.raises(bt.BpeError) as e:
        ctx.train(dev_sym(oracle.pretokenize(b"abc")), 65281)
    assert e.value.name == "ID_OVERFLOW"


def test_train_table_full_is_reported(ctx):
    import bpe_trie_encode_gb300 as bt
    rng = np.random.default_rng(5)
    data = rng.integers(97, 123, 200000, dtype=np.uint8)   # ~676 distinct pairs ... grows
    sym = oracle.pretokenize(data)
    ctx.set_option(bt.BPE_OPT_MERGE, bt.BPE_MERGE_TWO_PASS)   # the loop with the sized hash table
    ctx.set_option(bt.BPE_OPT_TABLE_LOG2, 12)
    try:
        with pytest.raises(bt.BpeError) as e:
            ctx.train(dev_sym(sym), 400)
        assert e.value.name == "TABLE_FULL"
    finally:
        ctx.set_option(bt.BPE_OPT_TABLE_LOG2, 0)
        ctx.set_option(bt.BPE_OPT_MERGE, bt.BPE_MERGE_LISTS)
    check_train(ctx, sym[:5000], 30)   # the context is still usable


@pytest.mark.parametrize("mode", ["graph", "eager", "profile"])
def test_train_launch_modes_agree(ctx, golden, mode):
    import bpe_trie_encode_gb300 as bt
    sym = oracle.pretokenize(synth.corpus("tiny"))
    ctx.set_option(bt.BPE_OPT_GRAPH, 1 if mode == "graph" else 0)
    ctx.set_option(bt.BPE_OPT_PROFILE, 1 if mode == "profile" else 0)
    try:
        m, f = ctx.train(dev_sym(sym), 256)
    finally:
        ctx.set_option(bt.BPE_OPT_GRAPH, 1)
        ctx.set_option(bt.BPE_OPT_PROFILE, 0)
    g = golden["tiny"]
    assert sha(m.astype(np.uint32)) == g["merges_sha256"]
    assert sha(host_u32(f)) == g["final_sha256"]
    if mode == "profile":
        st = ctx.stats()
        # every merge ran either in the single-CTA tail or on all SMs (scan + apply)
        assert st["pair_count"]["ms"] > 0 and st["merge_tail"]["launches"] + st["merge_scan"]["launches"] == 256
        assert st["merge_apply"]["launches"] == st["merge_scan"]["launches"] and st["compact"]["launches"] == 1


def train_workload(ctx, golden, name, checkpoints):
    g = golden[name]
    text = synth.corpus(name)
    assert sha(text) == g["corpus_sha256"], "generator output differs on this machine"
    sym = ctx.pretokenize(dev_u8(text))
    assert sha(host_u32(sym)) == g["symbols_sha256"]
    m, f = ctx.train(sym, g["n_merges"])
    assert m.shape[0] == g["n_done"]
    assert m[:8].tolist() == g["merges_head"]
    assert sha(m.astype(np.uint32)) == g["merges_sha256"]
    assert f.numel() == g["n_final"] and sha(host_u32(f)) == g["final_sha256"]
    for k in checkpoints:
        _, fk = ctx.train(sym, k)
        ck = g["checkpoints"][str(k)]
        assert fk.numel() == ck["n"] and sha(host_u32(fk)) == ck["sha256"], k
    return m


def test_train_tiny_workload(ctx, golden):
    train_workload(ctx, golden, "tiny", [0, 1, 2, 10, 100])


def test_train_med_workload(ctx, golden):
    train_workload(ctx, golden, "med", [1, 2, 10, 100, 1000])


@pytest.fixture(scope="module")
def large_merges(ctx, golden):
    """The large workload's merge table from the GPU, accepted only when it is
    bit-identical (by hash) to the oracle's recorded table."""
    return train_workload(ctx, golden, "large", [10, 1000])


def test_train_large_workload(large_merges, golden):
    assert large_merges.shape[0] == golden["large"]["n_done"]


# ------------------------------------------------------------------ encode --
def vocab_arrays(tokens):
    vb = b"".join(tokens)
    off = np.cumsum([0] + [len(t) for t in tokens]).astype(np.uint64)
    return np.frombuffer(vb, dtype=np.uint8).copy(), off


def check_encode(ctx, vb, off, docs, chunk=None):
    import bpe_trie_encode_gb300 as bt
    data = b"".join(docs)
    doc_off = np.cumsum([0] + [len(d) for d in docs]).astype(np.int64)
    trie = ctx.trie_build(vb, off)
    if chunk:
        ctx.set_option(bt.BPE_OPT_CHUNK, chunk)
    try:
        ids, id_off = ctx.encode(trie, dev_u8(data) if data else torch.empty(0, dtype=torch.uint8, device="cuda"),
                                 torch.from_numpy(doc_off).cuda())
    finally:
        ctx.set_option(bt.BPE_OPT_CHUNK, 256)
    wids, woff = oracle.Trie(vb, off).encode(data, doc_off.astype(np.uint64))
    assert np.array_equal(ids.cpu().numpy(), wids)
    assert np.array_equal(id_off.cpu().numpy().astype(np.uint64), woff)
    return ids


def test_encode_worked_examples(ctx):
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        ex = json.load(f)
    for e in ex["encode"]:
        toks = [bytes([b]) for b in range(256)] + [s.encode() for s in e["vocab_extra"]]
        vb, off = vocab_arrays(toks)
        ids = check_encode(ctx, vb, off, [e["text"].encode()])
        assert ids.cpu().tolist() == e["ids"], e["name"]


@pytest.mark.parametrize("seed", range(8))
def test_encode_random_vocab_ragged_docs(ctx, seed):
    rng = random.Random(seed)
    alpha = b"ab c" if seed % 2 else bytes(range(97, 103)) + b" ."
    toks = [bytes([b]) for b in range(256)]
    toks += [rand_bytes(rng, rng.randrange(2, 40), alpha) for _ in range(rng.randrange(5, 3000))]
    vb, off = vocab_arrays(toks)
    docs = [rand_bytes(rng, rng.choice([0, 1, 5, 127, 128, 129, 1000, 5000]), alpha) for _ in range(rng.randrange(1, 40))]
    check_encode(ctx, vb, off, docs)


@pytest.mark.parametrize("chunk", [64, 96, 128, 256])
def test_encode_chunk_sizes_agree(ctx, chunk):
    rng = random.Random(11)
    toks = [bytes([b]) for b in range(256)] + [rand_bytes(rng, rng.randrange(2, 30), b"abc ") for _ in range(500)]
    vb, off = vocab_arrays(toks)
    docs = [rand_bytes(rng, 20000, b"abc ") for _ in range(3)]
    check_encode(ctx, vb, off, docs, chunk=chunk)


def test_encode_tokens_longer_than_chunks(ctx):
    # tokens of 300 bytes make the previous chunk's last token cover whole chunks
    toks = [bytes([b]) for b in range(256)] + [b"x" * 300, b"x" * 299 + b"y", b"xy" * 100]
    vb, off = vocab_arrays(toks)
    docs = [b"x" * 5000 + b"y" + b"xy" * 700, b"x" * 299 + b"y" * 3]
    check_encode(ctx, vb, off, docs)


def test_encode_parses_that_never_meet(ctx):
    # with tokens {a, aa} parses started one byte apart never share a boundary:
    # every chunk needs the repair walk
    toks = [bytes([b]) for b in range(256)] + [b"aa", b"ab"]
    vb, off = vocab_arrays(toks)
    check_encode(ctx, vb, off, [b"a" * 100001 + b"b", b"a" * 1000, b"ba" * 3000])


def parity_shift_docs(rng, n_docs, lengths, c_rate):
    """Documents over {a, c} for the vocabulary {c, a, aa}: a 'c' moves the
    parse of the 'a' runs after it to the other parity, so a speculative parse
    from an even chunk start never meets the true one.  Chunks are flagged
    where the parity flips, and chains run until the next flip."""
    docs = []
    for _ in range(n_docs):
        n = rng.choice(lengths)
        docs.append(bytes(99 if (i == 0 or rng.random() < c_rate) else 97 for i in range(n)))
    return docs


PARITY_VOCAB = [bytes([b]) for b in range(256)] + [b"aa"]


@pytest.mark.parametrize("n_docs,lengths,c_rate", [
    (3000, [129, 300, 513], 0.0),      # one flag per document, under the flag list's capacity
    (5000, [300], 0.0),                # more flags than the list holds: sequential repair
    (4, [3000, 20000], 0.0),           # chains much longer than a walker records
    (64, [1, 2, 127, 128, 129, 5000], 0.004),   # flips at random: flagged chunks inside chains
])
def test_encode_repair_paths(ctx, n_docs, lengths, c_rate):
    rng = random.Random(n_docs * 7 + len(lengths))
    vb, off = vocab_arrays(PARITY_VOCAB)
    check_encode(ctx, vb, off, parity_shift_docs(rng, n_docs, lengths, c_rate))


def stream_encode(ctx, vb, off, text, cuts, trie=None):
    import bpe_trie_encode_gb300 as bt
    trie = trie or ctx.trie_build(vb, off)
    st = bt.Stream(ctx, trie)
    out = []
    bounds = [0] + sorted(cuts) + [len(text)]
    for i in range(len(bounds) - 1):
        piece = text[bounds[i]:bounds[i + 1]]
        d = dev_u8(piece) if piece else torch.empty(0, dtype=torch.uint8, device="cuda")
        out.append(st.push(d, last=(i == len(bounds) - 2)).cpu().numpy())
    st.close()
    return np.concatenate(out) if out else np.zeros(0, np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_encode_stream_slices_equal_whole_document(ctx, seed):
    # the ids of a document pushed in slices (empty, single-byte, shorter than
    # the longest token, cutting tokens) equal the oracle's on the whole text
    rng = random.Random(1000 + seed)
    alpha = b"ab c" if seed % 2 else bytes(range(97, 103)) + b" ."
    toks = [bytes([b]) for b in range(256)]
    toks += [rand_bytes(rng, rng.randrange(2, 60), alpha) for _ in range(rng.randrange(50, 2000))]
    vb, off = vocab_arrays(toks)
    text = rand_bytes(rng, rng.choice([0, 1, 7, 3000, 70000]), alpha)
    cuts = sorted(rng.randrange(0, len(text) + 1) for _ in range(rng.randrange(0, 40)))
    cuts += [c for c in cuts[:3]]   # repeated cuts: empty slices
    ids = stream_encode(ctx, vb, off, text, cuts)
    want, _ = oracle.Trie(vb, off).encode(text, np.array([0, len(text)], dtype=np.uint64))
    assert np.array_equal(ids, want)


def test_encode_stream_long_tokens_and_reuse(ctx):
    import bpe_trie_encode_gb300 as bt
    toks = [bytes([b]) for b in range(256)] + [b"x" * 300, b"x" * 299 + b"y", b"xy" * 100, b"aa"]
    vb, off = vocab_arrays(toks)
    trie = ctx.trie_build(vb, off)
    o = oracle.Trie(vb, off)
    st = bt.Stream(ctx, trie)
    for text, step in ((b"x" * 5000 + b"y" + b"xy" * 700, 7), (b"c" + b"a" * 2000, 5), (b"x" * 299, 1000)):
        got = []
        for i in range(0, len(text), step):   # slices far shorter than the longest token
            got.append(st.push(dev_u8(text[i:i + step])).cpu().numpy())
        got.append(st.push(torch.empty(0, dtype=torch.uint8, device="cuda"), last=True).cpu().numpy())
        want, _ = o.encode(text, np.array([0, len(text)], dtype=np.uint64))
        assert np.array_equal(np.concatenate(got), want)   # the stream is reused after each last push
    st.close()


def test_encode_stream_learned_vocab_megabytes(ctx, golden):
    merges, _ = oracle.train_words(oracle.pretokenize(synth.corpus("tiny")), 256)
    vb, off = oracle.vocab_from_merges(merges)
    text = synth.corpus("med")[: 6 << 20].tobytes()
    cuts = list(range(1 << 20, len(text), (1 << 20) + 12345))
    ids = stream_encode(ctx, vb, off, text, cuts)
    want, _ = oracle.Trie(vb, off).encode(text, np.array([0, len(text)], dtype=np.uint64))
    assert np.array_equal(ids, want)


@pytest.mark.parametrize("slice_bytes", [4096, 5000, 1 << 20])
def test_encode_host_pipeline(ctx, slice_bytes):
    # host buffers in, host buffers out: groups of whole documents and
    # documents longer than a slice, with empty documents mixed in
    import bpe_trie_encode_gb300 as bt
    rng = random.Random(slice_bytes)
    alpha = b"ab c."
    toks = [bytes([b]) for b in range(256)] + [rand_bytes(rng, rng.randrange(2, 40), alpha) for _ in range(800)]
    vb, off = vocab_arrays(toks)
    docs = [rand_bytes(rng, rng.choice([0, 1, 100, 3000, 20000, 70000]), alpha) for _ in range(60)]
    data = b"".join(docs)
    doc_off = np.cumsum([0] + [len(d) for d in docs]).astype(np.int64)
    trie = ctx.trie_build(vb, off)
    h = torch.from_numpy(np.frombuffer(data, dtype=np.uint8).copy()).pin_memory()
    ids, id_off = bt.encode_host(ctx, trie, h, torch.from_numpy(doc_off), slice_bytes=slice_bytes)
    wids, woff = oracle.Trie(vb, off).encode(data, doc_off.astype(np.uint64))
    assert np.array_equal(ids.numpy(), wids)
    assert np.array_equal(id_off.numpy().astype(np.uint64), woff)


def test_encode_capacity_error(ctx):
    import bpe_trie_encode_gb300 as bt
    toks = [bytes([b]) for b in range(256)]
    vb, off = vocab_arrays(toks)
    trie = ctx.trie_build(vb, off)
    with pytest.raises(bt.BpeError) as e:
        ctx.encode(trie, dev_u8(b"hello world"), capacity=5)
    assert e.value.name == "CAPACITY" and "11 ids" in str(e.value)


def test_encode_rejects_bad_inputs(ctx):
    import bpe_trie_encode_gb300 as bt
    partial = ctx.trie_build(*vocab_arrays([b"a", b"b"]))   # builds (Unigram can use it); greedy refuses it
    with pytest.raises(bt.BpeError) as e:
        ctx.encode(partial, dev_u8(b"ab"))
    assert e.value.name == "INVALID_ARG"
    trie = ctx.trie_build(*vocab_arrays([bytes([b]) for b in range(256)]))
    with pytest.raises(bt.BpeError) as e:
        ctx.encode(trie, dev_u8(b"abcdef"), torch.tensor([0, 4, 2], dtype=torch.int64, device="cuda"))
    assert e.value.name == "INVALID_ARG"


def test_encode_learned_vocab_tiny(ctx, golden):
    sym = oracle.pretokenize(synth.corpus("tiny"))
    wm, _ = oracle.train_words(sym, 256)
    vb, off = oracle.vocab_from_merges(wm)
    text = synth.lexicon("tiny").corpus(42, 300000)
    check_encode(ctx, vb, off, [text.tobytes()[:100000], text.tobytes()[100000:]])


def test_encode_large_vocab_workload(ctx, large_merges, golden):
    """1 GiB of text with the 32,256-token vocabulary learned on the large
    corpus (the merge table was verified against the oracle's by hash)."""
    g = golden["enc"]
    vb, off = oracle.vocab_from_merges(large_merges)
    assert sha(np.asarray(vb, dtype=np.uint8)) == g["vocab_sha256"]
    text = synth.corpus("enc")
    assert sha(text) == g["text_sha256"]
    trie = ctx.trie_build(vb, off)
    d = dev_u8(text)
    del text
    ids, id_off = ctx.encode(trie, d)
    assert ids.numel() == g["n_ids"]
    assert sha(ids.cpu().numpy()) == g["ids_sha256"]
    assert sha(id_off.cpu().numpy().astype(np.uint64)) == g["id_off_sha256"]
    # the same from host memory: 64 MiB slices streamed with the parse carried across them
    import bpe_trie_encode_gb300 as bt
    h = d.cpu().pin_memory()
    del d, ids
    hids, hoff = bt.encode_host(ctx, trie, h)
    assert hids.numel() == g["n_ids"] and sha(hids.numpy()) == g["ids_sha256"]
    assert sha(hoff.numpy().astype(np.uint64)) == g["id_off_sha256"]


def test_encode_batch_workload(ctx, golden):
    """512 documents of >= 64 KiB, 250,000-token substring vocabulary."""
    g = golden["batch"]
    big = synth.corpus("large")
    vb, off = synth.substring_vocab(big)
    del big
    assert sha(vb) == g["vocab_sha256"] and sha(off) == g["vocab_off_sha256"]
    data, doc_off = synth.batch_documents()
    assert sha(data) == g["text_sha256"]
    trie = ctx.trie_build(vb, off)
    ids, id_off = ctx.encode(trie, dev_u8(data), torch.from_numpy(doc_off.astype(np.int64)).cuda())
    assert ids.numel() == g["n_ids"]
    assert sha(ids.cpu().numpy()) == g["ids_sha256"]
    assert sha(id_off.cpu().numpy().astype(np.uint64)) == g["id_off_sha256"]


# ------------------------------------------------ bitmap-node trie layout --
@pytest.fixture
def bitmap_ctx(ctx):
    import bpe_trie_encode_gb300 as bt
    ctx.set_option(bt.BPE_OPT_TRIE_LAYOUT, bt.BPE_TRIE_BITMAP)
    yield ctx
    ctx.set_option(bt.BPE_OPT_TRIE_LAYOUT, bt.BPE_TRIE_DOUBLE_ARRAY)


@pytest.mark.parametrize("seed", range(4))
def test_bitmap_layout_random_vocab(bitmap_ctx, seed):
    test_encode_random_vocab_ragged_docs(bitmap_ctx, seed)


def test_bitmap_layout_edges(bitmap_ctx):
    # long tokens across chunks, parses that never meet (repair), the stream cut
    test_encode_tokens_longer_than_chunks(bitmap_ctx)
    test_encode_parses_that_never_meet(bitmap_ctx)
    test_encode_repair_paths(bitmap_ctx, 64, [1, 2, 127, 128, 129, 5000], 0.004)
    test_encode_stream_long_tokens_and_reuse(bitmap_ctx)
    test_encode_worked_examples(bitmap_ctx)


def test_bitmap_layout_batch_workload(bitmap_ctx, golden):
    test_encode_batch_workload(bitmap_ctx, golden)


# --------------------------------------------- word-frequency training path --
@pytest.fixture
def words_ctx(ctx):
    import bpe_trie_encode_gb300 as bt
    ctx.set_option(bt.BPE_OPT_TRAIN_WORDS, 1)
    yield ctx
    ctx.set_option(bt.BPE_OPT_TRAIN_WORDS, 0)


def test_words_worked_examples(words_ctx):
    test_train_worked_examples(words_ctx)


@pytest.mark.parametrize("seed", range(16))
def test_words_random_small(words_ctx, seed):
    test_train_random_small(words_ctx, seed)


@pytest.mark.parametrize("n", [2048 * 3 + 1, 1_000_001])
def test_words_identical_runs(words_ctx, n):
    test_train_identical_runs_cross_tiles(words_ctx, n)


def test_words_alternating_ties_degenerate(words_ctx):
    test_train_alternating_and_ties(words_ctx)
    test_train_degenerate(words_ctx)


def test_words_many_distinct_words(words_ctx):
    # every word distinct: the distinct-word table holds one entry per occurrence
    rng = np.random.default_rng(3)
    words = [bytes(rng.integers(97, 123, rng.integers(1, 9)).astype(np.uint8)) for _ in range(40000)]
    check_train(words_ctx, oracle.pretokenize(b" ".join(words)), 50)


def test_words_tiny_med_workloads(words_ctx, golden):
    train_workload(words_ctx, golden, "tiny", [0, 1, 10, 100])
    train_workload(words_ctx, golden, "med", [1, 100, 1000])


def test_words_large_workload(words_ctx, golden):
    train_workload(words_ctx, golden, "large", [1000])


# ------------------------------------------------------------------ decode --
def test_decode_streams_and_ids(ctx):
    """bpe_decode against the oracle's decode: a trained stream (symbols with
    WORD_START bits) and greedy ids decode to the corpus; empty input; an id
    outside the vocabulary and a short output are reported."""
    import bpe_trie_encode_gb300 as bt
    text = synth.corpus("tiny", 40_000)
    sym = oracle.pretokenize(text)
    m, fin = oracle.train_words(sym, 200)
    vb, voff = oracle.vocab_from_merges(m)
    got = ctx.decode(m, dev_sym(fin)).cpu().numpy()
    assert np.array_equal(got, text)
    assert oracle.decode(fin & np.uint32(0xFFFF), vb, voff) == text.tobytes()
    other = synth.lexicon("tiny").corpus(9, 30_000)
    ids, _ = oracle.Trie(vb, voff).encode(other)
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    assert np.array_equal(ctx.decode(m, d_ids).cpu().numpy(), other)
    assert ctx.decode(m, d_ids[:0]).numel() == 0
    bad = d_ids.clone()
    bad[17] = 256 + m.shape[0]
    with pytest.raises(bt.BpeError) as e:
        ctx.decode(m, bad)
    assert e.value.name == "INVALID_ARG"
    import ctypes
    from bpe_trie_encode_gb300 import _capi
    arr = (_capi.bpe_merge * m.shape[0]).from_buffer_copy(np.ascontiguousarray(m).tobytes())
    out = torch.empty(10, dtype=torch.uint8, device="cuda")
    n = ctypes.c_uint64(0)
    rc = _capi.load().bpe_decode(ctx._h, arr, m.shape[0], ctypes.c_void_p(d_ids.data_ptr()), d_ids.numel(),
                                 ctypes.c_void_p(out.data_ptr()), 10, ctypes.byref(n))
    assert rc == -6 and n.value == other.size
