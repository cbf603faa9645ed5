"""Pins of the CPU oracle against things other than itself.

* the byte-class table read by hand off the routine printed on the GPU BPE
  pipeline page ("Line by line", 1) bpe_word_boundary);
* hand-worked corpora (tests/golden/worked_examples.json);
* brute force on tiny inputs: an independent pure-Python merge loop
  (collections.Counter + a full sort for the argmax) and a greedy encoder that
  tries every vocabulary string at every position;
* the two oracle training forms (full stream, word frequency) against each
  other, including adversarial runs of identical symbols;
* invariants: the pair-count sum, WORD_START conservation, decode round trips,
  no learned token spanning a class transition, stream-length bookkeeping.
"""
import json
import os
import random
from collections import Counter

import numpy as np
import pytest

import oracle
import synth

WS = 0x10000
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_classes():
    cls = [None] * 256
    with open(os.path.join(GOLDEN, "char_class_ranges.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            a, b, c = line.split()
            for x in range(int(a, 16), int(b, 16) + 1):
                cls[x] = int(c)
    assert all(c is not None for c in cls)
    return cls


CLS = golden_classes()


# ---------------------------------------------------------------- brute force
def bf_pretokenize(text: bytes):
    return [b | (WS if i == 0 or CLS[b] != CLS[text[i - 1]] else 0) for i, b in enumerate(text)]


def bf_counts(s):
    c = Counter()
    for i in range(len(s) - 1):
        if not s[i + 1] & WS:
            c[(s[i] & 0xFFFF, s[i + 1] & 0xFFFF)] += 1
    return c


def bf_train(s, n_merges):
    s = list(s)
    merges = []
    for k in range(n_merges):
        c = bf_counts(s)
        if not c:
            break
        (l, r), cnt = sorted(c.items(), key=lambda kv: (-kv[1], kv[0]))[0]
        new, out, i = 256 + k, [], 0
        while i < len(s):
            if i + 1 < len(s) and (s[i] & 0xFFFF, s[i + 1] & 0xFFFF) == (l, r) and not s[i + 1] & WS:
                out.append(new | (s[i] & WS))
                i += 2
            else:
                out.append(s[i])
                i += 1
        merges.append([l, r, new, cnt])
        s = out
    return merges, s


def bf_vocab(merges):
    v = [bytes([b]) for b in range(256)]
    for l, r, _, _ in merges:
        v.append(v[l] + v[r])
    return v


def bf_encode(text: bytes, vocab):
    ids, p = [], 0
    while p < len(text):
        best, bl = -1, 0
        for t, s in enumerate(vocab):
            if len(s) > bl and text.startswith(s, p):
                best, bl = t, len(s)
        assert bl > 0
        ids.append(best)
        p += bl
    return ids


def rand_text(rng, n, alphabet):
    return bytes(rng.choice(alphabet) for _ in range(n))


# ----------------------------------------------------------------- byte class
def test_char_class_matches_page_table():
    for b in range(256):
        assert oracle.char_class(b) == CLS[b], hex(b)


def test_pretokenize_matches_hand_rule():
    rng = random.Random(1)
    alphabet = list(b"aZ09 \n\t.,\x7f") + [0x80, 0xC3, 0xA7, 0xFF, 0x00]
    for n in [0, 1, 2, 3, 17, 200]:
        for _ in range(5):
            t = rand_text(rng, n, alphabet)
            assert oracle.pretokenize(t).tolist() == bf_pretokenize(t)


def test_pretokenize_utf8_letters_are_letters():
    t = "çağ ış".encode()
    s = oracle.pretokenize(t)
    ws = [(x >> 16) & 1 for x in s.tolist()]
    # c3 a7 61 c4 9f | 20 | c4 b1 c5 9f : only the word starts carry the bit
    assert ws == [1, 0, 0, 0, 0, 1, 1, 0, 0, 0]


# ------------------------------------------------------------ worked examples
def load_examples():
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("form", ["stream", "words"])
def test_worked_training_examples(form):
    for ex in load_examples()["train"]:
        s = oracle.pretokenize(ex["text"].encode())
        fn = oracle.train_stream if form == "stream" else oracle.train_words
        m, f = fn(s, ex["n_merges"])
        assert m.tolist() == ex["merges"], ex["name"]
        assert [[x & 0xFFFF, x >> 16] for x in f.tolist()] == ex["final"], ex["name"]


def test_worked_encode_examples():
    for ex in load_examples()["encode"]:
        vocab = [bytes([b]) for b in range(256)] + [s.encode() for s in ex["vocab_extra"]]
        vb = b"".join(vocab)
        off = np.cumsum([0] + [len(v) for v in vocab]).astype(np.uint64)
        ids, id_off = oracle.Trie(vb, off).encode(ex["text"].encode())
        assert ids.tolist() == ex["ids"], ex["name"]
        assert id_off.tolist() == [0, len(ex["ids"])]


# ------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed", range(12))
def test_training_matches_brute_force(seed):
    rng = random.Random(seed)
    alphabets = [b"ab", b"aab ", b"abc a.\n1", b"a", b"ab1 "]
    t = rand_text(rng, rng.randrange(0, 90), alphabets[seed % len(alphabets)])
    s = oracle.pretokenize(t)
    want_m, want_f = bf_train(bf_pretokenize(t), 40)
    for fn in (oracle.train_stream, oracle.train_words):
        m, f = fn(s, 40)
        assert m.tolist() == want_m
        assert f.tolist() == want_f


def test_pair_counts_match_brute_force():
    rng = random.Random(7)
    for n in [0, 1, 2, 50, 400]:
        t = rand_text(rng, n, b"abcab a1.")
        s = oracle.pretokenize(t)
        keys, cnt = oracle.pair_counts(s)
        c = bf_counts(bf_pretokenize(t))
        want = sorted(((l << 16) | r, v) for (l, r), v in c.items())
        assert list(zip(keys.tolist(), cnt.tolist())) == want


@pytest.mark.parametrize("seed", range(8))
def test_greedy_encode_matches_brute_force(seed):
    rng = random.Random(100 + seed)
    # vocabulary: bytes + random short strings (with duplicates) over a small alphabet
    extra = [rand_text(rng, rng.randrange(2, 6), b"ab c") for _ in range(rng.randrange(1, 30))]
    vocab = [bytes([b]) for b in range(256)] + extra
    vb = b"".join(vocab)
    off = np.cumsum([0] + [len(v) for v in vocab]).astype(np.uint64)
    trie = oracle.Trie(vb, off)
    docs = [rand_text(rng, rng.randrange(0, 60), b"ab c") for _ in range(4)]
    data = b"".join(docs)
    doc_off = np.cumsum([0] + [len(d) for d in docs]).astype(np.uint64)
    ids, id_off = trie.encode(data, doc_off)
    want, want_off = [], [0]
    for d in docs:
        want += bf_encode(d, vocab)
        want_off.append(len(want))
    assert ids.tolist() == want
    assert id_off.tolist() == want_off
    assert oracle.decode(ids, vb, off) == data


def test_encode_reports_missing_byte():
    vocab = [b"a", b"b"]
    vb = b"ab"
    off = np.array([0, 1, 2], dtype=np.uint64)
    with pytest.raises(oracle.OracleError):
        oracle.Trie(vb, off).encode(b"abc")


def test_longest_match_is_greedy_step():
    vocab = [bytes([b]) for b in range(256)] + [b"ab", b"abcd"]
    vb = b"".join(vocab)
    off = np.cumsum([0] + [len(v) for v in vocab]).astype(np.uint64)
    t = oracle.Trie(vb, off)
    assert t.longest_match(b"abcab", 0) == (256, 2)
    assert t.longest_match(b"abcd", 0) == (257, 4)
    assert t.longest_match(b"abcd", 0, 3) == (256, 2)   # the document end cuts the walk


# ------------------------------------------------------------ adversarial runs
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 33, 64, 65, 1000, 1001])
def test_identical_runs_forms_agree(n):
    t = b"a" * n + b" " + b"a" * (n // 2 + 1)
    s = oracle.pretokenize(t)
    m1, f1 = oracle.train_stream(s, 20)
    m2, f2 = oracle.train_words(s, 20)
    assert np.array_equal(m1, m2) and np.array_equal(f1, f2)
    if n <= 65:
        bm, bf = bf_train(bf_pretokenize(t), 20)
        assert m1.tolist() == bm and f1.tolist() == bf


def test_all_equal_counts_tie():
    # every pair occurs once: the merge order must be ascending key order
    t = b"ab cd ef gh ba dc"
    m, _ = oracle.train_stream(oracle.pretokenize(t), 3)
    assert [(l, r) for l, r, _, _ in m.tolist()] == [(97, 98), (98, 97), (99, 100)]


# ------------------------------------------------------------------ invariants
@pytest.fixture(scope="module")
def tiny_run():
    text = synth.corpus("tiny")
    sym = oracle.pretokenize(text)
    cps = {}
    m, f = oracle.train_words(sym, 256, checkpoints=list(range(0, 257, 16)) + [1, 2, 3],
                              callback=lambda k, s: cps.__setitem__(k, s.copy()))
    return text, sym, m, f, cps


def test_invariant_pair_count_sum(tiny_run):
    text, sym, m, f, cps = tiny_run
    for k, s in cps.items():
        keys, cnt = oracle.pair_counts(s)
        n_ws = int(np.count_nonzero(s & WS))
        assert int(cnt.sum(dtype=np.uint64)) == s.size - n_ws
        if k < m.shape[0]:   # the chosen pair is the argmax of these counts
            best = max(zip(cnt.tolist(), (-keys.astype(np.int64)).tolist()))
            assert (m[k, 3], (m[k, 0] << 16) | m[k, 1]) == (best[0], -best[1])


def test_invariant_word_starts_and_decode(tiny_run):
    text, sym, m, f, cps = tiny_run
    vb, off = oracle.vocab_from_merges(m)
    ws0 = int(np.count_nonzero(sym & WS))
    for k, s in cps.items():
        assert int(np.count_nonzero(s & WS)) == ws0
        assert oracle.decode(s & 0xFFFF, vb, off) == text.tobytes()
        assert int(np.max(s & 0xFFFF)) < 256 + min(k, m.shape[0])


def test_invariant_tokens_within_one_class(tiny_run):
    text, sym, m, f, cps = tiny_run
    for tok in bf_vocab(m.tolist())[256:]:
        assert len({CLS[b] for b in tok}) == 1, tok


def test_invariant_length_bookkeeping(tiny_run):
    text, sym, m, f, cps = tiny_run
    for k in (0, 1, 2):
        l, r, _, cnt = m[k].tolist()
        applied = cps[k].size - cps[k + 1].size
        assert 0 < applied <= cnt
        if l != r:
            assert applied == cnt


def test_round_trip_encode_learned_vocab(tiny_run):
    text, sym, m, f, cps = tiny_run
    vb, off = oracle.vocab_from_merges(m)
    trie = oracle.Trie(vb, off)
    other = synth.lexicon("tiny").corpus(99, 20000)
    ids, _ = trie.encode(other)
    assert oracle.decode(ids, vb, off) == other.tobytes()
    # every emitted token is the longest match at its position
    p = 0
    for t in ids[:2000].tolist():
        assert trie.longest_match(other, p) == (t, int(off[t + 1] - off[t]))
        p += int(off[t + 1] - off[t])


def test_vocab_from_merges_brute_force(tiny_run):
    text, sym, m, f, cps = tiny_run
    vb, off = oracle.vocab_from_merges(m)
    want = bf_vocab(m.tolist())
    got = [bytes(vb[off[i]:off[i + 1]]) for i in range(len(want))]
    assert got == want
