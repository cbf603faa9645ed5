"""Pins of the oracle's Unigram (Viterbi) segmentation against things other
than itself ("Improving Unigram tokenizer CPU performance", "Unigram
tokenization": the most likely path over byte positions, tokens as edges,
UTF-8 continuation bytes skipped, <unk> when nothing matches):

* hand-worked vocabularies where the answer is read off by hand, including a
  tie and a case where greedy longest-match and Viterbi disagree;
* brute force: every segmentation of tiny inputs enumerated in pure Python,
  the best score compared exactly (sums taken left to right, as a path
  accumulates them) and the path compared wherever the best is unique;
* the UTF-8 readings: no token ends inside a character, and a character that
  no token starts becomes one <unk> spanning all its bytes;
* invariants on the synthetic batch workload: decode round trip, id offsets.
"""
import random

import numpy as np

import oracle
import synth


def vocab(tokens):
    data = b"".join(tokens)
    off = np.zeros(len(tokens) + 1, dtype=np.uint64)
    off[1:] = np.cumsum([len(t) for t in tokens])
    return np.frombuffer(data, dtype=np.uint8), off


def cont(b):
    return (b & 0xC0) == 0x80


def test_hand_worked():
    vb, off = vocab([b"a", b"b", b"ab"])
    T = oracle.Trie(vb, off)
    # ab (-1.5) beats a + b (-2)
    ids, io = T.unigram_encode(b"ab", [-1.0, -1.0, -1.5], 9, -50.0)
    assert ids.tolist() == [2] and io.tolist() == [0, 1]
    # a + b (-2) beats ab (-2.5)
    ids, _ = T.unigram_encode(b"ab", [-1.0, -1.0, -2.5], 9, -50.0)
    assert ids.tolist() == [0, 1]
    # a tie (-2 both ways): the path whose last token starts earliest wins
    ids, _ = T.unigram_encode(b"ab", [-1.0, -1.0, -2.0], 9, -50.0)
    assert ids.tolist() == [2]
    # an unmatched byte is one <unk>
    ids, _ = T.unigram_encode(b"abcab", [-1.0, -1.0, -1.5], 9, -50.0)
    assert ids.tolist() == [2, 9, 2]


def test_viterbi_is_not_greedy():
    vb, off = vocab([b"a", b"b", b"c", b"ab", b"bc"])
    T = oracle.Trie(vb, off)
    sc = [-1.0, -1.0, -5.0, -5.0, -1.0]
    assert T.encode(b"abc")[0].tolist() == [3, 2]          # greedy: ab c
    assert T.unigram_encode(b"abc", sc, 99, -50.0)[0].tolist() == [0, 4]   # a bc = -2


def test_utf8_boundaries():
    # 'ı' is C4 B1; tokens "\xc4" and "a\xc4" end inside it and never count
    vb, off = vocab([b"a", b"\xc4", b"a\xc4", b"\xb1"])
    T = oracle.Trie(vb, off)
    sc = [-1.0, -0.1, -0.1, -0.1]
    assert T.unigram_encode("aı".encode(), sc, 7, -20.0)[0].tolist() == [0, 7]
    assert T.unigram_encode("ıa".encode(), sc, 7, -20.0)[0].tolist() == [7, 0]
    # a 3-byte character with no token is one <unk>
    assert T.unigram_encode("a€a".encode(), sc, 7, -20.0)[0].tolist() == [0, 7, 0]
    # with the whole character in the vocabulary it is one token
    vb, off = vocab([b"a", "ı".encode(), "aı".encode()])
    T = oracle.Trie(vb, off)
    assert T.unigram_encode("aıı".encode(), [-1.0, -1.0, -1.5], 7, -20.0)[0].tolist() == [2, 1]


def brute_force(text, tokens, scores, unk_id, unk_score):
    """All paths from 0 to len(text): (best score, list of best paths)."""
    n = len(text)
    edges = {}
    for i in range(n):
        if cont(text[i]):
            continue
        out = []
        for t, tok in enumerate(tokens):
            j = i + len(tok)
            if j <= n and text[i:j] == tok and (j == n or not cont(text[j])):
                if all(not (text[i:j] == tokens[u] and u < t) for u in range(len(tokens))):
                    out.append((j, t, scores[t]))
        if not out:
            j = i + 1
            while j < n and cont(text[j]):
                j += 1
            out.append((j, unk_id, unk_score))
        edges[i] = out
    best, paths = None, []

    def walk(i, acc, path):
        nonlocal best, paths
        if i == n:
            if best is None or acc > best:
                best, paths = acc, [list(path)]
            elif acc == best:
                paths.append(list(path))
            return
        for j, t, s in edges.get(i, []):
            path.append(t)
            walk(j, acc + s, path)
            path.pop()

    walk(0, 0.0, [])
    return best, paths


def path_score(ids, tokens, scores, unk_id, unk_score):
    acc = 0.0
    for t in ids:
        acc = acc + (unk_score if t == unk_id else scores[t])
    return acc


def test_brute_force():
    rng = random.Random(11)
    alphabet = [b"a", b"b", b"c", "ı".encode(), "ş".encode()]
    for trial in range(300):
        n_tok = rng.randint(1, 10)
        tokens = []
        while len(tokens) < n_tok:
            t = b"".join(rng.choice(alphabet) for _ in range(rng.randint(1, 3)))
            if rng.random() < 0.2:                      # a token cut inside a character
                t = t[: rng.randint(1, len(t))]
            tokens.append(t)
        if trial % 3 == 0:
            scores = [float(-rng.randint(1, 4)) for _ in tokens]   # many ties
        else:
            scores = [-rng.random() * 8 for _ in tokens]
        text = b"".join(rng.choice(alphabet) for _ in range(rng.randint(0, 7)))
        unk_id, unk_score = len(tokens), -10.0 - rng.random()
        T = oracle.Trie(*vocab(tokens))
        ids, io = T.unigram_encode(text, scores, unk_id, unk_score)
        best, paths = brute_force(text, tokens, scores, unk_id, unk_score)
        got = ids.tolist()
        if not text:
            assert got == [] and io.tolist() == [0, 0]
            continue
        assert path_score(got, tokens, scores, unk_id, unk_score) == best, (text, tokens)
        assert got in paths
        if len(paths) == 1:
            assert got == paths[0]


def test_documents():
    vb, off = vocab([b"a", b"b", b"ab"])
    T = oracle.Trie(vb, off)
    text = b"ababba"
    doc = np.array([0, 2, 2, 5, 6], dtype=np.uint64)     # "ab", "", "abb", "a"
    ids, io = T.unigram_encode(text, [-1.0, -1.0, -1.5], 9, -50.0, doc)
    assert ids.tolist() == [2, 2, 1, 0] and io.tolist() == [0, 1, 1, 3, 4]


def test_batch_round_trip():
    data, doc = synth.batch_documents(n_docs=4, doc_bytes=4096)
    text = synth.corpus("large", 1 << 20)
    vb, off = synth.substring_vocab(text, n_tok=20000)
    scores = synth.unigram_scores(off.size - 1)
    n_tok = off.size - 1
    T = oracle.Trie(vb, off)
    ids, io = T.unigram_encode(data, scores, n_tok, synth.unigram_unk_score(scores), doc)
    assert io[0] == 0 and io[-1] == ids.size and np.all(np.diff(io.astype(np.int64)) >= 0)
    vbb = bytes(vb)
    for d in range(doc.size - 1):
        part = ids[int(io[d]):int(io[d + 1])].tolist()
        text_d = bytes(data[int(doc[d]):int(doc[d + 1])])
        if n_tok not in part:
            assert b"".join(vbb[int(off[t]):int(off[t + 1])] for t in part) == text_d
    # fewer tokens than greedy needs is not promised, but never more than characters
    chars = sum(1 for b in bytes(data) if not cont(b))
    assert ids.size <= chars


def test_scores_are_log_probabilities():
    s = synth.unigram_scores(5000)
    assert np.all(s < 0) and abs(np.exp(s).sum() - 1.0) < 1e-5
    assert np.array_equal(s, s.astype(np.float32).astype(np.float64))
    assert np.array_equal(s, synth.unigram_scores(5000))
    assert len(np.unique(s)) == s.size


def test_best_score_equals_shortest_path():
    """With scores <= 0 the best segmentation is a shortest path from 0 to n
    over positions (edge weight -score), found here by scipy's Dijkstra on
    texts of a few thousand bytes -- beyond what brute force enumerates.
    Scores are multiples of 1/8, so every sum is exact in either order."""
    from scipy.sparse import csr_matrix
    from scipy.sparse.csgraph import dijkstra
    rng = random.Random(21)
    for trial in range(12):
        tokens = []
        while len(tokens) < 200:
            t = b"".join(rng.choice([b"a", b"b", b"c", "ı".encode(), "ş".encode()])
                         for _ in range(rng.randint(1, 5)))
            if rng.random() < 0.1:
                t = t[: rng.randint(1, len(t))]
            tokens.append(t)
        scores = [-rng.randint(1, 80) / 8.0 for _ in tokens]
        unk_score = -20.0
        text = b"".join(rng.choice([b"a", b"b", b"c", b"d", "ı".encode(), "ş".encode()])
                        for _ in range(rng.randint(500, 3000)))
        n = len(text)
        first = {}
        for t, tok in enumerate(tokens):
            first.setdefault(tok, t)
        rows, cols, w = [], [], []
        for i in range(n):
            if cont(text[i]):
                continue
            matched = False
            for L in range(1, 16):
                j = i + L
                if j > n:
                    break
                t = first.get(text[i:j])
                if t is not None and (j == n or not cont(text[j])):
                    rows.append(i); cols.append(j); w.append(-scores[t]); matched = True
            if not matched:
                j = i + 1
                while j < n and cont(text[j]):
                    j += 1
                rows.append(i); cols.append(j); w.append(-unk_score)
        # every weight is at least 1/8: none vanishes from the sparse matrix
        g = csr_matrix((w, (rows, cols)), shape=(n + 1, n + 1))
        dist = dijkstra(g, directed=True, indices=0)[n]
        T = oracle.Trie(*vocab(tokens))
        ids, _ = T.unigram_encode(text, scores, len(tokens), unk_score)
        assert path_score(ids.tolist(), tokens, scores, len(tokens), unk_score) == -dist
