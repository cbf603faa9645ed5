"""C ABI checks that need no GPU: the library loads, exports every function the
header declares, refuses to run without a device, and builds a correct
double-array trie layout on the host (walked here in Python against the
oracle's plain trie)."""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import oracle
import synth
from bpe_trie_encode_gb300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TERM = 0x80000000


def header_functions():
    txt = open(os.path.join(ROOT, "include", "bpetrie.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_0-9]+)\s*\(", txt, flags=re.M)))


def test_library_exports_every_declared_function():
    lib = _capi.load()
    names = header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_capi.EXPORTS) == names


def test_no_gpu_is_an_error_not_a_fallback():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = _capi.load()
    h = ctypes.c_void_p()
    assert lib.bpe_ctx_create(ctypes.byref(h), 0, None) != 0
    import bpe_trie_encode_gb300 as bt
    with pytest.raises(RuntimeError):
        bt.Context()


def test_null_arguments_rejected():
    lib = _capi.load()
    assert lib.bpe_ctx_create(None, 0, None) == -1
    assert lib.bpe_ctx_set_option(None, 1, 0) == -1
    assert lib.bpe_train(None, None, 0, 0, None, None, None, None) == -1
    assert lib.trie_encode(None, None, None, None, 0, None, 0, None, None) == -1
    assert lib.unigram_create(None, None, None, 0, 0, 0.0, None) == -1
    assert lib.unigram_encode(None, None, None, None, 0, None, 0, None, None) == -1
    lib.bpe_ctx_destroy(None)
    lib.trie_free(None)
    lib.unigram_free(None)


def da_longest(check, base, tid, data: bytes, p: int, end: int):
    """Walk the double array: child of s on c is base[s]+c when check[..] == s."""
    node, best = 0, None
    q = p
    while q < end:
        b = base[node] & 0x7FFFFFFF if node else base[0]
        t = b + data[q]
        if node and (base[node] & 0x7FFFFFFF) == 0:
            break
        if t >= len(check) or check[t] != node:
            break
        node = t
        q += 1
        if base[node] & TERM:
            best = (int(tid[node]), q - p)
    return best


def vocab_arrays(tokens):
    vb = b"".join(tokens)
    off = np.cumsum([0] + [len(t) for t in tokens]).astype(np.uint64)
    return np.frombuffer(vb, dtype=np.uint8), off


@pytest.mark.parametrize("seed", range(6))
def test_double_array_matches_plain_trie(seed):
    rng = random.Random(seed)
    alpha = [b"ab", b"abc ", bytes(range(256))][seed % 3]
    toks = [bytes([b]) for b in range(256)]
    toks += [bytes(rng.choice(alpha) for _ in range(rng.randrange(2, 12))) for _ in range(rng.randrange(1, 400))]
    vb, off = vocab_arrays(toks)
    check, base, tid = _capi.trie_layout(vb, off)
    base = base.view(np.uint32)
    lc, lb, lt = check.tolist(), base.tolist(), tid.tolist()
    ref = oracle.Trie(vb, off)
    text = bytes(rng.choice(alpha) for _ in range(500))
    for p in range(len(text)):
        assert da_longest(lc, lb, lt, text, p, len(text)) == ref.longest_match(text, p), p
    # every used slot's parent is a used slot whose base reaches it
    used = np.nonzero(check >= 0)[0]
    par = check[used]
    assert np.all((base[par] & 0x7FFFFFFF) <= used)
    assert np.all(used - (base[par] & 0x7FFFFFFF) < 256)


def test_double_array_duplicates_keep_lowest_id():
    toks = [bytes([b]) for b in range(256)] + [b"xy", b"xy", b"x"]
    vb, off = vocab_arrays(toks)
    check, base, tid = _capi.trie_layout(vb, off)
    base = base.view(np.uint32)
    lc, lb, lt = check.tolist(), base.tolist(), tid.tolist()
    assert da_longest(lc, lb, lt, b"xyz", 0, 3) == (256, 2)
    assert da_longest(lc, lb, lt, b"xq", 0, 2) == (ord("x"), 1)


def test_layout_without_a_single_byte():
    """A vocabulary missing byte 0xFF lays out (Unigram encoding accepts it);
    the root's slot for 0xFF is then no token of the root."""
    toks = [bytes([b]) for b in range(255)] + [b"ab"]
    vb, off = vocab_arrays(toks)
    check, base, tid = _capi.trie_layout(vb, off)
    rb = int(base.view(np.uint32)[0] & 0x7FFFFFFF)
    for b in range(255):
        assert check[rb + b] == 0 and tid[rb + b] == b
    assert check[rb + 255] != 0 or tid[rb + 255] < 0


def test_layout_large_substring_vocab_sampled():
    """The 250,000-token substring vocabulary: sampled positions of a batch
    document agree with the oracle's plain trie."""
    text = synth.corpus("large", 8 << 20)
    vb, off = synth.substring_vocab(text)
    check, base, tid = _capi.trie_layout(vb, off)
    base = base.view(np.uint32)
    lc, lb, lt = check.tolist(), base.tolist(), tid.tolist()
    ref = oracle.Trie(vb, off)
    doc, _ = synth.batch_documents(1)
    d = doc.tobytes()
    rng = random.Random(3)
    for p in rng.sample(range(len(d)), 3000):
        assert da_longest(lc, lb, lt, d, p, len(d)) == ref.longest_match(d, p)


def test_vocab_from_merges_matches_oracle():
    """bpe_vocab_from_merges (the library, host only) against the oracle's
    vocabulary on the tiny workload's merge table and on the large corpus's
    stored table (32,000 merges)."""
    import bpe_trie_encode_gb300 as bt
    sym = oracle.pretokenize(synth.corpus("tiny"))
    m, _ = oracle.train_words(sym, 256)
    tables = [m, m[:0], m[:1]]
    lm = os.path.join(ROOT, "tests", "golden", "large_merges.npy")
    if os.path.exists(lm):
        lr = np.load(lm).astype(np.uint32)
        big = np.zeros((lr.shape[0], 4), dtype=np.uint32)
        big[:, :2] = lr[:, :2]
        big[:, 2] = 256 + np.arange(lr.shape[0], dtype=np.uint32)
        big[:, 3] = lr[:, 2]
        tables.append(big)
    for t in tables:
        vb, off = bt.vocab_from_merges(t)
        wb, woff = oracle.vocab_from_merges(t)
        assert np.array_equal(off, woff.astype(np.uint64))
        assert np.array_equal(vb, wb)


def test_vocab_from_merges_rejects_malformed_tables():
    lib = _capi.load()
    n = ctypes.c_uint64(0)

    def call(rows):
        arr = (_capi.bpe_merge * len(rows))(*[_capi.bpe_merge(*r) for r in rows])
        return lib.bpe_vocab_from_merges(arr, len(rows), None, 0, None, ctypes.byref(n))

    assert call([(97, 98, 256, 1)]) == -6            # valid: CAPACITY with the size
    assert n.value == 256 + 2
    assert call([(97, 98, 257, 1)]) == -1            # new_id must be 256 + k
    assert call([(97, 256, 256, 1)]) == -1           # an id no earlier merge made
    assert call([(97, 98, 256, 1), (256, 256, 257, 1)]) == -6
    assert n.value == 256 + 2 + 4
    assert lib.bpe_vocab_from_merges(None, 1, None, 0, None, ctypes.byref(n)) == -1
    assert lib.bpe_decode(None, None, 0, None, 0, None, 0, None) == -1
