"""trie_encode_noalloc: encoding for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: a plug-in handed only a
stream and device pointers by an application that owns all device memory, or
a latency-critical path that must not pay the synchronisation of cudaFree.
For them the library offers one entry point whose scratch is a fixed array
compiled into the library.  This test calls it through the C ABI and checks
it against trie_encode and the oracle's greedy encode, bit for bit, on two
calls in a row (the second on a smaller, different input, so stale contents
of the shared array would show), and checks that inputs beyond either stated
maximum (documents, chunks) are refused before any write.  It lives in a file
of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402


def _noalloc(lib, trie, data, doc_off, cap):
    n_docs = doc_off.numel() - 1
    ids = torch.full((max(cap, 1),), -7, dtype=torch.int32, device="cuda")
    id_off = torch.full((n_docs + 1,), -7, dtype=torch.int64, device="cuda")
    n = ctypes.c_uint64(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.trie_encode_noalloc(trie._h, ctypes.c_void_p(data.data_ptr()), ctypes.c_void_p(doc_off.data_ptr()),
                                 n_docs, ctypes.c_void_p(ids.data_ptr()), cap, ctypes.c_void_p(id_off.data_ptr()),
                                 ctypes.byref(n), stream)
    return rc, ids[: n.value], id_off


def _vocab(tokens):
    vb = np.frombuffer(b"".join(tokens), dtype=np.uint8).copy()
    return vb, np.cumsum([0] + [len(t) for t in tokens]).astype(np.uint64)


def test_noalloc_encode_matches_trie_encode():
    import bpe_trie_encode_gb300 as bt
    from bpe_trie_encode_gb300 import _capi
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    lib = _capi.load()
    ctx = bt.Context(0)
    merges, _ = oracle.train_words(oracle.pretokenize(synth.corpus("tiny")), 256)
    vb, off = oracle.vocab_from_merges(merges)
    trie = ctx.trie_build(vb, off)
    otrie = oracle.Trie(vb, off)
    lex = synth.lexicon("tiny")
    inputs = [
        [lex.corpus(100 + d, 40000 + 977 * d).tobytes() for d in range(40)],       # ~1.9 MB, 40 docs
        [lex.corpus(900 + d, 3000 + 31 * d).tobytes() for d in range(7)] + [b""],  # smaller, an empty doc
    ]
    for docs in inputs:
        data = torch.from_numpy(np.frombuffer(b"".join(docs), dtype=np.uint8).copy()).cuda()
        doc_off = torch.tensor(np.cumsum([0] + [len(d) for d in docs]), dtype=torch.int64, device="cuda")
        want_ids, want_off = ctx.encode(trie, data, doc_off)
        rc, ids, id_off = _noalloc(lib, trie, data, doc_off, data.numel())
        assert rc == 0
        assert torch.equal(ids, want_ids)
        assert torch.equal(id_off, want_off)
        o_ids, o_off = otrie.encode(b"".join(docs), doc_off.cpu().numpy())
        assert np.array_equal(ids.cpu().numpy(), o_ids)
        assert np.array_equal(id_off.cpu().numpy().astype(np.uint64), o_off)

    # documents whose parses flip parity at their first byte flag one chunk
    # each: the repair runs from the flag list, then past its capacity
    ptrie = ctx.trie_build(*_vocab([bytes([b]) for b in range(256)] + [b"aa"]))
    for n_docs in (3000, 5000, 300):
        docs = [b"c" + b"a" * (299 + d % 7) for d in range(n_docs)]
        data = torch.from_numpy(np.frombuffer(b"".join(docs), dtype=np.uint8).copy()).cuda()
        doc_off = torch.tensor(np.cumsum([0] + [len(d) for d in docs]), dtype=torch.int64, device="cuda")
        want_ids, want_off = ctx.encode(ptrie, data, doc_off)
        rc, ids, id_off = _noalloc(lib, ptrie, data, doc_off, data.numel())
        assert rc == 0
        assert torch.equal(ids, want_ids)
        assert torch.equal(id_off, want_off)

    # beyond the stated maximum (65,536 documents): refused before any write
    many = torch.zeros(65538, dtype=torch.int64, device="cuda")
    rc, _, id_off = _noalloc(lib, trie, data, many, 16)
    assert rc == -1 and int(id_off[0]) == -7

    # within the document limit but beyond the chunk limit: 65,536 documents
    # of 1,025 bytes take 9 chunks of 128 bytes each, 589,824 > 524,288
    big = torch.full((65536 * 1025,), ord("a"), dtype=torch.uint8, device="cuda")
    big_off = torch.arange(0, 65537, dtype=torch.int64, device="cuda") * 1025
    rc, ids, id_off = _noalloc(lib, trie, big, big_off, 64)
    assert rc == -1 and ids.numel() == 0
    assert bool((id_off == -7).all())
    # one document fewer is still refused (589,815 chunks); at 58,254
    # documents (524,286 chunks) the same bytes are accepted
    rc, _, _ = _noalloc(lib, trie, big, big_off[:65536], 64)
    assert rc == -1
    ok_off = big_off[:58255]
    rc, ids, id_off = _noalloc(lib, trie, big, ok_off, big.numel())
    assert rc == 0
    want_ids, want_off = ctx.encode(trie, big, ok_off)
    assert torch.equal(ids, want_ids) and torch.equal(id_off, want_off)
    ctx.close()
