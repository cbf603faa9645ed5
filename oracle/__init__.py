"""CPU oracle for byte-level BPE training and greedy trie encoding.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library
neither imports it nor shares code with it; the product path fails loudly
without its CUDA extension instead of falling back here.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, one function per
step of the method, each citing the web page and section it follows); this
module only marshals numpy arrays through ctypes.

Sources:
  [GPU-BPE]  "bpe -- GPU BPE Tokenizer Pipeline" (llm.istanbul, learn/tr/13_bpe)
  [UNIGRAM]  "Improving Unigram tokenizer CPU performance" (perplexity.ai hub)

Parity pins (tests/test_oracle_*.py): the byte-class table printed in
[GPU-BPE] (hand-derived fixture), hand-worked corpora, brute-force pair counts
and greedy matches on tiny inputs, the two training forms against each other,
and the invariants (pair-count sum, WORD_START conservation, decode round
trips, no token spanning a class transition).  Every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

WS = 0x10000
MAX_MERGES = 65280

_CKPT_FN = ctypes.CFUNCTYPE(None, ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32),
                            ctypes.c_uint64, ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        vp, u64, u32, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        lib.orc_char_class.restype = i32
        lib.orc_char_class.argtypes = [u32]
        lib.orc_pretokenize.argtypes = [vp, u64, vp]
        lib.orc_train_stream.restype = i32
        lib.orc_train_stream.argtypes = [vp, u64, u32, vp, vp, vp, vp]
        lib.orc_train_words.restype = i32
        lib.orc_train_words.argtypes = [vp, u64, u32, vp, vp, vp, vp, vp, u32, _CKPT_FN, vp]
        lib.orc_vocab_from_merges.restype = i32
        lib.orc_vocab_from_merges.argtypes = [vp, u32, vp, vp]
        lib.orc_trie_new.restype = vp
        lib.orc_trie_new.argtypes = [vp, vp, u32]
        lib.orc_trie_free.argtypes = [vp]
        lib.orc_trie_nodes.restype = u64
        lib.orc_trie_nodes.argtypes = [vp]
        lib.orc_trie_max_len.restype = u32
        lib.orc_trie_max_len.argtypes = [vp]
        lib.orc_longest_match.restype = i32
        lib.orc_longest_match.argtypes = [vp, vp, u64, u64, vp, vp]
        lib.orc_pair_counts.restype = ctypes.c_int64
        lib.orc_pair_counts.argtypes = [vp, u64, vp, vp, u64]
        lib.orc_encode.restype = i32
        lib.orc_encode.argtypes = [vp, vp, vp, u32, vp, u64, vp, vp]
        lib.orc_unigram_encode.restype = i32
        lib.orc_unigram_encode.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_double, vp, vp, u32,
                                           vp, u64, vp, vp]
        _lib = lib
        return lib


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def _u8(x) -> np.ndarray:
    if isinstance(x, (bytes, bytearray)):
        return np.frombuffer(bytes(x), dtype=np.uint8)
    return np.ascontiguousarray(x, dtype=np.uint8)


def char_class(b: int) -> int:
    """Byte class per [GPU-BPE] "Line by line" 1): 0 Letter, 1 Digit, 2 Space,
    3 Punct, 4 Newline."""
    return _load().orc_char_class(b)


def pretokenize(data) -> np.ndarray:
    """Bytes -> uint32 symbols with WORD_START (0x10000) at class transitions
    and at index 0 ([GPU-BPE] "What it does" 1.)."""
    b = _u8(data)
    out = np.empty(max(b.size, 1), dtype=np.uint32)
    _load().orc_pretokenize(_p(b), b.size, _p(out))
    return out[: b.size]


def pair_counts(symbols):
    """All adjacent-pair counts of a stream (pairs never end on a WORD_START):
    (keys uint32 = left << 16 | right, ascending; counts uint32)."""
    lib = _load()
    s = np.ascontiguousarray(symbols, dtype=np.uint32)
    cap = max(s.size, 1)
    keys = np.empty(cap, dtype=np.uint32)
    cnt = np.empty(cap, dtype=np.uint32)
    d = lib.orc_pair_counts(_p(s), s.size, _p(keys), _p(cnt), cap)
    if d < 0:
        raise OracleError("pair count failed")
    return keys[:d].copy(), cnt[:d].copy()


def _train(fn_name, symbols, n_merges, checkpoints=None, callback=None):
    lib = _load()
    s = np.ascontiguousarray(symbols, dtype=np.uint32)
    merges = np.zeros((max(n_merges, 1), 4), dtype=np.uint32)
    n_done = ctypes.c_uint32(0)
    out = np.empty(max(s.size, 1), dtype=np.uint32)
    n_out = ctypes.c_uint64(0)
    if fn_name == "stream":
        rc = lib.orc_train_stream(_p(s), s.size, n_merges, _p(merges), ctypes.byref(n_done),
                                  _p(out), ctypes.byref(n_out))
    else:
        cps = np.ascontiguousarray(sorted(checkpoints or []), dtype=np.uint32)

        def _cb(k, ptr, n, _user):
            if callback is not None:
                arr = np.ctypeslib.as_array(ptr, shape=(n,)) if n else np.empty(0, np.uint32)
                callback(int(k), arr)

        cfn = _CKPT_FN(_cb)
        rc = lib.orc_train_words(_p(s), s.size, n_merges, _p(merges), ctypes.byref(n_done),
                                 _p(out), ctypes.byref(n_out), _p(cps) if cps.size else None,
                                 cps.size, cfn, None)
    if rc != 0:
        raise OracleError(f"oracle training failed ({rc})")
    return merges[: n_done.value].copy(), out[: n_out.value].copy()


def train_stream(symbols, n_merges: int):
    """Full-stream BPE training.  Returns (merges[n_done, 4] = (left, right,
    new_id, count), final symbols)."""
    return _train("stream", symbols, n_merges)


def train_words(symbols, n_merges: int, checkpoints=None, callback=None):
    """Word-frequency BPE training (same result as ``train_stream``).

    ``callback(k, stream)`` is called for every k in ``checkpoints`` with the
    symbol stream after k merges (the array is only valid during the call)."""
    return _train("words", symbols, n_merges, checkpoints, callback)


def vocab_from_merges(merges):
    """Token byte strings for ids 0 .. 255 + len(merges): (bytes, offsets)."""
    lib = _load()
    m = np.ascontiguousarray(merges, dtype=np.uint32).reshape(-1, 4)
    off = np.zeros(256 + m.shape[0] + 1, dtype=np.uint64)
    rc = lib.orc_vocab_from_merges(_p(m) if m.size else None, m.shape[0], None, _p(off))
    if rc:
        raise OracleError("malformed merge table")
    data = np.empty(max(int(off[-1]), 1), dtype=np.uint8)
    lib.orc_vocab_from_merges(_p(m) if m.size else None, m.shape[0], _p(data), _p(off))
    return data[: int(off[-1])], off


def decode(ids, vocab_bytes, vocab_off) -> bytes:
    """Concatenate the byte strings of ``ids``."""
    vb = bytes(_u8(vocab_bytes))
    off = np.asarray(vocab_off, dtype=np.uint64)
    return b"".join(vb[off[i]:off[i + 1]] for i in np.asarray(ids).tolist())


class Trie:
    """Plain sorted-children byte trie over a vocabulary (token id = index)."""

    def __init__(self, vocab_bytes, vocab_off):
        self._lib = _load()
        self._vb = _u8(vocab_bytes)
        self._off = np.ascontiguousarray(vocab_off, dtype=np.uint64)
        n_tok = self._off.size - 1
        self.h = self._lib.orc_trie_new(_p(self._vb) if self._vb.size else None,
                                        _p(self._off), n_tok)
        if not self.h:
            raise OracleError("trie construction failed")

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self._lib.orc_trie_free(h)
            self.h = None

    @property
    def n_nodes(self) -> int:
        return self._lib.orc_trie_nodes(self.h)

    @property
    def max_len(self) -> int:
        return self._lib.orc_trie_max_len(self.h)

    def longest_match(self, data, pos: int, end: int | None = None):
        """(id, length) of the longest token prefixing data[pos:end]."""
        b = _u8(data)
        end = b.size if end is None else end
        tid, ln = ctypes.c_int32(0), ctypes.c_uint32(0)
        rc = self._lib.orc_longest_match(self.h, _p(b), end, pos, ctypes.byref(tid), ctypes.byref(ln))
        if rc:
            raise OracleError(f"no token matches at byte {pos}")
        return tid.value, ln.value

    def encode(self, data, doc_off=None):
        """Greedy longest-match ids of each document: (ids int32, id_off uint64)."""
        b = _u8(data)
        doc = (np.array([0, b.size], dtype=np.uint64) if doc_off is None
               else np.ascontiguousarray(doc_off, dtype=np.uint64))
        n_docs = doc.size - 1
        cap = b.size
        ids = np.empty(max(cap, 1), dtype=np.int32)
        id_off = np.zeros(n_docs + 1, dtype=np.uint64)
        n = ctypes.c_uint64(0)
        rc = self._lib.orc_encode(self.h, _p(b) if b.size else None, _p(doc), n_docs, _p(ids), cap,
                                  _p(id_off), ctypes.byref(n))
        if rc:
            raise OracleError(f"oracle encode failed ({rc})")
        return ids[: n.value].copy(), id_off

    def unigram_encode(self, data, scores, unk_id: int, unk_score: float, doc_off=None):
        """Most likely segmentation of each document under per-token f64 scores
        ([UNIGRAM] "Unigram tokenization"): (ids int32, id_off uint64).  Tokens
        end only on UTF-8 character boundaries; a character no token starts
        becomes one ``unk_id`` scored ``unk_score``."""
        b = _u8(data)
        sc = np.ascontiguousarray(scores, dtype=np.float64)
        if sc.size != self._off.size - 1:
            raise OracleError("one score per token")
        doc = (np.array([0, b.size], dtype=np.uint64) if doc_off is None
               else np.ascontiguousarray(doc_off, dtype=np.uint64))
        n_docs = doc.size - 1
        cap = b.size
        ids = np.empty(max(cap, 1), dtype=np.int32)
        id_off = np.zeros(n_docs + 1, dtype=np.uint64)
        n = ctypes.c_uint64(0)
        rc = self._lib.orc_unigram_encode(self.h, _p(sc) if sc.size else None, unk_id, unk_score,
                                          _p(b) if b.size else None, _p(doc), n_docs, _p(ids), cap,
                                          _p(id_off), ctypes.byref(n))
        if rc:
            raise OracleError(f"oracle unigram encode failed ({rc})")
        return ids[: n.value].copy(), id_off
