"""Seeded synthetic inputs for byte-level BPE training and trie encoding.

Test and benchmark infrastructure shared by the CPU oracle's scripts, the
tests and ``bench.py``.  It only produces bytes (corpora, documents, substring
vocabularies); it holds none of the tokenizer's arithmetic.  The generator is
C (``synth.c``) so that gigabyte inputs take seconds; its floating point is
architecture independent, so every machine produces the same bytes.

Workloads (sizes and seeds; the text recipe is in ``synth.c``):

====  =====================================================================
tiny  64 KiB corpus, lexicon seed 0, K = 2,000 ASCII words, text seed 0
med   16 MiB corpus, lexicon seed 1, K = 20,000 Turkish-mix words, seed 1
large 256 MiB corpus, lexicon seed 2, K = 50,000 Turkish-mix words, seed 2
enc   1 GiB text from the large lexicon, text seed 3
batch 512 documents of >= 64 KiB from the large lexicon, text seed 4,
      document d drawn from its own sub-stream d; vocabulary: 256 bytes plus
      distinct substrings (2..48 bytes, log-uniform length) of the large
      corpus drawn with seed 5, 250,000 tokens in all; Unigram scores for it:
      Zipf log-probabilities over a seed-6 random ranking (``unigram_scores``)
====  =====================================================================
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

KIB = 1 << 10
MIB = 1 << 20
GIB = 1 << 30

# (lexicon seed, K, turkish) per workload family
LEXICONS = {
    "tiny": (0, 2000, False),
    "med": (1, 20000, True),
    "large": (2, 50000, True),
}
CORPUS = {  # name -> (lexicon, text seed, bytes)
    "tiny": ("tiny", 0, 64 * KIB),
    "med": ("med", 1, 16 * MIB),
    "large": ("large", 2, 256 * MIB),
    "enc": ("large", 3, 1 * GIB),
}
BATCH_TEXT_SEED = 4
BATCH_DOCS = 512
BATCH_DOC_BYTES = 64 * KIB
BATCH_VOCAB_SEED = 5
BATCH_VOCAB_SIZE = 250000
BATCH_VOCAB_MIN_LEN = 2
BATCH_VOCAB_MAX_LEN = 48
UNIGRAM_SCORE_SEED = 6


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (gcc, no fp contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        vp, u64, u32, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        lib.syn_lexicon_new.restype = vp
        lib.syn_lexicon_new.argtypes = [u64, u32, i32]
        lib.syn_lexicon_free.argtypes = [vp]
        lib.syn_lexicon_bytes.restype = u64
        lib.syn_lexicon_bytes.argtypes = [vp]
        lib.syn_lexicon_size.restype = u32
        lib.syn_lexicon_size.argtypes = [vp]
        lib.syn_lexicon_export.argtypes = [vp, vp, vp]
        lib.syn_corpus.restype = u64
        lib.syn_corpus.argtypes = [vp, u64, u64, vp, u64]
        lib.syn_document.restype = u64
        lib.syn_document.argtypes = [vp, u64, u64, u64, vp, u64]
        lib.syn_substring_vocab.restype = u32
        lib.syn_substring_vocab.argtypes = [vp, u64, u64, u32, u32, u32, vp, u64, vp]
        lib.syn_unigram_scores.restype = i32
        lib.syn_unigram_scores.argtypes = [u32, u64, vp]
        lib.syn_ln_export.restype = ctypes.c_double
        lib.syn_ln_export.argtypes = [ctypes.c_double]
        lib.syn_exp_export.restype = ctypes.c_double
        lib.syn_exp_export.argtypes = [ctypes.c_double]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Lexicon:
    """K distinct words drawn from one seed (see ``synth.c``)."""

    def __init__(self, seed: int, k: int, turkish: bool):
        self._lib = _load()
        self.h = self._lib.syn_lexicon_new(seed, k, 1 if turkish else 0)
        if not self.h:
            raise ValueError("empty lexicon")
        self.seed, self.k, self.turkish = seed, k, turkish

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self._lib.syn_lexicon_free(h)
            self.h = None

    def words(self) -> list[bytes]:
        nb = self._lib.syn_lexicon_bytes(self.h)
        data = np.empty(max(nb, 1), dtype=np.uint8)
        off = np.empty(self.k + 1, dtype=np.uint64)
        self._lib.syn_lexicon_export(self.h, _ptr(data), _ptr(off))
        raw = data.tobytes()
        return [raw[off[i]:off[i + 1]] for i in range(self.k)]

    def corpus(self, text_seed: int, nbytes: int) -> np.ndarray:
        out = np.empty(max(nbytes, 1), dtype=np.uint8)
        n = self._lib.syn_corpus(self.h, text_seed, nbytes, _ptr(out), out.size)
        return out[:n]

    def document(self, text_seed: int, index: int, target: int) -> np.ndarray:
        out = np.empty(target + 64, dtype=np.uint8)
        n = self._lib.syn_document(self.h, text_seed, index, target, _ptr(out), out.size)
        if n == 0 and target > 0:
            raise RuntimeError("document buffer too small")
        return out[:n]


_lex_cache: dict = {}


def lexicon(name: str) -> Lexicon:
    if name not in _lex_cache:
        _lex_cache[name] = Lexicon(*LEXICONS[name])
    return _lex_cache[name]


def corpus(name: str, nbytes: int | None = None) -> np.ndarray:
    """The named corpus (``tiny``/``med``/``large``/``enc``), optionally a prefix
    recipe of another size (same lexicon and seed, cut at ``nbytes``)."""
    lex, seed, size = CORPUS[name]
    return lexicon(lex).corpus(seed, size if nbytes is None else nbytes)


def batch_documents(n_docs: int = BATCH_DOCS, doc_bytes: int = BATCH_DOC_BYTES,
                    first: int = 0):
    """Documents ``first .. first+n_docs-1`` of the batch workload.

    Returns (concatenated bytes uint8, doc offsets uint64 of length n_docs+1)."""
    lex = lexicon("large")
    docs = [lex.document(BATCH_TEXT_SEED, first + d, doc_bytes) for d in range(n_docs)]
    off = np.zeros(n_docs + 1, dtype=np.uint64)
    if docs:
        off[1:] = np.cumsum([d.size for d in docs], dtype=np.uint64)
        data = np.concatenate(docs)
    else:
        data = np.empty(0, dtype=np.uint8)
    return data, off


def substring_vocab(text: np.ndarray, n_tok: int = BATCH_VOCAB_SIZE,
                    seed: int = BATCH_VOCAB_SEED, min_len: int = BATCH_VOCAB_MIN_LEN,
                    max_len: int = BATCH_VOCAB_MAX_LEN):
    """256 single bytes + distinct substrings of ``text``.

    Returns (bytes uint8, offsets uint64 of length n+1) with n <= n_tok (n <
    n_tok only when ``text`` has too few distinct substrings)."""
    lib = _load()
    text = np.ascontiguousarray(text, dtype=np.uint8)
    cap = 256 + (n_tok - 256) * max_len
    data = np.empty(cap, dtype=np.uint8)
    off = np.zeros(n_tok + 1, dtype=np.uint64)
    n = lib.syn_substring_vocab(_ptr(text), text.size, seed, n_tok, min_len, max_len,
                                _ptr(data), cap, _ptr(off))
    if n < 256:
        raise ValueError("substring vocabulary needs >= 256 tokens and text >= 2 bytes")
    off = off[: n + 1].copy()
    return data[: int(off[-1])].copy(), off


def unigram_scores(n_tok: int, seed: int = UNIGRAM_SCORE_SEED) -> np.ndarray:
    """Seeded synthetic Unigram log-probabilities (float64, one per token):
    a Zipf law over a random ranking of the tokens, normalised to sum 1,
    each value a float32."""
    out = np.empty(max(n_tok, 1), dtype=np.float64)
    if _load().syn_unigram_scores(n_tok, seed, _ptr(out)) != 0:
        raise ValueError("unigram scores need n_tok >= 1")
    return out[:n_tok]


def unigram_unk_score(scores: np.ndarray) -> float:
    """Score of the unknown-character fallback: 10 below the lowest token."""
    return float(np.min(scores)) - 10.0


def ln(x: float) -> float:
    return _load().syn_ln_export(x)


def exp(x: float) -> float:
    return _load().syn_exp_export(x)
