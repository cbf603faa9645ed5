"""ctypes binding of libbpetrie.so (the C ABI declared in include/bpetrie.h).

Argument marshalling only: every step of training and encoding runs in the
library's CUDA kernels.  There is no CPU fallback -- if the library is not
built, or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libbpetrie.so")

BPE_OK = 0
ERRORS = {
    -1: "INVALID_ARG", -2: "OOM", -3: "CUDA", -4: "TABLE_FULL", -5: "ID_OVERFLOW",
    -6: "CAPACITY", -7: "TIMEOUT", -8: "CHECKED_OOB",
}
BPE_WORD_START = 0x10000
BPE_MAX_MERGES = 65280
BPE_OPT_TABLE_LOG2, BPE_OPT_GRAPH, BPE_OPT_PROFILE, BPE_OPT_CHUNK, BPE_OPT_TRAIN_WORDS = 1, 2, 3, 4, 5
BPE_OPT_MERGE, BPE_OPT_PERSISTENT, BPE_OPT_TRIE_LAYOUT, BPE_OPT_UNI_CHUNK = 6, 7, 8, 9
BPE_OPT_TEST_STALL_TILE, BPE_OPT_SPARSE_MERGE, BPE_OPT_LIST_FRONTIER, BPE_OPT_LIST_TAIL = 10, 11, 12, 13
BPE_TRIE_DOUBLE_ARRAY, BPE_TRIE_BITMAP = 0, 1
BPE_MERGE_TWO_PASS, BPE_MERGE_LOOKBACK, BPE_MERGE_TILES, BPE_MERGE_LISTS = 0, 1, 2, 3

# every symbol the header declares (checked by the tests)
EXPORTS = [
    "bpe_ctx_create", "bpe_ctx_set_stream", "bpe_ctx_destroy", "bpe_last_error",
    "bpe_ctx_set_option", "bpe_last_stats", "bpe_pretokenize", "bpe_train",
    "trie_build", "trie_layout", "trie_info", "trie_free", "trie_encode",
    "trie_encode_noalloc", "trie_stream_open", "trie_stream_push", "trie_stream_close",
    "trie_encode_host", "unigram_create", "unigram_encode", "unigram_free",
    "bpe_vocab_from_merges", "bpe_decode",
]


class BpeError(RuntimeError):
    def __init__(self, code: int, message: str):
        self.code = code
        self.name = ERRORS.get(code, str(code))
        super().__init__(f"{self.name}: {message}")


class bpe_merge(ctypes.Structure):
    _fields_ = [("left", ctypes.c_uint32), ("right", ctypes.c_uint32),
                ("new_id", ctypes.c_uint32), ("count", ctypes.c_uint32)]


class bpe_kernel_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_uint64),
                ("bytes", ctypes.c_double), ("ms", ctypes.c_double)]


class bpe_stats(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("kernel_launches", ctypes.c_uint64), ("k", bpe_kernel_stat * 8)]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libbpetrie.so (built by ``bpe_trie_encode_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, u32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
        P = ctypes.POINTER
        sig = {
            "bpe_ctx_create": (i32, [P(vp), i32, vp]),
            "bpe_ctx_set_stream": (i32, [vp, vp]),
            "bpe_ctx_destroy": (None, [vp]),
            "bpe_last_error": (ctypes.c_char_p, [vp]),
            "bpe_ctx_set_option": (i32, [vp, i32, ctypes.c_int64]),
            "bpe_last_stats": (i32, [vp, P(bpe_stats)]),
            "bpe_pretokenize": (i32, [vp, vp, u64, vp]),
            "bpe_train": (i32, [vp, vp, u64, u32, P(bpe_merge), P(u32), vp, P(u64)]),
            "trie_build": (i32, [vp, vp, vp, u32, P(vp)]),
            "trie_layout": (i32, [vp, vp, u32, vp, vp, vp, u64, P(u64)]),
            "trie_info": (i32, [vp, P(u64), P(u64), P(u32)]),
            "trie_free": (None, [vp]),
            "trie_encode": (i32, [vp, vp, vp, vp, u32, vp, u64, vp, P(u64)]),
            "trie_encode_noalloc": (i32, [vp, vp, vp, u32, vp, u64, vp, P(u64), vp]),
            "trie_stream_open": (i32, [vp, vp, P(vp)]),
            "trie_stream_push": (i32, [vp, vp, u64, i32, vp, u64, P(u64)]),
            "trie_stream_close": (None, [vp]),
            "trie_encode_host": (i32, [vp, vp, vp, vp, u32, vp, u64, vp, P(u64), u64]),
            "unigram_create": (i32, [vp, vp, vp, u32, ctypes.c_int32, ctypes.c_double, P(vp)]),
            "unigram_encode": (i32, [vp, vp, vp, vp, u32, vp, u64, vp, P(u64)]),
            "unigram_free": (None, [vp]),
            "bpe_vocab_from_merges": (i32, [vp, u32, vp, u64, vp, P(u64)]),
            "bpe_decode": (i32, [vp, vp, u32, vp, u64, vp, u64, P(u64)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(ctx, rc: int) -> None:
    if rc != BPE_OK:
        msg = load().bpe_last_error(ctx)
        raise BpeError(rc, msg.decode() if msg else "")


def trie_layout(vocab_bytes, vocab_off):
    """Host-side double-array layout (no GPU): (check, base, tid) int32 arrays."""
    import numpy as np
    lib = load()
    vb = np.ascontiguousarray(vocab_bytes, dtype=np.uint8)
    off = np.ascontiguousarray(vocab_off, dtype=np.uint64)
    n_tok = off.size - 1
    n = ctypes.c_uint64(0)
    vp = ctypes.c_void_p
    rc = lib.trie_layout(vp(vb.ctypes.data if vb.size else 0), vp(off.ctypes.data), n_tok,
                         None, None, None, 0, ctypes.byref(n))
    if rc not in (BPE_OK, -6):
        raise BpeError(rc, "trie_layout failed")
    check = np.empty(n.value, dtype=np.int32)
    base = np.empty(n.value, dtype=np.int32)
    tid = np.empty(n.value, dtype=np.int32)
    rc = lib.trie_layout(vp(vb.ctypes.data if vb.size else 0), vp(off.ctypes.data), n_tok,
                         vp(check.ctypes.data), vp(base.ctypes.data), vp(tid.ctypes.data), n.value,
                         ctypes.byref(n))
    if rc != BPE_OK:
        raise BpeError(rc, "trie_layout failed")
    return check, base, tid
