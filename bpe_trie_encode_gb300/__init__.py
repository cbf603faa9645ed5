"""bpe_trie_encode_gb300 -- byte-level BPE training and greedy trie encoding on
one GB300 (sm_103a).

The work happens in ``libbpetrie.so`` (hand-written CUDA kernels behind the C
ABI of ``include/bpetrie.h``); this package marshals torch tensors to it.
PyTorch is used only for device memory and streams.

    import torch, bpe_trie_encode_gb300 as bt
    ctx = bt.Context()
    sym = ctx.pretokenize(torch.frombuffer(text, dtype=torch.uint8).cuda())
    merges, final = ctx.train(sym, 4096)
    trie = ctx.trie_build(*bt.vocab_from_merges(merges))
    ids, id_off = ctx.encode(trie, data_u8_cuda, doc_off_i64_cuda)
    uni = ctx.unigram(trie, scores_f64, unk_id, unk_score)       # Viterbi model
    ids, id_off = ctx.unigram_encode(uni, data_u8_cuda, doc_off_i64_cuda)
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _capi
from ._capi import (BPE_MAX_MERGES, BPE_MERGE_LISTS, BPE_MERGE_LOOKBACK, BPE_MERGE_TILES,  # noqa: F401
                    BPE_MERGE_TWO_PASS, BPE_OPT_LIST_FRONTIER, BPE_OPT_LIST_TAIL,
                    BPE_OPT_CHUNK, BPE_OPT_GRAPH, BPE_OPT_MERGE, BPE_OPT_PERSISTENT, BPE_OPT_PROFILE,
                    BPE_OPT_SPARSE_MERGE, BPE_OPT_TABLE_LOG2, BPE_OPT_TRAIN_WORDS, BPE_OPT_TRIE_LAYOUT,
                    BPE_OPT_UNI_CHUNK, BPE_TRIE_BITMAP, BPE_TRIE_DOUBLE_ARRAY, BPE_WORD_START, BpeError)

__all__ = ["Context", "Trie", "Unigram", "BpeError", "vocab_from_merges", "BPE_WORD_START", "BPE_MAX_MERGES"]


def _stream_ptr(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(t: torch.Tensor, dtype: torch.dtype, name: str, device: torch.device) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the context is on {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.contiguous()


class Trie:
    """A double-array trie uploaded to the GPU (see ``Context.trie_build``)."""

    def __init__(self, handle: int, device: torch.device, n_tok: int):
        self._h = ctypes.c_void_p(handle)
        self.device = device
        self.n_tok = n_tok

    def info(self) -> dict:
        n_nodes, n_slots, max_len = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint32()
        _capi.load().trie_info(self._h, ctypes.byref(n_nodes), ctypes.byref(n_slots), ctypes.byref(max_len))
        return {"n_tok": self.n_tok, "n_nodes": n_nodes.value, "n_slots": n_slots.value,
                "max_token_len": max_len.value}

    def close(self):
        if self._h:
            _capi.load().trie_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Context:
    """A library context on one CUDA device.  Calls are ordered on the torch
    current stream of that device at the time of each call."""

    def __init__(self, device=None):
        if not torch.cuda.is_available():
            raise RuntimeError("bpe_trie_encode_gb300 needs a CUDA GPU")
        self.lib = _capi.load()
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        h = ctypes.c_void_p()
        rc = self.lib.bpe_ctx_create(ctypes.byref(h), self.device.index, ctypes.c_void_p(_stream_ptr(self.device)))
        if rc != 0:
            raise BpeError(rc, "bpe_ctx_create failed")
        self._h = h

    # -- plumbing -----------------------------------------------------------
    def _sync_stream(self):
        self.lib.bpe_ctx_set_stream(self._h, ctypes.c_void_p(_stream_ptr(self.device)))

    def close(self):
        if getattr(self, "_h", None):
            self.lib.bpe_ctx_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, option: int, value: int) -> None:
        _capi.check(self._h, self.lib.bpe_ctx_set_option(self._h, option, value))

    def stats(self) -> dict:
        s = _capi.bpe_stats()
        _capi.check(self._h, self.lib.bpe_last_stats(self._h, ctypes.byref(s)))
        out = {s.k[i].name.decode(): {"launches": s.k[i].launches, "bytes": s.k[i].bytes, "ms": s.k[i].ms}
               for i in range(s.n)}
        out["kernel_launches"] = s.kernel_launches
        return out

    # -- the C ABI --------------------------------------------------------
    def pretokenize(self, data: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        """uint8 bytes -> int32 tensor holding the uint32 symbols (bit 16 =
        WORD_START).  Asynchronous on the current stream."""
        data = _need_cuda(data, torch.uint8, "data", self.device)
        n = data.numel()
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device=self.device)
        out = _need_cuda(out, torch.int32, "out", self.device)
        if out.numel() < n:
            raise ValueError("out too small")
        self._sync_stream()
        _capi.check(self._h, self.lib.bpe_pretokenize(self._h, ctypes.c_void_p(data.data_ptr()), n,
                                                      ctypes.c_void_p(out.data_ptr())))
        return out[:n]

    def train(self, symbols: torch.Tensor, n_merges: int, final: bool = True):
        """BPE merge loop.  Returns (merges uint32 [n_done, 4] = (left, right,
        new_id, count), final symbols int32 tensor or None)."""
        symbols = _need_cuda(symbols, torch.int32, "symbols", self.device)
        n = symbols.numel()
        merges = (_capi.bpe_merge * max(n_merges, 1))()
        n_done = ctypes.c_uint32(0)
        n_final = ctypes.c_uint64(0)
        fin = torch.empty(max(n, 1), dtype=torch.int32, device=self.device) if final else None
        self._sync_stream()
        rc = self.lib.bpe_train(self._h, ctypes.c_void_p(symbols.data_ptr() if n else 0), n, n_merges,
                                merges, ctypes.byref(n_done),
                                ctypes.c_void_p(fin.data_ptr()) if fin is not None else None,
                                ctypes.byref(n_final))
        _capi.check(self._h, rc)
        m = np.frombuffer(merges, dtype=np.uint32).reshape(-1, 4)[: n_done.value].copy()
        return m, (fin[: n_final.value] if fin is not None else None)

    def trie_build(self, vocab_bytes, vocab_off) -> Trie:
        """Double-array trie of token strings vocab_bytes[off[t]:off[t+1]]."""
        vb = np.ascontiguousarray(np.frombuffer(bytes(vocab_bytes), dtype=np.uint8)
                                  if isinstance(vocab_bytes, (bytes, bytearray)) else vocab_bytes,
                                  dtype=np.uint8)
        off = np.ascontiguousarray(vocab_off, dtype=np.uint64)
        n_tok = off.size - 1
        h = ctypes.c_void_p()
        _capi.check(self._h, self.lib.trie_build(self._h, ctypes.c_void_p(vb.ctypes.data if vb.size else 0),
                                                 ctypes.c_void_p(off.ctypes.data), n_tok, ctypes.byref(h)))
        return Trie(h.value, self.device, n_tok)

    def encode(self, trie: Trie, data: torch.Tensor, doc_off: torch.Tensor | None = None,
               capacity: int | None = None, ids_out: torch.Tensor | None = None):
        """Greedy longest-match ids.  data: uint8 CUDA tensor; doc_off: int64
        CUDA tensor of n_docs+1 ascending offsets (default: one document).
        Returns (ids int32 [n_ids], id_off int64 [n_docs+1])."""
        data = _need_cuda(data, torch.uint8, "data", self.device)
        if doc_off is None:
            doc_off = torch.tensor([0, data.numel()], dtype=torch.int64, device=self.device)
        doc_off = _need_cuda(doc_off, torch.int64, "doc_off", self.device)
        n_docs = doc_off.numel() - 1
        if ids_out is None:
            cap = data.numel() if capacity is None else capacity
            ids_out = torch.empty(max(cap, 1), dtype=torch.int32, device=self.device)
        else:
            ids_out = _need_cuda(ids_out, torch.int32, "ids_out", self.device)
            cap = ids_out.numel() if capacity is None else min(capacity, ids_out.numel())
        id_off = torch.empty(max(n_docs + 1, 1), dtype=torch.int64, device=self.device)
        n_ids = ctypes.c_uint64(0)
        if data.numel() == 0:   # keep a valid device pointer for empty input
            data = torch.empty(16, dtype=torch.uint8, device=self.device)
        self._sync_stream()
        rc = self.lib.trie_encode(self._h, trie._h, ctypes.c_void_p(data.data_ptr()),
                                  ctypes.c_void_p(doc_off.data_ptr()), max(n_docs, 0),
                                  ctypes.c_void_p(ids_out.data_ptr()), cap,
                                  ctypes.c_void_p(id_off.data_ptr()), ctypes.byref(n_ids))
        if rc == -6:
            raise BpeError(rc, f"{n_ids.value} ids needed, capacity {cap}")
        _capi.check(self._h, rc)
        return ids_out[: n_ids.value], id_off[: n_docs + 1]

    def decode(self, merges, ids: torch.Tensor) -> torch.Tensor:
        """Bytes of ids or symbols (int32 CUDA tensor; WORD_START ignored)
        under the vocabulary of ``merges``: a uint8 CUDA tensor."""
        ids = _need_cuda(ids, torch.int32, "ids", self.device)
        arr, n = _merge_array(merges)
        n_bytes = ctypes.c_uint64(0)
        ptr = ctypes.c_void_p(ids.data_ptr() if ids.numel() else 0)
        self._sync_stream()
        rc = self.lib.bpe_decode(self._h, arr, n, ptr, ids.numel(), None, 0, ctypes.byref(n_bytes))
        if rc not in (0, -6):
            _capi.check(self._h, rc)
        out = torch.empty(max(n_bytes.value, 1), dtype=torch.uint8, device=self.device)
        if ids.numel():
            _capi.check(self._h, self.lib.bpe_decode(self._h, arr, n, ptr, ids.numel(),
                                                     ctypes.c_void_p(out.data_ptr()), out.numel(),
                                                     ctypes.byref(n_bytes)))
        return out[: n_bytes.value]


    def unigram(self, trie: Trie, scores, unk_id: int, unk_score: float) -> "Unigram":
        """A Unigram (Viterbi) model over ``trie``: one f64 score per token
        (host array), the id and score of the <unk> fallback."""
        sc = np.ascontiguousarray(scores, dtype=np.float64)
        h = ctypes.c_void_p()
        _capi.check(self._h, self.lib.unigram_create(self._h, trie._h,
                                                     ctypes.c_void_p(sc.ctypes.data if sc.size else 0),
                                                     sc.size, int(unk_id), float(unk_score), ctypes.byref(h)))
        return Unigram(h.value, self.device, trie)

    def unigram_encode(self, model: "Unigram", data: torch.Tensor, doc_off: torch.Tensor | None = None,
                       capacity: int | None = None, ids_out: torch.Tensor | None = None):
        """Most likely segmentation of each document (Viterbi).  Arguments and
        result as ``encode``."""
        data = _need_cuda(data, torch.uint8, "data", self.device)
        if doc_off is None:
            doc_off = torch.tensor([0, data.numel()], dtype=torch.int64, device=self.device)
        doc_off = _need_cuda(doc_off, torch.int64, "doc_off", self.device)
        n_docs = doc_off.numel() - 1
        if ids_out is None:
            cap = data.numel() if capacity is None else capacity
            ids_out = torch.empty(max(cap, 1), dtype=torch.int32, device=self.device)
        else:
            ids_out = _need_cuda(ids_out, torch.int32, "ids_out", self.device)
            cap = ids_out.numel() if capacity is None else min(capacity, ids_out.numel())
        id_off = torch.empty(max(n_docs + 1, 1), dtype=torch.int64, device=self.device)
        n_ids = ctypes.c_uint64(0)
        if data.numel() == 0:
            data = torch.empty(16, dtype=torch.uint8, device=self.device)
        self._sync_stream()
        rc = self.lib.unigram_encode(self._h, model._h, ctypes.c_void_p(data.data_ptr()),
                                     ctypes.c_void_p(doc_off.data_ptr()), max(n_docs, 0),
                                     ctypes.c_void_p(ids_out.data_ptr()), cap,
                                     ctypes.c_void_p(id_off.data_ptr()), ctypes.byref(n_ids))
        if rc == -6:
            raise BpeError(rc, f"{n_ids.value} ids needed, capacity {cap}")
        _capi.check(self._h, rc)
        return ids_out[: n_ids.value], id_off[: n_docs + 1]


class Unigram:
    """A Unigram model on the GPU (see ``Context.unigram``); keeps its trie alive."""

    def __init__(self, handle: int, device: torch.device, trie: Trie):
        self._h = ctypes.c_void_p(handle)
        self.device = device
        self.trie = trie

    def close(self):
        if self._h:
            _capi.load().unigram_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def encode_host(ctx: "Context", trie: "Trie", data, doc_off=None, ids_out=None, id_off_out=None,
                slice_bytes: int = 0):
    """Greedy longest-match ids from host memory (trie_encode_host: the
    copies overlap the encode).  data: uint8 CPU tensor (pinned for overlap);
    doc_off: int64 CPU tensor of n_docs+1 offsets (default: one document).
    Returns (ids int32 CPU tensor, id_off int64 CPU tensor)."""
    if not isinstance(data, torch.Tensor) or data.device.type != "cpu" or data.dtype != torch.uint8:
        raise TypeError("data must be a uint8 CPU tensor")
    if doc_off is None:
        doc_off = torch.tensor([0, data.numel()], dtype=torch.int64)
    doc_off = doc_off.to(torch.int64).contiguous()
    n_docs = doc_off.numel() - 1
    if ids_out is None:
        ids_out = torch.empty(max(data.numel(), 1), dtype=torch.int32, pin_memory=True)
    if id_off_out is None:
        id_off_out = torch.empty(max(n_docs + 1, 1), dtype=torch.int64)
    n = ctypes.c_uint64(0)
    ctx._sync_stream()
    rc = ctx.lib.trie_encode_host(ctx._h, trie._h, ctypes.c_void_p(data.data_ptr() if data.numel() else 0),
                                  ctypes.c_void_p(doc_off.data_ptr()), max(n_docs, 0),
                                  ctypes.c_void_p(ids_out.data_ptr()), ids_out.numel(),
                                  ctypes.c_void_p(id_off_out.data_ptr()), ctypes.byref(n), slice_bytes)
    if rc == -6:
        raise BpeError(rc, f"{n.value} ids needed, capacity {ids_out.numel()}")
    _capi.check(ctx._h, rc)
    return ids_out[: n.value], id_off_out[: n_docs + 1]


class Stream:
    """Streaming encode of one document arriving in slices (trie_stream_*):
    push() returns the ids that no later byte can change; the last push
    returns the rest.  The ids of all pushes, concatenated, equal
    Context.encode on the whole document."""

    def __init__(self, ctx: "Context", trie: Trie):
        self.ctx, self.trie = ctx, trie
        self._h = ctypes.c_void_p()
        _capi.check(ctx._h, ctx.lib.trie_stream_open(ctx._h, trie._h, ctypes.byref(self._h)))

    def push(self, data: torch.Tensor, last: bool = False, ids_out: torch.Tensor | None = None) -> torch.Tensor:
        data = _need_cuda(data, torch.uint8, "data", self.ctx.device)
        cap = data.numel() + self.trie.info()["max_token_len"] + 16   # one id per carried or new byte
        if ids_out is None:
            ids_out = torch.empty(cap, dtype=torch.int32, device=self.ctx.device)
        else:
            ids_out = _need_cuda(ids_out, torch.int32, "ids_out", self.ctx.device)
        n_ids = ctypes.c_uint64(0)
        ptr = data.data_ptr() if data.numel() else 0
        self.ctx._sync_stream()
        rc = self.ctx.lib.trie_stream_push(self._h, ctypes.c_void_p(ptr), data.numel(), 1 if last else 0,
                                           ctypes.c_void_p(ids_out.data_ptr()), ids_out.numel(), ctypes.byref(n_ids))
        if rc == -6:
            raise BpeError(rc, f"{n_ids.value} ids needed, capacity {ids_out.numel()}")
        _capi.check(self.ctx._h, rc)
        return ids_out[: n_ids.value]

    def close(self):
        if self._h:
            self.ctx.lib.trie_stream_close(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _merge_array(merges):
    """(n, 4) uint32 rows (left, right, new_id, count) as a bpe_merge array."""
    m = np.ascontiguousarray(np.asarray(merges, dtype=np.uint32).reshape(-1, 4))
    arr = (_capi.bpe_merge * max(m.shape[0], 1))()
    if m.shape[0]:
        ctypes.memmove(arr, m.ctypes.data, m.nbytes)
    return arr, m.shape[0]


def vocab_from_merges(merges):
    """Token byte strings of ids 0 .. 255 + len(merges), through the library's
    bpe_vocab_from_merges (host only).  Returns (uint8 array, uint64 offsets),
    the layout ``Context.trie_build`` takes."""
    lib = _capi.load()
    arr, n = _merge_array(merges)
    n_bytes = ctypes.c_uint64(0)
    rc = lib.bpe_vocab_from_merges(arr, n, None, 0, None, ctypes.byref(n_bytes))
    if rc not in (0, -6):
        raise BpeError(rc, "bpe_vocab_from_merges: malformed merge table")
    vb = np.empty(max(n_bytes.value, 1), dtype=np.uint8)
    off = np.empty(257 + n, dtype=np.uint64)
    rc = lib.bpe_vocab_from_merges(arr, n, ctypes.c_void_p(vb.ctypes.data), vb.size,
                                   ctypes.c_void_p(off.ctypes.data), ctypes.byref(n_bytes))
    if rc != 0:
        raise BpeError(rc, "bpe_vocab_from_merges failed")
    return vb[: n_bytes.value], off
