"""Write tests/golden/workloads.json: expected results of the CPU oracle on the
five synthetic workloads.

Calls only ``oracle`` (the CPU reference) and ``synth`` (the seeded input
generator); nothing here touches the GPU library.  Arrays are recorded by the
SHA-256 of their little-endian bytes, plus a few leading entries for reading.

    python tests/golden/make_golden.py                 # all workloads
    python tests/golden/make_golden.py tiny med        # a subset (merged in)

Workloads (see ``synth`` for the text recipe):
  tiny   64 KiB corpus, 256 merges (full-stream oracle and word-frequency
         oracle must agree; both are recorded)
  med    16 MiB corpus, 4,096 merges
  large  256 MiB corpus, 32,000 merges (the table itself is also stored,
         as large_merges.npy: rows of left, right, count)
  enc    1 GiB text, greedy encode with the vocabulary learned on ``large``
  batch  512 documents, 250,000-token substring vocabulary, per-document ids
  unigram      the batch documents and vocabulary, Viterbi ids under the
               synthetic scores (synth.unigram_scores; <unk> = the vocabulary
               size, scored synth.unigram_unk_score)
  unigram_doc  the first 64 MiB of the enc text as one document, same model
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "workloads.json")

TRAIN = {  # name -> (merges, checkpoints)
    "tiny": (256, [0, 1, 2, 10, 100, 256]),
    "med": (4096, [0, 1, 2, 10, 100, 1000, 4096]),
    "large": (32000, [0, 1, 2, 10, 100, 1000, 32000]),
}


def sha(a) -> str:
    if isinstance(a, np.ndarray):
        a = np.ascontiguousarray(a).tobytes()
    return hashlib.sha256(a).hexdigest()


def train_record(name: str) -> tuple[dict, np.ndarray]:
    n_merges, cps = TRAIN[name]
    text = synth.corpus(name)
    sym = oracle.pretokenize(text)
    ck = {}

    def cb(k, stream):
        ck[str(k)] = {"n": int(stream.size), "sha256": sha(stream)}

    t0 = time.time()
    merges, final = oracle.train_words(sym, n_merges, checkpoints=cps, callback=cb)
    dt = time.time() - t0
    rec = {
        "corpus_bytes": int(text.size),
        "corpus_sha256": sha(text),
        "symbols_sha256": sha(sym),
        "n_merges": n_merges,
        "n_done": int(merges.shape[0]),
        "merges_sha256": sha(merges.astype(np.uint32)),
        "merges_head": merges[:8].tolist(),
        "merges_tail": merges[-4:].tolist(),
        "n_final": int(final.size),
        "final_sha256": sha(final),
        "checkpoints": ck,
        "oracle": "word-frequency",
        "oracle_seconds": round(dt, 2),
    }
    if name == "tiny":   # the full-stream form must give the same result
        m2, f2 = oracle.train_stream(sym, n_merges)
        assert np.array_equal(m2, merges) and np.array_equal(f2, final)
        rec["oracle"] = "word-frequency == full-stream"
    return rec, merges


def encode_record(name: str, merges_large: np.ndarray | None) -> dict:
    if name == "enc":
        if merges_large is None:
            _, merges_large = train_record("large")
        vb, voff = oracle.vocab_from_merges(merges_large)
        text = synth.corpus("enc")
        doc_off = np.array([0, text.size], dtype=np.uint64)
    else:
        big = synth.corpus("large")
        vb, voff = synth.substring_vocab(big)
        del big
        text, doc_off = synth.batch_documents()
    trie = oracle.Trie(vb, voff)
    t0 = time.time()
    ids, id_off = trie.encode(text, doc_off)
    dt = time.time() - t0
    return {
        "text_bytes": int(text.size),
        "text_sha256": sha(text),
        "n_docs": int(doc_off.size - 1),
        "doc_off_sha256": sha(doc_off.astype(np.uint64)),
        "vocab_size": int(voff.size - 1),
        "vocab_sha256": sha(np.asarray(vb, dtype=np.uint8)),
        "vocab_off_sha256": sha(np.asarray(voff, dtype=np.uint64)),
        "trie_nodes": int(trie.n_nodes),
        "max_token_len": int(trie.max_len),
        "n_ids": int(ids.size),
        "ids_sha256": sha(ids.astype(np.int32)),
        "ids_head": ids[:16].tolist(),
        "id_off_sha256": sha(id_off.astype(np.uint64)),
        "oracle_seconds": round(dt, 2),
    }


UNIGRAM_DOC_BYTES = 64 << 20


def unigram_record(name: str) -> dict:
    big = synth.corpus("large")
    vb, voff = synth.substring_vocab(big)
    del big
    if name == "unigram":
        text, doc_off = synth.batch_documents()
    else:
        text = synth.corpus("enc", UNIGRAM_DOC_BYTES)
        doc_off = np.array([0, text.size], dtype=np.uint64)
    n_tok = int(voff.size - 1)
    scores = synth.unigram_scores(n_tok)
    unk = synth.unigram_unk_score(scores)
    trie = oracle.Trie(vb, voff)
    t0 = time.time()
    ids, id_off = trie.unigram_encode(text, scores, n_tok, unk, doc_off)
    dt = time.time() - t0
    return {
        "text_bytes": int(text.size),
        "text_sha256": sha(text),
        "n_docs": int(doc_off.size - 1),
        "vocab_size": n_tok,
        "vocab_sha256": sha(np.asarray(vb, dtype=np.uint8)),
        "scores_sha256": sha(np.asarray(scores, dtype=np.float64)),
        "unk_id": n_tok,
        "unk_score": unk,
        "n_ids": int(ids.size),
        "n_unk": int((ids == n_tok).sum()),
        "ids_sha256": sha(ids.astype(np.int32)),
        "ids_head": ids[:16].tolist(),
        "id_off_sha256": sha(id_off.astype(np.uint64)),
        "oracle_seconds": round(dt, 2),
    }


def main(names):
    data = {}
    if os.path.exists(OUT):
        with open(OUT) as f:
            data = json.load(f)
    merges_large = None
    for name in names:
        t0 = time.time()
        if name in TRAIN:
            rec, merges = train_record(name)
            if name == "large":
                merges_large = merges
                # (left, right, count) as uint32 for consumers that need the table
                np.save(os.path.join(os.path.dirname(OUT), "large_merges.npy"),
                        merges[:, [0, 1, 3]].astype(np.uint32))
        elif name.startswith("unigram"):
            rec = unigram_record(name)
        else:
            rec = encode_record(name, merges_large)
        data[name] = rec
        data["_about"] = ("Expected results of the CPU oracle (oracle/) on the seeded synth "
                          "workloads; written by tests/golden/make_golden.py.")
        with open(OUT, "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)
        print(f"{name}: {time.time() - t0:.1f}s", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:] or ["tiny", "med", "large", "enc", "batch"])
