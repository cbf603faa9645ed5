#!/usr/bin/env python
"""Benchmark: BPE training merges/s and trie-encode GB/s on one GB300.

One step is one pass of the whole hot path over one batch of synthetic input:
  train leg   pre-tokenize the large corpus (256 MiB, seed 2, 50,000-word
              Turkish-mix lexicon) and run 32,000 merges through the default
              full-stream loop (pair count, argmax, merge of the pair's
              occurrences) and the final compaction of the stream
  encode leg  greedy longest-match encode of 1 GiB of fresh text (seed 3) with
              the 32,256-token vocabulary learned on the large corpus (the
              oracle's stored table, hash-checked)
``value`` is the train leg's merges/s (the large training workload: the
largest training configuration, the one the metric's per-kernel figures are
asked for); the encode leg is reported in ``encode``.  Inputs are resident in
HBM when the timed region starts; L2 is flushed between steps.  The timed
steps replay the merge loop from CUDA graphs as a caller runs it.

Kernel figures (``rooflines``, ``kernels``) come from the same steps run again
with the library's profile option: a CUDA event on the launching stream around
each kernel that runs alone (pair count, list build, compaction, encode), and
event nodes inside the merge loop's graph (its kernels then run without the
launch overlap of the timed replay, so their sum exceeds the replayed loop).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (single-threaded C, pinned to one
core) on the same workload: each step pre-tokenizes the large corpus and runs
the word-frequency oracle's first merges, then its greedy encode of a 64 MiB
sample of the encode text.  N > 1 (torchrun) runs independent replicas, one
per GPU ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BPE train merges/s + trie_encode GB/s on 1 GB300; % of HBM roofline"
TRAIN = {"tiny": 256, "med": 4096, "large": 32000}
ENC_REF_SAMPLE = 64 << 20
REF_MERGES = 200          # word-frequency oracle merges per reference step (a bounded sample)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--train", default="large", choices=sorted(TRAIN))
    ap.add_argument("--encode", default="enc", choices=["enc", "batch", "none"])
    ap.add_argument("--merges", type=int, default=None, help="override the merge count (profiling cases)")
    ap.add_argument("--encode-bytes", type=int, default=None, help="encode only a prefix (profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the extra legs (word-frequency, other sizes, batch)")
    ap.add_argument("--merge-mode", type=int, choices=[0, 1, 2, 3], default=3,
                    help="BPE_OPT_MERGE for the train leg (3 = occurrence lists, the library default)")
    ap.add_argument("--sparse-merge", type=int, choices=[0, 1, 2], default=0,
                    help="BPE_OPT_SPARSE_MERGE (two-pass loop only)")
    ap.add_argument("--leg", choices=["unigram"], default=None,
                    help="run only that leg and print its JSON (profiling)")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


# ----------------------------------------------------------------- clocks ---
class Clocks:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.lines: list[str] = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.idx)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.th:
            self.th.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- helpers ------
def sha(a) -> str:
    import numpy as np
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def golden():
    try:
        with open(os.path.join(ROOT, "tests", "golden", "workloads.json")) as f:
            return json.load(f)
    except Exception:
        return {}


def traffic_record():
    """Per-launch DRAM bytes of each kernel from a committed ncu summary,
    valid only while the kernel's source is unchanged."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except Exception:
        return {}
    out = {}
    for name, r in rec.get("kernels", {}).items():
        src = os.path.join(ROOT, r["source"])
        try:
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        except Exception:
            continue
        if h == r.get("source_sha256"):
            out[name] = r
    return out


def kernel_roofline(stats: dict, fam: str, peak: float, peak_kind: str, traffic: dict, bound: str = "hbm",
                    scale: float = 1.0):
    """Roofline entry of one kernel family: algorithmic bytes per launch (the
    method's bytes, the library's stats) over the average launch duration
    from the profiled pass, times ``scale`` (for the merge loop's kernels: the
    factor that makes the families add up to the timed step).  ``traffic``
    from a committed ncu record of that kernel, scaled to this launch's
    algorithmic bytes, or null."""
    s = stats.get(fam)
    if not s or not s["launches"] or s["ms"] <= 0:
        return None
    ms = s["ms"] * scale
    achieved = s["bytes"] / (ms / 1e3) / 1e9
    per_launch_bytes = s["bytes"] / s["launches"]
    t = traffic.get(fam)
    tr = None
    if t:
        tr = t["dram_bytes"] * per_launch_bytes / t["algorithmic_bytes"] if t.get("scale") else t["dram_bytes"]
    return {"kernel": fam, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": f"of {peak_kind}",
            "traffic": round(tr, 1) if tr is not None else None,
            "algorithmic_bytes_per_launch": round(per_launch_bytes, 1),
            "avg_launch_ms": round(ms / s["launches"], 6), "launches": s["launches"],
            "profiled_avg_launch_ms": round(s["ms"] / s["launches"], 6), "timed_step_scale": round(scale, 4)}


def timed(stream, fn):
    """Run fn() between two CUDA events on the stream; returns (result, ms)."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    r = fn()
    b.record(stream)
    torch.cuda.synchronize()
    return r, a.elapsed_time(b)


def add_stats(acc: dict, st: dict):
    for k, v in st.items():
        if k == "kernel_launches":
            continue
        a = acc.setdefault(k, {"launches": 0, "bytes": 0.0, "ms": 0.0})
        for f in ("launches", "bytes", "ms"):
            a[f] += v[f]


def train_leg(args, ctx, stream, flush, name, steps, warmup):
    """W warm-up and K timed runs of pre-tokenize + full-stream training of a
    named corpus (final stream included), L2 flushed before each; then one
    profiled run for the kernel split."""
    import torch

    import bpe_trie_encode_gb300 as bt
    import synth
    text = synth.corpus(name)
    d_text = torch.from_numpy(text).to(stream.device)
    d_sym = torch.empty(text.size, dtype=torch.int32, device=stream.device)
    n_merges = TRAIN[name]
    ms_all, merges, steps_ms = 0.0, 0, []
    for i in range(warmup + steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        (m, _), ms = timed(stream, lambda: ctx.train(ctx.pretokenize(d_text, out=d_sym), n_merges))
        if i >= warmup:
            ms_all += ms
            merges += m.shape[0]
            steps_ms.append(round(ms, 3))
    ctx.set_option(bt.BPE_OPT_PROFILE, 1)
    ctx.train(ctx.pretokenize(d_text, out=d_sym), n_merges)
    kern = {}
    add_stats(kern, ctx.stats())
    ctx.set_option(bt.BPE_OPT_PROFILE, 0)
    return {"value": round(merges / (ms_all / 1e3), 2), "unit": "merges/s", "ms_per_step": round(ms_all / steps, 3),
            "us_per_merge": round(1e3 * ms_all / max(merges, 1), 3), "steps_ms": steps_ms,
            "workload": f"{name} training: {text.size} B corpus, {n_merges} merges, full stream",
            "kernels": {k: {"launches": v["launches"], "ms": round(v["ms"], 3)} for k, v in kern.items()}}


def extra_legs(args, ctx, dev, stream, flush, peak, peak_kind):
    import numpy as np
    import torch

    import bpe_trie_encode_gb300 as bt
    import synth
    out = {}
    # the medium (16 MiB, 4,096 merges) and tiny (64 KiB, 256 merges) training workloads, full stream
    out["train_med"] = train_leg(args, ctx, stream, flush, "med", args.steps, args.warmup)
    out["train_tiny"] = train_leg(args, ctx, stream, flush, "tiny", args.steps, args.warmup)
    # word-frequency training (the same merges) of the medium and large corpora
    ctx.set_option(bt.BPE_OPT_TRAIN_WORDS, 1)
    for name in ("med", "large"):
        text = synth.corpus(name)
        d_text = torch.from_numpy(text).to(dev)
        d_sym = torch.empty(text.size, dtype=torch.int32, device=dev)
        ctx.train(ctx.pretokenize(d_text, out=d_sym), 200, final=False)   # warm-up
        flush.fill_(1)
        torch.cuda.synchronize()
        (m, _), ms = timed(stream, lambda: ctx.train(ctx.pretokenize(d_text, out=d_sym), TRAIN[name], final=False))
        out[f"train_{name}_words"] = {"value": round(m.shape[0] / (ms / 1e3), 2), "unit": "merges/s",
                                      "ms": round(ms, 3),
                                      "workload": f"{name} training by distinct words: {text.size} B corpus, "
                                                  f"{m.shape[0]} merges (the full-stream merges)"}
        del d_text, d_sym
    ctx.set_option(bt.BPE_OPT_TRAIN_WORDS, 0)
    # the batch encode workload: 512 documents, 250,000-token substring vocabulary
    big = synth.corpus("large")
    vb, voff = synth.substring_vocab(big)
    del big
    data, doc_off = synth.batch_documents()
    trie = ctx.trie_build(vb, voff)
    d_data = torch.from_numpy(data).to(dev)
    d_off = torch.from_numpy(doc_off.astype(np.int64)).to(dev)
    ids = torch.empty(data.size, dtype=torch.int32, device=dev)
    ms_all = 0.0
    for i in range(args.warmup + args.steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        (r, _), ms = timed(stream, lambda: (ctx.encode(trie, d_data, d_off, ids_out=ids), None))
        if i >= args.warmup:
            ms_all += ms
    ctx.set_option(bt.BPE_OPT_PROFILE, 1)
    ctx.encode(trie, d_data, d_off, ids_out=ids)
    kern = {}
    add_stats(kern, ctx.stats())
    ctx.set_option(bt.BPE_OPT_PROFILE, 0)
    call_bytes = data.size + 4 * int(r[0].numel()) + 8 * doc_off.size
    call_gbs = call_bytes / (ms_all / args.steps / 1e3) / 1e9
    out["encode_batch"] = {"value": round(args.steps * data.size / (ms_all / 1e3) / 1e9, 3), "unit": "GB/s",
                           "ms_per_step": round(ms_all / args.steps, 3),
                           "roofline": {"kernel": "trie_encode (whole call)", "bound": "hbm",
                                        "achieved": round(call_gbs, 1), "peak": peak, "unit": "GB/s",
                                        "frac": round(call_gbs / peak, 4), "peak_kind": f"of {peak_kind}",
                                        "algorithmic_bytes_per_call": int(call_bytes)},
                           "workload": f"{doc_off.size - 1} documents, {data.size} B, 250,000-token substring vocabulary",
                           "n_ids": int(r[0].numel()), "trie": trie.info(),
                           "rooflines": {f: kernel_roofline(kern, f, peak, peak_kind, {})
                                         for f in ("encode_spec", "encode_emit")}}
    # the same batch through the bitmap-node trie layout, against the double array above
    ctx.set_option(bt.BPE_OPT_TRIE_LAYOUT, bt.BPE_TRIE_BITMAP)
    ms_bm = 0.0
    for i in range(args.warmup + args.steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        (r2, _), ms = timed(stream, lambda: (ctx.encode(trie, d_data, d_off, ids_out=ids), None))
        if i >= args.warmup:
            ms_bm += ms
    ctx.set_option(bt.BPE_OPT_TRIE_LAYOUT, bt.BPE_TRIE_DOUBLE_ARRAY)
    out["encode_batch_bitmap_layout"] = {
        "value": round(args.steps * data.size / (ms_bm / 1e3) / 1e9, 3), "unit": "GB/s",
        "ms_per_step": round(ms_bm / args.steps, 3), "n_ids": int(r2[0].numel()),
        "vs_double_array": round(ms_all / ms_bm, 3),
        "workload": "the batch encode above with 64-byte bitmap nodes instead of the double array"}
    out["unigram_batch"] = unigram_leg(args, ctx, stream, flush, trie, voff, d_data, d_off, ids, peak, peak_kind,
                                       vb=vb, data=data, doc_off=doc_off)
    out["unigram_doc"] = unigram_doc_leg(args, ctx, stream, flush, trie, voff)
    return out


def unigram_doc_leg(args, ctx, stream, flush, trie, voff):
    """Unigram encoding of one 64 MiB document (the first 64 MiB of the
    encode text) on the batch trie: the single-document case."""
    import torch

    import bpe_trie_encode_gb300 as bt
    import synth
    scores = synth.unigram_scores(voff.size - 1)
    unk = synth.unigram_unk_score(scores)
    model = ctx.unigram(trie, scores, voff.size - 1, unk)
    text = synth.corpus("enc", 64 << 20)
    d = torch.from_numpy(text).to(stream.device)
    ids = torch.empty(text.size, dtype=torch.int32, device=stream.device)
    ms_all = 0.0
    for i in range(args.warmup + args.steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        (r, _), ms = timed(stream, lambda: (ctx.unigram_encode(model, d, ids_out=ids), None))
        if i >= args.warmup:
            ms_all += ms
    ctx.set_option(bt.BPE_OPT_PROFILE, 1)
    ctx.unigram_encode(model, d, ids_out=ids)
    kern = {}
    add_stats(kern, ctx.stats())
    ctx.set_option(bt.BPE_OPT_PROFILE, 0)
    model.close()
    return {"value": round(args.steps * text.size / (ms_all / 1e3) / 1e9, 3), "unit": "GB/s",
            "ms_per_step": round(ms_all / args.steps, 3), "n_ids": int(r[0].numel()),
            "workload": f"one document of {text.size} B (the encode text's first 64 MiB), Viterbi under "
                        "synthetic Zipf log-probabilities, 250,000-token substring vocabulary",
            "kernels": {k: {"launches": v["launches"], "ms": round(v["ms"], 3)} for k, v in kern.items()}}


def unigram_leg(args, ctx, stream, flush, trie, voff, d_data, d_off, ids, peak, peak_kind, vb=None, data=None,
                doc_off=None):
    """Unigram (Viterbi) encoding of the batch documents on the batch trie,
    synthetic float32 Zipf log-probabilities; W warm-up and K timed steps,
    the L2 flushed before each.  With the host copies of the vocabulary and
    documents, the oracle is timed on the first 8 documents (rank 0)."""
    import torch

    import bpe_trie_encode_gb300 as bt
    import synth
    scores = synth.unigram_scores(voff.size - 1)
    unk = synth.unigram_unk_score(scores)
    model = ctx.unigram(trie, scores, voff.size - 1, unk)
    ms_u, kern = 0.0, {}
    ctx.set_option(bt.BPE_OPT_PROFILE, 1)
    for i in range(args.warmup + args.steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        (r3, _), ms = timed(stream, lambda: (ctx.unigram_encode(model, d_data, d_off, ids_out=ids), None))
        if i >= args.warmup:
            ms_u += ms
            for k2, v in ctx.stats().items():
                if k2 != "kernel_launches":
                    a = kern.setdefault(k2, {"launches": 0, "bytes": 0.0, "ms": 0.0})
                    for f in ("launches", "bytes", "ms"):
                        a[f] += v[f]
    ctx.set_option(bt.BPE_OPT_PROFILE, 0)
    model.close()
    nbytes = d_data.numel()
    fwd = kern.get("unigram_fwd", {"ms": 0.0, "launches": 1})
    fwd_ms = fwd["ms"] / max(fwd["launches"], 1)
    fwd_gbs = 5.0 * nbytes / (fwd_ms / 1e3) / 1e9 if fwd_ms else 0.0
    cpu = None
    if vb is not None and not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        import oracle
        n8 = int(doc_off[8])
        t0 = time.perf_counter()
        oracle.Trie(vb, voff).unigram_encode(data[:n8], scores, voff.size - 1, unk, doc_off[:9])
        dt = time.perf_counter() - t0
        cpu = {"value": round(n8 / dt / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"the first 8 documents ({n8} B), same model, single thread, {cpu_model()}",
               "seconds": round(dt, 2)}
    return {
        "value": round(args.steps * nbytes / (ms_u / 1e3) / 1e9, 3), "unit": "GB/s",
        "ms_per_step": round(ms_u / args.steps, 3), "n_ids": int(r3[0].numel()),
        "cpu_baseline": cpu,
        "workload": "the batch documents, most likely segmentation (Viterbi) under synthetic Zipf "
                    "log-probabilities (float32) for the 250,000 tokens",
        "kernels": {k2: {"launches": v["launches"], "ms": round(v["ms"], 3)} for k2, v in kern.items()},
        # the forward recurrence is bound by dependent trie-walk loads and integer
        # issue (ncu: ALU pipe ~53 %, issue ~72 % active), not by DRAM: its
        # algorithmic traffic -- text read, 4-byte back pointer per byte written --
        # over its duration is a small fraction of the copy bandwidth
        "fwd_hbm": {"bound": "latency/alu", "achieved": round(fwd_gbs, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(fwd_gbs / peak, 4), "peak_kind": f"of {peak_kind}",
                    "algorithmic_bytes_per_byte": 5.0},
    }


def run_unigram_only(args):
    """bench.py --leg unigram: only the Unigram leg (profiling and quick runs)."""
    import numpy as np
    import torch

    import bpe_trie_encode_gb300 as bt
    import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ctx = bt.Context(0)
    peak, peak_kind = peaks()
    big = synth.corpus("large")
    vb, voff = synth.substring_vocab(big)
    del big
    data, doc_off = synth.batch_documents()
    trie = ctx.trie_build(vb, voff)
    d_data = torch.from_numpy(data).to(dev)
    d_off = torch.from_numpy(doc_off.astype(np.int64)).to(dev)
    ids = torch.empty(data.size, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = unigram_leg(args, ctx, torch.cuda.current_stream(dev), flush, trie, voff, d_data, d_off, ids, peak,
                      peak_kind, vb=vb, data=data, doc_off=doc_off)
    out = {"leg": "unigram_batch", **out}
    ctx.close()
    return out


# ------------------------------------------------------------ ranks ---------
def reduce_ranks(times_ms: list, units: list, world: int, device) -> tuple[list, list]:
    """Whole-job figures over all ranks: the slowest rank's time for each
    entry of times_ms and the sum of units (merges, bytes) over ranks.  The
    tensors live on ``device`` (the GPU for NCCL, the CPU for gloo)."""
    if world <= 1:
        return [float(x) for x in times_ms], [float(x) for x in units]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    u = torch.tensor([float(x) for x in units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.cpu()], [float(x) for x in u.cpu()]


def throughput(units: float, ms: float) -> float:
    """Units per second from a duration in milliseconds (0 for no time)."""
    return units / (ms / 1e3) if ms > 0 else 0.0


# ---------------------------------------------------------------- ours ------
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    import bpe_trie_encode_gb300 as bt
    import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    ctx = bt.Context(local_rank)
    ctx.set_option(bt.BPE_OPT_MERGE, args.merge_mode)
    ctx.set_option(bt.BPE_OPT_SPARSE_MERGE, args.sparse_merge)
    peak, peak_kind = peaks()
    n_merges = args.merges or TRAIN[args.train]

    # ---- set-up (untimed)
    text = synth.corpus(args.train)
    h_text = torch.from_numpy(text.copy()).pin_memory()
    d_text = h_text.to(dev)
    d_sym = torch.empty(text.size, dtype=torch.int32, device=dev)
    enc = None
    vocab_check = None
    if args.encode != "none":
        if args.encode == "enc":
            m_big = large_merges_for_reference()       # the oracle's table (stored copy, hash checked)
            vocab_check = "the oracle's merge table of the large corpus"
            vb, voff = bt.vocab_from_merges(m_big)
            etext = synth.corpus("enc", args.encode_bytes)
            doc_off = np.array([0, etext.size], dtype=np.int64)
            wl = (f"{etext.size} B text (seed 3), 32,256-token vocabulary learned on the large corpus, "
                  "one document")
        else:
            big = synth.corpus("large")
            vb, voff = synth.substring_vocab(big)
            del big
            etext, doc_off = synth.batch_documents()
            doc_off = doc_off.astype(np.int64)
            vocab_check = "generator vocabulary"
            wl = "512 documents of >= 64 KiB (seed 4), 250,000-token substring vocabulary"
        trie = ctx.trie_build(vb, voff)
        h_enc = torch.from_numpy(etext).pin_memory()
        enc = {"trie": trie, "vb": vb, "voff": voff, "h": h_enc, "d": h_enc.to(dev),
               "h_off": torch.from_numpy(doc_off).pin_memory(), "d_off": torch.from_numpy(doc_off).to(dev),
               "workload": wl, "bytes": int(etext.size),
               "ids": torch.empty(int(etext.size), dtype=torch.int32, device=dev),
               # the end-to-end leg's host outputs, pinned at set-up next to its inputs
               "h_ids": torch.empty(int(etext.size), dtype=torch.int32, pin_memory=True),
               "h_ioff": torch.empty(doc_off.size, dtype=torch.int64)}
        del etext
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(timed_step: bool, acc: dict):
        flush.fill_(1)                         # L2 flush between steps (> 129 MB written)
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        ctx.pretokenize(d_text, out=d_sym)
        m, fin = ctx.train(d_sym, n_merges)    # the merge table and the final stream
        st_train = ctx.stats()
        e1.record(stream)
        st_enc = None
        n_ids = 0
        if enc:
            ids, _ = ctx.encode(enc["trie"], enc["d"], enc["d_off"], ids_out=enc["ids"])
            n_ids = ids.numel()
            st_enc = ctx.stats()
        e2.record(stream)
        torch.cuda.synchronize(dev)
        if timed_step:
            acc["train_ms"] += e0.elapsed_time(e1)
            acc["enc_ms"] += e1.elapsed_time(e2)
            acc["steps_ms"].append(round(e0.elapsed_time(e1), 3))
            acc["merges"] += m.shape[0]
            acc["launches"] += 1 + st_train["kernel_launches"] + (st_enc["kernel_launches"] if st_enc else 0)
            add_stats(acc["kern"], st_train)
            add_stats(acc["kern"], st_enc or {})
            acc["n_ids"] = n_ids
            acc["n_final"] = int(fin.numel())

    def fresh():
        return {"train_ms": 0.0, "enc_ms": 0.0, "merges": 0, "launches": 0, "kern": {}, "n_ids": 0,
                "steps_ms": [], "n_final": 0}

    # timed steps: graph replay, as a caller runs it
    for _ in range(args.warmup):
        step(False, fresh())
    acc = fresh()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = Clocks(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    for _ in range(args.steps):
        step(True, acc)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    # per-kernel device time: the same steps again with the profile option
    ctx.set_option(bt.BPE_OPT_PROFILE, 1)
    prof = fresh()
    step(False, prof)
    for _ in range(max(1, min(args.steps, 2))):
        step(True, prof)
    ctx.set_option(bt.BPE_OPT_PROFILE, 0)
    kern = prof["kern"]

    (train_ms, enc_ms), (merges_total, enc_bytes_total) = reduce_ranks(
        [acc["train_ms"], acc["enc_ms"]], [acc["merges"], enc["bytes"] * args.steps if enc else 0], world, dev)
    value = throughput(merges_total, train_ms)

    # ---- end to end through host buffers (graph replay, no profiling)
    e2e = None
    if not args.no_e2e:
        h_merges_bytes = n_merges * 16
        if enc:   # pinned host outputs of the end-to-end encode
            h_ids_buf, h_ioff_buf = enc["h_ids"], enc["h_ioff"]
        link = None
        if enc:   # the host link's own copy speed in this run: what bounds the end-to-end encode
            n_cp = max(acc["n_ids"], 1)
            h2d, d2h = [], []
            for _ in range(3):
                _, ms = timed(stream, lambda: enc["d"].copy_(enc["h"], non_blocking=True))
                h2d.append(enc["bytes"] / (ms / 1e3) / 1e9)
                _, ms = timed(stream, lambda: h_ids_buf[:n_cp].copy_(enc["ids"][:n_cp], non_blocking=True))
                d2h.append(4 * n_cp / (ms / 1e3) / 1e9)
            link = {"h2d_GBs": round(sorted(h2d)[1], 1), "d2h_GBs": round(sorted(d2h)[1], 1),
                    "copy_bound_ms": round(max(enc["bytes"] / sorted(h2d)[1], 4 * n_cp / sorted(d2h)[1]) / 1e6, 3)}
        tr_ms = en_ms = 0.0
        d2h_ids = 0
        en_steps = []
        for i in range(args.warmup + args.steps):
            flush.fill_(1)
            torch.cuda.synchronize(dev)
            a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            a.record(stream)
            dt = h_text.to(dev, non_blocking=True)
            ctx.pretokenize(dt, out=d_sym)
            m, _ = ctx.train(d_sym, n_merges, final=False)     # the merge table returns to the host
            b.record(stream)
            if enc:   # host buffers in and out through trie_encode_host (copies overlap the encode)
                h_ids, h_io = bt.encode_host(ctx, enc["trie"], enc["h"], enc["h_off"], ids_out=h_ids_buf,
                                             id_off_out=h_ioff_buf)
                d2h_ids = h_ids.numel() * 4 + h_io.numel() * 8
            c.record(stream)
            torch.cuda.synchronize(dev)
            if i >= args.warmup:
                tr_ms += a.elapsed_time(b)
                en_ms += b.elapsed_time(c)
                en_steps.append(round(b.elapsed_time(c), 2))
        (tr_ms, en_ms), (e2e_merges, e2e_bytes) = reduce_ranks(
            [tr_ms, en_ms], [args.steps * m.shape[0], args.steps * enc["bytes"] if enc else 0], world, dev)
        e2e = {"value": round(throughput(e2e_merges, tr_ms), 2), "unit": "merges/s",
               "h2d_bytes_per_step": int(text.size + (enc["bytes"] + enc["h_off"].numel() * 8 if enc else 0)),
               "d2h_bytes_per_step": int(h_merges_bytes + d2h_ids)}
        if enc:
            e2e["encode"] = {"value": round(throughput(e2e_bytes, en_ms) / 1e9, 3), "unit": "GB/s",
                             "steps_ms": en_steps,
                             "median_GBs": round(enc["bytes"] / (sorted(en_steps)[len(en_steps) // 2] / 1e3) / 1e9, 3)
                             if en_steps else None,
                             "mean_over_median": round((sum(en_steps) / len(en_steps)) /
                                                       sorted(en_steps)[len(en_steps) // 2], 3) if en_steps else None,
                             "host_link": link}

    # ---- extra legs: other training sizes, the word-frequency trainer (same
    # merges), the batch encode workload, Unigram
    extra = {}
    if not args.no_extra:
        extra = extra_legs(args, ctx, dev, stream, flush, peak, peak_kind)

    # ---- CPU baseline: the oracle as it stands, rank 0, N == 1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, text, enc, n_merges)

    if rank != 0:
        return None
    traffic = traffic_record()
    loop = ("merge_tail", "merge_scan", "merge_apply")
    loop_ms = sum(kern.get(f, {"ms": 0.0})["ms"] for f in loop)
    # The stand-alone kernels' times are exact (an event on each side). The
    # merge loop's kernels were profiled with event nodes between them, which
    # adds to each; their times are scaled so that, with the stand-alone ones,
    # they add up to the timed train leg.
    n_prof = max(1, min(args.steps, 2))
    alone = sum(kern.get(f, {"ms": 0.0})["ms"] for f in ("pair_count", "list_build", "compact")) / n_prof
    sc_loop = (train_ms / args.steps - alone) / (loop_ms / n_prof) if loop_ms > 0 else 1.0
    rooflines = {f: kernel_roofline(kern, f, peak, peak_kind, traffic, scale=sc_loop if f in loop else 1.0)
                 for f in ("pair_count", "list_build", "compact", "encode_spec", "encode_emit") + loop}
    # the timed step's dominant kernel: the merge loop's tail (most merges run there)
    dom = max((f for f in rooflines if rooflines[f]), key=lambda f: kern[f]["ms"])
    for f in loop:   # what the HBM fraction of the merge kernels means
        if rooflines.get(f):
            rooflines[f]["note"] = ("latency-bound: a chain of dependent gathers and barriers per merge "
                                    "(one CTA for the tail); HBM is nearly idle")
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "merges/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round((train_ms + enc_ms) / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic (seeded generator)",
        "config": {"workload": f"{args.train} training: {text.size} B corpus, {n_merges} merges, full stream "
                               f"(final compaction included); encode leg: {enc['workload'] if enc else 'none'}",
                   "train_corpus_bytes": int(text.size), "n_merges": n_merges,
                   "l2": "flushed between steps (256 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "vocab": vocab_check, "merge_mode": args.merge_mode, "sparse_merge": args.sparse_merge},
        "train": {"value": round(value, 2), "unit": "merges/s", "ms_per_step": round(train_ms / args.steps, 3),
                  "us_per_merge": round(1e3 * train_ms / max(merges_total, 1), 3), "steps_ms": acc["steps_ms"],
                  "n_final": acc["n_final"]},
        "roofline": rooflines[dom],
        "rooflines": rooflines,
        "gpu_launches": acc["launches"],
        "timing": ("value, e2e: CUDA events around each step, the merge loop replayed from CUDA graphs; "
                   "kernels and rooflines: a separate profiled pass of the same "
                   "steps (events around each stand-alone kernel, event nodes between the merge loop's kernels; "
                   "the loop's family times scaled by timed_step_scale so that all families add up to the "
                   "timed train leg)"),
        "profiled_merge_loop_ms_per_step": round(loop_ms / max(1, min(args.steps, 2)), 3),
        "kernels": {k: {"launches": v["launches"], "ms": round(v["ms"], 3),
                        "GB/s": round(v["bytes"] / (v["ms"] / 1e3) / 1e9, 1) if v["ms"] else None}
                    for k, v in kern.items()},
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    out.update(extra)
    if enc:
        gbs = throughput(enc_bytes_total, enc_ms) / 1e9
        # the whole call against HBM: its algorithmic bytes are the input once,
        # 4 per id and 8 per document offset
        call_bytes = enc["bytes"] + 4 * acc["n_ids"] + 8 * enc["h_off"].numel()
        call_gbs = call_bytes / (enc_ms / args.steps / 1e3) / 1e9
        out["encode"] = {"value": round(gbs, 3), "unit": "GB/s", "ms_per_step": round(enc_ms / args.steps, 3),
                         "workload": enc["workload"], "n_ids": acc["n_ids"],
                         "roofline": {"kernel": "trie_encode (whole call)", "bound": "hbm",
                                      "achieved": round(call_gbs, 1), "peak": peak, "unit": "GB/s",
                                      "frac": round(call_gbs / peak, 4), "peak_kind": f"of {peak_kind}",
                                      "algorithmic_bytes_per_call": int(call_bytes)},
                         "rooflines": {f: rooflines[f] for f in ("encode_spec", "encode_emit")}}
    return out


class one_core:
    """Pin this process to one host core while the oracle runs (the pages'
    measurement method: single-threaded, one pinned core), restoring the
    previous affinity afterwards."""

    def __enter__(self):
        self.before = None
        self.core = None
        try:
            self.before = os.sched_getaffinity(0)
            self.core = max(self.before)
            os.sched_setaffinity(0, {self.core})
        except (AttributeError, OSError):
            pass
        return self

    def __exit__(self, *exc):
        if self.before is not None:
            try:
                os.sched_setaffinity(0, self.before)
            except OSError:
                pass
        return False

    def info(self) -> dict:
        return {"affinity": [self.core] if self.core is not None else None, "nproc": os.cpu_count(),
                "cpu_model": cpu_model()}


def cpu_baseline(args, text, enc, n_merges):
    """The oracle as it stands, single-threaded and pinned to one core, on
    bounded samples: the word-frequency form on the headline workload's first
    merges (``value``); the full-stream form (like for like with the GPU loop)
    on the tiny workload in full and on the medium workload's first merges;
    and the greedy encode of the first 64 MiB of the encode text."""
    import oracle
    import synth

    with one_core() as pin:
        t0 = time.perf_counter()
        sym = oracle.pretokenize(text)
        m, _ = oracle.train_words(sym, min(REF_MERGES, n_merges))
        dt = time.perf_counter() - t0
        out = {"value": round(m.shape[0] / dt, 3), "unit": "merges/s", "cores": 1, "kind": "oracle",
               "sample": f"{args.train} training, pre-tokenize + the first {m.shape[0]} merges "
                         f"({text.size} B corpus), word-frequency oracle, single thread",
               "seconds": round(dt, 2), **pin.info()}
        tiny = oracle.pretokenize(synth.corpus("tiny"))
        t0 = time.perf_counter()
        mt, _ = oracle.train_stream(tiny, TRAIN["tiny"])
        dt = time.perf_counter() - t0
        out["full_stream_tiny"] = {"value": round(mt.shape[0] / dt, 2), "unit": "merges/s",
                                   "ms_per_merge": round(1e3 * dt / max(mt.shape[0], 1), 3),
                                   "sample": f"tiny training in full ({tiny.size} symbols, {mt.shape[0]} merges), "
                                             "full-stream oracle"}
        med = oracle.pretokenize(synth.corpus("med"))
        t0 = time.perf_counter()
        mm, _ = oracle.train_stream(med, 4)
        dt = time.perf_counter() - t0
        out["full_stream_med"] = {"value": round(mm.shape[0] / dt, 4), "unit": "merges/s",
                                  "sample": f"medium training, the first {mm.shape[0]} merges of {med.size} "
                                            "symbols, full-stream oracle (each merge costs about the same)"}
        if enc:
            sample = enc["h"][:ENC_REF_SAMPLE].numpy()
            trie = oracle.Trie(enc["vb"], enc["voff"])
            t0 = time.perf_counter()
            trie.encode(sample)
            dt = time.perf_counter() - t0
            out["encode"] = {"value": round(sample.size / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
                             "sample": f"first {sample.size} B of the encode text, same vocabulary"}
    return out


def large_merges_for_reference():
    """The oracle's merge table of the large corpus: the stored copy written by
    tests/golden/make_golden.py (checked by hash), else a fresh oracle run."""
    import numpy as np

    import oracle
    import synth
    g = golden().get("large", {})
    p = os.path.join(ROOT, "tests", "golden", "large_merges.npy")
    if os.path.exists(p) and g:
        lr = np.load(p).astype(np.uint32)
        m = np.zeros((lr.shape[0], 4), dtype=np.uint32)
        m[:, :2] = lr[:, :2]
        m[:, 2] = 256 + np.arange(lr.shape[0], dtype=np.uint32)
        m[:, 3] = lr[:, 2]
        if sha(m) == g.get("merges_sha256"):
            return m
    m, _ = oracle.train_words(oracle.pretokenize(synth.corpus("large")), TRAIN["large"])
    return m


def encode_reference_sample(args):
    """(vocab bytes, offsets, sample text, doc offsets) for the oracle's encode leg."""
    import numpy as np

    import oracle
    import synth
    if args.encode == "enc":
        vb, voff = oracle.vocab_from_merges(large_merges_for_reference())
        text = synth.corpus("enc", ENC_REF_SAMPLE)
        doc_off = np.array([0, text.size], dtype=np.uint64)
    else:
        big = synth.corpus("large")
        vb, voff = synth.substring_vocab(big)
        text, doc_off = synth.batch_documents(64)
    return vb, voff, text, doc_off


# ---------------------------------------------------------- reference -------
def run_reference(args, rank, world):
    """The CPU oracle on the same workload, pinned to one core: each step
    pre-tokenizes the training corpus and runs the word-frequency oracle's
    first merges (a bounded sample), then its greedy encode of a 64 MiB sample
    of the encode text."""
    import oracle
    import synth
    if rank != 0:
        return None
    n_merges = min(REF_MERGES, TRAIN[args.train])
    text = synth.corpus(args.train)
    enc = None
    if args.encode != "none":
        vb, voff, etext, doc_off = encode_reference_sample(args)
        enc = (oracle.Trie(vb, voff), etext, doc_off)

    def step():
        t0 = time.perf_counter()
        m, _ = oracle.train_words(oracle.pretokenize(text), n_merges)
        t1 = time.perf_counter()
        if enc:
            enc[0].encode(enc[1], enc[2])
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1, m.shape[0]

    with one_core() as pin:
        for _ in range(args.warmup):
            step()
        tr = en = 0.0
        merges = 0
        for _ in range(args.steps):
            a, b, m = step()
            tr += a
            en += b
            merges += m
    value = merges / tr
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "merges/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round((tr + en) / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
           "data": "synthetic (seeded generator)",
           "config": {"workload": f"{args.train} training: {text.size} B corpus, pre-tokenize + the first "
                                  f"{n_merges} merges per step; encode leg: {args.encode} "
                                  f"({'64 MiB sample' if args.encode == 'enc' else '64 documents'})",
                      "parallelism": "CPU oracle, rank 0 only"},
           "cpu_baseline": {"value": round(value, 3), "unit": "merges/s", "cores": 1, "kind": "oracle",
                            "sample": f"{args.train} training, pre-tokenize + the first {n_merges} merges per "
                                      "step, word-frequency oracle, single thread", **pin.info()},
           "e2e": {"value": round(value, 3), "unit": "merges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if enc:
        out["encode"] = {"value": round(args.steps * enc[1].size / en / 1e9, 4), "unit": "GB/s",
                         "sample_bytes": int(enc[1].size)}
    return out


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.leg == "unigram":
        out = run_unigram_only(args) if rank == 0 else None
    elif args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        import torch
        import torch.distributed as dist
        if world > 1:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            dist.destroy_process_group()
    if out is not None and rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
