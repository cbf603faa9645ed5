// internal.h -- context, scratch pool and error plumbing shared by the
// translation units of libbpetrie.so.  Host-side only (no device code).
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>
#include <vector>

#include "bpetrie.h"

namespace bpe {

// Named scratch slots of the context's pool.
enum Slot {
    S_TRAIN_BUF0, S_TRAIN_BUF1, S_TABLE_KEY, S_TABLE_CNT, S_LIST0, S_LIST1,
    S_STATUS0, S_STATUS1, S_BEST, S_STATE, S_NHIST,
    S_ENC_CHUNK_START, S_ENC_CHUNK_INFO, S_ENC_NOTOK, S_ENC_STATUS, S_ENC_PREFIX, S_ENC_STATE, S_ENC_SIDS,
    S_ENC_SBITS, S_HOST_IN0, S_HOST_IN1, S_HOST_OUT0, S_HOST_OUT1, S_HOST_OFF0, S_HOST_OFF1,
    S_W_BSUM, S_W_START, S_W_OCCSLOT, S_W_TABLE, S_W_UID, S_W_UINFO, S_W_SYM, S_W_OUTOFF,
    S_UNI_START, S_UNI_STATE, S_UNI_BACK, S_UNI_GBACK, S_UNI_CHUNK, S_UNI_FLAG, S_UNI_PREFIX, S_UNI_STATUS,
    S_UNI_TSTART,
    S_SPARSE_OCC,
    S_DEC_TOK, S_DEC_OFF, S_DEC_BSUM, S_DEC_STATE,
    S_L_STATE, S_L_OCC, S_L_EKEY, S_L_ECNT, S_L_ELEN, S_L_EOFF, S_L_VLEN, S_L_BFILL, S_L_EBEST, S_L_FRONT,
    S_L_HSLOT, S_L_HCNT, S_L_HENT, S_L_NS, S_L_CAND, S_L_APP, S_L_REC, S_L_CSTAT, S_L_KMODE, S_L_CBAR, S_L_CTILE,
    S_NUM
};

struct Scratch {
    void *p = nullptr;
    size_t cap = 0;
};

struct TrainGraph {
    cudaGraphExec_t exec = nullptr;
    // what the capture baked in; a mismatch forces a new capture
    std::vector<uintptr_t> key;
};

struct bpe_ctx_impl;

}  // namespace bpe

struct bpe_ctx {
    int device = 0;
    cudaStream_t stream = nullptr;
    cudaStream_t capture_stream = nullptr;  // private stream used only to capture graphs
    int sm_count = 0;
    std::string err;
    bpe::Scratch scratch[bpe::S_NUM];
    void *pinned = nullptr;                 // small pinned host staging area
    size_t pinned_cap = 0;
    // options
    int table_log2 = 0;
    int use_graph = 1;
    int profile = 0;
    int chunk = 256;   // trie_encode bytes per chunk (measured best on both encode workloads)
    int train_words = 0;
    int merge_mode = BPE_MERGE_LISTS;   // BPE_MERGE_*
    int persistent = 0;
    int sparse_merge = 0;   // BPE_OPT_SPARSE_MERGE
    int list_frontier = 0;  // BPE_OPT_LIST_FRONTIER (0: default)
    int list_tail = -1;     // BPE_OPT_LIST_TAIL (-1: default)
    int trie_layout = 0;   // BPE_TRIE_*
    int uni_chunk = 0;     // unigram_encode chunk bytes (0: default)
    long long test_stall_tile = -1;   // BPE_OPT_TEST_STALL_TILE
    // cached graph of merge iterations
    bpe::TrainGraph graph;
    bpe::TrainGraph graph_sparse;   // the same for occurrence-driven merge windows
    bpe::TrainGraph graph_lists;    // the same for the occurrence-list merge loop
    // profiling events (grown on demand)
    std::vector<cudaEvent_t> events;
    bpe_stats stats{};
    uint64_t pretok_launches = 0;   // running count of pre-tokenize launches
    // host pipeline of trie_encode_host, created on first use and kept: its
    // two copy streams, six events, pinned staging, and the streaming state
    // for documents longer than a slice (for one trie and longest-token length)
    cudaStream_t pipe_h2d = nullptr, pipe_d2h = nullptr;
    cudaEvent_t pipe_ev[6] = {};
    void *pipe_pinned = nullptr;
    size_t pipe_pinned_cap = 0;
    bpe_stream *pipe_stream = nullptr;
    const bpe_trie *pipe_trie = nullptr;
    uint32_t pipe_max_len = 0;
};

namespace bpe {

// Set ctx->err from a printf-style message and return `code`.
int fail(bpe_ctx *ctx, int code, const char *fmt, ...);

// Map a CUDA error to BPE_ERR_CUDA (or OOM) with context.
int cuda_fail(bpe_ctx *ctx, cudaError_t e, const char *what);

// Make scratch slot `s` at least `bytes` large (growth x1.5, contents are
// not preserved).  Waits for the context stream before freeing old storage.
int ensure(bpe_ctx *ctx, Slot s, size_t bytes, void **out);

// Pinned host staging of at least `bytes`.
int ensure_pinned(bpe_ctx *ctx, size_t bytes, void **out);

// Make sure ctx->events holds at least n timing events.
int ensure_events(bpe_ctx *ctx, size_t n);

// Stats helpers.
void stats_reset(bpe_ctx *ctx);
int stats_slot(bpe_ctx *ctx, const char *name);

// The bitmap-node layout of a trie, built on its first use (kept with the trie).
int trie_bitmap_nodes(bpe_ctx *ctx, const bpe_trie *trie);

// The merge loop over per-pair occurrence lists (train_lists.cu).  Needs
// byte-level input (ids < 256); *not_bytes is set, with nothing done, when a
// symbol is not one.
int train_lists(bpe_ctx *ctx, const uint32_t *d_symbols, uint64_t n, uint32_t n_merges, bpe_merge *h_merges_out,
                uint32_t *n_done, uint32_t *d_symbols_final, uint64_t *n_final, bool *not_bytes);

// Forget a stream's carried bytes (start a new document).
void stream_reset(bpe_stream *st);

// Streaming push of a slice with writable headroom of the trie's longest
// token length before it (the carried bytes are placed there).
int stream_push_in_place(bpe_stream *st, uint8_t *d_slice, uint64_t n, int last, int32_t *d_ids_out,
                         uint64_t ids_capacity, uint64_t *n_ids);

}  // namespace bpe

#define BPE_CUDA(ctx, call, what)                                  \
    do {                                                           \
        cudaError_t e__ = (call);                                  \
        if (e__ != cudaSuccess) return bpe::cuda_fail(ctx, e__, what); \
    } while (0)
