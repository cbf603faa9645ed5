// context.cpp -- bpe_ctx life cycle, options, errors, the scratch pool.
//
// The pool follows the persistent-buffer idea of [GPU-BPE] "Host
// architecture", 2.: buffers are made once and reused by later calls; a call
// that needs more grows the buffer to 1.5x the request.
#include <cstring>

#include "internal.h"

namespace bpe {

int fail(bpe_ctx *ctx, int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (ctx) ctx->err = buf;
    return code;
}

int cuda_fail(bpe_ctx *ctx, cudaError_t e, const char *what) {
    int code = (e == cudaErrorMemoryAllocation) ? BPE_ERR_OOM : BPE_ERR_CUDA;
    return fail(ctx, code, "%s: %s", what, cudaGetErrorString(e));
}

int ensure(bpe_ctx *ctx, Slot s, size_t bytes, void **out) {
    Scratch &sc = ctx->scratch[s];
    if (bytes == 0) bytes = 256;
    if (sc.cap < bytes) {
        if (sc.p) {
            BPE_CUDA(ctx, cudaStreamSynchronize(ctx->stream), "scratch grow: stream sync");
            cudaFree(sc.p);
            sc.p = nullptr;
            sc.cap = 0;
        }
        size_t want = bytes + bytes / 2;
        want = (want + 255) & ~size_t(255);
        void *p = nullptr;
        cudaError_t e = cudaMalloc(&p, want);
        if (e != cudaSuccess) {
            cudaGetLastError();
            want = (bytes + 255) & ~size_t(255);   // retry without headroom
            e = cudaMalloc(&p, want);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(ctx, BPE_ERR_OOM, "scratch: cudaMalloc of %zu bytes failed", want);
            }
        }
        sc.p = p;
        sc.cap = want;
        ctx->graph.key.clear();                    // pointers changed: recapture
        ctx->graph_sparse.key.clear();
        ctx->graph_lists.key.clear();
    }
    *out = sc.p;
    return BPE_OK;
}

int ensure_pinned(bpe_ctx *ctx, size_t bytes, void **out) {
    if (ctx->pinned_cap < bytes) {
        if (ctx->pinned) {
            BPE_CUDA(ctx, cudaStreamSynchronize(ctx->stream), "pinned grow: stream sync");
            cudaFreeHost(ctx->pinned);
            ctx->pinned = nullptr;
            ctx->pinned_cap = 0;
        }
        size_t want = bytes + bytes / 2 + 4096;
        BPE_CUDA(ctx, cudaMallocHost(&ctx->pinned, want), "cudaMallocHost");
        ctx->pinned_cap = want;
    }
    *out = ctx->pinned;
    return BPE_OK;
}

int ensure_events(bpe_ctx *ctx, size_t n) {
    while (ctx->events.size() < n) {
        cudaEvent_t ev;
        BPE_CUDA(ctx, cudaEventCreate(&ev), "cudaEventCreate");
        ctx->events.push_back(ev);
    }
    return BPE_OK;
}

void stats_reset(bpe_ctx *ctx) { memset(&ctx->stats, 0, sizeof ctx->stats); }

int stats_slot(bpe_ctx *ctx, const char *name) {
    for (int i = 0; i < ctx->stats.n; i++)
        if (!strcmp(ctx->stats.k[i].name, name)) return i;
    if (ctx->stats.n == BPE_MAX_STATS) return BPE_MAX_STATS - 1;
    int i = ctx->stats.n++;
    snprintf(ctx->stats.k[i].name, sizeof ctx->stats.k[i].name, "%s", name);
    return i;
}

}  // namespace bpe

using namespace bpe;

extern "C" int bpe_ctx_create(bpe_ctx **out, int device, void *cuda_stream) {
    if (!out) return BPE_ERR_INVALID_ARG;
    *out = nullptr;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) {
        cudaGetLastError();
        return BPE_ERR_INVALID_ARG;
    }
    bpe_ctx *ctx = new bpe_ctx();
    ctx->device = device;
    ctx->stream = (cudaStream_t)cuda_stream;
    cudaError_t e = cudaSetDevice(device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ctx->capture_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        delete ctx;
        return BPE_ERR_CUDA;
    }
    *out = ctx;
    return BPE_OK;
}

extern "C" int bpe_ctx_set_stream(bpe_ctx *ctx, void *cuda_stream) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    ctx->stream = (cudaStream_t)cuda_stream;
    return BPE_OK;
}

extern "C" void bpe_ctx_destroy(bpe_ctx *ctx) {
    if (!ctx) return;
    cudaSetDevice(ctx->device);
    cudaStreamSynchronize(ctx->stream);
    if (ctx->pipe_stream) trie_stream_close(ctx->pipe_stream);
    if (ctx->pipe_h2d) cudaStreamSynchronize(ctx->pipe_h2d);
    if (ctx->pipe_d2h) cudaStreamSynchronize(ctx->pipe_d2h);
    for (auto ev : ctx->pipe_ev)
        if (ev) cudaEventDestroy(ev);
    if (ctx->pipe_h2d) cudaStreamDestroy(ctx->pipe_h2d);
    if (ctx->pipe_d2h) cudaStreamDestroy(ctx->pipe_d2h);
    if (ctx->pipe_pinned) cudaFreeHost(ctx->pipe_pinned);
    if (ctx->graph.exec) cudaGraphExecDestroy(ctx->graph.exec);
    if (ctx->graph_sparse.exec) cudaGraphExecDestroy(ctx->graph_sparse.exec);
    if (ctx->graph_lists.exec) cudaGraphExecDestroy(ctx->graph_lists.exec);
    for (auto &s : ctx->scratch)
        if (s.p) cudaFree(s.p);
    for (auto ev : ctx->events) cudaEventDestroy(ev);
    if (ctx->pinned) cudaFreeHost(ctx->pinned);
    if (ctx->capture_stream) cudaStreamDestroy(ctx->capture_stream);
    delete ctx;
}

extern "C" const char *bpe_last_error(const bpe_ctx *ctx) { return ctx ? ctx->err.c_str() : "null context"; }

extern "C" int bpe_ctx_set_option(bpe_ctx *ctx, int option, int64_t value) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    switch (option) {
    case BPE_OPT_TABLE_LOG2:
        if (value != 0 && (value < 12 || value > 28))
            return fail(ctx, BPE_ERR_INVALID_ARG, "table log2 %lld outside 12..28", (long long)value);
        ctx->table_log2 = (int)value;
        return BPE_OK;
    case BPE_OPT_GRAPH:
        ctx->use_graph = value ? 1 : 0;
        return BPE_OK;
    case BPE_OPT_PROFILE:
        ctx->profile = value ? 1 : 0;
        return BPE_OK;
    case BPE_OPT_TRAIN_WORDS:
        ctx->train_words = value ? 1 : 0;
        return BPE_OK;
    case BPE_OPT_MERGE:
        if (value != BPE_MERGE_TILES && value != BPE_MERGE_LOOKBACK && value != BPE_MERGE_TWO_PASS &&
            value != BPE_MERGE_LISTS)
            return fail(ctx, BPE_ERR_INVALID_ARG, "unknown merge variant %lld", (long long)value);
        ctx->merge_mode = (int)value;
        return BPE_OK;
    case BPE_OPT_TRIE_LAYOUT:
        if (value != BPE_TRIE_DOUBLE_ARRAY && value != BPE_TRIE_BITMAP)
            return fail(ctx, BPE_ERR_INVALID_ARG, "unknown trie layout %lld", (long long)value);
        ctx->trie_layout = (int)value;
        return BPE_OK;
    case BPE_OPT_PERSISTENT:
        ctx->persistent = value ? 1 : 0;
        return BPE_OK;
    case BPE_OPT_SPARSE_MERGE:
        if (value < 0 || value > 2)
            return fail(ctx, BPE_ERR_INVALID_ARG, "sparse merge mode %lld is not 0, 1 or 2", (long long)value);
        ctx->sparse_merge = (int)value;
        return BPE_OK;
    case BPE_OPT_LIST_FRONTIER:
        if (value < 0 || value > 8192)
            return fail(ctx, BPE_ERR_INVALID_ARG, "list frontier %lld outside 0..8192", (long long)value);
        ctx->list_frontier = (int)value;
        return BPE_OK;
    case BPE_OPT_LIST_TAIL:
        if (value < -1 || value > 4096)
            return fail(ctx, BPE_ERR_INVALID_ARG, "list tail %lld outside -1..4096", (long long)value);
        ctx->list_tail = (int)value;
        return BPE_OK;
    case BPE_OPT_TEST_STALL_TILE:
        ctx->test_stall_tile = value < 0 ? -1 : value;
        return BPE_OK;
    case BPE_OPT_UNI_CHUNK:
        if (value != 0 && (value < 256 || value > 4096 || value % 64))
            return fail(ctx, BPE_ERR_INVALID_ARG, "unigram chunk %lld not 0 or in 256..4096 in steps of 64",
                        (long long)value);
        ctx->uni_chunk = (int)value;
        return BPE_OK;
    case BPE_OPT_CHUNK:
        if (value < 64 || value > 256 || value % 32)
            return fail(ctx, BPE_ERR_INVALID_ARG, "chunk %lld not in 64..256 or not a multiple of 32",
                        (long long)value);
        ctx->chunk = (int)value;
        return BPE_OK;
    default:
        return fail(ctx, BPE_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

extern "C" int bpe_last_stats(const bpe_ctx *ctx, bpe_stats *out) {
    if (!ctx || !out) return BPE_ERR_INVALID_ARG;
    *out = ctx->stats;
    return BPE_OK;
}
