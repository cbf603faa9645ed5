// pipeline.cpp -- trie_encode_host: greedy encoding from host buffers with the
// transfers overlapped, following "Async batching: when CPU and GPU work
// together" (three streams -- host to device, compute, device to host --
// ordered by CUDA events; two buffer slots so batch N+1 never overwrites
// batch N).  Whole documents are grouped into units of about slice_bytes and
// encoded with trie_encode; a document longer than that is streamed in
// slices through a bpe_stream ([GPU-BPE] "Host architecture", 3. multi-pass
// slicing, with the parse carried across slices).
#include <algorithm>
#include <cstring>
#include <vector>

#include "internal.h"
#include "trie.h"

namespace bpe {
namespace {

struct Unit {
    uint64_t b0, b1;    // bytes [b0, b1) of the input
    uint32_t d0, nd;    // documents d0 .. d0 + nd - 1 (a slice: the one document d0)
    bool slice, first, last;
    uint64_t stage;     // a group: where its id offsets land in the pinned staging area
};

// Waits for the pipeline's copy streams on every exit, so no copy still reads
// or writes the caller's host buffers after the call returns.
struct PipeSync {
    bpe_ctx *ctx;
    ~PipeSync() {
        if (ctx->pipe_h2d) cudaStreamSynchronize(ctx->pipe_h2d);
        if (ctx->pipe_d2h) cudaStreamSynchronize(ctx->pipe_d2h);
    }
};

// The context's pipeline resources, created on first use; pinned staging of
// at least `pinned` bytes (grown x1.5).
int pipe_resources(bpe_ctx *ctx, size_t pinned) {
    if (!ctx->pipe_h2d) BPE_CUDA(ctx, cudaStreamCreateWithFlags(&ctx->pipe_h2d, cudaStreamNonBlocking), "h2d stream");
    if (!ctx->pipe_d2h) BPE_CUDA(ctx, cudaStreamCreateWithFlags(&ctx->pipe_d2h, cudaStreamNonBlocking), "d2h stream");
    for (auto &ev : ctx->pipe_ev)
        if (!ev) BPE_CUDA(ctx, cudaEventCreateWithFlags(&ev, cudaEventDisableTiming), "event");
    if (ctx->pipe_pinned_cap < pinned) {
        if (ctx->pipe_pinned) {
            BPE_CUDA(ctx, cudaStreamSynchronize(ctx->pipe_d2h), "d2h sync");
            cudaFreeHost(ctx->pipe_pinned);
            ctx->pipe_pinned = nullptr;
            ctx->pipe_pinned_cap = 0;
        }
        const size_t cap = std::max(pinned, ctx->pipe_pinned_cap + ctx->pipe_pinned_cap / 2);
        BPE_CUDA(ctx, cudaMallocHost(&ctx->pipe_pinned, cap), "pinned staging");
        ctx->pipe_pinned_cap = cap;
    }
    return BPE_OK;
}

constexpr uint64_t kDefaultSlice = 128ull << 20;

}  // namespace
}  // namespace bpe

using namespace bpe;

extern "C" int trie_encode_host(bpe_ctx *ctx, const bpe_trie *trie, const uint8_t *h_bytes, const uint64_t *h_doc_off,
                                uint32_t n_docs, int32_t *h_ids_out, uint64_t ids_capacity, uint64_t *h_id_off_out,
                                uint64_t *n_ids, uint64_t slice_bytes) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (!trie || !n_ids) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode_host: null trie or n_ids");
    *n_ids = 0;
    if (n_docs && !h_doc_off) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode_host: null document offsets");
    if (ids_capacity && !h_ids_out) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode_host: null ids with capacity");
    for (uint32_t d = 0; d < n_docs; d++)
        if (h_doc_off[d + 1] < h_doc_off[d])
            return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode_host: document offsets descend at document %u", d);
    if (n_docs && h_doc_off[n_docs] > h_doc_off[0] && !h_bytes)
        return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode_host: null bytes");
    if (slice_bytes == 0) slice_bytes = kDefaultSlice;
    slice_bytes = std::max<uint64_t>(slice_bytes, 4096);
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");

    // units: groups of whole documents up to slice_bytes, slices of longer ones
    std::vector<Unit> units;
    uint32_t max_nd = 1;
    uint64_t max_bytes = 16, stage = 0;
    for (uint32_t d = 0; d < n_docs;) {
        const uint64_t len = h_doc_off[d + 1] - h_doc_off[d];
        if (len > slice_bytes) {
            for (uint64_t b = h_doc_off[d]; b < h_doc_off[d + 1]; b += slice_bytes) {
                const uint64_t e = std::min(h_doc_off[d + 1], b + slice_bytes);
                units.push_back({b, e, d, 1, true, b == h_doc_off[d], e == h_doc_off[d + 1], 0});
                max_bytes = std::max(max_bytes, e - b);
            }
            d++;
            continue;
        }
        uint32_t e = d + 1;
        while (e < n_docs && h_doc_off[e + 1] - h_doc_off[d] <= slice_bytes) e++;
        units.push_back({h_doc_off[d], h_doc_off[e], d, e - d, false, true, true, stage});
        stage += (uint64_t)(e - d) + 1;
        max_nd = std::max(max_nd, e - d);
        max_bytes = std::max(max_bytes, h_doc_off[e] - h_doc_off[d]);
        d = e;
    }

    PipeSync guard{ctx};
    const uint64_t id_slots = max_bytes + trie->max_len + 16;   // one id per byte, plus a carried tail
    const uint64_t head = ((uint64_t)trie->max_len + 15) & ~15ull;   // room for a slice's carried bytes
    void *din[2], *dout[2], *doff[2];
    int rc;
    if ((rc = ensure(ctx, S_HOST_IN0, head + max_bytes + 16, &din[0])) ||
        (rc = ensure(ctx, S_HOST_IN1, head + max_bytes + 16, &din[1])) ||
        (rc = ensure(ctx, S_HOST_OUT0, id_slots * 4, &dout[0])) || (rc = ensure(ctx, S_HOST_OUT1, id_slots * 4, &dout[1])) ||
        (rc = ensure(ctx, S_HOST_OFF0, ((uint64_t)max_nd + 1) * 16, &doff[0])) ||
        (rc = ensure(ctx, S_HOST_OFF1, ((uint64_t)max_nd + 1) * 16, &doff[1])))
        return rc;
    const size_t n_off = 2 * ((size_t)max_nd + 1), n_ioff = std::max<size_t>(stage, 1);
    if ((rc = pipe_resources(ctx, (n_off + n_ioff) * 8))) return rc;
    struct {
        cudaStream_t h2d, d2h;
        cudaEvent_t *in_ready, *computed, *out_free;
        uint64_t *h_off, *h_ioff;
    } pp{ctx->pipe_h2d, ctx->pipe_d2h, ctx->pipe_ev, ctx->pipe_ev + 2, ctx->pipe_ev + 4,
         (uint64_t *)ctx->pipe_pinned, (uint64_t *)ctx->pipe_pinned + n_off};
    for (int i = 0; i < 2; i++) BPE_CUDA(ctx, cudaEventRecord(pp.out_free[i], pp.d2h), "event");

    cudaStream_t cs = ctx->stream;
    const size_t noff = (size_t)max_nd + 1;
    // unit j's bytes (and, for a group, its rebased document offsets) into slot j & 1
    auto h2d = [&](size_t j) -> int {
        const Unit &u = units[j];
        const int sl = (int)(j & 1);
        if (u.b1 > u.b0)   // a slice lands after the room for the bytes carried into it
            BPE_CUDA(ctx, cudaMemcpyAsync((uint8_t *)din[sl] + (u.slice ? head : 0), h_bytes + u.b0, u.b1 - u.b0,
                                          cudaMemcpyHostToDevice, pp.h2d), "h2d");
        if (!u.slice) {
            uint64_t *ho = pp.h_off + sl * noff;
            for (uint32_t k = 0; k <= u.nd; k++) ho[k] = h_doc_off[u.d0 + k] - u.b0;
            BPE_CUDA(ctx, cudaMemcpyAsync(doff[sl], ho, (u.nd + 1) * 8, cudaMemcpyHostToDevice, pp.h2d), "h2d offsets");
        }
        BPE_CUDA(ctx, cudaEventRecord(pp.in_ready[sl], pp.h2d), "event");
        return BPE_OK;
    };
    std::vector<uint64_t> base(units.size() + 1, 0);   // ids before each unit
    uint64_t written = 0, launches = 0;
    if (!units.empty() && (rc = h2d(0))) return rc;
    for (size_t i = 0; i < units.size(); i++) {
        const Unit &u = units[i];
        const int sl = (int)(i & 1);
        // the next unit's copy overlaps this unit's encode (its slot was last
        // used by unit i-1, whose encode has returned)
        if (i + 1 < units.size() && (rc = h2d(i + 1))) return rc;
        BPE_CUDA(ctx, cudaStreamWaitEvent(cs, pp.in_ready[sl], 0), "wait input");
        BPE_CUDA(ctx, cudaStreamWaitEvent(cs, pp.out_free[sl], 0), "wait output slot");
        uint64_t n = 0;
        if (u.slice) {
            if (u.first) {   // the context's streaming state, reopened for another trie
                if (ctx->pipe_stream && (ctx->pipe_trie != trie || ctx->pipe_max_len != trie->max_len)) {
                    trie_stream_close(ctx->pipe_stream);
                    ctx->pipe_stream = nullptr;
                }
                if (!ctx->pipe_stream) {
                    if ((rc = trie_stream_open(ctx, trie, &ctx->pipe_stream))) return rc;
                    ctx->pipe_trie = trie;
                    ctx->pipe_max_len = trie->max_len;
                }
                stream_reset(ctx->pipe_stream);
            }
            rc = stream_push_in_place(ctx->pipe_stream, (uint8_t *)din[sl] + head, u.b1 - u.b0, u.last ? 1 : 0,
                                      (int32_t *)dout[sl], id_slots, &n);
        } else {
            rc = trie_encode(ctx, trie, (const uint8_t *)din[sl], (const uint64_t *)doff[sl], u.nd,
                             (int32_t *)dout[sl], id_slots, (uint64_t *)doff[sl] + noff, &n);
        }
        if (rc) return rc;
        launches += ctx->stats.kernel_launches;
        base[i] = written;
        BPE_CUDA(ctx, cudaEventRecord(pp.computed[sl], cs), "event");
        BPE_CUDA(ctx, cudaStreamWaitEvent(pp.d2h, pp.computed[sl], 0), "wait compute");
        if (written < ids_capacity && n) {
            const uint64_t m = std::min<uint64_t>(n, ids_capacity - written);
            BPE_CUDA(ctx, cudaMemcpyAsync(h_ids_out + written, dout[sl], m * 4, cudaMemcpyDeviceToHost, pp.d2h), "d2h");
        }
        if (!u.slice)
            BPE_CUDA(ctx, cudaMemcpyAsync(pp.h_ioff + u.stage, (uint64_t *)doff[sl] + noff, (u.nd + 1) * 8,
                                          cudaMemcpyDeviceToHost, pp.d2h), "d2h id offsets");
        BPE_CUDA(ctx, cudaEventRecord(pp.out_free[sl], pp.d2h), "event");
        written += n;
    }
    base[units.size()] = written;
    BPE_CUDA(ctx, cudaStreamSynchronize(pp.d2h), "d2h sync");
    BPE_CUDA(ctx, cudaStreamSynchronize(cs), "sync");
    if (h_id_off_out) {
        for (uint32_t d = 0; d <= n_docs; d++) h_id_off_out[d] = written;   // documents past the last unit: empty
        for (size_t i = units.size(); i-- > 0;) {
            const Unit &u = units[i];
            if (u.slice) {
                if (u.first) h_id_off_out[u.d0] = base[i];
            } else {
                for (uint32_t k = 0; k < u.nd; k++) h_id_off_out[u.d0 + k] = base[i] + pp.h_ioff[u.stage + k];
            }
        }
    }
    *n_ids = written;
    stats_reset(ctx);
    ctx->stats.kernel_launches = launches;
    if (written > ids_capacity)
        return fail(ctx, BPE_ERR_CAPACITY, "trie_encode_host: %llu ids exceed the capacity %llu",
                    (unsigned long long)written, (unsigned long long)ids_capacity);
    return BPE_OK;
}
