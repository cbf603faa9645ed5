// decode.cu -- the vocabulary a merge table defines, and ids back to bytes.
//
// [GPU-BPE] "What is this?": every merge gives the pair (left, right) one new
// symbol, so the vocabulary is the 256 single bytes followed by one token per
// merge whose bytes are its left token's bytes then its right token's bytes.
// [GPU-BPE] "Host architecture", 1. compiles that list of byte strings into
// the trie; bpe_vocab_from_merges writes the list (host only) and bpe_decode
// expands ids or symbols back into bytes on the device.
//
// bpe_decode kernels (ids in blocks of kDecItems per thread):
//   k_dec_len    per block: the byte length of its ids, and a flag for an
//                id outside the vocabulary
//   k_dec_scan   one CTA: exclusive 64-bit offsets of the block lengths and
//                the total, read back by the host to check the capacity
//   k_dec_write  per thread: its ids' offsets (warp and CTA scan on top of the
//                block offset), then each id's bytes copied from the table
#include <cstring>
#include <vector>

#include "device.cuh"
#include "internal.h"

namespace bpe {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecItems = 8;
constexpr int kDecBlock = kDecThreads * kDecItems;
constexpr uint32_t kDecIdMask = 0xFFFFu;

struct DecState {
    unsigned long long total;
    uint32_t bad;
    uint32_t pad;
};

struct DecParams {
    const uint32_t *ids;
    uint64_t n;
    const uint8_t *tok;        // token bytes, back to back
    const uint64_t *off;       // n_tok + 1 offsets into tok
    uint32_t n_tok;
    unsigned long long *bsum;  // per block: its length, then its exclusive offset
    DecState *st;
    uint8_t *out;
    uint64_t cap;
};

// The token id of one input value: bits 0..15, with WORD_START (bit 16)
// ignored; any other bit, or an id past the vocabulary, is invalid.
__device__ __forceinline__ bool dec_id(const DecParams &P, uint32_t v, uint32_t *id) {
    const uint32_t x = v & ~kWordStart;
    *id = x;
    return x <= kDecIdMask && x < P.n_tok;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long *s_w) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    if (lane == 0) s_w[warp] = v;
    __syncthreads();
    unsigned long long t = 0;
    if (threadIdx.x == 0)
        for (int w = 0; w < kDecThreads / 32; w++) t += s_w[w];
    return t;   // meaningful in thread 0
}

__global__ void __launch_bounds__(kDecThreads) k_dec_len(DecParams P) {
    __shared__ unsigned long long s_w[kDecThreads / 32];
    const uint64_t b0 = (uint64_t)blockIdx.x * kDecBlock;
    unsigned long long len = 0;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kDecItems; j++) {
        const uint64_t i = b0 + (uint64_t)j * kDecThreads + threadIdx.x;   // coalesced
        if (i < P.n) {
            uint32_t id;
            if (dec_id(P, P.ids[i], &id)) len += P.off[id + 1] - P.off[id];
            else bad = true;
        }
    }
    if (bad) atomicOr(&P.st->bad, 1u);
    const unsigned long long t = block_sum_u64(len, s_w);
    if (threadIdx.x == 0) P.bsum[blockIdx.x] = t;
}

__global__ void __launch_bounds__(1024) k_dec_scan(DecParams P, uint32_t nb) {
    __shared__ unsigned long long s_w[32];
    __shared__ unsigned long long s_carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (uint32_t c0 = 0; c0 < nb; c0 += 1024) {
        const uint32_t i = c0 + threadIdx.x;
        const unsigned long long v = i < nb ? P.bsum[i] : 0ull;
        unsigned long long incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long o = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) s_w[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            unsigned long long w = s_w[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long o = __shfl_up_sync(kFull, w, d);
                if (lane >= d) w += o;
            }
            s_w[lane] = w;   // inclusive over warps
        }
        __syncthreads();
        const unsigned long long base = s_carry + (warp ? s_w[warp - 1] : 0ull);
        if (i < nb) P.bsum[i] = base + incl - v;
        __syncthreads();
        if (threadIdx.x == 1023) s_carry = base + incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) P.st->total = s_carry;
}

__global__ void __launch_bounds__(kDecThreads) k_dec_write(DecParams P) {
    __shared__ unsigned long long s_w[kDecThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // this thread's ids are kDecItems consecutive ones, so its bytes are contiguous
    const uint64_t i0 = (uint64_t)blockIdx.x * kDecBlock + (uint64_t)threadIdx.x * kDecItems;
    uint32_t id[kDecItems];
    unsigned long long len = 0;
#pragma unroll
    for (int j = 0; j < kDecItems; j++) {
        id[j] = 0xFFFFFFFFu;
        if (i0 + j < P.n) {
            uint32_t x;
            if (dec_id(P, P.ids[i0 + j], &x)) {
                id[j] = x;
                len += P.off[x + 1] - P.off[x];
            }
        }
    }
    unsigned long long incl = len;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    unsigned long long wbase = 0;
    for (int w = 0; w < warp; w++) wbase += s_w[w];
    unsigned long long o = P.bsum[blockIdx.x] + wbase + incl - len;
#pragma unroll
    for (int j = 0; j < kDecItems; j++) {
        if (id[j] == 0xFFFFFFFFu) continue;
        const uint64_t a = P.off[id[j]], b = P.off[id[j] + 1];
        for (uint64_t t = a; t < b; t++, o++)
            if (o < P.cap) P.out[o] = P.tok[t];
    }
}

// Token byte strings of a merge table: ids 0..255 are the single bytes, id
// 256 + k the bytes of merge k's left token followed by its right token's.
// Returns false (with *why set) for a malformed table.
bool vocab_table(const bpe_merge *m, uint32_t n_merges, std::vector<uint64_t> &off, std::vector<uint8_t> *bytes,
                 const char **why) {
    const uint32_t n_tok = 256 + n_merges;
    off.assign((size_t)n_tok + 1, 0);
    for (uint32_t b = 0; b < 256; b++) off[b + 1] = b + 1;
    for (uint32_t k = 0; k < n_merges; k++) {
        const uint32_t id = 256 + k;
        if (m[k].new_id != id) {
            *why = "merge k must have new_id 256 + k";
            return false;
        }
        if (m[k].left >= id || m[k].right >= id) {
            *why = "a merge names an id that no earlier merge made";
            return false;
        }
        const uint64_t ll = off[m[k].left + 1] - off[m[k].left], lr = off[m[k].right + 1] - off[m[k].right];
        off[id + 1] = off[id] + ll + lr;
    }
    if (bytes) {
        bytes->resize(off[n_tok]);
        uint8_t *o = bytes->data();
        for (uint32_t b = 0; b < 256; b++) o[b] = (uint8_t)b;
        for (uint32_t k = 0; k < n_merges; k++) {
            const uint32_t id = 256 + k, l = m[k].left, r = m[k].right;
            const uint64_t ll = off[l + 1] - off[l];
            memcpy(o + off[id], o + off[l], ll);
            memcpy(o + off[id] + ll, o + off[r], off[r + 1] - off[r]);
        }
    }
    return true;
}

}  // namespace
}  // namespace bpe

using namespace bpe;

extern "C" int bpe_vocab_from_merges(const bpe_merge *h_merges, uint32_t n_merges, uint8_t *h_bytes_out,
                                     uint64_t bytes_capacity, uint64_t *h_off_out, uint64_t *n_bytes) {
    if ((n_merges && !h_merges) || !n_bytes) return BPE_ERR_INVALID_ARG;
    if (n_merges > BPE_MAX_MERGES) return BPE_ERR_ID_OVERFLOW;
    std::vector<uint64_t> off;
    const char *why = nullptr;
    if (!vocab_table(h_merges, n_merges, off, nullptr, &why)) return BPE_ERR_INVALID_ARG;
    *n_bytes = off.back();
    if (off.back() > bytes_capacity) return BPE_ERR_CAPACITY;
    if ((off.back() && !h_bytes_out) || !h_off_out) return BPE_ERR_INVALID_ARG;
    std::vector<uint8_t> bytes;
    vocab_table(h_merges, n_merges, off, &bytes, &why);
    if (!bytes.empty()) memcpy(h_bytes_out, bytes.data(), bytes.size());
    memcpy(h_off_out, off.data(), off.size() * sizeof(uint64_t));
    return BPE_OK;
}

extern "C" int bpe_decode(bpe_ctx *ctx, const bpe_merge *h_merges, uint32_t n_merges, const uint32_t *d_ids,
                          uint64_t n_ids, uint8_t *d_bytes_out, uint64_t bytes_capacity, uint64_t *n_bytes) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (!n_bytes || (n_merges && !h_merges) || (n_ids && !d_ids))
        return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_decode: null pointer");
    if (n_merges > BPE_MAX_MERGES) return fail(ctx, BPE_ERR_ID_OVERFLOW, "bpe_decode: %u merges", n_merges);
    std::vector<uint64_t> off;
    std::vector<uint8_t> tok;
    const char *why = nullptr;
    if (!vocab_table(h_merges, n_merges, off, &tok, &why)) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_decode: %s", why);
    *n_bytes = 0;
    if (n_ids == 0) return BPE_OK;
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    const uint64_t nb64 = (n_ids + kDecBlock - 1) / kDecBlock;
    if (nb64 > 0x7FFFFFFFull) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_decode: %llu ids", (unsigned long long)n_ids);
    const uint32_t nb = (uint32_t)nb64;
    void *p_tok, *p_off, *p_bsum, *p_st, *pin;
    int rc;
    if ((rc = ensure(ctx, S_DEC_TOK, tok.size(), &p_tok)) || (rc = ensure(ctx, S_DEC_OFF, off.size() * 8, &p_off)) ||
        (rc = ensure(ctx, S_DEC_BSUM, (size_t)nb * 8, &p_bsum)) || (rc = ensure(ctx, S_DEC_STATE, sizeof(DecState), &p_st)) ||
        (rc = ensure_pinned(ctx, sizeof(DecState), &pin)))
        return rc;
    cudaStream_t s = ctx->stream;
    // pageable sources: the copies complete before cudaMemcpyAsync returns
    BPE_CUDA(ctx, cudaMemcpyAsync(p_tok, tok.data(), tok.size(), cudaMemcpyHostToDevice, s), "vocab upload");
    BPE_CUDA(ctx, cudaMemcpyAsync(p_off, off.data(), off.size() * 8, cudaMemcpyHostToDevice, s), "offset upload");
    BPE_CUDA(ctx, cudaMemsetAsync(p_st, 0, sizeof(DecState), s), "state clear");
    DecParams P{d_ids, n_ids, (const uint8_t *)p_tok, (const uint64_t *)p_off, 256 + n_merges,
                (unsigned long long *)p_bsum, (DecState *)p_st, d_bytes_out, bytes_capacity};
    k_dec_len<<<nb, kDecThreads, 0, s>>>(P);
    k_dec_scan<<<1, 1024, 0, s>>>(P, nb);
    BPE_CUDA(ctx, cudaGetLastError(), "decode launch");
    BPE_CUDA(ctx, cudaMemcpyAsync(pin, p_st, sizeof(DecState), cudaMemcpyDeviceToHost, s), "state readback");
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "decode sync");
    DecState h;
    memcpy(&h, pin, sizeof h);
    if (h.bad) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_decode: an id outside the %u-token vocabulary", 256 + n_merges);
    *n_bytes = h.total;
    if (h.total > bytes_capacity)
        return fail(ctx, BPE_ERR_CAPACITY, "bpe_decode: %llu bytes needed, capacity %llu", h.total,
                    (unsigned long long)bytes_capacity);
    if (!d_bytes_out) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_decode: null output");
    k_dec_write<<<nb, kDecThreads, 0, s>>>(P);
    BPE_CUDA(ctx, cudaGetLastError(), "decode launch");
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "decode sync");
    return BPE_OK;
}
