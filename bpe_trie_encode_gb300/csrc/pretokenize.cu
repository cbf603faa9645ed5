// pretokenize.cu -- bytes -> uint32 symbols with WORD_START at class
// transitions ([GPU-BPE] "What it does", 1. GPU pre-tokenization; "Line by
// line", 1) bpe_word_boundary).
//
// One elementwise pass: each thread turns 16 bytes (one 128-bit load plus
// the byte before them) into 16 symbols (four 128-bit stores).  HBM bound:
// n bytes read, 4n bytes written.
#include "device.cuh"
#include "internal.h"

namespace bpe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t sym_of(uint32_t b, uint32_t prev_b, bool first) {
    return b | ((first || byte_class(b) != byte_class(prev_b)) ? kWordStart : 0u);
}

// Aligned path: bytes and symbols 16-byte aligned.
__global__ void __launch_bounds__(kThreads) k_pretok_vec(const uint8_t *__restrict__ bytes, uint64_t n,
                                                         uint32_t *__restrict__ sym) {
    const uint64_t groups = n >> 4;
    for (uint64_t g = blockIdx.x * (uint64_t)kThreads + threadIdx.x; g < groups;
         g += (uint64_t)gridDim.x * kThreads) {
        const uint64_t i0 = g << 4;
        uint4 v = __ldcs(reinterpret_cast<const uint4 *>(bytes + i0));
        uint32_t prev = (i0 > 0) ? bytes[i0 - 1] : 0u;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
            uint32_t b = (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
            out[j] = sym_of(b, prev, i0 + j == 0);
            prev = b;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(sym + i0);
#pragma unroll
        for (int q = 0; q < 4; q++) __stcs(dst + q, make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]));
    }
    // tail (n % 16 bytes) by the first threads of block 0
    if (blockIdx.x == 0 && threadIdx.x < (n & 15)) {
        uint64_t i = (groups << 4) + threadIdx.x;
        sym[i] = sym_of(bytes[i], i ? bytes[i - 1] : 0u, i == 0);
    }
}

// Any alignment: one symbol per thread.
__global__ void __launch_bounds__(kThreads) k_pretok_scalar(const uint8_t *__restrict__ bytes, uint64_t n,
                                                            uint32_t *__restrict__ sym) {
    for (uint64_t i = blockIdx.x * (uint64_t)kThreads + threadIdx.x; i < n; i += (uint64_t)gridDim.x * kThreads)
        sym[i] = sym_of(bytes[i], i ? bytes[i - 1] : 0u, i == 0);
}

}  // namespace
}  // namespace bpe

using namespace bpe;

extern "C" int bpe_pretokenize(bpe_ctx *ctx, const uint8_t *d_bytes, uint64_t n, uint32_t *d_symbols_out) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (n == 0) return BPE_OK;
    if (!d_bytes || !d_symbols_out) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_pretokenize: null pointer");
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    const bool aligned = ((uintptr_t)d_bytes % 16 == 0) && ((uintptr_t)d_symbols_out % 16 == 0);
    const uint64_t work = aligned ? (n >> 4) : n;
    uint64_t blocks = (work + kThreads - 1) / kThreads;
    const uint64_t cap = (uint64_t)ctx->sm_count * 16;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    if (aligned)
        k_pretok_vec<<<(unsigned)blocks, kThreads, 0, ctx->stream>>>(d_bytes, n, d_symbols_out);
    else
        k_pretok_scalar<<<(unsigned)blocks, kThreads, 0, ctx->stream>>>(d_bytes, n, d_symbols_out);
    BPE_CUDA(ctx, cudaGetLastError(), "bpe_pretokenize launch");
    ctx->pretok_launches++;
    return BPE_OK;
}
