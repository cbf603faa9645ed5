// device.cuh -- small device helpers shared by the kernels of libbpetrie.so.
#pragma once

#include <cstdint>

namespace bpe {

constexpr uint32_t kWordStart = 0x10000u;
constexpr uint32_t kEmptyKey = 0xFFFFFFFFu;
constexpr unsigned kFull = 0xFFFFFFFFu;

// Error bits a kernel may raise in a device-side status word.
enum : uint32_t { DERR_TABLE_FULL = 1u, DERR_TIMEOUT = 2u, DERR_OOB = 4u };

// Murmur3's 32-bit finaliser (Appleby, MurmurHash3, public domain): the
// hash the pair tables of [GPU-BPE] "What it does", 2. are keyed with.
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

// Relaxed, GPU-scope 64-bit status words for decoupled look-back.
__device__ __forceinline__ void st_relaxed(unsigned long long *a, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long *a) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}

// Acquire / release 32-bit words at GPU scope (grid barrier).
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *a) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *a, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// Weak 64-bit load served by L2 (no L1, no ordering): independent loads of
// look-back status words overlap; each word is one aligned 64-bit value, so a
// reader sees it either before or after its single store.
__device__ __forceinline__ unsigned long long ld_l2(const unsigned long long *a) {
    unsigned long long v;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(v) : "l"(a));
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        unsigned long long o = __shfl_xor_sync(kFull, v, d);
        v = o > v ? o : v;
    }
    return v;
}

// Inclusive warp sum via __shfl_up_sync.
__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

// Token byte class of [GPU-BPE] "Line by line", 1) bpe_word_boundary:
// 0 Letter (a-z, A-Z, >= 0x80), 1 Digit, 2 Space, 3 Punct, 4 Newline.
// Unsigned range tests, later tests take precedence (the classes are
// disjoint, so precedence never matters).
__device__ __forceinline__ uint32_t byte_class(uint32_t b) {
    uint32_t c = 3u;
    c = (b - 0x41u <= 25u) ? 0u : c;
    c = (b - 0x61u <= 25u) ? 0u : c;
    c = (b >= 0x80u) ? 0u : c;
    c = (b - 0x30u <= 9u) ? 1u : c;
    c = (b == 0x20u) ? 2u : c;
    c = (b == 0x0Au) ? 4u : c;
    return c;
}

}  // namespace bpe
