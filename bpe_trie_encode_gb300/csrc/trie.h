// trie.h -- the device-resident double-array trie shared by trie_build.cpp
// (construction, upload) and encode.cu (greedy longest-match).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

struct bpe_trie {
    int device = 0;
    uint32_t n_tok = 0;
    uint64_t n_nodes = 0;
    uint64_t n_slots = 0;
    uint32_t max_len = 0;
    int missing_byte = -1;     // lowest single byte that is not a token (-1: none; greedy encoding needs none)
    int2 *d_slot = nullptr;    // {check, base | TERM}, n_slots entries
    int32_t *d_tid = nullptr;  // token id per slot (-1: none)
    int4 *d_root = nullptr;    // 256 x {slot, base|TERM, tid, 0} of the depth-1 nodes
    // bitmap-node layout, built on first use: per slot one 64-byte node
    // {256-bit child bitmap, base|TERM} (the slot numbering of the double array)
    void *d_bm = nullptr;
};

namespace bpe {
struct alignas(64) BmNode {
    unsigned long long bits[4];   // bit c: this node has a child on byte c (at base + c)
    uint32_t by;                  // base | TERM, as in the double array
    uint32_t pad[7];
};
static_assert(sizeof(BmNode) == 64, "one cache line per node");
}

namespace bpe {
constexpr uint32_t kTermBit = 0x80000000u;
}
