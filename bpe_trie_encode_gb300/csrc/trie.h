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
    int2 *d_slot = nullptr;    // {check, base | TERM}, n_slots entries
    int32_t *d_tid = nullptr;  // token id per slot (-1: none)
    int4 *d_root = nullptr;    // 256 x {slot, base|TERM, tid, 0} of the depth-1 nodes
};

namespace bpe {
constexpr uint32_t kTermBit = 0x80000000u;
}
