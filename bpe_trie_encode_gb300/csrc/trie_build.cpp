// trie_build.cpp -- flattened double-array trie of a vocabulary.
//
// [UNIGRAM] (the double-array passage, after Aoe 1989): the trie lives in two
// flat integer arrays; the child of node s on byte c is slot base[s] + c and
// the link is real when check[base[s] + c] == s.  Construction places the
// children of every node in free slots of the shared array, so parents share
// space as long as their children differ.  The token id is stored with the
// node ([UNIGRAM], token id in the trie node), so no reverse lookup exists.
// [GPU-BPE] "Host architecture", 1.: nodes are placed in breadth-first order,
// children sorted by byte, which keeps each level's slots close together.
//
// Device layout (uploaded once, read only by trie_encode):
//   slot[i] = int2 { check, base | TERM }   check = parent slot (-1 free,
//             -2 root); TERM (bit 31) marks a token; base 0 = no children
//   tid[i]  = token id of slot i (-1 if none)
//   root[c] = int4 { slot, base|TERM, tid, 0 } of the depth-1 node of byte c
//             (the root LUT kept in shared memory by the encoder,
//             [GPU-BPE] "Line by line", 3) root LUT and depth-1 cache)
#include <algorithm>
#include <cstring>
#include <numeric>
#include <vector>

#include "internal.h"
#include "trie.h"

namespace bpe {
namespace {

struct Node {
    uint32_t first_child = 0;   // 0 = none (the root is node 0 and is nobody's child)
    uint32_t next_sibling = 0;
    uint32_t last_child = 0;
    int32_t tid = -1;
    uint8_t label = 0;
};

// Free-slot search over a growing array: a doubly linked list of free slots.
struct SlotArray {
    std::vector<int32_t> check, base, tid;
    std::vector<int64_t> nxt, prv;   // free list links (-1 = end)
    int64_t head = -1;               // first free slot
    int64_t tail = -1;               // last free slot
    int64_t size = 0;

    void grow(int64_t to) {
        int64_t old = size;
        if (to <= old) return;
        check.resize(to, -1);
        base.resize(to, 0);
        tid.resize(to, -1);
        nxt.resize(to, -1);
        prv.resize(to, -1);
        // append [old, to) to the free list
        for (int64_t i = old; i < to; i++) {
            prv[i] = tail;
            nxt[i] = -1;
            if (tail >= 0) nxt[tail] = i; else head = i;
            tail = i;
        }
        size = to;
    }
    void take(int64_t i) {
        if (prv[i] >= 0) nxt[prv[i]] = nxt[i]; else head = nxt[i];
        if (nxt[i] >= 0) prv[nxt[i]] = prv[i]; else tail = prv[i];
        nxt[i] = prv[i] = -2;
    }
    bool free_slot(int64_t i) const { return i < size && check[i] == -1; }
};

struct Layout {
    std::vector<int2> slots;
    std::vector<int32_t> tids;
    std::vector<int4> root;
    uint64_t n_nodes = 0;
    uint32_t max_len = 0;
    int missing_byte = -1;   // lowest byte that is not a token, -1 if none
};

// Host-side construction; ctx (nullable) only receives error messages.
int build_layout(bpe_ctx *ctx, const uint8_t *h_vocab_bytes, const uint64_t *h_vocab_off, uint32_t n_tok,
                 Layout &L) {
    if (!h_vocab_off || (n_tok && !h_vocab_bytes)) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_build: null pointer");
    for (uint32_t t = 0; t < n_tok; t++)
        if (h_vocab_off[t + 1] < h_vocab_off[t])
            return fail(ctx, BPE_ERR_INVALID_ARG, "trie_build: offsets descend at token %u", t);

    // 1. sort token strings (ties by id so the lowest id of equal strings wins)
    std::vector<uint32_t> order;
    order.reserve(n_tok);
    uint32_t max_len = 0;
    for (uint32_t t = 0; t < n_tok; t++) {
        uint64_t len = h_vocab_off[t + 1] - h_vocab_off[t];
        if (len == 0) continue;
        if (len > 0x7FFFFFFFull) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_build: token %u too long", t);
        max_len = std::max<uint32_t>(max_len, (uint32_t)len);
        order.push_back(t);
    }
    auto less = [&](uint32_t a, uint32_t b) {
        const uint8_t *pa = h_vocab_bytes + h_vocab_off[a], *pb = h_vocab_bytes + h_vocab_off[b];
        uint64_t la = h_vocab_off[a + 1] - h_vocab_off[a], lb = h_vocab_off[b + 1] - h_vocab_off[b];
        int c = memcmp(pa, pb, std::min(la, lb));
        if (c) return c < 0;
        if (la != lb) return la < lb;
        return a < b;
    };
    std::sort(order.begin(), order.end(), less);

    // 2. pointer trie, built along the sorted order (children appear in byte order)
    std::vector<Node> nodes(1);
    std::vector<uint32_t> path(1, 0);   // node at each depth of the previous string
    const uint8_t *prev = nullptr;
    uint64_t prev_len = 0;
    for (uint32_t t : order) {
        const uint8_t *s = h_vocab_bytes + h_vocab_off[t];
        uint64_t len = h_vocab_off[t + 1] - h_vocab_off[t];
        uint64_t lcp = 0;
        if (prev)
            while (lcp < len && lcp < prev_len && s[lcp] == prev[lcp]) lcp++;
        path.resize(lcp + 1);
        for (uint64_t i = lcp; i < len; i++) {
            uint32_t parent = path.back();
            uint32_t id = (uint32_t)nodes.size();
            nodes.emplace_back();
            nodes[id].label = s[i];
            if (nodes[parent].first_child == 0) nodes[parent].first_child = id;
            else nodes[nodes[parent].last_child].next_sibling = id;
            nodes[parent].last_child = id;
            path.push_back(id);
        }
        Node &end = nodes[path.back()];
        if (end.tid < 0) end.tid = (int32_t)t;   // lowest id (sorted by id on ties)
        prev = s;
        prev_len = len;
    }

    // whether every single byte is a token (greedy matching then never fails)
    {
        std::vector<int> seen(256, 0);
        for (uint32_t c = nodes[0].first_child; c; c = nodes[c].next_sibling)
            if (nodes[c].tid >= 0) seen[nodes[c].label] = 1;
        for (int b = 255; b >= 0; b--)
            if (!seen[b]) L.missing_byte = b;
    }

    // 3. double-array placement in breadth-first order
    SlotArray A;
    A.grow(std::max<int64_t>(1024, (int64_t)nodes.size() * 2));
    std::vector<int64_t> slot_of(nodes.size(), -1);
    slot_of[0] = 0;
    A.take(0);
    A.check[0] = -2;
    int64_t frontier = 1;
    std::vector<uint32_t> queue;
    queue.reserve(nodes.size());
    queue.push_back(0);
    std::vector<uint8_t> labels;
    std::vector<uint32_t> kids;
    for (size_t qi = 0; qi < queue.size(); qi++) {
        uint32_t u = queue[qi];
        int64_t su = slot_of[u];
        A.tid[su] = nodes[u].tid;
        labels.clear();
        kids.clear();
        for (uint32_t c = nodes[u].first_child; c; c = nodes[c].next_sibling) {
            labels.push_back(nodes[c].label);
            kids.push_back(c);
        }
        if (kids.empty()) {
            A.base[su] = 0;
            continue;
        }
        // first fit over the free list; a long scan falls back to the frontier
        // (the first slot after every used one), where all slots are free
        int64_t b = -1;
        int scanned = 0;
        for (int64_t q = A.head; q >= 0 && q < frontier; q = A.nxt[q]) {
            if (++scanned > 256) break;
            int64_t cand = q - labels[0];
            if (cand < 1) continue;
            bool ok = true;
            for (size_t i = 1; i < labels.size() && ok; i++) {
                int64_t x = cand + labels[i];
                if (x >= A.size) break;          // beyond the end: free after growth
                ok = A.check[x] == -1;
            }
            if (ok) {
                b = cand;
                break;
            }
        }
        if (b < 0) b = std::max<int64_t>(1, frontier - labels[0]);
        if (b + 256 > 0x7FFFFFFF) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_build: trie too large");
        if (b + 257 > A.size) A.grow(std::max<int64_t>(b + 257, A.size + A.size / 2));
        A.base[su] = (int32_t)b;
        for (size_t i = 0; i < kids.size(); i++) {
            int64_t x = b + labels[i];
            A.take(x);
            A.check[x] = (int32_t)su;
            frontier = std::max<int64_t>(frontier, x + 1);
            slot_of[kids[i]] = x;
            queue.push_back(kids[i]);
        }
    }
    // trim: every base + 255 must stay inside the array
    int64_t used = 0;
    for (int64_t i = 0; i < A.size; i++) {
        if (A.check[i] != -1) used = i + 1;
        if (A.check[i] != -1 && A.base[i] > 0) used = std::max<int64_t>(used, (int64_t)A.base[i] + 256);
    }
    used = std::max<int64_t>(used, 257);

    L.slots.resize(used);
    L.tids.resize(used);
    for (int64_t i = 0; i < used; i++) {
        uint32_t y = (uint32_t)A.base[i] | (A.tid[i] >= 0 ? kTermBit : 0u);
        L.slots[i] = make_int2(A.check[i], (int32_t)y);
        L.tids[i] = A.tid[i];
    }
    L.root.resize(256);
    const int32_t rb = A.base[0];
    for (int c = 0; c < 256; c++) {
        int64_t x = rb + c;
        L.root[c] = make_int4((int32_t)x, L.slots[x].y, L.tids[x], 0);
    }
    L.n_nodes = nodes.size();
    L.max_len = max_len;
    return BPE_OK;
}

}  // namespace
}  // namespace bpe

using namespace bpe;

extern "C" int trie_build(bpe_ctx *ctx, const uint8_t *h_vocab_bytes, const uint64_t *h_vocab_off, uint32_t n_tok,
                          bpe_trie **out) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (!out) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_build: out is null");
    *out = nullptr;
    Layout L;
    int rc = build_layout(ctx, h_vocab_bytes, h_vocab_off, n_tok, L);
    if (rc) return rc;
    const size_t used = L.slots.size();
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    bpe_trie *T = new bpe_trie();
    T->device = ctx->device;
    T->n_tok = n_tok;
    T->n_nodes = L.n_nodes;
    T->n_slots = (uint64_t)used;
    T->max_len = L.max_len;
    T->missing_byte = L.missing_byte;
    cudaError_t e = cudaMalloc(&T->d_slot, sizeof(int2) * used);
    if (e == cudaSuccess) e = cudaMalloc(&T->d_tid, sizeof(int32_t) * used);
    if (e == cudaSuccess) e = cudaMalloc(&T->d_root, sizeof(int4) * 256);
    if (e == cudaSuccess) e = cudaMemcpy(T->d_slot, L.slots.data(), sizeof(int2) * used, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(T->d_tid, L.tids.data(), sizeof(int32_t) * used, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(T->d_root, L.root.data(), sizeof(int4) * 256, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        trie_free(T);
        return cuda_fail(ctx, e, "trie_build upload");
    }
    *out = T;
    return BPE_OK;
}

extern "C" int trie_layout(const uint8_t *h_vocab_bytes, const uint64_t *h_vocab_off, uint32_t n_tok,
                           int32_t *check_out, int32_t *base_out, int32_t *tid_out, uint64_t capacity,
                           uint64_t *n_slots) {
    if (!n_slots) return BPE_ERR_INVALID_ARG;
    Layout L;
    int rc = build_layout(nullptr, h_vocab_bytes, h_vocab_off, n_tok, L);
    if (rc) return rc;
    *n_slots = L.slots.size();
    if (L.slots.size() > capacity) return BPE_ERR_CAPACITY;
    for (size_t i = 0; i < L.slots.size(); i++) {
        if (check_out) check_out[i] = L.slots[i].x;
        if (base_out) base_out[i] = L.slots[i].y;
        if (tid_out) tid_out[i] = L.tids[i];
    }
    return BPE_OK;
}

extern "C" int trie_info(const bpe_trie *T, uint64_t *n_nodes, uint64_t *n_slots, uint32_t *max_token_len) {
    if (!T) return BPE_ERR_INVALID_ARG;
    if (n_nodes) *n_nodes = T->n_nodes;
    if (n_slots) *n_slots = T->n_slots;
    if (max_token_len) *max_token_len = T->max_len;
    return BPE_OK;
}

extern "C" void trie_free(bpe_trie *T) {
    if (!T) return;
    cudaSetDevice(T->device);
    if (T->d_slot) cudaFree(T->d_slot);
    if (T->d_tid) cudaFree(T->d_tid);
    if (T->d_root) cudaFree(T->d_root);
    if (T->d_bm) cudaFree(T->d_bm);
    delete T;
}
