// encode.cu -- greedy longest-match encoding over the double-array trie
// ([GPU-BPE] "What it does", 4. trie-based inference; the inference pipeline
// trie_tokenizer_chunked -> trie_prefix_sum -> trie_tokenizer_compact).
//
// Every document is cut into chunks of C bytes; one thread parses one chunk.
// The exact result is the sequential greedy parse of each document, so a
// chunk must start where the previous chunk's last token ends, which is only
// known after that chunk is parsed.  The kernels resolve this without a
// sequential pass in the common case:
//
//   k_chunk_index   first chunk of every document (one CTA, exclusive scan)
//   k_spec          each thread parses its chunk speculatively from the chunk's
//                   first byte, remembering which positions start a token
//                   (bitmap in shared memory) and where the parse leaves the
//                   chunk (spec exit).  After a barrier each thread re-parses
//                   its chunk from the previous chunk's spec exit (the nominal
//                   entry) until that path meets a remembered token start --
//                   from there both paths are the same.  It records the
//                   chunk's token count and exit for the nominal entry, and
//                   flags the chunk when that exit differs from its own spec
//                   exit (the next chunk's nominal entry is then wrong).
//                   The first chunk of a CTA gets its nominal entry from a halo
//                   thread that parses the chunk before it.
//   k_repair_walk   only when some chunk was flagged (rare: the two parses of a
//                   chunk never meet inside it): one thread per flagged chunk
//                   re-parses the chunks after it, from that chunk's exit,
//                   until an exit agrees with the next nominal entry again,
//                   and keeps the chain privately.
//   k_repair_apply  one CTA sorts the flagged chunks and, in order, writes the
//                   chains of those whose own entry is true (a flagged chunk
//                   inside an applied chain is skipped); with more flags than
//                   the list holds it walks the chains sequentially instead.
//   k_emit          exclusive scan of the chunk counts (CTA scan + decoupled
//                   look-back over tiles taken in ticket order) and a final
//                   parse of every chunk from its true entry that writes ids at
//                   their global offsets.
//   k_doc_offsets   per-document id offsets.
//
// One trie step is: slot = base + byte, valid when check[slot] == node.  The
// root's 256 children are in a shared-memory LUT ([GPU-BPE] "Line by line",
// 3) root LUT), so the first byte of every token costs no global load.
#include <algorithm>
#include <mutex>

#include "device.cuh"
#include "internal.h"
#include "trie.h"

namespace bpe {
namespace {

constexpr int kSpecThreads = 256;          // 255 owned chunks + 1 halo chunk per CTA
constexpr int kEmitThreads = 256;
constexpr int kMaxChunk = 256;             // bytes per chunk (staging and bitmap bound)
constexpr unsigned kSpinLimit = 1u << 22;
constexpr uint32_t kBS = 256;   // stride between a thread's bitmap words (one column per thread: no bank conflicts)

struct EncState {
    unsigned long long n_chunks;
    unsigned long long total;
    uint32_t err;        // DERR_* bits
    uint32_t any_flag;   // some chunk's exit disagreed with the next nominal entry
    uint32_t flist_len;  // flagged chunks appended to the list
    uint32_t ticket;
    uint32_t bad_doc_off;
    unsigned long long span;     // doc_off[n_docs] - doc_off[0]
    unsigned long long text_lo;  // doc_off[0]
};

struct EncParams {
    const uint8_t *bytes;
    const uint64_t *doc_off;
    uint32_t n_docs;
    uint32_t chunk;              // C
    const unsigned long long *chunk_start;   // n_docs + 1
    const int2 *slot;
    const BmNode *bm;            // bitmap-node layout (null unless that layout is used)
    const int32_t *tid;
    const int4 *root;
    uint32_t *count;             // per chunk: tokens starting in the chunk (true path)
    uint32_t *exit_rel;          // per chunk: true exit - chunk start
    uint32_t *spec_rel;          // per chunk: spec exit - chunk start
    uint32_t *flag;              // bitmap of flagged chunks
    uint32_t *flist;             // flagged chunks, unordered (flist_cap entries; 0 = none kept)
    uint32_t flist_cap;
    uint32_t *wpriv;             // per flagged chunk: its repair walk (kWalkWords words)
    uint32_t *sbits;             // per chunk: C/32 words, token starts of the speculative parse
    int32_t *sids;               // per chunk: C words, the speculative parse's ids in order
                                 // (both null: the emit pass re-parses every chunk)
    unsigned long long *prefix;  // per chunk: global index of its first id
    unsigned long long *status;  // look-back words per emit tile
    int32_t *ids;
    unsigned long long cap;
    unsigned long long *id_off;
    EncState *st;
};

// -------------------------------------------------------------- matching ---

struct Match {
    uint32_t len;
    int32_t id;
};

// One trie step below the root: node -> its child on byte ch (at base + ch).
// L = 0, double array: the child slot's check must name node.  L = 1, bitmap
// nodes: node's bitmap has bit ch (both loads independent).  *ny: the
// child's base | TERM.
template <int L>
__device__ __forceinline__ bool trie_step(const EncParams &P, int32_t node, uint32_t base, uint32_t ch, int32_t *nt,
                                          uint32_t *ny) {
    const int32_t t = (int32_t)(base + ch);
    *nt = t;
    if (L == 0) {
        const int2 v = __ldg(P.slot + t);
        *ny = (uint32_t)v.y;
        return v.x == node;
    }
    const unsigned long long w = __ldg(&P.bm[node].bits[ch >> 6]);
    *ny = __ldg(&P.bm[t].by);
    return (w >> (ch & 63)) & 1ull;
}

// Longest token prefixing bytes[p, end) (p < end).
template <int L = 0>
__device__ __forceinline__ Match match_at(const EncParams &P, const int4 *lut, uint64_t p, uint64_t end) {
    const int4 r = lut[__ldg(P.bytes + p)];
    int32_t node = r.x;
    uint32_t y = (uint32_t)r.y;
    Match m{1u, r.z};
    int32_t best_node = -1;
    uint64_t q = p + 1;
    while (q < end) {
        const uint32_t base = y & ~kTermBit;
        if (base == 0) break;                       // no children
        int32_t t;
        uint32_t ny;
        if (!trie_step<L>(P, node, base, __ldg(P.bytes + q), &t, &ny)) break;
        node = t;
        y = ny;
        ++q;
        if (y & kTermBit) {
            m.len = (uint32_t)(q - p);
            best_node = node;
        }
    }
    if (best_node >= 0) m.id = __ldg(P.tid + best_node);
    return m;
}

// The longest token prefixing bytes[p, end) when that match is final: false
// when the trie walk ran into end with children still possible (more bytes
// could make the match longer).
template <int L = 0>
__device__ __forceinline__ bool match_final(const EncParams &P, const int4 *lut, uint64_t p, uint64_t end,
                                            uint32_t *len) {
    const int4 r = lut[__ldg(P.bytes + p)];
    int32_t node = r.x;
    uint32_t y = (uint32_t)r.y;
    *len = 1u;
    uint64_t q = p + 1;
    for (;;) {
        const uint32_t base = y & ~kTermBit;
        if (base == 0) return true;                 // no children: final
        if (q >= end) return false;                 // the next byte decides
        int32_t t;
        uint32_t ny;
        if (!trie_step<L>(P, node, base, __ldg(P.bytes + q), &t, &ny)) return true;   // mismatch: final
        node = t;
        y = ny;
        ++q;
        if (y & kTermBit) *len = (uint32_t)(q - p);
    }
}

__device__ __forceinline__ void load_lut(const EncParams &P, int4 *lut) {
    for (int c = threadIdx.x; c < 256; c += blockDim.x) lut[c] = P.root[c];
}

// document of a chunk: last d with chunk_start[d] <= k
__device__ __forceinline__ uint32_t doc_of_chunk(const EncParams &P, unsigned long long k) {
    uint32_t lo = 0, hi = P.n_docs;   // answer in [0, n_docs)
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (P.chunk_start[mid] <= k) lo = mid; else hi = mid;
    }
    return lo;
}

struct ChunkGeo {
    uint64_t cs, ce, de;   // chunk start, chunk end, document end
    bool doc_first;
};

__device__ __forceinline__ ChunkGeo chunk_geo(const EncParams &P, unsigned long long k) {
    const uint32_t d = doc_of_chunk(P, k);
    const uint64_t ds = P.doc_off[d], de = P.doc_off[d + 1];
    const uint64_t j = k - P.chunk_start[d];
    ChunkGeo g;
    g.cs = ds + j * P.chunk;
    g.ce = min(g.cs + P.chunk, de);
    g.de = de;
    g.doc_first = (j == 0);
    return g;
}

// ------------------------------------------------------------- parsing ---

// Sequential reads of a lane's bytes, four at a time: one aligned 32-bit load
// through L1 serves the next bytes (the word never leaves the allocation: it
// holds at least one byte of the text).  Offsets are 32-bit, from g.
struct ByteWin {
    const uint8_t *g;
    uint32_t at = 0xFFFFFFFFu;   // low word of the loaded word's address (never 4-aligned at start)
    uint32_t w = 0;
    __device__ __forceinline__ uint32_t operator()(uint32_t q) {
        const uintptr_t a = (uintptr_t)(g + q);
        const uint32_t al = (uint32_t)a & ~3u;
        if (al != at) {
            at = al;
            w = __ldg(reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3)));
        }
        return (w >> (8 * ((uint32_t)a & 3u))) & 0xFFu;
    }
};

// Greedy longest-match parse of the tokens that start in [p, ce) of a
// document ending at de.  Every loop iteration takes one trie step on every
// lane through the double array, so the lanes of a warp run the same
// instructions whatever their token lengths; a token ends when a step fails,
// and the next token's first step (through the shared LUT) is taken in the
// same iteration, from the byte that failed when the token ended there.  Positions are kept
// as 32-bit offsets from the chunk start cs (p >= cs; a parse never runs
// 2^31 bytes past it).
//   MODE 0 (speculative): mark token starts in bits (offsets from cs) and,
//          when sid is not null, store each token to sid[0 ...]: its id when
//          it is one byte long (from the root LUT), else 0x80000000 | its
//          trie slot, so the id lookup leaves the parse's critical path.
//          Tokens gather in the thread's column of shared memory (stage,
//          stride kBS) and go out eight at a time as one whole 32-byte
//          sector (sid is 32-byte aligned); the caller flushes the rest
//   MODE 1 (resync): stop early where a token start is already marked
//   MODE 2 (emit): write ids to ids[o ...] (below cap)
//   MODE 3 (emit head): MODE 2's writes, stopping like MODE 1
// Returns the position after the last token as an offset from cs; *cnt =
// tokens parsed (MODE 1 and 3: tokens up to the meeting point, *met = whether
// it met the marked path).
template <int MODE, int L = 0>
__device__ __forceinline__ uint32_t parse_tokens(const EncParams &P, const int4 *lut, uint64_t p_abs, uint64_t ce_abs,
                                                 uint64_t de_abs, uint64_t cs, uint32_t *bits, uint32_t *cnt,
                                                 unsigned long long o, bool *met, int32_t *sid = nullptr) {
    constexpr bool kMeet = MODE == 1 || MODE == 3, kWrite = MODE == 2 || MODE == 3;
    uint32_t p = (uint32_t)(p_abs - cs);
    const uint32_t ce = (uint32_t)(ce_abs - cs);
    const uint32_t de = de_abs - cs < 0x7FFFFFFFull ? (uint32_t)(de_abs - cs) : 0x7FFFFFFFu;
    uint32_t c = 0;
    if (kMeet) *met = false;
    if (p < ce && kMeet) {
        if ((bits[(p >> 5) * kBS] >> (p & 31)) & 1u) {
            *met = true;
            *cnt = 0;
            return p;
        }
    }
    ByteWin byte{P.bytes + cs};
    int32_t node = 0;
    uint32_t y = 0, blen = 0;     // base|TERM of node; length of the best token so far
    int32_t bnode = -1, btid = 0; // best token: its slot (id in tid[]) or, at depth 1, its id
    uint32_t q = p;
    uint32_t bw = 0;              // MODE 0: token starts in the word of the current token's start
    uint32_t *const stage = bits - 8 * kBS;   // MODE 0: the eight staged tokens sit just before bits
    // a token's first step, through the shared LUT (every byte is a token)
    auto root_step = [&](uint32_t ch) {
        const int4 r = lut[ch];
        node = r.x;
        y = (uint32_t)r.y;
        btid = r.z;
        blen = 1;
        bnode = -1;
        q = p + 1;
    };
    if (p < ce) root_step(byte(p));
    while (p < ce) {
        const uint32_t base = y & ~kTermBit;
        const bool load = q < de && base != 0;
        bool ok = false;
        int32_t nt = 0;
        uint32_t ny = 0, ch = 0;
        if (load) {
            ch = byte(q);
            ok = trie_step<L>(P, node, base, ch, &nt, &ny);
        }
        if (ok) {
            node = nt;
            y = ny;
            ++q;
            if (ny & kTermBit) {
                blen = q - p;
                bnode = nt;
            }
        } else {   // the token [p, p + blen) ends here; the next one starts in the same step
            if (MODE == 0) {
                bw |= 1u << (p & 31);
                if (sid) {
                    stage[(c & 7u) * kBS] = bnode >= 0 ? 0x80000000u | (uint32_t)bnode : (uint32_t)btid;
                    if ((c & 7u) == 7u) {   // a whole sector
                        uint4 *d = reinterpret_cast<uint4 *>(sid + (c & ~7u));
                        d[0] = make_uint4(stage[0], stage[kBS], stage[2 * kBS], stage[3 * kBS]);
                        d[1] = make_uint4(stage[4 * kBS], stage[5 * kBS], stage[6 * kBS], stage[7 * kBS]);
                    }
                }
            }
            if (kWrite && o < P.cap) P.ids[o] = bnode >= 0 ? __ldg(P.tid + bnode) : btid;
            ++o;
            ++c;
            const bool at_q = load && p + blen == q;   // the failed byte starts the next token
            p += blen;
            if (MODE == 0 && ((p ^ (p - blen)) >> 5)) {   // the next token starts in a later word
                bits[((p - blen) >> 5) * kBS] = bw;
                bw = 0;
            }
            if (kMeet && p < ce) {
                if ((bits[(p >> 5) * kBS] >> (p & 31)) & 1u) {
                    *met = true;
                    break;
                }
            }
            if (p < ce) root_step(at_q ? ch : byte(p));
        }
    }
    if (MODE == 0 && bw) bits[((p - blen) >> 5) * kBS] = bw;   // the last token's word
    *cnt = c;
    return p;
}

// k_spec's dynamic shared memory: the token-start bitmaps, then 8 staged
// tokens per thread (both one column per thread)
__host__ __device__ __forceinline__ size_t spec_smem_for(uint32_t C) {
    return (size_t)kSpecThreads * (C / 32) * 4 + (size_t)kSpecThreads * 8 * 4;
}
__host__ __device__ __forceinline__ size_t emit_smem_for(uint32_t C) { return (size_t)kEmitThreads * (C / 32) * 4; }
// Stored speculative ids take 4 bytes per input byte; above this the emit
// pass re-parses instead (also when the allocation fails).
constexpr uint64_t kMaxSpecIdBytes = 16ull << 30;

// ---------------------------------------------------------- chunk index ---

__global__ void __launch_bounds__(1024) k_chunk_index(EncParams P, unsigned long long *chunk_start) {
    __shared__ unsigned long long s_w[32];
    __shared__ unsigned long long s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (uint64_t base = 0; base < P.n_docs; base += 1024) {
        const uint64_t d = base + tid;
        unsigned long long v = 0;
        if (d < P.n_docs) {
            const uint64_t a = P.doc_off[d], b = P.doc_off[d + 1];
            if (b < a) {
                atomicOr(&P.st->err, DERR_OOB);
                P.st->bad_doc_off = (uint32_t)d;
            } else {
                v = (b - a + P.chunk - 1) / P.chunk;
            }
        }
        unsigned long long x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_w[warp] = x;
        __syncthreads();
        unsigned long long wpre = 0, tot = 0;
        for (int w = 0; w < 32; w++) {
            if (w < warp) wpre += s_w[w];
            tot += s_w[w];
        }
        const unsigned long long carry = s_carry;
        if (d < P.n_docs) chunk_start[d] = carry + wpre + x - v;
        __syncthreads();
        if (tid == 0) s_carry = carry + tot;
        __syncthreads();
    }
    if (tid == 0) {
        chunk_start[P.n_docs] = s_carry;
        P.st->n_chunks = s_carry;
        P.st->span = P.doc_off[P.n_docs] - P.doc_off[0];
        P.st->text_lo = P.doc_off[0];
    }
}

// ------------------------------------------------ speculative parse + fix ---

template <int L>
__global__ void __launch_bounds__(kSpecThreads, 8) k_spec(EncParams P, unsigned long long n_chunks, uint64_t text_end) {
    extern __shared__ uint32_t s_bits[];   // 8 staged tokens, then the C/32-word token-start bitmap: a column per thread
    __shared__ int4 lut[256];
    __shared__ uint32_t s_exit[kSpecThreads];   // each chunk's spec exit, from its start
    const int tid = threadIdx.x;
    const uint32_t words = P.chunk >> 5;
    uint32_t *stage = s_bits + tid, *bits = stage + 8 * kBS;
    const long long k = (long long)blockIdx.x * (kSpecThreads - 1) + tid - 1;
    const bool live = k >= 0 && (unsigned long long)k < n_chunks;
    load_lut(P, lut);

    __syncthreads();

    uint32_t spec_count = 0, spec_rel = 0;
    if (live) {
        const ChunkGeo g = chunk_geo(P, (unsigned long long)k);
        for (uint32_t w = 0; w < words; w++) bits[w * kBS] = 0;
        int32_t *sid = P.sids ? P.sids + (size_t)k * P.chunk : nullptr;
        spec_rel = parse_tokens<0, L>(P, lut, g.cs, g.ce, g.de, g.cs, bits, &spec_count, 0, nullptr, sid);
        if (sid)   // the last partial sector
            for (uint32_t i = spec_count & ~7u; i < spec_count; i++) sid[i] = (int32_t)stage[(i & 7u) * kBS];
        if (P.sbits)
            for (uint32_t w = 0; w < words; w++) P.sbits[(size_t)k * words + w] = bits[w * kBS];
    }
    s_exit[tid] = spec_rel;
    __syncthreads();
    if (!live || tid == 0) return;   // the halo thread only supplied its exit

    // the geometry again: reloaded rather than held in registers through the parse
    const ChunkGeo g = chunk_geo(P, (unsigned long long)k);
    uint32_t count, exit_rel;
    if (g.doc_first) {
        count = spec_count;
        exit_rel = spec_rel;
    } else {
        // re-parse from the nominal entry (previous chunk's spec exit) until the
        // two paths meet; from there the rest of the chunk is the spec path
        bool met = false;
        uint32_t c = 0;
        const uint32_t q =
            parse_tokens<1, L>(P, lut, (g.cs - P.chunk) + s_exit[tid - 1], g.ce, g.de, g.cs, bits, &c, 0, &met);
        if (met) {
            const uint32_t o = q;
            uint32_t rest = __popc(bits[(o >> 5) * kBS] >> (o & 31));
            for (uint32_t w = (o >> 5) + 1; w < words; w++) rest += __popc(bits[w * kBS]);
            c += rest;
            exit_rel = spec_rel;
        } else {
            exit_rel = q;
        }
        count = c;
    }
    P.count[k] = count;
    P.exit_rel[k] = exit_rel;
    P.spec_rel[k] = spec_rel;
    if (exit_rel != spec_rel) {
        atomicOr(P.flag + (k >> 5), 1u << (k & 31));
        P.st->any_flag = 1u;
        const uint32_t i = atomicAdd(&P.st->flist_len, 1u);
        if (i < P.flist_cap) P.flist[i] = (uint32_t)k;
    }
}

// ---------------------------------------------------------------- repair ---

// Parse [e, ce) of a chunk fully; returns the count and sets *exit.
template <int L>
__device__ uint32_t parse_from(const EncParams &P, const int4 *lut, uint64_t e, uint64_t ce, uint64_t de,
                               uint64_t *exit) {
    uint32_t c = 0;
    while (e < ce) {
        e += match_at<L>(P, lut, e, de).len;
        ++c;
    }
    *exit = e;
    return c;
}

// Sequential repair from flagged chunk f (whose entry is true): re-parse the
// chunks after it from their true entries until an exit agrees with the next
// chunk's nominal entry again or the document ends.  Returns the last chunk
// rewritten (f if none).
template <int L>
__device__ unsigned long long repair_chain(const EncParams &P, const int4 *lut, unsigned long long f,
                                           unsigned long long n_chunks) {
    const ChunkGeo gf = chunk_geo(P, f);
    uint64_t e = gf.cs + P.exit_rel[f];
    unsigned long long c = f + 1;
    for (; c < n_chunks; c++) {
        const ChunkGeo g = chunk_geo(P, c);
        if (g.doc_first) break;           // next document: entry resets
        uint64_t x;
        P.count[c] = parse_from<L>(P, lut, e, g.ce, g.de, &x);
        P.exit_rel[c] = (uint32_t)(x - g.cs);
        if (x == g.cs + P.spec_rel[c]) return c;   // agrees with the next nominal entry
        e = x;
    }
    return c - 1;
}

constexpr int kWalkMax = 8;                    // chunks a parallel walker records
constexpr int kWalkWords = 2 + 2 * kWalkMax;   // length, "continues", (count, exit) pairs
constexpr uint32_t kFlagListCap = 4096;

// One walker per flagged chunk, all in parallel: the chain as it would be if
// the chunk's entry is true, recorded privately (up to kWalkMax chunks).
template <int LY>
__global__ void k_repair_walk(EncParams P, unsigned long long n_chunks) {
    __shared__ int4 lut[256];
    const uint32_t L = P.st->flist_len;
    if (L == 0 || L > P.flist_cap) return;
    load_lut(P, lut);
    __syncthreads();
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < L; i += gridDim.x * blockDim.x) {
        const unsigned long long f = P.flist[i];
        uint32_t *w = P.wpriv + (size_t)i * kWalkWords;
        const ChunkGeo gf = chunk_geo(P, f);
        uint64_t e = gf.cs + P.exit_rel[f];
        uint32_t m = 0, more = 0;
        for (unsigned long long c = f + 1; c < n_chunks; c++) {
            const ChunkGeo g = chunk_geo(P, c);
            if (g.doc_first) break;
            if (m == kWalkMax) {
                more = 1;
                break;
            }
            uint64_t x;
            w[2 + 2 * m] = parse_from<LY>(P, lut, e, g.ce, g.de, &x);
            w[3 + 2 * m] = (uint32_t)(x - g.cs);
            ++m;
            if (x == g.cs + P.spec_rel[c]) break;
            e = x;
        }
        w[0] = m;
        w[1] = more;
    }
}

// Apply the walks of flagged chunks whose entry is true: in chunk order, a
// flagged chunk inside the chain of an earlier applied one has a wrong entry
// and is skipped.  With more flags than the list holds, repair sequentially.
template <int LY>
__global__ void __launch_bounds__(1024) k_repair_apply(EncParams P, unsigned long long n_chunks) {
    __shared__ int4 lut[256];
    __shared__ unsigned long long keys[kFlagListCap];
    const uint32_t L = P.st->flist_len;
    if (L == 0) return;
    load_lut(P, lut);
    if (L > P.flist_cap) {   // sequential repair over the flag bitmap
        __syncthreads();
        if (threadIdx.x != 0) return;
        const unsigned long long nw = (n_chunks + 31) >> 5;
        unsigned long long k = 0;
        for (;;) {
            unsigned long long w = k >> 5;
            uint32_t bitsw = w < nw ? (P.flag[w] & (~0u << (k & 31))) : 0u;
            while (w < nw && bitsw == 0) {
                ++w;
                if (w < nw) bitsw = P.flag[w];
            }
            if (w >= nw) break;
            const unsigned long long f = (w << 5) + (unsigned long long)(__ffs(bitsw) - 1);
            if (f >= n_chunks) break;
            k = repair_chain<LY>(P, lut, f, n_chunks) + 1;
        }
        return;
    }
    uint32_t n2 = 1;
    while (n2 < L) n2 <<= 1;
    for (uint32_t i = threadIdx.x; i < n2; i += blockDim.x)
        keys[i] = i < L ? (((unsigned long long)P.flist[i] << 12) | i) : ~0ull;
    __syncthreads();
    for (uint32_t k = 2; k <= n2; k <<= 1) {   // bitonic sort by chunk index
        for (uint32_t j = k >> 1; j > 0; j >>= 1) {
            for (uint32_t t = threadIdx.x; t < n2; t += blockDim.x) {
                const uint32_t x = t ^ j;
                if (x > t) {
                    const bool up = (t & k) == 0;
                    const unsigned long long a = keys[t], b = keys[x];
                    if ((a > b) == up) {
                        keys[t] = b;
                        keys[x] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    if (threadIdx.x != 0) return;
    long long cur_end = -1;   // last chunk settled by an applied chain
    for (uint32_t q = 0; q < L; q++) {
        const unsigned long long f = keys[q] >> 12;
        const uint32_t i = (uint32_t)(keys[q] & 0xFFFu);
        if ((long long)f <= cur_end) continue;
        const uint32_t *w = P.wpriv + (size_t)i * kWalkWords;
        const uint32_t m = w[0];
        for (uint32_t r = 0; r < m; r++) {
            P.count[f + 1 + r] = w[2 + 2 * r];
            P.exit_rel[f + 1 + r] = w[3 + 2 * r];
        }
        cur_end = (long long)(f + m);
        if (w[1]) cur_end = (long long)repair_chain<LY>(P, lut, f + m, n_chunks);   // a long chain goes on
    }
}

// ------------------------------------------------------------ scan + emit ---

template <int L>
__global__ void __launch_bounds__(kEmitThreads) k_emit(EncParams P, unsigned long long n_chunks, uint64_t text_end) {
    extern __shared__ uint32_t s_bits[];   // kEmitThreads x (C/32): each chunk's spec token starts
    __shared__ int4 lut[256];
    __shared__ unsigned long long s_csrc[kEmitThreads], s_cdst[kEmitThreads];   // per chunk: copy source, target
    __shared__ uint32_t s_cbeg[kEmitThreads];                                  // per chunk: start in the warp's range
    __shared__ uint32_t s_w[kEmitThreads / 32];
    __shared__ unsigned long long s_tile, s_off;
    load_lut(P, lut);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned long long ntiles = (n_chunks + kEmitThreads - 1) / kEmitThreads;
    if (tid == 0) s_tile = atomicAdd(&P.st->ticket, 1u);   // tiles in ticket order
    __syncthreads();
    const unsigned long long t = s_tile;
    if (t >= ntiles) return;
    const unsigned long long k = t * kEmitThreads + tid;
    const bool live = k < n_chunks;
    ChunkGeo g{0, 0, 0, true};
    if (live) g = chunk_geo(P, k);
    const uint32_t cnt = live ? P.count[k] : 0u;
    const uint32_t incl = warp_incl_sum(cnt, lane);
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    uint32_t wpre = 0, tsum = 0;
#pragma unroll
    for (int w = 0; w < kEmitThreads / 32; w++) {
        if (w < warp) wpre += s_w[w];
        tsum += s_w[w];
    }
    if (warp == 0) {   // publish, then look back 32 predecessors per round trip
        unsigned long long off = 0;
        if (t > 0) {
            if (lane == 0) st_relaxed(P.status + t, 1ull | ((unsigned long long)tsum << 2));
            long long jhi = (long long)t - 1;
            unsigned spins = 0;
            for (;;) {
                const long long j = jhi - lane;
                const unsigned long long w = (j >= 0) ? ld_l2(P.status + j) : 2ull;
                const uint32_t fl = (uint32_t)(w & 3ull);
                const unsigned incl_m = __ballot_sync(kFull, fl == 2);
                const int li = incl_m ? __ffs(incl_m) - 1 : 31;   // first lane holding an inclusive prefix
                const unsigned need = (li == 31) ? kFull : ((2u << li) - 1u);
                if (__ballot_sync(kFull, fl == 0) & need) {
                    if (++spins > kSpinLimit) {
                        if (lane == 0) atomicOr(&P.st->err, DERR_TIMEOUT);
                        break;
                    }
                    if (spins > 32) __nanosleep(64);
                    continue;
                }
                unsigned long long v = (lane <= li) ? (w >> 2) : 0ull;
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
                off += v;
                if (incl_m) break;
                jhi -= 32;
            }
        }
        if (lane == 0) {
            st_relaxed(P.status + t, 2ull | ((off + tsum) << 2));
            if (t == ntiles - 1) P.st->total = off + tsum;
            s_off = off;
        }
    }
    __syncthreads();
    const unsigned long long o = s_off + wpre + incl - cnt;
    if (live) P.prefix[k] = o;
    if (!P.sids) {   // re-parse the chunk from its true entry
        if (live) {
            const uint64_t e = g.doc_first ? g.cs : (g.cs - P.chunk) + P.exit_rel[k - 1];
            uint32_t c = 0;
            parse_tokens<2, L>(P, lut, e, g.ce, g.de, g.cs, nullptr, &c, o, nullptr);
        }
        return;
    }
    // Parse from the true entry only until the path meets a token start of the
    // speculative parse; the rest of the chunk's ids are the stored ones.
    uint32_t src_t = 0, n_copy = 0, c_head = 0;
    if (live) {
        const uint32_t words = P.chunk >> 5;
        uint32_t *bits = s_bits + tid;
        uint32_t n_spec = 0;
        for (uint32_t w = 0; w < words; w++) {
            bits[w * kBS] = P.sbits[(size_t)k * words + w];
            n_spec += __popc(bits[w * kBS]);
        }
        const uint64_t e = g.doc_first ? g.cs : (g.cs - P.chunk) + P.exit_rel[k - 1];
        bool met = false;
        const uint32_t off = parse_tokens<3, L>(P, lut, e, g.ce, g.de, g.cs, bits, &c_head, o, &met);
        if (met) {   // spec tokens before offset off are skipped
            uint32_t before = 0;
            for (uint32_t w = 0; w < (off >> 5); w++) before += __popc(bits[w * kBS]);
            before += __popc(bits[(off >> 5) * kBS] & ((1u << (off & 31)) - 1u));
            src_t = before;
            n_copy = n_spec - before;
        }
    }
    // The warp's 32 tails form one range of W ids: lane L copies ids L, L+32,
    // ... (coalesced reads and writes, four in flight), finding each id's
    // chunk by a binary search over the tails' starts.
    const unsigned long long dst = o + c_head;
    const uint32_t tincl = warp_incl_sum(n_copy, lane);
    const uint32_t W = __shfl_sync(kFull, tincl, 31);
    unsigned long long *wsrc = s_csrc + warp * 32, *wdst = s_cdst + warp * 32;
    uint32_t *wbeg = s_cbeg + warp * 32;
    wbeg[lane] = tincl - n_copy;
    wsrc[lane] = (unsigned long long)k * P.chunk + src_t;
    wdst[lane] = dst;
    __syncwarp();
    for (uint32_t w0 = 0; w0 < W; w0 += 4 * 32) {
        int32_t v[4];
        unsigned long long d[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const uint32_t w = w0 + u * 32 + lane;
            d[u] = ~0ull;
            if (w < W) {
                int j = 0;   // last lane whose tail starts at or before w
#pragma unroll
                for (int step = 16; step > 0; step >>= 1)
                    if (wbeg[j + step] <= w) j += step;
                const uint32_t r = w - wbeg[j];
                v[u] = __ldcs(P.sids + wsrc[j] + r);
                d[u] = wdst[j] + r;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; u++) {
            if (d[u] != ~0ull && d[u] < P.cap) {
                const int32_t x = v[u];
                P.ids[d[u]] = x < 0 ? __ldg(P.tid + (x & 0x7FFFFFFF)) : x;
            }
        }
    }
}

// Small transfers done by one CTA instead of a copy engine, so they never
// queue behind a large host transfer on another stream (the host side is
// pinned memory, which the device addresses directly).
__global__ void k_copy_small(const uint8_t *src, uint8_t *dst, uint32_t n) {
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}
__global__ void k_set_doc(uint64_t *off, uint64_t total) {
    off[0] = 0;
    off[1] = total;
}

__global__ void k_doc_offsets(EncParams P, unsigned long long n_chunks) {
    const uint64_t d = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    if (d > P.n_docs) return;
    const unsigned long long c = P.chunk_start[d];
    P.id_off[d] = c < n_chunks ? P.prefix[c] : P.st->total;
}

// Streaming ([GPU-BPE] "Host architecture", 3. multi-pass slicing, with the
// parse carried across slices): the prefix of one document's parse [0, end)
// that no later byte can change.  A token starting max_len or more bytes
// before the end is final (its walk stops within max_len bytes); from the
// last chunk exit at or before end - max_len the tokens are walked again
// until the first whose walk reached the end.  out[0]: number of final ids;
// out[1]: position of the first token that is not final (end if none).
template <int L>
__global__ void k_stream_cut(EncParams P, unsigned long long n_chunks, uint64_t end, uint32_t max_len,
                             unsigned long long *out) {
    __shared__ int4 lut[256];
    load_lut(P, lut);
    __syncthreads();
    if (threadIdx.x != 0) return;
    const uint64_t safe = end > max_len ? end - max_len : 0;
    long long lo = -1, hi = (long long)n_chunks;   // last chunk c with exit(c) <= safe
    while (hi - lo > 1) {
        const long long mid = (lo + hi) / 2;
        if ((uint64_t)mid * P.chunk + P.exit_rel[mid] <= safe) lo = mid;
        else hi = mid;
    }
    uint64_t b = 0;
    unsigned long long ids = 0;
    if (lo >= 0) {
        b = (uint64_t)lo * P.chunk + P.exit_rel[lo];
        ids = P.prefix[lo] + P.count[lo];
    }
    while (b < end) {
        uint32_t len;
        if (!match_final<L>(P, lut, b, end, &len)) break;
        b += len;
        ++ids;
    }
    out[0] = ids;
    out[1] = b;
}

// The bitmap-node layout from the double array ([UNIGRAM] "Bitmap and inline
// packing"): node i gets base | TERM and, for every slot j whose check names
// i, bit j - base(i) of its child bitmap.
__global__ void k_build_bm(const int2 *slot, unsigned long long n_slots, BmNode *bm) {
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n_slots;
         i += (unsigned long long)gridDim.x * blockDim.x) {
        const int2 v = slot[i];
        bm[i].by = (uint32_t)v.y;
        if (v.x >= 0) {   // a child of slot v.x
            const uint32_t c = (uint32_t)(i - (slot[v.x].y & ~kTermBit));
            atomicOr(&bm[v.x].bits[c >> 6], 1ull << (c & 63));
        }
    }
}

}  // namespace

int trie_bitmap_nodes(bpe_ctx *ctx, const bpe_trie *trie) {
    if (trie->d_bm) return BPE_OK;
    bpe_trie *t = const_cast<bpe_trie *>(trie);   // built once, on first use
    void *p = nullptr;
    BPE_CUDA(ctx, cudaMalloc(&p, trie->n_slots * sizeof(BmNode)), "bitmap nodes");
    BPE_CUDA(ctx, cudaMemsetAsync(p, 0, trie->n_slots * sizeof(BmNode), ctx->stream), "bitmap nodes clear");
    k_build_bm<<<(unsigned)std::min<unsigned long long>((trie->n_slots + 255) / 256, 65535), 256, 0, ctx->stream>>>(
        trie->d_slot, trie->n_slots, (BmNode *)p);
    BPE_CUDA(ctx, cudaGetLastError(), "k_build_bm launch");
    BPE_CUDA(ctx, cudaStreamSynchronize(ctx->stream), "bitmap nodes sync");
    t->d_bm = p;
    return BPE_OK;
}

namespace {
}  // namespace
}  // namespace bpe

using namespace bpe;

extern "C" int trie_encode(bpe_ctx *ctx, const bpe_trie *trie, const uint8_t *d_bytes, const uint64_t *d_doc_off,
                           uint32_t n_docs, int32_t *d_ids_out, uint64_t ids_capacity, uint64_t *d_id_off_out,
                           uint64_t *n_ids) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (!trie || !n_ids) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode: null trie or n_ids");
    if (trie->device != ctx->device) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode: trie on another device");
    if (trie->missing_byte >= 0)
        return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode: byte 0x%02X is not a token of the vocabulary",
                    trie->missing_byte);
    if (n_docs && (!d_doc_off || !d_bytes)) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode: null input");
    if (ids_capacity && !d_ids_out) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode: null ids with capacity");
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    cudaStream_t s = ctx->stream;
    stats_reset(ctx);
    *n_ids = 0;
    if (n_docs == 0) {
        if (d_id_off_out) BPE_CUDA(ctx, cudaMemsetAsync(d_id_off_out, 0, 8, s), "id_off");
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "sync");
        return BPE_OK;
    }
    const uint32_t C = (uint32_t)std::min(ctx->chunk, kMaxChunk);
    int rc;
    void *cstart, *state, *pin;
    if ((rc = ensure(ctx, S_ENC_CHUNK_START, ((uint64_t)n_docs + 1) * 8, &cstart)) ||
        (rc = ensure(ctx, S_ENC_STATE, sizeof(EncState), &state)) ||
        (rc = ensure_pinned(ctx, sizeof(EncState), &pin)))
        return rc;
    EncState *h = (EncState *)pin;
    const bool profile = ctx->profile != 0;
    if (profile && (rc = ensure_events(ctx, 6))) return rc;

    EncParams P{};
    P.bytes = d_bytes;
    P.doc_off = d_doc_off;
    P.n_docs = n_docs;
    P.chunk = C;
    P.chunk_start = (const unsigned long long *)cstart;
    P.slot = trie->d_slot;
    P.tid = trie->d_tid;
    P.root = trie->d_root;
    P.ids = d_ids_out;
    P.cap = ids_capacity;
    P.st = (EncState *)state;

    // phase 1: chunk index (needs the chunk count on the host to size the rest)
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "sync");
    BPE_CUDA(ctx, cudaMemsetAsync(state, 0, sizeof(EncState), s), "state clear");
    if (profile) cudaEventRecord(ctx->events[0], s);
    k_chunk_index<<<1, 1024, 0, s>>>(P, (unsigned long long *)cstart);
    if (profile) cudaEventRecord(ctx->events[1], s);
    BPE_CUDA(ctx, cudaGetLastError(), "k_chunk_index launch");
    k_copy_small<<<1, 128, 0, s>>>((const uint8_t *)state, (uint8_t *)h, (uint32_t)sizeof(EncState));   // state read
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "chunk index sync");
    if (h->err & DERR_OOB)
        return fail(ctx, BPE_ERR_INVALID_ARG, "trie_encode: document offsets descend at document %u", h->bad_doc_off);
    const unsigned long long nc = h->n_chunks;
    const uint64_t text_end = h->text_lo + h->span;   // end of the last document
    if (nc == 0) {
        if (d_id_off_out) BPE_CUDA(ctx, cudaMemsetAsync(d_id_off_out, 0, ((uint64_t)n_docs + 1) * 8, s), "id_off");
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "sync");
        return BPE_OK;
    }

    void *info, *flag, *status, *prefix, *idoff_tmp = nullptr;
    const unsigned long long spec_blocks = (nc + kSpecThreads - 2) / (kSpecThreads - 1);
    const unsigned long long emit_tiles = (nc + kEmitThreads - 1) / kEmitThreads;
    if ((rc = ensure(ctx, S_ENC_CHUNK_INFO, nc * 12, &info)) ||
        (rc = ensure(ctx, S_ENC_NOTOK, ((nc + 31) / 32) * 4, &flag)) ||
        (rc = ensure(ctx, S_ENC_STATUS, emit_tiles * 8, &status)) ||
        (rc = ensure(ctx, S_ENC_PREFIX, nc * 8 + ((uint64_t)n_docs + 1) * 8 +
                                                (uint64_t)kFlagListCap * (1 + kWalkWords) * 4, &prefix)))
        return rc;
    P.chunk_start = (const unsigned long long *)cstart;   // (ensure may not move it: distinct slot)
    P.count = (uint32_t *)info;
    P.exit_rel = P.count + nc;
    P.spec_rel = P.exit_rel + nc;
    P.flag = (uint32_t *)flag;
    P.status = (unsigned long long *)status;
    P.prefix = (unsigned long long *)prefix;
    idoff_tmp = (unsigned long long *)prefix + nc;
    P.flist = (uint32_t *)((unsigned long long *)idoff_tmp + n_docs + 1);
    P.flist_cap = kFlagListCap;
    P.wpriv = P.flist + kFlagListCap;
    P.id_off = d_id_off_out ? (unsigned long long *)d_id_off_out : (unsigned long long *)idoff_tmp;
    // the speculative parse's ids and token starts, so emit copies instead of re-parsing
    const uint64_t sid_bytes = nc * (uint64_t)C * 4, sbit_bytes = nc * (uint64_t)(C / 32) * 4;
    if (sid_bytes <= kMaxSpecIdBytes) {
        void *sids = nullptr, *sbits = nullptr;
        if (ensure(ctx, S_ENC_SIDS, sid_bytes, &sids) == BPE_OK && ensure(ctx, S_ENC_SBITS, sbit_bytes, &sbits) == BPE_OK) {
            P.sids = (int32_t *)sids;
            P.sbits = (uint32_t *)sbits;
        } else {
            ctx->err.clear();   // no room: the emit pass re-parses
        }
    }

    BPE_CUDA(ctx, cudaMemsetAsync(flag, 0, ((nc + 31) / 32) * 4, s), "flag clear");
    BPE_CUDA(ctx, cudaMemsetAsync(status, 0, emit_tiles * 8, s), "status clear");
    const size_t spec_smem = spec_smem_for(C), emit_smem = emit_smem_for(C);
    const bool bm = ctx->trie_layout == BPE_TRIE_BITMAP;
    if (bm) {
        if ((rc = trie_bitmap_nodes(ctx, trie))) return rc;
        P.bm = (const BmNode *)trie->d_bm;
    }
    auto spec_fn = bm ? k_spec<1> : k_spec<0>;
    auto emit_fn = bm ? k_emit<1> : k_emit<0>;
    BPE_CUDA(ctx, cudaFuncSetAttribute(spec_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)spec_smem),
             "k_spec smem");
    BPE_CUDA(ctx, cudaFuncSetAttribute(emit_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)emit_smem),
             "k_emit smem");

    const unsigned long long emit_grid = emit_tiles;   // one tile per CTA, ticket order

    if (profile) cudaEventRecord(ctx->events[2], s);
    spec_fn<<<(unsigned)spec_blocks, kSpecThreads, spec_smem, s>>>(P, nc, text_end);
    if (profile) cudaEventRecord(ctx->events[3], s);
    (bm ? k_repair_walk<1> : k_repair_walk<0>)<<<16, 256, 0, s>>>(P, nc);
    (bm ? k_repair_apply<1> : k_repair_apply<0>)<<<1, 1024, 0, s>>>(P, nc);
    if (profile) cudaEventRecord(ctx->events[4], s);
    emit_fn<<<(unsigned)emit_grid, kEmitThreads, emit_smem, s>>>(P, nc, text_end);
    if (profile) cudaEventRecord(ctx->events[5], s);
    k_doc_offsets<<<(unsigned)((n_docs + 1 + 255) / 256), 256, 0, s>>>(P, nc);
    BPE_CUDA(ctx, cudaGetLastError(), "trie_encode launch");
    k_copy_small<<<1, 128, 0, s>>>((const uint8_t *)state, (uint8_t *)h, (uint32_t)sizeof(EncState));   // state read
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "trie_encode sync");
    if (h->err & DERR_TIMEOUT) return fail(ctx, BPE_ERR_TIMEOUT, "trie_encode: look-back wait gave up");

    const uint64_t total = h->total;
    *n_ids = total;

    // statistics, in the encode's algorithmic bytes (the input once, 4 bytes
    // per id and 8 per document offset): the spec parse is charged the input,
    // the emit pass the ids and offsets it writes
    const int a = stats_slot(ctx, "encode_spec"), b = stats_slot(ctx, "encode_emit");
    ctx->stats.k[a].launches = 1;
    ctx->stats.k[b].launches = 1;
    const uint64_t in_bytes = h->span;
    ctx->stats.kernel_launches = 6;
    ctx->stats.k[a].bytes = (double)in_bytes;
    ctx->stats.k[b].bytes = 4.0 * (double)total + 8.0 * ((double)n_docs + 1.0);
    if (profile) {
        float x = 0, y = 0, z = 0;
        cudaEventElapsedTime(&x, ctx->events[2], ctx->events[3]);
        cudaEventElapsedTime(&y, ctx->events[4], ctx->events[5]);
        cudaEventElapsedTime(&z, ctx->events[3], ctx->events[4]);
        ctx->stats.k[a].ms = x;
        ctx->stats.k[b].ms = y;
        const int c = stats_slot(ctx, "encode_repair");
        ctx->stats.k[c].launches = 1;
        ctx->stats.k[c].ms = z;
        cudaGetLastError();
    }
    if (total > ids_capacity)
        return fail(ctx, BPE_ERR_CAPACITY, "trie_encode: %llu ids exceed the capacity %llu",
                    (unsigned long long)total, (unsigned long long)ids_capacity);
    return BPE_OK;
}

// ---------------------------------------------------------------------------
// Streaming encode of one document arriving in slices.  Each push encodes the
// carried bytes followed by the new slice as one document, hands back the ids
// no later byte can change and carries the bytes of the rest (fewer than the
// longest token) to the next push; the last push makes everything final.

struct bpe_stream {
    bpe_ctx *ctx = nullptr;
    const bpe_trie *trie = nullptr;
    uint8_t *d_buf = nullptr;          // carried bytes, then the slice
    size_t cap = 0;
    uint8_t *d_carry = nullptr;        // the carried bytes between pushes
    uint32_t carry = 0;
    uint64_t *d_off = nullptr;         // {0, total}: the one document
    unsigned long long *d_cut = nullptr;
    unsigned long long *h_cut = nullptr;   // pinned: final ids, cut position; then {0, total}
};

extern "C" int trie_stream_open(bpe_ctx *ctx, const bpe_trie *trie, bpe_stream **out) {
    if (!ctx || !trie || !out) return BPE_ERR_INVALID_ARG;
    *out = nullptr;
    if (trie->device != ctx->device) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_stream_open: trie on another device");
    if (trie->missing_byte >= 0)
        return fail(ctx, BPE_ERR_INVALID_ARG, "trie_stream_open: byte 0x%02X is not a token of the vocabulary",
                    trie->missing_byte);
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    bpe_stream *st = new bpe_stream();
    st->ctx = ctx;
    st->trie = trie;
    cudaError_t e = cudaMalloc(&st->d_carry, (size_t)trie->max_len + 16);
    if (e == cudaSuccess) e = cudaMalloc(&st->d_off, 2 * sizeof(uint64_t));
    if (e == cudaSuccess) e = cudaMalloc(&st->d_cut, 2 * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMallocHost(&st->h_cut, 4 * sizeof(unsigned long long));
    if (e != cudaSuccess) {
        trie_stream_close(st);
        return cuda_fail(ctx, e, "trie_stream_open");
    }
    *out = st;
    return BPE_OK;
}

extern "C" void trie_stream_close(bpe_stream *st) {
    if (!st) return;
    if (st->ctx) {
        cudaSetDevice(st->ctx->device);
        cudaStreamSynchronize(st->ctx->stream);
    }
    if (st->d_buf) cudaFree(st->d_buf);
    if (st->d_carry) cudaFree(st->d_carry);
    if (st->d_off) cudaFree(st->d_off);
    if (st->d_cut) cudaFree(st->d_cut);
    if (st->h_cut) cudaFreeHost(st->h_cut);
    delete st;
}

// Encode the document doc[0 .. total) (the carried bytes, then the slice) and
// keep the bytes after the final prefix of its parse as the next carry.
static int stream_encode(bpe_stream *st, const uint8_t *doc, uint64_t total, int last, int32_t *d_ids_out,
                         uint64_t ids_capacity, uint64_t *n_ids) {
    bpe_ctx *ctx = st->ctx;
    cudaStream_t s = ctx->stream;
    if (total == 0) {
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "sync");
        return BPE_OK;
    }
    k_set_doc<<<1, 1, 0, s>>>(st->d_off, total);
    uint64_t all = 0;
    int rc = trie_encode(ctx, st->trie, doc, st->d_off, 1, d_ids_out, ids_capacity, nullptr, &all);
    if (rc) {
        *n_ids = all;
        return rc;
    }
    if (last) {
        st->carry = 0;
        *n_ids = all;
        return BPE_OK;
    }
    // the final prefix of the parse: the chunk arrays of that encode are still in the pool
    const uint32_t C = (uint32_t)std::min(ctx->chunk, kMaxChunk);
    const unsigned long long nc = (total + C - 1) / C;
    EncParams P{};
    P.bytes = doc;
    P.chunk = C;
    P.slot = st->trie->d_slot;
    P.tid = st->trie->d_tid;
    P.root = st->trie->d_root;
    P.count = (uint32_t *)ctx->scratch[S_ENC_CHUNK_INFO].p;
    P.exit_rel = P.count + nc;
    P.prefix = (unsigned long long *)ctx->scratch[S_ENC_PREFIX].p;
    P.bm = (const BmNode *)st->trie->d_bm;   // built by the encode above when that layout is on
    (ctx->trie_layout == BPE_TRIE_BITMAP ? k_stream_cut<1> : k_stream_cut<0>)<<<1, 256, 0, s>>>(
        P, nc, total, st->trie->max_len, st->d_cut);
    BPE_CUDA(ctx, cudaGetLastError(), "k_stream_cut launch");
    k_copy_small<<<1, 32, 0, s>>>((const uint8_t *)st->d_cut, (uint8_t *)st->h_cut, 2 * sizeof(unsigned long long));
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "cut sync");
    const uint64_t cut = st->h_cut[1];
    st->carry = (uint32_t)(total - cut);   // below the longest token
    if (st->carry)
        k_copy_small<<<1, 256, 0, s>>>(doc + cut, st->d_carry, st->carry);   // carry keep
    *n_ids = st->h_cut[0];
    ctx->stats.kernel_launches += 1;
    return BPE_OK;
}

extern "C" int trie_stream_push(bpe_stream *st, const uint8_t *d_bytes, uint64_t n, int last, int32_t *d_ids_out,
                                uint64_t ids_capacity, uint64_t *n_ids) {
    if (!st || !n_ids) return BPE_ERR_INVALID_ARG;
    bpe_ctx *ctx = st->ctx;
    *n_ids = 0;
    if (n && !d_bytes) return fail(ctx, BPE_ERR_INVALID_ARG, "trie_stream_push: null bytes");
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    cudaStream_t s = ctx->stream;
    const uint64_t total = (uint64_t)st->carry + n;
    if (st->cap < total + 16) {   // grow the staging buffer (x1.5, like the context's pool)
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "stream grow sync");
        if (st->d_buf) cudaFree(st->d_buf);
        st->d_buf = nullptr;
        st->cap = 0;
        const size_t want = (size_t)(total + total / 2 + 256);
        BPE_CUDA(ctx, cudaMalloc(&st->d_buf, want), "trie_stream_push: staging buffer");
        st->cap = want;
    }
    if (st->carry)
        BPE_CUDA(ctx, cudaMemcpyAsync(st->d_buf, st->d_carry, st->carry, cudaMemcpyDeviceToDevice, s), "carry copy");
    if (n) BPE_CUDA(ctx, cudaMemcpyAsync(st->d_buf + st->carry, d_bytes, n, cudaMemcpyDeviceToDevice, s), "slice copy");
    return stream_encode(st, st->d_buf, total, last, d_ids_out, ids_capacity, n_ids);
}

namespace bpe {
void stream_reset(bpe_stream *st) {
    if (st) st->carry = 0;
}

// The slice already sits in device memory with at least the trie's longest
// token length of writable bytes before it: the carry goes there, so the
// slice itself is not copied.
int stream_push_in_place(bpe_stream *st, uint8_t *d_slice, uint64_t n, int last, int32_t *d_ids_out,
                         uint64_t ids_capacity, uint64_t *n_ids) {
    *n_ids = 0;
    uint8_t *doc = d_slice - st->carry;
    if (st->carry)
        k_copy_small<<<1, 256, 0, st->ctx->stream>>>(st->d_carry, doc, st->carry);   // carry copy
    return stream_encode(st, doc, (uint64_t)st->carry + n, last, d_ids_out, ids_capacity, n_ids);
}
}  // namespace bpe

// ---------------------------------------------------------------------------
// trie_encode_noalloc: the same kernels, with every scratch buffer carved out
// of one fixed device array instead of the context's pool, for callers that
// must not allocate device memory.  The array is part of the library's
// module: each GPU that loads the library holds it until the process exits.
namespace bpe {
namespace {

constexpr uint32_t kNaMaxDocs = 65536;
constexpr uint64_t kNaMaxChunks = 524288;          // 128-byte chunks: up to 64 MiB of text
constexpr uint32_t kNaChunk = 128;
constexpr size_t na_align(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kNaOffState = 0;
constexpr size_t kNaOffChunkStart = na_align(sizeof(EncState));
constexpr size_t kNaOffInfo = na_align(kNaOffChunkStart + 8 * ((size_t)kNaMaxDocs + 1));
constexpr size_t kNaOffFlag = na_align(kNaOffInfo + 12 * kNaMaxChunks);
constexpr size_t kNaOffStatus = na_align(kNaOffFlag + kNaMaxChunks / 8);
constexpr size_t kNaOffPrefix = na_align(kNaOffStatus + 8 * (kNaMaxChunks / kEmitThreads + 1));
constexpr size_t kNaOffIdOff = na_align(kNaOffPrefix + 8 * kNaMaxChunks);
constexpr size_t kNaOffFlist = na_align(kNaOffIdOff + 8 * ((size_t)kNaMaxDocs + 1));
constexpr size_t kNaBytes = na_align(kNaOffFlist + 4 * (size_t)kFlagListCap * (1 + kWalkWords));   // about 11.9 MB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

// Device address of g_noalloc_scratch per device, looked up once with that
// device current (the host-side name is only a stand-in, never a device
// address).
std::mutex g_na_mu;
void *g_na_addr[256] = {};

cudaError_t noalloc_scratch(int device, unsigned char **out) {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (device < 0 || device >= 256) return cudaErrorInvalidDevice;
    if (!g_na_addr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_na_addr[device] = p;
    }
    *out = (unsigned char *)g_na_addr[device];
    return cudaSuccess;
}

struct DeviceGuard {   // restores the caller's current device
    int prev = -1;
    explicit DeviceGuard(int d) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        cudaSetDevice(d);
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

int noalloc_body(const bpe_trie *trie, const uint8_t *d_bytes, const uint64_t *d_doc_off, uint32_t n_docs,
                 int32_t *d_ids_out, uint64_t ids_capacity, uint64_t *d_id_off_out, uint64_t *n_ids,
                 cudaStream_t s) {
    unsigned char *base = nullptr;
    if (noalloc_scratch(trie->device, &base) != cudaSuccess) return BPE_ERR_CUDA;
    EncParams P{};
    P.bytes = d_bytes;
    P.doc_off = d_doc_off;
    P.n_docs = n_docs;
    P.chunk = kNaChunk;
    P.chunk_start = (const unsigned long long *)(base + kNaOffChunkStart);
    P.slot = trie->d_slot;
    P.tid = trie->d_tid;
    P.root = trie->d_root;
    P.ids = d_ids_out;
    P.cap = ids_capacity;
    P.st = (EncState *)(base + kNaOffState);
    P.count = (uint32_t *)(base + kNaOffInfo);
    P.exit_rel = P.count + kNaMaxChunks;
    P.spec_rel = P.exit_rel + kNaMaxChunks;
    P.flag = (uint32_t *)(base + kNaOffFlag);
    P.status = (unsigned long long *)(base + kNaOffStatus);
    P.prefix = (unsigned long long *)(base + kNaOffPrefix);
    P.id_off = d_id_off_out ? (unsigned long long *)d_id_off_out : (unsigned long long *)(base + kNaOffIdOff);
    P.flist = (uint32_t *)(base + kNaOffFlist);
    P.flist_cap = kFlagListCap;
    P.wpriv = P.flist + kFlagListCap;

    // the array keeps the previous call's contents: zero what must start at zero
    if (cudaMemsetAsync(P.st, 0, sizeof(EncState), s) != cudaSuccess) return BPE_ERR_CUDA;
    k_chunk_index<<<1, 1024, 0, s>>>(P, (unsigned long long *)(base + kNaOffChunkStart));
    EncState h;
    if (cudaMemcpyAsync(&h, P.st, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BPE_ERR_CUDA;
    if (h.err & DERR_OOB) return BPE_ERR_INVALID_ARG;
    const unsigned long long nc = h.n_chunks;
    if (nc > kNaMaxChunks) return BPE_ERR_INVALID_ARG;
    if (nc == 0) {
        if (d_id_off_out && cudaMemsetAsync(d_id_off_out, 0, 8 * ((size_t)n_docs + 1), s) != cudaSuccess)
            return BPE_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return BPE_ERR_CUDA;
        *n_ids = 0;
        return BPE_OK;
    }
    const unsigned long long spec_blocks = (nc + kSpecThreads - 2) / (kSpecThreads - 1);
    const unsigned long long emit_tiles = (nc + kEmitThreads - 1) / kEmitThreads;
    if (cudaMemsetAsync(P.flag, 0, ((nc + 31) / 32) * 4, s) != cudaSuccess ||
        cudaMemsetAsync(P.status, 0, emit_tiles * 8, s) != cudaSuccess)
        return BPE_ERR_CUDA;
    const size_t spec_smem = spec_smem_for(kNaChunk), emit_smem = emit_smem_for(kNaChunk);
    if (cudaFuncSetAttribute(k_spec<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)spec_smem) != cudaSuccess ||
        cudaFuncSetAttribute(k_emit<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)emit_smem) != cudaSuccess)
        return BPE_ERR_CUDA;
    const uint64_t text_end = h.span + h.text_lo;
    k_spec<0><<<(unsigned)spec_blocks, kSpecThreads, spec_smem, s>>>(P, nc, text_end);
    k_repair_walk<0><<<16, 256, 0, s>>>(P, nc);
    k_repair_apply<0><<<1, 1024, 0, s>>>(P, nc);
    k_emit<0><<<(unsigned)emit_tiles, kEmitThreads, emit_smem, s>>>(P, nc, text_end);
    k_doc_offsets<<<(unsigned)((n_docs + 1 + 255) / 256), 256, 0, s>>>(P, nc);
    if (cudaGetLastError() != cudaSuccess) return BPE_ERR_CUDA;
    if (cudaMemcpyAsync(&h, P.st, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BPE_ERR_CUDA;
    if (h.err & DERR_TIMEOUT) return BPE_ERR_TIMEOUT;
    *n_ids = h.total;
    return h.total > ids_capacity ? BPE_ERR_CAPACITY : BPE_OK;
}

}  // namespace
}  // namespace bpe

extern "C" int trie_encode_noalloc(const bpe_trie *trie, const uint8_t *d_bytes, const uint64_t *d_doc_off,
                                   uint32_t n_docs, int32_t *d_ids_out, uint64_t ids_capacity,
                                   uint64_t *d_id_off_out, uint64_t *n_ids, void *cuda_stream) {
    if (!trie || !n_ids) return BPE_ERR_INVALID_ARG;
    *n_ids = 0;
    if (trie->missing_byte >= 0) return BPE_ERR_INVALID_ARG;   // greedy needs every single byte
    if (n_docs > bpe::kNaMaxDocs) return BPE_ERR_INVALID_ARG;
    if (n_docs && (!d_doc_off || !d_bytes)) return BPE_ERR_INVALID_ARG;
    if (ids_capacity && !d_ids_out) return BPE_ERR_INVALID_ARG;
    bpe::DeviceGuard guard(trie->device);
    cudaStream_t s = (cudaStream_t)cuda_stream;
    if (n_docs == 0) {
        if (d_id_off_out && cudaMemsetAsync(d_id_off_out, 0, 8, s) != cudaSuccess) return BPE_ERR_CUDA;
        return cudaStreamSynchronize(s) == cudaSuccess ? BPE_OK : BPE_ERR_CUDA;
    }
    return bpe::noalloc_body(trie, d_bytes, d_doc_off, n_docs, d_ids_out, ids_capacity, d_id_off_out, n_ids, s);
}
