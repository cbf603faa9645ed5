// unigram.cu -- Unigram (Viterbi) encoding over the double-array trie
// ([UNIGRAM] "Unigram tokenization": best[j] = max over tokens t = x[i..j) of
// best[i] + score(t), continuation bytes skipped, <unk> where nothing
// matches, a backtrack from the end; the token id and score live with the
// trie node, [UNIGRAM] "Baseline" and "Bitmap and inline packing").
//
// The recurrence is sequential along a document; the GPU splits every
// document into chunks of C bytes and makes the sequential result exact by
// speculation and repair.  Scores are summed in fixed point, so sums are
// associative and a path's decisions do not depend on the constant its
// values start from.
//
//   k_uni_index    first chunk of every document, longest document
//   k_uni_fwd_warp one warp per chunk runs the recurrence from the first
//                  character boundary G bytes before its chunk (value 0
//                  there, nothing reachable before) through its chunk: lanes
//                  walk the trie from 32 positions at once into shared
//                  memory, then relax them in order with the window of values
//                  in registers (int32, relative to the window's best).  It
//                  stores the back pointer of every position: the chunk's in
//                  the output array, the guard's in a private record with the
//                  guard positions whose edges reach the chunk ("crossing").
//                  (k_uni_fwd: the same with one thread per chunk and a
//                  64-bit ring, for spans over 63 bytes or wide scores.)
//   k_uni_fwd_wide the chunks whose 32-bit window spread (values more than
//                  2^30 units apart: many short tokens under scores of a fine
//                  unit) run again, a warp each, with 64-bit values.
//   k_uni_check    the guard ran from a wrong start value, but if the chains
//                  of the reachable crossing positions step like the true
//                  chains (the previous chunk's back pointers) until they
//                  meet at one position the true recurrence reaches, their
//                  values are the true ones plus one constant -- and so are
//                  the chunk's.  A chunk for which that fails is flagged.
//   k_uni_fix_coop one CTA per flagged chunk re-runs it from its
//                  predecessor's state (right when the predecessor is) and
//                  notes whether the next chunk then passes its check; eight
//                  warps walk the trie for eight batches at once while a
//                  ninth runs the recurrence.  (k_uni_fix_a: the same with
//                  one warp per chunk, when more chunks are flagged than
//                  the cooperative kernel has CTAs.)
//   k_uni_frepair_warp  one warp per document keeps those results where they
//                  hold and re-runs chains of chunks where they do not.
//   k_uni_bspec    each thread backtracks speculatively from a reachable
//                  position past its chunk's end; back-pointer chains merge,
//                  so where the chain enters the chunk (sx) is usually where
//                  the true path does.  It counts the chunk's tokens and
//                  records where the chain leaves it (bot).
//   k_uni_bcheck, k_uni_bfix_a, k_uni_brepair  the true sx of a chunk is the
//                  next chunk's bot (the document end for the last chunk):
//                  chunks where they differ are walked again, in parallel
//                  where the next chunk is right, right to left otherwise.
//   k_uni_emit     exclusive scan of the counts (decoupled look-back) and a
//                  walk of every chunk from its true sx that writes its ids;
//   k_uni_ids      one thread per id finds the ids the warp kernels left to
//                  the token's bytes.
//   k_uni_docoff   per-document id offsets.
//
// A back pointer is (length << 24) | id, with id 0xFFFFFF for <unk> and
// kNoTid where the id is found from the token's bytes; 0 marks an
// unreachable position and kRoot the start of a speculative run.
#include <algorithm>
#include <cmath>
#include <vector>

#include "device.cuh"
#include "internal.h"
#include "trie.h"

struct bpe_unigram {
    bpe_ctx *ctx = nullptr;
    const bpe_trie *trie = nullptr;
    int device = 0;
    int32_t unk_id = 0;
    long long unk = 0;          // unk_score in fixed-point units
    long long max_abs = 0;      // largest |score| in units (over tokens and unk)
    int q = 0;                  // units are 2^-q
    uint32_t span = 0;          // E: longest edge (token or <unk>) the kernels take
    void *d_leaf = nullptr;     // per trie slot: {score units, token id}
    void *d_fslot = nullptr;    // per trie slot: {check, base|TERM, score units (int32), token id};
                                // only when every |score| < 2^29 units (the warp kernels need it)
};

namespace bpe {
namespace {

constexpr int kUniThreads = 128;
constexpr uint32_t kRoot = 0x00FFFFFFu;    // speculative start (length 0 never occurs otherwise)
constexpr uint32_t kUnkTid = 0x00FFFFFFu;
constexpr uint32_t kNoTid = 0x00FFFFFEu;     // a token whose id the emit pass looks up from its bytes
constexpr long long kNeg = -0x7FFFFFFFFFFFFFFFll - 1;   // -inf
constexpr uint32_t kUniDefaultChunk = 768;   // measured on the batch workload: 512 3.90 ms, 768 3.69, 1024 3.99, 2048 4.73
constexpr unsigned kUniSpinLimit = 1u << 22;
enum : uint32_t { UERR_SPAN = 8u, UERR_OOB = 4u, UERR_TIMEOUT = 2u, UERR_CONT_START = 16u };

struct __align__(16) Leaf {
    long long score;
    int32_t tid;
    int32_t pad;
};

struct UniState {
    unsigned long long n_chunks;
    unsigned long long total;
    unsigned long long max_doc;
    unsigned long long span;      // doc_off[n_docs] - doc_off[0]
    unsigned long long text_lo;   // doc_off[0]
    uint32_t err;
    uint32_t any_fflag, any_bflag;
    uint32_t ticket;
    uint32_t bad_doc;
    uint32_t fwd_repairs, bwd_repairs;   // chunks re-run by the repair passes
    uint32_t flist_len;
    uint32_t wlist_len;   // chunks whose 32-bit window spread, for the wide re-run
};

struct UniParams {
    const uint8_t *bytes;
    const uint64_t *doc_off;
    uint32_t n_docs;
    uint32_t chunk;     // C
    uint32_t guard;     // G: guard bytes before a chunk (> E, <= 256, a multiple of 32)
    uint32_t grec;      // words per chunk of the guard record: G back pointers, G/32 crossing bits
    uint32_t E;         // longest edge
    uint32_t ahead;     // H: backtrack start past the chunk end
    const unsigned long long *chunk_start;   // n_docs + 1
    const int2 *slot;
    const int4 *root;
    const Leaf *leaf;
    const int4 *fslot;  // the slots with their token's score and id (warp kernels)
    long long unk;
    int32_t unk_id;
    unsigned long long stall_tile;   // testing: this emit tile never publishes (~0: none)
    unsigned long long text_lo;   // doc_off[0]
    unsigned long long text_end;  // doc_off[n_docs]
    uint32_t *back;     // per position (offset from text_lo), span + 1 words
    uint32_t *tstart;   // per id: its token's start for k_uni_ids (null: emit looks ids up itself)
    unsigned long long tstart_n;   // its entries
    uint32_t *gback;    // per chunk grec words: the guard's back pointers and crossing bits
    uint32_t *fflag, *bflag;   // bitmaps over chunks
    uint32_t *okn;             // bitmap: a flagged chunk's parallel repair was valid for its successor too
    uint32_t *okp;             // bitmap: a flagged chunk's parallel re-walk was valid for its predecessor too
    uint32_t *flist;           // flagged chunks (unordered; flist_cap entries kept)
    uint32_t flist_cap;
    uint32_t *wlist;           // chunks to run again in 64 bits (unordered; flist_cap entries kept)
    uint32_t *sx, *bot, *count;   // per chunk (sx, bot relative to the chunk start)
    unsigned long long *prefix;
    unsigned long long *status;
    int32_t *ids;
    unsigned long long cap;
    unsigned long long *id_off;
    UniState *st;
};

__device__ __forceinline__ bool is_cont(uint32_t b) { return (b & 0xC0u) == 0x80u; }
__device__ __forceinline__ uint32_t byte_at(const UniParams &P, uint64_t p) { return __ldg(P.bytes + p); }
__device__ __forceinline__ uint32_t &back_at(const UniParams &P, uint64_t p) {
    return P.back[p - P.text_lo];
}

// Root LUT with the depth-1 nodes that exist: entry x < 0 when byte c has no
// node below the root (the root is slot 0, its children's check is 0).
__device__ __forceinline__ void load_uni_lut(const UniParams &P, int4 *lut) {
    for (int c = threadIdx.x; c < 256; c += blockDim.x) {
        int4 r = P.root[c];
        if (__ldg(&P.slot[r.x].x) != 0) r.x = -1;
        lut[c] = r;
    }
}

// The same with each depth-1 node's score (int32 units) and token id:
// {slot or -1, base|TERM, score, tid}.
__device__ __forceinline__ void load_fat_lut(const UniParams &P, int4 *lut) {
    for (int c = threadIdx.x; c < 256; c += blockDim.x) {
        const int32_t x = P.root[c].x;
        const int4 f = P.fslot[x];
        lut[c] = make_int4(f.x == 0 ? x : -1, f.y, f.z, f.w);
    }
}

__device__ __forceinline__ uint32_t doc_of_chunk(const UniParams &P, unsigned long long k) {
    uint32_t lo = 0, hi = P.n_docs;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (P.chunk_start[mid] <= k) lo = mid; else hi = mid;
    }
    return lo;
}

struct UGeo {
    uint64_t ds, de, cs, ce;
    bool first, last;   // first / last chunk of its document
};

__device__ __forceinline__ UGeo uni_geo(const UniParams &P, unsigned long long k) {
    const uint32_t d = doc_of_chunk(P, k);
    UGeo g;
    g.ds = P.doc_off[d];
    g.de = P.doc_off[d + 1];
    const uint64_t j = k - P.chunk_start[d];
    g.cs = g.ds + j * P.chunk;
    g.ce = min(g.cs + P.chunk, g.de);
    g.first = j == 0;
    g.last = g.ce == g.de;
    return g;
}

// One run of the recurrence over positions [from, to) of a document ending
// at de, on a ring of R values and back pointers.  The caller has set the
// ring for the positions it starts from.  Position i is final when the run
// reaches it: its back pointer goes to sink(i, bp).  A reachable character
// start then relaxes every token that ends at a character boundary (trie
// walk) or, when there is none, the <unk> edge to the next boundary; every
// relaxed edge i -> j is reported to edge(i, j).  Back pointers carry the
// token id (kIds) or kNoTid, as the warp kernels write them.  Each loop iteration takes
// one trie step on every lane (finalising a position first where a walk has
// ended), so the lanes of a warp do not wait for each other's long walks.  A
// run of E continuation bytes could only be crossed by a longer edge: it
// raises UERR_SPAN (whichever run sees its last E bytes).
template <int R, bool kIds = true, typename Sink, typename Edge>
__device__ __forceinline__ void uni_run(const UniParams &P, const int4 *lut, long long *best, uint32_t *bk,
                                        uint64_t from, uint64_t to, uint64_t de, Sink sink, Edge edge) {
    uint32_t cont_run = 0;
    uint64_t i = from;
    int32_t node = -1;   // < 0: no walk in progress at i
    uint32_t y = 0, len = 0;
    long long b = 0;
    bool matched = false;
    auto relax = [&](uint64_t j, long long cand, uint32_t bp) {
        const uint32_t sj = (uint32_t)j & (R - 1);
        if (cand > best[sj]) {
            best[sj] = cand;
            bk[sj] = bp;
        }
        edge(i, j);
    };
    auto unk_edge = [&]() {
        uint64_t j = i + 1;
        while (j < de && is_cont(byte_at(P, j)) && j - i <= P.E) ++j;
        if (j - i > P.E) {
            atomicOr(&P.st->err, UERR_SPAN);
            j = i + P.E;   // keep the ring consistent; the call fails
        }
        relax(j, b + P.unk, ((uint32_t)(j - i) << 24) | kUnkTid);
    };
    for (;;) {
        if (node < 0) {
            if (i >= to) break;
            const uint32_t si = (uint32_t)i & (R - 1);
            b = best[si];
            const uint32_t bp = bk[si];
            best[si] = kNeg;
            bk[si] = 0;
            sink(i, b == kNeg ? 0u : bp);
            const uint32_t c0 = byte_at(P, i);
            cont_run = is_cont(c0) ? cont_run + 1 : 0u;
            if (cont_run >= P.E) atomicOr(&P.st->err, UERR_SPAN);
            if (b == kNeg || is_cont(c0)) {
                ++i;
                continue;
            }
            const int4 r = lut[c0];
            matched = false;
            if (r.x < 0) {
                unk_edge();
                ++i;
                continue;
            }
            node = r.x;
            y = (uint32_t)r.y;
            len = 1;
        }
        // the node for x[i .. i+len): its token, then one step down
        const uint64_t j = i + len;
        const uint32_t nb = j < de ? byte_at(P, j) : 0u;
        if ((y & kTermBit) && (j == de || !is_cont(nb))) {
            const Leaf lf = P.leaf[node];
            relax(j, b + lf.score, (len << 24) | (kIds ? (uint32_t)lf.tid : kNoTid));
            matched = true;
        }
        const uint32_t base = y & ~kTermBit;
        bool down = j < de && base != 0 && len < P.E;
        if (down) {
            const int32_t t = (int32_t)(base + nb);
            const int2 v = __ldg(P.slot + t);
            down = v.x == node;
            if (down) {
                node = t;
                y = (uint32_t)v.y;
                ++len;
            }
        }
        if (!down) {
            if (!matched) unk_edge();
            node = -1;
            ++i;
        }
    }
}

template <int R>
__device__ __forceinline__ void ring_clear(long long *best, uint32_t *bk) {
#pragma unroll 8
    for (int s = 0; s < R; s++) {
        best[s] = kNeg;
        bk[s] = 0;
    }
}

// First character boundary at or after p (p < de), or de.
__device__ __forceinline__ uint64_t next_boundary(const UniParams &P, uint64_t p, uint64_t de) {
    while (p < de && is_cont(byte_at(P, p))) ++p;
    return p;
}

// ---------------------------------------------------------- chunk index ---

// chunk_start (exclusive scan of ceil(len / C) per document), the longest
// document, the chunk count and the text span.
__global__ void __launch_bounds__(1024) k_uni_index(UniParams P, unsigned long long *chunk_start) {
    __shared__ unsigned long long s_w[32];
    __shared__ unsigned long long s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    unsigned long long longest = 0;
    for (uint64_t base = 0; base < P.n_docs; base += 1024) {
        const uint64_t d = base + tid;
        unsigned long long v = 0;
        if (d < P.n_docs) {
            const uint64_t a = P.doc_off[d], b = P.doc_off[d + 1];
            if (b < a) {
                atomicOr(&P.st->err, UERR_OOB);
                P.st->bad_doc = (uint32_t)d;
            } else {
                v = (b - a + P.chunk - 1) / P.chunk;
                longest = max(longest, (unsigned long long)(b - a));
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
    longest = warp_max_u64(longest);
    if (lane == 0 && longest) atomicMax(&P.st->max_doc, longest);
    if (tid == 0) {
        chunk_start[P.n_docs] = s_carry;
        P.st->n_chunks = s_carry;
        P.st->span = P.doc_off[P.n_docs] - P.doc_off[0];
        P.st->text_lo = P.doc_off[0];
    }
}

// ------------------------------------------------------------- forward ---

// Where chunk k's run starts: the document start when the chunk lies within
// G bytes of it (then the run is exact), else cs - G.
__device__ __forceinline__ uint64_t run_from(const UniParams &P, const UGeo &g) {
    return (g.cs - g.ds <= P.guard) ? g.ds : g.cs - P.guard;
}

template <int R>
__device__ __forceinline__ uint64_t start_run(const UniParams &P, const UGeo &g, uint64_t from, long long *best,
                                              uint32_t *bk) {
    ring_clear<R>(best, bk);
    const uint64_t s0 = from == g.ds ? g.ds : next_boundary(P, from, g.de);
    best[(uint32_t)s0 & (R - 1)] = 0;
    bk[(uint32_t)s0 & (R - 1)] = kRoot;
    return s0;
}

// The last position of a document is final after the run reaches it.
template <int R>
__device__ __forceinline__ void finish_doc(const UniParams &P, const UGeo &g, const long long *best,
                                           const uint32_t *bk) {
    const uint32_t s = (uint32_t)g.de & (R - 1);
    back_at(P, g.de) = best[s] == kNeg ? 0u : bk[s];
}

template <int R>
__global__ void __launch_bounds__(kUniThreads) k_uni_fwd(UniParams P, unsigned long long n_chunks) {
    __shared__ int4 lut[256];
    load_uni_lut(P, lut);
    __syncthreads();
    const unsigned long long k = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n_chunks) return;
    const UGeo g = uni_geo(P, k);
    long long best[R];
    uint32_t bk[R];
    const uint64_t from = run_from(P, g);
    const uint64_t s0 = start_run<R>(P, g, from, best, bk);
    uint32_t *gb = P.gback + k * (unsigned long long)P.grec;
    uint32_t cross[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // guard positions with an edge reaching cs or beyond
    const bool exact = from == g.ds;
    if (s0 >= g.cs && !exact) atomicOr(&P.st->err, UERR_SPAN);   // a guard of continuation bytes only
    if (g.first && is_cont(byte_at(P, g.ds))) atomicOr(&P.st->err, UERR_CONT_START);
    uni_run<R>(
        P, lut, best, bk, from, g.ce, g.de,
        [&](uint64_t i, uint32_t bp) {
            if (i >= g.cs) {
                if (i != g.ds) back_at(P, i) = bp;
            } else if (!exact) {
                gb[i - from] = bp;
            }
        },
        [&](uint64_t i, uint64_t j) {
            if (i < g.cs && j >= g.cs && !exact) {
                const uint32_t o = (uint32_t)(i - from);
                cross[o >> 5] |= 1u << (o & 31);
            }
        });
    if (!exact)
        for (uint32_t w = 0; w < (P.guard >> 5); w++) gb[P.guard + w] = cross[w];
    if (g.last) finish_doc<R>(P, g, best, bk);
}

// Whether chunk k's guard run (its record gr: back pointers over [cs - G,
// cs), then the crossing bits) agrees with the true back pointers up to a
// constant at cs.  Only positions with an edge reaching cs or beyond
// (crossing) influence the chunk.  Every reachable crossing position's chain
// must step like the true chain until all chains meet at one position z the
// true recurrence reaches; then their values are the true ones plus one
// constant.  A position of the last E bytes the run did not reach must be
// unreachable in truth too (its edges were never explored).
__device__ bool guard_agrees(const UniParams &P, const uint32_t *gr, uint64_t cs) {
    const uint64_t from = cs - P.guard;
    uint32_t mk[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // marked offsets (G <= 256)
    int n = 0;
    for (uint32_t o = P.guard - P.E; o < P.guard; o++) {
        if (gr[o] == 0) {
            if (back_at(P, from + o) != 0) return false;
        } else if ((gr[P.guard + (o >> 5)] >> (o & 31)) & 1u) {
            mk[o >> 5] |= 1u << (o & 31);
            ++n;
        }
    }
    if (n == 0) return false;
    for (int o = (int)P.guard - 1; o >= 0; o--) {
        if (!((mk[o >> 5] >> (o & 31)) & 1u)) continue;
        if (n == 1) return back_at(P, from + o) != 0;   // z: reachable in truth
        mk[o >> 5] &= ~(1u << (o & 31));
        const uint32_t v = gr[o];
        if (v == kRoot || back_at(P, from + o) != v) return false;
        const int po = o - (int)(v >> 24);
        if (po < 0) return false;
        if ((mk[po >> 5] >> (po & 31)) & 1u) --n;
        else mk[po >> 5] |= 1u << (po & 31);
    }
    return false;
}

// Guard bytes before a chunk for spans <= 63 (64 leaves the back-pointer
// chains too little room to meet: most chunks then need a repair; 128 almost
// none).
constexpr uint32_t kGuard64 = 128;

constexpr int kFwdWarps = 8;                 // warps per CTA of the warp-per-chunk kernels
constexpr int kEdgeStride = 33;              // a lane's edge row: lengths 1..32, odd stride (banks)
constexpr int kLongRows = 16;                // rows for lengths 33..63, claimed per batch by the lanes that need one
// per warp: 32 rows, the long rows, the long-row counter, the staged text
constexpr size_t kWarpEdgeBytes = (32 * kEdgeStride + kLongRows * 32 + 4) * sizeof(int32_t) + 128;

constexpr int32_t kNeg32 = -0x7FFFFFFF - 1;   // unreachable (relative values)
constexpr int32_t kSpread = 1 << 30;          // relative values stay within +-kSpread (else the run is redone)
constexpr int kTextStage = 128;               // bytes of text a warp stages per batch (32 positions + 63 + 1)

// The recurrence's window for spans E <= 63, held by a warp in registers.
// Only values of positions at most 63 apart are ever compared, so they are
// kept as int32 relative to the window's best, rebased every batch: with
// |score| < 2^29 and every value within 2^30 of 0 no sum wraps, and a value
// beyond that reports a spread (the run is redone exactly).  Before source s
// of the batch at b0, lane t holds in A the position b0 + t if t >= s, else
// b0 + 32 + t -- the one its length o1 = (t - s - 1) mod 32 + 1 edge reaches --
// and in B the position 32 further on (lengths o1 + 32).  When lane s is the
// source its A is final and B moves into A.  With each value, the source of
// its best edge as an offset from base (bit 31: the edge is <unk>); the
// edge's length is the distance to it.
//
// WideRing holds the same window in 64 bits, not rebased: it is what a run
// takes when the 32-bit window spread (values of a window more than 2^30
// units apart: many short tokens under scores of a fine unit), and it never
// spreads (a document's sums stay far below 2^62 units).
template <typename V>
struct WarpRingT {
    V a, b;
    uint32_t sa, sb;
    uint64_t base, b0;
};
using WarpRing = WarpRingT<int32_t>;
using WideRing = WarpRingT<long long>;
constexpr long long kNeg64 = -0x7FFFFFFFFFFFFFFFll - 1;   // unreachable (wide values)
template <typename V> __device__ __forceinline__ V ring_neg();
template <> __device__ __forceinline__ int32_t ring_neg<int32_t>() { return kNeg32; }
template <> __device__ __forceinline__ long long ring_neg<long long>() { return kNeg64; }

template <typename V>
__device__ __forceinline__ void ring_start(WarpRingT<V> &R, uint64_t base, uint64_t s0, int lane) {
    R.a = R.b = ring_neg<V>();
    R.sa = R.sb = 0;
    R.base = R.b0 = base;
    const uint64_t o = s0 - base;
    if (o < 64 && lane == (int)(o & 31)) {   // the start is its own source: length 0
        if (o >> 5) { R.b = 0; R.sb = (uint32_t)o; } else { R.a = 0; R.sa = (uint32_t)o; }
    }
}

// Back pointer of position pos given its value and source.
template <typename V>
__device__ __forceinline__ uint32_t ring_bp(const WarpRingT<V> &R, uint64_t pos, V v, uint32_t src) {
    if (v == ring_neg<V>()) return 0u;
    const uint32_t len = ((uint32_t)(pos - R.base) - src) & 0x7FFFFFFFu;
    return len == 0 ? kRoot : (len << 24) | ((src >> 31) ? kUnkTid : kNoTid);
}

// After a run: back pointer of the first position at or after its end that
// this lane holds (the document end, when the run ended there).
template <typename V>
__device__ __forceinline__ uint32_t ring_final(const WarpRingT<V> &R, uint64_t pos) {
    return ring_bp(R, pos, R.a, R.sa);
}

// One warp's shared memory: its edge rows (row l: lane l's position, entry
// len - 1 = the score, int32 units, of its edge of length len <= 32), a few
// rows for lengths 33..63 (entry len - 33) claimed by the lanes that have
// such an edge, and its text.
struct EdgeBuf {
    int32_t *score;
    int32_t *lrow;
    int *lcount;
    uint8_t *text;
    __device__ EdgeBuf(int32_t *base)
        : score(base), lrow(base + 32 * kEdgeStride), lcount((int *)(base + 32 * kEdgeStride + kLongRows * 32)),
          text((uint8_t *)(base + 32 * kEdgeStride + kLongRows * 32 + 4)) {}
};

// What one lane's walk of a batch leaves for the recurrence: its edge
// lengths as masks (1..32, 33..63), its long row, whether its only edge is
// <unk>, whether an edge reaches cs, and whether a long row was missing.
struct WalkOut {
    uint32_t X, Y;
    int lr;
    bool unk, crossing, norow;
};

// Walk: every lane walks the trie from its position b0 + lane (reachable or
// not) over the batch's text staged in shared memory, and records its edges'
// scores by length in its row (a long row for lengths over 32).
__device__ __forceinline__ WalkOut walk_batch(const UniParams &P, const int4 *lut, const EdgeBuf &eb, uint64_t b0,
                                              uint64_t to, uint64_t de, uint64_t cs) {
    const int lane = threadIdx.x & 31;
    int32_t *row = eb.score + lane * kEdgeStride;
    // stage text [b0, b0 + 128) (what lies before the text's end)
#pragma unroll
    for (int i = 0; i < kTextStage / 32; i++) {
        const uint64_t p = b0 + i * 32 + lane;
        eb.text[i * 32 + lane] = p < P.text_end ? byte_at(P, p) : 0u;
    }
    if (lane == 0) *eb.lcount = 0;
    __syncwarp();
    WalkOut w{0u, 0u, -1, false, false, false};
    const uint64_t q = b0 + lane;
    unsigned long long M = 0;   // bit len: an edge of that length
    if (q < to) {
        const uint32_t dlen = de - q < 64 ? (uint32_t)(de - q) : 64u;   // bytes to the document end (capped)
        const uint32_t lim = min(dlen, P.E);
        const uint32_t csr = q >= cs ? 0u : cs - q < 64 ? (uint32_t)(cs - q) : 64u;
        const uint8_t *tx = eb.text + lane;
        const uint32_t c0 = tx[0];
        if (!is_cont(c0)) {
            const int4 r = lut[c0];
            if (r.x >= 0) {
                int32_t node = r.x;
                uint32_t y = (uint32_t)r.y;
                int32_t sc = r.z;
                uint32_t len = 1;
                for (;;) {
                    const uint32_t nb = len < dlen ? tx[len] : 0u;
                    if ((y & kTermBit) && (len == dlen || !is_cont(nb))) {
                        if (len <= 32) {
                            row[len - 1] = sc;
                        } else {
                            if (w.lr < 0) w.lr = atomicAdd(eb.lcount, 1);
                            if (w.lr < kLongRows) eb.lrow[w.lr * 32 + (len - 33)] = sc;
                            else w.norow = true;   // no long row left: the run is redone exactly
                        }
                        M |= 1ull << len;
                        w.crossing |= len >= csr;
                    }
                    const uint32_t base = y & ~kTermBit;
                    if (len >= lim || base == 0) break;
                    const int32_t t = (int32_t)(base + nb);
                    const int4 v = __ldg(P.fslot + t);
                    if (v.x != node) break;
                    node = t;
                    y = (uint32_t)v.y;
                    sc = v.z;
                    ++len;
                }
            }
            if (M == 0) {   // <unk> to the next character boundary
                uint32_t len = 1;
                while (len < dlen && len <= P.E && is_cont(len < kTextStage - lane ? tx[len] : byte_at(P, q + len)))
                    ++len;
                if (len > P.E) {
                    atomicOr(&P.st->err, UERR_SPAN);
                    len = P.E;
                }
                if (len <= 32) {
                    row[len - 1] = (int32_t)P.unk;
                } else {
                    w.lr = atomicAdd(eb.lcount, 1);
                    if (w.lr < kLongRows) eb.lrow[w.lr * 32 + (len - 33)] = (int32_t)P.unk;
                    else w.norow = true;
                }
                M = 1ull << len;
                w.unk = true;
                w.crossing = len >= csr;
            }
        }
    }
    w.X = (uint32_t)(M >> 1);
    w.Y = (uint32_t)(M >> 33);
    return w;
}

// Recurrence over the batch at b0 (= R.b0) from the walk's rows in eb and
// this lane's walk results: the batch's positions in order; source s's value
// comes from lane s, and every lane relaxes its o1 and o1 + 32 targets (a bit
// of s's masks rotated by s + 1) from shared memory and shuffles only.
// sink(q, bp) receives every final position.  Returns whether this lane saw
// a value beyond kSpread (never in a wide ring).
template <typename V, typename Sink>
__device__ __forceinline__ bool dp_batch(const EdgeBuf &eb, WarpRingT<V> &R, uint64_t b0, uint64_t to,
                                         const WalkOut &w, Sink sink) {
    constexpr bool kNarrow = sizeof(V) == 4;
    const V neg = ring_neg<V>();
    const int lane = threadIdx.x & 31;
    const uint32_t mybit = 1u << lane;
    const uint64_t q = b0 + lane;
    bool spread = false;
    const uint32_t xrot = __funnelshift_l(w.X, w.X, lane + 1), yrot = __funnelshift_l(w.Y, w.Y, lane + 1);
    const uint32_t mycode = ((uint32_t)(q - R.base) & 0x7FFFFFFFu) | ((uint32_t)w.unk << 31);
    const int lr = w.lr;
    if constexpr (kNarrow) {   // rebase: the window's best reachable value becomes 0
        const int32_t mx = __reduce_max_sync(kFull, max((int32_t)R.a, (int32_t)R.b));
        if (mx != kNeg32) {
            if (R.a != kNeg32) {
                const long long v = (long long)R.a - mx;
                spread |= v < -kSpread;
                R.a = (V)max(v, (long long)-kSpread);
            }
            if (R.b != kNeg32) {
                const long long v = (long long)R.b - mx;
                spread |= v < -kSpread;
                R.b = (V)max(v, (long long)-kSpread);
            }
        }
    }
    __syncwarp();
    V fv = neg;
    uint32_t fs = 0;
    const uint32_t nsrc = (uint32_t)(to - b0 < 32 ? to - b0 : 32);
    const bool anylong = __any_sync(kFull, w.Y != 0u);   // some edge over 32 bytes (rare)
    // source s of the batch; o1 = this lane's length to reach its A position
    auto source = [&](uint32_t s, uint32_t o1) {
        const V b = __shfl_sync(kFull, R.a, s);
        const uint32_t xr = __shfl_sync(kFull, xrot, s);
        const uint32_t code = __shfl_sync(kFull, mycode, s);
        const uint32_t yr = anylong ? __shfl_sync(kFull, yrot, s) : 0u;
        const int slr = yr ? __shfl_sync(kFull, lr, s) : 0;   // s's long row (lengths 33..63)
        if (lane == (int)s) {   // position b0 + s is final; the next window position moves in
            fv = R.a;
            fs = R.sa;
            R.a = R.b;
            R.sa = R.sb;
            R.b = neg;
        }
        if (b == neg) return;
        if (xr & mybit) {
            const V cand = b + (V)eb.score[s * kEdgeStride + (o1 - 1)];
            if (cand > R.a) { R.a = cand; R.sa = code; }
        }
        if ((yr & mybit) && slr < kLongRows) {   // length o1 + 32
            const V cand = b + (V)eb.lrow[slr * 32 + (o1 - 1)];
            if (cand > R.b) { R.b = cand; R.sb = code; }
        }
    };
    const uint32_t o10 = lane == 0 ? 32u : (uint32_t)lane;   // this lane's length o1 from source 0
    if (nsrc == 32) {
#pragma unroll
        for (uint32_t s = 0; s < 32; s++) source(s, ((o10 - 1u - s) & 31u) + 1u);
    } else {
        for (uint32_t s = 0; s < nsrc; s++) source(s, ((o10 - 1u - s) & 31u) + 1u);
    }
    if constexpr (kNarrow) spread |= fv != neg && (fv < -kSpread || fv > kSpread);   // every source value stayed in range
    __syncwarp();
    if (q < to) sink(q, ring_bp(R, q, fv, fs));
    R.b0 = b0 + 32;
    return spread;
}

// The recurrence over positions [from, to) of a document ending at de, by one
// warp (from = R.b0), 32 positions at a time, on the slots that carry their
// token's score (fslot; lut: the depth-1 nodes): a walk, then the
// recurrence, per batch.  cross(m, bits) receives, per batch m, which
// positions have an edge reaching cs or beyond.  A back pointer holds the
// length and kNoTid (the emit pass finds the id from the token's bytes) or
// kUnkTid.  Returns 0 when the run is complete, else kRunLongRows when a
// long row was missing, kRunSpread when the values spread beyond kSpread
// (both: the run is incomplete).
constexpr uint32_t kRunLongRows = 1u, kRunSpread = 2u;
template <typename V, typename Sink, typename Cross>
__device__ uint32_t warp_dp(const UniParams &P, const int4 *lut, const EdgeBuf &eb, WarpRingT<V> &R, uint64_t from,
                            uint64_t to, uint64_t de, uint64_t cs, Sink sink, Cross cross) {
    const int lane = threadIdx.x & 31;
    bool rows = false, spread = false;
    for (uint64_t b0 = from; b0 < to; b0 += 32) {
        const WalkOut w = walk_batch(P, lut, eb, b0, to, de, cs);
        cross((uint32_t)((b0 - from) >> 5), __ballot_sync(kFull, w.crossing && b0 + lane < cs));
        rows |= w.norow;
        spread |= dp_batch(eb, R, b0, to, w, sink);
    }
    return (__any_sync(kFull, rows) ? kRunLongRows : 0u) | (__any_sync(kFull, spread) ? kRunSpread : 0u);
}

// The speculative forward run of chunk k by one warp (spans E <= 63):
// k_uni_fwd's work.  Returns warp_dp's code (0: complete).
template <typename V>
__device__ __forceinline__ uint32_t fwd_chunk(const UniParams &P, const int4 *lut, const EdgeBuf &eb,
                                              unsigned long long k) {
    const int lane = threadIdx.x & 31;
    const UGeo g = uni_geo(P, k);
    const uint64_t from = run_from(P, g);
    const bool exact = from == g.ds;
    if (g.first && lane == 0 && is_cont(byte_at(P, g.ds))) atomicOr(&P.st->err, UERR_CONT_START);
    const uint64_t s0 = exact ? g.ds : next_boundary(P, from, g.de);
    if (!exact && (s0 >= g.cs || s0 - from >= 64) && lane == 0) atomicOr(&P.st->err, UERR_SPAN);
    WarpRingT<V> R;
    ring_start(R, from, s0, lane);
    uint32_t *gb = P.gback + k * (unsigned long long)P.grec;
    const uint32_t code = warp_dp(
        P, lut, eb, R, from, g.ce, g.de, g.cs,
        [&](uint64_t q, uint32_t bp) {
            if (q >= g.cs) {
                if (q != g.ds) back_at(P, q) = bp;
            } else if (!exact) {
                gb[q - from] = bp;
            }
        },
        [&](uint32_t m, unsigned bits) {
            if (!exact && m < (P.guard >> 5) && lane == 0) gb[P.guard + m] = bits;
        });
    if (g.last && lane == (int)((g.de - from) & 31)) back_at(P, g.de) = ring_final(R, g.de);
    return code;
}

// A chunk whose run is incomplete for want of a long row: flagged, so the
// repair passes run it again.
__device__ __forceinline__ void flag_chunk(const UniParams &P, unsigned long long k) {
    atomicOr(P.fflag + (k >> 5), 1u << (k & 31));
    P.st->any_fflag = 1u;
    const uint32_t i = atomicAdd(&P.st->flist_len, 1u);
    if (i < P.flist_cap) P.flist[i] = (uint32_t)k;
}

// Warp-per-chunk speculative forward run in 32-bit windows; a chunk whose
// window spread is listed for k_uni_fwd_wide.
__global__ void __launch_bounds__(kFwdWarps * 32, 4) k_uni_fwd_warp(UniParams P, unsigned long long n_chunks) {
    __shared__ int4 lut[256];
    extern __shared__ int32_t s_rows[];   // kFwdWarps edge tables
    load_fat_lut(P, lut);
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned long long k = (unsigned long long)blockIdx.x * kFwdWarps + w;
    if (k >= n_chunks) return;
    const EdgeBuf eb(s_rows + w * (kWarpEdgeBytes / 4));
    const uint32_t code = fwd_chunk<int32_t>(P, lut, eb, k);
    if (lane == 0) {
        if (code & kRunLongRows) {
            flag_chunk(P, k);
        } else if (code & kRunSpread) {
            const uint32_t i = atomicAdd(&P.st->wlist_len, 1u);
            if (i < P.flist_cap) P.wlist[i] = (uint32_t)k;
            else flag_chunk(P, k);
        }
    }
}

// The listed chunks' forward runs again, in 64-bit windows (a warp each, all
// in parallel): their results replace the spread ones entirely.
__global__ void __launch_bounds__(kFwdWarps * 32) k_uni_fwd_wide(UniParams P) {
    __shared__ int4 lut[256];
    extern __shared__ int32_t s_rows[];
    const uint32_t n = min(P.st->wlist_len, P.flist_cap);
    if (n == 0) return;
    load_fat_lut(P, lut);
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const EdgeBuf eb(s_rows + w * (kWarpEdgeBytes / 4));
    for (uint32_t i = blockIdx.x * kFwdWarps + w; i < n; i += gridDim.x * kFwdWarps) {
        const unsigned long long k = P.wlist[i];
        const uint32_t code = fwd_chunk<long long>(P, lut, eb, k);
        if (code && lane == 0) flag_chunk(P, k);
    }
}

__global__ void __launch_bounds__(256) k_uni_check(UniParams P, unsigned long long n_chunks) {
    const unsigned long long k = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n_chunks) return;
    const UGeo g = uni_geo(P, k);
    if (g.cs - g.ds <= P.guard) return;   // exact run
    if (!guard_agrees(P, P.gback + k * (unsigned long long)P.grec, g.cs)) {
        const uint32_t old = atomicOr(P.fflag + (k >> 5), 1u << (k & 31));
        P.st->any_fflag = 1u;
        if (!((old >> (k & 31)) & 1u)) {   // not listed yet (an overflowed run lists itself)
            const uint32_t i = atomicAdd(&P.st->flist_len, 1u);
            if (i < P.flist_cap) P.flist[i] = (uint32_t)k;
        }
    }
}

__device__ __forceinline__ bool flag_bit(const uint32_t *flag, unsigned long long k) {
    return (flag[k >> 5] >> (k & 31)) & 1u;
}

// Next set bit of a chunk bitmap in [k, end) (end if none); one warp scans
// 32 words per step, all lanes get the answer.
__device__ __forceinline__ unsigned long long warp_next_flag(const uint32_t *flag, unsigned long long k,
                                                             unsigned long long end, int lane) {
    while (k < end) {
        const unsigned long long w0 = k >> 5;
        const unsigned long long w = w0 + lane;
        uint32_t bits = (w << 5) < end ? flag[w] : 0u;
        if (lane == 0) bits &= ~0u << (k & 31);
        if (((w + 1) << 5) > end) bits &= (end & 31) ? ((1u << (end & 31)) - 1u) : ~0u;
        const unsigned m = __ballot_sync(kFull, bits != 0);
        if (m) {
            const int l = __ffs(m) - 1;
            const uint32_t b = __shfl_sync(kFull, bits, l);
            return ((w0 + l) << 5) + (__ffs(b) - 1);
        }
        k = (w0 + 32) << 5;
    }
    return end;
}

// Previous set bit of a chunk bitmap in [begin, k] (or ~0 if none).
__device__ __forceinline__ unsigned long long warp_prev_flag(const uint32_t *flag, long long k, long long begin,
                                                             int lane) {
    while (k >= begin) {
        const long long w0 = k >> 5;
        const long long w = w0 - lane;
        uint32_t bits = (w >= 0 && ((w << 5) + 31) >= begin) ? flag[w] : 0u;
        if (lane == 0 && (k & 31) != 31) bits &= (2u << (k & 31)) - 1u;
        if (w >= 0 && (w << 5) < begin) bits &= ~0u << (begin & 31);
        const unsigned m = __ballot_sync(kFull, bits != 0);
        if (m) {
            const int l = __ffs(m) - 1;
            const uint32_t b = __shfl_sync(kFull, bits, l);
            return (unsigned long long)(((w0 - l) << 5) + (31 - __clz(b)));
        }
        k = ((w0 - 32) << 5) + 31;
    }
    return ~0ull;
}

// One warp per document; lane 0 does the runs.  For each flagged chunk f (in
// order) the recurrence is re-run from chunk f-1's start -- f-1 is correct:
// it passed its check, or the previous chain ended on it -- through chunk f
// and on through the chunks after it until one passes its check against the
// repaired back pointers (or the document ends).
template <int R>
__global__ void __launch_bounds__(128) k_uni_frepair(UniParams P) {
    __shared__ int4 lut[256];
    load_uni_lut(P, lut);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const uint32_t d = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (d >= P.n_docs) return;
    const unsigned long long c0 = P.chunk_start[d], c1 = P.chunk_start[d + 1];
    unsigned long long f = warp_next_flag(P.fflag, c0, c1, lane);
    uint32_t reruns = 0;
    while (f < c1) {
        unsigned long long m = f;
        if (lane == 0) {
            long long best[R];
            uint32_t bk[R];
            // the state at f's start: from f-1's run start, or exact from the
            // document start when f lies within G bytes of it
            const UGeo gf = uni_geo(P, f);
            const UGeo gp = gf.cs - gf.ds <= P.guard ? gf : uni_geo(P, f - 1);
            const uint64_t from = run_from(P, gp);
            start_run<R>(P, gp, from, best, bk);
            uni_run<R>(P, lut, best, bk, from, gf.cs, gf.de, [](uint64_t, uint32_t) {}, [](uint64_t, uint64_t) {});
            for (;;) {
                const UGeo g = uni_geo(P, m);
                uni_run<R>(
                    P, lut, best, bk, g.cs, g.ce, g.de, [&](uint64_t i, uint32_t bp) {
                        if (i != g.ds) back_at(P, i) = bp;
                    },
                    [](uint64_t, uint64_t) {});
                ++reruns;
                ++m;
                if (g.last) {
                    finish_doc<R>(P, g, best, bk);
                    break;
                }
                if (g.ce - g.ds <= P.guard || guard_agrees(P, P.gback + m * (unsigned long long)P.grec, g.ce))
                    break;
            }
        }
        m = __shfl_sync(kFull, m, 0);
        f = warp_next_flag(P.fflag, m + 1, c1, lane);   // chunk m is correct now
    }
    if (lane == 0 && reruns) atomicAdd(&P.st->fwd_repairs, reruns);
}

// Where the true back-pointer chains of every reachable crossing position
// of chunk f (its guard record gr: crossing bits; the chunk before it right)
// meet, within the G bytes before cs; ~0 if they do not.  Every such
// position's best path passes through it, so the recurrence started there
// (value 0, nothing else reachable) gives those positions their true values
// plus one constant -- and the chunk its true back pointers.
__device__ uint64_t true_meet(const UniParams &P, const uint32_t *gr, uint64_t cs) {
    const uint64_t from = cs - P.guard;
    uint32_t mk[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int n = 0;
    for (uint32_t o = P.guard - P.E; o < P.guard; o++)
        if (((gr[P.guard + (o >> 5)] >> (o & 31)) & 1u) && back_at(P, from + o) != 0) {
            mk[o >> 5] |= 1u << (o & 31);
            ++n;
        }
    if (n == 0) return ~0ull;
    for (int o = (int)P.guard - 1; o >= 0; o--) {
        if (!((mk[o >> 5] >> (o & 31)) & 1u)) continue;
        if (n == 1) return from + (uint64_t)o;
        mk[o >> 5] &= ~(1u << (o & 31));
        const uint32_t v = back_at(P, from + o);
        const int po = o - (int)(v >> 24);
        if ((v >> 24) == 0 || po < 0) return ~0ull;
        if ((mk[po >> 5] >> (po & 31)) & 1u) --n;
        else mk[po >> 5] |= 1u << (po & 31);
    }
    return ~0ull;
}

// Where a re-run of flagged chunk f starts, the chunk before it being right:
// where the true chains of f's crossing positions meet when they do (a few
// tokens back; the ring's base then lies a whole number of batches before
// cs), else f-1's run start (or the document start when f lies within G
// bytes of it).  Returns the ring's base; *s0 = the start position.
__device__ uint64_t repair_from(const UniParams &P, const UGeo &gf, unsigned long long f, uint64_t *s0) {
    if (gf.cs - gf.ds > P.guard) {
        const uint64_t z = true_meet(P, P.gback + f * (unsigned long long)P.grec, gf.cs);
        if (z != ~0ull) {
            *s0 = z;
            return gf.cs - ((gf.cs - z + 31) & ~31ull);
        }
    }
    const UGeo gp = gf.cs - gf.ds <= P.guard ? gf : uni_geo(P, f - 1);
    const uint64_t from = run_from(P, gp);
    *s0 = from == gp.ds ? gp.ds : next_boundary(P, from, gp.de);
    return from;
}

// The state at flagged chunk f's start, the chunk before it being right (the
// run from repair_from up to cs).  *code collects warp_dp's codes.
template <typename V>
__device__ __forceinline__ void warp_prefix(const UniParams &P, const int4 *lut, const EdgeBuf &eb, WarpRingT<V> &R,
                                            const UGeo &gf, unsigned long long f, uint32_t *code) {
    const int lane = threadIdx.x & 31;
    uint64_t base = 0, s0 = 0;
    if (lane == 0) base = repair_from(P, gf, f, &s0);
    base = __shfl_sync(kFull, base, 0);
    s0 = __shfl_sync(kFull, s0, 0);
    ring_start(R, base, s0, lane);
    *code |= warp_dp(P, lut, eb, R, base, gf.cs, gf.de, 0, [](uint64_t, uint32_t) {}, [](uint32_t, unsigned) {});
}

// Run chunk g (its start state in R), writing its true back pointers.
template <typename V>
__device__ __forceinline__ void warp_chunk(const UniParams &P, const int4 *lut, const EdgeBuf &eb, WarpRingT<V> &R,
                                           const UGeo &g, uint32_t *code) {
    *code |= warp_dp(
        P, lut, eb, R, g.cs, g.ce, g.de, 0,
        [&](uint64_t q, uint32_t bp) {
            if (q != g.ds) back_at(P, q) = bp;
        },
        [](uint32_t, unsigned) {});
    if (g.last && (int)(threadIdx.x & 31) == (int)((g.de - R.base) & 31)) back_at(P, g.de) = ring_final(R, g.de);
    __syncwarp();
}

// Whether chunk m + 1 (which starts where g ends) is right given the true
// back pointers before it; lane 0 checks, every lane gets the answer.
__device__ __forceinline__ bool warp_next_ok(const UniParams &P, const UGeo &g, unsigned long long m) {
    bool ok = false;
    if ((threadIdx.x & 31) == 0)
        ok = g.ce - g.ds <= P.guard || guard_agrees(P, P.gback + (m + 1) * (unsigned long long)P.grec, g.ce);
    return __shfl_sync(kFull, ok, 0);
}

// Parallel repair (spans E <= 63): one warp per listed flagged chunk f re-runs
// f from f-1's run start and writes f's back pointers -- right whenever f-1
// is -- and records in okn whether f + 1 then passes its check.
__global__ void __launch_bounds__(kFwdWarps * 32) k_uni_fix_a(UniParams P, uint32_t coop_max) {
    __shared__ int4 lut[256];
    extern __shared__ int32_t s_rows[];
    const uint32_t n = min(P.st->flist_len, P.flist_cap);
    if (n <= coop_max) return;   // k_uni_fix_coop runs them, a CTA each
    load_fat_lut(P, lut);
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const EdgeBuf eb(s_rows + w * (kWarpEdgeBytes / 4));
    for (uint32_t i = blockIdx.x * kFwdWarps + w; i < n; i += gridDim.x * kFwdWarps) {
        const unsigned long long f = P.flist[i];
        const UGeo gf = uni_geo(P, f);
        WarpRing R;
        uint32_t code = 0;
        warp_prefix(P, lut, eb, R, gf, f, &code);
        warp_chunk(P, lut, eb, R, gf, &code);
        if (code == kRunSpread) {   // the 32-bit window spread: the same run in 64 bits
            WideRing W;
            code = 0;
            warp_prefix(P, lut, eb, W, gf, f, &code);
            warp_chunk(P, lut, eb, W, gf, &code);
        }
        const bool ok = !code && (gf.last || warp_next_ok(P, gf, f));
        if (ok && lane == 0) atomicOr(P.okn + (f >> 5), 1u << (f & 31));
    }
}

// Cooperative parallel repair (spans E <= 63), used when the flagged chunks
// are no more than the CTAs: one CTA per listed flagged chunk f runs what
// k_uni_fix_a's warp runs (from where f's crossing chains truly meet, else
// from f-1's run start, through f's end).  Eight warps walk the trie for
// eight batches at a time into shared-memory buffers while a ninth runs the
// recurrence over the eight walked before, so the run costs about the
// recurrence's latency instead of a walk's chain of dependent trie loads per
// batch.
constexpr int kCoopWalkers = 8;
constexpr int kCoopBufWords = (kWarpEdgeBytes + 32 * 16) / 4;   // edge buffer + each lane's walk result

__global__ void __launch_bounds__((kCoopWalkers + 1) * 32) k_uni_fix_coop(UniParams P) {
    __shared__ int4 lut[256];
    __shared__ unsigned long long s_from, s_start;
    extern __shared__ int32_t s_buf[];
    load_fat_lut(P, lut);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool dp = w == kCoopWalkers;
    const uint32_t n = min(P.st->flist_len, P.flist_cap);
    if (n > gridDim.x) return;   // k_uni_fix_a runs them, a warp each
    for (uint32_t i = blockIdx.x; i < n; i += gridDim.x) {
        const unsigned long long f = P.flist[i];
        const UGeo gf = uni_geo(P, f);
        if (dp && lane == 0) {
            uint64_t s0;
            s_from = repair_from(P, gf, f, &s0);
            s_start = s0;
        }
        __syncthreads();
        const uint64_t from = s_from;
        const uint32_t npre = (uint32_t)((gf.cs - from + 31) >> 5);
        const uint32_t nb = npre + (uint32_t)((gf.ce - gf.cs + 31) >> 5);
        const uint32_t nr = (nb + kCoopWalkers - 1) / kCoopWalkers;
        // batch k: the prefix's batches up to cs, then the chunk's
        auto batch_b0 = [&](uint32_t k) { return k < npre ? from + 32ull * k : gf.cs + 32ull * (k - npre); };
        auto batch_to = [&](uint32_t k) { return k < npre ? gf.cs : gf.ce; };
        WarpRing R;
        bool rows = false, sp = false;
        if (dp) ring_start(R, from, s_start, lane);
        for (uint32_t r = 0; r <= nr; r++) {   // round r: walk group r, recurrence over group r - 1
            if (!dp) {
                const uint32_t k = r * kCoopWalkers + w;
                if (k < nb) {
                    int32_t *base = s_buf + ((r & 1) * kCoopWalkers + w) * kCoopBufWords;
                    const WalkOut wo = walk_batch(P, lut, EdgeBuf(base), batch_b0(k), batch_to(k), gf.de, 0);
                    ((uint4 *)(base + kWarpEdgeBytes / 4))[lane] =
                        make_uint4(wo.X, wo.Y, (uint32_t)wo.lr, (uint32_t)wo.unk | ((uint32_t)wo.norow << 1));
                }
            } else if (r > 0) {
                const uint32_t k1 = min(nb, r * kCoopWalkers);
                for (uint32_t k = (r - 1) * kCoopWalkers; k < k1; k++) {
                    const int32_t *base = s_buf + (((r - 1) & 1) * kCoopWalkers + (k % kCoopWalkers)) * kCoopBufWords;
                    const uint4 v = ((const uint4 *)(base + kWarpEdgeBytes / 4))[lane];
                    WalkOut wo;
                    wo.X = v.x;
                    wo.Y = v.y;
                    wo.lr = (int)v.z;
                    wo.unk = v.w & 1u;
                    wo.norow = (v.w >> 1) & 1u;
                    wo.crossing = false;
                    rows |= wo.norow;
                    sp |= dp_batch(EdgeBuf(const_cast<int32_t *>(base)), R, batch_b0(k), batch_to(k), wo,
                                   [&](uint64_t q, uint32_t bp) {
                                       if (q >= gf.cs && q != gf.ds) back_at(P, q) = bp;
                                   });
                }
            }
            __syncthreads();
        }
        if (dp) {
            if (gf.last && lane == (int)((gf.de - R.base) & 31)) back_at(P, gf.de) = ring_final(R, gf.de);
            __syncwarp();
            rows = __any_sync(kFull, rows);
            sp = __any_sync(kFull, sp);
            if (sp && !rows) {   // the 32-bit window spread: this warp runs the chunk again in 64 bits
                WideRing W;      // (the walkers' buffers are idle until every warp reaches the next chunk)
                uint32_t code = 0;
                const EdgeBuf eb(s_buf);
                warp_prefix(P, lut, eb, W, gf, f, &code);
                warp_chunk(P, lut, eb, W, gf, &code);
                sp = code != 0;
            }
            const bool ok = !rows && !sp && (gf.last || warp_next_ok(P, gf, f));
            if (ok && lane == 0) atomicOr(P.okn + (f >> 5), 1u << (f & 31));
        }
    }
}

// The chain of k_uni_frepair_warp run by one thread on a private 64-bit ring
// (back pointers in the warp kernels' format): from f's state through at
// least chunk wend, then on until a chunk passes its check; returns the chunk
// after the chain.
__device__ unsigned long long thread_chain(const UniParams &P, const int4 *lut, const UGeo &gf, unsigned long long f,
                                           unsigned long long wend) {
    long long best[64];
    uint32_t bk[64];
    const UGeo gp = gf.cs - gf.ds <= P.guard ? gf : uni_geo(P, f - 1);
    const uint64_t from = run_from(P, gp);
    start_run<64>(P, gp, from, best, bk);
    uni_run<64, false>(P, lut, best, bk, from, gf.cs, gf.de, [](uint64_t, uint32_t) {}, [](uint64_t, uint64_t) {});
    unsigned long long m = f;
    for (;;) {
        const UGeo g = uni_geo(P, m);
        uni_run<64, false>(
            P, lut, best, bk, g.cs, g.ce, g.de,
            [&](uint64_t i, uint32_t bp) {
                if (i != g.ds) back_at(P, i) = bp;
            },
            [](uint64_t, uint64_t) {});
        ++m;
        if (g.last) {
            finish_doc<64>(P, g, best, bk);
            return m;
        }
        if (m > wend && !flag_bit(P.fflag, m) &&
            (g.ce - g.ds <= P.guard || guard_agrees(P, P.gback + m * (unsigned long long)P.grec, g.ce)))
            return m;
    }
}

// A chain of k_uni_frepair_warp by the warp: from flagged chunk f's state,
// chunks f, f + 1, ... through at least chunk `through`, until one whose
// successor is not flagged and passes its check against the new back
// pointers (or the document ends); *last = the chain's last chunk.  Returns
// warp_dp's codes.
template <typename V>
__device__ uint32_t warp_chain(const UniParams &P, const int4 *lut, const EdgeBuf &eb, const UGeo &gf,
                               unsigned long long f, unsigned long long through, unsigned long long *last,
                               uint32_t *reruns) {
    WarpRingT<V> R;
    uint32_t code = 0;
    warp_prefix(P, lut, eb, R, gf, f, &code);
    unsigned long long m = f;
    for (;;) {
        const UGeo g = uni_geo(P, m);
        warp_chunk(P, lut, eb, R, g, &code);
        ++*reruns;
        if (g.last || (m >= through && !flag_bit(P.fflag, m + 1) && warp_next_ok(P, g, m))) break;
        ++m;
    }
    *last = m;
    return code;
}

// Sequential repair per document (spans E <= 63), one warp per document, in
// order over the flagged chunks.  Flagged chunk f was repaired by the
// parallel pass (k_uni_fix_coop or k_uni_fix_a) from f-1's state, which is
// right here (everything before f is).  If okn says f + 1 passes against f's
// new back pointers and f + 1 is not flagged itself, nothing is left to do.
// Otherwise the warp re-runs from f's state through the chunks after f until
// one passes its check and kept its own run's back pointers (the parallel
// pass rewrote every listed chunk).
__global__ void __launch_bounds__(128) k_uni_frepair_warp(UniParams P) {
    __shared__ int4 lut[256];
    extern __shared__ int32_t s_rows[];   // 4 edge tables
    load_fat_lut(P, lut);
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t d = blockIdx.x * 4 + w;
    if (d >= P.n_docs) return;
    const EdgeBuf eb(s_rows + w * (kWarpEdgeBytes / 4));
    const unsigned long long c0 = P.chunk_start[d], c1 = P.chunk_start[d + 1];
    unsigned long long f = warp_next_flag(P.fflag, c0, c1, lane);
    uint32_t reruns = 0;
    while (f < c1) {
        const UGeo gf = uni_geo(P, f);
        const bool fast = flag_bit(P.okn, f) && (gf.last || !flag_bit(P.fflag, f + 1));
        unsigned long long m = f + 1;
        if (!fast) {
            // after a call whose forward windows spread, chains go 64-bit at once
            const bool wide = __ldcg(&P.st->wlist_len) != 0;
            unsigned long long wend = f;   // last chunk the warp rewrote
            uint32_t code = wide ? kRunSpread : warp_chain<int32_t>(P, lut, eb, gf, f, f, &wend, &reruns);
            if (code == kRunSpread)   // the 32-bit window spread: the chain in 64 bits, through wend at least
                code = warp_chain<long long>(P, lut, eb, gf, f, wend, &wend, &reruns);
            m = wend + 1;
            if (code) {   // a long row was missing: lane 0 redoes the chain (through wend at least) on its own ring
                if (lane == 0) m = thread_chain(P, lut, gf, f, wend);
                m = __shfl_sync(kFull, m, 0);
            }
        }
        f = warp_next_flag(P.fflag, m, c1, lane);   // chunks before m are right
    }
    if (lane == 0 && reruns) atomicAdd(&P.st->fwd_repairs, reruns);
}

// ------------------------------------------------------------ backtrack ---

// Walk the back-pointer chain of chunk g from position x (>= ce, on the
// chain of a reachable position): tokens starting in [cs, ce) are counted
// (and passed to put(rank, back pointer, start), last first); returns the
// chain's last position at or after cs (the document start when the chunk is
// the first).
template <typename Put>
__device__ __forceinline__ uint64_t walk_chunk(const UniParams &P, const UGeo &g, uint64_t x, uint32_t *cnt,
                                               Put put) {
    uint32_t c = 0;
    while (x != g.ds) {
        const uint32_t v = back_at(P, x);
        const uint64_t nx = x - (v >> 24);
        if ((v >> 24) == 0 || nx < g.cs) break;   // unreachable or a run start: only on rejected input
        put(c, v, nx);
        ++c;
        x = nx;
    }
    *cnt = c;
    return x;
}

__global__ void __launch_bounds__(256) k_uni_bspec(UniParams P, unsigned long long n_chunks) {
    const unsigned long long k = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n_chunks) return;
    const UGeo g = uni_geo(P, k);
    uint64_t x = g.de;
    if (!g.last) {
        x = min(g.ce + P.ahead, g.de);
        while (x > g.ce && back_at(P, x) == 0) --x;
        // down the chain to its last position at or after ce
        for (;;) {
            const uint32_t v = back_at(P, x);
            if ((v >> 24) == 0) break;
            const uint64_t nx = x - (v >> 24);
            if (nx < g.ce) break;
            x = nx;
        }
    }
    uint32_t c;
    const uint64_t b = walk_chunk(P, g, x, &c, [](uint32_t, uint32_t, uint64_t) {});
    P.sx[k] = (uint32_t)(x - g.cs);
    P.bot[k] = (uint32_t)(b - g.cs);
    P.count[k] = c;
}

// chunk k's chain is the true path when it passes through the true sx, the
// next chunk's bot (true once that chunk is)
__global__ void __launch_bounds__(256) k_uni_bcheck(UniParams P, unsigned long long n_chunks) {
    const unsigned long long k = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k + 1 >= n_chunks) return;
    const UGeo g = uni_geo(P, k);
    if (g.last) return;
    if ((uint64_t)P.bot[k + 1] + P.chunk != (uint64_t)P.sx[k]) {   // both relative to their chunk starts
        atomicOr(P.bflag + (k >> 5), 1u << (k & 31));
        P.st->any_bflag = 1u;
    }
}

// Parallel re-walk: one thread per flagged chunk k walks it again from the
// next chunk's bot -- right whenever that chunk is -- and records in okp
// whether the chunk before k is then right too (not flagged, and its sx is
// k's new bot).
__global__ void __launch_bounds__(256) k_uni_bfix_a(UniParams P, unsigned long long n_chunks) {
    const unsigned long long k = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k + 1 >= n_chunks || !flag_bit(P.bflag, k)) return;
    const UGeo g = uni_geo(P, k);
    const uint64_t x = g.ce + P.bot[k + 1];
    uint32_t c;
    const uint64_t b = walk_chunk(P, g, x, &c, [](uint32_t, uint32_t, uint64_t) {});
    P.sx[k] = (uint32_t)(x - g.cs);
    P.bot[k] = (uint32_t)(b - g.cs);
    P.count[k] = c;
    if (!g.first && !flag_bit(P.bflag, k - 1) && (uint64_t)P.bot[k] + P.chunk == (uint64_t)P.sx[k - 1])
        atomicOr(P.okp + (k >> 5), 1u << (k & 31));
}

// One warp per document, right to left over the flagged chunks (everything
// to the right of the current one is right).  A flagged chunk k whose
// successor is not flagged was re-walked from a right bot by k_uni_bfix_a;
// with okp the chunk before it is right as well.  Otherwise k is walked again
// and so is every chunk before it until one that is not flagged and whose sx
// equals the new bot.
__global__ void __launch_bounds__(128) k_uni_brepair(UniParams P) {
    const int lane = threadIdx.x & 31;
    const uint32_t d = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (d >= P.n_docs) return;
    const long long c0 = (long long)P.chunk_start[d], c1 = (long long)P.chunk_start[d + 1];
    if (c1 - c0 < 2) return;
    unsigned long long f = warp_prev_flag(P.bflag, c1 - 2, c0, lane);
    uint32_t rewalks = 0;
    while (f != ~0ull) {
        long long k = (long long)f;
        const bool fast = !flag_bit(P.bflag, (unsigned long long)k + 1) && flag_bit(P.okp, (unsigned long long)k);
        if (!fast) {
            if (lane == 0) {
                for (;;) {
                    const UGeo g = uni_geo(P, (unsigned long long)k);
                    const uint64_t x = g.ce + P.bot[k + 1];   // the next chunk starts at ce
                    uint32_t c;
                    const uint64_t b = walk_chunk(P, g, x, &c, [](uint32_t, uint32_t, uint64_t) {});
                    P.sx[k] = (uint32_t)(x - g.cs);
                    P.bot[k] = (uint32_t)(b - g.cs);
                    P.count[k] = c;
                    ++rewalks;
                    if (k == c0 || (!flag_bit(P.bflag, (unsigned long long)k - 1) &&
                                    (uint64_t)P.bot[k] + P.chunk == (uint64_t)P.sx[k - 1]))
                        break;
                    --k;
                }
            }
            k = __shfl_sync(kFull, k, 0);
        }
        // chunk k - 1 is right now (or k is the document's first chunk)
        f = (k - 2 >= c0) ? warp_prev_flag(P.bflag, k - 2, c0, lane) : ~0ull;
    }
    if (lane == 0 && rewalks) atomicAdd(&P.st->bwd_repairs, rewalks);
}

// ----------------------------------------------------------------- emit ---

// Id of the token bytes[start, start + len) (a token: its path exists).
__device__ __forceinline__ int32_t token_id(const UniParams &P, uint64_t start, uint32_t len) {
    int32_t node = __ldg(&P.root[byte_at(P, start)].x);
    for (uint32_t i = 1; i < len; i++)
        node = (int32_t)(((uint32_t)__ldg(&P.fslot[node].y) & ~kTermBit) + byte_at(P, start + i));
    return __ldg(&P.fslot[node].w);
}

constexpr int kUniEmitThreads = 256;

// Exclusive scan of the chunk counts: tiles of 256 chunks taken in ticket
// order, each publishing its sum and then its inclusive prefix, the next
// looking back over 32 predecessors per round (bounded wait).  Then every
// chunk walks its chain from its true sx and writes its ids, last first.
__global__ void __launch_bounds__(kUniEmitThreads) k_uni_emit(UniParams P, unsigned long long n_chunks) {
    __shared__ uint32_t s_w[kUniEmitThreads / 32];
    __shared__ unsigned long long s_tile, s_off;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned long long ntiles = (n_chunks + kUniEmitThreads - 1) / kUniEmitThreads;
    if (tid == 0) s_tile = atomicAdd(&P.st->ticket, 1u);
    __syncthreads();
    const unsigned long long t = s_tile;
    if (t >= ntiles) return;
    const unsigned long long k = t * kUniEmitThreads + tid;
    const bool live = k < n_chunks;
    const uint32_t cnt = live ? P.count[k] : 0u;
    const uint32_t incl = warp_incl_sum(cnt, lane);
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    uint32_t wpre = 0, tsum = 0;
#pragma unroll
    for (int w = 0; w < kUniEmitThreads / 32; w++) {
        if (w < warp) wpre += s_w[w];
        tsum += s_w[w];
    }
    if (warp == 0) {
        unsigned long long off = 0;
        if (t > 0) {
            if (lane == 0 && t != P.stall_tile) st_relaxed(P.status + t, 1ull | ((unsigned long long)tsum << 2));
            long long jhi = (long long)t - 1;
            unsigned spins = 0;
            for (;;) {
                const long long j = jhi - lane;
                const unsigned long long w = (j >= 0) ? ld_l2(P.status + j) : 2ull;
                const uint32_t fl = (uint32_t)(w & 3ull);
                const unsigned incl_m = __ballot_sync(kFull, fl == 2);
                const int li = incl_m ? __ffs(incl_m) - 1 : 31;
                const unsigned need = (li == 31) ? kFull : ((2u << li) - 1u);
                if (__ballot_sync(kFull, fl == 0) & need) {
                    if (++spins > kUniSpinLimit) {
                        if (lane == 0) atomicOr(&P.st->err, UERR_TIMEOUT);
                        break;
                    }
                    if (spins > 32) __nanosleep(64);
                    continue;
                }
                unsigned long long v = (lane <= li) ? (w >> 2) : 0ull;
#pragma unroll
                for (int dd = 16; dd > 0; dd >>= 1) v += __shfl_xor_sync(kFull, v, dd);
                off += v;
                if (incl_m) break;
                jhi -= 32;
            }
        }
        if (lane == 0) {
            if (t != P.stall_tile) st_relaxed(P.status + t, 2ull | ((off + tsum) << 2));
            if (t == ntiles - 1) P.st->total = off + tsum;
            s_off = off;
        }
    }
    __syncthreads();
    if (!live) return;
    const unsigned long long o = s_off + wpre + incl - cnt;
    P.prefix[k] = o;
    const UGeo g = uni_geo(P, k);
    const unsigned long long last = o + cnt - 1;
    uint32_t c;
    walk_chunk(P, g, g.cs + P.sx[k], &c, [&](uint32_t r, uint32_t v, uint64_t start) {
        const unsigned long long w = last - r;
        if (w < P.cap) {
            const uint32_t id = v & 0x00FFFFFFu;
            if (id == kNoTid && P.tstart && w < P.tstart_n) {   // the id is looked up by k_uni_ids, one thread per id
                P.ids[w] = (int32_t)(v >> 24);
                P.tstart[w] = (uint32_t)(start - P.text_lo);
            } else {
                P.ids[w] = id == kUnkTid ? P.unk_id : id == kNoTid ? token_id(P, start, v >> 24) : (int32_t)id;
                if (P.tstart && w < P.tstart_n) P.tstart[w] = 0xFFFFFFFFu;
            }
        }
    });
}

// The ids k_uni_emit left to look up: ids[w] holds the token's length and
// tstart[w] its start (offset from text_lo; all ones: the id is final).
__global__ void __launch_bounds__(256) k_uni_ids(UniParams P) {
    const unsigned long long n = min(min(P.st->total, P.cap), P.tstart_n);
    for (unsigned long long w = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; w < n;
         w += (unsigned long long)gridDim.x * blockDim.x) {
        const uint32_t s = P.tstart[w];
        if (s != 0xFFFFFFFFu) P.ids[w] = token_id(P, P.text_lo + s, (uint32_t)P.ids[w]);
    }
}

__global__ void k_uni_docoff(UniParams P, unsigned long long n_chunks) {
    const uint64_t d = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    if (d > P.n_docs) return;
    const unsigned long long c = P.chunk_start[d];
    P.id_off[d] = c < n_chunks ? P.prefix[c] : P.st->total;
}

// Per trie slot: {check, base|TERM, score (int32 units), id} (scores that fit).
__global__ void k_uni_fat(const int2 *slot, const int32_t *tid, unsigned long long n_slots, const long long *units,
                          int4 *fslot) {
    const unsigned long long s = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
    if (s >= n_slots) return;
    const int2 v = slot[s];
    const int32_t t = tid[s];
    fslot[s] = make_int4(v.x, v.y, t >= 0 ? (int32_t)units[t] : 0, t);
}

// Per trie slot: the score (fixed-point units) and id of its token.
__global__ void k_uni_leaf(const int32_t *tid, unsigned long long n_slots, const long long *units, Leaf *leaf) {
    const unsigned long long s = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
    if (s >= n_slots) return;
    const int32_t t = tid[s];
    Leaf l;
    l.score = t >= 0 ? units[t] : 0;
    l.tid = t;
    l.pad = 0;
    leaf[s] = l;
}

__global__ void k_uni_copy(const uint8_t *src, uint8_t *dst, uint32_t n) {
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

}  // namespace
}  // namespace bpe

using namespace bpe;

namespace {
// Smallest q >= 0 with v * 2^q an integer (v finite): v = M * 2^(e - 53)
// with M the 53-bit mantissa; its trailing zeros lower the need.
int fraction_bits(double v) {
    if (v == 0.0) return 0;
    int e = 0;
    const double m = std::frexp(std::fabs(v), &e);   // |v| = m * 2^e, m in [0.5, 1)
    const uint64_t M = (uint64_t)std::ldexp(m, 53);
    int tz = 0;
    while (!((M >> tz) & 1ull)) ++tz;
    return std::max(0, 53 - tz - e);
}
}  // namespace

extern "C" int unigram_create(bpe_ctx *ctx, const bpe_trie *trie, const double *h_scores, uint32_t n_scores,
                              int32_t unk_id, double unk_score, bpe_unigram **out) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (!trie || !out || (n_scores && !h_scores)) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: null pointer");
    *out = nullptr;
    if (trie->device != ctx->device) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: trie on another device");
    if (n_scores != trie->n_tok)
        return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: %u scores for %u tokens", n_scores, trie->n_tok);
    if (trie->n_tok > 0xFFFFFEu) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: more than 16,777,214 tokens");
    if (trie->max_len > 255) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: a token longer than 255 bytes");
    int q = 0;
    for (uint32_t t = 0; t <= n_scores; t++) {
        const double v = t < n_scores ? h_scores[t] : unk_score;
        if (!std::isfinite(v)) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: score %u is not finite", t);
        q = std::max(q, fraction_bits(v));
    }
    if (q > 62) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: scores need %d fraction bits (at most 62)", q);
    std::vector<long long> units(std::max<uint32_t>(n_scores, 1));
    long long max_abs = 0;
    const double lim = std::ldexp(1.0, 62);
    for (uint32_t t = 0; t <= n_scores; t++) {
        const double v = std::ldexp(t < n_scores ? h_scores[t] : unk_score, q);
        if (std::fabs(v) >= lim)
            return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_create: score %u too large for 2^-%d units", t, q);
        const long long u = (long long)v;
        max_abs = std::max(max_abs, u < 0 ? -u : u);
        if (t < n_scores) units[t] = u;
    }
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    bpe_unigram *m = new bpe_unigram;
    m->ctx = ctx;
    m->trie = trie;
    m->device = ctx->device;
    m->unk_id = unk_id;
    m->unk = (long long)std::ldexp(unk_score, q);
    m->max_abs = max_abs;
    m->q = q;
    m->span = trie->max_len <= 63 ? 63u : 255u;
    void *d_units = nullptr;
    cudaError_t e = cudaMalloc(&m->d_leaf, sizeof(Leaf) * std::max<uint64_t>(trie->n_slots, 1));
    if (e == cudaSuccess) e = cudaMalloc(&d_units, sizeof(long long) * units.size());
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d_units, units.data(), sizeof(long long) * units.size(), cudaMemcpyHostToDevice, ctx->stream);
    if (e == cudaSuccess && trie->n_slots) {
        k_uni_leaf<<<(unsigned)((trie->n_slots + 255) / 256), 256, 0, ctx->stream>>>(
            trie->d_tid, trie->n_slots, (const long long *)d_units, (Leaf *)m->d_leaf);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && trie->n_slots && max_abs < (1ll << 29)) {   // the warp kernels' 32-bit sums
        e = cudaMalloc(&m->d_fslot, sizeof(int4) * trie->n_slots);
        if (e == cudaSuccess) {
            k_uni_fat<<<(unsigned)((trie->n_slots + 255) / 256), 256, 0, ctx->stream>>>(
                trie->d_slot, trie->d_tid, trie->n_slots, (const long long *)d_units, (int4 *)m->d_fslot);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    if (d_units) cudaFree(d_units);
    if (e != cudaSuccess) {
        unigram_free(m);
        return cuda_fail(ctx, e, "unigram_create");
    }
    *out = m;
    return BPE_OK;
}

extern "C" void unigram_free(bpe_unigram *model) {
    if (!model) return;
    if (model->d_leaf) cudaFree(model->d_leaf);
    if (model->d_fslot) cudaFree(model->d_fslot);
    delete model;
}

extern "C" int unigram_encode(bpe_ctx *ctx, const bpe_unigram *model, const uint8_t *d_bytes,
                              const uint64_t *d_doc_off, uint32_t n_docs, int32_t *d_ids_out, uint64_t ids_capacity,
                              uint64_t *d_id_off_out, uint64_t *n_ids) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (!model || !n_ids) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_encode: null model or n_ids");
    if (model->device != ctx->device) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_encode: model on another device");
    if (n_docs && (!d_doc_off || !d_bytes)) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_encode: null input");
    if (ids_capacity && !d_ids_out) return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_encode: null ids with capacity");
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    cudaStream_t s = ctx->stream;
    stats_reset(ctx);
    *n_ids = 0;
    if (n_docs == 0) {
        if (d_id_off_out) BPE_CUDA(ctx, cudaMemsetAsync(d_id_off_out, 0, 8, s), "id_off");
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "sync");
        return BPE_OK;
    }
    const bpe_trie *trie = model->trie;
    const uint32_t R = model->span == 63 ? 64u : 256u;
    const uint32_t C = std::max<uint32_t>(ctx->uni_chunk ? (uint32_t)ctx->uni_chunk : kUniDefaultChunk, 256u);
    int rc;
    void *cstart, *state, *pin;
    if ((rc = ensure(ctx, S_UNI_START, ((uint64_t)n_docs + 1) * 8, &cstart)) ||
        (rc = ensure(ctx, S_UNI_STATE, sizeof(UniState), &state)) || (rc = ensure_pinned(ctx, sizeof(UniState), &pin)))
        return rc;
    UniState *h = (UniState *)pin;
    const bool profile = ctx->profile != 0;
    if (profile && (rc = ensure_events(ctx, 5))) return rc;

    UniParams P{};
    P.bytes = d_bytes;
    P.doc_off = d_doc_off;
    P.n_docs = n_docs;
    P.chunk = C;
    P.guard = R == 64 ? kGuard64 : 256u;
    P.grec = P.guard + P.guard / 32;
    P.E = model->span;
    P.ahead = R;
    P.chunk_start = (const unsigned long long *)cstart;
    P.slot = trie->d_slot;
    P.root = trie->d_root;
    P.leaf = (const Leaf *)model->d_leaf;
    P.fslot = (const int4 *)model->d_fslot;
    P.unk = model->unk;
    P.unk_id = model->unk_id;
    P.stall_tile = ctx->test_stall_tile >= 0 ? (unsigned long long)ctx->test_stall_tile : ~0ull;
    P.ids = d_ids_out;
    P.cap = ids_capacity;
    P.st = (UniState *)state;

    BPE_CUDA(ctx, cudaMemsetAsync(state, 0, sizeof(UniState), s), "state clear");
    k_uni_index<<<1, 1024, 0, s>>>(P, (unsigned long long *)cstart);
    BPE_CUDA(ctx, cudaGetLastError(), "k_uni_index launch");
    k_uni_copy<<<1, 128, 0, s>>>((const uint8_t *)state, (uint8_t *)h, (uint32_t)sizeof(UniState));
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "chunk index sync");
    if (h->err & UERR_OOB)
        return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_encode: document offsets descend at document %u", h->bad_doc);
    const unsigned long long nc = h->n_chunks;
    if (nc == 0) {
        if (d_id_off_out) BPE_CUDA(ctx, cudaMemsetAsync(d_id_off_out, 0, ((uint64_t)n_docs + 1) * 8, s), "id_off");
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "sync");
        return BPE_OK;
    }
    if ((unsigned __int128)h->max_doc * (unsigned __int128)(model->max_abs + 1) >= ((unsigned __int128)1 << 62))
        return fail(ctx, BPE_ERR_INVALID_ARG,
                    "unigram_encode: a document of %llu bytes could overflow 64-bit sums of 2^-%d units",
                    (unsigned long long)h->max_doc, model->q);
    P.text_lo = h->text_lo;
    P.text_end = h->text_lo + h->span;
    const uint64_t words = (nc + 31) / 32, tiles = (nc + kUniEmitThreads - 1) / kUniEmitThreads;
    void *back, *gback, *info, *flag, *prefix, *status;
    if ((rc = ensure(ctx, S_UNI_BACK, (h->span + 1) * 4, &back)) ||
        (rc = ensure(ctx, S_UNI_GBACK, nc * (uint64_t)P.grec * 4, &gback)) ||
        (rc = ensure(ctx, S_UNI_CHUNK, nc * 12, &info)) || (rc = ensure(ctx, S_UNI_FLAG, words * 16 + nc * 8, &flag)) ||
        (rc = ensure(ctx, S_UNI_PREFIX, nc * 8 + ((uint64_t)n_docs + 1) * 8, &prefix)) ||
        (rc = ensure(ctx, S_UNI_STATUS, tiles * 8, &status)))
        return rc;
    // spans up to 63 bytes and 32-bit scores: the warp-per-chunk kernels;
    // otherwise one thread per chunk with a private ring
    const bool warp = R == 64 && model->d_fslot;
    if (warp && h->span < 0xFFFFFFFFull) {   // ids looked up by one thread each after the emit pass
        void *tst;
        P.tstart_n = std::max<uint64_t>(std::min<uint64_t>(ids_capacity, h->span + 1), 1);
        if ((rc = ensure(ctx, S_UNI_TSTART, P.tstart_n * 4, &tst))) return rc;
        P.tstart = (uint32_t *)tst;
    }
    P.back = (uint32_t *)back;
    P.gback = (uint32_t *)gback;
    P.sx = (uint32_t *)info;
    P.bot = P.sx + nc;
    P.count = P.bot + nc;
    P.fflag = (uint32_t *)flag;
    P.bflag = P.fflag + words;
    P.okn = P.bflag + words;
    P.okp = P.okn + words;
    P.flist = P.okp + words;
    P.flist_cap = (uint32_t)std::min<unsigned long long>(nc, 0xFFFFFFFFull);
    P.wlist = P.flist + nc;
    P.prefix = (unsigned long long *)prefix;
    P.status = (unsigned long long *)status;
    P.id_off = d_id_off_out ? (unsigned long long *)d_id_off_out : P.prefix + nc;
    BPE_CUDA(ctx, cudaMemsetAsync(flag, 0, words * 16, s), "flag clear");
    BPE_CUDA(ctx, cudaMemsetAsync(status, 0, tiles * 8, s), "status clear");

    const unsigned grid_c = (unsigned)((nc + kUniThreads - 1) / kUniThreads);
    const unsigned grid_c256 = (unsigned)((nc + 255) / 256);
    const unsigned grid_d = (n_docs + 3) / 4;   // one warp per document
    if (profile) cudaEventRecord(ctx->events[0], s);
    const size_t rep_smem = 4 * kWarpEdgeBytes, warp_smem = kFwdWarps * kWarpEdgeBytes;
    const size_t coop_smem = 2 * kCoopWalkers * kCoopBufWords * sizeof(int32_t);
    if (warp) {
        BPE_CUDA(ctx, cudaFuncSetAttribute(k_uni_fwd_warp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)warp_smem),
                 "k_uni_fwd_warp smem");
        BPE_CUDA(ctx, cudaFuncSetAttribute(k_uni_fix_a, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)warp_smem),
                 "k_uni_fix_a smem");
        BPE_CUDA(ctx, cudaFuncSetAttribute(k_uni_fix_coop, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)coop_smem),
                 "k_uni_fix_coop smem");
        BPE_CUDA(ctx, cudaFuncSetAttribute(k_uni_fwd_wide, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)warp_smem),
                 "k_uni_fwd_wide smem");
        k_uni_fwd_warp<<<(unsigned)((nc + kFwdWarps - 1) / kFwdWarps), kFwdWarps * 32, warp_smem, s>>>(P, nc);
        k_uni_fwd_wide<<<(unsigned)std::max(1, ctx->sm_count * 2), kFwdWarps * 32, warp_smem, s>>>(P);
    } else if (R == 64) {
        k_uni_fwd<64><<<grid_c, kUniThreads, 0, s>>>(P, nc);
    } else {
        k_uni_fwd<256><<<grid_c, kUniThreads, 0, s>>>(P, nc);
    }
    if (profile) cudaEventRecord(ctx->events[1], s);
    k_uni_check<<<grid_c256, 256, 0, s>>>(P, nc);
    if (warp) {
        const unsigned coop_grid = (unsigned)std::max(1, ctx->sm_count * 2);
        k_uni_fix_coop<<<coop_grid, (kCoopWalkers + 1) * 32, coop_smem, s>>>(P);
        k_uni_fix_a<<<(unsigned)std::max(1, ctx->sm_count * 3), kFwdWarps * 32, warp_smem, s>>>(P, coop_grid);
        k_uni_frepair_warp<<<grid_d, 128, rep_smem, s>>>(P);
    } else if (R == 64) {
        k_uni_frepair<64><<<grid_d, 128, 0, s>>>(P);
    } else {
        k_uni_frepair<256><<<grid_d, 128, 0, s>>>(P);
    }
    if (profile) cudaEventRecord(ctx->events[4], s);
    k_uni_bspec<<<grid_c256, 256, 0, s>>>(P, nc);
    k_uni_bcheck<<<grid_c256, 256, 0, s>>>(P, nc);
    k_uni_bfix_a<<<grid_c256, 256, 0, s>>>(P, nc);
    k_uni_brepair<<<grid_d, 128, 0, s>>>(P);
    if (profile) cudaEventRecord(ctx->events[2], s);
    k_uni_emit<<<(unsigned)tiles, kUniEmitThreads, 0, s>>>(P, nc);
    if (P.tstart) k_uni_ids<<<(unsigned)std::max(1, ctx->sm_count * 8), 256, 0, s>>>(P);
    if (profile) cudaEventRecord(ctx->events[3], s);
    k_uni_docoff<<<(unsigned)((n_docs + 1 + 255) / 256), 256, 0, s>>>(P, nc);
    BPE_CUDA(ctx, cudaGetLastError(), "unigram_encode launch");
    k_uni_copy<<<1, 128, 0, s>>>((const uint8_t *)state, (uint8_t *)h, (uint32_t)sizeof(UniState));
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "unigram_encode sync");
    if (h->err & UERR_CONT_START)
        return fail(ctx, BPE_ERR_INVALID_ARG, "unigram_encode: a document starts with a UTF-8 continuation byte");
    if (h->err & UERR_SPAN)
        return fail(ctx, BPE_ERR_INVALID_ARG,
                    "unigram_encode: a run of %u continuation bytes needs an edge longer than %u bytes", P.E, P.E);
    if (h->err & UERR_TIMEOUT) return fail(ctx, BPE_ERR_TIMEOUT, "unigram_encode: look-back wait gave up");

    const uint64_t total = h->total;
    *n_ids = total;
    // families, one pass each per call (launches counts passes): the forward
    // pass (with the wide re-run), its checks and repairs, the backward pass
    // (speculative backtrack, checks, re-walks), the emit pass
    const int a = stats_slot(ctx, "unigram_fwd"), b = stats_slot(ctx, "unigram_fix"), c = stats_slot(ctx, "unigram_emit");
    const int bk = stats_slot(ctx, "unigram_back");
    ctx->stats.k[a].launches = 1;
    ctx->stats.k[b].launches = 1;
    ctx->stats.k[bk].launches = 1;
    ctx->stats.k[c].launches = 1;
    const int wd = stats_slot(ctx, "unigram_wide");   // chunks whose forward run took 64-bit windows
    ctx->stats.k[wd].launches = h->wlist_len;
    ctx->stats.k[wd].bytes = (double)h->wlist_len * C;
    ctx->stats.k[a].bytes = (double)h->span;
    ctx->stats.k[b].bytes = (double)h->fwd_repairs * C;   // chunks re-run
    ctx->stats.k[bk].bytes = 4.0 * (double)h->span;        // back pointers read by the backtrack
    ctx->stats.k[c].bytes = 4.0 * (double)total;
    ctx->stats.kernel_launches = (warp ? 15 : 12) + (P.tstart ? 1 : 0);
    if (profile) {
        float x = 0, y = 0, z = 0, u = 0;
        cudaEventElapsedTime(&x, ctx->events[0], ctx->events[1]);
        cudaEventElapsedTime(&y, ctx->events[1], ctx->events[4]);
        cudaEventElapsedTime(&u, ctx->events[4], ctx->events[2]);
        cudaEventElapsedTime(&z, ctx->events[2], ctx->events[3]);
        ctx->stats.k[a].ms = x;
        ctx->stats.k[b].ms = y;
        ctx->stats.k[bk].ms = u;
        ctx->stats.k[c].ms = z;
        cudaGetLastError();
    }
    if (total > ids_capacity)
        return fail(ctx, BPE_ERR_CAPACITY, "unigram_encode: %llu ids exceed the capacity %llu",
                    (unsigned long long)total, (unsigned long long)ids_capacity);
    return BPE_OK;
}
