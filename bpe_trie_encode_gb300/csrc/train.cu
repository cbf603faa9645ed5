// train.cu -- the BPE merge loop on the GPU ([GPU-BPE] "What is this?",
// "What it does" 2.-3., and the training pipeline clear_table -> pair_count
// -> find_max -> setup_merge -> merge_reduce -> scan -> finalize_compact).
//
// Pair counts are kept exactly, for every pair ever seen, in one global table
// for the whole call:
//
//   k_count   (merge 0 only) counts every adjacent pair of the stream.  Each
//             CTA sums pairs in a shared-memory hash table (Murmur3
//             finaliser, triangular probing) and flushes it to the global
//             table when half full and once at the end ([GPU-BPE] "What it
//             does", 2. two-level pair counting).  atomicAdd returns each
//             key's running total; since counts only grow here, the largest
//             (count, -key) any flush sees is the argmax, which one
//             atomicMax per CTA records in best[0].
//   k_argmax  (merge k >= 1) max over the dense (key, count) arrays ->
//             best[k], tie-break count desc, left asc, right asc.
//   k_merge   merge + compaction + count update in one pass over the stream
//             ([GPU-BPE] "What it does", 3.; "Line by line", 2) subgroup
//             scan).  Tiles of 4,096 symbols are taken in ticket order; a tile
//             scans its items, publishes its aggregate, finds its prefix with
//             a warp-wide decoupled look-back and scatters the surviving
//             symbols.  Every pair the merge destroys or creates goes, as a
//             -1 or +1, through a shared-memory table of deltas into the
//             global counts, so the next argmax sees exact counts without a
//             full recount.
//
// Merge k's stream length, the stop flag (best[k] == 0) and the merge index
// live on the device, so iterations replay from a CUDA graph with no host
// round trip.
//
// Leftmost-first merging, the definition used: position i is a *valid start*
// when id(s[i]) == l, id(s[i+1]) == r and s[i+1] has no WORD_START.  Let c(i)
// be the number of consecutive valid starts ending at i (0 if none).  The
// left-to-right replacement merges exactly the starts with c(i) odd (for
// l != r every valid start has c(i) == 1; inside a run of l == r they
// alternate), and position i is consumed when i-1 merges.  Per position the
// parity of c is a function of the parity before it -- "negate" at a valid
// start, "zero" elsewhere -- so a tile is summarised by a 1-bit transducer
// plus its kept count for each incoming parity; these summaries compose, so
// they scan, within a tile and across tiles.
//
// Count deltas of one merge (exact): an old pair (j, j+1) (counted when
// s[j+1] has no WORD_START) disappears iff j-1, j or j+1 merges; in the new
// stream, the pair formed by a kept position j and the next kept position
// j + 1 + m(j) is new iff either side merged.
#include <algorithm>
#include <cstring>

#include "device.cuh"
#include "internal.h"

namespace bpe {
namespace {

constexpr int kCountThreads = 512;
constexpr int kCountSlots = 8192;                 // shared table slots per CTA (64 KiB)
constexpr int kCountItems = 8;
constexpr int kCountTile = kCountThreads * kCountItems;
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeItems = 16;
constexpr int kMergeTile = kMergeThreads * kMergeItems;  // 4,096 symbols per tile
// Warp-contiguous layout of a tile for l != r: warp w owns the 512 positions
// from wb = base + 512 w, in 4 rounds of 128; in round q lane L holds the 4
// positions p0 = wb + 128 q + 4 L .. p0 + 3 (one coalesced 128-bit load).
constexpr int kRounds = 4;
constexpr int kWarpSpan = 128 * kRounds;   // 512 positions per warp and tile
static_assert(kWarpSpan * kMergeWarps == kMergeTile, "tile geometry");
constexpr int kDeltaSlots = 2048;                 // shared delta table per merge CTA (16 KiB)
constexpr int kTileHalo = 16;                     // symbols staged past a tile
// Shared-memory tile layout: one padding word after every 16 symbols, so a
// thread reading its 16 consecutive symbols hits 32 different banks.
constexpr int kTileWords = (kMergeTile + kTileHalo) + (kMergeTile + kTileHalo) / 16;
__device__ __forceinline__ int padded(int i) { return i + (i >> 4); }
static_assert(kMergeItems == 16, "the padded tile layout assumes 16 symbols per thread");
constexpr int kArgmaxThreads = 256;
constexpr int kGraphIters = 32;                   // merge iterations per captured graph
constexpr int kLoopIters = 64;                    // merge iterations per persistent launch
constexpr int kBarGroups = 16;                    // first level of the grid barrier
constexpr int kPadSymbols = 64;                   // readable slack past the stream end
constexpr unsigned kSpinLimit = 1u << 22;         // look-back spins before giving up
constexpr int kInFlight = 3;                      // graph launches in flight before polling
constexpr unsigned long long kEmptySlot = ~0ull;

struct TrainState {
    uint32_t k_base;          // merges before the current graph replay
    uint32_t n_merges;
    uint32_t err;             // DERR_* bits
    uint32_t dense_len;       // entries of the dense key/count arrays
    unsigned long long n[2];  // stream length, by merge parity
    uint32_t ticket[2];       // tile tickets, by merge parity
    uint32_t msum_done;       // k_msum CTAs finished (the last one scans)
    uint32_t gactive[2];      // gapped tiles: tiles in use, by merge parity
    // occurrence-driven merges (merge sparse_from on): the stream sits in
    // buf[scur] as slen symbols, tombstones included
    uint32_t sparse_from;     // 0xFFFFFFFF: none
    uint32_t scur;
    unsigned long long slen, live, tombs;
    uint32_t occ_n[2];        // occurrences listed, by merge parity
    // grid barrier of the persistent merge loop: kBarGroups arrival counters,
    // the groups' counter and the release generation, each on its own
    // 128-byte line so arrivals and polling do not queue at one L2 slice
    alignas(128) uint32_t bar[32 * (kBarGroups + 2)];
};

struct TrainParams {
    uint32_t *buf[2];
    unsigned long long *tslot;   // hash slots: key << 32 | dense index
    uint32_t tmask;
    uint32_t *dkey;              // dense keys (l << 16 | r)
    uint32_t *dcnt;              // dense counts
    uint32_t dcap;
    unsigned long long *status[2];
    unsigned long long *rsum;    // two-pass merge: per-range summaries
    unsigned long long *rpre;    // two-pass merge: entering flag | offset << 1 per range
    unsigned long long *best;    // per merge: count << 32 | ~key ; 0 = stop
    unsigned long long *nhist;   // stream length after k merges
    uint32_t *dhist;             // dense entries scanned by argmax k
    TrainState *st;
    // gapped tiles: tile t's live symbols sit at buf + t * kMergeTile
    uint32_t *glen[2];           // live symbols per tile, by merge parity
    uint32_t *gsum;              // summary pass: tile summaries
    uint32_t *gcarry;            // summary pass: merge flag entering each tile
    unsigned long long *goff;    // summary pass: output offset of each tile (compacting merges)
    uint32_t gtiles;
    // occurrence-driven merges: each merge's occurrences as (i, j) position
    // pairs, by merge parity; compaction tiles' live counts and offsets
    uint32_t *occ[2];
    uint32_t occ_cap;
    uint32_t *ctile;
    unsigned long long *coff;
};

__device__ __forceinline__ unsigned long long pack_best(uint32_t count, uint32_t key) {
    return ((unsigned long long)count << 32) | (unsigned long long)(~key);
}

__device__ __forceinline__ uint32_t pair_key(uint32_t a, uint32_t b) { return ((a & 0xFFFFu) << 16) | (b & 0xFFFFu); }

// The global count table, as the kernels hand it around.
struct Table {
    unsigned long long *tslot;
    uint32_t *dkey, *dcnt;
    TrainState *st;
    uint32_t tmask, dcap;
};
__device__ __forceinline__ Table table_of(const TrainParams &p) {
    Table t;
    t.tslot = p.tslot; t.dkey = p.dkey; t.dcnt = p.dcnt; t.st = p.st; t.tmask = p.tmask; t.dcap = p.dcap;
    return t;
}

// Add delta (two's complement) to key's global count; returns the new total.
__device__ __forceinline__ uint32_t global_add(const Table p, uint32_t key, uint32_t delta) {
    uint32_t h = fmix32(key) & p.tmask;
    for (uint32_t probe = 1; probe <= 128; ++probe) {
        unsigned long long cur = __ldcg(p.tslot + h);
        if (cur == kEmptySlot) {
            const uint32_t idx = atomicAdd(&p.st->dense_len, 1u);
            if (idx >= p.dcap) {
                atomicOr(&p.st->err, DERR_TABLE_FULL);
                return 0;
            }
            p.dkey[idx] = key;
            const unsigned long long want = ((unsigned long long)key << 32) | idx;
            cur = atomicCAS(p.tslot + h, kEmptySlot, want);
            if (cur == kEmptySlot) cur = want;
            else p.dkey[idx] = kEmptyKey;   // lost the race: the entry stays a hole with count 0
        }
        if ((uint32_t)(cur >> 32) == key) return atomicAdd(p.dcnt + (uint32_t)cur, delta) + delta;
        h = (h + probe) & p.tmask;
    }
    atomicOr(&p.st->err, DERR_TABLE_FULL);
    return 0;
}

// Shared-memory accumulation; returns true when the key found no room in a
// crowded neighbourhood (the caller then adds it globally).
template <int SLOTS>
__device__ __forceinline__ bool smem_add(uint32_t *skey, uint32_t *sval, uint32_t *socc, uint32_t key, uint32_t delta) {
    uint32_t h = fmix32(key) & (SLOTS - 1);
#pragma unroll 1
    for (uint32_t probe = 1; probe <= 16; ++probe) {
        uint32_t cur = ((volatile uint32_t *)skey)[h];
        if (cur == kEmptyKey) {
            cur = atomicCAS(skey + h, kEmptyKey, key);
            if (cur == kEmptyKey) {
                atomicAdd(socc, 1u);
                cur = key;
            }
        }
        if (cur == key) {
            atomicAdd(sval + h, delta);
            return false;
        }
        h = (h + probe) & (SLOTS - 1);
    }
    return true;
}

// ------------------------------------------------------------ pair count ---

__global__ void __launch_bounds__(kCountThreads) k_count(TrainParams p) {
    extern __shared__ uint32_t smem[];
    uint32_t *skey = smem;
    uint32_t *scnt = smem + kCountSlots;
    __shared__ uint32_t socc;
    __shared__ unsigned long long sbest[kCountThreads / 32];

    TrainState *st = p.st;
    if (st->n_merges == 0 || st->err) return;
    const uint64_t n = st->n[0];
    const uint32_t *s = p.buf[0];
    const int tid = threadIdx.x, lane = tid & 31;

    for (int j = tid; j < kCountSlots; j += kCountThreads) {
        skey[j] = kEmptyKey;
        scnt[j] = 0;
    }
    if (tid == 0) socc = 0;
    __syncthreads();

    unsigned long long mybest = 0;
    auto flush = [&](bool clear) {
        for (int j = tid; j < kCountSlots; j += kCountThreads) {
            const uint32_t key = skey[j];
            if (key != kEmptyKey) {
                const uint32_t tot = global_add(table_of(p), key, scnt[j]);
                const unsigned long long b = pack_best(tot, key);
                mybest = b > mybest ? b : mybest;
                if (clear) {
                    skey[j] = kEmptyKey;
                    scnt[j] = 0;
                }
            }
        }
    };
    for (uint64_t base = (uint64_t)blockIdx.x * kCountTile; base < n; base += (uint64_t)gridDim.x * kCountTile) {
        const uint64_t pos = base + (uint64_t)kCountItems * tid;
        uint32_t a[kCountItems + 1];
        uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
        if (pos < n) {   // the buffer is padded: 8 symbols past pos are readable
            v0 = __ldcs(reinterpret_cast<const uint4 *>(s + pos));
            v1 = __ldcs(reinterpret_cast<const uint4 *>(s + pos + 4));
        }
        a[0] = v0.x; a[1] = v0.y; a[2] = v0.z; a[3] = v0.w;
        a[4] = v1.x; a[5] = v1.y; a[6] = v1.z; a[7] = v1.w;
        uint32_t nx = __shfl_down_sync(kFull, v0.x, 1);
        if (lane == 31) nx = (pos + kCountItems < n) ? __ldcs(s + pos + kCountItems) : kWordStart;
        a[8] = nx;
#pragma unroll
        for (int j = 0; j < kCountItems; j++) {
            if (pos + j + 1 < n && !(a[j + 1] & kWordStart)) {
                const uint32_t key = pair_key(a[j], a[j + 1]);
                if (smem_add<kCountSlots>(skey, scnt, &socc, key, 1u)) {
                    const uint32_t tot = global_add(table_of(p), key, 1u);
                    const unsigned long long b = pack_best(tot, key);
                    mybest = b > mybest ? b : mybest;
                }
            }
        }
        if (__syncthreads_or(tid == 0 && socc > kCountSlots / 2)) {
            flush(true);
            if (tid == 0) socc = 0;
            __syncthreads();
        }
    }
    __syncthreads();
    flush(false);
    mybest = warp_max_u64(mybest);
    if (lane == 0) sbest[tid >> 5] = mybest;
    __syncthreads();
    if (tid < 32) {
        unsigned long long b = tid < kCountThreads / 32 ? sbest[tid] : 0ull;
        b = warp_max_u64(b);
        if (tid == 0 && b) atomicMax(p.best, b);
    }
}

// ---------------------------------------------------------------- argmax ---

__global__ void __launch_bounds__(kArgmaxThreads) k_argmax(TrainParams p, uint32_t it) {
    __shared__ unsigned long long sbest[kArgmaxThreads / 32];
    TrainState *st = p.st;
    const uint32_t k = st->k_base + it;
    if (k == 0 || k >= st->n_merges || st->err) return;
    if ((p.best[k - 1] >> 32) == 0) return;   // training has stopped
    const uint32_t D = st->dense_len;
    if (blockIdx.x == 0 && threadIdx.x == 0) p.dhist[k] = D;
    // four counts per 128-bit load (entries past D are 0); a key is read only
    // for the largest count of the four (and its ties)
    unsigned long long b = 0;
    const uint32_t D4 = (D + 3) / 4;
    for (uint32_t i = blockIdx.x * kArgmaxThreads + threadIdx.x; i < D4; i += gridDim.x * kArgmaxThreads) {
        const uint4 c = __ldcg(reinterpret_cast<const uint4 *>(p.dcnt) + i);
        uint32_t cm = c.x > c.y ? c.x : c.y;
        cm = cm > c.z ? cm : c.z;
        cm = cm > c.w ? cm : c.w;
        if (cm == 0 || cm < (uint32_t)(b >> 32)) continue;
        const uint32_t cs[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (cs[j] == cm) {
                const unsigned long long v = pack_best(cm, __ldcg(p.dkey + 4 * i + j));
                b = v > b ? v : b;
            }
        }
    }
    b = warp_max_u64(b);
    if ((threadIdx.x & 31) == 0) sbest[threadIdx.x >> 5] = b;
    __syncthreads();
    if (threadIdx.x < 32) {
        unsigned long long x = threadIdx.x < kArgmaxThreads / 32 ? sbest[threadIdx.x] : 0ull;
        x = warp_max_u64(x);
        if (threadIdx.x == 0 && x) atomicMax(p.best + k, x);
    }
}

// -------------------------------------------------------- merge + compact ---

// 1-bit transducers: bit x of f is f(x).
constexpr uint32_t kFId = 2u;   // identity; 1 = negate, 0 = constant zero
__device__ __forceinline__ uint32_t fapply(uint32_t f, uint32_t x) { return (f >> x) & 1u; }
__device__ __forceinline__ uint32_t fcomp(uint32_t g, uint32_t f) {   // g after f
    return fapply(g, f & 1u) | (fapply(g, (f >> 1) & 1u) << 1);
}

// A summary of consecutive items packed in 32 bits: transducer f (2 bits),
// kept symbols for incoming parity 0 (15 bits) and 1 (15 bits).
constexpr uint32_t kSumId = kFId;
__device__ __forceinline__ uint32_t sum_pack(uint32_t f, uint32_t k0, uint32_t k1) { return f | (k0 << 2) | (k1 << 17); }
// b after a
__device__ __forceinline__ uint32_t sum_comp(uint32_t b, uint32_t a) {
    const uint32_t fa = a & 3u, fb = b & 3u;
    const uint32_t a0 = (a >> 2) & 0x7FFFu, a1 = a >> 17, b0 = (b >> 2) & 0x7FFFu, b1 = b >> 17;
    return sum_pack(fcomp(fb, fa), a0 + (fapply(fa, 0) ? b1 : b0), a1 + (fapply(fa, 1) ? b1 : b0));
}

// Look-back status words.
//   aggregate: 1 | f << 2 | kept(parity 0) << 4 | kept(parity 1) << 34
//   inclusive: 2 | parity << 2 | prefix << 4
__device__ __forceinline__ unsigned long long agg_word(uint32_t sum) {
    return 1ull | ((unsigned long long)(sum & 3u) << 2) | ((unsigned long long)((sum >> 2) & 0x7FFFu) << 4) |
           ((unsigned long long)(sum >> 17) << 34);
}
__device__ __forceinline__ unsigned long long inc_word(uint32_t par, unsigned long long prefix) {
    return 2ull | ((unsigned long long)par << 2) | (prefix << 4);
}

// Summary of many tiles in 64 bits: f (2 bits) | kept(parity 0) << 2 (31 bits)
// | kept(parity 1) << 33 (31 bits).  Identity: f = identity, counts 0.
__device__ __forceinline__ unsigned long long lsum_from_agg(unsigned long long w) {
    return ((w >> 2) & 3ull) | (((w >> 4) & 0x3FFFFFFFull) << 2) | (((w >> 34) & 0x3FFFFFFFull) << 33);
}
// b after a
__device__ __forceinline__ unsigned long long lsum_comp(unsigned long long b, unsigned long long a) {
    const uint32_t fa = (uint32_t)a & 3u, fb = (uint32_t)b & 3u;
    const unsigned long long a0 = (a >> 2) & 0x7FFFFFFFull, a1 = a >> 33, b0 = (b >> 2) & 0x7FFFFFFFull, b1 = b >> 33;
    const unsigned long long k0 = a0 + (fapply(fa, 0) ? b1 : b0), k1 = a1 + (fapply(fa, 1) ? b1 : b0);
    return (unsigned long long)fcomp(fb, fa) | (k0 << 2) | (k1 << 33);
}

// Warp-wide decoupled look-back for tile t (all 32 lanes call it).  Lane L
// reads the 8 status words of tiles jhi-8L-7 .. jhi-8L, so one round trip
// covers 256 predecessors; summaries are composed by a tree reduction.
// Returns false when the bounded wait gives up.
__device__ __forceinline__ bool lookback(const unsigned long long *status, uint64_t t, int lane, uint32_t *carry,
                         unsigned long long *off) {
    constexpr int kPer = 8;
    unsigned long long g = kFId;   // tiles newer than the current window, composed
    long long jhi = (long long)t - 1;
    unsigned spins = 0;
    for (;;) {
        unsigned long long w[kPer];
#pragma unroll
        for (int q = 0; q < kPer; q++) {   // q = 0 is the newest tile of this lane
            const long long j = jhi - kPer * lane - q;
            w[q] = (j >= 0) ? ld_l2(status + j) : inc_word(0, 0);
        }
        int qi = kPer;                      // newest inclusive of this lane
        bool ready = true;
#pragma unroll
        for (int q = kPer - 1; q >= 0; q--)
            if ((w[q] & 3ull) == 2) qi = q;
#pragma unroll
        for (int q = 0; q < kPer; q++)
            if (q <= qi && (w[q] & 3ull) == 0) ready = false;
        const unsigned incl_m = __ballot_sync(kFull, qi < kPer);
        const int Ls = incl_m ? __ffs(incl_m) - 1 : 32;   // first lane holding an inclusive
        const unsigned need = (Ls >= 31) ? kFull : ((2u << Ls) - 1u);
        if (__ballot_sync(kFull, !ready) & need) {
            if (++spins > kSpinLimit) return false;
            if (spins > 16) __nanosleep(32);
            continue;
        }
        // this lane's aggregates, oldest first (those newer than its inclusive)
        unsigned long long mine = kFId;
#pragma unroll
        for (int q = kPer - 1; q >= 0; q--)
            if (q < qi) mine = lsum_comp(lsum_from_agg(w[q]), mine);
        // ordered tree reduction over lanes 0 .. Ls-1 (higher lane = older)
        const int span = Ls < 32 ? Ls : 32;
        unsigned long long x = (lane < span) ? mine : (unsigned long long)kFId;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long y = __shfl_down_sync(kFull, x, d);
            if (lane + d < span) x = lsum_comp(x, y);
        }
        const unsigned long long newer = __shfl_sync(kFull, x, 0);   // lanes 0 .. span-1 composed
        if (Ls < 32) {
            // inclusive of lane Ls at its qi, then its newer aggregates, then lanes < Ls, then g
            unsigned long long wi = 0, part = 0;
            int q_i = __shfl_sync(kFull, qi, Ls);
            part = __shfl_sync(kFull, mine, Ls);
#pragma unroll
            for (int q = 0; q < kPer; q++) {
                const unsigned long long v = __shfl_sync(kFull, w[q], Ls);
                if (q == q_i) wi = v;
            }
            uint32_t par = (uint32_t)(wi >> 2) & 1u;
            unsigned long long o = wi >> 4;
            const unsigned long long chain = lsum_comp(g, lsum_comp(newer, part));
            o += par ? (chain >> 33) : ((chain >> 2) & 0x7FFFFFFFull);
            *carry = fapply((uint32_t)chain & 3u, par);
            *off = o;
            return true;
        }
        g = lsum_comp(g, newer);
        jhi -= 32 * kPer;
    }
}

// Count deltas of one thread's 16 positions (rare: only where a merge happened
// nearby), those before re only.  mm: bit j = m(pos+j) for j = 0..17; mprev =
// m(pos-1); sym(j) reads symbol pos+j from the padded tile; symbols exist
// below n.
__device__ __noinline__ void thread_deltas(const Table p, uint32_t *dkey, uint32_t *dval, uint32_t *socc,
                                           const uint32_t *mys, uint64_t pos, uint64_t re, uint64_t n, uint32_t mm,
                                           uint32_t mprev, uint32_t new_id) {
    auto sym = [&](int j) { return mys[j < 16 ? j : j + 1]; };
    auto add = [&](uint32_t kk, uint32_t d) {
        if (smem_add<kDeltaSlots>(dkey, dval, socc, kk, d)) global_add(p, kk, d);
    };
    const uint32_t mext = (mm << 1) | mprev;           // bit j: m(pos+j-1)
    // old pairs (j, j+1) touched by a merge at j-1, j or j+1
    uint32_t told = (mext | mm | (mm >> 1)) & 0xFFFFu;
    while (told) {
        const int j = __ffs(told) - 1;
        told &= told - 1;
        if (pos + j >= re || pos + j + 1 >= n) break;   // pairs owned by positions before re
        const uint32_t b = sym(j + 1);
        if (!(b & kWordStart)) add(pair_key(sym(j), b), 0xFFFFFFFFu);
    }
    // new pairs at kept positions j whose own or next kept symbol merged
    uint32_t tnew = ~mext & (mm | (mm >> 1)) & 0xFFFFu;
    while (tnew) {
        const int j = __ffs(tnew) - 1;
        tnew &= tnew - 1;
        if (pos + j >= re) break;
        const uint32_t mj = (mm >> j) & 1u;
        const int nk = j + 1 + (int)mj;
        if (pos + nk >= n) continue;
        const uint32_t b = sym(nk);
        if (b & kWordStart) continue;
        const uint32_t mk = (mm >> nk) & 1u;
        add(pair_key(mj ? new_id : sym(j), mk ? new_id : b), 1u);
    }
}

// Stage a tile (kMergeTile symbols from base) and its halo into padded shared
// memory with coalesced 128-bit loads; symbols at or past n read as 0.
__device__ __forceinline__ void stage_tile(uint32_t *stile, const uint32_t *in, uint64_t base, uint64_t n, int tid) {
#pragma unroll
    for (int q = 0; q < (kMergeTile + kTileHalo) / (4 * kMergeThreads) + 1; q++) {
        const int i4 = tid + q * kMergeThreads;
        if (i4 < (kMergeTile + kTileHalo) / 4) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (base + 4ull * i4 < n) v = __ldcg(reinterpret_cast<const uint4 *>(in + base + 4ull * i4));
            uint32_t *d = stile + padded(4 * i4);   // 4 symbols never straddle a padding word
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        }
    }
}

// Valid starts among a thread's 16 positions and the 2 after them (bit j:
// position pos + j, j = 0 .. 17), from the staged tile.
__device__ __forceinline__ uint32_t staged_valid(const uint32_t *mys, uint64_t pos, uint64_t n, uint32_t l, uint32_t r) {
    uint32_t isl = 0, isr = 0;   // id == l ; id == r without WORD_START
#pragma unroll
    for (int j = 0; j < kMergeItems + 3; j++) {
        const uint32_t x = mys[j < 16 ? j : j + 1];
        isl |= (uint32_t)((x & 0xFFFFu) == l) << j;
        isr |= (uint32_t)((x & 0x1FFFFu) == r) << j;
    }
    uint32_t valid = isl & (isr >> 1) & 0x3FFFFu;
    if (pos >= n) return 0u;
    const uint64_t lim = n - pos;   // positions pos+j with j + 1 < lim
    if (lim < kMergeItems + 3) valid &= (1u << (uint32_t)(lim - 1)) - 1u;
    return valid;
}

// Summary of one thread's 16 positions given their valid starts; positions
// at or past re (not this tile's) are left out.
__device__ __forceinline__ uint32_t thread_summary(uint32_t valid, uint64_t pos, uint64_t re) {
    uint32_t kept[2], fout[2];
#pragma unroll
    for (uint32_t c = 0; c < 2; c++) {
        uint32_t par = c, kc = 0;
#pragma unroll
        for (int j = 0; j < kMergeItems; j++) {
            if (pos + j < re) {
                kc += par ^ 1u;
                par = ((valid >> j) & 1u) ? (par ^ 1u) : 0u;
            }
        }
        kept[c] = kc;
        fout[c] = par;
    }
    return sum_pack(fout[0] | (fout[1] << 1), kept[0], kept[1]);
}

// Summary of a tile that owns no valid start: parity is 0 after every item,
// and only the first symbol can be consumed (by a merge just before the tile).
__device__ __forceinline__ uint32_t plain_tile_summary(uint32_t tile_len) {
    return sum_pack(0u, tile_len, tile_len - 1);
}

// In-tile ordered exclusive scan of the threads' summaries (all threads call
// it).  Returns the summary of the tile's items before this thread and leaves
// the tile's summary in *s_tilesum; ends with a barrier.
__device__ __forceinline__ uint32_t tile_scan(uint32_t mine, int lane, int warp, uint32_t *s_wsum,
                                              uint32_t *s_tilesum) {
    uint32_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl = sum_comp(incl, o);
    }
    uint32_t excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = kSumId;
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {   // exclusive scan of the warp totals
        uint32_t w = lane < kMergeWarps ? s_wsum[lane] : kSumId, wi = w;
#pragma unroll
        for (int d = 1; d < kMergeWarps; d <<= 1) {
            const uint32_t o = __shfl_up_sync(kFull, wi, d);
            if (lane >= d) wi = sum_comp(wi, o);
        }
        uint32_t we = __shfl_up_sync(kFull, wi, 1);
        if (lane == 0) we = kSumId;
        __syncwarp();
        if (lane < kMergeWarps) s_wsum[lane] = we;
        if (lane == kMergeWarps - 1) *s_tilesum = wi;
    }
    __syncthreads();
    return sum_comp(excl, s_wsum[warp]);
}

// A staged tile that owns no valid start: a shifted copy (a merge at the end
// of the previous tile consumed symbol 0, removing the pair it began).
__device__ __forceinline__ void emit_plain(const TrainParams &p, const uint32_t *stile, uint32_t carry,
                                           unsigned long long obase, uint64_t base, uint64_t n, uint32_t tile_len,
                                           uint32_t *out, int tid) {
    for (uint32_t i = tid; i + carry < tile_len; i += kMergeThreads) out[obase + i] = stile[padded(i + carry)];
    if (carry && tid == 0 && base + 1 < n && !(stile[1] & kWordStart))
        global_add(table_of(p), pair_key(stile[0], stile[1]), 0xFFFFFFFFu);
}

// Merge and compact a staged tile given each thread's merge flags (mm: bit j
// = m(pos+j), j = 0 .. 17; mprev = m(pos-1)), its tile-local output index e
// and the tile's kept count: count deltas, then the surviving symbols in
// order from out + obase.  Positions before re are the tile's own; symbols
// exist below n.  Needs the delta table cleared (by a barrier ago).
__device__ __forceinline__ void emit_full(const TrainParams &p, uint32_t *stile, uint32_t *dkey, uint32_t *dval,
                                          uint32_t *s_docc, uint32_t mm, uint32_t mprev, uint32_t e,
                                          uint32_t tile_kept, unsigned long long obase, uint64_t pos, uint64_t re,
                                          uint64_t n, uint32_t new_id, uint32_t *out, int tid) {
    const uint32_t *mys = stile + padded(kMergeItems * tid);
    if ((mm | mprev) & 0x1FFFFu)   // some merge touches this thread's pairs
        thread_deltas(table_of(p), dkey, dval, s_docc, mys, pos, re, n, mm, mprev, new_id);
    const uint32_t mext = (mm << 1) | mprev;   // bit j: position pos+j consumed
    uint32_t outv[kMergeItems];
#pragma unroll
    for (int j = 0; j < kMergeItems; j++) {
        const uint32_t x = mys[j];
        outv[j] = ((mm >> j) & 1u) ? (new_id | (x & kWordStart)) : x;
    }
    __syncthreads();   // every symbol of the tile is in registers: the tile buffer is free
#pragma unroll
    for (int j = 0; j < kMergeItems; j++)
        if (pos + j < re && !((mext >> j) & 1u)) stile[padded(e++)] = outv[j];
    __syncthreads();
    for (uint32_t i = tid; i < tile_kept; i += kMergeThreads) out[obase + i] = stile[padded(i)];
}

// Add a CTA's shared delta table to the global counts (after a barrier).
__device__ __forceinline__ void flush_deltas(const TrainParams &p, const uint32_t *dkey, const uint32_t *dval,
                                             const uint32_t *s_docc) {
    if (!*s_docc) return;
    for (int j = threadIdx.x; j < kDeltaSlots; j += kMergeThreads) {
        const uint32_t kk = dkey[j];
        if (kk != kEmptyKey && dval[j]) global_add(table_of(p), kk, dval[j]);
    }
}

// Merge flags of a thread's positions under the transducer scan (any l, r):
// m(pos-1) from the summary of the tile's items before the thread, then each
// valid start flips the parity and anything else clears it.
__device__ __forceinline__ uint32_t run_flags(uint32_t valid, uint32_t excl, uint32_t carry, uint32_t *mprev) {
    uint32_t par = fapply(excl & 3u, carry);
    *mprev = par;
    uint32_t mm = 0;
#pragma unroll
    for (int j = 0; j < kMergeItems + 2; j++) {
        par = ((valid >> j) & 1u) ? (par ^ 1u) : 0u;
        mm |= par << j;
    }
    return mm;
}

// Common prologue of the merge kernels: the merge to apply, or false when
// there is none (past the requested merges, an error, or training stopped).
struct MergeOp {
    uint32_t k, l, r, new_id;
    uint64_t n;
    const uint32_t *in;
    uint32_t *out;
};
// Merge k's operands, or false when training has stopped (best[k] == 0).
// Every word read here may have been written earlier in the same launch by
// the persistent loop, so the loads bypass L1.
__device__ __forceinline__ bool merge_op_at(const TrainParams &p, uint32_t k, MergeOp *op) {
    const unsigned long long bw = __ldcg(p.best + k);
    if ((bw >> 32) == 0) return false;
    const uint32_t key = ~(uint32_t)bw;
    op->k = k;
    op->l = key >> 16;
    op->r = key & 0xFFFFu;
    op->new_id = 256u + k;
    op->n = __ldcg(&p.st->n[k & 1]);
    op->in = (k & 1) ? p.buf[1] : p.buf[0];
    op->out = (k & 1) ? p.buf[0] : p.buf[1];
    return true;
}
__device__ __forceinline__ bool merge_op(const TrainParams &p, uint32_t it, MergeOp *op) {
    const TrainState *st = p.st;
    const uint32_t k = st->k_base + it;
    if (k >= st->n_merges || st->err) return false;
    return merge_op_at(p, k, op);
}

// Single pass with decoupled look-back: one tile per CTA in ticket order (a
// tile only waits on tiles that already run).
__global__ void __launch_bounds__(kMergeThreads, 4) k_merge(TrainParams p, uint32_t it) {
    extern __shared__ uint32_t dsm[];
    uint32_t *stile = dsm;                                // the tile and its halo (padded)
    uint32_t *dkey = dsm + kTileWords;                    // shared delta table
    uint32_t *dval = dkey + kDeltaSlots;
    __shared__ uint32_t s_wsum[kMergeWarps];
    __shared__ uint32_t s_tile, s_carry, s_docc, s_tilesum;
    __shared__ unsigned long long s_off;

    MergeOp op;
    if (!merge_op(p, it, &op)) return;
    TrainState *st = p.st;
    const uint32_t k = op.k;
    const uint64_t n = op.n;
    unsigned long long *status = (k & 1) ? p.status[1] : p.status[0];
    unsigned long long *next_status = (k & 1) ? p.status[0] : p.status[1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t ntiles = (n + kMergeTile - 1) / kMergeTile;

    if (tid == 0) {
        s_tile = atomicAdd(&st->ticket[k & 1], 1u);
        s_docc = 0;
        if (blockIdx.x == 0) st->ticket[(k + 1) & 1] = 0;
    }
    __syncthreads();
    const uint64_t t = s_tile;
    if (t >= ntiles) return;
    if (tid == 0) next_status[t] = 0ull;
    const uint64_t base = t * kMergeTile;
    const uint32_t tile_len = (n - base < (uint64_t)kMergeTile) ? (uint32_t)(n - base) : (uint32_t)kMergeTile;
    stage_tile(stile, op.in, base, n, tid);
    __syncthreads();
    const uint64_t pos = base + (uint64_t)kMergeItems * tid;
    const uint32_t valid = staged_valid(stile + padded(kMergeItems * tid), pos, n, op.l, op.r);
    // A tile takes the full path when it owns a valid start, or when the next
    // tile's first position is one: the merge there removes the pair (last,
    // first) and creates (last, new symbol), deltas this tile owes.
    const bool any = __syncthreads_or((valid & (tid == kMergeThreads - 1 ? 0x1FFFFu : 0xFFFFu)) != 0);
    uint32_t excl = kSumId;
    if (!any) {
        if (tid == 0) s_tilesum = plain_tile_summary(tile_len);
    } else {
        for (int j = tid; j < kDeltaSlots; j += kMergeThreads) {   // fenced by the barriers below
            dkey[j] = kEmptyKey;
            dval[j] = 0;
        }
        excl = tile_scan(thread_summary(valid, pos, n), lane, warp, s_wsum, &s_tilesum);
    }
    __syncthreads();
    const uint32_t tile = s_tilesum;

    // warp 0: publish the aggregate, look back over 256 predecessors per round trip
    if (warp == 0) {
        uint32_t carry = 0;
        unsigned long long off = 0;
        if (t > 0) {
            if (lane == 0) st_relaxed(status + t, agg_word(tile));
            if (!lookback(status, t, lane, &carry, &off)) {
                if (lane == 0) atomicOr(&st->err, DERR_TIMEOUT);
                carry = 0;
                off = 0;
            }
        }
        if (lane == 0) {
            const uint32_t t0 = (tile >> 2) & 0x7FFFu, t1 = tile >> 17;
            const unsigned long long total = off + (carry ? t1 : t0);
            st_relaxed(status + t, inc_word(fapply(tile & 3u, carry), total));
            if (t == ntiles - 1) {
                st->n[(k + 1) & 1] = total;
                p.nhist[k + 1] = total;
            }
            s_carry = carry;
            s_off = off;
        }
    }
    __syncthreads();
    const uint32_t carry = s_carry;
    if (!any) {
        emit_plain(p, stile, carry, s_off, base, n, tile_len, op.out, tid);
        return;
    }
    uint32_t mprev;
    const uint32_t mm = run_flags(valid, excl, carry, &mprev);
    const uint32_t e = carry ? (excl >> 17) : ((excl >> 2) & 0x7FFFu);
    const uint32_t tile_kept = carry ? (tile >> 17) : ((tile >> 2) & 0x7FFFu);
    emit_full(p, stile, dkey, dval, &s_docc, mm, mprev, e, tile_kept, s_off, pos, n, n, op.new_id, op.out, tid);
    flush_deltas(p, dkey, dval, &s_docc);
}

// ---- two-pass merge: per-range summaries, then apply (no inter-CTA wait) ---
//
// Both kernels give CTA b the same contiguous range of tiles.  k_msum
// summarises each range (the tile summaries composed in order); the last CTA
// to finish scans the range summaries into each range's entering merge flag
// and output offset, and the new stream length.  k_mapply then merges its
// range tile by tile, carrying flag and offset from one tile to the next with
// the tile summaries its own in-tile scans produce.

__device__ __forceinline__ unsigned long long lsum_from_sum(uint32_t s) {
    return (unsigned long long)(s & 3u) | ((unsigned long long)((s >> 2) & 0x7FFFu) << 2) |
           ((unsigned long long)(s >> 17) << 33);
}

// l != r: the stream is split into 512-symbol warp spans, balanced over the
// CTAs (ranges differ by at most one span); [r0, re) are the range's positions.
__device__ __forceinline__ void span_range(uint64_t n, uint64_t *r0, uint64_t *re) {
    const uint64_t nspans = (n + kWarpSpan - 1) / kWarpSpan;
    const uint64_t a = nspans * blockIdx.x / gridDim.x, b = nspans * (blockIdx.x + 1) / gridDim.x;
    *r0 = a * kWarpSpan;
    *re = b * kWarpSpan < n ? b * kWarpSpan : n;
    if (*r0 > *re) *r0 = *re;
}

__device__ __forceinline__ void tile_range(uint64_t ntiles, uint64_t *t0, uint64_t *t1) {
    const uint64_t per = (ntiles + gridDim.x - 1) / gridDim.x;
    const uint64_t a = (uint64_t)blockIdx.x * per;
    *t0 = a < ntiles ? a : ntiles;
    *t1 = a + per < ntiles ? a + per : ntiles;
}

// When l != r no two valid starts are adjacent (the position after one holds
// r, not l), so every valid start merges: a merge flag is the valid bit
// itself, and a range's summary is "the last position's valid bit" with kept
// count len - (valid starts before its last position), one less when its
// first symbol is consumed.
// Only l == r needs the transducer scan.


__device__ __forceinline__ uint32_t is_l(uint32_t x, uint32_t l) { return (x & 0xFFFFu) == l ? 1u : 0u; }
__device__ __forceinline__ uint32_t is_r(uint32_t x, uint32_t r) { return (x & 0x1FFFFu) == r ? 1u : 0u; }

// Valid-start bits (bit j: position p0 + j) of a lane's 4 positions for all
// rounds, with the 4 symbols per round in x[].  nx0: the symbol after the
// warp's span (read by lane 31).
__device__ __forceinline__ void quad_valid(const uint4 *x, uint32_t nx0, uint64_t wb, uint64_t n, uint32_t l,
                                           uint32_t r, int lane, uint32_t *v4) {
    uint32_t isl[kRounds], isr[kRounds];
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        isl[q] = is_l(x[q].x, l) | (is_l(x[q].y, l) << 1) | (is_l(x[q].z, l) << 2) | (is_l(x[q].w, l) << 3);
        isr[q] = is_r(x[q].x, r) | (is_r(x[q].y, r) << 1) | (is_r(x[q].z, r) << 2) | (is_r(x[q].w, r) << 3);
    }
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        uint32_t rn = __shfl_down_sync(kFull, isr[q], 1) & 1u;   // position p0 + 4
        const uint32_t rw = q + 1 < kRounds ? __shfl_sync(kFull, isr[q + 1 < kRounds ? q + 1 : q], 0) & 1u
                                            : is_r(nx0, r);
        if (lane == 31) rn = rw;
        uint32_t v = isl[q] & ((isr[q] >> 1) | (rn << 3));
        const uint64_t p0 = wb + 128ull * q + 4ull * lane;
        if (p0 >= n) v = 0;
        else if (n - p0 < 5) v &= (1u << (uint32_t)(n - p0 - 1)) - 1u;   // p0 + j + 1 < n
        v4[q] = v;
    }
}

// Count deltas of a lane's 4 positions p0 .. p0+3 (rare: only where a merge
// happened nearby), those before re (the end of the CTA's range) only.  mext
// bit j: m(p0 - 1 + j), j = 0 .. 6; sq[j]: symbol p0 + j, j = 0 .. 5.  For l != r every occurrence of the pair lr merges and
// none is created, so its count ends at exactly 0: its -1s are skipped and the
// count is cleared once instead (the hottest key would otherwise take one
// atomic per merge).
__device__ __noinline__ void quad_deltas(const Table p, uint32_t *dkey, uint32_t *dval, uint32_t *socc,
                                         const uint32_t *sq, uint64_t p0, uint64_t re, uint64_t n, uint32_t mext,
                                         uint32_t new_id, uint32_t lr) {
    auto add = [&](uint32_t kk, uint32_t d) {
        if (smem_add<kDeltaSlots>(dkey, dval, socc, kk, d)) global_add(p, kk, d);
    };
    const uint32_t mm = mext >> 1;   // bit j: m(p0 + j)
    // old pairs (j, j+1) touched by a merge at j-1, j or j+1
    uint32_t told = (mext | mm | (mm >> 1)) & 0xFu;
    while (told) {
        const int j = __ffs(told) - 1;
        told &= told - 1;
        if (p0 + j >= re || p0 + j + 1 >= n) break;   // pairs owned by positions of this range
        const uint32_t b = sq[j + 1];
        const uint32_t kk = pair_key(sq[j], b);
        if (!(b & kWordStart) && kk != lr) add(kk, 0xFFFFFFFFu);   // (l, r) itself is zeroed once
    }
    // new pairs at kept positions j whose own or next kept symbol merged
    uint32_t tnew = ~mext & (mm | (mm >> 1)) & 0xFu;
    while (tnew) {
        const int j = __ffs(tnew) - 1;
        tnew &= tnew - 1;
        if (p0 + j >= re) break;
        const uint32_t mj = (mm >> j) & 1u;
        const int nk = j + 1 + (int)mj;
        if (p0 + nk >= n) continue;
        const uint32_t b = sq[nk];
        if (b & kWordStart) continue;
        const uint32_t mk = (mm >> nk) & 1u;
        add(pair_key(mj ? new_id : sq[j], mk ? new_id : b), 1u);
    }
}

// Merge and compact one tile for l != r (every valid start merges, so the
// merge flags are the valid bits and no carry between tiles is needed: the
// flag before a warp's span is read from the data).  Survivors are packed
// into the warp's 512-word buffer wout, then copied to out + obase + (the
// warp's offset in the tile).  Returns the tile's kept count.  Deltas go to
// the CTA's shared table (cleared before, flushed by the caller).
__device__ __forceinline__ uint32_t apply_tile_distinct(const TrainParams &p, const MergeOp &op, uint64_t base,
                                                        uint64_t re, unsigned long long obase, uint32_t *wout,
                                                        uint32_t *s_wtot, uint32_t *dkey, uint32_t *dval,
                                                        uint32_t *s_docc, int lane, int warp) {
    const uint64_t n = op.n;
    const uint64_t wb = base + (uint64_t)kWarpSpan * warp;
    const bool live = wb < re;   // the warp's span lies in the CTA's range (re is span-aligned or n)
    uint4 x[kRounds];
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        const uint64_t p0 = wb + 128ull * q + 4ull * lane;
        x[q] = (live && p0 < n) ? __ldcg(reinterpret_cast<const uint4 *>(op.in + p0)) : make_uint4(0, 0, 0, 0);
    }
    // symbols past the span (lane 31) and before it (lane 0)
    uint32_t nx0 = 0, nx1 = 0, nx2 = 0, pv = 0;
    if (live && lane == 31) {
        const uint64_t e = wb + kWarpSpan;
        nx0 = e < n ? __ldcg(op.in + e) : 0u;
        nx1 = e + 1 < n ? __ldcg(op.in + e + 1) : 0u;
        nx2 = e + 2 < n ? __ldcg(op.in + e + 2) : 0u;
    }
    if (live && lane == 0 && wb > 0 && wb < n) pv = __ldcg(op.in + wb - 1);
    uint32_t v4[kRounds];
    quad_valid(x, nx0, wb, live ? n : 0, op.l, op.r, lane, v4);

    uint32_t packed = 0, kept4[kRounds], mext[kRounds];
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        const uint64_t p0 = wb + 128ull * q + 4ull * lane;
        // m(p0 - 1): the previous lane's last position, across rounds and spans
        uint32_t mp = (__shfl_up_sync(kFull, v4[q], 1) >> 3) & 1u;
        const uint32_t mw = q > 0 ? (__shfl_sync(kFull, v4[q > 0 ? q - 1 : 0], 31) >> 3) & 1u
                                  : ((wb > 0 && wb < n) ? (is_l(pv, op.l) & is_r(x[0].x, op.r)) : 0u);
        if (lane == 0) mp = mw;
        // m(p0 + 4), m(p0 + 5): the next lane's first positions
        uint32_t mn = __shfl_down_sync(kFull, v4[q], 1) & 3u;
        uint32_t mnw;
        if (q + 1 < kRounds) {
            mnw = __shfl_sync(kFull, v4[q + 1 < kRounds ? q + 1 : q], 0) & 3u;
        } else {
            const uint64_t e = wb + kWarpSpan;
            mnw = (e + 1 < n ? (is_l(nx0, op.l) & is_r(nx1, op.r)) : 0u) |
                  ((e + 2 < n ? (is_l(nx1, op.l) & is_r(nx2, op.r)) : 0u) << 1);
        }
        if (lane == 31) mn = mnw;
        mext[q] = mp | (v4[q] << 1) | (mn << 5);
        uint32_t kb = ~(mp | (v4[q] << 1)) & 0xFu;   // kept positions
        if (p0 >= re) kb = 0;
        else if (re - p0 < 4) kb &= (1u << (uint32_t)(re - p0)) - 1u;
        kept4[q] = kb;
        packed |= (uint32_t)__popc(kb) << (8 * q);
    }
    // one scan gives every round's lane offsets (8-bit fields, at most 128 each)
    const uint32_t incl = warp_incl_sum(packed, lane);
    const uint32_t excl = incl - packed;
    const uint32_t tot = __shfl_sync(kFull, incl, 31);
    uint32_t rbase = 0;
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        uint32_t o = rbase + ((excl >> (8 * q)) & 0xFFu);
        const uint32_t xs[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
        for (int j = 0; j < 4; j++)
            if ((kept4[q] >> j) & 1u) wout[o++] = ((v4[q] >> j) & 1u) ? (op.new_id | (xs[j] & kWordStart)) : xs[j];
        rbase += (tot >> (8 * q)) & 0xFFu;
    }
    // count deltas where a merge is near
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        uint32_t s4 = __shfl_down_sync(kFull, x[q].x, 1), s5 = __shfl_down_sync(kFull, x[q].y, 1);
        const uint32_t w4 = q + 1 < kRounds ? __shfl_sync(kFull, x[q + 1 < kRounds ? q + 1 : q].x, 0) : nx0;
        const uint32_t w5 = q + 1 < kRounds ? __shfl_sync(kFull, x[q + 1 < kRounds ? q + 1 : q].y, 0) : nx1;
        if (lane == 31) {
            s4 = w4;
            s5 = w5;
        }
        if (live && (mext[q] & 0x3Fu)) {
            const uint32_t sq[6] = {x[q].x, x[q].y, x[q].z, x[q].w, s4, s5};
            quad_deltas(table_of(p), dkey, dval, s_docc, sq, wb + 128ull * q + 4ull * lane, re, n, mext[q],
                        op.new_id, pair_key(op.l, op.r));
        }
    }
    if (lane == 0) s_wtot[warp] = rbase;
    __syncthreads();
    uint32_t wpre = 0, tile_kept = 0;
#pragma unroll
    for (int w = 0; w < kMergeWarps; w++) {
        const uint32_t t = s_wtot[w];
        wpre += w < warp ? t : 0u;
        tile_kept += t;
    }
    __syncwarp();
    for (uint32_t i = lane; i < rbase; i += 32) op.out[obase + wpre + i] = wout[i];
    return tile_kept;
}

// Shared words of the two-pass merge.
struct MergeShared {
    uint32_t wsum[kMergeWarps];
    unsigned long long lw[kMergeWarps];
    uint32_t lastv, docc, tilesum;
    int last;
};

// Summary of this CTA's range of tiles (valid in thread 0): for l != r the
// last position's valid bit and the kept counts, else the tile summaries
// composed in order.
__device__ __forceinline__ unsigned long long range_summary(const MergeOp &op, MergeShared &sh) {
    const uint64_t n = op.n;
    const uint32_t *in = op.in;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t ntiles = (n + kMergeTile - 1) / kMergeTile;
    const bool distinct = op.l != op.r;
    uint64_t t0, t1, r0, re;
    tile_range(ntiles, &t0, &t1);
    span_range(n, &r0, &re);
    if (tid == 0) sh.lastv = 0;
    __syncthreads();

    unsigned long long acc = kFId;   // l == r: this range's tiles so far, composed
    uint32_t cnt = 0;                // l != r: valid starts so far
    if (distinct) {
        // groups of 8 spans (one per warp), two groups' loads in flight
        for (uint64_t g = r0; g < re; g += 2 * kMergeTile) {
            uint4 x[2][kRounds];
            uint32_t nx0[2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint64_t wb = g + (uint64_t)h * kMergeTile + (uint64_t)kWarpSpan * warp;
                const bool live = wb < re;
#pragma unroll
                for (int q = 0; q < kRounds; q++) {
                    const uint64_t p0 = wb + 128ull * q + 4ull * lane;
                    x[h][q] = (live && p0 < n) ? __ldcg(reinterpret_cast<const uint4 *>(in + p0)) : make_uint4(0, 0, 0, 0);
                }
                nx0[h] = (live && lane == 31 && wb + kWarpSpan < n) ? __ldcg(in + wb + kWarpSpan) : 0u;
            }
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint64_t wb = g + (uint64_t)h * kMergeTile + (uint64_t)kWarpSpan * warp;
                if (wb >= re) continue;   // warp-uniform
                uint32_t v4[kRounds];
                quad_valid(x[h], nx0[h], wb, n, op.l, op.r, lane, v4);
#pragma unroll
                for (int q = 0; q < kRounds; q++) {
                    const uint64_t p0 = wb + 128ull * q + 4ull * lane;
                    uint32_t v = v4[q];
                    if (p0 >= re) v = 0;
                    else if (re - p0 < 4) v &= (1u << (uint32_t)(re - p0)) - 1u;   // positions of this range
                    cnt += __popc(v);
                    if (p0 < re && re - p0 <= 4) sh.lastv = (v4[q] >> (re - p0 - 1)) & 1u;
                }
            }
        }
    }
    for (uint64_t t = distinct ? t1 : t0; t < t1; t++) {
        const uint64_t base = t * kMergeTile;
        const uint64_t pos = base + (uint64_t)kMergeItems * tid;
        uint32_t isl = 0, isr = 0;
        if (pos < n) {   // the buffer is padded: 16 symbols past pos are readable
            const uint4 *src = reinterpret_cast<const uint4 *>(in + pos);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint4 v = __ldcg(src + q);
                const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    isl |= (uint32_t)((x[j] & 0xFFFFu) == op.l) << (4 * q + j);
                    isr |= (uint32_t)((x[j] & 0x1FFFFu) == op.r) << (4 * q + j);
                }
            }
        }
        uint32_t nxt = __shfl_down_sync(kFull, isr, 1) & 1u;   // position pos + 16
        if (lane == 31)
            nxt = (pos + kMergeItems < n) ? (uint32_t)((__ldcg(in + pos + kMergeItems) & 0x1FFFFu) == op.r) : 0u;
        uint32_t valid = isl & ((isr >> 1) | (nxt << 15)) & 0xFFFFu;
        if (pos >= n) valid = 0;
        else if (n - pos < kMergeItems + 1) valid &= (1u << (uint32_t)(n - pos - 1)) - 1u;   // pos+j+1 < n
        const uint32_t tile_len = (n - base < (uint64_t)kMergeTile) ? (uint32_t)(n - base) : (uint32_t)kMergeTile;
        uint32_t ts;
        if (!__syncthreads_or(valid != 0)) {
            ts = plain_tile_summary(tile_len);
        } else {
            // ordered reduction: lane L ends with lanes [L, L + 2d) composed
            uint32_t x = thread_summary(valid, pos, n);
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t y = __shfl_down_sync(kFull, x, d);
                if (lane + d < 32) x = sum_comp(y, x);
            }
            if (lane == 0) sh.wsum[warp] = x;
            __syncthreads();
            ts = sh.wsum[0];
#pragma unroll
            for (int w = 1; w < kMergeWarps; w++) ts = sum_comp(sh.wsum[w], ts);
            __syncthreads();   // wsum is reused by the next tile
        }
        acc = lsum_comp(lsum_from_sum(ts), acc);
    }
    if (distinct) {
        cnt = __reduce_add_sync(kFull, cnt);
        if (lane == 0) sh.wsum[warp] = cnt;
        __syncthreads();
        if (tid == 0) {
            uint32_t v = 0;
            for (int w = 0; w < kMergeWarps; w++) v += sh.wsum[w];
            const unsigned long long len = re - r0;
            if (len) {   // a valid start at the last position consumes the next range's first symbol
                const unsigned long long k0 = len - v + sh.lastv;
                acc = (sh.lastv ? 3ull : 0ull) | (k0 << 2) | ((k0 ? k0 - 1 : 0ull) << 33);
            }
        }
        __syncthreads();   // wsum is reused
    }
    return acc;
}

// Ordered exclusive scan of the threads' 64-bit summaries (all threads call
// it; ends with a barrier): the composition of the threads before this one.
__device__ __forceinline__ unsigned long long block_excl_lsum(unsigned long long mine, MergeShared &sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl = lsum_comp(incl, o);
    }
    unsigned long long excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = kFId;
    if (lane == 31) sh.lw[warp] = incl;
    __syncthreads();
    unsigned long long wpre = kFId;
    for (int w = 0; w < warp; w++) wpre = lsum_comp(sh.lw[w], wpre);
    __syncthreads();   // lw is reused
    return lsum_comp(excl, wpre);
}

// Entering merge flag and offset of range b from the G range summaries, and
// (by range G-1's owner thread) the new stream length.  Thread t takes the
// ranges [t*per, (t+1)*per).  write_all: also store every range's prefix.
__device__ __forceinline__ void scan_ranges(const TrainParams &p, uint32_t k, uint32_t G, bool write_all, uint32_t b_want,
                                            MergeShared &sh, uint32_t *carry_out, unsigned long long *off_out) {
    const int tid = threadIdx.x;
    const uint32_t per = (G + kMergeThreads - 1) / kMergeThreads;
    const uint32_t b0 = tid * per < G ? tid * per : G, b1 = b0 + per < G ? b0 + per : G;
    unsigned long long mine = kFId;
    for (uint32_t b = b0; b < b1; b++) mine = lsum_comp(__ldcg(p.rsum + b), mine);
    const unsigned long long excl = block_excl_lsum(mine, sh);
    // walk this thread's ranges from the stream start's state (flag 0, offset 0)
    uint32_t carry = fapply((uint32_t)excl & 3u, 0u);
    unsigned long long off = (excl >> 2) & 0x7FFFFFFFull;
    for (uint32_t b = b0; b < b1; b++) {
        if (write_all) p.rpre[b] = (off << 1) | carry;
        if (b == b_want) {
            sh.lw[0] = (off << 1) | carry;
        }
        const unsigned long long sb = __ldcg(p.rsum + b);
        off += carry ? (sb >> 33) : ((sb >> 2) & 0x7FFFFFFFull);
        carry = fapply((uint32_t)sb & 3u, carry);
    }
    if (b0 < b1 && b1 == G && (write_all || b_want == 0)) {
        p.st->n[(k + 1) & 1] = off;
        p.nhist[k + 1] = off;
    }
    __syncthreads();
    const unsigned long long pre = sh.lw[0];
    *carry_out = (uint32_t)pre & 1u;
    *off_out = pre >> 1;
    __syncthreads();   // lw is reused
}

// Merge and compact this CTA's range of tiles, entering with the merge flag
// carry and output offset off; count deltas go through one shared table,
// flushed once at the end.
__device__ __forceinline__ void apply_range(const TrainParams &p, const MergeOp &op, uint32_t carry,
                                            unsigned long long off, uint32_t *dsm, MergeShared &sh) {
    uint32_t *stile = dsm;   // l == r: the staged tile; l != r: the warps' output buffers
    uint32_t *dkey = dsm + kTileWords;
    uint32_t *dval = dkey + kDeltaSlots;
    const uint64_t n = op.n;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t ntiles = (n + kMergeTile - 1) / kMergeTile;
    const bool distinct = op.l != op.r;
    uint64_t t0, t1, r0, re;
    tile_range(ntiles, &t0, &t1);
    span_range(n, &r0, &re);
    if (distinct && blockIdx.x == 0 && tid == 0)   // every occurrence of (l, r) merges: its count ends at 0
        global_add(table_of(p), pair_key(op.l, op.r), 0u - (uint32_t)(__ldcg(p.best + op.k) >> 32));
    if (distinct ? r0 >= re : t0 >= t1) return;
    if (tid == 0) sh.docc = 0;
    for (int j = tid; j < kDeltaSlots; j += kMergeThreads) {
        dkey[j] = kEmptyKey;
        dval[j] = 0;
    }
    __syncthreads();
    if (distinct) {
        uint32_t *wout = stile + kWarpSpan * warp;
        for (uint64_t g = r0; g < re; g += kMergeTile) {
            off += apply_tile_distinct(p, op, g, re, off, wout, sh.wsum, dkey, dval, &sh.docc, lane, warp);
            __syncthreads();   // the output buffers and shared words are reused
        }
    } else {
        for (uint64_t t = t0; t < t1; t++) {
            const uint64_t base = t * kMergeTile;
            const uint32_t tile_len = (n - base < (uint64_t)kMergeTile) ? (uint32_t)(n - base) : (uint32_t)kMergeTile;
            stage_tile(stile, op.in, base, n, tid);
            __syncthreads();
            const uint64_t pos = base + (uint64_t)kMergeItems * tid;
            const uint32_t valid = staged_valid(stile + padded(kMergeItems * tid), pos, n, op.l, op.r);
            // the full path also when the next tile's first position merges: the
            // pair (last, first) it removes and (last, new) it creates are ours
            const bool any = __syncthreads_or((valid & (tid == kMergeThreads - 1 ? 0x1FFFFu : 0xFFFFu)) != 0);
            if (!any) {
                emit_plain(p, stile, carry, off, base, n, tile_len, op.out, tid);
                off += tile_len - carry;
                carry = 0;
                __syncthreads();   // the tile buffer is reused
                continue;
            }
            const uint32_t excl = tile_scan(thread_summary(valid, pos, n), lane, warp, sh.wsum, &sh.tilesum);
            const uint32_t tile = sh.tilesum;
            uint32_t mprev;
            const uint32_t mm = run_flags(valid, excl, carry, &mprev);
            const uint32_t e = carry ? (excl >> 17) : ((excl >> 2) & 0x7FFFu);
            const uint32_t tile_kept = carry ? (tile >> 17) : ((tile >> 2) & 0x7FFFu);
            emit_full(p, stile, dkey, dval, &sh.docc, mm, mprev, e, tile_kept, off, pos, n, n, op.new_id, op.out, tid);
            off += tile_kept;
            carry = fapply(tile & 3u, carry);
            __syncthreads();   // the tile buffer and shared words are reused
        }
    }
    flush_deltas(p, dkey, dval, &sh.docc);
}

__global__ void __launch_bounds__(kMergeThreads) k_msum(TrainParams p, uint32_t it) {
    __shared__ MergeShared sh;
    MergeOp op;
    if (!merge_op(p, it, &op)) return;
    TrainState *st = p.st;
    const unsigned long long acc = range_summary(op, sh);
    if (threadIdx.x == 0) p.rsum[blockIdx.x] = acc;
    // the last CTA to finish scans the range summaries
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) sh.last = atomicAdd(&st->msum_done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!sh.last) return;
    __threadfence();
    uint32_t c;
    unsigned long long o;
    scan_ranges(p, op.k, gridDim.x, true, 0, sh, &c, &o);
    if (threadIdx.x == 0) st->msum_done = 0;
}

__global__ void __launch_bounds__(kMergeThreads, 4) k_mapply(TrainParams p, uint32_t it) {
    extern __shared__ uint32_t dsm[];
    __shared__ MergeShared sh;
    MergeOp op;
    if (!merge_op(p, it, &op)) return;
    const unsigned long long pre = p.rpre[blockIdx.x];
    apply_range(p, op, (uint32_t)pre & 1u, pre >> 1, dsm, sh);
}

// ------------------------------------------- persistent two-pass merge loop ---
//
// One cooperative launch runs merges [k_begin, k_end): argmax, range
// summaries and apply, separated by grid barriers (all CTAs are resident).
// Each CTA finds its own range's prefix from the G summaries, so a merge
// costs three barriers and no kernel launch.

// Grid barrier with a bounded wait: false (and DERR_TIMEOUT) when it gives up.
// Two levels: CTA b arrives at counter b % kBarGroups; the last arrival of a
// group arrives at the groups' counter, whose last arrival bumps the
// generation the others poll.
__device__ __forceinline__ bool grid_sync(TrainState *st, int *s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t *grp = st->bar, *top = st->bar + 32 * kBarGroups, *gen_w = top + 32;
        const uint32_t G = gridDim.x, g = blockIdx.x % kBarGroups;
        const uint32_t ngroups = G < (uint32_t)kBarGroups ? G : (uint32_t)kBarGroups;
        const uint32_t gsize = (G - g + kBarGroups - 1) / kBarGroups;   // CTAs b < G with b % kBarGroups == g
        const uint32_t gen = ld_acquire_u32(gen_w);
        __threadfence();
        int ok = 1;
        if (atomicAdd(grp + 32 * g, 1u) == gsize - 1) {
            atomicExch(grp + 32 * g, 0u);
            if (atomicAdd(top, 1u) == ngroups - 1) {
                atomicExch(top, 0u);
                __threadfence();
                st_release_u32(gen_w, gen + 1);
            }
        }
        unsigned spins = 0;
        while (ld_acquire_u32(gen_w) == gen) {
            if (++spins > kSpinLimit) {
                atomicOr(&st->err, DERR_TIMEOUT);
                ok = 0;
                break;
            }
            if (spins > 4) __nanosleep(100);
        }
        __threadfence();
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Block max of (count, ~key) over the dense table, folded into best[k].
__device__ __forceinline__ void argmax_into(const TrainParams &p, uint32_t k, unsigned long long *sbest) {
    const uint32_t D = __ldcg(&p.st->dense_len);
    if (blockIdx.x == 0 && threadIdx.x == 0) p.dhist[k] = D;
    unsigned long long b = 0;
    const uint32_t D4 = (D + 3) / 4;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < D4; i += gridDim.x * blockDim.x) {
        const uint4 c = __ldcg(reinterpret_cast<const uint4 *>(p.dcnt) + i);
        uint32_t cm = c.x > c.y ? c.x : c.y;
        cm = cm > c.z ? cm : c.z;
        cm = cm > c.w ? cm : c.w;
        if (cm == 0 || cm < (uint32_t)(b >> 32)) continue;
        const uint32_t cs[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if (cs[j] == cm) {
                const unsigned long long v = pack_best(cm, __ldcg(p.dkey + 4 * i + j));
                b = v > b ? v : b;
            }
        }
    }
    b = warp_max_u64(b);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sbest[warp] = b;
    __syncthreads();
    if (threadIdx.x < 32) {
        unsigned long long x = threadIdx.x < blockDim.x / 32 ? sbest[threadIdx.x] : 0ull;
        x = warp_max_u64(x);
        if (threadIdx.x == 0 && x) atomicMax(p.best + k, x);
    }
}

// ------------------------------------------------ occurrence-driven merges ---
//
// Once the best pair is rare, rewriting the whole stream per merge costs far
// more than the merge changes.  From merge sparse_from on (chosen by the
// host), a merge instead
//   k_sscan     reads the stream once and, for each occurrence (i, j) of the
//               pair that merges (j: the next live position after i), applies
//               the exact count deltas from the old stream and lists (i, j);
//   k_sargmax   (the next merge's first kernel) writes new_id at i and a
//               tombstone at j for every listed occurrence, then runs that
//               merge's argmax.
// A pair is a live symbol and the next live one after it (tombstones are
// skipped); the stream is compacted when tombstones pass a quarter of it
// (k_ccount, k_cscan, k_cscatter, k_cdone, once per window of merges, after
// its first k_sargmax has applied the previous merge) and once at the end.
//
// Count deltas of one occurrence (i, j) that merges, taken from the old
// stream (p: the live position before i when i has no WORD_START; q: the
// live position after j when it has none):
//   own pair (l, r): -1 (for l != r all occurrences merge, so one thread
//       subtracts the whole count instead);
//   left edge (p, i): -(s[p], l), +(s[p]', new) where s[p]' = new when p is
//       the right half of another merging occurrence -- the edge between two
//       occurrences is counted by the right one;
//   right edge (j, q), unless q starts a merging occurrence: -(r, s[q]),
//       +(new, s[q]).
// For l == r only starts with an odd number of consecutive valid starts
// ending at them merge (leftmost first), and the first start of each run
// walks the run; the right half of the previous merging start and the next
// merging start are then exactly the cases the two tests above check.
constexpr uint32_t kTomb = 0xFFFFFFFFu;   // never a symbol: bits 17..31 of a symbol are 0
constexpr uint32_t kNoSparse = 0xFFFFFFFFu;
constexpr int kSparseThreads = 256;
constexpr uint64_t kSparseDiv = 64;   // automatic switch: best count below n / kSparseDiv

__device__ __forceinline__ uint32_t sym_id(uint32_t x) { return x & 0xFFFFu; }

__device__ __forceinline__ uint64_t next_live(const uint32_t *s, uint64_t a, uint64_t n) {
    uint64_t b = a + 1;
    while (b < n && __ldg(s + b) == kTomb) ++b;
    return b;
}

// The live position before a, or -1.
__device__ __forceinline__ long long prev_live(const uint32_t *s, uint64_t a) {
    long long b = (long long)a - 1;
    while (b >= 0 && __ldg(s + b) == kTomb) --b;
    return b;
}

// The count deltas of an occurrence (i, j) that merges, and its list entry.
__device__ void occurrence_deltas(const TrainParams &p, const Table &T, const uint32_t *s, uint64_t n, uint64_t i,
                                  uint64_t j, uint32_t l, uint32_t r, uint32_t nid, uint32_t k) {
    const uint32_t si = __ldg(s + i);
    if (l == r) global_add(T, pair_key(l, r), 0xFFFFFFFFu);
    if (!(si & kWordStart)) {
        const long long pp = prev_live(s, i);
        if (pp >= 0) {
            const uint32_t sp = __ldg(s + pp);
            bool pocc = false;   // p is the right half of a merging occurrence
            if (sym_id(sp) == r && !(sp & kWordStart)) {
                const long long p2 = prev_live(s, (uint64_t)pp);
                pocc = p2 >= 0 && sym_id(__ldg(s + p2)) == l;
            }
            global_add(T, pair_key(sp, l), 0xFFFFFFFFu);
            global_add(T, pair_key(pocc ? nid : sp, nid), 1u);
        }
    }
    const uint64_t q = next_live(s, j, n);
    if (q < n) {
        const uint32_t sq = __ldg(s + q);
        if (!(sq & kWordStart)) {
            bool qocc = false;   // q starts a merging occurrence
            if (sym_id(sq) == l) {
                const uint64_t q2 = next_live(s, q, n);
                qocc = q2 < n && sym_id(__ldg(s + q2)) == r && !(__ldg(s + q2) & kWordStart);
            }
            if (!qocc) {
                global_add(T, pair_key(r, sq), 0xFFFFFFFFu);
                global_add(T, pair_key(nid, sq), 1u);
            }
        }
    }
    const uint32_t x = atomicAdd(&p.st->occ_n[k & 1], 1u);
    if (x < p.occ_cap) {
        p.occ[k & 1][2 * (uint64_t)x] = (uint32_t)i;
        p.occ[k & 1][2 * (uint64_t)x + 1] = (uint32_t)j;
    } else {
        atomicOr(&p.st->err, DERR_OOB);   // the list is sized by a count no later merge exceeds
    }
}

// Whether live position x starts a pair with id r next: *y = the next live position.
__device__ __forceinline__ bool valid_start(const uint32_t *s, uint64_t n, uint64_t x, uint32_t r, uint64_t *y) {
    *y = next_live(s, x, n);
    return *y < n && sym_id(__ldg(s + *y)) == r && !(__ldg(s + *y) & kWordStart);
}

// Position i holds l (live).  For l != r: if (i, next live) is an
// occurrence, it merges.  For l == r only the first valid start of a run of
// consecutive valid starts proceeds: it walks the run and handles the starts
// that merge (every second one, leftmost first), so a run of length L costs
// O(L) steps in one thread.
__device__ void sparse_occurrence(const TrainParams &p, const Table &T, const uint32_t *s, uint64_t n, uint64_t i,
                                  uint32_t l, uint32_t r, uint32_t nid, uint32_t k) {
    uint64_t j;
    if (!valid_start(s, n, i, r, &j)) return;
    if (l != r) {
        occurrence_deltas(p, T, s, n, i, j, l, r, nid, k);
        return;
    }
    if (!(__ldg(s + i) & kWordStart)) {
        const long long pp = prev_live(s, i);
        if (pp >= 0 && sym_id(__ldg(s + pp)) == l) return;   // a valid start precedes i: not the run's first
    }
    uint64_t x = i, y = j;
    for (;;) {
        occurrence_deltas(p, T, s, n, x, y, l, r, nid, k);
        const uint64_t z = next_live(s, y, n);   // the next start that may merge
        if (z >= n || sym_id(__ldg(s + z)) != l || (__ldg(s + z) & kWordStart)) break;
        uint64_t w;
        if (!valid_start(s, n, z, r, &w)) break;
        x = z;
        y = w;
    }
}

__global__ void __launch_bounds__(kSparseThreads) k_sscan(TrainParams p, uint32_t it) {
    TrainState *st = p.st;
    const uint32_t k = st->k_base + it;
    if (k >= st->n_merges || st->err || k < st->sparse_from) return;
    const unsigned long long bw = __ldcg(p.best + k);
    const uint32_t cnt = (uint32_t)(bw >> 32);
    if (cnt == 0) return;
    const uint32_t key = ~(uint32_t)bw, l = key >> 16, r = key & 0xFFFFu, nid = 256u + k;
    const uint32_t *s = p.buf[st->scur];
    const uint64_t n = st->slen;
    const Table T = table_of(p);
    if (l != r && blockIdx.x == 0 && threadIdx.x == 0) global_add(T, key, 0u - cnt);   // its count ends at 0
    const uint64_t nq = (n + 3) / 4;   // the buffer is padded: a quad past n is readable
    for (uint64_t x = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; x < nq; x += (uint64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(s) + x);
        // positions of the quad holding l (rare): one call site for all four
        uint32_t m = (sym_id(v.x) == l && v.x != kTomb ? 1u : 0u) | (sym_id(v.y) == l && v.y != kTomb ? 2u : 0u) |
                     (sym_id(v.z) == l && v.z != kTomb ? 4u : 0u) | (sym_id(v.w) == l && v.w != kTomb ? 8u : 0u);
        while (m) {
            const uint32_t e = __ffs(m) - 1;
            m &= m - 1;
            if (4 * x + e < n) sparse_occurrence(p, T, s, n, 4 * x + e, l, r, nid, k);
        }
    }
}

// Apply merge k-1's listed occurrences (when it was occurrence-driven), then
// merge k's argmax.
__global__ void __launch_bounds__(kArgmaxThreads) k_sargmax(TrainParams p, uint32_t it) {
    __shared__ unsigned long long sbest[kArgmaxThreads / 32];
    TrainState *st = p.st;
    const uint32_t k = st->k_base + it;
    const uint32_t sf = st->sparse_from;
    if (k >= 1 && sf != kNoSparse && k - 1 >= sf && k - 1 < st->n_merges) {
        const uint32_t m = min(st->occ_n[(k - 1) & 1], p.occ_cap);
        uint32_t *s = p.buf[st->scur];
        const uint32_t nid = 256u + (k - 1);
        const uint32_t *L = p.occ[(k - 1) & 1];
        for (uint32_t x = blockIdx.x * blockDim.x + threadIdx.x; x < m; x += gridDim.x * blockDim.x) {
            const uint32_t i = L[2 * (uint64_t)x], j = L[2 * (uint64_t)x + 1];
            s[i] = nid | (s[i] & kWordStart);
            s[j] = kTomb;
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            st->live -= m;
            st->tombs += m;
            p.nhist[k] = st->live;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && sf != kNoSparse && k >= sf) st->occ_n[k & 1] = 0;   // merge k lists here
    if (k == 0 || k >= st->n_merges || st->err) return;
    if ((__ldcg(p.best + k - 1) >> 32) == 0) return;   // training has stopped
    argmax_into(p, k, sbest);
}

__global__ void __launch_bounds__(kMergeThreads, 4) k_train_loop(TrainParams p, uint32_t k_begin, uint32_t k_end) {
    extern __shared__ uint32_t dsm[];
    __shared__ MergeShared sh;
    __shared__ unsigned long long sbest[kMergeWarps];
    __shared__ int s_ok;
    TrainState *st = p.st;
    for (uint32_t k = k_begin; k < k_end; k++) {
        if (k > 0) argmax_into(p, k, sbest);   // merge 0's pair comes from the count pass
        if (!grid_sync(st, &s_ok)) return;
        // after the barrier every CTA reads the same best[k] and err (nothing
        // writes them until the next barrier)
        MergeOp op;
        if (__ldcg(&st->err) || !merge_op_at(p, k, &op)) return;
        const unsigned long long acc = range_summary(op, sh);
        if (threadIdx.x == 0) __stcg(p.rsum + blockIdx.x, acc);
        if (!grid_sync(st, &s_ok)) return;
        uint32_t carry;
        unsigned long long off;
        scan_ranges(p, k, gridDim.x, false, blockIdx.x, sh, &carry, &off);
        apply_range(p, op, carry, off, dsm, sh);
        if (!grid_sync(st, &s_ok)) return;
    }
}

// ------------------------------------------------------- gapped tile stream ---
//
// BPE_MERGE_TILES.  The stream is kept as fixed 4,096-slot tiles,
// each holding its live symbols at its start (a count per tile); the stream
// is the tiles' live parts in order.  A merge compacts each tile into the
// same tile of the other buffer, so no global offset is needed: for l != r
// one kernel does the whole merge, each tile reading the symbols around it
// from its neighbours' live parts.  For l == r a summary pass first gives
// each tile the merge flag entering it.  The contiguous stream is gathered
// once, at the end.

constexpr int kGapStage = 4 + kMergeTile + 16;   // [3] = symbol before the tile, [4 ..] = tile + halo

struct GapHalo {
    uint32_t prev, has_prev, nnext;
    uint32_t nx[3];
};

// The last live symbol before tile t and the first (up to 3) after it,
// skipping empty tiles.
__device__ __forceinline__ void gap_halo(const uint32_t *in, const uint32_t *lin, uint32_t T, uint32_t t,
                                         GapHalo *h) {
    h->has_prev = 0;
    h->prev = 0;
    for (uint32_t u = t; u-- > 0;) {
        const uint32_t lu = __ldcg(lin + u);
        if (lu) {
            h->prev = __ldcg(in + (uint64_t)u * kMergeTile + lu - 1);
            h->has_prev = 1;
            break;
        }
    }
    h->nnext = 0;
    for (uint32_t u = t + 1; u < T && h->nnext < 3; u++) {
        const uint32_t lu = __ldcg(lin + u);
        for (uint32_t i = 0; i < lu && h->nnext < 3; i++) h->nx[h->nnext++] = __ldcg(in + (uint64_t)u * kMergeTile + i);
    }
}

// Stage tile t's len live symbols and the halo symbols after them into the
// padded layout of the transducer path (tile-local positions).  Ends with a
// barrier.
__device__ __forceinline__ void stage_gapped_padded(uint32_t *stile, const uint32_t *tin, uint32_t len,
                                                    const GapHalo &h) {
    constexpr int kQuads = (kMergeTile + kTileHalo) / 4 / kMergeThreads + 1;
    uint4 v[kQuads];
#pragma unroll
    for (int u = 0; u < kQuads; u++) {   // all loads in flight before the first store
        const uint32_t i4 = threadIdx.x + u * blockDim.x;
        v[u] = 4 * i4 < len ? __ldcg(reinterpret_cast<const uint4 *>(tin) + i4) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuads; u++) {
        const uint32_t i4 = threadIdx.x + u * blockDim.x;
        if (i4 < (kMergeTile + kTileHalo) / 4) {
            uint32_t *d = stile + padded(4 * i4);
            d[0] = v[u].x; d[1] = v[u].y; d[2] = v[u].z; d[3] = v[u].w;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (uint32_t j = 0; j < h.nnext; j++) stile[padded(len + j)] = h.nx[j];
    __syncthreads();
}

__device__ __forceinline__ uint32_t bit_if(bool b, int j) { return b ? (1u << j) : 0u; }

// l != r, one tile: warp w takes tile positions [512 w, 512 w + 512) in four
// rounds of 128 (lane L: 4 positions from 128 q + 4 L), reading the staged
// tile (sdat[3]: the symbol before the tile, sdat[4 + i]: symbol i, halo after
// len).  Every read of sdat happens before the one barrier in here; after it
// each warp packs its survivors into its own part of sout and copies them to
// tout.  Returns the tile's kept count.
__device__ __forceinline__ uint32_t gap_tile_distinct(const TrainParams &p, const MergeOp &op, const uint32_t *sdat,
                                                      uint32_t len, uint32_t E, bool has_prev, uint32_t *sout,
                                                      uint32_t *tout, uint32_t *s_wtot, uint32_t *dkey,
                                                      uint32_t *dval, uint32_t *s_docc, int lane, int warp) {
    const uint32_t w0 = (uint32_t)kWarpSpan * warp;
    uint32_t packed = 0, kept4[kRounds] = {0, 0, 0, 0}, mext[kRounds] = {0, 0, 0, 0};
    uint4 xs[kRounds], xn[kRounds];
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        const uint32_t p0 = w0 + 128u * q + 4u * lane;
        xs[q] = make_uint4(0, 0, 0, 0);
        xn[q] = make_uint4(0, 0, 0, 0);
        if (p0 >= len) continue;
        xs[q] = *reinterpret_cast<const uint4 *>(sdat + 4 + p0);
        xn[q] = *reinterpret_cast<const uint4 *>(sdat + 8 + p0);
        const uint32_t sp = sdat[3 + p0];   // symbol p0 - 1
        const uint32_t sym[8] = {sp, xs[q].x, xs[q].y, xs[q].z, xs[q].w, xn[q].x, xn[q].y, xn[q].z};
        // bit j: m(p0 - 1 + j) = valid(p0 - 1 + j), j = 0 .. 6 (l != r: every valid start merges)
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 7; j++) {
            const uint32_t i1 = p0 + j;   // position of the right symbol of the pair starting at p0 - 1 + j
            const bool exists = i1 < E && (j > 0 || p0 > 0 || has_prev);
            m |= bit_if(exists && is_l(sym[j], op.l) && is_r(sym[j + 1], op.r), j);
        }
        mext[q] = m;
        uint32_t kb = ~m & 0xFu;   // position p0 + j is consumed when p0 + j - 1 merged
        if (len - p0 < 4) kb &= (1u << (len - p0)) - 1u;
        kept4[q] = kb;
        packed |= (uint32_t)__popc(kb) << (8 * q);
    }
    const uint32_t incl = warp_incl_sum(packed, lane);
    const uint32_t excl = incl - packed;
    const uint32_t tot = __shfl_sync(kFull, incl, 31);
    uint32_t wkept = 0;
#pragma unroll
    for (int q = 0; q < kRounds; q++) wkept += (tot >> (8 * q)) & 0xFFu;
    if (lane == 0) s_wtot[warp] = wkept;
    // count deltas where a merge is near (positions of this tile only)
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        if (mext[q] & 0x3Fu) {
            const uint32_t sq[6] = {xs[q].x, xs[q].y, xs[q].z, xs[q].w, xn[q].x, xn[q].y};
            quad_deltas(table_of(p), dkey, dval, s_docc, sq, w0 + 128u * q + 4u * lane, len, E, mext[q], op.new_id,
                        pair_key(op.l, op.r));
        }
    }
    __syncthreads();
    uint32_t wpre = 0, tile_kept = 0;
#pragma unroll
    for (int w = 0; w < kMergeWarps; w++) {
        const uint32_t t = s_wtot[w];
        wpre += w < warp ? t : 0u;
        tile_kept += t;
    }
    uint32_t rbase = wpre;
#pragma unroll
    for (int q = 0; q < kRounds; q++) {
        uint32_t o = rbase + ((excl >> (8 * q)) & 0xFFu);
        const uint32_t x4[4] = {xs[q].x, xs[q].y, xs[q].z, xs[q].w};
#pragma unroll
        for (int j = 0; j < 4; j++)
            if ((kept4[q] >> j) & 1u) sout[o++] = ((mext[q] >> (j + 1)) & 1u) ? (op.new_id | (x4[j] & kWordStart)) : x4[j];
        rbase += (tot >> (8 * q)) & 0xFFu;
    }
    __syncwarp();
    for (uint32_t i = wpre + lane; i < wpre + wkept; i += 32) tout[i] = sout[i];
    return tile_kept;
}

// l == r, one tile entering with merge flag carry: the transducer path over
// the padded staging (kept apart so its registers do not weigh on the l != r
// path).  Returns the tile's kept count; ends after its last barrier.
__device__ __noinline__ uint32_t gap_tile_runs(const TrainParams &p, const MergeOp &op, const uint32_t *tin,
                                               uint32_t *tout, uint32_t len, const GapHalo &h, uint32_t carry,
                                               uint32_t *stile, uint32_t *dkey, uint32_t *dval, MergeShared &sh,
                                               uint32_t *prev_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    stage_gapped_padded(stile, tin, len, h);
    const uint32_t E = len + h.nnext;
    const uint64_t pos = (uint64_t)kMergeItems * tid;
    const uint32_t valid = staged_valid(stile + padded(kMergeItems * tid), pos, E, op.l, op.r);
    // the full path also when the first position after the tile merges: the
    // pair (last, next) it removes and (last, new) it creates are ours
    const uint32_t upto = len >= pos ? (len - pos + 1 >= 18 ? 0x3FFFFu : (1u << (len - pos + 1)) - 1u) : 0u;
    const bool any = __syncthreads_or((valid & upto) != 0);
    *prev_out = stile[padded(len - 1)];
    uint32_t tile_kept;
    if (!any) {
        emit_plain(p, stile, carry, 0, 0, E, len, tout, tid);
        tile_kept = len - carry;
    } else {
        const uint32_t excl = tile_scan(thread_summary(valid, pos, len), lane, warp, sh.wsum, &sh.tilesum);
        const uint32_t tile = sh.tilesum;
        uint32_t mprev;
        const uint32_t mm = run_flags(valid, excl, carry, &mprev);
        const uint32_t e = carry ? (excl >> 17) : ((excl >> 2) & 0x7FFFu);
        tile_kept = carry ? (tile >> 17) : ((tile >> 2) & 0x7FFFu);
        emit_full(p, stile, dkey, dval, &sh.docc, mm, mprev, e, tile_kept, 0, pos, len, E, op.new_id, tout, tid);
    }
    __syncthreads();
    return tile_kept;
}

// A merge compacts the stream back into full tiles (its output at global
// offsets) when the live symbols fill less than 70% of the tiles in use, so
// the work per merge follows the live symbols, not the tiles.  Both merge
// kernels evaluate this on the same stored values.
__device__ __forceinline__ bool gap_pack(const TrainParams &p, uint32_t k, uint32_t active) {
    const unsigned long long nk = __ldcg(p.nhist + k);
    return nk * 10 < (unsigned long long)active * kMergeTile * 7;
}

// The summary pass, for merges that need it (l == r, or compacting): each
// tile's summary (the transducer over its live symbols); the last CTA scans
// them into each tile's entering merge flag and output offset, the new stream
// length and, for a compacting merge, the new number of tiles in use.
__global__ void __launch_bounds__(kMergeThreads) k_gsum(TrainParams p, uint32_t it) {
    extern __shared__ uint32_t dsm[];
    __shared__ MergeShared sh;
    __shared__ uint32_t s_tilesum;
    MergeOp op;
    if (!merge_op(p, it, &op)) return;
    const uint32_t Ta = __ldcg(&p.st->gactive[op.k & 1]);
    const bool pack = gap_pack(p, op.k, Ta);
    if (op.l != op.r && !pack) return;
    const uint32_t T = p.gtiles, t = blockIdx.x;
    const uint32_t *lin = (op.k & 1) ? p.glen[1] : p.glen[0];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t len = t < Ta ? __ldcg(lin + t) : 0u;
    uint32_t ts = kSumId;
    if (len) {
        __shared__ GapHalo s_h;
        if (tid == 0) gap_halo(op.in, lin, Ta, t, &s_h);
        __syncthreads();
        const GapHalo h = s_h;
        uint32_t *stile = dsm;
        stage_gapped_padded(stile, op.in + (uint64_t)t * kMergeTile, len, h);
        const uint32_t E = len + h.nnext;
        const uint64_t pos = (uint64_t)kMergeItems * tid;
        const uint32_t valid = staged_valid(stile + padded(kMergeItems * tid), pos, E, op.l, op.r);
        tile_scan(thread_summary(valid, pos, len), lane, warp, sh.wsum, &s_tilesum);
        ts = s_tilesum;
    }
    if (tid == 0) p.gsum[t] = ts;
    __threadfence();
    __syncthreads();
    if (tid == 0) sh.last = atomicAdd(&p.st->msum_done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!sh.last) return;
    __threadfence();
    // scan the tile summaries: thread t takes tiles [t*per, (t+1)*per)
    const uint32_t per = (T + kMergeThreads - 1) / kMergeThreads;
    const uint32_t b0 = tid * per < T ? tid * per : T, b1 = b0 + per < T ? b0 + per : T;
    unsigned long long mine = kFId;
    for (uint32_t b = b0; b < b1; b++) mine = lsum_comp(lsum_from_sum(__ldcg(p.gsum + b)), mine);
    const unsigned long long ex = block_excl_lsum(mine, sh);
    uint32_t carry = fapply((uint32_t)ex & 3u, 0u);
    unsigned long long off = (ex >> 2) & 0x7FFFFFFFull;
    for (uint32_t b = b0; b < b1; b++) {
        p.gcarry[b] = carry;
        p.goff[b] = off;
        const uint32_t sb = __ldcg(p.gsum + b);
        off += carry ? (sb >> 17) : ((sb >> 2) & 0x7FFFu);
        carry = fapply(sb & 3u, carry);
    }
    if (b0 < b1 && b1 == T) {
        p.st->n[(op.k + 1) & 1] = off;
        p.nhist[op.k + 1] = off;
        p.st->gactive[(op.k + 1) & 1] = pack ? (uint32_t)((off + kMergeTile - 1) / kMergeTile) : Ta;
    }
    if (tid == 0) p.st->msum_done = 0;
}

// One merge over the gapped tiles: CTA b compacts its contiguous range of
// tiles, each into its twin in the other buffer.  The range's live counts are
// read once; the symbol before a tile carries over from the tile before it,
// and the (up to 3) symbols after it are read with the tile itself.
constexpr int kGapMaxRange = 1024;   // tiles per CTA range (T / grid is far below)

__global__ void __launch_bounds__(kMergeThreads, 4) k_gmerge(TrainParams p, uint32_t it) {
    extern __shared__ uint32_t dsm[];
    uint32_t *sdat = dsm;                         // staged tile (linear) or, for l == r, the padded tile
    uint32_t *sout = dsm + kGapStage;             // l != r: survivors in order
    uint32_t *dkey = dsm + kGapStage + kMergeTile;
    uint32_t *dval = dkey + kDeltaSlots;
    __shared__ MergeShared sh;
    __shared__ GapHalo s_h;
    __shared__ uint32_t s_len[kGapMaxRange + 1];
    MergeOp op;
    if (!merge_op(p, it, &op)) return;
    const uint32_t T = __ldcg(&p.st->gactive[op.k & 1]);   // tiles in use (those after hold nothing)
    const bool pack = gap_pack(p, op.k, T);                 // compacting merge: the summary pass ran
    const bool distinct = op.l != op.r;
    const uint32_t *lin = (op.k & 1) ? p.glen[1] : p.glen[0];
    uint32_t *lout = (op.k & 1) ? p.glen[0] : p.glen[1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0 && tid == 0) {
        if (distinct) {   // every occurrence of (l, r) merges: its count ends at 0
            const uint32_t cnt = (uint32_t)(__ldcg(p.best + op.k) >> 32);
            global_add(table_of(p), pair_key(op.l, op.r), 0u - cnt);
            if (!pack) {   // the stream loses cnt symbols (a compacting merge's pass wrote the length)
                const unsigned long long nn = __ldcg(p.nhist + op.k) - cnt;
                p.st->n[(op.k + 1) & 1] = nn;
                p.nhist[op.k + 1] = nn;
            }
        }
        if (!pack) p.st->gactive[(op.k + 1) & 1] = T;
    }
    // a compacting merge leaves full tiles: the first n' / 4096 hold 4,096 symbols
    const unsigned long long n_new = pack ? __ldcg(p.nhist + op.k + 1) : 0ull;
    uint64_t t0, t1;
    tile_range(T, &t0, &t1);
    if (t0 >= t1) return;
    const uint32_t nt = (uint32_t)(t1 - t0);
    for (uint32_t i = tid; i <= nt; i += kMergeThreads) s_len[i] = (t0 + i < T) ? __ldcg(lin + t0 + i) : 0u;
    if (tid == 0) {
        sh.docc = 0;
        gap_halo(op.in, lin, T, (uint32_t)t0, &s_h);   // the symbol before the range
    }
    if (pack)   // the new live counts of this range's tiles
        for (uint32_t i = tid; i < (uint32_t)(t1 - t0); i += kMergeThreads) {
            const unsigned long long b = (t0 + i) * (unsigned long long)kMergeTile;
            lout[t0 + i] = b >= n_new ? 0u : (n_new - b < kMergeTile ? (uint32_t)(n_new - b) : (uint32_t)kMergeTile);
        }
    for (int j = tid; j < kDeltaSlots; j += kMergeThreads) {
        dkey[j] = kEmptyKey;
        dval[j] = 0;
    }
    __syncthreads();
    uint32_t prev = s_h.prev, has_prev = s_h.has_prev;
    for (uint32_t i = 0; i < nt; i++) {
        const uint32_t t = (uint32_t)t0 + i, len = s_len[i];
        // gapped: into the twin tile; compacting: at the tile's global offset
        uint32_t *tout = op.out + (pack ? __ldcg(p.goff + t) : (uint64_t)t * kMergeTile);
        if (len == 0) {
            if (tid == 0 && !pack) lout[t] = 0;
            continue;
        }
        const uint32_t *tin = op.in + (uint64_t)t * kMergeTile;
        const uint32_t ln = s_len[i + 1];
        uint32_t tile_kept;
        if (distinct) {
            // stage the live symbols exactly (the last quad element by element),
            // while thread 0 writes the symbols around the tile
            constexpr int kQuads = kMergeTile / 4 / kMergeThreads;   // 16-byte loads per thread
            uint4 v[kQuads];
#pragma unroll
            for (int u = 0; u < kQuads; u++) {   // all loads in flight before the first store
                const uint32_t i4 = tid + u * kMergeThreads;
                v[u] = 4 * i4 < len ? __ldcg(reinterpret_cast<const uint4 *>(tin) + i4) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kQuads; u++) {
                const uint32_t i4 = tid + u * kMergeThreads;
                if (4 * i4 + 4 <= len) {
                    *reinterpret_cast<uint4 *>(sdat + 4 + 4 * i4) = v[u];
                } else if (4 * i4 < len) {
                    const uint32_t e4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (uint32_t j = 0; j < 4; j++)
                        if (4 * i4 + j < len) sdat[4 + 4 * i4 + j] = e4[j];
                }
            }
            if (tid == 0) {
                uint32_t nx[3] = {0, 0, 0}, nn = 0;
                if (t + 1 < T && ln >= 3) {   // the next tile holds the three symbols after this one
                    const uint32_t *q = op.in + (uint64_t)(t + 1) * kMergeTile;
                    nx[0] = __ldcg(q);
                    nx[1] = __ldcg(q + 1);
                    nx[2] = __ldcg(q + 2);
                    nn = 3;
                } else {
                    GapHalo w;
                    gap_halo(op.in, lin, T, t, &w);
                    nn = w.nnext;
                    for (int j = 0; j < 3; j++) nx[j] = w.nx[j];
                }
                sdat[3] = prev;
                for (uint32_t j = 0; j < 3; j++) sdat[4 + len + j] = nx[j];
                s_h.nnext = nn;
                s_h.has_prev = has_prev;
            }
            __syncthreads();
            const uint32_t E = len + s_h.nnext;
            const bool hp = s_h.has_prev != 0;
            prev = sdat[4 + len - 1];
            tile_kept = gap_tile_distinct(p, op, sdat, len, E, hp, sout, tout, sh.wsum, dkey, dval, &sh.docc, lane,
                                          warp);
        } else {
            if (tid == 0) {
                GapHalo h;
                h.prev = prev;
                h.has_prev = has_prev;
                if (t + 1 < T && ln >= 3) {
                    const uint32_t *q = op.in + (uint64_t)(t + 1) * kMergeTile;
                    h.nx[0] = __ldcg(q);
                    h.nx[1] = __ldcg(q + 1);
                    h.nx[2] = __ldcg(q + 2);
                    h.nnext = 3;
                } else {
                    GapHalo w;
                    gap_halo(op.in, lin, T, t, &w);
                    h.nnext = w.nnext;
                    for (int j = 0; j < 3; j++) h.nx[j] = w.nx[j];
                }
                s_h = h;
            }
            __syncthreads();
            const GapHalo h = s_h;
            tile_kept = gap_tile_runs(p, op, tin, tout, len, h, __ldcg(p.gcarry + t), sdat, dkey, dval, sh, &prev);
        }
        has_prev = 1;
        if (tid == 0 && !pack) lout[t] = tile_kept;
    }
    __syncthreads();
    flush_deltas(p, dkey, dval, &sh.docc);
}

// Live symbols per tile at the start: the contiguous input.
__global__ void k_ginit(uint32_t *len0, uint32_t T, unsigned long long n) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < T) {
        const unsigned long long b = (unsigned long long)t * kMergeTile;
        len0[t] = n - b < (unsigned long long)kMergeTile ? (uint32_t)(n - b) : (uint32_t)kMergeTile;
    }
}

// Exclusive scan of T u32 counts into u64 offsets by one CTA of 1,024 threads.
__device__ __forceinline__ void exclusive_scan_1024(const uint32_t *len, uint32_t T, unsigned long long *off) {
    __shared__ unsigned long long s_w[32];
    __shared__ unsigned long long s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (uint32_t base = 0; base < T; base += 1024) {
        const uint32_t t = base + tid;
        const unsigned long long v = t < T ? len[t] : 0ull;
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
        if (t < T) off[t] = s_carry + wpre + x - v;
        __syncthreads();
        if (tid == 0) s_carry += tot;
        __syncthreads();
    }
}

// Exclusive scan of the tiles' live counts (one CTA).
__global__ void __launch_bounds__(1024) k_gscan(const uint32_t *len, uint32_t T, unsigned long long *off) {
    __shared__ unsigned long long s_w[32];
    __shared__ unsigned long long s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (uint32_t base = 0; base < T; base += 1024) {
        const uint32_t t = base + tid;
        const unsigned long long v = t < T ? len[t] : 0ull;
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
        if (t < T) off[t] = s_carry + wpre + x - v;
        __syncthreads();
        if (tid == 0) s_carry += tot;
        __syncthreads();
    }
}

// The contiguous stream: tile t's live symbols to out + off[t].
__global__ void k_gcopy(const uint32_t *buf, const uint32_t *len, const unsigned long long *off, uint32_t *out) {
    const uint32_t t = blockIdx.x, l = len[t];
    const uint32_t *src = buf + (uint64_t)t * kMergeTile;
    for (uint32_t i = threadIdx.x; i < l; i += blockDim.x) out[off[t] + i] = src[i];
}

__global__ void k_advance(TrainState *st, uint32_t by) { st->k_base += by; }

// Compaction of the tombstoned stream, in tiles of kCTile positions: live
// counts per tile, their exclusive scan, then each tile's live symbols in
// order.  Without force, all four kernels run only when tombstones exceed a
// quarter of the stream (the same test in each: nothing they read changes
// before k_cdone).
constexpr int kCTile = 4096;
constexpr int kCThreads = 256;
constexpr int kCItems = kCTile / kCThreads;

__device__ __forceinline__ bool compact_now(const TrainState *st, int force) {
    return force || (st->sparse_from != kNoSparse && st->tombs * 4 > st->slen);
}

__global__ void __launch_bounds__(kCThreads) k_ccount(TrainParams p, int force) {
    __shared__ uint32_t s_w[kCThreads / 32];
    const TrainState *st = p.st;
    if (!compact_now(st, force)) return;
    const uint64_t n = st->slen, base = (uint64_t)blockIdx.x * kCTile;
    if (base >= n) return;
    const uint32_t *s = p.buf[st->scur];
    uint32_t c = 0;
    for (int t = threadIdx.x; t < kCTile; t += kCThreads) {
        const uint64_t i = base + t;
        c += (i < n && s[i] != kTomb) ? 1u : 0u;
    }
    c = __reduce_add_sync(kFull, c);
    if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t tot = 0;
        for (int w = 0; w < kCThreads / 32; w++) tot += s_w[w];
        p.ctile[blockIdx.x] = tot;
    }
}

__global__ void __launch_bounds__(1024) k_cscan(TrainParams p, int force) {
    const TrainState *st = p.st;
    if (!compact_now(st, force)) return;
    const uint32_t T = (uint32_t)((st->slen + kCTile - 1) / kCTile);
    exclusive_scan_1024(p.ctile, T, p.coff);
}

// out: the other buffer (then k_cdone switches to it), or the caller's.
__global__ void __launch_bounds__(kCThreads) k_cscatter(TrainParams p, uint32_t *out, int force) {
    __shared__ uint32_t s_w[kCThreads / 32];
    const TrainState *st = p.st;
    if (!compact_now(st, force)) return;
    const uint64_t n = st->slen, base = (uint64_t)blockIdx.x * kCTile;
    if (base >= n) return;
    const uint32_t *s = p.buf[st->scur];
    if (!out) out = p.buf[st->scur ^ 1u];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t v[kCItems];
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < kCItems; e++) {
        const uint64_t i = base + (uint64_t)kCItems * tid + e;
        v[e] = i < n ? s[i] : kTomb;
        c += v[e] != kTomb ? 1u : 0u;
    }
    uint32_t x = c;   // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    uint32_t wpre = 0;
    for (int w = 0; w < warp; w++) wpre += s_w[w];
    uint64_t o = p.coff[blockIdx.x] + wpre + x - c;
#pragma unroll
    for (int e = 0; e < kCItems; e++)
        if (v[e] != kTomb) out[o++] = v[e];
}

__global__ void k_cdone(TrainParams p, int force) {
    TrainState *st = p.st;
    if (!compact_now(st, force)) return;
    st->slen = st->live;
    st->tombs = 0;
    if (!force) st->scur ^= 1u;
}

// Occurrence-driven merges from merge k on; the stream is in buf[k & 1].
__global__ void k_sparse_begin(TrainParams p, uint32_t k) {
    TrainState *st = p.st;
    st->sparse_from = k;
    st->scur = k & 1u;
    st->slen = st->n[k & 1];
    st->live = st->slen;
    st->tombs = 0;
    st->occ_n[0] = st->occ_n[1] = 0;
}

uint32_t ceil_log2(uint64_t x) {
    uint32_t l = 0;
    while ((1ull << l) < x) l++;
    return l;
}

struct Launch {
    TrainParams p;
    unsigned count_grid, merge_grid, argmax_grid;
    size_t count_smem, merge_smem, gmerge_smem, gsum_smem;
    unsigned gmerge_grid;
    int mode;   // BPE_MERGE_TWO_PASS, BPE_MERGE_LOOKBACK or BPE_MERGE_TILES
    unsigned sscan_grid, ctile_grid;   // occurrence-driven merges: scan CTAs, compaction tiles
};

constexpr size_t kGmergeSmem = (size_t)(kGapStage + kMergeTile + 2 * kDeltaSlots) * sizeof(uint32_t);
constexpr size_t kGsumSmem = (size_t)kTileWords * sizeof(uint32_t);

int occupancy(bpe_ctx *ctx, int *count_blocks, int *merge_blocks) {
    const size_t csm = 2 * kCountSlots * sizeof(uint32_t),
                 msm = (kTileWords + 2 * kDeltaSlots) * sizeof(uint32_t);
    BPE_CUDA(ctx, cudaFuncSetAttribute(k_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm),
             "k_count smem attribute");
    BPE_CUDA(ctx, cudaFuncSetAttribute(k_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msm),
             "k_merge smem attribute");
    BPE_CUDA(ctx, cudaFuncSetAttribute(k_mapply, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msm),
             "k_mapply smem attribute");
    BPE_CUDA(ctx, cudaFuncSetAttribute(k_gmerge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGmergeSmem),
             "k_gmerge smem attribute");
    BPE_CUDA(ctx, cudaFuncSetAttribute(k_gsum, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGsumSmem),
             "k_gsum smem attribute");
    BPE_CUDA(ctx, cudaOccupancyMaxActiveBlocksPerMultiprocessor(count_blocks, k_count, kCountThreads, csm),
             "k_count occupancy");
    BPE_CUDA(ctx, cudaOccupancyMaxActiveBlocksPerMultiprocessor(merge_blocks, k_mapply, kMergeThreads, msm),
             "k_mapply occupancy");
    *count_blocks = std::max(*count_blocks, 1);
    *merge_blocks = std::max(*merge_blocks, 1);
    return BPE_OK;
}

void launch_merge(const Launch &L, uint32_t it, cudaStream_t s) {
    if (L.mode == BPE_MERGE_TILES) {
        k_gsum<<<L.p.gtiles, kMergeThreads, L.gsum_smem, s>>>(L.p, it);   // returns at once unless l == r
        k_gmerge<<<L.gmerge_grid, kMergeThreads, L.gmerge_smem, s>>>(L.p, it);
    } else if (L.mode == BPE_MERGE_LOOKBACK) {
        k_merge<<<L.merge_grid, kMergeThreads, L.merge_smem, s>>>(L.p, it);
    } else {
        k_msum<<<L.merge_grid, kMergeThreads, 0, s>>>(L.p, it);
        k_mapply<<<L.merge_grid, kMergeThreads, L.merge_smem, s>>>(L.p, it);
    }
}

void launch_iteration(const Launch &L, uint32_t it, cudaStream_t s) {
    k_argmax<<<L.argmax_grid, kArgmaxThreads, 0, s>>>(L.p, it);
    launch_merge(L, it, s);
}

// Capture (or reuse) a graph of kGraphIters iterations plus the k_base advance.
int get_graph(bpe_ctx *ctx, const Launch &L, cudaGraphExec_t *out) {
    std::vector<uintptr_t> key = {
        (uintptr_t)L.p.buf[0], (uintptr_t)L.p.buf[1], (uintptr_t)L.p.tslot, (uintptr_t)L.p.tmask,
        (uintptr_t)L.p.dkey, (uintptr_t)L.p.dcnt, (uintptr_t)L.p.dcap, (uintptr_t)L.p.status[0],
        (uintptr_t)L.p.status[1], (uintptr_t)L.p.rsum, (uintptr_t)L.p.rpre, (uintptr_t)L.p.best,
        (uintptr_t)L.p.nhist, (uintptr_t)L.p.dhist, (uintptr_t)L.p.st, (uintptr_t)L.merge_grid,
        (uintptr_t)L.argmax_grid, (uintptr_t)L.mode, (uintptr_t)L.p.glen[0], (uintptr_t)L.p.glen[1],
        (uintptr_t)L.p.gsum, (uintptr_t)L.p.gcarry, (uintptr_t)L.p.goff, (uintptr_t)L.p.gtiles,
        (uintptr_t)L.gmerge_grid};
    if (ctx->graph.exec && ctx->graph.key == key) {
        *out = ctx->graph.exec;
        return BPE_OK;
    }
    if (ctx->graph.exec) {
        cudaGraphExecDestroy(ctx->graph.exec);
        ctx->graph.exec = nullptr;
    }
    cudaStream_t cs = ctx->capture_stream;
    BPE_CUDA(ctx, cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal), "begin capture");
    for (uint32_t i = 0; i < kGraphIters; i++) launch_iteration(L, i, cs);
    k_advance<<<1, 1, 0, cs>>>(L.p.st, kGraphIters);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(cs, &g);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "end capture");
    e = cudaGraphInstantiate(&ctx->graph.exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "graph instantiate");
    ctx->graph.key = key;
    *out = ctx->graph.exec;
    return BPE_OK;
}

// Compaction of the tombstoned stream: when due (force 0, into the other
// buffer), or always into out (force 1).
void launch_compaction(const Launch &L, uint32_t *out, int force, cudaStream_t s) {
    k_ccount<<<L.ctile_grid, kCThreads, 0, s>>>(L.p, force);
    k_cscan<<<1, 1024, 0, s>>>(L.p, force);
    k_cscatter<<<L.ctile_grid, kCThreads, 0, s>>>(L.p, out, force);
    k_cdone<<<1, 1, 0, s>>>(L.p, force);
}

// A window compacts after its first k_sargmax has applied the previous
// merge's occurrences (their positions are in the current buffer).
void launch_sparse_iteration(const Launch &L, uint32_t it, bool compact, cudaStream_t s) {
    k_sargmax<<<L.argmax_grid, kArgmaxThreads, 0, s>>>(L.p, it);
    if (compact) launch_compaction(L, nullptr, 0, s);
    k_sscan<<<L.sscan_grid, kSparseThreads, 0, s>>>(L.p, it);
}

// Capture (or reuse) a graph of one occurrence-driven window: kGraphIters
// merges (compaction when due after the first one's apply), the k_base
// advance.
int get_sparse_graph(bpe_ctx *ctx, const Launch &L, cudaGraphExec_t *out) {
    std::vector<uintptr_t> key = {
        (uintptr_t)L.p.buf[0], (uintptr_t)L.p.buf[1], (uintptr_t)L.p.tslot, (uintptr_t)L.p.tmask,
        (uintptr_t)L.p.dkey, (uintptr_t)L.p.dcnt, (uintptr_t)L.p.dcap, (uintptr_t)L.p.best,
        (uintptr_t)L.p.nhist, (uintptr_t)L.p.dhist, (uintptr_t)L.p.st, (uintptr_t)L.p.occ[0],
        (uintptr_t)L.p.occ[1], (uintptr_t)L.p.occ_cap, (uintptr_t)L.p.ctile, (uintptr_t)L.p.coff,
        (uintptr_t)L.sscan_grid, (uintptr_t)L.ctile_grid, (uintptr_t)L.argmax_grid};
    TrainGraph &G = ctx->graph_sparse;
    if (G.exec && G.key == key) {
        *out = G.exec;
        return BPE_OK;
    }
    if (G.exec) {
        cudaGraphExecDestroy(G.exec);
        G.exec = nullptr;
    }
    cudaStream_t cs = ctx->capture_stream;
    BPE_CUDA(ctx, cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal), "begin capture");
    for (uint32_t i = 0; i < kGraphIters; i++) launch_sparse_iteration(L, i, i == 0, cs);
    k_advance<<<1, 1, 0, cs>>>(L.p.st, kGraphIters);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(cs, &g);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "end capture");
    e = cudaGraphInstantiate(&G.exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "graph instantiate");
    G.key = key;
    *out = G.exec;
    return BPE_OK;
}

int train_once(bpe_ctx *ctx, const uint32_t *d_symbols, uint64_t n, uint32_t n_merges, uint32_t table_log2,
               bpe_merge *h_merges_out, uint32_t *n_done, uint32_t *d_symbols_final, uint64_t *n_final,
               bool *table_full) {
    *table_full = false;
    cudaStream_t s = ctx->stream;
    const uint64_t T = 1ull << table_log2;
    const uint64_t ntiles = (n + kMergeTile - 1) / kMergeTile;
    void *buf0, *buf1, *tslot, *dense, *st0, *st1, *best, *state, *nhist, *dhist;
    int rc;
    if ((rc = ensure(ctx, S_TRAIN_BUF0, (n + kPadSymbols) * 4, &buf0)) ||
        (rc = ensure(ctx, S_TRAIN_BUF1, (n + kPadSymbols) * 4, &buf1)) ||
        (rc = ensure(ctx, S_TABLE_KEY, T * 8, &tslot)) || (rc = ensure(ctx, S_TABLE_CNT, T * 8, &dense)) ||
        (rc = ensure(ctx, S_STATUS0, ntiles * 8, &st0)) || (rc = ensure(ctx, S_STATUS1, ntiles * 8, &st1)) ||
        (rc = ensure(ctx, S_BEST, (uint64_t)n_merges * 8, &best)) ||
        (rc = ensure(ctx, S_STATE, sizeof(TrainState), &state)) ||
        (rc = ensure(ctx, S_NHIST, ((uint64_t)n_merges + 1) * 8, &nhist)) ||
        (rc = ensure(ctx, S_LIST0, ((uint64_t)n_merges + 1) * 4, &dhist)))
        return rc;
    int cb, mb;
    if ((rc = occupancy(ctx, &cb, &mb))) return rc;
    // the list loop hands input it cannot take (ids past one byte) to the two-pass loop
    const int mode = ctx->merge_mode == BPE_MERGE_LISTS ? (int)BPE_MERGE_TWO_PASS : ctx->merge_mode;
    const bool lookback = mode == BPE_MERGE_LOOKBACK, gapped = mode == BPE_MERGE_TILES;
    const bool profile = ctx->profile != 0;
    const bool graph = ctx->use_graph && !profile;
    // merge windows replay from CUDA graphs, or (BPE_OPT_PERSISTENT, two-pass
    // merge only) from one persistent cooperative launch per window
    int coop = 0, pb = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, ctx->device);
    const bool persistent = ctx->persistent && graph && mode == BPE_MERGE_TWO_PASS && coop;
    if (persistent) {
        const size_t msm = (kTileWords + 2 * kDeltaSlots) * sizeof(uint32_t);
        BPE_CUDA(ctx, cudaFuncSetAttribute(k_train_loop, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msm),
                 "k_train_loop smem attribute");
        BPE_CUDA(ctx, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pb, k_train_loop, kMergeThreads, msm),
                 "k_train_loop occupancy");
        if (pb < 1) return fail(ctx, BPE_ERR_CUDA, "bpe_train: the persistent merge loop does not fit on an SM");
    }
    // occurrence-driven merges once the best count is rare (1) or from merge 0
    // (2); positions are 32-bit
    const int sparse_mode = ctx->sparse_merge;
    const bool sparse_ok = sparse_mode && mode == BPE_MERGE_TWO_PASS && !persistent && n > 0 &&
                           n + kPadSymbols < 0xFFFFFFFFull;
    void *occ = nullptr;
    uint64_t occ_cap = 0;   // a merge's occurrences never exceed the count that started the mode
    if (sparse_ok) {
        occ_cap = (sparse_mode == 2 ? n / 2 : n / kSparseDiv) + 1;
        if ((rc = ensure(ctx, S_SPARSE_OCC, occ_cap * 16, &occ))) return rc;
    }
    // persistent: every CTA resident (at least one per SM, for the argmax);
    // otherwise one range per CTA, at most as many ranges as tiles
    const uint64_t range_grid =
        persistent ? std::min<uint64_t>((uint64_t)ctx->sm_count * pb, std::max<uint64_t>(ntiles, ctx->sm_count))
                   : std::max<uint64_t>(1, std::min<uint64_t>(ntiles, (uint64_t)ctx->sm_count * mb));
    void *ranges;
    if ((rc = ensure(ctx, S_LIST1, range_grid * 16 + ntiles * 8, &ranges))) return rc;   // ranges, then tile offsets
    uint32_t *dkey = (uint32_t *)dense, *dcnt = dkey + T;   // dense keys, then dense counts
    const uint32_t G = persistent ? kLoopIters : kGraphIters;
    void *pin;
    const size_t pin_bytes = sizeof(TrainState) + 8 * kInFlight + (uint64_t)n_merges * 8 +
                             ((uint64_t)n_merges + 1) * 8 + ((uint64_t)n_merges + 1) * 4;
    if ((rc = ensure_pinned(ctx, pin_bytes, &pin))) return rc;
    TrainState *h_state = (TrainState *)pin;
    unsigned long long *h_poll = (unsigned long long *)(h_state + 1);
    unsigned long long *h_best = h_poll + kInFlight;
    unsigned long long *h_nhist = h_best + n_merges;
    uint32_t *h_dhist = (uint32_t *)(h_nhist + n_merges + 1);

    // Make sure nothing still reads the pinned area from an earlier call.
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "train: stream sync");
    memset(h_state, 0, sizeof *h_state);
    h_state->n_merges = n_merges;
    h_state->n[0] = n;
    h_state->gactive[0] = (uint32_t)ntiles;
    h_state->sparse_from = kNoSparse;
    h_nhist[0] = n;
    BPE_CUDA(ctx, cudaMemcpyAsync(state, h_state, sizeof *h_state, cudaMemcpyHostToDevice, s), "state upload");
    BPE_CUDA(ctx, cudaMemcpyAsync(nhist, h_nhist, 8, cudaMemcpyHostToDevice, s), "nhist upload");
    BPE_CUDA(ctx, cudaMemsetAsync(tslot, 0xFF, T * 8, s), "table clear");
    BPE_CUDA(ctx, cudaMemsetAsync(dcnt, 0, T * 4, s), "count clear");
    BPE_CUDA(ctx, cudaMemsetAsync(st0, 0, ntiles * 8, s), "status clear");
    BPE_CUDA(ctx, cudaMemsetAsync(best, 0, (uint64_t)n_merges * 8, s), "best clear");
    BPE_CUDA(ctx, cudaMemsetAsync(dhist, 0, ((uint64_t)n_merges + 1) * 4, s), "dhist clear");
    BPE_CUDA(ctx, cudaMemcpyAsync(buf0, d_symbols, n * 4, cudaMemcpyDeviceToDevice, s), "input copy");

    Launch L;
    L.mode = mode;
    // gapped tiles: live counts by parity (st0), l == r summaries and flags (st1)
    L.p.glen[0] = (uint32_t *)st0;
    L.p.glen[1] = (uint32_t *)st0 + ntiles;
    L.p.gsum = (uint32_t *)st1;
    L.p.gcarry = (uint32_t *)st1 + ntiles;
    L.p.goff = (unsigned long long *)ranges + 2 * range_grid;
    L.p.gtiles = (uint32_t)ntiles;
    L.gmerge_smem = kGmergeSmem;
    L.gsum_smem = kGsumSmem;
    {   // one range of tiles per CTA, every CTA resident
        int gb = 1;
        BPE_CUDA(ctx, cudaOccupancyMaxActiveBlocksPerMultiprocessor(&gb, k_gmerge, kMergeThreads, kGmergeSmem),
                 "k_gmerge occupancy");
        uint64_t g = std::min<uint64_t>(ntiles, (uint64_t)ctx->sm_count * std::max(gb, 1));
        g = std::max<uint64_t>(g, (ntiles + kGapMaxRange - 1) / kGapMaxRange);
        L.gmerge_grid = (unsigned)std::max<uint64_t>(1, g);
    }
    L.p.rsum = (unsigned long long *)ranges;
    L.p.rpre = L.p.rsum + range_grid;
    L.p.buf[0] = (uint32_t *)buf0;
    L.p.buf[1] = (uint32_t *)buf1;
    L.p.tslot = (unsigned long long *)tslot;
    L.p.tmask = (uint32_t)(T - 1);
    L.p.dkey = dkey;
    L.p.dcnt = dcnt;
    L.p.dcap = (uint32_t)T;
    L.p.status[0] = (unsigned long long *)st0;
    L.p.status[1] = (unsigned long long *)st1;
    L.p.best = (unsigned long long *)best;
    L.p.nhist = (unsigned long long *)nhist;
    L.p.dhist = (uint32_t *)dhist;
    L.p.st = (TrainState *)state;
    L.p.occ[0] = (uint32_t *)occ;
    L.p.occ[1] = occ ? (uint32_t *)occ + 2 * occ_cap : nullptr;
    L.p.occ_cap = (uint32_t)occ_cap;
    L.p.ctile = (uint32_t *)st0;                  // the look-back status words are unused here
    L.p.coff = (unsigned long long *)st1;
    L.sscan_grid = (unsigned)ctx->sm_count * (2048 / kSparseThreads);
    L.ctile_grid = (unsigned)std::max<uint64_t>(1, ntiles);
    const uint64_t count_work = (n + kCountTile - 1) / kCountTile;
    L.count_grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(count_work, (uint64_t)ctx->sm_count * cb));
    // look-back: one tile per CTA (spare CTAs exit); two passes: one range per CTA
    L.merge_grid = lookback ? (unsigned)std::max<uint64_t>(1, ntiles) : (unsigned)range_grid;
    L.argmax_grid = (unsigned)ctx->sm_count * 2;
    L.count_smem = 2 * kCountSlots * sizeof(uint32_t);
    L.merge_smem = (kTileWords + 2 * kDeltaSlots) * sizeof(uint32_t);

    // profile events: 0 before k_count, 1 after it; merge k: 2+2k after argmax, 3+2k after merge
    const size_t n_prof = profile ? 2 + 2 * (size_t)n_merges : 0;
    if ((rc = ensure_events(ctx, n_prof + kInFlight))) return rc;
    std::vector<cudaEvent_t> poll_ev(kInFlight);
    for (int i = 0; i < kInFlight; i++) poll_ev[i] = ctx->events[n_prof + i];

    cudaGraphExec_t exec = nullptr, sexec = nullptr;
    if (graph && !persistent && (rc = get_graph(ctx, L, &exec))) return rc;
    if (graph && sparse_ok && (rc = get_sparse_graph(ctx, L, &sexec))) return rc;
    if (gapped) k_ginit<<<(unsigned)((ntiles + 255) / 256), 256, 0, s>>>(L.p.glen[0], (uint32_t)ntiles, n);
    if (profile) BPE_CUDA(ctx, cudaEventRecord(ctx->events[0], s), "event");
    k_count<<<L.count_grid, kCountThreads, L.count_smem, s>>>(L.p);
    if (profile) BPE_CUDA(ctx, cudaEventRecord(ctx->events[1], s), "event");

    // Launch windows of G merges; keep at most kInFlight windows queued so a
    // stop (a merge with count 0) is noticed without a full drain.
    uint32_t launched = 0;
    uint64_t window = 0, sparse_windows = 0;
    bool stopped = false, sparse_on = false;
    uint32_t k_sparse = 0;   // first occurrence-driven merge
    auto sparse_begin = [&](uint32_t k) {
        k_sparse_begin<<<1, 1, 0, s>>>(L.p, k);
        sparse_on = true;
        k_sparse = k;
    };
    if (sparse_ok && sparse_mode == 2) sparse_begin(0);
    while (launched < n_merges && !stopped) {
        if (window >= (uint64_t)kInFlight) {
            const int slot = (int)(window % kInFlight);
            BPE_CUDA(ctx, cudaEventSynchronize(poll_ev[slot]), "poll sync");
            const uint64_t c = h_poll[slot] >> 32;   // best count of an earlier merge: later ones are no larger
            if (c == 0) stopped = true;
            if (stopped) break;
            if (sparse_ok && !sparse_on && c * kSparseDiv < n) sparse_begin(launched);
        }
        uint32_t end = std::min<uint32_t>(n_merges, launched + G);
        if (sparse_on) {
            ++sparse_windows;
            if (graph) {
                BPE_CUDA(ctx, cudaGraphLaunch(sexec, s), "graph launch");
            } else {
                for (uint32_t k = launched; k < end; k++) {
                    k_sargmax<<<L.argmax_grid, kArgmaxThreads, 0, s>>>(L.p, k);
                    if (k == launched) launch_compaction(L, nullptr, 0, s);
                    if (profile) cudaEventRecord(ctx->events[2 + 2 * (size_t)k], s);
                    k_sscan<<<L.sscan_grid, kSparseThreads, 0, s>>>(L.p, k);
                    if (profile) cudaEventRecord(ctx->events[3 + 2 * (size_t)k], s);
                }
            }
        } else if (persistent) {
            void *args[] = {&L.p, &launched, &end};
            BPE_CUDA(ctx, cudaLaunchCooperativeKernel((const void *)k_train_loop, L.merge_grid, kMergeThreads, args,
                                                      L.merge_smem, s),
                     "persistent merge launch");
        } else if (graph) {
            BPE_CUDA(ctx, cudaGraphLaunch(exec, s), "graph launch");
        } else {
            for (uint32_t k = launched; k < end; k++) {
                k_argmax<<<L.argmax_grid, kArgmaxThreads, 0, s>>>(L.p, k);
                if (profile) cudaEventRecord(ctx->events[2 + 2 * (size_t)k], s);
                launch_merge(L, k, s);
                if (profile) cudaEventRecord(ctx->events[3 + 2 * (size_t)k], s);
            }
        }
        BPE_CUDA(ctx, cudaGetLastError(), "train launch");
        const int slot = (int)(window % kInFlight);
        BPE_CUDA(ctx, cudaMemcpyAsync(h_poll + slot, L.p.best + (end - 1), 8, cudaMemcpyDeviceToHost, s),
                 "poll copy");
        BPE_CUDA(ctx, cudaEventRecord(poll_ev[slot], s), "poll event");
        launched = end;
        window++;
    }
    // the last occurrence-driven merge's occurrences (k_base is launched after
    // the graphs' advances, 0 with host launches)
    if (sparse_on) k_sargmax<<<L.argmax_grid, kArgmaxThreads, 0, s>>>(L.p, graph ? 0u : launched);
    BPE_CUDA(ctx, cudaMemcpyAsync(h_state, state, sizeof *h_state, cudaMemcpyDeviceToHost, s), "state read");
    BPE_CUDA(ctx, cudaMemcpyAsync(h_best, best, (uint64_t)n_merges * 8, cudaMemcpyDeviceToHost, s), "best read");
    BPE_CUDA(ctx, cudaMemcpyAsync(h_nhist, nhist, ((uint64_t)n_merges + 1) * 8, cudaMemcpyDeviceToHost, s),
             "nhist read");
    BPE_CUDA(ctx, cudaMemcpyAsync(h_dhist, dhist, ((uint64_t)n_merges + 1) * 4, cudaMemcpyDeviceToHost, s),
             "dhist read");
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "train sync");

    if (h_state->err & DERR_TABLE_FULL) {
        *table_full = true;
        return fail(ctx, BPE_ERR_TABLE_FULL, "bpe_train: pair table of 2^%u slots overflowed", table_log2);
    }
    if (h_state->err & DERR_TIMEOUT)
        return fail(ctx, BPE_ERR_TIMEOUT, "bpe_train: a look-back or grid-barrier wait gave up");
    if (h_state->err & DERR_OOB)
        return fail(ctx, BPE_ERR_CHECKED_OOB, "bpe_train: a merge's occurrences overflowed their list");
    uint32_t done = 0;
    while (done < n_merges && (h_best[done] >> 32) != 0) done++;
    for (uint32_t k = 0; k < done; k++) {
        const uint32_t key = ~(uint32_t)h_best[k];
        h_merges_out[k].left = key >> 16;
        h_merges_out[k].right = key & 0xFFFFu;
        h_merges_out[k].new_id = 256u + k;
        h_merges_out[k].count = (uint32_t)(h_best[k] >> 32);
    }
    *n_done = done;
    const uint64_t nf = h_nhist[done];
    if (n_final) *n_final = nf;
    const bool sparse_final = sparse_on && done > k_sparse;   // the stream holds tombstones
    if (d_symbols_final) {
        if (sparse_final) {
            launch_compaction(L, d_symbols_final, 1, s);
            BPE_CUDA(ctx, cudaGetLastError(), "compaction launch");
        } else if (gapped) {   // gather the tiles' live symbols
            void *goff;
            if ((rc = ensure(ctx, S_W_OUTOFF, ntiles * 8, &goff))) return rc;
            k_gscan<<<1, 1024, 0, s>>>(L.p.glen[done & 1], (uint32_t)ntiles, (unsigned long long *)goff);
            k_gcopy<<<(unsigned)ntiles, 256, 0, s>>>(L.p.buf[done & 1], L.p.glen[done & 1],
                                                      (const unsigned long long *)goff, d_symbols_final);
            BPE_CUDA(ctx, cudaGetLastError(), "gather launch");
        } else {
            BPE_CUDA(ctx, cudaMemcpyAsync(d_symbols_final, L.p.buf[done & 1], nf * 4, cudaMemcpyDeviceToDevice, s),
                     "final copy");
        }
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "final sync");
    }

    // statistics: algorithmic bytes per kernel family and (profiled) device time
    stats_reset(ctx);
    const uint64_t per_merge = lookback ? 2 : 3;
    const uint64_t full_windows = window - sparse_windows;
    const uint32_t full_merges = sparse_on ? std::min(k_sparse, launched) : launched;
    ctx->stats.kernel_launches =
        1 + (gapped ? 1 : 0) + (d_symbols_final && gapped ? 2 : 0) +
        (persistent ? (uint64_t)window
                    : graph ? full_windows * (per_merge * kGraphIters + 1) : per_merge * full_merges) +
        (sparse_on ? 2 + sparse_windows * 4 + (graph ? sparse_windows * (2 * kGraphIters + 1)
                                                      : 2 * (uint64_t)(launched - full_merges)) +
                         (sparse_final && d_symbols_final ? 4 : 0)
                   : 0);
    const int sc = stats_slot(ctx, "pair_count"), sa = stats_slot(ctx, "argmax"), sm = stats_slot(ctx, "merge_compact");
    const int ss = sparse_on ? stats_slot(ctx, "merge_scan") : sm;   // occurrence-driven merges: the scan
    ctx->stats.k[sc].launches = 1;
    ctx->stats.k[sc].bytes = 4.0 * (double)n;
    const uint32_t ran = std::min<uint32_t>(n_merges, done + 1);   // the argmax that found 0 ran too
    for (uint32_t k = 1; k < ran; k++) {
        ctx->stats.k[sa].launches++;
        ctx->stats.k[sa].bytes += 8.0 * (double)h_dhist[k];
    }
    for (uint32_t k = 0; k < done; k++) {
        // an occurrence-driven merge reads the live stream once (its few writes aside)
        const bool sp = sparse_on && k >= k_sparse;
        ctx->stats.k[sp ? ss : sm].launches++;
        ctx->stats.k[sp ? ss : sm].bytes += sp ? 4.0 * (double)h_nhist[k] : 4.0 * (double)h_nhist[k] + 4.0 * (double)h_nhist[k + 1];
    }
    if (profile) {
        float x = 0;
        if (cudaEventElapsedTime(&x, ctx->events[0], ctx->events[1]) == cudaSuccess) ctx->stats.k[sc].ms = x;
        for (uint32_t k = 0; k < launched; k++) {
            float a = 0, b = 0;
            cudaEvent_t before = ctx->events[k ? 3 + 2 * (size_t)(k - 1) : 1];
            if (k >= 1 && k < ran && cudaEventElapsedTime(&a, before, ctx->events[2 + 2 * (size_t)k]) == cudaSuccess)
                ctx->stats.k[sa].ms += a;
            if (k < done &&
                cudaEventElapsedTime(&b, ctx->events[2 + 2 * (size_t)k], ctx->events[3 + 2 * (size_t)k]) == cudaSuccess)
                ctx->stats.k[sparse_on && k >= k_sparse ? ss : sm].ms += b;
        }
        cudaGetLastError();
    }
    return BPE_OK;
}

// ----------------------------------------------- word-frequency training ---
//
// No pair is counted across a WORD_START and no merge crosses one, so the
// stream is a sequence of words (a word starts at index 0 and at every
// WORD_START symbol) and the merge loop can run over the distinct words,
// each weighted by its number of occurrences: the pair counts, the argmax,
// the merges and -- expanded back over the occurrences -- the final stream
// are exactly those of the full-stream loop.
//
//   k_wstarts_count / k_scan_top / k_wstarts_write   word start positions
//   k_whash / k_wverify     distinct words through a hash table of 64-bit
//                           content hashes; a verification pass compares
//                           every occurrence with its representative, a
//                           collision makes the host retry with a new seed
//   k_wassign / k_wgather   one compact copy of each distinct word
//   k_wcount                initial weighted pair counts (+ argmax of merge 0)
//   k_wmerge                per merge: every word holding the pair is merged
//                           left to right in place by one thread, and its
//                           pairs before and after go as -freq / +freq deltas
//                           into the count table (k_argmax finds the next pair)
//   k_wexpand               the final stream from the occurrences

constexpr int kWThreads = 256;
constexpr int kWItems = 16;
constexpr int kWBlock = kWThreads * kWItems;   // positions per scan block
constexpr uint32_t kWErrCollision = 8u;

struct WSlot {
    unsigned long long key;   // content hash | 1; 0 = empty
    uint32_t freq;
    uint32_t rep_inv;         // ~(first occurrence)
};

struct WordParams {
    const uint32_t *sym;      // the input stream
    uint64_t n;
    uint32_t *wstart;         // word starts, n_occ + 1 entries
    uint32_t *occ_slot;       // table slot of each occurrence
    WSlot *table;
    uint32_t tmask;
    uint32_t *uid;            // per table slot: distinct word id
    uint32_t *urep, *ufreq, *ulen, *uoff;   // per distinct word
    uint32_t *wsym;           // compact words
    uint32_t *bsum;           // scan block sums
    uint32_t *counter;        // [0] = n_occ, [1] = n_uniq, [2] = err, [3] = total of the last scan
};

// Block-wide exclusive scan of one value per thread (kWThreads threads).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *s_w, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t incl = warp_incl_sum(v, lane);
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    uint32_t pre = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWThreads / 32; w++) {
        const uint32_t x = s_w[w];
        pre += (w < warp) ? x : 0u;
        tot += x;
    }
    __syncthreads();
    *total = tot;
    return pre + incl - v;
}

__device__ __forceinline__ bool is_word_start(const uint32_t *sym, uint64_t i) { return i == 0 || (sym[i] & kWordStart); }

__global__ void __launch_bounds__(kWThreads) k_wstarts_count(WordParams W) {
    __shared__ uint32_t s_w[kWThreads / 32];
    const uint64_t base = (uint64_t)blockIdx.x * kWBlock + (uint64_t)threadIdx.x * kWItems;
    uint32_t c = 0;
    for (int j = 0; j < kWItems; j++)
        if (base + j < W.n && is_word_start(W.sym, base + j)) ++c;
    uint32_t tot;
    block_excl_scan(c, s_w, &tot);
    if (threadIdx.x == 0) W.bsum[blockIdx.x] = tot;
}

// Exclusive scan of nb block sums in place by one CTA; total -> *total.
__global__ void __launch_bounds__(1024) k_scan_top(uint32_t *bsum, uint32_t nb, uint32_t *total) {
    __shared__ uint32_t s_w[32];
    __shared__ uint32_t s_carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (uint32_t b0 = 0; b0 < nb; b0 += 1024) {
        const uint32_t i = b0 + threadIdx.x;
        const uint32_t v = i < nb ? bsum[i] : 0u;
        const uint32_t incl = warp_incl_sum(v, lane);
        if (lane == 31) s_w[warp] = incl;
        __syncthreads();
        uint32_t pre = 0, tot = 0;
        for (int w = 0; w < 32; w++) {
            pre += (w < warp) ? s_w[w] : 0u;
            tot += s_w[w];
        }
        const uint32_t carry = s_carry;
        if (i < nb) bsum[i] = carry + pre + incl - v;
        __syncthreads();
        if (threadIdx.x == 0) s_carry = carry + tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) *total = s_carry;
}

__global__ void __launch_bounds__(kWThreads) k_wstarts_write(WordParams W, uint32_t n_occ) {
    __shared__ uint32_t s_w[kWThreads / 32];
    const uint64_t base = (uint64_t)blockIdx.x * kWBlock + (uint64_t)threadIdx.x * kWItems;
    uint32_t c = 0;
    for (int j = 0; j < kWItems; j++)
        if (base + j < W.n && is_word_start(W.sym, base + j)) ++c;
    uint32_t tot;
    uint32_t o = W.bsum[blockIdx.x] + block_excl_scan(c, s_w, &tot);
    for (int j = 0; j < kWItems; j++)
        if (base + j < W.n && is_word_start(W.sym, base + j)) W.wstart[o++] = (uint32_t)(base + j);
    if (blockIdx.x == 0 && threadIdx.x == 0) W.wstart[n_occ] = (uint32_t)W.n;
}

__device__ __forceinline__ unsigned long long word_hash(const uint32_t *w, uint32_t len, unsigned long long seed) {
    unsigned long long h = seed ^ (0x9E3779B97F4A7C15ull * (len + 1));
    for (uint32_t i = 0; i < len; i++) {
        h ^= w[i];
        h *= 0x100000001B3ull;
        h ^= h >> 29;
    }
    h ^= h >> 33;       // a 64-bit finaliser (splitmix64's)
    h *= 0xFF51AFD7ED558CCDull;
    h ^= h >> 33;
    h *= 0xC4CEB9FE1A85EC53ull;
    h ^= h >> 33;
    return h | 1ull;
}

__global__ void k_whash(WordParams W, uint32_t n_occ, unsigned long long seed) {
    const uint32_t o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= n_occ) return;
    const uint32_t a = W.wstart[o], b = W.wstart[o + 1];
    const unsigned long long h = word_hash(W.sym + a, b - a, seed);
    uint32_t s = (uint32_t)(h >> 20) & W.tmask;
    for (uint32_t probe = 1; probe <= 256; ++probe) {
        const unsigned long long cur = atomicCAS(&W.table[s].key, 0ull, h);
        if (cur == 0ull || cur == h) {
            atomicAdd(&W.table[s].freq, 1u);
            atomicMax(&W.table[s].rep_inv, ~o);
            W.occ_slot[o] = s;
            return;
        }
        s = (s + probe) & W.tmask;
    }
    atomicOr(&W.counter[2], DERR_TABLE_FULL);
    W.occ_slot[o] = 0;
}

__global__ void k_wverify(WordParams W, uint32_t n_occ) {
    const uint32_t o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= n_occ) return;
    const uint32_t rep = ~W.table[W.occ_slot[o]].rep_inv;
    if (rep == o) return;
    const uint32_t a = W.wstart[o], len = W.wstart[o + 1] - a;
    const uint32_t ra = W.wstart[rep], rlen = W.wstart[rep + 1] - ra;
    bool same = (len == rlen);
    for (uint32_t i = 0; same && i < len; i++) same = (W.sym[a + i] == W.sym[ra + i]);
    if (!same) atomicOr(&W.counter[2], kWErrCollision);
}

__global__ void k_wassign(WordParams W, uint32_t tsize) {
    for (uint32_t s = blockIdx.x * blockDim.x + threadIdx.x; s < tsize; s += gridDim.x * blockDim.x) {
        const WSlot e = W.table[s];
        if (e.key == 0ull) continue;
        const uint32_t u = atomicAdd(&W.counter[1], 1u);
        const uint32_t rep = ~e.rep_inv;
        W.uid[s] = u;
        W.urep[u] = rep;
        W.ufreq[u] = e.freq;
        W.ulen[u] = W.wstart[rep + 1] - W.wstart[rep];
    }
}

// exclusive scan of len[0..n) into off (block part; k_scan_top completes it)
__global__ void __launch_bounds__(kWThreads) k_lens_partial(const uint32_t *len, uint32_t n, uint32_t *bsum) {
    __shared__ uint32_t s_w[kWThreads / 32];
    const uint64_t base = (uint64_t)blockIdx.x * kWBlock + (uint64_t)threadIdx.x * kWItems;
    uint32_t c = 0;
    for (int j = 0; j < kWItems; j++)
        if (base + j < n) c += len[base + j];
    uint32_t tot;
    block_excl_scan(c, s_w, &tot);
    if (threadIdx.x == 0) bsum[blockIdx.x] = tot;
}
__global__ void __launch_bounds__(kWThreads) k_lens_final(const uint32_t *len, uint32_t n, const uint32_t *bsum,
                                                          uint32_t *off) {
    __shared__ uint32_t s_w[kWThreads / 32];
    const uint64_t base = (uint64_t)blockIdx.x * kWBlock + (uint64_t)threadIdx.x * kWItems;
    uint32_t c = 0;
    for (int j = 0; j < kWItems; j++)
        if (base + j < n) c += len[base + j];
    uint32_t tot;
    uint32_t o = bsum[blockIdx.x] + block_excl_scan(c, s_w, &tot);
    for (int j = 0; j < kWItems; j++)
        if (base + j < n) {
            off[base + j] = o;
            o += len[base + j];
        }
}

__global__ void k_wgather(WordParams W, uint32_t U) {
    const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= U) return;
    const uint32_t a = W.wstart[W.urep[u]], len = W.ulen[u], o = W.uoff[u];
    for (uint32_t i = 0; i < len; i++) W.wsym[o + i] = W.sym[a + i];
}

// Per-thread word loop with a shared delta table flushed at the end.
template <bool COUNT>
__device__ __forceinline__ void word_deltas(const TrainParams &p, const WordParams &W, uint32_t U, uint32_t k,
                                            uint32_t l, uint32_t r, uint32_t new_id, uint32_t *dkey, uint32_t *dval,
                                            uint32_t *s_docc, unsigned long long &mybest) {
    const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
    auto add = [&](uint32_t kk, uint32_t d) {
        if (smem_add<kDeltaSlots>(dkey, dval, s_docc, kk, d)) {
            const uint32_t tot = global_add(table_of(p), kk, d);
            if (COUNT) {
                const unsigned long long b = pack_best(tot, kk);
                mybest = b > mybest ? b : mybest;
            }
        }
    };
    if (u < U) {
        uint32_t *w = W.wsym + W.uoff[u];
        const uint32_t len = W.ulen[u], f = W.ufreq[u];
        if (COUNT) {
            for (uint32_t i = 0; i + 1 < len; i++) add(pair_key(w[i], w[i + 1]), f);
        } else if (len >= 2) {
            bool hit = false;
            for (uint32_t i = 0; i + 1 < len && !hit; i++)
                hit = (w[i] & 0xFFFFu) == l && (w[i + 1] & 0xFFFFu) == r;
            if (hit) {
                const uint32_t neg = 0u - f;
                for (uint32_t i = 0; i + 1 < len; i++) add(pair_key(w[i], w[i + 1]), neg);
                uint32_t o = 0;   // left to right, non-overlapping, in place (o <= i)
                for (uint32_t i = 0; i < len;) {
                    if (i + 1 < len && (w[i] & 0xFFFFu) == l && (w[i + 1] & 0xFFFFu) == r) {
                        w[o++] = new_id | (w[i] & kWordStart);
                        i += 2;
                    } else {
                        w[o++] = w[i++];
                    }
                }
                W.ulen[u] = o;
                for (uint32_t i = 0; i + 1 < o; i++) add(pair_key(w[i], w[i + 1]), f);
            }
        }
    }
    __syncthreads();
    if (*s_docc) {
        for (int j = threadIdx.x; j < kDeltaSlots; j += blockDim.x) {
            const uint32_t kk = dkey[j];
            if (kk != kEmptyKey && dval[j]) {
                const uint32_t tot = global_add(table_of(p), kk, dval[j]);
                if (COUNT) {
                    const unsigned long long b = pack_best(tot, kk);
                    mybest = b > mybest ? b : mybest;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kWThreads) k_wcount(TrainParams p, WordParams W) {
    __shared__ uint32_t dkey[kDeltaSlots], dval[kDeltaSlots], s_docc;
    __shared__ unsigned long long sbest[kWThreads / 32];
    for (int j = threadIdx.x; j < kDeltaSlots; j += blockDim.x) {
        dkey[j] = kEmptyKey;
        dval[j] = 0;
    }
    if (threadIdx.x == 0) s_docc = 0;
    __syncthreads();
    unsigned long long mybest = 0;
    word_deltas<true>(p, W, W.counter[1], 0, 0, 0, 0, dkey, dval, &s_docc, mybest);
    mybest = warp_max_u64(mybest);
    if ((threadIdx.x & 31) == 0) sbest[threadIdx.x >> 5] = mybest;
    __syncthreads();
    if (threadIdx.x < 32) {
        unsigned long long b = threadIdx.x < kWThreads / 32 ? sbest[threadIdx.x] : 0ull;
        b = warp_max_u64(b);
        if (threadIdx.x == 0 && b) atomicMax(p.best, b);
    }
}

__global__ void __launch_bounds__(kWThreads) k_wmerge(TrainParams p, WordParams W, uint32_t it) {
    __shared__ uint32_t dkey[kDeltaSlots], dval[kDeltaSlots], s_docc;
    TrainState *st = p.st;
    const uint32_t k = st->k_base + it;
    if (k >= st->n_merges || st->err) return;
    const unsigned long long bw = p.best[k];
    if ((bw >> 32) == 0) return;   // training has stopped
    const uint32_t key = ~(uint32_t)bw;
    for (int j = threadIdx.x; j < kDeltaSlots; j += blockDim.x) {
        dkey[j] = kEmptyKey;
        dval[j] = 0;
    }
    if (threadIdx.x == 0) s_docc = 0;
    __syncthreads();
    unsigned long long unused = 0;
    word_deltas<false>(p, W, W.counter[1], k, key >> 16, key & 0xFFFFu, 256u + k, dkey, dval, &s_docc, unused);
}

// final stream: occurrence o's word, at its scanned offset
__global__ void k_occ_len(WordParams W, uint32_t n_occ, uint32_t *olen) {
    const uint32_t o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o < n_occ) olen[o] = W.ulen[W.uid[W.occ_slot[o]]];
}
__global__ void k_wexpand(WordParams W, uint32_t n_occ, const uint32_t *ooff, uint32_t *out) {
    const uint32_t o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= n_occ) return;
    const uint32_t u = W.uid[W.occ_slot[o]];
    const uint32_t *w = W.wsym + W.uoff[u];
    const uint32_t len = W.ulen[u], at = ooff[o];
    for (uint32_t i = 0; i < len; i++) out[at + i] = w[i];
}

// exclusive scan of a device u32 array (n <= 2^30) into off; returns the total
int scan_u32(bpe_ctx *ctx, const uint32_t *len, uint32_t n, uint32_t *off, uint32_t *bsum, uint32_t *d_total,
             uint32_t *h_total) {
    cudaStream_t s = ctx->stream;
    const uint32_t nb = (n + kWBlock - 1) / kWBlock;
    if (nb == 0) {
        *h_total = 0;
        return BPE_OK;
    }
    k_lens_partial<<<nb, kWThreads, 0, s>>>(len, n, bsum);
    k_scan_top<<<1, 1024, 0, s>>>(bsum, nb, d_total);
    k_lens_final<<<nb, kWThreads, 0, s>>>(len, n, bsum, off);
    BPE_CUDA(ctx, cudaMemcpyAsync(h_total, d_total, 4, cudaMemcpyDeviceToHost, s), "scan total");
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "scan sync");
    return BPE_OK;
}

int train_words_once(bpe_ctx *ctx, const uint32_t *d_symbols, uint64_t n, uint32_t n_merges, uint32_t table_log2,
                     bpe_merge *h_merges_out, uint32_t *n_done, uint32_t *d_symbols_final, uint64_t *n_final,
                     bool *table_full) {
    *table_full = false;
    cudaStream_t s = ctx->stream;
    int rc;
    void *bsum, *wstart, *occ_slot, *table, *uidv, *uinfo, *wsym, *state, *best, *tslot, *dense, *dhist, *cnt;
    const uint32_t nb = (uint32_t)((n + kWBlock - 1) / kWBlock);
    if ((rc = ensure(ctx, S_W_BSUM, ((uint64_t)nb + 1024) * 4 + 64, &bsum)) ||
        (rc = ensure(ctx, S_STATE, sizeof(TrainState) + 64, &state)))
        return rc;
    cnt = (uint32_t *)bsum + nb + 1024;   // 4 counters
    void *pin;
    const size_t pin_bytes = sizeof(TrainState) + 64 + 8 * kInFlight + (uint64_t)n_merges * 8 + ((uint64_t)n_merges + 1) * 4;
    if ((rc = ensure_pinned(ctx, pin_bytes, &pin))) return rc;
    uint32_t *h_cnt = (uint32_t *)pin;                     // 16 words
    TrainState *h_state = (TrainState *)(h_cnt + 16);
    unsigned long long *h_poll = (unsigned long long *)(h_state + 1);
    unsigned long long *h_best = h_poll + kInFlight;
    uint32_t *h_dhist = (uint32_t *)(h_best + n_merges);
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "train: stream sync");

    WordParams W{};
    W.sym = d_symbols;
    W.n = n;
    W.bsum = (uint32_t *)bsum;
    W.counter = (uint32_t *)cnt;
    BPE_CUDA(ctx, cudaMemsetAsync(cnt, 0, 16, s), "counters");
    // 1. word starts
    k_wstarts_count<<<nb, kWThreads, 0, s>>>(W);
    k_scan_top<<<1, 1024, 0, s>>>(W.bsum, nb, W.counter);
    BPE_CUDA(ctx, cudaMemcpyAsync(h_cnt, cnt, 16, cudaMemcpyDeviceToHost, s), "count read");
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "word count sync");
    const uint32_t n_occ = h_cnt[0];
    if ((rc = ensure(ctx, S_W_START, ((uint64_t)n_occ + 1) * 4, &wstart)) ||
        (rc = ensure(ctx, S_W_OCCSLOT, (uint64_t)n_occ * 4 + 4, &occ_slot)))
        return rc;
    W.wstart = (uint32_t *)wstart;
    W.occ_slot = (uint32_t *)occ_slot;
    k_wstarts_write<<<nb, kWThreads, 0, s>>>(W, n_occ);
    // 2. distinct words (retry on a hash collision or a full table)
    uint32_t tlog = 16;
    while ((1u << tlog) < 2u * std::min<uint32_t>(n_occ, 1u << 26) && tlog < 27) tlog++;
    uint32_t U = 0;
    for (int attempt = 0;; attempt++) {
        const uint64_t tsize = 1ull << tlog;
        if ((rc = ensure(ctx, S_W_TABLE, tsize * sizeof(WSlot), &table)) ||
            (rc = ensure(ctx, S_W_UID, tsize * 4, &uidv)))
            return rc;
        W.table = (WSlot *)table;
        W.tmask = (uint32_t)(tsize - 1);
        W.uid = (uint32_t *)uidv;
        BPE_CUDA(ctx, cudaMemsetAsync(table, 0, tsize * sizeof(WSlot), s), "word table clear");
        BPE_CUDA(ctx, cudaMemsetAsync(cnt, 0, 16, s), "counters");
        const unsigned long long seed = 0x243F6A8885A308D3ull * (attempt + 1);
        const uint32_t gb = (n_occ + 255) / 256;
        if (gb) {
            k_whash<<<gb, 256, 0, s>>>(W, n_occ, seed);
            k_wverify<<<gb, 256, 0, s>>>(W, n_occ);
        }
        BPE_CUDA(ctx, cudaMemcpyAsync(h_cnt, cnt, 16, cudaMemcpyDeviceToHost, s), "count read");
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "word hash sync");
        if (h_cnt[2] == 0) break;
        if (attempt >= 4) return fail(ctx, BPE_ERR_TABLE_FULL, "bpe_train: distinct-word table failed");
        if (h_cnt[2] & DERR_TABLE_FULL) tlog = std::min<uint32_t>(tlog + 2, 28);
    }
    {
        const uint64_t tsize = 1ull << tlog;
        const uint32_t Umax = std::min<uint32_t>(n_occ, (uint32_t)tsize);
        if ((rc = ensure(ctx, S_W_UINFO, ((uint64_t)Umax + 1) * 16, &uinfo))) return rc;
        W.urep = (uint32_t *)uinfo;
        W.ufreq = W.urep + Umax + 1;
        W.ulen = W.ufreq + Umax + 1;
        W.uoff = W.ulen + Umax + 1;
        k_wassign<<<std::max<uint32_t>(1, std::min<uint64_t>(tsize / 256, 4096)), 256, 0, s>>>(W, (uint32_t)tsize);
        BPE_CUDA(ctx, cudaMemcpyAsync(h_cnt, cnt, 16, cudaMemcpyDeviceToHost, s), "count read");
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "assign sync");
        U = h_cnt[1];
    }
    uint32_t usym = 0;
    if ((rc = scan_u32(ctx, W.ulen, U, W.uoff, W.bsum, W.counter + 3, &usym))) return rc;
    if ((rc = ensure(ctx, S_W_SYM, (uint64_t)usym * 4 + 16, &wsym))) return rc;
    W.wsym = (uint32_t *)wsym;
    if (U) k_wgather<<<(U + 255) / 256, 256, 0, s>>>(W, U);

    // 3. the merge loop over distinct words
    const uint64_t T = 1ull << table_log2;
    if ((rc = ensure(ctx, S_TABLE_KEY, T * 8, &tslot)) || (rc = ensure(ctx, S_TABLE_CNT, T * 8, &dense)) ||
        (rc = ensure(ctx, S_BEST, (uint64_t)n_merges * 8, &best)) ||
        (rc = ensure(ctx, S_LIST0, ((uint64_t)n_merges + 1) * 4, &dhist)))
        return rc;
    uint32_t *dkey = (uint32_t *)dense, *dcnt = dkey + T;
    memset(h_state, 0, sizeof *h_state);
    h_state->n_merges = n_merges;
    BPE_CUDA(ctx, cudaMemcpyAsync(state, h_state, sizeof *h_state, cudaMemcpyHostToDevice, s), "state upload");
    BPE_CUDA(ctx, cudaMemsetAsync(tslot, 0xFF, T * 8, s), "table clear");
    BPE_CUDA(ctx, cudaMemsetAsync(dcnt, 0, T * 4, s), "count clear");
    BPE_CUDA(ctx, cudaMemsetAsync(best, 0, (uint64_t)n_merges * 8, s), "best clear");
    BPE_CUDA(ctx, cudaMemsetAsync(dhist, 0, ((uint64_t)n_merges + 1) * 4, s), "dhist clear");
    TrainParams P{};
    P.tslot = (unsigned long long *)tslot;
    P.tmask = (uint32_t)(T - 1);
    P.dkey = dkey;
    P.dcnt = dcnt;
    P.dcap = (uint32_t)T;
    P.best = (unsigned long long *)best;
    P.dhist = (uint32_t *)dhist;
    P.st = (TrainState *)state;
    const unsigned wgrid = std::max<uint32_t>(1, (U + kWThreads - 1) / kWThreads);
    const unsigned agrid = (unsigned)ctx->sm_count * 2;
    const bool profile = ctx->profile != 0;
    const bool graph = ctx->use_graph && !profile;
    const size_t n_prof = profile ? 2 + 2 * (size_t)n_merges : 0;
    if ((rc = ensure_events(ctx, n_prof + kInFlight))) return rc;
    std::vector<cudaEvent_t> poll_ev(kInFlight);
    for (int i = 0; i < kInFlight; i++) poll_ev[i] = ctx->events[n_prof + i];

    cudaGraphExec_t exec = nullptr;
    if (graph) {
        std::vector<uintptr_t> key = {0x57u /* word loop */, (uintptr_t)P.tslot, (uintptr_t)P.tmask, (uintptr_t)P.dkey,
                                      (uintptr_t)P.dcnt, (uintptr_t)P.best, (uintptr_t)P.dhist, (uintptr_t)P.st,
                                      (uintptr_t)W.wsym, (uintptr_t)W.ulen, (uintptr_t)W.counter, wgrid, agrid};
        if (!(ctx->graph.exec && ctx->graph.key == key)) {
            if (ctx->graph.exec) cudaGraphExecDestroy(ctx->graph.exec);
            ctx->graph.exec = nullptr;
            cudaStream_t cs = ctx->capture_stream;
            BPE_CUDA(ctx, cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal), "begin capture");
            for (uint32_t i = 0; i < kGraphIters; i++) {
                k_argmax<<<agrid, kArgmaxThreads, 0, cs>>>(P, i);
                k_wmerge<<<wgrid, kWThreads, 0, cs>>>(P, W, i);
            }
            k_advance<<<1, 1, 0, cs>>>(P.st, kGraphIters);
            cudaGraph_t g = nullptr;
            cudaError_t e = cudaStreamEndCapture(cs, &g);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "end capture");
            e = cudaGraphInstantiate(&ctx->graph.exec, g, 0);
            cudaGraphDestroy(g);
            if (e != cudaSuccess) return cuda_fail(ctx, e, "graph instantiate");
            ctx->graph.key = key;
        }
        exec = ctx->graph.exec;
    }
    if (profile) BPE_CUDA(ctx, cudaEventRecord(ctx->events[0], s), "event");
    k_wcount<<<wgrid, kWThreads, 0, s>>>(P, W);
    if (profile) BPE_CUDA(ctx, cudaEventRecord(ctx->events[1], s), "event");
    uint32_t launched = 0;
    uint64_t window = 0;
    bool stopped = false;
    while (launched < n_merges && !stopped) {
        if (window >= (uint64_t)kInFlight) {
            const int slot = (int)(window % kInFlight);
            BPE_CUDA(ctx, cudaEventSynchronize(poll_ev[slot]), "poll sync");
            if ((h_poll[slot] >> 32) == 0) stopped = true;
            if (stopped) break;
        }
        const uint32_t end = std::min<uint32_t>(n_merges, launched + kGraphIters);
        if (graph) {
            BPE_CUDA(ctx, cudaGraphLaunch(exec, s), "graph launch");
        } else {
            for (uint32_t k = launched; k < end; k++) {
                k_argmax<<<agrid, kArgmaxThreads, 0, s>>>(P, k);
                if (profile) cudaEventRecord(ctx->events[2 + 2 * (size_t)k], s);
                k_wmerge<<<wgrid, kWThreads, 0, s>>>(P, W, k);
                if (profile) cudaEventRecord(ctx->events[3 + 2 * (size_t)k], s);
            }
        }
        BPE_CUDA(ctx, cudaGetLastError(), "train launch");
        const int slot = (int)(window % kInFlight);
        BPE_CUDA(ctx, cudaMemcpyAsync(h_poll + slot, P.best + (end - 1), 8, cudaMemcpyDeviceToHost, s), "poll copy");
        BPE_CUDA(ctx, cudaEventRecord(poll_ev[slot], s), "poll event");
        launched = end;
        window++;
    }
    BPE_CUDA(ctx, cudaMemcpyAsync(h_state, state, sizeof *h_state, cudaMemcpyDeviceToHost, s), "state read");
    BPE_CUDA(ctx, cudaMemcpyAsync(h_best, best, (uint64_t)n_merges * 8, cudaMemcpyDeviceToHost, s), "best read");
    BPE_CUDA(ctx, cudaMemcpyAsync(h_dhist, dhist, ((uint64_t)n_merges + 1) * 4, cudaMemcpyDeviceToHost, s),
             "dhist read");
    BPE_CUDA(ctx, cudaStreamSynchronize(s), "train sync");
    if (h_state->err & DERR_TABLE_FULL) {
        *table_full = true;
        return fail(ctx, BPE_ERR_TABLE_FULL, "bpe_train: pair table of 2^%u slots overflowed", table_log2);
    }
    uint32_t done = 0;
    while (done < n_merges && (h_best[done] >> 32) != 0) done++;
    for (uint32_t k = 0; k < done; k++) {
        const uint32_t key = ~(uint32_t)h_best[k];
        h_merges_out[k].left = key >> 16;
        h_merges_out[k].right = key & 0xFFFFu;
        h_merges_out[k].new_id = 256u + k;
        h_merges_out[k].count = (uint32_t)(h_best[k] >> 32);
    }
    *n_done = done;

    // 4. the final stream (expanded over the occurrences) and its length
    void *ooff;
    if ((rc = ensure(ctx, S_W_OUTOFF, (uint64_t)n_occ * 8 + 16, &ooff))) return rc;
    uint32_t *olen = (uint32_t *)ooff, *ooffs = olen + n_occ + 1;
    if (n_occ) k_occ_len<<<(n_occ + 255) / 256, 256, 0, s>>>(W, n_occ, olen);
    uint32_t total = 0;
    if ((rc = scan_u32(ctx, olen, n_occ, ooffs, W.bsum, W.counter + 3, &total))) return rc;
    if (n_final) *n_final = total;
    if (d_symbols_final && n_occ) {
        k_wexpand<<<(n_occ + 255) / 256, 256, 0, s>>>(W, n_occ, ooffs, d_symbols_final);
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "expand sync");
    }

    stats_reset(ctx);
    const uint64_t per_merge = 2;   // argmax + word merge
    ctx->stats.kernel_launches = 1 + (graph ? (uint64_t)window * (per_merge * kGraphIters + 1) : per_merge * launched);
    const int sc = stats_slot(ctx, "word_count"), sa = stats_slot(ctx, "argmax"), sm = stats_slot(ctx, "word_merge");
    ctx->stats.k[sc].launches = 1;
    ctx->stats.k[sc].bytes = 8.0 * (double)usym;
    const uint32_t ran = std::min<uint32_t>(n_merges, done + 1);
    for (uint32_t k = 1; k < ran; k++) {
        ctx->stats.k[sa].launches++;
        ctx->stats.k[sa].bytes += 8.0 * (double)h_dhist[k];
    }
    ctx->stats.k[sm].launches = done;
    ctx->stats.k[sm].bytes = 4.0 * (double)usym * done;   // every word read once per merge (upper bound)
    if (profile) {
        float x = 0;
        if (cudaEventElapsedTime(&x, ctx->events[0], ctx->events[1]) == cudaSuccess) ctx->stats.k[sc].ms = x;
        for (uint32_t k = 0; k < launched; k++) {
            float a = 0, b = 0;
            cudaEvent_t before = ctx->events[k ? 3 + 2 * (size_t)(k - 1) : 1];
            if (k >= 1 && k < ran && cudaEventElapsedTime(&a, before, ctx->events[2 + 2 * (size_t)k]) == cudaSuccess)
                ctx->stats.k[sa].ms += a;
            if (k < done &&
                cudaEventElapsedTime(&b, ctx->events[2 + 2 * (size_t)k], ctx->events[3 + 2 * (size_t)k]) == cudaSuccess)
                ctx->stats.k[sm].ms += b;
        }
        cudaGetLastError();
    }
    return BPE_OK;
}

}  // namespace
}  // namespace bpe

using namespace bpe;

extern "C" int bpe_train(bpe_ctx *ctx, const uint32_t *d_symbols, uint64_t n, uint32_t n_merges,
                         bpe_merge *h_merges_out, uint32_t *n_done, uint32_t *d_symbols_final, uint64_t *n_final) {
    if (!ctx) return BPE_ERR_INVALID_ARG;
    if (!n_done) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_train: n_done is null");
    if (n_merges > BPE_MAX_MERGES)
        return fail(ctx, BPE_ERR_ID_OVERFLOW, "bpe_train: %u merges exceed %u (ids must fit 16 bits)", n_merges,
                    BPE_MAX_MERGES);
    if (n && !d_symbols) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_train: d_symbols is null");
    if (n_merges && !h_merges_out) return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_train: h_merges_out is null");
    if (n >= BPE_MAX_TRAIN_SYMBOLS)
        return fail(ctx, BPE_ERR_INVALID_ARG, "bpe_train: %llu symbols exceed the limit", (unsigned long long)n);
    BPE_CUDA(ctx, cudaSetDevice(ctx->device), "cudaSetDevice");
    *n_done = 0;
    if (n < 2 || n_merges == 0) {   // no pair to count
        stats_reset(ctx);
        if (n_final) *n_final = n;
        if (d_symbols_final && n) {
            BPE_CUDA(ctx, cudaMemcpyAsync(d_symbols_final, d_symbols, n * 4, cudaMemcpyDeviceToDevice, ctx->stream),
                     "final copy");
            BPE_CUDA(ctx, cudaStreamSynchronize(ctx->stream), "final sync");
        }
        return BPE_OK;
    }
    if (ctx->merge_mode == BPE_MERGE_LISTS && !ctx->train_words) {
        bool not_bytes = false;
        const int rc = train_lists(ctx, d_symbols, n, n_merges, h_merges_out, n_done, d_symbols_final, n_final,
                                   &not_bytes);
        if (rc != BPE_OK || !not_bytes) return rc;
        // ids beyond one byte: the full-stream loop with the hash-table count
    }
    uint32_t lg = ctx->table_log2;
    const bool automatic = (lg == 0);
    if (automatic) lg = std::min<uint32_t>(22, std::max<uint32_t>(16, ceil_log2(n)));
    for (;;) {
        bool full = false;
        int rc = ctx->train_words
                     ? train_words_once(ctx, d_symbols, n, n_merges, lg, h_merges_out, n_done, d_symbols_final,
                                        n_final, &full)
                     : train_once(ctx, d_symbols, n, n_merges, lg, h_merges_out, n_done, d_symbols_final, n_final,
                                  &full);
        if (rc == BPE_OK || !full || !automatic || lg >= 28) return rc;
        lg += 2;   // automatic size was too small: retry with a larger table
    }
}
