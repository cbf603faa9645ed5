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
constexpr int kDeltaSlots = 1024;                 // shared delta table per merge CTA (8 KiB)
constexpr int kTileHalo = 16;                     // symbols staged past a tile
// Shared-memory tile layout: one padding word after every 16 symbols, so a
// thread reading its 16 consecutive symbols hits 32 different banks.
constexpr int kTileWords = (kMergeTile + kTileHalo) + (kMergeTile + kTileHalo) / 16;
__device__ __forceinline__ int padded(int i) { return i + (i >> 4); }
static_assert(kMergeItems == 16, "the padded tile layout assumes 16 symbols per thread");
constexpr int kArgmaxThreads = 256;
constexpr int kGraphIters = 32;                   // merge iterations per captured graph
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
};

struct TrainParams {
    uint32_t *buf[2];
    unsigned long long *tslot;   // hash slots: key << 32 | dense index
    uint32_t tmask;
    uint32_t *dkey;              // dense keys (l << 16 | r)
    uint32_t *dcnt;              // dense counts
    uint32_t dcap;
    unsigned long long *status[2];
    unsigned long long *best;    // per merge: count << 32 | ~key ; 0 = stop
    unsigned long long *nhist;   // stream length after k merges
    uint32_t *dhist;             // dense entries scanned by argmax k
    TrainState *st;
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
    unsigned long long b = 0;
    for (uint32_t i = blockIdx.x * kArgmaxThreads + threadIdx.x; i < D; i += gridDim.x * kArgmaxThreads) {
        const uint32_t c = __ldcg(p.dcnt + i);
        if (c != 0) {
            const unsigned long long v = pack_best(c, __ldcg(p.dkey + i));
            b = v > b ? v : b;
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
// nearby).  mm: bit j = m(pos+j) for j = 0..17; mprev = m(pos-1); sym(j) reads
// symbol pos+j from the padded tile.
__device__ __noinline__ void thread_deltas(const Table p, uint32_t *dkey, uint32_t *dval, uint32_t *socc,
                                           const uint32_t *mys, uint64_t pos, uint64_t n, uint32_t mm,
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
        if (pos + j + 1 >= n) break;
        const uint32_t b = sym(j + 1);
        if (!(b & kWordStart)) add(pair_key(sym(j), b), 0xFFFFFFFFu);
    }
    // new pairs at kept positions j whose own or next kept symbol merged
    uint32_t tnew = ~mext & (mm | (mm >> 1)) & 0xFFFFu;
    while (tnew) {
        const int j = __ffs(tnew) - 1;
        tnew &= tnew - 1;
        if (pos + j >= n) break;
        const uint32_t mj = (mm >> j) & 1u;
        const int nk = j + 1 + (int)mj;
        if (pos + nk >= n) continue;
        const uint32_t b = sym(nk);
        if (b & kWordStart) continue;
        const uint32_t mk = (mm >> nk) & 1u;
        add(pair_key(mj ? new_id : sym(j), mk ? new_id : b), 1u);
    }
}

__global__ void __launch_bounds__(kMergeThreads, 4) k_merge(TrainParams p, uint32_t it) {
    extern __shared__ uint32_t dsm[];
    uint32_t *stile = dsm;                                // the tile and its halo (padded)
    uint32_t *dkey = dsm + kTileWords;                    // shared delta table
    uint32_t *dval = dkey + kDeltaSlots;
    __shared__ uint32_t s_wsum[kMergeWarps];
    __shared__ uint32_t s_tile, s_carry, s_docc, s_tilesum;
    __shared__ unsigned long long s_off;

    TrainState *st = p.st;
    const uint32_t k = st->k_base + it;
    if (k >= st->n_merges || st->err) return;
    const unsigned long long bw = p.best[k];
    if ((bw >> 32) == 0) return;  // nothing to merge: training has stopped
    const uint32_t key = ~(uint32_t)bw;
    const uint32_t l = key >> 16, r = key & 0xFFFFu, new_id = 256u + k;
    const uint64_t n = st->n[k & 1];
    const uint32_t *in = (k & 1) ? p.buf[1] : p.buf[0];
    uint32_t *out = (k & 1) ? p.buf[0] : p.buf[1];
    unsigned long long *status = (k & 1) ? p.status[1] : p.status[0];
    unsigned long long *next_status = (k & 1) ? p.status[0] : p.status[1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t ntiles = (n + kMergeTile - 1) / kMergeTile;

    // one tile per CTA, in ticket order (a tile only waits on tiles that run)
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

    // coalesced 128-bit loads of the tile and its halo into shared memory
#pragma unroll
    for (int q = 0; q < (kMergeTile + kTileHalo) / (4 * kMergeThreads) + 1; q++) {
        const int i4 = tid + q * kMergeThreads;
        if (i4 < (kMergeTile + kTileHalo) / 4) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (base + 4ull * i4 < n) v = __ldcs(reinterpret_cast<const uint4 *>(in + base + 4ull * i4));
            uint32_t *d = stile + padded(4 * i4);   // 4 symbols never straddle a padding word
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        }
    }
    __syncthreads();

    // valid starts among this thread's 16 positions and the 2 after them
    const uint64_t pos = base + (uint64_t)kMergeItems * tid;
    const uint32_t *mys = stile + padded(kMergeItems * tid);
    uint32_t valid = 0;   // bit j: position pos + j is a valid start, j = 0 .. 17
    {
        uint32_t isl = 0, isr = 0;   // id == l ; id == r without WORD_START
#pragma unroll
        for (int j = 0; j < kMergeItems + 3; j++) {
            const uint32_t x = mys[j < 16 ? j : j + 1];
            isl |= (uint32_t)((x & 0xFFFFu) == l) << j;
            isr |= (uint32_t)((x & 0x1FFFFu) == r) << j;
        }
        valid = isl & (isr >> 1) & 0x3FFFFu;
        const uint64_t lim = n - pos;   // positions pos+j with j + 1 < lim
        if (lim < kMergeItems + 3) valid &= (lim >= 1) ? ((1u << (uint32_t)(lim - 1)) - 1u) : 0u;
    }
    // A tile takes the full path when it owns a valid start, or when the next
    // tile's first position is one: the merge there removes the pair (last,
    // first) and creates (last, new symbol), deltas this tile owes.
    const bool any = __syncthreads_or((valid & (tid == kMergeThreads - 1 ? 0x1FFFFu : 0xFFFFu)) != 0);

    uint32_t excl = kSumId;   // summary of this tile's items before this thread
    if (!any) {
        // no valid start owned by the tile: parity is 0 after every item, only
        // the first symbol can be consumed (by a merge at the end of the tile before)
        if (tid == 0) s_tilesum = sum_pack(0u, tile_len, tile_len - 1);
    } else {
        for (int j = tid; j < kDeltaSlots; j += kMergeThreads) {   // fenced by the barriers below
            dkey[j] = kEmptyKey;
            dval[j] = 0;
        }
        uint32_t kept[2], fout[2];
#pragma unroll
        for (uint32_t c = 0; c < 2; c++) {
            uint32_t par = c, kc = 0;
#pragma unroll
            for (int j = 0; j < kMergeItems; j++) {
                if (pos + j < n) kc += par ^ 1u;
                par = ((valid >> j) & 1u) ? (par ^ 1u) : 0u;
            }
            kept[c] = kc;
            fout[c] = par;
        }
        const uint32_t mine = sum_pack(fout[0] | (fout[1] << 1), kept[0], kept[1]);
        uint32_t incl = mine;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(kFull, incl, d);
            if (lane >= d) incl = sum_comp(incl, o);
        }
        excl = __shfl_up_sync(kFull, incl, 1);
        if (lane == 0) excl = kSumId;
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {   // exclusive scan of the 8 warp totals
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
            if (lane == kMergeWarps - 1) s_tilesum = wi;
        }
        __syncthreads();
        excl = sum_comp(excl, s_wsum[warp]);
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
    const unsigned long long obase = s_off;

    if (!any) {
        // shifted copy; a merge at the end of the previous tile consumed symbol 0
        for (uint32_t i = tid; i + carry < tile_len; i += kMergeThreads) out[obase + i] = stile[padded(i + carry)];
        if (carry && tid == 0 && base + 1 < n && !(stile[1] & kWordStart))
            global_add(table_of(p), pair_key(stile[0], stile[1]), 0xFFFFFFFFu);
        return;
    }

    // merge flags m(pos-1 .. pos+17) under the real carry
    uint32_t par = fapply(excl & 3u, carry);
    const uint32_t mprev = par;   // m(pos-1)
    uint32_t mm = 0;              // bit j: m(pos+j)
#pragma unroll
    for (int j = 0; j < kMergeItems + 2; j++) {
        par = ((valid >> j) & 1u) ? (par ^ 1u) : 0u;
        mm |= par << j;
    }
    if ((mm | mprev) & 0x1FFFFu)   // some merge touches this thread's pairs
        thread_deltas(table_of(p), dkey, dval, &s_docc, mys, pos, n, mm, mprev, new_id);
    const uint32_t mext = (mm << 1) | mprev;   // bit j: position pos+j consumed
    uint32_t outv[kMergeItems];
#pragma unroll
    for (int j = 0; j < kMergeItems; j++) {
        const uint32_t x = mys[j];
        outv[j] = ((mm >> j) & 1u) ? (new_id | (x & kWordStart)) : x;
    }
    uint32_t e = carry ? (excl >> 17) : ((excl >> 2) & 0x7FFFu);   // tile-local output index
    const uint32_t tile_kept = carry ? (tile >> 17) : ((tile >> 2) & 0x7FFFu);
    __syncthreads();   // every symbol of the tile is in registers: the tile buffer is free
#pragma unroll
    for (int j = 0; j < kMergeItems; j++)
        if (pos + j < n && !((mext >> j) & 1u)) stile[padded(e++)] = outv[j];
    __syncthreads();
    for (uint32_t i = tid; i < tile_kept; i += kMergeThreads) out[obase + i] = stile[padded(i)];
    if (s_docc) {
        for (int j = tid; j < kDeltaSlots; j += kMergeThreads) {
            const uint32_t kk = dkey[j];
            if (kk != kEmptyKey && dval[j]) global_add(table_of(p), kk, dval[j]);
        }
    }
}

__global__ void k_advance(TrainState *st, uint32_t by) { st->k_base += by; }

uint32_t ceil_log2(uint64_t x) {
    uint32_t l = 0;
    while ((1ull << l) < x) l++;
    return l;
}

struct Launch {
    TrainParams p;
    unsigned count_grid, merge_grid, argmax_grid;
    size_t count_smem, merge_smem;
};

int occupancy(bpe_ctx *ctx, int *count_blocks, int *merge_blocks) {
    const size_t csm = 2 * kCountSlots * sizeof(uint32_t),
                 msm = (kTileWords + 2 * kDeltaSlots) * sizeof(uint32_t);
    BPE_CUDA(ctx, cudaFuncSetAttribute(k_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csm),
             "k_count smem attribute");
    BPE_CUDA(ctx, cudaFuncSetAttribute(k_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msm),
             "k_merge smem attribute");
    BPE_CUDA(ctx, cudaOccupancyMaxActiveBlocksPerMultiprocessor(count_blocks, k_count, kCountThreads, csm),
             "k_count occupancy");
    BPE_CUDA(ctx, cudaOccupancyMaxActiveBlocksPerMultiprocessor(merge_blocks, k_merge, kMergeThreads, msm),
             "k_merge occupancy");
    *count_blocks = std::max(*count_blocks, 1);
    *merge_blocks = std::max(*merge_blocks, 1);
    return BPE_OK;
}

void launch_iteration(const Launch &L, uint32_t it, cudaStream_t s) {
    k_argmax<<<L.argmax_grid, kArgmaxThreads, 0, s>>>(L.p, it);
    k_merge<<<L.merge_grid, kMergeThreads, L.merge_smem, s>>>(L.p, it);
}

// Capture (or reuse) a graph of kGraphIters iterations plus the k_base advance.
int get_graph(bpe_ctx *ctx, const Launch &L, cudaGraphExec_t *out) {
    std::vector<uintptr_t> key = {
        (uintptr_t)L.p.buf[0], (uintptr_t)L.p.buf[1], (uintptr_t)L.p.tslot, (uintptr_t)L.p.tmask,
        (uintptr_t)L.p.dkey, (uintptr_t)L.p.dcnt, (uintptr_t)L.p.dcap, (uintptr_t)L.p.status[0],
        (uintptr_t)L.p.status[1], (uintptr_t)L.p.best, (uintptr_t)L.p.nhist, (uintptr_t)L.p.dhist,
        (uintptr_t)L.p.st, (uintptr_t)L.merge_grid, (uintptr_t)L.argmax_grid};
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
    uint32_t *dkey = (uint32_t *)dense, *dcnt = dkey + T;   // dense keys, then dense counts
    const uint32_t G = kGraphIters;
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
    h_nhist[0] = n;
    BPE_CUDA(ctx, cudaMemcpyAsync(state, h_state, sizeof *h_state, cudaMemcpyHostToDevice, s), "state upload");
    BPE_CUDA(ctx, cudaMemcpyAsync(nhist, h_nhist, 8, cudaMemcpyHostToDevice, s), "nhist upload");
    BPE_CUDA(ctx, cudaMemsetAsync(tslot, 0xFF, T * 8, s), "table clear");
    BPE_CUDA(ctx, cudaMemsetAsync(dcnt, 0, T * 4, s), "count clear");
    BPE_CUDA(ctx, cudaMemsetAsync(st0, 0, ntiles * 8, s), "status clear");
    BPE_CUDA(ctx, cudaMemsetAsync(best, 0, (uint64_t)n_merges * 8, s), "best clear");
    BPE_CUDA(ctx, cudaMemsetAsync(dhist, 0, ((uint64_t)n_merges + 1) * 4, s), "dhist clear");
    BPE_CUDA(ctx, cudaMemcpyAsync(buf0, d_symbols, n * 4, cudaMemcpyDeviceToDevice, s), "input copy");

    int cb, mb;
    if ((rc = occupancy(ctx, &cb, &mb))) return rc;
    Launch L;
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
    const uint64_t count_work = (n + kCountTile - 1) / kCountTile;
    L.count_grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(count_work, (uint64_t)ctx->sm_count * cb));
    L.merge_grid = (unsigned)std::max<uint64_t>(1, ntiles);   // one tile per CTA; spare CTAs exit
    L.argmax_grid = (unsigned)ctx->sm_count * 2;
    L.count_smem = 2 * kCountSlots * sizeof(uint32_t);
    L.merge_smem = (kTileWords + 2 * kDeltaSlots) * sizeof(uint32_t);

    const bool profile = ctx->profile != 0;
    const bool graph = ctx->use_graph && !profile;
    // profile events: 0 before k_count, 1 after it; merge k: 2+2k after argmax, 3+2k after merge
    const size_t n_prof = profile ? 2 + 2 * (size_t)n_merges : 0;
    if ((rc = ensure_events(ctx, n_prof + kInFlight))) return rc;
    std::vector<cudaEvent_t> poll_ev(kInFlight);
    for (int i = 0; i < kInFlight; i++) poll_ev[i] = ctx->events[n_prof + i];

    cudaGraphExec_t exec = nullptr;
    if (graph && (rc = get_graph(ctx, L, &exec))) return rc;
    if (profile) BPE_CUDA(ctx, cudaEventRecord(ctx->events[0], s), "event");
    k_count<<<L.count_grid, kCountThreads, L.count_smem, s>>>(L.p);
    if (profile) BPE_CUDA(ctx, cudaEventRecord(ctx->events[1], s), "event");

    // Launch windows of G merges; keep at most kInFlight windows queued so a
    // stop (a merge with count 0) is noticed without a full drain.
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
        const uint32_t end = std::min<uint32_t>(n_merges, launched + G);
        if (graph) {
            BPE_CUDA(ctx, cudaGraphLaunch(exec, s), "graph launch");
        } else {
            for (uint32_t k = launched; k < end; k++) {
                k_argmax<<<L.argmax_grid, kArgmaxThreads, 0, s>>>(L.p, k);
                if (profile) cudaEventRecord(ctx->events[2 + 2 * (size_t)k], s);
                k_merge<<<L.merge_grid, kMergeThreads, L.merge_smem, s>>>(L.p, k);
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
        return fail(ctx, BPE_ERR_TIMEOUT, "bpe_train: decoupled look-back wait gave up");
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
    if (d_symbols_final) {
        BPE_CUDA(ctx, cudaMemcpyAsync(d_symbols_final, L.p.buf[done & 1], nf * 4, cudaMemcpyDeviceToDevice, s),
                 "final copy");
        BPE_CUDA(ctx, cudaStreamSynchronize(s), "final sync");
    }

    // statistics: algorithmic bytes per kernel family and (profiled) device time
    stats_reset(ctx);
    ctx->stats.kernel_launches = 1 + (graph ? (uint64_t)window * (2 * kGraphIters + 1) : 2ull * launched);
    const int sc = stats_slot(ctx, "pair_count"), sa = stats_slot(ctx, "argmax"), sm = stats_slot(ctx, "merge_compact");
    ctx->stats.k[sc].launches = 1;
    ctx->stats.k[sc].bytes = 4.0 * (double)n;
    const uint32_t ran = std::min<uint32_t>(n_merges, done + 1);   // the argmax that found 0 ran too
    for (uint32_t k = 1; k < ran; k++) {
        ctx->stats.k[sa].launches++;
        ctx->stats.k[sa].bytes += 8.0 * (double)h_dhist[k];
    }
    for (uint32_t k = 0; k < done; k++) {
        ctx->stats.k[sm].launches++;
        ctx->stats.k[sm].bytes += 4.0 * (double)h_nhist[k] + 4.0 * (double)h_nhist[k + 1];
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
                ctx->stats.k[sm].ms += b;
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
    ctx->stats.kernel_launches = 1 + (graph ? (uint64_t)window * (2 * kGraphIters + 1) : 2ull * launched);
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
