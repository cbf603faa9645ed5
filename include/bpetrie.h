/*
 * bpetrie.h -- byte-level BPE training, greedy trie encoding and Unigram
 * (Viterbi) encoding on one GPU.
 *
 * C ABI of libbpetrie.so (sm_103a).  Plain pointers and sizes only.
 *
 * Sources (web pages; section names as printed there):
 *   [GPU-BPE]  "bpe -- GPU BPE Tokenizer Pipeline" (llm.istanbul, learn/tr/13_bpe)
 *   [UNIGRAM]  "Improving Unigram tokenizer CPU performance" (perplexity.ai hub)
 *
 * Conventions for every call
 *   - d_ pointers are device pointers on the context's device; h_ pointers are
 *     host pointers.  The caller owns every input and output buffer; the
 *     library owns the context, its scratch pool and tries.
 *   - Work is ordered on the context's stream.  A call returns only after its
 *     work is complete when it returns a host-side result (n_done, n_ids...);
 *     bpe_pretokenize returns as soon as its kernel is queued.
 *   - Return value: BPE_OK (0) or a negative BPE_ERR_* code; the message of
 *     the last failure is available from bpe_last_error().  On failure no
 *     output beyond what the code describes is meaningful.
 *   - Symbols are uint32: bits 0-15 a token id, bit 16 BPE_WORD_START
 *     ([GPU-BPE] "What it does", 1. GPU pre-tokenization), bits 17-31 zero.
 */
#ifndef BPETRIE_H
#define BPETRIE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BPE_WORD_START 0x10000u
#define BPE_MAX_MERGES 65280u          /* ids 256 .. 65535 fit in 16 bits */
#define BPE_MAX_TRAIN_SYMBOLS (1ull << 30)

enum {
    BPE_OK = 0,
    BPE_ERR_INVALID_ARG = -1,  /* null pointer, bad size, malformed vocabulary */
    BPE_ERR_OOM = -2,          /* device or host allocation failed */
    BPE_ERR_CUDA = -3,         /* a CUDA runtime call failed */
    BPE_ERR_TABLE_FULL = -4,   /* the global pair table overflowed (raise BPE_OPT_TABLE_LOG2) */
    BPE_ERR_ID_OVERFLOW = -5,  /* n_merges > BPE_MAX_MERGES */
    BPE_ERR_CAPACITY = -6,     /* output buffer too small; required size reported */
    BPE_ERR_TIMEOUT = -7,      /* a bounded device-side wait gave up */
    BPE_ERR_CHECKED_OOB = -8   /* a device bounds check failed (internal error) */
};

typedef struct bpe_ctx bpe_ctx;
typedef struct bpe_trie bpe_trie;

/* One learned merge: the pair (left, right) becomes new_id = 256 + k; count
 * is the pair's number of occurrences when it was chosen.  Ids carry no
 * WORD_START bit. */
typedef struct {
    uint32_t left, right, new_id, count;
} bpe_merge;

/* ------------------------------------------------------------- context --- */

/* Create a context on `device` that orders its work on `cuda_stream` (a
 * cudaStream_t; NULL means the legacy default stream).  The context keeps a
 * persistent scratch pool that grows by 1.5x when a call needs more
 * ([GPU-BPE] "Host architecture", 2. persistent buffer pool).
 * Errors: INVALID_ARG (out NULL, bad device), CUDA. */
int bpe_ctx_create(bpe_ctx **out, int device, void *cuda_stream);

/* Change the stream later calls are ordered on. */
int bpe_ctx_set_stream(bpe_ctx *ctx, void *cuda_stream);

/* Release the context and its scratch (waits for its stream first). */
void bpe_ctx_destroy(bpe_ctx *ctx);

/* Message of the last failed call on this context ("" if none).  The string
 * lives until the next call on the context. */
const char *bpe_last_error(const bpe_ctx *ctx);

/* Tuning and measurement options (bpe_ctx_set_option):
 *   BPE_OPT_TABLE_LOG2   log2 of the global pair-table slots (12..28;
 *                        0 = automatic from the stream length)
 *   BPE_OPT_GRAPH        1 = replay merge iterations from CUDA graphs
 *                        (default), 0 = launch every kernel from the host
 *   BPE_OPT_PROFILE      1 = record a CUDA event after every kernel of
 *                        bpe_train / trie_encode so bpe_last_stats() reports
 *                        per-kernel device time (implies host launches)
 *   BPE_OPT_CHUNK        trie_encode bytes per chunk (64..256, multiple
 *                        of 32; default 256; chunks shorter than a few of
 *                        the vocabulary's longest tokens resynchronise badly)
 *   BPE_OPT_TRAIN_WORDS  1 = bpe_train runs the merge loop over distinct
 *                        words weighted by their number of occurrences
 *                        (the same merges and final stream: no count or merge
 *                        crosses a WORD_START); 0 = over the full symbol
 *                        stream (default)
 *   BPE_OPT_MERGE        the merge loop (all give the same results):
 *                        BPE_MERGE_LISTS (default): every pair occurrence
 *                          is filed, when it forms, in its pair's list; a
 *                          merge reads only its pair's list, rewrites those
 *                          positions in place (the right token's positions
 *                          marked dead) and keeps counts by exact deltas; the
 *                          argmax scans a frontier of the highest counts;
 *                          the stream is compacted once at the end.  Needs
 *                          byte-level input (ids < 256, bits 17-31 zero);
 *                          other input runs BPE_MERGE_TWO_PASS
 *                        BPE_MERGE_TWO_PASS: per merge, range
 *                          summaries (the last CTA scans them into offsets),
 *                          then each range merges and compacts; no CTA waits
 *                          on another
 *                        BPE_MERGE_LOOKBACK: one pass, each tile finding its
 *                          output offset by decoupled look-back
 *                        BPE_MERGE_TILES: the stream is kept as 4,096-slot
 *                          tiles with a live count each; a merge compacts
 *                          every tile into its twin in the other buffer (no
 *                          global offsets), compacting into full tiles when
 *                          they fall below 70% full; gathered at the end
 *   BPE_OPT_TRIE_LAYOUT  the trie layout trie_encode walks (same results):
 *                        BPE_TRIE_DOUBLE_ARRAY (default): a step loads the
 *                          child slot {check, base|TERM} and compares check;
 *                        BPE_TRIE_BITMAP: 64-byte nodes with a 256-bit child
 *                          bitmap ([UNIGRAM] "Bitmap and inline packing"), a
 *                          step tests the parent's bit and loads the child's
 *                          base|TERM; built on a trie's first use (n_slots x
 *                          64 bytes, kept until trie_free)
 *   BPE_OPT_UNI_CHUNK    bytes per chunk of unigram_encode (256 .. 4096, a
 *                        multiple of 64; 0 = default 768)
 *   BPE_OPT_TEST_STALL_TILE  testing only: in unigram_encode the scan tile
 *                        with this ticket never publishes its prefix, so the
 *                        tiles after it wait until their bounded wait gives up
 *                        and the call returns BPE_ERR_TIMEOUT (the context
 *                        stays usable); -1 = off (default)
 *   BPE_OPT_PERSISTENT   1 = with BPE_MERGE_TWO_PASS, the merge loop runs as one cooperative
 *                        launch per window of merges (all CTAs resident,
 *                        phases separated by grid barriers) instead of a CUDA
 *                        graph of per-phase kernels; default 0
 *   BPE_OPT_SPARSE_MERGE occurrence-driven merges (with BPE_MERGE_TWO_PASS;
 *                        same results): a merge reads the stream once to
 *                        find the pair's occurrences and rewrites only those
 *                        (the right symbol becomes a tombstone; the stream
 *                        is compacted when tombstones pass a quarter of it,
 *                        and at the end).  0 = off, every merge rewrites the
 *                        whole stream (default); 1 = from the first window
 *                        after the best pair's count falls below 1/64 of the
 *                        input length; 2 = from merge 0
 *   BPE_OPT_LIST_FRONTIER  testing: the occurrence-list loop's argmax
 *                        frontier capacity (1 .. 8192; 0 = default 8192);
 *                        small values force its overflow and rescan paths
 *   BPE_OPT_LIST_TAIL    the occurrence-list loop runs a merge whose list
 *                        holds at most this many entries in one CTA, many
 *                        merges per launch (0 = every merge on all SMs;
 *                        -1 = default 4096; at most 4096) */
enum {
    BPE_OPT_TABLE_LOG2 = 1,
    BPE_OPT_GRAPH = 2,
    BPE_OPT_PROFILE = 3,
    BPE_OPT_CHUNK = 4,
    BPE_OPT_TRAIN_WORDS = 5,
    BPE_OPT_MERGE = 6,
    BPE_OPT_PERSISTENT = 7,
    BPE_OPT_TRIE_LAYOUT = 8,
    BPE_OPT_UNI_CHUNK = 9,
    BPE_OPT_TEST_STALL_TILE = 10,
    BPE_OPT_SPARSE_MERGE = 11,
    BPE_OPT_LIST_FRONTIER = 12,
    BPE_OPT_LIST_TAIL = 13
};
enum { BPE_TRIE_DOUBLE_ARRAY = 0, BPE_TRIE_BITMAP = 1 };
enum { BPE_MERGE_TWO_PASS = 0, BPE_MERGE_LOOKBACK = 1, BPE_MERGE_TILES = 2, BPE_MERGE_LISTS = 3 };
int bpe_ctx_set_option(bpe_ctx *ctx, int option, int64_t value);

/* Statistics of the last bpe_train or trie_encode call on this context.
 * Per kernel family: launches, algorithmic DRAM bytes (the bytes the method
 * must move: 4 per symbol read or written, input bytes, 4 per id written)
 * and, with BPE_OPT_PROFILE, summed device milliseconds between the events
 * bracketing each launch (0 otherwise). */
typedef struct {
    char name[32];
    uint64_t launches;
    double bytes;
    double ms;
} bpe_kernel_stat;
enum { BPE_MAX_STATS = 8 };
typedef struct {
    int n;
    uint64_t kernel_launches;   /* every kernel launch of the call, graph nodes included */
    bpe_kernel_stat k[BPE_MAX_STATS];
} bpe_stats;
int bpe_last_stats(const bpe_ctx *ctx, bpe_stats *out);

/* -------------------------------------------------------- pre-tokenize --- */

/* [GPU-BPE] "What it does", 1. GPU pre-tokenization, and "Line by line",
 * 1) bpe_word_boundary.  symbols[i] = bytes[i] | WORD_START when i == 0 or
 * class(bytes[i]) != class(bytes[i-1]); classes: Newline 0x0A, Space 0x20,
 * Digit '0'-'9', Letter a-z A-Z and every byte >= 0x80, Punct otherwise.
 * d_bytes: n bytes; d_symbols_out: n uint32 (may not alias d_bytes).
 * n == 0 is a no-op.  Asynchronous.  Errors: INVALID_ARG, CUDA. */
int bpe_pretokenize(bpe_ctx *ctx, const uint8_t *d_bytes, uint64_t n, uint32_t *d_symbols_out);

/* --------------------------------------------------------------- train --- */

/* The BPE merge loop ([GPU-BPE] "What is this?" and "What it does" 2.-3.;
 * the 9-dispatch training pipeline).  For k = 0 .. n_merges-1: count every
 * adjacent pair (i, i+1) whose right symbol has no WORD_START (overlapping
 * occurrences all count), choose the highest count (ties: lowest left id,
 * then lowest right id), stop if that count is 0, otherwise replace the
 * pair's occurrences left to right, non-overlapping, by 256 + k keeping the
 * left symbol's WORD_START bit, and compact the stream.
 *
 * d_symbols: n input symbols (read only; n < BPE_MAX_TRAIN_SYMBOLS).
 * h_merges_out: host array with room for n_merges entries; the first
 *   *n_done are written.
 * d_symbols_final (nullable): device array with room for n symbols; receives
 *   the stream after *n_done merges, *n_final (nullable) its length.
 * Blocks until done.  Errors: INVALID_ARG, ID_OVERFLOW (n_merges >
 * BPE_MAX_MERGES), OOM, TABLE_FULL, TIMEOUT, CUDA. */
int bpe_train(bpe_ctx *ctx, const uint32_t *d_symbols, uint64_t n, uint32_t n_merges,
              bpe_merge *h_merges_out, uint32_t *n_done,
              uint32_t *d_symbols_final, uint64_t *n_final);

/* -------------------------------------------------------- vocabulary --- */

/* The vocabulary a merge table defines ([GPU-BPE] "What is this?": each
 * merge gives its pair one new symbol; "Host architecture", 1.: the
 * vocabulary, as byte strings, is what the trie is compiled from).  Token
 * b < 256 is the single byte b; token 256 + k is merge k's left token's bytes
 * followed by its right token's bytes.  Host only, needs no GPU.
 *
 * h_merges: n_merges entries as bpe_train writes them (merge k must have
 * new_id 256 + k and left, right < 256 + k).  h_bytes_out: bytes_capacity
 * bytes; h_off_out: 257 + n_merges uint64 offsets, token t being
 * h_bytes_out[h_off_out[t] .. h_off_out[t+1]) -- the layout trie_build takes.
 * *n_bytes receives the total; when it exceeds bytes_capacity nothing is
 * written and BPE_ERR_CAPACITY is returned (call with capacity 0 to size the
 * buffer).  Errors: INVALID_ARG (malformed table, null pointer), ID_OVERFLOW,
 * CAPACITY. */
int bpe_vocab_from_merges(const bpe_merge *h_merges, uint32_t n_merges, uint8_t *h_bytes_out,
                          uint64_t bytes_capacity, uint64_t *h_off_out, uint64_t *n_bytes);

/* Ids or symbols back to bytes on the device: the concatenation of the byte
 * strings (as bpe_vocab_from_merges defines them) of d_ids[0 .. n_ids).  Bits
 * 0-15 of each value are the id and WORD_START (bit 16) is ignored, so a
 * symbol stream from bpe_pretokenize / bpe_train and the int32 ids of
 * trie_encode with the same vocabulary both decode; decode(encode(x)) == x.
 *
 * d_ids: n_ids uint32 (device); d_bytes_out: bytes_capacity bytes (device).
 * *n_bytes (host) receives the total; when it exceeds bytes_capacity nothing
 * is written and BPE_ERR_CAPACITY is returned with the required size.  Blocks
 * until done.  Errors: INVALID_ARG (malformed table, a value with bits above
 * 16 or an id past 255 + n_merges), ID_OVERFLOW, CAPACITY, OOM, CUDA. */
int bpe_decode(bpe_ctx *ctx, const bpe_merge *h_merges, uint32_t n_merges, const uint32_t *d_ids,
               uint64_t n_ids, uint8_t *d_bytes_out, uint64_t bytes_capacity, uint64_t *n_bytes);

/* ---------------------------------------------------------------- trie --- */

/* Build a flattened double-array trie ([UNIGRAM], the double-array passage:
 * child = base[node] + byte, valid when check[child] == node; token id kept
 * in the node) over a vocabulary, and upload it to the context's device.
 * Token t is the byte string h_vocab_bytes[h_vocab_off[t] .. h_vocab_off[t+1]);
 * the id of a token is its index.  Greedy encoding (trie_encode and the calls
 * built on it) needs every single byte 0..255 to be a token -- byte-level
 * vocabularies always are, and greedy matching then never fails -- and rejects
 * a trie without; Unigram encoding does not.  When two tokens have the same
 * bytes the lower id is kept.  Empty strings are ignored.  The trie is usable
 * with any context on the same device.
 * Errors: INVALID_ARG (offsets not ascending), OOM, CUDA. */
int trie_build(bpe_ctx *ctx, const uint8_t *h_vocab_bytes, const uint64_t *h_vocab_off,
               uint32_t n_tok, bpe_trie **out);

/* Host-only: the double-array layout trie_build would upload, written to
 * caller arrays of `capacity` entries (check = parent slot, -1 free, -2 root;
 * base = child offset | 0x80000000 when the slot is a token; tid = token id
 * or -1).  *n_slots receives the layout size; BPE_ERR_CAPACITY when it
 * exceeds capacity (call with capacity 0 to size the arrays).  Needs no GPU.
 * Errors: INVALID_ARG (as trie_build), CAPACITY. */
int trie_layout(const uint8_t *h_vocab_bytes, const uint64_t *h_vocab_off, uint32_t n_tok,
                int32_t *check_out, int32_t *base_out, int32_t *tid_out, uint64_t capacity,
                uint64_t *n_slots);

/* Sizes of a built trie (any pointer may be NULL). */
int trie_info(const bpe_trie *trie, uint64_t *n_nodes, uint64_t *n_slots, uint32_t *max_token_len);

void trie_free(bpe_trie *trie);

/* Greedy longest-match encoding ([GPU-BPE] "What it does", 4. trie-based
 * inference, and the 3-dispatch inference pipeline).  Each document
 * d_bytes[d_doc_off[d] .. d_doc_off[d+1]) is encoded independently from its
 * first byte: at position p the id of the longest token that prefixes the
 * rest of the document is emitted and p advances by its length.
 *
 * d_doc_off: n_docs+1 ascending uint64 (device); d_ids_out: ids_capacity
 * int32; d_id_off_out (nullable): n_docs+1 uint64, d_id_off_out[d] = index
 * of document d's first id, [n_docs] = total.  *n_ids (host) receives the
 * total.  When the total exceeds ids_capacity no id beyond the capacity is
 * written, *n_ids holds the required size and BPE_ERR_CAPACITY is returned.
 * Blocks until done.  Errors: INVALID_ARG, CAPACITY, OOM, TIMEOUT, CUDA. */
int trie_encode(bpe_ctx *ctx, const bpe_trie *trie, const uint8_t *d_bytes,
                const uint64_t *d_doc_off, uint32_t n_docs, int32_t *d_ids_out,
                uint64_t ids_capacity, uint64_t *d_id_off_out, uint64_t *n_ids);

/* Streaming encode of one document that arrives in slices ([GPU-BPE] "Host
 * architecture", 3. multi-pass slicing; the parse is carried across slices so
 * the ids equal trie_encode's on the whole document).
 *
 * trie_stream_open: a stream bound to ctx (its device, stream and pool) and
 * trie; both must outlive it.  trie_stream_push: encode the bytes carried from
 * the previous push followed by d_bytes[0 .. n) (device), write the ids that
 * no later byte can change to d_ids_out[0 .. *n_ids) and carry the rest of
 * the bytes (fewer than the longest token) to the next push; with last != 0
 * every id is final and the stream is ready for a new document.  The ids of
 * the carried tail may also be written past *n_ids, so ids_capacity must
 * hold one id per carried or new byte; when it does not, BPE_ERR_CAPACITY is
 * returned with the required size in *n_ids and the carry is kept (the push
 * can be repeated).  Blocks until done.  Errors: INVALID_ARG, CAPACITY, OOM,
 * TIMEOUT, CUDA.  trie_stream_close releases the stream (NULL is ignored). */
typedef struct bpe_stream bpe_stream;
int trie_stream_open(bpe_ctx *ctx, const bpe_trie *trie, bpe_stream **out);
int trie_stream_push(bpe_stream *stream, const uint8_t *d_bytes, uint64_t n, int last, int32_t *d_ids_out,
                     uint64_t ids_capacity, uint64_t *n_ids);
void trie_stream_close(bpe_stream *stream);

/* Greedy encoding from host buffers, with the transfers overlapped ("Async
 * batching", three streams ordered by events: host to device, compute,
 * device to host; two device buffer slots).  Same result as trie_encode on
 * the same documents.  Whole documents are grouped into units of about
 * slice_bytes (0: 128 MiB) and encoded together; a longer document is streamed
 * in slices of slice_bytes with the parse carried across them.
 *
 * h_bytes, h_doc_off (n_docs+1 ascending offsets): host input (pinned memory
 * lets the copies overlap the encode); h_ids_out: ids_capacity int32 (host,
 * pinned for the same reason); h_id_off_out (nullable): n_docs+1 uint64.
 * *n_ids receives the total; past ids_capacity nothing is written and
 * BPE_ERR_CAPACITY is returned with the required size.  Blocks until done.
 * Errors: INVALID_ARG, CAPACITY, OOM, TIMEOUT, CUDA. */
int trie_encode_host(bpe_ctx *ctx, const bpe_trie *trie, const uint8_t *h_bytes, const uint64_t *h_doc_off,
                     uint32_t n_docs, int32_t *h_ids_out, uint64_t ids_capacity, uint64_t *h_id_off_out,
                     uint64_t *n_ids, uint64_t slice_bytes);

/* Encoding that allocates nothing.  The pages have no counterpart: this entry
 * point exists for callers of the library that cannot allocate device memory,
 * for example a plug-in that receives only a stream and raw device pointers
 * from a host application which owns all device memory through its own
 * allocator or a fixed budget, or a latency-critical path that must not
 * trigger the device-wide synchronisation that cudaFree implies.
 *
 * Same inputs, outputs, result and errors as trie_encode, but no context is
 * used and nothing is allocated (no cudaMalloc, cudaFree, pinned host memory
 * or allocating library routine): the scratch lives in one fixed array inside
 * the library, about 11.9 MB, which every GPU that loads the library holds
 * until the process exits.  The work is ordered on `cuda_stream` (a
 * cudaStream_t, NULL = legacy default stream); the trie's device is made
 * current for the call and the caller's current device is restored.
 *
 * Limits: n_docs <= 65,536 and at most 524,288 chunks of 128 bytes, where a
 * document of L bytes uses ceil(L / 128) chunks (up to 64 MiB of text in
 * all).  A larger input returns BPE_ERR_INVALID_ARG before any id is written.
 * The first call on a device looks up the array's device address, once per
 * device with that device current; make that first call before any stream
 * capture.  Every call shares the array, which keeps the last call's contents
 * (each call clears what must start at zero), so calls that overlap on the GPU
 * -- on different streams or threads -- race: the caller must serialise them.
 * Blocks until done.  Errors: INVALID_ARG, CAPACITY (with *n_ids = required
 * size), TIMEOUT, CUDA; there is no context, so no message is kept. */
int trie_encode_noalloc(const bpe_trie *trie, const uint8_t *d_bytes, const uint64_t *d_doc_off,
                        uint32_t n_docs, int32_t *d_ids_out, uint64_t ids_capacity,
                        uint64_t *d_id_off_out, uint64_t *n_ids, void *cuda_stream);

/* --------------------------------------------------------- Unigram ------ */

/* Unigram (Viterbi) encoding ([UNIGRAM] "Unigram tokenization": the most
 * likely segmentation, best[j] = max over tokens t = bytes[i..j) of best[i] +
 * score(t), with best[0] = 0, then a backtrack from the end) over the same
 * double-array trie.  Per document, exactly as that recurrence states:
 *   - a position that holds a UTF-8 continuation byte (10xxxxxx) starts no
 *     token, and a token counts only when it ends at a character boundary
 *     (the document end or a byte that is not a continuation byte);
 *   - a reachable position from which no token counts is followed by one
 *     unk_id spanning to the next character boundary, scored unk_score;
 *   - on equal scores the path whose last token starts earliest wins (the
 *     strict comparison of the recurrence, positions taken in order).
 *
 * unigram_create: a model bound to ctx's device and to trie (which must
 * outlive it).  h_scores: trie's n_tok f64 scores (host), one per token id.
 * The GPU sums scores exactly in 64-bit fixed point: with q the smallest
 * exponent for which every score and unk_score times 2^q is an integer, q
 * must be at most 62 and every |score| * 2^q below 2^62 (any float32 value of
 * magnitude at least 2^-39 qualifies).  Sums are then exact, so the result
 * equals the recurrence evaluated in f64 whenever that evaluation rounds
 * nothing.  Errors: INVALID_ARG (bad
 * pointer, a score that is not finite or not representable as above, more
 * than 16,777,214 tokens, a token longer than 255 bytes), OOM, CUDA.
 *
 * unigram_encode: inputs and outputs as trie_encode (d_doc_off: n_docs+1
 * ascending offsets; ids_capacity; d_id_off_out nullable; *n_ids = total,
 * BPE_ERR_CAPACITY with the required size when it exceeds the capacity).
 * A token or an <unk> span longer than the model's span limit (63 bytes when
 * the longest token has at most 63 bytes, else 255) returns INVALID_ARG, as
 * does a document whose length times the largest |score| * 2^q reaches 2^62.
 * Blocks until done.  Errors: INVALID_ARG, CAPACITY, OOM, TIMEOUT, CUDA.
 * unigram_free releases the model (NULL is ignored). */
typedef struct bpe_unigram bpe_unigram;
int unigram_create(bpe_ctx *ctx, const bpe_trie *trie, const double *h_scores, uint32_t n_scores,
                   int32_t unk_id, double unk_score, bpe_unigram **out);
int unigram_encode(bpe_ctx *ctx, const bpe_unigram *model, const uint8_t *d_bytes, const uint64_t *d_doc_off,
                   uint32_t n_docs, int32_t *d_ids_out, uint64_t ids_capacity, uint64_t *d_id_off_out,
                   uint64_t *n_ids);
void unigram_free(bpe_unigram *model);

#ifdef __cplusplus
}
#endif
#endif /* BPETRIE_H */
