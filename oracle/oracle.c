/*
 * oracle.c -- plain, slow, single-threaded CPU reference for byte-level BPE.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The GPU library never
 * calls it, links it or shares a line with it.
 *
 * Sources (web pages; section names as printed there):
 *   [GPU-BPE]  "bpe -- GPU BPE Tokenizer Pipeline" (llm.istanbul, learn/tr/13_bpe)
 *   [UNIGRAM]  "Improving Unigram tokenizer CPU performance" (perplexity.ai hub)
 *
 * Symbols are uint32: bits 0-15 hold a token id, bit 16 is WORD_START
 * (0x10000, [GPU-BPE] "What it does", 1. GPU pre-tokenization).
 *
 * Every function follows the plain definition; no blocking, fusion or reuse
 * between merges.  Readings where the pages are silent:
 *   - WORD_START is set at index 0 (a text starts a word) and wherever the
 *     class of byte i differs from the class of byte i-1.
 *   - pair counts are overlapping: every adjacent position (i, i+1) with no
 *     WORD_START on i+1 counts once ("aaa" holds the pair (a,a) twice).
 *   - the chosen pair is the highest count, ties to the lowest left id, then
 *     the lowest right id; training stops when the highest count is 0.
 *   - merge k creates id 256 + k; occurrences are replaced left to right,
 *     non-overlapping (leftmost first), and the merged symbol keeps the
 *     WORD_START bit of its left part.
 *   - greedy encoding emits, at each position, the longest vocabulary string
 *     that prefixes the rest of the document; duplicate strings keep the
 *     lowest id; a position no token matches is an error.
 *   - Unigram (Viterbi) segmentation: see orc_unigram_encode.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define WS 0x10000u
#define ID(s) ((s) & 0xFFFFu)

enum { ORC_OK = 0, ORC_EARG = -1, ORC_ENOMEM = -2, ORC_ENOMATCH = -3, ORC_ECAP = -4 };

/* ------------------------------------------------------------------------
 * [GPU-BPE] "Line by line", 1) bpe_word_boundary -- byte classification.
 * Classes: 0 Letter (a-z, A-Z and every byte >= 0x80), 1 Digit, 2 Space,
 * 3 Punct (everything else, including tab, CR and DEL), 4 Newline.
 * Written out as the page's cascade of tests, in the page's order.
 * ---------------------------------------------------------------------- */
int orc_char_class(uint32_t b) {
    if (b == 0x0A) return 4;
    if (b == 0x20) return 2;
    if (b >= 0x30 && b <= 0x39) return 1;
    if (b >= 0x80) return 0;
    if (b >= 0x61 && b <= 0x7A) return 0;
    if (b >= 0x41 && b <= 0x5A) return 0;
    return 3;
}

/* [GPU-BPE] "What it does", 1. GPU pre-tokenization (bpe_word_boundary):
 * each byte becomes a symbol; WORD_START marks class transitions. */
void orc_pretokenize(const uint8_t *bytes, uint64_t n, uint32_t *sym) {
    for (uint64_t i = 0; i < n; i++) {
        uint32_t s = bytes[i];
        if (i == 0 || orc_char_class(bytes[i]) != orc_char_class(bytes[i - 1])) s |= WS;
        sym[i] = s;
    }
}

/* ------------------------------------------------------------------------
 * One merge step shared by both training forms: left-to-right scan,
 * non-overlapping.  Returns the new length; *applied = merges done.
 * ---------------------------------------------------------------------- */
static uint64_t apply_merge(const uint32_t *in, uint64_t n, uint32_t l, uint32_t r,
                            uint32_t new_id, uint32_t *out, uint64_t *applied) {
    uint64_t o = 0, a = 0, i = 0;
    while (i < n) {
        if (i + 1 < n && ID(in[i]) == l && ID(in[i + 1]) == r && !(in[i + 1] & WS)) {
            out[o++] = new_id | (in[i] & WS);
            i += 2;
            a++;
        } else {
            out[o++] = in[i];
            i += 1;
        }
    }
    if (applied) *applied = a;
    return o;
}

static int cmp_u32(const void *a, const void *b) {
    uint32_t x = *(const uint32_t *)a, y = *(const uint32_t *)b;
    return (x > y) - (x < y);
}

/*
 * Full-stream training ("O-naive").  [GPU-BPE] "What is this?": find the most
 * frequent adjacent pair, give it a new symbol, repeat; pair counting stops
 * at WORD_START ("What it does", 1. and 2.).  Counting is done by sorting the
 * list of pair keys (l << 16 | r) and measuring runs; the first longest run
 * in ascending key order is the tie-break winner.
 *
 * merges: 4 uint32 per merge (left, right, new id, count).
 * sym_out (nullable, capacity n) receives the stream after n_done merges.
 */
int orc_train_stream(const uint32_t *sym_in, uint64_t n, uint32_t n_merges,
                     uint32_t *merges, uint32_t *n_done, uint32_t *sym_out, uint64_t *n_out) {
    if ((n && !sym_in) || (n_merges && !merges) || !n_done) return ORC_EARG;
    if (n_merges > 65280u) return ORC_EARG;
    uint32_t *a = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));
    uint32_t *b = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));
    uint32_t *keys = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));
    if (!a || !b || !keys) { free(a); free(b); free(keys); return ORC_ENOMEM; }
    if (n) memcpy(a, sym_in, sizeof(uint32_t) * n);
    uint32_t k = 0;
    for (; k < n_merges; k++) {
        uint64_t m = 0;
        for (uint64_t i = 0; i + 1 < n; i++)
            if (!(a[i + 1] & WS)) keys[m++] = (ID(a[i]) << 16) | ID(a[i + 1]);
        if (m == 0) break;
        qsort(keys, m, sizeof(uint32_t), cmp_u32);
        uint32_t best_key = 0;
        uint64_t best = 0, run = 1;
        for (uint64_t i = 1; i <= m; i++) {
            if (i < m && keys[i] == keys[i - 1]) { run++; continue; }
            if (run > best) { best = run; best_key = keys[i - 1]; }
            run = 1;
        }
        uint32_t l = best_key >> 16, r = best_key & 0xFFFFu, id = 256u + k;
        merges[4 * k + 0] = l;
        merges[4 * k + 1] = r;
        merges[4 * k + 2] = id;
        merges[4 * k + 3] = (uint32_t)best;
        n = apply_merge(a, n, l, r, id, b, NULL);
        uint32_t *t = a; a = b; b = t;
    }
    *n_done = k;
    if (sym_out && n) memcpy(sym_out, a, sizeof(uint32_t) * n);
    if (n_out) *n_out = n;
    free(a); free(b); free(keys);
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Word-frequency training ("O-wordfreq").  Because no pair is counted across
 * a WORD_START and no merge crosses one, the stream is a sequence of words
 * (a word starts at index 0 and at every WORD_START symbol); counting every
 * distinct word once, weighted by its number of occurrences, gives the same
 * pair counts as the full stream, and merging inside each distinct word gives
 * the same stream.  Same merge step, same tie-break.
 * ---------------------------------------------------------------------- */
typedef struct {            /* growable open-addressing map: pair key -> count */
    uint32_t *key;
    uint64_t *cnt;
    uint32_t *used;         /* slots in use, to clear them cheaply */
    uint64_t cap, n;
} pairmap;

static uint32_t mix32(uint32_t h) {    /* any decent integer hash will do */
    h ^= h >> 16; h *= 0x7FEB352Du; h ^= h >> 15; h *= 0x846CA68Bu; h ^= h >> 16;
    return h;
}
static int pm_init(pairmap *m, uint64_t cap) {
    m->cap = cap; m->n = 0;
    m->key = (uint32_t *)malloc(sizeof(uint32_t) * cap);
    m->cnt = (uint64_t *)malloc(sizeof(uint64_t) * cap);
    m->used = (uint32_t *)malloc(sizeof(uint32_t) * cap);
    if (!m->key || !m->cnt || !m->used) return ORC_ENOMEM;
    memset(m->key, 0xFF, sizeof(uint32_t) * cap);
    return ORC_OK;
}
static void pm_free(pairmap *m) { free(m->key); free(m->cnt); free(m->used); }
static void pm_clear(pairmap *m) {
    for (uint64_t i = 0; i < m->n; i++) m->key[m->used[i]] = 0xFFFFFFFFu;
    m->n = 0;
}
static int pm_add(pairmap *m, uint32_t key, uint64_t c);
static int pm_grow(pairmap *m) {
    pairmap g;
    if (pm_init(&g, m->cap * 2)) { pm_free(&g); return ORC_ENOMEM; }
    for (uint64_t i = 0; i < m->n; i++) {
        uint32_t s = m->used[i];
        pm_add(&g, m->key[s], m->cnt[s]);
    }
    pm_free(m);
    *m = g;
    return ORC_OK;
}
static int pm_add(pairmap *m, uint32_t key, uint64_t c) {
    if (2 * (m->n + 1) > m->cap && pm_grow(m)) return ORC_ENOMEM;
    uint64_t s = mix32(key) & (m->cap - 1);
    while (m->key[s] != 0xFFFFFFFFu && m->key[s] != key) s = (s + 1) & (m->cap - 1);
    if (m->key[s] == 0xFFFFFFFFu) {
        m->key[s] = key; m->cnt[s] = 0; m->used[m->n++] = (uint32_t)s;
    }
    m->cnt[s] += c;
    return ORC_OK;
}

typedef void (*orc_checkpoint_fn)(uint32_t k, const uint32_t *sym, uint64_t n, void *user);

typedef struct {            /* distinct words */
    uint32_t **w;           /* symbols of each distinct word */
    uint32_t *len;
    uint64_t *freq;
    uint64_t nw, capw;
} wordset;

static uint64_t hash_syms(const uint32_t *s, uint32_t n) {
    uint64_t h = 1469598103934665603ull;
    for (uint32_t i = 0; i < n; i++) { h ^= s[i]; h *= 1099511628211ull; }
    return h;
}

/* Expand the occurrence list back into the stream. */
static uint64_t expand(const wordset *W, const uint32_t *occ, uint64_t n_occ, uint32_t *out) {
    uint64_t o = 0;
    for (uint64_t i = 0; i < n_occ; i++) {
        const uint32_t *w = W->w[occ[i]];
        uint32_t L = W->len[occ[i]];
        memcpy(out + o, w, sizeof(uint32_t) * L);
        o += L;
    }
    return o;
}

/*
 * checkpoints (nullable): ascending merge counts k at which fn(k, stream)
 * is called with the stream after k merges (k may exceed n_done: then the
 * final stream is reported for it).
 */
int orc_train_words(const uint32_t *sym_in, uint64_t n, uint32_t n_merges,
                    uint32_t *merges, uint32_t *n_done, uint32_t *sym_out, uint64_t *n_out,
                    const uint32_t *checkpoints, uint32_t n_checkpoints,
                    orc_checkpoint_fn fn, void *user) {
    if ((n && !sym_in) || (n_merges && !merges) || !n_done) return ORC_EARG;
    if (n_merges > 65280u) return ORC_EARG;
    int rc = ORC_OK;
    /* 1. split into words and intern them */
    uint64_t n_occ = 0;
    for (uint64_t i = 0; i < n; i++) if (i == 0 || (sym_in[i] & WS)) n_occ++;
    uint32_t *occ = (uint32_t *)malloc(sizeof(uint32_t) * (n_occ ? n_occ : 1));
    wordset W = {0};
    W.capw = 1024;
    W.w = (uint32_t **)malloc(sizeof(uint32_t *) * W.capw);
    W.len = (uint32_t *)malloc(sizeof(uint32_t) * W.capw);
    W.freq = (uint64_t *)malloc(sizeof(uint64_t) * W.capw);
    uint64_t hcap = 1 << 16;
    uint32_t *ht = (uint32_t *)malloc(sizeof(uint32_t) * hcap);
    if (!occ || !W.w || !W.len || !W.freq || !ht) { rc = ORC_ENOMEM; goto out; }
    memset(ht, 0xFF, sizeof(uint32_t) * hcap);
    uint64_t o = 0;
    for (uint64_t i = 0; i < n;) {
        uint64_t j = i + 1;
        while (j < n && !(sym_in[j] & WS)) j++;
        uint32_t L = (uint32_t)(j - i);
        uint64_t h = hash_syms(sym_in + i, L), s = h & (hcap - 1);
        while (ht[s] != 0xFFFFFFFFu) {
            uint32_t w = ht[s];
            if (W.len[w] == L && !memcmp(W.w[w], sym_in + i, sizeof(uint32_t) * L)) break;
            s = (s + 1) & (hcap - 1);
        }
        uint32_t w = ht[s];
        if (w == 0xFFFFFFFFu) {
            if (W.nw == W.capw) {
                W.capw *= 2;
                W.w = (uint32_t **)realloc(W.w, sizeof(uint32_t *) * W.capw);
                W.len = (uint32_t *)realloc(W.len, sizeof(uint32_t) * W.capw);
                W.freq = (uint64_t *)realloc(W.freq, sizeof(uint64_t) * W.capw);
            }
            w = (uint32_t)W.nw++;
            W.w[w] = (uint32_t *)malloc(sizeof(uint32_t) * L);
            memcpy(W.w[w], sym_in + i, sizeof(uint32_t) * L);
            W.len[w] = L;
            W.freq[w] = 0;
            ht[s] = w;
            if (2 * W.nw > hcap) {       /* rehash */
                uint64_t nc = hcap * 2;
                uint32_t *nt = (uint32_t *)malloc(sizeof(uint32_t) * nc);
                memset(nt, 0xFF, sizeof(uint32_t) * nc);
                for (uint64_t q = 0; q < W.nw; q++) {
                    uint64_t t = hash_syms(W.w[q], W.len[q]) & (nc - 1);
                    while (nt[t] != 0xFFFFFFFFu) t = (t + 1) & (nc - 1);
                    nt[t] = (uint32_t)q;
                }
                free(ht); ht = nt; hcap = nc;
            }
        }
        W.freq[w]++;
        occ[o++] = w;
        i = j;
    }
    /* 2. merge loop over distinct words */
    pairmap pm;
    if (pm_init(&pm, 1 << 16)) { pm_free(&pm); rc = ORC_ENOMEM; goto out; }
    uint32_t maxlen = 1;
    for (uint64_t w = 0; w < W.nw; w++) if (W.len[w] > maxlen) maxlen = W.len[w];
    uint32_t *tmp = (uint32_t *)malloc(sizeof(uint32_t) * maxlen);
    uint32_t *stream = NULL;
    if (n_checkpoints) stream = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));
    uint32_t cp = 0, k = 0;
    for (;; k++) {
        while (cp < n_checkpoints && checkpoints[cp] == k) {
            uint64_t sn = expand(&W, occ, n_occ, stream);
            fn(k, stream, sn, user);
            cp++;
        }
        if (k == n_merges) break;
        pm_clear(&pm);
        for (uint64_t w = 0; w < W.nw; w++)
            for (uint32_t i = 0; i + 1 < W.len[w]; i++)
                if (pm_add(&pm, (ID(W.w[w][i]) << 16) | ID(W.w[w][i + 1]), W.freq[w])) {
                    rc = ORC_ENOMEM; break;
                }
        if (rc) break;
        uint64_t best = 0;
        uint32_t best_key = 0;
        for (uint64_t i = 0; i < pm.n; i++) {
            uint32_t s = pm.used[i];
            if (pm.cnt[s] > best || (pm.cnt[s] == best && pm.key[s] < best_key)) {
                best = pm.cnt[s]; best_key = pm.key[s];
            }
        }
        if (best == 0) break;
        uint32_t l = best_key >> 16, r = best_key & 0xFFFFu, id = 256u + k;
        merges[4 * k + 0] = l;
        merges[4 * k + 1] = r;
        merges[4 * k + 2] = id;
        merges[4 * k + 3] = (uint32_t)best;
        for (uint64_t w = 0; w < W.nw; w++) {
            if (W.len[w] < 2) continue;
            uint64_t nl = apply_merge(W.w[w], W.len[w], l, r, id, tmp, NULL);
            memcpy(W.w[w], tmp, sizeof(uint32_t) * nl);
            W.len[w] = (uint32_t)nl;
        }
    }
    if (!rc) {
        *n_done = k;
        while (cp < n_checkpoints) {   /* checkpoints past the end: final stream */
            uint64_t sn = expand(&W, occ, n_occ, stream);
            fn(checkpoints[cp], stream, sn, user);
            cp++;
        }
        uint64_t total = 0;
        for (uint64_t i = 0; i < n_occ; i++) total += W.len[occ[i]];
        if (sym_out) expand(&W, occ, n_occ, sym_out);
        if (n_out) *n_out = total;
    }
    free(stream);
    free(tmp);
    pm_free(&pm);
out:
    for (uint64_t w = 0; w < W.nw; w++) free(W.w[w]);
    free(W.w); free(W.len); free(W.freq); free(ht); free(occ);
    return rc;
}

/* ------------------------------------------------------------------------
 * Vocabulary strings from a merge table: bytes(b) = [b] for b < 256,
 * bytes(256 + k) = bytes(left_k) ++ bytes(right_k).
 * off has 256 + n_merges + 1 entries; out has room for off[last] bytes
 * (call with out = NULL first to size it).
 * ---------------------------------------------------------------------- */
int orc_vocab_from_merges(const uint32_t *merges, uint32_t n_merges, uint8_t *out, uint64_t *off) {
    uint64_t V = 256u + n_merges;
    uint64_t *len = (uint64_t *)malloc(sizeof(uint64_t) * V);
    if (!len) return ORC_ENOMEM;
    for (uint64_t t = 0; t < 256; t++) len[t] = 1;
    for (uint64_t k = 0; k < n_merges; k++) {
        uint32_t l = merges[4 * k], r = merges[4 * k + 1];
        if (l >= 256 + k || r >= 256 + k || merges[4 * k + 2] != 256 + k) { free(len); return ORC_EARG; }
        len[256 + k] = len[l] + len[r];
    }
    off[0] = 0;
    for (uint64_t t = 0; t < V; t++) off[t + 1] = off[t] + len[t];
    if (out) {
        for (uint64_t t = 0; t < 256; t++) out[t] = (uint8_t)t;
        for (uint64_t k = 0; k < n_merges; k++) {
            uint32_t l = merges[4 * k], r = merges[4 * k + 1];
            uint8_t *dst = out + off[256 + k];
            memcpy(dst, out + off[l], len[l]);
            memcpy(dst + len[l], out + off[r], len[r]);
        }
    }
    free(len);
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Plain byte trie with sorted child lists and the token id in the node
 * ([UNIGRAM], token id stored in the trie node; [GPU-BPE] "Host
 * architecture", 1. children sorted by byte).  No double array here: the
 * oracle walks the plain tree.
 * ---------------------------------------------------------------------- */
typedef struct {
    uint32_t *child;   /* node indices, sorted by label */
    uint8_t *label;
    uint32_t nchild, capchild;
    int32_t tid;       /* -1 if not a token */
} tnode;

typedef struct {
    tnode *nodes;
    uint64_t n, cap;
    uint32_t max_len;
} orc_trie;

static uint32_t trie_new_node(orc_trie *T) {
    if (T->n == T->cap) {
        T->cap = T->cap ? T->cap * 2 : 1024;
        T->nodes = (tnode *)realloc(T->nodes, sizeof(tnode) * T->cap);
    }
    tnode *nd = &T->nodes[T->n];
    memset(nd, 0, sizeof(*nd));
    nd->tid = -1;
    return (uint32_t)T->n++;
}

/* binary search for label c among node's children; returns node or UINT32_MAX */
static uint32_t trie_find(const orc_trie *T, uint32_t node, uint8_t c) {
    const tnode *nd = &T->nodes[node];
    uint32_t lo = 0, hi = nd->nchild;
    while (lo < hi) {
        uint32_t mid = (lo + hi) / 2;
        if (nd->label[mid] < c) lo = mid + 1; else hi = mid;
    }
    if (lo < nd->nchild && nd->label[lo] == c) return nd->child[lo];
    return UINT32_MAX;
}

void orc_trie_free(orc_trie *T) {
    if (!T) return;
    for (uint64_t i = 0; i < T->n; i++) { free(T->nodes[i].child); free(T->nodes[i].label); }
    free(T->nodes);
    free(T);
}

orc_trie *orc_trie_new(const uint8_t *vocab, const uint64_t *off, uint32_t n_tok) {
    orc_trie *T = (orc_trie *)calloc(1, sizeof(orc_trie));
    if (!T) return NULL;
    trie_new_node(T);                      /* root = 0 */
    for (uint32_t t = 0; t < n_tok; t++) {
        uint64_t a = off[t], b = off[t + 1];
        if (b <= a) continue;              /* empty strings are never matched */
        uint32_t node = 0;
        for (uint64_t i = a; i < b; i++) {
            uint8_t c = vocab[i];
            uint32_t nx = trie_find(T, node, c);
            if (nx == UINT32_MAX) {
                nx = trie_new_node(T);
                tnode *nd = &T->nodes[node];   /* (after a possible realloc) */
                if (nd->nchild == nd->capchild) {
                    nd->capchild = nd->capchild ? nd->capchild * 2 : 2;
                    nd->child = (uint32_t *)realloc(nd->child, sizeof(uint32_t) * nd->capchild);
                    nd->label = (uint8_t *)realloc(nd->label, nd->capchild);
                }
                uint32_t p = nd->nchild;
                while (p > 0 && nd->label[p - 1] > c) {
                    nd->label[p] = nd->label[p - 1]; nd->child[p] = nd->child[p - 1]; p--;
                }
                nd->label[p] = c; nd->child[p] = nx; nd->nchild++;
            }
            node = nx;
        }
        if (T->nodes[node].tid < 0) T->nodes[node].tid = (int32_t)t;   /* lowest id wins */
        if (b - a > T->max_len) T->max_len = (uint32_t)(b - a);
    }
    return T;
}

uint64_t orc_trie_nodes(const orc_trie *T) { return T->n; }
uint32_t orc_trie_max_len(const orc_trie *T) { return T->max_len; }

/* Longest vocabulary string that prefixes bytes[pos..end): walk the trie as
 * far as it goes, remembering the last node that is a token. */
int orc_longest_match(const orc_trie *T, const uint8_t *bytes, uint64_t end, uint64_t pos,
                      int32_t *id, uint32_t *len) {
    uint32_t node = 0, best_len = 0;
    int32_t best_id = -1;
    for (uint64_t q = pos; q < end; q++) {
        node = trie_find(T, node, bytes[q]);
        if (node == UINT32_MAX) break;
        if (T->nodes[node].tid >= 0) { best_id = T->nodes[node].tid; best_len = (uint32_t)(q + 1 - pos); }
    }
    if (best_len == 0) return ORC_ENOMATCH;
    *id = best_id;
    *len = best_len;
    return ORC_OK;
}

/*
 * Greedy longest-match encoding of a batch of documents ([GPU-BPE] "What is
 * this?", inference: walk the trie one byte at a time and take the longest
 * match; "What it does", 4. trie-based inference).  Each document
 * [doc_off[d], doc_off[d+1]) is encoded independently from its first byte.
 * ids (capacity cap) receive all ids back to back; id_off[d] is the index of
 * document d's first id, id_off[n_docs] the total.  When the total exceeds
 * cap nothing beyond cap is written and ORC_ECAP is returned with *n_ids set
 * to the required size.
 */
int orc_encode(const orc_trie *T, const uint8_t *bytes, const uint64_t *doc_off, uint32_t n_docs,
               int32_t *ids, uint64_t cap, uint64_t *id_off, uint64_t *n_ids) {
    uint64_t m = 0;
    for (uint32_t d = 0; d < n_docs; d++) {
        if (id_off) id_off[d] = m;
        uint64_t p = doc_off[d], end = doc_off[d + 1];
        if (end < p) return ORC_EARG;
        while (p < end) {
            int32_t id; uint32_t len;
            if (orc_longest_match(T, bytes, end, p, &id, &len)) return ORC_ENOMATCH;
            if (m < cap && ids) ids[m] = id;
            m++;
            p += len;
        }
    }
    if (id_off) id_off[n_docs] = m;
    *n_ids = m;
    return m > cap ? ORC_ECAP : ORC_OK;
}

/* ------------------------------------------------------------------------
 * All pair counts of a stream (the counting step of the merge loop on its
 * own, for tests): distinct keys (l << 16 | r) ascending with their counts.
 * Returns the number of distinct pairs (only the first cap are written).
 * ---------------------------------------------------------------------- */
int64_t orc_pair_counts(const uint32_t *sym, uint64_t n, uint32_t *keys_out,
                        uint32_t *counts_out, uint64_t cap) {
    uint32_t *keys = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));
    if (!keys) return ORC_ENOMEM;
    uint64_t m = 0;
    for (uint64_t i = 0; i + 1 < n; i++)
        if (!(sym[i + 1] & WS)) keys[m++] = (ID(sym[i]) << 16) | ID(sym[i + 1]);
    qsort(keys, m, sizeof(uint32_t), cmp_u32);
    int64_t d = 0;
    for (uint64_t i = 0; i < m;) {
        uint64_t j = i;
        while (j < m && keys[j] == keys[i]) j++;
        if ((uint64_t)d < cap) { keys_out[d] = keys[i]; counts_out[d] = (uint32_t)(j - i); }
        d++;
        i = j;
    }
    free(keys);
    return d;
}

/* ------------------------------------------------------------------------
 * Unigram (Viterbi) segmentation ([UNIGRAM] "Unigram tokenization": the most
 * likely path, best[i] = max over tokens t = x[j..i) of best[j] + score(t)).
 * Per document, following the page's recurrence:
 *   best[0] = 0, best[i] = -inf otherwise;
 *   for each position i in order that is reachable and not a UTF-8
 *   continuation byte (10xxxxxx): walk the trie from i; every token t ending
 *   at j relaxes best[j] with best[i] + score[t] when strictly larger
 *   (ties keep the earlier start);
 *   then backtrack from the document end.
 * Readings of what the page leaves open:
 *   - a token counts only when it ends at a character boundary (j is the end
 *     or byte j is not a continuation byte): a path through the middle of a
 *     character could never be continued;
 *   - "no token matched" means no such token: then <unk> (id unk_id, score
 *     unk_score) spans i .. the next character boundary, so every document
 *     has a path.
 * Scores are f64 (the page's node holds an f64 score).  ids / id_off as in
 * orc_encode.
 * ---------------------------------------------------------------------- */
static int is_cont(uint8_t b) { return (b & 0xC0) == 0x80; }

int orc_unigram_encode(const orc_trie *T, const double *score, int32_t unk_id, double unk_score,
                       const uint8_t *bytes, const uint64_t *doc_off, uint32_t n_docs,
                       int32_t *ids, uint64_t cap, uint64_t *id_off, uint64_t *n_ids) {
    uint64_t m = 0;
    for (uint32_t d = 0; d < n_docs; d++) {
        if (id_off) id_off[d] = m;
        const uint64_t s = doc_off[d], e = doc_off[d + 1];
        if (e < s) return ORC_EARG;
        const uint64_t n = e - s;
        const uint8_t *x = bytes + s;
        double *best = (double *)malloc(sizeof(double) * (n + 1));
        uint64_t *from = (uint64_t *)malloc(sizeof(uint64_t) * (n + 1));
        int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (n + 1));
        if (!best || !from || !tok) { free(best); free(from); free(tok); return ORC_ENOMEM; }
        for (uint64_t i = 0; i <= n; i++) best[i] = -INFINITY;
        best[0] = 0.0;
        for (uint64_t i = 0; i < n; i++) {
            if (best[i] == -INFINITY || is_cont(x[i])) continue;
            int matched = 0;
            uint32_t node = 0;
            for (uint64_t q = i; q < n; q++) {
                node = trie_find(T, node, x[q]);
                if (node == UINT32_MAX) break;
                const uint64_t j = q + 1;
                const int32_t t = T->nodes[node].tid;
                if (t < 0 || (j < n && is_cont(x[j]))) continue;
                matched = 1;
                const double cand = best[i] + score[t];
                if (cand > best[j]) { best[j] = cand; from[j] = i; tok[j] = t; }
            }
            if (!matched) {
                uint64_t j = i + 1;
                while (j < n && is_cont(x[j])) j++;
                const double cand = best[i] + unk_score;
                if (cand > best[j]) { best[j] = cand; from[j] = i; tok[j] = unk_id; }
            }
        }
        if (best[n] == -INFINITY) {   /* cannot happen: every character has an edge */
            free(best); free(from); free(tok);
            return ORC_ENOMATCH;
        }
        /* backtrack: count, then write in order */
        uint64_t k = 0;
        for (uint64_t j = n; j > 0; j = from[j]) k++;
        uint64_t w = m + k;
        for (uint64_t j = n; j > 0; j = from[j]) {
            w--;
            if (w < cap && ids) ids[w] = tok[j];
        }
        m += k;
        free(best); free(from); free(tok);
    }
    if (id_off) id_off[n_docs] = m;
    *n_ids = m;
    return m > cap ? ORC_ECAP : ORC_OK;
}
