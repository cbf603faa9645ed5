/*
 * synth.c -- seeded synthetic text for byte-level BPE workloads.
 *
 * Test and benchmark input only.  This file holds none of the tokenizer's
 * arithmetic (no character classes, no pair counting, no merging, no trie):
 * it only writes bytes.  Both the CPU oracle and the GPU library consume what
 * it writes; neither is used here.
 *
 * Text model (one recipe for every workload):
 *   lexicon   K distinct words; word length ~ Geometric(p = 1/5) on {1,2,...},
 *             redrawn while > 12; each letter uniform over a-z, or, when the
 *             lexicon is "Turkish", with probability 0.30 one of the six
 *             two-byte UTF-8 letters c-cedilla, g-breve, dotless i, o-umlaut,
 *             s-cedilla, u-umlaut (uniformly).  Duplicate words are redrawn.
 *   stream    each token is, with probability 0.03, a number of 1-4 digits
 *             (length and digits uniform), otherwise the lexicon word of
 *             Zipf(s = 1.1) rank over the ranks 1..K (inverse CDF); every
 *             token is followed by one separator: space 0.85, one of the 32
 *             ASCII punctuation characters 0.10 (uniform), newline 0.05.
 *   corpus    tokens are appended until the target size is reached; the text
 *             is cut at the target and a dangling UTF-8 lead byte is dropped.
 *   document  tokens are appended until the text is at least the target size
 *             right after a separator (the document ends with that separator).
 *   substring vocabulary: the 256 single bytes, then substrings of a corpus
 *             (start uniform, length round(exp(U[ln 2, ln 48])) clipped to the
 *             corpus end), deduplicated, until the requested size.
 *
 * Randomness is splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  Floating point uses only IEEE-754 basic
 * operations (+ - * /, which are correctly rounded), our own ln/exp series and
 * exact scaling, and this file is compiled with -ffp-contract=off: the bytes
 * are identical on every architecture (x86_64 and aarch64 alike).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ rng -- */
typedef struct { uint64_t s; } syn_rng;

static uint64_t rng_next(syn_rng *r) {
    uint64_t z = (r->s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
/* uniform double in [0,1) from the top 53 bits */
static double rng_unit(syn_rng *r) { return (double)(rng_next(r) >> 11) * (1.0 / 9007199254740992.0); }
/* uniform integer in [0, n) by 128-bit multiply (no modulo bias worth naming) */
static uint32_t rng_below(syn_rng *r, uint32_t n) {
    return (uint32_t)(((unsigned __int128)(rng_next(r) >> 32) * n) >> 32);
}
/* domain-separated stream: tag keeps lexicon/text/vocab draws independent */
static syn_rng rng_make(uint64_t seed, uint64_t tag) {
    syn_rng r;
    r.s = seed * 0xD1B54A32D192ED03ull + tag * 0x9E3779B97F4A7C15ull + 0x1234567ull;
    rng_next(&r);
    return r;
}

/* ------------------------------------------------- portable ln and exp -- */
static const double LN2 = 0.6931471805599453094;

/* scale by 2^e exactly (e small) */
static double pow2i(int e) {
    double v = 1.0, b = (e >= 0) ? 2.0 : 0.5;
    int n = (e >= 0) ? e : -e;
    while (n--) v *= b;
    return v;
}
/* ln(x) for x > 0: x = m * 2^e with m in [1,2); ln m = 2 atanh((m-1)/(m+1)) */
static double syn_ln(double x) {
    int e = 0;
    while (x >= 2.0) { x *= 0.5; e++; }
    while (x < 1.0) { x *= 2.0; e--; }
    double z = (x - 1.0) / (x + 1.0), z2 = z * z, term = z, sum = 0.0;
    for (int k = 1; k < 60; k += 2) { sum += term / (double)k; term *= z2; }
    return 2.0 * sum + (double)e * LN2;
}
/* exp(y): y = n ln2 + r, |r| <= ln2/2, Taylor series for exp(r) */
static double syn_exp(double y) {
    double q = y / LN2;
    int n = (int)(q >= 0 ? q + 0.5 : q - 0.5);
    double r = y - (double)n * LN2, term = 1.0, sum = 1.0;
    for (int k = 1; k < 30; k++) { term = term * r / (double)k; sum += term; }
    return sum * pow2i(n);
}

/* -------------------------------------------------------------- lexicon -- */
typedef struct {
    uint32_t K;
    uint8_t *bytes;      /* concatenated words */
    uint64_t *off;       /* K+1 offsets */
    double *cdf;         /* cumulative Zipf weights, cdf[K-1] = total */
    uint32_t *guide;     /* guide[b] = first k with cdf[k] > b/GUIDE * total */
} syn_lexicon;
#define GUIDE 65536

static const char PUNCT[33] = "!\"#$%&'()*+,-./:;<=>?@[\\]^_`{|}~";
static const uint8_t TR[6][2] = {
    {0xC3, 0xA7}, /* c-cedilla */
    {0xC4, 0x9F}, /* g-breve */
    {0xC4, 0xB1}, /* dotless i */
    {0xC3, 0xB6}, /* o-umlaut */
    {0xC5, 0x9F}, /* s-cedilla */
    {0xC3, 0xBC}, /* u-umlaut */
};

static uint64_t fnv1a(const uint8_t *p, size_t n) {
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < n; i++) { h ^= p[i]; h *= 1099511628211ull; }
    return h;
}

void syn_lexicon_free(syn_lexicon *L) {
    if (!L) return;
    free(L->bytes); free(L->off); free(L->cdf); free(L->guide); free(L);
}

syn_lexicon *syn_lexicon_new(uint64_t seed, uint32_t K, int turkish) {
    if (K == 0) return NULL;
    syn_rng r = rng_make(seed, 1);
    syn_lexicon *L = (syn_lexicon *)calloc(1, sizeof(*L));
    L->K = K;
    L->bytes = (uint8_t *)malloc((size_t)K * 24);
    L->off = (uint64_t *)malloc(sizeof(uint64_t) * ((size_t)K + 1));
    L->cdf = (double *)malloc(sizeof(double) * (size_t)K);
    size_t hcap = 1; while (hcap < 4 * (size_t)K) hcap <<= 1;
    uint32_t *hs = (uint32_t *)malloc(sizeof(uint32_t) * hcap);
    memset(hs, 0xFF, sizeof(uint32_t) * hcap);
    uint64_t pos = 0;
    L->off[0] = 0;
    for (uint32_t w = 0; w < K;) {
        uint32_t len;
        do {                      /* Geometric(1/5) on {1,2,...}, <= 12 */
            len = 1;
            while (rng_below(&r, 5) != 0) len++;
        } while (len > 12);
        uint8_t buf[24];
        size_t n = 0;
        for (uint32_t i = 0; i < len; i++) {
            if (turkish && rng_below(&r, 100) < 30) {
                const uint8_t *t = TR[rng_below(&r, 6)];
                buf[n++] = t[0]; buf[n++] = t[1];
            } else {
                buf[n++] = (uint8_t)('a' + rng_below(&r, 26));
            }
        }
        uint64_t h = fnv1a(buf, n);
        size_t j = h & (hcap - 1);
        int dup = 0;
        while (hs[j] != 0xFFFFFFFFu) {
            uint32_t o = hs[j];
            size_t ol = L->off[o + 1] - L->off[o];
            if (ol == n && memcmp(L->bytes + L->off[o], buf, n) == 0) { dup = 1; break; }
            j = (j + 1) & (hcap - 1);
        }
        if (dup) continue;        /* redraw duplicates */
        hs[j] = w;
        memcpy(L->bytes + pos, buf, n);
        pos += n;
        L->off[++w] = pos;
    }
    free(hs);
    double acc = 0.0;
    for (uint32_t k = 0; k < K; k++) {   /* weight of rank k+1 = (k+1)^-1.1 */
        acc += syn_exp(-1.1 * syn_ln((double)(k + 1)));
        L->cdf[k] = acc;
    }
    L->guide = (uint32_t *)malloc(sizeof(uint32_t) * (GUIDE + 1));
    uint32_t k = 0;
    for (uint32_t b = 0; b <= GUIDE; b++) {
        double u = ((double)b / (double)GUIDE) * acc;
        while (k < K - 1 && !(L->cdf[k] > u)) k++;
        L->guide[b] = k;
    }
    return L;
}

uint64_t syn_lexicon_bytes(const syn_lexicon *L) { return L->off[L->K]; }
uint32_t syn_lexicon_size(const syn_lexicon *L) { return L->K; }
void syn_lexicon_export(const syn_lexicon *L, uint8_t *bytes, uint64_t *off) {
    memcpy(bytes, L->bytes, L->off[L->K]);
    memcpy(off, L->off, sizeof(uint64_t) * ((size_t)L->K + 1));
}

static uint32_t zipf_rank(const syn_lexicon *L, syn_rng *r) {
    double x = rng_unit(r), u = x * L->cdf[L->K - 1];
    uint32_t b = (uint32_t)(x * (double)GUIDE);  /* cdf[k] > u fails below guide[b] */
    uint32_t lo = L->guide[b], hi = L->guide[b + 1];  /* first k with cdf[k] > u */
    while (lo < hi) {
        uint32_t mid = lo + (hi - lo) / 2;
        if (L->cdf[mid] > u) hi = mid; else lo = mid + 1;
    }
    return lo;
}

/* Append one token and its separator; returns bytes written (<= 40). */
static size_t emit_token(const syn_lexicon *L, syn_rng *r, uint8_t *dst) {
    size_t n = 0;
    if (rng_below(r, 100) < 3) {
        uint32_t nd = 1 + rng_below(r, 4);
        for (uint32_t i = 0; i < nd; i++) dst[n++] = (uint8_t)('0' + rng_below(r, 10));
    } else {
        uint32_t w = zipf_rank(L, r);
        size_t wl = L->off[w + 1] - L->off[w];
        memcpy(dst, L->bytes + L->off[w], wl);
        n = wl;
    }
    uint32_t s = rng_below(r, 100);
    if (s < 85) dst[n++] = ' ';
    else if (s < 95) dst[n++] = (uint8_t)PUNCT[rng_below(r, 32)];
    else dst[n++] = '\n';
    return n;
}

/*
 * Corpus of exactly min(target, cap) bytes, minus one if that cut leaves a
 * UTF-8 lead byte without its continuation.  Returns the length written.
 */
uint64_t syn_corpus(const syn_lexicon *L, uint64_t text_seed, uint64_t target,
                    uint8_t *out, uint64_t cap) {
    if (target > cap) target = cap;
    syn_rng r = rng_make(text_seed, 2);
    uint8_t tok[48];
    uint64_t n = 0;
    while (n < target) {
        size_t t = emit_token(L, &r, tok);
        size_t c = (n + t > target) ? (size_t)(target - n) : t;
        memcpy(out + n, tok, c);
        n += c;
    }
    if (n > 0 && out[n - 1] >= 0xC0) n--;   /* drop a dangling lead byte */
    return n;
}

/* Document: tokens until length >= target right after a separator. */
uint64_t syn_document(const syn_lexicon *L, uint64_t text_seed, uint64_t doc_index,
                      uint64_t target, uint8_t *out, uint64_t cap) {
    syn_rng r = rng_make(text_seed * 0x100000000ull + doc_index, 3);
    uint8_t tok[48];
    uint64_t n = 0;
    while (n < target) {
        size_t t = emit_token(L, &r, tok);
        if (n + t > cap) return 0;           /* caller buffer too small */
        memcpy(out + n, tok, t);
        n += t;
    }
    return n;
}

/*
 * Substring vocabulary over `text`: entries 0..255 are the single bytes, the
 * rest are distinct substrings (length >= 2).  Writes at most `bytes_cap`
 * bytes; returns the number of tokens written (== n_tok on success).
 */
uint32_t syn_substring_vocab(const uint8_t *text, uint64_t text_len, uint64_t seed,
                             uint32_t n_tok, uint32_t min_len, uint32_t max_len,
                             uint8_t *bytes, uint64_t bytes_cap, uint64_t *off) {
    if (n_tok < 256 || text_len < 2 || min_len < 2 || max_len < min_len) return 0;
    syn_rng r = rng_make(seed, 4);
    size_t hcap = 1; while (hcap < 4 * (size_t)n_tok) hcap <<= 1;
    uint32_t *hs = (uint32_t *)malloc(sizeof(uint32_t) * hcap);
    memset(hs, 0xFF, sizeof(uint32_t) * hcap);
    uint64_t pos = 0;
    off[0] = 0;
    for (uint32_t b = 0; b < 256; b++) { bytes[pos++] = (uint8_t)b; off[b + 1] = pos; }
    double lo = syn_ln((double)min_len), hi = syn_ln((double)max_len);
    uint32_t t = 256;
    uint64_t guard = 0;
    while (t < n_tok) {
        if (++guard > 64ull * n_tok) break;            /* text too small */
        uint64_t start = (uint64_t)(rng_unit(&r) * (double)text_len);
        if (start >= text_len) start = text_len - 1;
        double x = syn_exp(lo + rng_unit(&r) * (hi - lo));
        uint64_t len = (uint64_t)(x + 0.5);
        if (len < min_len) len = min_len;
        if (len > max_len) len = max_len;
        if (start + len > text_len) len = text_len - start;
        if (len < 2) continue;
        if (pos + len > bytes_cap) break;
        const uint8_t *s = text + start;
        uint64_t h = fnv1a(s, len);
        size_t j = h & (hcap - 1);
        int dup = 0;
        while (hs[j] != 0xFFFFFFFFu) {
            uint32_t o = hs[j];
            uint64_t ol = off[o + 1] - off[o];
            if (ol == len && memcmp(bytes + off[o], s, len) == 0) { dup = 1; break; }
            j = (j + 1) & (hcap - 1);
        }
        if (dup) continue;
        hs[j] = t;
        memcpy(bytes + pos, s, len);
        pos += len;
        off[++t] = pos;
    }
    free(hs);
    return t;
}

/* Exposed for a determinism check of the float helpers. */
double syn_ln_export(double x) { return syn_ln(x); }
double syn_exp_export(double x) { return syn_exp(x); }

/*
 * Synthetic Unigram log-probabilities for n_tok tokens: a Zipf law over a
 * seeded random ranking, score[t] = ln(1 / ((rank(t) + 1) * H)) with H the
 * harmonic number of n_tok, so that exp(score) sums to 1, each rounded to a
 * float32 value (the precision Unigram models store scores in).  Returns 0 on
 * success, -1 when n_tok is 0.
 */
int syn_unigram_scores(uint32_t n_tok, uint64_t seed, double *score) {
    if (n_tok == 0) return -1;
    uint32_t *rank = (uint32_t *)malloc(sizeof(uint32_t) * n_tok);
    if (!rank) return -1;
    for (uint32_t t = 0; t < n_tok; t++) rank[t] = t;
    syn_rng r = rng_make(seed, 5);
    for (uint32_t t = n_tok - 1; t > 0; t--) {          /* Fisher-Yates */
        uint32_t k = rng_below(&r, t + 1);
        uint32_t x = rank[t]; rank[t] = rank[k]; rank[k] = x;
    }
    double H = 0.0;
    for (uint32_t k = n_tok; k > 0; k--) H += 1.0 / (double)k;
    const double lnH = syn_ln(H);
    for (uint32_t t = 0; t < n_tok; t++) score[t] = (double)(float)-(lnH + syn_ln((double)rank[t] + 1.0));
    free(rank);
    return 0;
}
