/*
 * ecc_oracle.c -- reference oracle for lossless fixed-codebook coding of
 * e4m3 byte tensors (Quad Length Codes and single-stage canonical Huffman).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library.
 * It shares no code, header, table or constant with the CUDA library; the
 * two meet only on the seeded inputs of the workload generators.
 *
 * Everything here is deliberately plain and slow: tables are built by
 * selection loops, codes are written and read one bit at a time.  Each
 * function names the passage of the pages it follows:
 *
 *   [QLC]  "Quad Length Codes for Lossless Compression of e4m3"
 *          (gist.science summary of arXiv 2602.17849), section 2
 *          "Metodologia" (areas, 3-bit prefix, per-area length, 256-entry
 *          rank LUT, prefix -> length -> offset -> second LUT decode,
 *          adaptation keeping 4 distinct lengths) and section 5
 *          ("Future Directions": optimise the areas and lengths).
 *   [SSH]  "Single-Stage Huffman Encoder for ML Compression"
 *          (arXiv 2601.10673), TL;DR and abstract (fixed codebook from the
 *          average PMF of earlier batches; compared with per-shard Huffman
 *          and the Shannon bound; KL divergence of Figure 3), and the
 *          euno.news summary, Methodology steps 1-4.
 *   [LLH]  length-limited Huffman, to bound decode tables ([QLC] section 5
 *          "Future Directions" asks for the lengths to be optimised under the
 *          speed constraint): the package-merge algorithm of Larmore and
 *          Hirschberg (J. ACM 37(3), 1990), whose result is an optimal code
 *          among those with no length above the limit.
 *   [ZIP]  "ZipCCL" (gist.science summary of arXiv 2604.27844), section 2.B
 *          "Tecnica di Codifica degli Esponenti": sign and mantissa bits
 *          kept as they are, the 7 most frequent exponents coded in 3 bits
 *          (001-111), any other exponent as the code 000 plus the exponent
 *          itself.
 *
 * Where the pages are silent the readings used are:
 *   - area k is named by the 3-bit prefix equal to k in binary, areas are
 *     filled in rank order, the last non-empty area may be partial and its
 *     unused suffixes are invalid codes;
 *   - ranks sort by count descending, ties by byte value ascending, and
 *     every byte gets a rank (zero-count bytes included);
 *   - Huffman merges the two nodes with the smallest (weight, smallest byte
 *     in the subtree) keys; a lone symbol gets length 1; zero-weight bytes
 *     get no code; codes are canonical (sorted by length, then byte);
 *   - package-merge ties: leaves sort by (weight, byte); when a leaf and a
 *     package weigh the same, the leaf comes first; packages pair items
 *     0-1, 2-3, ... of the previous list; a lone symbol gets length 1;
 *   - escape code on e4m3 (sign bit 7, exponent bits 6-3, mantissa bits
 *     2-0): the page codes BF16's 8-bit exponent and keeps escaped
 *     exponents in a separate array; here the exponent field has 4 bits and
 *     an escaped exponent follows its 000 code in the stream, so a byte's
 *     codeword is [exponent code][4-bit exponent if escaped][sign]
 *     [mantissa] (7 or 11 bits).  The top 7 are the exponents with the
 *     largest summed counts, ties to the smaller exponent; the one ranked r
 *     gets code r + 1.  000 followed by a top-7 exponent is no codeword;
 *   - codewords are written most significant bit first, bits are packed
 *     most significant bit first into bytes;
 *   - the container splits the tensor into chunks of C symbols, pads each
 *     chunk's payload with zero bits to a multiple of 16 bytes, and records
 *     chunk byte offsets (chunk_off[0] = 0, chunk_off[c+1] = chunk_off[c] +
 *     padded bytes of chunk c) and the exact bit count of every sub-block of
 *     S symbols (sub_bits).
 *
 * Return codes: 0 ok, 1 bad argument, 2 capacity, 3 corrupt stream,
 * 4 codebook (symbol without a code, over-long or over-full code).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EO_OK 0
#define EO_ARG 1
#define EO_CAPACITY 2
#define EO_CORRUPT 3
#define EO_CODEBOOK 4

/* ------------------------------------------------------------------ */
/* Histogram ([SSH] Methodology step 1: record symbol frequencies).    */
/* ------------------------------------------------------------------ */
void eo_histogram(const uint8_t *x, uint64_t n, uint64_t *count)
{
    for (int b = 0; b < 256; b++)
        count[b] = 0;
    for (uint64_t i = 0; i < n; i++)
        count[x[i]] += 1;
}

/* ------------------------------------------------------------------ */
/* Rank LUT ([QLC] section 2, "Implementazione tramite LUT": symbols   */
/* sorted by decreasing probability get indices 0..255).               */
/* rank[b] = rank of byte b; by_rank[r] = byte holding rank r.         */
/* ------------------------------------------------------------------ */
void eo_rank(const uint64_t *count, uint8_t *rank, uint8_t *by_rank)
{
    int taken[256];
    for (int b = 0; b < 256; b++)
        taken[b] = 0;
    for (int r = 0; r < 256; r++) {
        int best = -1;
        for (int b = 0; b < 256; b++) {
            if (taken[b])
                continue;
            /* strictly larger count wins, so the smaller byte wins ties */
            if (best < 0 || count[b] > count[best])
                best = b;
        }
        taken[best] = 1;
        rank[best] = (uint8_t)r;
        by_rank[r] = (uint8_t)best;
    }
}

/* ------------------------------------------------------------------ */
/* Area layout ([QLC] section 2, "Partizionamento in Aree" and the     */
/* base example: five areas of 8, one of 16, one of 32, the remaining  */
/* 168).  With p prefix bits there are 2^p areas ([QLC] section 5:     */
/* optimise the number of areas; the page's code has p = 3).  Area k   */
/* can hold 2^width[k] ranks; areas are filled in order.  Returns the   */
/* number of ranks the areas can hold, capped at 256.                  */
/* ------------------------------------------------------------------ */
int eo_gqlc_layout(int p, const uint8_t *width, int32_t *start, int32_t *size)
{
    int next = 0;
    for (int k = 0; k < (1 << p); k++) {
        int cap = 1 << width[k];
        int left = 256 - next;
        int take = cap < left ? cap : left;
        if (take < 0)
            take = 0;
        start[k] = next;
        size[k] = take;
        next += take;
    }
    return next;
}

int eo_qlc_layout(const uint8_t *width, int32_t *start, int32_t *size)
{
    return eo_gqlc_layout(3, width, start, size);
}

/* Code of every byte under widths of 2^p areas: rank r in area k gets the
 * code (k << width[k]) | (r - start[k]) of length p + width[k]. */
int eo_gqlc_codebook(const uint64_t *count, int p, const uint8_t *width, uint8_t *len,
                     uint64_t *code, uint8_t *by_rank)
{
    int32_t start[8], size[8];
    uint8_t rank[256];
    if (p < 1 || p > 3)
        return EO_ARG;
    for (int k = 0; k < (1 << p); k++)
        if (width[k] > 8)
            return EO_ARG;
    if (eo_gqlc_layout(p, width, start, size) < 256)
        return EO_ARG;
    eo_rank(count, rank, by_rank);
    for (int b = 0; b < 256; b++) {
        int r = rank[b];
        int k = 0;
        while (!(r >= start[k] && r < start[k] + size[k]))
            k++;
        len[b] = (uint8_t)(p + width[k]);
        code[b] = ((uint64_t)k << width[k]) | (uint64_t)(r - start[k]);
    }
    return EO_OK;
}

int eo_qlc_codebook(const uint64_t *count, const uint8_t *width, uint8_t *len,
                    uint64_t *code, uint8_t *by_rank)
{
    return eo_gqlc_codebook(count, 3, width, len, code, by_rank);
}

/* Expected-length cost (integer sum of count x length) of widths b of the
 * 2^p areas when ranks are filled in order; counts_by_rank is sorted
 * descending.  Also reports how many distinct lengths the non-empty areas
 * use. */
static uint64_t qlc_cost(int p, const uint64_t *counts_by_rank, const uint8_t *b, int *distinct, int *capacity)
{
    int32_t start[8], size[8];
    int cap = 0;
    for (int k = 0; k < (1 << p); k++)
        cap += 1 << b[k];
    *capacity = cap;
    eo_gqlc_layout(p, b, start, size);
    uint64_t cost = 0;
    int seen[12] = {0};
    int nd = 0;
    for (int k = 0; k < (1 << p); k++) {
        if (size[k] == 0)
            continue;
        int L = p + b[k];
        if (!seen[L]) {
            seen[L] = 1;
            nd++;
        }
        for (int r = start[k]; r < start[k] + size[k]; r++)
            cost += counts_by_rank[r] * (uint64_t)L;
    }
    *distinct = nd;
    return cost;
}

/* Adapted QLC ([QLC] section 2 "Adattabilita": change the symbols per area
 * and the lengths, keep 4 distinct lengths; section 5: optimise the areas
 * and lengths).  Exhaustive search over widths in 0..8 for the 2^p areas
 * with capacity >= 256 (require_full: capacity == 256) and at most
 * max_distinct distinct lengths, minimising the integer cost; ties go to the
 * lexicographically smallest width vector.  nondecreasing_only restricts the
 * search to b0 <= b1 <= ...; 0 tries all 9^(2^p).  Returns EO_ARG if no
 * vector qualifies. */
int eo_gqlc_search(const uint64_t *count, int p, int max_distinct, int require_full,
                   int nondecreasing_only, uint8_t *width_out, uint64_t *cost_out)
{
    uint8_t rank[256], by_rank[256];
    uint64_t sorted[256];
    if (p < 1 || p > 3)
        return EO_ARG;
    const int A = 1 << p;
    eo_rank(count, rank, by_rank);
    for (int r = 0; r < 256; r++)
        sorted[r] = count[by_rank[r]];

    int found = 0;
    uint64_t best = 0;
    uint8_t bestb[8] = {0};
    uint8_t b[8] = {0};
    /* odometer over 9^A width vectors in lexicographic order */
    for (;;) {
        int ok = 1;
        if (nondecreasing_only)
            for (int k = 1; k < A; k++)
                if (b[k] < b[k - 1])
                    ok = 0;
        if (ok) {
            int nd, cap;
            uint64_t c = qlc_cost(p, sorted, b, &nd, &cap);
            int cap_ok = require_full ? (cap == 256) : (cap >= 256);
            if (cap_ok && nd <= max_distinct && (!found || c < best)) {
                found = 1;
                best = c;
                memcpy(bestb, b, 8);
            }
        }
        int k = A - 1;
        while (k >= 0 && b[k] == 8) {
            b[k] = 0;
            k--;
        }
        if (k < 0)
            break;
        b[k]++;
    }
    if (!found)
        return EO_ARG;
    memcpy(width_out, bestb, (size_t)A);
    for (int k = A; k < 8; k++)
        width_out[k] = 0;
    *cost_out = best;
    return EO_OK;
}

int eo_qlc_search(const uint64_t *count, int max_distinct, int require_full,
                  int nondecreasing_only, uint8_t *width_out, uint64_t *cost_out)
{
    return eo_gqlc_search(count, 3, max_distinct, require_full, nondecreasing_only, width_out, cost_out);
}

/* ------------------------------------------------------------------ */
/* Huffman code lengths ([QLC] section 1 and [SSH] Methodology step 3: */
/* build the Huffman tree of a distribution).  Textbook construction:  */
/* repeatedly merge the two live nodes with the smallest keys; a       */
/* leaf's length is its depth.  Found by linear scans, no heap.        */
/* ------------------------------------------------------------------ */
int eo_huffman_lengths(const uint64_t *weight, uint8_t *len)
{
    uint64_t w[511];
    int minsym[511], parent[511], live[511];
    int nodes = 0, nlive = 0;
    int leaf_of[256];

    for (int b = 0; b < 256; b++) {
        len[b] = 0;
        leaf_of[b] = -1;
        if (weight[b] == 0)
            continue;
        w[nodes] = weight[b];
        minsym[nodes] = b;
        parent[nodes] = -1;
        live[nodes] = 1;
        leaf_of[b] = nodes;
        nodes++;
        nlive++;
    }
    if (nodes == 0)
        return EO_OK;
    if (nodes == 1) {
        for (int b = 0; b < 256; b++)
            if (leaf_of[b] >= 0)
                len[b] = 1;
        return EO_OK;
    }
    while (nlive > 1) {
        int pick[2];
        for (int t = 0; t < 2; t++) {
            int best = -1;
            for (int i = 0; i < nodes; i++) {
                if (!live[i])
                    continue;
                if (best < 0 || w[i] < w[best] ||
                    (w[i] == w[best] && minsym[i] < minsym[best]))
                    best = i;
            }
            live[best] = 0;
            pick[t] = best;
        }
        /* weights are counts; a sum that wraps would break the order */
        if (w[pick[0]] > UINT64_MAX - w[pick[1]])
            return EO_ARG;
        w[nodes] = w[pick[0]] + w[pick[1]];
        minsym[nodes] = minsym[pick[0]] < minsym[pick[1]] ? minsym[pick[0]] : minsym[pick[1]];
        parent[nodes] = -1;
        live[nodes] = 1;
        parent[pick[0]] = nodes;
        parent[pick[1]] = nodes;
        nodes++;
        nlive--;
    }
    for (int b = 0; b < 256; b++) {
        if (leaf_of[b] < 0)
            continue;
        int d = 0;
        for (int i = leaf_of[b]; parent[i] >= 0; i = parent[i])
            d++;
        if (d > 255)
            return EO_CODEBOOK;
        len[b] = (uint8_t)d;
    }
    return EO_OK;
}

/* Canonical codes from lengths: visit bytes by (length, byte); the first
 * gets all-zero bits, each next one is (previous + 1) shifted left by the
 * length increase.  Lengths above 64 or an over-full set fail. */
int eo_canonical_codes(const uint8_t *len, uint64_t *code)
{
    int first = 1, prev_len = 0;
    uint64_t c = 0;
    for (int b = 0; b < 256; b++)
        code[b] = 0;
    for (int L = 1; L <= 255; L++) {
        for (int b = 0; b < 256; b++) {
            if (len[b] != L)
                continue;
            if (L > 64)
                return EO_CODEBOOK;
            if (first) {
                c = 0;
                first = 0;
            } else {
                c = c + 1;
                for (int s = prev_len; s < L; s++) {
                    if (c >> 63)
                        return EO_CODEBOOK;
                    c <<= 1;
                }
            }
            if (L < 64 && (c >> L) != 0)
                return EO_CODEBOOK; /* more codes than the lengths allow */
            code[b] = c;
            prev_len = L;
        }
    }
    return EO_OK;
}

/* ------------------------------------------------------------------ */
/* Container checks shared by encode and decode of this file.          */
/* ------------------------------------------------------------------ */
static int pow2_in(uint64_t v, uint64_t lo, uint64_t hi)
{
    if (v < lo || v > hi)
        return 0;
    return (v & (v - 1)) == 0;
}

static int container_args(uint32_t C, uint32_t S)
{
    if (!pow2_in(C, 1024, 65536) || !pow2_in(S, 64, 1024) || S > C)
        return 0;
    return 1;
}

static uint64_t pad16(uint64_t bytes)
{
    return (bytes + 15) / 16 * 16;
}

/* ------------------------------------------------------------------ */
/* Encode ([QLC] "Codifica": the encoder looks the code up in the LUT; */
/* [SSH] Methodology step 4: encode with the precomputed codebook).    */
/* One bit at a time.                                                  */
/* ------------------------------------------------------------------ */
int eo_encode(const uint8_t *x, uint64_t n, const uint8_t *len, const uint64_t *code,
              uint32_t C, uint32_t S, uint8_t *out, uint64_t cap,
              uint64_t *chunk_off, uint16_t *sub_bits, uint64_t *total_bits)
{
    if (!container_args(C, S))
        return EO_ARG;
    for (int b = 0; b < 256; b++)
        if (len[b] > 64)
            return EO_CODEBOOK;
    for (uint64_t i = 0; i < cap; i++)
        out[i] = 0;
    uint64_t n_chunks = (n + C - 1) / C;
    uint64_t pos = 0; /* byte offset of the current chunk */
    uint64_t total = 0;
    int err = EO_OK;
    chunk_off[0] = 0;
    for (uint64_t c = 0; c < n_chunks; c++) {
        uint64_t lo = c * C, hi = lo + C < n ? lo + C : n;
        uint64_t bit = 0;       /* bit offset within the chunk */
        uint64_t sub_start = 0; /* bit offset where the sub-block began */
        for (uint64_t i = lo; i < hi; i++) {
            uint8_t s = x[i];
            if (len[s] == 0)
                return EO_CODEBOOK;
            if (i % S == 0)
                sub_start = bit;
            for (int t = len[s] - 1; t >= 0; t--) {
                int v = (int)((code[s] >> t) & 1);
                uint64_t at = pos * 8 + bit;
                if (at / 8 < cap) {
                    if (v)
                        out[at / 8] |= (uint8_t)(0x80u >> (at % 8));
                } else {
                    err = EO_CAPACITY;
                }
                bit++;
            }
            if ((i + 1) % S == 0 || i + 1 == hi) {
                uint64_t sb = bit - sub_start;
                if (sb > 65535)
                    return EO_ARG;
                sub_bits[i / S] = (uint16_t)sb;
            }
        }
        uint64_t bytes = pad16((bit + 7) / 8);
        if (pos + bytes > cap)
            err = EO_CAPACITY;
        pos += bytes;
        chunk_off[c + 1] = pos;
        total += bit;
    }
    *total_bits = total;
    return err;
}

/* MSB-first bit reader over one chunk: bits [at, limit) of buf. */
typedef struct {
    const uint8_t *buf;
    uint64_t at, limit;
} eo_reader;

static int read_bit(eo_reader *r, int *v)
{
    if (r->at >= r->limit)
        return -1;
    *v = (r->buf[r->at / 8] >> (7 - (r->at % 8))) & 1;
    r->at++;
    return 0;
}

static int read_bits(eo_reader *r, int nbits, uint64_t *v)
{
    uint64_t acc = 0;
    for (int t = 0; t < nbits; t++) {
        int bitv;
        if (read_bit(r, &bitv))
            return -1;
        acc = (acc << 1) | (uint64_t)bitv;
    }
    *v = acc;
    return 0;
}

/* Common container walk: checks offsets, calls the symbol decoder once per
 * symbol, checks every sub-block's bit count and every chunk's padding. */
typedef int (*eo_symbol_fn)(eo_reader *r, const void *ctx, uint8_t *sym);

static int decode_container(const uint8_t *in, uint64_t in_bytes, const uint64_t *chunk_off,
                            const uint16_t *sub_bits, uint64_t n, uint32_t C, uint32_t S,
                            eo_symbol_fn fn, const void *ctx, uint8_t *out)
{
    if (!container_args(C, S))
        return EO_ARG;
    uint64_t n_chunks = (n + C - 1) / C;
    if (chunk_off[0] != 0)
        return EO_CORRUPT;
    for (uint64_t c = 0; c < n_chunks; c++) {
        uint64_t b0 = chunk_off[c], b1 = chunk_off[c + 1];
        if (b1 < b0 || b1 > in_bytes || (b0 % 16) || (b1 % 16))
            return EO_CORRUPT;
        eo_reader r = {in, b0 * 8, b1 * 8};
        uint64_t lo = c * C, hi = lo + C < n ? lo + C : n;
        uint64_t sub_start = r.at;
        for (uint64_t i = lo; i < hi; i++) {
            if (i % S == 0)
                sub_start = r.at;
            if (fn(&r, ctx, &out[i]))
                return EO_CORRUPT;
            if ((i + 1) % S == 0 || i + 1 == hi)
                if (r.at - sub_start != sub_bits[i / S])
                    return EO_CORRUPT;
        }
        /* the chunk must end where its padded payload says */
        if (pad16((r.at - b0 * 8 + 7) / 8) != b1 - b0)
            return EO_CORRUPT;
        while (r.at < r.limit) {
            int v;
            read_bit(&r, &v);
            if (v)
                return EO_CORRUPT; /* padding must be zero */
        }
    }
    return EO_OK;
}

/* ------------------------------------------------------------------ */
/* QLC decode ([QLC] "Decodifica": read the first 3 bits -> area ->    */
/* total length; read the remaining bits; add the area's offset; a     */
/* second LUT maps the rank back to the symbol).                       */
/* ------------------------------------------------------------------ */
typedef struct {
    int p;
    uint8_t width[8];
    int32_t start[8], size[8];
    const uint8_t *by_rank;
} qlc_ctx;

static int qlc_symbol(eo_reader *r, const void *vctx, uint8_t *sym)
{
    const qlc_ctx *q = (const qlc_ctx *)vctx;
    uint64_t k, v;
    if (read_bits(r, q->p, &k))
        return -1;
    if (read_bits(r, q->width[k], &v))
        return -1;
    if (v >= (uint64_t)q->size[k])
        return -1; /* unused suffix of a partial or empty area */
    *sym = q->by_rank[q->start[k] + (int)v];
    return 0;
}

int eo_decode_gqlc(const uint8_t *in, uint64_t in_bytes, const uint64_t *chunk_off,
                   const uint16_t *sub_bits, uint64_t n, uint32_t C, uint32_t S,
                   int p, const uint8_t *width, const uint8_t *by_rank, uint8_t *out)
{
    qlc_ctx q;
    if (p < 1 || p > 3)
        return EO_ARG;
    q.p = p;
    for (int k = 0; k < (1 << p); k++) {
        if (width[k] > 8)
            return EO_ARG;
        q.width[k] = width[k];
    }
    if (eo_gqlc_layout(p, width, q.start, q.size) < 256)
        return EO_ARG;
    q.by_rank = by_rank;
    return decode_container(in, in_bytes, chunk_off, sub_bits, n, C, S, qlc_symbol, &q, out);
}

int eo_decode_qlc(const uint8_t *in, uint64_t in_bytes, const uint64_t *chunk_off,
                  const uint16_t *sub_bits, uint64_t n, uint32_t C, uint32_t S,
                  const uint8_t *width, const uint8_t *by_rank, uint8_t *out)
{
    return eo_decode_gqlc(in, in_bytes, chunk_off, sub_bits, n, C, S, 3, width, by_rank, out);
}

/* ------------------------------------------------------------------ */
/* Huffman decode: bit-serial canonical walk, one bit per step, which   */
/* is the binary-tree traversal [QLC] section 1 describes.  After L    */
/* bits the value v is a code of length L exactly when                 */
/* first[L] <= v < first[L] + count[L].                                */
/* ------------------------------------------------------------------ */
typedef struct {
    int maxlen;
    uint64_t first[65];
    int count[65];
    int index[65];
    uint8_t sorted[256];
} huff_ctx;

static int huff_symbol(eo_reader *r, const void *vctx, uint8_t *sym)
{
    const huff_ctx *h = (const huff_ctx *)vctx;
    uint64_t v = 0;
    for (int L = 1; L <= h->maxlen; L++) {
        int bitv;
        if (read_bit(r, &bitv))
            return -1;
        v = (v << 1) | (uint64_t)bitv;
        if (h->count[L] > 0 && v >= h->first[L] && v - h->first[L] < (uint64_t)h->count[L]) {
            *sym = h->sorted[h->index[L] + (int)(v - h->first[L])];
            return 0;
        }
    }
    return -1;
}

int eo_decode_huffman(const uint8_t *in, uint64_t in_bytes, const uint64_t *chunk_off,
                      const uint16_t *sub_bits, uint64_t n, uint32_t C, uint32_t S,
                      const uint8_t *len, uint8_t *out)
{
    huff_ctx h;
    uint64_t code[256];
    if (eo_canonical_codes(len, code))
        return EO_CODEBOOK;
    memset(&h, 0, sizeof h);
    int m = 0;
    for (int L = 1; L <= 64; L++) {
        h.index[L] = m;
        for (int b = 0; b < 256; b++) {
            if (len[b] != L)
                continue;
            if (h.count[L] == 0)
                h.first[L] = code[b];
            h.count[L]++;
            h.sorted[m++] = (uint8_t)b;
            h.maxlen = L;
        }
    }
    return decode_container(in, in_bytes, chunk_off, sub_bits, n, C, S, huff_symbol, &h, out);
}

/* ------------------------------------------------------------------ */
/* Length-limited Huffman by package-merge ([LLH]).  List 1 holds the   */
/* leaves sorted by weight; list d merges the leaves with the packages  */
/* of list d-1 (pairs of consecutive items).  The first 2n-2 items of   */
/* list max_len are selected; a symbol's length is the number of times */
/* it occurs in them, counting inside packages.                        */
/* ------------------------------------------------------------------ */
typedef struct {
    uint64_t w;
    int sym;  /* >= 0: a leaf */
    int a, b; /* package: items a and b of the previous list */
} llh_item;

static void llh_count(llh_item **lists, int level, int i, uint8_t *len)
{
    const llh_item *it = &lists[level][i];
    if (it->sym >= 0) {
        len[it->sym]++;
        return;
    }
    llh_count(lists, level - 1, it->a, len);
    llh_count(lists, level - 1, it->b, len);
}

int eo_huffman_limited(const uint64_t *weight, int max_len, uint8_t *len)
{
    int leaf_sym[256], n = 0;
    uint64_t total = 0;
    for (int b = 0; b < 256; b++) {
        len[b] = 0;
        if (weight[b]) {
            if (weight[b] >= ((uint64_t)1 << 62) - total)
                return EO_ARG; /* sums of packages must fit 64 bits */
            total += weight[b];
            leaf_sym[n++] = b;
        }
    }
    if (n == 0 || max_len < 1 || max_len > 64)
        return EO_ARG;
    if (n == 1) {
        len[leaf_sym[0]] = 1;
        return EO_OK;
    }
    if (max_len < 63 && ((uint64_t)1 << max_len) < (uint64_t)n)
        return EO_CODEBOOK; /* no prefix code of n words fits max_len bits */
    /* leaves by (weight, byte): selection sort */
    for (int i = 0; i < n; i++) {
        int m = i;
        for (int j = i + 1; j < n; j++) {
            const uint64_t wj = weight[leaf_sym[j]], wm = weight[leaf_sym[m]];
            if (wj < wm || (wj == wm && leaf_sym[j] < leaf_sym[m]))
                m = j;
        }
        const int t = leaf_sym[i];
        leaf_sym[i] = leaf_sym[m];
        leaf_sym[m] = t;
    }
    llh_item *lists[65];
    int cnt[65];
    for (int d = 1; d <= max_len; d++)
        lists[d] = (llh_item *)malloc(sizeof(llh_item) * 2 * 256);
    for (int i = 0; i < n; i++) {
        lists[1][i].w = weight[leaf_sym[i]];
        lists[1][i].sym = leaf_sym[i];
        lists[1][i].a = lists[1][i].b = -1;
    }
    cnt[1] = n;
    for (int d = 2; d <= max_len; d++) {
        const int npk = cnt[d - 1] / 2;
        int i = 0, j = 0, k = 0;
        while (i < n || j < npk) {
            const uint64_t pw = j < npk ? lists[d - 1][2 * j].w + lists[d - 1][2 * j + 1].w : 0;
            if (i < n && (j >= npk || weight[leaf_sym[i]] <= pw)) { /* leaf first on a tie */
                lists[d][k].w = weight[leaf_sym[i]];
                lists[d][k].sym = leaf_sym[i];
                lists[d][k].a = lists[d][k].b = -1;
                i++;
            } else {
                lists[d][k].w = pw;
                lists[d][k].sym = -1;
                lists[d][k].a = 2 * j;
                lists[d][k].b = 2 * j + 1;
                j++;
            }
            k++;
        }
        cnt[d] = k;
    }
    for (int i = 0; i < 2 * n - 2; i++)
        llh_count(lists, max_len, i, len);
    for (int d = 1; d <= max_len; d++)
        free(lists[d]);
    return EO_OK;
}

/* ------------------------------------------------------------------ */
/* Escape code on e4m3 exponents ([ZIP] section 2.B): top-7 exponents   */
/* in 3 bits, others as 000 plus the 4-bit exponent; sign and mantissa  */
/* follow as they are.                                                 */
/* ------------------------------------------------------------------ */
int eo_escape_codebook(const uint64_t *count, uint8_t *len, uint64_t *code, uint8_t *top)
{
    uint64_t ecount[16] = {0};
    int taken[16] = {0};
    for (int b = 0; b < 256; b++)
        ecount[(b >> 3) & 15] += count[b];
    int rank_of[16];
    for (int e = 0; e < 16; e++)
        rank_of[e] = -1;
    for (int r = 0; r < 7; r++) { /* selection: largest count, then smaller exponent */
        int best = -1;
        for (int e = 0; e < 16; e++)
            if (!taken[e] && (best < 0 || ecount[e] > ecount[best]))
                best = e;
        taken[best] = 1;
        rank_of[best] = r;
        top[r] = (uint8_t)best;
    }
    for (int b = 0; b < 256; b++) {
        const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
        const uint64_t sm = ((uint64_t)s << 3) | (uint64_t)m; /* 4 bits */
        if (rank_of[e] >= 0) {
            code[b] = ((uint64_t)(rank_of[e] + 1) << 4) | sm;
            len[b] = 7;
        } else {
            code[b] = ((uint64_t)e << 4) | sm; /* 000 eeee s mmm */
            len[b] = 11;
        }
    }
    return EO_OK;
}

typedef struct {
    int rank_of[16];
    uint8_t top[7];
} esc_ctx;

static int escape_symbol(eo_reader *r, const void *vctx, uint8_t *sym)
{
    const esc_ctx *q = (const esc_ctx *)vctx;
    uint64_t p, e, s, m;
    if (read_bits(r, 3, &p))
        return -1;
    if (p == 0) {
        if (read_bits(r, 4, &e))
            return -1;
        if (q->rank_of[e] >= 0)
            return -1; /* a top-7 exponent has a short code: not a codeword */
    } else {
        e = q->top[p - 1];
    }
    if (read_bits(r, 1, &s) || read_bits(r, 3, &m))
        return -1;
    *sym = (uint8_t)((s << 7) | (e << 3) | m);
    return 0;
}

int eo_decode_escape(const uint8_t *in, uint64_t in_bytes, const uint64_t *chunk_off,
                     const uint16_t *sub_bits, uint64_t n, uint32_t C, uint32_t S,
                     const uint8_t *top, uint8_t *out)
{
    esc_ctx q;
    for (int e = 0; e < 16; e++)
        q.rank_of[e] = -1;
    for (int r = 0; r < 7; r++) {
        if (top[r] > 15 || q.rank_of[top[r]] >= 0)
            return EO_ARG;
        q.rank_of[top[r]] = r;
        q.top[r] = top[r];
    }
    return decode_container(in, in_bytes, chunk_off, sub_bits, n, C, S, escape_symbol, &q, out);
}

/* ------------------------------------------------------------------ */
/* Figures in float64 ([SSH] TL;DR: compressibility against the        */
/* Shannon bound; Figure 3: KL divergence of shard PMFs from the        */
/* average PMF).                                                       */
/* ------------------------------------------------------------------ */

/* Shannon entropy in bits per symbol: -sum p log2 p. */
double eo_entropy_bits(const uint64_t *count)
{
    double n = 0.0, h = 0.0;
    for (int b = 0; b < 256; b++)
        n += (double)count[b];
    if (n == 0.0)
        return 0.0;
    for (int b = 0; b < 256; b++) {
        if (count[b] == 0)
            continue;
        double p = (double)count[b] / n;
        h -= p * log2(p);
    }
    return h;
}

/* D(P || Q) in bits, P and Q given as counts; +inf if Q misses a symbol
 * that P has. */
double eo_kl_bits(const uint64_t *p_count, const uint64_t *q_count)
{
    double np = 0.0, nq = 0.0, d = 0.0;
    for (int b = 0; b < 256; b++) {
        np += (double)p_count[b];
        nq += (double)q_count[b];
    }
    for (int b = 0; b < 256; b++) {
        if (p_count[b] == 0)
            continue;
        if (q_count[b] == 0)
            return INFINITY;
        double p = (double)p_count[b] / np;
        double q = (double)q_count[b] / nq;
        d += p * log2(p / q);
    }
    return d;
}

/* Total code bits sum(count x length); UINT64_MAX if a counted byte has no
 * code. */
uint64_t eo_code_bits(const uint64_t *count, const uint8_t *len)
{
    uint64_t bits = 0;
    for (int b = 0; b < 256; b++) {
        if (count[b] == 0)
            continue;
        if (len[b] == 0)
            return UINT64_MAX;
        bits += count[b] * (uint64_t)len[b];
    }
    return bits;
}

/* ------------------------------------------------------------------ */
/* Escape code on BF16 exponents ([ZIP] section 2.A and 2.B).  A BF16   */
/* value is sign (bit 15), exponent (bits 14-7, bias 127) and mantissa   */
/* (bits 6-0).  The 7 exponents of the table get the 3-bit codes        */
/* 001-111 by rank; any other exponent is coded 000 followed by its 8    */
/* bits (the page moves escaped exponents to a separate array; here     */
/* they follow their 000 code in the stream, as in the e4m3 variant).   */
/* Sign and mantissa follow as they are: a value's codeword is          */
/* [code][exponent if escaped][sign][mantissa], 11 or 19 bits.  The      */
/* container is the byte container's, with 16-bit symbols.              */
/* ------------------------------------------------------------------ */

/* Histogram of the exponent field. */
int eo_bf16_exponent_counts(const uint16_t *x, uint64_t n, uint64_t *count)
{
    for (int e = 0; e < 256; e++)
        count[e] = 0;
    for (uint64_t i = 0; i < n; i++)
        count[(x[i] >> 7) & 0xFF]++;
    return EO_OK;
}

/* Top 7 exponents by count ([ZIP] 2.A: the 7 most frequent exponents):
 * selection, largest count first, ties to the smaller exponent. */
int eo_bf16_top7_from_counts(const uint64_t *count, uint8_t *top)
{
    int taken[256] = {0};
    for (int r = 0; r < 7; r++) {
        int best = -1;
        for (int e = 0; e < 256; e++)
            if (!taken[e] && (best < 0 || count[e] > count[best]))
                best = e;
        taken[best] = 1;
        top[r] = (uint8_t)best;
    }
    return EO_OK;
}

/* Probability that x ~ N(0, sigma^2), rounded to BF16 (round to nearest,
 * ties to even), has exponent field e ([ZIP] 2.A: the table follows from
 * the standard deviation alone).  A BF16 value with exponent field e
 * (1..254) has magnitude in [2^(e-127), 2^(e-126)); rounding moves each
 * boundary 2^k down to the midpoint 2^k (1 - 2^-9) between 2^k and the
 * largest BF16 below it (the tie goes to 2^k, whose mantissa is even).
 * Field 0 holds zero and the subnormals (|x| below 2^-126 (1 - 2^-9)); field
 * 255 the values that round past the largest finite BF16 (not reached by
 * any sigma a tensor has).  P(|x| >= a) = erfc(a / (sigma sqrt 2)). */
static double bf16_tail(double a, double sigma)
{
    return erfc(a / (sigma * sqrt(2.0)));
}

int eo_bf16_exponent_probs(double sigma, double *prob)
{
    if (!(sigma > 0.0))
        return EO_ARG;
    const double shrink = 1.0 - ldexp(1.0, -9);
    for (int e = 0; e < 256; e++) {
        double lo, hi;
        if (e == 0) {
            lo = 0.0;
            hi = ldexp(1.0, -126) * shrink;
        } else if (e == 255) {
            lo = ldexp(1.0, 128) * shrink;
            hi = INFINITY;
        } else {
            lo = ldexp(1.0, e - 127) * shrink;
            hi = ldexp(1.0, e - 126) * shrink;
        }
        prob[e] = bf16_tail(lo, sigma) - (isinf(hi) ? 0.0 : bf16_tail(hi, sigma));
    }
    return EO_OK;
}

/* Top 7 exponents of N(0, sigma^2): the 7 largest probabilities, ties to
 * the smaller exponent. */
int eo_bf16_top7_from_sigma(double sigma, uint8_t *top)
{
    double prob[256];
    if (eo_bf16_exponent_probs(sigma, prob))
        return EO_ARG;
    int taken[256] = {0};
    for (int r = 0; r < 7; r++) {
        int best = -1;
        for (int e = 0; e < 256; e++)
            if (!taken[e] && (best < 0 || prob[e] > prob[best]))
                best = e;
        taken[best] = 1;
        top[r] = (uint8_t)best;
    }
    return EO_OK;
}

static int bf16_rank_table(const uint8_t *top, int *rank_of)
{
    for (int e = 0; e < 256; e++)
        rank_of[e] = -1;
    for (int r = 0; r < 7; r++) {
        if (rank_of[top[r]] >= 0)
            return EO_ARG; /* an exponent listed twice */
        rank_of[top[r]] = r;
    }
    return EO_OK;
}

/* Code and length of one BF16 value. */
static void bf16_code(uint16_t v, const int *rank_of, uint64_t *code, int *len)
{
    const uint64_t s = (v >> 15) & 1, e = (v >> 7) & 0xFF, m = v & 0x7F;
    const uint64_t sm = (s << 7) | m; /* 8 bits */
    if (rank_of[e] >= 0) {
        *code = ((uint64_t)(rank_of[e] + 1) << 8) | sm; /* ccc s mmmmmmm */
        *len = 11;
    } else {
        *code = (e << 8) | sm; /* 000 eeeeeeee s mmmmmmm */
        *len = 19;
    }
}

/* Encode n BF16 values into the container, one bit at a time. */
int eo_bf16_escape_encode(const uint16_t *x, uint64_t n, const uint8_t *top, uint32_t C, uint32_t S,
                          uint8_t *out, uint64_t cap, uint64_t *chunk_off, uint16_t *sub_bits,
                          uint64_t *total_bits)
{
    int rank_of[256];
    if (!container_args(C, S) || bf16_rank_table(top, rank_of))
        return EO_ARG;
    for (uint64_t i = 0; i < cap; i++)
        out[i] = 0;
    uint64_t n_chunks = (n + C - 1) / C;
    uint64_t pos = 0, total = 0;
    int err = EO_OK;
    chunk_off[0] = 0;
    for (uint64_t c = 0; c < n_chunks; c++) {
        uint64_t lo = c * C, hi = lo + C < n ? lo + C : n;
        uint64_t bit = 0, sub_start = 0;
        for (uint64_t i = lo; i < hi; i++) {
            uint64_t code;
            int len;
            bf16_code(x[i], rank_of, &code, &len);
            if (i % S == 0)
                sub_start = bit;
            for (int t = len - 1; t >= 0; t--) {
                uint64_t at = pos * 8 + bit;
                if (at / 8 < cap) {
                    if ((code >> t) & 1)
                        out[at / 8] |= (uint8_t)(0x80u >> (at % 8));
                } else {
                    err = EO_CAPACITY;
                }
                bit++;
            }
            if ((i + 1) % S == 0 || i + 1 == hi)
                sub_bits[i / S] = (uint16_t)(bit - sub_start);
        }
        uint64_t bytes = pad16((bit + 7) / 8);
        if (pos + bytes > cap)
            err = EO_CAPACITY;
        pos += bytes;
        chunk_off[c + 1] = pos;
        total += bit;
    }
    *total_bits = total;
    return err;
}

/* Decode the container back to BF16 values, one bit at a time, with the
 * same checks as the byte container (offsets, sub-block bit counts, zero
 * padding); 000 followed by an exponent of the table is no codeword. */
int eo_bf16_escape_decode(const uint8_t *in, uint64_t in_bytes, const uint64_t *chunk_off,
                          const uint16_t *sub_bits, uint64_t n, uint32_t C, uint32_t S, const uint8_t *top,
                          uint16_t *out)
{
    int rank_of[256];
    if (!container_args(C, S) || bf16_rank_table(top, rank_of))
        return EO_ARG;
    uint64_t n_chunks = (n + C - 1) / C;
    if (chunk_off[0] != 0)
        return EO_CORRUPT;
    for (uint64_t c = 0; c < n_chunks; c++) {
        uint64_t b0 = chunk_off[c], b1 = chunk_off[c + 1];
        if (b1 < b0 || b1 > in_bytes || (b0 % 16) || (b1 % 16))
            return EO_CORRUPT;
        eo_reader r = {in, b0 * 8, b1 * 8};
        uint64_t lo = c * C, hi = lo + C < n ? lo + C : n;
        uint64_t sub_start = r.at;
        for (uint64_t i = lo; i < hi; i++) {
            uint64_t p, e, s, m;
            if (i % S == 0)
                sub_start = r.at;
            if (read_bits(&r, 3, &p))
                return EO_CORRUPT;
            if (p == 0) {
                if (read_bits(&r, 8, &e))
                    return EO_CORRUPT;
                if (rank_of[e] >= 0)
                    return EO_CORRUPT;
            } else {
                e = top[p - 1];
            }
            if (read_bits(&r, 1, &s) || read_bits(&r, 7, &m))
                return EO_CORRUPT;
            out[i] = (uint16_t)((s << 15) | (e << 7) | m);
            if ((i + 1) % S == 0 || i + 1 == hi)
                if (r.at - sub_start != sub_bits[i / S])
                    return EO_CORRUPT;
        }
        if (pad16((r.at - b0 * 8 + 7) / 8) != b1 - b0)
            return EO_CORRUPT;
        while (r.at < r.limit) {
            int v;
            read_bit(&r, &v);
            if (v)
                return EO_CORRUPT;
        }
    }
    return EO_OK;
}
