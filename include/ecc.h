/*
 * ecc.h -- C ABI of the GB300 library for lossless fixed-codebook coding of
 * e4m3 byte tensors.
 *
 * Three codebook families, all fixed before the data is seen:
 *
 *  - the Quad Length Code (QLC) of "Quad Length Codes for Lossless
 *    Compression of e4m3" (gist.science summary of arXiv 2602.17849),
 *    section 2 "Metodologia": the 256 byte values are ranked by decreasing
 *    probability, the ranks are split into 8 areas named by a 3-bit prefix,
 *    every area has one fixed suffix width, so there are at most 4 distinct
 *    code lengths and the decoder learns the length from the first 3 bits;
 *  - the single-stage canonical Huffman code of "Single-Stage Huffman
 *    Encoder for ML Compression" (arXiv 2601.10673), abstract and TL;DR: one
 *    codebook built from the average symbol distribution of earlier batches
 *    and reused for every later tensor, with no per-tensor frequency
 *    analysis and no codebook sent with the data;
 *  - the exponent escape code of ZipCCL (gist.science summary of arXiv
 *    2604.27844), section 2.B, on the e4m3 exponent field (see
 *    escape_build_tables).
 *
 * Conventions (all entry points):
 *  - Every function returns an ecc_status.  A host-side return value reports
 *    argument and launch errors only; errors that depend on the data are
 *    written by the kernels to a caller-provided device word `status`, which
 *    the call first sets to ECC_OK.  Read it after the stream has reached the
 *    end of the call.  The first error written wins.
 *  - Device buffers are plain device pointers owned by the caller.  Buffers
 *    that hold bytes (tensor, payload) and the device codebook must start on
 *    a 16-byte boundary.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Device calls only enqueue work: they never synchronise and,
 *    apart from the batched calls' one host-to-device copy of their
 *    descriptors, never copy between host and device.  The library allocates
 *    no device memory; scratch space is the caller's workspace.
 *  - Calls keep no state between invocations and may be made from several
 *    host threads; calls on one stream run in order.
 *
 * Container format written by ecc_encode and read by ecc_decode (the pages
 * fix no format; this one is the library's own):
 *  - the n input bytes are split into chunks of C symbols (C a power of two,
 *    1024 <= C <= 65536), chunk c holding symbols [cC, min(n, (c+1)C));
 *  - a chunk's payload is its codewords in symbol order, each written most
 *    significant bit first, packed most significant bit first into bytes and
 *    zero-padded to a multiple of 16 bytes; payloads follow each other;
 *  - chunk_off has n_chunks + 1 entries: chunk_off[0] = 0 and
 *    chunk_off[c + 1] = chunk_off[c] + padded payload bytes of chunk c;
 *  - sub_bits has ceil(n / S) entries: the exact payload bits of the
 *    symbols [jS, min(n, (j+1)S)) (S a power of two, 64 <= S <= 1024,
 *    S <= C), which lets a decoder start in the middle of a chunk;
 *  - total_bits is the sum of all code lengths, i.e. sum over bytes of
 *    count x length.
 */
#ifndef ECC_H
#define ECC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ecc_status;

enum {
    ECC_OK = 0,
    ECC_ERR_ARG = 1,      /* bad size, alignment, null pointer or workspace */
    ECC_ERR_CAPACITY = 2, /* the payload does not fit in out_cap bytes */
    ECC_ERR_CORRUPT = 3,  /* stream, offsets or sub-block bits inconsistent */
    ECC_ERR_CODEBOOK = 4, /* bad codebook, or a byte the codebook does not code */
    ECC_ERR_TIMEOUT = 5,  /* a bounded device wait ran out (the kernel returned) */
    ECC_ERR_CUDA = 6,     /* a CUDA runtime call failed */
    ECC_ERR_CHECK = 7     /* an internal check failed: in index-checked builds (-DECC_CHECKED) a
                             kernel index was out of range and the access skipped; in any build,
                             chunks of more than 16384 symbols coded to other sizes than their
                             length pass counted, or a batched encode's second pass (chunks
                             with long codes) sizing a chunk otherwise than its first pass
                             placed it (nothing is written for such a chunk) */
};

enum { ECC_FAMILY_QLC = 1, ECC_FAMILY_HUFFMAN = 2, ECC_FAMILY_ESCAPE = 3 };

#define ECC_CODEBOOK_MAGIC 0x45434342u /* "ECCB" */
#define ECC_MAX_CODE_LEN 48            /* longest code the device path accepts */
#define ECC_PEEK_BITS 14               /* first-level decode table index width */

/*
 * Codebook: a fixed-size, pointer-free record built on the host by
 * qlc_build_tables, huff_build_canonical or escape_build_tables (or on the
 * device by huff_build_device) and copied as raw bytes to the
 * device (cudaMemcpy of ecc_codebook_bytes()).  Serialising it is a memcpy.
 * Fields marked "derived" are lookup tables the kernels stage in shared
 * memory; they follow from len/code and are filled by the builders.
 */
typedef struct ecc_codebook {
    uint32_t magic;       /* ECC_CODEBOOK_MAGIC */
    uint32_t family;      /* ECC_FAMILY_QLC, ECC_FAMILY_HUFFMAN or ECC_FAMILY_ESCAPE */
    uint32_t max_len;     /* longest code length in bits */
    uint32_t min_len;     /* shortest code length in bits */
    uint32_t n_coded;     /* number of byte values that have a code */
    uint32_t prefix_bits; /* QLC: prefix bits p, 2^p areas (the page's code: 3); 0 for other families */
    uint32_t reserved[2];
    uint64_t code[256];   /* code of each byte value, right-aligned */
    uint64_t first[64];   /* Huffman: first canonical code of each length */
    uint32_t enc_code[256]; /* derived: code << (32 - len) (first bit in bit 31) if 1 <= len <= 31, else 0 */
    uint32_t enc_mul[256];  /* derived: 2^(32 - len) if 1 <= len <= 31, else 0 (the exact path codes it) */
    uint32_t area[8];     /* derived, QLC: per prefix k, start | len << 16 | width << 24 */
    uint16_t dec[16384];  /* derived: 14-bit peek -> byte | len << 8; 0 = not resolved */
    uint16_t count[64];   /* Huffman: number of codes of each length */
    uint16_t index[64];   /* Huffman: position in sorted[] of the first code of each length */
    uint16_t area_start[8]; /* QLC: first rank of each area */
    uint16_t area_size[8];  /* QLC: ranks held by each area (0 = empty) */
    uint8_t width[8];     /* QLC: suffix width of each area, 0..8 */
    uint8_t len[256];     /* code length of each byte value, 0 = no code */
    uint8_t rank[256];    /* QLC: rank of each byte value */
    uint8_t by_rank[256]; /* QLC: byte value holding each rank; escape code: the 7 exponents by rank */
    uint8_t sorted[256];  /* Huffman: coded byte values sorted by (length, value) */
} ecc_codebook;

/* Size in bytes of ecc_codebook (what to copy to the device). */
size_t ecc_codebook_bytes(void);

/* ------------------------------------------------------------------------
 * Host codebook builders (pure CPU, no CUDA calls)
 * ---------------------------------------------------------------------- */

/*
 * qlc_build_tables -- Quad Length Code tables ("Quad Length Codes ...",
 * section 2: LUT paragraph and area bullets; "Adattabilita" for other widths).
 *   count[256]  occurrences of each byte value (any scale; only the order
 *               matters).  Ranks sort by count descending, ties by byte value
 *               ascending; every byte gets a rank.
 *   width[8]    suffix width of each area, 0..8; areas are filled with ranks
 *               in order, area k taking min(2^width[k], ranks left).  The base
 *               code is {3,3,3,3,3,4,5,8}: areas of 8,8,8,8,8,16,32,168 ranks
 *               and lengths 6,6,6,6,6,7,8,11.  Rank r in area k gets the code
 *               (k << width[k]) | (r - start_k), length 3 + width[k].
 *   out         filled codebook (caller-owned host memory).
 * Errors: ECC_ERR_ARG if a pointer is NULL, a width exceeds 8, or the areas
 * hold fewer than 256 ranks.
 */
ecc_status qlc_build_tables(const uint64_t count[256], const uint8_t width[8], ecc_codebook *out);

/*
 * qlc_search_widths -- adapted QLC ("Quad Length Codes ...", section 2
 * "Adattabilita", section 3 case 2 and section 5 "Future Directions"):
 * exhaustive search over non-decreasing width vectors (0..8 each) whose
 * areas hold at least 256 ranks (require_full != 0: exactly 256), whose
 * non-empty areas use at most max_distinct distinct lengths, minimising
 * sum(count x length); ties go to the lexicographically smallest vector.
 *   width_out[8]  best widths; cost_bits (may be NULL) its sum(count x len).
 * Errors: ECC_ERR_ARG for NULL inputs, max_distinct == 0, or no vector.
 */
ecc_status qlc_search_widths(const uint64_t count[256], uint32_t max_distinct, uint32_t require_full,
                             uint8_t width_out[8], uint64_t *cost_bits);

/*
 * gqlc_build_tables, gqlc_search_widths -- QLC with p = 1, 2 or 3 prefix
 * bits, i.e. 2, 4 or 8 areas ("Quad Length Codes ...", section 5 "Future
 * Directions": optimise the number of areas and the code lengths).  As
 * qlc_build_tables / qlc_search_widths (which are the p = 3 case) with
 * lengths p + width[k] over the first 2^p entries of width (the rest are
 * ignored on input, 0 on output).  The decoder's QLC fast path serves
 * p = 3; other codebooks decode through the first-level table.
 * Errors: as for the p = 3 calls, and ECC_ERR_ARG for p outside 1..3.
 */
ecc_status gqlc_build_tables(const uint64_t count[256], uint32_t prefix_bits, const uint8_t width[8],
                             ecc_codebook *out);
ecc_status gqlc_search_widths(const uint64_t count[256], uint32_t prefix_bits, uint32_t max_distinct,
                              uint32_t require_full, uint8_t width_out[8], uint64_t *cost_bits);

/*
 * huff_build_canonical -- the fixed Huffman codebook of the single-stage
 * encoder ("Single-Stage Huffman Encoder ...", abstract: codebook built once
 * from the average probability distribution of earlier batches; euno.news
 * summary, Methodology step 3).
 *   weight[256]  integer PMF numerators, e.g. pooled warm-up counts plus one
 *                per byte; weight 0 = byte absent (gets no code).  The two
 *                nodes with the smallest (weight, smallest byte below) keys
 *                merge first, so equal weights resolve deterministically.  A
 *                lone coded byte gets length 1.  Codes are canonical: sorted
 *                by (length, byte value), consecutive within a length.
 *   max_len      longest code accepted, 1..ECC_MAX_CODE_LEN; a longer tree
 *                is an error, not a silent length limit.
 *   out          filled codebook (caller-owned host memory).
 * Errors: ECC_ERR_ARG (NULL, max_len out of range, all weights 0, weights
 * whose sum overflows 64 bits), ECC_ERR_CODEBOOK (tree deeper than max_len).
 */
ecc_status huff_build_canonical(const uint64_t weight[256], uint32_t max_len, ecc_codebook *out);

/*
 * huff_build_limited -- canonical Huffman code with no length above max_len
 * (the decode tables stay bounded: "Quad Length Codes ...", section 5
 * "Future Directions", asks for code lengths optimised under the decoder's
 * constraints), from the package-merge algorithm of Larmore and Hirschberg
 * (J. ACM 37(3), 1990): optimal among codes within the limit.  Leaves sort
 * by (weight, byte value); a package and a leaf of equal weight: the leaf
 * first.  With max_len at least the unlimited tree's depth the cost equals
 * huff_build_canonical's (the lengths may differ on ties).
 *   weight[256], out  as for huff_build_canonical (family ECC_FAMILY_HUFFMAN);
 *   max_len   1..ECC_MAX_CODE_LEN.
 * Errors: ECC_ERR_ARG (NULL, max_len out of range, all weights 0, a weight
 * sum of 2^62 or more), ECC_ERR_CODEBOOK (more coded bytes than 2^max_len).
 */
ecc_status huff_build_limited(const uint64_t weight[256], uint32_t max_len, ecc_codebook *out);

/*
 * escape_build_tables -- the exponent escape code of ZipCCL (gist.science
 * summary of arXiv 2604.27844, section 2.B "Tecnica di Codifica degli
 * Esponenti") as a fixed codebook for e4m3 bytes (sign bit 7, exponent bits
 * 6-3, mantissa bits 2-0): the 7 exponents with the largest summed counts
 * (ties to the smaller exponent) get the 3-bit codes 001..111 by rank; any
 * other exponent is coded 000 followed by its 4 bits (the page keeps such
 * exponents in a separate array; here they stay in the stream).  Sign and
 * mantissa follow as they are, so every byte has a 7- or 11-bit code.
 *   count[256]  byte counts (e.g. pooled warm-up histograms).
 *   out         filled codebook (family ECC_FAMILY_ESCAPE); by_rank[0..6]
 *               holds the 7 exponents in rank order.
 * Errors: ECC_ERR_ARG for NULL pointers.
 */
ecc_status escape_build_tables(const uint64_t count[256], ecc_codebook *out);

/* ------------------------------------------------------------------------
 * Host figures in float64 ("Single-Stage Huffman ...", TL;DR: compressibility
 * against per-shard Huffman and the Shannon bound; Figure 3: KL divergence
 * of shard distributions from the average one)
 * ---------------------------------------------------------------------- */

/* Shannon entropy -sum p log2 p (bits/symbol) of a count vector. */
double ecc_entropy_bits(const uint64_t count[256]);

/* D(P || Q) in bits of two count vectors; +inf if Q lacks a byte P has. */
double ecc_kl_bits(const uint64_t p_count[256], const uint64_t q_count[256]);

/* Exact payload bits sum(count x len) of a codebook on a histogram.
 * Errors: ECC_ERR_CODEBOOK if a counted byte has no code, ECC_ERR_ARG. */
ecc_status ecc_code_bits(const uint64_t count[256], const ecc_codebook *cb, uint64_t *bits);

/* ------------------------------------------------------------------------
 * Sizes
 * ---------------------------------------------------------------------- */
size_t ecc_num_chunks(size_t n, uint32_t C);     /* ceil(n / C) */
size_t ecc_num_subblocks(size_t n, uint32_t S);  /* ceil(n / S) */
/* Payload bytes that always suffice: every symbol at max_len bits, every
 * chunk padded to 16 bytes. */
size_t ecc_max_encoded_bytes(size_t n, uint32_t C, uint32_t max_len);
/* Device workspace ecc_encode needs for n symbols in chunks of C: 256 bytes,
 * 8 a chunk and, when C > 16384, 8 per 16384 symbols. */
size_t ecc_encode_workspace_bytes(size_t n, uint32_t C);

/* ------------------------------------------------------------------------
 * Device calls
 * ---------------------------------------------------------------------- */

/*
 * e4m3_histogram -- count of each byte value ("Single-Stage Huffman ...",
 * euno.news summary, Methodology step 1: record symbol frequencies of
 * warm-up batches; also the rank input of qlc_build_tables).
 *   in     device bytes [n] (any alignment);
 *   count  device uint64[256]; the counts of `in` are ADDED to it, so
 *          several tensors can be pooled (zero it first for one tensor).
 * Errors (host): ECC_ERR_ARG for NULL pointers with n > 0, ECC_ERR_CUDA.
 */
ecc_status e4m3_histogram(const uint8_t *in, size_t n, uint64_t *count, void *stream);

/*
 * huff_build_device -- the canonical Huffman codebook built on the device,
 * stream-ordered after e4m3_histogram, so that frequency analysis, codebook
 * construction and encoding (the three stages a per-tensor Huffman pipeline
 * runs, "Single-Stage Huffman Encoder for ML Compression", introduction)
 * need no host round trip; also a codebook refresh from fresh counts when
 * the data drift (same page, discussion).  One CTA, a few tens of
 * microseconds.
 *   count    device uint64[256] (e.g. the histogram); read only.
 *   add      pseudocount added to every count: the weights are
 *            count[b] + add, with the meaning huff_build_canonical gives
 *            them; the output is byte-identical to that builder's.
 *   max_len  1..ECC_MAX_CODE_LEN, as for huff_build_canonical.
 *   out      device ecc_codebook, 16-byte aligned; always rewritten.  On a
 *            device error it is left all zero (no magic word), so every call
 *            that is handed it reports ECC_ERR_CODEBOOK.
 *   status   device uint32[1]; ECC_OK, or ECC_ERR_ARG (a weight or the
 *            weight sum does not fit 64 bits, all weights 0) or
 *            ECC_ERR_CODEBOOK (tree deeper than max_len).
 * Host errors: ECC_ERR_ARG (NULL, misaligned out, max_len out of range),
 * ECC_ERR_CUDA.  Calls that read `out` must be ordered after this one.
 */
ecc_status huff_build_device(const uint64_t *count, uint64_t add, uint32_t max_len, ecc_codebook *out,
                             uint32_t *status, void *stream);

/*
 * ecc_encode -- single-stage encode with a fixed codebook ("Quad Length
 * Codes ...", section 2 "Codifica": the encoder looks the code up in the
 * LUT; "Single-Stage Huffman ...", Methodology step 4: encode with the
 * precomputed codebook, no analysis, no codebook transmission).
 *   in, n        device bytes [n], 16-byte aligned.
 *   cb           device copy of an ecc_codebook (max_len <= 48).
 *   C, S         chunk and sub-block sizes (see the container format).
 *   out, out_cap device payload buffer, 16-byte aligned, out_cap bytes;
 *                ecc_max_encoded_bytes() always suffices.
 *   chunk_off    device uint64[ceil(n/C) + 1]; written.
 *   sub_bits     device uint16[ceil(n/S)]; written.
 *   total_bits   device uint64[1]; written (sum of all code lengths).
 *   ws, ws_bytes device workspace of at least ecc_encode_workspace_bytes();
 *                its contents need not be initialised and are clobbered.
 *   status       device uint32[1]; set to ECC_OK, then to the first error.
 * Device errors: ECC_ERR_CODEBOOK (bad magic or a byte without a code),
 * ECC_ERR_CAPACITY (payload exceeds out_cap; chunk_off still holds the sizes
 * the payload needs, nothing is written past out_cap), ECC_ERR_TIMEOUT (the
 * chunk-offset look-back waited more than about a second).
 * Host errors: ECC_ERR_ARG (sizes, alignment, NULL, small workspace),
 * ECC_ERR_CUDA.  n = 0 writes chunk_off[0] = 0 and total_bits = 0.
 * Launches (all on `stream`, after a prologue that clears the workspace):
 * one kernel codes and places the symbols in units of 16384 (a chunk,
 * whole smaller chunks, or part of a larger chunk; decoupled look-back over
 * units, or over chunks when a chunk spans units), followed by a deferred
 * pass that codes the units (or chunks) whose codes were too long to stage
 * (it only reads the look-back words when there are none).  On a device
 * where that kernel cannot run, larger chunks take a length pass, a scan of
 * the offsets and a coding kernel (ECC_ERR_CHECK if the two ever disagree).
 */
ecc_status ecc_encode(const uint8_t *in, size_t n, const ecc_codebook *cb, uint32_t C, uint32_t S,
                      uint8_t *out, size_t out_cap, uint64_t *chunk_off, uint16_t *sub_bits,
                      uint64_t *total_bits, void *ws, size_t ws_bytes, uint32_t *status, void *stream);

/*
 * ecc_decode -- chunk-parallel decode ("Quad Length Codes ...", section 2
 * "Decodifica": read 3 bits -> area -> length, read the suffix, add the
 * area's offset, a second LUT gives the byte; section 4 items 2-3; Huffman
 * codes resolve through a 14-bit first-level table, then a second-level
 * table over the few 14-bit prefixes longer codes start with, then the
 * canonical per-length ranges).
 *   in, in_bytes device payload [in_bytes], 16-byte aligned.
 *   chunk_off    device uint64[ceil(n/C) + 1] and sub_bits device
 *                uint16[ceil(n/S)] as written by ecc_encode.
 *   n, C, S      symbol count and the sizes used at encode time.
 *   cb           device codebook used at encode time.
 *   out          device bytes [n], 16-byte aligned; written.
 *   status       device uint32[1]; set to ECC_OK, then to the first error.
 * Device errors: ECC_ERR_CORRUPT (offsets out of range, a code the codebook
 * lacks, a sub-block whose bit count differs from sub_bits, a chunk whose
 * padded size differs from its offsets); output bytes of a corrupt chunk are
 * unspecified but nothing is written outside out[0, n).  ECC_ERR_CODEBOOK.
 */
ecc_status ecc_decode(const uint8_t *in, size_t in_bytes, const uint64_t *chunk_off,
                      const uint16_t *sub_bits, size_t n, uint32_t C, uint32_t S,
                      const ecc_codebook *cb, uint8_t *out, uint32_t *status, void *stream);

/* ------------------------------------------------------------------------
 * The exponent escape code on BF16 tensors (ZipCCL, gist.science summary of
 * arXiv 2604.27844, section 2.B "Tecnica di Codifica degli Esponenti"; the
 * exponent table of section 2.A).  Values are BF16 bit patterns (uint16:
 * sign bit 15, exponent bits 14-7, mantissa bits 6-0).  A value whose
 * exponent is one of the 7 of the table is written as the 3-bit code r + 1
 * (its rank r in the table), any other as 000 followed by its 8-bit
 * exponent; the sign bit and the 7 mantissa bits follow as they are: 11 or 19
 * bits a value, most significant bit first (the page keeps escaped exponents
 * in a separate array; here they stay in the stream).  The container is the
 * byte container above with BF16 values as the symbols: chunks of C values
 * (1024 <= C <= 16384), sub_bits per S values, chunk payloads padded to 16
 * bytes.
 * ---------------------------------------------------------------------- */

/*
 * bf16_escape_table_sigma -- the table from the layer's standard deviation
 * alone (section 2.A: no statistics of the data): the 7 exponent fields of
 * largest probability under N(0, sigma^2) rounded to BF16 (round to nearest
 * even: a field's magnitude range [2^(e-127), 2^(e-126)) has its edges at the
 * rounding midpoints 2^k (1 - 2^-9)), in decreasing probability, ties to the
 * smaller field.
 *   sigma  > 0, finite.   top7  host uint8[7], written.
 * Errors: ECC_ERR_ARG.
 */
ecc_status bf16_escape_table_sigma(double sigma, uint8_t top7[7]);

/*
 * bf16_escape_table_counts -- the table from exponent counts (section 2.A:
 * the 7 most frequent exponents): count descending, ties to the smaller
 * field.   count  host uint64[256] (e.g. from bf16_exponent_histogram).
 * Errors: ECC_ERR_ARG.
 */
ecc_status bf16_escape_table_counts(const uint64_t count[256], uint8_t top7[7]);

/*
 * bf16_exponent_histogram -- count of each exponent field, ADDED to count.
 *   in  device uint16[n], 16-byte aligned;  count  device uint64[256].
 * Errors: ECC_ERR_ARG (NULL, misaligned), ECC_ERR_CUDA.
 */
ecc_status bf16_exponent_histogram(const uint16_t *in, size_t n, uint64_t *count, void *stream);

/* Payload bytes that always suffice for n values in chunks of C: 19 bits a
 * value, each chunk padded to 16 bytes. */
size_t bf16_escape_max_encoded_bytes(size_t n, uint32_t C);

/*
 * bf16_escape_encode -- code n BF16 values with the table top7 (host array
 * of 7 distinct exponent fields, rank order).  Arguments, outputs, workspace
 * (ecc_encode_workspace_bytes(n, C)) and device errors as for ecc_encode;
 * out_cap: bf16_escape_max_encoded_bytes() always suffices.
 * Host errors: ECC_ERR_ARG (sizes, C above 16384, alignment, NULL, a table
 * exponent listed twice, small workspace), ECC_ERR_CUDA.
 */
ecc_status bf16_escape_encode(const uint16_t *in, size_t n, const uint8_t top7[7], uint32_t C, uint32_t S,
                              uint8_t *out, size_t out_cap, uint64_t *chunk_off, uint16_t *sub_bits,
                              uint64_t *total_bits, void *ws, size_t ws_bytes, uint32_t *status, void *stream);

/*
 * bf16_escape_decode -- the inverse: out (device uint16[n], 16-byte
 * aligned) from the container written with the same table, C and S; in
 * (the payload) 16-byte aligned.  Device errors:
 * ECC_ERR_CORRUPT (offsets, a sub-block whose bit count differs from
 * sub_bits, 000 followed by a table exponent, a chunk whose padded size or
 * zero padding is wrong); nothing is read outside each chunk's payload.
 * Host errors as for ecc_decode.
 */
ecc_status bf16_escape_decode(const uint8_t *in, size_t in_bytes, const uint64_t *chunk_off,
                              const uint16_t *sub_bits, size_t n, uint32_t C, uint32_t S, const uint8_t top7[7],
                              uint16_t *out, uint32_t *status, void *stream);

/* ------------------------------------------------------------------------
 * Batched calls: many tensors, one call for encode and one for decode (each
 * tensor an independent container, each with its own codebook)
 * ---------------------------------------------------------------------- */
typedef struct ecc_desc {
    const uint8_t *in;     /* encode: symbols [n]; decode: payload [in_bytes] */
    uint8_t *out;          /* encode: payload [out_cap]; decode: symbols [n] */
    uint64_t n;            /* symbols */
    uint64_t cap;          /* encode: out_cap; decode: in_bytes */
    uint64_t *chunk_off;   /* [ceil(n/C) + 1] */
    uint16_t *sub_bits;    /* [ceil(n/S)] */
    uint64_t *total_bits;  /* encode: [1], written; decode: ignored (may be NULL) */
    const ecc_codebook *cb;/* device codebook */
    uint32_t *status;      /* device word, set to ECC_OK then the first error */
    uint64_t *t_done_ns;   /* optional device word: %globaltimer (ns) when the
                              tensor's last chunk finished; NULL = not recorded */
    uint32_t C, S;         /* container sizes of this tensor */
} ecc_desc;

/* Workspace the batched calls need for these descriptors (host array). */
size_t ecc_batched_workspace_bytes(const ecc_desc *descs, uint32_t count);

/*
 * ecc_encode_batched / ecc_decode_batched -- the calls above over `count`
 * tensors in one coding launch over all of them (after a prologue; the
 * encode adds a second launch for the chunks whose codes were too long to
 * stage -- when every tensor has 16 KiB chunks, the unit encoder again with
 * larger stages, else a deferred pass of a warp a chunk -- and a tensor's
 * t_done_ns is stamped by whichever launch finishes its last chunk).  `descs` is a host array; the call copies it and a
 * chunk prefix table into `ws` with one asynchronous host-to-device copy,
 * so `descs` may be reused once the call returns.  Every tensor obeys the
 * rules of ecc_encode / ecc_decode; its errors go to its own status word.
 * Optionally `t_start_ns` (device word, may be NULL) receives %globaltimer
 * at the coding kernel's start, for per-tensor latency = t_done_ns -
 * t_start_ns.
 * Host errors: ECC_ERR_ARG (bad descriptor, small workspace), ECC_ERR_CUDA.
 */
ecc_status ecc_encode_batched(const ecc_desc *descs, uint32_t count, void *ws, size_t ws_bytes,
                              uint64_t *t_start_ns, void *stream);
ecc_status ecc_decode_batched(const ecc_desc *descs, uint32_t count, void *ws, size_t ws_bytes,
                              uint64_t *t_start_ns, void *stream);

/*
 * ecc_selftest_wait -- failure-detection self-test of the bounded wait used
 * by the encoder's chunk-offset look-back.  Runs the look-back of chunk
 * `chunk` on the caller's device array flags[chunk + 1] (uint64, zero = not
 * published) with a time limit of timeout_ns; writes the exclusive prefix it
 * found to *prefix and ECC_ERR_TIMEOUT to *status if the limit ran out.  A
 * flags array in which no predecessor is ever published must return
 * ECC_ERR_TIMEOUT, not hang.  Host errors: ECC_ERR_ARG, ECC_ERR_CUDA.
 */
ecc_status ecc_selftest_wait(uint64_t *flags, uint64_t chunk, uint64_t aggregate, uint64_t timeout_ns,
                             uint64_t *prefix, uint32_t *status, void *stream);

/*
 * ecc_encode_static -- ecc_encode without a workspace argument, for callers
 * that cannot allocate device memory on their call path: latency-critical
 * communication code (cudaMalloc can synchronise the whole device) and code
 * embedded in a framework whose allocator owns all device memory.  The pages
 * have no counterpart; this is a property of the library, not of the method.
 *   Arguments, outputs and errors are those of ecc_encode.  The scratch
 *   space (a ticket, one 64-bit look-back word per chunk and, for chunks of
 *   more than 16384 symbols, one per 16384 symbols) is a file-scope device
 *   array of 5 x ECC_STATIC_MAX_CHUNKS + 32 words (about 2.5 MiB) that
 *   every GPU loading the library holds until the process exits; the call
 *   allocates and frees nothing.  Inputs with more than ECC_STATIC_MAX_CHUNKS
 *   chunks (n > 65536 * C) are rejected with ECC_ERR_ARG.
 *   Every call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress, with that device current), so a context reset
 *   that reloads the library's module does not leave a stale address; the
 *   first call on a device may load the module, so make it before any stream
 *   capture.  Every call clears the scratch words it uses
 *   before use, but all calls share the one array: calls that can overlap on
 *   the GPU (other streams, other host threads) race and must be ordered by
 *   the caller.
 */
#define ECC_STATIC_MAX_CHUNKS 65536u
ecc_status ecc_encode_static(const uint8_t *in, size_t n, const ecc_codebook *cb, uint32_t C, uint32_t S,
                             uint8_t *out, size_t out_cap, uint64_t *chunk_off, uint16_t *sub_bits,
                             uint64_t *total_bits, uint32_t *status, void *stream);

/* Human-readable name of a status code (static string). */
const char *ecc_status_string(ecc_status s);

#ifdef __cplusplus
}
#endif

#endif /* ECC_H */
