// ecc_host.cpp -- host-side codebook builders, figures and size helpers of
// the e4m3 entropy-coding library (see include/ecc.h for the contract).
//
// Codebooks are built once, off the critical path ("Single-Stage Huffman
// Encoder for ML Compression", TL;DR: precomputed off the critical path and
// shared), so this is plain C++ on the CPU.  Besides the codes themselves it
// fills the lookup tables the kernels stage in shared memory.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <queue>
#include <vector>

#include "../../include/ecc.h"

static_assert(sizeof(ecc_codebook) % 16 == 0 || sizeof(ecc_codebook) % 8 == 0, "codebook padding");

namespace {

constexpr int kPeek = ECC_PEEK_BITS;

void clear(ecc_codebook *cb, uint32_t family)
{
    std::memset(cb, 0, sizeof(*cb));
    cb->magic = ECC_CODEBOOK_MAGIC;
    cb->family = family;
}

// Fill the derived tables from len[]/code[]: the encode entries (the code
// with its first bit in bit 31, and the multiplier 2^(32 - len) that shifts
// a following code behind it) and the 14-bit first-level decode table
// (byte | len << 8 for codes of at most 14 bits; entries under a longer
// code's prefix and unused entries stay 0).
void fill_derived(ecc_codebook *cb)
{
    uint32_t mx = 0, mn = 255, nc = 0;
    for (int b = 0; b < 256; ++b) {
        uint32_t L = cb->len[b];
        cb->enc_code[b] = 0;
        cb->enc_mul[b] = 0;
        if (!L)
            continue;
        ++nc;
        mx = std::max(mx, L);
        mn = std::min(mn, L);
        if (L <= 31) {
            cb->enc_code[b] = (uint32_t)(cb->code[b] << (32 - L));
            cb->enc_mul[b] = 1u << (32 - L);
        }
        if (L <= (uint32_t)kPeek) {
            uint32_t lo = (uint32_t)cb->code[b] << (kPeek - L);
            uint32_t hi = lo + (1u << (kPeek - L));
            for (uint32_t i = lo; i < hi; ++i)
                cb->dec[i] = (uint16_t)(b | (L << 8));
        }
    }
    cb->max_len = mx;
    cb->min_len = nc ? mn : 0;
    cb->n_coded = nc;
}

bool valid_widths(const uint8_t *width, int areas)
{
    for (int k = 0; k < areas; ++k)
        if (width[k] > 8)
            return false;
    return true;
}

// Ranks held by the first `areas` areas filled in order, capped at 256.
int layout(const uint8_t *width, int areas, int start[8], int size[8])
{
    int used = 0;
    for (int k = 0; k < areas; ++k) {
        int room = 256 - used;
        int n = std::min(1 << width[k], room);
        start[k] = used;
        size[k] = n;
        used += n;
    }
    return used;
}

// Byte values ordered by count descending; stable sort keeps equal counts
// in ascending byte order.
void order_by_count(const uint64_t *count, uint8_t by_rank[256])
{
    int idx[256];
    for (int b = 0; b < 256; ++b)
        idx[b] = b;
    std::stable_sort(idx, idx + 256, [count](int a, int b) { return count[a] > count[b]; });
    for (int r = 0; r < 256; ++r)
        by_rank[r] = (uint8_t)idx[r];
}

// Canonical Huffman codebook from code lengths (RFC 1951 section 3.2.2):
// codes of one length are consecutive in byte order, the first code of each
// length follows the last of the shorter ones, shifted.
void canonical_fill(const uint8_t len[256], ecc_codebook *out)
{
    clear(out, ECC_FAMILY_HUFFMAN);
    uint32_t bl_count[65] = {0};
    for (int b = 0; b < 256; ++b)
        if (len[b])
            ++bl_count[len[b]];
    // first code of each length: first[1] = 0, first[L] = (first[L-1] + count[L-1]) << 1
    uint64_t next[65] = {0};
    for (int L = 2; L <= 64; ++L)
        next[L] = (next[L - 1] + bl_count[L - 1]) << 1;
    int pos = 0;
    for (int L = 1; L <= (int)ECC_MAX_CODE_LEN; ++L) {
        out->index[L] = (uint16_t)pos;
        out->count[L] = (uint16_t)bl_count[L];
        out->first[L] = next[L];
        for (int b = 0; b < 256; ++b)
            if (len[b] == L)
                out->sorted[pos++] = (uint8_t)b;
    }
    for (int b = 0; b < 256; ++b) {
        if (!len[b])
            continue;
        out->len[b] = len[b];
        out->code[b] = next[len[b]]++;
    }
    fill_derived(out);
}

} // namespace

extern "C" {

size_t ecc_codebook_bytes(void) { return sizeof(ecc_codebook); }

ecc_status gqlc_build_tables(const uint64_t count[256], uint32_t prefix_bits, const uint8_t width[8],
                             ecc_codebook *out)
{
    if (!count || !width || !out || prefix_bits < 1 || prefix_bits > 3)
        return ECC_ERR_ARG;
    const int areas = 1 << prefix_bits;
    if (!valid_widths(width, areas))
        return ECC_ERR_ARG;
    int start[8], size[8];
    if (layout(width, areas, start, size) < 256)
        return ECC_ERR_ARG;
    clear(out, ECC_FAMILY_QLC);
    out->prefix_bits = prefix_bits;
    order_by_count(count, out->by_rank);
    for (int k = 0; k < areas; ++k) {
        out->width[k] = width[k];
        out->area_start[k] = (uint16_t)start[k];
        out->area_size[k] = (uint16_t)size[k];
        uint32_t L = prefix_bits + width[k];
        out->area[k] = (uint32_t)start[k] | (L << 16) | ((uint32_t)width[k] << 24);
        for (int v = 0; v < size[k]; ++v) {
            int r = start[k] + v;
            uint8_t b = out->by_rank[r];
            out->rank[b] = (uint8_t)r;
            out->len[b] = (uint8_t)L;
            out->code[b] = ((uint64_t)k << width[k]) + (uint64_t)v;
        }
    }
    fill_derived(out);
    return ECC_OK;
}

ecc_status qlc_build_tables(const uint64_t count[256], const uint8_t width[8], ecc_codebook *out)
{
    return gqlc_build_tables(count, 3, width, out);
}

namespace {

struct Search {
    uint64_t sorted[257]; // prefix sums of counts in rank order
    uint32_t p;           // prefix bits: 2^p areas
    uint32_t max_distinct;
    bool full;
    bool found = false;
    uint64_t best = 0;
    uint8_t best_w[8];
    uint8_t w[8];

    // cost of the current w, or false if it does not qualify
    bool evaluate(uint64_t &cost) const
    {
        const int areas = 1 << p;
        uint32_t cap = 0;
        for (int k = 0; k < areas; ++k)
            cap += 1u << w[k];
        if (full ? cap != 256 : cap < 256)
            return false;
        uint32_t lengths_used = 0; // bit L set if some non-empty area uses length L
        uint64_t c = 0;
        int at = 0;
        for (int k = 0; k < areas && at < 256; ++k) {
            int take = std::min(1 << w[k], 256 - at);
            uint32_t L = p + w[k];
            lengths_used |= 1u << L;
            c += (sorted[at + take] - sorted[at]) * L;
            at += take;
        }
        if ((uint32_t)__builtin_popcount(lengths_used) > max_distinct)
            return false;
        cost = c;
        return true;
    }

    // widths non-decreasing, generated in lexicographic order
    void walk(int k, int lo)
    {
        if (k == (1 << p)) {
            uint64_t c;
            if (evaluate(c) && (!found || c < best)) {
                found = true;
                best = c;
                std::memcpy(best_w, w, 8);
            }
            return;
        }
        for (int v = lo; v <= 8; ++v) {
            w[k] = (uint8_t)v;
            walk(k + 1, v);
        }
    }
};

} // namespace

ecc_status gqlc_search_widths(const uint64_t count[256], uint32_t prefix_bits, uint32_t max_distinct,
                              uint32_t require_full, uint8_t width_out[8], uint64_t *cost_bits)
{
    if (!count || !width_out || max_distinct == 0 || prefix_bits < 1 || prefix_bits > 3)
        return ECC_ERR_ARG;
    Search s;
    uint8_t by_rank[256];
    order_by_count(count, by_rank);
    s.sorted[0] = 0;
    for (int r = 0; r < 256; ++r)
        s.sorted[r + 1] = s.sorted[r] + count[by_rank[r]];
    s.p = prefix_bits;
    s.max_distinct = max_distinct;
    s.full = require_full != 0;
    std::memset(s.w, 0, 8);
    s.walk(0, 0);
    if (!s.found)
        return ECC_ERR_ARG;
    std::memcpy(width_out, s.best_w, 8);
    if (cost_bits)
        *cost_bits = s.best;
    return ECC_OK;
}

ecc_status qlc_search_widths(const uint64_t count[256], uint32_t max_distinct, uint32_t require_full,
                             uint8_t width_out[8], uint64_t *cost_bits)
{
    return gqlc_search_widths(count, 3, max_distinct, require_full, width_out, cost_bits);
}

ecc_status huff_build_canonical(const uint64_t weight[256], uint32_t max_len, ecc_codebook *out)
{
    if (!weight || !out || max_len < 1 || max_len > ECC_MAX_CODE_LEN)
        return ECC_ERR_ARG;
    uint64_t total = 0;
    for (int b = 0; b < 256; ++b) {
        if (weight[b] > std::numeric_limits<uint64_t>::max() - total)
            return ECC_ERR_ARG;
        total += weight[b];
    }
    if (total == 0)
        return ECC_ERR_ARG;

    // Binary min-heap of (weight, smallest byte in the subtree, node).
    struct Node {
        uint64_t w;
        int minb;
        int id;
    };
    auto later = [](const Node &a, const Node &b) {
        return a.w != b.w ? a.w > b.w : a.minb > b.minb;
    };
    std::priority_queue<Node, std::vector<Node>, decltype(later)> heap(later);
    std::vector<int> parent;
    parent.reserve(512);
    int leaf[256];
    for (int b = 0; b < 256; ++b) {
        leaf[b] = -1;
        if (weight[b]) {
            leaf[b] = (int)parent.size();
            parent.push_back(-1);
            heap.push({weight[b], b, leaf[b]});
        }
    }
    uint8_t len[256] = {0};
    if (heap.size() == 1) {
        len[heap.top().minb] = 1;
    } else {
        while (heap.size() > 1) {
            Node a = heap.top();
            heap.pop();
            Node b = heap.top();
            heap.pop();
            int id = (int)parent.size();
            parent.push_back(-1);
            parent[a.id] = id;
            parent[b.id] = id;
            heap.push({a.w + b.w, std::min(a.minb, b.minb), id});
        }
        // depth of every node, computed root-down (children have smaller ids)
        std::vector<int> depth(parent.size(), 0);
        for (int i = (int)parent.size() - 2; i >= 0; --i)
            depth[i] = depth[parent[i]] + 1;
        for (int b = 0; b < 256; ++b) {
            if (leaf[b] < 0)
                continue;
            if ((uint32_t)depth[leaf[b]] > max_len)
                return ECC_ERR_CODEBOOK;
            len[b] = (uint8_t)depth[leaf[b]];
        }
    }

    canonical_fill(len, out);
    return ECC_OK;
}

ecc_status huff_build_limited(const uint64_t weight[256], uint32_t max_len, ecc_codebook *out)
{
    if (!weight || !out || max_len < 1 || max_len > ECC_MAX_CODE_LEN)
        return ECC_ERR_ARG;
    std::vector<int> leaves;
    uint64_t total = 0;
    for (int b = 0; b < 256; ++b)
        if (weight[b]) {
            if (weight[b] >= (1ull << 62) - total)
                return ECC_ERR_ARG; // package sums must fit 64 bits
            total += weight[b];
            leaves.push_back(b);
        }
    const int n = (int)leaves.size();
    if (n == 0)
        return ECC_ERR_ARG;
    uint8_t len[256] = {0};
    if (n == 1) {
        len[leaves[0]] = 1;
        canonical_fill(len, out);
        return ECC_OK;
    }
    if (max_len < 63 && (1ull << max_len) < (uint64_t)n)
        return ECC_ERR_CODEBOOK; // n codewords need more than max_len bits
    std::stable_sort(leaves.begin(), leaves.end(), [&](int a, int b) { return weight[a] < weight[b]; });
    // Package-merge (Larmore and Hirschberg): list d merges the leaves with
    // the packages (consecutive pairs) of list d - 1, a leaf first on equal
    // weight; a symbol's length is its number of occurrences among the
    // first 2n - 2 items of the last list.
    struct Item {
        uint64_t w;
        int sym;  // >= 0: leaf
        int a, b; // package of items a, b of the previous list
    };
    std::vector<std::vector<Item>> lists(max_len + 1);
    for (int b : leaves)
        lists[1].push_back({weight[b], b, -1, -1});
    for (uint32_t d = 2; d <= max_len; ++d) {
        const std::vector<Item> &prev = lists[d - 1];
        std::vector<Item> &cur = lists[d];
        const size_t npk = prev.size() / 2;
        size_t i = 0, j = 0;
        while (i < leaves.size() || j < npk) {
            const uint64_t pw = j < npk ? prev[2 * j].w + prev[2 * j + 1].w : 0;
            if (i < leaves.size() && (j >= npk || weight[leaves[i]] <= pw)) {
                cur.push_back({weight[leaves[i]], leaves[i], -1, -1});
                ++i;
            } else {
                cur.push_back({pw, -1, (int)(2 * j), (int)(2 * j + 1)});
                ++j;
            }
        }
    }
    // count occurrences: an explicit stack of (list, item)
    std::vector<std::pair<uint32_t, int>> stack;
    for (int i = 0; i < 2 * n - 2; ++i)
        stack.push_back({max_len, i});
    while (!stack.empty()) {
        const auto [d, i] = stack.back();
        stack.pop_back();
        const Item &it = lists[d][i];
        if (it.sym >= 0) {
            ++len[it.sym];
        } else {
            stack.push_back({d - 1, it.a});
            stack.push_back({d - 1, it.b});
        }
    }
    canonical_fill(len, out);
    return ECC_OK;
}

ecc_status escape_build_tables(const uint64_t count[256], ecc_codebook *out)
{
    if (!count || !out)
        return ECC_ERR_ARG;
    uint64_t ecount[16] = {0};
    for (int b = 0; b < 256; ++b)
        ecount[(b >> 3) & 15] += count[b];
    int order[16];
    for (int e = 0; e < 16; ++e)
        order[e] = e;
    std::stable_sort(order, order + 16, [&](int a, int b) { return ecount[a] > ecount[b]; });
    int code_of[16]; // 1..7 for the top exponents, 0 for the escaped ones
    for (int e = 0; e < 16; ++e)
        code_of[e] = 0;
    clear(out, ECC_FAMILY_ESCAPE);
    for (int r = 0; r < 7; ++r) {
        code_of[order[r]] = r + 1;
        out->by_rank[r] = (uint8_t)order[r];
    }
    for (int b = 0; b < 256; ++b) {
        const int e = (b >> 3) & 15;
        const uint64_t tail = (uint64_t)(b >> 7) << 3 | (uint64_t)(b & 7); // sign, mantissa
        if (code_of[e]) {
            out->len[b] = 7;
            out->code[b] = (uint64_t)code_of[e] << 4 | tail;
        } else {
            out->len[b] = 11;
            out->code[b] = (uint64_t)e << 4 | tail; // 000, exponent, sign, mantissa
        }
    }
    fill_derived(out);
    return ECC_OK;
}

double ecc_entropy_bits(const uint64_t count[256])
{
    if (!count)
        return std::nan("");
    long double n = 0;
    for (int b = 0; b < 256; ++b)
        n += (long double)count[b];
    if (n == 0)
        return 0.0;
    double h = 0.0;
    for (int b = 0; b < 256; ++b) {
        if (!count[b])
            continue;
        double p = (double)count[b] / (double)n;
        h -= p * std::log2(p);
    }
    return h;
}

double ecc_kl_bits(const uint64_t p_count[256], const uint64_t q_count[256])
{
    if (!p_count || !q_count)
        return std::nan("");
    double np = 0, nq = 0;
    for (int b = 0; b < 256; ++b) {
        np += (double)p_count[b];
        nq += (double)q_count[b];
    }
    double d = 0.0;
    for (int b = 0; b < 256; ++b) {
        if (!p_count[b])
            continue;
        if (!q_count[b])
            return std::numeric_limits<double>::infinity();
        double p = (double)p_count[b] / np, q = (double)q_count[b] / nq;
        d += p * std::log2(p / q);
    }
    return d;
}

ecc_status ecc_code_bits(const uint64_t count[256], const ecc_codebook *cb, uint64_t *bits)
{
    if (!count || !cb || !bits || cb->magic != ECC_CODEBOOK_MAGIC)
        return ECC_ERR_ARG;
    uint64_t s = 0;
    for (int b = 0; b < 256; ++b) {
        if (!count[b])
            continue;
        if (!cb->len[b])
            return ECC_ERR_CODEBOOK;
        s += count[b] * (uint64_t)cb->len[b];
    }
    *bits = s;
    return ECC_OK;
}

size_t ecc_num_chunks(size_t n, uint32_t C) { return C ? (n + C - 1) / C : 0; }
size_t ecc_num_subblocks(size_t n, uint32_t S) { return S ? (n + S - 1) / S : 0; }

size_t ecc_max_encoded_bytes(size_t n, uint32_t C, uint32_t max_len)
{
    if (!C)
        return 0;
    auto chunk = [max_len](size_t L) { return ((L * max_len + 7) / 8 + 15) / 16 * 16; };
    size_t full = n / C, tail = n % C;
    return full * chunk(C) + (tail ? chunk(tail) : 0);
}

const char *ecc_status_string(ecc_status s)
{
    switch (s) {
    case ECC_OK: return "ok";
    case ECC_ERR_ARG: return "invalid argument";
    case ECC_ERR_CAPACITY: return "output capacity exceeded";
    case ECC_ERR_CORRUPT: return "corrupt stream";
    case ECC_ERR_CODEBOOK: return "codebook error";
    case ECC_ERR_TIMEOUT: return "device wait timed out";
    case ECC_ERR_CUDA: return "CUDA error";
    case ECC_ERR_CHECK: return "kernel index out of range (checked build)";
    default: return "unknown status";
    }
}

} // extern "C"
