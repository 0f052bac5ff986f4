// ecc_build.cu -- canonical Huffman codebook built on the device from a
// device histogram, so that histogram -> codebook -> encode runs in one
// stream with no host round trip.  This is the three-stage pipeline
// ("Single-Stage Huffman Encoder for ML Compression", introduction: frequency
// analysis, codebook construction, encoding, per tensor) that the
// single-stage method avoids, and the codebook refresh its discussion asks
// for when the data drift.  The result is byte-identical to the host builder
// huff_build_canonical given the weights count[b] + add.
//
// One CTA of 256 threads, thread t owning byte value t.  The codebook is
// assembled in shared memory and copied out once, coalesced.
//   1. weights, the overflow checks;
//   2. leaves sorted by key (a bitonic network);
//   3. the n - 1 merges in one thread over two queues (see merge_queues);
//   4. code lengths (leaf depths), canonical codes, the derived tables.

#include <cstdint>

#include "ecc_device.cuh"
#include "ecc_launch.h"

namespace ecc {

constexpr int kBuildThreads = 256;
constexpr int kBuildWarps = kBuildThreads / 32;
constexpr int kMaxNodes = 511; // 256 leaves + 255 merges

struct BuildShared {
    uint64_t aw[257];     // leaves sorted by key: weight, or the packed key;
                          // aw[256] = ~0 ends the queue when all 256 are leaves
    uint64_t bw[256];     // internal nodes in creation order: same
    uint16_t ab[257];     // leaves: byte value (unpacked keys only)
    uint16_t bb[256];     // internal nodes: smallest byte below (unpacked only)
    int16_t parent[512];  // node -> internal node index; leaves are nodes
                          // 0..255 (by byte), internal node k is 256 + k
    uint8_t sorted[256];  // coded byte values by (length, value)
    uint32_t bl_count[65];
    uint32_t warp_len[kBuildWarps][ECC_MAX_CODE_LEN + 1]; // bytes of each length per warp
    uint64_t next[65];    // first canonical code of each length
    uint32_t index[65];   // position in sorted[] of the first code of each length
    uint32_t dec_lo[ECC_PEEK_BITS + 1], dec_hi[ECC_PEEK_BITS + 1]; // peek range of each length
    uint64_t warp_sum[kBuildWarps]; // weight sum of each warp's bytes
    uint32_t warp_wrap[kBuildWarps]; // ... did not fit 64 bits
    uint32_t warp_n[kBuildWarps];
    uint32_t err;
};

constexpr size_t kBuildCbOffset = (sizeof(BuildShared) + 15) / 16 * 16;
constexpr size_t kBuildSmem = kBuildCbOffset + sizeof(ecc_codebook);

// The heap order of the host builder: smaller weight first, then the
// smaller byte value below the node.  Live subtrees are disjoint, so no two
// live nodes share a key and the order is total.  When the total weight is
// below 2^55 the key packs into one word, weight << 8 | byte, whose integer
// order is the same and whose sum for a merged node is the sum of the
// weights' parts plus the smaller byte.
__device__ __forceinline__ bool key_less(uint64_t wa, uint32_t ba, uint64_t wb, uint32_t bb)
{
    return (wa < wb) | ((wa == wb) & (ba < bb));
}

__device__ __forceinline__ void fail(BuildShared &sh, ecc_status e) { atomicCAS(&sh.err, 0u, (uint32_t)e); }

// Bitonic sort of one key a thread across the block (ascending; thread t
// ends with the t-th smallest).  Partners within a warp by shuffles, across
// warps through the aw/ab arrays.
template <bool kPacked>
__device__ __forceinline__ void bitonic(BuildShared &sh, uint64_t &kw, uint32_t &kb)
{
    const uint32_t t = threadIdx.x;
    for (uint32_t k = 2; k <= 256; k <<= 1)
        for (uint32_t j = k >> 1; j; j >>= 1) {
            uint64_t pw;
            uint32_t pb = 0;
            if (j < 32) {
                pw = __shfl_xor_sync(~0u, kw, j);
                if (!kPacked)
                    pb = __shfl_xor_sync(~0u, kb, j);
            } else {
                __syncthreads();
                sh.aw[t] = kw;
                if (!kPacked)
                    sh.ab[t] = (uint16_t)kb;
                __syncthreads();
                pw = sh.aw[t ^ j];
                if (!kPacked)
                    pb = sh.ab[t ^ j];
            }
            const bool p_less = kPacked ? pw < kw : key_less(pw, pb, kw, kb);
            const bool k_less = kPacked ? kw < pw : key_less(kw, kb, pw, pb);
            const bool take = ((t & j) == 0) == ((t & k) == 0) ? p_less : k_less;
            kw = take ? pw : kw;
            kb = take ? pb : kb;
        }
}

// The merges.  The heap pops keys in increasing order and each pushed sum
// outweighs what was popped, so internal nodes are created in increasing key
// order (equal weights included: an internal node with the same weight as an
// earlier one would need children no smaller than the earlier one's, which
// forces a larger smallest byte).  Two queues, the sorted leaves and the
// internal nodes in creation order, therefore reproduce the heap exactly:
// each pop takes the smaller head.  Each queue keeps its head and the next
// node in registers plus a pending load of the node after that (index
// clamped; a node not yet created reads as ~0 and is replaced when it is
// created), so a pop consumes a load issued one pop earlier and the loop's
// dependency chain holds compares and selects only.  Run by one thread.
template <bool kPacked>
__device__ __noinline__ void merge_queues(BuildShared &sh, uint32_t n)
{
    uint32_t ia = 0, ib = 0, nb = 0;
    uint64_t a0w = sh.aw[0], a1w = sh.aw[1], paw = sh.aw[2], b0w = ~0ull, b1w = ~0ull, pbw = ~0ull;
    uint32_t a0b = 0, a1b = 0, pab = 0, b0b = 0, b1b = 0, pbb = 0;
    if (!kPacked)
        a0b = sh.ab[0], a1b = sh.ab[1], pab = sh.ab[2];
    for (uint32_t m = 0; m + 1 < n; ++m) {
        uint64_t w2[2];
        uint32_t b2[2], id2[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            // packed: leaves past the last and internal nodes not yet
            // created hold the key ~0, above every real key, so the compare
            // alone decides
            const bool take_a =
                kPacked ? a0w < b0w : (ia < n) & ((ib == nb) | key_less(a0w, a0b, b0w, b0b));
            w2[p] = take_a ? a0w : b0w;
            b2[p] = take_a ? a0b : b0b;
            id2[p] = take_a ? (kPacked ? (uint32_t)(a0w & 255u) : a0b) : 256u + ib;
            a0w = take_a ? a1w : a0w, a1w = take_a ? paw : a1w;
            b0w = take_a ? b0w : b1w, b1w = take_a ? b1w : pbw;
            if (!kPacked) {
                a0b = take_a ? a1b : a0b, a1b = take_a ? pab : a1b;
                b0b = take_a ? b0b : b1b, b1b = take_a ? b1b : pbb;
            }
            ia += take_a ? 1u : 0u;
            ib += take_a ? 0u : 1u;
            const uint32_t ja = min(ia + 2, 256u), jb = min(ib + 2, 255u);
            paw = sh.aw[ja];
            pbw = sh.bw[jb];
            if (!kPacked)
                pab = sh.ab[ja], pbb = sh.bb[jb];
        }
        sh.parent[id2[0]] = (int16_t)nb;
        sh.parent[id2[1]] = (int16_t)nb;
        uint64_t nw;
        uint32_t nbyte = 0;
        if (kPacked) {
            nw = (w2[0] & ~255ull) + (w2[1] & ~255ull) + min(w2[0] & 255u, w2[1] & 255u);
        } else {
            nw = w2[0] + w2[1];
            nbyte = min(b2[0], b2[1]);
            sh.bb[nb] = (uint16_t)nbyte;
        }
        sh.bw[nb] = nw;
        // the new node heads the internal queue, follows its head, or is the
        // pending one
        b0w = ib == nb ? nw : b0w;
        b1w = ib + 1 == nb ? nw : b1w;
        pbw = ib + 2 == nb ? nw : pbw;
        if (!kPacked) {
            b0b = ib == nb ? nbyte : b0b;
            b1b = ib + 1 == nb ? nbyte : b1b;
            pbb = ib + 2 == nb ? nbyte : pbb;
        }
        ++nb;
    }
}

// Copy the shared codebook to the output (16-byte words, then the last
// 8 bytes when its size is 8 modulo 16).
__device__ __forceinline__ void copy_out(const ecc_codebook *cbs, ecc_codebook *out)
{
    constexpr uint32_t n16 = sizeof(ecc_codebook) / 16;
    static_assert(sizeof(ecc_codebook) % 8 == 0, "codebook size");
    const uint4 *s = reinterpret_cast<const uint4 *>(cbs);
    uint4 *d = reinterpret_cast<uint4 *>(out);
    for (uint32_t i = threadIdx.x; i < n16; i += kBuildThreads)
        d[i] = s[i];
    if (sizeof(ecc_codebook) % 16 == 8 && threadIdx.x == 0)
        reinterpret_cast<uint2 *>(out)[2 * n16] = reinterpret_cast<const uint2 *>(cbs)[2 * n16];
}

__global__ void __launch_bounds__(kBuildThreads) huff_build_kernel(const uint64_t *count, uint64_t add,
                                                                  uint32_t max_len, ecc_codebook *out,
                                                                  uint32_t *status)
{
    extern __shared__ __align__(16) uint8_t build_smem[];
    BuildShared &sh = *reinterpret_cast<BuildShared *>(build_smem);
    ecc_codebook *cbs = reinterpret_cast<ecc_codebook *>(build_smem + kBuildCbOffset);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;

    // ---- 1. weights; the codebook starts all zero, as the host builder's
    // (on an error it is copied out so, without its magic word, and every
    // call that is handed it rejects it)
    const uint64_t c = count[t];
    {
        uint2 *z = reinterpret_cast<uint2 *>(cbs);
        for (uint32_t i = t; i < sizeof(ecc_codebook) / 8; i += kBuildThreads)
            z[i] = make_uint2(0, 0);
    }
    const uint64_t wb = c + add;
    const bool present = wb != 0;
    const unsigned ball = __ballot_sync(~0u, present);
    // the total weight must fit 64 bits and be nonzero: a butterfly sum per
    // warp that notes any wrap, then the eight warp sums
    {
        uint64_t sum = wb;
        bool wrap = c > ~0ull - add;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const uint64_t s2 = __shfl_xor_sync(~0u, sum, o);
            wrap = __shfl_xor_sync(~0u, (int)wrap, o) != 0 || wrap || s2 > ~0ull - sum;
            sum += s2;
        }
        if (lane == 0) {
            sh.warp_n[warp] = __popc(ball);
            sh.warp_sum[warp] = sum;
            sh.warp_wrap[warp] = wrap;
        }
    }
    if (t <= 64)
        sh.bl_count[t] = 0;
    for (int k = t; k < kBuildWarps * (ECC_MAX_CODE_LEN + 1); k += kBuildThreads)
        (&sh.warp_len[0][0])[k] = 0;
    sh.parent[t] = -1;
    sh.parent[t + 256] = -1;
    sh.bw[t] = ~0ull; // internal nodes not yet created: keys above every node's
    sh.bb[t] = 0;
    if (t == 0) {
        sh.err = 0;
        sh.aw[256] = ~0ull;
        sh.ab[256] = 0;
    }
    __syncthreads();
    uint32_t n_leaves = 0;
    uint64_t total = 0;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kBuildWarps; ++k) {
        n_leaves += sh.warp_n[k];
        bad |= sh.warp_wrap[k] != 0 || sh.warp_sum[k] > ~0ull - total;
        total += sh.warp_sum[k];
    }
    if (bad || total == 0) {
        copy_out(cbs, out);
        if (t == 0)
            *status = ECC_ERR_ARG;
        return;
    }
    const bool packed = (total >> 55) == 0;

    // ---- 2-3. sorted leaves (absent bytes last), then the merges
    if (packed) {
        uint64_t kw = present ? (wb << 8 | (uint32_t)t) : ~0ull;
        uint32_t kb = 0;
        bitonic<true>(sh, kw, kb);
        __syncthreads();
        sh.aw[t] = kw;
        __syncthreads();
        if (t == 0 && n_leaves > 1)
            merge_queues<true>(sh, n_leaves);
    } else {
        uint64_t kw = present ? wb : ~0ull;
        uint32_t kb = present ? (uint32_t)t : 256u + (uint32_t)t;
        bitonic<false>(sh, kw, kb);
        __syncthreads();
        sh.aw[t] = kw;
        sh.ab[t] = (uint16_t)kb;
        __syncthreads();
        if (t == 0 && n_leaves > 1)
            merge_queues<false>(sh, n_leaves);
    }
    __syncthreads();

    // ---- 4. code lengths: the depth of each leaf; a lone symbol gets 1
    uint32_t L = 0;
    if (present) {
        if (n_leaves == 1) {
            L = 1;
        } else {
            int x = t;
            while (sh.parent[x] >= 0 && L <= kMaxNodes) {
                x = 256 + sh.parent[x];
                ++L;
            }
        }
        if (L > max_len) {
            fail(sh, ECC_ERR_CODEBOOK);
            L = 0;
        }
    }
    // canonical codes (RFC 1951 section 3.2.2): codes of one length are
    // consecutive in byte order.  r = bytes before t of the same length:
    // within the warp by a match mask, across warps by per-warp counts.
    const unsigned same = __match_any_sync(~0u, L);
    const uint32_t r_in = __popc(same & ((1u << lane) - 1));
    if (L && r_in == 0) {
        sh.warp_len[warp][L] = __popc(same);
        atomicAdd(&sh.bl_count[L], __popc(same));
    }
    __syncthreads();
    if (sh.err) {
        copy_out(cbs, out);
        if (t == 0)
            *status = sh.err;
        return;
    }
    if (warp == 0) {
        // lane handles lengths k1 = lane + 1 and k2 = lane + 33.  The first
        // code of length k is (first[k-1] + count[k-1]) << 1 from first[1] = 0,
        // i.e. the sum over j < k of count[j] << (k - j), modulo 2^64.
        const uint32_t k1 = lane + 1, k2 = lane + 33;
        uint64_t f1 = 0, f2 = 0;
        uint32_t i1 = 0, i2 = 0;
#pragma unroll
        for (uint32_t j = 1; j < 64; ++j) {
            const uint32_t bl = sh.bl_count[j];
            const bool below1 = j < k1, below2 = j < k2;
            f1 += below1 ? (uint64_t)bl << ((k1 - j) & 63) : 0ull;
            i1 += below1 ? bl : 0u;
            f2 += below2 ? (uint64_t)bl << ((k2 - j) & 63) : 0ull;
            i2 += below2 ? bl : 0u;
        }
        sh.next[k1] = f1;
        sh.next[k2] = f2;
        sh.index[k1] = i1;
        sh.index[k2] = i2;
        const uint32_t c1 = sh.bl_count[k1], c2 = k2 <= ECC_MAX_CODE_LEN ? sh.bl_count[k2] : 0u;
        cbs->index[k1] = (uint16_t)i1;
        cbs->count[k1] = (uint16_t)c1;
        cbs->first[k1] = f1;
        if (k2 <= ECC_MAX_CODE_LEN) {
            cbs->index[k2] = (uint16_t)i2;
            cbs->count[k2] = (uint16_t)c2;
            cbs->first[k2] = f2;
        }
        if (k1 <= ECC_PEEK_BITS) {
            sh.dec_lo[k1] = (uint32_t)(f1 << (ECC_PEEK_BITS - k1));
            sh.dec_hi[k1] = (uint32_t)((f1 + c1) << (ECC_PEEK_BITS - k1));
        }
        const unsigned m1 = __ballot_sync(~0u, c1 != 0), m2 = __ballot_sync(~0u, c2 != 0);
        if (lane == 0) {
            cbs->min_len = m1 ? __ffs(m1) : 32 + __ffs(m2);
            cbs->max_len = m2 ? 64 - __clz(m2) : 32 - __clz(m1);
            cbs->n_coded = n_leaves;
            cbs->family = ECC_FAMILY_HUFFMAN;
            cbs->magic = ECC_CODEBOOK_MAGIC;
        }
    }
    __syncthreads();
    if (L) {
        uint32_t r = r_in;
        for (int k = 0; k < warp; ++k)
            r += sh.warp_len[k][L];
        const uint64_t code = sh.next[L] + r;
        cbs->len[t] = (uint8_t)L;
        cbs->code[t] = code;
        sh.sorted[sh.index[L] + r] = (uint8_t)t;
        cbs->sorted[sh.index[L] + r] = (uint8_t)t;
        if (L <= 31) {
            cbs->enc_code[t] = (uint32_t)(code << (32 - L));
            cbs->enc_mul[t] = 1u << (32 - L);
        }
    }
    __syncthreads();
    // the 14-bit first-level decode table.  Canonical codes of length
    // k <= 14, left-aligned to 14 bits, tile [dec_lo[k], dec_hi[k]) in order
    // of k; entry i holds byte | k << 8 of the code that prefixes i.  Entries
    // under longer codes stay 0.
    for (uint32_t k = 1; k <= ECC_PEEK_BITS; ++k) {
        const uint32_t lo = sh.dec_lo[k], hi = sh.dec_hi[k], base = sh.index[k];
#pragma unroll 4
        for (uint32_t i = lo + t; i < hi; i += kBuildThreads)
            cbs->dec[i] = (uint16_t)(sh.sorted[base + ((i - lo) >> (ECC_PEEK_BITS - k))] | (k << 8));
    }
    __syncthreads();
    copy_out(cbs, out);
    if (t == 0)
        *status = ECC_OK;
}

} // namespace ecc

using namespace ecc;

extern "C" ecc_status huff_build_device(const uint64_t *count, uint64_t add, uint32_t max_len, ecc_codebook *out,
                                        uint32_t *status, void *stream)
{
    if (!count || !out || !status || !aligned16(out) || max_len < 1 || max_len > ECC_MAX_CODE_LEN)
        return ECC_ERR_ARG;
    if (occupancy((const void *)huff_build_kernel, kBuildThreads, kBuildSmem) <= 0)
        return launch_status(cudaErrorInvalidConfiguration);
    huff_build_kernel<<<1, kBuildThreads, kBuildSmem, (cudaStream_t)stream>>>(count, add, max_len, out, status);
    return launch_status(cudaGetLastError());
}
