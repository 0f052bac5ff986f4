// ecc_bf16.cu -- the exponent escape code on BF16 tensors (ZipCCL, gist.science
// summary of arXiv 2604.27844, section 2.B "Tecnica di Codifica degli
// Esponenti"): a BF16 value (sign bit 15, exponent bits 14-7, mantissa bits
// 6-0) is written as a 3-bit code 001..111 when its exponent is one of a
// table of 7, else as 000 followed by the 8-bit exponent; its sign and its 7
// mantissa bits follow as they are (11 or 19 bits a value).  Section 2.A:
// the table is the 7 exponents a Gaussian of the layer's standard deviation
// makes most probable (no histogram of the data), or the 7 most frequent ones
// of a histogram.  The stream uses the library's container (chunks of C
// values, 16-byte padded payloads, chunk_off, sub_bits per S values).
//
// Kernels: an exponent histogram (lane-private shared counters); the encoder
// (chunks of at most 4096 values: a warp a chunk, claimed by ticket, coded in
// rounds of 16 values a lane placed by a warp scan, packed into the warp's
// zeroed shared stage, placed by decoupled look-back and written out
// byte-swapped with 16-byte stores; larger chunks: the same with a CTA of 256
// threads a chunk and block scans); the decoder (a warp per chunk, a lane per
// sub-block, codes read through a three-word window, eight values a 16-byte
// store).

#include <algorithm>
#include <cmath>

#include "ecc_device.cuh"
#include "ecc_launch.h"

namespace ecc {

constexpr int kBfThreads = 256;
constexpr uint32_t kBfPerThread = 16;                    // values a thread codes in a tile
constexpr uint32_t kBfTile = kBfThreads * kBfPerThread;  // 4096 values
constexpr uint32_t kBfMaxC = 16384;

// ---------------------------------------------------------------- histogram
__global__ void __launch_bounds__(kBfThreads) bf16_hist_kernel(const uint16_t *in, uint64_t n,
                                                               unsigned long long *count)
{
    __shared__ uint32_t h[256 * 32]; // counter e of lane l at word e * 32 + l
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 256 * 32; i += kBfThreads)
        h[i] = 0;
    __syncthreads();
    const uint64_t nv = n / 8; // 16-byte vectors
    const uint4 *v4 = reinterpret_cast<const uint4 *>(in);
    for (uint64_t i = (uint64_t)blockIdx.x * kBfThreads + tid; i < nv; i += (uint64_t)gridDim.x * kBfThreads) {
        const uint4 v = ld_stream16(v4 + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            atomicAdd(&h[((w[k] >> 7) & 0xFFu) * 32 + lane], 1u);
            atomicAdd(&h[((w[k] >> 23) & 0xFFu) * 32 + lane], 1u);
        }
    }
    if (blockIdx.x == 0)
        for (uint64_t i = nv * 8 + tid; i < n; i += kBfThreads)
            atomicAdd(&h[((in[i] >> 7) & 0xFFu) * 32 + lane], 1u);
    __syncthreads();
    for (int e = warp; e < 256; e += kBfThreads / 32) {
        uint32_t c = h[e * 32 + lane];
#pragma unroll
        for (int o = 16; o; o >>= 1)
            c += __shfl_xor_sync(~0u, c, o);
        if (lane == 0 && c)
            atomicAdd(count + e, (unsigned long long)c);
    }
}

// ---------------------------------------------------------------- encoder
struct BfTable {
    uint8_t top[8]; // the 7 exponents in rank order (top[7] unused)
};

struct BfEncParams {
    const uint16_t *in;
    uint64_t n;
    BfTable tab;
    uint32_t C, S;
    uint8_t *out;
    uint64_t out_cap;
    uint64_t *chunk_off;
    uint16_t *sub_bits;
    uint64_t *total_bits;
    uint64_t *flags;
    uint32_t *ticket;
    uint32_t *status;
    uint64_t n_chunks;
    uint32_t stage_bytes;
    uint64_t timeout_ns;
};

// code of one value: (code, length) with rank[e] = 1..7 for table exponents, 0 else
__device__ __forceinline__ uint32_t bf_code(uint32_t v, const uint8_t *rank, uint32_t &len)
{
    const uint32_t e = (v >> 7) & 0xFFu;
    const uint32_t sm = ((v >> 8) & 0x80u) | (v & 0x7Fu); // sign, mantissa
    const uint32_t r = rank[e];
    len = r ? 11u : 19u;
    return r ? (r << 8) | sm : (e << 8) | sm;
}

__global__ void __launch_bounds__(kBfThreads) bf16_encode_kernel(BfEncParams p)
{
    extern __shared__ __align__(16) uint8_t bf_smem[];
    uint32_t *stage = reinterpret_cast<uint32_t *>(bf_smem);
    __shared__ uint8_t rank[256];
    __shared__ uint32_t warp_tot[kBfThreads / 32];
    __shared__ uint32_t incl_s[kBfThreads];
    __shared__ uint64_t prefix_s;
    __shared__ uint32_t ticket_s, flags_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < 256; e += kBfThreads)
        rank[e] = 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 7; ++r) // static indices: the parameter block stays out of local memory
        if (tid == r)
            rank[p.tab.top[r]] = (uint8_t)(r + 1);
    for (uint32_t i = tid; i < p.stage_bytes / 16; i += kBfThreads)
        reinterpret_cast<uint4 *>(stage)[i] = make_uint4(0, 0, 0, 0);
    const uint32_t s_shift = 31u - __clz(p.S);
    for (;;) {
        if (tid == 0) {
            ticket_s = atomicAdd(p.ticket, 1u);
            flags_s = 0;
        }
        __syncthreads();
        const uint64_t c = ticket_s;
        if (c >= p.n_chunks)
            break;
        const uint64_t base = c * p.C;
        const uint32_t L = (uint32_t)min((uint64_t)p.C, p.n - base);
        uint32_t run = 0; // bits of the chunk's earlier tiles
        for (uint32_t t0 = 0; t0 < L; t0 += kBfTile) {
            const uint32_t my0 = t0 + (uint32_t)tid * kBfPerThread;
            const uint32_t cnt = my0 < L ? min(kBfPerThread, L - my0) : 0u;
            uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (cnt == kBfPerThread) {
                const uint4 a = ld_stream16(p.in + base + my0), b = ld_stream16(p.in + base + my0 + 8);
                w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
            } else {
                for (uint32_t j = 0; j < cnt; ++j)
                    w[j >> 1] |= (uint32_t)p.in[base + my0 + j] << (16 * (j & 1));
            }
            uint32_t bits = 0;
#pragma unroll
            for (uint32_t j = 0; j < kBfPerThread; ++j) {
                uint32_t len;
                (void)bf_code((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, rank, len);
                bits += j < cnt ? len : 0u;
            }
            uint32_t incl = bits;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(~0u, incl, o);
                if (lane >= o)
                    incl += y;
            }
            if (lane == 31)
                warp_tot[warp] = incl;
            __syncthreads();
            uint32_t before = 0, tile = 0;
#pragma unroll
            for (int u = 0; u < kBfThreads / 32; ++u) {
                before += u < warp ? warp_tot[u] : 0u;
                tile += warp_tot[u];
            }
            incl += before;
            incl_s[tid] = incl;
            __syncthreads();
            // sub-blocks of S values: S / 16 threads each (4 .. 64)
            const uint32_t tps = p.S / kBfPerThread;
            if (cnt && (tid & (tps - 1)) == 0) {
                const uint32_t last = min((uint32_t)tid + tps - 1, (uint32_t)kBfThreads - 1);
                p.sub_bits[(base + my0) >> s_shift] = (uint16_t)(incl_s[last] - (incl - bits));
            }
            const uint32_t pos = run + incl - bits;
            if (cnt) {
                if ((uint64_t)(pos + bits + 31) / 32 * 4 <= p.stage_bytes) {
                    Packer<false> pk;
                    pk.start(stage, pos);
                    for (uint32_t j = 0; j < cnt; ++j) {
                        uint32_t len;
                        const uint32_t code = bf_code((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, rank, len);
                        pk.put(code, len);
                    }
                    pk.finish();
                } else {
                    atomicOr(&flags_s, 1u); // cannot happen: the stage holds C values at 19 bits
                }
            }
            run += tile;
            __syncthreads(); // warp_tot and incl_s are rewritten by the next tile
        }
        const uint64_t bytes = ((uint64_t)run + 127u) / 128u * 16u;
        if (warp == 0) {
            bool to;
            const uint64_t prefix = lookback(p.flags, c, bytes, p.timeout_ns, &to);
            if (lane == 0) {
                prefix_s = prefix;
                if (to) {
                    atomicOr(&flags_s, 2u);
                    set_status(p.status, ECC_ERR_TIMEOUT);
                }
                p.chunk_off[c + 1] = prefix + bytes;
                if (c == 0)
                    p.chunk_off[0] = 0;
                atomicAdd((unsigned long long *)p.total_bits, (unsigned long long)run);
            }
        }
        __syncthreads();
        const uint64_t prefix = prefix_s;
        const bool fits = prefix + bytes <= p.out_cap;
        if (!fits && tid == 0 && !(flags_s & 2u))
            set_status(p.status, ECC_ERR_CAPACITY);
        if (flags_s & 1u && tid == 0)
            set_status(p.status, ECC_ERR_CHECK);
        const bool write = fits && !flags_s;
        uint4 *st4 = reinterpret_cast<uint4 *>(stage);
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + prefix);
        for (uint32_t i = tid; i < (uint32_t)(bytes / 16); i += kBfThreads) {
            const uint4 v = st4[i];
            st4[i] = make_uint4(0, 0, 0, 0);
            if (write)
                st_stream16(dst + i, bswap4(v));
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- warp encoder
// Chunks of at most kBfWarpC values, a warp a chunk: rounds of 512 values
// (16 a lane) placed by a warp scan of the code lengths and packed into the
// warp's own zeroed stage; the chunk's sub-block counts from the bit
// positions where its sub-blocks start; then its offset by the look-back, and
// the stage written out and cleared.  After the start no CTA barrier: a warp
// waiting on its look-back holds up no other warp.
constexpr uint32_t kBfWarpC = 4096;
constexpr int kBfWarpThreads = 128;
constexpr uint32_t kBfRound = 32 * kBfPerThread;   // 512 values
constexpr uint32_t kBfSubMax = kBfWarpC / 64 + 1;  // sub-blocks of a chunk (S >= 64)

__global__ void __launch_bounds__(kBfWarpThreads) bf16_encode_warp_kernel(BfEncParams p)
{
    extern __shared__ __align__(16) uint8_t bfw_smem[];
    __shared__ uint8_t rank[256];
    __shared__ uint32_t subpos[kBfWarpThreads / 32][kBfSubMax]; // bit where each sub-block starts
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < 256; e += kBfWarpThreads)
        rank[e] = 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 7; ++r) // static indices: the parameter block stays out of local memory
        if (tid == r)
            rank[p.tab.top[r]] = (uint8_t)(r + 1);
    __syncthreads();
    uint32_t *stage = reinterpret_cast<uint32_t *>(bfw_smem + (size_t)warp * p.stage_bytes);
    uint4 *st4 = reinterpret_cast<uint4 *>(stage);
    for (uint32_t i = lane; i < p.stage_bytes / 16; i += 32)
        st4[i] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    const uint32_t s_shift = 31u - __clz(p.S);
    uint32_t *sp = subpos[warp];
    for (;;) {
        uint32_t tk = 0;
        if (lane == 0)
            tk = atomicAdd(p.ticket, 1u);
        const uint64_t c = __shfl_sync(~0u, tk, 0);
        if (c >= p.n_chunks)
            break;
        const uint64_t base = c * p.C;
        const uint32_t L = (uint32_t)min((uint64_t)p.C, p.n - base);
        // the lane's 16 values of the round starting at t0 (zeros past the chunk)
        auto load_round = [&](uint32_t t0, uint32_t (&w)[8]) {
            const uint32_t my0 = t0 + (uint32_t)lane * kBfPerThread;
            const uint32_t cnt = my0 < L ? min(kBfPerThread, L - my0) : 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                w[k] = 0;
            if (cnt == kBfPerThread) {
                const uint4 a = ld_stream16(p.in + base + my0), b = ld_stream16(p.in + base + my0 + 8);
                w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
            } else {
#pragma unroll
                for (uint32_t j = 0; j < kBfPerThread; ++j) // unrolled: w stays in registers
                    if (j < cnt)
                        w[j >> 1] |= (uint32_t)p.in[base + my0 + j] << (16 * (j & 1));
            }
        };
        uint32_t wn[8]; // the next round's values, loaded one round ahead
        load_round(0, wn);
        uint32_t run = 0; // bits of the chunk's earlier rounds
        for (uint32_t t0 = 0; t0 < L; t0 += kBfRound) {
            const uint32_t my0 = t0 + (uint32_t)lane * kBfPerThread;
            const uint32_t cnt = my0 < L ? min(kBfPerThread, L - my0) : 0u;
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                w[k] = wn[k];
            if (t0 + kBfRound < L)
                load_round(t0 + kBfRound, wn);
            uint32_t bits = 0;
#pragma unroll
            for (uint32_t j = 0; j < kBfPerThread; ++j) {
                uint32_t len;
                (void)bf_code((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, rank, len);
                bits += j < cnt ? len : 0u;
            }
            uint32_t incl = bits;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(~0u, incl, o);
                if (lane >= o)
                    incl += y;
            }
            const uint32_t pos = run + incl - bits;
            if (cnt && (my0 & (p.S - 1u)) == 0)
                sp[my0 >> s_shift] = pos;
            if (cnt) {
                Packer<false> pk;
                pk.start(stage, pos);
#pragma unroll
                for (uint32_t j = 0; j < kBfPerThread; ++j) {
                    if (j < cnt) {
                        uint32_t len;
                        const uint32_t code = bf_code((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, rank, len);
                        pk.put(code, len);
                    }
                }
                pk.finish();
            }
            run += __shfl_sync(~0u, incl, 31);
        }
        __syncwarp(); // the stage and the sub-block starts are complete
        const uint32_t nsub = (L + p.S - 1u) >> s_shift;
        for (uint32_t k = lane; k < nsub; k += 32) {
            const uint32_t e = k + 1 < nsub ? sp[k + 1] : run;
            p.sub_bits[(base >> s_shift) + k] = (uint16_t)(e - sp[k]);
        }
        const uint64_t bytes = ((uint64_t)run + 127u) / 128u * 16u;
        bool to;
        const uint64_t prefix = lookback(p.flags, c, bytes, p.timeout_ns, &to);
        if (lane == 0) {
            if (to)
                set_status(p.status, ECC_ERR_TIMEOUT);
            p.chunk_off[c + 1] = prefix + bytes;
            if (c == 0)
                p.chunk_off[0] = 0;
            atomicAdd((unsigned long long *)p.total_bits, (unsigned long long)run);
        }
        const bool fits = prefix + bytes <= p.out_cap;
        if (!fits && !to && lane == 0)
            set_status(p.status, ECC_ERR_CAPACITY);
        const bool write = fits && !to;
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + prefix);
        for (uint32_t i = lane; i < (uint32_t)(bytes / 16); i += 32) {
            const uint4 v = st4[i];
            st4[i] = make_uint4(0, 0, 0, 0);
            if (write)
                st_stream16(dst + i, bswap4(v));
        }
        __syncwarp(); // the stage is clear and the sub-block starts are read
    }
}

// ---------------------------------------------------------------- decoder
struct BfDecParams {
    const uint8_t *in;
    uint64_t in_bytes;
    const uint64_t *chunk_off;
    const uint16_t *sub_bits;
    uint64_t n;
    uint32_t C, S;
    BfTable tab;
    uint16_t *out;
    uint32_t *status;
    uint64_t n_chunks;
};

// One value of a lane's stream: the window (hi, lo, nx, nn) holds the next
// 128 bits from bit o of hi (o < 32), wi is the index of the word after nn.
// A value takes 11 or 19 bits, so the window moves by at most one word; when
// it does, the word after nn is loaded (word(wi)), and its value is needed
// only at a later move, two or more values on, which hides the load.
// tA/tB: the table's exponents 0-3 and 4-6, one a byte.  Returns the BF16
// value; sets bad for 000 followed by a table exponent.
template <typename WordFn>
__device__ __forceinline__ uint32_t bf_step(uint32_t &hi, uint32_t &lo, uint32_t &nx, uint32_t &nn, uint32_t &o,
                                            uint32_t &wi, const WordFn &word, uint32_t tA, uint32_t tB,
                                            const uint8_t *rank, bool &bad)
{
    const uint32_t top = __funnelshift_l(lo, hi, o);
    const uint32_t code = top >> 29;
    const bool esc = code == 0;
    const uint32_t et = __byte_perm(tA, tB, (code - 1u) & 7u) & 0xFFu; // code - 1 = 7 for an escape (unused byte)
    const uint32_t e = esc ? (top >> 21) & 0xFFu : et;
    const uint32_t tail = esc ? (top >> 13) & 0xFFu : (top >> 21) & 0xFFu;
    if (esc)
        bad |= rank[e] != 0; // a table exponent has a short code
    o += esc ? 19u : 11u;
    const bool adv = o >= 32u;
    hi = adv ? lo : hi;
    lo = adv ? nx : lo;
    nx = adv ? nn : nx;
    if (adv) {
        nn = word(wi);
        ++wi;
    }
    o &= 31u;
    return ((tail & 0x80u) << 8) | (e << 7) | (tail & 0x7Fu);
}

// A warp per chunk, a lane per sub-block (rounds of 32 sub-blocks): each lane
// decodes its sub-block from a three-word window over the chunk's words
// (read through the read-only path, clamped to the chunk), eight values at a
// time, written as one 16-byte store.
__global__ void __launch_bounds__(256) bf16_decode_kernel(BfDecParams p)
{
    __shared__ uint8_t rank[256];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int e = tid; e < 256; e += 256)
        rank[e] = 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 7; ++r) // static indices: the parameter block stays out of local memory
        if (tid == r)
            rank[p.tab.top[r]] = (uint8_t)(r + 1);
    __syncthreads();
    const uint32_t tA = p.tab.top[0] | (uint32_t)p.tab.top[1] << 8 | (uint32_t)p.tab.top[2] << 16 |
                        (uint32_t)p.tab.top[3] << 24;
    const uint32_t tB = p.tab.top[4] | (uint32_t)p.tab.top[5] << 8 | (uint32_t)p.tab.top[6] << 16;
    const uint64_t gw = (uint64_t)blockIdx.x * (blockDim.x / 32) + (tid >> 5);
    const uint64_t nw = (uint64_t)gridDim.x * (blockDim.x / 32);
    const uint32_t s_shift = 31u - __clz(p.S);
    for (uint64_t c = gw; c < p.n_chunks; c += nw) {
        const uint64_t c0 = p.chunk_off[c], c1 = p.chunk_off[c + 1];
        const uint64_t base = c * p.C;
        const uint32_t L = (uint32_t)min((uint64_t)p.C, p.n - base);
        const uint32_t nsub = (L + p.S - 1) >> s_shift;
        // a chunk of at least one value holds at least 16 bytes
        bool bad = c1 < c0 + 16 || c1 > p.in_bytes || (c0 & 15) || (c1 & 15) || (c == 0 && c0 != 0);
        if (__any_sync(~0u, bad)) {
            if (lane == 0)
                set_status(p.status, ECC_ERR_CORRUPT);
            continue;
        }
        const uint32_t *words = reinterpret_cast<const uint32_t *>(p.in + c0);
        const uint32_t wlast = (uint32_t)((c1 - c0) / 4) - 1u;
        auto word = [&](uint32_t k) { return bswap32(__ldg(words + min(k, wlast))); };
        uint64_t run = 0; // bits of the sub-blocks before this round
        for (uint32_t r0 = 0; r0 < nsub; r0 += 32) {
            const uint32_t j = r0 + lane;
            const uint32_t sb = j < nsub ? p.sub_bits[((base >> s_shift) + j)] : 0u;
            uint32_t incl = sb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(~0u, incl, o);
                if (lane >= o)
                    incl += y;
            }
            const uint64_t start = run + incl - sb; // bit offset in the chunk
            run += __shfl_sync(~0u, incl, 31);
            if (j >= nsub)
                continue;
            if (start + sb > (uint64_t)(wlast + 1u) * 32u) { // more bits than the chunk holds
                bad = true;
                continue;
            }
            const uint32_t v0 = j << s_shift, v1 = min(v0 + p.S, L);
            uint32_t wi = (uint32_t)(start >> 5), o = (uint32_t)start & 31u;
            uint32_t hi = word(wi), lo = word(wi + 1), nx = word(wi + 2), nn = word(wi + 3);
            wi += 4; // the next word to load
            uint16_t *dst = p.out + base;
            uint32_t v = v0;
            for (; v + 8 <= v1; v += 8) { // p.out + base + v is 16-byte aligned (C, S multiples of 8)
                uint32_t q[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint32_t a = bf_step(hi, lo, nx, nn, o, wi, word, tA, tB, rank, bad);
                    const uint32_t b = bf_step(hi, lo, nx, nn, o, wi, word, tA, tB, rank, bad);
                    q[h] = a | b << 16;
                }
#ifdef ECC_CHECKED
                if (base + v + 8 > p.n) {
                    set_status(p.status, ECC_ERR_CHECK);
                    break;
                }
#endif
                *reinterpret_cast<uint4 *>(dst + v) = make_uint4(q[0], q[1], q[2], q[3]);
            }
            for (; v < v1; ++v)
                dst[v] = (uint16_t)bf_step(hi, lo, nx, nn, o, wi, word, tA, tB, rank, bad);
            // consumed bits: (words loaded - 4) * 32 + o
            bad |= (uint64_t)(wi - 4u) * 32u + o - start != sb;
        }
        // the chunk ends at its padded size, and the padding is zero
        if (lane == 0) {
            bad |= ((run + 127) / 128) * 16 != c1 - c0;
            if (!bad) {
                uint64_t wk = run >> 5;
                if (run & 31)
                    bad |= (word((uint32_t)(wk++)) << (run & 31)) != 0;
                for (; wk <= wlast; ++wk)
                    bad |= word((uint32_t)wk) != 0;
            }
        }
        if (__any_sync(~0u, bad) && lane == 0)
            set_status(p.status, ECC_ERR_CORRUPT);
    }
}

} // namespace ecc

using namespace ecc;

namespace {
bool bf_table_ok(const uint8_t top[7])
{
    bool seen[256] = {};
    for (int r = 0; r < 7; ++r) {
        if (seen[top[r]])
            return false;
        seen[top[r]] = true;
    }
    return true;
}
} // namespace

extern "C" {

ecc_status bf16_escape_table_counts(const uint64_t count[256], uint8_t top7[7])
{
    if (!count || !top7)
        return ECC_ERR_ARG;
    int order[256];
    for (int e = 0; e < 256; ++e)
        order[e] = e;
    std::stable_sort(order, order + 256, [&](int a, int b) { return count[a] > count[b]; });
    for (int r = 0; r < 7; ++r)
        top7[r] = (uint8_t)order[r];
    return ECC_OK;
}

ecc_status bf16_escape_table_sigma(double sigma, uint8_t top7[7])
{
    if (!top7 || !(sigma > 0.0) || !std::isfinite(sigma))
        return ECC_ERR_ARG;
    // P(field e) = P(|x| in [lo_e, hi_e)) with the edges 2^k moved to the
    // round-to-nearest midpoints 2^k (1 - 2^-9): erfc(lo / (sigma sqrt 2)) -
    // erfc(hi / (sigma sqrt 2))
    double pr[256];
    const double m = 1.0 - std::ldexp(1.0, -9), d = sigma * std::sqrt(2.0);
    for (int e = 0; e < 256; ++e) {
        const double lo = e == 0 ? 0.0 : std::ldexp(1.0, e - 127) * m;
        const double hi_tail = e == 255 ? 0.0 : std::erfc(std::ldexp(1.0, e == 0 ? -126 : e - 126) * m / d);
        pr[e] = std::erfc(lo / d) - hi_tail;
    }
    int order[256];
    for (int e = 0; e < 256; ++e)
        order[e] = e;
    std::stable_sort(order, order + 256, [&](int a, int b) { return pr[a] > pr[b]; });
    for (int r = 0; r < 7; ++r)
        top7[r] = (uint8_t)order[r];
    return ECC_OK;
}

size_t bf16_escape_max_encoded_bytes(size_t n, uint32_t C)
{
    if (!C)
        return 0;
    const size_t full = n / C, tail = n % C;
    const size_t per = ((size_t)C * 19 + 7) / 8;
    return full * ((per + 15) / 16 * 16) + (tail ? (((tail * 19 + 7) / 8) + 15) / 16 * 16 : 0);
}

ecc_status bf16_exponent_histogram(const uint16_t *in, size_t n, uint64_t *count, void *stream)
{
    if (!count || (n && !in) || (n && ((uintptr_t)in & 15)))
        return ECC_ERR_ARG;
    if (!n)
        return ECC_OK;
    const int sms = sm_count();
    if (sms <= 0)
        return ECC_ERR_CUDA;
    const uint64_t blocks = std::max<uint64_t>(1, std::min<uint64_t>((n / 8 + kBfThreads - 1) / kBfThreads,
                                                                      (uint64_t)sms * 4));
    bf16_hist_kernel<<<(unsigned)blocks, kBfThreads, 0, (cudaStream_t)stream>>>(in, n, (unsigned long long *)count);
    return launch_status(cudaGetLastError());
}

ecc_status bf16_escape_encode(const uint16_t *in, size_t n, const uint8_t top7[7], uint32_t C, uint32_t S,
                              uint8_t *out, size_t out_cap, uint64_t *chunk_off, uint16_t *sub_bits,
                              uint64_t *total_bits, void *ws, size_t ws_bytes, uint32_t *status, void *stream)
{
    if (!top7 || !bf_table_ok(top7) || !chunk_off || !total_bits || !status || !ws || !valid_sizes(C, S) ||
        C > kBfMaxC)
        return ECC_ERR_ARG;
    if (n && (!in || !out || !sub_bits || !aligned16(in) || !aligned16(out)))
        return ECC_ERR_ARG;
    if (!aligned16(ws) || ws_bytes < ecc_encode_workspace_bytes(n, C))
        return ECC_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const uint64_t n_chunks = ecc_num_chunks(n, C);
    uint32_t *ticket = (uint32_t *)ws;
    uint64_t *flags = (uint64_t *)((uint8_t *)ws + 256);
    // the ticket, the look-back words and the outputs the kernel adds to
    if (cudaMemsetAsync(ws, 0, 256 + n_chunks * sizeof(uint64_t), st) != cudaSuccess ||
        cudaMemsetAsync(total_bits, 0, sizeof(uint64_t), st) != cudaSuccess ||
        cudaMemsetAsync(chunk_off, 0, sizeof(uint64_t), st) != cudaSuccess ||
        cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess)
        return launch_status(cudaErrorUnknown);
    if (!n)
        return ECC_OK;
    BfEncParams p;
    p.in = in;
    p.n = n;
    for (int r = 0; r < 7; ++r)
        p.tab.top[r] = top7[r];
    p.tab.top[7] = 0;
    p.C = C;
    p.S = S;
    p.out = out;
    p.out_cap = out_cap;
    p.chunk_off = chunk_off;
    p.sub_bits = sub_bits;
    p.total_bits = total_bits;
    p.flags = flags;
    p.ticket = ticket;
    p.status = status;
    p.n_chunks = n_chunks;
    p.stage_bytes = pad16((C * 19u + 7u) / 8u) + 16u; // C values at 19 bits
    p.timeout_ns = kWaitLimitNs;
    const int sms = sm_count();
    if (sms <= 0)
        return ECC_ERR_CUDA;
    if (C <= kBfWarpC) { // a warp a chunk, persistent
        const size_t smem = (size_t)(kBfWarpThreads / 32) * p.stage_bytes;
        const int occ = occupancy((const void *)bf16_encode_warp_kernel, kBfWarpThreads, smem);
        if (occ <= 0)
            return ECC_ERR_CUDA;
        const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, (n_chunks + kBfWarpThreads / 32 - 1) /
                                                                          (kBfWarpThreads / 32));
        bf16_encode_warp_kernel<<<(unsigned)grid, kBfWarpThreads, smem, st>>>(p);
        return launch_status(cudaGetLastError());
    }
    const int occ = occupancy((const void *)bf16_encode_kernel, kBfThreads, p.stage_bytes);
    if (occ <= 0)
        return ECC_ERR_CUDA;
    const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, n_chunks);
    bf16_encode_kernel<<<(unsigned)grid, kBfThreads, p.stage_bytes, st>>>(p);
    return launch_status(cudaGetLastError());
}

ecc_status bf16_escape_decode(const uint8_t *in, size_t in_bytes, const uint64_t *chunk_off,
                              const uint16_t *sub_bits, size_t n, uint32_t C, uint32_t S, const uint8_t top7[7],
                              uint16_t *out, uint32_t *status, void *stream)
{
    if (!top7 || !bf_table_ok(top7) || !status || !chunk_off || !valid_sizes(C, S) || C > kBfMaxC)
        return ECC_ERR_ARG;
    if (n && (!in || !out || !sub_bits || !aligned16(in) || !aligned16(out)))
        return ECC_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess)
        return launch_status(cudaErrorUnknown);
    if (!n)
        return ECC_OK;
    BfDecParams p;
    p.in = in;
    p.in_bytes = in_bytes;
    p.chunk_off = chunk_off;
    p.sub_bits = sub_bits;
    p.n = n;
    p.C = C;
    p.S = S;
    for (int r = 0; r < 7; ++r)
        p.tab.top[r] = top7[r];
    p.tab.top[7] = 0;
    p.out = out;
    p.status = status;
    p.n_chunks = ecc_num_chunks(n, C);
    const int sms = sm_count();
    if (sms <= 0)
        return ECC_ERR_CUDA;
    const uint64_t grid = std::max<uint64_t>(1, std::min<uint64_t>((p.n_chunks + 7) / 8, (uint64_t)sms * 8));
    bf16_decode_kernel<<<(unsigned)grid, 256, 0, st>>>(p);
    return launch_status(cudaGetLastError());
}

} // extern "C"
