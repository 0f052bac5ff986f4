// ecc_device.cuh -- device building blocks of the e4m3 entropy coder for
// sm_103a: the chunk encoder (LUT lookup, scans of code lengths, decoupled
// look-back for chunk offsets, bit packing) and the warp-per-chunk decoder
// (first-level peek table, canonical long-code ranges).  Included by the
// single-tensor and the batched translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ecc.h"

namespace ecc {

// ---------------------------------------------------------------- constants
constexpr int kEncThreads = 256;
constexpr int kEncWarps = kEncThreads / 32;
constexpr int kSymPerThread = 16;                     // one 16-byte load
constexpr int kTile = kEncThreads * kSymPerThread;    // symbols per tile
constexpr uint32_t kLutRows = 256;                    // byte values
constexpr uint64_t kFlagAggregate = 1ull << 62;       // look-back states
constexpr uint64_t kFlagPrefix = 2ull << 62;
constexpr uint64_t kFlagDeferred = 1ull << 61;        // with kFlagPrefix: the deferred pass codes the unit's payload
constexpr uint64_t kValueMask = (1ull << 61) - 1;
constexpr uint64_t kWaitLimitNs = 1000000000ull;      // bounded waits: 1 s

__host__ __device__ constexpr uint32_t pad16(uint32_t b) { return (b + 15u) & ~15u; }

// Zeroed bytes after a staged chunk: the decoder reads ahead into them.
constexpr uint32_t kStageGuard = 96;

// Worst-case staging bytes for one chunk of C symbols at up to 11 bits
// (every QLC code fits; longer Huffman chunks take the unstaged path), with
// a zeroed guard so peeks past a payload's end read zeros.
__host__ __device__ constexpr uint32_t stage_bytes_for(uint32_t C) { return pad16((C * 11u + 7u) / 8u) + kStageGuard; }

// Decoder stage of one warp: a chunk at up to 9.25 bits a symbol (larger
// chunks are staged 32 sub-blocks at a time), and never less than 32
// sub-blocks at 11 bits; when a chunk has fewer than 32 sub-blocks, the whole
// chunk at 11 bits.
__host__ __device__ constexpr uint32_t dec_stage_bytes(uint32_t C, uint32_t S)
{
    return C / S < 32 ? stage_bytes_for(C)
                      : (pad16((C * 37u + 31u) / 32u) > pad16((32u * S * 11u + 7u) / 8u) + 16u
                             ? pad16((C * 37u + 31u) / 32u)
                             : pad16((32u * S * 11u + 7u) / 8u) + 16u) +
                            kStageGuard;
}

// ---------------------------------------------------------------- memory ops
__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t *p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream16(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t bswap32(uint32_t x) { return __byte_perm(x, 0, 0x0123); }
__device__ __forceinline__ uint4 bswap4(uint4 v) { return make_uint4(bswap32(v.x), bswap32(v.y), bswap32(v.z), bswap32(v.w)); }

// ---------------------------------------------------------------- bulk copies
// One-instruction global -> shared copies through the bulk-copy (TMA) engine,
// completion tracked by an mbarrier transaction count.  Sizes are multiples
// of 16 bytes, addresses 16-byte aligned.
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// order this thread's earlier generic accesses to shared memory before later
// bulk-copy writes to it
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false if limit_ns
// passed first (the copy is then still in flight: wait again before the
// buffer is reused or the CTA exits).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (globaltimer() - t0 > limit_ns)
            return false;
    }
}

// byte k (0..3) of x, zero-extended
__device__ __forceinline__ uint32_t byte_of(uint32_t x, int k) { return __byte_perm(x, 0, 0x4440 | k); }

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t code)
{
    if (status)
        atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------- look-back
// Decoupled look-back over chunk offsets, run by one full warp.  flags[c]
// holds (state << 62) | value: state 1 = chunk aggregate published, 2 =
// inclusive prefix published.  Returns the exclusive prefix of chunk c and
// publishes c's inclusive prefix.  Every wait is bounded: past timeout_ns the
// warp reports ECC_ERR_TIMEOUT through *timed_out, still publishes (so that
// successors finish), and the caller writes nothing for the chunk.
__device__ __forceinline__ uint64_t lookback(uint64_t *flags, uint64_t c, uint64_t aggregate, uint64_t timeout_ns,
                                             bool *timed_out)
{
    const int lane = threadIdx.x & 31;
    *timed_out = false;
    if (c == 0) {
        if (lane == 0)
            st_relaxed(flags, kFlagPrefix | (aggregate & kValueMask));
        return 0;
    }
    if (lane == 0)
        st_relaxed(flags + c, kFlagAggregate | (aggregate & kValueMask));
    uint64_t prefix = 0;
    int64_t j = (int64_t)c - 1;
    uint64_t t0 = 0;
    bool expired = false;
    for (;;) {
        const int64_t idx = j - lane;
        const uint64_t f = idx >= 0 ? ld_relaxed(flags + idx) : kFlagPrefix;
        const uint32_t state = (uint32_t)(f >> 62);
        const unsigned pmask = __ballot_sync(~0u, state == 2);
        const unsigned zmask = __ballot_sync(~0u, state == 0);
        const int fp = pmask ? __ffs(pmask) - 1 : 32;          // nearest prefix
        const unsigned need = fp >= 31 ? ~0u : ((2u << fp) - 1u); // lanes 0..fp
        if (zmask & need) {
            const uint64_t now = globaltimer();
            if (t0 == 0)
                t0 = now;
            if (__any_sync(~0u, now - t0 > timeout_ns)) {
                expired = true;
                break;
            }
            __nanosleep(64);
            continue;
        }
        uint64_t v = lane <= fp ? (f & kValueMask) : 0;
#pragma unroll
        for (int o = 16; o; o >>= 1)
            v += __shfl_xor_sync(~0u, v, o);
        prefix += v;
        if (fp < 32)
            break;
        j -= 32;
    }
    if (lane == 0)
        st_relaxed(flags + c, kFlagPrefix | ((prefix + aggregate) & kValueMask));
    *timed_out = expired;
    return prefix;
}

// Resolve the exclusive prefix of chunk c (c > 0) whose aggregate was
// already published, then publish its inclusive prefix.  One full warp.
__device__ __forceinline__ uint64_t resolve_prefix(uint64_t *flags, uint64_t c, uint64_t aggregate,
                                                   uint64_t timeout_ns, bool *timed_out)
{
    const int lane = threadIdx.x & 31;
    uint64_t prefix = 0;
    int64_t j = (int64_t)c - 1;
    uint64_t t0 = 0;
    bool expired = false;
    for (;;) {
        const int64_t idx = j - lane;
        const uint64_t f = idx >= 0 ? ld_relaxed(flags + idx) : kFlagPrefix;
        const uint32_t state = (uint32_t)(f >> 62);
        const unsigned pmask = __ballot_sync(~0u, state == 2);
        const unsigned zmask = __ballot_sync(~0u, state == 0);
        const int fp = pmask ? __ffs(pmask) - 1 : 32;
        const unsigned need = fp >= 31 ? ~0u : ((2u << fp) - 1u);
        if (zmask & need) {
            const uint64_t now = globaltimer();
            if (t0 == 0)
                t0 = now;
            if (__any_sync(~0u, now - t0 > timeout_ns)) {
                expired = true;
                break;
            }
            __nanosleep(32);
            continue;
        }
        uint64_t v = lane <= fp ? (f & kValueMask) : 0;
#pragma unroll
        for (int o = 16; o; o >>= 1)
            v += __shfl_xor_sync(~0u, v, o);
        prefix += v;
        if (fp < 32)
            break;
        j -= 32;
    }
    if (lane == 0)
        st_relaxed(flags + c, kFlagPrefix | ((prefix + aggregate) & kValueMask));
    *timed_out = expired;
    return prefix;
}

// ---------------------------------------------------------------- named barriers
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t n)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// barrier over n threads that also returns the AND of p over them
__device__ __forceinline__ bool bar_red_and(uint32_t id, uint32_t n, bool p)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\tbar.red.and.pred b, %2, %3, a;\n\t"
                 "selp.u32 %0, 1, 0, b;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)p), "r"(id), "r"(n)
                 : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- encoder
struct EncJob {
    const uint8_t *in;
    uint64_t n;
    const ecc_codebook *cb;
    uint32_t C, S;
    uint8_t *out;
    uint64_t out_cap;
    uint64_t *chunk_off;
    uint16_t *sub_bits;
    uint64_t *total_bits;
    uint64_t *flags;
    uint32_t *status;
};

// One chunk claimed by the warp-specialised encoder.
struct EncSlot {
    EncJob job;       // many-tensor kernel: the chunk's tensor (flags already offset to it)
    uint64_t c;       // chunk index within its tensor
    uint64_t *t_done; // many-tensor kernel: the tensor's completion stamp (may be null)
    uint32_t tensor;  // many-tensor kernel: tensor index (completion counters)
    uint32_t state;   // kSlotEnd: no more work; kSlotChunk; kSlotBadCodebook
    uint32_t staged;  // its input was bulk-copied into input buffer k % 2
    uint32_t parity;  // phase parity of that copy on the buffer's mbarrier
};
constexpr uint32_t kSlotEnd = 0, kSlotChunk = 1, kSlotBadCodebook = 2;
constexpr uint32_t kEncSlots = 4; // claimed two chunks ahead: slots k .. k + 2 live at once

// Shared state of one encoder CTA.  lut holds 16 replicas of the 256 encode
// entries {code << (32 - len), 2^(32 - len)}: entry s for lane l is
// lut[s * 16 + (l & 15)].  A warp's 64-bit loads are served half a warp at a
// time, and the 16 lanes of each half read 16 different bank pairs whatever
// bytes they look up.
constexpr uint32_t kLutReplicas = 16;
// The warp-segmented encoder takes chunks smaller than kGroupSyms symbols in
// groups of consecutive chunks and codes and places a group as one unit of
// kEncWarps segments (one a compute warp): at most kMaxGroup chunks.
constexpr uint32_t kGroupSyms = 16384;
constexpr uint32_t kMaxGroup = kEncWarps;
struct EncShared {
    uint2 lut[kLutRows * kLutReplicas];
    alignas(16) uint32_t warp_tot[2][kEncWarps]; // per tile parity: one barrier per tile suffices
    uint64_t prefix;
    uint64_t bar[2];            // input-buffer mbarriers
    uint32_t slot_bits[2];      // warp-specialised encoder: payload bits of the chunk in each stage slot
    uint32_t slot_flags[2];     // bit 0: staging overflow
    uint32_t issued[2];         // bulk copies issued into each input buffer
    uint32_t nostage;           // set once a copy timed out: issue no more copies
    const ecc_codebook *loaded; // codebook currently in lut
    uint32_t ticket;
    uint32_t flags; // bit 0: staging overflow, bit 1: skip the write
    EncSlot slot[kEncSlots];
    // warp-segmented encoder: each warp's segment of unit k, its payload
    // bits and the first word of its region, in entry k % 4 (two units are
    // in flight, and a warp may code the next one while another still
    // copies the one before)
    uint32_t seg_bits[4][kEncWarps];
    uint32_t seg_first[4][kEncWarps];
    uint64_t out_prefix[2];          // byte offset of the slot's chunk or group in the output (resolved look-back)
    uint32_t out_copy[2];            // 1: the compute warps copy the slot out to the output
    uint32_t chunk_rel[2][kMaxGroup + 1]; // byte offsets of a group's chunks in its output (last: the group's bytes)
};

__host__ __device__ constexpr uint32_t enc_shared_bytes() { return (sizeof(EncShared) + 15u) & ~15u; }

// Fill the shared encode table from the codebook; threads [0, nthreads).
__device__ __forceinline__ void load_encode_lut(EncShared &sh, const ecc_codebook *cb, uint32_t nthreads)
{
    const uint32_t tid = threadIdx.x;
    if (tid >= nthreads)
        return;
    for (uint32_t i = tid; i < kLutRows * kLutReplicas; i += nthreads) {
        const uint32_t s = i / kLutReplicas;
        sh.lut[i] = make_uint2(cb->enc_code[s], cb->enc_mul[s]);
    }
}

// Load up to 16 input bytes: a full group from the chunk source (shared
// stage or global memory, 16-byte aligned), a partial one (the tensor's last
// bytes) from global memory.
template <bool kSharedSrc>
__device__ __forceinline__ uint4 load_symbols(const uint8_t *chunk_src, const uint8_t *global_src, uint32_t cnt)
{
    if (cnt == kSymPerThread) {
        if (kSharedSrc)
            return *reinterpret_cast<const uint4 *>(chunk_src);
        return ld_stream16(global_src);
    }
    const uint8_t *src = global_src;
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < kSymPerThread; ++i)
        if ((uint32_t)i < cnt)
            w[i >> 2] |= (uint32_t)src[i] << (8 * (i & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// x << n with n >= 32 giving 0 (PTX shift semantics)
__device__ __forceinline__ uint32_t shl_clamp(uint32_t x, uint32_t n)
{
    uint32_t r;
    asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(n));
    return r;
}

// hi32(a * b) + c
__device__ __forceinline__ uint32_t mad_hi(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// ---- fast path: codes as multiplications
// A code of length l is held as v = code << (32 - l) (first bit in bit 31)
// with the multiplier q = 2^(32 - l).  Appending code 2 behind code 1 is
// v1 + hi32(v2 * q1), and the pair's multiplier is hi32(q1 * q2) =
// 2^(32 - l1 - l2), which is 0 exactly when the pair is longer than 32 bits
// (or when either entry is 0, a byte the fast path does not code).

// Encode entries of the 16 symbols in `in`, joined in 8 consecutive pairs
// (v[k], q[k]).  Returns the bit total; *slow when the group is partial or
// some pair has q == 0 (the exact path must code the group).
__device__ __forceinline__ uint32_t lookup_pairs(const uint2 *lut, uint4 in, uint32_t cnt, uint32_t v[8],
                                                 uint32_t q[8], bool *slow)
{
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t zsum = 0, zor = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint2 e1 = lut[byte_of(w[k >> 1], (2 * k) & 3) * kLutReplicas];
        const uint2 e2 = lut[byte_of(w[k >> 1], (2 * k + 1) & 3) * kLutReplicas];
        v[k] = mad_hi(e2.x, e1.y, e1.x);
        q[k] = __umulhi(e1.y, e2.y);
        const uint32_t z = __clz(q[k]); // pair length - 1 (32: no fast code)
        zsum += z;
        zor |= z;
    }
    *slow = cnt < kSymPerThread || (zor & 32u);
    return zsum + 8;
}

// Bit total of the 16 symbols in `in` coded one by one from the table (a
// group whose pairs do not all fit 32 bits); *exact when some byte has no
// code of at most 31 bits (multiplier 0), which only the exact path codes.
__device__ __forceinline__ uint32_t single_bits(const uint2 *lut, uint4 in, bool *exact)
{
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t zsum = 0, zor = 0;
#pragma unroll
    for (int j = 0; j < kSymPerThread; ++j) {
        const uint32_t z = __clz(lut[byte_of(w[j >> 2], j & 3) * kLutReplicas].y); // length - 1
        zsum += z;
        zor |= z;
    }
    *exact = (zor & 32u) != 0;
    return zsum + kSymPerThread;
}

// Predicated or-reduction into a shared word (addr: shared-window address):
// done when `gate` is 0.  Written as one predicated instruction so that no
// branch surrounds it.
__device__ __forceinline__ void red_or_shared_if_zero(uint32_t addr, uint32_t v, uint32_t gate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %2, 0;\n\t@p red.shared.or.b32 [%0], %1;\n\t}" ::"r"(addr),
                 "r"(v), "r"(gate)
                 : "memory");
}

__device__ __forceinline__ void red_or_shared(uint32_t addr, uint32_t v)
{
    asm volatile("red.shared.or.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// predicated 32-bit shared store (addr: shared-window address)
__device__ __forceinline__ void st_shared_if(uint32_t addr, uint32_t v, bool p)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.shared.b32 [%0], %1;\n\t}" ::"r"(addr),
                 "r"(v), "r"((uint32_t)p)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4_zero(uint32_t addr)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Bit sink of the fast path, a shared stage of 32-bit words in register
// order (bit 31 of a word is its first bit; whoever copies the stage out
// swaps the bytes).  The partial word cur (its first nb bits used,
// 1 <= nb <= 32, first bit in bit 31) belongs at shared address a, and
// K = 2^(32 - nb).  Appending (v, q) of length l: v * K + (cur << 32) holds
// in its high word cur with v's leading bits behind it and in its low word
// v's remaining bits; K * q = 2^(64 - nb - l) says whether the word filled
// up (high word 0) and gives the next K (whichever word is non-zero).
// Completed words are or-ed into the zeroed stage, which also merges the
// first and last words a thread shares with its neighbours.  A start at a
// word boundary begins as a full, empty word just before it (for bit 0 of
// the stage: a zero guard word in front of it, only ever or-ed with 0).
struct MulPacker {
    uint32_t a;
    uint32_t cur, K;

    __device__ __forceinline__ void start(uint32_t sink_addr, uint32_t bitpos)
    {
        const uint32_t pm1 = bitpos - 1u;
        a = sink_addr + (uint32_t)(((int32_t)pm1 >> 5) * 4);
        K = 1u << (31u - (pm1 & 31u));
        cur = 0;
    }
    __device__ __forceinline__ void put(uint32_t v, uint32_t q)
    {
        const uint64_t x = (uint64_t)v * K + ((uint64_t)cur << 32);
        const uint64_t y = (uint64_t)K * q;
        const uint32_t xhi = (uint32_t)(x >> 32), xlo = (uint32_t)x;
        const uint32_t yhi = (uint32_t)(y >> 32), ylo = (uint32_t)y;
        red_or_shared_if_zero(a, xhi, yhi);
        const bool full = yhi == 0;
        cur = full ? xlo : xhi;
        a += full ? 4u : 0u;
        K = yhi + ylo;
    }
    __device__ __forceinline__ void finish() { red_or_shared(a, cur); }
};

// ---- exact path: any code length up to ECC_MAX_CODE_LEN, codes read from
// the codebook (global memory).  Packing sink: 32-bit words, in memory byte
// order when kSwap (a final destination), else in register order (a shared
// stage, swapped when copied out); a thread's first and last words are
// merged with atomicOr into a zeroed destination, every word in between
// belongs to this thread alone and is stored once.  The accumulator is kept
// as two 32-bit halves shifted with funnel shifts.
template <bool kSwap>
struct Packer {
    uint32_t *dst;
    uint32_t wi0, wi; // first word, word being filled
    uint32_t nb;      // pending bits in (ahi:alo), right-aligned, < 32 between appends
    uint32_t ahi, alo;
    uint32_t fw;      // the first word, once completed

    __device__ __forceinline__ void start(uint32_t *d, uint32_t bitpos)
    {
        dst = d;
        wi0 = wi = bitpos >> 5;
        nb = bitpos & 31; // the predecessor's bits count as zeros here
        ahi = alo = 0;
        fw = 0;
    }
    // append up to 32 bits (len <= 32)
    __device__ __forceinline__ void put(uint32_t code, uint32_t len)
    {
        ahi = __funnelshift_lc(alo, ahi, len);
        alo = shl_clamp(alo, len) | code;
        nb += len;
        const bool full = nb >= 32;
        nb &= 31;
        const uint32_t w0 = __funnelshift_r(alo, ahi, nb);
        const uint32_t w = kSwap ? bswap32(w0) : w0;
        const bool first = wi == wi0;
        if (full && !first)
            dst[wi] = w;
        fw = (full && first) ? w : fw;
        wi += full ? 1u : 0u;
    }
    // append up to 48 bits
    __device__ __forceinline__ void put_long(uint64_t code, uint32_t len)
    {
        if (len > 24) {
            put((uint32_t)(code >> 24), len - 24);
            put((uint32_t)(code & 0xFFFFFFu), 24);
        } else {
            put((uint32_t)code, len);
        }
    }
    __device__ __forceinline__ void finish()
    {
        if (wi != wi0)
            atomicOr(dst + wi0, fw);
        if (nb)
            atomicOr(dst + wi, kSwap ? bswap32(shl_clamp(alo, 32 - nb)) : shl_clamp(alo, 32 - nb));
    }
};

// Exact bit total of the cnt symbols in `in`; *bad if some byte has no code.
__device__ __forceinline__ uint32_t exact_bits(uint4 in, uint32_t cnt, const ecc_codebook *cb, bool *bad)
{
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t bits = 0;
    bool nocode = false;
#pragma unroll
    for (int j = 0; j < kSymPerThread; ++j) {
        if ((uint32_t)j >= cnt)
            continue;
        const uint32_t L = min((uint32_t)cb->len[byte_of(w[j >> 2], j & 3)], (uint32_t)ECC_MAX_CODE_LEN);
        nocode |= L == 0;
        bits += L;
    }
    *bad = nocode;
    return bits;
}

// Exact packing of the cnt symbols in `in` at bit `pos` of dst.
template <bool kSwap>
__device__ __forceinline__ void exact_pack(uint32_t *dst, uint32_t pos, uint4 in, uint32_t cnt,
                                           const ecc_codebook *cb)
{
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    Packer<kSwap> pk;
    pk.start(dst, pos);
#pragma unroll 1
    for (int j = 0; j < kSymPerThread; ++j) {
        if ((uint32_t)j >= cnt)
            break;
        const uint32_t b = byte_of(w[j >> 2], j & 3);
        const uint32_t L = min((uint32_t)cb->len[b], (uint32_t)ECC_MAX_CODE_LEN);
        if (L)
            pk.put_long(cb->code[b] & ((1ull << L) - 1), L);
    }
    pk.finish();
}

constexpr uint32_t kBarCompute = 1;   // the encoder's compute warps
constexpr uint32_t kBarFull = 2;      // + slot: stage slot filled (compute -> output warp)
constexpr int kEncThreadsWS = kEncThreads + 32;

__device__ __forceinline__ void compute_barrier(bool named)
{
    if (named)
        bar_sync(kBarCompute, kEncThreads);
    else
        __syncthreads();
}

// Bytes in front of each stage slot: a zero guard word the multiplying
// packer may or 0 into when a thread starts at bit 0 of the slot.
constexpr uint32_t kStageLead = 16;

// Encode one tile (kTile symbols from t0) of a chunk of L symbols at bit
// `run` of sink; returns the tile's bits.  kFast: full groups are coded with
// the shared table and the multiplying packer (the sink is a shared stage
// slot with its guard word in front); otherwise every group takes the exact
// path (any sink).  kCheckRoom: a group that would pass sink_bits is not
// written and raises bit 0 of *flag_word (or sh.flags).
template <bool kCheckRoom, bool kSharedSrc, bool kNamed = false, bool kFast = true>
__device__ __forceinline__ uint32_t encode_tile(EncShared &sh, const EncJob &job, const uint8_t *src, uint64_t base,
                                                uint32_t L, uint32_t t0, uint32_t run, uint32_t *sink,
                                                uint32_t sink_bits, bool write_sub, bool *bad_out,
                                                uint32_t *flag_word = nullptr)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t parity = (t0 / kTile) & 1;
    const uint32_t my0 = t0 + (uint32_t)tid * kSymPerThread;
    const uint32_t cnt = my0 < L ? min((uint32_t)kSymPerThread, L - my0) : 0u;
    const uint4 v = cnt ? load_symbols<kSharedSrc>(src + my0, job.in + base + my0, cnt) : make_uint4(0, 0, 0, 0);
    uint32_t pv[8], pq[8];
    bool slow = true, bad = false;
    uint32_t bits = 0;
    if (kFast)
        bits = lookup_pairs(sh.lut + (lane & (kLutReplicas - 1)), v, cnt, pv, pq, &slow);
    if (slow) // rare: a partial group or a code the fast path leaves out
        bits = exact_bits(v, cnt, job.cb, &bad);
    *bad_out |= bad;

    uint32_t incl = bits;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(~0u, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        sh.warp_tot[parity][warp] = incl;
    compute_barrier(kNamed);
    uint32_t before = 0, tile_total = 0;
    {
        const uint4 w03 = *reinterpret_cast<const uint4 *>(&sh.warp_tot[parity][0]);
        const uint4 w47 = *reinterpret_cast<const uint4 *>(&sh.warp_tot[parity][4]);
        const uint32_t t[8] = {w03.x, w03.y, w03.z, w03.w, w47.x, w47.y, w47.z, w47.w};
#pragma unroll
        for (int w = 0; w < kEncWarps; ++w) {
            before += w < warp ? t[w] : 0u;
            tile_total += t[w];
        }
    }
    const uint32_t excl = before + incl - bits;
    if (write_sub) {
        // bits of each sub-block of S symbols = S/16 consecutive threads
        const uint32_t tps = job.S / kSymPerThread; // a power of two, 4..64
        uint32_t sb;
        if (tps <= 32) {
            sb = __shfl_sync(~0u, incl, lane | (int)(tps - 1)) - (incl - bits);
        } else { // S = 1024: two whole warps
            sb = sh.warp_tot[parity][warp] + sh.warp_tot[parity][warp | 1];
        }
        if (cnt && ((uint32_t)tid & (tps - 1)) == 0)
            job.sub_bits[(base + my0) >> (31 - __clz(job.S))] = (uint16_t)sb;
    }
    const uint32_t pos = run + excl;
    if (cnt) {
        if (!kCheckRoom || pos + bits <= sink_bits) {
            if (!slow) {
                MulPacker pk;
                pk.start(smem_u32(sink), pos);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    pk.put(pv[k], pq[k]);
                pk.finish();
            } else {
                exact_pack<!kFast>(sink, pos, v, cnt, job.cb);
            }
        } else {
            atomicOr(flag_word ? flag_word : &sh.flags, 1u);
        }
    }
    return tile_total;
}

// Encode chunk c of job into its place in job.out.  src holds the chunk's
// input (its whole 16-byte groups) in shared memory when kSharedSrc, else
// src is unused and the input is read from global memory.  `stage` is a
// zeroed shared-memory buffer of stage_bytes; it is zeroed again on return.
template <bool kSharedSrc>
__device__ __forceinline__ void encode_chunk(EncShared &sh, uint32_t *stage, uint32_t stage_bytes, const EncJob &job,
                                             const uint8_t *src, uint64_t c, uint64_t timeout_ns)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t base = c * job.C;
    const uint32_t L = (uint32_t)min((uint64_t)job.C, job.n - base);
    if (tid == 0)
        sh.flags = 0;
    __syncthreads();

    bool bad = false;
    uint32_t run = 0;
    for (uint32_t t0 = 0; t0 < L; t0 += kTile)
        run += encode_tile<true, kSharedSrc>(sh, job, src, base, L, t0, run, stage, stage_bytes * 8u, true, &bad);
    if (bad)
        set_status(job.status, ECC_ERR_CODEBOOK);

    const uint64_t bytes = ((uint64_t)run + 127u) / 128u * 16u;
    if (warp == 0) {
        bool to;
        const uint64_t prefix = lookback(job.flags, c, bytes, timeout_ns, &to);
        if (lane == 0) {
            sh.prefix = prefix;
            if (to) {
                atomicOr(&sh.flags, 2u);
                set_status(job.status, ECC_ERR_TIMEOUT);
            }
            job.chunk_off[c + 1] = prefix + bytes;
            if (c == 0)
                job.chunk_off[0] = 0;
            atomicAdd((unsigned long long *)job.total_bits, (unsigned long long)run);
        }
    }
    __syncthreads();
    const uint64_t prefix = sh.prefix;
    const uint32_t fl = sh.flags;
    uint4 *st4 = reinterpret_cast<uint4 *>(stage);
    const uint32_t nvec = (uint32_t)(bytes / 16);
    const bool fits = prefix + bytes <= job.out_cap;
    if (!fits && !(fl & 2u) && tid == 0)
        set_status(job.status, ECC_ERR_CAPACITY);
    if (!(fl & 1u)) {
        uint4 *dst = reinterpret_cast<uint4 *>(job.out + prefix);
        const bool write = fits && !(fl & 2u);
        for (uint32_t i = tid; i < nvec; i += kEncThreads) {
            const uint4 w = st4[i];
            st4[i] = make_uint4(0, 0, 0, 0);
            if (write)
                st_stream16(dst + i, bswap4(w));
        }
    } else {
        // the payload outgrew the staging buffer: re-encode straight into
        // global memory (zeroed first), then clear the whole stage
        for (uint32_t i = tid; i < stage_bytes / 16; i += kEncThreads)
            st4[i] = make_uint4(0, 0, 0, 0);
        if (fits && !(fl & 2u)) {
            uint4 *dst = reinterpret_cast<uint4 *>(job.out + prefix);
            for (uint32_t i = tid; i < nvec; i += kEncThreads)
                dst[i] = make_uint4(0, 0, 0, 0);
            __syncthreads();
            bool bad2 = false;
            uint32_t run2 = 0;
            uint32_t *gsink = reinterpret_cast<uint32_t *>(job.out + prefix);
            for (uint32_t t0 = 0; t0 < L; t0 += kTile)
                run2 += encode_tile<false, kSharedSrc, false, false>(sh, job, src, base, L, t0, run2, gsink, 0, false,
                                                                     &bad2);
        }
    }
    __syncthreads();
}

// Re-encode chunk c with one warp straight into global memory at dst (the
// chunk's place in the output, `words` 32-bit words, zeroed here first):
// the path for chunks whose payload outgrew the shared staging buffer.
// Codes come from the codebook in global memory (the exact path), never
// from the shared table, which the compute warps may be reloading.
static __device__ __noinline__ void encode_chunk_warp(const EncJob &job, uint64_t c, uint32_t *dst, uint32_t words)
{
    const int lane = threadIdx.x & 31;
    for (uint32_t i = lane; i < words; i += 32)
        dst[i] = 0;
    __syncwarp();
    const uint64_t base = c * job.C;
    const uint32_t L = (uint32_t)min((uint64_t)job.C, job.n - base);
    uint32_t run = 0;
    for (uint32_t t0 = 0; t0 < L; t0 += 32 * kSymPerThread) {
        const uint32_t my0 = t0 + (uint32_t)lane * kSymPerThread;
        const uint32_t cnt = my0 < L ? min((uint32_t)kSymPerThread, L - my0) : 0u;
        const uint4 v = cnt ? load_symbols<false>(nullptr, job.in + base + my0, cnt) : make_uint4(0, 0, 0, 0);
        bool bad;
        const uint32_t bits = exact_bits(v, cnt, job.cb, &bad);
        if (bad)
            set_status(job.status, ECC_ERR_CODEBOOK);
        uint32_t incl = bits;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(~0u, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (cnt)
            exact_pack<true>(dst, run + incl - bits, v, cnt, job.cb);
        run += __shfl_sync(~0u, incl, 31);
    }
}

// The deferred pass: units an encoder could not stage (long codes) were
// sized, their offsets resolved and their flag word marked kFlagPrefix |
// kFlagDeferred; here one warp codes each chunk of such a unit straight into
// the output at chunk_off (the encoder checked the capacity before marking).
// Unit u holds chunks [u * G, u * G + G).  Returns the chunks it coded.
__device__ __forceinline__ uint32_t code_deferred_unit(const EncJob &job, uint64_t u, uint32_t G, uint64_t n_chunks)
{
    uint32_t k = 0;
    for (uint64_t c = u * G; c < n_chunks && c < (u + 1) * G; ++c, ++k) {
        const uint64_t o0 = job.chunk_off[c], o1 = job.chunk_off[c + 1];
        if (o0 > o1 || o1 > job.out_cap) // offsets not published (an error status is set)
            continue;
        encode_chunk_warp(job, c, reinterpret_cast<uint32_t *>(job.out + o0), (uint32_t)((o1 - o0) / 4u));
    }
    return k;
}

__device__ __forceinline__ bool is_deferred(uint64_t f)
{
    return (f & (3ull << 62)) == kFlagPrefix && (f & kFlagDeferred);
}

// Bulk-copy the whole 16-byte groups of the input of chunks c .. c + g - 1
// into buf (thread 0); completion arrives on bar.  The last chunk's trailing
// bytes (fewer than 16) are read from global memory by the thread that owns
// them.
__device__ __forceinline__ void issue_chunk_input(const EncJob &job, uint64_t c, uint8_t *buf, uint64_t *bar,
                                                  uint32_t g = 1)
{
    const uint64_t base = c * job.C;
    const uint32_t L = (uint32_t)min((uint64_t)job.C * g, job.n - base);
    const uint32_t whole = L & ~15u;
    fence_proxy_async();
    mbar_expect_tx(bar, whole);
    if (whole)
        bulk_g2s(buf, job.in + base, whole, bar);
}

// ---------------------------------------------------------------- warp-segmented encoder
// Each compute warp codes one contiguous segment of a chunk into a region of
// its own in a shared stage slot, in rounds of 32 lanes x 16 symbols: a warp
// scan of the lanes' bit counts places every lane, so no CTA-wide barrier
// is needed until the chunk ends.  A segment is at least 512 symbols (one
// full round) and at least one sub-block, so sub-blocks never straddle
// warps.  Regions hold 32-bit words in register order (bit 31 first).  Once
// the chunk's offset in the output is known each compute warp copies its
// region out, shifted to where its segment starts in the chunk's bitstream
// (the stream is the segments' bits end to end).

constexpr uint32_t kRoundSyms = 32 * kSymPerThread; // 512

__host__ __device__ constexpr uint32_t seg_symbols(uint32_t C, uint32_t S)
{
    return (C / kEncWarps > S ? C / kEncWarps : S) > kRoundSyms ? (C / kEncWarps > S ? C / kEncWarps : S)
                                                                  : kRoundSyms;
}
// a region: room for the segment at up to 11 bits a symbol, plus one zero
// word of slack that the out-copy may read past the payload
__host__ __device__ constexpr uint32_t region_cap_bytes(uint32_t seg) { return pad16((seg * 11u + 7u) / 8u); }
__host__ __device__ constexpr uint32_t region_bytes(uint32_t seg) { return region_cap_bytes(seg) + 16u; }
__host__ __device__ constexpr uint32_t enc_ws_slot_bytes(uint32_t C, uint32_t S)
{
    return (C / seg_symbols(C, S)) * region_bytes(seg_symbols(C, S));
}
// Segments of chunks coded in groups (chunks of fewer than kGroupSyms
// symbols): kGroupSyms / kEncWarps symbols, or the whole chunk when it is
// smaller (and at least one sub-block and one round); a group holds
// kEncWarps of them, one a compute warp.
__host__ __device__ constexpr uint32_t seg_symbols_grouped(uint32_t C, uint32_t S)
{
    if (C >= kGroupSyms)
        return seg_symbols(C, S);
    uint32_t seg = C < kGroupSyms / kEncWarps ? C : kGroupSyms / kEncWarps;
    seg = seg > S ? seg : S;
    return seg > kRoundSyms ? seg : kRoundSyms;
}
// Chunks of a group, and the stage slot of a group.
__host__ __device__ constexpr uint32_t enc_group_chunks(uint32_t C, uint32_t S)
{
    return C >= kGroupSyms ? 1u : kEncWarps / (C / seg_symbols_grouped(C, S));
}
__host__ __device__ constexpr uint32_t enc_ws_group_slot_bytes(uint32_t C, uint32_t S)
{
    return kEncWarps * region_bytes(seg_symbols_grouped(C, S));
}

// Fast-path sink for one lane's group: the multiplying packer with plain
// stores.  State: the partial word cur (its first nb bits used, 1 <= nb <=
// 32) at word index a of the region, K = 2^(32 - nb).  A group that starts
// at a word boundary takes its first pair as the initial partial word, so
// no lane ever writes a word before the one holding its first bit.  A
// completed word is stored whole, the predecessor's bits in it as zeros:
// the lane that ends in a word merges its partial word into it afterwards
// (or-reduction after a warp barrier), which also covers a word completed
// by the next lane.
struct SegPacker {
    uint32_t addr, cur, K; // addr: shared-window address of the word holding cur
#ifdef ECC_CHECKED
    uint32_t lim = ~0u;  // index-checked builds: stores must end at or below lim
    bool bad_index = false;
#endif

    // one append's tail: store w at addr when gate == 0 (the word filled up),
    // then take xlo (the code's remaining bits) as the partial word and move
    // to the next word; else w stays the partial word
    __device__ __forceinline__ void tail(uint32_t w, uint32_t xlo, uint32_t gate)
    {
#ifdef ECC_CHECKED
        if (gate == 0 && addr + 4u > lim) { // skip the store, keep the stream going
            bad_index = true;
            cur = xlo;
            addr += 4u;
            return;
        }
#endif
        asm volatile("{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %4, 0;\n\t@p st.shared.b32 [%0], %2;\n\t"
                     "selp.b32 %1, %3, %2, p;\n\t@p add.u32 %0, %0, 4;\n\t}"
                     : "+r"(addr), "=r"(cur)
                     : "r"(w), "r"(xlo), "r"(gate)
                     : "memory");
    }
    // pairs (v[k], q[k]) of one group at bit pos of the region (word base
    // `region`, shared-window address); c0 = the bits already in the word
    // holding pos (merged there by an earlier round, else 0)
    __device__ __forceinline__ void pack(uint32_t region, uint32_t pos, uint32_t c0, const uint32_t v[8],
                                         const uint32_t q[8])
    {
        const uint32_t nb0 = pos & 31u;
        addr = region + (pos >> 5) * 4u;
        {   // first pair: a normal append unless the group starts a word
            const uint32_t K0 = 1u << ((32u - nb0) & 31u); // nb0 = 0: unused
            const uint64_t x = (uint64_t)v[0] * K0;
            const uint64_t y = (uint64_t)K0 * q[0];
            const uint32_t yhi = (uint32_t)(y >> 32), ylo = (uint32_t)y;
            tail((uint32_t)(x >> 32) | c0, (uint32_t)x, nb0 ? yhi : 1u);
            cur = nb0 ? cur : v[0];
            K = nb0 ? yhi + ylo : q[0];
        }
#pragma unroll
        for (int k = 1; k < 8; ++k) {
            const uint64_t x = (uint64_t)v[k] * K;
            const uint64_t y = (uint64_t)K * q[k];
            const uint32_t yhi = (uint32_t)(y >> 32), ylo = (uint32_t)y;
            tail((uint32_t)(x >> 32) | cur, (uint32_t)x, yhi);
            K = yhi + ylo;
        }
    }
    // the same for the 16 codes of `in` one by one (table entries of codes of
    // at most 31 bits; a group with a longer pair)
    __device__ __forceinline__ void pack_singles(const uint2 *lut, uint32_t region, uint32_t pos, uint32_t c0,
                                                 uint4 in)
    {
        const uint32_t w[4] = {in.x, in.y, in.z, in.w};
        const uint32_t nb0 = pos & 31u;
        addr = region + (pos >> 5) * 4u;
        {
            const uint2 e = lut[byte_of(w[0], 0) * kLutReplicas];
            const uint32_t K0 = 1u << ((32u - nb0) & 31u);
            const uint64_t x = (uint64_t)e.x * K0;
            const uint64_t y = (uint64_t)K0 * e.y;
            const uint32_t yhi = (uint32_t)(y >> 32), ylo = (uint32_t)y;
            tail((uint32_t)(x >> 32) | c0, (uint32_t)x, nb0 ? yhi : 1u);
            cur = nb0 ? cur : e.x;
            K = nb0 ? yhi + ylo : e.y;
        }
#pragma unroll
        for (int j = 1; j < kSymPerThread; ++j) {
            const uint2 e = lut[byte_of(w[j >> 2], j & 3) * kLutReplicas];
            const uint64_t x = (uint64_t)e.x * K;
            const uint64_t y = (uint64_t)K * e.y;
            const uint32_t yhi = (uint32_t)(y >> 32), ylo = (uint32_t)y;
            tail((uint32_t)(x >> 32) | cur, (uint32_t)x, yhi);
            K = yhi + ylo;
        }
    }
};

// Exact-path sink for one lane's group (rare: partial groups, long codes):
// same protocol as SegPacker, codes read from the codebook.  Returns the
// final partial word (first bit in bit 31), its word index and its bit count
// (0: the group ended on a word boundary).
struct PackEnd {
    uint32_t word, wa, nb;
};
static __device__ __noinline__ PackEnd seg_exact_pack(uint32_t *region, uint32_t pos, uint32_t c0, uint4 in,
                                                      uint32_t cnt, const ecc_codebook *cb)
{
    const uint32_t w4[4] = {in.x, in.y, in.z, in.w};
    uint32_t wi = pos >> 5, nb = pos & 31u;
    uint32_t alo = nb ? c0 >> (32u - nb) : 0u, ahi = 0;
    auto put = [&](uint32_t code, uint32_t len) { // len <= 32
        ahi = __funnelshift_lc(alo, ahi, len);
        alo = shl_clamp(alo, len) | code;
        nb += len;
        if (nb >= 32) {
            nb -= 32;
            region[wi++] = __funnelshift_r(alo, ahi, nb);
        }
    };
    for (uint32_t j = 0; j < cnt; ++j) {
        const uint32_t b = byte_of(w4[j >> 2], j & 3);
        const uint32_t L = min((uint32_t)cb->len[b], (uint32_t)ECC_MAX_CODE_LEN);
        if (!L)
            continue;
        const uint64_t code = cb->code[b] & ((1ull << L) - 1);
        if (L > 24) {
            put((uint32_t)(code >> 24), L - 24);
            put((uint32_t)(code & 0xFFFFFFu), 24);
        } else {
            put((uint32_t)code, L);
        }
    }
    return PackEnd{nb ? shl_clamp(alo, 32u - nb) : 0u, wi, nb};
}

// Bit total of a slow group (bits 0-29), coded one code at a time from the
// table when it is full and every code has at most 31 bits (bit 30), else by
// the exact path from the codebook; bit 31: some byte has no code.
static __device__ __noinline__ uint32_t slow_group_bits(const uint2 *lut, uint4 in, uint32_t cnt,
                                                        const ecc_codebook *cb)
{
    bool exact = cnt < kSymPerThread;
    if (!exact) {
        const uint32_t bits = single_bits(lut, in, &exact);
        if (!exact)
            return bits | 1u << 30;
    }
    bool nocode = false;
    const uint32_t bits = exact_bits(in, cnt, cb, &nocode);
    return bits | (nocode ? 1u << 31 : 0u);
}

// Slow-group sink coded one code at a time from the table (SegPacker's
// protocol); returns the final partial word and its shared-window address.
static __device__ __noinline__ PackEnd seg_single_pack(const uint2 *lut, uint32_t region, uint32_t pos,
                                                       uint32_t c0, uint4 in, uint32_t lim)
{
    SegPacker pk;
#ifdef ECC_CHECKED
    pk.lim = lim;
#endif
    pk.pack_singles(lut, region, pos, c0, in);
#ifdef ECC_CHECKED
    if (pk.bad_index)
        return PackEnd{pk.cur, pk.addr, 0xFFFFFFFFu};
#endif
    return PackEnd{pk.cur, pk.addr, 1u};
}

// Code the rounds of one warp's segment [s0, s1) of chunk symbols (s1 > s0)
// into its region (shared-window address `region`, cap_bits of room).
// src: the chunk's staged input (kSharedSrc) else unused; the tensor's bytes
// come from job.in + base.  Writes the segment's sub-block bit counts.
// Returns the segment's bit total; raises bit 0 of *flag_word (and writes
// nothing more) if the segment outgrows its region; *bad if some byte has no
// code.
template <bool kSharedSrc>
__device__ __forceinline__ uint32_t encode_segment(EncShared &sh, const EncJob &job, const uint8_t *src,
                                                   uint64_t base, uint32_t s0, uint32_t s1, uint32_t region,
                                                   uint32_t cap_bits, uint32_t *flag_word, bool *bad)
{
    const int lane = threadIdx.x & 31;
    const uint2 *lut = sh.lut + (lane & (kLutReplicas - 1));
    const uint32_t s_shift = 31 - __clz(job.S);
    const uint32_t tps = job.S / kSymPerThread; // lanes per sub-block (64 for S = 1024: two rounds)
    uint16_t *sub = job.sub_bits + (base >> s_shift);
    uint32_t run = 0, half = 0;
    bool room = true;
    for (uint32_t r0 = s0; r0 < s1; r0 += kRoundSyms) {
        const bool full_round = r0 + kRoundSyms <= s1; // the same for every lane
        const uint32_t my0 = r0 + (uint32_t)lane * kSymPerThread;
        const uint32_t cnt = full_round ? kSymPerThread : my0 < s1 ? min((uint32_t)kSymPerThread, s1 - my0) : 0u;
        uint4 in = make_uint4(0, 0, 0, 0);
        if (full_round)
            in = load_symbols<kSharedSrc>(src + my0, job.in + base + my0, kSymPerThread);
        else if (cnt)
            in = load_symbols<kSharedSrc>(src + my0, job.in + base + my0, cnt);
        uint32_t pv[8], pq[8];
        bool slow;
        uint32_t bits = lookup_pairs(lut, in, cnt, pv, pq, &slow);
        // the common case, every group of the round full and coded by the
        // table, runs without a branch that splits the warp
        const bool fast = __all_sync(~0u, !slow);
        bool single = false; // slow group coded one code at a time from the table
        if (!fast && slow) {
            const uint32_t r = slow_group_bits(lut, in, cnt, job.cb);
            bits = r & 0x3FFFFFFFu;
            single = (r >> 30) & 1u;
            *bad |= (r >> 31) != 0;
        }
        uint32_t incl = bits;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(~0u, incl, o);
            incl += lane >= o ? y : 0u;
        }
        const uint32_t rtot = __shfl_sync(~0u, incl, 31);
        // sub-block bit counts
        if (tps <= 32) {
            const uint32_t sb = __shfl_sync(~0u, incl, lane | (int)(tps - 1)) - (incl - bits);
            if (cnt && (lane & (tps - 1)) == 0)
                sub[my0 >> s_shift] = (uint16_t)sb;
        } else {
            if (((r0 - s0) / kRoundSyms) & 1) {
                if (lane == 0)
                    sub[(my0 - kRoundSyms) >> s_shift] = (uint16_t)(half + rtot);
            } else if (r0 + kRoundSyms >= s1 && lane == 0) { // a final half sub-block
                sub[my0 >> s_shift] = (uint16_t)rtot;
            }
            half = rtot;
        }
        room = room && run + rtot <= cap_bits;
        if (room) {
            const uint32_t pos = run + incl - bits;
            // the word holding a lane's first bit may already hold bits of
            // the previous round (merged there): every lane reads it before
            // any lane of this round stores, so whichever lane completes it
            // keeps those bits (the others merge them again, harmlessly)
            const uint32_t lim = region + cap_bits / 8u + 16u; // the region's end (capacity + slack)
#ifdef ECC_CHECKED
            bool bad_index = region + (pos >> 5) * 4u + 4u > lim;
            const uint32_t cw = bad_index ? 0u : ld_shared_u32(region + (pos >> 5) * 4u);
#else
            const uint32_t cw = ld_shared_u32(region + (pos >> 5) * 4u);
#endif
            const uint32_t c0 = (pos & 31u) ? cw : 0u;
            __syncwarp();
            if (fast) {
                SegPacker pk;
#ifdef ECC_CHECKED
                pk.lim = lim;
#endif
                pk.pack(region, pos, c0, pv, pq);
                __syncwarp(); // every store of the round precedes every merge
#ifdef ECC_CHECKED
                bad_index |= pk.bad_index || pk.addr + 4u > lim;
                if (pk.addr + 4u <= lim)
#endif
                    red_or_shared(pk.addr, pk.cur);
            } else {
                uint32_t word = 0, wa = 0, nb = 0;
                if (cnt) {
                    if (!slow) {
                        SegPacker pk;
#ifdef ECC_CHECKED
                        pk.lim = lim;
#endif
                        pk.pack(region, pos, c0, pv, pq);
#ifdef ECC_CHECKED
                        bad_index |= pk.bad_index;
#endif
                        word = pk.cur;
                        wa = pk.addr;
                        nb = 1; // 1..32 bits: always a partial word to merge
                    } else if (single) {
                        const PackEnd e = seg_single_pack(lut, region, pos, c0, in, lim);
#ifdef ECC_CHECKED
                        bad_index |= e.nb != 1u;
#endif
                        word = e.word;
                        wa = e.wa;
                        nb = 1;
                    } else {
                        const PackEnd e = seg_exact_pack(
                            reinterpret_cast<uint32_t *>(__cvta_shared_to_generic(region)), pos, c0, in, cnt, job.cb);
                        word = e.word;
                        wa = region + e.wa * 4u;
                        nb = e.nb;
#ifdef ECC_CHECKED
                        bad_index |= wa > lim; // its stores ended below wa
#endif
                    }
                }
                __syncwarp();
#ifdef ECC_CHECKED
                bad_index |= nb && wa + 4u > lim;
                if (nb && wa + 4u <= lim)
#else
                if (nb)
#endif
                    red_or_shared(wa, word);
            }
#ifdef ECC_CHECKED
            if (bad_index)
                set_status(job.status, ECC_ERR_CHECK);
#endif
            __syncwarp();
        } else if (lane == 0) {
            atomicOr(flag_word, 1u);
        }
        run += rtot;
    }
    return run;
}

// Copy region w of a finished chunk from its stage slot (shared-window
// address `slot`, regions of region_words) to the chunk's payload at dst
// (global, 16-byte aligned); one warp.  seg_bits[0..nseg) are the segments'
// bit totals; the chunk's bitstream is their bits end to end.  Region w
// supplies the output words whose first bit lies in its segment, shifted
// from the region's word grid to the stream's; the last of them may also
// take the first bits of the segments after it (the first words of their
// regions, or seg_first[u] when given, which leaves the other regions free
// for reuse).  Region 0 also zeroes the
// words up to the 16-byte boundary after the stream.  Each lane takes four
// region words at a time (one 16-byte load).
// A pass of a larger chunk (P0 > 0: the slot's segments are the chunk's bits
// from bit P0 on): the word holding bit P0 was stored by the previous pass,
// with zeros for this pass's bits, and region 0 or-s its first bits into it
// (the caller orders the two); `pad`: the slot ends the chunk, so region 0
// zeroes the padding.
// Returns true (index-checked builds only) if the region or the chunk's
// padded payload would be overrun; nothing is copied then.
__device__ __forceinline__ bool copy_region_out(uint32_t slot, uint32_t region_words, const uint32_t *seg_bits,
                                                uint32_t nseg, uint32_t w, uint32_t *dst, uint32_t P0 = 0,
                                                bool pad = true, const uint32_t *seg_first = nullptr)
{
    const int lane = threadIdx.x & 31;
    uint32_t P = P0, total = P0;
    for (uint32_t u = 0; u < nseg; ++u) {
        P += u < w ? seg_bits[u] : 0u;
        total += seg_bits[u];
    }
    const uint32_t T = seg_bits[w];
    const uint32_t j0 = (P + 31) >> 5, nw = ((P + T + 31) >> 5) - j0;
#ifdef ECC_CHECKED
    if (nw && (nw >= region_words || j0 + nw > (pad16((total + 7) >> 3) >> 2)))
        return true;
#endif
    if (w == 0 && (P0 & 31u) && T && lane == 0) // the first word, shared with the previous pass
        atomicOr(dst + (P0 >> 5), bswap32(ld_shared_u32(slot) >> (P0 & 31u)));
    // nw = 0: the segment's bits all lie inside a word that starts in an
    // earlier segment, whose last word takes them
    if (nw) {
        const uint32_t src = slot + w * region_words * 4u;
        const uint32_t r = (0u - P) & 31u;
        const uint32_t nlast = nw - 1; // words [0, nlast) here, the last one below
        uint32_t *d = dst + j0;
        // output word i takes region words i and i + 1 (i + 1 <= nw stays
        // inside the region: nw <= its capacity in words + 1)
#pragma unroll 2
        for (uint32_t i0 = (uint32_t)lane * 4u; i0 < ((nlast + 127u) & ~127u); i0 += 128u) {
            const uint4 v = i0 <= nw ? ld_shared_v4(src + i0 * 4u) : make_uint4(0, 0, 0, 0);
            uint32_t nx = __shfl_down_sync(~0u, v.x, 1);
            if (lane == 31)
                nx = i0 + 4u <= nw ? ld_shared_u32(src + (i0 + 4u) * 4u) : 0u;
            const uint32_t o[4] = {__funnelshift_l(v.y, v.x, r), __funnelshift_l(v.z, v.y, r),
                                   __funnelshift_l(v.w, v.z, r), __funnelshift_l(nx, v.w, r)};
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (i0 + (uint32_t)t < nlast)
                    d[i0 + t] = bswap32(o[t]);
        }
        if (lane == 0) {
            uint32_t val = __funnelshift_l(ld_shared_u32(src + nw * 4u), ld_shared_u32(src + nlast * 4u), r);
            const uint32_t jj = j0 + nlast;
            uint32_t Pv = P + T; // first bits of the following segments inside this word
            for (uint32_t u = w + 1; u < nseg && Pv < 32 * jj + 32; ++u) {
                if (seg_bits[u])
                    val |= (seg_first ? seg_first[u] : ld_shared_u32(slot + u * region_words * 4u)) >> (Pv - 32 * jj);
                Pv += seg_bits[u];
            }
            d[nlast] = bswap32(val);
        }
    }
    if (w == 0 && pad) {
        const uint32_t jend = (total + 31) >> 5, jpad = pad16((total + 7) >> 3) >> 2;
        if (jend + (uint32_t)lane < jpad)
            dst[jend + lane] = 0;
    }
    return false;
}

// Zero one warp's region (shared-window address, region_words words, a
// multiple of 4).
__device__ __forceinline__ void zero_region(uint32_t region, uint32_t region_words)
{
    const int lane = threadIdx.x & 31;
    for (uint32_t i = (uint32_t)lane * 4u; i < region_words; i += 128u)
        st_shared_v4_zero(region + i * 4u);
}

// ---------------------------------------------------------------- warp-specialised encoder
// 8 compute warps encode chunk k into stage slot k % 2 (one segment each)
// and publish its aggregate at once; one output warp resolves the chunk's
// offset (decoupled look-back), writes chunk_off/total_bits/status and
// claims chunk k + 2 (ticket, then a bulk copy of its input into the input
// buffer chunk k has just released), while the compute warps code chunk
// k + 1 into the other slot; right after that they copy chunk k's regions
// out to their places in its bitstream, so the look-back has a whole
// chunk's time to resolve.  Named barriers: kBarFull + slot (compute ->
// output: the chunk is coded) and kBarReady + slot (output -> compute: its
// offset is known).  Claiming in the output warp keeps the ticket's round
// trip off the compute warps' critical path.

// Source of chunks of the many-tensor encoder: one ticket over the chunks of
// all tensors (workspace order), item[t] = tensor << 32 | chunk.
struct EncBatch {
    uint32_t *ticket;
    uint64_t total;
    const uint64_t *item;
    const ecc_desc *descs;
    uint64_t *flags; // look-back words, one per ticket
    uint32_t *done;  // chunks finished, per tensor
};

__device__ __forceinline__ void claim_single(EncSlot &s, uint32_t *ticket, uint64_t n_chunks)
{
    const uint32_t t = atomicAdd(ticket, 1u);
    s.c = t;
    s.state = t < n_chunks ? kSlotChunk : kSlotEnd;
}

__device__ __forceinline__ void claim_batched(EncSlot &s, const EncBatch &bt)
{
    const uint32_t t = atomicAdd(bt.ticket, 1u);
    if (t >= bt.total) {
        s.state = kSlotEnd;
        return;
    }
    const uint64_t m = bt.item[t];
    const uint32_t k = (uint32_t)(m >> 32);
    const uint64_t c = m & 0xFFFFFFFFull;
    const ecc_desc &d = bt.descs[k];
    const ecc_codebook *cb = d.cb;
    s.job = EncJob{d.in,     d.n,        cb,           d.C,  d.S, d.out, d.cap, d.chunk_off, d.sub_bits,
                   d.total_bits, bt.flags + (t - c), d.status};
    s.c = c;
    s.t_done = d.t_done_ns;
    s.tensor = k;
    s.state = (cb->magic == ECC_CODEBOOK_MAGIC && cb->max_len <= ECC_MAX_CODE_LEN) ? kSlotChunk : kSlotBadCodebook;
}

// Shared memory of the warp-specialised kernels: EncShared | 2 input buffers
// of cmax bytes | 2 stage slots of slot_bytes (see enc_ws_slot_bytes).
__host__ __device__ constexpr size_t enc_ws_smem_bytes(uint32_t cmax, uint32_t slot_bytes)
{
    return enc_shared_bytes() + 2 * (size_t)cmax + 2 * (size_t)slot_bytes;
}

constexpr uint32_t kBarReady = 4; // + slot: the chunk's output offset is known (output warp -> compute)

// kBatched: chunks of many tensors from bt (each chunk's job in its slot);
// else the chunks of `single`, one at a time or (kGrouped) in groups of gsz
// consecutive chunks, claimed with `ticket` (one ticket a group).  A group is coded
// as one unit: its chunks' segments spread over the compute warps (segment q
// of the group to warp q % kEncWarps), one look-back word and one output
// offset for the group, its chunks placed back to back from that offset.
template <bool kBatched, bool kGrouped = false>
__device__ __forceinline__ void encode_ws_body(const EncJob &single, uint64_t n_chunks, uint32_t *ticket,
                                               const EncBatch &bt, uint32_t slot_bytes, uint32_t cmax,
                                               uint64_t timeout_ns, uint32_t gsz = 1)
{
    extern __shared__ __align__(16) uint8_t smem[];
    EncShared &sh = *reinterpret_cast<EncShared *>(smem);
    uint8_t *inbuf = smem + enc_shared_bytes();
    const uint32_t stage0 = smem_u32(inbuf + 2 * (size_t)cmax);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t G = kGrouped && !kBatched ? gsz : 1u;
    const uint64_t n_units = kBatched ? 0 : (n_chunks + G - 1) / G; // groups
    if (!kBatched && (single.cb->magic != ECC_CODEBOOK_MAGIC || single.cb->max_len > ECC_MAX_CODE_LEN)) {
        if (tid == 0 && blockIdx.x == 0)
            set_status(single.status, ECC_ERR_CODEBOOK);
        return;
    }
    if (tid == 0) {
        mbar_init(&sh.bar[0], 1);
        mbar_init(&sh.bar[1], 1);
        fence_mbar_init();
        sh.issued[0] = sh.issued[1] = 0;
        sh.nostage = 0;
        sh.slot_flags[0] = sh.slot_flags[1] = 0;
    }
    if (!kBatched)
        load_encode_lut(sh, single.cb, kEncThreadsWS);
    for (uint32_t i = tid; i < 2 * slot_bytes / 16; i += kEncThreadsWS)
        st_shared_v4_zero(stage0 + i * 16u);
    // one thread: claim the unit (group or chunk) of iteration k into slot
    // k % 4 and, unless staging was given up, bulk-copy its input into buffer
    // k % 2
    auto claim = [&](uint32_t k) {
        EncSlot &s = sh.slot[k % kEncSlots];
        if (kBatched)
            claim_batched(s, bt);
        else
            claim_single(s, ticket, n_units);
        s.staged = 0;
        if (s.state != kSlotEnd && !sh.nostage) {
            issue_chunk_input(kBatched ? s.job : single, s.c * G, inbuf + (size_t)(k & 1) * cmax, &sh.bar[k & 1],
                              G);
            s.parity = sh.issued[k & 1] & 1u;
            s.staged = 1;
            ++sh.issued[k & 1];
        }
    };
    if (tid == 0) {
        claim(0);
        if (sh.slot[0].state != kSlotEnd)
            claim(1);
        else
            sh.slot[1].state = kSlotEnd;
    }
    __syncthreads(); // the last CTA-wide barrier before the warps split

    if (warp == kEncWarps) { // ---------------- output warp
        for (uint32_t k = 0;; ++k) {
            const uint32_t b = k & 1;
            bar_sync(kBarFull + b, kEncThreadsWS);
            const EncSlot &s = sh.slot[k % kEncSlots];
            if (s.state == kSlotEnd)
                break;
            if (lane == 0) { // unit k's input buffer is free: claim unit k + 2 into it
                if (sh.slot[(k + 1) % kEncSlots].state != kSlotEnd)
                    claim(k + 2);
                else
                    sh.slot[(k + 2) % kEncSlots].state = kSlotEnd;
            }
            const EncJob &job = kBatched ? s.job : single;
            const uint64_t u = s.c;
            const uint64_t c0 = u * G;
            const uint32_t gc = kGrouped ? (uint32_t)min((uint64_t)G, n_chunks - c0) : 1u; // chunks in the unit
            const uint32_t run = sh.slot_bits[b];
            const uint32_t fl = sh.slot_flags[b];
            __syncwarp();
            if (lane == 0)
                sh.slot_flags[b] = 0; // read; unit k + 2 is coded after this warp's arrival below
            const uint64_t bytes = kGrouped ? (uint64_t)sh.chunk_rel[b][gc] : ((uint64_t)run + 127u) / 128u * 16u;
            bool to = false;
            const uint64_t prefix = u == 0 ? 0 : resolve_prefix(job.flags, u, bytes, timeout_ns, &to);
            const bool fits = prefix + bytes <= job.out_cap;
            const bool write = fits && !to;
            if (kGrouped && (uint32_t)lane < gc)
                job.chunk_off[c0 + lane + 1] = prefix + sh.chunk_rel[b][lane + 1];
            if (lane == 0) {
                if (!kGrouped)
                    job.chunk_off[u + 1] = prefix + bytes;
                if (u == 0)
                    job.chunk_off[0] = 0;
                atomicAdd((unsigned long long *)job.total_bits, (unsigned long long)run);
                if (to)
                    set_status(job.status, ECC_ERR_TIMEOUT);
                else if (!fits)
                    set_status(job.status, ECC_ERR_CAPACITY);
            }
            const bool copy = write && !(fl & 1u);
            if (lane == 0) {
                sh.out_prefix[b] = prefix;
                sh.out_copy[b] = copy ? 1u : 0u;
            }
            // a segment outgrew its region (long codes): the unit is left to
            // the deferred pass (a warp a unit over the whole GPU, after this
            // kernel), so this warp's pipeline does not stall on it
            const bool deferred = (fl & 1u) && write;
            if (deferred && lane == 0)
                st_relaxed(job.flags + u, kFlagPrefix | kFlagDeferred | ((prefix + bytes) & kValueMask));
            if (kBatched && s.t_done && !copy && !deferred) {
                // completion counts one per segment: the copying warps count
                // their own, else this warp counts the chunk's
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t nseg = job.C / seg_symbols(job.C, job.S);
                    const uint32_t want = nseg * (uint32_t)((job.n + job.C - 1) >> (31 - __clz(job.C)));
                    if (atomicAdd(bt.done + s.tensor, nseg) + nseg == want)
                        *s.t_done = globaltimer();
                }
            }
            bar_arrive(kBarReady + b, kEncThreadsWS);
        }
    } else { // ---------------- compute warps
        const ecc_codebook *loaded = kBatched ? nullptr : single.cb;
        // copy this warp's regions of unit j (slot j % 2) out once the output
        // warp has resolved the unit's offset
        auto copy_out = [&](uint32_t j) {
            const uint32_t pb = j & 1;
            bar_sync(kBarReady + pb, kEncThreadsWS);
            const EncSlot &ps = sh.slot[j % kEncSlots];
            const EncJob &pjob = kBatched ? ps.job : single;
            const uint32_t seg = kGrouped ? seg_symbols_grouped(pjob.C, pjob.S) : seg_symbols(pjob.C, pjob.S);
            const uint32_t nseg = pjob.C / seg;
            const uint32_t gc = kGrouped ? (uint32_t)min((uint64_t)G, n_chunks - ps.c * G) : 1u;
            const uint32_t rwords = region_bytes(seg) / 4u;
            const uint32_t q = (uint32_t)warp; // the unit's segment q: chunk i, segment w of the chunk
            if (sh.out_copy[pb] && q < gc * nseg) {
                const uint32_t i = kGrouped ? q >> (31 - __clz(nseg)) : 0u, w = q - i * nseg; // nseg: a power of 2
                const bool bad_index = copy_region_out(
                    stage0 + pb * slot_bytes + i * nseg * rwords * 4u, rwords, sh.seg_bits[j & 3u] + i * nseg, nseg, w,
                    reinterpret_cast<uint32_t *>(pjob.out + sh.out_prefix[pb] + (kGrouped ? sh.chunk_rel[pb][i] : 0u)),
                    0u, true, sh.seg_first[j & 3u] + i * nseg);
                if (bad_index && lane == 0)
                    set_status(pjob.status, ECC_ERR_CHECK);
                if (kBatched && ps.t_done) {
                    __threadfence(); // this lane's payload stores before the completion count
                    __syncwarp();
                    const uint32_t want = nseg * (uint32_t)((pjob.n + pjob.C - 1) >> (31 - __clz(pjob.C)));
                    if (lane == 0 && atomicAdd(bt.done + ps.tensor, 1u) + 1u == want)
                        *ps.t_done = globaltimer();
                }
            }
        };
        for (uint32_t k = 0;; ++k) {
            const uint32_t b = k & 1;
            const EncSlot &s = sh.slot[k % kEncSlots];
            const uint32_t state = s.state;
            if (state == kSlotEnd) {
                bar_arrive(kBarFull + b, kEncThreadsWS);
                if (k >= 1)
                    copy_out(k - 1);
                break;
            }
            const EncJob &job = kBatched ? s.job : single;
            const uint64_t u = s.c;
            const uint64_t c0 = u * G;
            const uint32_t gc = kGrouped ? (uint32_t)min((uint64_t)G, n_chunks - c0) : 1u;
            const uint32_t seg = kGrouped ? seg_symbols_grouped(job.C, job.S) : seg_symbols(job.C, job.S);
            const uint32_t nseg = job.C / seg;
            const uint32_t rwords = region_bytes(seg) / 4u;
            // this warp's segment: segment w of the unit's chunk i (i = 0 unless
            // grouped; nseg is a power of two)
            const uint32_t i = kGrouped ? (uint32_t)warp >> (31 - __clz(nseg)) : 0u;
            const uint32_t w = (uint32_t)warp - i * nseg;
            const uint32_t region = stage0 + b * slot_bytes + (uint32_t)warp * rwords * 4u;
#ifdef ECC_CHECKED
            // index-checked builds: the warp's region must lie inside its
            // stage slot (a slot sized for another layout would run past the
            // shared memory the launch gave); otherwise nothing is staged and
            // the chunk takes the output warp's direct path
            const bool region_ok = (uint32_t)(warp + 1) * rwords * 4u <= slot_bytes;
            if (!region_ok && lane == 0)
                set_status(job.status, ECC_ERR_CHECK);
#else
            constexpr bool region_ok = true;
#endif
            if (k >= 2) {
                // unit k - 2 left this slot: this warp has copied its region
                // out (after coding unit k - 1), and the others' copies read
                // only their own regions and seg_first, so the region is free.
                // The many-tensor kernel also keeps every warp past its
                // lookups before a codebook change.
                if (kBatched)
                    bar_sync(kBarCompute, kEncThreads);
                if ((uint32_t)warp < G * nseg && region_ok)
                    zero_region(region, rwords);
            }
            if (kBatched && state == kSlotChunk && job.cb != loaded) {
                // every compute warp is past the last lookup of the previous
                // chunk (the chunk barrier); the output warp's overflow path
                // reads the codebook in global memory
                bar_sync(kBarCompute, kEncThreads);
                load_encode_lut(sh, job.cb, kEncThreads);
                loaded = job.cb;
                bar_sync(kBarCompute, kEncThreads);
            }
            const uint64_t base = (c0 + i) * job.C;
            const uint32_t L =
                state == kSlotChunk && i < gc ? (uint32_t)min((uint64_t)job.C, job.n - base) : 0u;
            const uint32_t s0 = w * seg, s1 = min(s0 + seg, L);
            bool bad = state == kSlotBadCodebook;
            uint32_t bits = 0;
            if (s0 < s1) {
                bool ok = false;
                if (s.staged) {
                    ok = __all_sync(~0u, mbar_wait(&sh.bar[b], s.parity, timeout_ns));
                    if (!ok && lane == 0) { // never expected: the copy reads valid memory
                        set_status(job.status, ECC_ERR_TIMEOUT);
                        sh.nostage = 1;
                    }
                }
                const uint8_t *src = inbuf + (size_t)b * cmax + (size_t)i * job.C;
                const uint32_t cap = region_ok ? region_cap_bytes(seg) * 8u : 0u;
                bits = ok ? encode_segment<true>(sh, job, src, base, s0, s1, region, cap, &sh.slot_flags[b], &bad)
                          : encode_segment<false>(sh, job, nullptr, base, s0, s1, region, cap, &sh.slot_flags[b],
                                                  &bad);
            }
            if (lane == 0) {
                sh.seg_bits[k & 3u][warp] = bits;
                sh.seg_first[k & 3u][warp] = bits && region_ok ? ld_shared_u32(region) : 0u;
            }
            if (bad && lane == 0)
                set_status(job.status, ECC_ERR_CODEBOOK);
            bar_sync(kBarCompute, kEncThreads); // the unit is coded
            if (tid == 0) {
                uint32_t run = 0;
                uint64_t bytes;
                if (kGrouped) { // the chunks' padded offsets in the group
                    uint32_t rel = 0;
                    sh.chunk_rel[b][0] = 0;
                    for (uint32_t i = 0; i < gc; ++i) {
                        uint32_t r = 0;
                        for (uint32_t w = 0; w < nseg; ++w)
                            r += sh.seg_bits[k & 3u][i * nseg + w];
                        run += r;
                        rel += (r + 127u) / 128u * 16u;
                        sh.chunk_rel[b][i + 1] = rel;
                    }
                    bytes = rel;
                } else {
#pragma unroll
                    for (uint32_t w = 0; w < kEncWarps; ++w)
                        run += w < nseg ? sh.seg_bits[k & 3u][w] : 0u;
                    bytes = ((uint64_t)run + 127u) / 128u * 16u;
                }
                st_relaxed(job.flags + u, (u == 0 ? kFlagPrefix : kFlagAggregate) | (bytes & kValueMask));
                sh.slot_bits[b] = run;
            }
            bar_arrive(kBarFull + b, kEncThreadsWS);
            // unit k - 1's offset has had a whole unit to resolve
            if (k >= 1)
                copy_out(k - 1);
        }
    }
    // never exit with a bulk copy still writing into this CTA's shared memory
    // (only after a timed-out wait can an issued copy be left unconsumed)
    __syncthreads();
    if (tid == 0)
        for (uint32_t q = 0; q < 2; ++q)
            if (sh.issued[q])
                (void)mbar_wait(&sh.bar[q], (sh.issued[q] - 1u) & 1u, timeout_ns);
}

// ---------------------------------------------------------------- chunks of more than kGroupSyms symbols
// Three launches: a length pass writes each chunk's payload bits into the
// look-back words (flags[c], bit 63 set when a segment of the chunk needs
// more than its stage region), a scan turns them into chunk_off and
// total_bits, and then encode_pass_body codes each chunk in passes of
// kGroupSyms symbols (kEncWarps segments of kPassSeg, one a compute warp)
// into a stage slot and copies every pass out at its place in the chunk's
// bitstream, which is known before the pass is coded: no pass waits for a
// look-back, and a stage slot holds one pass instead of a whole chunk.  A
// chunk's passes go to one CTA in order, so the word that two passes share
// is stored by the earlier pass and or-ed into by the later one after a CTA
// barrier.  A flagged chunk is coded by the output warp straight into the
// output.
constexpr uint32_t kPassSeg = kGroupSyms / kEncWarps;
constexpr uint32_t kSlotDirect = 3; // a chunk the output warp codes straight into the output
constexpr uint64_t kLenOverflow = 1ull << 63;

// Bulk-copy the whole 16-byte groups of the L input bytes at src into buf
// (thread 0); completion arrives on bar.  Trailing bytes (fewer than 16, the
// tensor's end) are read from global memory by the thread that owns them.
__device__ __forceinline__ void issue_input(const uint8_t *src, uint32_t L, uint8_t *buf, uint64_t *bar)
{
    const uint32_t whole = L & ~15u;
    fence_proxy_async();
    mbar_expect_tx(bar, whole);
    if (whole)
        bulk_g2s(buf, src, whole, bar);
}

// Passes of chunk c.
__device__ __forceinline__ uint32_t chunk_passes(const EncJob &job, uint64_t c)
{
    const uint32_t L = (uint32_t)min((uint64_t)job.C, job.n - c * job.C);
    return (L + kGroupSyms - 1) / kGroupSyms;
}

// The pass encoder (C > kGroupSyms): slots and barriers as in
// encode_ws_body, a unit being one pass (EncSlot::c the chunk,
// EncSlot::tensor the pass) or one flagged chunk (kSlotDirect).
// chunk_rel[b][0] / [1] hold the slot's bit offset in its chunk and whether
// it ends the chunk.
__device__ __forceinline__ void encode_pass_body(const EncJob &job, uint64_t n_chunks, uint32_t *ticket,
                                                 uint32_t slot_bytes, uint64_t timeout_ns)
{
    extern __shared__ __align__(16) uint8_t smem[];
    EncShared &sh = *reinterpret_cast<EncShared *>(smem);
    uint8_t *inbuf = smem + enc_shared_bytes();
    constexpr uint32_t cmax = kGroupSyms;
    const uint32_t stage0 = smem_u32(inbuf + 2 * (size_t)cmax);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (job.cb->magic != ECC_CODEBOOK_MAGIC || job.cb->max_len > ECC_MAX_CODE_LEN) {
        if (tid == 0 && blockIdx.x == 0)
            set_status(job.status, ECC_ERR_CODEBOOK);
        return;
    }
    if (tid == 0) {
        mbar_init(&sh.bar[0], 1);
        mbar_init(&sh.bar[1], 1);
        fence_mbar_init();
        sh.issued[0] = sh.issued[1] = 0;
        sh.nostage = 0;
        sh.slot_flags[0] = sh.slot_flags[1] = 0;
    }
    load_encode_lut(sh, job.cb, kEncThreadsWS);
    for (uint32_t i = tid; i < 2 * slot_bytes / 16; i += kEncThreadsWS)
        st_shared_v4_zero(stage0 + i * 16u);
    // one thread: the unit of iteration k into slot k % 4 -- the next pass
    // of iteration k - 1's chunk, else a new chunk by ticket -- and, unless
    // staging was given up, its input into buffer k % 2
    auto claim = [&](uint32_t k) {
        EncSlot &s = sh.slot[k % kEncSlots];
        const EncSlot &prev = sh.slot[(k + kEncSlots - 1) % kEncSlots];
        if (k > 0 && prev.state == kSlotChunk && prev.tensor + 1 < chunk_passes(job, prev.c)) {
            s.c = prev.c;
            s.tensor = prev.tensor + 1;
            s.state = kSlotChunk;
        } else {
            claim_single(s, ticket, n_chunks);
            s.tensor = 0;
            if (s.state == kSlotChunk && (ld_relaxed(job.flags + s.c) & kLenOverflow))
                s.state = kSlotDirect;
        }
        s.staged = 0;
        if (s.state == kSlotChunk && !sh.nostage) {
            const uint64_t base = s.c * job.C + (uint64_t)s.tensor * kGroupSyms;
            issue_input(job.in + base, (uint32_t)min((uint64_t)kGroupSyms, job.n - base),
                        inbuf + (size_t)(k & 1) * cmax, &sh.bar[k & 1]);
            s.parity = sh.issued[k & 1] & 1u;
            s.staged = 1;
            ++sh.issued[k & 1];
        }
    };
    if (tid == 0) {
        claim(0);
        if (sh.slot[0].state != kSlotEnd)
            claim(1);
        else
            sh.slot[1].state = kSlotEnd;
    }
    __syncthreads(); // the last CTA-wide barrier before the warps split

    const uint32_t seg = kPassSeg;
    const uint32_t rwords = region_bytes(seg) / 4u;
    if (warp == kEncWarps) { // ---------------- output warp
        uint32_t pos = 0; // bits of the current chunk's earlier passes
        for (uint32_t k = 0;; ++k) {
            const uint32_t b = k & 1;
            bar_sync(kBarFull + b, kEncThreadsWS);
            const EncSlot &s = sh.slot[k % kEncSlots];
            if (s.state == kSlotEnd)
                break;
            if (lane == 0) { // unit k's input buffer is free: claim unit k + 2 into it
                if (sh.slot[(k + 1) % kEncSlots].state != kSlotEnd)
                    claim(k + 2);
                else
                    sh.slot[(k + 2) % kEncSlots].state = kSlotEnd;
            }
            const uint64_t c = s.c;
            const uint64_t prefix = job.chunk_off[c], end = job.chunk_off[c + 1]; // written by the scan
            const bool write = end <= job.out_cap;
            bool copy = false;
            if (s.state == kSlotDirect) {
                if (write)
                    encode_chunk_warp(job, c, reinterpret_cast<uint32_t *>(job.out + prefix),
                                      (uint32_t)((end - prefix) / 4));
            } else {
                const uint32_t run = sh.slot_bits[b];
                if (s.tensor == 0)
                    pos = 0;
                const uint32_t P0 = pos;
                pos += run;
                const bool last = s.tensor + 1 == chunk_passes(job, c);
                // the coded bits must be the length pass's (the same lookups)
                const bool mismatch = (sh.slot_flags[b] & 1u) ||
                                      (last && (uint64_t)pos != (ld_relaxed(job.flags + c) & ~kLenOverflow));
                if (mismatch && lane == 0)
                    set_status(job.status, ECC_ERR_CHECK);
                copy = write && !mismatch;
                if (lane == 0) {
                    sh.chunk_rel[b][0] = P0;
                    sh.chunk_rel[b][1] = last ? 1u : 0u;
                    sh.out_prefix[b] = prefix;
                }
            }
            if (lane == 0)
                sh.out_copy[b] = copy ? 1u : 0u;
            bar_arrive(kBarReady + b, kEncThreadsWS);
        }
    } else { // ---------------- compute warps
        // copy this warp's region of unit j (slot j % 2) out
        auto copy_out = [&](uint32_t j) {
            const uint32_t pb = j & 1;
            bar_sync(kBarReady + pb, kEncThreadsWS);
            if (sh.out_copy[pb]) {
                const bool bad_index = copy_region_out(
                    stage0 + pb * slot_bytes, rwords, sh.seg_bits[pb], kEncWarps, (uint32_t)warp,
                    reinterpret_cast<uint32_t *>(job.out + sh.out_prefix[pb]), sh.chunk_rel[pb][0],
                    sh.chunk_rel[pb][1] != 0);
                if (bad_index && lane == 0)
                    set_status(job.status, ECC_ERR_CHECK);
            }
        };
        for (uint32_t k = 0;; ++k) {
            const uint32_t b = k & 1;
            const EncSlot &s = sh.slot[k % kEncSlots];
            const uint32_t state = s.state;
            if (state == kSlotEnd) {
                bar_arrive(kBarFull + b, kEncThreadsWS);
                if (k >= 1)
                    copy_out(k - 1);
                break;
            }
            const uint32_t region = stage0 + b * slot_bytes + (uint32_t)warp * rwords * 4u;
            if (k >= 2) {
                // unit k - 2 left this slot: every warp has copied its region
                // out (after coding unit k - 1) and is past its lookups; the
                // barrier also orders the copies of consecutive passes
                bar_sync(kBarCompute, kEncThreads);
                if (tid == 0)
                    sh.slot_flags[b] = 0; // the output warp has read it
                zero_region(region, rwords);
            }
            // a flagged chunk (the output warp codes it): this warp's eighth of
            // the chunk, for its sub-block counts only (a region of no room
            // packs nothing)
            const bool direct = state == kSlotDirect;
            const uint64_t base = s.c * job.C + (direct ? 0ull : (uint64_t)s.tensor * kGroupSyms);
            const uint32_t span = direct ? job.C / kEncWarps : seg;
            const uint32_t L = (uint32_t)min((uint64_t)(direct ? job.C : kGroupSyms), job.n - base);
            const uint32_t s0 = (uint32_t)warp * span, s1 = min(s0 + span, L);
            bool bad = false;
            uint32_t bits = 0;
            if (direct && s0 < s1) {
                (void)encode_segment<false>(sh, job, nullptr, base, s0, s1, region, 0u, &sh.slot_flags[b], &bad);
            } else if (s0 < s1) {
                bool ok = false;
                if (s.staged) {
                    ok = __all_sync(~0u, mbar_wait(&sh.bar[b], s.parity, timeout_ns));
                    if (!ok && lane == 0) { // never expected: the copy reads valid memory
                        set_status(job.status, ECC_ERR_TIMEOUT);
                        sh.nostage = 1;
                    }
                }
                const uint8_t *src = inbuf + (size_t)b * cmax;
                const uint32_t cap = region_cap_bytes(seg) * 8u;
                bits = ok ? encode_segment<true>(sh, job, src, base, s0, s1, region, cap, &sh.slot_flags[b], &bad)
                          : encode_segment<false>(sh, job, nullptr, base, s0, s1, region, cap, &sh.slot_flags[b],
                                                  &bad);
            }
            if (bad && lane == 0)
                set_status(job.status, ECC_ERR_CODEBOOK);
            if (lane == 0)
                sh.seg_bits[b][warp] = bits;
            bar_sync(kBarCompute, kEncThreads); // the unit is coded
            if (tid == 0) {
                uint32_t run = 0;
#pragma unroll
                for (uint32_t w = 0; w < kEncWarps; ++w)
                    run += sh.seg_bits[b][w];
                sh.slot_bits[b] = run;
            }
            bar_arrive(kBarFull + b, kEncThreadsWS);
            if (k >= 1)
                copy_out(k - 1);
        }
    }
    // never exit with a bulk copy still writing into this CTA's shared memory
    // (only after a timed-out wait can an issued copy be left unconsumed)
    __syncthreads();
    if (tid == 0)
        for (uint32_t q = 0; q < 2; ++q)
            if (sh.issued[q])
                (void)mbar_wait(&sh.bar[q], (sh.issued[q] - 1u) & 1u, timeout_ns);
}

// ---------------------------------------------------------------- decoder
// One warp decodes one chunk: lane l runs the sub-blocks l, l + 32, ... of
// the chunk as independent bit streams, starting at offsets given by a warp
// scan of sub_bits.  Each step peeks 12 bits and resolves the code through
// the first-level table; longer Huffman codes fall back to canonical
// per-length ranges.
struct DecJob {
    const uint8_t *in;
    uint64_t in_bytes;
    const uint64_t *chunk_off;
    const uint16_t *sub_bits;
    uint64_t n;
    uint32_t C, S;
    const ecc_codebook *cb;
    uint8_t *out;
    uint32_t *status;
};

// Canonical ranges of the codes longer than the first-level table, staged in
// shared memory for the decoder's slow path.  For a length L the L-bit
// prefix v of the stream is a code of length L exactly when v < first[L] +
// count[L] and no shorter length matched; the test is monotone in L, so the
// code length is the number of lengths that fail plus the first length tried.
//
// Second level: a canonical code's longer codes are its numerically largest,
// so the codes longer than the first-level table start with the few 14-bit
// prefixes from first[14] + count[14] up (about 2^14 times their share of
// the code space: two or three for a code whose long codes are rare under
// its own statistics, however often the data meets them).  For those
// sub_np prefixes, each followed by sub_kb more bits, sub[] holds
// byte | length << 8 of the code those 14 + sub_kb bits start, or 0 when
// the code is longer (or there is none): one lookup in place of the search
// over the ranges.  sub_np = 0: no second level (a QLC codebook, codes
// longer than 32 bits, or too many prefixes for kLongSubEntries).
constexpr uint32_t kLongSubEntries = 2048;
struct LongTable {
    uint64_t lim32[33];    // (first[L] + count[L]) << (32 - L), L <= 32
    uint64_t first[ECC_MAX_CODE_LEN + 1];
    uint16_t index[ECC_MAX_CODE_LEN + 1];
    uint16_t count[ECC_MAX_CODE_LEN + 1];
    uint8_t sorted[256];
    uint32_t max_len;
    uint32_t family;
    uint32_t sub_p0, sub_np, sub_kb;
    uint16_t sub[kLongSubEntries];
};

__device__ __forceinline__ void load_long_table(LongTable &lt, const ecc_codebook *cb)
{
    const int t = threadIdx.x;
    const uint32_t maxl = min(cb->max_len, (uint32_t)ECC_MAX_CODE_LEN);
    for (int L = t; L <= ECC_MAX_CODE_LEN; L += blockDim.x) {
        const uint64_t f = cb->first[L];
        const uint32_t k = (uint32_t)L <= maxl ? cb->count[L] : 0u;
        lt.first[L] = f;
        lt.index[L] = cb->index[L];
        lt.count[L] = (uint16_t)k;
        if (L <= 32)
            lt.lim32[L] = L == 0 ? 0ull : (f + k) << (32 - L);
    }
    for (int i = t; i < 256; i += blockDim.x)
        lt.sorted[i] = cb->sorted[i];
    if (t == 0) {
        lt.max_len = maxl;
        lt.family = cb->family;
        // the second level's extent (its entries: fill_long_sub, once the
        // ranges above are in place)
        uint32_t np = 0, kb = 0;
        const uint64_t p0 = cb->first[ECC_PEEK_BITS] + (ECC_PEEK_BITS <= maxl ? cb->count[ECC_PEEK_BITS] : 0u);
        if (cb->family == ECC_FAMILY_HUFFMAN && maxl > ECC_PEEK_BITS && maxl <= 32 && p0 < (1u << ECC_PEEK_BITS)) {
            const uint64_t end = (cb->first[maxl] + cb->count[maxl]) << (32 - maxl); // past the last long code
            const uint64_t lo = p0 << (32 - ECC_PEEK_BITS);
            if (end > lo && end <= (1ull << 32)) {
                np = (uint32_t)(((end - 1) >> (32 - ECC_PEEK_BITS)) - p0 + 1);
                while (kb < maxl - ECC_PEEK_BITS && ((uint64_t)np << (kb + 1)) <= kLongSubEntries)
                    ++kb;
                if (kb == 0)
                    np = 0;
            }
        }
        lt.sub_p0 = (uint32_t)p0;
        lt.sub_np = np;
        lt.sub_kb = kb;
    }
}

// The second level's entries from the ranges (threads i0, i0 + stride, ...,
// after a barrier that follows load_long_table; a barrier follows before
// any lookup).
__device__ __forceinline__ uint32_t decode_long32(uint32_t p32, const LongTable &lt);
__device__ __forceinline__ void fill_long_sub(LongTable &lt, uint32_t i0, uint32_t stride)
{
    const uint32_t kb = lt.sub_kb, n = lt.sub_np << kb;
    for (uint32_t j = i0; j < n; j += stride) {
        // the 32-bit window of prefix sub_p0 + (j >> kb), then j's low kb bits, then zeros
        const uint32_t v = ((lt.sub_p0 + (j >> kb)) << (32 - ECC_PEEK_BITS)) |
                           ((j & ((1u << kb) - 1u)) << (32 - ECC_PEEK_BITS - kb));
        const uint32_t e = decode_long32(v, lt);
        lt.sub[j] = (uint16_t)((e >> 8) <= ECC_PEEK_BITS + kb ? e : 0u);
    }
}

// Resolve a code longer than the first-level table.  p32 holds the next 32
// stream bits and win the next 64, MSB first.  Returns byte | len << 8, or 0
// for a code the codebook lacks.
static __device__ __noinline__ uint32_t decode_long(uint32_t p32, uint64_t win, const LongTable &lt)
{
    if (lt.family != ECC_FAMILY_HUFFMAN)
        return 0;
    const uint32_t maxl = lt.max_len;
    uint32_t L = ECC_PEEK_BITS + 1;
    if (maxl <= 32) {
        // count the lengths in (12, maxl) whose range lies below the window
#pragma unroll
        for (uint32_t j = ECC_PEEK_BITS + 1; j < 32; ++j)
            L += (j < maxl) & ((uint64_t)p32 >= lt.lim32[j]);
        if (L > maxl)
            return 0;
        const uint32_t v = p32 >> (32 - L);
        const uint64_t d = (uint64_t)v - lt.first[L];
        if (d >= lt.count[L])
            return 0;
        const uint32_t at = lt.index[L] + (uint32_t)d;
        return at < 256 ? (uint32_t)lt.sorted[at] | (L << 8) : 0u;
    }
    for (; L <= maxl; ++L) {
        const uint32_t k = lt.count[L];
        if (!k)
            continue;
        const uint64_t d = (win >> (64 - L)) - lt.first[L];
        if (d < k) {
            const uint32_t at = lt.index[L] + (uint32_t)d;
            return at < 256 ? (uint32_t)lt.sorted[at] | (L << 8) : 0u;
        }
    }
    return 0;
}

// Bit stream of one sub-block, read from 32-bit words in memory byte order
// through a sliding window: (hi, lo) are words wp-3 and wp-2, nx (word wp-1)
// is already loaded, o is the bit offset into hi.  Word reads are clamped to
// [0, wlast], so a corrupt stream can never read outside its chunk.
struct Stream {
    uint32_t hi, lo, nx, o, wp;
};

template <bool kShared>
__device__ __forceinline__ uint32_t load_word(const uint32_t *words, uint32_t i, uint32_t wlast)
{
    const uint32_t k = min(i, wlast);
    return bswap32(kShared ? words[k] : __ldg(words + k));
}

template <bool kShared>
__device__ __forceinline__ void stream_start(Stream &s, const uint32_t *words, uint32_t wlast, uint32_t bit)
{
    const uint32_t w0 = bit >> 5;
    s.o = bit & 31;
    s.hi = load_word<kShared>(words, w0, wlast);
    s.lo = load_word<kShared>(words, w0 + 1, wlast);
    s.nx = load_word<kShared>(words, w0 + 2, wlast);
    s.wp = w0 + 3;
}

__device__ __forceinline__ uint32_t stream_pos(const Stream &s) { return (s.wp - 3) * 32 + s.o; }

// Long or invalid code at the window (hi:lo:nx << o): byte | len << 8, or 0.
static __device__ __noinline__ uint32_t decode_long_at(uint32_t hi, uint32_t lo, uint32_t nx, uint32_t o,
                                                       const LongTable &lt)
{
    const uint64_t two = ((uint64_t)hi << 32) | lo;
    const uint64_t win = o ? (two << o) | ((uint64_t)nx >> (32 - o)) : two;
    return decode_long((uint32_t)(win >> 32), win, lt);
}

// Decode one symbol: returns byte | len << 8 (byte in the low 8 bits).
// kLong: the codebook has codes longer than the 12-bit first-level table, so
// an empty entry sends the lane to the slow path; otherwise an empty entry
// is an invalid code, recorded in emin (the minimum entry seen) and decoded
// as a zero-length code -- the sub-block's bit count then fails too.
template <bool kShared, bool kLong>
__device__ __forceinline__ uint32_t step(Stream &s, const uint32_t *words, uint32_t wlast, const uint16_t *dec,
                                         const LongTable &lt, bool &bad, uint32_t &emin)
{
    const uint32_t p = __funnelshift_l(s.lo, s.hi, s.o);
    uint32_t e = dec[p >> (32 - ECC_PEEK_BITS)];
    if (kLong) {
        if (e == 0) { // rare: a long or invalid code
            e = decode_long_at(s.hi, s.lo, s.nx, s.o, lt);
            if (e == 0) {
                bad = true;
                e = 1u << 8; // consume one bit and go on; the chunk is flagged
            }
            s.o += e >> 8;
            while (s.o >= 32) {
                s.hi = s.lo;
                s.lo = s.nx;
                s.nx = load_word<kShared>(words, s.wp, wlast);
                ++s.wp;
                s.o -= 32;
            }
            return e;
        }
    } else {
        emin = min(emin, e);
    }
    // a code of at most 12 bits moves the window by at most one word; the
    // word after nx is loaded every step, so no lane ever branches here
    s.o += e >> 8;
    const bool adv = s.o >= 32;
    const uint32_t w = load_word<kShared>(words, s.wp, wlast);
    s.hi = adv ? s.lo : s.hi;
    s.lo = adv ? s.nx : s.lo;
    s.nx = adv ? w : s.nx;
    s.wp += adv ? 1u : 0u;
    s.o &= 31;
    return e;
}

// Stream of the hot loop, reading the staged chunk in shared memory: the
// next three words (hi, lo, nx) in stream order, o the bit offset in hi
// (< 32), wa the shared-memory address of the word after nx.
struct FastStream {
    uint32_t hi, lo, nx, o, wa;
};

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// predicated shared load: v when p is false
__device__ __forceinline__ uint32_t lds_u32_if(uint32_t addr, bool p, uint32_t v)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q ld.shared.u32 %0, [%1];\n\t}"
                 : "+r"(v)
                 : "r"(addr), "r"((uint32_t)p));
    return v;
}

// predicated 16-bit shared load (zero-extended): v when p is false
__device__ __forceinline__ uint32_t lds_u16_if(uint32_t addr, bool p, uint32_t v)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q ld.shared.u16 %0, [%1];\n\t}"
                 : "+r"(v)
                 : "r"(addr), "r"((uint32_t)p));
    return v;
}

// Hot-loop step: two codes the 14-bit table resolves, one window refill.
// The first code starts at o < 32 and ends by bit 45, so the second one's
// 14-bit peek lies in (hi, lo) or (lo, nx); after both the stream has moved
// at most 59 bits, i.e. by at most one word.  Only a stream that moved on
// loads the refill word, after the lookups: the next step's first lookup
// reads (hi, lo) alone and hides the load, and the lanes that stay add no
// bank conflicts to the load (QLC steps, with no lookup on the stream's
// path, load first instead).  An empty entry (a longer or an
// invalid code) has length 0, so the stream stays where it is; emin records
// it and the caller redoes the iteration with fstep_slow.  Returns the two
// bytes in the low half (first code's in byte 0).
__device__ __forceinline__ uint32_t fstep2(FastStream &s, const uint16_t *dec, uint32_t &emin)
{
    const uint32_t p1 = __funnelshift_l(s.lo, s.hi, s.o);
    const uint32_t e1 = dec[p1 >> (32 - ECC_PEEK_BITS)];
    const uint32_t o1 = s.o + (e1 >> 8);
    const bool in2 = o1 >= 32;
    const uint32_t p2 = __funnelshift_l(in2 ? s.nx : s.lo, in2 ? s.lo : s.hi, o1); // shift taken mod 32
    const uint32_t e2 = dec[p2 >> (32 - ECC_PEEK_BITS)];
    emin = min(emin, min(e1, e2));
    const uint32_t o2 = o1 + (e2 >> 8);
    const bool adv = o2 >= 32;
    const uint32_t w = lds_u32_if(s.wa, adv, 0u);
    s.hi = adv ? s.lo : s.hi;
    s.lo = adv ? s.nx : s.lo;
    s.nx = adv ? bswap32(w) : s.nx;
    s.wa += adv ? 4u : 0u;
    s.o = o2 & 31;
    return __byte_perm(e1, e2, 0x0040);
}

// Any code, long ones through the canonical ranges; invalid codes set bad.
__device__ __forceinline__ uint32_t fstep_slow(FastStream &s, const uint16_t *dec, const LongTable &lt, bool &bad)
{
    const uint32_t p = __funnelshift_l(s.lo, s.hi, s.o);
    uint32_t e = dec[p >> (32 - ECC_PEEK_BITS)];
    if (e == 0) {
        e = decode_long_at(s.hi, s.lo, s.nx, s.o, lt);
        if (e == 0) {
            bad = true;
            e = 1u << 8; // consume one bit and go on; the chunk is flagged
        }
    }
    s.o += e >> 8;
    while (s.o >= 32) {
        s.hi = s.lo;
        s.lo = s.nx;
        s.nx = bswap32(lds_u32(s.wa));
        s.wa += 4;
        s.o -= 32;
    }
    return e;
}

// A code of at most 32 bits longer than the first-level table, from the
// next 32 stream bits p32; byte | len << 8, or 0 when the codebook has longer
// codes or p32 starts no code.  The length is 15 plus the number of lengths
// j in [15, max_len) whose canonical range lies below p32 (lim32 rises with
// j), found by a binary search.
__device__ __forceinline__ uint32_t decode_long32(uint32_t p32, const LongTable &lt)
{
    const uint32_t maxl = lt.max_len;
    if (maxl > 32 || maxl <= ECC_PEEK_BITS || lt.family != ECC_FAMILY_HUFFMAN)
        return 0;
    const uint32_t n = maxl - (ECC_PEEK_BITS + 1); // candidates j = 15 .. maxl - 1
    uint32_t c = 0;
#pragma unroll
    for (uint32_t step = 16; step; step >>= 1)
        if (c + step <= n && (uint64_t)p32 >= lt.lim32[ECC_PEEK_BITS + c + step])
            c += step;
    const uint32_t L = ECC_PEEK_BITS + 1 + c;
    const uint32_t v = L == 32 ? p32 : p32 >> (32 - L);
    const uint64_t d = (uint64_t)v - lt.first[L];
    if (d >= lt.count[L])
        return 0;
    const uint32_t at = lt.index[L] + (uint32_t)d;
    return at < 256 ? (uint32_t)lt.sorted[at] | (L << 8) : 0u;
}

// The second level's extent, read once per redo.
struct SubHdr {
    uint32_t p0, np, kb;
};

// A code the two table levels do not resolve: longer ones through the
// canonical ranges, byte | length << 8; an invalid code gives a one-bit step
// with bit 16 set (the chunk is flagged).
static __device__ __noinline__ uint32_t redo_long(uint32_t hi, uint32_t lo, uint32_t nx, uint32_t o, uint32_t p,
                                                  const LongTable &lt)
{
    uint32_t e = decode_long32(p, lt);
    if (e == 0)
        e = decode_long_at(hi, lo, nx, o, lt);
    return e ? e : (1u << 16) | (1u << 8);
}

// The redo of an iteration that met a code the first-level table does not
// resolve: one code at a time; the second level resolves most long codes in
// line, the rest go out of line.
__device__ __forceinline__ uint32_t fstep_redo(FastStream &s, const uint16_t *dec, const LongTable &lt,
                                               const SubHdr &h, bool &bad)
{
    const uint32_t p = __funnelshift_l(s.lo, s.hi, s.o);
    const uint32_t top = p >> (32 - ECC_PEEK_BITS);
    uint32_t e = dec[top];
    const uint32_t j = top - h.p0;
    if (e == 0 && j < h.np)
        e = lt.sub[(j << h.kb) | ((p << ECC_PEEK_BITS) >> (31u - h.kb) >> 1)];
    if (e == 0) {
        e = redo_long(s.hi, s.lo, s.nx, s.o, p, lt);
        bad |= (e >> 16) != 0;
        e &= 0xFFFFu;
    }
    s.o += e >> 8;
    while (s.o >= 32) {
        s.hi = s.lo;
        s.lo = s.nx;
        s.nx = bswap32(lds_u32(s.wa));
        s.wa += 4;
        s.o -= 32;
    }
    return e;
}

// Step of an iteration in long-code mode: one code through both table
// levels, the second-level load predicated on the first missing (no
// branch, so the R streams interleave).  A code either level resolves has
// at most 32 bits, so the window moves by at most one word; an unresolved
// one has length 0 (the stream stays) and sets emin to 0 for the redo.
// long2 records that some code took the second level.
__device__ __forceinline__ uint32_t fstep_long(FastStream &s, const uint16_t *dec, const LongTable &lt,
                                               const SubHdr &h, uint32_t &emin, bool &long2)
{
    const uint32_t p = __funnelshift_l(s.lo, s.hi, s.o);
    const uint32_t top = p >> (32 - ECC_PEEK_BITS);
    uint32_t e = dec[top];
    const uint32_t j = top - h.p0;
    const bool use2 = e == 0 && j < h.np;
    // (kb = 0 when there is no second level: the shifts stay below 32)
    const uint32_t idx = (j << h.kb) | ((p << ECC_PEEK_BITS) >> (31u - h.kb) >> 1);
    e = lds_u16_if(smem_u32(lt.sub) + 2u * idx, use2, e);
    long2 |= use2;
    emin = min(emin, e);
    const uint32_t o = s.o + (e >> 8);
    const bool adv = o >= 32;
    const uint32_t w = lds_u32_if(s.wa, adv, 0u);
    s.hi = adv ? s.lo : s.hi;
    s.lo = adv ? s.nx : s.lo;
    s.nx = adv ? bswap32(w) : s.nx;
    s.wa += adv ? 4u : 0u;
    s.o = o & 31;
    return e;
}

// QLC codes need no first-level table: the 3-bit prefix fixes the code
// length (a byte of two registers, selected by the prefix), and the rank is
// the whole code plus a per-prefix offset (start of the area minus prefix <<
// width).  The stream's next position then never waits for a shared-memory
// load; the rank -> byte lookups run beside it, in a table with one replica
// per lane (rank r of lane l at word r * 32 + l), free of bank conflicts.
// A rank of 256 or more is no code (an empty area, or past the last rank).
// Ranks stay below 512 (an empty area's offset maps its codes to 256 +
// suffix), so the lookup needs no clamp: it reads within the first 64 KiB
// of the CTA's shared memory, which the launch always provides.
struct QlcShared {
    int32_t off[8];
    uint32_t len[2]; // code length of prefixes 0..3 and 4..7, one byte each
};
// shared memory a decoder launch always provides, covering QLC rank lookups
constexpr uint32_t kDecMinSmem = 64u * 1024u + 128u;

// The decoder's tables for one codebook.
struct DecTables {
    const uint16_t *dec; // 14-bit first-level table: shared, or (QLC mode) the codebook's own in global memory
    const LongTable *lt; // shared
    uint32_t len0, len1; // QLC: code length by prefix
    uint32_t lg;         // QLC: the upper bytes a byte-permute of (len0, len1) by a prefix leaves (byte 0 of len0 in each)
    const int32_t *off;  // QLC: shared, rank = code + off[prefix]
    uint32_t rt;         // QLC: shared-window address of the rank table + lane * 4
};

// Whether the QLC path can decode with this codebook.
__device__ __forceinline__ bool qlc_mode(const ecc_codebook *cb)
{
    return cb->family == ECC_FAMILY_QLC && cb->prefix_bits == 3 && cb->max_len <= 11;
}

// Fill the QLC tables from the codebook: the rank table over the 32 KB of
// the first-level table (threads [0, nthreads)).
__device__ __forceinline__ void load_qlc_tables(uint32_t *rt, QlcShared &q, const ecc_codebook *cb, uint32_t nthreads)
{
    const uint32_t t = threadIdx.x;
    for (uint32_t i = t; i < 256 * 32; i += nthreads)
        rt[i] = cb->by_rank[i >> 5];
    if (t < 8) {
        const uint32_t w = cb->width[t];
        q.off[t] = (cb->area_size[t] ? (int32_t)cb->area_start[t] : 256) - (int32_t)(t << w);
    }
    if (t == 0) {
        uint32_t l0 = 0, l1 = 0;
        for (int k = 0; k < 4; ++k) {
            l0 |= (3u + cb->width[k]) << (8 * k);
            l1 |= (3u + cb->width[k + 4]) << (8 * k);
        }
        q.len[0] = l0;
        q.len[1] = l1;
    }
}

__device__ __forceinline__ DecTables qlc_tables(const uint16_t *gdec, const LongTable *lt, const QlcShared &q,
                                                const uint32_t *rt)
{
    DecTables T;
    T.dec = gdec;
    T.lt = lt;
    T.len0 = q.len[0];
    T.len1 = q.len[1];
    T.lg = (q.len[0] & 0xFFu) * 0x01010100u;
    T.off = q.off;
    T.rt = smem_u32(rt) + (threadIdx.x & 31) * 4u;
    return T;
}

// QLC hot-loop step: two codes, one window refill, as fstep2.  vmax collects
// the ranks (one of 256 or more: no code, the chunk is corrupt).
__device__ __forceinline__ uint32_t qstep2(FastStream &s, const DecTables &T, uint32_t &vmax)
{
    const uint32_t w = lds_u32(s.wa); // the refill word, loaded first: nothing else hides its latency here
    // the permute leaves len[prefix] in byte 0 and byte 0 of len0 in bytes
    // 1..3: lg removes those; a funnel shift only uses the low 5 bits anyway
    const uint32_t p1 = __funnelshift_l(s.lo, s.hi, s.o);
    const uint32_t a1 = p1 >> 29;
    const uint32_t l1 = __byte_perm(T.len0, T.len1, a1);
    const uint32_t o1 = s.o + l1 - T.lg;
    const bool in2 = o1 >= 32;
    const uint32_t p2 = __funnelshift_l(in2 ? s.nx : s.lo, in2 ? s.lo : s.hi, o1); // shift taken mod 32
    const uint32_t a2 = p2 >> 29;
    const uint32_t l2 = __byte_perm(T.len0, T.len1, a2);
    const uint32_t o2 = o1 + l2 - T.lg;
    const bool adv = o2 >= 32;
    s.hi = adv ? s.lo : s.hi;
    s.lo = adv ? s.nx : s.lo;
    s.nx = adv ? bswap32(w) : s.nx;
    s.wa += adv ? 4u : 0u;
    s.o = o2 & 31;
    // beside the stream: ranks and bytes
    const uint32_t r1 = __funnelshift_l(p1, 0u, l1) + (uint32_t)T.off[a1];
    const uint32_t r2 = __funnelshift_l(p2, 0u, l2) + (uint32_t)T.off[a2];
    vmax = max(vmax, max(r1, r2));
    const uint32_t b1 = lds_u32(T.rt + r1 * 128u);
    const uint32_t b2 = lds_u32(T.rt + r2 * 128u);
    return __byte_perm(b1, b2, 0x0040);
}

// Hot loop: R full sub-blocks per lane from a staged chunk, 8 symbols per
// stream per iteration, output as 16-byte stores every second iteration.
// The loop body has no branch, so the R streams interleave; a lane that met
// a code the table cannot resolve redoes the iteration from its saved state
// with fstep_slow (rare: codes longer than 14 bits, or corrupt data).
// wmax: the highest word index a stream may reach at an iteration start; a
// stream moves at most 16 words per iteration, into the zeroed guard.
template <int R, bool kQlc, bool kLong = false>
__device__ __forceinline__ void decode_group_fast(const DecJob &job, const DecTables &T, const uint32_t *words,
                                                  uint32_t wmax, uint64_t base, uint32_t g0,
                                                  const uint32_t (&st)[R], const uint32_t (&nb)[R], bool &bad)
{
    const uint16_t *dec = T.dec;
    const LongTable &lt = *T.lt;
    uint32_t vmax = 0;
    const int lane = threadIdx.x & 31;
    const uint32_t w_base = smem_u32(words);
    const uint32_t a_max = w_base + wmax * 4;
    FastStream s[R];
    uint8_t *dst[R];
    uint32_t q0[R], q1[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t w0 = min(st[r] >> 5, wmax);
        s[r].o = st[r] & 31;
        s[r].hi = bswap32(words[w0]);
        s[r].lo = bswap32(words[w0 + 1]);
        s[r].nx = bswap32(words[w0 + 2]);
        s[r].wa = w_base + (w0 + 3) * 4;
        dst[r] = job.out + base + (uint64_t)(g0 + (uint32_t)(r * 32 + lane)) * job.S;
        q0[r] = q1[r] = 0;
    }
    // Long-code mode (table-decoded codes; the same in every lane of the
    // warp): after an iteration in which some lane met a code longer than
    // the first-level table, the next one decodes a code at a time through
    // both table levels instead of two codes a step through the first,
    // until an iteration takes no code from the second level.  Chunks whose
    // data meets a codebook's long codes often (a codebook fitted to other
    // data) then skip the fast attempt that the redo would discard.
    bool lmode = false;
    for (uint32_t i = 0; i < job.S; i += 8) {
        FastStream s0[R];
        uint32_t a[R], b[R], emin[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            s[r].wa = min(s[r].wa, a_max);
            s0[r] = s[r];
            a[r] = b[r] = 0;
            emin[r] = ~0u;
        }
        bool long2 = false; // some code of this lane took the second level
        const bool was_long = !kQlc && kLong && lmode;
        if (was_long) {
            const SubHdr sh{lt.sub_p0, lt.sub_np, lt.sub_kb};
#pragma unroll
            for (int t = 0; t < 8; ++t)
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t e = fstep_long(s[r], dec, lt, sh, emin[r], long2);
                    if (t < 4)
                        a[r] = __byte_perm(a[r], e, 0x4321);
                    else
                        b[r] = __byte_perm(b[r], e, 0x4321);
                }
        } else {
            uint32_t h[R][4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int r = 0; r < R; ++r)
                    h[r][t] = kQlc ? qstep2(s[r], T, vmax) : fstep2(s[r], dec, emin[r]);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                a[r] = __byte_perm(h[r][0], h[r][1], 0x5410);
                b[r] = __byte_perm(h[r][2], h[r][3], 0x5410);
            }
        }
        uint32_t esc = 0; // streams of this lane that met an unresolved code
#pragma unroll
        for (int r = 0; r < R; ++r)
            esc |= (!kQlc && emin[r] == 0) ? (1u << r) : 0u;
        // (fast mode: the one vote, as before long-code mode existed)
        const bool any_esc = !kQlc && __any_sync(~0u, esc != 0);
        if (!kQlc && kLong)
            lmode = was_long ? __any_sync(~0u, esc != 0 || long2) : any_esc;
        if (any_esc) {
            // the lane's streams that met one, from their saved states, a
            // code at a time (one stream after the other: interleaving the
            // streams was slower, for the long-code chunks and the rest)
            const SubHdr sh{lt.sub_p0, lt.sub_np, lt.sub_kb};
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (!(esc & (1u << r)))
                    continue;
                s[r] = s0[r];
                a[r] = b[r] = 0;
#pragma unroll 1
                for (int t = 0; t < 8; ++t) {
                    const uint32_t e = fstep_redo(s[r], dec, lt, sh, bad);
                    if (t < 4)
                        a[r] = __byte_perm(a[r], e, 0x4321);
                    else
                        b[r] = __byte_perm(b[r], e, 0x4321);
                }
            }
        }
#ifdef ECC_CHECKED
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (s[r].wa > a_max + 16u * 4u) // past the guard the stage keeps after wmax
                set_status(job.status, ECC_ERR_CHECK);
#endif
        if (i & 8) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
#ifdef ECC_CHECKED
                if (dst[r] + i + 8 > job.out + job.n) {
                    set_status(job.status, ECC_ERR_CHECK);
                    continue;
                }
#endif
                st_stream16(dst[r] + i - 8, make_uint4(q0[r], q1[r], a[r], b[r]));
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            q0[r] = a[r];
            q1[r] = b[r];
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
        if ((s[r].wa - w_base) / 4 * 32 - 96 + s[r].o - st[r] != nb[r]) // position = (word of hi) * 32 + o
            bad = true;
    if (kQlc && vmax > 255)
        bad = true;
}

// Any other sub-block (the tensor's last, partial chunk, or a chunk read
// straight from global memory): one symbol at a time, byte stores.
// Returns true if the stream was inconsistent.
template <bool kShared>
static __device__ __noinline__ bool decode_stream_generic(const uint32_t *words, uint32_t wlast, uint32_t start,
                                                          uint32_t cnt, uint32_t expect, uint8_t *dst,
                                                          const uint16_t *dec, const LongTable &lt)
{
    bool bad = false;
    uint32_t emin = ~0u;
    Stream s;
    stream_start<kShared>(s, words, wlast, start);
    for (uint32_t i = 0; i < cnt; ++i)
        dst[i] = (uint8_t)step<kShared, true>(s, words, wlast, dec, lt, bad, emin);
    return bad || stream_pos(s) - start != expect;
}

constexpr uint32_t kDecTableBytes = sizeof(((ecc_codebook *)0)->dec);
constexpr uint32_t kLongTableBytes = (sizeof(LongTable) + 15u) & ~15u;
constexpr uint32_t kDecBarSlots = 24; // one mbarrier per warp
constexpr uint32_t kQlcSharedBytes = (sizeof(QlcShared) + 15u) & ~15u;
constexpr uint32_t kDecHeadBytes = kDecTableBytes + kLongTableBytes + kQlcSharedBytes + kDecBarSlots * 8;

// Per-warp staging state: the chunk buffer, its mbarrier and phase.
struct WarpStage {
    uint32_t *buf;
    uint32_t bytes; // capacity
    uint64_t *bar;
    uint32_t phase;
};

__device__ __forceinline__ bool chunk_range_ok(const DecJob &job, uint64_t c, uint64_t &b0, uint64_t &b1)
{
    b0 = job.chunk_off[c];
    b1 = job.chunk_off[c + 1];
    return b1 > b0 && b1 <= job.in_bytes && !((b0 | b1) & 15) && (b1 - b0) <= (uint64_t)job.C * 8;
}

// End of a chunk's stream after its last code at bit `carry`: the chunk's
// size must be the stream padded to 16 bytes, and the padding zero bits (read
// from global memory by lane 0).  Returns true if not (lane 0's answer;
// skipped when the stream is already known bad).
__device__ __forceinline__ bool chunk_tail_bad(const DecJob &job, uint64_t b0, uint32_t bytes, uint32_t carry,
                                               bool known_bad)
{
    bool bad = pad16((carry + 7) / 8) != bytes;
    if (!bad && !known_bad && (threadIdx.x & 31) == 0) {
        const uint32_t *words = reinterpret_cast<const uint32_t *>(job.in + b0);
        for (uint32_t wi = carry >> 5; wi < bytes / 4; ++wi) {
            uint32_t w = bswap32(__ldg(words + wi));
            if (wi == (carry >> 5))
                w &= 0xFFFFFFFFu >> (carry & 31);
            bad |= w != 0;
        }
    }
    return bad;
}

// Sub-blocks [g_begin, g_end) of a chunk (a multiple of 32, all full) too big
// for the warp's stage: stage and decode them 32 sub-blocks at a time (one
// stream per lane); each group's bytes fit, since a stage holds at least 32
// sub-blocks at the longest fast code lengths.  carry0: the chunk's bits
// before g_begin; `last`: the range ends the chunk, so its end is checked
// against the chunk's size and zero padding.
template <bool kQlc, bool kLong = false>
static __device__ __noinline__ void decode_chunk_in_groups(const DecJob &job, const DecTables &T, WarpStage &ws,
                                                           uint64_t base, uint32_t g_begin, uint32_t g_end,
                                                           uint64_t sub0, uint64_t b0, uint32_t bytes,
                                                           uint32_t carry0, bool last)
{
    const uint16_t *dec = T.dec;
    const LongTable &lt = *T.lt;
    const int lane = threadIdx.x & 31;
    bool bad = false;
    uint32_t carry = carry0; // bits of the chunk's earlier groups
    for (uint32_t g0 = g_begin; g0 < g_end; g0 += 32) {
        const uint32_t v = job.sub_bits[sub0 + g0 + lane];
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(~0u, incl, o);
            incl += lane >= o ? y : 0u;
        }
        const uint32_t gbits = __shfl_sync(~0u, incl, 31);
        // the group's bytes, widened to 16-byte boundaries of the chunk
        const uint32_t s0 = (carry >> 3) & ~15u;
        const uint32_t s1 = min(pad16((carry + gbits + 7) >> 3), bytes);
        if (carry + gbits > bytes * 8u || gbits == 0) { // sub_bits claim more bits than the chunk holds, or none
            bad = true;
            break;
        }
        if (s1 - s0 + kStageGuard > ws.bytes) {
            // long codes: the group does not fit either; read it from global memory
            bad |= decode_stream_generic<false>(reinterpret_cast<const uint32_t *>(job.in + b0), bytes / 4 - 1,
                                                carry + incl - v, job.S, v,
                                                job.out + base + (uint64_t)(g0 + lane) * job.S, dec, lt);
            carry += gbits;
            continue;
        }
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async();
            mbar_expect_tx(ws.bar, s1 - s0);
            bulk_g2s(ws.buf, job.in + b0 + s0, s1 - s0, ws.bar);
        }
        bool ok = __all_sync(~0u, mbar_wait(ws.bar, ws.phase, kWaitLimitNs));
        if (!ok) // never expected: the copy reads valid memory; wait once more
            ok = __all_sync(~0u, mbar_wait(ws.bar, ws.phase, kWaitLimitNs));
        ws.phase ^= 1;
        if (!ok) {
            if (lane == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            ws.buf = nullptr; // the copy may still land: stop using this buffer
            return;
        }
        if (lane < kStageGuard / 4)
            ws.buf[(s1 - s0) / 4 + lane] = 0; // guard: reads past the end see 0
        __syncwarp();
        const uint32_t st[1] = {carry + incl - v - s0 * 8u}, nb[1] = {v};
        decode_group_fast<1, kQlc, kLong>(job, T, ws.buf, (s1 - s0) / 4 + 4, base, g0, st, nb, bad);
        carry += gbits;
    }
    if (last)
        bad |= chunk_tail_bad(job, b0, bytes, carry, bad);
    if (__any_sync(~0u, bad) && lane == 0)
        set_status(job.status, ECC_ERR_CORRUPT);
    __syncwarp();
}

// Decode chunk c with one warp.  The compressed chunk is staged into the
// warp's shared buffer by one bulk copy (when it fits), while the lanes scan
// sub_bits; next_c (if valid) is prefetched into L2 for the warp's next call.
template <int R, bool kQlc, bool kLong = false>
__device__ __forceinline__ void decode_chunk(const DecJob &job, const DecTables &T, WarpStage &ws, uint64_t c,
                                             uint64_t next_c, uint64_t n_chunks)
{
    const uint16_t *dec = T.dec;
    const LongTable &lt = *T.lt;
    const int lane = threadIdx.x & 31;
    const uint64_t base = c * job.C;
    const uint32_t L = (uint32_t)min((uint64_t)job.C, job.n - base);
    const uint32_t s_shift = 31 - __clz(job.S); // S is a power of two
    const uint32_t nsub = (L + job.S - 1) >> s_shift;
    const uint64_t sub0 = base >> s_shift;
    uint64_t b0, b1;
    if (!chunk_range_ok(job, c, b0, b1)) {
        if (lane == 0)
            set_status(job.status, ECC_ERR_CORRUPT);
        return;
    }
    const uint32_t bytes = (uint32_t)(b1 - b0);
    const bool staged = ws.buf != nullptr && bytes + kStageGuard <= ws.bytes;
    if (!staged && ws.buf != nullptr && L == job.C && nsub >= 32 && (nsub & 31) == 0) {
        decode_chunk_in_groups<kQlc, kLong>(job, T, ws, base, 0, nsub, sub0, b0, bytes, 0, true);
        return;
    }
    if (staged) {
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async();
            mbar_expect_tx(ws.bar, bytes);
            bulk_g2s(ws.buf, job.in + b0, bytes, ws.bar);
        }
    }
    if (lane == 0 && next_c < n_chunks) {
        uint64_t n0, n1;
        if (chunk_range_ok(job, next_c, n0, n1))
            prefetch_l2(job.in + n0, (uint32_t)(n1 - n0));
    }
    const uint32_t *words;
    uint32_t wlast;
    if (staged) {
        bool ok = __all_sync(~0u, mbar_wait(ws.bar, ws.phase, kWaitLimitNs));
        if (!ok) // never expected: the copy reads valid memory; wait once more
            ok = __all_sync(~0u, mbar_wait(ws.bar, ws.phase, kWaitLimitNs));
        ws.phase ^= 1;
        if (!ok) {
            if (lane == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            ws.buf = nullptr; // the copy may still land: stop using this buffer
            return;
        }
        if (lane < kStageGuard / 4)
            ws.buf[bytes / 4 + lane] = 0; // guard: reads past the end see 0
        __syncwarp();
        words = ws.buf;
        wlast = bytes / 4 + kStageGuard / 4 - 1;
    } else {
        words = reinterpret_cast<const uint32_t *>(job.in + b0);
        wlast = bytes / 4 - 1;
    }

    bool bad = false;
    uint32_t carry = 0;
    for (uint32_t g0 = 0; g0 < nsub; g0 += 32 * R) {
        uint32_t st[R], nb[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t k = g0 + (uint32_t)(r * 32 + lane);
            const uint32_t v = k < nsub ? job.sub_bits[sub0 + k] : 0u;
            uint32_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(~0u, incl, o);
                if (lane >= o)
                    incl += y;
            }
            st[r] = carry + incl - v;
            nb[r] = v;
            carry += __shfl_sync(~0u, incl, 31);
        }
        // the hot loop needs every lane to own R full sub-blocks
        if (staged && L == job.C && nsub - g0 >= 32u * R) {
            const uint32_t wmax = bytes / 4 + 4; // + up to 2 words per step x 8 steps < guard
            decode_group_fast<R, kQlc, kLong>(job, T, words, wmax, base, g0, st, nb, bad);
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t k = g0 + (uint32_t)(r * 32 + lane);
                if (k * job.S >= L)
                    continue;
                const uint32_t cnt = min(job.S, L - k * job.S);
                uint8_t *dst = job.out + base + (uint64_t)k * job.S;
                bad |= staged ? decode_stream_generic<true>(words, wlast, st[r], cnt, nb[r], dst, dec, lt)
                              : decode_stream_generic<false>(words, wlast, st[r], cnt, nb[r], dst, dec, lt);
            }
        }
    }
    if (pad16((carry + 7) / 8) != bytes)
        bad = true;
    // the padding after the last code must be zero bits
    if (!bad && lane == 0) {
        for (uint32_t wi = carry >> 5; wi < bytes / 4; ++wi) {
            uint32_t w = bswap32(staged ? words[wi] : __ldg(words + wi));
            if (wi == (carry >> 5))
                w &= 0xFFFFFFFFu >> (carry & 31);
            bad |= w != 0;
        }
    }
    if (__any_sync(~0u, bad) && lane == 0)
        set_status(job.status, ECC_ERR_CORRUPT);
    __syncwarp();
}

// Decode piece `piece` of chunk c with one warp: the sub-blocks [piece * ps,
// (piece + 1) * ps) of the chunk, ps = (C / S) >> pshift (32 * R of them in a
// full piece).  Splitting a large chunk into pieces lets each warp stage
// only a piece, so that as many warps fit an SM as for a small chunk.  The
// piece starts at the sum of the chunk's sub_bits before it; its bytes,
// widened to 16-byte boundaries of the chunk, are staged by one bulk copy
// when they fit.  The piece that ends the chunk also checks the chunk's size
// and zero padding.
template <int R, bool kQlc, bool kLong = false>
__device__ __forceinline__ void decode_piece(const DecJob &job, const DecTables &T, WarpStage &ws, uint64_t c,
                                             uint32_t piece, uint32_t pshift)
{
    const uint16_t *dec = T.dec;
    const LongTable &lt = *T.lt;
    const int lane = threadIdx.x & 31;
    const uint64_t base = c * job.C;
    const uint32_t L = (uint32_t)min((uint64_t)job.C, job.n - base);
    const uint32_t s_shift = 31 - __clz(job.S); // S is a power of two
    const uint32_t nsub = (L + job.S - 1) >> s_shift;
    const uint32_t ps = (job.C >> s_shift) >> pshift;
    const uint32_t g_begin = piece * ps;
    if (g_begin >= nsub) // past the end of the tensor's last, partial chunk
        return;
    const uint32_t g_end = min(g_begin + ps, nsub);
    const bool last = g_end == nsub;
    const uint64_t sub0 = base >> s_shift;
    uint64_t b0, b1;
    if (!chunk_range_ok(job, c, b0, b1)) {
        if (lane == 0)
            set_status(job.status, ECC_ERR_CORRUPT);
        return;
    }
    const uint32_t bytes = (uint32_t)(b1 - b0);
    // (no L2 prefetch of the next piece: estimated from the chunk's size, it
    // fetched about a sixth of the payload twice and saved no time)
    // the chunk's bits before the piece
    uint32_t carry0 = 0;
    for (uint32_t k = (uint32_t)lane; k < g_begin; k += 32)
        carry0 += job.sub_bits[sub0 + k];
#pragma unroll
    for (int o = 16; o; o >>= 1)
        carry0 += __shfl_xor_sync(~0u, carry0, o);
    // the piece's streams: lane l runs sub-blocks g_begin + r * 32 + l
    uint32_t st[R], nb[R];
    uint32_t carry = carry0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t k = g_begin + (uint32_t)(r * 32 + lane);
        const uint32_t v = k < g_end ? job.sub_bits[sub0 + k] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(~0u, incl, o);
            if (lane >= o)
                incl += y;
        }
        st[r] = carry + incl - v;
        nb[r] = v;
        carry += __shfl_sync(~0u, incl, 31);
    }
    if ((uint64_t)carry > (uint64_t)bytes * 8u || carry == carry0) { // more bits than the chunk holds, or none
        if (lane == 0)
            set_status(job.status, ECC_ERR_CORRUPT);
        return;
    }
    // every stream of a full piece is a full sub-block
    const bool full = g_end - g_begin == 32u * R && g_end * job.S <= L;
    const uint32_t s0 = (carry0 >> 3) & ~15u;
    const uint32_t s1 = min(pad16((carry + 7) >> 3), bytes);
    const bool staged = ws.buf != nullptr && s1 - s0 + kStageGuard <= ws.bytes;
    if (!staged && ws.buf != nullptr && full && ((g_end - g_begin) & 31) == 0) {
        decode_chunk_in_groups<kQlc, kLong>(job, T, ws, base, g_begin, g_end, sub0, b0, bytes, carry0, last);
        return;
    }
    const uint32_t *words;
    uint32_t wlast, off = 0; // off: the stage's first bit in the chunk
    if (staged) {
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async();
            mbar_expect_tx(ws.bar, s1 - s0);
            bulk_g2s(ws.buf, job.in + b0 + s0, s1 - s0, ws.bar);
        }
        bool ok = __all_sync(~0u, mbar_wait(ws.bar, ws.phase, kWaitLimitNs));
        if (!ok) // never expected: the copy reads valid memory; wait once more
            ok = __all_sync(~0u, mbar_wait(ws.bar, ws.phase, kWaitLimitNs));
        ws.phase ^= 1;
        if (!ok) {
            if (lane == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            ws.buf = nullptr; // the copy may still land: stop using this buffer
            return;
        }
        if (lane < kStageGuard / 4)
            ws.buf[(s1 - s0) / 4 + lane] = 0; // guard: reads past the end see 0
        __syncwarp();
        words = ws.buf;
        wlast = (s1 - s0) / 4 + kStageGuard / 4 - 1;
        off = s0 * 8u;
    } else {
        words = reinterpret_cast<const uint32_t *>(job.in + b0);
        wlast = bytes / 4 - 1;
    }
    bool bad = false;
#pragma unroll
    for (int r = 0; r < R; ++r)
        st[r] -= off;
    if (staged && full) {
        decode_group_fast<R, kQlc, kLong>(job, T, words, (s1 - s0) / 4 + 4, base, g_begin, st, nb, bad);
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t k = g_begin + (uint32_t)(r * 32 + lane);
            if (k >= g_end)
                continue;
            const uint32_t cnt = min(job.S, L - k * job.S);
            uint8_t *dst = job.out + base + (uint64_t)k * job.S;
            bad |= staged ? decode_stream_generic<true>(words, wlast, st[r], cnt, nb[r], dst, dec, lt)
                          : decode_stream_generic<false>(words, wlast, st[r], cnt, nb[r], dst, dec, lt);
        }
    }
    if (last)
        bad |= chunk_tail_bad(job, b0, bytes, carry, bad);
    if (__any_sync(~0u, bad) && lane == 0)
        set_status(job.status, ECC_ERR_CORRUPT);
    __syncwarp();
}

} // namespace ecc
