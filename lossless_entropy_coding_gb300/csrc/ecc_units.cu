// ecc_units.cu -- the unit encoder: a tensor coded in units of 16384
// consecutive symbols (one chunk of 16384, 2..16 whole smaller chunks, or a
// quarter or half of a chunk of 65536 or 32768), the codewords of each chunk
// packed at their final places in a shared stage and the unit's payload
// written with one bulk copy.
//
// The coding follows "Quad Length Codes for Lossless Compression of e4m3",
// section 2 "Codifica" (a table gives each byte its code; codes are written
// one after the other), and "Single-Stage Huffman Encoder for ML
// Compression", Methodology step 4 (the precomputed codebook is applied with
// no analysis of the tensor).  Chunk offsets, sub-block bit counts and the
// padding are the library's container (include/ecc.h).
//
// A CTA is one pipeline: 16 compute warps, a loader warp and a storer warp;
// two CTAs run on an SM.
//  * compute thread t of a unit owns symbols [32 t, 32 t + 32).  Phase A sums
//    its 32 code lengths from a 256-byte shared length table (one byte-sized
//    load a symbol, at the byte value rotated by one bit).
//  * phase B: a warp scan of the counts and one barrier over the compute
//    warps give every thread its bit position inside its chunk, every chunk
//    its padded place in the unit, and the unit its padded size, which is
//    published at once for the decoupled look-back over units; sub-block bit
//    counts are written here.
//  * phase C: each thread reads its 32 bytes again, looks them up in a
//    16-way replicated shared table of {code << (32 - len), 2^(32 - len)},
//    joins them into 16 code pairs (v1 + hi32(v2 * q1), hi32(q1 * q2)) and
//    appends the pairs at their final bit positions in the stage (two wide
//    multiplies an append, a predicated store of each completed word,
//    byte-swapped to memory order).  A word two threads share
//    is stored by the later one: the earlier passes its last partial word on
//    with a shuffle (across warps, through the storer).
//  * the loader warp claims units in ticket order as phase C frees an input
//    buffer and bulk-copies their input; the storer warp resolves each unit's
//    offset from its predecessors' published sizes while the compute warps
//    pack it, writes chunk_off and total_bits, finishes the words shared
//    across warps and the chunks' zero padding, and stores the stage to the
//    output with one cp.async.bulk shared -> global copy.
// A unit whose payload outgrows the stage (long codes only) is sized and
// placed like any other and marked in its look-back word; a second kernel
// (the deferred pass) codes it, a warp a unit, from the codebook in global
// memory.
//
// Chunks of more than 16384 symbols (split chunks) are coded a unit at a
// time, units of one chunk running on different CTAs at once.  The look-back
// runs over chunks: each unit adds its bit count to its chunk's word in
// phase B, and the unit that completes the count publishes the chunk's
// padded size there.  Inside a chunk a unit starts at any bit.  Its compute
// warps pack it from bit 0 of the stage, without waiting for anything; its
// storer learns the bit counts of the chunk's earlier units (published in
// their phase B, a word a unit) and writes the stage shifted to that bit:
// the words that are wholly the unit's (16-byte stores in the middle, single
// words at either end).  Two consecutive units of a chunk share a word (the
// earlier one's last bits, the later one's first): each ors its part into
// the earlier unit's word with one atomic, and the one that comes second
// writes the whole word.  The chunk's last unit pads the chunk; a chunk with
// a unit too long to stage is marked and left whole to the deferred pass.
//
// Many tensors at once (every tensor with chunks of 16384 symbols): the same
// pipeline over an item map, a chunk a unit.  The loader resolves each unit
// it claims into a shared record (its tensor's job, its chunk, the codebook
// check, the completion stamp) and fills the slot's length table; the
// compute warps reload the code table after the phase-B barrier of a unit
// whose codebook differs; the look-back runs over the unit's tensor.  The
// units too long to stage are listed, and a second launch of the pipeline,
// one CTA an SM with stages of up to 32 bits a symbol, codes them at the
// places the first gave them.

#include <algorithm>

#include "ecc_device.cuh"
#include "ecc_launch.h"

namespace ecc {

constexpr uint32_t kUSyms = kUnitSyms;               // symbols of a unit
constexpr uint32_t kUThr = 32;                       // symbols of a compute thread
constexpr uint32_t kUWarps = kUSyms / (32 * kUThr);  // compute warps (16)
constexpr uint32_t kUCompute = 32 * kUWarps;         // compute threads (512)
constexpr uint32_t kUThreads = kUCompute + 64;       // + the loader and the storer
constexpr uint64_t kUEnd = ~0ull;                    // slot holds no unit: the pipeline ends
constexpr uint32_t kULutBytes = kLutRows * kLutReplicas * 8u;
constexpr uint32_t kUBarCompute = 1;                 // named barrier of the compute warps
constexpr uint32_t kUBarTables = 2;                  // ... around a reload of the code tables
// what a unit holds: a whole chunk, whole smaller chunks, or part of a chunk
constexpr int kUnitOne = 0, kUnitGroup = 1, kUnitSplit = 2;
// Word of a unit of a split chunk that is not the chunk's last: kFlagAggregate
// | bits once sized (bits 0..20); then the word the unit shares with the
// next one (memory order, bits 21..52), or-ed in by both, with a bit for
// each that has (kHandPrev: this unit, kHandNext: the next).  The word of a
// chunk's last unit is the chunk's deferred mark (kMarkDeferred: some unit
// of the chunk could not be staged).
constexpr uint32_t kUBitsShift = 21;
constexpr uint64_t kUBitsMask = (1ull << kUBitsShift) - 1;
constexpr uint64_t kHandPrev = 1ull << 53, kHandNext = 1ull << 54;
constexpr uint64_t kMarkDeferred = 1;
// A split chunk's look-back word before it is published (state 0): the
// units sized so far (<< kUCountShift) and their bits.  Every later change
// of the word raises it (atomicMax): the size (by the unit counted last,
// after its count, so a published size means every unit is counted), the
// inclusive prefix, the deferred mark.
constexpr uint32_t kUCountShift = 32;
static_assert((uint64_t)kUSyms * ECC_MAX_CODE_LEN <= kUBitsMask, "a unit's bit count fits its field");
// Stage bytes a unit of a split chunk needs: its words from bit 0, and 8
// words more that the storer clears and reads past them when it shifts the
// unit to its bit in the output (the shifted unit spans at most 4 words more,
// and its 16-byte blocks are read whole).
__host__ __device__ constexpr uint32_t split_stage_bytes(uint32_t bits) { return (bits + 31u) / 32u * 4u + 32u; }
static_assert(kUWarps == 16, "phase B scans the warp totals over the lanes of one half-warp");

// Shared state of the pipeline.  Slot s = k % 2 of the CTA's k-th unit holds
// its input buffer and its stage; the per-unit records the storer reads, and
// the mbarrier that hands them over, are kept four deep (k % 4): the compute
// warps may size unit k + 2 before the storer, busy with unit k's look-back,
// has taken unit k's records (at the start, when both stages are free), but
// never unit k + 4.
struct UPipe {
    uint64_t full[2];      // input buffer s filled: one arrival (loader) + the copy's bytes
    uint64_t st_free[2];   // stage s read by its bulk store: one arrival (storer)
    uint64_t agg[4];       // unit k sized and published: one arrival (compute thread 0), in agg[k % 4]
    uint64_t done[2];      // unit of slot s packed (its input read, its stage written): one arrival per compute thread
    uint64_t unit[2];      // loader -> compute: unit of slot s, or kUEnd
    uint64_t sunit[4];     // compute -> storer: unit k, or kUEnd
    uint32_t wtot[4][kUWarps];  // compute -> storer: bit totals of the compute warps of unit k
    uint32_t wtail[2][kUWarps]; // lane 31's last partial word (stage word order) when the next warp continues its chunk
};
static_assert(sizeof(UPipe) % 16 == 0, "buffers stay 16-byte aligned");

struct UnitParams {
    EncJob job;
    uint64_t n_units;
    uint64_t *uflags;     // split chunks: a word per unit (job.flags holds a word per chunk)
    uint32_t mlog;        // split chunks: log2 of the units of a chunk
    uint32_t *ticket;
    uint32_t stage_bytes; // payload bytes a stage holds (multiple of 16)
    uint64_t timeout_ns;
    // Many-tensor launch (chunks of kUSyms symbols, a unit each): unit k is
    // chunk items[k] & 0xFFFFFFFF of tensor items[k] >> 32; job.flags holds
    // a look-back word per unit, job.status receives the errors of waits
    // that end before their unit is known; done counts each tensor's coded
    // segments for its completion stamp; *t_start (may be null) is stamped
    // at the start.
    const uint64_t *items;
    const ecc_desc *descs;
    uint32_t *done;
    uint64_t *t_start;
    // the units the first pass sized and placed but could not stage (their
    // positions, *n_deferred of them), coded by the second pass
    uint32_t *deferred;
    uint32_t *n_deferred;
};

// Unit k of a many-tensor launch: its chunk as a job of its own (look-back
// words offset to its tensor's), the chunk's index in its tensor, and the
// tensor's.
struct UItem {
    EncJob job;
    uint64_t c;
    uint32_t tensor;
};
__device__ __forceinline__ UItem unit_item(const UnitParams &p, uint64_t k)
{
    const uint64_t it = p.items[k];
    const uint32_t t = (uint32_t)(it >> 32);
    const uint64_t c = it & 0xFFFFFFFFull;
    const ecc_desc &d = p.descs[t];
    return UItem{EncJob{d.in, d.n, d.cb, d.C, d.S, d.out, d.cap, d.chunk_off, d.sub_bits, d.total_bits,
                        p.job.flags + (k - c), d.status},
                 c, t};
}

// A many-tensor launch's unit as the loader resolves it when it claims the
// unit (the CTA's k-th unit in recs[k % 4], the depth of the storer's
// records): the compute warps and the storer then start the unit without
// dependent global loads.  The loader claims unit k + 4 only once the
// storer is past unit k (see the UPipe records).
struct UUnitRec {
    EncJob job;
    uint64_t c;        // the unit's chunk in its tensor
    uint64_t *t_done;  // the tensor's completion stamp (may be null)
    uint32_t tensor;
    uint32_t cb_ok;    // the codebook is valid
};
constexpr uint32_t kURecs = 4;

// The job of the CTA's unit with record slot r: the launch's, or (a
// many-tensor launch) the record's in shared memory.
template <bool kBatch>
__device__ __forceinline__ const EncJob &unit_job(const UnitParams &p, const UUnitRec *recs, uint32_t r)
{
    if constexpr (kBatch)
        return recs[r].job;
    else
        return p.job;
}

__device__ __forceinline__ bool codebook_ok(const ecc_codebook *cb)
{
    return cb->magic == ECC_CODEBOOK_MAGIC && cb->max_len <= ECC_MAX_CODE_LEN;
}

__host__ __device__ constexpr size_t unit_smem_bytes(uint32_t stage_bytes)
{
    return kULutBytes + sizeof(UPipe) + 2u * kUSyms + 2u * (size_t)stage_bytes;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// expected transaction bytes without an arrival (the arrival follows)
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// the stage may be reused once every bulk store has read it
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// predicated shared store (one instruction, no branch)
__device__ __forceinline__ void st_shared_pred(uint32_t addr, uint32_t v, bool p)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.shared.b32 [%0], %1;\n\t}" ::"r"(addr), "r"(v),
                 "r"((uint32_t)p)
                 : "memory");
}

// predicated shared or-reduction
__device__ __forceinline__ void red_or_pred(uint32_t addr, uint32_t v, bool p)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q red.shared.or.b32 [%0], %1;\n\t}" ::"r"(addr),
                 "r"(v), "r"((uint32_t)p)
                 : "memory");
}

// predicated shared 64-bit store, mbarrier arrival, relaxed global store and
// 16-bit global store (single instructions under a predicate, no branch)
__device__ __forceinline__ void st_shared_u64_pred(void *addr, uint64_t v, bool p)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.shared.u64 [%0], %1;\n\t}" ::"r"(smem_u32(addr)),
                 "l"(v), "r"((uint32_t)p)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_pred(uint64_t *bar, bool p)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t@q mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"((uint32_t)p)
                 : "memory");
}
__device__ __forceinline__ void st_relaxed_pred(uint64_t *addr, uint64_t v, bool p)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.relaxed.gpu.global.u64 [%0], %1;\n\t}" ::"l"(addr),
                 "l"(v), "r"((uint32_t)p)
                 : "memory");
}
__device__ __forceinline__ void st_global_u16_pred(uint16_t *addr, uint32_t v, bool p)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.u16 [%0], %1;\n\t}" ::"l"(addr),
                 "h"((uint16_t)v), "r"((uint32_t)p)
                 : "memory");
}

// index of the highest set bit, 0xFFFFFFFF for 0
__device__ __forceinline__ uint32_t bfind(uint32_t x)
{
    uint32_t r;
    asm("bfind.u32 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// inclusive scan over the 32 lanes (shfl.up with its in-range predicate)
__device__ __forceinline__ uint32_t warp_incl(uint32_t x)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y;
        asm volatile("{\n\t.reg .pred p;\n\tshfl.sync.up.b32 %0|p, %1, %2, 0, -1;\n\t@!p mov.b32 %0, 0;\n\t}"
                     : "=r"(y)
                     : "r"(x), "r"(o));
        x += y;
    }
    return x;
}

// inclusive scan over lanes 0..15 (lanes 16..31 get sums of their own half)
__device__ __forceinline__ uint32_t half_incl(uint32_t x)
{
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
        uint32_t y;
        asm volatile("{\n\t.reg .pred p;\n\tshfl.sync.up.b32 %0|p, %1, %2, 0, -1;\n\t@!p mov.b32 %0, 0;\n\t}"
                     : "=r"(y)
                     : "r"(x), "r"(o));
        x += y;
    }
    return x;
}

// barrier over the compute warps that also returns the OR of p over them
__device__ __forceinline__ bool compute_bar_or(bool p)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\tbar.red.or.pred b, %2, %3, a;\n\t"
                 "selp.u32 %0, 1, 0, b;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)p), "n"(kUBarCompute), "n"(kUCompute)
                 : "memory");
    return r != 0;
}

// Bit count of the 32 bytes of (a, b) coded one code at a time from the
// lane's table replica (a thread with a pair longer than 32 bits); bit 31 set
// when some byte has no code of at most 31 bits in the table (the exact path
// from the codebook must code the thread).
static __device__ __noinline__ uint32_t unit_bits_single(const uint2 *lt, uint4 a, uint4 b)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t f = 0, fo = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t ff = bfind(lt[byte_of(w[j >> 2], j & 3) * kLutReplicas].y); // 32 - length, or ~0
        f += ff;
        fo |= ff;
    }
    return (fo >> 31) ? 1u << 31 : 32u * 32u - f;
}

// End state of a thread's packing: its last partial word (register order,
// first bit in bit 31; 0 when the thread ended on a word boundary) and the
// shared-window address of the word that holds it (else of the next word).
struct UEnd {
    uint32_t tail, addr;
    bool partial; // tail holds 1..31 bits (it may still be all zeros)
};

#ifdef ECC_CHECKED
// index-checked builds: a stage store at or past lim is skipped and reported
__device__ __forceinline__ void ust(uint32_t addr, uint32_t v, uint32_t lim, bool &bad)
{
    if (addr + 4u > lim) {
        bad = true;
        return;
    }
    st_shared_u32(addr, v);
}
#endif

// Packer of codes given as (v, q): v = code << (32 - l) (first bit in bit
// 31), q = 2^(32 - l), l <= 32.  State: the partial word cur (its first nb
// bits used, 1 <= nb <= 32, first bit in bit 31) at shared address addr, K =
// 2^(32 - nb).  Appending (v, q): v * K + (cur << 32) holds cur completed by
// v's leading bits in its high word and v's remaining bits in its low word;
// K * q = 2^(64 - nb - l) has a zero high word exactly when the word filled
// up (it is then stored, byte-swapped to memory order unless kSwap is
// false, and the low word becomes the partial one) and holds the next K in
// whichever word is non-zero.  The store, the select and the address step
// are one predicated block (no branch).
template <bool kSwap>
__device__ __forceinline__ uint32_t word_order(uint32_t w) { return kSwap ? bswap32(w) : w; }

template <bool kSwap>
struct UPacker {
    uint32_t addr, cur, K, nb0;
#ifdef ECC_CHECKED
    uint32_t lim;
    bool bad = false;
#endif

    // position at bit pos of the stage; the first code follows with
    // start_pending: when pos is inside a word, its first nb0 bits belong to
    // an earlier thread (zeros here) and the code is appended to them; when
    // pos starts a word, the code is the partial word
    __device__ __forceinline__ void begin(uint32_t stage, uint32_t pos)
    {
        nb0 = pos & 31u;
        addr = stage + (pos >> 5) * 4u;
        cur = 0;
        K = 1u << ((32u - nb0) & 31u); // nb0 = 0: 1, as if a full word came first
    }
    __device__ __forceinline__ void start_pending(uint32_t v0, uint32_t q0)
    {
        const uint64_t x = (uint64_t)v0 * K;
        const uint64_t y = (uint64_t)K * q0;
        const uint32_t xhi = (uint32_t)(x >> 32), xlo = (uint32_t)x;
        const uint32_t yhi = (uint32_t)(y >> 32), ylo = (uint32_t)y;
        emit(xhi, xlo, nb0 ? yhi : 1u); // nb0 = 0: nothing to store, the word is v0
        cur = nb0 ? cur : v0;
        K = nb0 ? yhi + ylo : q0;
    }
    // begin + start_pending
    __device__ __forceinline__ void start(uint32_t stage, uint32_t pos, uint32_t v0, uint32_t q0)
    {
        begin(stage, pos);
        start_pending(v0, q0);
    }
    // the append's tail: the word w = cur completed by the code's leading
    // bits is stored when gate == 0 (it filled up), and the code's remaining
    // bits xlo become the partial word; else w stays the partial word
    __device__ __forceinline__ void emit(uint32_t xhi, uint32_t xlo, uint32_t gate)
    {
        const uint32_t w = xhi | cur;
#ifdef ECC_CHECKED
        if (gate == 0)
            ust(addr, word_order<kSwap>(w), lim, bad);
        cur = gate == 0 ? xlo : w;
        addr += gate == 0 ? 4u : 0u;
#else
        if (kSwap)
            asm volatile("{\n\t.reg .pred p;\n\t.reg .b32 s;\n\tsetp.eq.u32 p, %3, 0;\n\tprmt.b32 s, %2, 0, 0x0123;\n\t"
                         "@p st.shared.b32 [%0], s;\n\tselp.b32 %1, %4, %2, p;\n\t@p add.u32 %0, %0, 4;\n\t}"
                         : "+r"(addr), "=r"(cur)
                         : "r"(w), "r"(gate), "r"(xlo)
                         : "memory");
        else
            asm volatile("{\n\t.reg .pred p;\n\tsetp.eq.u32 p, %3, 0;\n\t"
                         "@p st.shared.b32 [%0], %2;\n\tselp.b32 %1, %4, %2, p;\n\t@p add.u32 %0, %0, 4;\n\t}"
                         : "+r"(addr), "=r"(cur)
                         : "r"(w), "r"(gate), "r"(xlo)
                         : "memory");
#endif
    }
    __device__ __forceinline__ void put(uint32_t v, uint32_t q)
    {
        const uint64_t x = (uint64_t)v * K;
        const uint64_t y = (uint64_t)K * q;
        emit((uint32_t)(x >> 32), (uint32_t)x, (uint32_t)(y >> 32));
        K = (uint32_t)(y >> 32) + (uint32_t)y;
    }
    // store a completed last word; the end state
    __device__ __forceinline__ UEnd finish()
    {
        const bool complete = K == 1u;
#ifdef ECC_CHECKED
        if (complete)
            ust(addr, word_order<kSwap>(cur), lim, bad);
#else
        st_shared_pred(addr, word_order<kSwap>(cur), complete);
#endif
        return complete ? UEnd{0u, addr + 4u, false} : UEnd{cur, addr, true};
    }
};

// The 32 bytes of (a, b) packed one code at a time from the lane's table
// replica (every code at most 31 bits).
template <bool kSwap>
static __device__ __noinline__ UEnd unit_pack_single(const uint2 *lt, uint32_t stage, uint32_t pos, uint4 a, uint4 b,
                                                     uint32_t lim, uint32_t *status)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    UPacker<kSwap> pk;
#ifdef ECC_CHECKED
    pk.lim = lim;
#endif
    const uint2 e0 = lt[byte_of(w[0], 0) * kLutReplicas];
    pk.start(stage, pos, e0.x, e0.y);
#pragma unroll
    for (int j = 1; j < 32; ++j) {
        const uint2 e = lt[byte_of(w[j >> 2], j & 3) * kLutReplicas];
        pk.put(e.x, e.y);
    }
    const UEnd e = pk.finish();
#ifdef ECC_CHECKED
    if (pk.bad)
        set_status(status, ECC_ERR_CHECK);
#endif
    return e;
}

// Slow-path packing of the cnt bytes of (a, b) at bit pos of the stage (codes
// from the codebook in global memory, up to ECC_MAX_CODE_LEN bits): the same
// word protocol.
template <bool kSwap>
static __device__ __noinline__ UEnd unit_pack_slow(uint32_t stage, uint32_t pos, uint4 a, uint4 b, uint32_t cnt,
                                                   const ecc_codebook *cb, uint32_t lim, uint32_t *status)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t addr = stage + (pos >> 5) * 4u;
    uint32_t nb = pos & 31u; // bits of the current word already used (by an earlier thread: zeros here)
    uint64_t acc = 0;        // the current word in bits 63..32, first bit in bit 63
    bool bad = false;
    auto put = [&](uint32_t code, uint32_t len) { // len <= 24
        acc |= (uint64_t)code << (64u - nb - len);
        nb += len;
        if (nb >= 32u) {
#ifdef ECC_CHECKED
            ust(addr, word_order<kSwap>((uint32_t)(acc >> 32)), lim, bad);
#else
            st_shared_u32(addr, word_order<kSwap>((uint32_t)(acc >> 32)));
#endif
            addr += 4u;
            acc <<= 32;
            nb -= 32u;
        }
    };
    bool nocode = false;
    for (uint32_t j = 0; j < cnt; ++j) {
        const uint32_t b8 = byte_of(w[j >> 2], j & 3);
        const uint32_t L = min((uint32_t)cb->len[b8], (uint32_t)ECC_MAX_CODE_LEN);
        if (!L) { // a byte the codebook does not code (its length counted 0 bits)
            nocode = true;
            continue;
        }
        const uint64_t code = cb->code[b8] & ((1ull << L) - 1);
        if (L > 24) {
            put((uint32_t)(code >> 24), L - 24);
            put((uint32_t)(code & 0xFFFFFFu), 24);
        } else {
            put((uint32_t)code, L);
        }
    }
    if (nocode)
        set_status(status, ECC_ERR_CODEBOOK);
    if (bad)
        set_status(status, ECC_ERR_CHECK);
    return UEnd{nb ? (uint32_t)(acc >> 32) : 0u, addr, nb != 0};
}

// Chunk layout of a unit from the compute warps' bit totals (x = total of
// warp `lane`, lanes 0..15; wpc warps per chunk): for lane l, E = bits of
// its chunk before warp l, base = byte offset of its chunk in the unit's
// stage, cbits = its chunk's bits (valid on the chunk's last lane), Y =
// inclusive sum of padded chunk sizes (lane 15: the unit's bytes).
struct ULayout {
    uint32_t E, base, cbits, Y;
};
template <bool kOne>
__device__ __forceinline__ ULayout unit_layout(uint32_t x, uint32_t lane, uint32_t wpc)
{
    ULayout o;
    const uint32_t X = half_incl(x);
    if (kOne) {
        o.E = X - x;
        o.base = 0;
        o.cbits = X;
        o.Y = (X + 127u) / 128u * 16u;
        return o;
    }
    const uint32_t sl = lane & ~(wpc - 1u);                    // first lane of this lane's chunk
    const uint32_t xp = __shfl_sync(~0u, X, (sl + 31u) & 31u); // inclusive total before the chunk
    const uint32_t before = sl ? xp : 0u;
    o.E = X - x - before;
    o.cbits = X - before;
    const bool last = (lane & (wpc - 1u)) == wpc - 1u && lane < kUWarps;
    o.Y = half_incl(last ? (o.cbits + 127u) / 128u * 16u : 0u);
    const uint32_t yp = __shfl_sync(~0u, o.Y, (sl + 31u) & 31u);
    o.base = sl ? yp : 0u;
    return o;
}

// Exclusive prefix (bytes) of unit u from its predecessors' published sizes
// (decoupled look-back over units, one warp, one flag a lane per step, so a
// step spans 32 predecessors: the nearest published inclusive prefix is
// usually that close, and a poll that reads fewer flags adds less traffic to
// the cache lines every storer is polling); the caller then publishes u's
// inclusive prefix.  The look-back stops at the first
// inclusive prefix it meets, or at unit `known` (< u, or -1 for none) whose
// inclusive prefix known_incl the caller already holds (the CTA's previous
// unit, about one ticket round back): it never depends on how far other CTAs
// have got with their own look-backs.  Waits for a predecessor that has
// published nothing yet, at most timeout_ns in all (then *timed_out).
__device__ __forceinline__ uint64_t unit_lookback(const uint64_t *flags, uint64_t u, int64_t known,
                                                  uint64_t known_incl, uint64_t timeout_ns, bool *timed_out)
{
    constexpr int kPer = 1;
    const uint32_t lane = threadIdx.x & 31;
    uint64_t prefix = 0;
    int64_t j = (int64_t)u - 1; // highest unit this step reads
    uint64_t t0 = 0;
    bool expired = false;
    while (j >= 0) {
        uint64_t f[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int64_t idx = j - kPer * (int64_t)lane - i;
            // before unit 0: a prefix of 0; the known unit: its inclusive prefix
            f[i] = idx < 0 ? kFlagPrefix
                           : idx == known ? (kFlagPrefix | known_incl)
                                          : (idx < known ? kFlagPrefix : ld_relaxed(const_cast<uint64_t *>(flags) + idx));
        }
        // this lane's flags, newest first, up to and including the first prefix
        bool have = false, zero = false;
        uint64_t sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (!have) {
                const uint32_t state = (uint32_t)(f[i] >> 62);
                zero |= state == 0;
                sum += f[i] & kValueMask;
                have = state == 2;
            }
        }
        const unsigned pmask = __ballot_sync(~0u, have);
        const int fp = pmask ? __ffs(pmask) - 1 : 32; // first lane holding a prefix
        const bool need = (int)lane <= fp;
        if (__any_sync(~0u, need && zero)) {
            const uint64_t now = globaltimer();
            if (t0 == 0)
                t0 = now;
            if (__any_sync(~0u, now - t0 > timeout_ns)) {
                expired = true;
                break;
            }
            __nanosleep(128); // polls compete with the compute warps for issue slots
            continue;
        }
        uint64_t v = need ? sum : 0;
#pragma unroll
        for (int o = 16; o; o >>= 1)
            v += __shfl_xor_sync(~0u, v, o);
        prefix += v;
        if (fp < 32)
            break;
        j -= 32 * kPer;
    }
    *timed_out = expired;
    return prefix;
}

// The word of a unit of a split chunk once its state is at least `state` (1:
// the unit is sized, 2: its tail word is published), polled by the calling
// lane; 0 after timeout_ns (ECC_ERR_TIMEOUT).
__device__ __forceinline__ uint64_t unit_wait_word(const uint64_t *f, uint32_t state, uint64_t timeout_ns,
                                                   uint32_t *status)
{
    uint64_t v = ld_relaxed(f);
    if ((uint32_t)(v >> 62) >= state)
        return v;
    const uint64_t t0 = globaltimer();
    for (;;) {
        __nanosleep(32);
        v = ld_relaxed(f);
        if ((uint32_t)(v >> 62) >= state)
            return v;
        if (globaltimer() - t0 > timeout_ns) {
            set_status(status, ECC_ERR_TIMEOUT);
            return 0;
        }
    }
}

// ---------------------------------------------------------------- compute warps
// The 4 bytes of w as two code pairs (v, q) from the lane's table replica;
// qm tracks the smallest pair multiplier (0: some pair longer than 32 bits,
// or a byte without a table code).
__device__ __forceinline__ void unit_join(const uint2 *lt, uint32_t w, uint32_t &v0, uint32_t &q0, uint32_t &v1,
                                          uint32_t &q1, uint32_t &qm)
{
    const uint2 e0 = lt[byte_of(w, 0) * kLutReplicas];
    const uint2 e1 = lt[byte_of(w, 1) * kLutReplicas];
    const uint2 e2 = lt[byte_of(w, 2) * kLutReplicas];
    const uint2 e3 = lt[byte_of(w, 3) * kLutReplicas];
    v0 = mad_hi(e1.x, e0.y, e0.x);
    q0 = __umulhi(e0.y, e1.y);
    v1 = mad_hi(e3.x, e2.y, e2.x);
    q1 = __umulhi(e2.y, e3.y);
    qm = min(qm, min(q0, q1));
}

// The length table is indexed by each byte rotated left by one bit
// (len_rot), which puts a byte's sign bit beside its lowest bit: a value and
// its negation, equally frequent in these tensors, then share one word of
// the table instead of two words of one bank.  A byte's bank is set by bits
// 1..5, and only bit 6 (the exponent's top bit, rarely set in a gradient or
// an activation) splits a bank's bytes over two words.
__host__ __device__ constexpr uint32_t len_rot(uint32_t b) { return ((b << 1) | (b >> 7)) & 0xFFu; }
// the four bytes of w rotated alike (three instructions for four bytes)
__device__ __forceinline__ uint32_t len_rot4(uint32_t w) { return ((w << 1) & 0xFEFEFEFEu) | ((w >> 7) & 0x01010101u); }

// sum of the 4 code lengths of the bytes of w (len: the shared length table)
__device__ __forceinline__ uint32_t len4(const uint8_t *len, uint32_t w)
{
    w = len_rot4(w);
    return (uint32_t)len[byte_of(w, 0)] + len[byte_of(w, 1)] + len[byte_of(w, 2)] + len[byte_of(w, 3)];
}

// The shared tables of codebook cb (valid), filled by the threads i0,
// i0 + stride, ...: the code table (each code replicated kLutReplicas
// times) and the length table (at the rotated byte values).
__device__ __forceinline__ void unit_load_lut(const ecc_codebook *cb, uint2 *lut, uint32_t i0, uint32_t stride)
{
    for (uint32_t i = i0; i < kLutRows * kLutReplicas; i += stride) {
        const uint32_t s = i / kLutReplicas;
        lut[i] = make_uint2(cb->enc_code[s], cb->enc_mul[s]);
    }
}
__device__ __forceinline__ void unit_load_len(const ecc_codebook *cb, uint8_t *len, uint32_t i0, uint32_t stride)
{
    for (uint32_t i = i0; i < kLutRows; i += stride)
        len[len_rot(i)] = (uint8_t)min((uint32_t)cb->len[i], (uint32_t)ECC_MAX_CODE_LEN);
}

// (lens: the length table; a many-tensor launch: one a slot, and the unit
// records recs)
template <int kMode, bool kBatch = false, bool kFixed = false>
__device__ __forceinline__ void unit_compute(const UnitParams &p, UPipe &P, uint2 *lut, const uint8_t *lens,
                                             [[maybe_unused]] const UUnitRec *recs, uint32_t in0, uint32_t st0,
                                             uint32_t w, uint32_t lane)
{
    static_assert(!kBatch || kMode == kUnitOne, "a many-tensor launch codes a chunk a unit");
    static_assert(!kFixed || kBatch, "the second pass is a many-tensor launch's");
    constexpr bool kOne = kMode != kUnitGroup; // the unit's codes are one run (one chunk, or part of one)
    // stage words in memory order (the storer copies them out as they are),
    // or in register order (split chunks: the storer shifts them first)
    constexpr bool kSwap = kMode != kUnitSplit;
    const uint2 *lt = lut + (lane & (kLutReplicas - 1u));
    const uint32_t wpc = kOne ? kUWarps : p.job.C / (32u * kUThr); // warps per chunk: 1..16
    const uint32_t t = w * 32u + lane;
    const uint32_t s0 = t * kUThr;
    [[maybe_unused]] const ecc_codebook *loaded = nullptr; // many-tensor launch: the code table's codebook
    for (uint64_t k = 0; k <= p.n_units; ++k) {
        const uint32_t slot = (uint32_t)k & 1u, par = (uint32_t)(k >> 1) & 1u, r = (uint32_t)k & 3u;
        const bool ok = mbar_wait(&P.full[slot], par, p.timeout_ns);
        if (!ok)
            set_status(p.job.status, ECC_ERR_TIMEOUT);
        const uint64_t u = ok ? (uint64_t)*(volatile uint64_t *)&P.unit[slot] : (uint64_t)kUEnd;
        const bool end = u == kUEnd;
        // the unit's job, and the unit's index in it (a many-tensor launch:
        // its chunk of its tensor)
        // (a many-tensor launch reads its record even at the end, stale or
        // never written: no address in it is used before the pipeline ends)
        const EncJob &job = unit_job<kBatch>(p, recs, r);
        const uint64_t uc = kBatch ? recs[r].c : u;
        const uint32_t s_shift = 31u - __clz(job.S);
        const uint32_t tps = job.S / kUThr; // threads per sub-block: 2..32
        // a many-tensor launch: a broken codebook codes nothing; the length
        // table is the slot's (the loader fills it with the input)
        const bool cb_ok = !kBatch || recs[r].cb_ok;
        const uint64_t ubase = end ? 0 : uc * kUSyms;
        const uint32_t L = end || !cb_ok ? 0u : (uint32_t)min((uint64_t)kUSyms, job.n - ubase);
        const uint32_t cnt = s0 < L ? min(kUThr, L - s0) : 0u;
        const uint32_t src = in0 + slot * kUSyms + s0;

        // ---- phase A: the thread's bit count from the length table
        uint32_t B;
        {
            const uint4 a = ld_shared_v4(src), b = ld_shared_v4(src + 16u);
            auto count = [&](const uint8_t *len) {
                if (cnt == kUThr)
                    return len4(len, a.x) + len4(len, a.y) + len4(len, a.z) + len4(len, a.w) + len4(len, b.x) +
                           len4(len, b.y) + len4(len, b.z) + len4(len, b.w);
                const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                uint32_t n = 0;
#pragma unroll
                for (uint32_t j = 0; j < kUThr; ++j)
                    n += j < cnt ? (uint32_t)len[byte_of(len_rot4(wd[j >> 2]), j & 3)] : 0u;
                return n;
            };
            // (a many-tensor launch: the slot's table, each at a fixed
            // address, so that the lookups take it as an immediate offset)
            if constexpr (kBatch)
                B = slot ? count(lens + kLutRows) : count(lens);
            else
                B = count(lens);
        }

        // ---- phase B: positions, sub-block counts, the unit's size
        const uint32_t incl = warp_incl(B);
        st_shared_pred(smem_u32(&P.wtot[r][w]), incl, lane == 31);
        if (compute_bar_or(end)) { // the pipeline ends (the same decision in every compute warp)
            if (t == 0) {
                P.sunit[r] = kUEnd;
                mbar_arrive(&P.agg[r]);
            }
            break;
        }
        if constexpr (kBatch) {
            // A codebook other than the code table's: every compute warp is
            // past the last unit's phase C (and holds this unit: none has
            // ended), so the table is reloaded here, the same decision in
            // every compute warp, before this unit's phase C reads it.
            if (cb_ok && job.cb != loaded) {
                unit_load_lut(job.cb, lut, t, kUCompute);
                bar_sync(kUBarTables, kUCompute);
                loaded = job.cb;
            }
        }
        const uint32_t x = lane < kUWarps ? P.wtot[r][lane] : 0u;
        const ULayout lay = unit_layout<kOne>(x, lane, wpc);
        const uint32_t wE = __shfl_sync(~0u, lay.E, w);
        const uint32_t cbase = kOne ? 0u : __shfl_sync(~0u, lay.base, w);
        const uint32_t utot = __shfl_sync(~0u, lay.cbits, kUWarps - 1u); // the unit's bits (kOne)
        // stage bytes the unit needs (split chunks: its words and the storer's 8)
        const uint32_t ubytes = kMode == kUnitSplit ? split_stage_bytes(utot) : __shfl_sync(~0u, lay.Y, kUWarps - 1u);
        // publish the unit's size for the look-back (split chunks: its bits,
        // for the chunk's later units, unless it is the chunk's last); hand
        // the unit to the storer
        if (kMode == kUnitSplit) {
            if (t == 0) {
                const uint32_t m1 = (1u << p.mlog) - 1u;
                const uint64_t c = u >> p.mlog;
                const bool clast = ((uint32_t)u & m1) == m1 || u + 1 == p.n_units;
                const uint64_t units = min((uint64_t)m1 + 1u, p.n_units - (c << p.mlog)); // units of chunk c
                // count the unit into its chunk's word; the last one counted publishes the chunk's size
                const uint64_t old = atomicAdd((unsigned long long *)(job.flags + c),
                                               (1ull << kUCountShift) | (uint64_t)utot);
                if ((old >> kUCountShift) + 1u == units) {
                    const uint64_t cb = ((old & ((1ull << kUCountShift) - 1u)) + utot + 127u) / 128u * 16u;
                    atomicMax((unsigned long long *)(job.flags + c), (c ? kFlagAggregate : kFlagPrefix) | cb);
                }
                // the unit's bits, for the chunk's later units
                if (!clast)
                    st_relaxed(p.uflags + u, kFlagAggregate | utot);
            }
        } else if (!kFixed) { // (the second pass: the first published it)
            st_relaxed_pred(job.flags + uc, kFlagAggregate | ubytes, t == 0 && uc != 0);
        }
        st_shared_u64_pred(&P.sunit[r], u, t == 0);
        mbar_arrive_pred(&P.agg[r], t == 0);
        {
            const uint32_t sb = __shfl_sync(~0u, incl, lane | (tps - 1u)) - (incl - B);
            const uint64_t sidx = (ubase + s0) >> s_shift;
            const uint64_t n_sub = (job.n + job.S - 1) >> s_shift;
            st_global_u16_pred(job.sub_bits + sidx, sb,
                               !kFixed && cnt && (lane & (tps - 1u)) == 0 && sidx < n_sub);
        }
        const bool over = ubytes > p.stage_bytes;
        // the stage of this slot is free once the unit two back has been stored
        if (!mbar_wait(&P.st_free[slot], par ^ 1u, p.timeout_ns))
            set_status(job.status, ECC_ERR_TIMEOUT);

        // ---- phase C: codes at their final places in the stage
        const uint32_t pos = cbase * 8u + wE + incl - B;
        const uint32_t st = st0 + slot * p.stage_bytes;
        const uint32_t lim = st + p.stage_bytes;
        UEnd e{0u, 0u, false};
        [[maybe_unused]] bool bad_index = false;
        // the code pairs, 8 at a time (16 bytes); a partial thread, or one
        // with a pair the table cannot code, takes the paths below, which
        // rewrite every word of its range
        UPacker<kSwap> pk;
#ifdef ECC_CHECKED
        pk.lim = lim;
#endif
        pk.begin(st, pos);
        bool fast = !over && cnt == kUThr;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t v[8], q[8], qm = 0xFFFFFFFFu;
            const uint4 x = ld_shared_v4(src + 16u * h);
            unit_join(lt, x.x, v[0], q[0], v[1], q[1], qm);
            unit_join(lt, x.y, v[2], q[2], v[3], q[3], qm);
            unit_join(lt, x.z, v[4], q[4], v[5], q[5], qm);
            unit_join(lt, x.w, v[6], q[6], v[7], q[7], qm);
            fast = fast && qm != 0;
            if (__all_sync(~0u, fast)) { // the common case: straight-line appends
                if (h == 0)
                    pk.start_pending(v[0], q[0]);
                else
                    pk.put(v[0], q[0]);
#pragma unroll
                for (int i = 1; i < 8; ++i)
                    pk.put(v[i], q[i]);
            } else if (fast) {
                if (h == 0)
                    pk.start_pending(v[0], q[0]);
                else
                    pk.put(v[0], q[0]);
#pragma unroll
                for (int i = 1; i < 8; ++i)
                    pk.put(v[i], q[i]);
            }
        }
        if (__all_sync(~0u, fast)) {
            e = pk.finish();
#ifdef ECC_CHECKED
            bad_index = pk.bad;
#endif
        } else if (fast) {
            e = pk.finish();
#ifdef ECC_CHECKED
            bad_index = pk.bad;
#endif
        } else if (!over && cnt) {
            const uint4 a = ld_shared_v4(src), b = ld_shared_v4(src + 16u);
            const uint32_t bs = cnt == kUThr ? unit_bits_single(lt, a, b) : 1u << 31;
            if (!(bs >> 31))
                e = unit_pack_single<kSwap>(lt, st, pos, a, b, lim, job.status);
            else
                e = unit_pack_slow<kSwap>(st, pos, a, b, cnt, job.cb, lim, job.status);
        }
        // The thread's last partial word: the next lane or-s it into its first
        // word; lane 31 leaves it to the storer; the chunk's last thread
        // stores it (the storer writes the zero padding after it).
        const uint32_t cend = kOne ? L : min(L, (w / wpc + 1u) * wpc * 32u * kUThr); // this chunk's end in the unit
        const bool clast = cnt && s0 + cnt == cend;
        const uint32_t prev = __shfl_up_sync(~0u, clast ? 0u : e.tail, 1);
        if (!over) {
#ifdef ECC_CHECKED
            if (clast && e.partial)
                ust(e.addr, word_order<kSwap>(e.tail), lim, bad_index);
#else
            st_shared_pred(e.addr, word_order<kSwap>(e.tail), clast && e.partial);
#endif
            st_shared_pred(smem_u32(&P.wtail[slot][w]), word_order<kSwap>(e.tail), lane == 31 && !clast);
            red_or_pred(st + (pos >> 5) * 4u, word_order<kSwap>(prev), cnt && lane && (pos & 31u));
        }
#ifdef ECC_CHECKED
        if (bad_index)
            set_status(job.status, ECC_ERR_CHECK);
#endif
        fence_proxy_async(); // this thread's stage stores before the bulk store that reads them
        mbar_arrive(&P.done[slot]); // also: this thread has read the input buffer
    }
}

// ---------------------------------------------------------------- loader warp
// Claims units in ticket order, one slot at a time as the compute warps finish
// the unit in it (phase C reads the input again) and size the next one, and
// bulk-copies each unit's input (lane 0 alone).
// A many-tensor launch: the loader also writes the unit's record and fills
// the slot's length table for the unit's codebook (when it is not the one
// the slot's table holds) before the slot's arrival, as it does the input
// bytes it copies itself.
template <bool kBatch = false, bool kFixed = false>
__device__ __forceinline__ void unit_loader(const UnitParams &p, UPipe &P, uint8_t *in0,
                                            [[maybe_unused]] uint8_t *lens, [[maybe_unused]] UUnitRec *recs,
                                            uint32_t lane)
{
    if (lane != 0)
        return;
    [[maybe_unused]] const ecc_codebook *held0 = nullptr, *held1 = nullptr; // codebooks of the slots' length tables
    // the second pass: its units are the first pass's deferred list (written
    // by the previous launch)
    const uint64_t n_claims = kFixed ? (uint64_t)*(volatile uint32_t *)p.n_deferred : p.n_units;
    for (uint64_t k = 0; k <= p.n_units; ++k) {
        const uint32_t slot = (uint32_t)k & 1u;
        bool stop = false;
        if (k >= 2 && !mbar_wait(&P.done[slot], (uint32_t)((k - 2) >> 1) & 1u, p.timeout_ns)) {
            set_status(p.job.status, ECC_ERR_TIMEOUT);
            stop = true;
        }
        // claim late, once the compute warps have sized the unit in the other
        // slot: a unit is then sized soon after its ticket, and the
        // look-backs of later units wait less for it
        if (k >= 2 && !stop && !mbar_wait(&P.agg[(k - 1) & 3u], (uint32_t)((k - 1) >> 2) & 1u, p.timeout_ns)) {
            set_status(p.job.status, ECC_ERR_TIMEOUT);
            stop = true;
        }
        const uint32_t tk = stop ? 0xFFFFFFFFu : atomicAdd(p.ticket, 1u);
        if (tk >= n_claims) {
            P.unit[slot] = kUEnd;
            mbar_arrive(&P.full[slot]);
            return;
        }
        const uint64_t u = kFixed ? (uint64_t)p.deferred[tk] : (uint64_t)tk;
        P.unit[slot] = u;
        const UItem I = kBatch ? unit_item(p, u) : UItem{p.job, u, 0u};
        const EncJob &job = I.job;
        uint8_t *buf = in0 + slot * kUSyms;
        const uint64_t ubase = I.c * kUSyms;
        const uint32_t L = (uint32_t)min((uint64_t)kUSyms, job.n - ubase);
        const uint32_t whole = L & ~15u;
        for (uint32_t i = whole; i < L; ++i) // the tensor's last bytes (fewer than 16)
            buf[i] = job.in[ubase + i];
        fence_proxy_async();
        if constexpr (kBatch) {
            // the input copy first; the record and the length table (more
            // dependent loads) while it runs, published by the arrival
            mbar_expect_tx_only(&P.full[slot], whole);
            if (whole)
                bulk_g2s(buf, job.in + ubase, whole, &P.full[slot]);
            const bool ok = codebook_ok(job.cb);
            recs[k & (kURecs - 1u)] = UUnitRec{job, I.c, p.descs[I.tensor].t_done_ns, I.tensor, ok ? 1u : 0u};
            if (job.cb != (slot ? held1 : held0) && ok) {
                unit_load_len(job.cb, lens + slot * kLutRows, 0u, 1u);
                if (slot)
                    held1 = job.cb;
                else
                    held0 = job.cb;
            }
            mbar_arrive(&P.full[slot]);
        } else {
            mbar_expect_tx(&P.full[slot], whole);
            if (whole)
                bulk_g2s(buf, job.in + ubase, whole, &P.full[slot]);
        }
    }
}

// ---------------------------------------------------------------- storer warp
// For each unit: its offset (look-back, while the compute warps pack it),
// chunk_off, total_bits, then the stage to the output with one bulk copy.
template <bool kOne, bool kBatch = false>
__device__ __forceinline__ void unit_storer(const UnitParams &p, UPipe &P, [[maybe_unused]] const UUnitRec *recs,
                                            uint32_t st0, uint32_t lane)
{
    const uint32_t G = kOne ? 1u : kUSyms / p.job.C;
    const uint32_t wpc = kOne ? kUWarps : p.job.C / (32u * kUThr);
    int64_t known = -1; // the CTA's previous unit, whose inclusive prefix is known_incl
    uint64_t known_incl = 0;
    [[maybe_unused]] uint32_t known_t = 0xFFFFFFFFu; // many-tensor launch: the previous unit's tensor
    for (uint64_t k = 0; k <= p.n_units; ++k) {
        const uint32_t slot = (uint32_t)k & 1u, par = (uint32_t)(k >> 1) & 1u, r = (uint32_t)k & 3u;
        if (!mbar_wait(&P.agg[r], (uint32_t)(k >> 2) & 1u, p.timeout_ns)) {
            if (lane == 0)
                set_status(p.job.status, ECC_ERR_TIMEOUT);
            break;
        }
        const uint64_t u = *(volatile uint64_t *)&P.sunit[r];
        const uint32_t x = lane < kUWarps ? P.wtot[r][lane] : 0u;
        __syncwarp();
        // The previous unit's stage is free again once its bulk store has
        // read it.  Released only now that unit k's records are read: the
        // compute warps cannot hand over unit k + 4 (same records) before
        // they have packed unit k + 3, whose stage this releases.
        if (k > 0 && lane == 0) {
            bulk_wait_read();
            mbar_arrive(&P.st_free[slot ^ 1u]);
        }
        if (u == kUEnd)
            break;
        // the unit's job, and the unit's index in it (a many-tensor launch:
        // its chunk of its tensor, whose look-back it runs)
        const EncJob &job = unit_job<kBatch>(p, recs, r);
        const uint64_t uc = kBatch ? recs[r].c : u;
        const uint64_t n_chunks = (job.n + job.C - 1) / job.C;
        const bool cb_ok = !kBatch || recs[r].cb_ok; // else the compute warps coded nothing
        const uint64_t ubase = uc * kUSyms;
        const uint32_t L = cb_ok ? (uint32_t)min((uint64_t)kUSyms, job.n - ubase) : 0u;
        const ULayout lay = unit_layout<kOne>(x, lane, wpc);
        const uint32_t ubytes = __shfl_sync(~0u, lay.Y, kUWarps - 1u);
        uint32_t ubits = x;
#pragma unroll
        for (int o = 16; o; o >>= 1)
            ubits += __shfl_xor_sync(~0u, ubits, o);
        bool to = false;
        const uint32_t tensor = kBatch ? recs[r].tensor : 0u;
        const int64_t kn = kBatch && known_t != tensor ? -1 : known;
        const uint64_t prefix = unit_lookback(job.flags, uc, kn, known_incl, p.timeout_ns, &to);
        if (lane == 0) // the unit's inclusive prefix, for the look-backs of later units
            st_relaxed(job.flags + uc, kFlagPrefix | ((prefix + ubytes) & kValueMask));
        known = (int64_t)uc;
        known_incl = prefix + ubytes;
        if constexpr (kBatch)
            known_t = tensor;
        const uint64_t c0 = uc * G;
        const bool chunk_end = lane < kUWarps && (lane & (wpc - 1u)) == wpc - 1u; // a chunk's last lane
        const bool chunk_real = chunk_end && c0 + lane / wpc < n_chunks;
        if (chunk_real)
            job.chunk_off[c0 + lane / wpc + 1] = prefix + lay.Y;
        if (lane == 0) {
            if (uc == 0)
                job.chunk_off[0] = 0;
            atomicAdd((unsigned long long *)job.total_bits, (unsigned long long)ubits);
            if (to)
                set_status(job.status, ECC_ERR_TIMEOUT);
            if (!cb_ok)
                set_status(job.status, ECC_ERR_CODEBOOK);
        }
        const bool fits = prefix + ubytes <= job.out_cap;
        if (!fits && !to && lane == 0)
            set_status(job.status, ECC_ERR_CAPACITY);
        const bool write = fits && !to;
        if (!mbar_wait(&P.done[slot], par, p.timeout_ns)) { // the compute warps have packed the unit
            if (lane == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            break;
        }
        const bool deferred = ubytes > p.stage_bytes;
        if (deferred) {
            // the unit outgrew the stage (long codes): left to the deferred
            // pass, a warp a unit over the whole GPU after this kernel
            if (write && lane == 0) {
                st_relaxed(job.flags + uc, kFlagPrefix | kFlagDeferred | ((prefix + ubytes) & kValueMask));
                if constexpr (kBatch) // for the second pass
                    p.deferred[atomicAdd(p.n_deferred, 1u)] = (uint32_t)u;
            }
        } else if (write) {
            const uint32_t st = st0 + slot * p.stage_bytes;
            // words shared across warps: warp `lane`'s first word takes the
            // previous warp's last partial word
            if (lane > 0 && lane < kUWarps && (lane & (wpc - 1u)) != 0 && lane * 32u * kUThr < L) {
                const uint32_t bit = lay.base * 8u + lay.E;
                if (bit & 31u)
                    red_or_shared(st + (bit >> 5) * 4u, P.wtail[slot][lane - 1]);
            }
            // each chunk's zero padding: from the word after its last bit to its 16-byte end
            if (chunk_real) {
                const uint32_t cb0 = lay.Y - (lay.cbits + 127u) / 128u * 16u; // the chunk's base
                for (uint32_t a2 = cb0 + (lay.cbits + 31u) / 32u * 4u; a2 < lay.Y; a2 += 4u)
                    st_shared_u32(st + a2, 0u);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0 && (!kBatch || ubytes)) // (a broken codebook's chunk has no bytes)
                bulk_s2g(job.out + prefix, st, ubytes);
        }
        if constexpr (kBatch) {
            // the tensor's completion stamp: its segments counted as the
            // deferred pass counts them, by whichever launch codes the chunk
            uint64_t *t_done = recs[r].t_done;
            if (lane == 0 && t_done && !(deferred && write)) {
                __threadfence();
                const uint32_t nseg = job.C / seg_symbols(job.C, job.S);
                if (atomicAdd(p.done + tensor, nseg) + nseg == nseg * (uint32_t)n_chunks)
                    *t_done = globaltimer();
            }
        }
        __syncwarp();
    }
    if (lane == 0)
        bulk_wait_all();
}

// The second pass's storer (many-tensor launch): its units are chunks the
// first pass sized and placed at chunk_off but could not stage; with the
// larger stage of one CTA an SM they are staged and stored like any other
// (a unit still too long, more than 32 bits a symbol, is coded by this warp
// into the output directly).  No look-back: the places are known.
__device__ __forceinline__ void unit_storer_fixed(const UnitParams &p, UPipe &P, const UUnitRec *recs, uint32_t st0,
                                                  uint32_t lane)
{
    for (uint64_t k = 0; k <= p.n_units; ++k) {
        const uint32_t slot = (uint32_t)k & 1u, par = (uint32_t)(k >> 1) & 1u, r = (uint32_t)k & 3u;
        if (!mbar_wait(&P.agg[r], (uint32_t)(k >> 2) & 1u, p.timeout_ns)) {
            if (lane == 0)
                set_status(p.job.status, ECC_ERR_TIMEOUT);
            break;
        }
        const uint64_t u = *(volatile uint64_t *)&P.sunit[r];
        const uint32_t x = lane < kUWarps ? P.wtot[r][lane] : 0u;
        __syncwarp();
        if (k > 0 && lane == 0) { // the previous unit's stage is free again (as unit_storer)
            bulk_wait_read();
            mbar_arrive(&P.st_free[slot ^ 1u]);
        }
        if (u == kUEnd)
            break;
        const UUnitRec &R = recs[r];
        const EncJob &job = R.job;
        const uint64_t uc = R.c;
        const uint64_t n_chunks = (job.n + job.C - 1) / job.C;
        const uint32_t L = (uint32_t)min((uint64_t)kUSyms, job.n - uc * kUSyms);
        const ULayout lay = unit_layout<true>(x, lane, kUWarps);
        const uint32_t ubytes = __shfl_sync(~0u, lay.Y, kUWarps - 1u);
        const uint64_t o0 = job.chunk_off[uc], o1 = job.chunk_off[uc + 1];
        const bool placed = o0 + ubytes == o1 && o1 <= job.out_cap; // where the first pass put it
        if (!placed && lane == 0)
            set_status(job.status, ECC_ERR_CHECK);
        if (!mbar_wait(&P.done[slot], par, p.timeout_ns)) { // the compute warps have packed the unit
            if (lane == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            break;
        }
        if (ubytes > p.stage_bytes) {
            if (placed)
                encode_chunk_warp(job, uc, reinterpret_cast<uint32_t *>(job.out + o0), (uint32_t)((o1 - o0) / 4u));
        } else if (placed) {
            const uint32_t st = st0 + slot * p.stage_bytes;
            // words shared across warps, then the chunk's zero padding (as unit_storer)
            if (lane > 0 && lane < kUWarps && lane * 32u * kUThr < L) {
                const uint32_t bit = lay.base * 8u + lay.E;
                if (bit & 31u)
                    red_or_shared(st + (bit >> 5) * 4u, P.wtail[slot][lane - 1]);
            }
            if (lane == kUWarps - 1u) {
                const uint32_t cb0 = lay.Y - (lay.cbits + 127u) / 128u * 16u;
                for (uint32_t a2 = cb0 + (lay.cbits + 31u) / 32u * 4u; a2 < lay.Y; a2 += 4u)
                    st_shared_u32(st + a2, 0u);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0 && ubytes)
                bulk_s2g(job.out + o0, st, ubytes);
        }
        // the tensor's completion stamp (the first pass left these chunks' segments to be counted here)
        if (lane == 0 && R.t_done) {
            __threadfence();
            const uint32_t nseg = job.C / seg_symbols(job.C, job.S);
            if (atomicAdd(p.done + R.tensor, nseg) + nseg == nseg * (uint32_t)n_chunks)
                *R.t_done = globaltimer();
        }
        __syncwarp();
    }
    if (lane == 0)
        bulk_wait_all();
}

__device__ __forceinline__ void st_global_u32(uint8_t *addr, uint32_t v)
{
    asm volatile("st.global.b32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_global_v4(uint8_t *addr, uint4 v)
{
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// The output word (memory order) whose first r bits are the last r bits of
// hi and whose other 32 - r bits are the first bits of lo (stage words, in
// register order: first bit in bit 31).
__device__ __forceinline__ uint32_t shift_word(uint32_t hi, uint32_t lo, uint32_t r)
{
    return bswap32(__funnelshift_r(lo, hi, r));
}

// Output blocks [b_first, b_end) (16 bytes each, relative to g0) of a unit
// of a split chunk whose stage holds its bits from bit 0 (register-order
// words) and whose first bit is bit s = 32 Q + r of block 0: block b takes
// stage words 4b - Q - 1 .. 4b - Q + 3, read as the two aligned 16-byte
// groups around them.  A lane a block; b_first >= 1.
template <int Q>
__device__ __forceinline__ void split_blocks(uint8_t *g0, uint32_t st, uint32_t r, uint32_t b_first, uint32_t b_end,
                                             uint32_t lane)
{
#pragma unroll 4
    for (uint32_t b = b_first + lane; b < b_end; b += 32u) {
        const uint4 A = ld_shared_v4(st + 16u * (b - 1u)), B = ld_shared_v4(st + 16u * b);
        const uint32_t w[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
        uint32_t v[5];
#pragma unroll
        for (int i = 0; i < 5; ++i)
            v[i] = w[i + 3 - Q];
        uint4 o;
        o.x = bswap32(__funnelshift_r(v[1], v[0], r));
        o.y = bswap32(__funnelshift_r(v[2], v[1], r));
        o.z = bswap32(__funnelshift_r(v[3], v[2], r));
        o.w = bswap32(__funnelshift_r(v[4], v[3], r));
        st_global_v4(g0 + 16u * b, o);
    }
}

// Storer of split chunks.  For unit u (the j-th of chunk c): the bits of the
// chunk's earlier units, the chunk's offset (look-back over chunks), then the
// unit's stage shifted to its bit in the output: the words that are wholly
// the unit's, and its part of each word it shares with a neighbour.  The
// chunk's last unit also publishes the chunk's inclusive prefix, writes
// chunk_off and pads the chunk.  A unit that could not be staged marks its
// chunk for the deferred pass.
__device__ __forceinline__ void unit_storer_split(const UnitParams &p, UPipe &P, uint32_t st0, uint32_t lane)
{
    const EncJob &job = p.job;
    const uint32_t m1 = (1u << p.mlog) - 1u;
    int64_t known = -1; // a chunk whose inclusive prefix known_incl the CTA holds
    uint64_t known_incl = 0;
    for (uint64_t k = 0; k <= p.n_units; ++k) {
        const uint32_t slot = (uint32_t)k & 1u, par = (uint32_t)(k >> 1) & 1u, r4 = (uint32_t)k & 3u;
        if (!mbar_wait(&P.agg[r4], (uint32_t)(k >> 2) & 1u, p.timeout_ns)) {
            if (lane == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            break;
        }
        const uint64_t u = *(volatile uint64_t *)&P.sunit[r4];
        const uint32_t x = lane < kUWarps ? P.wtot[r4][lane] : 0u;
        __syncwarp();
        if (k > 0 && lane == 0) { // as in unit_storer
            bulk_wait_read();
            mbar_arrive(&P.st_free[slot ^ 1u]);
        }
        if (u == kUEnd)
            break;
        const uint64_t c = u >> p.mlog;
        const uint32_t j = (uint32_t)u & m1;
        const bool clast = j == m1 || u + 1 == p.n_units;
        const uint32_t L = (uint32_t)min((uint64_t)kUSyms, job.n - u * kUSyms);
        const ULayout lay = unit_layout<true>(x, lane, kUWarps);
        const uint32_t ubits = __shfl_sync(~0u, lay.cbits, kUWarps - 1u);
        // the bits of the chunk's earlier units (lane i waits for the i-th)
        const uint64_t fb = lane < j ? unit_wait_word(p.uflags + (u - j + lane), 1, p.timeout_ns, job.status) : 0;
        const uint32_t intra = __reduce_add_sync(~0u, (uint32_t)(fb & kUBitsMask));
        const uint32_t cbytes = (intra + ubits + 127u) / 128u * 16u; // the chunk's size (its last unit)
        bool to = false;
        const uint64_t prefix = unit_lookback(job.flags, c, known, known_incl, p.timeout_ns, &to);
        if (clast) {
            if (lane == 0) {
                // raise the chunk's word to the inclusive prefix once every
                // unit has been counted into it (it holds the chunk's size)
                unit_wait_word(job.flags + c, 1, p.timeout_ns, job.status);
                atomicMax((unsigned long long *)(job.flags + c), kFlagPrefix | ((prefix + cbytes) & kValueMask));
                job.chunk_off[c + 1] = prefix + cbytes;
            }
            known = (int64_t)c;
            known_incl = prefix + cbytes;
        } else {
            known = (int64_t)c - 1;
            known_incl = prefix;
        }
        if (lane == 0) {
            if (u == 0)
                job.chunk_off[0] = 0;
            atomicAdd((unsigned long long *)job.total_bits, (unsigned long long)ubits);
            if (to)
                set_status(job.status, ECC_ERR_TIMEOUT);
        }
        // the unit's first bit is bit s = 32 q + r of output block g0
        const uint32_t s = intra & 127u, q = s >> 5, r = s & 31u, e = s + ubits;
        uint8_t *const g0 = job.out + prefix + (intra >> 7) * 16u;
        // output words (from g0) the unit writes, from word q: every word
        // through the chunk's padding (last unit), else its complete words
        // (the partial last one, word e / 32, is shared with the next unit)
        const uint32_t nwe = clast ? (e + 127u) / 128u * 4u : e / 32u;
        const bool fits = prefix + (intra >> 7) * 16u + 4ull * nwe <= job.out_cap;
        if (!fits && !to && lane == 0)
            set_status(job.status, ECC_ERR_CAPACITY);
        const bool write = fits && !to;
        if (!mbar_wait(&P.done[slot], par, p.timeout_ns)) { // the compute warps have packed the unit
            if (lane == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            break;
        }
        const uint32_t st = st0 + slot * p.stage_bytes;
        const uint32_t nst = (ubits + 31u) / 32u; // stage words holding the unit's bits
        if (split_stage_bytes(ubits) > p.stage_bytes) {
            // not staged: the deferred pass codes the whole chunk (the chunk's
            // last unit marks the chunk's word, once the chunk fits; the
            // others the mark word)
            if (lane == 0) {
                if (!clast)
                    atomicOr((unsigned long long *)(p.uflags + min(((c + 1) << p.mlog) - 1u, p.n_units - 1u)),
                             (unsigned long long)kMarkDeferred);
                else if (write)
                    atomicMax((unsigned long long *)(job.flags + c),
                              kFlagPrefix | kFlagDeferred | ((prefix + cbytes) & kValueMask));
            }
            __syncwarp();
            continue;
        }
        // words shared across warps (as in unit_storer; the unit starts at stage bit 0)
        if (lane > 0 && lane < kUWarps && lane * 32u * kUThr < L && (lay.E & 31u))
            red_or_shared(st + (lay.E >> 5) * 4u, P.wtail[slot][lane - 1]);
        // zeros after the unit's last word: the shifted unit reads up to 4
        // words past it (its last partial word, the chunk's padding)
        if (lane < 4u)
            st_shared_u32(st + 4u * (nst + lane), 0u);
        __syncwarp();
        if (!write)
            continue;
        // output word W (q <= W, W - q <= nst + 3): the unit's bits that
        // fall in it, shifted from the stage (word q: zeros in the first r bits)
        auto out_word = [&](uint32_t W) -> uint32_t {
            const uint32_t lo = ld_shared_u32(st + 4u * (W - q));
            const uint32_t hi = W > q ? ld_shared_u32(st + 4u * (W - q - 1u)) : 0u;
            return shift_word(hi, lo, r);
        };
        // whole 16-byte blocks after block 0 (a lane a block)
        const uint32_t b_end = nwe / 4u;
        switch (q) {
        case 0: split_blocks<0>(g0, st, r, 1u, b_end, lane); break;
        case 1: split_blocks<1>(g0, st, r, 1u, b_end, lane); break;
        case 2: split_blocks<2>(g0, st, r, 1u, b_end, lane); break;
        default: split_blocks<3>(g0, st, r, 1u, b_end, lane); break;
        }
        // single words: block 0 after word q (from word q when r = 0: nothing
        // of the previous unit's in it), and the complete words of a last
        // partial block
        const uint32_t hw = q + (r ? 1u : 0u) + lane;          // lanes 0..3
        const uint32_t tw = max(4u, 4u * b_end) + (lane - 4u); // lanes 4..7
        if (lane < 4u && hw < min(4u, nwe))
            st_global_u32(g0 + 4u * hw, out_word(hw));
        if (lane >= 4u && lane < 8u && tw < nwe)
            st_global_u32(g0 + 4u * tw, out_word(tw));
        // the words shared with the previous unit of the chunk (word q, lane
        // 8) and with the next (word e / 32, lane 9): or this unit's part into
        // the earlier unit's word; the second to do so writes the word
        const bool head = lane == 8u && j > 0 && r;
        const bool tail = lane == 9u && !clast && (e & 31u);
        if (head || tail) {
            const uint32_t W = head ? q : e >> 5;
            const uint32_t part = out_word(W);
            const uint64_t old = atomicOr((unsigned long long *)(p.uflags + (head ? u - 1 : u)),
                                          (unsigned long long)((head ? kHandNext : kHandPrev) |
                                                               ((uint64_t)part << kUBitsShift)));
            if (old & (head ? kHandPrev : kHandNext))
                st_global_u32(g0 + 4u * W, part | (uint32_t)(old >> kUBitsShift));
        }
        __syncwarp();
    }
}

// The pipeline of one CTA: tables, barriers, then the warps' roles.  A
// many-tensor launch loads the code tables at each unit whose codebook is
// not the last one's (the units come sorted by codebook).
template <int kMode, bool kBatch, bool kFixed = false>
__device__ __forceinline__ void unit_pipeline(const UnitParams &p, uint8_t *unit_smem, uint8_t *len_table,
                                              UUnitRec *recs)
{
    uint2 *lut = reinterpret_cast<uint2 *>(unit_smem);
    UPipe &P = *reinterpret_cast<UPipe *>(unit_smem + kULutBytes);
    uint8_t *const base = unit_smem + kULutBytes + sizeof(UPipe);
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if constexpr (kBatch) {
        if (!kFixed && p.t_start && blockIdx.x == 0 && threadIdx.x == 0)
            *p.t_start = globaltimer();
    } else {
        const ecc_codebook *cb = p.job.cb;
        if (!codebook_ok(cb)) {
            if (threadIdx.x == 0 && blockIdx.x == 0)
                set_status(p.job.status, ECC_ERR_CODEBOOK);
            return;
        }
    }
#ifdef ECC_CHECKED
    {   // the layout must lie inside the dynamic shared memory the launch gave
        uint32_t dyn;
        asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        if (unit_smem_bytes(p.stage_bytes) > dyn) {
            if (threadIdx.x == 0)
                set_status(p.job.status, ECC_ERR_CHECK);
            return;
        }
    }
#endif
    if constexpr (!kBatch) {
        unit_load_lut(p.job.cb, lut, threadIdx.x, blockDim.x);
        unit_load_len(p.job.cb, len_table, threadIdx.x, blockDim.x);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < 4; ++s)
            mbar_init(&P.agg[s], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&P.full[s], 1);
            mbar_init(&P.st_free[s], 1);
            mbar_init(&P.done[s], kUCompute);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t st0 = smem_u32(base + 2 * kUSyms);
    if (warp < kUWarps)
        unit_compute<kMode, kBatch, kFixed>(p, P, lut, len_table, recs, smem_u32(base), st0, warp, lane);
    else if (warp == kUWarps)
        unit_loader<kBatch, kFixed>(p, P, base, len_table, recs, lane);
    else if constexpr (kMode == kUnitSplit)
        unit_storer_split(p, P, st0, lane);
    else if constexpr (kFixed)
        unit_storer_fixed(p, P, recs, st0, lane);
    else
        unit_storer<kMode == kUnitOne, kBatch>(p, P, recs, st0, lane);
}

// Two CTAs an SM (56 registers a thread): one CTA's barrier waits and
// pipeline stalls are covered by the other's warps.
template <int kMode>
__global__ void __launch_bounds__(kUThreads, 2) encode_unit_kernel(UnitParams p)
{
    extern __shared__ __align__(128) uint8_t unit_smem[];
    __shared__ uint8_t len_table[kLutRows]; // code length of byte b at len_rot(b) (at most ECC_MAX_CODE_LEN; 0: no code)
    unit_pipeline<kMode, false>(p, unit_smem, len_table, nullptr);
}

// The many-tensor launch: tensors of chunks of kUSyms symbols, a chunk a
// unit, in the order of the item map.
__global__ void __launch_bounds__(kUThreads, 2) encode_unit_batched_kernel(UnitParams p)
{
    extern __shared__ __align__(128) uint8_t unit_smem[];
    __shared__ uint8_t len_table[2 * kLutRows]; // a length table for each input slot
    __shared__ UUnitRec recs[kURecs];           // the records of the units in flight
    unit_pipeline<kUnitOne, true>(p, unit_smem, len_table, recs);
}

// Its second pass: the units the first could not stage, with the stage of
// one CTA an SM.
__global__ void __launch_bounds__(kUThreads, 1) encode_unit_fixed_kernel(UnitParams p)
{
    extern __shared__ __align__(128) uint8_t unit_smem[];
    __shared__ uint8_t len_table[2 * kLutRows];
    __shared__ UUnitRec recs[kURecs];
    unit_pipeline<kUnitOne, true, true>(p, unit_smem, len_table, recs);
}

// ---------------------------------------------------------------- host side
// static shared bytes of the kernels, rounded up (the length tables, the
// unit records)
constexpr uint32_t kUStaticOne = 512, kUStaticBatch = 1024;
static_assert(kLutRows <= kUStaticOne && 2 * kLutRows + kURecs * sizeof(UUnitRec) <= kUStaticBatch,
              "static shared bytes");
// Largest stage (multiple of 16; at most 16 bits a symbol for two CTAs an
// SM, 32 for one) with which `ctas` CTAs fit one SM beside static_bytes of
// static shared memory each; 0 if none.
uint32_t unit_stage_bytes(uint32_t static_bytes, int ctas = 2)
{
    int dev = 0, per_sm = 0, reserved = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const int64_t per_cta = std::min<int64_t>(per_sm / ctas - reserved, (int64_t)kMaxDynSmem) - static_bytes;
    const int64_t room = per_cta - (int64_t)unit_smem_bytes(0);
    if (room < 2 * 16)
        return 0;
    return (uint32_t)std::min<int64_t>(room / 2 / 16 * 16, (ctas == 1 ? 4 : 2) * kUSyms);
}

// Launch the unit encoder (the prologue has cleared the flags, the ticket
// and the outputs; for chunks of more than kUSyms symbols job.flags holds a
// word per chunk and then a word per unit).  *unit_chunks: the chunks of a
// unit of the deferred pass.  Returns ECC_ERR_CUDA if it cannot run on this
// device.
ecc_status launch_unit_encoder(const EncJob &job, uint32_t *ticket, cudaStream_t st, uint32_t *unit_chunks)
{
    UnitParams p{};
    p.job = job;
    p.n_units = (job.n + kUSyms - 1) / kUSyms;
    p.uflags = job.flags + (job.n + job.C - 1) / job.C;
    p.mlog = job.C > kUSyms ? 31u - __builtin_clz(job.C / kUSyms) : 0u;
    p.ticket = ticket;
    p.timeout_ns = kWaitLimitNs;
    p.stage_bytes = unit_stage_bytes(kUStaticOne);
    if (p.stage_bytes < 16u)
        return ECC_ERR_CUDA;
    const int mode = job.C == kUSyms ? kUnitOne : job.C < kUSyms ? kUnitGroup : kUnitSplit;
    const void *kfn = mode == kUnitOne     ? (const void *)encode_unit_kernel<kUnitOne>
                      : mode == kUnitGroup ? (const void *)encode_unit_kernel<kUnitGroup>
                                           : (const void *)encode_unit_kernel<kUnitSplit>;
    const size_t smem = unit_smem_bytes(p.stage_bytes);
    const int occ = occupancy(kfn, kUThreads, smem);
    const int sms = sm_count();
    if (occ <= 0 || sms <= 0)
        return ECC_ERR_CUDA;
    // persistent: every CTA resident, so a unit's predecessors are always being coded
    const uint64_t need = (p.n_units + 1) / 2;
    const uint64_t grid = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)occ * sms, need));
    if (mode == kUnitOne)
        encode_unit_kernel<kUnitOne><<<(unsigned)grid, kUThreads, smem, st>>>(p);
    else if (mode == kUnitGroup)
        encode_unit_kernel<kUnitGroup><<<(unsigned)grid, kUThreads, smem, st>>>(p);
    else
        encode_unit_kernel<kUnitSplit><<<(unsigned)grid, kUThreads, smem, st>>>(p);
    *unit_chunks = mode == kUnitSplit ? 1u : kUSyms / job.C;
    return launch_status(cudaGetLastError());
}

// The many-tensor launch over n_units chunks of kUSyms symbols (the prologue
// has cleared flags, done and the tensors' outputs; *ticket is 0).  Returns
// ECC_ERR_CUDA with *launched false, having launched nothing, if it cannot
// run on this device; *launched true once its first kernel is launched.
ecc_status launch_unit_encoder_batched(const UnitBatch &b, cudaStream_t st, bool *launched)
{
    *launched = false;
    UnitParams p{};
    // only its look-back words and status are read (the waits that end
    // before their unit is known report there)
    p.job.flags = b.flags;
    p.job.status = b.status;
    p.job.C = kUSyms;
    p.job.S = kUSyms;
    p.n_units = b.n_units;
    p.ticket = b.ticket;
    p.timeout_ns = kWaitLimitNs;
    p.stage_bytes = unit_stage_bytes(kUStaticBatch);
    p.items = b.items;
    p.descs = b.descs;
    p.done = b.done;
    p.t_start = b.t_start;
    if (p.stage_bytes < 16u || b.n_units == 0)
        return ECC_ERR_CUDA;
    const size_t smem = unit_smem_bytes(p.stage_bytes);
    const int occ = occupancy((const void *)encode_unit_batched_kernel, kUThreads, smem);
    const int sms = sm_count();
    if (occ <= 0 || sms <= 0)
        return ECC_ERR_CUDA;
    const uint64_t need = (p.n_units + 1) / 2;
    const uint64_t grid = std::max<uint64_t>(1, std::min<uint64_t>((uint64_t)occ * sms, need));
    p.deferred = b.deferred;
    p.n_deferred = b.n_deferred;
    // the second pass: a CTA an SM, each with stages of up to 32 bits a
    // symbol (checked before the first launches: the caller's other route
    // must find the workspace untouched)
    UnitParams q = p;
    q.ticket = b.ticket2;
    q.stage_bytes = unit_stage_bytes(kUStaticBatch, 1);
    q.t_start = nullptr;
    const size_t smem2 = unit_smem_bytes(q.stage_bytes);
    const int occ2 = q.stage_bytes < 16u ? 0 : occupancy((const void *)encode_unit_fixed_kernel, kUThreads, smem2);
    if (occ2 <= 0)
        return ECC_ERR_CUDA;
    encode_unit_batched_kernel<<<(unsigned)grid, kUThreads, smem, st>>>(p);
    const ecc_status e = launch_status(cudaGetLastError());
    if (e != ECC_OK)
        return e;
    *launched = true; // from here on an error is the call's: no other route may follow
    encode_unit_fixed_kernel<<<(unsigned)(occ2 * sms), kUThreads, smem2, st>>>(q);
    return launch_status(cudaGetLastError());
}

} // namespace ecc
