// ecc_batched.cu -- one-launch encode and decode of many tensors, each with
// its own codebook and container sizes (the message regime of collective
// communication: many tensors of very different sizes).  See ecc.h.
//
// The host orders the tensors by codebook (stable: equal codebooks keep the
// caller's order) and lays their chunks (decode: the pieces of their chunks,
// as the single-tensor decoder splits them) end to end in that order.  A
// prologue kernel writes item[i] = tensor << 32 | chunk (or piece) for every
// position, so a kernel finds its work with one load instead of a search,
// and a CTA reloads its shared code tables only where the codebook changes
// (a few times per launch) instead of at almost every chunk.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#include "ecc_device.cuh"
#include "ecc_launch.h"

namespace ecc {

// Workspace layout (all offsets 16-byte aligned):
//   header | descs[count] | prefix[count + 1] | done[count] | item[n_items] | flags[total_chunks]
//   | deferred[total_chunks]
// descs are in workspace order (sorted by codebook); prefix[d] = first item
// of tensor d; flags = look-back words, deferred = the positions of the
// chunks the unit encoder left to its second pass (encode only).
struct BatchHeader {
    uint32_t ticket;
    uint32_t count;
    uint32_t warps;       // decode: chunks per group (warps per CTA)
    uint32_t stage_bytes;
    uint32_t max_C;
    uint32_t encode;
    uint32_t ws_slot_bytes; // encode: stage slot of the warp-specialised kernel (largest over the tensors)
    uint32_t n_deferred;    // encode: entries of deferred[]
    uint32_t ticket2;       // encode: the unit encoder's second pass
    uint32_t pad;
    uint64_t n_items;     // encode: chunks; decode: pieces, each codebook run padded to a multiple of warps
    uint64_t total_chunks;
    uint64_t desc_off, prefix_off, done_off, item_off, flags_off, deferred_off;
};

constexpr uint64_t kNoItem = ~0ull; // item of a padding position

struct BatchLayout {
    size_t desc_off, prefix_off, done_off, item_off, flags_off, deferred_off, bytes;
};

static size_t up16(size_t v) { return (v + 15) & ~size_t(15); }

static BatchLayout layout_for(uint32_t count, uint64_t n_items, uint64_t flag_words)
{
    BatchLayout L;
    L.desc_off = up16(sizeof(BatchHeader));
    L.prefix_off = up16(L.desc_off + (size_t)count * sizeof(ecc_desc));
    L.done_off = up16(L.prefix_off + ((size_t)count + 1) * sizeof(uint64_t));
    L.item_off = up16(L.done_off + (size_t)count * sizeof(uint32_t));
    L.flags_off = up16(L.item_off + n_items * sizeof(uint64_t));
    L.deferred_off = up16(L.flags_off + flag_words * sizeof(uint64_t));
    L.bytes = up16(L.deferred_off + flag_words * sizeof(uint32_t));
    return L;
}

__device__ __forceinline__ uint64_t chunks_of(const ecc_desc &d) { return (d.n + d.C - 1) >> (31 - __clz(d.C)); }

// The batched decoder's split of a tensor's chunks: one or two streams a
// lane, pieces of at most kDecPieceSyms symbols.
__host__ __device__ inline DecSplit batch_split(const ecc_desc &d) { return dec_split(d.C, d.S, 2); }

__global__ void batch_prologue_kernel(uint8_t *ws)
{
    const BatchHeader *h = reinterpret_cast<const BatchHeader *>(ws);
    const ecc_desc *descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    const uint64_t *prefix = reinterpret_cast<const uint64_t *>(ws + h->prefix_off);
    uint32_t *done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    uint64_t *item = reinterpret_cast<uint64_t *>(ws + h->item_off);
    uint64_t *flags = reinterpret_cast<uint64_t *>(ws + h->flags_off);
    const uint32_t count = h->count;
    const uint64_t i0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = i0; i < count; i += stride) {
        const ecc_desc &d = descs[i];
        *d.status = ECC_OK;
        done[i] = 0;
        if (h->encode) {
            *d.total_bits = 0;
            d.chunk_off[0] = 0;
        }
        if (d.t_done_ns && d.n == 0)
            *d.t_done_ns = 0;
    }
    for (uint64_t i = i0; i < h->n_items; i += stride) {
        // the tensor of position i: largest d with prefix[d] <= i (empty
        // tensors share their successor's prefix and are passed over)
        uint32_t lo = 0, hi = count;
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (prefix[mid] <= i)
                lo = mid;
            else
                hi = mid;
        }
        const uint64_t c = i - prefix[lo]; // the chunk (decode: the piece) within its tensor
        const uint32_t ps = h->encode ? 0u : batch_split(descs[lo]).ps;
        item[i] = c < (chunks_of(descs[lo]) << ps) ? ((uint64_t)lo << 32 | c) : kNoItem;
    }
    if (h->encode)
        for (uint64_t i = i0; i < h->total_chunks; i += stride)
            flags[i] = 0;
}

// ---------------------------------------------------------------- encode
// Warp-specialised many-tensor encoder: the single-tensor kernel's body with
// each claimed chunk's job taken from the item map and its descriptor.
__global__ void __maxnreg__(96) encode_batched_ws_kernel(uint8_t *ws, uint64_t *t_start)
{
    BatchHeader *h = reinterpret_cast<BatchHeader *>(ws);
    if (t_start && blockIdx.x == 0 && threadIdx.x == 0)
        *t_start = globaltimer();
    EncBatch bt;
    bt.ticket = &h->ticket;
    bt.total = h->total_chunks;
    bt.item = reinterpret_cast<const uint64_t *>(ws + h->item_off);
    bt.descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    bt.flags = reinterpret_cast<uint64_t *>(ws + h->flags_off);
    bt.done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    const EncJob none{};
    encode_ws_body<true>(none, 0, nullptr, bt, h->ws_slot_bytes, h->max_C, kWaitLimitNs);
}

// The deferred pass of the many-tensor encoder: warp w of W takes chunk
// positions w, w + W, w + 2W, ... (the marked chunks come in runs: the
// tensors are grouped by codebook, and long codes are a codebook's), 32 at a
// time, a lane each reading a look-back word; it codes each chunk the
// encoder marked (long codes), then counts its segments toward the tensor's
// completion stamp as the encoder would have.
__global__ void __launch_bounds__(256) encode_batched_deferred_kernel(uint8_t *ws)
{
    const BatchHeader *h = reinterpret_cast<const BatchHeader *>(ws);
    const uint64_t *item = reinterpret_cast<const uint64_t *>(ws + h->item_off);
    const ecc_desc *descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    uint64_t *flags = reinterpret_cast<uint64_t *>(ws + h->flags_off);
    uint32_t *done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t total = h->total_chunks;
    const uint64_t w0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nw = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t p0 = w0; p0 < total; p0 += 32 * nw) {
        const uint64_t mine = p0 + lane * nw;
        const bool marked = mine < total && is_deferred(flags[mine]);
        for (uint32_t m = __ballot_sync(~0u, marked); m; m &= m - 1) {
            const uint64_t pos = p0 + (uint64_t)(__ffs(m) - 1) * nw;
            const uint64_t it = item[pos];
            if (it == kNoItem)
                continue;
            const uint32_t t = (uint32_t)(it >> 32);
            const uint64_t c = it & 0xFFFFFFFFull;
            const ecc_desc &d = descs[t];
            const EncJob job{d.in, d.n, d.cb, d.C, d.S, d.out, d.cap, d.chunk_off, d.sub_bits, d.total_bits,
                             flags + (pos - c), d.status};
            code_deferred_unit(job, c, 1, chunks_of(d));
            if (d.t_done_ns) {
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t nseg = d.C / seg_symbols(d.C, d.S);
                    const uint32_t want = nseg * (uint32_t)chunks_of(d);
                    if (atomicAdd(done + t, nseg) + nseg == want)
                        *d.t_done_ns = globaltimer();
                }
            }
        }
    }
}

__device__ __forceinline__ void stamp_done(const ecc_desc &d, uint32_t *done, uint32_t k)
{
    if (!d.t_done_ns)
        return;
    __threadfence();
    if (atomicAdd(done + k, 1u) + 1u == chunks_of(d))
        *d.t_done_ns = globaltimer();
}

// Single-slot many-tensor encoder, for chunk sizes whose two input buffers
// and two stage slots exceed shared memory (C = 64 KiB).  Thread 0 claims
// one chunk ahead into a shared slot and bulk-copies its input.
struct BatchSlot {
    ecc_desc d;
    uint64_t item;   // ticket
    uint64_t c;      // chunk within its tensor
    uint32_t tensor;
    uint32_t pad;
};
constexpr uint32_t kBatchSlotBytes = 2 * ((sizeof(BatchSlot) + 15) & ~15u);

__global__ void __launch_bounds__(kEncThreads) encode_batched_kernel(uint8_t *ws, uint64_t *t_start)
{
    extern __shared__ __align__(16) uint8_t smem[];
    EncShared &sh = *reinterpret_cast<EncShared *>(smem);
    BatchHeader *h = reinterpret_cast<BatchHeader *>(ws);
    const ecc_desc *descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    const uint64_t *item = reinterpret_cast<const uint64_t *>(ws + h->item_off);
    uint32_t *done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    uint64_t *flags = reinterpret_cast<uint64_t *>(ws + h->flags_off);
    const uint32_t stage_bytes = h->stage_bytes;
    const uint32_t cmax = h->max_C;
    const uint64_t total = h->total_chunks;
    BatchSlot *slot = reinterpret_cast<BatchSlot *>(smem + enc_shared_bytes());
    uint8_t *inbuf = smem + enc_shared_bytes() + kBatchSlotBytes;
    uint32_t *stage = reinterpret_cast<uint32_t *>(inbuf + cmax + kStageLead);
    const int tid = threadIdx.x;
    if (t_start && blockIdx.x == 0 && tid == 0)
        *t_start = globaltimer();
    if (tid == 0) {
        mbar_init(&sh.bar[0], 1);
        fence_mbar_init();
    }
    uint4 *st4 = reinterpret_cast<uint4 *>(inbuf + cmax); // the guard word and the stage
    for (uint32_t i = tid; i < (kStageLead + stage_bytes) / 16; i += kEncThreads)
        st4[i] = make_uint4(0, 0, 0, 0);
    auto job_of = [&](const BatchSlot &s) {
        const ecc_desc &d = s.d;
        return EncJob{d.in,         d.n, d.cb, d.C, d.S, d.out, d.cap, d.chunk_off, d.sub_bits,
                      d.total_bits, flags + (s.item - s.c), d.status};
    };
    // thread 0: claim the next chunk into slot q, and bulk-copy its input
    bool pending = false;
    auto claim = [&](uint32_t q, bool copy) {
        const uint32_t t = atomicAdd(&h->ticket, 1u);
        slot[q].item = t;
        if (t < total) {
            const uint64_t m = item[t];
            slot[q].tensor = (uint32_t)(m >> 32);
            slot[q].c = m & 0xFFFFFFFFull;
            slot[q].d = descs[m >> 32];
            if (copy) {
                issue_chunk_input(job_of(slot[q]), slot[q].c, inbuf, &sh.bar[0]);
                pending = true;
            }
        }
    };
    if (tid == 0)
        claim(0, true);
    __syncthreads();
    uint32_t phase = 0;
    bool staging = true;
    const ecc_codebook *loaded = nullptr;
    for (uint32_t b = 0;; b ^= 1) {
        if (slot[b].item >= total)
            break;
        const BatchSlot s = slot[b];
        const EncJob job = job_of(s);
        const bool cb_ok = s.d.cb->magic == ECC_CODEBOOK_MAGIC && s.d.cb->max_len <= ECC_MAX_CODE_LEN;
        if (cb_ok && s.d.cb != loaded) {
            __syncthreads(); // the previous chunk's lookups are done
            load_encode_lut(sh, s.d.cb, kEncThreads);
            loaded = s.d.cb;
            __syncthreads();
        }
        bool ok = staging && mbar_wait(&sh.bar[0], phase, kWaitLimitNs);
        ok = __syncthreads_and(ok) != 0;
        if (ok) {
            phase ^= 1u;
            if (tid == 0)
                pending = false;
        } else {
            if (staging && tid == 0)
                set_status(job.status, ECC_ERR_TIMEOUT);
            staging = false;
        }
        if (cb_ok) {
            if (ok)
                encode_chunk<true>(sh, stage, stage_bytes, job, inbuf, s.c, kWaitLimitNs);
            else
                encode_chunk<false>(sh, stage, stage_bytes, job, nullptr, s.c, kWaitLimitNs);
        } else if (tid < 32) {
            // keep the tensor's look-back moving; its status says why it is empty
            bool to;
            const uint64_t pre = lookback(job.flags, s.c, 0, kWaitLimitNs, &to);
            if (tid == 0) {
                set_status(job.status, ECC_ERR_CODEBOOK);
                job.chunk_off[s.c + 1] = pre;
            }
        }
        if (tid == 0) {
            stamp_done(s.d, done, s.tensor);
            claim(b ^ 1, staging); // the input buffer is free again
        }
        __syncthreads();
    }
    if (tid == 0 && pending)
        (void)mbar_wait(&sh.bar[0], phase, kWaitLimitNs);
}

// ---------------------------------------------------------------- decode
// Groups of `warps` consecutive items; CTA x decodes groups x, x + grid, ...
// (warp w the group's item w), the schedule of the single-tensor decoder.
// Codebook runs are padded to whole groups, so a group has one codebook and
// every warp of a CTA meets the codebook changes at the same groups.
// An item is a piece of a chunk (dec_split with at most 2 streams a lane,
// per tensor): the warp decodes it with its own streams a lane.  At most 128
// registers (batched message workload, decode GB/s: 417 at 96, 430 at 112,
// 437 at 128, 358 at 144 and 363 uncapped at 168, with fewer warps).
__global__ void __maxnreg__(128) decode_batched_kernel(uint8_t *ws, uint64_t *t_start)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *dec = reinterpret_cast<uint16_t *>(smem);
    LongTable &lt = *reinterpret_cast<LongTable *>(smem + kDecTableBytes);
    QlcShared &qs = *reinterpret_cast<QlcShared *>(smem + kDecTableBytes + kLongTableBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kDecTableBytes + kLongTableBytes + kQlcSharedBytes);
    const BatchHeader *h = reinterpret_cast<const BatchHeader *>(ws);
    const ecc_desc *descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    const uint64_t *item = reinterpret_cast<const uint64_t *>(ws + h->item_off);
    uint32_t *done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    const uint32_t stage_bytes = h->stage_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t W = blockDim.x >> 5;
    if (t_start && blockIdx.x == 0 && threadIdx.x == 0)
        *t_start = globaltimer();
    if (lane == 0) {
        mbar_init(&bars[warp], 1);
        fence_mbar_init();
    }
    __syncthreads();
    WarpStage wst{reinterpret_cast<uint32_t *>(smem + kDecHeadBytes + (size_t)warp * stage_bytes), stage_bytes,
                  &bars[warp], 0};
    const uint64_t groups = h->n_items / W;
    const ecc_codebook *loaded = nullptr;
    bool loaded_ok = false, loaded_qlc = false;
    for (uint64_t g = blockIdx.x; g < groups; g += gridDim.x) {
        const uint64_t m0 = item[g * W]; // a group never starts on padding
        const uint64_t m = item[g * W + warp];
        const ecc_codebook *cb = descs[m0 >> 32].cb;
        if (cb != loaded) {
            __syncthreads(); // every warp is done with the previous tables
            loaded = cb;
            loaded_ok = cb->magic == ECC_CODEBOOK_MAGIC && cb->max_len <= ECC_MAX_CODE_LEN;
            loaded_qlc = loaded_ok && qlc_mode(cb);
            if (loaded_qlc) {
                load_qlc_tables(reinterpret_cast<uint32_t *>(smem), qs, cb, blockDim.x);
                load_long_table(lt, cb);
            } else if (loaded_ok) {
                const uint4 *src = reinterpret_cast<const uint4 *>(cb->dec);
                uint4 *dst = reinterpret_cast<uint4 *>(dec);
                for (int i = threadIdx.x; i < (int)(kDecTableBytes / 16); i += blockDim.x)
                    dst[i] = src[i];
                load_long_table(lt, cb);
            }
            __syncthreads();
            if (loaded_ok && lt.sub_np) { // the long codes' second level (the same decision in every thread)
                fill_long_sub(lt, threadIdx.x, blockDim.x);
                __syncthreads();
            }
        }
        if (m == kNoItem)
            continue;
        const uint32_t k = (uint32_t)(m >> 32);
        const uint64_t local = m & 0xFFFFFFFFull;
        const ecc_desc &d = descs[k];
        const uint64_t nch = chunks_of(d);
        const DecSplit sp = batch_split(d);
        const uint64_t c = local >> sp.ps;
        const uint32_t piece = (uint32_t)local & ((1u << sp.ps) - 1u);
        if (loaded_ok) {
            const DecJob job{d.in, d.cap, d.chunk_off, d.sub_bits, d.n, d.C, d.S, d.cb, d.out, d.status};
            // (the next item is another warp's: no L2 prefetch)
            auto run = [&](const DecTables &T, auto qlc) {
                constexpr bool kQ = decltype(qlc)::value;
                if (sp.ps == 0) {
                    if (sp.R == 2)
                        decode_chunk<2, kQ, true>(job, T, wst, c, nch, nch);
                    else
                        decode_chunk<1, kQ, true>(job, T, wst, c, nch, nch);
                } else if (sp.R == 2) {
                    decode_piece<2, kQ, true>(job, T, wst, c, piece, sp.ps);
                } else {
                    decode_piece<1, kQ, true>(job, T, wst, c, piece, sp.ps);
                }
            };
            if (loaded_qlc) {
                run(qlc_tables(cb->dec, &lt, qs, reinterpret_cast<const uint32_t *>(smem)), std::true_type{});
            } else {
                DecTables T{};
                T.dec = dec;
                T.lt = &lt;
                run(T, std::false_type{});
            }
        } else if (lane == 0) {
            set_status(d.status, ECC_ERR_CODEBOOK);
        }
        if (d.t_done_ns) {
            __threadfence(); // this lane's output stores before the completion count
            __syncwarp();
            if (lane == 0 && atomicAdd(done + k, 1u) + 1u == (uint32_t)(nch << sp.ps))
                *d.t_done_ns = globaltimer();
        }
    }
}

} // namespace ecc

using namespace ecc;

namespace {

constexpr uint64_t kMaxItems = 1ull << 31; // tickets are 32-bit

struct BatchPlan {
    std::vector<uint32_t> order; // workspace position -> caller's index
    std::vector<uint64_t> prefix;
    uint64_t n_items = 0, total_chunks = 0;
    uint32_t max_C = 1024, warps = 1, stage = 0, ws_slot = 0, dec_stage = 0;
    bool units = true; // every tensor's chunks are of kUnitSyms symbols: the unit encoder codes the batch
};

// as many warps as shared memory holds stages for, and registers allow
uint32_t batch_decode_warps(uint32_t stage)
{
    int warps = decode_warps(stage);
    while (warps > 1 &&
           (kDecHeadBytes + (size_t)warps * stage > kMaxDynSmem - kStaticSmemReserve ||
            occupancy((const void *)decode_batched_kernel, warps * 32,
                      std::max<size_t>(kDecMinSmem, kDecHeadBytes + (size_t)warps * stage)) <= 0))
        --warps;
    return (uint32_t)warps;
}

ecc_status plan_batch(const ecc_desc *descs, uint32_t count, bool encode, bool check, BatchPlan *P)
{
    if (!descs || count == 0)
        return ECC_ERR_ARG;
    for (uint32_t i = 0; i < count; ++i) {
        const ecc_desc &d = descs[i];
        if (check) {
            if (!valid_sizes(d.C, d.S) || !d.cb || !aligned16(d.cb) || !d.status || !d.chunk_off)
                return ECC_ERR_ARG;
            if (encode && !d.total_bits)
                return ECC_ERR_ARG;
            if (d.n && (!d.in || !d.out || !d.sub_bits || !aligned16(d.in) || !aligned16(d.out)))
                return ECC_ERR_ARG;
        } else if (!valid_sizes(d.C, d.S)) {
            continue;
        }
        const uint64_t nc = ecc_num_chunks(d.n, d.C);
        if (nc >= kMaxItems)
            return ECC_ERR_ARG;
        P->total_chunks += nc;
        P->units = P->units && (d.n == 0 || d.C == kUnitSyms);
        P->max_C = std::max(P->max_C, d.C);
        P->ws_slot = std::max(P->ws_slot, enc_ws_slot_bytes(d.C, d.S));
        // decode stage: the single-tensor decoder's for a piece (at up to 9.25
        // bits a symbol, larger ones 32 sub-blocks at a time), for every shape
        P->dec_stage = std::max(P->dec_stage, dec_stage_bytes(d.C >> batch_split(d).ps, d.S));
    }
    P->stage = encode ? stage_bytes_for(P->max_C) : P->dec_stage;
    P->warps = encode ? 1u : batch_decode_warps(P->stage);
    P->order.resize(count);
    std::iota(P->order.begin(), P->order.end(), 0u);
    std::stable_sort(P->order.begin(), P->order.end(), [&](uint32_t a, uint32_t b) {
        return reinterpret_cast<uintptr_t>(descs[a].cb) < reinterpret_cast<uintptr_t>(descs[b].cb);
    });
    P->prefix.assign((size_t)count + 1, 0);
    uint64_t acc = 0;
    for (uint32_t j = 0; j < count; ++j) {
        const ecc_desc &d = descs[P->order[j]];
        // decode: pad each codebook run to whole groups
        if (!encode && j > 0 && d.cb != descs[P->order[j - 1]].cb)
            acc = (acc + P->warps - 1) / P->warps * P->warps;
        P->prefix[j] = acc;
        acc += valid_sizes(d.C, d.S) ? ecc_num_chunks(d.n, d.C) << (encode ? 0u : batch_split(d).ps) : 0;
    }
    if (!encode)
        acc = (acc + P->warps - 1) / P->warps * P->warps;
    P->prefix[count] = acc;
    P->n_items = acc;
    if (acc >= kMaxItems)
        return ECC_ERR_ARG;
    return ECC_OK;
}

ecc_status run_batched(const ecc_desc *descs, uint32_t count, void *ws, size_t ws_bytes, uint64_t *t_start,
                       void *stream, bool encode)
{
    BatchPlan P;
    ecc_status e = plan_batch(descs, count, encode, true, &P);
    if (e != ECC_OK)
        return e;
    const BatchLayout L = layout_for(count, P.n_items, encode ? P.total_chunks : 0);
    if (!ws || !aligned16(ws) || ws_bytes < L.bytes)
        return ECC_ERR_ARG;
    // host image of header | descs | prefix, copied with one async copy
    std::vector<uint8_t> img(L.done_off, 0);
    BatchHeader *h = reinterpret_cast<BatchHeader *>(img.data());
    h->ticket = 0;
    h->count = count;
    h->warps = P.warps;
    h->stage_bytes = P.stage;
    h->max_C = P.max_C;
    h->encode = encode ? 1u : 0u;
    h->ws_slot_bytes = P.ws_slot;
    h->n_items = P.n_items;
    h->total_chunks = P.total_chunks;
    h->desc_off = L.desc_off;
    h->prefix_off = L.prefix_off;
    h->done_off = L.done_off;
    h->item_off = L.item_off;
    h->flags_off = L.flags_off;
    h->deferred_off = L.deferred_off;
    ecc_desc *sorted = reinterpret_cast<ecc_desc *>(img.data() + L.desc_off);
    for (uint32_t j = 0; j < count; ++j)
        sorted[j] = descs[P.order[j]];
    std::memcpy(img.data() + L.prefix_off, P.prefix.data(), P.prefix.size() * sizeof(uint64_t));
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(ws, img.data(), img.size(), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return launch_status(cudaErrorUnknown);
    const int sms = sm_count();
    if (sms <= 0)
        return ECC_ERR_CUDA;
    {
        const uint64_t work = std::max<uint64_t>(count, P.n_items);
        const uint64_t nb = std::max<uint64_t>(1, std::min<uint64_t>((work + 255) / 256, 1024));
        batch_prologue_kernel<<<(unsigned)nb, 256, 0, st>>>((uint8_t *)ws);
        if ((e = launch_status(cudaGetLastError())) != ECC_OK)
            return e;
    }
    if (P.n_items == 0)
        return ECC_OK;
    if (encode) {
        // the chunks it leaves to the deferred pass (long codes)
        auto deferred = [&]() {
            const uint64_t blocks = std::max<uint64_t>(1, std::min<uint64_t>((P.n_items + 7) / 8, (uint64_t)sms * 8));
            encode_batched_deferred_kernel<<<(unsigned)blocks, 256, 0, st>>>((uint8_t *)ws);
            return launch_status(cudaGetLastError());
        };
        if (P.units) {
            uint8_t *w = (uint8_t *)ws;
            BatchHeader *wh = reinterpret_cast<BatchHeader *>(w);
            const UnitBatch ub{reinterpret_cast<const uint64_t *>(w + L.item_off),
                               reinterpret_cast<const ecc_desc *>(w + L.desc_off),
                               reinterpret_cast<uint64_t *>(w + L.flags_off),
                               reinterpret_cast<uint32_t *>(w + L.done_off),
                               &wh->ticket,
                               sorted[0].status,
                               t_start,
                               P.total_chunks,
                               reinterpret_cast<uint32_t *>(w + L.deferred_off),
                               &wh->n_deferred,
                               &wh->ticket2};
            // (its second pass codes the chunks it could not stage); the
            // warp-segmented route below only if it launched nothing
            bool launched = false;
            const ecc_status ue = launch_unit_encoder_batched(ub, st, &launched);
            if (ue == ECC_OK || launched)
                return ue;
        }
        const size_t ws_smem = enc_ws_smem_bytes(P.max_C, P.ws_slot);
        const int occ_ws = ws_smem <= kMaxDynSmem - kStaticSmemReserve
                               ? occupancy((const void *)encode_batched_ws_kernel, kEncThreadsWS, ws_smem)
                               : 0;
        if (occ_ws > 0) {
            const uint64_t grid = std::min<uint64_t>((uint64_t)occ_ws * sms, P.n_items);
            encode_batched_ws_kernel<<<(unsigned)grid, kEncThreadsWS, ws_smem, st>>>((uint8_t *)ws, t_start);
            if ((e = launch_status(cudaGetLastError())) != ECC_OK)
                return e;
            return deferred();
        }
        const size_t smem = enc_shared_bytes() + kBatchSlotBytes + (size_t)P.max_C + kStageLead + P.stage;
        const int occ = occupancy((const void *)encode_batched_kernel, kEncThreads, smem);
        if (occ <= 0)
            return ECC_ERR_CUDA;
        const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, P.n_items);
        encode_batched_kernel<<<(unsigned)grid, kEncThreads, smem, st>>>((uint8_t *)ws, t_start);
        return launch_status(cudaGetLastError());
    }
    const size_t smem = std::max<size_t>(kDecMinSmem, kDecHeadBytes + (size_t)P.warps * P.stage);
    const int occ = occupancy((const void *)decode_batched_kernel, (int)P.warps * 32, smem);
    if (occ <= 0)
        return ECC_ERR_CUDA;
    const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, P.n_items / P.warps);
    decode_batched_kernel<<<(unsigned)grid, P.warps * 32, smem, st>>>((uint8_t *)ws, t_start);
    return launch_status(cudaGetLastError());
}

} // namespace

extern "C" {

size_t ecc_batched_workspace_bytes(const ecc_desc *descs, uint32_t count)
{
    // room for both directions: encode needs the look-back words, decode
    // the padded item map
    BatchPlan pe, pd;
    if (plan_batch(descs, count, true, false, &pe) != ECC_OK || plan_batch(descs, count, false, false, &pd) != ECC_OK)
        return 0;
    return std::max(layout_for(count, pe.n_items, pe.total_chunks).bytes, layout_for(count, pd.n_items, 0).bytes);
}

ecc_status ecc_encode_batched(const ecc_desc *descs, uint32_t count, void *ws, size_t ws_bytes, uint64_t *t_start_ns,
                              void *stream)
{
    return run_batched(descs, count, ws, ws_bytes, t_start_ns, stream, true);
}

ecc_status ecc_decode_batched(const ecc_desc *descs, uint32_t count, void *ws, size_t ws_bytes, uint64_t *t_start_ns,
                              void *stream)
{
    return run_batched(descs, count, ws, ws_bytes, t_start_ns, stream, false);
}

} // extern "C"
