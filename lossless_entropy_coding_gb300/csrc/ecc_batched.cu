// ecc_batched.cu -- one-launch encode and decode of many tensors, each with
// its own codebook and container sizes (the message regime of collective
// communication: many tensors of very different sizes).  See ecc.h.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "ecc_device.cuh"
#include "ecc_launch.h"

namespace ecc {

// Workspace layout (all offsets 16-byte aligned):
//   header | descs[count] | prefix[count + 1] | done[count] | flags[total]
// prefix[d] = first global work item of tensor d (chunks for encode, groups
// of `warps` chunks for decode); flags = look-back words (encode only).
struct BatchHeader {
    uint32_t ticket;
    uint32_t count;
    uint32_t warps;       // decode: chunks per work item
    uint32_t stage_bytes;
    uint32_t max_C;
    uint32_t nbuf; // encode: shared input buffers (2 = next chunk prefetched)
    uint64_t total_items;
    uint64_t total_chunks;
    uint64_t desc_off, prefix_off, done_off, flags_off;
};

struct BatchLayout {
    size_t desc_off, prefix_off, done_off, flags_off, bytes;
};

static size_t up16(size_t v) { return (v + 15) & ~size_t(15); }

static BatchLayout layout_for(uint32_t count, uint64_t total_chunks)
{
    BatchLayout L;
    L.desc_off = up16(sizeof(BatchHeader));
    L.prefix_off = up16(L.desc_off + (size_t)count * sizeof(ecc_desc));
    L.done_off = up16(L.prefix_off + ((size_t)count + 1) * sizeof(uint64_t));
    L.flags_off = up16(L.done_off + (size_t)count * sizeof(uint32_t));
    L.bytes = up16(L.flags_off + total_chunks * sizeof(uint64_t));
    return L;
}

__device__ __forceinline__ uint32_t find_tensor(const uint64_t *prefix, uint32_t count, uint64_t item)
{
    // largest d with prefix[d] <= item (prefix is non-decreasing; empty
    // tensors share a prefix with their successor and are skipped)
    uint32_t lo = 0, hi = count; // invariant: prefix[lo] <= item < prefix[hi]
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (prefix[mid] <= item)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__global__ void batch_prologue_kernel(uint8_t *ws, int encode)
{
    BatchHeader *h = reinterpret_cast<BatchHeader *>(ws);
    const ecc_desc *descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    uint32_t *done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    uint64_t *flags = reinterpret_cast<uint64_t *>(ws + h->flags_off);
    const uint64_t i0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = i0; i < h->count; i += stride) {
        const ecc_desc &d = descs[i];
        *d.status = ECC_OK;
        done[i] = 0;
        if (encode) {
            *d.total_bits = 0;
            d.chunk_off[0] = 0;
        }
        if (d.t_done_ns && d.n == 0)
            *d.t_done_ns = 0;
    }
    if (encode)
        for (uint64_t i = i0; i < h->total_chunks; i += stride)
            flags[i] = 0;
}

__device__ __forceinline__ void stamp_done(const ecc_desc &d, uint32_t *done, uint32_t k, uint64_t n_chunks,
                                           uint32_t items)
{
    if (!d.t_done_ns)
        return;
    __threadfence();
    if (atomicAdd(done + k, items) + items == n_chunks)
        *d.t_done_ns = globaltimer();
}

__device__ __forceinline__ EncJob batch_job(const ecc_desc &d, uint64_t *flags, const uint64_t *prefix, uint32_t k)
{
    return EncJob{d.in, d.n, d.cb, d.C, d.S, d.out, d.cap, d.chunk_off, d.sub_bits, d.total_bits,
                  flags + prefix[k], d.status};
}

// Work items are claimed one ahead by thread 0, which also finds the item's
// tensor (binary search over the prefix table) and copies its descriptor
// into shared memory, so the other threads never wait on that search.
struct BatchSlot {
    ecc_desc d;
    uint64_t item;   // global work item (ticket)
    uint32_t tensor; // index of the tensor it belongs to
    uint32_t pad;
};
constexpr uint32_t kBatchSlotBytes = 2 * ((sizeof(BatchSlot) + 15) & ~15u);

__global__ void __launch_bounds__(kEncThreads) encode_batched_kernel(uint8_t *ws, uint64_t *t_start)
{
    extern __shared__ __align__(16) uint8_t smem[];
    EncShared &sh = *reinterpret_cast<EncShared *>(smem);
    BatchHeader *h = reinterpret_cast<BatchHeader *>(ws);
    const ecc_desc *descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    const uint64_t *prefix = reinterpret_cast<const uint64_t *>(ws + h->prefix_off);
    uint32_t *done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    uint64_t *flags = reinterpret_cast<uint64_t *>(ws + h->flags_off);
    const uint32_t stage_bytes = h->stage_bytes;
    const uint32_t cmax = h->max_C;
    const uint32_t nbuf = h->nbuf;
    BatchSlot *slot = reinterpret_cast<BatchSlot *>(smem + enc_shared_bytes());
    uint8_t *inbuf = smem + enc_shared_bytes() + kBatchSlotBytes;
    uint32_t *stage = reinterpret_cast<uint32_t *>(inbuf + (size_t)nbuf * cmax);
    const int tid = threadIdx.x;
    if (t_start && blockIdx.x == 0 && tid == 0)
        *t_start = globaltimer();
    if (tid == 0) {
        sh.loaded = nullptr;
        mbar_init(&sh.bar[0], 1);
        mbar_init(&sh.bar[1], 1);
        fence_mbar_init();
    }
    uint4 *st4 = reinterpret_cast<uint4 *>(stage);
    for (uint32_t i = tid; i < stage_bytes / 16; i += kEncThreads)
        st4[i] = make_uint4(0, 0, 0, 0);
    // thread 0: claim the next chunk into slot q (and bulk-copy its input)
    uint32_t pending = 0;
    auto claim = [&](uint32_t q, bool copy) {
        const uint32_t t = atomicAdd(&h->ticket, 1u);
        slot[q].item = t;
        if (t < h->total_chunks) {
            const uint32_t k = find_tensor(prefix, h->count, t);
            slot[q].tensor = k;
            slot[q].d = descs[k];
            if (copy) {
                issue_chunk_input(batch_job(slot[q].d, flags, prefix, k), t - prefix[k],
                                  inbuf + (size_t)q * cmax, &sh.bar[q]);
                pending |= 1u << q;
            }
        }
    };
    if (tid == 0)
        claim(0, true);
    __syncthreads();
    uint32_t b = 0, phase = 0;
    bool staging = true;
    for (;;) {
        const uint64_t t = slot[b].item;
        if (t >= h->total_chunks)
            break;
        const uint32_t k = slot[b].tensor;
        const ecc_desc d = slot[b].d;
        __syncthreads(); // every thread has read slot b before it is refilled
        if (tid == 0 && nbuf == 2)
            claim(b ^ 1, staging);
        const uint64_t c = t - prefix[k];
        const EncJob job = batch_job(d, flags, prefix, k);
        const bool cb_ok = d.cb->magic == ECC_CODEBOOK_MAGIC && d.cb->max_len <= ECC_MAX_CODE_LEN;
        if (cb_ok && d.cb != sh.loaded) {
            load_encode_lut(sh, d.cb);
            __syncthreads();
            if (tid == 0)
                sh.loaded = d.cb;
        }
        const uint32_t ib = nbuf == 2 ? b : 0u;
        bool ok = staging && mbar_wait(&sh.bar[ib], (phase >> ib) & 1u, kWaitLimitNs);
        ok = __syncthreads_and(ok) != 0;
        if (ok) {
            phase ^= 1u << ib;
            if (tid == 0)
                pending &= ~(1u << ib);
        } else {
            if (staging && tid == 0)
                set_status(d.status, ECC_ERR_TIMEOUT);
            staging = false;
        }
        if (cb_ok) {
            if (ok)
                encode_chunk<true>(sh, stage, stage_bytes, job, inbuf + (size_t)ib * cmax, c, kWaitLimitNs);
            else
                encode_chunk<false>(sh, stage, stage_bytes, job, nullptr, c, kWaitLimitNs);
        } else if (tid < 32) {
            // keep the tensor's look-back moving; its status says why it is empty
            bool to;
            const uint64_t pre = lookback(job.flags, c, 0, kWaitLimitNs, &to);
            if (tid == 0) {
                set_status(d.status, ECC_ERR_CODEBOOK);
                d.chunk_off[c + 1] = pre;
            }
        }
        if (tid == 0) {
            stamp_done(d, done, k, (d.n + d.C - 1) / d.C, 1);
            if (nbuf == 1)
                claim(0, staging); // the single buffer is free again
        }
        __syncthreads();
        if (nbuf == 2)
            b ^= 1;
    }
    if (tid == 0)
        for (uint32_t q = 0; q < 2; ++q)
            if (pending & (1u << q))
                (void)mbar_wait(&sh.bar[q], (phase >> q) & 1u, kWaitLimitNs);
}

__global__ void decode_batched_kernel(uint8_t *ws, uint64_t *t_start)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *dec = reinterpret_cast<uint16_t *>(smem);
    LongTable &lt = *reinterpret_cast<LongTable *>(smem + kDecTableBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kDecTableBytes + kLongTableBytes);
    BatchSlot *slot = reinterpret_cast<BatchSlot *>(smem + kDecHeadBytes);
    __shared__ const ecc_codebook *loaded;
    BatchHeader *h = reinterpret_cast<BatchHeader *>(ws);
    const ecc_desc *descs = reinterpret_cast<const ecc_desc *>(ws + h->desc_off);
    const uint64_t *prefix = reinterpret_cast<const uint64_t *>(ws + h->prefix_off);
    uint32_t *done = reinterpret_cast<uint32_t *>(ws + h->done_off);
    const uint32_t stage_bytes = h->stage_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t warps = h->warps;
    if (t_start && blockIdx.x == 0 && threadIdx.x == 0)
        *t_start = globaltimer();
    if (lane == 0) {
        mbar_init(&bars[warp], 1);
        fence_mbar_init();
    }
    auto claim = [&](uint32_t q) {
        const uint32_t g = atomicAdd(&h->ticket, 1u);
        slot[q].item = g;
        if (g < h->total_items) {
            const uint32_t k = find_tensor(prefix, h->count, g);
            slot[q].tensor = k;
            slot[q].d = descs[k];
        }
    };
    if (threadIdx.x == 0) {
        loaded = nullptr;
        claim(0);
    }
    __syncthreads();
    WarpStage wst{reinterpret_cast<uint32_t *>(smem + kDecHeadBytes + kBatchSlotBytes + (size_t)warp * stage_bytes),
                  stage_bytes, &bars[warp], 0};
    for (uint32_t b = 0;; b ^= 1) {
        const uint64_t g = slot[b].item;
        if (g >= h->total_items)
            break;
        const uint32_t k = slot[b].tensor;
        const ecc_desc d = slot[b].d;
        __syncthreads(); // every thread has read slot b
        if (threadIdx.x == 0)
            claim(b ^ 1);
        const uint64_t n_chunks = (d.n + d.C - 1) / d.C;
        const uint64_t c = (g - prefix[k]) * warps + warp;
        const bool cb_ok = d.cb->magic == ECC_CODEBOOK_MAGIC && d.cb->max_len <= ECC_MAX_CODE_LEN;
        if (cb_ok && d.cb != loaded) {
            const uint4 *src = reinterpret_cast<const uint4 *>(d.cb->dec);
            uint4 *dst = reinterpret_cast<uint4 *>(dec);
            for (int i = threadIdx.x; i < (int)(kDecTableBytes / 16); i += blockDim.x)
                dst[i] = src[i];
            load_long_table(lt, d.cb);
            __syncthreads();
            if (threadIdx.x == 0)
                loaded = d.cb;
        }
        if (c < n_chunks) {
            if (cb_ok) {
                DecJob job{d.in, d.cap, d.chunk_off, d.sub_bits, d.n, d.C, d.S, d.cb, d.out, d.status};
                const uint32_t per_lane = (d.C >> (31 - __clz(d.S))) >> 5; // (C/S)/32
                if (per_lane >= 4)
                    decode_chunk<4>(job, dec, lt, wst, c, c + warps, n_chunks);
                else if (per_lane >= 2)
                    decode_chunk<2>(job, dec, lt, wst, c, c + warps, n_chunks);
                else
                    decode_chunk<1>(job, dec, lt, wst, c, c + warps, n_chunks);
            } else if (lane == 0) {
                set_status(d.status, ECC_ERR_CODEBOOK);
            }
            if (lane == 0)
                stamp_done(d, done, k, n_chunks, 1);
        }
        __syncthreads();
    }
}

} // namespace ecc

using namespace ecc;

namespace {

ecc_status check_descs(const ecc_desc *descs, uint32_t count, bool encode, uint64_t *total_chunks, uint32_t *max_C)
{
    if (!descs || count == 0)
        return ECC_ERR_ARG;
    uint64_t tot = 0;
    uint32_t mc = 1024;
    for (uint32_t i = 0; i < count; ++i) {
        const ecc_desc &d = descs[i];
        if (!valid_sizes(d.C, d.S) || !d.cb || !aligned16(d.cb) || !d.status || !d.chunk_off)
            return ECC_ERR_ARG;
        if (encode && !d.total_bits)
            return ECC_ERR_ARG;
        if (d.n && (!d.in || !d.out || !d.sub_bits || !aligned16(d.in) || !aligned16(d.out)))
            return ECC_ERR_ARG;
        tot += ecc_num_chunks(d.n, d.C);
        mc = std::max(mc, d.C);
    }
    *total_chunks = tot;
    *max_C = mc;
    return ECC_OK;
}

ecc_status run_batched(const ecc_desc *descs, uint32_t count, void *ws, size_t ws_bytes, uint64_t *t_start,
                       void *stream, bool encode)
{
    uint64_t total_chunks;
    uint32_t max_C;
    ecc_status e = check_descs(descs, count, encode, &total_chunks, &max_C);
    if (e != ECC_OK)
        return e;
    BatchLayout L = layout_for(count, total_chunks);
    if (!ws || !aligned16(ws) || ws_bytes < L.bytes)
        return ECC_ERR_ARG;
    const uint32_t stage = stage_bytes_for(max_C);
    int warps = decode_warps(stage);
    while (warps > 1 && kDecHeadBytes + kBatchSlotBytes + (size_t)warps * stage > kMaxDynSmem - kStaticSmemReserve)
        --warps;
    // host image of header | descs | prefix, copied with one async copy
    std::vector<uint8_t> img(L.done_off, 0);
    BatchHeader *h = reinterpret_cast<BatchHeader *>(img.data());
    h->ticket = 0;
    h->count = count;
    h->warps = (uint32_t)warps;
    h->stage_bytes = stage;
    h->max_C = max_C;
    h->nbuf = enc_input_buffers(max_C);
    h->total_chunks = total_chunks;
    h->desc_off = L.desc_off;
    h->prefix_off = L.prefix_off;
    h->done_off = L.done_off;
    h->flags_off = L.flags_off;
    std::memcpy(img.data() + L.desc_off, descs, (size_t)count * sizeof(ecc_desc));
    uint64_t *prefix = reinterpret_cast<uint64_t *>(img.data() + L.prefix_off);
    uint64_t acc = 0;
    for (uint32_t i = 0; i < count; ++i) {
        prefix[i] = acc;
        const uint64_t nc = ecc_num_chunks(descs[i].n, descs[i].C);
        acc += encode ? nc : (nc + warps - 1) / warps;
    }
    prefix[count] = acc;
    h->total_items = acc;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(ws, img.data(), img.size(), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return launch_status(cudaErrorUnknown);
    const int sms = sm_count();
    if (sms <= 0)
        return ECC_ERR_CUDA;
    {
        const uint64_t work = std::max<uint64_t>(count, encode ? total_chunks : 0);
        const uint64_t nb = std::max<uint64_t>(1, std::min<uint64_t>((work + 255) / 256, 1024));
        batch_prologue_kernel<<<(unsigned)nb, 256, 0, st>>>((uint8_t *)ws, encode ? 1 : 0);
        if ((e = launch_status(cudaGetLastError())) != ECC_OK)
            return e;
    }
    if (acc == 0)
        return ECC_OK;
    if (encode) {
        const size_t smem = enc_shared_bytes() + kBatchSlotBytes + (size_t)h->nbuf * max_C + stage;
        const int occ = occupancy((const void *)encode_batched_kernel, kEncThreads, smem);
        if (occ <= 0)
            return ECC_ERR_CUDA;
        const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, acc);
        encode_batched_kernel<<<(unsigned)grid, kEncThreads, smem, st>>>((uint8_t *)ws, t_start);
    } else {
        const size_t smem = kDecHeadBytes + kBatchSlotBytes + (size_t)warps * stage;
        const int occ = occupancy((const void *)decode_batched_kernel, warps * 32, smem);
        if (occ <= 0)
            return ECC_ERR_CUDA;
        const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, acc);
        decode_batched_kernel<<<(unsigned)grid, warps * 32, smem, st>>>((uint8_t *)ws, t_start);
    }
    return launch_status(cudaGetLastError());
}

} // namespace

extern "C" {

size_t ecc_batched_workspace_bytes(const ecc_desc *descs, uint32_t count)
{
    if (!descs || !count)
        return 0;
    uint64_t tot = 0;
    for (uint32_t i = 0; i < count; ++i)
        tot += ecc_num_chunks(descs[i].n, descs[i].C ? descs[i].C : 1);
    return layout_for(count, tot).bytes;
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
