// ecc_kernels.cu -- sm_103a kernels and C-ABI launchers for single tensors:
// byte histogram, chunk-parallel encode with decoupled look-back, and
// warp-per-chunk decode.  See include/ecc.h for the contract.

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "ecc_device.cuh"
#include "ecc_launch.h"

namespace ecc {

// ---------------------------------------------------------------- histogram
// e4m3_histogram: lane-private counters in shared memory, counter b of lane
// l at word b * 32 + l, so every lane of a shared atomic hits its own bank
// and no two lanes of one instruction share an address (one pass per warp
// instruction, whatever the byte distribution).  All 16 warps of a CTA
// share the one 32 KB set: atomics of different instructions to one address
// cost no extra pass.  Each warp streams 4 KB chunks (8 16-byte vectors a
// lane, the next chunk's loads in flight while this one is counted) and asks
// L2 for the chunk after that with a bulk prefetch.  At the end one warp per
// bin sums the 32 lanes' counters and adds them to the 64-bit count with one
// global atomic per non-empty bin per CTA.  A counter sums the bytes of one
// lane position of 16 warps, about n / (CTAs x 32): it fits 32 bits while n
// < 2^37 x CTAs, for any tensor that fits in device memory.
constexpr int kHistWarps = 16;
constexpr int kHistThreads = kHistWarps * 32;
constexpr int kHistVec = 8;                                // 16-byte vectors a lane per chunk
constexpr uint32_t kHistChunk = 32 * kHistVec * 16;        // bytes a warp counts per chunk
constexpr size_t kHistSmem = 256 * 32 * 4;

// L2 prefetch of the chunk at byte offset off of the body, if any
__device__ __forceinline__ void prefetch_chunk(const uint8_t *body, uint64_t off, uint64_t body_bytes)
{
    if (off < body_bytes)
        prefetch_l2(body + off, (uint32_t)(body_bytes - off < kHistChunk ? body_bytes - off : kHistChunk));
}

__device__ __forceinline__ void count_word(uint32_t *mine, uint32_t w)
{
#pragma unroll
    for (int k = 0; k < 4; ++k)
        atomicAdd(mine + (byte_of(w, k) << 5), 1u);
}

__global__ void __launch_bounds__(kHistThreads, 1) hist_kernel(const uint8_t *in, uint64_t n, uint64_t head,
                                                              unsigned long long *count)
{
    extern __shared__ __align__(16) uint32_t hist_smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t *const mine = hist_smem + lane;
    for (int i = tid; i < 256 * 32 / 4; i += kHistThreads)
        reinterpret_cast<uint4 *>(hist_smem)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    // unaligned head and the tail bytes: CTA 0
    const uint64_t nvec = (n - head) / 16;
    const uint64_t tail0 = head + nvec * 16;
    if (blockIdx.x == 0) {
        for (uint64_t i = tid; i < head; i += kHistThreads)
            atomicAdd(mine + ((uint32_t)in[i] << 5), 1u);
        for (uint64_t i = tail0 + tid; i < n; i += kHistThreads)
            atomicAdd(mine + ((uint32_t)in[i] << 5), 1u);
    }
    const uint4 *body = reinterpret_cast<const uint4 *>(in + head);
    const uint64_t body_bytes = nvec * 16;
    const uint64_t W = (uint64_t)gridDim.x * kHistWarps;
    constexpr uint64_t kv = 32 * kHistVec; // vectors a chunk
    uint64_t ch = (uint64_t)blockIdx.x * kHistWarps + warp;
    if (lane == 0) {
        prefetch_chunk((const uint8_t *)body, ch * kHistChunk, body_bytes);
        prefetch_chunk((const uint8_t *)body, (ch + W) * kHistChunk, body_bytes);
    }
    uint4 cur[kHistVec];
#pragma unroll
    for (int u = 0; u < kHistVec; ++u) {
        const uint64_t v = ch * kv + u * 32 + lane;
        cur[u] = v < nvec ? ld_stream16(body + v) : make_uint4(0, 0, 0, 0);
    }
    for (; ch * kv < nvec; ch += W) {
        const uint64_t nx = ch + W;
        if (lane == 0)
            prefetch_chunk((const uint8_t *)body, (nx + W) * kHistChunk, body_bytes);
        uint4 nxt[kHistVec];
#pragma unroll
        for (int u = 0; u < kHistVec; ++u) {
            const uint64_t v = nx * kv + u * 32 + lane;
            nxt[u] = v < nvec ? ld_stream16(body + v) : make_uint4(0, 0, 0, 0);
        }
        if (ch * kv + kv <= nvec) {
#pragma unroll
            for (int u = 0; u < kHistVec; ++u) {
                count_word(mine, cur[u].x);
                count_word(mine, cur[u].y);
                count_word(mine, cur[u].z);
                count_word(mine, cur[u].w);
            }
        } else {
#pragma unroll
            for (int u = 0; u < kHistVec; ++u)
                if (ch * kv + u * 32 + lane < nvec) {
                    count_word(mine, cur[u].x);
                    count_word(mine, cur[u].y);
                    count_word(mine, cur[u].z);
                    count_word(mine, cur[u].w);
                }
        }
#pragma unroll
        for (int u = 0; u < kHistVec; ++u)
            cur[u] = nxt[u];
    }
    __syncthreads();
    for (int b = warp; b < 256; b += kHistWarps) {
        uint32_t c = hist_smem[b * 32 + lane];
#pragma unroll
        for (int o = 16; o; o >>= 1)
            c += __shfl_xor_sync(~0u, c, o);
        if (lane == 0 && c)
            atomicAdd(count + b, (unsigned long long)c);
    }
}

// ---------------------------------------------------------------- encode
struct EncParams {
    EncJob job;
    uint64_t n_chunks;
    uint32_t *ticket;
    uint32_t stage_bytes;
    uint32_t nbuf; // shared input buffers of C bytes: 2 = next chunk prefetched
    uint64_t timeout_ns;
    uint32_t group; // warp-specialised kernel: chunks coded as one unit
};

// zero the look-back flags, the ticket and the outputs the kernel accumulates
__global__ void enc_prologue_kernel(uint64_t *flags, uint64_t n_flags, uint32_t *ticket, uint64_t *total_bits,
                                    uint64_t *chunk_off, uint32_t *status)
{
    const uint64_t i0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (uint64_t i = i0; i < n_flags; i += (uint64_t)gridDim.x * blockDim.x)
        flags[i] = 0;
    if (i0 == 0) {
        *ticket = 0;
        *total_bits = 0;
        chunk_off[0] = 0;
        *status = ECC_OK;
    }
}

// Persistent CTAs take chunks in ticket order, so a chunk's predecessors have
// always been claimed by running CTAs when it looks back.  Each CTA claims
// its next chunk one chunk ahead and bulk-copies that chunk's input into the
// second shared buffer while it encodes the current one.
__global__ void __launch_bounds__(kEncThreads, 2) encode_kernel(EncParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    EncShared &sh = *reinterpret_cast<EncShared *>(smem);
    uint8_t *inbuf = smem + enc_shared_bytes();
    uint32_t *stage = reinterpret_cast<uint32_t *>(inbuf + (size_t)p.nbuf * p.job.C + kStageLead);
    const int tid = threadIdx.x;
    if (p.job.cb->magic != ECC_CODEBOOK_MAGIC || p.job.cb->max_len > ECC_MAX_CODE_LEN) {
        if (tid == 0 && blockIdx.x == 0)
            set_status(p.job.status, ECC_ERR_CODEBOOK);
        return;
    }
    if (tid == 0) {
        mbar_init(&sh.bar[0], 1);
        mbar_init(&sh.bar[1], 1);
        fence_mbar_init();
    }
    load_encode_lut(sh, p.job.cb, kEncThreads);
    uint4 *st4 = reinterpret_cast<uint4 *>(inbuf + (size_t)p.nbuf * p.job.C); // the guard word and the stage
    for (uint32_t i = tid; i < (kStageLead + p.stage_bytes) / 16; i += kEncThreads)
        st4[i] = make_uint4(0, 0, 0, 0);
    uint32_t pending = 0; // thread 0: buffers with a copy not yet waited for
    if (tid == 0) {
        const uint32_t t = atomicAdd(p.ticket, 1u);
        sh.ticket = t;
        if (t < p.n_chunks) {
            issue_chunk_input(p.job, t, inbuf, &sh.bar[0]);
            pending = 1;
        }
    }
    __syncthreads();
    uint64_t c = sh.ticket;
    uint32_t b = 0, phase = 0;
    bool staging = true;
    while (c < p.n_chunks) {
        __syncthreads(); // every thread has read sh.ticket
        if (tid == 0) {
            const uint32_t t = atomicAdd(p.ticket, 1u);
            sh.ticket = t;
            if (t < p.n_chunks && p.nbuf == 2 && staging) {
                issue_chunk_input(p.job, t, inbuf + (size_t)(b ^ 1) * p.job.C, &sh.bar[b ^ 1]);
                pending |= 1u << (b ^ 1);
            }
        }
        bool ok = staging && mbar_wait(&sh.bar[b], (phase >> b) & 1u, p.timeout_ns);
        ok = __syncthreads_and(ok) != 0;
        if (ok) {
            phase ^= 1u << b;
            if (tid == 0)
                pending &= ~(1u << b);
            encode_chunk<true>(sh, stage, p.stage_bytes, p.job, inbuf + (size_t)b * p.job.C, c, p.timeout_ns);
        } else {
            // the copy did not arrive in time: report it, stop staging, and
            // read this and later chunks from global memory
            if (staging && tid == 0)
                set_status(p.job.status, ECC_ERR_TIMEOUT);
            staging = false;
            encode_chunk<false>(sh, stage, p.stage_bytes, p.job, nullptr, c, p.timeout_ns);
        }
        const uint64_t nc = sh.ticket;
        if (p.nbuf == 1 && staging && tid == 0 && nc < p.n_chunks) {
            issue_chunk_input(p.job, nc, inbuf, &sh.bar[0]);
            pending |= 1u;
        }
        if (p.nbuf == 2)
            b ^= 1;
        c = nc;
    }
    // never exit with a bulk copy still writing into this CTA's shared memory
    if (tid == 0)
        for (uint32_t k = 0; k < 2; ++k)
            if (pending & (1u << k))
                (void)mbar_wait(&sh.bar[k], (phase >> k) & 1u, p.timeout_ns);
}

// Warp-specialised encoder over one tensor: see encode_ws_body.  At most 96
// registers a thread, so that two 288-thread CTAs fit one SM.
template <bool kGrouped>
__global__ void __maxnreg__(96) encode_ws_kernel(EncParams p)
{
    const EncBatch none{};
    encode_ws_body<false, kGrouped>(p.job, p.n_chunks, p.ticket, none, p.stage_bytes, p.job.C * p.group,
                                    p.timeout_ns, p.group);
}

// ---------------------------------------------------------------- chunks of more than kGroupSyms symbols
// Length pass: flags[c] = the payload bits of chunk c (the same table
// lookups as the encoder's), bit 63 set when one of its segments of kPassSeg
// symbols needs more than its stage region.  A CTA takes one chunk at a
// time; warp w sums segments w, w + 8, ... reading the input straight from
// global memory, a segment's four 16-byte loads a lane issued together.
__global__ void __launch_bounds__(kEncThreads) enc_len_kernel(const uint8_t *in, uint64_t n, const ecc_codebook *cb,
                                                              uint32_t C, uint64_t n_chunks, uint64_t *flags)
{
    extern __shared__ __align__(16) uint8_t smem[];
    EncShared &sh = *reinterpret_cast<EncShared *>(smem);
    __shared__ uint32_t wbits[kEncWarps], wover[kEncWarps];
    if (cb->magic != ECC_CODEBOOK_MAGIC || cb->max_len > ECC_MAX_CODE_LEN)
        return; // the encoder reports it
    load_encode_lut(sh, cb, kEncThreads);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint2 *lut = sh.lut + (lane & (kLutReplicas - 1));
    const uint32_t cap = region_cap_bytes(kPassSeg) * 8u;
    for (uint64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
        const uint64_t base = c * C;
        const uint32_t L = (uint32_t)min((uint64_t)C, n - base);
        uint32_t bits = 0, over = 0;
        for (uint32_t s0 = (uint32_t)warp * kPassSeg; s0 < L; s0 += kEncWarps * kPassSeg) {
            const uint32_t s1 = min(s0 + kPassSeg, L);
            uint4 v[kPassSeg / kRoundSyms];
            uint32_t cnt[kPassSeg / kRoundSyms];
#pragma unroll
            for (uint32_t r = 0; r < kPassSeg / kRoundSyms; ++r) {
                const uint32_t my0 = s0 + r * kRoundSyms + (uint32_t)lane * kSymPerThread;
                cnt[r] = my0 < s1 ? min((uint32_t)kSymPerThread, s1 - my0) : 0u;
                v[r] = cnt[r] ? load_symbols<false>(nullptr, in + base + my0, cnt[r]) : make_uint4(0, 0, 0, 0);
            }
            uint32_t sb = 0;
#pragma unroll
            for (uint32_t r = 0; r < kPassSeg / kRoundSyms; ++r) {
                uint32_t pv[8], pq[8];
                bool slow;
                uint32_t g = lookup_pairs(lut, v[r], cnt[r], pv, pq, &slow);
                if (slow)
                    g = cnt[r] ? slow_group_bits(lut, v[r], cnt[r], cb) & 0x3FFFFFFFu : 0u;
                sb += g;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1)
                sb += __shfl_xor_sync(~0u, sb, o);
            bits += sb;
            over |= sb > cap ? 1u : 0u;
        }
        if (lane == 0) {
            wbits[warp] = bits;
            wover[warp] = over;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            uint64_t t = 0;
            uint32_t o = 0;
            for (int w = 0; w < kEncWarps; ++w) {
                t += wbits[w];
                o |= wover[w];
            }
            flags[c] = t | (o ? kLenOverflow : 0ull);
        }
        __syncthreads();
    }
}

// Scan of the length pass (one CTA of 1024 threads, 1024 chunks a step):
// chunk_off[c + 1] = the padded bytes of chunks 0 .. c, total_bits, and
// ECC_ERR_CAPACITY when the payload exceeds out_cap.
__global__ void __launch_bounds__(1024) enc_scan_kernel(const uint64_t *flags, uint64_t n_chunks, uint64_t *chunk_off,
                                                        uint64_t *total_bits, uint64_t out_cap, uint32_t *status)
{
    __shared__ uint64_t wsum[32];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    uint64_t carry = 0, tbits = 0;
    for (uint64_t t0 = 0; t0 < n_chunks; t0 += 1024) {
        const uint64_t c = t0 + (uint64_t)t;
        const uint64_t bits = c < n_chunks ? flags[c] & ~kLenOverflow : 0ull;
        tbits += bits;
        uint64_t incl = (bits + 127u) / 128u * 16u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(~0u, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane == 31)
            wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            uint64_t v = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint64_t y = __shfl_up_sync(~0u, v, o);
                if (lane >= o)
                    v += y;
            }
            wsum[lane] = v;
        }
        __syncthreads();
        if (c < n_chunks)
            chunk_off[c + 1] = carry + (warp ? wsum[warp - 1] : 0ull) + incl;
        carry += wsum[31];
        __syncthreads(); // wsum is rewritten by the next step
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        tbits += __shfl_xor_sync(~0u, tbits, o);
    if (lane == 0)
        wsum[warp] = tbits;
    __syncthreads();
    if (t == 0) {
        uint64_t sum = 0;
        for (int w = 0; w < 32; ++w)
            sum += wsum[w];
        *total_bits = sum;
        chunk_off[0] = 0;
        if (carry > out_cap)
            set_status(status, ECC_ERR_CAPACITY);
    }
}

// Pass encoder over one tensor (C > kGroupSyms): see encode_pass_body.
__global__ void __maxnreg__(96) encode_pass_kernel(EncParams p)
{
    encode_pass_body(p.job, p.n_chunks, p.ticket, p.stage_bytes, p.timeout_ns);
}

// ---------------------------------------------------------------- decode
struct DecParams {
    DecJob job;
    uint64_t n_chunks;
    uint32_t stage_bytes;
    uint32_t pshift; // log2(pieces per chunk): warps take chunks (0) or pieces of chunks
};

// kPieces: the warps take pieces of chunks (p.pshift > 0), else chunks.
// One or two streams a lane: at most 96 registers, so that up to 21 warps
// fit an SM where the stages allow (smaller chunks); four: at most 136.
template <int R, bool kPieces>
__global__ void __maxnreg__(R >= 4 ? 136 : 96) decode_kernel(DecParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *dec = reinterpret_cast<uint16_t *>(smem);
    LongTable &lt = *reinterpret_cast<LongTable *>(smem + kDecTableBytes);
    QlcShared &qs = *reinterpret_cast<QlcShared *>(smem + kDecTableBytes + kLongTableBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kDecTableBytes + kLongTableBytes + kQlcSharedBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ecc_codebook *cb = p.job.cb;
    if (cb->magic != ECC_CODEBOOK_MAGIC || cb->max_len > ECC_MAX_CODE_LEN) {
        if (threadIdx.x == 0 && blockIdx.x == 0)
            set_status(p.job.status, ECC_ERR_CODEBOOK);
        return;
    }
    const bool qlc = qlc_mode(cb);
    if (qlc) {
        load_qlc_tables(reinterpret_cast<uint32_t *>(smem), qs, cb, blockDim.x);
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(cb->dec);
        uint4 *dst = reinterpret_cast<uint4 *>(dec);
        for (int i = threadIdx.x; i < (int)(kDecTableBytes / 16); i += blockDim.x)
            dst[i] = src[i];
    }
    load_long_table(lt, cb);
    __shared__ uint32_t next_item; // the CTA's chunks blockIdx.x + k * gridDim.x, claimed by k in turn
    if (lane == 0) {
        mbar_init(&bars[warp], 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0)
        next_item = 0;
    __syncthreads();
    if (lt.sub_np) { // the long codes' second level (the same decision in every thread)
        fill_long_sub(lt, threadIdx.x, blockDim.x);
        __syncthreads();
    }
    WarpStage ws{reinterpret_cast<uint32_t *>(smem + kDecHeadBytes + (size_t)warp * p.stage_bytes), p.stage_bytes,
                 &bars[warp], 0};
    // The warps of a CTA claim its chunks one at a time, so a warp that
    // drew chunks with many long codes does not hold up the CTA's end; a
    // warp claims its next chunk before decoding the current one, so that
    // (whole chunks) the next one's L2 prefetch starts early.
    auto claim = [&]() -> uint64_t {
        uint32_t k = 0;
        if (lane == 0)
            k = atomicAdd(&next_item, 1u);
        return blockIdx.x + (uint64_t)__shfl_sync(~0u, k, 0) * gridDim.x;
    };
    uint64_t c = claim();
    const uint32_t ps = p.pshift, pm = (1u << ps) - 1u;
    const uint64_t n_items = p.n_chunks << ps;
    if (qlc) {
        const DecTables T = qlc_tables(cb->dec, &lt, qs, reinterpret_cast<const uint32_t *>(smem));
        if constexpr (kPieces) {
            while (c < n_items) {
                const uint64_t nc = claim();
                decode_piece<R, true>(p.job, T, ws, c >> ps, (uint32_t)c & pm, ps);
                c = nc;
            }
        } else {
            while (c < p.n_chunks) {
                const uint64_t nc = claim();
                decode_chunk<R, true>(p.job, T, ws, c, nc, p.n_chunks);
                c = nc;
            }
        }
    } else {
        DecTables T{};
        T.dec = dec;
        T.lt = &lt;
        if constexpr (kPieces) {
            while (c < n_items) {
                const uint64_t nc = claim();
                decode_piece<R, false>(p.job, T, ws, c >> ps, (uint32_t)c & pm, ps);
                c = nc;
            }
        } else {
            while (c < p.n_chunks) {
                const uint64_t nc = claim();
                decode_chunk<R, false>(p.job, T, ws, c, nc, p.n_chunks);
                c = nc;
            }
        }
    }
}

// ---------------------------------------------------------------- self-test
__global__ void selftest_wait_kernel(uint64_t *flags, uint64_t chunk, uint64_t aggregate, uint64_t timeout_ns,
                                     uint64_t *prefix, uint32_t *status)
{
    bool to;
    const uint64_t pre = lookback(flags, chunk, aggregate, timeout_ns, &to);
    if (threadIdx.x == 0) {
        *prefix = pre;
        *status = to ? ECC_ERR_TIMEOUT : ECC_OK;
    }
}

// ---------------------------------------------------------------- host side
namespace {

struct DevInfo {
    int sms = 0;
    std::map<std::tuple<const void *, int, size_t>, int> occ; // (kernel, threads, smem) -> blocks/SM
};

std::mutex g_mu;
std::map<int, DevInfo> g_dev;

DevInfo *device_info()
{
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &d = g_dev[dev];
    if (!d.sms && cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        d.sms = 0;
        return nullptr;
    }
    return &d;
}

bool pow2_in(uint64_t v, uint64_t lo, uint64_t hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

} // namespace

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool valid_sizes(uint32_t C, uint32_t S) { return pow2_in(C, 1024, 65536) && pow2_in(S, 64, 1024) && S <= C; }

uint32_t enc_input_buffers(uint32_t C)
{
    // two CTAs per SM must fit: LUT + two input buffers + output staging
    const size_t two = enc_shared_bytes() + 2 * (size_t)C + kStageLead + stage_bytes_for(C);
    return two <= kMaxDynSmem / 2 - kStaticSmemReserve ? 2u : 1u;
}

static_assert(kDecMaxWarps <= (int)kDecBarSlots, "one stage mbarrier per decoding warp");

int decode_warps(uint32_t stage_bytes)
{
    const size_t room = kMaxDynSmem - kStaticSmemReserve - kDecHeadBytes;
    const int w = (int)std::min<size_t>(kDecMaxWarps, room / stage_bytes);
    return std::max(w, 1);
}

ecc_status launch_status(cudaError_t e)
{
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return ECC_ERR_CUDA;
    }
    return ECC_OK;
}

int sm_count()
{
    DevInfo *d = device_info();
    return d ? d->sms : 0;
}

int occupancy(const void *kernel, int threads, size_t smem)
{
    DevInfo *d = device_info();
    if (!d)
        return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(kernel, threads, smem);
    auto it = d->occ.find(key);
    if (it != d->occ.end())
        return it->second;
    int nb = 0;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess || fa.sharedSizeBytes + smem > kMaxDynSmem ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kMaxDynSmem - fa.sharedSizeBytes)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        nb = 0;
    }
    d->occ[key] = nb;
    return nb;
}

// The deferred pass (code_deferred_unit): warp w of W takes units w, w + W,
// w + 2W, ... (marked units come in runs: the long codes of one part of a
// tensor), 32 at a time, a lane each reading a look-back word, and codes the
// marked ones.  Chunks coded in parts (marks != NULL: chunks of 2^mlog parts,
// n_parts in all) are also coded when the mark word of the chunk (the word
// of its last part) is set and the chunk's offsets are published within the
// output.  A launch over a tensor with no marked unit only reads its
// look-back (and mark) words, all of a warp's at once.
__global__ void __launch_bounds__(256) encode_deferred_kernel(EncJob job, uint64_t n_chunks, uint32_t G,
                                                               const uint64_t *marks, uint32_t mlog, uint64_t n_parts)
{
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t n_units = (n_chunks + G - 1) / G;
    const uint64_t w0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nw = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t u0 = w0; u0 < n_units; u0 += 32 * nw) {
        const uint64_t u = u0 + lane * nw;
        bool d = false;
        if (u < n_units) {
            const uint64_t f = job.flags[u];
            d = is_deferred(f);
            if (!d && marks && (marks[min(((u + 1) << mlog) - 1u, n_parts - 1u)] & 1u) && (f >> 62) == 2u)
                d = job.chunk_off[u] <= job.chunk_off[u + 1] && job.chunk_off[u + 1] <= job.out_cap;
        }
        for (uint32_t m = __ballot_sync(~0u, d); m; m &= m - 1)
            code_deferred_unit(job, u0 + (uint64_t)(__ffs(m) - 1) * nw, G, n_chunks);
    }
}

ecc_status launch_deferred(const EncJob &job, uint64_t n_chunks, uint32_t G, cudaStream_t st, const uint64_t *marks,
                           uint32_t mlog, uint64_t n_parts)
{
    const int sms = sm_count();
    if (sms <= 0)
        return ECC_ERR_CUDA;
    const uint64_t n_units = (n_chunks + G - 1) / G;
    // a warp a unit, up to 8 CTAs of 8 warps an SM
    const uint64_t blocks = std::max<uint64_t>(1, std::min<uint64_t>((n_units + 7) / 8, (uint64_t)sms * 8));
    encode_deferred_kernel<<<(unsigned)blocks, 256, 0, st>>>(job, n_chunks, G, marks, mlog, n_parts);
    return launch_status(cudaGetLastError());
}

} // namespace ecc

using namespace ecc;

extern "C" {

size_t ecc_encode_workspace_bytes(size_t n, uint32_t C)
{
    if (!C)
        return 0;
    // a ticket; a look-back word per chunk; for chunks of more than kGroupSyms
    // symbols, also a word per kGroupSyms symbols (the unit encoder's units)
    const uint64_t units = C > kGroupSyms ? ecc_num_chunks(n, kGroupSyms) : 0;
    return 256 + (ecc_num_chunks(n, C) + units) * sizeof(uint64_t);
}

ecc_status e4m3_histogram(const uint8_t *in, size_t n, uint64_t *count, void *stream)
{
    if (!count || (n && !in))
        return ECC_ERR_ARG;
    if (!n)
        return ECC_OK;
    const int sms = sm_count();
    if (!sms)
        return ECC_ERR_CUDA;
    const uint64_t head = std::min<uint64_t>(n, (16 - ((uintptr_t)in & 15)) & 15);
    const uint64_t nvec = (n - head) / 16;
    if (occupancy((const void *)hist_kernel, kHistThreads, kHistSmem) <= 0)
        return launch_status(cudaErrorInvalidConfiguration);
    const uint64_t chunks = (nvec + 32 * kHistVec - 1) / (32 * kHistVec);
    const uint64_t blocks = std::max<uint64_t>(1, std::min<uint64_t>((chunks + kHistWarps - 1) / kHistWarps, sms));
    hist_kernel<<<(unsigned)blocks, kHistThreads, kHistSmem, (cudaStream_t)stream>>>(in, n, head,
                                                                                      (unsigned long long *)count);
    return launch_status(cudaGetLastError());
}

ecc_status ecc_encode(const uint8_t *in, size_t n, const ecc_codebook *cb, uint32_t C, uint32_t S, uint8_t *out,
                      size_t out_cap, uint64_t *chunk_off, uint16_t *sub_bits, uint64_t *total_bits, void *ws,
                      size_t ws_bytes, uint32_t *status, void *stream)
{
    if (!cb || !aligned16(cb) || !chunk_off || !total_bits || !status || !ws || !valid_sizes(C, S))
        return ECC_ERR_ARG;
    if (n && (!in || !out || !sub_bits || !aligned16(in) || !aligned16(out)))
        return ECC_ERR_ARG;
    if (!aligned16(ws) || ws_bytes < ecc_encode_workspace_bytes(n, C))
        return ECC_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const uint64_t n_chunks = ecc_num_chunks(n, C);
    uint32_t *ticket = (uint32_t *)ws;
    uint64_t *flags = (uint64_t *)((uint8_t *)ws + 256);
    {
        const uint64_t n_flags = (ecc_encode_workspace_bytes(n, C) - 256) / sizeof(uint64_t);
        const uint64_t nb = std::max<uint64_t>(1, std::min<uint64_t>((n_flags + 255) / 256, 1024));
        enc_prologue_kernel<<<(unsigned)nb, 256, 0, st>>>(flags, n_flags, ticket, total_bits, chunk_off, status);
        ecc_status e = launch_status(cudaGetLastError());
        if (e != ECC_OK || !n)
            return e;
    }
    EncParams p;
    p.job = EncJob{in, n, cb, C, S, out, out_cap, chunk_off, sub_bits, total_bits, flags, status};
    p.n_chunks = n_chunks;
    p.ticket = ticket;
    p.stage_bytes = stage_bytes_for(C);
    p.timeout_ns = kWaitLimitNs;
    p.group = 1;
    const int sms = sm_count();
    if (sms <= 0)
        return ECC_ERR_CUDA;
    // the unit encoder (ecc_units.cu), then the deferred pass over the units
    // (or split chunks) it could not stage
    uint32_t unit_chunks = 1;
    if (launch_unit_encoder(p.job, ticket, st, &unit_chunks) == ECC_OK) {
        if (C <= kGroupSyms)
            return launch_deferred(p.job, n_chunks, unit_chunks, st, nullptr, 0, 0);
        // chunks coded in parts of kGroupSyms symbols: their mark words follow the chunks' words
        return launch_deferred(p.job, n_chunks, 1, st, flags + n_chunks, 31u - __builtin_clz(C / kGroupSyms),
                               ecc_num_chunks(n, kGroupSyms));
    }
    // a device where it cannot run.  Chunks of more than kGroupSyms symbols:
    // length pass, scan, pass encoder
    if (C > kGroupSyms) {
        const uint32_t slot = enc_ws_slot_bytes(kGroupSyms, S);
        const size_t smem = enc_ws_smem_bytes(kGroupSyms, slot);
        const int occ = smem <= kMaxDynSmem - kStaticSmemReserve
                            ? occupancy((const void *)encode_pass_kernel, kEncThreadsWS, smem)
                            : 0;
        const int occ_len = occupancy((const void *)enc_len_kernel, kEncThreads, enc_shared_bytes());
        if (occ > 0 && occ_len > 0) {
            const uint64_t grid_len = std::min<uint64_t>((uint64_t)occ_len * sms, n_chunks);
            enc_len_kernel<<<(unsigned)grid_len, kEncThreads, enc_shared_bytes(), st>>>(in, n, cb, C, n_chunks, flags);
            enc_scan_kernel<<<1, 1024, 0, st>>>(flags, n_chunks, chunk_off, total_bits, out_cap, status);
            EncParams q = p;
            q.nbuf = 2;
            q.stage_bytes = slot;
            const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, n_chunks);
            encode_pass_kernel<<<(unsigned)grid, kEncThreadsWS, smem, st>>>(q);
            return launch_status(cudaGetLastError());
        }
    }
    // Smaller chunks: the warp-specialised kernel (two input buffers, two
    // stage slots of warp regions) when it fits, else the single-slot kernel;
    // chunks smaller than kGroupSyms symbols are coded in groups of
    // consecutive chunks
    {
        const uint32_t G = enc_group_chunks(C, S);
        const uint32_t slot = G > 1 ? enc_ws_group_slot_bytes(C, S) : enc_ws_slot_bytes(C, S);
        const size_t smem = enc_ws_smem_bytes(C * G, slot);
        const void *kfn = G > 1 ? (const void *)encode_ws_kernel<true> : (const void *)encode_ws_kernel<false>;
        const int occ = smem <= kMaxDynSmem - kStaticSmemReserve ? occupancy(kfn, kEncThreadsWS, smem) : 0;
        if (occ > 0) {
            EncParams q = p;
            q.nbuf = 2;
            q.stage_bytes = slot;
            q.group = G;
            const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, (n_chunks + G - 1) / G);
            if (G > 1)
                encode_ws_kernel<true><<<(unsigned)grid, kEncThreadsWS, smem, st>>>(q);
            else
                encode_ws_kernel<false><<<(unsigned)grid, kEncThreadsWS, smem, st>>>(q);
            const ecc_status e = launch_status(cudaGetLastError());
            return e != ECC_OK ? e : launch_deferred(p.job, n_chunks, G, st, nullptr, 0, 0);
        }
    }
    p.nbuf = enc_input_buffers(C);
    const size_t smem = enc_shared_bytes() + (size_t)p.nbuf * C + kStageLead + p.stage_bytes;
    const int occ = occupancy((const void *)encode_kernel, kEncThreads, smem);
    if (occ <= 0)
        return ECC_ERR_CUDA;
    const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, n_chunks);
    encode_kernel<<<(unsigned)grid, kEncThreads, smem, st>>>(p);
    return launch_status(cudaGetLastError());
}

ecc_status ecc_decode(const uint8_t *in, size_t in_bytes, const uint64_t *chunk_off, const uint16_t *sub_bits,
                      size_t n, uint32_t C, uint32_t S, const ecc_codebook *cb, uint8_t *out, uint32_t *status,
                      void *stream)
{
    if (!cb || !aligned16(cb) || !status || !chunk_off || !valid_sizes(C, S))
        return ECC_ERR_ARG;
    if (n && (!in || !out || !sub_bits || !aligned16(in) || !aligned16(out)))
        return ECC_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess)
        return launch_status(cudaErrorUnknown);
    if (!n)
        return ECC_OK;
    DecParams p;
    p.job = DecJob{in, in_bytes, chunk_off, sub_bits, n, C, S, cb, out, status};
    p.n_chunks = ecc_num_chunks(n, C);
    // streams per lane and pieces of a chunk (up to 4 streams)
    const DecSplit split = dec_split(C, S, 4);
    const uint32_t per_lane = split.R;
    p.pshift = split.ps;
    p.stage_bytes = dec_stage_bytes(C >> p.pshift, S);
    const bool pieces = p.pshift > 0;
    const void *kfn = per_lane == 4   ? (pieces ? (const void *)decode_kernel<4, true> : (const void *)decode_kernel<4, false>)
                      : per_lane == 2 ? (pieces ? (const void *)decode_kernel<2, true> : (const void *)decode_kernel<2, false>)
                                      : (pieces ? (const void *)decode_kernel<1, true> : (const void *)decode_kernel<1, false>);
    // as many warps as shared memory holds stages for, and registers allow
    int warps = decode_warps(p.stage_bytes);
    auto smem_for = [&](int w) { return std::max<size_t>(kDecMinSmem, kDecHeadBytes + (size_t)w * p.stage_bytes); };
    while (warps > 1 && occupancy(kfn, warps * 32, smem_for(warps)) <= 0)
        --warps;
    const size_t smem = smem_for(warps);
    const int occ = occupancy(kfn, warps * 32, smem);
    const int sms = sm_count();
    if (occ <= 0 || sms <= 0)
        return ECC_ERR_CUDA;
    const uint64_t need = ((p.n_chunks << p.pshift) + warps - 1) / warps;
    const uint64_t grid = std::min<uint64_t>((uint64_t)occ * sms, need);
    if (per_lane == 4 && pieces)
        decode_kernel<4, true><<<(unsigned)grid, warps * 32, smem, st>>>(p);
    else if (per_lane == 4)
        decode_kernel<4, false><<<(unsigned)grid, warps * 32, smem, st>>>(p);
    else if (per_lane == 2 && pieces)
        decode_kernel<2, true><<<(unsigned)grid, warps * 32, smem, st>>>(p);
    else if (per_lane == 2)
        decode_kernel<2, false><<<(unsigned)grid, warps * 32, smem, st>>>(p);
    else if (pieces)
        decode_kernel<1, true><<<(unsigned)grid, warps * 32, smem, st>>>(p);
    else
        decode_kernel<1, false><<<(unsigned)grid, warps * 32, smem, st>>>(p);
    return launch_status(cudaGetLastError());
}

ecc_status ecc_selftest_wait(uint64_t *flags, uint64_t chunk, uint64_t aggregate, uint64_t timeout_ns,
                             uint64_t *prefix, uint32_t *status, void *stream)
{
    if (!flags || !prefix || !status || timeout_ns == 0 || timeout_ns > 10ull * kWaitLimitNs)
        return ECC_ERR_ARG;
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(flags, chunk, aggregate, timeout_ns, prefix, status);
    return launch_status(cudaGetLastError());
}

} // extern "C"

// ---------------------------------------------------------------- encode without allocation
// ecc_encode_static: ecc_encode for callers that cannot allocate device
// memory on their call path.  Its workspace (ticket + one look-back word per
// chunk, and one per 16384 symbols for larger chunks) is a file-scope
// device array instead of a caller buffer.
namespace ecc {

constexpr uint64_t kStaticMaxChunks = ECC_STATIC_MAX_CHUNKS;
// a ticket, a word per chunk and, for chunks of 65536 symbols, 4 per chunk
constexpr uint64_t kStaticScratchWords = 256 / sizeof(uint64_t) + kStaticMaxChunks * (1 + 65536 / kGroupSyms);

// Held by every GPU that loads the library until the process exits.  Host
// code must not pass this name to a kernel: on the host it is only a
// stand-in; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint64_t g_encode_scratch[kStaticScratchWords];

namespace {
// The array's device address on the current device, resolved on every call
// with that device current: a host-side lookup, cheap once the module is
// loaded, and never stale (a context reset reloads the module elsewhere).
// The first call on a device may load the module; make it before any stream
// capture.
ecc_status static_scratch(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_encode_scratch);
    if (e != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return ECC_ERR_CUDA;
    }
    *out = p;
    return ECC_OK;
}
} // namespace

} // namespace ecc

extern "C" ecc_status ecc_encode_static(const uint8_t *in, size_t n, const ecc_codebook *cb, uint32_t C, uint32_t S,
                                        uint8_t *out, size_t out_cap, uint64_t *chunk_off, uint16_t *sub_bits,
                                        uint64_t *total_bits, uint32_t *status, void *stream)
{
    if (!valid_sizes(C, S) || ecc_num_chunks(n, C) > ecc::kStaticMaxChunks)
        return ECC_ERR_ARG;
    void *scratch = nullptr;
    const ecc_status e = ecc::static_scratch(&scratch);
    if (e != ECC_OK)
        return e;
    return ecc_encode(in, n, cb, C, S, out, out_cap, chunk_off, sub_bits, total_bits, scratch,
                      sizeof(ecc::g_encode_scratch), status, stream);
}
