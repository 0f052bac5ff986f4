// ecc_launch.h -- host-side launch helpers shared by the kernel translation
// units (device properties, occupancy, argument checks).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ecc.h"

namespace ecc {

struct EncJob;

constexpr size_t kMaxDynSmem = 227 * 1024; // per-CTA shared memory opt-in limit (static + dynamic)
constexpr size_t kStaticSmemReserve = 64;  // static shared bytes a kernel may add on top
constexpr int kDecMaxWarps = 22;
constexpr uint32_t kDecPieceSyms = 8192; // symbols one decoding warp stages at most (but 32 sub-blocks)
constexpr uint32_t kUnitSyms = 16384;    // symbols of a unit of the unit encoder

// How a decoding warp splits a chunk of C symbols in sub-blocks of S: R
// streams a lane (C / S sub-blocks over 32 lanes, at most rmax, with a
// warp's 32 R sub-blocks at most kDecPieceSyms symbols), and chunks of more
// than 32 R sub-blocks in 2^ps pieces of 32 R sub-blocks, one warp a piece,
// so that a warp's stage stays as small as for a chunk of that size.
struct DecSplit {
    uint32_t R, ps;
};
__host__ __device__ inline DecSplit dec_split(uint32_t C, uint32_t S, uint32_t rmax)
{
    uint32_t R = C / S / 32u;
    R = R < 1u ? 1u : (R > rmax ? rmax : R);
    while (R > 1u && 32u * R * S > kDecPieceSyms)
        R >>= 1;
    uint32_t ps = 0;
    while ((C / S >> ps) > 32u * R)
        ++ps;
    return DecSplit{R, ps};
}

bool valid_sizes(uint32_t C, uint32_t S);
// shared input buffers of the encoder (2 = the next chunk is prefetched)
uint32_t enc_input_buffers(uint32_t C);
// warps of a decoder CTA whose per-warp staging buffers hold stage_bytes
int decode_warps(uint32_t stage_bytes);
bool aligned16(const void *p);
ecc_status launch_status(cudaError_t e);
int sm_count();
// CTAs of `kernel` that fit on one SM (raises the kernel's dynamic shared
// memory limit on first use on the current device).
int occupancy(const void *kernel, int threads, size_t smem);
// The unit encoder for chunks of at most 16384 symbols (ecc_units.cu).
// (unit_chunks: the chunks of a unit, for the deferred pass)
ecc_status launch_unit_encoder(const EncJob &job, uint32_t *ticket, cudaStream_t st, uint32_t *unit_chunks);
// The unit encoder over many tensors whose chunks are all of 16384 symbols,
// a chunk a unit (ecc_units.cu), in two launches: unit k is chunk items[k] &
// 0xFFFFFFFF of tensor descs[items[k] >> 32]; flags: a look-back word per
// unit (zeroed); done: a counter per tensor (zeroed) for the completion
// stamps; status: where waits that end before their unit is known report;
// deferred[*n_deferred] (zeroed count): the units the first launch sized
// and placed but could not stage, which the second one codes (its tickets
// from *ticket2, zeroed).
struct UnitBatch {
    const uint64_t *items;
    const ecc_desc *descs;
    uint64_t *flags;
    uint32_t *done;
    uint32_t *ticket;
    uint32_t *status;
    uint64_t *t_start;
    uint64_t n_units;
    uint32_t *deferred;
    uint32_t *n_deferred;
    uint32_t *ticket2;
};
ecc_status launch_unit_encoder_batched(const UnitBatch &b, cudaStream_t st, bool *launched);

} // namespace ecc
