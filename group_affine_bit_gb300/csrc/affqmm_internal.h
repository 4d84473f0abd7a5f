// affqmm_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "affqmm.h"

namespace affqmm {

// One projection of a decode (M <= 16) launch.  Its 128-deep blocks are
// grouped into "stages" of up to `su` consecutive blocks of one 16-row tile
// (ceil(KB / su) stages per tile); the stages, numbered tile-major, are cut
// into `nctas` contiguous runs, one per CTA.  The cut depends only on the
// projection, M and the device, never on what else shares the launch.
struct DecProj {
    const uint8_t* packed;
    uint16_t* y;
    int64_t N;
    int32_t tiles;        // ceil(N / 16)
    int32_t stages;       // tiles * stages per tile
    int32_t nctas;        // CTAs working on this projection (<= stages)
    int32_t cta_begin;    // first CTA of this projection in the grid
    int32_t ctr_begin;    // first merge counter (one per tile)
    int32_t slot_begin;   // first partial slot (two per CTA)
};

struct DecParams {
    DecProj proj[AFFQMM_MAX_STACK];
    int32_t nproj;
    int32_t KB;              // k-blocks of 128
    int64_t K;
    int32_t M;
    int32_t block_bytes;     // bytes of one (tile, k-block) block
    int32_t group;
    int32_t su;              // blocks per stage = consumer warps per CTA
    int32_t spt;             // stages per tile = ceil(KB / su)
    int32_t ring;            // stages in the shared-memory ring
    int32_t stage_bytes;     // ring stage stride (su * block_bytes rounded up to 128)
    const uint16_t* x;
    uint32_t* status;        // device status word (bit 0: a bounded wait gave up)
    uint32_t* counters;
    float* partials;         // slot = 32 lanes x 8 floats
};

// Dynamic shared memory of one decode CTA: the ring, two reduction buffers
// (su warps x 32 lanes x 8 floats) and the mbarriers.
inline size_t decode_smem_bytes(int ring, int stage_bytes, int su) {
    return (size_t)ring * stage_bytes + 2 * (size_t)su * 32 * 8 * sizeof(float) + (2 * (size_t)ring + 4) * 8 + 128;
}

constexpr int DEC_MAX_SU = 8;   // at most 8 consumer warps (+1 producer) per decode CTA

// Workspace layout shared by every kernel: a status word, then a fixed region
// of merge counters (zero between calls: the last user of a counter resets
// it), then per-launch partial-sum slots whose contents between calls do not
// matter.  The fixed counter region keeps one plan's slots from ever
// overlapping another plan's counters.
constexpr size_t kStatusBytes = 256;
constexpr size_t kMaxCounters = 65536;
constexpr size_t kCounterBytes = kMaxCounters * sizeof(uint32_t);
constexpr size_t kSlotsOffset = kStatusBytes + kCounterBytes;

// One projection of a prompt (M = 17..128 per launch) launch: its units are
// (256-row tile, 128-deep block) pairs, numbered tile-major, cut into `nctas`
// contiguous runs, one per CTA.
struct PromptProj {
    const uint8_t* packed;
    uint16_t* y;
    int64_t N;
    int32_t tiles16;      // ceil(N / 16): 16-row blocks present in `packed`
    int32_t tiles;        // ceil(N / 256)
    int32_t units;        // tiles * k-blocks
    int32_t nctas;        // CTAs working on this projection (<= units)
    int32_t cta_begin;    // first CTA of this projection in the grid
    int32_t ctr_begin;    // first tile of this projection's merge counters (four per tile)
    int32_t slot_begin;   // first partial slot (two per CTA)
};

struct PromptParams {
    PromptProj proj[AFFQMM_MAX_STACK];
    int32_t nproj;
    int32_t KB;
    int64_t K;
    int32_t M;               // activation rows of this launch (1..128)
    int32_t block_bytes;
    int32_t group;
    uint32_t* status;
    uint32_t* counters;
    float* slots;            // slot = 128 x 256 floats
};

constexpr size_t kPromptSlotFloats = 128 * 256;

// Launchers (decode.cu, pack.cu).  They return a cudaError_t of the launch.
cudaError_t launch_decode(int bits, int mt, const DecParams& p, int grid, cudaStream_t st);
// Resident CTAs per SM of the decode kernel with `su` consumer warps and
// `smem` bytes of dynamic shared memory.
int decode_ctas_per_sm(int bits, int mt, int su, size_t smem);
// Let every decode instantiation use up to `bytes` of dynamic shared memory.
cudaError_t decode_allow_smem(int bytes);
constexpr int kDecodeSmemMax = 200 * 1024;
// prompt.cu: the tensor map describes x [M, K] bf16 with a 64 x 128 box.
size_t prompt_smem_bytes();
cudaError_t prompt_allow_smem();
cudaError_t launch_prompt(int bits, const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st);
cudaError_t launch_pack(int bits, int group, int64_t N, int64_t K, const uint8_t* codes,
                        const uint16_t* scales, const uint16_t* biases, void* packed,
                        cudaStream_t st);
cudaError_t launch_dequant(int bits, int group, int64_t N, int64_t K, const void* packed,
                           uint16_t* out, cudaStream_t st);

}  // namespace affqmm
