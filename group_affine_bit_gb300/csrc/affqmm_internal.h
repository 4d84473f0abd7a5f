// affqmm_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "affqmm.h"

namespace affqmm {

// One projection of a decode (M <= 16) launch.  The projection's units (one
// 16-row x 128-deep block each, numbered tile-major) are split into `nwarps`
// contiguous runs, one per warp; the split depends only on the projection,
// M and the device, never on what else shares the launch.
struct DecProj {
    const uint8_t* packed;
    uint16_t* y;
    int64_t N;
    int32_t tiles;        // ceil(N / 16)
    int32_t units;        // tiles * k-blocks
    int32_t nwarps;       // warps working on this projection (<= units)
    int32_t warp_begin;   // first global warp of this projection
    int32_t ctr_begin;    // first merge counter (one per tile)
    int32_t slot_begin;   // first partial slot (two per warp)
};

struct DecParams {
    DecProj proj[AFFQMM_MAX_STACK];
    int32_t nproj;
    int32_t KB;              // k-blocks of 128
    int64_t K;
    int32_t M;
    int32_t block_bytes;     // bytes of one (tile, k-block) block
    int32_t group;
    int32_t total_warps;
    int32_t stages;          // shared-memory ring depth per warp
    int32_t stage_bytes;     // ring stage stride (block_bytes rounded up to 128)
    const uint16_t* x;
    uint32_t* status;        // device status word (bit 0: a bounded wait gave up)
    uint32_t* counters;
    float* partials;         // slot = 32 lanes x 8 floats
};

// Shared memory of one decode CTA for a given ring.
inline size_t decode_smem_bytes(int stages, int stage_bytes) {
    return (size_t)4 * stages * (stage_bytes + 8) + 16;
}

constexpr int DEC_WARPS = 4;

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
// Resident CTAs per SM of the decode kernel with `smem` bytes of ring.
int decode_ctas_per_sm(int bits, int mt, size_t smem);
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
