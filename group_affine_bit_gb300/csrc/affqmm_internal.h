// affqmm_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI).
#pragma once
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

// Launchers (decode.cu, pack.cu).  They return a cudaError_t of the launch.
cudaError_t launch_decode(int bits, int mt, const DecParams& p, int grid, cudaStream_t st);
// Resident CTAs per SM of the decode kernel with `smem` bytes of ring.
int decode_ctas_per_sm(int bits, int mt, size_t smem);
// Let every decode instantiation use up to `bytes` of dynamic shared memory.
cudaError_t decode_allow_smem(int bytes);
constexpr int kDecodeSmemMax = 200 * 1024;
cudaError_t launch_pack(int bits, int group, int64_t N, int64_t K, const uint8_t* codes,
                        const uint16_t* scales, const uint16_t* biases, void* packed,
                        cudaStream_t st);
cudaError_t launch_dequant(int bits, int group, int64_t N, int64_t K, const void* packed,
                           uint16_t* out, cudaStream_t st);

}  // namespace affqmm
