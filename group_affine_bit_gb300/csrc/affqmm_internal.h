// affqmm_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "affqmm.h"

namespace affqmm {

// One projection of a decode (M <= 16) launch.
struct DecProj {
    const uint8_t* packed;
    uint16_t* y;
    int64_t N;
    int32_t tiles;       // ceil(N / 16)
    int32_t S;           // K slices across CTAs (1 = no cross-CTA merge)
    int32_t cta_begin;   // first CTA of this projection in the grid
    int32_t ctr_begin;   // first merge counter (used when S > 1)
    int64_t part_begin;  // first partial slot (used when S > 1)
};

struct DecParams {
    DecProj proj[AFFQMM_MAX_STACK];
    int32_t nproj;
    int32_t KB;              // k-blocks of 128
    int64_t K;
    int32_t M;
    int32_t block_bytes;     // bytes of one (tile, k-block) block
    int32_t group;
    const uint16_t* x;
    uint32_t* counters;
    float* partials;         // slot = 32 lanes x 8 floats
};

constexpr int DEC_WARPS = 4;

// Launchers (decode.cu, pack.cu).  They return a cudaError_t of the launch.
cudaError_t launch_decode(int bits, int mt, const DecParams& p, int grid, cudaStream_t st);
int decode_ctas_per_sm(int bits, int mt);
cudaError_t launch_pack(int bits, int group, int64_t N, int64_t K, const uint8_t* codes,
                        const uint16_t* scales, const uint16_t* biases, void* packed,
                        cudaStream_t st);
cudaError_t launch_dequant(int bits, int group, int64_t N, int64_t K, const void* packed,
                           uint16_t* out, cudaStream_t st);

}  // namespace affqmm
