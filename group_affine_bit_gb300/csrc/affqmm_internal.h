// affqmm_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "affqmm.h"

namespace affqmm {

// One projection of a decode (M <= 16) launch: its units are
// (128-row tile, 128-deep block) pairs, numbered tile-major (the order they
// sit in memory), cut into `nctas` contiguous runs, one per CTA.  The cut
// depends only on the projection, M and the device, never on what else
// shares the launch.
struct DecProj {
    const uint8_t* packed;
    uint16_t* y;
    int64_t N;
    int32_t tiles;        // ceil(N / 128)
    int32_t units;        // tiles * k-blocks
    int32_t nctas;        // CTAs working on this projection (<= units)
    int32_t cta_begin;    // first CTA of this projection in the grid
    int32_t ctr_begin;    // first tile of this projection's merge counters (eight per tile)
    int32_t slot_begin;   // first partial slot (two per CTA)
};

struct DecParams {
    DecProj proj[AFFQMM_MAX_STACK];
    int32_t nproj;
    int32_t KB;              // k-blocks of 128
    int64_t K;
    int32_t M;               // activation rows (1..16)
    const uint16_t* x;       // x [M, K] bf16 (read directly in exact-codes mode)
    const float* xsums;      // exact-codes mode: [M, K/group] fp32 sums of x written by x's producer, or null
    int32_t epi;             // 0: y = bf16(sums); 1: GeGLU of a gate/up stack interleaved in 16-row blocks
    uint32_t* status;        // device status word (bit 0: a bounded wait gave up)
    uint32_t* counters;
    float* partials;         // slot = 128 rows x 16 floats
    int64_t fault_wait;      // test hook (0 = off): cycles the consumers wait on a barrier nothing completes
};

constexpr size_t kDecSlotFloats = 128 * 16;
constexpr int kDecCountersPerTile = 8;   // one per 16-row group of a tile

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
    int32_t ltiles;       // ceil(N / 128): 128-row layout tiles present in `packed`
    int32_t tiles;        // ceil(N / 256)
    int32_t units;        // tiles * k-blocks
    int32_t nctas;        // CTAs working on this projection (<= units)
    int32_t cta_begin;    // first CTA of this projection in the grid
    int32_t ctr_begin;    // first 256-row tile of this projection in the merge kernel's grid
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

// Launch `kernel` with programmatic stream serialization: it may begin while
// the previous kernel in the stream finishes, and resolves the dependency
// itself (griddepcontrol.wait) before it touches data that kernel may use.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, int threads, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (decode.cu, prompt.cu, pack.cu).  They return the launch's error.
// decode.cu: the tensor map describes x [M, K] bf16 with a 136 x M box, no
// swizzle.  decode_allow_smem sets the kernels' shared-memory attributes and
// reports how many decode CTAs one SM holds.
cudaError_t decode_allow_smem(int* ctas_per_sm);
// The decode launches' fault_wait test hook (affqmm_test_fault_wait).
int64_t decode_fault_wait();
void decode_set_fault_wait(int64_t cycles);
cudaError_t launch_decode(int bits, int group, const DecParams& p, const CUtensorMap& map, int grid, cudaStream_t st,
                          bool exact = false);
// prompt.cu: the tensor map describes x [M, K] bf16 with a 64 x 128 box.
cudaError_t prompt_allow_smem();
cudaError_t launch_prompt(int bits, const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st);
cudaError_t launch_pack(int bits, int group, int64_t N, int64_t K, const uint8_t* codes,
                        const uint16_t* scales, const uint16_t* biases, void* packed,
                        cudaStream_t st);
cudaError_t launch_dequant(int bits, int group, int64_t N, int64_t K, const void* packed,
                           uint16_t* out, cudaStream_t st);
// embed.cu: rows ids[0..T) of the table (the packed blocks, or their
// row-contiguous copy when `rowcopy`), optionally times a bf16 scale; and the
// row-contiguous copy of a packed table.
cudaError_t launch_embed(int bits, int group, bool rowcopy, const void* table, int64_t N, int64_t K,
                         const int32_t* ids, int64_t T, int has_scale, uint16_t scale, uint16_t* out, uint32_t* status,
                         cudaStream_t st);
cudaError_t launch_pack_rows(int bits, int group, const void* packed, int64_t N, int64_t K, void* rows,
                             cudaStream_t st);
// plan.cu: how a launch is cut (see there).  Rows per launch: the decode
// kernel takes up to 16 activation rows, the prompt kernel up to 128; a prompt
// unit covers 256 weight rows.
constexpr int64_t kDecodeRows = 16;
constexpr int64_t kPromptRows = 128;
constexpr int kPromptTileN = 256;
struct DecodePlan {
    DecParams p;
    int grid = 0;
    size_t ws_bytes = 0;
};
struct PromptPlan {
    PromptParams p;
    int grid = 0;
    size_t ws_bytes = 0;
};
int plan_decode(int sms, int ctas_per_sm, int count, const affqmm_weight* ws, int64_t M, DecodePlan* plan);
int plan_prompt(int sms, int count, const affqmm_weight* ws, int64_t M, PromptPlan* plan);

// hostio.cu: the host-buffer entry point's transfers as kernels (the host
// pointers are the GPU's addresses of page-locked host memory).
cudaError_t launch_host_upload(const void* host_src, void* dev_dst, size_t bytes, cudaStream_t st);
cudaError_t launch_host_download(const void* dev_src, void* host_dst, size_t bytes, cudaStream_t st);

}  // namespace affqmm
