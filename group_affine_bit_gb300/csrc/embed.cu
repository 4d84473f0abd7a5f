// embed.cu -- scaled embedding rows gathered from a packed affine table:
//
//     out[t, k] = bf16( W[ids[t], k] * scale ),   W[n, k] = bf16(s * q + b)
//
// ("cuda gemma4: images on the 12B" page, the embed_rows commit: MLX affine
// tables at 2..8 bits, each dequantized bf16 value multiplied by a bf16
// scale -- Gemma's bf16(sqrt(hidden)) -- and rounded again.)  Both roundings
// are of exact values: fma.rn.bf16x2 for the weight (affqmm_format.cuh, the
// arithmetic of the projection kernels) and mul.rn.bf16x2 for the product.
//
// One thread per (row t, 128-deep block): it loads the row's codes and
// scale/bias words of that block, makes the 128 values and writes them as 16
// contiguous 16-byte stores.  Memory-bound: the packed bytes of the gathered
// rows in, 2 bytes per value out.  The words come from either
//   * the packed table itself (the layout the projections read, so a tied
//     head serves as the embedding table without a copy): a row's 16-byte
//     chunks sit between those of 31 other rows, so each one costs a whole
//     DRAM burst of which it uses a fraction; or
//   * its row-contiguous copy (affqmm_format.cuh, rows_stride), which
//     pack_rows_kernel makes once from the packed table: a warp's 32 threads
//     then read 32 consecutive blocks of one row, one contiguous range, and
//     the gather reads only the bytes it needs.
#include <cuda_bf16.h>

#include "affqmm_format.cuh"
#include "affqmm_internal.h"

namespace affqmm {
namespace {

constexpr int E_THREADS = 128;

__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void st_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int BITS, int GROUP, bool ROWCOPY>
__global__ void __launch_bounds__(E_THREADS) embed_kernel(const uint8_t* __restrict__ packed, int64_t N, int64_t K,
                                                          int KB, const int32_t* __restrict__ ids, int64_t T,
                                                          int has_scale, uint32_t scale2, uint16_t* __restrict__ out,
                                                          uint32_t* status) {
    const int64_t item = (int64_t)blockIdx.x * E_THREADS + threadIdx.x;
    if (item >= T * KB) return;
    const int64_t t = item / KB;
    const int kb = (int)(item - t * KB);
    const int64_t n = ids[t];
    uint16_t* dst = out + t * K + (int64_t)kb * KBLK;
    const int64_t kleft = K - (int64_t)kb * KBLK;  // values of this block inside the row (8-aligned, >= 32)
    uint32_t w[KBLK / 2];
    if (n < 0 || n >= N) {  // not a row of the table: zeros, and say so
#pragma unroll
        for (int c = 0; c < KBLK / 2; ++c) w[c] = 0u;
        if (status && kb == 0) atomicOr(status, 2u);
    } else {
        uint32_t cw[4 * BITS];
        uint32_t sbw[sb_words(GROUP)];
        if constexpr (ROWCOPY) {
            const uint8_t* row = packed + n * rows_stride(BITS, GROUP, KB);
            load_rowcopy_codes<BITS>(row + rows_codes_offset(BITS, kb), cw);
            load_row_sb<GROUP>(row + rows_sb_offset(BITS, GROUP, KB, kb), sbw);
        } else {
            const uint8_t* blk = packed + ((n / TILE_N) * KB + kb) * (int64_t)block_bytes(BITS, GROUP);
            const int r = (int)(n % TILE_N);
            load_row_codes<BITS>(blk, r, cw);
            load_row_sb<GROUP>(blk + sb_offset(BITS, GROUP, r), sbw);
        }
        weight_pairs<BITS, GROUP, 0, KBLK / 2>(cw, sbw, w);
        if (has_scale) {
#pragma unroll
            for (int c = 0; c < KBLK / 2; ++c) w[c] = bf2_mul(w[c], scale2);
        }
    }
    // When the depth is whole blocks, item i's values are out[128 i ..
    // 128 i + 127], so a warp's 32 items are one contiguous 8 KB range: the
    // warp stages its items in shared memory and writes the range as 16
    // stores of 512 contiguous bytes.  (A thread's own 16 stores would put
    // 16 bytes in each of 32 lines per instruction.)  The 16-byte slot of
    // piece c of lane L is L*16 + (c ^ (L & 7)), so that the eight lanes of
    // one store phase, either way round, touch eight different bank groups.
    __shared__ uint4 stage[E_THREADS / 32][32 * 16];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t item0 = item - lane;
    if (KB * (int64_t)KBLK == K && item0 + 31 < T * KB) {
        uint4* st = stage[wid];
#pragma unroll
        for (int c = 0; c < KBLK / 8; ++c)
            st[lane * 16 + (c ^ (lane & 7))] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        __syncwarp();
        uint16_t* base = out + item0 * KBLK;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int u = 32 * i + lane;  // 16-byte piece of the warp's range
            const int owner = u >> 4, c = u & 15;
            const uint4 v = st[owner * 16 + (c ^ (owner & 7))];
            st_v4(base + 8 * u, v.x, v.y, v.z, v.w);
        }
    } else {
#pragma unroll
        for (int c = 0; c < KBLK / 8; ++c)  // 8 values (16 bytes) per store
            if (8 * c < kleft) st_v4(dst + 8 * c, w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

// The row-contiguous copy: one thread per (row n, 128-deep block) moves the
// row's code words and scale/bias words of that block, unchanged, from the
// packed table to their places in the copy.
template <int BITS, int GROUP>
__global__ void __launch_bounds__(E_THREADS) pack_rows_kernel(const uint8_t* __restrict__ packed, int64_t N, int KB,
                                                              uint8_t* __restrict__ rows) {
    const int64_t item = (int64_t)blockIdx.x * E_THREADS + threadIdx.x;
    if (item >= N * KB) return;
    const int64_t n = item / KB;
    const int kb = (int)(item - n * KB);
    const uint8_t* blk = packed + ((n / TILE_N) * KB + kb) * (int64_t)block_bytes(BITS, GROUP);
    const int r = (int)(n % TILE_N);
    uint32_t cw[4 * BITS];
    load_row_codes<BITS>(blk, r, cw);
    uint32_t sbw[sb_words(GROUP)];
    load_row_sb<GROUP>(blk + sb_offset(BITS, GROUP, r), sbw);
    uint8_t* row = rows + n * rows_stride(BITS, GROUP, KB);
    uint4* dc = reinterpret_cast<uint4*>(row + rows_codes_offset(BITS, kb));
#pragma unroll
    for (int v = 0; v < BITS; ++v) dc[v] = make_uint4(cw[4 * v], cw[4 * v + 1], cw[4 * v + 2], cw[4 * v + 3]);
    uint32_t* ds = reinterpret_cast<uint32_t*>(row + rows_sb_offset(BITS, GROUP, KB, kb));
#pragma unroll
    for (int v = 0; v < sb_words(GROUP); ++v) ds[v] = sbw[v];
    // the padding at the end of a row (at most 12 bytes) is written as zeros
    // by the block that ends the row
    if (kb == KB - 1) {
        const int64_t used = rows_sb_offset(BITS, GROUP, KB, KB);
        for (int64_t b = used; b < rows_stride(BITS, GROUP, KB); b += 4) *reinterpret_cast<uint32_t*>(row + b) = 0u;
    }
    __threadfence();  // the copy is complete device-wide before a gather enqueued after it starts
}

template <int BITS, int GROUP>
void embed_bg(bool rowcopy, unsigned grid, const uint8_t* src, int64_t N, int64_t K, int KB, const int32_t* ids,
              int64_t T, int has_scale, uint32_t scale2, uint16_t* out, uint32_t* status, cudaStream_t st) {
    if (rowcopy)
        embed_kernel<BITS, GROUP, true><<<grid, E_THREADS, 0, st>>>(src, N, K, KB, ids, T, has_scale, scale2, out,
                                                                    status);
    else
        embed_kernel<BITS, GROUP, false><<<grid, E_THREADS, 0, st>>>(src, N, K, KB, ids, T, has_scale, scale2, out,
                                                                     status);
}

template <int BITS>
cudaError_t embed_bits(int group, bool rowcopy, const uint8_t* src, int64_t N, int64_t K, int KB, const int32_t* ids,
                       int64_t T, int has_scale, uint32_t scale2, uint16_t* out, uint32_t* status, cudaStream_t st) {
    const int64_t items = T * KB;
    const unsigned grid = (unsigned)((items + E_THREADS - 1) / E_THREADS);
    if (group == 32) embed_bg<BITS, 32>(rowcopy, grid, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
    else if (group == 64) embed_bg<BITS, 64>(rowcopy, grid, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
    else embed_bg<BITS, 128>(rowcopy, grid, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t pack_rows_bits(int group, const uint8_t* packed, int64_t N, int KB, uint8_t* rows, cudaStream_t st) {
    const int64_t items = N * KB;
    const unsigned grid = (unsigned)((items + E_THREADS - 1) / E_THREADS);
    if (group == 32) pack_rows_kernel<BITS, 32><<<grid, E_THREADS, 0, st>>>(packed, N, KB, rows);
    else if (group == 64) pack_rows_kernel<BITS, 64><<<grid, E_THREADS, 0, st>>>(packed, N, KB, rows);
    else pack_rows_kernel<BITS, 128><<<grid, E_THREADS, 0, st>>>(packed, N, KB, rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_embed(int bits, int group, bool rowcopy, const void* table, int64_t N, int64_t K,
                         const int32_t* ids, int64_t T, int has_scale, uint16_t scale, uint16_t* out, uint32_t* status,
                         cudaStream_t st) {
    const int KB = (int)((K + KBLK - 1) / KBLK);
    if (T == 0 || KB == 0) return cudaSuccess;
    const uint8_t* src = static_cast<const uint8_t*>(table);
    const uint32_t scale2 = (uint32_t)scale * 0x00010001u;  // the scale in both halves
    switch (bits) {
        case 2: return embed_bits<2>(group, rowcopy, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
        case 3: return embed_bits<3>(group, rowcopy, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
        case 4: return embed_bits<4>(group, rowcopy, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
        case 5: return embed_bits<5>(group, rowcopy, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
        case 6: return embed_bits<6>(group, rowcopy, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
        case 8: return embed_bits<8>(group, rowcopy, src, N, K, KB, ids, T, has_scale, scale2, out, status, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_pack_rows(int bits, int group, const void* packed, int64_t N, int64_t K, void* rows,
                             cudaStream_t st) {
    const int KB = (int)((K + KBLK - 1) / KBLK);
    if (N == 0 || KB == 0) return cudaSuccess;
    const uint8_t* src = static_cast<const uint8_t*>(packed);
    uint8_t* dst = static_cast<uint8_t*>(rows);
    switch (bits) {
        case 2: return pack_rows_bits<2>(group, src, N, KB, dst, st);
        case 3: return pack_rows_bits<3>(group, src, N, KB, dst, st);
        case 4: return pack_rows_bits<4>(group, src, N, KB, dst, st);
        case 5: return pack_rows_bits<5>(group, src, N, KB, dst, st);
        case 6: return pack_rows_bits<6>(group, src, N, KB, dst, st);
        case 8: return pack_rows_bits<8>(group, src, N, KB, dst, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace affqmm
