// pack.cu -- canonical affine table -> the library's packed blocks, and the
// dequantization test hook that reads them back with the run kernels' own
// device arithmetic (affqmm_format.cuh).
#include "affqmm_format.cuh"
#include "affqmm_internal.h"

namespace affqmm {
namespace {

// One CTA per (128-row tile, 128-deep block), one thread per row.
template <int BITS>
__global__ void __launch_bounds__(TILE_N) pack_kernel(int group, int64_t N, int64_t K, int KB,
                                                      const uint8_t* __restrict__ codes,
                                                      const uint16_t* __restrict__ scales,
                                                      const uint16_t* __restrict__ biases,
                                                      uint8_t* __restrict__ packed) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
    const int n = threadIdx.x;
    const int64_t blk = blockIdx.x;
    const int64_t tile = blk / KB;
    const int kb = (int)(blk % KB);
    uint8_t* out = packed + blk * block_bytes(BITS, group);
    const int64_t row = tile * TILE_N + n;
    const int64_t G = K / group;
    const uint32_t qmask = (1u << BITS) - 1u;

    auto code = [&](int kk) -> uint32_t {
        const int64_t k = (int64_t)kb * KBLK + kk;
        if (row >= N || k >= K) return 0u;
        return codes[row * K + k] & qmask;
    };

    for (int plane = 0; plane < (P1 ? 2 : 1); ++plane) {
        const int p = plane ? P1 : P0;
        const int shift_in = plane ? P0 : 0;
        const uint32_t fmask = (1u << p) - 1u;
        for (int w = 0; w < 4 * p; ++w) {
            // class-major words: word p*c + v holds class c's pairs j = v*(16/p) + i,
            // pair C = 4j + c at k = 2C
            const int c = w / p, v = w % p;
            uint32_t word = 0;
            for (int i = 0; i < 16 / p; ++i) {
                const int k0 = 2 * (4 * (v * (16 / p) + i) + c);
                word |= ((code(k0) >> shift_in) & fmask) << (p * i);
                word |= ((code(k0 + 1) >> shift_in) & fmask) << (16 + p * i);
            }
            *reinterpret_cast<uint32_t*>(out + word_offset(BITS, plane, n, w)) = word;
        }
    }
    const int gw = sb_words(group);
    uint32_t* sb = reinterpret_cast<uint32_t*>(out + sb_offset(BITS, group, n));
    for (int gi = 0; gi < gw; ++gi) {
        const int64_t k = (int64_t)kb * KBLK + gi * group;
        uint32_t v = 0u;
        if (row < N && k < K) {
            const int64_t j = k / group;
            v = (uint32_t)scales[row * G + j] | ((uint32_t)biases[row * G + j] << 16);
        }
        sb[gi] = v;
    }
    // The run kernels start copying packed weights before they wait on the
    // kernel ahead of them in the stream (programmatic dependent launch): make
    // this thread's writes visible GPU-wide before the block exits, which is
    // when this kernel (it never triggers early) lets a dependent start.
    __threadfence();
}

// One CTA per block, one thread per row: the run kernels' loads and
// dequantization, written out as bf16 [N, K].
template <int BITS, int GROUP>
__global__ void __launch_bounds__(TILE_N) dequant_kernel(int64_t N, int64_t K, int KB, const uint8_t* __restrict__ packed,
                                                         uint16_t* __restrict__ out) {
    const int n = threadIdx.x;
    const int64_t blk = blockIdx.x;
    const int64_t tile = blk / KB;
    const int kb = (int)(blk % KB);
    const uint8_t* src = packed + blk * block_bytes(BITS, GROUP);
    const int64_t row = tile * TILE_N + n;
    if (row >= N) return;
    uint32_t cw[4 * BITS];
    load_row_codes<BITS>(src, n, cw);
    uint32_t sbw[sb_words(GROUP)];
    load_row_sb<GROUP>(src + sb_offset(BITS, GROUP, n), sbw);
    uint32_t w[KBLK / 2];
    weight_pairs<BITS, GROUP, 0, KBLK / 2>(cw, sbw, w);
#pragma unroll
    for (int c = 0; c < KBLK / 2; ++c) {
        const int64_t k = (int64_t)kb * KBLK + 2 * c;
        if (k < K) {
            out[row * K + k] = (uint16_t)(w[c] & 0xFFFFu);
            out[row * K + k + 1] = (uint16_t)(w[c] >> 16);
        }
    }
}

template <int BITS>
cudaError_t dequant_bits(int group, int64_t N, int64_t K, int KB, int64_t blocks, const uint8_t* src,
                         uint16_t* out, cudaStream_t st) {
    if (group == 32) dequant_kernel<BITS, 32><<<(unsigned)blocks, TILE_N, 0, st>>>(N, K, KB, src, out);
    else if (group == 64) dequant_kernel<BITS, 64><<<(unsigned)blocks, TILE_N, 0, st>>>(N, K, KB, src, out);
    else dequant_kernel<BITS, 128><<<(unsigned)blocks, TILE_N, 0, st>>>(N, K, KB, src, out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(int bits, int group, int64_t N, int64_t K, const uint8_t* codes,
                        const uint16_t* scales, const uint16_t* biases, void* packed, cudaStream_t st) {
    const int64_t tiles = (N + TILE_N - 1) / TILE_N;
    const int KB = (int)((K + KBLK - 1) / KBLK);
    const int64_t blocks = tiles * KB;
    if (blocks == 0) return cudaSuccess;
    uint8_t* dst = static_cast<uint8_t*>(packed);
    switch (bits) {
        case 2: pack_kernel<2><<<(unsigned)blocks, TILE_N, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 3: pack_kernel<3><<<(unsigned)blocks, TILE_N, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 4: pack_kernel<4><<<(unsigned)blocks, TILE_N, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 5: pack_kernel<5><<<(unsigned)blocks, TILE_N, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 6: pack_kernel<6><<<(unsigned)blocks, TILE_N, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 8: pack_kernel<8><<<(unsigned)blocks, TILE_N, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_dequant(int bits, int group, int64_t N, int64_t K, const void* packed, uint16_t* out,
                           cudaStream_t st) {
    const int64_t tiles = (N + TILE_N - 1) / TILE_N;
    const int KB = (int)((K + KBLK - 1) / KBLK);
    const int64_t blocks = tiles * KB;
    if (blocks == 0) return cudaSuccess;
    const uint8_t* src = static_cast<const uint8_t*>(packed);
    switch (bits) {
        case 2: return dequant_bits<2>(group, N, K, KB, blocks, src, out, st);
        case 3: return dequant_bits<3>(group, N, K, KB, blocks, src, out, st);
        case 4: return dequant_bits<4>(group, N, K, KB, blocks, src, out, st);
        case 5: return dequant_bits<5>(group, N, K, KB, blocks, src, out, st);
        case 6: return dequant_bits<6>(group, N, K, KB, blocks, src, out, st);
        case 8: return dequant_bits<8>(group, N, K, KB, blocks, src, out, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace affqmm
