// pack.cu -- canonical affine table -> the library's packed blocks, and the
// dequantization test hook that reads them back with the run kernels' own
// device arithmetic (affqmm_format.cuh).
#include "affqmm_format.cuh"
#include "affqmm_internal.h"

namespace affqmm {
namespace {

// One warp per (tile, k-block).  Lane l = 4r + t packs rows r, r+8 and
// k = 32t .. 32t+31 of the block (see affqmm_format.cuh).
template <int BITS>
__global__ void pack_kernel(int group, int64_t N, int64_t K, int KB, const uint8_t* __restrict__ codes,
                            const uint16_t* __restrict__ scales, const uint16_t* __restrict__ biases,
                            uint8_t* __restrict__ packed) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int64_t blk = blockIdx.x;
    const int64_t tile = blk / KB;
    const int kb = (int)(blk % KB);
    uint8_t* out = packed + blk * block_bytes(BITS, group);
    const int64_t G = K / group;
    const uint32_t qmask = (1u << BITS) - 1u;

    auto code = [&](int row_off, int kk) -> uint32_t {
        const int64_t n = tile * TILE_N + r + row_off;
        const int64_t k = (int64_t)kb * KBLK + 32 * t + kk;
        if (n >= N || k >= K) return 0u;
        return codes[n * K + k] & qmask;
    };

#pragma unroll
    for (int plane = 0; plane < (P1 ? 2 : 1); ++plane) {
        const int p = plane ? P1 : P0;
        const int shift_in = plane ? P0 : 0;
        const uint32_t fmask = (1u << p) - 1u;
        const int cs = chunk_bytes(p);
        for (int w = 0; w < 2 * p; ++w) {
            uint32_t word = 0;
            const int steps = 4 / p;  // k-steps per word
            for (int ds = 0; ds < steps; ++ds) {
                const int s = w * steps + ds;
                for (int reg = 0; reg < 4; ++reg) {
                    const int i = ds * 4 + reg;
                    const int row_off = (reg & 1) ? 8 : 0;
                    const int kk = 4 * s + (reg >> 1) * 2;
                    const uint32_t lo = (code(row_off, kk) >> shift_in) & fmask;
                    const uint32_t hi = (code(row_off, kk + 1) >> shift_in) & fmask;
                    word |= lo << (p * i);
                    word |= hi << (16 + p * i);
                }
            }
            const int off = plane_offset(BITS, plane) + (w * 4 / cs) * (32 * cs) + lane * cs + (w * 4) % cs;
            *reinterpret_cast<uint32_t*>(out + off) = word;
        }
    }
    // scale/bias words: one lane per (group slot, row pair) writes them
    if ((32 * t) % group == 0) {
        const int64_t k = (int64_t)kb * KBLK + 32 * t;
        const int64_t j = k / group;
        uint32_t v[2];
        for (int h = 0; h < 2; ++h) {
            const int64_t n = tile * TILE_N + r + 8 * h;
            v[h] = 0u;
            if (n < N && k < K) v[h] = (uint32_t)scales[n * G + j] | ((uint32_t)biases[n * G + j] << 16);
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(out + sb_offset(BITS, group, t, r));
        dst[0] = v[0];
        dst[1] = v[1];
    }
}

// One warp per (tile, k-block): the same loads and dequantization as the run
// kernels, written out as bf16 [N, K].
template <int BITS>
__global__ void dequant_kernel(int group, int64_t N, int64_t K, int KB, const uint8_t* __restrict__ packed,
                               uint16_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;
    const int64_t blk = blockIdx.x;
    const int64_t tile = blk / KB;
    const int kb = (int)(blk % KB);
    const uint8_t* src = packed + blk * block_bytes(BITS, group);
    uint32_t cw[2 * BITS];
    load_lane_codes<BITS>(src, lane, cw);
    const uint2 sb = *reinterpret_cast<const uint2*>(src + sb_offset(BITS, group, t, r));
    const uint32_t sg = bcast_lo(sb.x), bg = bcast_hi(sb.x), sg8 = bcast_lo(sb.y), bg8 = bcast_hi(sb.y);
    uint32_t a[8][4];
    dequant_kstep<BITS, 0>(cw, sg, bg, sg8, bg8, a[0]);
    dequant_kstep<BITS, 1>(cw, sg, bg, sg8, bg8, a[1]);
    dequant_kstep<BITS, 2>(cw, sg, bg, sg8, bg8, a[2]);
    dequant_kstep<BITS, 3>(cw, sg, bg, sg8, bg8, a[3]);
    dequant_kstep<BITS, 4>(cw, sg, bg, sg8, bg8, a[4]);
    dequant_kstep<BITS, 5>(cw, sg, bg, sg8, bg8, a[5]);
    dequant_kstep<BITS, 6>(cw, sg, bg, sg8, bg8, a[6]);
    dequant_kstep<BITS, 7>(cw, sg, bg, sg8, bg8, a[7]);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int reg = 0; reg < 4; ++reg) {
            const int64_t n = tile * TILE_N + r + ((reg & 1) ? 8 : 0);
            const int64_t k = (int64_t)kb * KBLK + 32 * t + 4 * s + (reg >> 1) * 2;
            if (n < N && k < K) {
                out[n * K + k] = (uint16_t)(a[s][reg] & 0xFFFFu);
                out[n * K + k + 1] = (uint16_t)(a[s][reg] >> 16);
            }
        }
    }
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
        case 2: pack_kernel<2><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 3: pack_kernel<3><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 4: pack_kernel<4><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 5: pack_kernel<5><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 6: pack_kernel<6><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
        case 8: pack_kernel<8><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, codes, scales, biases, dst); break;
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
        case 2: dequant_kernel<2><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, src, out); break;
        case 3: dequant_kernel<3><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, src, out); break;
        case 4: dequant_kernel<4><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, src, out); break;
        case 5: dequant_kernel<5><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, src, out); break;
        case 6: dequant_kernel<6><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, src, out); break;
        case 8: dequant_kernel<8><<<(unsigned)blocks, 32, 0, st>>>(group, N, K, KB, src, out); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace affqmm
