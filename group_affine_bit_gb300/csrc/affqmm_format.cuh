// affqmm_format.cuh -- the packed affine-table layout and the device-side
// dequantization shared by every libaffqmm kernel.
//
// Layout (one layout for the decode and the prompt kernels, as the pages'
// AffineN tiles serve both paths -- "cuda gemma4: images on the 12B" page,
// the widths commit):
//
//   * rows are cut into tiles of 16 (TILE_N), the depth into blocks of 128
//     (KBLK); a (tile, k-block) "block" is contiguous and the blocks of one
//     tile follow each other in k order, tiles in n order;
//   * a block holds the codes of its 16 x 128 weights as bit planes (a width
//     is 4+4, 4+2, 4+1, 4, 2+1 or 2 bits), then the scale/bias words;
//   * inside a plane, 32 "lanes" each own the codes of two rows (r, r+8) and
//     32 consecutive k, the operand fragment one lane of an m16n8k16 MMA
//     holds over 8 k-steps; a warp reads each plane chunk with one coalesced
//     vector load;
//   * a scale/bias word is s | b << 16 (two bf16 patterns); a lane's 32 k sit
//     inside one group for every group size 32, 64, 128.
//
// Lane l = 4*r + t (r = 0..7, t = 0..3) owns rows r and r+8 and k = 32t..32t+31
// of the block.  For k-step s (0..7) the MMA slots {2t, 2t+1, 2t+8, 2t+9} of
// the 16-deep step hold k = 32t + 4s + {0, 1, 2, 3}: the contraction is the
// same sum over k in another order of the terms inside one MMA.
//
// A k-step needs four bf16x2 registers: reg0 = W[r][k0..k0+1],
// reg1 = W[r+8][k0..k0+1], reg2 = W[r][k0+2..k0+3], reg3 = W[r+8][k0+2..k0+3]
// (k0 = 32t + 4s).  In a plane of p bits one 32-bit word holds 16/p such
// register pairs: pair i = (s mod (4/p)) * 4 + reg keeps its low element at
// bits [p*i, p*i + p) and its high element at bits [16 + p*i, 16 + p*i + p);
// word index (within the lane's plane) is s*p/4.
#pragma once
#include <cstdint>

namespace affqmm {

constexpr int TILE_N = 16;
constexpr int KBLK = 128;

__host__ __device__ constexpr int plane0_bits(int bits) { return bits <= 3 ? 2 : 4; }
__host__ __device__ constexpr int plane1_bits(int bits) { return bits - plane0_bits(bits); }
__host__ __device__ constexpr int code_bytes(int bits) { return 256 * bits; }
__host__ __device__ constexpr int sb_bytes(int group) { return 8192 / group; }
__host__ __device__ constexpr int block_bytes(int bits, int group) {
    return code_bytes(bits) + sb_bytes(group);
}
// Bytes one lane owns in a plane of p bits, and the vector chunk it is read in.
__host__ __device__ constexpr int lane_plane_bytes(int p) { return 8 * p; }
__host__ __device__ constexpr int chunk_bytes(int p) { return p >= 2 ? 16 : 8; }
__host__ __device__ constexpr int plane_offset(int bits, int plane) {
    return plane == 0 ? 0 : 256 * plane0_bits(bits);
}
// Byte offset, inside a block, of word w (0 .. 2p-1) of lane `lane` in a plane.
__host__ __device__ constexpr int plane_word_offset(int bits, int plane, int lane, int w) {
    return plane_offset(bits, plane) +
           (w * 4 / chunk_bytes(plane ? plane1_bits(bits) : plane0_bits(bits))) *
               (32 * chunk_bytes(plane ? plane1_bits(bits) : plane0_bits(bits))) +
           lane * chunk_bytes(plane ? plane1_bits(bits) : plane0_bits(bits)) +
           (w * 4) % chunk_bytes(plane ? plane1_bits(bits) : plane0_bits(bits));
}
// Scale/bias words of a block: [group slot gi][row pair r][row r, row r+8].
__host__ __device__ constexpr int sb_offset(int bits, int group, int t, int r) {
    return code_bytes(bits) + (((32 * t) / group) * 8 + r) * 8;
}

#if defined(__CUDACC__)

// ---------------------------------------------------------------- bf16x2 ops
__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// (a & mask) | magic, one LOP3
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t magic) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
    return d;
}
// (a & mask) | c, same LOP3, named for merging a second field
__device__ __forceinline__ uint32_t merge_field(uint32_t a, uint32_t mask, uint32_t c) {
    return and_or(a, mask, c);
}
__device__ __forceinline__ uint32_t bcast_lo(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

constexpr uint32_t BF2_MAGIC = 0x43004300u;    // 128.0 in both halves: ulp 1
constexpr uint32_t BF2_ONE = 0x3F803F80u;      // 1.0
constexpr uint32_t BF2_MINUS_MAGIC = 0xC300C300u;  // -128.0
constexpr uint32_t BF2_SIXTEEN = 0x41804180u;  // 16.0

template <int SH>
__device__ __forceinline__ uint32_t shr(uint32_t v) {
    if constexpr (SH == 0) return v;
    else if constexpr (SH > 0) return v >> SH;
    else return v << (-SH);
}

// The exact code pair of register `reg` (0..3) of k-step s (0..7) as bf16x2,
// from a lane's code words cw[]: plane 0 words first (2*p0 of them), then
// plane 1.  128 + q is exact in bf16 for q < 128 (the 0x4300 magic with q in
// the mantissa), and subtracting 128 leaves q exactly.  An 8-bit code is
// 16*hi + lo, also exact (at most 255 needs 8 significant bits).
template <int BITS, int S, int REG>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* cw) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
    constexpr int W0 = S * P0 / 4;
    constexpr int I0 = (S % (4 / P0)) * 4 + REG;
    constexpr uint32_t M0 = ((1u << P0) - 1u) * 0x00010001u;
    const uint32_t lo = shr<P0 * I0>(cw[W0]);
    if constexpr (P1 == 0) {
        return bf2_fma(and_or(lo, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
    } else if constexpr (BITS < 8) {
        constexpr int W1 = S * P1 / 4;
        constexpr int I1 = (S % (4 / P1)) * 4 + REG;
        constexpr uint32_t M1 = (((1u << P1) - 1u) << P0) * 0x00010001u;
        const uint32_t hi = shr<P1 * I1 - P0>(cw[2 * P0 + W1]);
        const uint32_t qm = merge_field(hi, M1, and_or(lo, M0, BF2_MAGIC));
        return bf2_fma(qm, BF2_ONE, BF2_MINUS_MAGIC);
    } else {
        const uint32_t hi = shr<P1 * I0>(cw[2 * P0 + W0]);
        const uint32_t ql = bf2_fma(and_or(lo, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
        const uint32_t qh = bf2_fma(and_or(hi, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
        return bf2_fma(qh, BF2_SIXTEEN, ql);
    }
}

// The four A-fragment registers of k-step S: W = bf16(fma(s, q, b)), ONE
// rounding (fma.rn.bf16x2 rounds the exact s*q + b once).  sg/bg are the row-r
// scale and bias broadcast to both halves, sg8/bg8 those of row r+8.
template <int BITS, int S>
__device__ __forceinline__ void dequant_kstep(const uint32_t* cw, uint32_t sg, uint32_t bg,
                                              uint32_t sg8, uint32_t bg8, uint32_t (&a)[4]) {
    a[0] = bf2_fma(code_pair<BITS, S, 0>(cw), sg, bg);
    a[1] = bf2_fma(code_pair<BITS, S, 1>(cw), sg8, bg8);
    a[2] = bf2_fma(code_pair<BITS, S, 2>(cw), sg, bg);
    a[3] = bf2_fma(code_pair<BITS, S, 3>(cw), sg8, bg8);
}

// Load one lane's code words of one block (2*BITS words) with vector loads.
// Streaming: the weights are read once, so they bypass L1.
__device__ __forceinline__ void ld_stream_v4(const void* p, uint32_t& a, uint32_t& b, uint32_t& c,
                                             uint32_t& d) {
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "l"(p));
}
__device__ __forceinline__ void ld_stream_v2(const void* p, uint32_t& a, uint32_t& b) {
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(a), "=r"(b)
                 : "l"(p));
}

template <int BITS>
__device__ __forceinline__ void load_lane_codes(const uint8_t* blk, int lane, uint32_t* cw) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
#pragma unroll
    for (int c = 0; c < lane_plane_bytes(P0) / chunk_bytes(P0); ++c) {
        const uint8_t* p = blk + plane_offset(BITS, 0) + c * 32 * chunk_bytes(P0) + lane * chunk_bytes(P0);
        if constexpr (chunk_bytes(P0) == 16)
            ld_stream_v4(p, cw[4 * c], cw[4 * c + 1], cw[4 * c + 2], cw[4 * c + 3]);
        else
            ld_stream_v2(p, cw[2 * c], cw[2 * c + 1]);
    }
    if constexpr (P1 > 0) {
#pragma unroll
        for (int c = 0; c < lane_plane_bytes(P1) / chunk_bytes(P1); ++c) {
            const uint8_t* p = blk + plane_offset(BITS, 1) + c * 32 * chunk_bytes(P1) + lane * chunk_bytes(P1);
            uint32_t* d = cw + 2 * P0;
            if constexpr (chunk_bytes(P1) == 16)
                ld_stream_v4(p, d[4 * c], d[4 * c + 1], d[4 * c + 2], d[4 * c + 3]);
            else
                ld_stream_v2(p, d[2 * c], d[2 * c + 1]);
        }
    }
}

// The same lane words read from a block staged in shared memory (same layout).
template <int BITS>
__device__ __forceinline__ void load_lane_codes_smem(uint32_t blk, int lane, uint32_t* cw) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
#pragma unroll
    for (int c = 0; c < lane_plane_bytes(P0) / chunk_bytes(P0); ++c) {
        const uint32_t a = blk + plane_offset(BITS, 0) + c * 32 * chunk_bytes(P0) + lane * chunk_bytes(P0);
        if constexpr (chunk_bytes(P0) == 16)
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(cw[4 * c]), "=r"(cw[4 * c + 1]), "=r"(cw[4 * c + 2]), "=r"(cw[4 * c + 3])
                         : "r"(a));
        else
            asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(cw[2 * c]), "=r"(cw[2 * c + 1]) : "r"(a));
    }
    if constexpr (P1 > 0) {
#pragma unroll
        for (int c = 0; c < lane_plane_bytes(P1) / chunk_bytes(P1); ++c) {
            const uint32_t a = blk + plane_offset(BITS, 1) + c * 32 * chunk_bytes(P1) + lane * chunk_bytes(P1);
            uint32_t* d = cw + 2 * P0;
            if constexpr (chunk_bytes(P1) == 16)
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(d[4 * c]), "=r"(d[4 * c + 1]), "=r"(d[4 * c + 2]), "=r"(d[4 * c + 3])
                             : "r"(a));
            else
                asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(d[2 * c]), "=r"(d[2 * c + 1]) : "r"(a));
        }
    }
}

#endif  // __CUDACC__

}  // namespace affqmm
