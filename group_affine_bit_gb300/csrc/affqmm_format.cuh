// affqmm_format.cuh -- the packed affine-table layout and the device-side
// dequantization shared by every libaffqmm kernel.
//
// One layout serves the decode and the prompt kernels, as the pages' AffineN
// tiles serve both paths ("cuda gemma4: images on the 12B" page, the widths
// commit):
//
//   * rows are cut into tiles of 128 (TILE_N), the depth into blocks of 128
//     (KBLK); a (tile, k-block) "block" is contiguous, the blocks of one tile
//     follow each other in k order and tiles follow in n order, so any run of
//     consecutive blocks is one contiguous range of bytes (one bulk copy);
//   * one thread owns one row of a block: the 128 codes of its row as bit
//     planes (a width is 4+4, 4+2, 4+1, 4, 2+1 or 2 bits), read as 16-byte
//     chunks that 32 consecutive rows store side by side (a warp's read is
//     one coalesced 512-byte access), then its row's scale/bias words;
//   * a scale/bias word is s | b << 16 (two bf16 patterns), one per group of
//     `group` k in the block, stored row-major after the codes.
//
// In a plane of p bits a row's 128 codes fill 4p words.  Word w holds the
// codes of k in [w*32/p, (w+1)*32/p) as 16/p pairs: pair i (k = w*32/p + 2i
// and the next k) keeps the first code at bits [p*i, p*i + p) and the second
// at bits [16 + p*i, 16 + p*i + p), so one AND/OR gives both as a bf16x2.
// Pair c of the row (k = 2c, 2c + 1) is what the kernels hold in one 32-bit
// register: column c of a tensor-memory row, or 4 bytes of a shared-memory
// row.
#pragma once
#include <cstdint>

namespace affqmm {

constexpr int TILE_N = 128;
constexpr int KBLK = 128;

__host__ __device__ constexpr int plane0_bits(int bits) { return bits <= 3 ? 2 : 4; }
__host__ __device__ constexpr int plane1_bits(int bits) { return bits - plane0_bits(bits); }
// bytes of codes in one block, and of one row's codes in one plane
__host__ __device__ constexpr int code_bytes(int bits) { return 2048 * bits; }
__host__ __device__ constexpr int row_plane_bytes(int p) { return 16 * p; }
__host__ __device__ constexpr int sb_words(int group) { return KBLK / group; }
__host__ __device__ constexpr int sb_bytes(int group) { return TILE_N * 4 * sb_words(group); }
__host__ __device__ constexpr int block_bytes(int bits, int group) { return code_bytes(bits) + sb_bytes(group); }
__host__ __device__ constexpr int plane_offset(int bits, int plane) { return plane == 0 ? 0 : 2048 * plane0_bits(bits); }
// Byte offset inside a block of 16-byte chunk c (0 .. p-1) of row n's plane.
__host__ __device__ constexpr int chunk_offset(int bits, int plane, int n, int c) {
    return plane_offset(bits, plane) + ((n >> 5) * (plane ? plane1_bits(bits) : plane0_bits(bits)) + c) * 512 +
           (n & 31) * 16;
}
// Byte offset inside a block of row n's scale/bias words.
__host__ __device__ constexpr int sb_offset(int bits, int group, int n) {
    return code_bytes(bits) + n * 4 * sb_words(group);
}

#if defined(__CUDACC__)

// ---------------------------------------------------------------- bf16x2 ops
__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// (a & mask) | c in one LOP3
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t bcast_lo(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

constexpr uint32_t BF2_MAGIC = 0x43004300u;        // 128.0 in both halves: ulp 1
constexpr uint32_t BF2_ONE = 0x3F803F80u;          // 1.0
constexpr uint32_t BF2_MINUS_MAGIC = 0xC300C300u;  // -128.0
constexpr uint32_t BF2_SIXTEEN = 0x41804180u;      // 16.0

template <int SH>
__device__ __forceinline__ uint32_t shr(uint32_t v) {
    if constexpr (SH == 0) return v;
    else if constexpr (SH > 0) return v >> SH;
    else return v << (-SH);
}

// The exact codes of pair C (k = 2C, 2C + 1) of a row as bf16x2, from the
// row's words cw[] (plane 0's 4*p0 words, then plane 1's).  128 + q is exact
// in bf16 for q < 128 (q in the mantissa of the 0x4300 magic) and taking 128
// away leaves q exactly; an 8-bit code is 16*hi + lo, also exact.
template <int BITS, int C>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* cw) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
    constexpr int W0 = C / (16 / P0), I0 = C % (16 / P0);
    constexpr uint32_t M0 = ((1u << P0) - 1u) * 0x00010001u;
    const uint32_t lo = shr<P0 * I0>(cw[W0]);
    if constexpr (P1 == 0) {
        return bf2_fma(and_or(lo, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
    } else if constexpr (BITS < 8) {
        constexpr int W1 = C / (16 / P1), I1 = C % (16 / P1);
        constexpr uint32_t M1 = (((1u << P1) - 1u) << P0) * 0x00010001u;
        const uint32_t hi = shr<P1 * I1 - P0>(cw[4 * P0 + W1]);
        return bf2_fma(and_or(hi, M1, and_or(lo, M0, BF2_MAGIC)), BF2_ONE, BF2_MINUS_MAGIC);
    } else {
        const uint32_t hi = shr<P1 * I0>(cw[4 * P0 + W0]);
        const uint32_t ql = bf2_fma(and_or(lo, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
        const uint32_t qh = bf2_fma(and_or(hi, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
        return bf2_fma(qh, BF2_SIXTEEN, ql);
    }
}

// Weight pair C of a row: bf16(fma(s, q, b)), ONE rounding (fma.rn.bf16x2
// rounds the exact s*q + b once).  sbw[] are the row's scale/bias words.
template <int BITS, int GROUP, int C>
__device__ __forceinline__ uint32_t weight_pair(const uint32_t* cw, const uint32_t* sbw) {
    constexpr int GI = (2 * C) / GROUP;
    return bf2_fma(code_pair<BITS, C>(cw), bcast_lo(sbw[GI]), bcast_hi(sbw[GI]));
}

// Pairs [C0, C0 + NC) of a row into w[0 .. NC).
template <int BITS, int GROUP, int C0, int NC>
__device__ __forceinline__ void weight_pairs(const uint32_t* cw, const uint32_t* sbw, uint32_t* w) {
    if constexpr (NC > 0) {
        w[0] = weight_pair<BITS, GROUP, C0>(cw, sbw);
        weight_pairs<BITS, GROUP, C0 + 1, NC - 1>(cw, sbw, w + 1);
    }
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ void ld_stream_v4(const void* p, uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "l"(p));
}
__device__ __forceinline__ void lds_v4(uint32_t a, uint32_t& x, uint32_t& y, uint32_t& z, uint32_t& w) {
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(x), "=r"(y), "=r"(z), "=r"(w) : "r"(a) : "memory");
}
__device__ __forceinline__ void lds_v2(uint32_t a, uint32_t& x, uint32_t& y) {
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(x), "=r"(y) : "r"(a) : "memory");
}
__device__ __forceinline__ void lds_v1(uint32_t a, uint32_t& x) {
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(a) : "memory");
}

// Row n's code words (4*BITS) of a block in global memory.
template <int BITS>
__device__ __forceinline__ void load_row_codes(const uint8_t* blk, int n, uint32_t* cw) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
#pragma unroll
    for (int c = 0; c < P0; ++c) {
        const uint8_t* q = blk + chunk_offset(BITS, 0, n, c);
        ld_stream_v4(q, cw[4 * c], cw[4 * c + 1], cw[4 * c + 2], cw[4 * c + 3]);
    }
#pragma unroll
    for (int c = 0; c < P1; ++c) {
        const uint8_t* q = blk + chunk_offset(BITS, 1, n, c);
        uint32_t* d = cw + 4 * P0;
        ld_stream_v4(q, d[4 * c], d[4 * c + 1], d[4 * c + 2], d[4 * c + 3]);
    }
}

// The same words from a block staged in shared memory (same layout).
template <int BITS>
__device__ __forceinline__ void load_row_codes_smem(uint32_t blk, int n, uint32_t* cw) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
#pragma unroll
    for (int c = 0; c < P0; ++c) lds_v4(blk + chunk_offset(BITS, 0, n, c), cw[4 * c], cw[4 * c + 1], cw[4 * c + 2], cw[4 * c + 3]);
#pragma unroll
    for (int c = 0; c < P1; ++c) {
        uint32_t* d = cw + 4 * P0;
        lds_v4(blk + chunk_offset(BITS, 1, n, c), d[4 * c], d[4 * c + 1], d[4 * c + 2], d[4 * c + 3]);
    }
}

// Row n's scale/bias words (KBLK / GROUP of them) from global or shared memory.
template <int GROUP>
__device__ __forceinline__ void load_row_sb(const uint8_t* p, uint32_t* sbw) {
    if constexpr (GROUP == 32) ld_stream_v4(p, sbw[0], sbw[1], sbw[2], sbw[3]);
    else if constexpr (GROUP == 64) {
        uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
        sbw[0] = v.x;
        sbw[1] = v.y;
    } else {
        sbw[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
    }
}
template <int GROUP>
__device__ __forceinline__ void load_row_sb_smem(uint32_t a, uint32_t* sbw) {
    if constexpr (GROUP == 32) lds_v4(a, sbw[0], sbw[1], sbw[2], sbw[3]);
    else if constexpr (GROUP == 64) lds_v2(a, sbw[0], sbw[1]);
    else lds_v1(a, sbw[0]);
}

#endif  // __CUDACC__

}  // namespace affqmm
