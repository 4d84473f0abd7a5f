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
//   * a row's 128 codes are stored as bit planes (a width is 4+4, 4+2, 4+1,
//     4, 2+1 or 2 bits); in a plane of p bits the row has 4p words, read as p
//     16-byte chunks that 32 consecutive rows store side by side, each row's
//     chunk at a row slot swizzled by the chunk index, so that a warp reading
//     one chunk of 32 rows (one thread per row) and a warp reading the four
//     k-classes of 8 rows (the tensor-core fragment order below) both touch
//     every shared-memory bank once;
//   * a scale/bias word is s | b << 16 (two bf16 patterns), one per group of
//     `group` k in the block, stored row-major after the codes.
//
// Pairs and classes.  Pair C of a row holds k = 2C and 2C + 1 as a bf16x2 (the
// first code at bits [p*i, p*i + p) of its word, the second at [16 + p*i, ...),
// so one AND/OR gives both).  Pair C belongs to class C mod 4: the pairs a
// thread of a warp-level matrix fragment (16 rows x 16 k per step, thread t
// holding k = 2(t mod 4) and 2(t mod 4) + 8 of its rows) uses across the 8
// steps of a block.  Words are class-major: word p*c + v of a plane holds
// class c's pairs j = v*(16/p) .. v*(16/p) + 16/p - 1 (pair C = 4j + c), so a
// fragment thread reads its class as p consecutive words of each row and a
// row-per-thread reader reads all 4p words.
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
// Row-slot swizzle of chunk c in a plane of p bits: the fragment reader's
// eight rows x four classes land on distinct 16-byte bank groups.
__host__ __device__ constexpr int chunk_swizzle(int p, int c) { return (c * (8 / p)) & 7; }
// Byte offset inside a block of 16-byte chunk c (0 .. p-1) of row n's plane.
__host__ __device__ constexpr int chunk_offset(int bits, int plane, int n, int c) {
    return plane_offset(bits, plane) + ((n >> 5) * (plane ? plane1_bits(bits) : plane0_bits(bits)) + c) * 512 +
           ((n & 31) ^ chunk_swizzle(plane ? plane1_bits(bits) : plane0_bits(bits), c)) * 16;
}
// Byte offset inside a block of word w (0 .. 4p-1) of row n's plane.
__host__ __device__ constexpr int word_offset(int bits, int plane, int n, int w) {
    return chunk_offset(bits, plane, n, w >> 2) + 4 * (w & 3);
}
// Byte offset inside a block of row n's scale/bias words.
__host__ __device__ constexpr int sb_offset(int bits, int group, int n) {
    return code_bytes(bits) + n * 4 * sb_words(group);
}

// The row-contiguous copy of a packed table that the embedding gather reads
// (affqmm_pack_rows): the same words as the blocks above, regrouped by row so
// that one row's bytes are one contiguous range.  Row n starts at
// n * rows_stride; in it come the 4*bits code words of each 128-deep block
// in block order (the words load_row_codes returns, in that order), then the
// scale/bias words of every block in block order; the stride is padded to
// 16 bytes.
__host__ __device__ constexpr int64_t rows_stride(int bits, int group, int KB) {
    return ((int64_t)KB * (16 * bits + 4 * sb_words(group)) + 15) / 16 * 16;
}
__host__ __device__ constexpr int64_t rows_codes_offset(int bits, int kb) { return (int64_t)kb * 16 * bits; }
__host__ __device__ constexpr int64_t rows_sb_offset(int bits, int group, int KB, int kb) {
    return (int64_t)KB * 16 * bits + (int64_t)kb * 4 * sb_words(group);
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

// The exact codes of class pair J (pair C = 4J + c of class c) as bf16x2,
// from the class's words: w0[] its p0 words of plane 0, w1[] its p1 words of
// plane 1.  128 + q is exact in bf16 for q < 128 (q in the mantissa of the
// 0x4300 magic) and taking 128 away leaves q exactly; an 8-bit code is
// 16*hi + lo, also exact.
template <int BITS, int J>
__device__ __forceinline__ uint32_t class_code_pair(const uint32_t* w0, const uint32_t* w1) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
    constexpr int V0 = J / (16 / P0), I0 = J % (16 / P0);
    constexpr uint32_t M0 = ((1u << P0) - 1u) * 0x00010001u;
    const uint32_t lo = shr<P0 * I0>(w0[V0]);
    if constexpr (P1 == 0) {
        return bf2_fma(and_or(lo, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
    } else if constexpr (BITS < 8) {
        constexpr int V1 = J / (16 / P1), I1 = J % (16 / P1);
        constexpr uint32_t M1 = (((1u << P1) - 1u) << P0) * 0x00010001u;
        const uint32_t hi = shr<P1 * I1 - P0>(w1[V1]);
        return bf2_fma(and_or(hi, M1, and_or(lo, M0, BF2_MAGIC)), BF2_ONE, BF2_MINUS_MAGIC);
    } else {
        const uint32_t hi = shr<P1 * I0>(w1[V0]);
        const uint32_t ql = bf2_fma(and_or(lo, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
        const uint32_t qh = bf2_fma(and_or(hi, M0, BF2_MAGIC), BF2_ONE, BF2_MINUS_MAGIC);
        return bf2_fma(qh, BF2_SIXTEEN, ql);
    }
}

// The exact codes of pair C (k = 2C, 2C + 1) of a row from the row's words
// cw[] (plane 0's 4*p0 words, then plane 1's).
template <int BITS, int C>
__device__ __forceinline__ uint32_t code_pair(const uint32_t* cw) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
    return class_code_pair<BITS, C / 4>(cw + P0 * (C % 4), cw + 4 * P0 + P1 * (C % 4));
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

// The same words from a row of the row-contiguous copy (16-byte aligned).
template <int BITS>
__device__ __forceinline__ void load_rowcopy_codes(const uint8_t* p, uint32_t* cw) {
#pragma unroll
    for (int v = 0; v < BITS; ++v) ld_stream_v4(p + 16 * v, cw[4 * v], cw[4 * v + 1], cw[4 * v + 2], cw[4 * v + 3]);
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

// ---------------------------------------------------------------- fragment (class) form
// A matrix-fragment thread of class c (its index mod 4) holds, for each of
// its rows, the class's p words of every plane: pairs j = 0..15 of the class,
// k = 8j + 2c and the next.
template <int P>
__device__ __forceinline__ void lds_words(uint32_t a, uint32_t* w) {
    if constexpr (P == 4) lds_v4(a, w[0], w[1], w[2], w[3]);
    else if constexpr (P == 2) lds_v2(a, w[0], w[1]);
    else lds_v1(a, w[0]);
}
// Class c's words of row n (plane 0's p0, then plane 1's p1) from a block
// staged in shared memory.
template <int BITS>
__device__ __forceinline__ void load_class_words_smem(uint32_t blk, int n, int c, uint32_t* w) {
    constexpr int P0 = plane0_bits(BITS);
    constexpr int P1 = plane1_bits(BITS);
    lds_words<P0>(blk + word_offset(BITS, 0, n, P0 * c), w);
    if constexpr (P1 > 0) lds_words<P1>(blk + word_offset(BITS, 1, n, P1 * c), w + P0);
}
// Weight pair J of a row's class: bf16(fma(s, q, b)), one rounding.  The
// class offset 2c < 8 never crosses a group boundary (groups are multiples
// of 32), so the group is that of k = 8J.
template <int BITS, int GROUP, int J>
__device__ __forceinline__ uint32_t class_weight_pair(const uint32_t* w, const uint32_t* sbw) {
    constexpr int GI = (8 * J) / GROUP;
    return bf2_fma(class_code_pair<BITS, J>(w, w + plane0_bits(BITS)), bcast_lo(sbw[GI]), bcast_hi(sbw[GI]));
}

#endif  // __CUDACC__

}  // namespace affqmm
