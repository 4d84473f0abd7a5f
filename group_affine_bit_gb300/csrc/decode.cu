// decode.cu -- the memory-bound projection for M = 1..16 activation rows.
//
// Each CTA owns one 16-row tile of W and one slice of the depth; its warps
// split the slice's 128-deep blocks.  A warp streams its blocks' code words
// and scale/bias words straight from HBM into registers (a ring of DEC_DEPTH
// blocks in flight), dequantizes every weight once as bf16(fma(s, q, b))
// (affqmm_format.cuh) and contracts on the tensor cores with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate): the weights are the A
// operand (16 rows x 16 k), the activation rows the B operand (8 rows, or two
// MMAs for 9..16 rows).  Prior art: the "reg variant" lane projection of the
// "Gemma 4 12B on the native Metal engine" page (4-bit groups in tensor-op
// registers, K split per shape); unlike it, the weights here are rounded to
// bf16 before the contraction.
//
// Reduction order is fixed: warps of a CTA add in warp order through shared
// memory; when the depth is split across S CTAs each writes an fp32 partial
// and the last CTA to arrive (an atomic counter, no waiting) adds the S
// partials in slice order, converts to bf16 and re-zeroes the counter.  The
// same inputs therefore give the same bits on every run.
#include <cuda_bf16.h>

#include "affqmm_format.cuh"
#include "affqmm_internal.h"

namespace affqmm {
namespace {

constexpr int DEC_DEPTH = 3;  // blocks of codes in flight per warp

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ld_x16(const uint16_t* p, uint32_t* v) {
    // 32 consecutive bf16 of one activation row (64 bytes); read-only, L1-cached
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v[4 * i]), "=r"(v[4 * i + 1]), "=r"(v[4 * i + 2]), "=r"(v[4 * i + 3])
                     : "l"(p + 8 * i));
}

template <int BITS, int MT, int S>
__device__ __forceinline__ void kstep(const uint32_t* cw, uint32_t sg, uint32_t bg, uint32_t sg8, uint32_t bg8,
                                      const uint32_t* xa, const uint32_t* xb, float (&acc)[MT][4]) {
    uint32_t a[4];
    dequant_kstep<BITS, S>(cw, sg, bg, sg8, bg8, a);
    mma_16816(acc[0], a, xa[2 * S], xa[2 * S + 1]);
    if constexpr (MT == 2) mma_16816(acc[1], a, xb[2 * S], xb[2 * S + 1]);
}

template <int BITS, int MT>
__device__ __forceinline__ void block_contract(const uint32_t* cw, uint2 sb, const uint32_t* xa, const uint32_t* xb,
                                               float (&acc)[MT][4]) {
    const uint32_t sg = bcast_lo(sb.x), bg = bcast_hi(sb.x);
    const uint32_t sg8 = bcast_lo(sb.y), bg8 = bcast_hi(sb.y);
    kstep<BITS, MT, 0>(cw, sg, bg, sg8, bg8, xa, xb, acc);
    kstep<BITS, MT, 1>(cw, sg, bg, sg8, bg8, xa, xb, acc);
    kstep<BITS, MT, 2>(cw, sg, bg, sg8, bg8, xa, xb, acc);
    kstep<BITS, MT, 3>(cw, sg, bg, sg8, bg8, xa, xb, acc);
    kstep<BITS, MT, 4>(cw, sg, bg, sg8, bg8, xa, xb, acc);
    kstep<BITS, MT, 5>(cw, sg, bg, sg8, bg8, xa, xb, acc);
    kstep<BITS, MT, 6>(cw, sg, bg, sg8, bg8, xa, xb, acc);
    kstep<BITS, MT, 7>(cw, sg, bg, sg8, bg8, xa, xb, acc);
}

__device__ __forceinline__ uint2 ld_sb(const uint8_t* p) {
    uint32_t a, b;
    ld_stream_v2(p, a, b);
    return make_uint2(a, b);
}

template <int BITS, int MT>
__global__ void __launch_bounds__(DEC_WARPS * 32) decode_kernel(const __grid_constant__ DecParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, t = lane & 3;

    int pi = 0;
    for (int i = 1; i < p.nproj; ++i)
        if ((int)blockIdx.x >= p.proj[i].cta_begin) pi = i;
    const DecProj& P = p.proj[pi];
    const int local = (int)blockIdx.x - P.cta_begin;
    const int S = P.S;
    const int tile = local / S, slice = local - (local / S) * S;
    const int KB = p.KB;
    const int kb_lo = (int)((int64_t)slice * KB / S);
    const int kb_hi = (int)((int64_t)(slice + 1) * KB / S);
    const int nkb = kb_hi - kb_lo;
    const int w_lo = kb_lo + warp * nkb / DEC_WARPS;
    const int w_hi = kb_lo + (warp + 1) * nkb / DEC_WARPS;

    const uint8_t* tbase = P.packed + (size_t)tile * KB * p.block_bytes;
    const int sb_off = sb_offset(BITS, p.group, t, r);
    const bool row0 = r < p.M;
    const bool row1 = (MT == 2) && (r + 8 < p.M);
    const uint16_t* x0 = p.x + (size_t)r * p.K + 32 * t;
    const uint16_t* x1 = p.x + (size_t)(r + 8) * p.K + 32 * t;

    float acc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    uint32_t cw[DEC_DEPTH][2 * BITS];
    uint2 sb[DEC_DEPTH];
#pragma unroll
    for (int i = 0; i < DEC_DEPTH - 1; ++i) {
        if (w_lo + i < w_hi) {
            const uint8_t* blk = tbase + (size_t)(w_lo + i) * p.block_bytes;
            load_lane_codes<BITS>(blk, lane, cw[i]);
            sb[i] = ld_sb(blk + sb_off);
        }
    }
    for (int kb0 = w_lo; kb0 < w_hi; kb0 += DEC_DEPTH) {
#pragma unroll
        for (int i = 0; i < DEC_DEPTH; ++i) {
            const int kb = kb0 + i;
            if (kb < w_hi) {
                const int nxt = kb + DEC_DEPTH - 1;
                if (nxt < w_hi) {
                    const uint8_t* blk = tbase + (size_t)nxt * p.block_bytes;
                    load_lane_codes<BITS>(blk, lane, cw[(i + DEC_DEPTH - 1) % DEC_DEPTH]);
                    sb[(i + DEC_DEPTH - 1) % DEC_DEPTH] = ld_sb(blk + sb_off);
                }
                uint32_t xa[16], xb[16];
                const int64_t kpos = (int64_t)kb * KBLK;
                const bool kin = kpos + 32 * t < p.K;
                if (row0 && kin) {
                    ld_x16(x0 + kpos, xa);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) xa[j] = 0u;
                }
                if constexpr (MT == 2) {
                    if (row1 && kin) {
                        ld_x16(x1 + kpos, xb);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) xb[j] = 0u;
                    }
                }
                block_contract<BITS, MT>(cw[i], sb[i], xa, xb, acc);
            }
        }
    }

    // Fixed-order reduction over the CTA's warps.
    __shared__ float red[DEC_WARPS][MT * 4][32];
    __shared__ int s_last;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[warp][mt * 4 + i][lane] = acc[mt][i];
    __syncthreads();

    float v[MT * 4];
    if (warp == 0) {
#pragma unroll
        for (int j = 0; j < MT * 4; ++j) {
            float s = red[0][j][lane];
#pragma unroll
            for (int w = 1; w < DEC_WARPS; ++w) s += red[w][j][lane];
            v[j] = s;
        }
        if (S > 1) {
            float* slot = p.partials + (size_t)(P.part_begin + (int64_t)tile * S + slice) * 256 + lane * 8;
#pragma unroll
            for (int j = 0; j < MT * 4; ++j) slot[j] = v[j];
            __threadfence();
        }
    }
    if (S > 1) {
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned prev = atomicAdd(&p.counters[P.ctr_begin + tile], 1u);
            s_last = (prev == (unsigned)(S - 1));
        }
        __syncthreads();
        if (!s_last || warp != 0) return;
        __threadfence();
#pragma unroll
        for (int j = 0; j < MT * 4; ++j) v[j] = 0.f;
        for (int sl = 0; sl < S; ++sl) {
            const float* slot = p.partials + (size_t)(P.part_begin + (int64_t)tile * S + sl) * 256 + lane * 8;
#pragma unroll
            for (int j = 0; j < MT * 4; ++j) v[j] += __ldcg(slot + j);
        }
        if (lane == 0) p.counters[P.ctr_begin + tile] = 0u;
    } else if (warp != 0) {
        return;
    }

    // y[m, n]: lane (r, t) holds n = r (+8) and m = 8*mt + 2t (+1).
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t n = (int64_t)tile * TILE_N + r + (i >= 2 ? 8 : 0);
            const int m = mt * 8 + 2 * t + (i & 1);
            if (n < P.N && m < p.M) {
                const __nv_bfloat16 h = __float2bfloat16_rn(v[mt * 4 + i]);
                P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(h);
            }
        }
    }
}

template <int BITS>
cudaError_t launch_bits(int mt, const DecParams& p, int grid, cudaStream_t st) {
    if (mt == 1)
        decode_kernel<BITS, 1><<<grid, DEC_WARPS * 32, 0, st>>>(p);
    else
        decode_kernel<BITS, 2><<<grid, DEC_WARPS * 32, 0, st>>>(p);
    return cudaGetLastError();
}

template <int BITS>
int occupancy_bits(int mt) {
    int n = 0;
    cudaError_t e = mt == 1 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, 1>, DEC_WARPS * 32, 0)
                            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, 2>, DEC_WARPS * 32, 0);
    return e == cudaSuccess ? n : -1;
}

}  // namespace

cudaError_t launch_decode(int bits, int mt, const DecParams& p, int grid, cudaStream_t st) {
    switch (bits) {
        case 2: return launch_bits<2>(mt, p, grid, st);
        case 3: return launch_bits<3>(mt, p, grid, st);
        case 4: return launch_bits<4>(mt, p, grid, st);
        case 5: return launch_bits<5>(mt, p, grid, st);
        case 6: return launch_bits<6>(mt, p, grid, st);
        case 8: return launch_bits<8>(mt, p, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

int decode_ctas_per_sm(int bits, int mt) {
    switch (bits) {
        case 2: return occupancy_bits<2>(mt);
        case 3: return occupancy_bits<3>(mt);
        case 4: return occupancy_bits<4>(mt);
        case 5: return occupancy_bits<5>(mt);
        case 6: return occupancy_bits<6>(mt);
        case 8: return occupancy_bits<8>(mt);
        default: return -1;
    }
}

}  // namespace affqmm
