// decode.cu -- the memory-bound projection for M = 1..16 activation rows.
//
// A CTA is one producer warp and `su` (<= 8) consumer warps.  The projection's
// 128-deep weight blocks are grouped into stages of up to `su` consecutive
// blocks of one 16-row tile; the stages are cut into one contiguous run per
// resident CTA ("stream-K"), so every SM streams the same number of bytes.
// The producer moves each stage from HBM into a ring of shared-memory slots
// with ONE 1-D bulk copy (TMA) -- a few large copies in flight keep HBM busy
// where many small ones do not -- and consumer warp w takes block w of the
// stage: it reads its fragment words back from shared memory, dequantizes
// every weight once as bf16(fma(s, q, b)) (affqmm_format.cuh) and contracts
// on the tensor cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate): the
// weights are the A operand (16 rows x 16 k), the activation rows the B
// operand (8 rows, or two MMAs for 9..16 rows).  Prior art: the "reg
// variant" lane projection of the "Gemma 4 12B on the native Metal engine"
// page (4-bit groups in tensor-op registers, K split per shape); unlike it,
// the weights here are rounded to bf16 before the contraction, as the same
// page's prompt GEMM does.
//
// Reduction order is fixed: each consumer warp sums its blocks in k order in
// interleaved chains (k-step s of every block into chain s mod CH);
// at the end of a tile's segment the warps' sums are added in warp order
// through shared memory; a tile cut by CTA run boundaries gets one fp32
// partial per run, and the last CTA to arrive (an atomic counter, no
// waiting) adds them in run order and re-zeroes the counter.  The cut
// depends only on the projection, M and the device, so the same inputs give
// the same bits on every call, alone or stacked with other projections.
// Every wait is on an mbarrier with a bounded wait; a wait that gives up sets
// the workspace status word and the CTA stops.
#include <cuda_bf16.h>

#include "affqmm_async.cuh"
#include "affqmm_format.cuh"
#include "affqmm_internal.h"

namespace affqmm {
namespace {

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

// Independent accumulator chains: k-step s of a block adds into chain
// s % CH, so several tensor-core MMAs are in flight instead of one dependent
// sequence (four chains for up to 8 rows, two for 9..16 rows, whose two MMAs
// per k-step are already independent).  The chains are added in a fixed
// order when a tile segment ends.
template <int MT>
constexpr int dec_chains() { return MT == 1 ? 4 : 2; }

template <int BITS, int MT, int S>
__device__ __forceinline__ void kstep(const uint32_t* cw, uint32_t sg, uint32_t bg, uint32_t sg8, uint32_t bg8,
                                      const uint32_t* xa, const uint32_t* xb,
                                      float (&acc)[dec_chains<MT>()][MT][4]) {
    constexpr int CH = dec_chains<MT>();
    uint32_t a[4];
    dequant_kstep<BITS, S>(cw, sg, bg, sg8, bg8, a);
    mma_16816(acc[S % CH][0], a, xa[2 * S], xa[2 * S + 1]);
    if constexpr (MT == 2) mma_16816(acc[S % CH][1], a, xb[2 * S], xb[2 * S + 1]);
}

template <int BITS, int MT>
__device__ __forceinline__ void block_contract(const uint32_t* cw, uint2 sb, const uint32_t* xa, const uint32_t* xb,
                                               float (&acc)[dec_chains<MT>()][MT][4]) {
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

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* addr, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// y[m, n] from a lane's accumulator: lane (r, t) holds n = r (+8) and
// m = 8*mt + 2t (+1).
template <int MT>
__device__ __forceinline__ void store_y(const DecProj& P, int M, int tile, int r, int t, const float* v) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t n = (int64_t)tile * TILE_N + r + (i >= 2 ? 8 : 0);
            const int m = mt * 8 + 2 * t + (i & 1);
            if (n < P.N && m < M) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[mt * 4 + i]));
        }
    }
}

// The CTA whose run holds stage g of a projection with S stages cut into PC
// runs: the largest c with floor(c*S/PC) <= g.
__device__ __forceinline__ int cta_of(int g, int S, int PC) {
    return (int)(((int64_t)(g + 1) * PC - 1) / S);
}

// Publish a partial tile segment of this CTA's run: store its fp32 sums in one
// of the CTA's two slots, count it on the tile's counter, and if it is the last
// of the tile's segments to arrive, add all of them in run (k) order, store y
// and reset the counter.  Executed by one warp.
template <int MT>
__device__ __forceinline__ void publish_partial(const DecParams& p, const DecProj& P, int c, int tile, bool first_seg,
                                                int lane, const float* v_in) {
    const int r = lane >> 2, t = lane & 3;
    const int S = P.stages, PC = P.nctas;
    const int slot = P.slot_begin + 2 * c + (first_seg ? 0 : 1);
    float* sp = p.partials + (size_t)slot * 256 + lane * 8;
#pragma unroll
    for (int j = 0; j < MT * 4; ++j) __stcg(sp + j, v_in[j]);
    // Lane 0's release publishes the warp's stores (ordered by __syncwarp);
    // the acquire side makes every earlier partial visible to the last CTA.
    __syncwarp();
    unsigned prev = 0;
    if (lane == 0) prev = atom_add_acq_rel(&p.counters[P.ctr_begin + tile], 1u);
    __syncwarp();
    prev = __shfl_sync(0xffffffffu, prev, 0);
    const int g0 = tile * p.spt, g1 = g0 + p.spt - 1;
    const int cf = cta_of(g0, S, PC), cl = cta_of(g1, S, PC);
    if (prev != (unsigned)(cl - cf)) return;
    float v[MT * 4];
#pragma unroll
    for (int j = 0; j < MT * 4; ++j) v[j] = 0.f;
    for (int cb = cf; cb <= cl; ++cb) {
        const int b0 = (int)((int64_t)cb * S / PC);
        const int sc = P.slot_begin + 2 * cb + (b0 >= g0 ? 0 : 1);
        const float* cp = p.partials + (size_t)sc * 256 + lane * 8;
#pragma unroll
        for (int j = 0; j < MT * 4; ++j) v[j] += __ldcg(cp + j);
    }
    store_y<MT>(P, p.M, tile, r, t, v);
    if (lane == 0) p.counters[P.ctr_begin + tile] = 0u;
}

template <int BITS, int MT>
__global__ void __launch_bounds__((DEC_MAX_SU + 1) * 32) decode_kernel(const __grid_constant__ DecParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int SU = p.su, NS = p.ring, SBY = p.stage_bytes, KB = p.KB, SPT = p.spt;
    const int bb = p.block_bytes;

    int pi = 0;
    for (int i = 1; i < p.nproj; ++i)
        if ((int)blockIdx.x >= p.proj[i].cta_begin) pi = i;
    const DecProj& P = p.proj[pi];
    const int c = (int)blockIdx.x - P.cta_begin;
    const int S = P.stages, PC = P.nctas;
    const int g_lo = (int)((int64_t)c * S / PC);
    const int g_hi = (int)((int64_t)(c + 1) * S / PC);

    // shared memory: ring | reduction buffers [2][SU][MT*4][32] | barriers
    const uint32_t s_base = smem_u32(smem);
    float* red = reinterpret_cast<float*>(smem + (size_t)NS * SBY);
    const uint32_t bar0 = s_base + (uint32_t)((size_t)NS * SBY + 2 * (size_t)SU * 32 * 8 * sizeof(float));
    auto bar_full = [&](int s) { return bar0 + 8u * s; };
    auto bar_empty = [&](int s) { return bar0 + 8u * (NS + s); };
    auto bar_red_full = [&](int b) { return bar0 + 8u * (2 * NS + b); };
    auto bar_red_free = [&](int b) { return bar0 + 8u * (2 * NS + 2 + b); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), SU);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_red_full(b), SU);
            mbar_init(bar_red_free(b), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();  // the weights are read once
            int s = 0;
            uint32_t ph = 0;
            const int tile0 = g_lo / SPT;
            int kb0 = (g_lo - tile0 * SPT) * SU;
            const uint8_t* src = P.packed + ((size_t)tile0 * KB + kb0) * bb;  // stages are contiguous
            for (int g = g_lo; g < g_hi; ++g) {
                if (!mbar_wait(bar_empty(s), ph ^ 1u)) {
                    atomicOr(p.status, 1u);
                    break;
                }
                const int cnt = min(SU, KB - kb0);
                const uint32_t bytes = (uint32_t)(cnt * bb);
                mbar_arrive_expect_tx(bar_full(s), bytes);
                bulk_g2s_hint(s_base + (uint32_t)(s * SBY), src, bytes, bar_full(s), policy);
                src += bytes;
                kb0 = (kb0 + cnt == KB) ? 0 : kb0 + SU;
                if (++s == NS) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int cw = warp - 1;  // block cw of every stage
    const int r = lane >> 2, t = lane & 3;
    const int sb_off = sb_offset(BITS, p.group, t, r);
    // Activation rows past M feed only output columns that are never stored,
    // so those lanes read row 0 instead of branching around the load.
    const uint16_t* x0 = p.x + (size_t)(r < p.M ? r : 0) * p.K + 32 * t;
    const uint16_t* x1 = p.x + (size_t)(r + 8 < p.M ? r + 8 : 0) * p.K + 32 * t;
    const bool ragged_k = (p.K % KBLK) != 0;  // only then can a lane's 32 k pass K

    constexpr int CH = dec_chains<MT>();
    float acc[CH][MT][4];
#pragma unroll
    for (int ch = 0; ch < CH; ++ch)
#pragma unroll
        for (int i = 0; i < MT; ++i) acc[ch][i][0] = acc[ch][i][1] = acc[ch][i][2] = acc[ch][i][3] = 0.f;
    float first_v[MT * 4];
    int first_tile = -1;
    int seg = 0;                 // tile segments finished by this CTA
    int seg_first_g = g_lo;      // first stage of the current segment
    bool failed = false;
    int s = 0;
    uint32_t ph = 0;
    int tile = g_lo / SPT;
    int kb0 = (g_lo - tile * SPT) * SU;
    for (int g = g_lo; g < g_hi; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar_full(s), ph))) {
            failed = true;
            break;
        }
        const int cnt = min(SU, KB - kb0);
        if (cw < cnt) {
            const uint32_t blk = s_base + (uint32_t)(s * SBY + cw * bb);
            uint32_t cw_words[2 * BITS];
            load_lane_codes_smem<BITS>(blk, lane, cw_words);
            uint2 sb;
            lds_v2(blk + sb_off, sb.x, sb.y);
            uint32_t xa[16], xb[16];
            const int kpos = (kb0 + cw) * KBLK;
            if (!ragged_k || kpos + 32 * t < p.K) {
                ld_x16(x0 + kpos, xa);
                if constexpr (MT == 2) ld_x16(x1 + kpos, xb);
            } else {  // depth padding: the weights there are zero, so are these
#pragma unroll
                for (int q = 0; q < 16; ++q) xa[q] = xb[q] = 0u;
            }
            block_contract<BITS, MT>(cw_words, sb, xa, xb, acc);
        }
        // this warp is done with the stage's shared memory
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty(s));

        const bool tile_end = kb0 + cnt == KB;
        const int cur_tile = tile;
        kb0 = tile_end ? 0 : kb0 + SU;
        tile += tile_end ? 1 : 0;
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
        if (!(tile_end || g == g_hi - 1)) continue;
        // ---- end of a tile segment: add the warps' sums in warp order
        const int b = seg & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar_red_free(b), (uint32_t)((seg >> 1) & 1) ^ 1u))) {
            failed = true;
            break;
        }
        float* rb = red + (size_t)b * SU * 32 * 8;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                rb[((size_t)cw * 8 + mt * 4 + q) * 32 + lane] =
                    CH == 4 ? (acc[0][mt][q] + acc[1][mt][q]) + (acc[CH > 2 ? 2 : 0][mt][q] + acc[CH - 1][mt][q])
                            : acc[0][mt][q] + acc[1][mt][q];
#pragma unroll
        for (int ch = 0; ch < CH; ++ch)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) acc[ch][mt][0] = acc[ch][mt][1] = acc[ch][mt][2] = acc[ch][mt][3] = 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_red_full(b));
        if (cw == 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_red_full(b), (uint32_t)((seg >> 1) & 1)))) {
                failed = true;
                break;
            }
            float v[MT * 4];
#pragma unroll
            for (int j = 0; j < MT * 4; ++j) {
                float sum = rb[(size_t)j * 32 + lane];
                for (int w = 1; w < SU; ++w) sum += rb[((size_t)w * 8 + j) * 32 + lane];
                v[j] = sum;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_red_free(b));
            const bool whole = (seg_first_g == cur_tile * SPT) && tile_end;
            if (whole) {
                store_y<MT>(P, p.M, cur_tile, r, t, v);
            } else if (seg_first_g == g_lo && g != g_hi - 1) {
                // the run's first segment ends mid-run: publish it after the
                // run so the stream never waits on a merge
#pragma unroll
                for (int j = 0; j < MT * 4; ++j) first_v[j] = v[j];
                first_tile = cur_tile;
            } else {
                publish_partial<MT>(p, P, c, cur_tile, seg_first_g == g_lo, lane, v);
            }
        }
        ++seg;
        seg_first_g = g + 1;
    }
    if (failed) {
        if (lane == 0) atomicOr(p.status, 1u);
        return;
    }
    if (cw == 0 && first_tile >= 0) publish_partial<MT>(p, P, c, first_tile, true, lane, first_v);
}

template <int BITS>
cudaError_t launch_bits(int mt, const DecParams& p, int grid, cudaStream_t st) {
    const size_t smem = decode_smem_bytes(p.ring, p.stage_bytes, p.su);
    const int threads = (p.su + 1) * 32;
    if (mt == 1)
        decode_kernel<BITS, 1><<<grid, threads, smem, st>>>(p);
    else
        decode_kernel<BITS, 2><<<grid, threads, smem, st>>>(p);
    return cudaGetLastError();
}

template <int BITS>
int occupancy_bits(int mt, int su, size_t smem) {
    int n = 0;
    const int threads = (su + 1) * 32;
    cudaError_t e = mt == 1 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, 1>, threads, smem)
                            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, 2>, threads, smem);
    return e == cudaSuccess ? n : -1;
}

template <int BITS>
cudaError_t allow_smem_bits(int bytes) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<BITS, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_kernel<BITS, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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

int decode_ctas_per_sm(int bits, int mt, int su, size_t smem) {
    switch (bits) {
        case 2: return occupancy_bits<2>(mt, su, smem);
        case 3: return occupancy_bits<3>(mt, su, smem);
        case 4: return occupancy_bits<4>(mt, su, smem);
        case 5: return occupancy_bits<5>(mt, su, smem);
        case 6: return occupancy_bits<6>(mt, su, smem);
        case 8: return occupancy_bits<8>(mt, su, smem);
        default: return -1;
    }
}

cudaError_t decode_allow_smem(int bytes) {
    for (cudaError_t e : {allow_smem_bits<2>(bytes), allow_smem_bits<3>(bytes), allow_smem_bits<4>(bytes),
                          allow_smem_bits<5>(bytes), allow_smem_bits<6>(bytes), allow_smem_bits<8>(bytes)})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace affqmm
