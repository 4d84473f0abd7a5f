// decode.cu -- the memory-bound projection for M = 1..16 activation rows.
//
// The weight blocks of one projection (16 rows x 128 k each, stored tile-major)
// are cut into contiguous runs, one run per warp, with all of the device's
// resident warps busy ("stream-K" at warp granularity).  A warp streams its
// run's blocks from HBM into its own ring of shared-memory stages with 1-D
// bulk copies (TMA, one mbarrier per stage, every wait bounded), keeping up
// to `stages` blocks in flight; each lane reads its fragment words back from
// shared memory, dequantizes every weight once as
// bf16(fma(s, q, b)) (affqmm_format.cuh) and contracts on the tensor cores
// with mma.sync m16n8k16 (bf16 in, fp32 accumulate): the weights are the A
// operand (16 rows x 16 k), the activation rows the B operand (8 rows, or two
// MMAs for 9..16 rows).  Prior art: the "reg variant" lane projection of the
// "Gemma 4 12B on the native Metal engine" page (4-bit groups in tensor-op
// registers, K split per shape); unlike it, the weights here are rounded to
// bf16 before the contraction, as the same page's prompt GEMM does.
//
// Reduction order is fixed: a tile whose blocks all fall in one warp's run is
// summed in k order and stored directly; a tile cut by run boundaries gets one
// fp32 partial per run, and the last of those warps to arrive (an atomic
// counter, no waiting) adds the partials in run order, converts to bf16 and
// re-zeroes the counter.  The runs depend only on the projection, M and the
// device, so the same inputs give the same bits on every call, alone or
// stacked with other projections.
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

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* addr, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// The warp whose run holds unit u: the largest w with floor(w*U/PW) <= u.
__device__ __forceinline__ int warp_of(int u, int U, int PW) {
    return (int)(((int64_t)(u + 1) * PW - 1) / U);
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

// Publish a partial segment [seg_start, seg_end] of tile `tile` from this
// warp's run [u0, u1): store its fp32 sums in the warp's slot, count it on the
// tile's counter, and if it is the last of the tile's segments to arrive, add
// all of them in run (k) order, store y and re-zero what it used.
template <int MT>
__device__ __forceinline__ void publish_partial(const DecParams& p, const DecProj& P, int w, int u0, int tile,
                                                int seg_start, int lane, const float* v_in) {
    const int r = lane >> 2, t = lane & 3;
    const int KB = p.KB;
    const int t0 = tile * KB, t1 = t0 + KB - 1;
    const int U = P.units, PW = P.nwarps;
    const int slot = P.slot_begin + 2 * w + (seg_start == u0 ? 0 : 1);
    float* sp = p.partials + (size_t)slot * 256 + lane * 8;
#pragma unroll
    for (int j = 0; j < MT * 4; ++j) __stcg(sp + j, v_in[j]);
    // The warp's partial is published by lane 0's release (ordered after the
    // other lanes' stores by __syncwarp); the acquire side of the same atomic
    // makes every earlier partial visible to the last warp to arrive.
    __syncwarp();
    unsigned prev = 0;
    if (lane == 0) prev = atom_add_acq_rel(&p.counters[P.ctr_begin + tile], 1u);
    __syncwarp();
    prev = __shfl_sync(0xffffffffu, prev, 0);
    const int wf = warp_of(t0, U, PW), wl = warp_of(t1, U, PW);
    if (prev != (unsigned)(wl - wf)) return;
    float v[MT * 4];
#pragma unroll
    for (int j = 0; j < MT * 4; ++j) v[j] = 0.f;
    for (int c = wf; c <= wl; ++c) {
        const int bc = (int)((int64_t)c * U / PW);
        const int sc = P.slot_begin + 2 * c + (bc >= t0 ? 0 : 1);
        const float* cp = p.partials + (size_t)sc * 256 + lane * 8;
#pragma unroll
        for (int j = 0; j < MT * 4; ++j) v[j] += __ldcg(cp + j);
    }
    store_y<MT>(P, p.M, tile, r, t, v);
    if (lane == 0) p.counters[P.ctr_begin + tile] = 0u;
}

template <int BITS, int MT>
__global__ void __launch_bounds__(DEC_WARPS * 32) decode_kernel(const __grid_constant__ DecParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int r = lane >> 2, t = lane & 3;
    const int gw = (int)blockIdx.x * DEC_WARPS + wid;
    if (gw >= p.total_warps) return;
    int pi = 0;
    for (int i = 1; i < p.nproj; ++i)
        if (gw >= p.proj[i].warp_begin) pi = i;
    const DecProj& P = p.proj[pi];
    const int w = gw - P.warp_begin;
    const int U = P.units, PW = P.nwarps;
    const int u0 = (int)((int64_t)w * U / PW);
    const int u1 = (int)((int64_t)(w + 1) * U / PW);
    const int n = u1 - u0;
    const int KB = p.KB;
    const int bb = p.block_bytes;
    const int NS = p.stages, SBY = p.stage_bytes;
    const uint8_t* base = P.packed;
    const int sb_off = sb_offset(BITS, p.group, t, r);
    const bool row0 = r < p.M;
    const bool row1 = (MT == 2) && (r + 8 < p.M);
    const uint16_t* x0 = p.x + (size_t)r * p.K + 32 * t;
    const uint16_t* x1 = p.x + (size_t)(r + 8) * p.K + 32 * t;

    // This warp's ring: NS stages of SBY bytes, then NS mbarriers.
    const uint32_t ring = smem_u32(smem) + (uint32_t)(wid * NS * SBY);
    const uint32_t bars = smem_u32(smem) + (uint32_t)(DEC_WARPS * NS * SBY + wid * NS * 8);
    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t policy = policy_evict_first();  // weights are read once
    auto issue = [&](int j) {                       // unit u0 + j into stage j % NS
        const int s = j % NS;
        mbar_arrive_expect_tx(bars + 8 * s, (uint32_t)bb);
        bulk_g2s_hint(ring + (uint32_t)(s * SBY), base + (size_t)(u0 + j) * bb, (uint32_t)bb, bars + 8 * s, policy);
    };
    if (lane == 0)
        for (int j = 0; j < NS && j < n; ++j) issue(j);

    float acc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    int tile = u0 / KB;
    int kb = u0 - tile * KB;
    int seg_start = u0;
    int stage = 0;
    uint32_t parity = 0;
    int j = 0;
    // partial segments of this run, published after it
    float first_v[MT * 4], last_v[MT * 4];
    int first_tile = -1, last_tile = -1, last_start = 0;
    for (; j < n; ++j) {
        const int u = u0 + j;
        const bool ok = mbar_wait(bars + 8 * stage, parity);
        if (!__all_sync(0xffffffffu, ok)) break;
        uint32_t cw[2 * BITS];
        const uint32_t blk = ring + (uint32_t)(stage * SBY);
        load_lane_codes_smem<BITS>(blk, lane, cw);
        uint2 sb;
        lds_v2(blk + sb_off, sb.x, sb.y);
        uint32_t xa[16], xb[16];
        const int64_t kpos = (int64_t)kb * KBLK;
        const bool kin = kpos + 32 * t < p.K;
        if (row0 && kin) {
            ld_x16(x0 + kpos, xa);
        } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) xa[q] = 0u;
        }
        if constexpr (MT == 2) {
            if (row1 && kin) {
                ld_x16(x1 + kpos, xb);
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) xb[q] = 0u;
            }
        }
        // every lane has its words in registers: refill this stage NS units ahead
        __syncwarp();
        if (lane == 0 && j + NS < n) {
            fence_proxy_async_smem();
            issue(j + NS);
        }
        block_contract<BITS, MT>(cw, sb, xa, xb, acc);
        if (kb == KB - 1 || u == u1 - 1) {
            float v[MT * 4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) v[mt * 4 + i] = acc[mt][i];
            if (seg_start == tile * KB && kb == KB - 1) {
                store_y<MT>(P, p.M, tile, r, t, v);  // the whole tile was ours
            } else if (seg_start == u0 && u != u1 - 1) {
                // the run's first segment ends mid-run: keep it in registers and
                // publish it after the run, so the stream never stalls on a merge
#pragma unroll
                for (int q = 0; q < MT * 4; ++q) first_v[q] = v[q];
                first_tile = tile;
            } else {
                last_tile = tile;
                last_start = seg_start;
#pragma unroll
                for (int q = 0; q < MT * 4; ++q) last_v[q] = v[q];
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
            seg_start = u + 1;
        }
        if (++kb == KB) {
            kb = 0;
            ++tile;
        }
        if (++stage == NS) {
            stage = 0;
            parity ^= 1u;
        }
    }
    if (j == n) {
        if (first_tile >= 0) publish_partial<MT>(p, P, w, u0, first_tile, u0, lane, first_v);
        if (last_tile >= 0) publish_partial<MT>(p, P, w, u0, last_tile, last_start, lane, last_v);
    } else {
        // A bounded wait gave up: record it and let the copies still in flight
        // land (again bounded) before this CTA's shared memory is released.
        if (lane == 0) {
            atomicOr(p.status, 1u);
            for (int q = j; q < n && q < j + NS; ++q) {
                const int s = q % NS;
                (void)mbar_wait(bars + 8 * s, (uint32_t)((q / NS) & 1));
            }
        }
        __syncwarp();
    }
}

template <int BITS>
cudaError_t launch_bits(int mt, const DecParams& p, int grid, cudaStream_t st) {
    const size_t smem = decode_smem_bytes(p.stages, p.stage_bytes);
    if (mt == 1)
        decode_kernel<BITS, 1><<<grid, DEC_WARPS * 32, smem, st>>>(p);
    else
        decode_kernel<BITS, 2><<<grid, DEC_WARPS * 32, smem, st>>>(p);
    return cudaGetLastError();
}

template <int BITS>
int occupancy_bits(int mt, size_t smem) {
    int n = 0;
    cudaError_t e = mt == 1 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, 1>, DEC_WARPS * 32, smem)
                            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, 2>, DEC_WARPS * 32, smem);
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

int decode_ctas_per_sm(int bits, int mt, size_t smem) {
    switch (bits) {
        case 2: return occupancy_bits<2>(mt, smem);
        case 3: return occupancy_bits<3>(mt, smem);
        case 4: return occupancy_bits<4>(mt, smem);
        case 5: return occupancy_bits<5>(mt, smem);
        case 6: return occupancy_bits<6>(mt, smem);
        case 8: return occupancy_bits<8>(mt, smem);
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
