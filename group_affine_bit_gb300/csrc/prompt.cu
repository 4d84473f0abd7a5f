// prompt.cu -- the compute-bound projection for prompt chunks of up to 128
// activation rows, on the 5th-generation tensor cores (tcgen05, TMEM).
//
// One CTA per SM.  Its work is a contiguous run of (256-row tile, 128-deep
// block) units ("stream-K"), cut so every SM gets the same number of units.
// Per unit:
//   * a TMA warp loads the 128 x 128 activation tile (two 64-wide panels,
//     128-byte swizzle, rows past M and depth past K filled with zeros);
//   * eight dequantization warps read the unit's sixteen packed 16-row blocks
//     from HBM (one unit ahead, in registers), round every weight once as
//     bf16(fma(s, q, b)) -- the same device arithmetic as the decode kernel
//     -- and write them into shared memory in the tensor core's K-major,
//     128-byte-swizzled layout (prior art: the affine_mm prompt GEMM of the
//     "Gemma 4 12B on the native Metal engine" page, which dequantizes into
//     the threadgroup tile and lets the tensor unit accumulate over the whole
//     depth);
//   * one thread issues tcgen05.mma (kind::f16, M = 128 activation rows,
//     N = 256 weight rows, K = 16) accumulating in fp32 in TMEM, and commits
//     to the stage's "empty" barrier;
//   * at the end of a tile's segment four epilogue warps read TMEM with
//     tcgen05.ld and either store bf16 y (the whole tile was this CTA's) or
//     an fp32 partial that the last CTA to finish the tile adds up in k order
//     (an atomic counter per tile and 32-row quarter, no waiting).
// Two shared-memory stages of 96 KB (32 KB activations + 64 KB weights).
// Every mbarrier wait is bounded; a wait that gives up sets the workspace
// status word and a CTA-wide abort flag, and every role then finishes.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstddef>
#include <type_traits>

#include "affqmm_async.cuh"
#include "affqmm_format.cuh"
#include "affqmm_internal.h"

namespace affqmm {
namespace {

constexpr int P_THREADS = 14 * 32;   // TMA, MMA, 8 dequant, 4 epilogue warps
constexpr int P_DEQ_WARP0 = 2;
constexpr int P_EPI_WARP0 = 10;
constexpr int P_TILE_N = 256;        // weight rows per tile (MMA N)
constexpr int P_TILE_M = 128;        // activation rows (MMA M)
constexpr int P_STAGES = 2;
constexpr uint32_t P_A_BYTES = P_TILE_M * KBLK * 2;   // 32 KB
constexpr uint32_t P_B_BYTES = P_TILE_N * KBLK * 2;   // 64 KB
constexpr uint32_t P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr uint32_t P_A_PANEL = P_TILE_M * 128;         // one 64-deep panel
constexpr uint32_t P_B_PANEL = P_TILE_N * 128;
constexpr uint32_t P_TMEM_COLS = 256;

// instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major,
// N = 256, M = 128
constexpr uint32_t P_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(P_TILE_N >> 3) << 17) |
                             ((uint32_t)(P_TILE_M >> 4) << 24);

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// whose 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
           ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void sts_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel_p(unsigned* addr, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// A bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            atomicOr(status, 1u);
            return false;
        }
    }
    return true;
}

struct PromptSmem {
    uint64_t full_a[P_STAGES];
    uint64_t full_b[P_STAGES];
    uint64_t empty[P_STAGES];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint32_t tmem_base;
    int abort_flag;
};

template <int BITS>
__global__ void __launch_bounds__(P_THREADS, 1)
    prompt_kernel(const __grid_constant__ PromptParams p, const __grid_constant__ CUtensorMap xmap) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled panels
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    PromptSmem* sh = reinterpret_cast<PromptSmem*>(base_ptr + P_STAGES * P_STAGE_BYTES);
    const uint32_t sh_addr = base + P_STAGES * P_STAGE_BYTES;
    auto bar_full_a = [&](int s) { return sh_addr + (uint32_t)offsetof(PromptSmem, full_a) + 8u * s; };
    auto bar_full_b = [&](int s) { return sh_addr + (uint32_t)offsetof(PromptSmem, full_b) + 8u * s; };
    auto bar_empty = [&](int s) { return sh_addr + (uint32_t)offsetof(PromptSmem, empty) + 8u * s; };
    const uint32_t bar_acc_full = sh_addr + (uint32_t)offsetof(PromptSmem, acc_full);
    const uint32_t bar_acc_empty = sh_addr + (uint32_t)offsetof(PromptSmem, acc_empty);
    auto stage_a = [&](int s) { return base + (uint32_t)s * P_STAGE_BYTES; };
    auto stage_b = [&](int s) { return base + (uint32_t)s * P_STAGE_BYTES + P_A_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int pi = 0;
    for (int i = 1; i < p.nproj; ++i)
        if ((int)blockIdx.x >= p.proj[i].cta_begin) pi = i;
    const PromptProj& P = p.proj[pi];
    const int c = (int)blockIdx.x - P.cta_begin;
    const int U = P.units, PC = P.nctas, KB = p.KB;
    const int u0 = (int)((int64_t)c * U / PC);
    const int u1 = (int)((int64_t)(c + 1) * U / PC);

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(bar_full_a(s), 1);
            mbar_init(bar_full_b(s), 8);  // one arrival per dequantization warp
            mbar_init(bar_empty(s), 1);
        }
        mbar_init(bar_acc_full, 1);
        mbar_init(bar_acc_empty, 4);      // one arrival per epilogue warp
        sh->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {  // TMEM for the fp32 accumulator: 128 lanes x 256 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sh_addr + (uint32_t)offsetof(PromptSmem, tmem_base)),
                     "r"(P_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort_flag = &sh->abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
            for (int u = u0, i = 0; u < u1; ++u, ++i) {
                const int s = i % P_STAGES;
                const uint32_t ph = (uint32_t)((i / P_STAGES) & 1);
                if (!wait_or_abort(bar_empty(s), ph ^ 1u, abort_flag, p.status)) break;
                const int kb = u % KB;
                mbar_arrive_expect_tx(bar_full_a(s), P_A_BYTES);
                tma_load_2d(stage_a(s), &xmap, kb * KBLK, 0, bar_full_a(s));
                tma_load_2d(stage_a(s) + P_A_PANEL, &xmap, kb * KBLK + 64, 0, bar_full_a(s));
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int seg = 0;
            bool seg_open = false;
            for (int u = u0, i = 0; u < u1; ++u, ++i) {
                const int s = i % P_STAGES;
                const uint32_t ph = (uint32_t)((i / P_STAGES) & 1);
                const int kb = u % KB;
                const bool first = !seg_open;
                if (first) {  // the accumulator must have been drained
                    if (!wait_or_abort(bar_acc_empty, (uint32_t)(seg & 1) ^ 1u, abort_flag, p.status)) break;
                    tc_fence_after();
                    seg_open = true;
                }
                if (!wait_or_abort(bar_full_a(s), ph, abort_flag, p.status)) break;
                if (!wait_or_abort(bar_full_b(s), ph, abort_flag, p.status)) break;
                tc_fence_after();
#pragma unroll
                for (int pnl = 0; pnl < 2; ++pnl) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sw128_desc(stage_a(s) + pnl * P_A_PANEL + kk * 32);
                        const uint64_t bd = sw128_desc(stage_b(s) + pnl * P_B_PANEL + kk * 32);
                        umma_f16(tmem, ad, bd, P_IDESC, (first && pnl == 0 && kk == 0) ? 0u : 1u);
                    }
                }
                umma_commit(bar_empty(s));
                if (kb == KB - 1 || u == u1 - 1) {
                    umma_commit(bar_acc_full);
                    ++seg;
                    seg_open = false;
                }
            }
        }
    } else if (warp < P_EPI_WARP0) {
        // ---------------------------------------------------------- dequantization
        const int dw = warp - P_DEQ_WARP0;            // sub-tiles 2*dw, 2*dw + 1 of 16
        const int q = lane >> 3, j = lane & 7;        // conflict-free store order
        const int pl = 4 * j + q;                     // the packed lane this thread reads
        const int r = j, t = q;
        const int sb_off = sb_offset(BITS, p.group, t, r);
        const int bb = p.block_bytes;
        uint32_t cw[2][2][2 * BITS];
        uint2 sb[2][2];
        auto load_unit = [&](int u, auto bufc) {
            constexpr int buf = decltype(bufc)::value;
            const int tile = u / KB, kb = u % KB;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int st = tile * (P_TILE_N / TILE_N) + 2 * dw + h;
                if (st < P.tiles16) {
                    const uint8_t* blk = P.packed + ((size_t)st * KB + kb) * bb;
                    load_lane_codes<BITS>(blk, pl, cw[buf][h]);
                    uint32_t a, b2;
                    ld_stream_v2(blk + sb_off, a, b2);
                    sb[buf][h] = make_uint2(a, b2);
                } else {
#pragma unroll
                    for (int w = 0; w < 2 * BITS; ++w) cw[buf][h][w] = 0u;
                    sb[buf][h] = make_uint2(0u, 0u);
                }
            }
        };
        auto store_unit = [&](int s, auto bufc) {
            constexpr int buf = decltype(bufc)::value;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t sg = bcast_lo(sb[buf][h].x), bg = bcast_hi(sb[buf][h].x);
                const uint32_t sg8 = bcast_lo(sb[buf][h].y), bg8 = bcast_hi(sb[buf][h].y);
                uint32_t a[8][4];
                dequant_kstep<BITS, 0>(cw[buf][h], sg, bg, sg8, bg8, a[0]);
                dequant_kstep<BITS, 1>(cw[buf][h], sg, bg, sg8, bg8, a[1]);
                dequant_kstep<BITS, 2>(cw[buf][h], sg, bg, sg8, bg8, a[2]);
                dequant_kstep<BITS, 3>(cw[buf][h], sg, bg, sg8, bg8, a[3]);
                dequant_kstep<BITS, 4>(cw[buf][h], sg, bg, sg8, bg8, a[4]);
                dequant_kstep<BITS, 5>(cw[buf][h], sg, bg, sg8, bg8, a[5]);
                dequant_kstep<BITS, 6>(cw[buf][h], sg, bg, sg8, bg8, a[6]);
                dequant_kstep<BITS, 7>(cw[buf][h], sg, bg, sg8, bg8, a[7]);
                const int n0 = 16 * (2 * dw + h) + r;  // row r of the sub-tile; row r + 8 is n0 + 8
                const uint32_t pbase = stage_b(s) + (uint32_t)(t >> 1) * P_B_PANEL;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t chunk = (uint32_t)((4 * (t & 1) + i) ^ r) << 4;
                    sts_v4(pbase + (uint32_t)(n0 >> 3) * 1024u + (uint32_t)r * 128u + chunk, a[2 * i][0],
                           a[2 * i][2], a[2 * i + 1][0], a[2 * i + 1][2]);
                    sts_v4(pbase + (uint32_t)((n0 + 8) >> 3) * 1024u + (uint32_t)r * 128u + chunk, a[2 * i][1],
                           a[2 * i][3], a[2 * i + 1][1], a[2 * i + 1][3]);
                }
            }
        };
        using B0 = std::integral_constant<int, 0>;
        using B1 = std::integral_constant<int, 1>;
        if (u0 < u1) load_unit(u0, B0{});
        for (int u = u0, i = 0; u < u1; ++u, ++i) {
            const int s = i % P_STAGES;
            const uint32_t ph = (uint32_t)((i / P_STAGES) & 1);
            const bool even = (i & 1) == 0;
            if (u + 1 < u1) {  // next unit's codes in flight while this one is dequantized
                if (even) load_unit(u + 1, B1{});
                else load_unit(u + 1, B0{});
            }
            if (!__all_sync(0xffffffffu, wait_or_abort(bar_empty(s), ph ^ 1u, abort_flag, p.status))) break;
            if (even) store_unit(s, B0{});
            else store_unit(s, B1{});
            fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_full_b(s));
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int m = 32 * quarter + lane;       // activation row of this thread
        const int M = p.M;
        int seg = 0;
        int seg_start = u0;
        for (int u = u0; u < u1; ++u) {
            const int kb = u % KB;
            if (!(kb == KB - 1 || u == u1 - 1)) continue;
            const int tile = u / KB;
            const bool whole = (seg_start == tile * KB) && (kb == KB - 1);
            if (!__all_sync(0xffffffffu, wait_or_abort(bar_acc_full, (uint32_t)(seg & 1), abort_flag, p.status))) break;
            tc_fence_after();
            const int64_t n_base = (int64_t)tile * P_TILE_N;
            const int slot = P.slot_begin + 2 * c + (seg_start == u0 ? 0 : 1);
            float* srow = p.slots + (size_t)slot * (P_TILE_M * P_TILE_N) + (size_t)m * P_TILE_N;
#pragma unroll 1
            for (int cc = 0; cc < P_TILE_N / 32; ++cc) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(32 * cc), v);
                if (whole) {
                    if (m < M) {
                        for (int e = 0; e < 32; ++e) {
                            const int64_t n = n_base + 32 * cc + e;
                            if (n < P.N) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[e]));
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        __stcg(reinterpret_cast<float4*>(srow + 32 * cc + e), make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]));
                }
            }
            // accumulator drained: the MMA warp may start the next segment
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_empty);
            if (!whole) {
                // Publish this warp's 32 rows of the partial; the last CTA to
                // arrive (per tile and row quarter) adds them in k order.
                __syncwarp();
                unsigned prev = 0;
                unsigned* ctr = &p.counters[(size_t)(P.ctr_begin + tile) * 4 + quarter];
                if (lane == 0) prev = atom_add_acq_rel_p(ctr, 1u);
                __syncwarp();
                prev = __shfl_sync(0xffffffffu, prev, 0);
                const int t0 = tile * KB, t1 = t0 + KB - 1;
                const int cf = (int)(((int64_t)(t0 + 1) * PC - 1) / U);
                const int cl = (int)(((int64_t)(t1 + 1) * PC - 1) / U);
                if (prev == (unsigned)(cl - cf)) {
#pragma unroll 1
                    for (int cc = 0; cc < P_TILE_N / 32; ++cc) {
                        float acc[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[e] = 0.f;
                        for (int cb = cf; cb <= cl; ++cb) {
                            const int bcb = (int)((int64_t)cb * U / PC);
                            const int sc = P.slot_begin + 2 * cb + (bcb >= t0 ? 0 : 1);
                            const float* row = p.slots + (size_t)sc * (P_TILE_M * P_TILE_N) + (size_t)m * P_TILE_N + 32 * cc;
#pragma unroll
                            for (int e = 0; e < 32; e += 4) {
                                const float4 f = __ldcg(reinterpret_cast<const float4*>(row + e));
                                acc[e] += f.x;
                                acc[e + 1] += f.y;
                                acc[e + 2] += f.z;
                                acc[e + 3] += f.w;
                            }
                        }
                        if (m < M) {
                            for (int e = 0; e < 32; ++e) {
                                const int64_t n = n_base + 32 * cc + e;
                                if (n < P.N) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[e]));
                            }
                        }
                    }
                    if (lane == 0) *ctr = 0u;
                }
            }
            ++seg;
            seg_start = u + 1;
        }
    }

    // teardown: every role has left its loop
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P_TMEM_COLS)
                     : "memory");
    }
}

template <int BITS>
cudaError_t launch_prompt_bits(const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    prompt_kernel<BITS><<<grid, P_THREADS, prompt_smem_bytes(), st>>>(p, map);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t allow_prompt_bits() {
    return cudaFuncSetAttribute(prompt_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)prompt_smem_bytes());
}

}  // namespace

size_t prompt_smem_bytes() { return (size_t)P_STAGES * P_STAGE_BYTES + sizeof(PromptSmem) + 1024; }

cudaError_t prompt_allow_smem() {
    for (cudaError_t e : {allow_prompt_bits<2>(), allow_prompt_bits<3>(), allow_prompt_bits<4>(),
                          allow_prompt_bits<5>(), allow_prompt_bits<6>(), allow_prompt_bits<8>()})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_prompt(int bits, const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    switch (bits) {
        case 2: return launch_prompt_bits<2>(p, map, grid, st);
        case 3: return launch_prompt_bits<3>(p, map, grid, st);
        case 4: return launch_prompt_bits<4>(p, map, grid, st);
        case 5: return launch_prompt_bits<5>(p, map, grid, st);
        case 6: return launch_prompt_bits<6>(p, map, grid, st);
        case 8: return launch_prompt_bits<8>(p, map, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace affqmm
