// prompt.cu -- the compute-bound projection for prompt chunks of up to 128
// activation rows, on the 5th-generation tensor cores (tcgen05, TMEM).
//
// One CTA per SM.  Its work is a contiguous run of (256-row tile, 128-deep
// block) units ("stream-K"), cut so every SM gets the same number of units.
// Per unit:
//   * a TMA warp loads the 128 x 128 activation tile (two 64-wide panels,
//     128-byte swizzle, rows past M and depth past K filled with zeros);
//   * eight dequantization warps, one thread per weight row, read the row's
//     codes of the unit's two packed 128-row blocks from HBM (one unit
//     ahead, in registers), round every weight once as
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
#include "affqmm_tc.cuh"

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

constexpr uint32_t P_IDESC = idesc_bf16_f32(P_TILE_M, P_TILE_N);

__device__ __forceinline__ void sts_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// The 16 chunks (8 weights each) of one dequantized row into the 128-byte-
// swizzled K-major layout: chunk c holds k = 8c .. 8c + 7, lives in panel
// c / 8 at 16-byte position (c mod 8) xor (row mod 8) of the row's 128 bytes.
template <int BITS, int GROUP, int C>
__device__ __forceinline__ void store_chunks(const uint32_t* cw, const uint32_t* sbw, uint32_t rowbase, int r8) {
    if constexpr (C < KBLK / 8) {
        uint32_t w[4];
        weight_pairs<BITS, GROUP, 4 * C, 4>(cw, sbw, w);
        sts_v4(rowbase + (uint32_t)(C >> 3) * P_B_PANEL + ((uint32_t)((C & 7) ^ r8) << 4), w[0], w[1], w[2], w[3]);
        store_chunks<BITS, GROUP, C + 1>(cw, sbw, rowbase, r8);
    }
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

template <int BITS, int GROUP>
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
    if (warp == 1)  // TMEM for the fp32 accumulator: 128 lanes x 256 columns
        tmem_alloc(sh_addr + (uint32_t)offsetof(PromptSmem, tmem_base), P_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort_flag = &sh->abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&xmap);
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
                        umma_ss(tmem, ad, bd, P_IDESC, (first && pnl == 0 && kk == 0) ? 0u : 1u);
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
        // thread = weight row n of the 256-row tile (two 128-row layout tiles)
        const int n = 32 * (warp - P_DEQ_WARP0) + lane;
        const int sub = n >> 7, nn = n & 127;
        constexpr int BB = block_bytes(BITS, GROUP);
        uint32_t cw[2][4 * BITS];
        uint32_t sbw[2][sb_words(GROUP)];
        auto load_unit = [&](int u, auto bufc) {
            constexpr int buf = decltype(bufc)::value;
            const int tile = u / KB, kb = u % KB;
            const int lt = 2 * tile + sub;  // layout tile of this row
            if (lt < P.ltiles) {
                const uint8_t* blk = P.packed + ((size_t)lt * KB + kb) * BB;
                load_row_codes<BITS>(blk, nn, cw[buf]);
                load_row_sb<GROUP>(blk + sb_offset(BITS, GROUP, nn), sbw[buf]);
            } else {  // rows past the last tile: zero weights
#pragma unroll
                for (int w = 0; w < 4 * BITS; ++w) cw[buf][w] = 0u;
#pragma unroll
                for (int w = 0; w < sb_words(GROUP); ++w) sbw[buf][w] = 0u;
            }
        };
        auto store_unit = [&](int s, auto bufc) {
            constexpr int buf = decltype(bufc)::value;
            const uint32_t rowbase = stage_b(s) + (uint32_t)(n >> 3) * 1024u + (uint32_t)(n & 7) * 128u;
            store_chunks<BITS, GROUP, 0>(cw[buf], sbw[buf], rowbase, n & 7);
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
                uint32_t vr[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(32 * cc), vr);
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(vr[e]);
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
                if (lane == 0) prev = atom_add_acq_rel(ctr, 1u);
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
        tmem_dealloc(tmem, P_TMEM_COLS);
    }
}

template <int BITS, int GROUP>
cudaError_t launch_prompt_bg(const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    prompt_kernel<BITS, GROUP><<<grid, P_THREADS, prompt_smem_bytes(), st>>>(p, map);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_prompt_b(const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    if (p.group == 32) return launch_prompt_bg<BITS, 32>(p, map, grid, st);
    if (p.group == 64) return launch_prompt_bg<BITS, 64>(p, map, grid, st);
    return launch_prompt_bg<BITS, 128>(p, map, grid, st);
}

template <int BITS>
cudaError_t allow_prompt_b() {
    for (cudaError_t e : {cudaFuncSetAttribute(prompt_kernel<BITS, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)prompt_smem_bytes()),
                          cudaFuncSetAttribute(prompt_kernel<BITS, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)prompt_smem_bytes()),
                          cudaFuncSetAttribute(prompt_kernel<BITS, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)prompt_smem_bytes())})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

size_t prompt_smem_bytes() { return (size_t)P_STAGES * P_STAGE_BYTES + sizeof(PromptSmem) + 1024; }

cudaError_t prompt_allow_smem() {
    for (cudaError_t e : {allow_prompt_b<2>(), allow_prompt_b<3>(), allow_prompt_b<4>(), allow_prompt_b<5>(),
                          allow_prompt_b<6>(), allow_prompt_b<8>()})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_prompt(int bits, const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    switch (bits) {
        case 2: return launch_prompt_b<2>(p, map, grid, st);
        case 3: return launch_prompt_b<3>(p, map, grid, st);
        case 4: return launch_prompt_b<4>(p, map, grid, st);
        case 5: return launch_prompt_b<5>(p, map, grid, st);
        case 6: return launch_prompt_b<6>(p, map, grid, st);
        case 8: return launch_prompt_b<8>(p, map, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace affqmm
