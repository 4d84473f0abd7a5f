// prompt.cu -- the compute-bound projection for prompt chunks of 17..128
// activation rows, on the 5th-generation tensor cores (tcgen05, TMEM).
//
// The weights are the A operand and live in tensor memory; the activations
// are the B operand in shared memory.  One CTA per SM works on a contiguous
// run of units (an even cut of all units, "stream-K", or a whole number of
// runs per tile: the launch planner's choice, plan.cu); a unit is a 256-row
// tile pair (two 128-row layout tiles) x one 128-deep block.  Per unit:
//   * one producer thread copies the unit's 128 x 128 activation tile (TMA,
//     two 64-wide panels, 128-byte swizzle, rows past M and depth past K read
//     as zero) into a ring of activation stages, another the two packed
//     weight blocks (one bulk copy each, about 9 KB at 4 bits) into a deeper
//     ring of weight stages;
//   * two dequantization groups of four warps -- one per 128-row layout
//     tile, one thread per weight row -- read their row's codes back, round
//     every weight once as bf16(fma(s, q, b)) (affqmm_format.cuh, the same
//     device arithmetic as the decode kernel) and store the row into a
//     tensor-memory A buffer with tcgen05.st.  Units alternate between two
//     such pairs of groups, each with its own A buffers, so one unit is
//     dequantized while the MMAs of the previous one run;
//   * two threads (one per layout tile) issue the unit's MMAs (M = 128
//     weight rows, N = activation rows rounded up to 16, K = 16), each into
//     its own fp32 accumulator in tensor memory over the tile's whole depth
//     (one issuing thread cannot keep the tensor pipe busy at these sizes);
//   * at the end of a tile's segment four epilogue warps read the two
//     accumulators with tcgen05.ld and store bf16 y, or, when several runs
//     share the tile, an fp32 partial; a second, small kernel then adds each
//     shared tile's partials in run (k) order, every output in parallel.
// Prior art: the affine_mm prompt GEMM of the "Gemma 4 12B on the native
// Metal engine" page, which dequantizes each weight as bf16(fma(scale, code,
// bias)) into the tile and lets the tensor unit accumulate over the whole
// depth; on GB300 the dequantized tile goes to tensor memory, which keeps
// the shared-memory traffic to the activations and the packed codes.
// Every mbarrier wait is bounded; a wait that gives up sets the workspace
// status word and a CTA-wide abort flag, and every role then finishes.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstddef>

#include "affqmm_async.cuh"
#include "affqmm_format.cuh"
#include "affqmm_internal.h"
#include "affqmm_tc.cuh"

namespace affqmm {
namespace {

constexpr int P_DEQ_GROUPS = 4;                                  // (layout tile, unit parity)
constexpr int P_DEQ_WARP0 = 3;                                   // warp 0: weights producer, 1-2: MMA issuers
constexpr int P_EPI_WARP0 = P_DEQ_WARP0 + 4 * P_DEQ_GROUPS;      // 19
constexpr int P_XPROD = P_EPI_WARP0 + 4;                         // 23: activations producer
constexpr int P_THREADS = (P_XPROD + 1) * 32;                    // 768
constexpr int P_TILE_N = 256;                                    // weight rows per unit
constexpr int P_ROWS = 128;                                      // activation rows per launch (max)
constexpr uint32_t P_X_PANEL = P_ROWS * 128;                     // 128 rows x 64 k bf16, 16 KB
constexpr uint32_t P_X_BYTES = 2 * P_X_PANEL;                    // one 128-deep block of x
constexpr uint32_t P_TMEM_COLS = 512;
constexpr uint32_t P_ACC_COLS = 128;                             // fp32 accumulator per layout tile
constexpr uint32_t P_A_COL0 = 2 * P_ACC_COLS;                    // A buffers after the two accumulators
constexpr uint32_t P_A_COLS = KBLK / 2;                          // 128 bf16 per row
constexpr int P_RING_MAX = 8;

struct PromptSmem {
    uint64_t xfull[P_RING_MAX];
    uint64_t xempty[P_RING_MAX];
    uint64_t wfull[P_RING_MAX];
    uint64_t wempty[P_RING_MAX];
    uint64_t a_full[P_DEQ_GROUPS];
    uint64_t a_empty[P_DEQ_GROUPS];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint32_t tmem_base;
    int abort_flag;
};

// Two rings in shared memory: activation blocks (32 KB each, 1024-byte
// aligned for the swizzle; held until the unit's MMAs are done) and packed
// weight blocks (the unit's two blocks; held only until the dequantization
// warps have read them, so that ring runs further ahead of the HBM latency).
// The weight ring has an even depth: its stage s always serves units of
// parity s mod 2, whose dequantization groups are the only readers.
constexpr uint32_t kPromptSmemBudget = 210u * 1024u;
template <int BITS, int GROUP>
constexpr uint32_t prm_wstage() {
    return 2u * (uint32_t)block_bytes(BITS, GROUP);
}
template <int BITS, int GROUP>
constexpr int prm_wring_for(int nx) {
    return (int)((kPromptSmemBudget - (uint32_t)nx * P_X_BYTES) / prm_wstage<BITS, GROUP>()) / 2 * 2 > P_RING_MAX
               ? P_RING_MAX
               : (int)((kPromptSmemBudget - (uint32_t)nx * P_X_BYTES) / prm_wstage<BITS, GROUP>()) / 2 * 2;
}
template <int BITS, int GROUP>
constexpr int prm_xring() {  // activations come from L2 but wait for the MMAs: as deep as leaves 2 weight stages
    return prm_wring_for<BITS, GROUP>(4) >= 2 ? 4 : prm_wring_for<BITS, GROUP>(3) >= 2 ? 3 : 2;
}
template <int BITS, int GROUP>
constexpr int prm_wring() {
    return prm_wring_for<BITS, GROUP>(prm_xring<BITS, GROUP>());
}
template <int BITS, int GROUP>
constexpr size_t prm_ring_bytes() {
    return (size_t)prm_xring<BITS, GROUP>() * P_X_BYTES + (size_t)prm_wring<BITS, GROUP>() * prm_wstage<BITS, GROUP>();
}

template <int BITS, int GROUP>
__global__ void __launch_bounds__(P_THREADS, 1)
    prompt_kernel(const __grid_constant__ PromptParams p, const __grid_constant__ CUtensorMap xmap) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int BB = block_bytes(BITS, GROUP);
    constexpr int NX = prm_xring<BITS, GROUP>();
    constexpr int NW = prm_wring<BITS, GROUP>();
    constexpr uint32_t WSTAGE = prm_wstage<BITS, GROUP>();
    static_assert(NX >= 2 && NW >= 2 && NW % 2 == 0, "ring depths");
    static_assert(BB % 16 == 0, "bulk copies move multiples of 16 bytes");
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;        // activation ring
    const uint32_t wbase = base + (uint32_t)NX * P_X_BYTES;  // weight ring
    PromptSmem* sh = reinterpret_cast<PromptSmem*>(smem_raw + (base - raw) + prm_ring_bytes<BITS, GROUP>());
    const uint32_t sh_addr = base + (uint32_t)prm_ring_bytes<BITS, GROUP>();
#define BAR(field, i) (sh_addr + (uint32_t)offsetof(PromptSmem, field) + 8u * (uint32_t)(i))
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
        for (int s = 0; s < NX; ++s) {
            mbar_init(BAR(xfull, s), 1);
            mbar_init(BAR(xempty, s), 2);  // the two issuers' MMAs read the activations
        }
        for (int s = 0; s < NW; ++s) {
            mbar_init(BAR(wfull, s), 1);
            mbar_init(BAR(wempty, s), 8);  // the 8 dequantization warps of the unit read the packed blocks
        }
        for (int g = 0; g < P_DEQ_GROUPS; ++g) {
            mbar_init(BAR(a_full, g), 4);
            mbar_init(BAR(a_empty, g), 1);
        }
        mbar_init(BAR(acc_full, 0), 2);   // both issuers commit at every segment end
        mbar_init(BAR(acc_empty, 0), 4);  // one arrival per epilogue warp
        sh->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(sh_addr + (uint32_t)offsetof(PromptSmem, tmem_base), P_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort_flag = &sh->abort_flag;
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (warp == 0) {
        // ---------------------------------------------------------- weights producer
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();  // the weights are read once
            for (int u = u0, i = 0; u < u1; ++u, ++i) {
                const int s = i % NW;
                const uint32_t ph = (uint32_t)((i / NW) & 1);
                if (!wait_or_abort_lazy(BAR(wempty, s), ph ^ 1u, abort_flag, p.status)) break;
                const int tile = u / KB, kb = u - (u / KB) * KB;
                const int lt0 = 2 * tile;
                const bool two = lt0 + 1 < P.ltiles;
                const uint32_t st = wbase + (uint32_t)s * WSTAGE;
                mbar_arrive_expect_tx(BAR(wfull, s), (two ? 2u : 1u) * (uint32_t)BB);
                bulk_g2s_hint(st, P.packed + ((size_t)lt0 * KB + kb) * BB, (uint32_t)BB, BAR(wfull, s), policy);
                if (two)
                    bulk_g2s_hint(st + (uint32_t)BB, P.packed + ((size_t)(lt0 + 1) * KB + kb) * BB, (uint32_t)BB,
                                  BAR(wfull, s), policy);
            }
        }
    } else if (warp == P_XPROD) {
        // ---------------------------------------------------------- activations producer
        if (lane == 0) {
            prefetch_tmap(&xmap);
            pdl_wait();  // x may come from the previous kernel
            int kb = u0 % KB;
            for (int u = u0, i = 0; u < u1; ++u, ++i) {
                const int s = i % NX;
                const uint32_t ph = (uint32_t)((i / NX) & 1);
                if (!wait_or_abort_lazy(BAR(xempty, s), ph ^ 1u, abort_flag, p.status)) break;
                const uint32_t st = base + (uint32_t)s * P_X_BYTES;
                mbar_arrive_expect_tx(BAR(xfull, s), P_X_BYTES);
                tma_load_2d(st, &xmap, kb * KBLK, 0, BAR(xfull, s));
                tma_load_2d(st + P_X_PANEL, &xmap, kb * KBLK + 64, 0, BAR(xfull, s));
                if (++kb == KB) kb = 0;
            }
        }
    } else if (warp < P_DEQ_WARP0) {
        // ---------------------------------------------------------- MMA issuers
        // issuer `sub` accumulates layout tile `sub` of every unit (one
        // issuing thread per accumulator keeps the fp32 order fixed)
        if (lane == 0) {
            const int sub = warp - 1;
            const int nn = p.M <= 16 ? 16 : (p.M + 15) / 16 * 16;  // MMA N: activation rows
            const uint32_t idesc = idesc_bf16_f32(128, nn);
            int seg = 0;
            bool open = false, first = false;
            int kb = u0 % KB;
            for (int u = u0, i = 0; u < u1; ++u, ++i) {
                if (!open) {  // both accumulators must have been drained
                    if (!wait_or_abort(BAR(acc_empty, 0), (uint32_t)(seg & 1) ^ 1u, abort_flag, p.status)) break;
                    tc_fence_after();
                    open = first = true;
                }
                const int s = i % NX;
                const uint32_t ph = (uint32_t)((i / NX) & 1);
                const int par = i & 1;
                const uint32_t aph = (uint32_t)((i >> 1) & 1);
                if (!wait_or_abort(BAR(xfull, s), ph, abort_flag, p.status)) break;
                if (!wait_or_abort(BAR(a_full, 2 * sub + par), aph, abort_flag, p.status)) break;
                tc_fence_after();
                const uint64_t bd0 = sw128_desc(base + (uint32_t)s * P_X_BYTES);
                const uint32_t dcol = tmem + (uint32_t)sub * P_ACC_COLS;
                const uint32_t acol = tmem + P_A_COL0 + (uint32_t)(2 * sub + par) * P_A_COLS;
#pragma unroll
                for (int k = 0; k < KBLK / 16; ++k) {
                    // +32 bytes per 16-deep step, +16 KB per 64-deep panel (descriptor units of 16 bytes)
                    const uint64_t bd = bd0 + (uint64_t)((k >> 2) * (P_X_PANEL >> 4) + (k & 3) * 2);
                    umma_ts(dcol, acol + 8u * k, bd, idesc, (first && k == 0) ? 0u : 1u);
                }
                first = false;
                umma_commit(BAR(a_empty, 2 * sub + par));
                umma_commit(BAR(xempty, s));
                if (kb == KB - 1 || u == u1 - 1) {
                    umma_commit(BAR(acc_full, 0));
                    ++seg;
                    open = false;
                }
                if (++kb == KB) kb = 0;
            }
        }
    } else if (warp < P_EPI_WARP0) {
        // ---------------------------------------------------------- dequantization
        // group g: layout tile `sub` of the units of parity `par`; thread =
        // weight row 32q + lane of that layout tile (TMEM lane quarter q)
        const int g = (warp - P_DEQ_WARP0) >> 2;
        const int sub = g >> 1, par = g & 1;
        const int abuf = 2 * sub + par;
        const int q = warp & 3;
        const int n_in = 32 * q + lane;
        for (int u = u0 + par, i = par; u < u1; u += 2, i += 2) {
            const int s = i % NW;
            const uint32_t ph = (uint32_t)((i / NW) & 1);
            const uint32_t aph = (uint32_t)((i >> 1) & 1);
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(wfull, s), ph, abort_flag, p.status))) break;
            const int tile = u / KB;
            const bool present = 2 * tile + sub < P.ltiles;
            uint32_t cw[4 * BITS];
            uint32_t sbw[sb_words(GROUP)];
            if (present) {
                const uint32_t blk = wbase + (uint32_t)s * WSTAGE + (uint32_t)(sub * BB);
                load_row_codes_smem<BITS>(blk, n_in, cw);
                load_row_sb_smem<GROUP>(blk + sb_offset(BITS, GROUP, n_in), sbw);
            } else {  // rows past the last layout tile: zero weights
#pragma unroll
                for (int w = 0; w < 4 * BITS; ++w) cw[w] = 0u;
#pragma unroll
                for (int w = 0; w < sb_words(GROUP); ++w) sbw[w] = 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(wempty, s));  // codes are in registers
            uint32_t w[32];
            weight_pairs<BITS, GROUP, 0, 32>(cw, sbw, w);
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(a_empty, abuf), aph ^ 1u, abort_flag, p.status))) break;
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + P_A_COL0 + (uint32_t)abuf * P_A_COLS;
            tmem_st32(ta, w);
            tmem_st_wait();
            weight_pairs<BITS, GROUP, 32, 32>(cw, sbw, w);
            tmem_st32(ta + 32, w);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(a_full, abuf));
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;               // TMEM lanes 32q .. 32q + 31: weight rows
        const int n_in = 32 * q + lane;
        const int M = p.M;
        const int nchunks = (M + 31) / 32;    // 32-column pieces of the accumulators to read
        pdl_wait();  // y and the partial slots may still be in use by the previous kernel
        int seg = 0;
        int seg_start = u0;
        for (int u = u0; u < u1; ++u) {
            const int tile = u / KB;
            const int kb = u - tile * KB;
            if (!(kb == KB - 1 || u == u1 - 1)) continue;
            const bool whole = (seg_start == tile * KB) && (kb == KB - 1);
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(acc_full, 0), (uint32_t)(seg & 1), abort_flag, p.status)))
                break;
            tc_fence_after();
            const int slot = P.slot_begin + 2 * c + (seg_start == u0 ? 0 : 1);
            float* sp = p.slots + (size_t)slot * kPromptSlotFloats;
#pragma unroll 1
            for (int sub = 0; sub < 2; ++sub) {
                const int64_t n = (int64_t)tile * P_TILE_N + sub * 128 + n_in;
#pragma unroll 1
                for (int cc = 0; cc < nchunks; ++cc) {
                    uint32_t vr[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)sub * P_ACC_COLS + 32u * cc, vr);
                    const int mb = 32 * cc;
                    if (whole) {
                        if (n < P.N) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (mb + e < M)
                                    P.y[(int64_t)(mb + e) * P.N + n] =
                                        __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(vr[e])));
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (mb + e < M) __stcg(sp + (size_t)(mb + e) * P_TILE_N + sub * 128 + n_in, __uint_as_float(vr[e]));
                    }
                }
            }
            // accumulators drained: the MMA thread may start the next segment
            // (a partial is added to the other runs' by prompt_merge_kernel)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(acc_empty, 0));
            ++seg;
            seg_start = u + 1;
        }
    }
#undef BAR

    // teardown: every role has left its loop and nothing is in flight
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, P_TMEM_COLS);
    }
}

// The tiles that several runs share: y = the runs' fp32 partials added in run
// order.  Grid: (4-row blocks of the activation rows, every tile of every
// projection); a thread owns four consecutive weight rows n of one activation
// row m (a 16-byte load from each run's partial: a warp reads 512 contiguous
// bytes), so the whole merge is a few rounds of fully parallel L2 reads.
// Tiles that one run owned were stored by prompt_kernel and are skipped.
// RB runs' loads are issued before they are added: 4, or 8 for launches whose
// tiles have more than four runs (every partial of a 7-run tile in one round
// of loads; with few runs the wider body costs more than it saves).
constexpr int P_MERGE_THREADS = 256;
template <int RB>
__global__ void __launch_bounds__(P_MERGE_THREADS) prompt_merge_kernel(const __grid_constant__ PromptParams p) {
    pdl_launch_dependents();  // the next kernel's prologue and weight copies may start
    pdl_wait();               // the partials of prompt_kernel are complete and visible
    const int t_all = (int)blockIdx.y;
    int pi = 0;
    for (int i = 1; i < p.nproj; ++i)
        if (t_all >= p.proj[i].ctr_begin) pi = i;
    const PromptProj& P = p.proj[pi];
    const int tile = t_all - P.ctr_begin;
    const int U = P.units, PC = P.nctas, KB = p.KB;
    const int t0 = tile * KB, t1 = t0 + KB - 1;
    const int cf = run_of(t0, U, PC), cl = run_of(t1, U, PC);
    if (cf == cl) return;
    const int m = 4 * (int)blockIdx.x + ((int)threadIdx.x >> 6);
    const int n4 = 4 * ((int)threadIdx.x & 63);  // weight row within the 256-row tile
    const int64_t n = (int64_t)tile * P_TILE_N + n4;
    if (m >= p.M || n >= P.N) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cb0 = cf; cb0 <= cl; cb0 += RB) {
        float4 f[RB];
#pragma unroll
        for (int d = 0; d < RB; ++d) {
            const int cb = cb0 + d;
            if (cb > cl) break;
            const int b0 = (int)((int64_t)cb * U / PC);
            const int sc = P.slot_begin + 2 * cb + (b0 >= t0 ? 0 : 1);
            f[d] = __ldcg(
                reinterpret_cast<const float4*>(p.slots + (size_t)sc * kPromptSlotFloats + (size_t)m * P_TILE_N + n4));
        }
#pragma unroll
        for (int d = 0; d < RB; ++d) {
            if (cb0 + d > cl) break;
            acc.x += f[d].x;
            acc.y += f[d].y;
            acc.z += f[d].z;
            acc.w += f[d].w;
        }
    }
    uint16_t* yr = P.y + (int64_t)m * P.N + n;
    const float av[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (n + e < P.N) yr[e] = __bfloat16_as_ushort(__float2bfloat16_rn(av[e]));
}

template <int BITS, int GROUP>
size_t prompt_smem_for() {
    return prm_ring_bytes<BITS, GROUP>() + sizeof(PromptSmem) + 1024;
}

template <int BITS, int GROUP>
cudaError_t launch_prompt_bg(const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    cudaError_t e = launch_pdl(prompt_kernel<BITS, GROUP>, grid, P_THREADS, prompt_smem_for<BITS, GROUP>(), st, p, map);
    if (e != cudaSuccess) return e;
    const PromptProj& last = p.proj[p.nproj - 1];
    const dim3 mgrid((unsigned)((p.M + 3) / 4), (unsigned)(last.ctr_begin + last.tiles));
    int runs = 0;  // most runs sharing one tile in this launch (a bound)
    for (int i = 0; i < p.nproj; ++i)
        if (p.proj[i].tiles > 0) runs = max(runs, (p.proj[i].nctas + p.proj[i].tiles - 1) / p.proj[i].tiles + 1);
    if (runs > 4) return launch_pdl(prompt_merge_kernel<8>, mgrid, P_MERGE_THREADS, 0, st, p);
    return launch_pdl(prompt_merge_kernel<4>, mgrid, P_MERGE_THREADS, 0, st, p);
}

template <int BITS>
cudaError_t launch_prompt_b(const PromptParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    if (p.group == 32) return launch_prompt_bg<BITS, 32>(p, map, grid, st);
    if (p.group == 64) return launch_prompt_bg<BITS, 64>(p, map, grid, st);
    return launch_prompt_bg<BITS, 128>(p, map, grid, st);
}

template <int BITS, int GROUP>
cudaError_t allow_prompt_bg() {
    return cudaFuncSetAttribute(prompt_kernel<BITS, GROUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)prompt_smem_for<BITS, GROUP>());
}

template <int BITS>
cudaError_t allow_prompt_b() {
    for (cudaError_t e : {allow_prompt_bg<BITS, 32>(), allow_prompt_bg<BITS, 64>(), allow_prompt_bg<BITS, 128>()})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

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
