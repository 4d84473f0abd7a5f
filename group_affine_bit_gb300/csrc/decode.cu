// decode.cu -- the memory-bound projection for M = 1..16 activation rows, on
// the 5th-generation tensor cores.
//
// Each 128-row x 128-deep weight block is one tcgen05.mma problem:
// D[128 weight rows, 16 activation rows] += W (tensor memory) * x^T (shared
// memory), fp32 in tensor memory.  Per CTA:
//   * two producer threads stream the blocks (9 KB for 4-bit codes and bf16
//     scale/bias words) two at a time with 1-D bulk copies into a ring of
//     weight slots, and a third loads each block's M x 128 activation rows
//     (TMA, 128-byte swizzle) into a ring of 16-row tiles whose other rows
//     stay zero;
//   * four lanes of work take blocks i = 0, 1, 2, 3 (mod 4) of the run; each
//     has a group of four dequantization warps -- one thread per weight row
//     reads the row's codes back, rounds every weight once as
//     bf16(fma(s, q, b)) (affqmm_format.cuh) and stores the row into the
//     lane's tensor-memory buffer with tcgen05.st, so the A operand never
//     touches shared memory -- and an MMA warp that issues the block's MMAs
//     (M = 128, N = 16, K = 16) into the lane's accumulator chain and
//     commits (at N = 16 a single issuing thread cannot keep up);
//   * the group that dequantized a tile segment's last block adds the four
//     chains with tcgen05.ld and stores bf16 y (coalesced along n).
// One CTA per SM owns all 512 tensor-memory columns.  Every barrier has one
// owner per phase sequence (stage s always belongs to lane s mod 4), so no
// parity wait can be satisfied by a phase one round too old.
// Prior art: the "reg variant" lane projection of the "Gemma 4 12B on the
// native Metal engine" page (4-bit groups in tensor-op registers, K split per
// shape); unlike it, every weight is rounded to bf16 before the contraction,
// as that page's prompt GEMM does.
//
// Work split: the projection's blocks, numbered tile-major, are cut into one
// contiguous run per resident CTA ("stream-K").  A tile cut by run boundaries
// gets one fp32 partial per run (its accumulator chains added first, in chain
// order); the last CTA to arrive (an atomic counter per
// tile and 32-row quarter, no waiting) adds them in run order and resets the
// counter.  The cut depends only on the projection, M and the device, so the
// same inputs give the same bits on every call, alone or stacked.  Every wait
// is on an mbarrier with a bound; a wait that gives up sets the workspace
// status word and an abort flag, and every role of the CTA finishes.
#include <cuda_bf16.h>

#include <cstddef>
#include <type_traits>

#include "affqmm_async.cuh"
#include "affqmm_format.cuh"
#include "affqmm_internal.h"
#include "affqmm_tc.cuh"

namespace affqmm {
namespace {

constexpr int D_LANES = 4;            // (dequant group, MMA issuer, A buffer, chain) lanes of work
constexpr int D_ISSUER0 = 1;                       // warp 0: weights producer of the even blocks
constexpr int D_DEQ_WARP0 = 1 + D_LANES;           // then 4 issuers, 4 groups of 4 dequant warps
constexpr int D_WPROD1 = D_DEQ_WARP0 + 4 * D_LANES; // weights producer of the odd blocks
constexpr int D_XPROD = D_WPROD1 + 1;              // activations producer
constexpr int D_THREADS = (D_XPROD + 1) * 32;
constexpr int D_MMA_N = 16;           // activation rows per MMA (M <= 16)
constexpr uint32_t D_X_PANEL = D_MMA_N * 128;      // 16 rows x 64 k bf16, 2 KB
constexpr uint32_t D_X_BYTES = 2 * D_X_PANEL;      // one 128-deep block of x
constexpr uint32_t D_TMEM_COLS = 512;
constexpr int D_A_HALVES = 3;                      // A buffers per lane, each half a block deep
constexpr uint32_t D_A_HALF_COLS = KBLK / 4;        // 32 columns: 64 bf16 per row
constexpr uint32_t D_A_COLS = D_A_HALVES * D_A_HALF_COLS;  // 96 columns per lane
constexpr uint32_t D_ACC_COL0 = D_LANES * D_A_COLS;
// Accumulators: one chain per lane of work (its blocks of the segment), and
// two segments' worth so the next segment starts while the last one is
// drained: column D_ACC_COL0 + 16 * (D_LANES * segment buffer + chain).
constexpr uint32_t D_IDESC = idesc_bf16_f32(128, D_MMA_N);
// Two rings: activation blocks (held until the block's MMAs are done) and
// packed weight blocks (held only until the dequantization warps have the
// codes in registers, so the weight ring covers the HBM latency).  Both
// depths are multiples of the lanes: slot s always belongs to lane s mod 4,
// so no barrier is waited on by two threads that could be a phase apart.
constexpr int D_XRING = 16;
constexpr int D_WRING_MAX = 24;
constexpr uint32_t kDecRingBudget = 210u * 1024u;

struct DecSmem {
    uint64_t wfull[D_WRING_MAX];
    uint64_t wempty[D_WRING_MAX];
    uint64_t xfull[D_XRING];
    uint64_t xempty[D_XRING];
    uint64_t a_full[D_A_HALVES * D_LANES];   // (lane, A buffer)
    uint64_t a_empty[D_A_HALVES * D_LANES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ void sts_zero16(uint32_t a) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
}

constexpr int dec_wring_for(int block) {
    return (int)((kDecRingBudget - D_XRING * D_X_BYTES) / (uint32_t)block) / D_LANES * D_LANES > D_WRING_MAX
               ? D_WRING_MAX
               : (int)((kDecRingBudget - D_XRING * D_X_BYTES) / (uint32_t)block) / D_LANES * D_LANES;
}
template <int BITS, int GROUP>
constexpr int dec_wring() {
    return dec_wring_for(block_bytes(BITS, GROUP));
}

template <int BITS, int GROUP>
__global__ void __launch_bounds__(D_THREADS, 1)
    decode_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap xmap) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int BB = block_bytes(BITS, GROUP);
    constexpr int NW = dec_wring<BITS, GROUP>();
    constexpr int NP = NW / 2;  // weight slots go in pairs: slot pair q serves lanes 2(q mod 2), 2(q mod 2) + 1
    constexpr int NX = D_XRING;
    static_assert(NW >= D_LANES && NW % D_LANES == 0 && NX % D_LANES == 0, "ring depths");
    static_assert(BB % 16 == 0, "bulk copies move multiples of 16 bytes");
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;          // activation ring (1024-aligned for the swizzle)
    const uint32_t wbase = base + (uint32_t)NX * D_X_BYTES;  // weight ring
    const uint32_t ring_bytes = (uint32_t)NX * D_X_BYTES + (uint32_t)NW * BB;
    DecSmem* sh = reinterpret_cast<DecSmem*>(smem_raw + (base - raw) + ring_bytes);
    const uint32_t sh_addr = base + ring_bytes;
#define BAR(field, i) (sh_addr + (uint32_t)offsetof(DecSmem, field) + 8u * (uint32_t)(i))
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int pi = 0;
    for (int i = 1; i < p.nproj; ++i)
        if ((int)blockIdx.x >= p.proj[i].cta_begin) pi = i;
    const DecProj& P = p.proj[pi];
    const int c = (int)blockIdx.x - P.cta_begin;
    const int U = P.units, PC = P.nctas, KB = p.KB;
    const int u0 = (int)((int64_t)c * U / PC);
    const int u1 = (int)((int64_t)(c + 1) * U / PC);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NP; ++s) {
            mbar_init(BAR(wfull, s), 1);
            mbar_init(BAR(wempty, s), 8);  // the four warps of each of the pair's two groups read the codes
        }
        for (int s = 0; s < NX; ++s) {
            mbar_init(BAR(xfull, s), 1);
            mbar_init(BAR(xempty, s), 1);  // the block's MMAs read x
        }
        for (int l = 0; l < D_A_HALVES * D_LANES; ++l) {
            mbar_init(BAR(a_full, l), 4);
            mbar_init(BAR(a_empty, l), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR(acc_full, b), D_LANES);  // every issuer commits at every segment end
            mbar_init(BAR(acc_empty, b), 4);       // the four warps of the group draining it
        }
        sh->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == D_ISSUER0) tmem_alloc(sh_addr + (uint32_t)offsetof(DecSmem, tmem_base), D_TMEM_COLS);
    // The activation tiles' rows M..15 stay zero for the whole launch: the
    // TMA loads write rows 0..M-1 only (the tensor map's box is M rows).
    for (uint32_t off = 16u * threadIdx.x; off < (uint32_t)NX * D_X_BYTES; off += 16u * D_THREADS)
        sts_zero16(base + off);
    fence_proxy_async_smem();  // generic-proxy zeros -> TMA writes and tensor-core reads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort_flag = &sh->abort_flag;
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (warp == 0 || warp == D_WPROD1) {
        // ---------------------------------------------------------- weights producers
        // Blocks go in pairs (two consecutive blocks are contiguous, ~18 KB:
        // a bulk copy moves data faster the larger it is), and two threads in
        // two warps take alternate pairs.  The weights never depend on an
        // earlier kernel, so these threads start before the grid dependency
        // is resolved.
        if (lane == 0) {
            const int pp = warp == 0 ? 0 : 1;
            const uint64_t policy = policy_evict_first();  // the weights are read once
            const int n = u1 - u0;
            for (int j = pp; 2 * j < n; j += 2) {
                const int ps = j % NP;
                const uint32_t ph = (uint32_t)((j / NP) & 1);
                if (!wait_or_abort_lazy(BAR(wempty, ps), ph ^ 1u, abort_flag, p.status)) break;
                const uint32_t bytes = (2 * j + 1 < n ? 2u : 1u) * (uint32_t)BB;
                mbar_arrive_expect_tx(BAR(wfull, ps), bytes);
                bulk_g2s_hint(wbase + (uint32_t)ps * (2u * BB), P.packed + (size_t)(u0 + 2 * j) * BB, bytes,
                              BAR(wfull, ps), policy);
            }
        }
    } else if (warp == D_XPROD) {
        // ---------------------------------------------------------- activations producer
        if (lane == 0) {
            prefetch_tmap(&xmap);
            pdl_wait();  // x may come from the previous kernel
            const uint32_t x_bytes = 2u * 64u * 2u * (uint32_t)p.M;  // two panels of M rows
            int kb = u0 % KB;
            for (int u = u0, i = 0; u < u1; ++u, ++i) {
                const int s = i % NX;
                const uint32_t ph = (uint32_t)((i / NX) & 1);
                if (!wait_or_abort_lazy(BAR(xempty, s), ph ^ 1u, abort_flag, p.status)) break;
                const uint32_t st = base + (uint32_t)s * D_X_BYTES;
                mbar_arrive_expect_tx(BAR(xfull, s), x_bytes);
                tma_load_2d(st, &xmap, kb * KBLK, 0, BAR(xfull, s));
                tma_load_2d(st + D_X_PANEL, &xmap, kb * KBLK + 64, 0, BAR(xfull, s));
                if (++kb == KB) kb = 0;
            }
        }
    } else if (warp < D_DEQ_WARP0) {
        // ---------------------------------------------------------- MMA issuers
        // Issuer e takes the blocks i = e (mod 4) of the run (the ones group e
        // dequantizes into A buffer e) and accumulates them into chain e of
        // the segment.  Every issuer waits for the segment's accumulators to
        // be drained and commits at every segment end, so none runs a segment
        // ahead of another.
        if (lane == 0) {
            const int e = warp - D_ISSUER0;
            int seg = 0, seg_start = u0;
            int kb = u0 % KB;
            bool open = false;
            for (int u = u0, i = 0; u < u1; ++u, ++i) {
                const bool seg_end = (kb == KB - 1) || (u == u1 - 1);
                const int db = seg & 1;
                if (!open) {
                    if (!wait_or_abort(BAR(acc_empty, db), (uint32_t)((seg >> 1) & 1) ^ 1u, abort_flag, p.status))
                        break;
                    open = true;
                }
                if ((i & (D_LANES - 1)) == e) {
                    const int s = i % NX;
                    const uint32_t ph = (uint32_t)((i / NX) & 1);
                    const int jl = i / D_LANES;  // this lane's block count; its halves are 2 jl, 2 jl + 1
                    if (!wait_or_abort(BAR(xfull, s), ph, abort_flag, p.status)) break;
                    const int j = u - seg_start;  // block index within the segment
                    const uint32_t dcol = tmem + D_ACC_COL0 + (uint32_t)(D_LANES * db + e) * D_MMA_N;
                    const uint32_t acol = tmem + (uint32_t)e * D_A_COLS;
                    const uint64_t bd0 = sw128_desc(base + (uint32_t)s * D_X_BYTES);
                    bool ok = true;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {  // each half of the depth as soon as it is in TMEM
                        const int t = 2 * jl + h;  // the lane's half number: buffer t mod 3, use t / 3
                        const int b = t % D_A_HALVES;
                        if (!wait_or_abort(BAR(a_full, D_A_HALVES * e + b), (uint32_t)((t / D_A_HALVES) & 1), abort_flag,
                                           p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int k = 4 * h; k < 4 * h + 4; ++k) {
                            // +32 bytes per 16-deep step, +2 KB per 64-deep panel (descriptor units of 16 bytes)
                            const uint64_t bd = bd0 + (uint64_t)((k >> 2) * (D_X_PANEL >> 4) + (k & 3) * 2);
                            umma_ts(dcol, acol + (uint32_t)b * D_A_HALF_COLS + 8u * (k - 4 * h), bd, D_IDESC,
                                    (j < D_LANES && k == 0) ? 0u : 1u);
                        }
                        umma_commit(BAR(a_empty, D_A_HALVES * e + b));
                    }
                    if (!ok) break;
                    umma_commit(BAR(xempty, s));
                }
                if (seg_end) {
                    umma_commit(BAR(acc_full, db));  // this issuer's MMAs of the segment (maybe none)
                    ++seg;
                    open = false;
                    seg_start = u + 1;
                }
                if (++kb == KB) kb = 0;
            }
        }
    } else {
        // ------------------------------------------ dequantization (+ epilogue)
        const int g = (warp - D_DEQ_WARP0) >> 2;  // group: blocks i = g (mod 4)
        const int q = warp & 3;                   // tensor-memory lanes 32q .. 32q + 31
        const int n_in = 32 * q + lane;           // weight row of this thread within the tile
        const int M = p.M;
        const int tile0 = u0 / KB;
        pdl_wait();  // y, the partials and the counters may still be in use by the previous kernel
        for (int u = u0 + g, i = g; u < u1; u += D_LANES, i += D_LANES) {
            const int ps = (i >> 1) % NP;  // pair slot of this block
            const uint32_t ph = (uint32_t)(((i >> 1) / NP) & 1);
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(wfull, ps), ph, abort_flag, p.status))) break;
            const uint32_t st = wbase + (uint32_t)ps * (2u * BB) + (uint32_t)(i & 1) * BB;
            uint32_t cw[4 * BITS];
            load_row_codes_smem<BITS>(st, n_in, cw);
            uint32_t sbw[sb_words(GROUP)];
            load_row_sb_smem<GROUP>(st + sb_offset(BITS, GROUP, n_in), sbw);
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(wempty, ps));  // codes are in registers
            // Each half of the row's depth goes to the next of the lane's three
            // half-block A buffers, so the dequantization runs up to a block
            // and a half ahead of the lane's MMAs.
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)g * D_A_COLS;
            auto half = [&](auto hc) -> bool {
                constexpr int H = decltype(hc)::value;
                uint32_t w[32];
                weight_pairs<BITS, GROUP, 32 * H, 32>(cw, sbw, w);
                const int t = 2 * (i / D_LANES) + H;  // the lane's half number: buffer t mod 3, use t / 3
                const int b = t % D_A_HALVES;
                if (!__all_sync(0xffffffffu, wait_or_abort(BAR(a_empty, D_A_HALVES * g + b),
                                                           (uint32_t)((t / D_A_HALVES) & 1) ^ 1u, abort_flag, p.status)))
                    return false;
                tc_fence_after();
                tmem_st32(ta + (uint32_t)b * D_A_HALF_COLS, w);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(a_full, D_A_HALVES * g + b));
                return true;
            };
            if (!half(std::integral_constant<int, 0>{})) break;
            if (!half(std::integral_constant<int, 1>{})) break;

            // ---- this block ends a tile segment: drain the accumulators
            const int tile = u / KB;
            const int kb = u - tile * KB;
            if (!(kb == KB - 1 || u == u1 - 1)) continue;
            const int seg = tile - tile0;
            const int db = seg & 1;
            const int seg_start = seg == 0 ? u0 : tile * KB;  // first block of the segment
            const int len = u - seg_start + 1;
            const int i_start = seg_start - u0;
            if (!__all_sync(0xffffffffu,
                            wait_or_abort(BAR(acc_full, db), (uint32_t)((seg >> 1) & 1), abort_flag, p.status)))
                break;
            tc_fence_after();
            // chain l holds the segment's blocks with run index = l (mod 4);
            // add the chains that received a block, in chain order
            float v[D_MMA_N];
            bool any = false;
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + D_ACC_COL0 + (uint32_t)(D_LANES * db) * D_MMA_N;
#pragma unroll
            for (int l = 0; l < D_LANES; ++l) {
                const bool used = len >= D_LANES || ((l - i_start) & (D_LANES - 1)) < len;
                uint32_t r[16];
                tmem_ld16(trow + (uint32_t)l * D_MMA_N, r);
                if (used) {
#pragma unroll
                    for (int e2 = 0; e2 < D_MMA_N; ++e2) v[e2] = any ? v[e2] + __uint_as_float(r[e2]) : __uint_as_float(r[e2]);
                    any = true;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(acc_empty, db));  // accumulators drained
            const int64_t n = (int64_t)tile * TILE_N + n_in;
            const bool whole = (seg_start == tile * KB) && (kb == KB - 1);
            if (whole) {
                if (n < P.N)
                    for (int m = 0; m < M; ++m)
                        P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[m]));
                continue;
            }
            // publish this run's partial of the tile; the last run to arrive
            // adds them all in run (k) order
            const int slot = P.slot_begin + 2 * c + (seg_start == u0 ? 0 : 1);
            float4* sp = reinterpret_cast<float4*>(p.partials + ((size_t)slot * TILE_N + n_in) * D_MMA_N);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) __stcg(sp + e2, make_float4(v[4 * e2], v[4 * e2 + 1], v[4 * e2 + 2], v[4 * e2 + 3]));
            __syncwarp();
            unsigned prev = 0;
            unsigned* ctr = &p.counters[(size_t)(P.ctr_begin + tile) * 4 + q];
            if (lane == 0) prev = atom_add_acq_rel(ctr, 1u);
            __syncwarp();
            prev = __shfl_sync(0xffffffffu, prev, 0);
            const int t0 = tile * KB, t1 = t0 + KB - 1;
            const int cf = run_of(t0, U, PC), cl = run_of(t1, U, PC);
            if (prev != (unsigned)(cl - cf)) continue;
            float acc[D_MMA_N];
#pragma unroll
            for (int e2 = 0; e2 < D_MMA_N; ++e2) acc[e2] = 0.f;
            for (int cb = cf; cb <= cl; ++cb) {
                const int b0 = (int)((int64_t)cb * U / PC);
                const int sc = P.slot_begin + 2 * cb + (b0 >= t0 ? 0 : 1);
                const float4* cp = reinterpret_cast<const float4*>(p.partials + ((size_t)sc * TILE_N + n_in) * D_MMA_N);
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float4 f = __ldcg(cp + e2);
                    acc[4 * e2] += f.x;
                    acc[4 * e2 + 1] += f.y;
                    acc[4 * e2 + 2] += f.z;
                    acc[4 * e2 + 3] += f.w;
                }
            }
            if (n < P.N)
                for (int m = 0; m < M; ++m) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
            if (lane == 0) *ctr = 0u;
        }
    }
#undef BAR
    // teardown: every role has left its loop and nothing is in flight
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == D_ISSUER0) {
        tc_fence_after();
        tmem_dealloc(tmem, D_TMEM_COLS);
    }
}

template <int BITS, int GROUP>
size_t dec_smem() {
    return (size_t)D_XRING * D_X_BYTES + (size_t)dec_wring<BITS, GROUP>() * block_bytes(BITS, GROUP) + sizeof(DecSmem) +
           1024;
}

template <int BITS, int GROUP>
cudaError_t launch_bg(const DecParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    const size_t smem = dec_smem<BITS, GROUP>();
    return launch_pdl(decode_kernel<BITS, GROUP>, grid, D_THREADS, smem, st, p, map);
}

template <int BITS>
cudaError_t launch_b(int group, const DecParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    if (group == 32) return launch_bg<BITS, 32>(p, map, grid, st);
    if (group == 64) return launch_bg<BITS, 64>(p, map, grid, st);
    return launch_bg<BITS, 128>(p, map, grid, st);
}

template <int BITS, int GROUP>
cudaError_t allow_bg() {
    return cudaFuncSetAttribute(decode_kernel<BITS, GROUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)dec_smem<BITS, GROUP>());
}

template <int BITS>
cudaError_t allow_b() {
    for (cudaError_t e : {allow_bg<BITS, 32>(), allow_bg<BITS, 64>(), allow_bg<BITS, 128>()})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

cudaError_t decode_allow_smem() {
    for (cudaError_t e : {allow_b<2>(), allow_b<3>(), allow_b<4>(), allow_b<5>(), allow_b<6>(), allow_b<8>()})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_decode(int bits, int group, const DecParams& p, const CUtensorMap& map, int grid,
                          cudaStream_t st) {
    switch (bits) {
        case 2: return launch_b<2>(group, p, map, grid, st);
        case 3: return launch_b<3>(group, p, map, grid, st);
        case 4: return launch_b<4>(group, p, map, grid, st);
        case 5: return launch_b<5>(group, p, map, grid, st);
        case 6: return launch_b<6>(group, p, map, grid, st);
        case 8: return launch_b<8>(group, p, map, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace affqmm
