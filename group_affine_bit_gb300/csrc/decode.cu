// decode.cu -- the memory-bound projection for M = 1..16 activation rows.
//
// y[m, n] = bf16( sum_k x[m, k] * bf16(s * q[n, k] + b) ), fp32 sums.
//
// At M <= 16 the work is a stream of packed weights: every byte is read once
// and the dequantization arithmetic (three bf16x2 operations per two weights)
// is what the SMs must keep up with.  The dot products go through the warp-
// level matrix instruction (mma.sync m16n8k16, bf16 in, fp32 accumulate) with
// the weights as the A fragment straight from the registers that rounded
// them, so nothing is written back to shared or tensor memory: one
// instruction does the 256 multiply-adds of 16 rows x 16 k for up to 8
// activation rows, where fp32 FMAs would cost one instruction per weight and
// row.
//
// Each CTA (two per SM) works through one contiguous run of (128-row tile,
// 128-deep block) units, numbered tile-major, from its last unit down to its
// first.  A ring of slots in shared memory holds two consecutive blocks each
// (one bulk copy, 9 KB a block at 4 bits, group 64) and their activation
// tiles:
//   * a weights producer thread copies the slot's blocks; an activation
//     producer thread loads the slot's activation tiles with TMA -- M rows x
//     136 k, 272 bytes a row so that the eight rows of a matrix load sit on
//     distinct banks -- into tiles whose rows M..15 stay zero;
//   * eight consumer warps each own 16 rows of every block: thread t
//     (g = t/4, class c = t mod 4) reads class c's code words of rows g and
//     g + 8 and their scale/bias words (affqmm_format.cuh), loads the
//     activation fragments with ldmatrix, releases the slot after its last
//     read, and for each of the 8 16-deep steps rounds four weight pairs --
//     bf16(fma(s, q, b)), one rounding -- and issues one mma (two when
//     M > 8) into fp32 registers;
//   * at the end of each tile segment (the part of a tile inside the run)
//     every consumer warp writes its fp32 sums to a staging buffer in shared
//     memory and goes on; an epilogue warp stores the tile as bf16 y, or, for
//     a tile that several runs share, publishes the run's fp32 partial and
//     counts in on the tile's counter.  The last run to arrive adds every
//     run's partial in run order and stores y.  Only the epilogue warp waits
//     on global memory (a round trip to L2 is about a microsecond under full
//     load), so the consumers never do.
// Runs are walked downwards, so a tile's lower runs reach it at their start
// and the highest run reaches it at its very end: that run's epilogue finds
// the other partials already published, adds them ahead of time and skips
// the counter.  Same inputs, same bits, alone or stacked: the cut, the order
// within a run and the order of the merge are fixed.
// The exact-codes instantiation (the pages' lane projection) puts the exact
// codes into the A fragments and adds s * sum(q x) + b * sum(x) per group;
// its activation warp loads the tiles itself and writes each group's sum of
// x next to them (or copies sums that the kernel producing x wrote).  The
// epilogue can also apply GeGLU to a gate/up stack interleaved in 16-row
// blocks (h = gelu_approx(gate) * up as bf16 operations).
// Every wait is on an mbarrier with a bound; a wait that gives up sets the
// workspace status word and an abort flag, and every role finishes.
// Prior art: the "reg variant" lane projection of the "Gemma 4 12B on the
// native Metal engine" page (4-bit groups held in registers for the
// matrix-op, K split per shape, geglu as the gate/up projection's epilogue
// on a stack interleaved in 16-row blocks); unlike it, every weight of
// affqmm_run is rounded to bf16 before the contraction, as that page's
// prompt GEMM does.
#include <cuda_bf16.h>

#include <cstddef>
#include <type_traits>

#include "affqmm_async.cuh"
#include "affqmm_format.cuh"
#include "affqmm_internal.h"
#include "affqmm_tc.cuh"

namespace affqmm {
namespace {

// Consumer groups per CTA.  1: two CTAs per SM, eight consumer warps each,
// every warp taking both blocks of a slot.  2: one CTA per SM, sixteen
// consumer warps; group 0 takes the upper block of each slot, group 1 the
// lower one, and the epilogue adds the groups' sums in that order.
#ifndef AFFQMM_DECODE_GROUPS
#define AFFQMM_DECODE_GROUPS 1
#endif
constexpr int D_GROUPS = AFFQMM_DECODE_GROUPS;
static_assert(D_GROUPS == 1 || D_GROUPS == 2, "one or two consumer groups");
constexpr int D_CWARPS = 8 * D_GROUPS;        // consumer warp w owns rows 16 (w mod 8) .. + 15 of its blocks
constexpr int D_WPROD = D_CWARPS;             // weights producer warp
constexpr int D_XPROD = D_CWARPS + 1;         // activations producer warp
constexpr int D_EPI = D_CWARPS + 2;           // epilogue warp
constexpr int D_THREADS = (D_CWARPS + 3) * 32;
constexpr uint32_t D_XROW = 272;              // bytes per activation row of a tile (128 k + 8 of padding)
constexpr int D_SLOTS_MAX = 16;
constexpr int D_CTAS_PER_SM = D_GROUPS == 1 ? 2 : 1;
constexpr uint32_t D_SMEM = D_GROUPS == 1 ? 112u * 1024u : 227u * 1024u;   // dynamic shared memory per CTA
constexpr uint32_t D_BARS = 1024u;            // barriers and flags; the staging buffers and the ring follow
constexpr uint32_t D_XSUM = 256;              // per block, exact-codes mode: [4 groups][16 rows] fp32 sums of x

// A ring slot: the lower block (position 0), the upper block (position 1),
// their activation tiles in the same order, then their group sums.  The
// consumers take the upper block first (the run is walked downwards).
struct DecSmem {
    uint64_t full[D_SLOTS_MAX];    // both producers' bytes (arrivals: 2)
    uint64_t empty[D_SLOTS_MAX];   // every consumer warp (8)
    uint64_t stage_full[2];        // every consumer warp has staged its sums (8)
    uint64_t stage_empty[2];       // the epilogue is done with the buffer (1)
    uint64_t never;                // completed by nothing: the fault_wait test hook waits on it
    uint64_t merge;                // the last segment's copies of other runs' partials (1)
    int issued[2];                 // slots armed by the weights producer [0] and the activation producer [1]
    int abort_flag;
};
static_assert(sizeof(DecSmem) <= D_BARS, "barriers fit in their area");

template <int NB>
constexpr uint32_t x_tile_bytes() { return 8u * NB * D_XROW; }   // 8 rows per activation block of the mma
template <int NB>
constexpr uint32_t stage_bytes() { return D_GROUPS * TILE_N * 8u * NB * 4u; }   // [group][128 rows][8 NB] fp32
template <int NB>
constexpr uint32_t ring_offset() { return D_BARS + 2u * stage_bytes<NB>(); }
template <int BITS, int GROUP, int NB>
constexpr uint32_t slot_bytes() {
    return 2u * (uint32_t)block_bytes(BITS, GROUP) + 2u * x_tile_bytes<NB>() + 2u * D_XSUM;
}
template <int BITS, int GROUP, int NB>
constexpr int ring_slots() {
    return (int)((D_SMEM - 128u - ring_offset<NB>()) / slot_bytes<BITS, GROUP, NB>()) > D_SLOTS_MAX
               ? D_SLOTS_MAX
               : (int)((D_SMEM - 128u - ring_offset<NB>()) / slot_bytes<BITS, GROUP, NB>());
}

__device__ __forceinline__ void sts_zero16(uint32_t a) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
}
__device__ __forceinline__ void sts_v2f(uint32_t a, float x, float y) {
    asm volatile("st.shared.v2.f32 [%0], {%1,%2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void lds_v4f(uint32_t a, float (&v)[4]) {
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(a)
                 : "memory");
}
__device__ __forceinline__ void sts_v4f(uint32_t a, const float (&v)[4]) {
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3])
                 : "memory");
}
// Order this thread's earlier global accesses before its later ones at GPU
// scope (release and acquire; lighter than the sequentially consistent fence).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Whether the phase of parity `parity` of `bar` has completed (no waiting).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a)
                 : "memory");
}
// d (+)= a (16 x 16 bf16, row) * b (16 x 8 bf16, col), fp32
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The 16-deep step S of a block: weight pairs 2S and 2S + 1 of the thread's
// class for its two rows (the A fragment: row g k-low, row g + 8 k-low, row g
// k-high, row g + 8 k-high) times the activation fragments.
template <int BITS, int GROUP, int NB, int S>
__device__ __forceinline__ void mma_step(const uint32_t* wl, const uint32_t* wh, const uint32_t* sl,
                                         const uint32_t* sh, const uint32_t (&b)[NB][8][2], float* acc) {
    const uint32_t a0 = class_weight_pair<BITS, GROUP, 2 * S>(wl, sl);
    const uint32_t a1 = class_weight_pair<BITS, GROUP, 2 * S>(wh, sh);
    const uint32_t a2 = class_weight_pair<BITS, GROUP, 2 * S + 1>(wl, sl);
    const uint32_t a3 = class_weight_pair<BITS, GROUP, 2 * S + 1>(wh, sh);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) mma_bf16(acc + 4 * nb, a0, a1, a2, a3, b[nb][S][0], b[nb][S][1]);
}
template <int BITS, int GROUP, int NB, int S = 0>
__device__ __forceinline__ void mma_steps(const uint32_t* wl, const uint32_t* wh, const uint32_t* sl,
                                          const uint32_t* sh, const uint32_t (&b)[NB][8][2], float* acc) {
    if constexpr (S < 8) {
        mma_step<BITS, GROUP, NB, S>(wl, wh, sl, sh, b, acc);
        mma_steps<BITS, GROUP, NB, S + 1>(wl, wh, sl, sh, b, acc);
    }
}
// Exact-codes mode (the pages' lane projection): the A fragment holds the
// exact codes q (no rounding of s*q + b), the mmas of one group accumulate
// sum_k q x in accg, and at the group's end
//     acc += s_row * accg + b_row * sum_{k in group} x[m, k]
// with the group sums xs (fp32 [group][16 rows]) written by the activation
// producer.  sl/sh hold the rows' s | b << 16 words.
template <int BITS, int GROUP, int NB, int S = 0>
__device__ __forceinline__ void mma_steps_exact(const uint32_t* wl, const uint32_t* wh, const uint32_t* sl,
                                                const uint32_t* sh, const uint32_t (&b)[NB][8][2], uint32_t xs, int c,
                                                float* acc, float* accg) {
    if constexpr (S < 8) {
        constexpr int P0 = plane0_bits(BITS);
        const uint32_t a0 = class_code_pair<BITS, 2 * S>(wl, wl + P0);
        const uint32_t a1 = class_code_pair<BITS, 2 * S>(wh, wh + P0);
        const uint32_t a2 = class_code_pair<BITS, 2 * S + 1>(wl, wl + P0);
        const uint32_t a3 = class_code_pair<BITS, 2 * S + 1>(wh, wh + P0);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma_bf16(accg + 4 * nb, a0, a1, a2, a3, b[nb][S][0], b[nb][S][1]);
        constexpr int SPG = GROUP / 16;  // 16-deep steps per group
        if constexpr ((S + 1) % SPG == 0) {
            constexpr int GI = S / SPG;
            const float s_lo = __uint_as_float(sl[GI] << 16), b_lo = __uint_as_float(sl[GI] & 0xFFFF0000u);
            const float s_hi = __uint_as_float(sh[GI] << 16), b_hi = __uint_as_float(sh[GI] & 0xFFFF0000u);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                uint32_t x0u, x1u;  // the group sums of activation rows 8nb + 2c, 8nb + 2c + 1
                lds_v2(xs + (uint32_t)(GI * 16 + 8 * nb + 2 * c) * 4u, x0u, x1u);
                const float x0 = __uint_as_float(x0u), x1 = __uint_as_float(x1u);
                float* a = acc + 4 * nb;
                float* q = accg + 4 * nb;
                a[0] = fmaf(b_lo, x0, fmaf(s_lo, q[0], a[0]));
                a[1] = fmaf(b_lo, x1, fmaf(s_lo, q[1], a[1]));
                a[2] = fmaf(b_hi, x0, fmaf(s_hi, q[2], a[2]));
                a[3] = fmaf(b_hi, x1, fmaf(s_hi, q[3], a[3]));
                q[0] = q[1] = q[2] = q[3] = 0.f;
            }
        }
        mma_steps_exact<BITS, GROUP, NB, S + 1>(wl, wh, sl, sh, b, xs, c, acc, accg);
    }
}

// The activation fragments of one block: 8 steps x (k low, k high) for each
// 8-row activation block.  xa is this lane's ldmatrix row address in the tile.
template <int NB>
__device__ __forceinline__ void load_x_frags(uint32_t xa, uint32_t (&b)[NB][8][2]) {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            ldmatrix_x4(xa + 8u * D_XROW * nb + 64u * q, b[nb][2 * q][0], b[nb][2 * q][1], b[nb][2 * q + 1][0],
                        b[nb][2 * q + 1][1]);
}

// bf16 rounding of an fp32 value, back in fp32.
__device__ __forceinline__ float bf16r(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// mlx_lm's GeGLU on one pair of bf16 values (gate g, up u, as floats):
// h = gelu_approx(g) * u with gelu_approx(g) = 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))), every
// operation rounded to bf16 as MLX evaluates it on bf16 arrays, the constants taken as bf16.  The products of
// two bf16 values and the cube of one are exact in fp32, and so is the sum of two unless they lie more than 16
// binades apart, where the smaller cannot move the larger's bf16 rounding: each fp32 result rounded to bf16 is
// the single rounding of the exact value (results below fp32's normal range excepted).  tanh is tanhf.
__device__ __forceinline__ uint16_t geglu_bf16(float g, float u) {
    constexpr float C1 = 0.044677734375f;   // bf16(0.044715)
    constexpr float C2 = 0.796875f;         // bf16(sqrt(2 / pi))
    const float cube = bf16r(g * g * g);
    const float a = bf16r(C1 * cube);
    const float z = bf16r(g + a);
    const float v = bf16r(C2 * z);
    const float t = bf16r(tanhf(v));
    const float e = bf16r(1.0f + t);
    const float h = bf16r(0.5f * g);
    const float r = bf16r(h * e);
    return __bfloat16_as_ushort(__float2bfloat16_rn(r * u));
}

// The epilogue's output for one weight row of a tile and activation rows
// [8 mc, 8 mc + 8): v[e] is the fp32 value of weight row n = 128 tile + 32 i +
// lane, activation row 8 mc + e.  Plain form: y[m, n] = bf16(v).  GeGLU form
// (rows interleaved in 16-row blocks: rows 32 j .. 32 j + 15 are gate rows of
// hidden units 16 j .. 16 j + 15, rows 32 j + 16 .. 32 j + 31 their up rows):
// lanes 0-15 hold gate rows and take the up values from lane + 16, and
// h[m, 16 j + lane] = geglu(gate, up).  Every lane calls this with the same
// (tile, mc, i).
__device__ __forceinline__ void store_row_chunk(const DecParams& p, const DecProj& P, int tile, int mc, int i,
                                                int lane, const float (&v)[8]) {
    const int M = p.M;
    const int64_t n = (int64_t)tile * TILE_N + 32 * i + lane;
    if (p.epi == 0) {
        if (n >= P.N) return;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int m = 8 * mc + e;
            if (m < M) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[e]));
        }
    } else {
        const int64_t F = P.N / 2;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float gv = bf16r(v[e]);
            const float uv = __shfl_down_sync(0xffffffffu, gv, 16);
            const int m = 8 * mc + e;
            if (lane < 16 && m < M && n < P.N) P.y[(int64_t)m * F + 16 * (n / 32) + lane] = geglu_bf16(gv, uv);
        }
    }
}

__device__ __forceinline__ void add_partial(float (&v)[8], const float* q) {
    const float4 q0 = __ldcg(reinterpret_cast<const float4*>(q)), q1 = __ldcg(reinterpret_cast<const float4*>(q) + 1);
    v[0] += q0.x; v[1] += q0.y; v[2] += q0.z; v[3] += q0.w;
    v[4] += q1.x; v[5] += q1.y; v[6] += q1.z; v[7] += q1.w;
}

template <int BITS, int GROUP, int NB, bool EXACT>
__global__ void __launch_bounds__(D_THREADS, D_CTAS_PER_SM)
    decode_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap xmap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    constexpr int BB = block_bytes(BITS, GROUP);
    constexpr int SBW = sb_words(GROUP);
    constexpr int MP = 8 * NB;                       // staged activation rows per weight row
    constexpr uint32_t XT = x_tile_bytes<NB>();
    constexpr uint32_t SLOT = slot_bytes<BITS, GROUP, NB>();
    constexpr uint32_t STG = stage_bytes<NB>();
    constexpr int NS = ring_slots<BITS, GROUP, NB>();
    static_assert(BB % 128 == 0 && SLOT % 128 == 0 && XT % 128 == 0, "bulk copies and tiles 128-byte aligned");
    static_assert(NS >= 2, "at least two ring slots");
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sh_addr = (raw + 127u) & ~127u;
    DecSmem* sh = reinterpret_cast<DecSmem*>(smem_raw + (sh_addr - raw));
    const uint32_t stage0 = sh_addr + D_BARS;               // staging buffer b at stage0 + b * STG
    const uint32_t ring = sh_addr + ring_offset<NB>();      // slot s at ring + s * SLOT
    const int M = p.M;
#define BAR(field, i) (sh_addr + (uint32_t)offsetof(DecSmem, field) + 8u * (uint32_t)(i))
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int pi = 0;
    for (int i = 1; i < p.nproj; ++i)
        if ((int)blockIdx.x >= p.proj[i].cta_begin) pi = i;
    const DecProj& P = p.proj[pi];
    const int cta = (int)blockIdx.x - P.cta_begin;
    const int U = P.units, PC = P.nctas, KB = p.KB;
    const int u0 = (int)((int64_t)cta * U / PC);
    const int u1 = (int)((int64_t)(cta + 1) * U / PC);
    const int nslots = (u1 - u0 + 1) / 2;       // slot j: units u1-1-2j (upper) and u1-2-2j (lower)
    const int tile_top = (u1 - 1) / KB, tile_bot = u0 / KB;
    const int nsegs = tile_top - tile_bot + 1;  // segment k: the run's part of tile tile_top - k

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(BAR(full, s), 2);
            mbar_init(BAR(empty, s), D_CWARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR(stage_full, b), D_CWARPS);
            mbar_init(BAR(stage_empty, b), 1);
        }
        mbar_init(BAR(never, 0), 1);
        mbar_init(BAR(merge, 0), 1);
        sh->issued[0] = sh->issued[1] = 0;
        sh->abort_flag = 0;
        fence_mbar_init();
    }
    // Activation rows M..8NB-1 (and their group sums) stay zero for the whole
    // launch: the producers write rows 0..M-1 only.
    for (int s = 0; s < NS; ++s)
        for (uint32_t off = 16u * threadIdx.x; off < 2u * XT + 2u * D_XSUM; off += 16u * D_THREADS)
            sts_zero16(ring + (uint32_t)s * SLOT + 2u * BB + off);
    fence_proxy_async_smem();  // generic-proxy zeros -> TMA writes
    __syncthreads();
    volatile int* abort_flag = &sh->abort_flag;
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (warp == D_WPROD || (warp == D_XPROD && !EXACT)) {
        // ---------------------------------------------------------- producers
        // The weights never depend on an earlier kernel (see affqmm_run on
        // weights written by the preceding kernel), so their producer starts
        // before the grid dependency is resolved; the activations may come
        // from the previous kernel.
        if (lane == 0) {
            const bool wprod = warp == D_WPROD;
            const uint64_t policy = policy_evict_first();  // the weights are read once
            if (!wprod) {
                prefetch_tmap(&xmap);
                pdl_wait();
            }
            int issued = 0;
            for (int j = 0; j < nslots; ++j) {
                const int s = j % NS;
                if (!wait_or_abort_lazy(BAR(empty, s), (uint32_t)((j / NS) & 1) ^ 1u, abort_flag, p.status)) break;
                const int uh = u1 - 1 - 2 * j, ul = uh - 1;
                const bool two = ul >= u0;
                const uint32_t st = ring + (uint32_t)s * SLOT;
                if (wprod) {
                    const uint32_t bytes = (two ? 2u : 1u) * (uint32_t)BB;
                    mbar_arrive_expect_tx(BAR(full, s), bytes);
                    bulk_g2s_hint(two ? st : st + (uint32_t)BB, P.packed + (size_t)(two ? ul : uh) * BB, bytes,
                                  BAR(full, s), policy);
                } else {
                    mbar_arrive_expect_tx(BAR(full, s), (two ? 2u : 1u) * D_XROW * (uint32_t)M);
                    tma_load_2d(st + 2u * BB + XT, &xmap, (uh % KB) * KBLK, 0, BAR(full, s));
                    if (two) tma_load_2d(st + 2u * BB, &xmap, (ul % KB) * KBLK, 0, BAR(full, s));
                }
                issued = j + 1;
            }
            sh->issued[wprod ? 0 : 1] = issued;
        }
    } else if (warp == D_XPROD) {
        // ------------------------- activations and their group sums (exact-codes mode)
        // The whole warp loads the slot's M rows of x (lane l: k = 4l .. 4l + 3
        // of each block), stores them in the tile layout, and writes each
        // group's sum of x: added by the lanes of the group in a fixed tree,
        // or copied from p.xsums when the kernel that produced x wrote them.
        pdl_wait();  // x may come from the previous kernel
        constexpr int LPG = GROUP / 4;  // lanes per group
        constexpr int GPB = KBLK / GROUP;
        const int64_t G = p.K / GROUP;
        for (int j = 0; j < nslots; ++j) {
            const int s = j % NS;
            int okw = 1;
            if (lane == 0) okw = wait_or_abort_lazy(BAR(empty, s), (uint32_t)((j / NS) & 1) ^ 1u, abort_flag, p.status);
            if (!__shfl_sync(0xffffffffu, okw, 0)) break;
            const int uh = u1 - 1 - 2 * j, ul = uh - 1;
            const bool two = ul >= u0;
            const uint32_t st = ring + (uint32_t)s * SLOT;
            // both blocks' loads first (one round trip to L2 per slot), then the stores and sums
            uint32_t xw[2][8 * NB][2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {                  // h = slot position: 0 lower block, 1 upper block
                const int u = h ? uh : ul;
                const int64_t k0 = (int64_t)(u % KB) * KBLK + 4 * lane;
                const bool in = (h == 1 || two) && k0 < p.K;  // K is a multiple of 32: a lane's values are all in or out
#pragma unroll
                for (int m = 0; m < 8 * NB; ++m) {
                    xw[h][m][0] = xw[h][m][1] = 0u;
                    if (m < M && in) {
                        const uint2 v = __ldg(reinterpret_cast<const uint2*>(p.x + (int64_t)m * p.K + k0));
                        xw[h][m][0] = v.x;
                        xw[h][m][1] = v.y;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h == 0 && !two) continue;
                const int u = h ? uh : ul;
                const uint32_t tile = st + 2u * BB + (uint32_t)h * XT;
                const uint32_t sums = st + 2u * BB + 2u * XT + (uint32_t)h * D_XSUM;
#pragma unroll
                for (int m = 0; m < 8 * NB; ++m) {
                    if (m >= M) break;
                    asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(tile + (uint32_t)m * D_XROW + 8u * lane),
                                 "r"(xw[h][m][0]), "r"(xw[h][m][1])
                                 : "memory");
                    if (p.xsums == nullptr) {
                        float v = __uint_as_float(xw[h][m][0] << 16) + __uint_as_float(xw[h][m][0] & 0xFFFF0000u) +
                                  __uint_as_float(xw[h][m][1] << 16) + __uint_as_float(xw[h][m][1] & 0xFFFF0000u);
#pragma unroll
                        for (int off = 1; off < LPG; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                        if (lane % LPG == 0)
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sums + (uint32_t)((lane / LPG) * 16 + m) * 4u),
                                         "f"(v)
                                         : "memory");
                    }
                }
                if (p.xsums != nullptr) {  // the producer's sums of this block's groups, as given
                    for (int i = lane; i < GPB * M; i += 32) {
                        const int gi = i / M, m = i - gi * M;
                        const int64_t gg = (int64_t)(u % KB) * GPB + gi;
                        const float v = gg < G ? __ldg(p.xsums + (int64_t)m * G + gg) : 0.f;
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(sums + (uint32_t)(gi * 16 + m) * 4u), "f"(v)
                                     : "memory");
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(BAR(full, s));  // the tiles and sums are written
                sh->issued[1] = j + 1;
            }
        }
    } else if (warp == D_EPI) {
        // ---------------------------------------------------------- epilogue
        // Lane l owns weight rows l, l + 32, l + 64, l + 96 of each tile.
        pdl_wait();  // y, the partials and the counters may still be in use by the previous kernel
        for (int k = 0; k < nsegs; ++k) {
            const int t = tile_top - k;
            const int lo = max(u0, t * KB), hi = min(u1, t * KB + KB);
            const bool whole = lo == t * KB && hi == t * KB + KB;
            const int cf = run_of(t * KB, U, PC), cl = run_of(t * KB + KB - 1, U, PC);
            unsigned* ctr = &p.counters[P.ctr_begin + t];
            const int b = k & 1;
            // The highest run of a shared tile reaches it last.  While its
            // consumers finish the run's last segment the epilogue watches the
            // tile's counter; once every lower run has published its partial it
            // adds them in run order, into the other staging buffer (free: this
            // is the last segment), and this run then needs no counter at all.
            bool fast = false;
            const uint32_t prefix = stage0 + (uint32_t)(1 - b) * STG;
            auto all_published = [&]() -> bool {
                unsigned cnt = 0;
                if (lane == 0) cnt = ld_acquire_gpu(ctr);
                cnt = __shfl_sync(0xffffffffu, cnt, 0);
                return cnt == (unsigned)(cl - cf);
            };
            auto take_prefix = [&]() {
                fence_acq_rel_gpu();  // every lane reads the partials after the acquire
                for (int mc = 0; mc < NB; ++mc)
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        float pre[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) pre[e] = 0.f;
                        const int r = 32 * i + lane;
                        for (int run = cf; run < cl; ++run) {
                            const int ub = (int)((int64_t)run * U / PC);
                            const int sc = P.slot_begin + 2 * run + (t == ub / KB ? 0 : 1);
                            add_partial(pre, p.partials + (size_t)sc * kDecSlotFloats + (size_t)r * 16 + 8 * mc);
                        }
                        const uint32_t a = prefix + ((uint32_t)r * MP + 8u * mc) * 4u;
                        sts_v4f(a, {pre[0], pre[1], pre[2], pre[3]});
                        sts_v4f(a + 16u, {pre[4], pre[5], pre[6], pre[7]});
                    }
            };
            const bool candidate = !whole && k == nsegs - 1 && cta == cl && cf < cl;
            if (candidate) {
                const uint32_t par = (uint32_t)((k >> 1) & 1);
                const long long t_start = clock64();
                for (;;) {
                    const bool ready = __all_sync(0xffffffffu, mbar_test(BAR(stage_full, b), par));
                    if (all_published()) {
                        take_prefix();
                        fast = true;
                        break;
                    }
                    if (ready || *abort_flag || clock64() - t_start > kWaitLimitCycles) break;
                    __nanosleep(500);
                }
            }
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(stage_full, b), (uint32_t)((k >> 1) & 1), abort_flag,
                                                       p.status)))
                break;
            // this run's value of weight row 32 i + lane, as the consumers staged it
            auto own = [&](int mc, int i, float (&v)[8]) {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = 0.f;
#pragma unroll
                for (int gr = 0; gr < D_GROUPS; ++gr) {  // group 0's sums, then group 1's
                    const uint32_t ra = stage0 + (uint32_t)b * STG + (uint32_t)gr * (STG / D_GROUPS) +
                                        ((uint32_t)(32 * i + lane) * MP + 8u * mc) * 4u;
                    float a0[4], a1[4];
                    lds_v4f(ra, a0);
                    lds_v4f(ra + 16u, a1);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[e] += a0[e];
                        v[4 + e] += a1[e];
                    }
                }
            };
            auto partial_of = [&](int run, int mc, int i) -> const float* {
                const int ub = (int)((int64_t)run * U / PC);
                const int sc = P.slot_begin + 2 * run + (t == ub / KB ? 0 : 1);
                return p.partials + (size_t)sc * kDecSlotFloats + (size_t)(32 * i + lane) * 16 + 8 * mc;
            };
            if (whole) {
                for (int mc = 0; mc < NB; ++mc)
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        float v[8];
                        own(mc, i, v);
                        store_row_chunk(p, P, t, mc, i, lane, v);
                    }
            } else if (fast) {
                for (int mc = 0; mc < NB; ++mc)
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        float v[8], q0[4], q1[4];
                        own(mc, i, v);
                        const uint32_t a = prefix + ((uint32_t)(32 * i + lane) * MP + 8u * mc) * 4u;
                        lds_v4f(a, q0);
                        lds_v4f(a + 16u, q1);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[e] = q0[e] + v[e];
                            v[4 + e] = q1[e] + v[4 + e];
                        }
                        store_row_chunk(p, P, t, mc, i, lane, v);
                    }
                if (lane == 0) *ctr = 0u;  // every other run has arrived; none will again
            } else {
                const int sc_own = P.slot_begin + 2 * cta + (t == tile_bot ? 0 : 1);
                float* sp = p.partials + (size_t)sc_own * kDecSlotFloats;
                for (int mc = 0; mc < NB; ++mc)
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        float v[8];
                        own(mc, i, v);
                        float4* q = reinterpret_cast<float4*>(sp + (size_t)(32 * i + lane) * 16 + 8 * mc);
                        __stcg(q, make_float4(v[0], v[1], v[2], v[3]));
                        __stcg(q + 1, make_float4(v[4], v[5], v[6], v[7]));
                    }
                fence_acq_rel_gpu();  // every lane's partial is visible GPU-wide before the arrival
                __syncwarp();
                unsigned prev = 0;
                if (lane == 0) prev = atom_add_acq_rel(ctr, 1u);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev == (unsigned)(cl - cf)) {  // the last run to arrive adds every run's partial in run order
                    fence_acq_rel_gpu();
                    // At the run's last segment the ring is free (every block has
                    // been consumed): one bulk copy per other run lands all of
                    // their partials in it in one round trip.  Otherwise the
                    // partials are read run by run, all four rows of a run at once.
                    const int cap = (int)((uint32_t)NS * SLOT / (uint32_t)(kDecSlotFloats * 4));
                    const bool landed = k == nsegs - 1 && cl - cf <= cap;
                    if (landed) {
                        if (lane == 0) {
                            asm volatile("fence.proxy.async.global;" ::: "memory");  // the acquire, then the copies' reads
                            mbar_arrive_expect_tx(BAR(merge, 0), (uint32_t)(cl - cf) * (uint32_t)(kDecSlotFloats * 4));
                            int slot_i = 0;
                            for (int run = cf; run <= cl; ++run) {
                                if (run == cta) continue;
                                const int ub = (int)((int64_t)run * U / PC);
                                const int sc = P.slot_begin + 2 * run + (t == ub / KB ? 0 : 1);
                                bulk_g2s(ring + (uint32_t)slot_i++ * (uint32_t)(kDecSlotFloats * 4),
                                         p.partials + (size_t)sc * kDecSlotFloats, (uint32_t)(kDecSlotFloats * 4),
                                         BAR(merge, 0));
                            }
                        }
                        if (!__all_sync(0xffffffffu, wait_or_abort(BAR(merge, 0), 0u, abort_flag, p.status))) break;
                    }
                    for (int mc = 0; mc < NB; ++mc)
#pragma unroll 1
                        for (int ih = 0; ih < 2; ++ih) {  // weight rows 32 i + lane, i = 2 ih, 2 ih + 1
                            float v[2][8];
#pragma unroll
                            for (int i = 0; i < 2; ++i)
#pragma unroll
                                for (int e = 0; e < 8; ++e) v[i][e] = 0.f;
                            int slot_i = 0;
                            for (int run = cf; run <= cl; ++run) {
                                // this run's partial: its own staged sums, a copy in the ring, or global memory
                                const bool mine = run == cta;
                                if (mine) {
#pragma unroll
                                    for (int i = 0; i < 2; ++i) {
                                        float o[8];
                                        own(mc, 2 * ih + i, o);
#pragma unroll
                                        for (int e = 0; e < 8; ++e) v[i][e] += o[e];
                                    }
                                } else if (landed) {
                                    const uint32_t sbase = ring + (uint32_t)slot_i++ * (uint32_t)(kDecSlotFloats * 4);
#pragma unroll
                                    for (int i = 0; i < 2; ++i) {
                                        float a0[4], a1[4];
                                        const uint32_t a = sbase + ((uint32_t)(32 * (2 * ih + i) + lane) * 16u + 8u * mc) * 4u;
                                        lds_v4f(a, a0);
                                        lds_v4f(a + 16u, a1);
#pragma unroll
                                        for (int e = 0; e < 4; ++e) {
                                            v[i][e] += a0[e];
                                            v[i][4 + e] += a1[e];
                                        }
                                    }
                                } else {
                                    const int ub = (int)((int64_t)run * U / PC);
                                    const int sc = P.slot_begin + 2 * run + (t == ub / KB ? 0 : 1);
                                    const float4* src = reinterpret_cast<const float4*>(p.partials + (size_t)sc * kDecSlotFloats) +
                                                        (size_t)(64 * ih + lane) * 4 + 2 * mc;
                                    // both rows' loads first: one round trip a run
                                    const float4 q0 = __ldcg(src), q1 = __ldcg(src + 1);
                                    const float4 q2 = __ldcg(src + 32 * 4), q3 = __ldcg(src + 32 * 4 + 1);
                                    v[0][0] += q0.x; v[0][1] += q0.y; v[0][2] += q0.z; v[0][3] += q0.w;
                                    v[0][4] += q1.x; v[0][5] += q1.y; v[0][6] += q1.z; v[0][7] += q1.w;
                                    v[1][0] += q2.x; v[1][1] += q2.y; v[1][2] += q2.z; v[1][3] += q2.w;
                                    v[1][4] += q3.x; v[1][5] += q3.y; v[1][6] += q3.z; v[1][7] += q3.w;
                                }
                            }
                            store_row_chunk(p, P, t, mc, 2 * ih, lane, v[0]);
                            store_row_chunk(p, P, t, mc, 2 * ih + 1, lane, v[1]);
                        }
                    if (lane == 0) *ctr = 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(stage_empty, b));
        }
    } else {
        // ---------------------------------------------------------- consumers
        const int grp = warp >> 3;                 // this warp's consumer group
        const int g = lane >> 2, c = lane & 3;
        const int r_lo = 16 * (warp & 7) + g, r_hi = r_lo + 8;  // this thread's rows within the tile
        // ldmatrix: lanes 8j .. 8j + 7 address matrix j's eight rows; matrix j
        // of a pair of steps is (step 2p + j/2, k half j mod 2)
        const uint32_t xlane = (uint32_t)(lane & 7) * D_XROW + (uint32_t)((lane >> 3) & 1) * 16u + (uint32_t)(lane >> 4) * 32u;
        float acc[4 * NB], accg[4 * NB];  // accg: the current group's sum of q x (exact-codes mode)
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) acc[e] = accg[e] = 0.f;
        // Stage this warp's sums of segment k (and clear them): rows r_lo,
        // r_hi, activation rows 8 nb + 2c and 8 nb + 2c + 1.
        auto stage = [&](int k) -> bool {
            const int b = k & 1;
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(stage_empty, b), (uint32_t)((k >> 1) & 1) ^ 1u, abort_flag,
                                                       p.status)))
                return false;
            const uint32_t base = stage0 + (uint32_t)b * STG + (uint32_t)grp * (STG / D_GROUPS);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                sts_v2f(base + ((uint32_t)r_lo * MP + 8u * nb + 2u * c) * 4u, acc[4 * nb + 0], acc[4 * nb + 1]);
                sts_v2f(base + ((uint32_t)r_hi * MP + 8u * nb + 2u * c) * 4u, acc[4 * nb + 2], acc[4 * nb + 3]);
            }
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e) acc[e] = 0.f;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(stage_full, b));
            return true;
        };
        // Test hook: wait, bounded by p.fault_wait cycles, on a barrier that
        // nothing completes; the wait runs out, sets the status word and the
        // abort flag, and the CTA finishes without output.
        bool run = p.fault_wait <= 0 ||
                   __all_sync(0xffffffffu,
                              wait_or_abort_within(BAR(never, 0), 0u, abort_flag, p.status, p.fault_wait));
        int cur = 0;  // the segment acc belongs to
        // the segment and depth block of this warp's next block (walked downwards)
        const int ufirst = max(u1 - 1 - (D_GROUPS == 2 ? grp : 0), u0);
        int seg = tile_top - ufirst / KB, kbu = ufirst % KB;
        for (int j = 0; run && j < nslots; ++j) {
            const int s = j % NS;
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(full, s), (uint32_t)((j / NS) & 1), abort_flag, p.status))) {
                run = false;
                break;
            }
            const uint32_t st = ring + (uint32_t)s * SLOT;
            const int uh = u1 - 1 - 2 * j;
            const bool two = uh - 1 >= u0;
#pragma unroll
            for (int h = 1; h >= 0; --h) {  // the upper block, then the lower one
                if (D_GROUPS == 2 && h != 1 - grp) continue;  // each group its own block
                if (h == 0 && !two) {
                    if (D_GROUPS == 2) {  // group 1 has no block in the run's odd last slot
                        __syncwarp();
                        if (lane == 0) mbar_arrive(BAR(empty, s));
                    }
                    break;
                }
                while (run && cur < seg) run = stage(cur++);
                if (!run) break;
                const uint32_t blk = st + (uint32_t)h * (uint32_t)BB;
                uint32_t wl[BITS], wh[BITS], sl[SBW], sh2[SBW];
                load_class_words_smem<BITS>(blk, r_lo, c, wl);
                load_class_words_smem<BITS>(blk, r_hi, c, wh);
                load_row_sb_smem<GROUP>(blk + sb_offset(BITS, GROUP, r_lo), sl);
                load_row_sb_smem<GROUP>(blk + sb_offset(BITS, GROUP, r_hi), sh2);
                uint32_t b[NB][8][2];
                load_x_frags<NB>(st + 2u * BB + (uint32_t)h * XT + xlane, b);
                if (!EXACT && (D_GROUPS == 2 || h == 0 || !two)) {  // every read of the slot is issued: release it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(empty, s));
                }
                if constexpr (EXACT)
                    mma_steps_exact<BITS, GROUP, NB>(wl, wh, sl, sh2, b, st + 2u * BB + 2u * XT + (uint32_t)h * D_XSUM,
                                                     c, acc, accg);
                else
                    mma_steps<BITS, GROUP, NB>(wl, wh, sl, sh2, b, acc);
                if (EXACT && (D_GROUPS == 2 || h == 0 || !two)) {  // the group sums are read too: release the slot
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(empty, s));
                }
                kbu -= D_GROUPS;
                while (kbu < 0) {
                    kbu += KB;
                    ++seg;
                }
            }
        }
        while (run && cur < nsegs) run = stage(cur++);
    }
    // teardown: every role has left its loop.  After an abort, no copy may
    // still be landing when the CTA exits: one thread waits for each slot a
    // producer armed, making the arrival the other producer never made (a
    // slot's phase needs both), so every wait ends once the bytes are in.
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        const int iw = sh->issued[0], ix = sh->issued[1];
        const int hi = max(iw, ix), lo = min(iw, ix);
        for (int j = max(0, hi - NS); j < hi; ++j) {
            if (j >= lo) mbar_arrive(BAR(full, j % NS));
            (void)mbar_wait(BAR(full, j % NS), (uint32_t)((j / NS) & 1));
        }
    }
#undef BAR
}

template <int BITS, int GROUP, bool EXACT>
cudaError_t launch_bge(const DecParams& p, const CUtensorMap& map, int grid, cudaStream_t st) {
    if (p.M > 8) return launch_pdl(decode_kernel<BITS, GROUP, 2, EXACT>, grid, D_THREADS, (size_t)D_SMEM, st, p, map);
    return launch_pdl(decode_kernel<BITS, GROUP, 1, EXACT>, grid, D_THREADS, (size_t)D_SMEM, st, p, map);
}
template <int BITS, int GROUP>
cudaError_t launch_bg(const DecParams& p, const CUtensorMap& map, int grid, cudaStream_t st, bool exact) {
    return exact ? launch_bge<BITS, GROUP, true>(p, map, grid, st) : launch_bge<BITS, GROUP, false>(p, map, grid, st);
}

template <int BITS>
cudaError_t launch_b(int group, const DecParams& p, const CUtensorMap& map, int grid, cudaStream_t st, bool exact) {
    if (group == 32) return launch_bg<BITS, 32>(p, map, grid, st, exact);
    if (group == 64) return launch_bg<BITS, 64>(p, map, grid, st, exact);
    return launch_bg<BITS, 128>(p, map, grid, st, exact);
}

// The kernel's shared-memory limit, the largest shared-memory carveout (two
// CTAs of 112 KB per SM), and how many CTAs of it an SM holds (min over the
// instantiations, which differ only in registers).
template <int BITS, int GROUP, int NB, bool EXACT>
cudaError_t allow_bgn(int* per_sm) {
    auto* k = decode_kernel<BITS, GROUP, NB, EXACT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)D_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, D_THREADS, (size_t)D_SMEM);
    if (e != cudaSuccess) return e;
    *per_sm = min(*per_sm, n);
    return cudaSuccess;
}
template <int BITS, int GROUP>
cudaError_t allow_bg(int* per_sm) {
    for (cudaError_t e : {allow_bgn<BITS, GROUP, 1, false>(per_sm), allow_bgn<BITS, GROUP, 2, false>(per_sm),
                          allow_bgn<BITS, GROUP, 1, true>(per_sm), allow_bgn<BITS, GROUP, 2, true>(per_sm)})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

template <int BITS>
cudaError_t allow_b(int* per_sm) {
    for (cudaError_t e : {allow_bg<BITS, 32>(per_sm), allow_bg<BITS, 64>(per_sm), allow_bg<BITS, 128>(per_sm)})
        if (e != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace

static long long g_fault_wait = 0;  // affqmm_test_fault_wait

int64_t decode_fault_wait() { return __atomic_load_n(&g_fault_wait, __ATOMIC_RELAXED); }

void decode_set_fault_wait(int64_t cycles) { __atomic_store_n(&g_fault_wait, (long long)cycles, __ATOMIC_RELAXED); }

cudaError_t decode_allow_smem(int* ctas_per_sm) {
    int n = D_CTAS_PER_SM;
    for (cudaError_t e : {allow_b<2>(&n), allow_b<3>(&n), allow_b<4>(&n), allow_b<5>(&n), allow_b<6>(&n), allow_b<8>(&n)})
        if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    *ctas_per_sm = n;
    return cudaSuccess;
}

cudaError_t launch_decode(int bits, int group, const DecParams& p, const CUtensorMap& map, int grid,
                          cudaStream_t st, bool exact) {
    switch (bits) {
        case 2: return launch_b<2>(group, p, map, grid, st, exact);
        case 3: return launch_b<3>(group, p, map, grid, st, exact);
        case 4: return launch_b<4>(group, p, map, grid, st, exact);
        case 5: return launch_b<5>(group, p, map, grid, st, exact);
        case 6: return launch_b<6>(group, p, map, grid, st, exact);
        case 8: return launch_b<8>(group, p, map, grid, st, exact);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace affqmm
