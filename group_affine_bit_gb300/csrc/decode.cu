// decode.cu -- the memory-bound projection for M = 1..16 activation rows.
//
// y[m, n] = bf16( sum_k x[m, k] * bf16(s * q[n, k] + b) ), fp32 sums.
//
// At M <= 16 the work is a stream of packed weights: every byte is read once
// and the dequantization arithmetic (three bf16x2 operations per two weights)
// is what the SMs must keep up with.  The dot products go through the warp-
// level matrix instruction (mma.sync m16n8k16, bf16 in, fp32 accumulate) with
// the weights as the A fragment straight from the registers that rounded
// them, so nothing is written back to shared or tensor memory and no warp
// waits on another warp's arithmetic: one instruction does the 256
// multiply-adds of 16 rows x 16 k for up to 8 activation rows, where fp32
// FMAs on the CUDA cores would cost one instruction per weight and row.
//
// Per CTA (two per SM), one ring of slots, each holding two consecutive
// blocks of the run (9 KB each at 4 bits, group 64) and their two activation
// tiles:
//   * one producer thread fills a slot's blocks with one 1-D bulk copy, and
//     another loads the slot's activation tiles -- M rows x 136 k, 272 bytes a
//     row so that the eight rows of a matrix load sit on distinct banks --
//     with TMA into tiles whose rows M..15 stay zero;
//   * eight consumer warps each own 16 rows of every block: thread t (group
//     g = t/4, class c = t mod 4) reads class c's code words of rows g and
//     g + 8 and the rows' scale/bias words (affqmm_format.cuh), loads the
//     activation fragments with ldmatrix, releases the slot after its last
//     read, and for each of the 8 16-deep steps rounds four weight pairs --
//     bf16(fma(s, q, b)), one rounding -- and issues one mma (two when M > 8)
//     into fp32 registers.
// At the launch's start a CTA requests two slots' weights and waits for the
// first to land before it requests the rest of its ring, so that the first
// slots of all CTAs are not queued behind everyone's later ones.
// The exact-codes instantiation (the pages' lane projection) puts the exact
// codes into the A fragments and adds s * sum(q x) + b * sum(x) per group;
// each group's sum of x comes from one more mma per step with an A fragment
// of ones, or from the sums that the kernel producing x wrote (copied into
// the slot with cp.async).
// The GeGLU form treats the projection as a gate/up stack whose rows are
// interleaved in 16-row blocks: the two warps of a pair own a gate block and
// its up block; for a whole tile they meet in shared memory, for a cut tile
// they count in on one counter; the gate warp, or the last to arrive, stores
// h = gelu_approx(gate) * up as bf16 operations.
// Work split: the projection's blocks, numbered tile-major, are cut into one
// contiguous run per CTA; how many runs (one whole tile each, a whole number
// per tile, or an even cut of all blocks, "stream-K") is the launch planner's
// choice (plan.cu).  A tile cut by run boundaries gets one
// fp32 partial per run; the last warp to arrive (an atomic counter per tile
// and 16-row group, no waiting) adds them in run order and resets the
// counter.  The run that holds a tile's first blocks reaches them at its
// end, usually after the other runs have counted in: it then adds their
// partials to its own registers at once.  The cut depends only on the projection, M and the device, so the
// same inputs give the same bits on every call, alone or stacked.  Every
// wait is on an mbarrier with a bound; a wait that gives up sets the
// workspace status word and an abort flag, and every role finishes.
// Prior art: the reg variant of the lane projection on the "Gemma 4 12B on the
// native Metal engine" page (4-bit groups held in registers for the
// matrix-op, K split per shape); unlike it, every weight is rounded to bf16
// before the contraction, as that page's prompt GEMM does.
#include <cuda_bf16.h>

#include <cstddef>
#include <type_traits>

#include "affqmm_async.cuh"
#include "affqmm_format.cuh"
#include "affqmm_internal.h"
#include "affqmm_tc.cuh"

namespace affqmm {
namespace {

constexpr int D_CWARPS = 8;                   // consumer warp w owns rows 16w .. 16w + 15 of every block
constexpr int D_WPROD = D_CWARPS;             // weights producer warp
constexpr int D_XPROD = D_CWARPS + 1;         // activations producer warp
constexpr int D_THREADS = (D_CWARPS + 2) * 32;
constexpr int D_CTAS_PER_SM = 2;
constexpr int D_FILL_GATE = 2;                // weight slots a CTA requests before its first has landed
constexpr uint32_t D_XROW = 272;              // bytes per activation row of a tile (128 k + 8 of padding)
constexpr int D_SLOTS_MAX = 16;
constexpr uint32_t D_SMEM = 110u * 1024u;     // dynamic shared memory per CTA
constexpr uint32_t D_XCHG0 = 1024u;           // the GeGLU pair exchange area starts here; the barriers sit below
constexpr uint32_t D_XCHG_PAIR = 32u * 8u * 4u;  // one warp's sums: 32 lanes x up to 8 fp32
constexpr uint32_t D_RING0 = D_XCHG0 + 4u * D_XCHG_PAIR;   // the ring starts here

// A ring slot holds two consecutive blocks of the run (contiguous in memory:
// one bulk copy) and their two activation tiles.  Its full barrier waits for
// both producers' bytes; its empty barrier for every consumer warp.
struct DecSmem {
    uint64_t full[D_SLOTS_MAX];
    uint64_t empty[D_SLOTS_MAX];
    uint64_t never;      // completed by nothing: the fault_wait test hook waits on it
    uint64_t xfull[4];   // GeGLU: warp 2i + 1 has put its up sums of a whole tile in the exchange area (1)
    uint64_t xempty[4];  // GeGLU: warp 2i has read them (1)
    int issued[2];       // slots armed by the weights producer [0] and the activation producer [1]
    int abort_flag;
};
static_assert(sizeof(DecSmem) <= D_XCHG0, "barriers fit below the exchange area");

template <int NB>
constexpr uint32_t x_tile_bytes() { return 8u * NB * D_XROW; }  // 8 rows per activation block of the mma
constexpr uint32_t D_XSUM = 256;  // per block, exact-codes mode: sums of x over each group, [4 groups][16 rows] fp32
template <int BITS, int GROUP, int NB>
constexpr uint32_t slot_bytes() {
    return 2u * (uint32_t)block_bytes(BITS, GROUP) + 2u * x_tile_bytes<NB>() + 2u * D_XSUM;
}
template <int BITS, int GROUP, int NB>
constexpr int ring_slots() {
    return (int)((D_SMEM - 128u - D_RING0) / slot_bytes<BITS, GROUP, NB>()) > D_SLOTS_MAX
               ? D_SLOTS_MAX
               : (int)((D_SMEM - 128u - D_RING0) / slot_bytes<BITS, GROUP, NB>());
}

__device__ __forceinline__ void sts_zero16(uint32_t a) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
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
// sum_k q x in accg and, against an A fragment of ones, sum_k x in accx (the
// same value in every weight row), and at the group's end
//     acc += s_row * accg + b_row * (sum of x over the group)
// with the sum of x from accx, or, when the kernel that produced x wrote the
// sums (given), from xs (fp32 [group][16 rows] in the slot).  sl/sh hold the
// rows' s | b << 16 words.
template <int BITS, int GROUP, int NB, int S = 0>
__device__ __forceinline__ void mma_steps_exact(const uint32_t* wl, const uint32_t* wh, const uint32_t* sl,
                                                const uint32_t* sh, const uint32_t (&b)[NB][8][2], uint32_t xs,
                                                bool given, int c, float* acc, float* accg, float* accx) {
    if constexpr (S < 8) {
        constexpr int P0 = plane0_bits(BITS);
        const uint32_t a0 = class_code_pair<BITS, 2 * S>(wl, wl + P0);
        const uint32_t a1 = class_code_pair<BITS, 2 * S>(wh, wh + P0);
        const uint32_t a2 = class_code_pair<BITS, 2 * S + 1>(wl, wl + P0);
        const uint32_t a3 = class_code_pair<BITS, 2 * S + 1>(wh, wh + P0);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            mma_bf16(accg + 4 * nb, a0, a1, a2, a3, b[nb][S][0], b[nb][S][1]);
            mma_bf16(accx + 4 * nb, BF2_ONE, BF2_ONE, BF2_ONE, BF2_ONE, b[nb][S][0], b[nb][S][1]);
        }
        constexpr int SPG = GROUP / 16;  // 16-deep steps per group
        if constexpr ((S + 1) % SPG == 0) {
            constexpr int GI = S / SPG;
            const float s_lo = __uint_as_float(sl[GI] << 16), b_lo = __uint_as_float(sl[GI] & 0xFFFF0000u);
            const float s_hi = __uint_as_float(sh[GI] << 16), b_hi = __uint_as_float(sh[GI] & 0xFFFF0000u);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                float x0 = accx[4 * nb], x1 = accx[4 * nb + 1];  // activation rows 8nb + 2c, 8nb + 2c + 1
                if (given) {
                    uint32_t x0u, x1u;
                    lds_v2(xs + (uint32_t)(GI * 16 + 8 * nb + 2 * c) * 4u, x0u, x1u);
                    x0 = __uint_as_float(x0u);
                    x1 = __uint_as_float(x1u);
                }
                float* a = acc + 4 * nb;
                float* q = accg + 4 * nb;
                a[0] = fmaf(b_lo, x0, fmaf(s_lo, q[0], a[0]));
                a[1] = fmaf(b_lo, x1, fmaf(s_lo, q[1], a[1]));
                a[2] = fmaf(b_hi, x0, fmaf(s_hi, q[2], a[2]));
                a[3] = fmaf(b_hi, x1, fmaf(s_hi, q[3], a[3]));
                q[0] = q[1] = q[2] = q[3] = 0.f;
                accx[4 * nb] = accx[4 * nb + 1] = accx[4 * nb + 2] = accx[4 * nb + 3] = 0.f;
            }
        }
        mma_steps_exact<BITS, GROUP, NB, S + 1>(wl, wh, sl, sh, b, xs, given, c, acc, accg, accx);
    }
}

// 4-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on `bar` once every earlier cp.async of this thread has completed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
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

// The run's partial of a tile for this thread: activation rows m (e & 1 and
// e >> 2 pick 8 nb + 2c + ...), weight rows r_lo (e & 2 == 0) or r_hi.
__device__ __forceinline__ int acc_m(int e, int c) { return 8 * (e >> 2) + 2 * c + (e & 1); }

// Add the partials of runs cf .. cl of a tile (slot of run cb: two per CTA,
// the first for the segment that starts its run) for this thread's
// activation rows m < M and weight rows rows[e], in run order; `mine` stands
// for run `me`.  Four runs' loads are issued before their adds, so a merge
// over R runs costs about R / 4 round trips to L2.
template <int NB>
__device__ __forceinline__ void add_runs(const DecParams& p, const DecProj& P, int t0, int cf, int cl, int U, int PC,
                                         int me, const float* mine, const int* rows, int M, int c, float* sum) {
#pragma unroll
    for (int e = 0; e < 4 * NB; ++e) sum[e] = 0.f;
    for (int cb0 = cf; cb0 <= cl; cb0 += 4) {
        float q[4][4 * NB];
#pragma unroll
        for (int d = 0; d < 4; ++d) {
            const int cb = cb0 + d;
            const bool ld = cb <= cl && cb != me;
            const int b0 = (int)((int64_t)cb * U / PC);
            const int sc = P.slot_begin + 2 * cb + (b0 >= t0 ? 0 : 1);
            const float* src = p.partials + (size_t)sc * kDecSlotFloats;
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e) {
                const int m = acc_m(e, c);
                q[d][e] = (ld && m < M) ? __ldcg(src + rows[e] * 16 + m) : 0.f;
                if (cb == me) q[d][e] = mine[e];
            }
        }
#pragma unroll
        for (int d = 0; d < 4; ++d)
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e)
                if (cb0 + d <= cl) sum[e] += q[d][e];
    }
}

// End of a tile segment (the run's last block of a tile, or of the run): store
// y, or publish this run's partial and, if it is the last to arrive, add all
// runs' partials in run order.  acc[4 nb + e]: weight row (e < 2 ? lo : hi),
// activation row 8 nb + 2c + (e & 1).  In the GeGLU form (p.epi == 1) every
// segment goes through the partials: warps 2i and 2i + 1 (a gate block and
// its up block) count in on warp 2i's counter, and the last of the pair's
// arrivals over all runs stores h for both.
template <int NB>
__device__ __forceinline__ void segment_end(const DecParams& p, const DecProj& P, float* acc, int tile, bool whole,
                                            bool first_seg, int cta, int U, int PC, int KB, int M, int warp,
                                            int lane, int r_lo, int c, uint32_t xchg, uint32_t xfull,
                                            uint32_t xempty, int& nxchg, volatile int* abort_flag) {
    const int r_hi = r_lo + 8;
    const int64_t n_lo = (int64_t)tile * TILE_N + r_lo;
    const bool geglu = p.epi != 0;
    if (whole && geglu) {
        // The pair's sums of a whole tile meet in shared memory: warp 2i + 1
        // (up rows) puts its sums there, warp 2i (gate rows, the same lanes)
        // takes them and stores h.
        const uint32_t a = xchg + (uint32_t)lane * 32u;
        const uint32_t ph = (uint32_t)(nxchg++ & 1);
        if (warp & 1) {
            if (!__all_sync(0xffffffffu, wait_or_abort(xempty, ph ^ 1u, abort_flag, p.status))) return;
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e)
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(a + 4u * e), "f"(acc[e]) : "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(xfull);
        } else {
            if (!__all_sync(0xffffffffu, wait_or_abort(xfull, ph, abort_flag, p.status))) return;
            float up[4 * NB];
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e) {
                uint32_t v;
                lds_v1(a + 4u * e, v);
                up[e] = __uint_as_float(v);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xempty);
            const int64_t F = P.N / 2;
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e) {
                const int m = acc_m(e, c);
                const int64_t n = n_lo + ((e & 2) ? 8 : 0);   // a gate row: 32 j + (0 .. 15)
                if (m < M && n < P.N)
                    P.y[(int64_t)m * F + 16 * (n / 32) + (n % 32)] = geglu_bf16(bf16r(acc[e]), bf16r(up[e]));
            }
        }
        return;
    }
    if (whole && !geglu) {
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) {
            const int m = acc_m(e, c);
            const int64_t n = n_lo + ((e & 2) ? 8 : 0);
            if (m < M && n < P.N) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[e]));
        }
        return;
    }
    const int t0 = tile * KB, t1 = t0 + KB - 1;
    const int cf = run_of(t0, U, PC), cl = run_of(t1, U, PC);
    // A run reaches the tile that begins inside it only at its very end, while
    // the later runs of that tile had it at their start: when they have all
    // counted in already, this warp adds their partials and its own at once,
    // without publishing its own or counting in.
    if (!geglu && !whole && cta == cf && cf < cl && t1 > (int)((int64_t)(cta + 1) * U / PC) - 1) {
        unsigned* ctr_f = &p.counters[(size_t)(P.ctr_begin + tile) * D_CWARPS + warp];
        unsigned cnt = 0;
        if (lane == 0) cnt = ld_acquire_gpu(ctr_f);
        cnt = __shfl_sync(0xffffffffu, cnt, 0);
        if (cnt == (unsigned)(cl - cf)) {
            fence_acq_rel_gpu();
            int rows[4 * NB];
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e) rows[e] = (e & 2) ? r_hi : r_lo;
            float sum[4 * NB];
            add_runs<NB>(p, P, t0, cf, cl, U, PC, cta, acc, rows, M, c, sum);
#pragma unroll
            for (int e = 0; e < 4 * NB; ++e) {
                const int m = acc_m(e, c);
                const int64_t n = n_lo + ((e & 2) ? 8 : 0);
                if (m < M && n < P.N) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum[e]));
            }
            __syncwarp();
            if (lane == 0) *ctr_f = 0u;
            return;
        }
    }
    const int slot = P.slot_begin + 2 * cta + (first_seg ? 0 : 1);
    float* sp = p.partials + (size_t)slot * kDecSlotFloats;
#pragma unroll
    for (int e = 0; e < 4 * NB; ++e) {
        const int m = acc_m(e, c);
        const int r = (e & 2) ? r_hi : r_lo;
        if (m < M) __stcg(sp + r * 16 + m, acc[e]);
    }
    fence_acq_rel_gpu();  // every lane's partial is visible GPU-wide before the arrival
    __syncwarp();
    const int cw = geglu ? (warp & ~1) : warp;      // the counter this warp arrives on
    unsigned prev = 0;
    unsigned* ctr = &p.counters[(size_t)(P.ctr_begin + tile) * D_CWARPS + cw];
    if (lane == 0) prev = atom_add_acq_rel(ctr, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    const unsigned arrivals = (unsigned)(cl - cf + 1) * (geglu ? 2u : 1u);
    if (prev != arrivals - 1u) return;
    fence_acq_rel_gpu();  // the last arrival: every lane reads the other runs' partials after it
    if (!geglu) {
        int rows[4 * NB];
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) rows[e] = (e & 2) ? r_hi : r_lo;
        float sum[4 * NB];
        add_runs<NB>(p, P, t0, cf, cl, U, PC, cta, acc, rows, M, c, sum);
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) {
            const int m = acc_m(e, c);
            const int64_t n = n_lo + ((e & 2) ? 8 : 0);
            if (m < M && n < P.N) P.y[(int64_t)m * P.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum[e]));
        }
    } else {
        // gate rows of warp cw, up rows of warp cw + 1; this warp's own values
        // come from the slot (both warps of the pair stored theirs above)
        const int g_lo = 16 * cw + (lane >> 2), u_lo = g_lo + 16;
        int rg[4 * NB], ru[4 * NB];
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) {
            rg[e] = (e & 2) ? g_lo + 8 : g_lo;
            ru[e] = (e & 2) ? u_lo + 8 : u_lo;
        }
        float gs[4 * NB], us[4 * NB];
        add_runs<NB>(p, P, t0, cf, cl, U, PC, -1, nullptr, rg, M, c, gs);
        add_runs<NB>(p, P, t0, cf, cl, U, PC, -1, nullptr, ru, M, c, us);
        const int64_t F = P.N / 2;
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) {
            const int m = acc_m(e, c);
            const int64_t n = (int64_t)tile * TILE_N + rg[e];   // a gate row: 32 j + (0 .. 15)
            if (m < M && n < P.N)
                P.y[(int64_t)m * F + 16 * (n / 32) + (n % 32)] = geglu_bf16(bf16r(gs[e]), bf16r(us[e]));
        }
    }
    __syncwarp();
    if (lane == 0) *ctr = 0u;
}

template <int BITS, int GROUP, int NB, bool EXACT>
__global__ void __launch_bounds__(D_THREADS, D_CTAS_PER_SM)
    decode_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap xmap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    constexpr int BB = block_bytes(BITS, GROUP);
    constexpr int SBW = sb_words(GROUP);
    constexpr uint32_t XT = x_tile_bytes<NB>();
    constexpr uint32_t SLOT = slot_bytes<BITS, GROUP, NB>();
    constexpr int NS = ring_slots<BITS, GROUP, NB>();
    static_assert(BB % 16 == 0 && SLOT % 128 == 0, "bulk copies move multiples of 16 bytes; tiles 128-aligned");
    static_assert(NS >= 2, "at least two ring slots");
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sh_addr = (raw + 127u) & ~127u;
    DecSmem* sh = reinterpret_cast<DecSmem*>(smem_raw + (sh_addr - raw));
    const uint32_t ring = sh_addr + D_RING0;  // slot s: two weight blocks, then two activation tiles
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
    const int nblk = u1 - u0;
    const int npairs = (nblk + 1) / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(BAR(full, s), (EXACT && p.xsums != nullptr) ? 3 : 2);  // both producers (and the sums' copies)
            mbar_init(BAR(empty, s), D_CWARPS);  // every consumer warp
        }
        mbar_init(BAR(never, 0), 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(BAR(xfull, i), 1);
            mbar_init(BAR(xempty, i), 1);
        }
        sh->issued[0] = sh->issued[1] = 0;
        sh->abort_flag = 0;
        fence_mbar_init();
    }
    // Activation rows M..8NB-1 (and their group sums) stay zero for the whole
    // launch: the producers write rows 0..M-1 only (the tensor map's box is M
    // rows).
    for (int s = 0; s < NS; ++s)
        for (uint32_t off = 16u * threadIdx.x; off < 2u * XT + 2u * D_XSUM; off += 16u * D_THREADS)
            sts_zero16(ring + (uint32_t)s * SLOT + 2u * BB + off);
    fence_proxy_async_smem();  // generic-proxy zeros -> TMA writes
    __syncthreads();
    volatile int* abort_flag = &sh->abort_flag;
    if (threadIdx.x == 0) pdl_launch_dependents();

    if (warp == D_WPROD || warp == D_XPROD) {
        // ---------------------------------------------------------- producers
        // The weights never depend on an earlier kernel, so their producer
        // starts before the grid dependency is resolved; the activations may
        // come from the previous kernel.
        if (lane == 0) {
            const bool wprod = warp == D_WPROD;
            const uint64_t policy = policy_evict_first();  // the weights are read once
            if (!wprod) {
                prefetch_tmap(&xmap);
                pdl_wait();
            }
            int issued = 0;
            for (int j = 0; j < npairs; ++j) {
                const int s = j % NS;
                if (!wait_or_abort_lazy(BAR(empty, s), (uint32_t)((j / NS) & 1) ^ 1u, abort_flag, p.status)) break;
                // Launch start: every CTA would ask for its whole ring at once;
                // the weights past the first D_FILL_GATE slots wait until the
                // first slot has landed, so that each CTA's first slot is not
                // queued behind the other CTAs' later ones.  (Slot 0 has
                // completed at most its first phase here: its refill is pair NS.)
                if (wprod && j == D_FILL_GATE && D_FILL_GATE < NS &&
                    !wait_or_abort_lazy(BAR(full, 0), 0u, abort_flag, p.status))
                    break;
                const int nb2 = min(2, nblk - 2 * j);
                const uint32_t st = ring + (uint32_t)s * SLOT;
                if (wprod) {
                    const uint32_t bytes = (uint32_t)nb2 * BB;
                    mbar_arrive_expect_tx(BAR(full, s), bytes);
                    bulk_g2s_hint(st, P.packed + (size_t)(u0 + 2 * j) * BB, bytes, BAR(full, s), policy);
                } else {
                    mbar_arrive_expect_tx(BAR(full, s), (uint32_t)nb2 * D_XROW * (uint32_t)M);
                    for (int h = 0; h < nb2; ++h)
                        tma_load_2d(st + 2u * BB + (uint32_t)h * XT, &xmap, ((u0 + 2 * j + h) % KB) * KBLK, 0,
                                    BAR(full, s));
                    if (EXACT && p.xsums != nullptr) {
                        // the group sums of x that x's producer wrote, 4 bytes each, into the
                        // blocks' sum areas ([group][16 rows]); past K the copies fill zeros
                        constexpr int GPB = KBLK / GROUP;
                        const int64_t G = p.K / GROUP;
                        for (int h = 0; h < nb2; ++h) {
                            const int64_t g0 = (int64_t)((u0 + 2 * j + h) % KB) * GPB;
                            const uint32_t sums = st + 2u * BB + 2u * XT + (uint32_t)h * D_XSUM;
                            for (int gi = 0; gi < GPB; ++gi)
                                for (int m = 0; m < M; ++m) {
                                    const bool in = g0 + gi < G;
                                    cp_async_4(sums + (uint32_t)(gi * 16 + m) * 4u,
                                               in ? p.xsums + (int64_t)m * G + g0 + gi : p.xsums, in ? 4u : 0u);
                                }
                        }
                        cp_async_arrive_noinc(BAR(full, s));  // arrives once these copies have landed
                    }
                }
                issued = j + 1;
            }
            sh->issued[wprod ? 0 : 1] = issued;
        }
    } else {
        // ---------------------------------------------------------- consumers
        const int g = lane >> 2, c = lane & 3;
        const int r_lo = 16 * warp + g, r_hi = r_lo + 8;  // this thread's rows within the tile
        // ldmatrix: lanes 8j .. 8j + 7 address matrix j's eight rows; matrix j
        // of a pair of steps is (step 2p + j/2, k half j mod 2)
        const uint32_t xlane = (uint32_t)(lane & 7) * D_XROW + (uint32_t)((lane >> 3) & 1) * 16u + (uint32_t)(lane >> 4) * 32u;
        // exact-codes mode: accg the current group's sum of q x, accx its sum of x
        float acc[4 * NB], accg[4 * NB], accx[4 * NB];
#pragma unroll
        for (int e = 0; e < 4 * NB; ++e) acc[e] = accg[e] = accx[e] = 0.f;
        const bool given = p.xsums != nullptr;
        pdl_wait();  // y, the partials and the counters may still be in use by the previous kernel
        // Test hook: wait, bounded by p.fault_wait cycles, on a barrier that
        // nothing completes; the wait runs out, sets the status word and the
        // abort flag, and the CTA finishes without output.
        const bool run = p.fault_wait <= 0 ||
                         __all_sync(0xffffffffu, wait_or_abort_within(BAR(never, 0), 0u, abort_flag, p.status,
                                                                      p.fault_wait));
        int kb = u0 % KB, tile = u0 / KB, seg_start = u0;
        int nxchg = 0;  // whole tiles exchanged through shared memory (GeGLU form)
        for (int j = 0; run && j < npairs; ++j) {
            const int s = j % NS;
            if (!__all_sync(0xffffffffu, wait_or_abort(BAR(full, s), (uint32_t)((j / NS) & 1), abort_flag, p.status)))
                break;
            const uint32_t st = ring + (uint32_t)s * SLOT;
            const bool pair = 2 * j + 1 < nblk;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h == 1 && !pair) break;
                const uint32_t blk = st + (uint32_t)h * BB;
                uint32_t wl[BITS], wh[BITS], sl[SBW], sh2[SBW];
                load_class_words_smem<BITS>(blk, r_lo, c, wl);
                load_class_words_smem<BITS>(blk, r_hi, c, wh);
                load_row_sb_smem<GROUP>(blk + sb_offset(BITS, GROUP, r_lo), sl);
                load_row_sb_smem<GROUP>(blk + sb_offset(BITS, GROUP, r_hi), sh2);
                uint32_t b[NB][8][2];
                load_x_frags<NB>(st + 2u * BB + (uint32_t)h * XT + xlane, b);
                if (!EXACT && (h == 1 || !pair)) {  // every read of the slot is issued: release it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(empty, s));
                }
                if constexpr (EXACT)
                    mma_steps_exact<BITS, GROUP, NB>(wl, wh, sl, sh2, b, st + 2u * BB + 2u * XT + (uint32_t)h * D_XSUM,
                                                     given, c, acc, accg, accx);
                else
                    mma_steps<BITS, GROUP, NB>(wl, wh, sl, sh2, b, acc);
                if (EXACT && (h == 1 || !pair)) {  // the group sums are read too: release the slot
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(empty, s));
                }
                const int u = u0 + 2 * j + h;
                if (kb == KB - 1 || u == u1 - 1) {  // this block ends a tile segment
                    segment_end<NB>(p, P, acc, tile, (seg_start == tile * KB) && (kb == KB - 1), seg_start == u0, cta,
                                    U, PC, KB, M, warp, lane, r_lo, c,
                                    sh_addr + D_XCHG0 + (uint32_t)(warp >> 1) * D_XCHG_PAIR, BAR(xfull, warp >> 1),
                                    BAR(xempty, warp >> 1), nxchg, abort_flag);
#pragma unroll
                    for (int e = 0; e < 4 * NB; ++e) acc[e] = 0.f;
                    seg_start = u + 1;
                }
                if (++kb == KB) {
                    kb = 0;
                    ++tile;
                }
            }
        }
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
// CTAs of 110 KB per SM), and how many CTAs of it an SM holds (min over the
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
