// plan.cu -- how a launch is cut: the decomposition of each projection's
// (tile, depth block) units into the runs of the decode and prompt kernels'
// CTAs.  Host code only; the cut depends on the projection's shape, M and the
// device's SM count, never on the data, so one input gives one answer.
#include <algorithm>
#include <cstring>

#include "affqmm_format.cuh"
#include "affqmm_internal.h"

namespace affqmm {

namespace {
// Least share (%) of the resident CTAs that a tile-aligned decode cut must
// fill: several runs per tile, or one whole tile per CTA (no merge at all).
constexpr int64_t kDecodeAlignPct = 90;
constexpr int64_t kDecodeWholePct = 75;
}  // namespace

// Decomposition of a decode launch over `count` projections (M <= 16) on a
// device with `sms` SMs holding `ctas_per_sm` decode CTAs each: each
// projection's (128-row tile, 128-deep block) units are cut into contiguous
// runs, one per CTA (the three cuts below).  The cut of one projection does
// not depend on the others in the launch.
int plan_decode(int sms, int ctas_per_sm, int count, const affqmm_weight* ws, int64_t M, DecodePlan* plan) {
    std::memset(&plan->p, 0, sizeof(plan->p));
    const int64_t K = ws[0].K;
    const int KB = (int)((K + KBLK - 1) / KBLK);
    DecParams& p = plan->p;
    p.nproj = count;
    p.KB = KB;
    p.K = K;
    p.M = (int32_t)M;
    p.fault_wait = decode_fault_wait();
    const int64_t resident = (int64_t)sms * ctas_per_sm;
    int64_t ctas = 0, tiles_total = 0;
    for (int i = 0; i < count; ++i) {
        DecProj& P = p.proj[i];
        P.N = ws[i].N;
        P.packed = static_cast<const uint8_t*>(ws[i].packed);
        const int64_t tiles = (ws[i].N + TILE_N - 1) / TILE_N;
        P.tiles = (int32_t)tiles;
        P.units = (int32_t)(tiles * KB);
        P.nctas = (int32_t)std::min<int64_t>(resident, P.units);
        // Fewer tiles than resident CTAs: when a whole number S > 1 of runs
        // per tile still fills 90 % of them, every tile is cut into S depth
        // runs, so that each run lies inside one tile (one segment, one
        // merge); when the tiles alone fill 75 %, each CTA takes one whole
        // tile (no merge at all).  Otherwise one contiguous run of units per
        // resident CTA ("stream-K").
        if (tiles > 0 && tiles < resident) {
            const int64_t S = std::min<int64_t>(resident / tiles, KB);
            if (S > 1 && tiles * S * 100 >= resident * kDecodeAlignPct)
                P.nctas = (int32_t)(tiles * S);
            else if (tiles * 100 >= resident * kDecodeWholePct)
                P.nctas = (int32_t)tiles;
        }
        P.cta_begin = (int32_t)ctas;
        P.ctr_begin = (int32_t)tiles_total;
        P.slot_begin = (int32_t)(2 * ctas);
        ctas += P.nctas;
        tiles_total += tiles;
    }
    if (kDecCountersPerTile * tiles_total > (int64_t)kMaxCounters) return AFFQMM_E_SHAPE;
    plan->grid = (int)ctas;
    plan->ws_bytes = ctas > 0 ? kSlotsOffset + (size_t)(2 * ctas) * kDecSlotFloats * sizeof(float) : 0;
    return AFFQMM_OK;
}



// Decomposition of a prompt launch (M <= 128 rows) on a device with `sms`
// SMs: each projection's (256-row tile, block) units are cut into contiguous
// runs, one per CTA (one CTA per SM).
int plan_prompt(int sms, int count, const affqmm_weight* ws, int64_t M, PromptPlan* plan) {
    std::memset(&plan->p, 0, sizeof(plan->p));
    PromptParams& p = plan->p;
    const int bits = ws[0].bits, group = ws[0].group;
    const int64_t K = ws[0].K;
    const int KB = (int)((K + KBLK - 1) / KBLK);
    p.nproj = count;
    p.KB = KB;
    p.K = K;
    p.M = (int32_t)M;
    p.block_bytes = block_bytes(bits, group);
    p.group = group;
    int64_t ctas = 0, tiles_total = 0;
    for (int i = 0; i < count; ++i) {
        PromptProj& P = p.proj[i];
        P.N = ws[i].N;
        P.packed = static_cast<const uint8_t*>(ws[i].packed);
        P.ltiles = (int32_t)((ws[i].N + TILE_N - 1) / TILE_N);
        const int64_t tiles = (ws[i].N + kPromptTileN - 1) / kPromptTileN;
        P.tiles = (int32_t)tiles;
        P.units = (int32_t)(tiles * KB);
        // Fewer tiles than SMs: every tile is cut into the same number S of
        // depth runs and the grid is tiles x S CTAs, so that each run lies
        // inside one tile (one segment, one partial, no pipeline drain in the
        // middle of a run).  Otherwise one contiguous run of units per SM.
        if (tiles > 0 && tiles < sms)
            P.nctas = (int32_t)(tiles * std::min<int64_t>(sms / tiles, KB));
        else
            P.nctas = (int32_t)std::min<int64_t>(sms, P.units);
        P.cta_begin = (int32_t)ctas;
        P.ctr_begin = (int32_t)tiles_total;
        P.slot_begin = (int32_t)(2 * ctas);
        ctas += P.nctas;
        tiles_total += tiles;
    }
    if (tiles_total > 65535) return AFFQMM_E_SHAPE;  // one merge-kernel grid row per 256-row tile
    plan->grid = (int)ctas;
    plan->ws_bytes = ctas > 0 ? kSlotsOffset + (size_t)(2 * ctas) * kPromptSlotFloats * sizeof(float) : 0;
    return AFFQMM_OK;
}

}  // namespace affqmm
