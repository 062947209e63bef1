// stream_k_plan.h -- host-side choice of the stream-K partition (the planner
// in fa_decode_host.cu; no device code includes this file).
#pragma once

#include "fa_decode_internal.h"

namespace fad {

// Clusters of the stream-K partition for `units` units of `nv` tiles each
// (cluster size P, at most `most` clusters resident, `slots` scratch slots of
// two per cluster), or 0 when it does not apply.
//  - Fewer units than resident clusters: the resident clusters, fewer while a
//    rank would keep fewer than kChunkMinTilesPerRank tiles or a unit would be
//    shared by more than kMaxSplit clusters.
//  - At least as many: every resident cluster, when whole-unit rounds would
//    give a cluster more than 5/4 of an equal share of the tiles (the shared
//    units' merge through global memory and the partial units' start-up cost
//    more than smaller imbalances; measured on 128 units of 32 tiles over 36
//    clusters: 4 rounds beat the equal share). Each cluster's range then spans
//    at least one unit's worth of tiles, so a unit is shared by at most two
//    clusters.
inline int sk_choose_clusters(int64_t units, int64_t nv, int P, int64_t most, int64_t slots)
{
    if (units < 1 || nv < 1 || nv > INT32_MAX || most < 1) return 0;
    const int64_t total = units * nv;
    if (units >= most) {
        const int64_t rounds = (units + most - 1) / most, share = (total + most - 1) / most;
        if (4 * rounds * nv <= 5 * share || total / (most * P) < kChunkMinTilesPerRank) return 0;
        return 2 * most <= slots ? (int)most : 0;
    }
    int64_t G = total / ((int64_t)kChunkMinTilesPerRank * P);
    if (G > most) G = most;
    for (; G > units; --G) {
        int widest = 0;
        for (int64_t u = 0; u < units; ++u) {
            const int n = sk_cluster_of(total, (int)G, (u + 1) * nv - 1) - sk_cluster_of(total, (int)G, u * nv) + 1;
            if (n > widest) widest = n;
        }
        if (widest <= kMaxSplit) break;
    }
    return (G > units && 2 * G <= slots) ? (int)G : 0;
}

}  // namespace fad
