// Host check of the stream-K partition that the tensor-core decode kernel
// takes with a fixed split when whole (sequence, kv head) units would leave
// resident clusters idle (sk_begin and sk_cluster_of of fa_decode_internal.h,
// which the kernel and the planner call, and the planner's
// sk_choose_clusters of stream_k_plan.h), and the scratch slots that the
// merge of a unit shared by several clusters uses (splitk_combine.cuh).
// Built and run by tests/test_stream_k_partition.py; prints "ok <cases>" or
// the first violated property, and exits non-zero on a violation.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "stream_k_plan.h"

using namespace fad;

static int fail(const char* what, long long a, long long b, long long c, long long d)
{
    std::printf("FAIL %s (%lld %lld %lld %lld)\n", what, a, b, c, d);
    return 1;
}

int main()
{
    // sk_cluster_of(x) is the cluster whose range [sk_begin(c), sk_begin(c + 1)) holds x.
    for (int G = 1; G <= 40; ++G)
        for (long long total = G; total <= 400; total += 7)
            for (long long x = 0; x < total; ++x) {
                const int c = sk_cluster_of(total, G, x);
                if (c < 0 || c >= G || sk_begin(total, G, c) > x || sk_begin(total, G, c + 1) <= x)
                    return fail("cluster_of", G, total, x, c);
            }
    unsigned long long seed = 12345;
    auto rnd = [&](long long lo, long long hi) {
        seed = seed * 6364136223846793005ull + 1442695040888963407ull;
        return lo + (long long)((seed >> 33) % (unsigned long long)(hi - lo + 1));
    };
    const int splits[5] = {1, 2, 4, 8, 16};
    int cases = 0;
    for (int trial = 0; trial < 20000; ++trial) {
        const long long units = (trial & 1) ? rnd(1, 48) : rnd(1, 400), nv = rnd(1, 4096), most = rnd(1, 160);
        const int P = splits[rnd(0, 4)];
        const long long slots = 2 * most;
        const int G = sk_choose_clusters(units, nv, P, most, slots);
        if (G == 0) {
            // At least as many units as clusters: refused only when whole rounds
            // stay within 5/4 of an equal share or ranks would keep too few tiles.
            if (units >= most) {
                const long long rounds = (units + most - 1) / most, share = (units * nv + most - 1) / most;
                if (4 * rounds * nv > 5 * share && units * nv / (most * P) >= kChunkMinTilesPerRank)
                    return fail("many-unit partition refused", units, nv, P, most);
            }
            // Not taken: no idle clusters, or already the largest admissible count <= units.
            if (units < most && units * nv / ((long long)kChunkMinTilesPerRank * P) > units) {
                // every count in (units, min(most, total / 4P)] must share some unit more than kMaxSplit ways
                long long top = units * nv / ((long long)kChunkMinTilesPerRank * P);
                if (top > most) top = most;
                const long long total = units * nv;
                for (long long g = units + 1; g <= top; ++g) {
                    int widest = 0;
                    for (long long u = 0; u < units; ++u) {
                        const int n = sk_cluster_of(total, (int)g, (u + 1) * nv - 1) - sk_cluster_of(total, (int)g, u * nv) + 1;
                        if (n > widest) widest = n;
                    }
                    if (widest <= kMaxSplit) return fail("admissible count refused", units, nv, P, g);
                }
            }
            continue;
        }
        ++cases;
        const long long total = units * nv;
        if (units < most && (G <= units || G > most)) return fail("cluster count bounds", units, nv, most, G);
        if (units >= most && G != most) return fail("every resident cluster", units, nv, most, G);
        if (units >= most && 4 * ((units + most - 1) / most) * nv <= 5 * ((total + most - 1) / most))
            return fail("balanced rounds taken over", units, nv, most, G);
        if (2 * G > slots) return fail("scratch slots", units, nv, most, G);
        if (total / G < (long long)kChunkMinTilesPerRank * P) return fail("tiles per rank", units, nv, P, G);
        // Every cluster's range is non-empty and touches one or two units; the
        // ranges tile [0, total) in order.
        long long next = 0;
        for (int c = 0; c < G; ++c) {
            const long long g0 = sk_begin(total, G, c), g1 = sk_begin(total, G, c + 1);
            if (g0 != next || g1 <= g0) return fail("ranges tile the units", units, nv, G, c);
            next = g1;
            const long long u0 = g0 / nv, u1 = (g1 - 1) / nv;
            if (units < most && u1 - u0 > 1) return fail("more than two units in a range", units, nv, G, c);
        }
        if (next != total) return fail("ranges end at total", units, nv, G, next);
        // Every unit is shared by at most kMaxSplit clusters, and the clusters
        // touching it are exactly sk_cluster_of(first tile) .. sk_cluster_of(last tile).
        for (long long u = 0; u < units; ++u) {
            const int cf = sk_cluster_of(total, G, u * nv), cl = sk_cluster_of(total, G, (u + 1) * nv - 1);
            if (cl - cf + 1 > kMaxSplit) return fail("unit shared too widely", units, nv, G, u);
            if (units >= most && cl - cf > 1) return fail("unit shared by more than two", units, nv, G, u);
            for (int c = 0; c < G; ++c) {
                const bool touches = sk_begin(total, G, c) < (u + 1) * nv && sk_begin(total, G, c + 1) > u * nv;
                if (touches != (c >= cf && c <= cl)) return fail("touching clusters", units, nv, G, c);
            }
        }
        // Scratch slots of the shared units (the merge's rule): cluster c's
        // chunk of unit u sits at 2c, or 2c + 1 when c is the unit's first
        // cluster and its range began in an earlier unit; the unit's count
        // sits at its first cluster's slot. Every (cluster, unit) pair gets a
        // slot of its own below 2G.
        std::vector<int> used(2 * G, 0);
        for (long long u = 0; u < units; ++u) {
            const int cf = sk_cluster_of(total, G, u * nv), cl = sk_cluster_of(total, G, (u + 1) * nv - 1);
            if (cl == cf) continue;
            const int first_second = sk_begin(total, G, cf) < u * nv ? 1 : 0;
            for (int c = cf; c <= cl; ++c) {
                const long long slot = 2LL * c + (c == cf ? first_second : 0);
                if (slot < 0 || slot >= 2 * G || used[slot]++) return fail("scratch slot reused", units, nv, G, slot);
            }
        }
    }
    if (cases < 1000) return fail("too few partitions exercised", cases, 0, 0, 0);
    std::printf("ok %d\n", cases);
    return 0;
}
