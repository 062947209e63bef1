// Host check of the stream-K partition that the tensor-core decode kernel
// takes when a fixed split has fewer (sequence, kv head) units than resident
// clusters (sk_begin and sk_cluster_of of fa_decode_internal.h, which the
// kernel and the planner call, and the planner's sk_choose_clusters of
// stream_k_plan.h).
// Built and run by tests/test_stream_k_partition.py; prints "ok <cases>" or
// the first violated property, and exits non-zero on a violation.
#include <cstdio>
#include <cstdlib>

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
        const long long units = rnd(1, 48), nv = rnd(1, 4096), most = rnd(1, 160);
        const int P = splits[rnd(0, 4)];
        const long long slots = 2 * most;
        const int G = sk_choose_clusters(units, nv, P, most, slots);
        if (G == 0) {
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
        if (G <= units || G > most || 2 * G > slots) return fail("cluster count bounds", units, nv, most, G);
        if (total / G < (long long)kChunkMinTilesPerRank * P) return fail("tiles per rank", units, nv, P, G);
        // Every cluster's range is non-empty and touches one or two units; the
        // ranges tile [0, total) in order.
        long long next = 0;
        for (int c = 0; c < G; ++c) {
            const long long g0 = sk_begin(total, G, c), g1 = sk_begin(total, G, c + 1);
            if (g0 != next || g1 <= g0) return fail("ranges tile the units", units, nv, G, c);
            next = g1;
            const long long u0 = g0 / nv, u1 = (g1 - 1) / nv;
            if (u1 - u0 > 1) return fail("more than two units in a range", units, nv, G, c);
        }
        if (next != total) return fail("ranges end at total", units, nv, G, next);
        // Every unit is shared by at most kMaxSplit clusters, and the clusters
        // touching it are exactly sk_cluster_of(first tile) .. sk_cluster_of(last tile).
        for (long long u = 0; u < units; ++u) {
            const int cf = sk_cluster_of(total, G, u * nv), cl = sk_cluster_of(total, G, (u + 1) * nv - 1);
            if (cl - cf + 1 > kMaxSplit) return fail("unit shared too widely", units, nv, G, u);
            for (int c = 0; c < G; ++c) {
                const bool touches = sk_begin(total, G, c) < (u + 1) * nv && sk_begin(total, G, c + 1) > u * nv;
                if (touches != (c >= cf && c <= cl)) return fail("touching clusters", units, nv, G, c);
            }
        }
    }
    if (cases < 1000) return fail("too few partitions exercised", cases, 0, 0, 0);
    std::printf("ok %d\n", cases);
    return 0;
}
