// Host check of the work partition used by the kernels (rr_internal.h):
// every vector / byte is covered exactly once, in whole 256-byte granules,
// for the one-shot chunks, the two-shot owned segments and their per-block
// chunks, and the gather byte regions.  Compiled with g++ (no GPU).
#include <cstdio>
#include <vector>

#include "rr_internal.h"

using namespace rr;

static int failures = 0;
#define CHECK(c, ...)                                   \
    do {                                                \
        if (!(c)) {                                     \
            if (failures < 20) std::printf(__VA_ARGS__); \
            ++failures;                                 \
        }                                               \
    } while (0)

int main()
{
    const int64_t sizes[] = {0, 1, 15, 16, 17, 255, 256, 257, 4096, 12345, 65536 + 7, 1 << 21, 3000017};
    const int Ws[] = {1, 2, 3, 5, 8, 16};
    const int Bs[] = {1, 2, 3, 7, 19, 64, 152};
    for (int64_t n : sizes) {
        for (int B : Bs) {
            std::vector<int> cover(n, 0);
            int64_t prev = 0;
            for (int b = 0; b < B; ++b) {
                int64_t v0, v1;
                part_range(n, B, b, v0, v1);
                CHECK(v0 == prev, "part_range gap n=%lld B=%d b=%d\n", (long long)n, B, b);
                CHECK(v0 % kGranuleVec == 0 || v0 == n, "part_range unaligned start\n");
                for (int64_t v = v0; v < v1; ++v) cover[v]++;
                prev = v1;
            }
            CHECK(prev == n, "part_range does not end at n=%lld B=%d\n", (long long)n, B);
            for (int64_t v = 0; v < n; ++v) CHECK(cover[v] == 1, "part_range cover n=%lld v=%lld\n", (long long)n, (long long)v);

            std::vector<int> bcover(n, 0);
            for (int b = 0; b < B; ++b) {
                int64_t x0, x1;
                byte_region(n, B, b, x0, x1);
                CHECK(x0 % kGranuleBytes == 0 || x0 == n, "byte_region unaligned\n");
                for (int64_t x = x0; x < x1; ++x) bcover[x]++;
            }
            for (int64_t x = 0; x < n; ++x) CHECK(bcover[x] == 1, "byte_region cover n=%lld x=%lld\n", (long long)n, (long long)x);

            for (int W : Ws) {
                std::vector<int> tcover(n, 0);
                for (int c = 0; c < W; ++c) {
                    int64_t s0, s1;
                    owned_segment(n, W, c, s0, s1);
                    for (int b = 0; b < B; ++b) {
                        int64_t c0, c1;
                        owned_chunk(n, W, B, c, b, c0, c1);
                        CHECK(c0 >= s0 && c1 <= s1 && c0 <= c1, "owned_chunk outside its segment\n");
                        CHECK((c0 - s0) % kGranuleVec == 0 || c0 == c1, "owned_chunk unaligned\n");
                        for (int64_t v = c0; v < c1; ++v) tcover[v]++;
                    }
                }
                for (int64_t v = 0; v < n; ++v)
                    CHECK(tcover[v] == 1, "two-shot cover n=%lld W=%d B=%d v=%lld\n", (long long)n, W, B, (long long)v);
            }
        }
    }
    // Staged copy_mode kernel: every output vector is reduced exactly once,
    // by a block of index b after every rank's block b has published the unit
    // that staged it; a block's units stay below 2^kRoundBits.
    struct Case {
        int64_t n;
        int W, B;
        int64_t opt;
    };
    std::vector<Case> cases;
    const int64_t ssizes[] = {0, 1, 15, 16, 17, 255, 256, 257, 1023, 1024, 1025, 4096, 12345, 65543};
    const int sWs[] = {1, 2, 3, 5, 8, 16};
    const int sBs[] = {1, 2, 3, 7, 19};
    const int64_t opts[] = {0, 256, 4096, 65536};
    for (int64_t n : ssizes)
        for (int W : sWs)
            for (int B : sBs)
                for (int64_t o : opts) cases.push_back({n, W, B, o});
    cases.push_back({(1 << 21) / 8 + 3, 8, 19, 0});   // W=8, 2^21 bf16 + a few vectors
    cases.push_back({(1 << 21) + 7, 8, 19, 0});
    cases.push_back({(int64_t)40000000, 2, 1, 256});  // P grows: one block, 16-byte option
    for (const Case &cs : cases) {
        const int64_t n = cs.n;
        for (int twoshot = 0; twoshot < 2; ++twoshot) {
            const int W = cs.W, B = cs.B, nr = twoshot ? W : 1;
            std::vector<int64_t> r0(nr), r1(nr);
            for (int j = 0; j < nr; ++j) {
                if (twoshot) owned_segment(n, W, j, r0[j], r1[j]);
                else { r0[j] = 0; r1[j] = n; }
            }
            const int64_t P = staged_piece_vectors(cs.opt, r1[0] - r0[0], nr, B);
            CHECK(P % kGranuleVec == 0 && P >= kGranuleVec, "staged P=%lld not in granules\n", (long long)P);
            if (n > 4000000) continue;  // the size only checks that P grows
            // producer: the block and unit that stage each vector (same on every rank)
            std::vector<int> sb(n, -1), su(n, -1);
            for (int b = 0; b < B; ++b) {
                const int units = staged_rounds(r1[0] - r0[0], P, B, b) * nr;
                CHECK(units < (1 << kRoundBits), "staged units %d\n", units);
                for (int u = 0; u < units; ++u) {
                    int64_t ps, pe;
                    staged_piece(r0[u % nr], r1[u % nr], P, B, b, u / nr, ps, pe);
                    for (int64_t v = ps; v < pe; ++v) {
                        CHECK(sb[v] < 0, "vector %lld staged twice\n", (long long)v);
                        sb[v] = b;
                        su[v] = u;
                    }
                }
            }
            for (int64_t v = 0; v < n; ++v) CHECK(sb[v] >= 0, "vector %lld never staged n=%lld W=%d B=%d\n", (long long)v, (long long)n, W, B);
            if (cs.opt == 0 && r1[0] > r0[0]) {
                // default pieces: no block stages more than its even share of a
                // range plus a granule per round
                const int64_t len = r1[0] - r0[0];
                const int K = staged_rounds(len, P, B, 0);
                for (int b = 0; b < B; ++b) {
                    int64_t mine = 0;
                    for (int k = 0; k < staged_rounds(len, P, B, b); ++k) {
                        int64_t ps, pe;
                        staged_piece(r0[0], r1[0], P, B, b, k, ps, pe);
                        mine += pe - ps;
                    }
                    CHECK(mine <= (len + B - 1) / B + (int64_t)K * kGranuleVec,
                          "block %d stages %lld of %lld vectors over %d blocks (P=%lld)\n", b, (long long)mine,
                          (long long)len, B, (long long)P);
                }
            }
            const int nouts[] = {1, W};
            for (int nout : nouts) {
                if (twoshot && nout != W) continue;
                std::vector<int> red((size_t)n * nout, 0);
                for (int r = 0; r < W; ++r)
                    for (int b = 0; b < B; ++b) {
                        StagedItems it;
                        const int jo = twoshot ? r : 0;
                        it.init(twoshot != 0, r0[jo], r1[jo], P, B, b, r, W, nout);
                        int prev_unit = -1;
                        for (int64_t i = 0; i < it.total; ++i) {
                            int unit, m;
                            int64_t v;
                            it.item(i, unit, m, v);
                            CHECK(v >= 0 && v < n, "item vector %lld out of range\n", (long long)v);
                            if (v < 0 || v >= n) continue;
                            CHECK(unit >= prev_unit, "items not in unit order\n");
                            prev_unit = unit;
                            CHECK(sb[v] == b && su[v] <= unit,
                                  "item reads vector %lld before its unit (block %d unit %d, staged by %d unit %d)\n",
                                  (long long)v, b, unit, sb[v], su[v]);
                            if (twoshot) {
                                CHECK(m == -1 && v >= r0[r] && v < r1[r], "two-shot item outside own segment\n");
                                red[v]++;
                            } else {
                                CHECK(m >= 0 && m < nout, "output index %d\n", m);
                                if (m >= 0 && m < nout) red[(size_t)m * n + v]++;
                            }
                        }
                    }
                const int64_t expect = twoshot ? n : (int64_t)nout * n;
                for (int64_t x = 0; x < expect; ++x)
                    CHECK(red[x] == 1, "staged %s n=%lld W=%d B=%d P=%lld nout=%d: item %lld reduced %d times\n",
                          twoshot ? "two-shot" : "one-shot", (long long)n, W, B, (long long)P, nout, (long long)x, red[x]);
            }
        }
    }

    // Automatic engines: the rules at their boundaries.
    const int64_t MiB = (int64_t)1 << 20;
    CHECK(!auto_staged(false, 2, 64 * MiB, 1) && !auto_staged(false, 2, 1024 * MiB, 1), "one-shot W=2 staged\n");
    CHECK(!auto_staged(false, 4, 16 * MiB - 16, 1) && auto_staged(false, 4, 16 * MiB, 1), "one-shot W=4 boundary\n");
    CHECK(!auto_staged(false, 8, 8 * MiB - 16, 1) && auto_staged(false, 8, 8 * MiB, 1), "one-shot W=8 boundary\n");
    CHECK(!auto_staged(false, 16, 4 * MiB - 16, 1) && auto_staged(false, 16, 4 * MiB, 1), "one-shot W=16 boundary\n");
    CHECK(auto_staged(true, 2, 16, 2) && auto_staged(true, 1, 16, 1), "two-shot W<=2 not staged\n");
    CHECK(!auto_staged(true, 4, 8 * MiB - 16, 4) && auto_staged(true, 4, 8 * MiB, 4) && auto_staged(true, 16, 8 * MiB, 16),
          "two-shot 8 MiB boundary\n");
    CHECK(!auto_bulk_oneshot(8, 1024 * MiB, 1) && !auto_bulk_oneshot(2, 1024 * MiB, 1), "copy-off bulk one-shot at W<=8\n");
    CHECK(!auto_bulk_oneshot(16, 8 * MiB - 16, 1) && auto_bulk_oneshot(16, 8 * MiB, 1) && auto_bulk_oneshot(9, 15 * MiB, 1),
          "copy-off bulk one-shot boundary\n");
    CHECK(auto_staged(false, 8, 32 * MiB, 2) && !auto_staged(false, 8, 32 * MiB, 3) &&
              !auto_staged(false, 4, 32 * MiB, 2) && auto_staged(false, 16, 8 * MiB, 4) &&
              !auto_staged(false, 16, 32 * MiB, 16), "one-shot staged with several outputs\n");
    CHECK(auto_bulk_oneshot(16, 8 * MiB, 2) && auto_bulk_oneshot(16, 8 * MiB, 8) && !auto_bulk_oneshot(16, 8 * MiB, 9) &&
              !auto_bulk_oneshot(16, 32 * MiB - 16, 16) && auto_bulk_oneshot(16, 32 * MiB, 16),
          "copy-off bulk one-shot with several outputs\n");
    {
        GatherArgs g{};
        g.W = 8;
        g.nout = 1;
        g.nsplit = 1;
        g.off[0] = 0;
        g.off[1] = 16 * MiB;
        CHECK(auto_gather_engine(g, 16 * MiB) == 2, "gather 256 MiB moved not bulk\n");
        g.off[1] = 16 * MiB - 16;
        CHECK(auto_gather_engine(g, 16 * MiB - 16) == 1, "gather below 256 MiB moved is bulk\n");
        g.nout = 2;  // 24 x 11 MiB = 264 MiB moved
        g.off[1] = 11 * MiB;
        CHECK(auto_gather_engine(g, 11 * MiB) == 2, "gather with two outputs not bulk\n");
        g.off[1] = (MiB / 3) & ~(int64_t)15;  // 24 x 349,520 B: just under 8 MiB moved
        CHECK(auto_gather_engine(g, g.off[1]) == 1, "gather with two outputs below 8 MiB moved is bulk\n");
        g.off[1] = MiB;  // 24 MiB moved
        CHECK(auto_gather_engine(g, MiB) == 2, "gather with two outputs from 8 MiB moved not bulk\n");
        g.nsplit = 2;
        g.off[1] = 5 * MiB + 8;  // a split boundary off 16 bytes
        g.off[2] = 11 * MiB;
        CHECK(auto_gather_engine(g, 11 * MiB) == 1, "gather with a split off 16 bytes is bulk\n");
        g.W = 2;
        g.nout = 1;
        g.nsplit = 1;
        g.off[1] = 32 * MiB;
        CHECK(auto_gather_engine(g, 32 * MiB) == 1 && (g.off[1] = 64 * MiB, auto_gather_engine(g, 64 * MiB) == 2),
              "gather W=2 boundary\n");
    }

    if (failures) {
        std::printf("%d failures\n", failures);
        return 1;
    }
    std::printf("partition ok\n");
    return 0;
}
