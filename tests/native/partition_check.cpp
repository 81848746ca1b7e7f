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
    if (failures) {
        std::printf("%d failures\n", failures);
        return 1;
    }
    std::printf("partition ok\n");
    return 0;
}
