// Host-side check of the Q8_0 cache layout (kvq.cuh): the position functions are permutations, and the
// 16-byte chunks that the attention kernel stages and reads hand every MMA lane exactly the codes of its
// tensor-core fragments, with every 128-bit read phase (8 lanes) on distinct bank groups.  The staging and
// read address arithmetic below restates the attention kernel's, for hd 64 and 128.  Exit status 0 = pass.
#include <cstdio>
#include <vector>

#include "../../block_quantized_token_gb300/csrc/kvq.cuh"

using er::kvq_code_off;

static int fails = 0;
#define CHECK(c)                                                         \
    do {                                                                 \
        if (!(c)) {                                                      \
            std::printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #c);      \
            if (++fails > 20) return 1;                                  \
        }                                                                \
    } while (0)

static int check(int hd) {
    // a plane of 32 rows; value id = row * hd + dim
    const int rows = 32;
    std::vector<int> plane[2];
    for (int v = 0; v < 2; ++v) {
        plane[v].assign((size_t)rows * hd, -1);
        for (int r = 0; r < rows; ++r)
            for (int d = 0; d < hd; ++d) {
                const size_t o = kvq_code_off(v != 0, r, d, hd);
                CHECK(o < plane[v].size());
                CHECK(plane[v][o] == -1);  // each place taken once
                plane[v][o] = r * hd + d;
            }
    }
    const int NQ = hd / 32;
    for (int tile = 0; tile < rows / 16; ++tile) {
        const int rb = tile * 16;
        // stage: 16-byte chunks, K with chunk j of row r at j ^ (r & 1), V chunk (L, q) at q ^ key(L)
        std::vector<int> sk(16 * hd, -1), sv(16 * hd, -1);
        for (int ci = 0; ci < hd; ++ci) {
            const int row = ci / (hd / 16), j = ci % (hd / 16);
            for (int b = 0; b < 16; ++b)
                sk[row * hd + ((j ^ (row & 1)) << 4) + b] = plane[0][(size_t)(rb + row) * hd + j * 16 + b];
            const int L = ci / NQ, q = ci % NQ, key = (L * NQ / 8) % NQ;
            for (int b = 0; b < 16; ++b)
                sv[L * (hd / 2) + ((q ^ key) << 4) + b] = plane[1][(size_t)rb * hd + ci * 16 + b];
        }
        for (int lane = 0; lane < 32; ++lane) {
            const int g = lane >> 2, t = lane & 3;
            for (int h = 0; h < 2; ++h) {  // K: rows g and g + 8
                const int row = 8 * h + g;
                for (int c = 0; c < hd / 16; ++c) {
                    const int ch = (hd / 64) * t + c / 4, w = c % 4;
                    const int base = row * hd + ((ch ^ (row & 1)) << 4) + 4 * w;
                    const int dims[4] = {16 * c + 2 * t, 16 * c + 2 * t + 1, 16 * c + 2 * t + 8, 16 * c + 2 * t + 9};
                    for (int b = 0; b < 4; ++b) CHECK(sk[base + b] == (rb + row) * hd + dims[b]);
                }
            }
            const int key = (lane * NQ / 8) % NQ;  // V: rows 2t, 2t+1, 2t+8, 2t+9 of dim 8j + g
            for (int j = 0; j < hd / 8; ++j) {
                const int q = j / 4, w = j % 4;
                const int base = lane * (hd / 2) + ((q ^ key) << 4) + 4 * w;
                const int rr[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
                for (int b = 0; b < 4; ++b) CHECK(sv[base + b] == (rb + rr[b]) * hd + 8 * j + g);
            }
        }
    }
    // 128-bit read phases: 8 lanes, 8 distinct 16-byte bank groups
    for (int h = 0; h < 2; ++h)
        for (int k2 = 0; k2 < hd / 64; ++k2)
            for (int p = 0; p < 4; ++p) {
                int seen = 0;
                for (int lane = 8 * p; lane < 8 * p + 8; ++lane) {
                    const int g = lane >> 2, t = lane & 3, row = 8 * h + g, ch = (hd / 64) * t + k2;
                    seen |= 1 << (((row * hd + ((ch ^ (row & 1)) << 4)) >> 4) & 7);
                }
                CHECK(seen == 0xFF);
            }
    for (int q = 0; q < NQ; ++q)
        for (int p = 0; p < 4; ++p) {
            int seen = 0;
            for (int lane = 8 * p; lane < 8 * p + 8; ++lane) {
                const int key = (lane * NQ / 8) % NQ;
                seen |= 1 << (((lane * (hd / 2) + ((q ^ key) << 4)) >> 4) & 7);
            }
            CHECK(seen == 0xFF);
        }
    return 0;
}

int main() {
    if (check(64) || check(128) || fails) {
        std::printf("kvq layout: %d failures\n", fails);
        return 1;
    }
    std::printf("kvq layout: ok\n");
    return 0;
}
