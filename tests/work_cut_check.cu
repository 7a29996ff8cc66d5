// Host-side check of the split decode's cost-weighted cut (WorkCut in
// decode_kernel.cuh): for many length mixes (empty sequences included), head
// counts and grid sizes, the ranges start_unit(c) .. start_unit(c + 1) must
// partition the units in order, range_of(u, s) must name the range holding
// unit u of segment s, and a segment's ranges must be consecutive with none
// of them empty.  Prints "ok" or the first violation; exit status 0 / 1.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "decode_kernel.cuh"

using pagedkv::dec::WorkCut;

static int check(const std::vector<int>& nb, int H, int W) {
    const int B = (int)nb.size();
    std::vector<int> pre(B + 1, 0);
    for (int b = 0; b < B; ++b) pre[b + 1] = pre[b] + nb[b];
    const int U = pre[B] * H;
    const WorkCut cut(pre.data(), B, H, W);
    // unit -> (segment) and the range each unit falls in, in order
    int prev_range = -1, prev_start = 0;
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < H; ++g) {
            const int s = b * H + g, first = pre[b] * H + g * nb[b];
            int last_c = -1;
            for (int k = 0; k < nb[b]; ++k) {
                const int u = first + k, c = cut.range_of(u, s);
                if (c < prev_range || c >= W) {
                    std::printf("B=%d H=%d W=%d: unit %d in range %d after %d\n", B, H, W, u, c, prev_range);
                    return 1;
                }
                if (c != prev_range) {            // u is the first unit of range c
                    if (cut.start_unit(c) != u) {
                        std::printf("B=%d H=%d W=%d: range %d starts at %d, start_unit says %d\n", B, H, W,
                                    c, u, cut.start_unit(c));
                        return 1;
                    }
                    for (int e = prev_range + 1; e < c; ++e)   // empty ranges in between
                        if (cut.start_unit(e) != u) {
                            std::printf("B=%d H=%d W=%d: empty range %d starts at %d, not %d\n", B, H,
                                        W, e, cut.start_unit(e), u);
                            return 1;
                        }
                    if (last_c >= 0 && c != last_c + 1) {
                        std::printf("B=%d H=%d W=%d: segment %d skips from range %d to %d\n", B, H, W,
                                    s, last_c, c);
                        return 1;
                    }
                    prev_range = c;
                    prev_start = u;
                }
                last_c = c;
            }
        }
    for (int e = prev_range + 1; e <= W; ++e)
        if (cut.start_unit(e) != U) {
            std::printf("B=%d H=%d W=%d: range %d after the last starts at %d, not U = %d\n", B, H, W, e,
                        cut.start_unit(e), U);
            return 1;
        }
    (void)prev_start;
    return 0;
}

int main() {
    std::srand(12345);
    long long cases = 0;
    for (int trial = 0; trial < 400; ++trial) {
        const int B = 1 + std::rand() % 300;
        std::vector<int> nb(B);
        for (int b = 0; b < B; ++b) {
            const int kind = std::rand() % 10;
            nb[b] = kind == 0 ? 0 : kind < 6 ? std::rand() % 8 : std::rand() % 600;
        }
        for (int H : {1, 2, 8})
            for (int W : {1, 4, 96, 1824}) {
                if (check(nb, H, W)) return 1;
                ++cases;
            }
    }
    std::printf("ok %lld cases\n", cases);
    return 0;
}
