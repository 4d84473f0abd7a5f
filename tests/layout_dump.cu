// Prints the packed block layout of affqmm_format.cuh for every width and
// group: one line per 32-bit code word ("w bits plane row word offset") and
// per scale/bias word ("s bits group row word offset"), so that
// tests/test_layout.py can check the layout's claims on the host.
#include <cstdio>

#include "affqmm_format.cuh"

using namespace affqmm;

int main() {
    const int widths[] = {2, 3, 4, 5, 6, 8};
    const int groups[] = {32, 64, 128};
    for (int bits : widths) {
        for (int plane = 0; plane < 2; ++plane) {
            const int p = plane ? plane1_bits(bits) : plane0_bits(bits);
            for (int n = 0; n < TILE_N; ++n)
                for (int w = 0; w < 4 * p; ++w) std::printf("w %d %d %d %d %d\n", bits, plane, n, w, word_offset(bits, plane, n, w));
        }
        for (int group : groups)
            for (int n = 0; n < TILE_N; ++n)
                for (int j = 0; j < sb_words(group); ++j)
                    std::printf("s %d %d %d %d %d %d\n", bits, group, n, j, sb_offset(bits, group, n) + 4 * j,
                                block_bytes(bits, group));
    }
    return 0;
}
