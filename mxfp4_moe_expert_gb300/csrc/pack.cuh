// Packed (tile-major) layout of one layer's expert matrices.  The expert kernels
// stream, per stage, the 256 weight rows of one work item over 256 K (32 KB of E2M1
// codes: the gate and the up rows of a 128-row block, or 256 down rows), and per
// group of stages those rows' E8M0 scales.  In the canonical row-major layout each of
// those is 256 short runs spread over one or two matrices (two tensor maps, two or
// four copies); here each is one contiguous run, read by a single copy through one
// tensor map.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace moe {

// 256-K stages per scale group for contraction length K (a multiple of 512): the
// largest of 8, 6, 4, 2 that divides K / 256 (a scale row of a group is 8 G bytes).
__host__ __device__ constexpr int pack_scale_group(int K) {
    return (K / 256) % 8 == 0 ? 8 : (K / 256) % 6 == 0 ? 6 : (K / 256) % 4 == 0 ? 4 : 2;
}

// Byte offsets of the sections of a packed buffer (256-byte aligned each):
//   codes     gate/up tiles [E][I/128][H/256][256 rows: 128 gate, 128 up][128 B], then
//             down tiles    [E][H/256][I/256][256 rows][128 B]          (down_codes = offset)
//   scales_gu [E][I/128][H/256/G_H][256 rows: 128 gate, 128 up][8 G_H B]
//   scales_d  [E][H/256][I/256/G_I][256 rows][8 G_I B]
struct PackLayout {
    size_t codes, down_codes, scales_gu, scales_d, total;
};

inline PackLayout pack_layout(int H, int I, int E) {
    auto up256 = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t hi = (size_t)H * I;
    PackLayout L;
    L.codes = 0;
    L.down_codes = (size_t)E * hi;                   // gate + up codes: 2 x E * I * H / 2
    L.scales_gu = up256(L.down_codes + (size_t)E * hi / 2);
    L.scales_d = up256(L.scales_gu + (size_t)E * hi / 16);
    L.total = up256(L.scales_d + (size_t)E * hi / 32);
    return L;
}

}  // namespace moe
