// mma.sync operand fragments of one 128-wide K slice of a 16-row weight tile
// (rows g and g + 8 of the tile for lane (g = lane / 4, t = lane % 4)).
//
// Operand mapping inside a slice: thread t holds 32 consecutive K (16 code
// bytes, or 32 bf16) of each of its two rows.  Each 8-code word yields four
// bf16x2 pairs (codes i, i + 4); the activation vector is permuted the same
// way (byte_perm of its 16-byte chunks), so every product pairs matching K.
// NVFP4 rows are dequantised exactly: each pair is built as e2m1 * 2^-126
// (bit placement) and multiplied by bf16(scale * 2^119), giving
// e2m1 * scale * 2^-7; the fp32 accumulator is scaled back by 2^7 (exact).
#pragma once

#include "common.cuh"

namespace flint {

constexpr int kSliceK = 128;  // K per slice: 4 threads x 32

struct Fp4Slice {
  uint4 c0, c1;     // codes of rows g and g + 8 (32 each)
  uint32_t s0, s1;  // their two e4m3 block scales (one per 16 codes)
};
struct Bf16Slice {
  uint4 r0[4], r1[4];  // 32 bf16 of rows g and g + 8
};

// A fragments of the slice: af[q][r][0..3] for word q (0..3), half r (0, 1).
FLINT_DEV void a_frags(const Fp4Slice& d, uint32_t (&af)[4][2][4]) {
  const uint32_t sc0 = e4m3x2_to_bf16x2_x2p119(d.s0);
  const uint32_t sc1 = e4m3x2_to_bf16x2_x2p119(d.s1);
  const uint32_t wg[4] = {d.c0.x, d.c0.y, d.c0.z, d.c0.w};
  const uint32_t wg8[4] = {d.c1.x, d.c1.y, d.c1.z, d.c1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t sg = bf16x2_bcast(sc0, q >= 2);
    const uint32_t sg8 = bf16x2_bcast(sc1, q >= 2);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      af[q][r][0] = bf16x2_mul(e2m1_pair(wg[q], 2 * r), sg);
      af[q][r][1] = bf16x2_mul(e2m1_pair(wg8[q], 2 * r), sg8);
      af[q][r][2] = bf16x2_mul(e2m1_pair(wg[q], 2 * r + 1), sg);
      af[q][r][3] = bf16x2_mul(e2m1_pair(wg8[q], 2 * r + 1), sg8);
    }
  }
}

FLINT_DEV void a_frags(const Bf16Slice& d, uint32_t (&af)[4][2][4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 a = d.r0[q], b = d.r1[q];
    af[q][0][0] = __byte_perm(a.x, a.z, 0x5410);
    af[q][0][2] = __byte_perm(a.x, a.z, 0x7632);
    af[q][1][0] = __byte_perm(a.y, a.w, 0x5410);
    af[q][1][2] = __byte_perm(a.y, a.w, 0x7632);
    af[q][0][1] = __byte_perm(b.x, b.z, 0x5410);
    af[q][0][3] = __byte_perm(b.x, b.z, 0x7632);
    af[q][1][1] = __byte_perm(b.y, b.w, 0x5410);
    af[q][1][3] = __byte_perm(b.y, b.w, 0x7632);
  }
}

}  // namespace flint
