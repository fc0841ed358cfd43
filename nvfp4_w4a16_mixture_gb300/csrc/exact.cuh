// Exactly rounded sums and certified roundings shared by the decode kernels.
//
// The gate/up sums of the MoE block feed BF16 roundings whose outcome moves a
// whole row of outputs, so the decode kernels form them as the exact sum of
// the exact products, rounded once to fp32: products are split so that their
// high parts are integers on a common grid (a chained mma of them is exact),
// the remaining small products go to a compensation term, and partial sums
// are added with TwoSum.  The sigmoid steps use the correctly rounded fp32
// exp wherever the BF16 result depends on it.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace flint {
namespace {

constexpr int kMargin = 64;  // fp32 ulps kept clear of a BF16 rounding boundary

// ------------------------------------------------------------ numerics --
// s += v with the rounding error of the addition kept in c (TwoSum: s + e
// equals the exact sum of the old s and v).
FLINT_DEV void two_sum(float& s, float& c, float v) {
  const float t = __fadd_rn(s, v);
  const float z = __fsub_rn(t, s);
  const float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(v, z));
  c = __fadd_rn(c, e);
  s = t;
}

// fp32 ulps between v and the nearest BF16 rounding boundary (the midpoint
// between two BF16 neighbours, where round-to-nearest-even decides).
FLINT_DEV int bf16_margin(float v) {
  return abs((int)(__float_as_uint(v) & 0xFFFFu) - 0x8000);
}

// exp(v) correctly rounded to fp32 but for a double-ulp window at the fp32
// rounding boundaries: double-precision exp, rounded once.
__device__ __noinline__ float exp_f32_rn(float v) { return (float)exp((double)v); }

// act = bf16(silu(g) * u), silu(g) = g * (1 / (1 + exp(-g))), every step one
// fp32 rounding.  expf is within 2 ulps of the rounded exp; that moves the
// product by at most about 16 ulps, so a result more than kMargin ulps from a
// BF16 boundary rounds as the correctly rounded exp would make it round.
FLINT_DEV uint32_t act_bits(float g, float u) {
  float e = expf(-g);
  float v = __fmul_rn(__fmul_rn(g, __fdiv_rn(1.0f, __fadd_rn(1.0f, e))), u);
  if (bf16_margin(v) <= kMargin) {
    e = exp_f32_rn(-g);
    v = __fmul_rn(__fmul_rn(g, __fdiv_rn(1.0f, __fadd_rn(1.0f, e))), u);
  }
  return f32_to_bf16_bits(v);
}

// shared expert: sact = bf16((gS / (1 + exp(-gS))) * uS) with gS, uS BF16
// values (the stock SiLU form), same certification.
FLINT_DEV uint32_t sact_bits(float gS, float uS) {
  float e = expf(-gS);
  float v = __fmul_rn(__fdiv_rn(gS, __fadd_rn(1.0f, e)), uS);
  if (bf16_margin(v) <= kMargin) {
    e = exp_f32_rn(-gS);
    v = __fmul_rn(__fdiv_rn(gS, __fadd_rn(1.0f, e)), uS);
  }
  return f32_to_bf16_bits(v);
}

// bf16x2 arithmetic, round to nearest even
FLINT_DEV uint32_t bf2_add(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
FLINT_DEV uint32_t bf2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest biased exponent field among the 32 bf16 values of v (two per word).
FLINT_DEV int max_exp_field(const uint4 (&v)[4]) {
  int m = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = max(m, (int)max((w[i] >> 23) & 0xFFu, (w[i] >> 7) & 0xFFu));
  }
  return m;
}

// Split 32 bf16 values as v = hi + lo, exactly: hi is v rounded to the grid
// 2^(ef - 132) (ef = the largest biased exponent field among the values that
// share the grid), so |hi| / grid <= 64, and lo = v - hi holds the rest (at
// most 8 significant bits, a BF16 value).  The rounding adds and subtracts
// C = 1.5 * 2^(ef - 125): v + C stays in one binade whose BF16 spacing is the
// grid.
FLINT_DEV void split_hi_lo(const uint4 (&v)[4], int ef, uint4 (&hi)[4], uint4 (&lo)[4]) {
  ef = min(max(ef, 1), 252);
  const uint32_t cb = ((uint32_t)(ef + 2) << 7) | 0x40u;
  const uint32_t c2 = cb | (cb << 16);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    hi[q].x = bf2_sub(bf2_add(v[q].x, c2), c2);
    hi[q].y = bf2_sub(bf2_add(v[q].y, c2), c2);
    hi[q].z = bf2_sub(bf2_add(v[q].z, c2), c2);
    hi[q].w = bf2_sub(bf2_add(v[q].w, c2), c2);
    lo[q].x = bf2_sub(v[q].x, hi[q].x);
    lo[q].y = bf2_sub(v[q].y, hi[q].y);
    lo[q].z = bf2_sub(v[q].z, hi[q].z);
    lo[q].w = bf2_sub(v[q].w, hi[q].w);
  }
}

// The activation column of lane (g, t) for one 128-K slice (32 K values at K
// offset 32 t), split hi / lo on the grid of the column's largest value over
// the whole slice (the four lanes of column g agree).
FLINT_DEV void split_column(const uint4 (&xb)[4], uint4 (&xh)[4], uint4 (&xl)[4]) {
  int ef = max_exp_field(xb);
  ef = max(ef, __shfl_xor_sync(0xffffffffu, ef, 1));
  ef = max(ef, __shfl_xor_sync(0xffffffffu, ef, 2));
  split_hi_lo(xb, ef, xh, xl);
}

// B operand registers of word q on the BF16 path (the K permutation of the
// A fragments in frag.cuh: pairs (0, 4), (1, 5) for the first mma, (2, 6),
// (3, 7) for the second).
FLINT_DEV void b_regs(const uint4& x, uint32_t (&b)[2][2]) {
  b[0][0] = __byte_perm(x.x, x.z, 0x5410);
  b[0][1] = __byte_perm(x.x, x.z, 0x7632);
  b[1][0] = __byte_perm(x.y, x.w, 0x5410);
  b[1][1] = __byte_perm(x.y, x.w, 0x7632);
}

// A fragments of word q from natural-order bf16 rows (row g: a, row g + 8:
// b), as a_frags(Bf16Slice) builds them.
FLINT_DEV void a_regs_bf16(const uint4& a, const uint4& b, uint32_t (&af)[2][4]) {
  af[0][0] = __byte_perm(a.x, a.z, 0x5410);
  af[0][2] = __byte_perm(a.x, a.z, 0x7632);
  af[1][0] = __byte_perm(a.y, a.w, 0x5410);
  af[1][2] = __byte_perm(a.y, a.w, 0x7632);
  af[0][1] = __byte_perm(b.x, b.z, 0x5410);
  af[0][3] = __byte_perm(b.x, b.z, 0x7632);
  af[1][1] = __byte_perm(b.y, b.w, 0x5410);
  af[1][3] = __byte_perm(b.y, b.w, 0x7632);
}

FLINT_DEV void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  mma_bf16_16816(d, a[0], a[1], a[2], a[3], b0, b1);
}
FLINT_DEV void mmah(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  mma_f16_16816(d, a[0], a[1], a[2], a[3], b0, b1);
}

// Largest biased exponent field among the 8 bf16 values of one word.
FLINT_DEV int max_exp_word(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  int m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, (int)max((w[i] >> 23) & 0xFFu, (w[i] >> 7) & 0xFFu));
  return m;
}

// split_hi_lo of one word with the rounding constant c2 of the grid.
FLINT_DEV void split_word(const uint4& v, uint32_t c2, uint4& hi, uint4& lo) {
  hi.x = bf2_sub(bf2_add(v.x, c2), c2);
  hi.y = bf2_sub(bf2_add(v.y, c2), c2);
  hi.z = bf2_sub(bf2_add(v.z, c2), c2);
  hi.w = bf2_sub(bf2_add(v.w, c2), c2);
  lo.x = bf2_sub(v.x, hi.x);
  lo.y = bf2_sub(v.y, hi.y);
  lo.z = bf2_sub(v.z, hi.z);
  lo.w = bf2_sub(v.w, hi.w);
}

// The rounding constant C = 1.5 * 2^(ef - 125) of split_hi_lo, twice.
FLINT_DEV uint32_t split_const(int ef) {
  ef = min(max(ef, 1), 252);
  const uint32_t cb = ((uint32_t)(ef + 2) << 7) | 0x40u;
  return cb | (cb << 16);
}

// One 128-K slice of a 16-row tile against xb, exactly: rows g and g + 8
// are read through la(q) / lb(q) (word q = K 32 t + 8 q .. + 7 of the slice
// as 8 bf16 in natural order), the lane's activations are xb.  Weights and
// activations are split per row / column over the slice (split_hi_lo grids),
// w_hi * x_hi accumulates exactly in one chained mma (products of two <= 6-bit
// integers, 128 of them), the rest goes to C.  The grids come first (one pass
// over the words); the words are then split one at a time, so few registers
// stay live.
template <class RowA, class RowB>
FLINT_DEV void slice_exact(float (&S)[4], float (&C)[4], RowA la, RowB lb, const uint4 (&xb)[4]) {
  int ex = 0, ea = 0, eb = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    ex = max(ex, max_exp_word(xb[q]));
    ea = max(ea, max_exp_word(la(q)));
    eb = max(eb, max_exp_word(lb(q)));
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    ex = max(ex, __shfl_xor_sync(0xffffffffu, ex, o));
    ea = max(ea, __shfl_xor_sync(0xffffffffu, ea, o));
    eb = max(eb, __shfl_xor_sync(0xffffffffu, eb, o));
  }
  const uint32_t cx = split_const(ex), ca = split_const(ea), cb = split_const(eb);
  float hh[4] = {0.0f, 0.0f, 0.0f, 0.0f}, ap[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 wa = la(q), wb = lb(q);
    uint4 xh, xl, wah, wal, wbh, wbl;
    split_word(xb[q], cx, xh, xl);
    split_word(wa, ca, wah, wal);
    split_word(wb, cb, wbh, wbl);
    uint32_t bh[2][2], bl[2][2], ah[2][4], alo[2][4], aw[2][4];
    b_regs(xh, bh);
    b_regs(xl, bl);
    a_regs_bf16(wah, wbh, ah);
    a_regs_bf16(wal, wbl, alo);
    a_regs_bf16(wa, wb, aw);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mma16(hh, ah[r], bh[r][0], bh[r][1]);
      mma16(ap, alo[r], bh[r][0], bh[r][1]);
      mma16(ap, aw[r], bl[r][0], bl[r][1]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    two_sum(S[i], C[i], hh[i]);
    C[i] = __fadd_rn(C[i], ap[i]);
  }
}

// The slice of a 16-row BF16 tile (rows g, g + 8 in natural order at ra /
// rb, this lane's 32 K at offset 32 t of the slice).
FLINT_DEV void slice_bf16_exact(float (&S)[4], float (&C)[4], const uint16_t* ra, const uint16_t* rb,
                                const uint4 (&xb)[4]) {
  slice_exact(S, C, [&](int q) { return *reinterpret_cast<const uint4*>(ra + 8 * q); },
              [&](int q) { return *reinterpret_cast<const uint4*>(rb + 8 * q); }, xb);
}

// 8 NVFP4 weights (one word of codes, K 2b in the low nibble of byte b) as
// 8 bf16 e2m1 * scale * 2^-7 in natural order, exactly; sc: bf16x2 of the
// block's scale * 2^119 (twice).
FLINT_DEV uint4 nvfp4_word_bf16(uint32_t w, uint32_t sc) {
  uint32_t o[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t byte = (w >> (8 * b)) & 0xFFu;
    o[b] = bf16x2_mul(e2m1x2_to_bf16x2_scaled((byte & 0xFu) | ((byte >> 4) << 16)), sc);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The slice of a 16-row NVFP4 tile: ca / cb this lane's 16 code bytes of
// rows g, g + 8 (K 32 t .. 32 t + 31 of the slice), sa / sb their two block
// scale bytes (blocks 2 t, 2 t + 1).  The sums are of the weights times
// 2^-7: the caller scales them back.
FLINT_DEV void slice_nvfp4_exact(float (&S)[4], float (&C)[4], const uint8_t* ca, const uint8_t* cb,
                                 uint32_t sa, uint32_t sb, const uint4 (&xb)[4]) {
  const uint32_t a2 = e4m3x2_to_bf16x2_x2p119(sa), b2 = e4m3x2_to_bf16x2_x2p119(sb);
  const uint4 wa = *reinterpret_cast<const uint4*>(ca), wb = *reinterpret_cast<const uint4*>(cb);
  const uint32_t wa4[4] = {wa.x, wa.y, wa.z, wa.w}, wb4[4] = {wb.x, wb.y, wb.z, wb.w};
  slice_exact(S, C, [&](int q) { return nvfp4_word_bf16(wa4[q], bf16x2_bcast(a2, q >> 1)); },
              [&](int q) { return nvfp4_word_bf16(wb4[q], bf16x2_bcast(b2, q >> 1)); }, xb);
}

// K split over warps: a tile of 8 token columns is summed by kw warps, warp
// w0 + p taking the slices s = p (mod kw).  Each warp leaves its (sum,
// compensation) pair in red (float4 sum, then float4 compensation, per lane:
// 64 float4 per warp); after a CTA barrier the first warp of the tile adds
// the others' pairs to its own in warp order with TwoSum, so the result
// does not depend on which warp finished first.
FLINT_DEV void store_pair(float4* red, int warp, int lane, const float (&S)[4], const float (&C)[4]) {
  red[(2 * warp) * 32 + lane] = make_float4(S[0], S[1], S[2], S[3]);
  red[(2 * warp + 1) * 32 + lane] = make_float4(C[0], C[1], C[2], C[3]);
}
FLINT_DEV void add_pairs(float (&S)[4], float (&C)[4], const float4* red, int w0, int kw, int lane) {
  for (int p = 1; p < kw; ++p) {
    const float4 s = red[(2 * (w0 + p)) * 32 + lane], c = red[(2 * (w0 + p) + 1) * 32 + lane];
    two_sum(S[0], C[0], s.x);
    two_sum(S[1], C[1], s.y);
    two_sum(S[2], C[2], s.z);
    two_sum(S[3], C[3], s.w);
    C[0] = __fadd_rn(C[0], c.x);
    C[1] = __fadd_rn(C[1], c.y);
    C[2] = __fadd_rn(C[2], c.z);
    C[3] = __fadd_rn(C[3], c.w);
  }
}

}  // namespace
}  // namespace flint
