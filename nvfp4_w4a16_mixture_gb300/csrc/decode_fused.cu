// Single-launch decode path for a few tokens (M <= 8, M * top_k <= 64):
// router, top-k, routed gate/up with SiLU * up, shared-expert gate/up, routed
// and shared down projections and the weighted combine, all in one
// cooperative launch of one CTA per SM.
//
// Page "vllm.models.flint.ops.moe": _router_kernel and _topk_row (BF16
// logits, ties to the lowest expert index, s / (sum + 1e-20) rounded to BF16),
// _gate_up_gemv_kernel (act = bf16(silu(g) * u), global scale on the fp32
// accumulator), _down_gemv_kernel (y = bf16(acc * gs), out = bf16(bf16(sum_j
// tw_j y_j) + shared)), and the module docstring's Numerics paragraph.
//
// Phases (every CTA runs all of them; two grid-wide barriers on workspace
// counters, possible because the cooperative launch keeps every CTA resident):
//   A  the producer warp streams, before any dependency, the CTA's router
//      rows, its shared-expert gate/up tiles and its rows of the shared down
//      projection.  The consumer warps compute the CTA's router logits for
//      every token (barrier 1 follows), split every token row into the
//      exact hi / lo operands of the routed gate/up (below), and compute the
//      shared gate/up tiles.
//   B  after barrier 1 every CTA reads all logits and runs the same top-k and
//      expert grouping, so every CTA knows the routing without another
//      round trip; CTA 0 writes the caller's ids / weights.
//   C  the routed gate/up items (8 gate + 8 up rows of one expert) are split
//      over the CTAs in proportion to their load; act rows go to the
//      workspace; then barrier 2.  Each ring record (a shared tile, an item,
//      a down stage) belongs to one consumer warp, which sums all of its K
//      in registers and writes its results itself.
//   D  CTA c < H / 16 owns output rows 16c .. 16c + 15: the shared down rows
//      (resident since phase A) and the routed down blocks of every routed
//      expert (prefetched behind the gate/up items), then
//      out = bf16(bf16(sum_j tw_j y_j) + ys) in rank order.
//
// Rounding.  The gate/up sums feed a BF16 rounding whose outcome moves a whole
// row of outputs (one activation of the shared expert reaches every output of
// its token, one of a routed expert every output of that expert's pair), so
// they are formed as the exact sum rounded once to fp32:
//   - every token row is split per 128-wide K slice as x = 2^q (X_hi + x_lo):
//     X_hi = round(x 2^-q) an integer |X_hi| <= 32 (q from the slice's
//     largest value), x_lo the rest, both held as f16;
//   - NVFP4 weights are block floating point (e2m1 times an e4m3 scale, an
//     integer of at most 8 bits on the block's grid), so the hi products of
//     a slice are integers on the grid of its smallest scale, and their sum
//     stays below 2^24 when the slice's block scales span at most 2^4: one
//     chained mma from a zero accumulator is then exact; with a wider span
//     every mma is taken alone (16 products, exact for spans up to 2^7);
//     the slice results are added into a (sum, compensation) pair with
//     TwoSum;
//   - BF16 shared weights are split the same way per row and slice (w_hi on
//     6-bit integers) so w_hi * x_hi accumulates exactly in one chained mma;
//   - the small remaining products (x_lo, w_lo) go to the compensation term.
// The down sums feed one output element each: every 128-K slice is one
// chained mma and the slices are added with TwoSum.
// The sigmoid / SiLU steps are evaluated as 1 / (1 + e), every step one fp32
// rounding, with e the correctly rounded fp32 exp: the fast fp32 exp is used
// when the result is far from a BF16 rounding boundary, else exp is
// recomputed in double precision and rounded once.
//
// Every wait is bounded: on expiry the kernel records FLINT_ERR_TIMEOUT in the
// status word, later waits return at once and every loop exits, so a launch
// always ends; the last CTA to leave returns the grid counters to zero.
#include <atomic>

#include "common.cuh"
#include "exact.cuh"
#include "frag.cuh"
#include "internal.h"

namespace flint {
namespace {

constexpr int kCons = 15;                  // consumer warps
constexpr int kProd = kCons;               // producer warp
constexpr int kThreads = (kCons + 1) * 32;
constexpr int kStageBytes = 20480;         // 16 NVFP4 rows of 2048 K with scales, or down blocks
constexpr int kMaxStages = 10;
constexpr int kShKst = 512;                // K per shared gate/up stage (16 bf16 rows)
constexpr int kShPitch = 2 * kShKst + 16;  // smem bytes per shared row (padded)
constexpr int kMaxPairs = 64;              // M * top_k
constexpr int kMaxM = 8;
constexpr int kMaxSlices = 16;             // H / 128
constexpr int kMaxRouterRows = 2;          // router rows per CTA (E <= 2 * grid)
constexpr int kMaxSmem = 232448;
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms
constexpr uint32_t kSuspendNs = 50000;

// wait sites recorded with a timeout (status word 1)
enum {
  kSiteSlot = 1, kSiteFull = 2, kSiteBar1 = 3, kSiteBar2 = 4, kSiteRouted = 5, kSiteLogits = 6,
  kSiteTopk = 7, kSiteSplit = 8, kSiteRdone = 9, kSiteRows = 10, kSiteAct = 11, kSiteDrain = 12,
};

enum { kKindShared = 0, kKindRouted = 1, kKindDown = 2 };

// A record is the unit of work of one consumer warp: a shared gate/up tile
// (sh_stages ring stages), a routed gate/up item, the shared down, or a
// routed down stage (one ring stage each).  Records are issued in this order
// and record r belongs to consumer warp kCons - 1 - r % kCons, so the first
// records (the shared tiles, before any routing) go to the last warps while
// warps 0 .. M - 1 run the top-k.
struct Stage {
  int seq;          // stage number: set before the slot's barrier phase opens
  int kind;
  int k0, kst;      // kind 0: K offset and extent
  int tile;         // kind 0: shared tile j (intermediate rows 8j .. 8j + 7)
  int u, r0;        // kind 1: expert slot and first intermediate row; kind 2: u
  int act_in;       // kind 2: the stage's copies include the activation rows
};

struct Route {
  int U;
  int item_lo, item_hi;
  int e[kMaxPairs], cnt[kMaxPairs], off[kMaxPairs];
  unsigned char tok[kMaxPairs][kMaxM];
  float tw[kMaxM][kMaxTopK];
  int pos[kMaxM][kMaxTopK];
  unsigned emask[kMaxE];              // tokens routed to expert e (bit t)
  unsigned char jslot[kMaxM][kMaxE];  // rank j of expert e in token t
};

struct Ctl {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t xfull, rfull, sdfull;
  uint64_t rdone, split_done, topk_done, logits_ready, routed_ready, act_ready;
  uint64_t abar[kCons];  // per consumer warp: its bulk copies of activation rows
  int abort;
  int ca_done;   // records whose act / sact are written (+1 once the routing is known)
  int all_done;  // records finished (+1 once the routing is known)
  int ca_target, all_target;
  int left;      // the CTA has counted itself out of the grid
  int parts;     // warps sharing one routed gate/up item (its K split)
  int pcnt[kMaxStages];  // parts of the slot's item finished
  Stage info[kMaxStages];
  float xp2[kMaxM][kMaxSlices];  // 2^q of token t, slice s
  float xp2zero[kMaxSlices];     // a column that holds no token
  Route rt;
};

struct Layout {
  int stages;
  size_t xr, xh, xl, xpitch, rrow, sdown, ysm, yss, ctl, total;
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }

__host__ __device__ inline Layout fused_layout(int M, int H, int SI) {
  Layout L;
  L.xpitch = 2 * (size_t)H + 16;
  const size_t xsplit = al16((size_t)M * L.xpitch);
  const size_t rrow = (size_t)kMaxRouterRows * 2 * H;
  const size_t sdown = al16((size_t)16 * (SI > 0 ? SI : 0) * 2);
  const size_t ysm = (size_t)kMaxPairs * 16 * 2;
  const size_t yss = al16((size_t)kMaxM * 16 * 2);
  const size_t xraw = al16((size_t)M * H * 2);
  const size_t fixed = xraw + 2 * xsplit + rrow + sdown + ysm + yss + al16(sizeof(Ctl));
  const size_t room = fixed < (size_t)kMaxSmem ? kMaxSmem - fixed : 0;
  L.stages = (int)(room / kStageBytes);
  if (L.stages > kMaxStages) L.stages = kMaxStages;
  L.xr = (size_t)L.stages * kStageBytes;
  L.xh = L.xr + xraw;
  L.xl = L.xh + xsplit;
  L.rrow = L.xl + xsplit;
  L.sdown = L.rrow + rrow;
  L.ysm = L.sdown + sdown;
  L.yss = L.ysm + ysm;
  L.ctl = L.yss + yss;
  L.total = L.ctl + al16(sizeof(Ctl));
  return L;
}

// --------------------------------------------------------------- waits --
__device__ __noinline__ void record_timeout(int* status, int site, int n) {
  if (atomicCAS(status, 0, FLINT_ERR_TIMEOUT) == 0) {
    status[1] = site;
    status[2] = (int)blockIdx.x;
    status[3] = n;
  }
}

__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                          int site, int n) {
  if (*abort) return false;
  unsigned long long t0 = 0;
  for (;;) {
    if (mbar_try_wait(bar, parity, kSuspendNs)) return true;
    if (*abort) return false;
    const unsigned long long now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > kWaitNs) {
      *abort = 1;
      record_timeout(status, site, n);
      return false;
    }
  }
}

__device__ __noinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status, int lane,
                         int site, int n) {
  int ok = 0;
  if (lane == 0) ok = wait_phase(bar, parity, abort, status, site, n);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait for a phase that must complete whatever happened elsewhere
// (it counts bulk copies in flight, which may not outlive the CTA): on
// expiry it records the timeout and returns.
__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status, int n) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity, kSuspendNs))
    if (globaltimer_ns() - t0 > kWaitNs) {
      *abort = 1;
      record_timeout(status, kSiteDrain, n);
      return;
    }
}

// Bounded poll until a ring slot carries stage number nn.  The stamp comes
// at least a copy's latency before the data, so the poll backs off to 512 ns:
// a waiting warp then costs the compute warps of its SM almost no issue slots.
__device__ __noinline__ bool wait_stamp(const int* seq, int nn, volatile int* abort, int* status) {
  const volatile int* sq = seq;
  unsigned long long t0 = 0;
  unsigned sleep_ns = 32;
  while (*sq != nn) {
    if (*abort) return false;
    const unsigned long long now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > kWaitNs) {
      *abort = 1;
      record_timeout(status, kSiteFull, nn);
      return false;
    }
    __nanosleep(sleep_ns);
    sleep_ns = min(2 * sleep_ns, 512u);
  }
  return true;
}

// Spin (bounded) until the grid counter reaches `target` (acquire, GPU scope).
__device__ __noinline__ bool wait_counter(const int* p, int target, volatile int* abort, int* status, int site) {
  unsigned long long t0 = 0;
  for (;;) {
    if (ld_acquire(p) >= target) return true;
    if (*abort) return false;
    const unsigned long long now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > kWaitNs) {
      *abort = 1;
      record_timeout(status, site, target);
      return false;
    }
    __nanosleep(32);
  }
}

// A fragments of one slice on the f16 path: byte b of a row's 16 code bytes
// of this thread -> (K 2b, 2b + 1) by the hardware e2m1 -> f16 conversion,
// times the f16 block scale (exact: at most 6 significant bits, inside f16's
// normal range); mma r of word q gets K {2r, 2r + 1} and {2r + 4, 2r + 5} of
// the word, matching the natural-order B registers (x, z) and (y, w).
FLINT_DEV void a_frags_f16(uint32_t (&af)[4][2][4], const uint4& c0, const uint4& c1, uint32_t s0b,
                           uint32_t s1b) {
  const uint32_t s0 = e4m3x2_to_f16x2(s0b), s1 = e4m3x2_to_f16x2(s1b);
  const uint32_t wg[4] = {c0.x, c0.y, c0.z, c0.w};
  const uint32_t wg8[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t sq = f16x2_bcast(s0, q >= 2), sq8 = f16x2_bcast(s1, q >= 2);
    uint32_t p[4], p8[4];
    e2m1x8_to_f16x2(wg[q], p);
    e2m1x8_to_f16x2(wg8[q], p8);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      af[q][r][0] = f16x2_mul(p[r], sq);
      af[q][r][1] = f16x2_mul(p8[r], sq8);
      af[q][r][2] = f16x2_mul(p[r + 2], sq);
      af[q][r][3] = f16x2_mul(p8[r + 2], sq8);
    }
  }
}

FLINT_DEV void load_col_smem(uint4 (&xb)[4], const uint8_t* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    xb[q] = p ? *reinterpret_cast<const uint4*>(p + 16 * q) : make_uint4(0, 0, 0, 0);
}
FLINT_DEV void load_col_global(uint4 (&xb)[4], const uint16_t* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q) xb[q] = p ? ldg_cg_v4(p + 8 * q) : make_uint4(0, 0, 0, 0);
}

// Min / max exponent field of the non-zero e4m3 block scales among the two
// bytes of `two` (subnormal scales share field 1's grid).
FLINT_DEV void scale_fields(uint32_t two, int& lo, int& hi) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t b = (two >> (8 * i)) & 0x7Fu;
    if (b) {
      const int f = max((int)(b >> 3), 1);
      lo = min(lo, f);
      hi = max(hi, f);
    }
  }
}

// Routed gate/up of one item part: a 16-row NVFP4 tile (rows g, g + 8 of
// lane (g, t): gate row g and up row g) over the 128-K slices s_lo .. s_hi - 1,
// against the activation columns on the f16 path.  bcol: this lane's column
// of X_hi (integers), or, with `combined`, X_hi for columns 0..3 and x_lo for
// columns 4..7; lcol: x_lo (not combined); p2[s][c]: 2^q of the lane's two
// columns in slice s.  hi products go exactly into (S, C), lo ones into C.
//
// Exactness of the hi sums: X_hi is an integer of at most 5 bits and a
// weight an integer of at most 8 bits on its block's grid, so a slice's 128
// hi products are integers on the grid of its smallest block scale and sum
// to less than 2^24 when the block scales span at most 2^4 binades (checked
// over both rows and the part's slices): the slice's mma's then run in two
// exact chains (words 0-1 and 2-3) whose fp32 sum is exact too, and the
// slice total is added with one TwoSum.  With a wider span every mma (16
// products, exact for spans up to 2^7) is added alone.
FLINT_DEV void item_gateup(float (&S)[4], float (&C)[4], const uint8_t* st, int H, int g, int t,
                           const uint8_t* bcol, const uint8_t* lcol, bool combined,
                           const float* p2c0, const float* p2c1, int s_lo, int s_hi) {
  const uint8_t* rg = st + g * (H / 2);
  const uint8_t* rg8 = st + (g + 8) * (H / 2);
  const uint8_t* sg = st + 16 * (H / 2) + g * (H / 16);
  const uint8_t* sg8 = st + 16 * (H / 2) + (g + 8) * (H / 16);
  // block-scale span of rows g and g + 8 over the part's slices
  int lo0 = 99, hi0 = -1, lo1 = 99, hi1 = -1;
  for (int s = s_lo; s < s_hi; ++s) {
    scale_fields(*reinterpret_cast<const uint16_t*>(sg + s * 8 + 2 * t), lo0, hi0);
    scale_fields(*reinterpret_cast<const uint16_t*>(sg8 + s * 8 + 2 * t), lo1, hi1);
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    lo0 = min(lo0, __shfl_xor_sync(0xffffffffu, lo0, o));
    hi0 = max(hi0, __shfl_xor_sync(0xffffffffu, hi0, o));
    lo1 = min(lo1, __shfl_xor_sync(0xffffffffu, lo1, o));
    hi1 = max(hi1, __shfl_xor_sync(0xffffffffu, hi1, o));
  }
  const bool wide = __any_sync(0xffffffffu, hi0 - lo0 > 4 || hi1 - lo1 > 4);

  for (int s = s_lo; s < s_hi; ++s) {
    const uint4 c0 = *reinterpret_cast<const uint4*>(rg + s * (kSliceK / 2) + 16 * t);
    const uint4 c1 = *reinterpret_cast<const uint4*>(rg8 + s * (kSliceK / 2) + 16 * t);
    const uint32_t s0b = *reinterpret_cast<const uint16_t*>(sg + s * (kSliceK / 16) + 2 * t);
    const uint32_t s1b = *reinterpret_cast<const uint16_t*>(sg8 + s * (kSliceK / 16) + 2 * t);
    uint4 bh[4];
    load_col_smem(bh, bcol ? bcol + 2 * (s * kSliceK + 32 * t) : nullptr);
    const float pa = p2c0[s], pb = p2c1[s];
    uint32_t af[4][2][4];
    a_frags_f16(af, c0, c1, s0b, s1b);
    if (!wide) {
      float da[4] = {0.0f, 0.0f, 0.0f, 0.0f}, db[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        mmah(da, af[q][0], bh[q].x, bh[q].z);
        mmah(db, af[q + 2][0], bh[q + 2].x, bh[q + 2].z);
        mmah(da, af[q][1], bh[q].y, bh[q].w);
        mmah(db, af[q + 2][1], bh[q + 2].y, bh[q + 2].w);
      }
      // (the x_lo columns of a combined item round in the mma already; their
      // sum is about 2^-5 of the hi one, so one more rounding costs nothing)
#pragma unroll
      for (int i = 0; i < 4; ++i) two_sum(S[i], C[i], __fadd_rn(da[i], db[i]) * ((i & 1) ? pb : pa));
    } else {
      // (rare: block scales spread over more than 2^4; kept compact)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mmah(d, af[q][r], r ? bh[q].y : bh[q].x, r ? bh[q].w : bh[q].z);
#pragma unroll
          for (int i = 0; i < 4; ++i) two_sum(S[i], C[i], d[i] * ((i & 1) ? pb : pa));
        }
      }
    }
    if (!combined) {
      uint4 bl[4];
      load_col_smem(bl, lcol ? lcol + 2 * (s * kSliceK + 32 * t) : nullptr);
      float dl[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        mmah(dl, af[q][0], bl[q].x, bl[q].z);
        mmah(dl, af[q][1], bl[q].y, bl[q].w);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) C[i] = __fadd_rn(C[i], dl[i] * ((i & 1) ? pb : pa));
    }
  }
}

// One 128-K slice of an NVFP4 down block (bf16 path, weights scaled by 2^-7)
// against bf16 activation columns: one chained mma, then TwoSum.
FLINT_DEV void slice_down_fp4(float (&S)[4], float (&C)[4], const uint8_t* rg, const uint8_t* rg8,
                              const uint8_t* sg, const uint8_t* sg8, int s, int t, const uint4 (&xb)[4]) {
  Fp4Slice d;
  d.c0 = *reinterpret_cast<const uint4*>(rg + s * (kSliceK / 2) + 16 * t);
  d.c1 = *reinterpret_cast<const uint4*>(rg8 + s * (kSliceK / 2) + 16 * t);
  d.s0 = *reinterpret_cast<const uint16_t*>(sg + s * (kSliceK / 16) + 2 * t);
  d.s1 = *reinterpret_cast<const uint16_t*>(sg8 + s * (kSliceK / 16) + 2 * t);
  uint32_t af[4][2][4];
  a_frags(d, af);
  float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // words 0-1 and 2-3 in two chains
    uint32_t b[2][2];
    b_regs(xb[q], b);
    mma16(acc[q >> 1], af[q][0], b[0][0], b[0][1]);
    mma16(acc[q >> 1], af[q][1], b[1][0], b[1][1]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    two_sum(S[i], C[i], acc[0][i]);
    two_sum(S[i], C[i], acc[1][i]);
  }
}

// The same for a BF16 down block in natural row order (shared expert).
FLINT_DEV void slice_down_bf16(float (&S)[4], float (&C)[4], const uint16_t* ra, const uint16_t* rb,
                               const uint4 (&xb)[4]) {
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 wa = *reinterpret_cast<const uint4*>(ra + 8 * q);
    const uint4 wb = *reinterpret_cast<const uint4*>(rb + 8 * q);
    uint32_t af[2][4], b[2][2];
    a_regs_bf16(wa, wb, af);
    b_regs(xb[q], b);
    mma16(acc, af[0], b[0][0], b[0][1]);
    mma16(acc, af[1], b[1][0], b[1][1]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) two_sum(S[i], C[i], acc[i]);
}

// ---------------------------------------------------------- top-k warp --
// Top-k of one token (lane j < k ends with rank j's expert and weight),
// sigmoid and renormalisation with the correctly rounded exp, certified like
// act_bits.
template <class Get>
FLINT_DEV void topk_token(Get get, int E, int k, int lane, int& out_e, float& out_w) {
  int key[kMaxE / 32];
#pragma unroll
  for (int q = 0; q < kMaxE / 32; ++q) {
    const int ee = q * 32 + lane;
    key[q] = -1;
    if (ee < E) key[q] = (int)((ordered_bf16(get(ee)) << 8) | (uint32_t)(E - 1 - ee));
  }
  int my_e = 0, my_key = 0;
  for (int j = 0; j < k; ++j) {
    int lm = key[0];
#pragma unroll
    for (int q = 1; q < kMaxE / 32; ++q) lm = max(lm, key[q]);
    const int best = __reduce_max_sync(0xffffffffu, lm);
#pragma unroll
    for (int q = 0; q < kMaxE / 32; ++q)
      if (key[q] == best) key[q] = -1;
    if (lane == j) { my_key = best; my_e = E - 1 - (best & 0xFF); }
  }
  float logit = 0.0f;
  if (lane < k) {
    const uint32_t o = (uint32_t)my_key >> 8;
    const uint32_t b16 = (o & 0x8000u) ? (o ^ 0x8000u) : (o ^ 0xFFFFu);
    logit = bf16_bits_to_f32(b16);
  }
  float w = 0.0f;
  for (int pass = 0; pass < 2; ++pass) {
    float s = 0.0f;
    if (lane < k) {
      const float e = pass == 0 ? expf(-logit) : exp_f32_rn(-logit);
      s = __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
    }
    float sum = 0.0f;  // in rank order
    for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, s, j));
    const float q = __fdiv_rn(s, __fadd_rn(sum, 1e-20f));
    w = round_bf16(q);
    // expf moves s by at most a few ulps and the quotient by at most about 40
    const bool near = lane < k && bf16_margin(q) <= kMargin;
    if (!__any_sync(0xffffffffu, near)) break;
  }
  out_e = my_e;
  out_w = w;
}

// ---------------------------------------------------- work assignment --
struct Items {
  int lo, hi;
};

// The routed gate/up items (T = U * I / 8) are split evenly over the CTAs:
// the down work comes after the grid barrier that ends the gate/up phase, so
// each phase is balanced on its own.
FLINT_DEV Items item_range(int c, int G, int U, int I) {
  const int T = U * (I / 8);  // T * G < 2^31 (U <= 256, I <= 2048, G <= 1024)
  Items r;
  r.lo = T * c / G;
  r.hi = T * (c + 1) / G;
  return r;
}

// Parts per item for a CTA with ni items: the number (1 .. 4, at most the
// slice count, within the stage's spare room) that minimises the slices the
// busiest warp sums when the ni * Q part records go round-robin over the
// consumer warps; fewer parts on ties.
FLINT_DEV int item_parts(int ni, int nsl, int room, bool wide_cols) {
  int best = 1, best_cost = 0x7fffffff;
  for (int q = 1; q <= 4 && q <= nsl; ++q) {
    if (q > 1 && q * (wide_cols ? 1024 : 512) > room) break;
    const int cost = (ni * q + kCons - 1) / kCons * ((nsl + q - 1) / q);
    if (cost < best_cost) { best_cost = cost; best = q; }
  }
  return best;
}

// ======================================================================
// Records of this CTA in issue order: the shared gate/up tiles, the routed
// gate/up items, the shared down (CTAs owning output rows, SI > 0), the
// routed down stages.  nrec_dn: routed down stages.
struct RecPlan {
  int n_sh, n_items, n_shd, n_dn, total;
};

__global__ void __launch_bounds__(kThreads, 1) moe_decode_fused_kernel(MoEArgs a) {
  SpanGuard<kSpanSingle> span_guard;
  extern __shared__ __align__(128) uint8_t smem[];
  const int M = a.M, H = a.H, E = a.E, k = a.k, I = a.I, SI = a.SI;
  const Layout L = fused_layout(M, H, SI);
  const int S = L.stages;
  uint8_t* ring = smem;
  const uint16_t* xr = reinterpret_cast<const uint16_t*>(smem + L.xr);  // bf16 x [token][H]
  uint8_t* xh = smem + L.xh;  // f16 X_hi [token][H]
  uint8_t* xl = smem + L.xl;  // f16 x_lo [token][H]
  const int xpitch = (int)L.xpitch;
  const uint16_t* rrow = reinterpret_cast<const uint16_t*>(smem + L.rrow);
  const uint16_t* sdown = reinterpret_cast<const uint16_t*>(smem + L.sdown);
  uint16_t* ysm = reinterpret_cast<uint16_t*>(smem + L.ysm);
  uint16_t* yss = reinterpret_cast<uint16_t*>(smem + L.yss);
  Ctl& SM = *reinterpret_cast<Ctl*>(smem + L.ctl);
  Route& RT = SM.rt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = gridDim.x, c = blockIdx.x;
  int* status = a.ws.status;
  int* cnt = a.ws.fd_cnt;  // [0] barrier 1, [1] barrier 2, [2] CTAs done
  volatile int* abort = &SM.abort;

  const int n_dn_ctas = min(H / 16, G);  // CTAs owning output rows
  const bool has_dn = c < n_dn_ctas;
  const int h0 = 16 * c;
  const int nSh = SI / 8;  // shared tiles
  const int sh_stages = (H + kShKst - 1) / kShKst;
  const int nsl_h = H / kSliceK;
  int my_sh_tiles = 0;
  for (int j = c; j < nSh; j += G) ++my_sh_tiles;
  int my_rrows = 0;
  for (int e = c; e < E; e += G) ++my_rrows;

  for (int i = threadIdx.x; i < kMaxE; i += kThreads) RT.emask[i] = 0u;
  for (int i = threadIdx.x; i < kMaxSlices; i += kThreads) SM.xp2zero[i] = 0.0f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&SM.full[i], 1);
      mbar_init(&SM.empty[i], 1);
      SM.info[i].seq = -1;
      SM.pcnt[i] = 0;
    }
    mbar_init(&SM.xfull, 1);
    mbar_init(&SM.rfull, 1);
    mbar_init(&SM.sdfull, 1);
    mbar_init(&SM.rdone, kCons);
    mbar_init(&SM.split_done, kCons);
    mbar_init(&SM.topk_done, M);
    mbar_init(&SM.logits_ready, 1);
    mbar_init(&SM.routed_ready, 1);
    mbar_init(&SM.act_ready, 1);
    for (int w = 0; w < kCons; ++w) mbar_init(&SM.abar[w], 1);
    SM.abort = 0;
    SM.ca_done = 0;
    SM.all_done = 0;
    SM.ca_target = 0x7fffffff;
    SM.all_target = 0x7fffffff;
    SM.left = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // Producer side of ring slot n % S: wait until its previous use was consumed.
  auto acquire_slot = [&](int n) -> bool {
    if (n < S) return !*abort;
    return wait_phase(&SM.empty[n % S], ((n / S) - 1) & 1, abort, status, kSiteSlot, n);
  };

  if (warp == kProd) {
    // ================================================================ producer
    bool dead = false;
    pdl_wait();  // x belongs to the stream's earlier work
    if (lane == 0) {
      // phase A: the token rows, then weights that depend on no routing
      mbar_arrive_expect_tx(&SM.xfull, (uint32_t)M * 2u * H);
      bulk_g2s(smem + L.xr, a.x, (uint32_t)M * 2u * H, &SM.xfull);
      mbar_arrive_expect_tx(&SM.rfull, (uint32_t)my_rrows * 2u * H);
      int i = 0;
      for (int e = c; e < E; e += G, ++i)
        bulk_g2s(smem + L.rrow + (size_t)i * 2 * H, a.router_w + (size_t)e * H, 2u * H, &SM.rfull);
      // the shared expert's weights go out once the router rows have landed,
      // so that the routing, on the critical path, does not queue behind them
      if (!wait_phase(&SM.rfull, 0, abort, status, kSiteRows, 0)) dead = true;
      const uint32_t sb = (!dead && has_dn && SI > 0) ? 16u * (uint32_t)SI * 2u : 0u;
      mbar_arrive_expect_tx(&SM.sdfull, sb);
      if (sb) bulk_g2s(smem + L.sdown, a.shared_down + (size_t)h0 * SI, sb, &SM.sdfull);
    }
    dead = __shfl_sync(0xffffffffu, dead, 0);
    int n = 0;
    // shared gate/up tiles: a stage is 8 gate + 8 up rows over up to 512 K
    for (int j = c; j < nSh && !dead; j += G) {
      for (int sidx = 0; sidx < sh_stages && !dead; ++sidx) {
        int ok = 1;
        if (lane == 0) ok = acquire_slot(n);
        if (!__shfl_sync(0xffffffffu, ok, 0)) { dead = true; break; }
        const int sl = n % S;
        const int k0 = sidx * kShKst, kst = min(kShKst, H - k0);
        Stage& inf = SM.info[sl];
        if (lane == 0) {
          inf.kind = kKindShared; inf.k0 = k0; inf.kst = kst; inf.tile = j;
          inf.seq = n;
          mbar_arrive_expect_tx(&SM.full[sl], 16u * 2u * (uint32_t)kst);
        }
        __syncwarp();
        if (lane < 16) {
          const int row = lane < 8 ? 8 * j + lane : SI + 8 * j + (lane - 8);
          bulk_g2s(ring + (size_t)sl * kStageBytes + (size_t)lane * kShPitch,
                   a.shared_gu + (size_t)row * H + k0, 2u * (uint32_t)kst, &SM.full[sl]);
        }
        ++n;
      }
    }
    // barrier 1: this CTA's logits are written (consumers), then every CTA's
    if (lane == 0) {
      if (wait_phase(&SM.rdone, 0, abort, status, kSiteRdone, 0)) {
        red_release_add(cnt + 0, 1);
        if (wait_counter(cnt + 0, G, abort, status, kSiteBar1)) mbar_arrive(&SM.logits_ready);
      } else {
        red_release_add(cnt + 0, 1);  // so that no other CTA waits in vain
      }
    }
    __syncwarp();
    // phase C: this CTA's routed gate/up items (routing from the consumers)
    if (!dead && !warp_wait(&SM.routed_ready, 0, abort, status, lane, kSiteRouted, 0)) dead = true;
    if (!dead) {
      const int U = RT.U, lo = RT.item_lo, hi = RT.item_hi;
      const int ipe = I / 8;
      for (int it = lo; it < hi; ++it) {
        int ok = 1;
        if (lane == 0) ok = acquire_slot(n);
        if (!__shfl_sync(0xffffffffu, ok, 0)) { dead = true; break; }
        const int sl = n % S;
        const int u = it / ipe, r0 = (it % ipe) * 8;
        const size_t g0 = (size_t)RT.e[u] * 2 * I + r0, u0 = g0 + I;
        Stage& inf = SM.info[sl];
        uint8_t* st = ring + (size_t)sl * kStageBytes;
        if (lane == 0) {
          inf.kind = kKindRouted; inf.u = u; inf.r0 = r0;
          inf.seq = n;
          mbar_arrive_expect_tx(&SM.full[sl], 16u * (H / 2) + 16u * (H / 16));
        }
        __syncwarp();
        if (lane == 0) bulk_g2s(st, a.w13 + g0 * (H / 2), 8u * (H / 2), &SM.full[sl]);
        if (lane == 1) bulk_g2s(st + 8 * (H / 2), a.w13 + u0 * (H / 2), 8u * (H / 2), &SM.full[sl]);
        if (lane == 2)
          bulk_g2s(st + 16 * (H / 2), a.w13_sf + g0 * (H / 16), 8u * (H / 16), &SM.full[sl]);
        if (lane == 3)
          bulk_g2s(st + 16 * (H / 2) + 8 * (H / 16), a.w13_sf + u0 * (H / 16), 8u * (H / 16),
                   &SM.full[sl]);
        ++n;
      }
      // phase D stages: the routed down blocks of the output tile (the shared
      // down needs none: its weight rows are resident since phase A)
      if (has_dn && !dead) {
        // one routed expert per stage; once the activation rows are
        // complete (barrier 2 passed) their copies join the stage's weights
        const int wb = 16 * (I / 2) + I;  // weight bytes of a block
        for (int ub = 0; ub < U && !dead; ++ub) {
          int ok = 1;
          if (lane == 0) ok = acquire_slot(n);
          if (!__shfl_sync(0xffffffffu, ok, 0)) { dead = true; break; }
          const int sl = n % S;
          Stage& inf = SM.info[sl];
          uint8_t* st = ring + (size_t)sl * kStageBytes;
          int act_in = 0;
          if (lane == 0) act_in = mbar_test_wait(&SM.act_ready, 0) ? 1 : 0;
          act_in = __shfl_sync(0xffffffffu, act_in, 0);
          const int cn = RT.cnt[ub];
          if (lane == 0) {
            inf.kind = kKindDown; inf.u = ub; inf.act_in = act_in;
            inf.seq = n;
            mbar_arrive_expect_tx(&SM.full[sl], (uint32_t)(wb + (act_in ? cn * 2 * I : 0)));
          }
          __syncwarp();
          const size_t row0 = (size_t)RT.e[ub] * H + h0;
          if (lane == 0) bulk_g2s(st, a.w2 + row0 * (I / 2), 16u * (I / 2), &SM.full[sl]);
          if (lane == 1) bulk_g2s(st + 16 * (I / 2), a.w2_sf + row0 * (I / 16), 16u * (I / 16), &SM.full[sl]);
          if (act_in) {
            // the rows were written by other CTAs before barrier 2 (generic
            // proxy); the proxy fence orders them before these copies
            fence_proxy_async_global();
            for (int r = lane; r < cn; r += 32)
              bulk_g2s(st + wb + (size_t)r * (2 * I + 16), a.ws.act + (size_t)(RT.off[ub] + r) * I, 2u * I,
                       &SM.full[sl]);
          }
          ++n;
        }
      }
    }
    if (lane == 0) {
      // no bulk copy may outlive the CTA: wait (bounded) for the stages that
      // may still be in flight and for the phase-A copies
      for (int i = (n - S > 0 ? n - S : 0); i < n; ++i)
        drain_wait(&SM.full[i % S], (i / S) & 1, abort, status, i);
      drain_wait(&SM.xfull, 0, abort, status, -1);
      drain_wait(&SM.rfull, 0, abort, status, -2);
      drain_wait(&SM.sdfull, 0, abort, status, -3);
    }
    return;
  }

  // =================================================================== consumers
  bool ok = true;
  uint32_t aphase = 0;  // passes of this warp's activation-copy barrier

  // ---- phase A.1: router logits of this CTA's experts, task = (row, token);
  // lane l sums the products of h = 256 c + 8 l + i ascending in (c, i) with
  // fmaf (exact products), then the xor butterfly 16 .. 1
  pdl_wait();  // the workspace belongs to the stream's earlier work
  ok = warp_wait(&SM.xfull, 0, abort, status, lane, kSiteRows, 0);
  if (ok && my_rrows * M > warp) ok = warp_wait(&SM.rfull, 0, abort, status, lane, kSiteRows, 0);
  for (int task = warp; ok && task < my_rrows * M; task += kCons) {
    const int i = task / M, tt = task % M, e = c + i * G;
    const uint16_t* wr = rrow + (size_t)i * H;
    const uint16_t* xt = xr + (size_t)tt * H;
    float acc = 0.0f;
#pragma unroll
    for (int cch = 0; cch < 8; ++cch) {
      const int h = 256 * cch + 8 * lane;
      if (h >= H) break;
      const uint4 xv = *reinterpret_cast<const uint4*>(xt + h);
      const uint4 wv = *reinterpret_cast<const uint4*>(wr + h);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc = fmaf(__uint_as_float(xw[q] << 16), __uint_as_float(ww[q] << 16), acc);
        acc = fmaf(__uint_as_float(xw[q] & 0xFFFF0000u), __uint_as_float(ww[q] & 0xFFFF0000u), acc);
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.ws.logits[(size_t)tt * E + e] = (uint16_t)f32_to_bf16_bits(acc);
  }
  __syncwarp();
  // the arrive (release, CTA scope) orders the logit stores before the
  // producer's GPU-scope release of barrier 1
  if (lane == 0) mbar_arrive(&SM.rdone);

  // ---- phase A.2: the routed gate/up operands, task = (token, slice):
  // q = (largest exponent of the slice) - 4, X_hi = round(x 2^-q) (|X_hi| <=
  // 32), x_lo = x 2^-q - X_hi, both f16 in natural K order
  for (int task = warp; ok && task < M * nsl_h; task += kCons) {
    const int tt = task / nsl_h, s = task % nsl_h;
    const uint2 raw = *reinterpret_cast<const uint2*>(xr + (size_t)tt * H + s * kSliceK + 4 * lane);
    const uint32_t w2[2] = {raw.x, raw.y};
    int ef = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) ef = max(ef, (int)max((w2[i] >> 23) & 0xFFu, (w2[i] >> 7) & 0xFFu));
    ef = __reduce_max_sync(0xffffffffu, ef);
    const int q = max(ef - 127 - 4, -126);
    const float sc = pow2f(-q);
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float v0 = __uint_as_float(w2[i] << 16) * sc;
      const float v1 = __uint_as_float(w2[i] & 0xFFFF0000u) * sc;
      const float h0f = rintf(v0), h1f = rintf(v1);
      const __half2 hh = __floats2half2_rn(h0f, h1f);
      const __half2 ll = __floats2half2_rn(v0 - h0f, v1 - h1f);
      hw[i] = *reinterpret_cast<const uint32_t*>(&hh);
      lw[i] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    const size_t o = (size_t)tt * xpitch + 2 * (s * kSliceK + 4 * lane);
    *reinterpret_cast<uint2*>(xh + o) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(xl + o) = make_uint2(lw[0], lw[1]);
    if (lane == 0) SM.xp2[tt][s] = pow2f(q);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&SM.split_done);

  // ---- phase B: top-k of token t on warp t, then the expert grouping on warp 0
  if (warp < M) {
    if (ok) ok = warp_wait(&SM.logits_ready, 0, abort, status, lane, kSiteLogits, 0);
    if (ok) {
      const int tt = warp;
      int my_e = 0;
      float my_w = 0.0f;
      topk_token([&](int ee) { return ldg_cg_u16(a.ws.logits + (size_t)tt * E + ee); }, E, k, lane,
                 my_e, my_w);
      if (lane < k) {
        RT.tw[tt][lane] = my_w;
        RT.jslot[tt][my_e] = (unsigned char)lane;
        atomicOr(&RT.emask[my_e], 1u << tt);
        if (c == 0) {
          if (a.ids_out) a.ids_out[tt * k + lane] = my_e;
          if (a.tw_out) a.tw_out[tt * k + lane] = my_w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&SM.topk_done);
    }
  }
  if (warp == 0 && ok) ok = warp_wait(&SM.topk_done, 0, abort, status, lane, kSiteTopk, 0);
  if (warp == 0 && ok) {
    // experts in ascending order get consecutive slots u and sorted pair
    // positions; the pairs of one expert in ascending token order.  Lane l
    // takes experts l * per .. l * per + per - 1; one packed scan gives every
    // lane its first pair position (high half) and slot (low half).
    const int per = (E + 31) / 32;
    int tot = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      const int ce = e < E ? __popc(RT.emask[e]) : 0;
      tot += (ce << 16) | (ce > 0 ? 1 : 0);
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int off = (incl - tot) >> 16, u = (incl - tot) & 0xFFFF;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      const unsigned mask = e < E ? RT.emask[e] : 0u;
      if (mask) {
        const int base = off;
        RT.e[u] = e;
        RT.cnt[u] = __popc(mask);
        RT.off[u] = base;
        for (unsigned m = mask; m; m &= m - 1, ++off) {
          const int tt = __ffs(m) - 1;
          RT.tok[u][off - base] = (unsigned char)tt;
          RT.pos[tt][RT.jslot[tt][e]] = off;
        }
        ++u;
      }
    }
    const int run_u = __shfl_sync(0xffffffffu, incl & 0xFFFF, 31);
    if (lane == 0) {
      RT.U = run_u;
      const Items r = item_range(c, G, run_u, I);
      RT.item_lo = r.lo;
      RT.item_hi = r.hi;
      // few items per CTA: split each one's K over up to 4 warps; a part's
      // (sum, compensation) pairs take 512 bytes of the stage's spare room
      // (1 KB when the item has more than 4 tokens)
      bool wide_cols = false;
      for (int it = r.lo; it < r.hi; ++it) wide_cols |= RT.cnt[it / (I / 8)] > 4;
      SM.parts = item_parts(r.hi - r.lo, nsl_h, kStageBytes - 16 * (H / 2 + H / 16), wide_cols);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&SM.routed_ready);
  }

  // ---- the records of this warp, in issue order
  // Finishing a record: `ca` marks records whose act / sact rows feed other
  // CTAs.  The thread that completes the CTA's act / sact count releases
  // barrier 2 and, once every CTA has, opens the down phase; the one that
  // completes the CTA's record count writes the output rows and leaves.
  auto finish = [&](bool ca) {
    __syncwarp();
    int last_ca = 0, last_all = 0;
    if (lane == 0) {
      // the acq_rel shared-memory atomics order this warp's act / sact / y
      // writes (made visible to lane 0 by the __syncwarp above) before the
      // last finisher's GPU-scope release of barrier 2; no GPU-scope fence is
      // needed here (one would wait for the SM's bulk copies in flight)
      volatile int* tg = &SM.ca_target;
      if (ca) {
        const int old = atom_add_acqrel_cta_smem(&SM.ca_done, 1);
        last_ca = old + 1 == tg[0];
      }
      const int old = atom_add_acqrel_cta_smem(&SM.all_done, 1);
      last_all = old + 1 == tg[1];
    }
    return make_int2(__shfl_sync(0xffffffffu, last_ca, 0), __shfl_sync(0xffffffffu, last_all, 0));
  };
  auto open_down = [&]() {  // lane 0 of the last act / sact writer of the CTA
    red_release_add(cnt + 1, 1);
    if (wait_counter(cnt + 1, G, abort, status, kSiteBar2) &&
        a.fault != FLINT_FAULT_DOWN_HANDOVER)  // test hook: leave the hand-over out
      mbar_arrive(&SM.act_ready);
  };
  auto final_rows = [&]() {  // out = bf16(bf16(sum_j tw_j y_j) + ys), rank order
    __syncwarp();  // lane 0's acquire covers every lane's reads below
    if (!has_dn) return;
    for (int idx = lane; idx < M * 8; idx += 32) {
      const int tt = idx >> 3, rp = idx & 7;
      uint32_t o[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int row = 2 * rp + cc;
        float R = 0.0f;
#pragma unroll 1
        for (int j = 0; j < k; ++j)
          R = __fadd_rn(R, __fmul_rn(RT.tw[tt][j], bf16_bits_to_f32(ysm[RT.pos[tt][j] * 16 + row])));
        const float ysv = SI > 0 ? bf16_bits_to_f32(yss[tt * 16 + row]) : 0.0f;
        o[cc] = f32_to_bf16_bits(__fadd_rn(round_bf16(R), ysv));
      }
      *reinterpret_cast<uint32_t*>(a.out + (size_t)tt * H + h0 + 2 * rp) = o[0] | (o[1] << 16);
    }
  };
  auto leave = [&]() {  // the last CTA returns the grid counters to zero
    __syncwarp();
    if (lane == 0 && atomicExch(&SM.left, 1) == 0) {
      __threadfence();
      if (atomicAdd(cnt + 2, 1) == G - 1) {
        cnt[0] = 0;
        cnt[1] = 0;
        cnt[2] = 0;
        __threadfence();
      }
    }
  };
  // A stage's owner may come to its slot while the slot still holds an
  // earlier stage (up to a whole phase behind, where a parity wait would pass
  // at once), so it first waits for the producer to stamp the slot with its
  // stage number: from then on the barrier's open phase is this stage's.
  auto wait_full = [&](int nn) -> bool {
    int ok2 = 1;
    if (lane == 0) ok2 = wait_stamp(&SM.info[nn % S].seq, nn, abort, status);
    if (!__shfl_sync(0xffffffffu, ok2, 0)) return false;
    return warp_wait(&SM.full[nn % S], (nn / S) & 1, abort, status, lane, kSiteFull, nn);
  };
  auto release = [&](int nn) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&SM.empty[nn % S]);
  };
  // Bulk-copy `rows` activation rows of `len` bf16 from global `src` (row
  // stride len) into smem `dst` (row pitch 2 len + 16) through this warp's
  // barrier, and wait for them.  The rows were written by other CTAs before
  // barrier 2 (generic proxy); the proxy fence orders them before the copies.
  auto copy_rows = [&](uint8_t* dst, const uint16_t* src, int rows, int len) -> bool {
    fence_proxy_async_global();
    if (lane == 0) mbar_arrive_expect_tx(&SM.abar[warp], (uint32_t)rows * 2u * len);
    __syncwarp();
    for (int r = lane; r < rows; r += 32)
      bulk_g2s(dst + (size_t)r * (2 * len + 16), src + (size_t)r * len, 2u * len, &SM.abar[warp]);
    const bool got = warp_wait(&SM.abar[warp], aphase & 1, abort, status, lane, kSiteAct, 0);
    ++aphase;
    return got;
  };

  const int sh_stage_total = my_sh_tiles * sh_stages;
  int n_items = 0, n_shd = 0, n_dn = 0, total = sh_stage_total, Q = 1;
  bool routed = false, act_ok = false;
  bool closing = false;  // this warp finished the CTA's last record
  for (int r = kCons - 1 - warp; ok; r += kCons) {
    if (r >= sh_stage_total && !routed) {
      // the routing (and the operand split) are needed from here on
      ok = warp_wait(&SM.routed_ready, 0, abort, status, lane, kSiteRouted, 0) &&
           warp_wait(&SM.split_done, 0, abort, status, lane, kSiteSplit, 0);
      if (!ok) break;
      routed = true;
      n_items = RT.item_hi - RT.item_lo;
      Q = SM.parts;
      n_shd = (has_dn && SI > 0) ? 1 : 0;
      n_dn = 0;
      if (has_dn) n_dn = RT.U;  // one routed expert per down stage
      total = sh_stage_total + n_items * Q + n_shd + n_dn;
      if (warp == 0 && lane == 0) {
        SM.ca_target = my_sh_tiles + n_items + 1;
        SM.all_target = total + 1;
      }
      if (warp == 0) {  // the routing is known: count it once on both counters
        const int2 fl = finish(true);
        if (fl.x && lane == 0) open_down();
        if (fl.y) { closing = true; break; }
      }
    }
    if (routed && r >= total) break;
    if (r < sh_stage_total) {
      // ---- shared gate/up stage: 8 gate + 8 up rows over up to 512 K.  The
      // sh_stages stages of a tile are records of their own; their pairs
      // meet in the stages' spare bytes and the last one to finish adds them
      // up in K order, releases the tile's stages and writes sact
      const int n = r, part = r % sh_stages, n0 = r - part;
      if (!wait_full(n)) { ok = false; break; }
      const Stage& inf = SM.info[n % S];
      uint8_t* st = ring + (size_t)(n % S) * kStageBytes;
      const int tile = inf.tile;
      float S_[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C_[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int s = 0; s < inf.kst / kSliceK; ++s) {
        uint4 xb[4];
        load_col_smem(xb, g < M ? reinterpret_cast<const uint8_t*>(xr + (size_t)g * H + inf.k0 + s * kSliceK + 32 * t)
                                : nullptr);
        const uint16_t* ra = reinterpret_cast<const uint16_t*>(st + g * kShPitch) + s * kSliceK + 32 * t;
        const uint16_t* rb = reinterpret_cast<const uint16_t*>(st + (g + 8) * kShPitch) + s * kSliceK + 32 * t;
        slice_bf16_exact(S_, C_, ra, rb, xb);
      }
      if (sh_stages > 1) {
        float* area = reinterpret_cast<float*>(st + 16 * kShPitch);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          area[i * 32 + lane] = S_[i];
          area[(4 + i) * 32 + lane] = C_[i];
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          last = atom_add_acqrel_cta_smem(&SM.pcnt[n0 % S], 1) == sh_stages - 1;
          if (last) SM.pcnt[n0 % S] = 0;
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) {
          const int2 fl = finish(false);
          if (fl.y) { closing = true; break; }
          continue;
        }
        __syncwarp();  // lane 0's acquire covers every lane's reads below
        for (int pp = 0; pp < sh_stages; ++pp) {
          const float* ar =
              reinterpret_cast<const float*>(ring + (size_t)((n0 + pp) % S) * kStageBytes + 16 * kShPitch);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (pp == 0) {
              S_[i] = ar[i * 32 + lane];
              C_[i] = ar[(4 + i) * 32 + lane];
            } else {
              two_sum(S_[i], C_[i], ar[i * 32 + lane]);
              C_[i] = __fadd_rn(C_[i], ar[(4 + i) * 32 + lane]);
            }
          }
        }
        __syncwarp();
        if (lane == 0)
          for (int pp = 0; pp < sh_stages; ++pp) mbar_arrive(&SM.empty[(n0 + pp) % S]);
      } else {
        release(n);
      }
      const int row = 8 * tile + g;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int tt = 2 * t + cc;
        if (tt < M) {
          const float gS = round_bf16(__fadd_rn(S_[cc], C_[cc]));
          const float uS = round_bf16(__fadd_rn(S_[2 + cc], C_[2 + cc]));
          a.ws.sact[(size_t)tt * SI + row] = (uint16_t)sact_bits(gS, uS);
        }
      }
      const int2 fl = finish(true);
      if (fl.x && lane == 0) open_down();
      if (fl.y) { closing = true; break; }
      continue;
    }
    // item records: Q parts of one stage each; the shared down (no stage);
    // then one record per routed down stage
    const int rr = r - sh_stage_total;
    if (n_shd && rr == n_items * Q) {
      // ---- shared down: rows h0 .. h0 + 15 (resident) against sact, copied
      // into the split activations' room (every item of the CTA is done)
      if (!act_ok) {
        if (!warp_wait(&SM.act_ready, 0, abort, status, lane, FLINT_FAULT_DOWN_HANDOVER, r)) {
          ok = false;
          break;
        }
        act_ok = true;
      }
      // (the room was last read through the generic proxy: fence it before
      // the bulk copies write it)
      fence_proxy_async_smem();
      if (!warp_wait(&SM.sdfull, 0, abort, status, lane, kSiteRows, r) ||
          !copy_rows(xh, a.ws.sact, M, SI)) { ok = false; break; }
      float S_[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C_[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int s = 0; s < SI / kSliceK; ++s) {
        uint4 xb[4];
        load_col_smem(xb, g < M ? xh + (size_t)g * (2 * SI + 16) + 2 * (s * kSliceK + 32 * t) : nullptr);
        slice_down_bf16(S_, C_, sdown + (size_t)g * SI + s * kSliceK + 32 * t,
                        sdown + (size_t)(g + 8) * SI + s * kSliceK + 32 * t, xb);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int tt = 2 * t + cc;
        if (tt < M) {
          yss[tt * 16 + g] = (uint16_t)f32_to_bf16_bits(__fadd_rn(S_[cc], C_[cc]));
          yss[tt * 16 + g + 8] = (uint16_t)f32_to_bf16_bits(__fadd_rn(S_[2 + cc], C_[2 + cc]));
        }
      }
      const int2 fl = finish(false);
      if (fl.y) { closing = true; break; }
      continue;
    }
    const int n = sh_stage_total + (rr < n_items * Q ? rr / Q : rr - n_items * (Q - 1) - n_shd);
    if (!wait_full(n)) { ok = false; break; }
    const Stage& inf = SM.info[n % S];
    uint8_t* st = ring + (size_t)(n % S) * kStageBytes;
    const int kind = inf.kind;
    if (kind == kKindRouted) {
      // ---- routed gate/up item part: 16 rows (8 gate, 8 up) over 1 / Q of K
      const int u = inf.u, r0 = inf.r0, cn = RT.cnt[u], part = rr % Q;
      const bool combined = cn <= 4;
      // B column g: X_hi of token g, or (combined) X_hi of token g for g < 4
      // and x_lo of token g - 4 for g >= 4
      const int col = combined ? (g & 3) : g;
      const bool live = col < cn;
      const uint8_t* bcol = live ? (combined && g >= 4 ? xl : xh) + (size_t)RT.tok[u][col] * xpitch : nullptr;
      const uint8_t* lcol = live ? xl + (size_t)RT.tok[u][col] * xpitch : nullptr;
      int ctok[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int n2 = 2 * t + cc, c2 = combined ? (n2 & 3) : n2;
        ctok[cc] = c2 < cn ? RT.tok[u][c2] : -1;
      }
      float S_[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C_[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const float* p2a = ctok[0] >= 0 ? SM.xp2[ctok[0]] : SM.xp2zero;
      const float* p2b = ctok[1] >= 0 ? SM.xp2[ctok[1]] : SM.xp2zero;
      item_gateup(S_, C_, st, H, g, t, bcol, lcol, combined, p2a, p2b, part * nsl_h / Q,
                  (part + 1) * nsl_h / Q);
      if (combined) {
        // lanes t = 2, 3 hold the x_lo columns of lanes t - 2's tokens
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __shfl_down_sync(0xffffffffu, __fadd_rn(S_[i], C_[i]), 2);
          C_[i] = __fadd_rn(C_[i], lo);
        }
      }
      if (Q > 1) {
        // every part leaves its pairs in the stage's spare bytes; the last
        // one to finish adds them up in part order (the same result whichever
        // part comes last) and finishes the item
        float* area = reinterpret_cast<float*>(st + 16 * (H / 2 + H / 16));
        const int per = combined ? 16 : 32;
        const bool keep = !combined || t < 2;
        const int li = combined ? 2 * g + t : lane;
        if (keep) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            area[(part * 8 + i) * per + li] = S_[i];
            area[(part * 8 + 4 + i) * per + li] = C_[i];
          }
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          last = atom_add_acqrel_cta_smem(&SM.pcnt[n % S], 1) == Q - 1;
          if (last) SM.pcnt[n % S] = 0;
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) {
          const int2 fl = finish(false);
          if (fl.y) { closing = true; break; }
          continue;
        }
        __syncwarp();  // lane 0's acquire covers every lane's reads below
        if (keep) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            S_[i] = area[i * per + li];
            C_[i] = area[(4 + i) * per + li];
          }
          for (int pp = 1; pp < Q; ++pp) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              two_sum(S_[i], C_[i], area[(pp * 8 + i) * per + li]);
              C_[i] = __fadd_rn(C_[i], area[(pp * 8 + 4 + i) * per + li]);
            }
          }
        }
      }
      release(n);
      const float gsc = a.w13_gs[RT.e[u]];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int nn = 2 * t + cc;
        if (nn < cn && (!combined || t < 2)) {
          const float gv = __fmul_rn(__fadd_rn(S_[cc], C_[cc]), gsc);
          const float uv = __fmul_rn(__fadd_rn(S_[2 + cc], C_[2 + cc]), gsc);
          a.ws.act[(size_t)(RT.off[u] + nn) * I + r0 + g] = (uint16_t)act_bits(gv, uv);
        }
      }
      const int2 fl = finish(true);
      if (fl.x && lane == 0) open_down();
      if (fl.y) { closing = true; break; }
      continue;
    }
    // down records: every CTA's act and sact are in the workspace
    if (!act_ok && !(kind == kKindDown && inf.act_in)) {
      if (!warp_wait(&SM.act_ready, 0, abort, status, lane, FLINT_FAULT_DOWN_HANDOVER, n)) {
        ok = false;
        break;
      }
      act_ok = true;
    }
    {
      // ---- routed down stage: rows h0 .. h0 + 15 of one expert
      const int u = inf.u, cn = RT.cnt[u], wb = 16 * (I / 2) + I;
      uint8_t* arow = st + wb;
      if (!inf.act_in && !copy_rows(arow, a.ws.act + (size_t)RT.off[u] * I, cn, I)) { ok = false; break; }
      const uint8_t* sc = st + 16 * (I / 2);
      float S_[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C_[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int s = 0; s < I / kSliceK; ++s) {
        uint4 xb[4];
        load_col_smem(xb, g < cn ? arow + (size_t)g * (2 * I + 16) + 2 * (s * kSliceK + 32 * t) : nullptr);
        slice_down_fp4(S_, C_, st + g * (I / 2), st + (g + 8) * (I / 2), sc + g * (I / 16),
                       sc + (g + 8) * (I / 16), s, t, xb);
      }
      const float gs2 = a.w2_gs[RT.e[u]];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int nn = 2 * t + cc;
        if (nn < cn) {
          const int p = RT.off[u] + nn;
          ysm[p * 16 + g] = (uint16_t)f32_to_bf16_bits(__fmul_rn(__fadd_rn(S_[cc], C_[cc]) * 128.0f, gs2));
          ysm[p * 16 + g + 8] =
              (uint16_t)f32_to_bf16_bits(__fmul_rn(__fadd_rn(S_[2 + cc], C_[2 + cc]) * 128.0f, gs2));
        }
      }
      release(n);
    }
    const int2 fl = finish(false);
    if (fl.y) { closing = true; break; }
  }
  // the output rows are written once, after the loop, by the warp that
  // finished the CTA's last record
  if (closing) {
    final_rows();
    leave();
  }
  if (!ok) {
    // a wait gave up: count this warp out once so that the CTA still leaves
    // (the outputs of the call are undefined; the status word says why)
    __syncwarp();
    int last = 0;
    if (lane == 0) last = 1;
    if (__shfl_sync(0xffffffffu, last, 0)) leave();
  }
}

}  // namespace

bool fused_supported(const flint_moe_shape& s, int sms) {
  if (s.M < 1 || s.M > kFusedMaxTokens || s.M * s.top_k > kMaxPairs) return false;
  if (s.H > 2048 || s.H % 128 != 0 || s.H / 16 > sms) return false;
  if (s.I > 2048 || s.I % 128 != 0 || s.SI > 1024 || s.SI % 128 != 0) return false;
  if (s.E > kMaxRouterRows * sms) return false;
  // a routed down block with all M of its activation rows fits one stage
  if (16 * (s.I / 2) + s.I + s.M * (2 * s.I + 16) > kStageBytes) return false;
  // the shared down's activation rows fit the split activations' room
  if (2 * s.SI + 16 > 2 * (2 * s.H + 16)) return false;
  const Layout L = fused_layout(s.M, s.H, s.SI);
  // the (up to 4) stages of a shared gate/up tile are resident together
  return L.stages >= 4 && L.total <= (size_t)kMaxSmem;
}

cudaError_t launch_fused(const MoEArgs& a, cudaStream_t st, int sms) {
  static std::atomic<bool> attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute((const void*)moe_decode_fused_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  MoEArgs aa = a;
  void* args[] = {&aa};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = fused_layout(a.M, a.H, a.SI).total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barriers need every CTA resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, (const void*)moe_decode_fused_kernel, args);
}

FLINT_SPAN_SETTER(fused)

}  // namespace flint
