// Decode-path expert kernels for few tokens (M <= 64): NVFP4 gate/up with
// SiLU * up, and the down projection with the weighted combine and the
// shared-expert add.
//
// Page "vllm.models.flint.ops.moe": _gate_up_gemv_kernel
// (act[p] = silu(x[t] Wg[e]^T) * (x[t] Wu[e]^T), global scale on the fp32
// accumulator), _down_gemv_kernel (y_j = bf16(act W2[e_j]^T * gs),
// out = bf16(bf16(sum_j tw_j y_j) + shared)), and the module's Numerics rule.
//
// Both kernels stream weights through a ring of shared-memory stages filled
// by 1-D bulk copies (cp.async.bulk, completion counted on an mbarrier) from
// one producer warp; sixteen consumer warps run the products on the tensor
// cores (mma.sync m16n8k16, weights as the 16-row A operand, up to 8 tokens
// per B tile); in the gate/up kernel a further warp runs the tile epilogues.  The producer runs ahead by the whole ring, so every SM keeps
// well over 100 KB of weight reads in flight.
//
// Chaining (programmatic dependent launch):
//   router (loads its weight rows, then waits for every earlier kernel, and
//   only then releases the gate/up grid -- so x is final when gate/up starts)
//     -> gate/up: launched early; before its dependency wait it computes the
//        whole shared-expert gate/up (x and the weights are inputs), then
//        streams the routed experts' tiles named by the router's records.
//     -> down: launched when every gate/up CTA is past its wait (so the
//        routing records are final); its producer fills the ring with down
//        weights before the dependency wait, the consumers wait for act.
// Every wait is bounded: on expiry the kernel records FLINT_ERR_TIMEOUT in
// the status word, later waits return at once, and the control flow of all
// warps stays identical (no barrier is skipped), so the launch always ends.
#include "common.cuh"
#include "exact.cuh"
#include "frag.cuh"
#include "internal.h"

namespace flint {
namespace {

constexpr int kCons = 16;                   // consumer warps
constexpr int kThreads = (kCons + 1) * 32;  // + one producer warp
constexpr int kEpi = kCons + 1;               // gate/up: the tile-epilogue warp
constexpr int kGuThreads = (kCons + 2) * 32;  // gate/up: + producer + epilogue warp
constexpr int kXsMaxBytes = 67584;            // gate/up: staged activations, at most
constexpr int kPad = 16;                    // smem row padding (bank spread)
constexpr int kMaxSmem = 232448;            // opt-in shared memory per CTA
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // 200 ms
constexpr uint32_t kSuspendNs = 50000;  // suspend-time hint of one try_wait

// ---- gate/up ring: a stage holds 32 NVFP4 rows (16 gate + 16 up) of up to
// 2048 K with their scales, or 16 BF16 rows (8 gate + 8 up) of up to 1024 K.
constexpr int kGuMaxStages = 5;
constexpr int kGuKst4 = 2048;
constexpr int kGuKst16 = 1024;
constexpr int kGuStageBytes = 32 * (kGuKst4 / 2 + kPad) + 32 * (kGuKst4 / 16);  // 37376
static_assert(16 * (2 * kGuKst16 + kPad) <= kGuStageBytes, "bf16 stage fits");
constexpr int kKP = kCons / 2;  // K parts of a routed stage (x 2 A tiles)

// ---- down ring: a stage holds up to 8 weight blocks of 16 output rows.
constexpr int kDnStages = 3;
// down stages whose weights are requested before the dependency wait (the
// kernel starts while gate/up is still running, so they have landed by the
// time the activation copies go out)
constexpr int kDnPrefetch = 3;
static_assert(kDnPrefetch <= kDnStages, "prefetched stages fit the ring");
constexpr int kDnStageBytes = 57344;
constexpr int kDnMaxBlocks = 8;
constexpr int kDnMaxItems = 64;

struct GuInfo {
  int kind;   // 0 shared (bf16), 1 routed (nvfp4), -1 end of work
  int first;  // first / last stage of its tile
  int last;
  int k0;     // K offset of the stage within the rows
  int kst;    // K covered by the stage
  int pitch;  // smem bytes per weight row
  int sf_off; // byte offset of the scale rows (routed)
  int sf_pitch;
  int r0;     // first intermediate row of the tile
  int e;      // expert (routed)
  int cnt;    // tokens
  int off;    // sorted position of the expert's first pair (routed)
  int x16;    // 1: the router's f16 copy of x is exact (routed, M <= kX16MaxTokens)
  short tok[kDecodeMaxTokens];
};

struct DnBlock {
  int kind;      // 0 shared (bf16), 1 routed (nvfp4)
  int e;
  int u;         // routed: index of the expert's routing record
  int cnt;
  int off;
  int smem;      // byte offset of the weight rows in the stage
  int pitch;
  int act_smem;  // byte offset of the block's activation rows, -1 = read from global
};

struct DnInfo {
  int nblocks;  // 0 = end of work
  int nitems;
  int abytes;   // bytes of activation rows staged with the block weights
  unsigned char item_blk[kDnMaxItems];
  unsigned char item_nt[kDnMaxItems];
  DnBlock blk[kDnMaxBlocks];
};

struct Ctl {
  uint64_t full[kGuMaxStages];
  uint64_t empty[kGuMaxStages];
  uint64_t bar[2];  // CTA barriers among warps (bounded, unlike bar.sync)
  int abort;
};

// Records a timeout: status[0] = FLINT_ERR_TIMEOUT, and for the first one
// status[1] = wait site, status[2] = CTA, status[3] = stage.
FLINT_DEV void record_timeout(int* status, int site, int n) {
  if (atomicCAS(status, 0, FLINT_ERR_TIMEOUT) == 0) {
    status[1] = site;
    status[2] = (int)blockIdx.x;
    status[3] = n;
  }
}

// Bounded wait on an mbarrier phase.  Returns false (and records the
// timeout) once the deadline passes or another warp has given up.
FLINT_DEV bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                          int site, int n) {
  if (*abort) return false;
  unsigned long long t0 = 0;
  for (;;) {
    // suspends until the phase completes (or the hint runs out), so idle
    // warps leave the issue slots to the working ones
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

FLINT_DEV bool warp_wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                               int lane, int site, int n) {
  int ok = 0;
  if (lane == 0) ok = wait_phase(bar, parity, abort, status, site, n);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Barrier among the `count` warps that share mbarrier `bar` (lane 0 of each
// arrives); `phase` is the warp's own count of passed barriers on it.
FLINT_DEV void warp_barrier(uint64_t* bar, uint32_t& phase, volatile int* abort, int* status,
                            int lane, int site) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  warp_wait_phase(bar, phase & 1, abort, status, lane, site, (int)phase);
  ++phase;
}

// Producer side of slot `n % S`: wait until the consumers released its
// previous use.
FLINT_DEV bool acquire_slot(Ctl& c, int n, int S, volatile int* abort, int* status, int site) {
  if (n < S) return !*abort;
  return wait_phase(&c.empty[n % S], ((n / S) - 1) & 1, abort, status, site, n);
}

// Before the CTA exits, wait (bounded) for the copies of the stages issued
// last, so that no bulk copy lands after the CTA has left.  `n` is the end
// marker's stage: it reused the slot of stage n - S, whose copies had landed
// (acquiring the slot waited for its consumers), so stages n - S + 1 .. n - 1
// remain.
FLINT_DEV void drain_slots(Ctl& c, int n, int S, volatile int* abort, int* status) {
  for (int i = (n - S + 1 > 0 ? n - S + 1 : 0); i < n; ++i) {
    const uint32_t parity = (i / S) & 1;
    unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(&c.full[i % S], parity, kSuspendNs)) {
      if (globaltimer_ns() - t0 > kWaitNs) {
        *abort = 1;
        record_timeout(status, 9, i);
        break;
      }
    }
  }
}

// The lane's 32 B-operand K values of one slice (token row `brow`, already
// offset to the slice; nullptr = zero column).
FLINT_DEV void load_b(uint4 (&xb)[4], const uint16_t* brow, int t, bool l2_only) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (!brow) xb[q] = make_uint4(0, 0, 0, 0);
    else xb[q] = l2_only ? ldg_cg_v4(brow + 32 * t + 8 * q) : ldg_nc_v4(brow + 32 * t + 8 * q);
  }
}

// The same from activation rows staged in shared memory.
FLINT_DEV void load_b_smem(uint4 (&xb)[4], const uint16_t* brow, int t) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    xb[q] = brow ? *reinterpret_cast<const uint4*>(brow + 32 * t + 8 * q) : make_uint4(0, 0, 0, 0);
}

// 8 mma of one 128-K slice against one 8-token B tile.  The slice is
// accumulated from zero and then added to `acc` with an fp32 add, so the
// tensor core's own accumulation only ever spans 128 products.
FLINT_DEV void mma_b(float (&acc)[4], const uint32_t (&af)[4][2][4], const uint4 (&xb)[4]) {
  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t b00 = __byte_perm(xb[q].x, xb[q].z, 0x5410);
    const uint32_t b01 = __byte_perm(xb[q].x, xb[q].z, 0x7632);
    const uint32_t b10 = __byte_perm(xb[q].y, xb[q].w, 0x5410);
    const uint32_t b11 = __byte_perm(xb[q].y, xb[q].w, 0x7632);
    mma_bf16_16816(d, af[q][0][0], af[q][0][1], af[q][0][2], af[q][0][3], b00, b01);
    mma_bf16_16816(d, af[q][1][0], af[q][1][1], af[q][1][2], af[q][1][3], b10, b11);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] += d[i];
}

// A fragments of slice s from smem rows `rg` (row g) and `rg8` (row g + 8).
FLINT_DEV void frags_fp4(uint32_t (&af)[4][2][4], const uint8_t* rg, const uint8_t* rg8,
                         const uint8_t* sg, const uint8_t* sg8, int s, int t) {
  Fp4Slice d;
  d.c0 = *reinterpret_cast<const uint4*>(rg + s * (kSliceK / 2) + 16 * t);
  d.c1 = *reinterpret_cast<const uint4*>(rg8 + s * (kSliceK / 2) + 16 * t);
  d.s0 = *reinterpret_cast<const uint16_t*>(sg + s * (kSliceK / 16) + 2 * t);
  d.s1 = *reinterpret_cast<const uint16_t*>(sg8 + s * (kSliceK / 16) + 2 * t);
  a_frags(d, af);
}

FLINT_DEV void frags_bf16(uint32_t (&af)[4][2][4], const uint8_t* rg, const uint8_t* rg8, int s,
                          int t) {
  Bf16Slice d;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    d.r0[q] = *reinterpret_cast<const uint4*>(rg + 2 * (s * kSliceK + 32 * t + 8 * q));
    d.r1[q] = *reinterpret_cast<const uint4*>(rg8 + 2 * (s * kSliceK + 32 * t + 8 * q));
  }
  a_frags(d, af);
}

// A fragments of slice s on the f16 path (the few-token gate/up when the f16
// copy of x is exact): byte b of a row's 16 code bytes of this thread ->
// (K 2b, 2b + 1) by the hardware e2m1 -> f16 conversion, times the f16 block
// scale; each mma gets the same K set as on the bf16 path (bytes 0, 2 of a
// word, then 1, 3), so it sums the same products.
FLINT_DEV void frags_fp4_f16(uint32_t (&af)[4][2][4], const uint8_t* rg, const uint8_t* rg8,
                             const uint8_t* sg, const uint8_t* sg8, int s, int t) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(rg + s * (kSliceK / 2) + 16 * t);
  const uint4 c1 = *reinterpret_cast<const uint4*>(rg8 + s * (kSliceK / 2) + 16 * t);
  const uint32_t s0 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sg + s * (kSliceK / 16) + 2 * t));
  const uint32_t s1 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sg8 + s * (kSliceK / 16) + 2 * t));
  const uint32_t wg[4] = {c0.x, c0.y, c0.z, c0.w};
  const uint32_t wg8[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t sq = f16x2_bcast(s0, q >= 2), sq8 = f16x2_bcast(s1, q >= 2);
    uint32_t p[4], p8[4];
    e2m1x8_to_f16x2(wg[q], p);
    e2m1x8_to_f16x2(wg8[q], p8);
#pragma unroll
    for (int r = 0; r < 2; ++r) {  // mma r: K {2r, 2r + 1} and {2r + 4, 2r + 5} of the word
      af[q][r][0] = f16x2_mul(p[r], sq);
      af[q][r][1] = f16x2_mul(p8[r], sq8);
      af[q][r][2] = f16x2_mul(p[r + 2], sq);
      af[q][r][3] = f16x2_mul(p8[r + 2], sq8);
    }
  }
}

// 8 mma of one 128-K slice on the f16 path: B is the f16 copy of x in natural
// order (word 0 of a 16-byte chunk holds K 0, 1, word 2 K 4, 5, ...).
FLINT_DEV void mma_b16(float (&acc)[4], const uint32_t (&af)[4][2][4], const uint4 (&xb)[4]) {
  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    mma_f16_16816(d, af[q][0][0], af[q][0][1], af[q][0][2], af[q][0][3], xb[q].x, xb[q].z);
    mma_f16_16816(d, af[q][1][0], af[q][1][1], af[q][1][2], af[q][1][3], xb[q].y, xb[q].w);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] += d[i];
}

// =============================================================== gate/up ==
// Tiles: shared expert, 8 intermediate rows each (tile rows 0..7 gate rows
// r0.., rows 8..15 up rows SI + r0..), stages of up to 1024 K; then routed
// (expert u, 16 intermediate rows), smem rows 0..15 gate, 16..31 up, stages
// of up to 2048 K.  Shared tiles go round-robin over the CTAs; the routed
// tiles (U * I / 16 of them, expert-major) in contiguous chunks, so that
// consecutive tiles of a CTA share an expert.  For few tokens the routed
// tiles' activation rows are copied into shared memory once per CTA.
//
// Consumer warp w: routed stages -> 16-row A tile a = w & 1 (gate/up rows
// 8a..8a+7), K slices s = w >> 1 (mod 8); shared stages -> the one A tile,
// K slices s = w (mod 8), warps 8..15 idle.  Token n-tiles are taken NTG at
// a time in registers; each warp adds its partial sums for the tile into its
// own smem rows of one of two alternating buffers (red) and goes on; the
// epilogue warp sums them over the warps in a fixed order, writes act (or
// sact) and releases the buffer.
// What the epilogue warp needs of a finished tile (the stage's info may be
// overwritten by then).
struct EpiRec {
  int kind;  // 0 shared, 1 routed, -1 no more tiles
  int r0, e, off, cnt, f16p;
  float gs;  // routed, few tokens: the expert's global scale (loaded while the tile is summed)
  int exp[32];  // f16 path: scale exponent of pair nn's token (nn < cnt <= 16)
};

struct GuSmem {
  Ctl ctl;              // bar[b]: the consumers' partials of a tile of parity b are written
  uint64_t redfree[2];  // the epilogue warp has read partial-sum buffer b
  uint64_t xfull;       // the staged activation rows have landed
  EpiRec er[2];
  GuInfo info[kGuMaxStages];
};

struct GuLayout {
  int stages;
  size_t red, xs, xpitch, ctl, total;  // xpitch = 0: activations not staged
};

// Activation rows of the routed tiles are staged in shared memory once per
// CTA when they fit (few tokens): M rows, padded by 16 bytes against bank
// conflicts between tokens.
__host__ __device__ inline GuLayout gu_layout(int M, int H) {
  const int ntmax = (M + 7) / 8;
  GuLayout L;
  const size_t red_bytes = size_t(kCons) * ntmax * 32 * 16;
  L.xpitch = 0;
  size_t xs_bytes = 0;
  if (M <= kX16MaxTokens && size_t(M) * (2 * H + 16) <= kXsMaxBytes) {
    L.xpitch = 2 * size_t(H) + 16;
    xs_bytes = size_t(M) * L.xpitch;
  }
  const size_t room = kMaxSmem - sizeof(GuSmem) - 2 * red_bytes - xs_bytes;
  L.stages = (int)(room / kGuStageBytes);
  if (L.stages > kGuMaxStages) L.stages = kGuMaxStages;
  L.red = size_t(L.stages) * kGuStageBytes;
  L.xs = L.red + 2 * red_bytes;
  L.ctl = L.xs + xs_bytes;
  L.total = L.ctl + sizeof(GuSmem);
  return L;
}

FLINT_DEV void gu_issue_shared(const MoEArgs& a, uint8_t* stage, GuInfo& inf, uint64_t* full,
                               int tile, int k0, int lane) {
  const int H = a.H, SI = a.SI;
  const int kst = min(H - k0, kGuKst16);
  const int pitch = 2 * kst + kPad;
  const int r0 = tile * 8;
  if (lane == 0) {
    inf.kind = 0; inf.first = (k0 == 0); inf.last = (k0 + kst >= H);
    inf.k0 = k0; inf.kst = kst; inf.pitch = pitch; inf.sf_off = 0; inf.sf_pitch = 0;
    inf.r0 = r0; inf.e = -1; inf.cnt = a.M; inf.off = 0;
    mbar_arrive_expect_tx(full, 16u * 2u * kst);
  }
  __syncwarp();
  if (lane < 16) {
    const int row = lane < 8 ? r0 + lane : SI + r0 + (lane - 8);
    bulk_g2s(stage + lane * pitch, a.shared_gu + (size_t)row * H + k0, 2u * kst, full);
  }
}

FLINT_DEV void gu_issue_routed(const MoEArgs& a, uint8_t* stage, GuInfo& inf, uint64_t* full,
                               int e, int r0, int k0, int lane) {
  const int H = a.H, I = a.I;
  const int kst = min(H - k0, kGuKst4);
  const bool whole = (kst == H);  // whole rows: 16 gate (up) rows are one block
  const int pitch = whole ? kst / 2 : kst / 2 + kPad;
  const int sf_off = 32 * pitch;
  const int sfp = kst / 16;
  const size_t g0 = (size_t)e * 2 * I + r0;  // first gate row
  const size_t u0 = g0 + I;                  // first up row
  if (lane == 0) {
    inf.kind = 1; inf.first = (k0 == 0); inf.last = (k0 + kst >= H);
    inf.k0 = k0; inf.kst = kst; inf.pitch = pitch; inf.sf_off = sf_off; inf.sf_pitch = sfp;
    inf.r0 = r0; inf.e = e;
    mbar_arrive_expect_tx(full, 32u * (kst / 2) + 32u * sfp);
  }
  __syncwarp();
  if (whole) {  // four copies in one instruction: lanes 0, 1 the gate and up
                // codes, lanes 2, 3 their scale rows
    if (lane < 4) {
      const size_t row = (lane & 1) ? u0 : g0;
      const bool sc = lane >= 2;
      uint8_t* dst = stage + (sc ? sf_off + (lane & 1) * 16 * sfp : (lane & 1) * 16 * pitch);
      const uint8_t* src = sc ? a.w13_sf + row * (H / 16) : a.w13 + row * (H / 2);
      bulk_g2s(dst, src, sc ? 16u * sfp : 16u * (H / 2), full);
    }
  } else {  // a K chunk of each row, rows padded against bank conflicts
    const size_t row = lane < 16 ? g0 + lane : u0 + (lane - 16);
    bulk_g2s(stage + lane * pitch, a.w13 + row * (H / 2) + k0 / 2, kst / 2, full);
    bulk_g2s(stage + sf_off + lane * sfp, a.w13_sf + row * (H / 16) + k0 / 16, sfp, full);
  }
}

// NTG: token n-tiles held in registers at a time (1 when M <= 8).
template <int NTG>
__global__ void __launch_bounds__(kGuThreads, 1) gate_up2_kernel(MoEArgs a) {
  SpanGuard<kSpanGateUp> span_guard;
  extern __shared__ __align__(128) uint8_t smem[];
  const GuLayout L = gu_layout(a.M, a.H);
  const int S = L.stages;
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + L.red);
  uint8_t* xs = smem + L.xs;
  const int xpitch = (int)L.xpitch;
  GuSmem& SM = *reinterpret_cast<GuSmem*>(smem + L.ctl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int H = a.H, I = a.I, SI = a.SI, M = a.M;
  const int ntmax = (M + 7) / 8;
  const int G = gridDim.x, c = blockIdx.x;
  int* status = a.ws.status;
  volatile int* abort = &SM.ctl.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&SM.ctl.full[i], 1);
      mbar_init(&SM.ctl.empty[i], kCons);
    }
    mbar_init(&SM.ctl.bar[0], kCons);
    mbar_init(&SM.ctl.bar[1], kCons);
    mbar_init(&SM.redfree[0], 1);
    mbar_init(&SM.redfree[1], 1);
    mbar_init(&SM.xfull, 1);
    SM.ctl.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // two partial-sum buffers, alternating per tile: the epilogue warp reads
  // one while the consumers fill the other
  const size_t red_floats = (size_t)kCons * ntmax * 32 * 4;

  if (warp == kEpi) {
    // ---------------------------------------------------------- epilogue
    // Tile j: sum the consumers' partials in a fixed order, apply the
    // scales and the activation, write act (routed) or sact (shared).
    bool triggered = false;
    for (int j = 0;; ++j) {
      const int b = j & 1;
      if (!warp_wait_phase(&SM.ctl.bar[b], (j >> 1) & 1, abort, status, lane, 5, j)) break;
      const EpiRec& er = SM.er[b];
      const int kind = er.kind;
      if (kind < 0) break;
      if (kind == 1 && !triggered) {  // routed tiles follow the router's completion
        pdl_launch_dependents();
        triggered = true;
      }
      const float4* red4 = reinterpret_cast<const float4*>(red + b * red_floats);
      const int cnt = er.cnt, ntiles = (cnt + 7) / 8, r0 = er.r0, off = er.off;
      if (kind == 1) {
        // bf16 path: 2^7 undoes the operand scaling; f16 path: 2^-exp of the
        // token undoes the activations' scaling
        // (many tokens: the consumers have no register to spare for it)
        const float egs = NTG == 1 ? er.gs : a.w13_gs[er.e];
        const float gs = er.f16p ? egs : egs * 128.0f;
        for (int it = 0; it < 2 * ntiles; ++it) {
          const int at = it & 1, nt = it >> 1;
          float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          for (int kp = 0; kp < kKP; ++kp) {
            const float4 p = red4[((size_t)(at + 2 * kp) * ntmax + nt) * 32 + lane];
            v[0] += p.x; v[1] += p.y; v[2] += p.z; v[3] += p.w;
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int nn = nt * 8 + 2 * t + cc;
            if (nn < cnt) {
              const float f = er.f16p ? gs * pow2f(-er.exp[nn]) : gs;
              const float gv = v[cc] * f, uv = v[2 + cc] * f;
              a.ws.act[(size_t)(off + nn) * I + r0 + 8 * at + g] = (uint16_t)act_bits(gv, uv);
            }
          }
        }
      } else {
        // shared tile: warp w < 8 left the (sum, compensation) pair of its K
        // slices in its own slots and in warp w + 8's; they are added in warp
        // order with TwoSum
        for (int nt = 0; nt < ntiles; ++nt) {
          float S[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          for (int w = 0; w < 8; ++w) {
            const float4 p = red4[((size_t)w * ntmax + nt) * 32 + lane];
            const float4 q = red4[((size_t)(w + 8) * ntmax + nt) * 32 + lane];
            two_sum(S[0], C[0], p.x); two_sum(S[1], C[1], p.y);
            two_sum(S[2], C[2], p.z); two_sum(S[3], C[3], p.w);
            C[0] = __fadd_rn(C[0], q.x); C[1] = __fadd_rn(C[1], q.y);
            C[2] = __fadd_rn(C[2], q.z); C[3] = __fadd_rn(C[3], q.w);
          }
          const float v[4] = {__fadd_rn(S[0], C[0]), __fadd_rn(S[1], C[1]), __fadd_rn(S[2], C[2]),
                              __fadd_rn(S[3], C[3])};
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int nn = nt * 8 + 2 * t + cc;
            if (nn < cnt) {
              // stock BF16 SwiGLU: gS, uS rounded, silu(gS) = gS / (1 + exp(-gS))
              const float gS = round_bf16(v[cc]), uS = round_bf16(v[2 + cc]);
              a.ws.sact[(size_t)nn * SI + r0 + g] = (uint16_t)sact_bits(gS, uS);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&SM.redfree[b]);  // buffer b (and er[b]) free again
    }
    if (!triggered) pdl_launch_dependents();
    return;
  }

  if (warp == kCons) {
    // ------------------------------------------------------------ producer
    int n = 0;
    const int nS = SI / 8;
    for (int tile = c; tile < nS; tile += G) {
      for (int k0 = 0; k0 < H; k0 += kGuKst16) {
        int ok = 1;
        if (lane == 0) ok = acquire_slot(SM.ctl, n, S, abort, status, 1);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int sl = n % S;
        gu_issue_shared(a, stages + (size_t)sl * kGuStageBytes, SM.info[sl], &SM.ctl.full[sl],
                        tile, k0, lane);
        ++n;
      }
    }
    pdl_wait();  // router finished: routing records are final
    pdl_launch_dependents();
    // one token routes to k distinct experts, so U needs no read then, and
    // the first record's loads go out with the f16-copy report
    const int U = M == 1 ? a.k : ldg_cg_i32(a.ws.uniq);
    const int tpe = I / 16;  // tiles per expert
    const int T = U * tpe;
    const int lo = (int)((long long)T * c / G), hi = (int)((long long)T * (c + 1) / G);
    int r_hdr = 0, r_p0 = 0, r_p1 = 0;  // the record of expert slot lo / tpe, in flight
    auto load_record = [&](int u) {
      const int* rec = a.ws.urec + (size_t)u * kUrecInts;
      r_hdr = lane < 3 ? ldg_cg_i32(rec + lane) : 0;
      r_p0 = ldg_cg_i32(rec + 4 + lane);
      r_p1 = ldg_cg_i32(rec + 36 + lane);
    };
    if (lo < hi) load_record(lo / tpe);
    const int x16 = (M <= kX16MaxTokens && ldg_cg_i32(a.ws.glob_cnt + 1) == 0) ? 1 : 0;
    const bool staged = xpitch && lo < hi;
    if (staged) {  // the routed tiles' activation rows, once: the f16 copy or x
      fence_proxy_async_global();  // the router's f16 copy, read by bulk copies
      const uint16_t* src = x16 ? a.ws.x16 : a.x;
      if (lane == 0) mbar_arrive_expect_tx(&SM.xfull, (uint32_t)M * 2u * H);
      __syncwarp();
      for (int tk = lane; tk < M; tk += 32)
        bulk_g2s(xs + (size_t)tk * xpitch, src + (size_t)tk * H, 2u * H, &SM.xfull);
    }
    int cur_u = -1, e = 0, cnt = 0, off = 0;
    short tok0 = 0, tok1 = 0;
    for (int tile = lo; tile < hi; ++tile) {
      const int u = tile / tpe, r0 = (tile % tpe) * 16;
      if (u != cur_u) {  // the expert's record: one round trip, lanes in parallel
        if (tile != lo) load_record(u);
        e = __shfl_sync(0xffffffffu, r_hdr, 0);
        cnt = __shfl_sync(0xffffffffu, r_hdr, 1);
        off = __shfl_sync(0xffffffffu, r_hdr, 2);
        tok0 = lane < cnt ? (short)(r_p0 / a.k) : 0;
        tok1 = lane + 32 < cnt ? (short)(r_p1 / a.k) : 0;
        cur_u = u;
      }
      for (int k0 = 0; k0 < H; k0 += kGuKst4) {
        int ok = 1;
        if (lane == 0) ok = acquire_slot(SM.ctl, n, S, abort, status, 2);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int sl = n % S;
        GuInfo& inf = SM.info[sl];
        inf.tok[lane] = tok0;
        inf.tok[lane + 32] = tok1;
        if (lane == 0) { inf.cnt = cnt; inf.off = off; inf.x16 = x16; }
        __syncwarp();  // info complete before the arrive that publishes it
        gu_issue_routed(a, stages + (size_t)sl * kGuStageBytes, inf, &SM.ctl.full[sl], e, r0, k0,
                        lane);
        ++n;
      }
    }
    // end marker: a stage with no copies (consumers that gave up have
    // left already; the bounded waits keep this from blocking)
    if (lane == 0) {
      if (acquire_slot(SM.ctl, n, S, abort, status, 3)) {
        const int sl = n % S;
        SM.info[sl].kind = -1;
        mbar_arrive(&SM.ctl.full[sl]);
      }
      drain_slots(SM.ctl, n, S, abort, status);
      if (staged) {  // no copy outlives the CTA
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(&SM.xfull, 0, kSuspendNs)) {
          if (globaltimer_ns() - t0 > kWaitNs) {
            *abort = 1;
            record_timeout(status, 7, n);
            break;
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  bool triggered = false, waited = false, xready = false;
  int ep = 0;  // tiles handed to the epilogue warp
  for (int n = 0;; ++n) {
    const int sl = n % S;
    if (!warp_wait_phase(&SM.ctl.full[sl], (n / S) & 1, abort, status, lane, 4, n)) break;
    const GuInfo& inf = SM.info[sl];
    const int kind = inf.kind;
    if (kind != 0 && !triggered) {  // past the producer's dependency wait
      pdl_launch_dependents();
      triggered = true;
    }
    if (kind == 1 && !waited) {  // the router's outputs (the f16 copy of x) are visible
      pdl_wait();
      waited = true;
    }
    const int b = ep & 1;
    // buffer b (partials and the epilogue record) was last used by tile ep - 2
    if ((kind < 0 || inf.first) && ep >= 2 &&
        !warp_wait_phase(&SM.redfree[b], ((ep >> 1) - 1) & 1, abort, status, lane, 10, ep))
      break;
    if (kind < 0) {  // no more tiles: tell the epilogue warp
      if (warp == 0 && lane == 0) SM.er[b].kind = -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&SM.ctl.bar[b]);
      break;
    }
    const bool xsm = kind == 1 && xpitch;  // activations from the staged rows
    if (xsm && !xready) {
      if (!warp_wait_phase(&SM.xfull, 0, abort, status, lane, 6, n)) break;
      xready = true;
    }
    float4* myred = reinterpret_cast<float4*>(red + b * red_floats) + (size_t)warp * ntmax * 32 + lane;
    const int first = inf.first, last = inf.last, k0 = inf.k0, kst = inf.kst;
    const int pitch = inf.pitch, cnt = inf.cnt;
    const int ntiles = (cnt + 7) / 8;
    const uint8_t* st = stages + (size_t)sl * kGuStageBytes;
    const int nsl = kst / kSliceK;
    // this warp's rows and K slices
    int s0, sstep;
    const uint8_t *rg, *rg8, *sg = nullptr, *sg8 = nullptr;
    if (kind == 1) {
      const int at = warp & 1;
      s0 = warp >> 1;
      sstep = kKP;
      rg = st + (8 * at + g) * pitch;
      rg8 = st + (16 + 8 * at + g) * pitch;
      sg = st + inf.sf_off + (8 * at + g) * inf.sf_pitch;
      sg8 = st + inf.sf_off + (16 + 8 * at + g) * inf.sf_pitch;
    } else {
      s0 = warp < 8 ? warp : nsl;
      sstep = 8;
      rg = st + g * pitch;
      rg8 = st + (8 + g) * pitch;
    }
    if (kind == 0) {
      // ---- shared tile: warp w < 8 sums its K slices s = w (mod 8) of
      // every token tile exactly (the shared activation of a token feeds all
      // of its outputs) into a (sum, compensation) pair, carried from stage
      // to stage in the partial buffer: the sum in its own slot, the
      // compensation in idle warp w + 8's
      if (warp < 8) {
        for (int nt = 0; nt < ntiles; ++nt) {
          float S_[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C_[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          float4* rs = reinterpret_cast<float4*>(red + b * red_floats) + ((size_t)warp * ntmax + nt) * 32 + lane;
          float4* rc =
              reinterpret_cast<float4*>(red + b * red_floats) + ((size_t)(warp + 8) * ntmax + nt) * 32 + lane;
          if (!first) {
            const float4 o = *rs, q = *rc;
            S_[0] = o.x; S_[1] = o.y; S_[2] = o.z; S_[3] = o.w;
            C_[0] = q.x; C_[1] = q.y; C_[2] = q.z; C_[3] = q.w;
          }
          const int nn = nt * 8 + g;
          const uint16_t* brow = nn < cnt ? a.x + (size_t)nn * H + k0 : nullptr;
          for (int s = warp; s < nsl; s += 8) {
            uint4 xb[4];
            load_b(xb, brow ? brow + s * kSliceK : nullptr, t, false);
            slice_bf16_exact(S_, C_, reinterpret_cast<const uint16_t*>(rg) + s * kSliceK + 32 * t,
                             reinterpret_cast<const uint16_t*>(rg8) + s * kSliceK + 32 * t, xb);
          }
          *rs = make_float4(S_[0], S_[1], S_[2], S_[3]);
          *rc = make_float4(C_[0], C_[1], C_[2], C_[3]);
        }
      }
      if (last && warp == 0) {  // the tile's record, before the stage slot is released
        EpiRec& er = SM.er[b];
        if (lane == 0) {
          er.kind = kind; er.r0 = inf.r0; er.e = inf.e; er.off = inf.off; er.cnt = cnt;
          er.f16p = 0;
        }
        er.exp[lane] = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&SM.ctl.empty[sl]);  // stage consumed
      if (!last) continue;
      if (lane == 0) mbar_arrive(&SM.ctl.bar[b]);  // partials (and record) of tile ep written
      ++ep;
      continue;
    }
    const bool f16p = kind == 1 && inf.x16;
    // the scale exponent of this lane's pair (f16 path) and the expert's
    // global scale, for the epilogue record: loaded now, used after the sums
    const int cexp =
        f16p && last && warp == 0 && lane < cnt ? ldg_cg_i32(a.ws.x16_exp + inf.tok[lane]) : 0;
    const float egs = NTG == 1 && last && warp == 0 && lane == 0 ? ldg_cg_f32(a.w13_gs + inf.e) : 0.0f;
    for (int n0 = 0; n0 < ntiles; n0 += NTG) {
      float acc[NTG][4];
      const uint16_t* brow[NTG];
#pragma unroll
      for (int i = 0; i < NTG; ++i) {
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        const int nn = (n0 + i) * 8 + g;
        if (nn >= cnt) brow[i] = nullptr;
        else if (xsm) brow[i] = reinterpret_cast<const uint16_t*>(xs + (size_t)inf.tok[nn] * xpitch) + k0;
        else brow[i] = (f16p ? a.ws.x16 : a.x) + (size_t)(kind ? inf.tok[nn] : nn) * H + k0;
      }
      for (int s = s0; s < nsl; s += sstep) {
        // activations first: their load latency hides behind the dequant
        uint4 xb[NTG][4];
#pragma unroll
        for (int i = 0; i < NTG; ++i) {
          const uint16_t* bp = (n0 + i < ntiles && brow[i]) ? brow[i] + s * kSliceK : nullptr;
          if (xsm) load_b_smem(xb[i], bp, t);
          else load_b(xb[i], bp, t, false);
        }
        uint32_t af[4][2][4];
        if (f16p) {
          frags_fp4_f16(af, rg, rg8, sg, sg8, s, t);
#pragma unroll
          for (int i = 0; i < NTG; ++i)
            if (n0 + i < ntiles) mma_b16(acc[i], af, xb[i]);
        } else {
          if (kind == 1) frags_fp4(af, rg, rg8, sg, sg8, s, t);
          else frags_bf16(af, rg, rg8, s, t);
#pragma unroll
          for (int i = 0; i < NTG; ++i)
            if (n0 + i < ntiles) mma_b(acc[i], af, xb[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < NTG; ++i) {
        if (n0 + i < ntiles) {
          float4* r = myred + (size_t)(n0 + i) * 32;
          float4 v = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
          if (!first) {
            const float4 o = *r;
            v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
          }
          *r = v;
        }
      }
    }
    if (last && warp == 0) {  // the tile's record, before the stage slot is released
      EpiRec& er = SM.er[b];
      if (lane == 0) {
        er.kind = kind; er.r0 = inf.r0; er.e = inf.e; er.off = inf.off; er.cnt = cnt;
        er.f16p = f16p ? 1 : 0;
        er.gs = egs;
      }
      er.exp[lane] = cexp;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&SM.ctl.empty[sl]);  // stage consumed
    if (!last) continue;
    if (lane == 0) mbar_arrive(&SM.ctl.bar[b]);  // partials (and record) of tile ep written
    ++ep;
  }
  if (!triggered) pdl_launch_dependents();
}

// ================================================================== down ==
// CTA hb owns output rows h0 = 16 hb .. h0 + 15 for every token.  Weight
// blocks: the shared expert's 16 rows (BF16, SI <= 1024 K) and, per routed
// expert u < U, its 16 rows of w2 (NVFP4, I <= 2048 K) with their scales,
// packed in order into stages of up to 8 blocks.  Work items are (block,
// 8-token n-tile); warp w takes items w, w + 16, ... of a stage and runs the
// whole K of its item, so no cross-warp reduction is needed.  Results go to
// smem: y (bf16, per pair t * k + j) and ys (bf16, per token); after the last
// stage the CTA forms out = bf16(bf16(sum_j tw_j y_j) + ys) for its rows.
// A stage with at most 8 items gives each item P = 2 warps, one per half of
// its K slices; parts 1 .. P - 1 hand their fp32 partials to
// part 0 through shared memory (a float4 per lane) and a per-part flag
// holding the stage number + 1; part 0 adds them in part order.
constexpr int kDnPartSlots = kCons / 2;  // items * (P - 1) when P = 2

struct DnSmem {
  Ctl ctl;
  DnInfo info[kDnStages];
  int flag[kDnStages][kDnPartSlots];
  float4 part[kDnStages][kDnPartSlots][32];
};

// Byte offsets in the down kernel's dynamic smem: stages, y, ys, control.
struct DnLayout {
  size_t y, ys, tw, ctl, total;
};
__host__ __device__ inline DnLayout dn_layout(int M, int k) {
  DnLayout L;
  L.y = size_t(kDnStages) * kDnStageBytes;
  L.ys = L.y + (size_t(M) * k * 16 * 2 + 15) / 16 * 16;
  L.tw = L.ys + (size_t(M) * 16 * 2 + 15) / 16 * 16;
  L.ctl = L.tw + (size_t(M) * k * 4 + 15) / 16 * 16;
  L.total = L.ctl + sizeof(DnSmem);
  return L;
}

// Weight rows of a block sit unpadded in smem (16 consecutive rows are one
// contiguous block in global memory, so one copy brings them in).
FLINT_DEV int dn_block_bytes(int kind, int I, int SI) {
  return kind ? 16 * (I / 2) + I : 16 * (2 * SI);
}

__global__ void __launch_bounds__(kThreads, 1) down2_kernel(MoEArgs a) {
  SpanGuard<kSpanDown> span_guard;
  extern __shared__ __align__(128) uint8_t smem[];
  // the next kernel may start now: a router launched after this one loads
  // only its weights before its own dependency wait
  pdl_launch_dependents();
  uint8_t* stages = smem;
  const DnLayout L = dn_layout(a.M, a.k);
  uint16_t* ysm = reinterpret_cast<uint16_t*>(smem + L.y);
  uint16_t* yss = reinterpret_cast<uint16_t*>(smem + L.ys);
  float* tws = reinterpret_cast<float*>(smem + L.tw);
  DnSmem& SM = *reinterpret_cast<DnSmem*>(smem + L.ctl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int H = a.H, I = a.I, SI = a.SI, k = a.k, M = a.M;
  const int h0 = blockIdx.x * 16;
  int* status = a.ws.status;
  volatile int* abort = &SM.ctl.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDnStages; ++i) {
      mbar_init(&SM.ctl.full[i], 1);
      mbar_init(&SM.ctl.empty[i], kCons);
      for (int j = 0; j < kDnPartSlots; ++j) SM.flag[i][j] = 0;
    }
    mbar_init(&SM.ctl.bar[0], kCons + 1);
    SM.ctl.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCons) {
    // ------------------------------------------------------------ producer
    // The gate/up grid released this grid only after its own dependency
    // wait, which follows the router's completion: the records are final.
    // headers of routed units [win, win + 32), one per lane; the first window
    // is read with U (records past U are allocated but unused)
    const int urows = min(a.E, M * k);  // records the workspace holds
    int win = 0, hdr_e = 0, hdr_c = 0, hdr_o = 0;
    auto load_window = [&](int w0) {
      const int ul = w0 + lane;
      if (ul < urows) {
        const int* rec = a.ws.urec + (size_t)ul * kUrecInts;
        hdr_e = ldg_cg_i32(rec);
        hdr_c = ldg_cg_i32(rec + 1);
        hdr_o = ldg_cg_i32(rec + 2);
      }
      win = w0;
    };
    load_window(0);
    const int U = ldg_cg_i32(a.ws.uniq);
    const int nsh = SI > 0 ? 1 : 0;
    const int nunits = U + nsh;
    int n = 0, unit = 0, pend = 0;  // stages [pend, n) still need their activations
    bool waited = false;
    // Activation rows of a stage: copied once the gate/up grid has finished,
    // one copy per block, all issued by one instruction of the warp (lane =
    // block); then the producer's arrival completes the stage.
    auto finish = [&](int m) {
      const int sl = m % kDnStages;
      const DnInfo& inf = SM.info[sl];
      uint8_t* st = stages + (size_t)sl * kDnStageBytes;
      if (lane == 0) mbar_expect_tx(&SM.ctl.full[sl], (uint32_t)inf.abytes);
      __syncwarp();
      if (lane < inf.nblocks && inf.blk[lane].act_smem >= 0) {
        const DnBlock& b = inf.blk[lane];
        const uint16_t* srcp = b.kind == 0 ? a.ws.sact : a.ws.act + (size_t)b.off * I;
        bulk_g2s(st + b.act_smem, srcp, (uint32_t)b.cnt * (b.kind == 0 ? SI : I) * 2u, &SM.ctl.full[sl]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&SM.ctl.full[sl]);
    };
    // Stage n takes units unit, unit + 1, ...: the longest run (at most
    // kDnMaxBlocks) whose weight rows and activation rows fit the stage and
    // whose items fit its table; a first unit whose activations alone do not
    // fit is taken with them read from global memory.  Lane l looks at unit
    // unit + l, so the plan is a few prefix sums over the lanes, and every
    // block's copies go out in one instruction of the warp: a warp issuing
    // bulk copies one lane at a time pays a round trip per copy.
    auto prefix = [&](int v) {  // inclusive prefix sum over lanes 0 .. kDnMaxBlocks - 1
#pragma unroll
      for (int o = 1; o < kDnMaxBlocks; o <<= 1) {
        const int w = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += w;
      }
      return v;
    };
    while (unit < nunits) {
      int ok = 1;
      if (lane == 0) ok = acquire_slot(SM.ctl, n, kDnStages, abort, status, 11);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int sl = n % kDnStages;
      uint8_t* st = stages + (size_t)sl * kDnStageBytes;
      DnInfo& inf = SM.info[sl];
      // a stage holds at most kDnMaxBlocks units: move the window if needed
      if (unit - nsh + kDnMaxBlocks > win + 32) load_window(max(unit - nsh, 0));
      const int cu = unit + lane;
      const bool cand = lane < kDnMaxBlocks && cu < nunits;
      const bool shared = nsh && cu == 0;
      const int hl = (cu - nsh - win) & 31;  // lane holding this unit's header
      const int he = __shfl_sync(0xffffffffu, hdr_e, hl);
      const int hc = __shfl_sync(0xffffffffu, hdr_c, hl);
      const int ho = __shfl_sync(0xffffffffu, hdr_o, hl);
      const int cnt = shared ? M : hc;
      const int wb = cand ? dn_block_bytes(shared ? 0 : 1, I, SI) : 0;
      const int ab = cand ? cnt * (shared ? SI : I) * 2 : 0;
      const int nit = cand ? (cnt + 7) / 8 : 0;
      const int pit = prefix(nit);
      int sz = wb + ab;
      int pre = prefix(sz);
      bool fit = cand && pre <= kDnStageBytes && pit <= kDnMaxItems;
      const bool lone = __shfl_sync(0xffffffffu, fit ? 1 : 0, 0) == 0;
      if (lone) {  // the first unit with its activations read from global memory
        if (lane == 0) sz = wb;
        pre = prefix(sz);
        fit = cand && pre <= kDnStageBytes && pit <= kDnMaxItems;
      }
      const int nb = __popc(__ballot_sync(0xffffffffu, fit));  // fit holds for lanes 0 .. nb - 1
      if (nb == 0) {  // cannot happen for supported shapes; never spin on it
        if (lane == 0) { *abort = 1; record_timeout(status, 12, n); }
        break;
      }
      const bool mine = lane < nb;
      const bool staged = mine && !(lone && lane == 0);
      const int at = pre - sz;  // byte offset of this block's weight rows in the stage
      if (mine) {
        DnBlock& b = inf.blk[lane];
        b.kind = shared ? 0 : 1; b.e = shared ? -1 : he; b.u = cu - nsh;
        b.cnt = cnt; b.off = ho; b.smem = at;
        b.pitch = shared ? 2 * SI : I / 2;
        b.act_smem = staged ? at + wb : -1;
        for (int i = 0; i < nit; ++i) {
          inf.item_blk[pit - nit + i] = (unsigned char)lane;
          inf.item_nt[pit - nit + i] = (unsigned char)i;
        }
      }
      const uint32_t wbytes = __reduce_add_sync(0xffffffffu, mine ? (uint32_t)wb : 0u);
      const uint32_t abytes = __reduce_add_sync(0xffffffffu, staged ? (uint32_t)ab : 0u);
      const int ni = __shfl_sync(0xffffffffu, pit, nb - 1);
      if (lane == 0) {
        inf.nblocks = nb; inf.nitems = ni; inf.abytes = (int)abytes;
        mbar_expect_tx(&SM.ctl.full[sl], wbytes);
      }
      __syncwarp();
      // weights (known before the dependency wait): the block's rows, then
      // a routed block's scale rows
      const size_t row0 = (size_t)he * H + h0;
      if (mine) {
        const uint8_t* srcp = shared ? reinterpret_cast<const uint8_t*>(a.shared_down + (size_t)h0 * SI)
                                     : a.w2 + row0 * (I / 2);
        bulk_g2s(st + at, srcp, shared ? 16u * 2u * SI : 16u * (I / 2), &SM.ctl.full[sl]);
      }
      if (mine && !shared)
        bulk_g2s(st + at + 16 * (I / 2), a.w2_sf + row0 * (I / 16), 16u * (I / 16), &SM.ctl.full[sl]);
      unit += nb;
      ++n;
      if (waited) {
        finish(n - 1);
        pend = n;
      } else if (n - pend == kDnPrefetch || unit >= nunits) {
        pdl_wait();  // gate/up finished: act and sact are complete
        fence_proxy_async_global();
        waited = true;
        for (; pend < n; ++pend) finish(pend);
      }
    }
    if (!waited) {  // nothing was planned (or the ring gave up): keep the order
      pdl_wait();
      waited = true;
      for (; pend < n; ++pend) finish(pend);
    }
    if (lane == 0) {
      if (acquire_slot(SM.ctl, n, kDnStages, abort, status, 13)) {
        const int sl = n % kDnStages;
        SM.info[sl].nblocks = 0;
        mbar_arrive(&SM.ctl.full[sl]);
      }
      drain_slots(SM.ctl, n, kDnStages, abort, status);
    }
    // the combine's weights (final since the router finished), staged while
    // the consumers work
    for (int i = lane; i < M * k; i += 32) tws[i] = ldg_cg_f32(a.ws.tw + i);
    // the combine below needs every consumer's results
    uint32_t ph = 0;
    warp_barrier(&SM.ctl.bar[0], ph, abort, status, lane, 14);
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();  // gate/up finished: act and sact are complete
  if (blockIdx.x == 0 && threadIdx.x == 0) a.ws.glob_cnt[1] = 0;  // f16-copy report consumed
  for (int n = 0;; ++n) {
    const int sl = n % kDnStages;
    if (!warp_wait_phase(&SM.ctl.full[sl], (n / kDnStages) & 1, abort, status, lane, 15, n)) break;
    const DnInfo& inf = SM.info[sl];
    if (inf.nblocks == 0) break;
    const uint8_t* st = stages + (size_t)sl * kDnStageBytes;
    const int P = inf.nitems <= kCons / 2 ? 2 : 1;  // K parts per item
    const int kp = warp % P;                                     // this warp's part
    for (int it = warp / P; it < inf.nitems; it += kCons / P) {
      const DnBlock& b = inf.blk[inf.item_blk[it]];
      const int nt = inf.item_nt[it];
      const int nn = nt * 8 + g;  // token column of this lane
      const uint8_t* rg = st + b.smem + g * b.pitch;
      const uint8_t* rg8 = st + b.smem + (8 + g) * b.pitch;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const bool routed = b.kind == 1;
      const int K = routed ? I : SI;
      const int ncnt = routed ? b.cnt : M;
      // this lane's pair ids (routed), read early: used only at the end
      int pr[2] = {0, 0};
      if (routed) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tok = nt * 8 + 2 * t + c;
          if (tok < ncnt) pr[c] = ldg_cg_i32(a.ws.urec + (size_t)b.u * kUrecInts + 4 + tok);
        }
      }
      const uint16_t* brow = nullptr;  // global B row (activations not staged)
      const uint8_t* bsm = nullptr;    // staged B row
      if (nn < ncnt) {
        if (b.act_smem >= 0) bsm = st + b.act_smem + (size_t)nn * K * 2;
        else brow = routed ? a.ws.act + (size_t)(b.off + nn) * I : a.ws.sact + (size_t)nn * SI;
      }
      // the global scale, used only after the sums (2^7 undoes the operand scaling)
      const float gs2 = routed ? ldg_cg_f32(a.w2_gs + b.e) : 0.0f;
      const uint8_t* sg = st + b.smem + 16 * b.pitch + g * (I / 16);
      const uint8_t* sg8 = sg + 8 * (I / 16);
      const int nsl = K / kSliceK;
      const int s_lo = nsl * kp / P, s_hi = nsl * (kp + 1) / P;
      for (int s = s_lo; s < s_hi; ++s) {
        uint4 xb[4];
        if (bsm) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            xb[q] = *reinterpret_cast<const uint4*>(bsm + 2 * (s * kSliceK + 32 * t + 8 * q));
        } else {
          load_b(xb, brow ? brow + s * kSliceK : nullptr, t, true);
        }
        uint32_t af[4][2][4];
        if (routed) frags_fp4(af, rg, rg8, sg, sg8, s, t);
        else frags_bf16(af, rg, rg8, s, t);
        mma_b(acc, af, xb);
      }
      if (P > 1) {
        const int slot0 = it * (P - 1);  // slots of parts 1 .. P - 1
        if (kp) {  // hand the partials over; part 0 writes y
          SM.part[sl][slot0 + kp - 1][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
          __threadfence_block();
          __syncwarp();
          if (lane == 0 && a.fault != FLINT_FAULT_DOWN_HANDOVER)  // test hook leaves it out
            reinterpret_cast<volatile int*>(SM.flag[sl])[slot0 + kp - 1] = n + 1;
          continue;
        }
        int ok = 1;
        if (lane == 0) {
          const unsigned long long t0 = globaltimer_ns();
          for (int q = 1; q < P && ok; ++q) {
            volatile int* fl = &SM.flag[sl][slot0 + q - 1];
            while (*fl != n + 1) {
              if (*abort || globaltimer_ns() - t0 > kWaitNs) {
                if (!*abort) { *abort = 1; record_timeout(status, 17, n); }
                ok = 0;
                break;
              }
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __threadfence_block();
        for (int q = 1; q < P; ++q) {
          const float4 o = SM.part[sl][slot0 + q - 1][lane];
          acc[0] += o.x; acc[1] += o.y; acc[2] += o.z; acc[3] += o.w;
        }
      }
      if (routed) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = nt * 8 + 2 * t + (i & 1);
          if (tok < ncnt)
            ysm[(size_t)pr[i & 1] * 16 + g + (i >> 1) * 8] =
                (uint16_t)f32_to_bf16_bits(__fmul_rn(acc[i], gs2) * 128.0f);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = nt * 8 + 2 * t + (i & 1);
          if (tok < M) yss[(size_t)tok * 16 + g + (i >> 1) * 8] = (uint16_t)f32_to_bf16_bits(acc[i]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&SM.ctl.empty[sl]);
  }
  uint32_t ph = 0;
  warp_barrier(&SM.ctl.bar[0], ph, abort, status, lane, 16);
  if (*abort) return;

  // ---- combine: out = bf16(bf16(sum_j tw_j y_j) + ys), j in rank order
  for (int idx = threadIdx.x; idx < M * 16; idx += kCons * 32) {
    const int tt = idx >> 4, h = idx & 15;
    float R = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float w = tws[tt * k + j];
      R = R + w * bf16_bits_to_f32(ysm[(size_t)(tt * k + j) * 16 + h]);
    }
    const float ys = SI > 0 ? bf16_bits_to_f32(yss[tt * 16 + h]) : 0.0f;
    a.out[(size_t)tt * H + h0 + h] = (uint16_t)f32_to_bf16_bits(round_bf16(R) + ys);
  }
}

// ------------------------------------------------------------------ launch
struct DevCache {
  int sms = 0;
  bool attrs = false;
};
DevCache g_dev[64];

cudaError_t launch_ex(const void* fn, dim3 grid, int threads, size_t smem, void** args,
                      cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

bool decode2_supported(const flint_moe_shape& s) {
  return s.M <= kDecodeMaxTokens && s.M * s.top_k <= 1024 && s.I <= kGuKst4 &&
         s.SI <= kGuKst16 && (s.H <= kGuKst4 || s.H % 256 == 0) &&
         dn_layout(s.M, s.top_k).total <= (size_t)kMaxSmem &&
         gu_layout(s.M, s.H).stages >= 2 && 16 * (s.I / 2 + kPad) + s.I <= kDnStageBytes;
}

cudaError_t launch_decode2(const MoEArgs& a, cudaStream_t st) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  DevCache& dc = g_dev[dev];
  if (!dc.attrs) {
    err = cudaDeviceGetAttribute(&dc.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute((const void*)gate_up2_kernel<1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute((const void*)gate_up2_kernel<2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute((const void*)down2_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (err != cudaSuccess) return err;
    dc.attrs = true;
  }
  MoEArgs aa = a;
  void* args[] = {&aa};
  err = route_cluster_supported(a) ? launch_route_cluster(a, st) : launch_route(a, true, st, false);
  if (err != cudaSuccess) return err;
  const void* gu = a.M <= 8 ? (const void*)gate_up2_kernel<1> : (const void*)gate_up2_kernel<2>;
  err = launch_ex(gu, dim3(dc.sms), kGuThreads, gu_layout(a.M, a.H).total, args, st, true);
  if (err != cudaSuccess) return err;
  return launch_ex((const void*)down2_kernel, dim3(a.H / 16), kThreads, dn_layout(a.M, a.k).total,
                   args, st, true);
}

FLINT_SPAN_SETTER(decode2)

}  // namespace flint
