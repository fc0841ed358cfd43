// Grouped path for many tokens (M > 64): token permutation by expert,
// grouped NVFP4 GEMMs on the tensor cores (tcgen05, TMEM accumulators), the
// shared expert's BF16 GEMMs in the same launches, and the weighted combine.
//
// Page "vllm.models.flint.ops.moe": flint_moe for large M (per-expert
// grouped GEMMs over the permuted tokens, then _combine_kernel), with the
// module's Numerics rule: weights dequantised exactly (e2m1 x e4m3 block
// scale), fp32 accumulation, the per-expert global scale on the
// accumulator, act = bf16(silu(g) * u), y = bf16(acc * gs2),
// out = bf16(bf16(sum_j tw_j y_j) + shared).
//
// Launches (chained with programmatic dependent launch):
//   router + grouping (route.cu)  ->  plan  ->  gather  ->  GEMM1  ->  GEMM2  ->  combine
// plan:    per expert, tiles of up to 256 of its sorted rows (token tiles).
// gather:  x_perm[pos] = x[token of sorted pair pos] (so GEMM1 reads its A
//          operand as plain 2-D TMA tiles).
// GEMM1:   routed units (token tile, 128 intermediate rows): D = X W13^T over
//          256 weight rows (128 gate + the 128 matching up rows), epilogue
//          SwiGLU -> act; shared units (256 tokens, 32 rows): BF16 weights,
//          -> sact.
// GEMM2:   routed units (token tile, 256 output rows): D = act W2^T, epilogue
//          y = bf16(acc * gs2); shared units likewise: sact Wsd^T -> ys.
// combine: out[t] = bf16(bf16(sum_j tw_j y[row of (t, j)]) + ys[t]).
//
// GEMM kernel: persistent clusters of two CTAs on two SMs (one pair per two
// SMs), 640 threads per CTA.  Every unit is a pair unit: 256 token rows
// (CTA c owns rows 128 c ..) by n weight rows (CTA c dequantises n / 2 of
// them); one thread of the leader CTA issues tcgen05.mma.cta_group::2
// (M = 256), which reads A and B halves from both CTAs' shared memory and
// writes each CTA's 128 token rows into its own TMEM.
//   warp 13: TMA producer of the stages (A tiles; the shared expert's BF16
//           B tiles),
//   warp 17: TMA producer of the NVFP4 code tiles (a ring of their own),
//   warp 9:  leader: MMA issuer and TMEM owner (two 256-column accumulator
//           buffers, so one unit's epilogue overlaps the next unit's MMAs);
//           peer: relays "this CTA's half of stage s is in" to the leader's
//           barrier,
//   8 dequantising warps: two groups of 4 taking alternate K blocks; one
//           thread per B row: 128 codes of a K block -> bf16 e2m1 * scale *
//           2^-7, exact, the first half before the stage is free and the
//           second after, stored into the 128-byte swizzled K-major layout,
//   8 epilogue warps: TMEM -> registers (tcgen05.ld), scales, SwiGLU, BF16
//           stores (lane quarter warp % 4, two column groups).
// Rings: 3 stages of {A 2 x 16 KB, B 2 x 16 KB} (K blocks of 128); 3 code
// tiles of 8 KB; the dequantising threads' block scales (asynchronous 8-byte
// copies three K blocks ahead, across unit boundaries).
// Every wait is bounded (FLINT_ERR_TIMEOUT in the status word on expiry).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace flint {
namespace {

// Roles by warp.  A warp runs on scheduler warp % 4; the single MMA-issuing
// thread shares its scheduler only with light warps (the two producers and the
// two epilogue warps that must sit there for TMEM lane quarter 1), so its
// instructions are not queued behind dequantisation math.
//   scheduler 0: dequant 0, 3, 6; epilogue q0 (12, 16)
//   scheduler 1: epilogue q1 (1, 5); MMA 9; stage producer 13; code producer 17
//   scheduler 2: dequant 1, 4, 7; epilogue q2 (14, 18)
//   scheduler 3: dequant 2, 5; epilogue q3 (11, 15); warp 19 idle
constexpr int kGWarps = 20;
constexpr int kWarpMma = 9, kWarpProd = 13, kWarpCodes = 17;
constexpr int kGThreads = kGWarps * 32;
// dequantising warp index (0..7: group = index / 4) or -1
FLINT_DEV int dq_index(int warp) {
  switch (warp) {
    case 0: return 0;
    case 2: return 1;
    case 3: return 2;
    case 4: return 3;
    case 6: return 4;
    case 7: return 5;
    case 8: return 6;
    case 10: return 7;
    default: return -1;
  }
}
// epilogue column group (0, 1) of an epilogue warp, or -1; its TMEM lane
// quarter is warp % 4
FLINT_DEV int epi_group(int warp) {
  switch (warp) {
    case 1: case 11: case 12: case 14: return 0;
    case 5: case 15: case 16: case 18: return 1;
    default: return -1;
  }
}
constexpr int kKB = 128;                          // K per stage
constexpr int kStages = 3;
constexpr int kATile = 128 * 128;                  // one 128-row x 64-column bf16 tile
constexpr int kBRows = 128;                        // B rows per CTA: N = 256 per pair
constexpr int kOffA = 0;                           // A: tiles of K 0..63, 64..127
constexpr int kOffB = 2 * kATile;                  // B: likewise
constexpr int kStageBytes = 4 * kATile;            // 65536
static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
// NVFP4 code tiles (kBRows rows x 64 bytes per K block) have a ring of their
// own, so they land well before they are dequantised.
constexpr int kCStages = 3;
constexpr int kCodeBytes = kBRows * (kKB / 2);
constexpr int kOffCodes = kStages * kStageBytes;
// Block-scale ring of the 256 dequantising threads (thread = B row of its
// group): slot j of thread t at bytes 8 (j * 256 + t), filled by
// asynchronous 8-byte copies kScaleAhead of the thread's K blocks ahead of
// use (slot j % kScaleSlots, never the one read).
constexpr int kScaleSlots = 4;
constexpr int kScaleAhead = 3;
constexpr int kDqThreads = 256;
constexpr int kOffScale = kOffCodes + kCStages * kCodeBytes;
constexpr int kScaleBytes = kScaleSlots * kDqThreads * 8;
constexpr int kTokTile = 256;   // token rows of a pair unit: 128 per CTA
constexpr int kTmemBuf = 256;   // TMEM columns of one accumulator buffer (two buffers)
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;
constexpr uint32_t kSuspendNs = 50000;
constexpr int kStWords = 4;  // token-tile table entry: e, row0, row_end, unused

struct GCtl {
  uint64_t full[kStages];      // this CTA's stage is in: A (and BF16 B) bytes, and the
                               // dequantising group's 4 warps (count 1 + 4, + tx); the
                               // leader's also counts the peer's relay (+ 1)
  uint64_t empty[kStages];     // the pair's MMAs are done with the stage (commit, both CTAs)
  uint64_t cfull[kCStages];    // code tile landed (count 1 + tx)
  uint64_t cempty[kCStages];   // code tile read by its 4 dequantising warps
  uint64_t acc_full[2];        // all MMAs of a unit done (commit, both CTAs)
  uint64_t acc_empty[2];       // leader: the pair's 16 epilogue warps read the buffer
  uint32_t tmem;
  int abort;
};
constexpr size_t kGSmem = (size_t)kOffScale + kScaleBytes + sizeof(GCtl) + 1024;

// Bounded waits (FLINT_ERR_TIMEOUT in the status word on expiry).  CL: the
// barrier also receives the peer CTA's arrivals.
template <bool CL = false>
FLINT_DEV bool gwait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
  if (CL ? tc::mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity)) return true;
  unsigned long long t0 = 0;
  for (;;) {
    if (*abort) return false;
    if (CL ? tc::mbar_try_wait_cluster(bar, parity, kSuspendNs) : mbar_try_wait(bar, parity, kSuspendNs))
      return true;
    const unsigned long long now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > kWaitNs) {
      *abort = 1;
      atomicCAS(status, 0, FLINT_ERR_TIMEOUT);
      return false;
    }
  }
}
FLINT_DEV bool gwait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int* status, int lane) {
  int ok = 0;
  if (lane == 0) ok = gwait(bar, parity, abort, status);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

struct TMaps {
  CUtensorMap a_routed;  // x_perm [np, H] (GEMM1) / act [np, I] (GEMM2), box {64, 128}
  CUtensorMap a_shared;  // x [M, H] / sact [M, SI], box {64, 128}
  CUtensorMap b_shared;  // shared_gu [2 SI, H] box {64, 32} / shared_down [H, SI] box {64, 128}
  CUtensorMap codes;     // w13 [E 2I, H/2] bytes / w2 [E H, I/2], box {64, 128}
};

// One pair unit, the same in every role of both CTAs: 256 token rows (CTA c
// takes rows row0 + 128 c ..) by n weight rows (CTA c holds n / 2 of them).
struct Unit {
  int shared;   // 0 routed, 1 shared expert
  int e;        // routed expert
  int row0;     // first row of the token tile (sorted position / token)
  int row_end;  // one past its last valid row
  int nt;       // N tile
  int K;        // reduction length
  int parts;    // accumulators (K block kb -> kb % parts)
  int n;        // B rows of the pair (MMA N): n / 2 from each CTA
  int w;        // TMEM buffers taken (n * parts = w * kTmemBuf; two start at column 0)
};

template <int STAGE>
FLINT_DEV Unit unit_of(const MoEArgs& a, int u, int R, int NT, int NTs) {
  Unit x;
  if (u < R) {
    const int st = u / NT;
    const int* ent = a.ws.st_table + (size_t)st * kStWords;
    x.shared = 0;
    x.e = ldg_cg_i32(ent);
    x.row0 = ldg_cg_i32(ent + 1);
    x.row_end = ldg_cg_i32(ent + 2);
    x.nt = u % NT;
    x.K = STAGE == 1 ? a.H : a.I;
  } else {
    const int v = u - R;
    x.shared = 1;
    x.e = -1;
    x.row0 = (v / NTs) * kTokTile;
    x.row_end = min(a.M, x.row0 + kTokTile);
    x.nt = v % NTs;
    x.K = STAGE == 1 ? a.H : a.SI;
  }
  // Routed units: N = 256 (GEMM1: 128 gate + 128 up rows of tile nt; GEMM2:
  // output rows 256 nt ..), one accumulator, one TMEM buffer.  The shared
  // expert keeps more accumulators (both buffers): its gate/up eight at
  // N = 64 (its bf16(gS), bf16(uS) roundings feed every output of the token),
  // its down two (its rounded ys is added to every output).
  const bool sgu = x.shared && STAGE == 1;
  x.parts = sgu ? 8 : (x.shared ? 2 : 1);
  x.n = sgu ? 64 : 256;
  x.w = x.shared ? 2 : 1;
  return x;
}

// Dequantise half j of one K block of a B row (32 codes, their 2 scale
// bytes) to bf16 e2m1 * scale * 2^-7, exactly: v[i] holds K 32 j + 8 i .. + 7.
FLINT_DEV void dequant_half(uint4 (&v)[4], const uint4 c0, uint32_t sc2) {
  const uint32_t s01 = e4m3x2_to_bf16x2_x2p119(sc2 & 0xFFFFu);
  const uint32_t w[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // word i: K 32 j + 8 i .. + 7, scale block i / 2
    const uint32_t sc = bf16x2_bcast(s01, i >> 1);
    const uint32_t p0 = bf16x2_mul(e2m1_pair(w[i], 0), sc);  // K 8 i + 0, 8 i + 4
    const uint32_t p1 = bf16x2_mul(e2m1_pair(w[i], 1), sc);  // 1, 5
    const uint32_t p2 = bf16x2_mul(e2m1_pair(w[i], 2), sc);  // 2, 6
    const uint32_t p3 = bf16x2_mul(e2m1_pair(w[i], 3), sc);  // 3, 7
    v[i].x = __byte_perm(p0, p1, 0x5410);  // K 0, 1
    v[i].y = __byte_perm(p2, p3, 0x5410);  // 2, 3
    v[i].z = __byte_perm(p0, p1, 0x7632);  // 4, 5
    v[i].w = __byte_perm(p2, p3, 0x7632);  // 6, 7
  }
}

template <int STAGE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGThreads, 1)
    grouped_gemm_kernel(const MoEArgs a, const __grid_constant__ TMaps tm, int NT, int NTs,
                        int n_shared_tiles) {
  SpanGuard<(STAGE == 1 ? kSpanGemm1 : kSpanGemm2)> span_guard;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  GCtl& C = *reinterpret_cast<GCtl*>(smem + (size_t)kOffScale + kScaleBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  int* status = a.ws.status;
  volatile int* abort = &C.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&C.full[i], 1 + 4 + (leader ? 1 : 0));
      mbar_init(&C.empty[i], 1);
    }
    for (int i = 0; i < kCStages; ++i) {
      mbar_init(&C.cfull[i], 1);
      mbar_init(&C.cempty[i], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&C.acc_full[b], 1);
      mbar_init(&C.acc_empty[b], 16);
    }
    C.abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tc::tmem_alloc_pair(&C.tmem, 2 * kTmemBuf);
  tc::fence_before_sync();
  tc::cluster_sync();  // both CTAs: barriers initialised, TMEM allocated
  tc::fence_after_sync();
  const uint32_t tmem = C.tmem;

  pdl_wait();  // routing, plan and the previous GEMM are complete
  pdl_launch_dependents();
  const int ST = ldg_cg_i32(a.ws.st_count);
  const int R = ST * NT;
  const int total = R + n_shared_tiles * NTs;

  if (warp == kWarpProd) {
    // ------------------------------------------------------- stage producer
    int it = 0;
    for (int u = pair; u < total && !*abort; u += npairs) {
      const Unit x = unit_of<STAGE>(a, u, R, NT, NTs);
      const int nkb = x.K / kKB;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % kStages;
        int ok = 1;
        if (it >= kStages) ok = gwait_warp(&C.empty[s], ((it / kStages) - 1) & 1, abort, status, lane);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = smem + (size_t)s * kStageBytes;
          const CUtensorMap* ta = x.shared ? &tm.a_shared : &tm.a_routed;
          uint32_t bytes = 2 * kATile;
          if (x.shared) bytes += 2u * (uint32_t)(x.n / 2) * 128u;
          mbar_arrive_expect_tx(&C.full[s], bytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // the two 64-wide halves of the K block
            const int k0 = kb * kKB + 64 * h;
            tc::tma_load_2d(st + kOffA + h * kATile, ta, k0, x.row0 + 128 * (int)rank, &C.full[s]);
            if (x.shared) {
              if (STAGE == 1)  // leader 32 gate rows, peer the 32 matching up rows
                tc::tma_load_2d(st + kOffB + h * kATile, &tm.b_shared, k0, (leader ? 0 : a.SI) + 32 * x.nt, &C.full[s]);
              else  // rows past H (last tile) read as zeros
                tc::tma_load_2d(st + kOffB + h * kATile, &tm.b_shared, k0, 256 * x.nt + 128 * (int)rank, &C.full[s]);
            }
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == kWarpCodes) {
    // ----------------------------------------------------- code-tile producer
    // Runs up to kCStages K blocks ahead of dequantisation; K blocks of the
    // shared expert (no codes) only advance the ring.
    int it = 0;
    for (int u = pair; u < total && !*abort; u += npairs) {
      const Unit x = unit_of<STAGE>(a, u, R, NT, NTs);
      const int nkb = x.K / kKB;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int c = it % kCStages;
        int ok = 1;
        if (it >= kCStages) ok = gwait_warp(&C.cempty[c], ((it / kCStages) - 1) & 1, abort, status, lane);
        if (!ok) break;
        if (lane == 0) {
          if (x.shared) {
            mbar_arrive(&C.cfull[c]);
          } else {
            // GEMM1: leader the expert's 128 gate rows of tile nt, peer its up
            // rows; GEMM2: 128 output rows each (past H: the next expert's
            // rows, or zeros past the tensor; never stored)
            const int row = STAGE == 1 ? x.e * 2 * a.I + (leader ? 0 : a.I) + 128 * x.nt
                                       : x.e * a.H + 256 * x.nt + 128 * (int)rank;
            mbar_arrive_expect_tx(&C.cfull[c], (uint32_t)kCodeBytes);
            tc::tma_load_2d(smem + kOffCodes + c * kCodeBytes, &tm.codes, kb * (kKB / 2), row, &C.cfull[c]);
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0 && leader) {
      // ------------------------------------------------- MMA issuer (leader)
      // descriptors of stage 0's tiles; a stage's are these plus its byte
      // offset / 16 (shared addresses stay below 2^18, inside the 14-bit field)
      const uint64_t dA = tc::desc_sw128(smem + kOffA), dB = tc::desc_sw128(smem + kOffB);
      // buffer uses are counted over both buffers: use sl goes to buffer
      // sl % 2 and is that buffer's (sl / 2)-th
      int s = 0, slot = 0;
      uint32_t ph = 0;
      uint64_t so = 0;
      for (int u = pair; u < total && !*abort; u += npairs) {
        const Unit x = unit_of<STAGE>(a, u, R, NT, NTs);
        const int nkb = x.K / kKB;
        const uint32_t idesc = tc::idesc_bf16(256, x.n);
        const uint32_t dwrap = (uint32_t)(x.n * x.parts);
        bool ok = true;
        // the buffers' previous units have been read out by both CTAs
        for (int i = 0; i < x.w && ok; ++i) {
          const int sl = slot + i;
          if (sl >= 2) ok = gwait<true>(&C.acc_empty[sl & 1], ((sl >> 1) - 1) & 1, abort, status);
        }
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t dbuf = tmem + (x.w == 2 ? 0u : (uint32_t)(kTmemBuf * (slot & 1)));
        uint32_t dcol = 0;  // accumulator of K block kb: columns n * (kb % parts)
        for (int kb = 0; kb < nkb; ++kb) {
          if (!gwait<true>(&C.full[s], ph, abort, status)) {  // both CTAs' parts
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t da = dA + so, db = dB + so;
          const uint32_t d = dbuf + dcol;
          const bool acc = kb >= x.parts;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // K 16 kk: tile kk / 4, 32-byte step kk % 4
            const uint64_t o = (uint64_t)((kk >> 2) * (kATile >> 4) + 2 * (kk & 3));
            tc::mma_bf16_pair(d, da + o, db + o, idesc, acc || kk > 0);
          }
          tc::commit_pair(&C.empty[s]);
          dcol += (uint32_t)x.n;
          if (dcol == dwrap) dcol = 0;
          so += (uint64_t)(kStageBytes >> 4);
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
            so = 0;
          }
        }
        if (!ok) break;
        for (int i = 0; i < x.w; ++i) tc::commit_pair(&C.acc_full[(slot + i) & 1]);
        slot += x.w;
      }
    } else if (lane == 0) {
      // --------------------------------------------------- relay (peer CTA)
      // tells the leader when this CTA's part of each stage is in
      int s = 0;
      uint32_t ph = 0;
      for (int u = pair; u < total && !*abort; u += npairs) {
        const Unit x = unit_of<STAGE>(a, u, R, NT, NTs);
        const int nkb = x.K / kKB;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!gwait(&C.full[s], ph, abort, status)) {
            ok = false;
            break;
          }
          // the stage's A (TMA) and B (dequantised, made visible to the async
          // proxy) are writes to this CTA's shared memory
          tc::mbar_arrive_remote_smem(tc::mapa(&C.full[s], 0));
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (dq_index(warp) >= 0) {
    // ------------------------------------------------------- dequantisation
    // Two groups of 4 warps take alternate K blocks (global K block index
    // it: group it % 2), so each warp has two K blocks' time for one.
    const int dq = dq_index(warp);
    const int grp = dq >> 2;
    const int dqt = dq * 32 + lane;      // 0..255
    const int r = dqt & 127;             // B row of this CTA
    // block scales of the row (8 bytes per K block), or null (shared expert,
    // rows past H)
    auto scale_row = [&](const Unit& x) -> const uint8_t* {
      if (x.shared) return nullptr;
      if (STAGE == 1)
        return a.w13_sf + ((size_t)x.e * 2 * a.I + (leader ? 0 : a.I) + 128 * x.nt + r) * (a.H / 16);
      if (256 * x.nt + 128 * (int)rank + r >= a.H) return nullptr;
      return a.w2_sf + ((size_t)x.e * a.H + 256 * x.nt + 128 * rank + r) * (a.I / 16);
    };
    // The scale copies run kScaleAhead of this group's K blocks ahead of their
    // use as one stream over the units (no wait at a unit's start); the
    // fetch cursor: unit fu (its first global K block fit), K block fkb.
    uint2* ring = reinterpret_cast<uint2*>(smem + kOffScale) + dqt;
    int fu = pair, fit = 0, fkb = grp, fnkb = 0, jf = 0;
    const uint8_t* frow = nullptr;
    if (fu < total) {
      const Unit fx = unit_of<STAGE>(a, fu, R, NT, NTs);
      fnkb = fx.K / kKB;
      frow = scale_row(fx);
    }
    auto fetch_next = [&]() {
      while (fu < total && fkb >= fnkb) {  // on to this group's first K block of the next unit
        fit += fnkb;
        fu += npairs;
        if (fu < total) {
          const Unit fx = unit_of<STAGE>(a, fu, R, NT, NTs);
          fnkb = fx.K / kKB;
          frow = scale_row(fx);
          fkb = (grp - fit) & 1;
        }
      }
      if (fu < total && frow) cp_async8(ring + (jf % kScaleSlots) * kDqThreads, frow + 8 * fkb);
      cp_async_commit();
      ++jf;
      fkb += 2;
    };
#pragma unroll 1
    for (int d = 0; d < kScaleAhead; ++d) fetch_next();
    int it = 0, jc = 0;
    for (int u = pair; u < total && !*abort; u += npairs) {
      const Unit x = unit_of<STAGE>(a, u, R, NT, NTs);
      const int nkb = x.K / kKB;
      const bool has_sf = scale_row(x) != nullptr;
      const int kb0 = (grp - it) & 1;  // this group's first K block of the unit
      const int nmine = (nkb - kb0 + 1) / 2;
      bool ok = true;
      for (int j = 0; j < nmine; ++j, ++jc) {
        const int itk = it + kb0 + 2 * j;
        const int s = itk % kStages, c = itk % kCStages;
        cp_async_wait_group<kScaleAhead - 1>();  // this K block's copy has landed
        const uint2 sc = has_sf ? ring[(jc % kScaleSlots) * kDqThreads] : make_uint2(0, 0);  // 8 block scales
        fetch_next();
        // codes of the K block (landed well ahead): into registers, slot released
        if (!gwait_warp(&C.cfull[c], (itk / kCStages) & 1, abort, status, lane)) {
          ok = false;
          break;
        }
        uint4 cq[4];  // codes of K 0..31, 32..63, 64..95, 96..127
        if (!x.shared) {
          const uint4* cr = reinterpret_cast<const uint4*>(smem + kOffCodes + c * kCodeBytes + r * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) cq[i] = cr[i];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.cempty[c]);
        uint4 bv0[4], bv1[4];  // K 0..31, 32..63 (dequantised before the stage is free)
        if (!x.shared) {
          dequant_half(bv0, cq[0], sc.x & 0xFFFFu);
          dequant_half(bv1, cq[1], sc.x >> 16);
        }
        // the stage's previous MMAs are done: its B area is free
        if (itk >= kStages && !gwait_warp(&C.empty[s], ((itk / kStages) - 1) & 1, abort, status, lane)) {
          ok = false;
          break;
        }
        if (!x.shared) {
          uint8_t* bt = smem + (size_t)s * kStageBytes + kOffB;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            *reinterpret_cast<uint4*>(bt + tc::sw128_offset(r, 8 * i)) = bv0[i];
            *reinterpret_cast<uint4*>(bt + tc::sw128_offset(r, 32 + 8 * i)) = bv1[i];
          }
          dequant_half(bv0, cq[2], sc.y & 0xFFFFu);  // second tile: K 64..127
          dequant_half(bv1, cq[3], sc.y >> 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            *reinterpret_cast<uint4*>(bt + kATile + tc::sw128_offset(r, 8 * i)) = bv0[i];
            *reinterpret_cast<uint4*>(bt + kATile + tc::sw128_offset(r, 32 + 8 * i)) = bv1[i];
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.full[s]);
      }
      if (!ok) break;
      it += nkb;
    }
    cp_async_wait_all();  // no copy may land after the block has exited
  } else if (epi_group(warp) >= 0) {
    // ------------------------------------------------------------ epilogue
    // TMEM lane quarter warp % 4 (lane = token row of this CTA), column half
    // epi_group(warp) of the unit's outputs, 16 columns at a time; the
    // accumulator buffers alternate, so this overlaps the next unit's MMAs.
    const int q = warp & 3, cg = epi_group(warp);
    int slot = 0;
    for (int u = pair; u < total && !*abort; u += npairs) {
      const Unit x = unit_of<STAGE>(a, u, R, NT, NTs);
      bool ok = true;
      for (int i = 0; i < x.w && ok; ++i) {
        const int sl = slot + i;
        ok = gwait_warp(&C.acc_full[sl & 1], (sl >> 1) & 1, abort, status, lane);
      }
      if (!ok) break;
      tc::fence_after_sync();
      const int row = x.row0 + 128 * (int)rank + 32 * q + lane;
      const bool valid = row < x.row_end;
      const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (x.w == 2 ? 0u : (uint32_t)(kTmemBuf * (slot & 1)));
      const int nparts = min(x.parts, x.K / kKB);
      if (STAGE == 1) {
        const int I = x.shared ? a.SI : a.I;
        const int hw = x.n / 2;  // intermediate columns of the unit: gate [0, hw), up [hw, n)
        uint16_t* dst = (x.shared ? a.ws.sact : a.ws.act) + (size_t)row * I + hw * x.nt;
        const float gs = x.shared ? 1.0f : a.w13_gs[x.e] * 128.0f;
        const int cw = hw / 2 < 16 ? 16 : hw / 2;  // columns of this column group
        for (int c0 = cg * cw; c0 < min(hw, (cg + 1) * cw); c0 += 16) {
          uint32_t gv[16], uv[16], t2[16], t3[16];
          tc::tmem_ld16_async(tb + c0, gv);       // gate, partial 0
          tc::tmem_ld16_async(tb + hw + c0, uv);  // up, partial 0
          tc::tmem_wait_ld();
          tc::tmem_regs_ready16(gv);
          tc::tmem_regs_ready16(uv);
          for (int p = 1; p < nparts; ++p) {  // each partial's gate and up together
            tc::tmem_ld16_async(tb + x.n * p + c0, t2);
            tc::tmem_ld16_async(tb + x.n * p + hw + c0, t3);
            tc::tmem_wait_ld();
            tc::tmem_regs_ready16(t2);
            tc::tmem_regs_ready16(t3);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              gv[i] = __float_as_uint(__uint_as_float(gv[i]) + __uint_as_float(t2[i]));
              uv[i] = __float_as_uint(__uint_as_float(uv[i]) + __uint_as_float(t3[i]));
            }
          }
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float v[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float gg = __uint_as_float(gv[i + j]), uu = __uint_as_float(uv[i + j]);
              if (x.shared) {
                // stock BF16 SwiGLU: gS, uS rounded, silu(gS) = gS / (1 + exp(-gS))
                const float gS = round_bf16(gg), uS = round_bf16(uu);
                v[j] = __fdiv_rn(gS, 1.0f + expf(-gS)) * uS;
              } else {
                v[j] = silu_approx(gg * gs) * (uu * gs);
              }
            }
            pk[i / 2] = f32_to_bf16_bits(v[0]) | (f32_to_bf16_bits(v[1]) << 16);
          }
          if (valid) {
            reinterpret_cast<uint4*>(dst + c0)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            reinterpret_cast<uint4*>(dst + c0)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else {
        uint16_t* dst = (x.shared ? a.ws.ys : a.ws.y) + (size_t)row * a.H + x.n * x.nt;
        const float gs = x.shared ? 1.0f : a.w2_gs[x.e] * 128.0f;
        const int ncols = min(x.n, a.H - x.n * x.nt);  // the last tile of H may be partial
        for (int c0 = cg * (x.n / 2); c0 < min(ncols, (cg + 1) * (x.n / 2)); c0 += 16) {
          uint32_t v[16], t2[16];
          tc::tmem_ld16_async(tb + c0, v);
          if (nparts > 1) tc::tmem_ld16_async(tb + x.n + c0, t2);
          tc::tmem_wait_ld();
          tc::tmem_regs_ready16(v);
          tc::tmem_regs_ready16(t2);
          for (int p = 1; p < nparts; ++p) {
            if (p > 1) {
              tc::tmem_ld16_async(tb + x.n * p + c0, t2);
              tc::tmem_wait_ld();
              tc::tmem_regs_ready16(t2);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(t2[i]));
          }
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 16; i += 2)
            pk[i / 2] = f32_to_bf16_bits(__uint_as_float(v[i]) * gs) |
                        (f32_to_bf16_bits(__uint_as_float(v[i + 1]) * gs) << 16);
          if (valid) {
            reinterpret_cast<uint4*>(dst + c0)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            reinterpret_cast<uint4*>(dst + c0)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        for (int i = 0; i < x.w; ++i) {
          const int b = (slot + i) & 1;
          if (leader) mbar_arrive(&C.acc_empty[b]);
          else tc::mbar_arrive_remote(tc::mapa(&C.acc_empty[b], 0));
        }
      }
      slot += x.w;
    }
  }

  tc::fence_before_sync();
  tc::cluster_sync();  // no CTA leaves while its peer may still reach its memory
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, 2 * kTmemBuf);
  }
}

// ------------------------------------------------------------- small kernels
// Token tiles: per expert, ceil(cnt / 256) entries {e, row0, row_end}.
__global__ void __launch_bounds__(256) plan_kernel(MoEArgs a) {
  SpanGuard<kSpanPlan> span_guard;
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_n[kMaxE], s_start[kMaxE + 1];
  const int E = a.E, tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) s_n[e] = (ldg_cg_i32(a.ws.e_cnt + e) + kTokTile - 1) / kTokTile;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) { s_start[e] = run; run += s_n[e]; }
    s_start[E] = run;
    a.ws.st_count[0] = run;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    const int off = ldg_cg_i32(a.ws.e_off + e), cnt = ldg_cg_i32(a.ws.e_cnt + e);
    for (int i = 0; i < s_n[e]; ++i) {
      int* ent = a.ws.st_table + (size_t)(s_start[e] + i) * kStWords;
      ent[0] = e;
      ent[1] = off + kTokTile * i;
      ent[2] = off + cnt;
      ent[3] = 0;
    }
  }
}

// x_perm[pos] = x[sorted_pairs[pos] / k], one warp per row.
__global__ void __launch_bounds__(256) gather_kernel(MoEArgs a) {
  SpanGuard<kSpanGather> span_guard;
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pos = blockIdx.x * 8 + warp;
  if (pos >= a.M * a.k) return;
  const int t = ldg_cg_i32(a.ws.sorted_pairs + pos) / a.k;
  const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H);
  uint4* dst = reinterpret_cast<uint4*>(a.ws.x_perm + (size_t)pos * a.H);
  for (int i = lane; i < a.H / 8; i += 32) dst[i] = ldg_cg_v4(src + i);
}

// out[t, h..h+7] = bf16(bf16(sum_j tw_j y[row(t, j), h]) + ys[t, h]), j in rank order.
__global__ void __launch_bounds__(256) combine_kernel(MoEArgs a) {
  SpanGuard<kSpanCombine> span_guard;
  pdl_wait();
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int hv = a.H / 8;
  if (idx >= (size_t)a.M * hv) return;
  const int t = (int)(idx / hv), h = (int)(idx % hv) * 8;
  float R[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int j = 0; j < a.k; ++j) {
    const int p = t * a.k + j;
    const float w = ldg_cg_f32(a.ws.tw + p);
    const int row = ldg_cg_i32(a.ws.rowof + p);
    const uint4 yv = ldg_cg_v4(a.ws.y + (size_t)row * a.H + h);
    const uint32_t ys_[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      R[2 * i] = R[2 * i] + w * bf16_bits_to_f32(ys_[i] & 0xFFFFu);
      R[2 * i + 1] = R[2 * i + 1] + w * bf16_bits_to_f32(ys_[i] >> 16);
    }
  }
  uint32_t o[4];
  uint4 sv = make_uint4(0, 0, 0, 0);
  if (a.SI > 0) sv = ldg_cg_v4(a.ws.ys + (size_t)t * a.H + h);
  const uint32_t s_[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = round_bf16(R[2 * i]) + bf16_bits_to_f32(s_[i] & 0xFFFFu);
    const float hi = round_bf16(R[2 * i + 1]) + bf16_bits_to_f32(s_[i] >> 16);
    o[i] = f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
  }
  *reinterpret_cast<uint4*>(a.out + (size_t)t * a.H + h) = make_uint4(o[0], o[1], o[2], o[3]);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// 2-D map over a row-major [rows, cols] matrix; bf16 tiles use the 128-byte
// swizzle, byte (code) tiles none.
bool make_map(CUtensorMap* m, const void* base, bool bf16, uint64_t rows, uint64_t cols,
              uint32_t box_cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (bf16 ? 2 : 1)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, void** args,
                       cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

struct GDev {
  int sms = 0;
  int pairs = 0;  // CTA pairs of the GEMM grid (all co-resident)
  bool attrs = false;
};
GDev g_gdev[64];

}  // namespace

bool grouped_supported(const flint_moe_shape& s) {
  // 128-wide K blocks over H, I and SI; 128-row intermediate tiles of GEMM1
  // (32 for the shared expert); GEMM2's last 256-row output tile may be half
  return s.I % 128 == 0 && s.H % 128 == 0 && s.SI % 128 == 0;
}

size_t grouped_st_entries(const flint_moe_shape& s) {
  return (size_t)s.M * s.top_k / kTokTile + s.E + 1;
}

cudaError_t launch_grouped(const MoEArgs& a, cudaStream_t st) {
  if (!get_encoder()) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  GDev& gd = g_gdev[dev];
  if (!gd.attrs) {
    err = cudaDeviceGetAttribute(&gd.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute((const void*)grouped_gemm_kernel<1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute((const void*)grouped_gemm_kernel<2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (err != cudaSuccess) return err;
    // persistent pairs: as many clusters of two as can be resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gd.sms & ~1);
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = kGSmem;
    int nclusters = 0;
    err = cudaOccupancyMaxActiveClusters(&nclusters, (const void*)grouped_gemm_kernel<1>, &cfg);
    if (err != cudaSuccess) return err;
    if (nclusters < 1) return cudaErrorNotSupported;
    gd.pairs = nclusters < gd.sms / 2 ? nclusters : gd.sms / 2;
    gd.attrs = true;
  }
  const uint64_t np = (uint64_t)a.M * a.k;
  const int H = a.H, I = a.I, SI = a.SI, E = a.E;
  TMaps t1{}, t2{};
  bool ok = make_map(&t1.a_routed, a.ws.x_perm, true, np, H, 64, 128) &&
            make_map(&t1.a_shared, a.x, true, a.M, H, 64, 128) &&
            make_map(&t1.codes, a.w13, false, (uint64_t)E * 2 * I, H / 2, kKB / 2, 128) &&
            make_map(&t2.a_routed, a.ws.act, true, np, I, 64, 128) &&
            make_map(&t2.codes, a.w2, false, (uint64_t)E * H, I / 2, kKB / 2, 128);
  if (ok && SI > 0)
    ok = make_map(&t1.b_shared, a.shared_gu, true, 2 * (uint64_t)SI, H, 64, 32) &&
         make_map(&t2.a_shared, a.ws.sact, true, a.M, SI, 64, 128) &&
         make_map(&t2.b_shared, a.shared_down, true, H, SI, 64, 128);
  if (!ok) return cudaErrorInvalidValue;

  err = launch_route(a, true, st, false);
  if (err != cudaSuccess) return err;
  MoEArgs aa = a;
  void* args0[] = {&aa};
  err = launch_pdl((const void*)plan_kernel, dim3(1), dim3(256), 0, args0, st);
  if (err != cudaSuccess) return err;
  err = launch_pdl((const void*)gather_kernel, dim3((unsigned)((np + 7) / 8)), dim3(256), 0, args0, st);
  if (err != cudaSuccess) return err;
  // pair units: 256 token rows by 256 weight rows (GEMM1: 128 gate + 128 up
  // intermediate rows; the shared expert's gate/up 32 + 32), GEMM2 256
  // output rows (the last tile of H may be half)
  const int nsh = SI > 0 ? (a.M + kTokTile - 1) / kTokTile : 0;
  int NT1 = I / 128, NTs1 = SI > 0 ? SI / 32 : 1, NT2 = (H + 255) / 256, NTs2 = NT2;
  const dim3 grid(2 * gd.pairs);
  void* args1[] = {&aa, &t1, &NT1, &NTs1, (void*)&nsh};
  err = launch_pdl((const void*)grouped_gemm_kernel<1>, grid, dim3(kGThreads), kGSmem, args1, st);
  if (err != cudaSuccess) return err;
  void* args2[] = {&aa, &t2, &NT2, &NTs2, (void*)&nsh};
  err = launch_pdl((const void*)grouped_gemm_kernel<2>, grid, dim3(kGThreads), kGSmem, args2, st);
  if (err != cudaSuccess) return err;
  const size_t nthr = (size_t)a.M * (H / 8);
  return launch_pdl((const void*)combine_kernel, dim3((unsigned)((nthr + 255) / 256)), dim3(256), 0,
                    args0, st);
}

FLINT_SPAN_SETTER(grouped)

}  // namespace flint
