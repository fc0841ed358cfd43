// Decode megakernel: the whole MoE block for M <= kDecodeMaxTokens tokens in
// one persistent launch.
//
// Page "vllm.models.flint.ops.moe": the decode path is _router_kernel
// (router GEMV, top-k by the token's last program), _gate_up_gemv_kernel
// (per (token, expert) NVFP4 gate/up + SiLU * up) and _down_gemv_kernel
// (down GEMV over the top-k experts, weighted combine, shared-expert add),
// with the shared expert on an auxiliary stream.  Here the same steps are
// work tiles of one kernel, chained by device-side counters, so the weight
// stream never drains between steps.  Tile order (every tile depends only on
// tiles of lower index):
//
//   static (round robin over CTAs; weights staged before the PDL wait)
//     ROUTER  router row e: logits of every token, fixed fp32 order
//     SGU     shared expert gate/up: 8 intermediate rows (gate + up), a K part
//             -> fp32 partial sums
//     TOPK    top-k + sigmoid renormalisation + expert grouping -> routing flag
//   dynamic (atomic work counter, decoded once the routing flag is up)
//     RGU     routed expert u: 8 intermediate rows, all K -> act
//     SFIN    64 shared intermediate rows: sact = bf16(silu(gS) * uS)
//     SDN     shared expert down: 16 output rows, a K part -> fp32 partials
//     RDN     routed expert u: 16 output rows -> y
//     COMBINE 128 output rows: out = bf16(bf16(sum_j tw_j y_j) + ys)
//
// CTA: 16 consumer warps, 1 producer warp, 1 epilogue warp.  The producer
// copies each tile's weight rows (NVFP4 codes + E4M3 scales, or BF16 rows)
// into a 3-stage shared-memory ring with cp.async.bulk, stages x once, and
// for down tiles also stages the activation rows once their producers have
// finished.  Inside a tile, consumer warp w takes n-tile (w mod nn) and every
// (16 / nn)-th 128-wide K slice, multiplies on the tensor cores (mma.sync
// m16n8k16, bf16 operands, fp32 accumulate) and leaves its partial in shared
// memory; the epilogue warp sums the partials in fixed warp order, applies the
// tile's epilogue and frees the stage, so consumers never stall on it.
// Completion is signalled with release adds; every wait is bounded (status
// FLINT_ERR_TIMEOUT on expiry).
#include "common.cuh"
#include "internal.h"

namespace flint {

namespace {

constexpr int kCW = 16;                   // consumer warps
constexpr int kProducer = kCW;            // warp index of the producer
constexpr int kEpilogue = kCW + 1;        // warp index of the epilogue warp
constexpr int kThreads = (kCW + 2) * 32;
constexpr int kStages = 3;
constexpr int kStageBytes = 40 * 1024;
constexpr int kXsBytes = 64 * 1024;       // staged x (M * H * 2 <= this)
constexpr int kSliceK = 128;
constexpr int kSfinRows = 64;             // shared intermediate rows per SFIN tile
constexpr int kCombineBlocks = 8;         // 16-row output blocks per COMBINE tile
constexpr unsigned long long kWaitNs = 2000000000ull;

enum : int { T_END = 0, T_ROUTER, T_SGU, T_TOPK, T_RGU, T_SFIN, T_SDN, T_RDN, T_COMBINE };

// counters (int32, workspace control block)
enum : int { C_WORK = 0, C_ROUTER = 1, C_ROUTED = 2, C_SGU = 3, C_SFIN = 4, C_EXIT = 5, C_N = 8 };

constexpr int kMaxPairs = kDecodeMaxTokens * kMaxTopK;

struct Tile {
  int type;
  int u, e;      // unique-expert slot, expert id (routed tiles)
  int row0;      // first intermediate / output row
  int part;      // K part (shared tiles)
  int s0, ns;    // first K slice and slice count
  int cnt, off;  // routed tiles: tokens of the expert, their first sorted row
  int boff;      // byte offset of activation rows staged after the weights, or -1
};

struct Smem {
  alignas(128) uint8_t stage[kStages][kStageBytes];
  alignas(128) uint8_t xs[kXsBytes];
  alignas(16) float red[kStages][kCW][32][4];
  Tile info[kStages];
  uint64_t full[kStages];   // producer -> consumers (weights landed)
  uint64_t done[kStages];   // consumers -> epilogue warp (partials written)
  uint64_t empty[kStages];  // epilogue warp -> producer (stage free)
  uint64_t xbar;
  uint64_t metabar;
  int cnt[kMaxE];
  int base[kMaxE];
  int off_s[kMaxE];
  alignas(16) int uniq_s[kMaxE + 4];
  alignas(16) int ecnt_s[kMaxE + 4];
  alignas(16) int eoff_s[kMaxE + 4];
  alignas(16) int pairs_s[kMaxPairs];
};

static_assert(sizeof(Smem) <= 227 * 1024, "decode megakernel shared memory exceeds one CTA's limit");

struct Geo {
  int nsl_H, nsl_I, nsl_SI;  // K slices of 128
  int P_sg, spp_sg;          // shared gate/up: K parts, slices per part
  int P_sd, spp_sd;          // shared down: K parts, slices per part
  int NSG, N1;               // shared gate/up tiles, static tiles
  int NSF, NCB;              // SFIN and COMBINE tiles
  int xs;                    // x staged in shared memory
};

}  // namespace

struct MkArgs {
  MoEArgs a;
  Geo G;
  int* ctr;        // [C_N]
  int* gu_done;    // [E]   RGU tiles done per routed-expert slot (x 32)
  int* down_cnt;   // [H/16] SDN parts + RDN tiles done per output block (x 32)
  float* part_sg;  // [SI/8][P_sg][16][64]
  float* part_sd;  // [H/16][P_sd][16][64]
};

namespace {

// Bounded wait (one lane) until *p >= target.
__device__ __noinline__ bool wait_ge(const int* p, int target, int* status) {
  if (ld_acquire(p) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned ns = 32;
  for (int i = 0;; ++i) {
    __nanosleep(ns);
    if (ns < 512) ns <<= 1;
    if (ld_acquire(p) >= target) return true;
    if ((i & 15) == 15) {
      if (ld_acquire(status) != 0) return false;
      if (globaltimer_ns() - t0 > kWaitNs) {
        atomicCAS(status, 0, FLINT_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Warp-uniform bounded wait (lane 0 polls).
__device__ __noinline__ bool warp_wait_ge(const int* p, int target, int* status, int lane) {
  int ok = 1;
  if (lane == 0) ok = wait_ge(p, target, status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    // suspended until the phase completes (or 0.1 ms passes): no spinning
    if (mbar_try_wait(bar, parity, 100000u)) return true;
    if (globaltimer_ns() - t0 > kWaitNs) {
      atomicCAS(status, 0, FLINT_ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform mbarrier wait: lane 0 polls, the warp follows.
__device__ __noinline__ bool warp_mbar_wait(uint64_t* bar, uint32_t parity, int* status, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity, status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// ------------------------------------------------------------ tile list
__device__ __noinline__ Tile static_tile(const MoEArgs& a, const Geo& G, int idx) {
  Tile t{};
  t.boff = -1;
  if (idx < a.E) {
    t.type = T_ROUTER;
    t.e = idx;
  } else if (idx < a.E + G.NSG) {
    const int d = idx - a.E;
    t.type = T_SGU;
    t.row0 = (d / G.P_sg) * 8;
    t.part = d % G.P_sg;
    t.s0 = t.part * G.spp_sg;
    t.ns = min(G.spp_sg, G.nsl_H - t.s0);
  } else {
    t.type = T_TOPK;
  }
  return t;
}

__device__ __noinline__ Tile dynamic_tile(const MoEArgs& a, const Geo& G, int d, int U) {
  Tile t{};
  const int nrg = U * (a.I / 8);
  const int nsf = G.NSF;
  const int nsd = a.SI > 0 ? (a.H / 16) * G.P_sd : 0;
  const int nrd = U * (a.H / 16);
  const int ncb = G.NCB;
  if (d < nrg) {
    t.type = T_RGU;
    t.u = d / (a.I / 8);
    t.row0 = (d % (a.I / 8)) * 8;
    t.ns = G.nsl_H;
    return t;
  }
  d -= nrg;
  if (d < nsf) {
    t.type = T_SFIN;
    t.row0 = d * kSfinRows;
    return t;
  }
  d -= nsf;
  if (d < nsd) {
    t.type = T_SDN;
    t.row0 = (d / G.P_sd) * 16;
    t.part = d % G.P_sd;
    t.s0 = t.part * G.spp_sd;
    t.ns = min(G.spp_sd, G.nsl_SI - t.s0);
    return t;
  }
  d -= nsd;
  if (d < nrd) {
    t.type = T_RDN;
    t.u = d / (a.H / 16);
    t.row0 = (d % (a.H / 16)) * 16;
    t.ns = G.nsl_I;
    return t;
  }
  d -= nrd;
  if (d < ncb) {
    t.type = T_COMBINE;
    t.row0 = d * kCombineBlocks * 16;
    return t;
  }
  t.type = T_END;
  return t;
}

// Bulk copies of a tile's weights into a stage; completion on `bar`.
__device__ __noinline__ void issue_tile(const MoEArgs& a, const Geo& G, const Tile& t, uint8_t* buf,
                          uint64_t* bar) {
  const int H = a.H, I = a.I, SI = a.SI;
  switch (t.type) {
    case T_ROUTER:
      mbar_arrive_expect_tx(bar, H * 2);
      bulk_g2s(buf, a.router_w + (size_t)t.e * H, H * 2, bar);
      break;
    case T_SGU: {
      const int pk = t.ns * kSliceK;
      mbar_arrive_expect_tx(bar, 16 * pk * 2);
      if (G.P_sg == 1) {
        bulk_g2s(buf, a.shared_gu + (size_t)t.row0 * H, 8 * H * 2, bar);
        bulk_g2s(buf + 8 * H * 2, a.shared_gu + (size_t)(SI + t.row0) * H, 8 * H * 2, bar);
      } else {
#pragma unroll 1
        for (int i = 0; i < 16; ++i) {
          const size_t row = i < 8 ? (size_t)(t.row0 + i) : (size_t)(SI + t.row0 + i - 8);
          bulk_g2s(buf + i * pk * 2, a.shared_gu + row * H + t.s0 * kSliceK, pk * 2, bar);
        }
      }
      break;
    }
    case T_RGU: {
      const size_t rg = (size_t)t.e * 2 * I + t.row0, ru = rg + I;
      mbar_arrive_expect_tx(bar, 16 * (H / 2) + 16 * (H / 16));
      bulk_g2s(buf, a.w13 + rg * (H / 2), 8 * (H / 2), bar);
      bulk_g2s(buf + 8 * (H / 2), a.w13 + ru * (H / 2), 8 * (H / 2), bar);
      bulk_g2s(buf + 16 * (H / 2), a.w13_sf + rg * (H / 16), 8 * (H / 16), bar);
      bulk_g2s(buf + 16 * (H / 2) + 8 * (H / 16), a.w13_sf + ru * (H / 16), 8 * (H / 16), bar);
      break;
    }
    case T_SDN: {
      const int pk = t.ns * kSliceK;
      const uint32_t bbytes = t.boff >= 0 ? (uint32_t)(a.M * SI * 2) : 0u;
      mbar_arrive_expect_tx(bar, 16 * pk * 2 + bbytes);
      if (bbytes) bulk_g2s(buf + t.boff, a.ws.sact, bbytes, bar);
      if (G.P_sd == 1) {
        bulk_g2s(buf, a.shared_down + (size_t)t.row0 * SI, 16 * SI * 2, bar);
      } else {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
          bulk_g2s(buf + i * pk * 2, a.shared_down + (size_t)(t.row0 + i) * SI + t.s0 * kSliceK,
                   pk * 2, bar);
      }
      break;
    }
    case T_RDN: {
      const size_t r = (size_t)t.e * H + t.row0;
      const uint32_t bbytes = t.boff >= 0 ? (uint32_t)(t.cnt * I * 2) : 0u;
      mbar_arrive_expect_tx(bar, 16 * (I / 2) + 16 * (I / 16) + bbytes);
      if (bbytes) bulk_g2s(buf + t.boff, a.ws.act + (size_t)t.off * I, bbytes, bar);
      bulk_g2s(buf, a.w2 + r * (I / 2), 16 * (I / 2), bar);
      bulk_g2s(buf + 16 * (I / 2), a.w2_sf + r * (I / 16), 16 * (I / 16), bar);
      break;
    }
    default:
      mbar_arrive(bar);  // tiles without weights
  }
}



// ------------------------------------------------------------ A operand
// NVFP4 rows g and g + 8 of a tile, one 128-wide K slice: the codes of the
// two rows (16 bytes each) and their two E4M3 block scales.
struct Fp4Slice {
  uint4 c0, c1;
  uint32_t sc0, sc1;  // bf16x2 of scale * 2^119 (lo = first 16 codes)
};

FLINT_DEV Fp4Slice fp4_slice(const uint8_t* cg, const uint8_t* cg8, const uint8_t* sg,
                             const uint8_t* sg8, int s, int t) {
  Fp4Slice d;
  d.c0 = *reinterpret_cast<const uint4*>(cg + s * (kSliceK / 2) + 16 * t);
  d.c1 = *reinterpret_cast<const uint4*>(cg8 + s * (kSliceK / 2) + 16 * t);
  d.sc0 = e4m3x2_to_bf16x2_x2p119(*reinterpret_cast<const uint16_t*>(sg + s * (kSliceK / 16) + 2 * t));
  d.sc1 = e4m3x2_to_bf16x2_x2p119(*reinterpret_cast<const uint16_t*>(sg8 + s * (kSliceK / 16) + 2 * t));
  return d;
}

FLINT_DEV uint32_t word_of(const uint4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// Two m16n8k16 products for word q of the slice (K offsets 8q .. 8q+7 of
// this thread's 32): A from NVFP4 codes (exactly dequantised, x 2^-7) or BF16
// rows, B from the activation vector xq (8 consecutive 16-bit values).
FLINT_DEV void mma_word_fp4(float (&acc)[4], const Fp4Slice& d, int q, uint4 xq) {
  const uint32_t wg = word_of(d.c0, q), wg8 = word_of(d.c1, q);
  const uint32_t sg = bf16x2_bcast(d.sc0, q >= 2), sg8 = bf16x2_bcast(d.sc1, q >= 2);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t a0 = bf16x2_mul(e2m1_pair(wg, 2 * r), sg);
    const uint32_t a1 = bf16x2_mul(e2m1_pair(wg8, 2 * r), sg8);
    const uint32_t a2 = bf16x2_mul(e2m1_pair(wg, 2 * r + 1), sg);
    const uint32_t a3 = bf16x2_mul(e2m1_pair(wg8, 2 * r + 1), sg8);
    const uint32_t xlo = r ? xq.y : xq.x, xhi = r ? xq.w : xq.z;
    mma_bf16_16816(acc, a0, a1, a2, a3, __byte_perm(xlo, xhi, 0x5410), __byte_perm(xlo, xhi, 0x7632));
  }
}

FLINT_DEV void mma_word_bf16(float (&acc)[4], uint4 a, uint4 b, uint4 xq) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t alo = r ? a.y : a.x, ahi = r ? a.w : a.z;
    const uint32_t blo = r ? b.y : b.x, bhi = r ? b.w : b.z;
    const uint32_t xlo = r ? xq.y : xq.x, xhi = r ? xq.w : xq.z;
    mma_bf16_16816(acc, __byte_perm(alo, ahi, 0x5410), __byte_perm(blo, bhi, 0x5410),
                   __byte_perm(alo, ahi, 0x7632), __byte_perm(blo, bhi, 0x7632),
                   __byte_perm(xlo, xhi, 0x5410), __byte_perm(xlo, xhi, 0x7632));
  }
}

// 8 activations (16-bit) of one row at K offset koff + 32 t + 8 q.
FLINT_DEV uint4 load_bq(const uint16_t* row, bool smem, int koff, int t, int q) {
  if (!row) return make_uint4(0, 0, 0, 0);
  const uint16_t* p = row + koff + 32 * t + 8 * q;
  return smem ? *reinterpret_cast<const uint4*>(p) : ldg_cg_v4(p);
}

// ----------------------------------------------------------- routing
FLINT_DEV void topk_token(const MoEArgs& a, int t, int lane, int* ids_s) {
  const int E = a.E, k = a.k;
  int key[kMaxE / 32];
#pragma unroll
  for (int q = 0; q < kMaxE / 32; ++q) {
    const int ee = q * 32 + lane;
    key[q] = -1;
    if (ee < E) {
      const uint32_t b = ldg_cg_u16(a.ws.logits + (size_t)t * E + ee);
      key[q] = (int)((ordered_bf16(b) << 8) | (uint32_t)(E - 1 - ee));
    }
  }
  float sum = 0.0f, my_s = 0.0f;
  int my_e = 0;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    int lm = key[0];
#pragma unroll
    for (int q = 1; q < kMaxE / 32; ++q) lm = max(lm, key[q]);
    const int best = __reduce_max_sync(0xffffffffu, lm);
#pragma unroll
    for (int q = 0; q < kMaxE / 32; ++q)
      if (key[q] == best) key[q] = -1;
    const uint32_t o = (uint32_t)best >> 8;
    const uint32_t b16 = (o & 0x8000u) ? (o ^ 0x8000u) : (o ^ 0xFFFFu);
    const float s = __fdiv_rn(1.0f, 1.0f + expf(-bf16_bits_to_f32(b16)));
    sum = sum + s;  // rank order
    if (lane == j) { my_s = s; my_e = E - 1 - (best & 0xFF); }
  }
  if (lane < k) {
    const float w = round_bf16(__fdiv_rn(my_s, sum + 1e-20f));
    a.ws.ids[t * k + lane] = my_e;
    ids_s[t * k + lane] = my_e;
    a.ws.tw[t * k + lane] = w;
    if (a.ids_out) a.ids_out[t * k + lane] = my_e;
    if (a.tw_out) a.tw_out[t * k + lane] = w;
  }
}

// Expert grouping of the M*k pairs (one warp).  Every token lists an expert at
// most once, so the rank of pair (t, j) among the pairs of its expert is the
// number of earlier tokens that chose the same expert: a popcount over a
// per-expert token bitmask.  Outputs: counts, exclusive offsets, the routed
// experts in ascending order, the pairs stable-sorted by expert and the
// inverse map.
FLINT_DEV void group_pairs(const MoEArgs& a, Smem& S, const int* ids_s, int lane) {
  const int E = a.E, k = a.k, np = a.M * a.k;
  uint32_t* mlo = reinterpret_cast<uint32_t*>(S.cnt);   // tokens 0..31
  uint32_t* mhi = reinterpret_cast<uint32_t*>(S.base);  // tokens 32..63
#pragma unroll 1
  for (int e = lane; e < E; e += 32) { mlo[e] = 0u; mhi[e] = 0u; }
  __syncwarp();
#pragma unroll 1
  for (int p = lane; p < np; p += 32) {
    const int t = p / k;
    atomicOr(t < 32 ? &mlo[ids_s[p]] : &mhi[ids_s[p]], 1u << (t & 31));
  }
  __syncwarp();
  int run = 0, urun = 0;
#pragma unroll 1
  for (int b = 0; b < E; b += 32) {
    const int e = b + lane;
    const int c = e < E ? __popc(mlo[e]) + __popc(mhi[e]) : 0, u = c > 0;
    int ic = c, iu = u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vc = __shfl_up_sync(0xffffffffu, ic, o), vu = __shfl_up_sync(0xffffffffu, iu, o);
      if (lane >= o) { ic += vc; iu += vu; }
    }
    if (e < E) {
      S.off_s[e] = run + ic - c;
      a.ws.e_cnt[e] = c;
      a.ws.e_off[e] = run + ic - c;
      if (u) a.ws.uniq[1 + urun + iu - u] = e;
    }
    run += __shfl_sync(0xffffffffu, ic, 31);
    urun += __shfl_sync(0xffffffffu, iu, 31);
  }
  if (lane == 0) { a.ws.e_off[E] = run; a.ws.uniq[0] = urun; }
  __syncwarp();
#pragma unroll 1
  for (int p = lane; p < np; p += 32) {
    const int e = ids_s[p], t = p / k;
    const int rank = t < 32 ? __popc(mlo[e] & ((1u << t) - 1u))
                            : __popc(mlo[e]) + __popc(mhi[e] & ((1u << (t - 32)) - 1u));
    const int pos = S.off_s[e] + rank;
    a.ws.sorted_pairs[pos] = p;
    a.ws.rowof[p] = pos;
  }
}

// ------------------------------------------------------------ producer
FLINT_DEV void run_producer(const MkArgs& A, Smem& S) {
  const MoEArgs& a = A.a;
  const Geo& G = A.G;
  int* status = a.ws.status;
  const int I = a.I, SI = a.SI, E = a.E, k = a.k, M = a.M, H = a.H;
  int n = 0;
  bool ok = true;
  auto slot = [&](int& st) {
    st = n % kStages;
    if (n >= kStages && !mbar_wait(&S.empty[st], ((n / kStages) - 1) & 1, status)) ok = false;
    return ok;
  };
  int idx = blockIdx.x;
  // weights of the first static tiles do not depend on earlier grids
  for (; idx < G.N1 && n < kStages; idx += gridDim.x, ++n) {
    const Tile tl = static_tile(a, G, idx);
    S.info[n] = tl;
    if (tl.type != T_TOPK) issue_tile(a, G, tl, S.stage[n], &S.full[n]);
  }
  pdl_wait();
  for (int i = 0; i < n; ++i)  // a TOPK tile reads the workspace: release it after the wait
    if (S.info[i].type == T_TOPK) mbar_arrive(&S.full[i]);
  if (G.xs) {
    mbar_arrive_expect_tx(&S.xbar, M * H * 2);
    bulk_g2s(S.xs, a.x, M * H * 2, &S.xbar);
  }
  for (; idx < G.N1; idx += gridDim.x) {
    int st;
    if (!slot(st)) break;
    const Tile tl = static_tile(a, G, idx);
    S.info[st] = tl;
    issue_tile(a, G, tl, S.stage[st], &S.full[st]);
    ++n;
  }
  int U = -1;
  for (;;) {
    int st;
    if (!slot(st)) {
      S.info[st].type = T_END;
      mbar_arrive(&S.full[st]);
      break;
    }
    const int d = atomicAdd(&A.ctr[C_WORK], 1);
    if (U < 0) {
      U = 0;
      if (wait_ge(&A.ctr[C_ROUTED], 1, status)) {
        // routing metadata into shared memory, once
        fence_proxy_async_global();
        const uint32_t b1 = ((E + 1) * 4 + 15) & ~15u, b2 = (E * 4 + 15) & ~15u;
        const uint32_t b3 = ((M * k) * 4 + 15) & ~15u;
        mbar_arrive_expect_tx(&S.metabar, 2 * b1 + b2 + b3);
        bulk_g2s(S.uniq_s, a.ws.uniq, b1, &S.metabar);
        bulk_g2s(S.ecnt_s, a.ws.e_cnt, b2, &S.metabar);
        bulk_g2s(S.eoff_s, a.ws.e_off, b1, &S.metabar);
        bulk_g2s(S.pairs_s, a.ws.sorted_pairs, b3, &S.metabar);
        if (mbar_wait(&S.metabar, 0, status)) U = S.uniq_s[0];
      }
    }
    Tile tl = dynamic_tile(a, G, d, U);
    tl.boff = -1;
    if (tl.type == T_RGU || tl.type == T_RDN) {
      tl.e = S.uniq_s[1 + tl.u];
      tl.cnt = S.ecnt_s[tl.e];
      tl.off = S.eoff_s[tl.e];
    }
    // stage the activation rows of down tiles next to their weights
    if (tl.type == T_RDN && 9 * I + tl.cnt * I * 2 <= kStageBytes) {
      if (wait_ge(&A.gu_done[tl.u], 32 * (I / 8), status)) {
        fence_proxy_async_global();
        tl.boff = 9 * I;
      }
    } else if (tl.type == T_SDN && 16 * tl.ns * kSliceK * 2 + M * SI * 2 <= kStageBytes) {
      if (wait_ge(&A.ctr[C_SFIN], 32 * kCW * G.NSF, status)) {
        fence_proxy_async_global();
        tl.boff = 16 * tl.ns * kSliceK * 2;
      }
    }
    S.info[st] = tl;
    issue_tile(a, G, tl, S.stage[st], &S.full[st]);
    ++n;
    if (tl.type == T_END) break;
  }
}

// ------------------------------------------------------ consumer bodies
FLINT_DEV void c_router(const MkArgs& A, Smem& S, const Tile& tl, const uint8_t* buf,
                                      int cw, int lane) {
  const MoEArgs& a = A.a;
  const int H = a.H, E = a.E, M = a.M;
  // logits[t, e]: lane l owns h = 256 c + 8 l, partial over (c, i) ascending
  // with fmaf, then the xor butterfly 16, 8, 4, 2, 1
  const uint16_t* w = reinterpret_cast<const uint16_t*>(buf);
  for (int tok = cw; tok < M; tok += kCW) {
    const uint16_t* xr = A.G.xs ? reinterpret_cast<const uint16_t*>(S.xs) + (size_t)tok * H
                                : a.x + (size_t)tok * H;
    float acc = 0.0f;
#pragma unroll 1
    for (int c = 0; 256 * c < H; ++c) {
      const int h = 256 * c + 8 * lane;
      if (h < H) {
        const uint4 xv = A.G.xs ? *reinterpret_cast<const uint4*>(xr + h) : ldg_cg_v4(xr + h);
        const uint4 wv = *reinterpret_cast<const uint4*>(w + h);
        const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc = fmaf(__uint_as_float(xs[q] << 16), __uint_as_float(ws[q] << 16), acc);
          acc = fmaf(__uint_as_float(xs[q] & 0xFFFF0000u), __uint_as_float(ws[q] & 0xFFFF0000u), acc);
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) a.ws.logits[(size_t)tok * E + tl.e] = (uint16_t)f32_to_bf16_bits(acc);
  }
  // one count per logit, released by the lane that wrote it
  if (lane == 0 && cw < M) red_release_add(&A.ctr[C_ROUTER], (M - 1 - cw) / kCW + 1);
}

FLINT_DEV void c_topk(const MkArgs& A, Smem& S, int st, int cw, int lane) {
  const MoEArgs& a = A.a;
  int* ids_s = reinterpret_cast<int*>(S.stage[st]);  // this tile carries no weights
  if (warp_wait_ge(&A.ctr[C_ROUTER], a.E * a.M, a.ws.status, lane))
    for (int tok = cw; tok < a.M; tok += kCW) topk_token(a, tok, lane, ids_s);
}

FLINT_DEV void c_sfin(const MkArgs& A, const Tile& tl, int cw, int lane) {
  const MoEArgs& a = A.a;
  const Geo& G = A.G;
  const int SI = a.SI, M = a.M;
  if (warp_wait_ge(&A.ctr[C_SGU], 32 * G.NSG, a.ws.status, lane)) {
    const int nr = min(kSfinRows, SI - tl.row0);
    for (int idx = cw * 32 + lane; idx < nr * M; idx += kCW * 32) {
      const int r = tl.row0 + idx / M, tok = idx % M;
      const float* part = A.part_sg + (size_t)(r / 8) * G.P_sg * 16 * 64;
      float gsum = 0.0f, usum = 0.0f;
      for (int pp = 0; pp < G.P_sg; ++pp) {
        gsum += ldg_cg_f32(part + ((size_t)pp * 16 + r % 8) * 64 + tok);
        usum += ldg_cg_f32(part + ((size_t)pp * 16 + 8 + r % 8) * 64 + tok);
      }
      // stock BF16 SwiGLU: gS, uS rounded, silu(gS) = gS / (1 + exp(-gS))
      const float gS = round_bf16(gsum), uS = round_bf16(usum);
      const float v = __fdiv_rn(gS, 1.0f + expf(-gS)) * uS;
      a.ws.sact[(size_t)tok * SI + r] = (uint16_t)f32_to_bf16_bits(v);
    }
  }
  red_release_add(&A.ctr[C_SFIN], 1);  // every lane, after its own stores
}

FLINT_DEV void c_combine(const MkArgs& A, Smem& S, const Tile& tl, int cw, int lane) {
  const MoEArgs& a = A.a;
  const Geo& G = A.G;
  const int H = a.H, SI = a.SI, M = a.M, k = a.k;
  const int U = S.uniq_s[0];
  const int expect = 32 * (U + (SI > 0 ? G.P_sd : 0));
  const int h_end = min(H, tl.row0 + kCombineBlocks * 16);
  bool ok2 = true;
  for (int hb = tl.row0 / 16; hb < h_end / 16 && ok2; ++hb)
    ok2 = warp_wait_ge(&A.down_cnt[hb], expect, a.ws.status, lane);
  if (!ok2) return;
  const int nh = h_end - tl.row0;
  for (int idx = cw * 32 + lane; idx < nh * M; idx += kCW * 32) {
    const int tok = idx / nh, h = tl.row0 + idx % nh;
    float R = 0.0f;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      const int p = tok * k + j;
      const float w = ldg_cg_f32(a.ws.tw + p);
      const int row = ldg_cg_i32(a.ws.rowof + p);
      R = R + w * bf16_bits_to_f32(ldg_cg_u16(a.ws.y + (size_t)row * H + h));  // rank order
    }
    float ys = 0.0f;
    if (SI > 0) {
      const float* part = A.part_sd + (size_t)(h / 16) * G.P_sd * 16 * 64;
      float sum = 0.0f;
      for (int pp = 0; pp < G.P_sd; ++pp) sum += ldg_cg_f32(part + ((size_t)pp * 16 + h % 16) * 64 + tok);
      ys = round_bf16(sum);
    }
    a.out[(size_t)tok * H + h] = (uint16_t)f32_to_bf16_bits(round_bf16(R) + ys);
  }
}

// NVFP4 K loop of one warp: slices s = s_first, s_first + step, ...
FLINT_DEV void k_loop_fp4(float (&acc)[4], const uint8_t* buf, int K2, int ns,
                                        int s_first, int step, int s0, const uint16_t* brow,
                                        bool bsm, int g, int t) {
  const uint8_t* cg = buf + g * K2;
  const uint8_t* cg8 = buf + (8 + g) * K2;
  const uint8_t* sg = buf + 16 * K2 + g * (K2 / 8);
  const uint8_t* sg8 = buf + 16 * K2 + (8 + g) * (K2 / 8);
#pragma unroll 1
  for (int s = s_first; s < ns; s += step) {
    const int koff = (s0 + s) * kSliceK;
    uint4 xq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) xq[q] = load_bq(brow, bsm, koff, t, q);
    const Fp4Slice d = fp4_slice(cg, cg8, sg, sg8, s, t);
#pragma unroll
    for (int q = 0; q < 4; ++q) mma_word_fp4(acc, d, q, xq[q]);
  }
}

// BF16 K loop of one warp (rows stored with pk elements each).
FLINT_DEV void k_loop_bf16(float (&acc)[4], const uint8_t* buf, int pk, int ns,
                                         int s_first, int step, int s0, const uint16_t* brow,
                                         bool bsm, int g, int t) {
  const uint16_t* rg = reinterpret_cast<const uint16_t*>(buf) + g * pk;
  const uint16_t* rg8 = reinterpret_cast<const uint16_t*>(buf) + (8 + g) * pk;
#pragma unroll 1
  for (int s = s_first; s < ns; s += step) {
    const int koff = (s0 + s) * kSliceK;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 xq = load_bq(brow, bsm, koff, t, q);
      const uint4 ra = *reinterpret_cast<const uint4*>(rg + s * kSliceK + 32 * t + 8 * q);
      const uint4 rb = *reinterpret_cast<const uint4*>(rg8 + s * kSliceK + 32 * t + 8 * q);
      mma_word_bf16(acc, ra, rb, xq);
    }
  }
}

FLINT_DEV void c_mma(const MkArgs& A, Smem& S, const Tile& tl, const uint8_t* buf,
                                   int st, int cw, int lane, bool& meta_ok) {
  const MoEArgs& a = A.a;
  const Geo& G = A.G;
  int* status = a.ws.status;
  const int H = a.H, I = a.I, SI = a.SI, k = a.k, M = a.M;
  const int g = lane >> 2, t = lane & 3;
  const bool fp4 = (tl.type == T_RGU || tl.type == T_RDN);
  int ntok = M, off = 0;
  if (fp4) {
    ntok = tl.cnt;
    off = tl.off;
    if (!meta_ok) meta_ok = warp_mbar_wait(&S.metabar, 0, status, lane);
  }
  const int nn = max(1, min((ntok + 7) / 8, 8));  // n-tiles (ntok <= 64)
  const int nk = kCW / nn;                        // K groups
  const int nw = cw % nn, kw = cw / nn;
  bool dep_ok = true;  // staged activations: the producer already waited
  if (tl.type == T_SDN && tl.boff < 0) dep_ok = warp_wait_ge(&A.ctr[C_SFIN], 32 * kCW * G.NSF, status, lane);
  if (tl.type == T_RDN && tl.boff < 0) dep_ok = warp_wait_ge(&A.gu_done[tl.u], 32 * (I / 8), status, lane);
  if (cw >= nn * nk) return;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (dep_ok) {
    const int n_ = nw * 8 + g;  // token column of this lane
    const uint16_t* brow = nullptr;
    bool bsm = false;
    if (n_ < ntok) {
      if (tl.type == T_RGU) {
        const int tok = S.pairs_s[off + n_] / k;
        bsm = G.xs;
        brow = bsm ? reinterpret_cast<const uint16_t*>(S.xs) + (size_t)tok * H : a.x + (size_t)tok * H;
      } else if (tl.type == T_SGU) {
        bsm = G.xs;
        brow = bsm ? reinterpret_cast<const uint16_t*>(S.xs) + (size_t)n_ * H : a.x + (size_t)n_ * H;
      } else if (tl.type == T_RDN) {
        bsm = tl.boff >= 0;
        brow = bsm ? reinterpret_cast<const uint16_t*>(buf + tl.boff) + (size_t)n_ * I
                   : a.ws.act + (size_t)(off + n_) * I;
      } else {
        bsm = tl.boff >= 0;
        brow = bsm ? reinterpret_cast<const uint16_t*>(buf + tl.boff) + (size_t)n_ * SI
                   : a.ws.sact + (size_t)n_ * SI;
      }
    }
    if (fp4)
      k_loop_fp4(acc, buf, (tl.type == T_RGU ? H : I) / 2, tl.ns, kw, nk, tl.s0, brow, bsm, g, t);
    else
      k_loop_bf16(acc, buf, tl.ns * kSliceK, tl.ns, kw, nk, tl.s0, brow, bsm, g, t);
  }
  *reinterpret_cast<float4*>(&S.red[st][cw][lane][0]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
}

// ------------------------------------------------------ epilogue bodies
FLINT_DEV void e_mma(const MkArgs& A, Smem& S, const Tile& tl, int st, int lane) {
  const MoEArgs& a = A.a;
  const Geo& G = A.G;
  const int H = a.H, I = a.I, M = a.M;
  const int g = lane >> 2, t = lane & 3;
  const bool fp4 = (tl.type == T_RGU || tl.type == T_RDN);
  const int ntok = fp4 ? tl.cnt : M, off = fp4 ? tl.off : 0;
  const int nn = max(1, min((ntok + 7) / 8, 8)), nk = kCW / nn;
#pragma unroll 1
  for (int nt = 0; nt < nn; ++nt) {
    // partials of the K groups in fixed order
    float4 r4 = *reinterpret_cast<const float4*>(&S.red[st][nt][lane][0]);
#pragma unroll 1
    for (int q = 1; q < nk; ++q) {
      const float4 o = *reinterpret_cast<const float4*>(&S.red[st][q * nn + nt][lane][0]);
      r4.x += o.x; r4.y += o.y; r4.z += o.z; r4.w += o.w;
    }
    const float v[4] = {r4.x, r4.y, r4.z, r4.w};
    if (tl.type == T_RGU) {
      const float gs = a.w13_gs[tl.e];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int nn_ = nt * 8 + 2 * t + c;
        if (nn_ < ntok) {
          const float gv = v[c] * 128.0f * gs, uv = v[2 + c] * 128.0f * gs;
          a.ws.act[(size_t)(off + nn_) * I + tl.row0 + g] = (uint16_t)f32_to_bf16_bits(silu_approx(gv) * uv);
        }
      }
    } else if (tl.type == T_RDN) {
      const float gs2 = a.w2_gs[tl.e];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int nn_ = nt * 8 + 2 * t + (i & 1);
        if (nn_ < ntok)
          a.ws.y[(size_t)(off + nn_) * H + tl.row0 + g + (i >> 1) * 8] =
              (uint16_t)f32_to_bf16_bits(v[i] * 128.0f * gs2);
      }
    } else {
      float* part = tl.type == T_SGU
                        ? A.part_sg + ((size_t)(tl.row0 / 8) * G.P_sg + tl.part) * 16 * 64
                        : A.part_sd + ((size_t)(tl.row0 / 16) * G.P_sd + tl.part) * 16 * 64;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int nn_ = nt * 8 + 2 * t + (i & 1);
        if (nn_ < ntok) part[(g + (i >> 1) * 8) * 64 + nn_] = v[i];
      }
    }
  }
  // every lane releases its own stores
  if (tl.type == T_RGU) red_release_add(&A.gu_done[tl.u], 1);
  else if (tl.type == T_SGU) red_release_add(&A.ctr[C_SGU], 1);
  else red_release_add(&A.down_cnt[tl.row0 / 16], 1);
}

FLINT_DEV void e_topk(const MkArgs& A, Smem& S, int st, int lane) {
  group_pairs(A.a, S, reinterpret_cast<const int*>(S.stage[st]), lane);
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    st_release(&A.ctr[C_ROUTED], 1);
  }
}

FLINT_DEV void run_epilogue(const MkArgs& A, Smem& S, int lane) {
  int* status = A.a.ws.status;
  for (int n = 0;; ++n) {
    const int st = n % kStages;
    if (!warp_mbar_wait(&S.full[st], (n / kStages) & 1, status, lane)) break;
    const Tile tl = S.info[st];
    if (tl.type == T_END) break;
    if (!warp_mbar_wait(&S.done[st], (n / kStages) & 1, status, lane)) break;
    if (tl.type == T_TOPK) e_topk(A, S, st, lane);
    else if (tl.type == T_SGU || tl.type == T_RGU || tl.type == T_SDN || tl.type == T_RDN)
      e_mma(A, S, tl, st, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[st]);
  }
  // exit: the last CTA returns every counter to zero
  int last = 0;
  if (lane == 0) {
    __threadfence();
    last = (atomicAdd(&A.ctr[C_EXIT], 1) == (int)gridDim.x - 1);
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  for (int i = lane; i < C_N; i += 32)
    if (i != C_EXIT) A.ctr[i] = 0;
  for (int i = lane; i < A.a.E; i += 32) A.gu_done[i] = 0;
  for (int i = lane; i < A.a.H / 16; i += 32) A.down_cnt[i] = 0;
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    A.ctr[C_EXIT] = 0;
  }
}

FLINT_DEV void run_consumer(const MkArgs& A, Smem& S, int cw, int lane) {
  int* status = A.a.ws.status;
  bool xs_ok = true;
  if (A.G.xs) xs_ok = warp_mbar_wait(&S.xbar, 0, status, lane);
  bool meta_ok = false;
  for (int n = 0; xs_ok; ++n) {
    const int st = n % kStages;
    if (!warp_mbar_wait(&S.full[st], (n / kStages) & 1, status, lane)) break;
    const Tile tl = S.info[st];
    if (tl.type == T_END) break;
    const uint8_t* buf = S.stage[st];
    if (tl.type == T_ROUTER) c_router(A, S, tl, buf, cw, lane);
    else if (tl.type == T_TOPK) c_topk(A, S, st, cw, lane);
    else if (tl.type == T_SFIN) c_sfin(A, tl, cw, lane);
    else if (tl.type == T_COMBINE) c_combine(A, S, tl, cw, lane);
    else c_mma(A, S, tl, buf, st, cw, lane, meta_ok);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.done[st]);
  }
}

}  // namespace

// ======================================================================
__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ MkArgs A) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.done[s], kCW);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.xbar, 1);
    mbar_init(&S.metabar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kProducer) {
    if (lane == 0) run_producer(A, S);
    return;
  }
  pdl_wait();
  pdl_launch_dependents();
  if (warp == kEpilogue) run_epilogue(A, S, lane);
  else run_consumer(A, S, warp, lane);
}

// ---------------------------------------------------------------- launch
static int g_num_sms = 0;

static Geo make_geo(int M, int H, int I, int SI, int E) {
  Geo G{};
  G.nsl_H = H / kSliceK;
  G.nsl_I = I / kSliceK;
  G.nsl_SI = SI / kSliceK;
  const int max_sl = kStageBytes / (16 * kSliceK * 2);  // slices of 16 BF16 rows per stage
  G.P_sg = (G.nsl_H + max_sl - 1) / max_sl;
  G.spp_sg = (G.nsl_H + G.P_sg - 1) / G.P_sg;
  G.P_sg = (G.nsl_H + G.spp_sg - 1) / G.spp_sg;
  if (SI > 0) {
    G.P_sd = (G.nsl_SI + max_sl - 1) / max_sl;
    G.spp_sd = (G.nsl_SI + G.P_sd - 1) / G.P_sd;
    G.P_sd = (G.nsl_SI + G.spp_sd - 1) / G.spp_sd;
  } else {
    G.P_sd = 1;
    G.spp_sd = 1;
  }
  G.NSG = (SI / 8) * G.P_sg;
  G.N1 = E + G.NSG + 1;
  G.NSF = (SI + kSfinRows - 1) / kSfinRows;
  G.NCB = (H / 16 + kCombineBlocks - 1) / kCombineBlocks;
  G.xs = (size_t)M * H * 2 <= (size_t)kXsBytes ? 1 : 0;
  return G;
}

bool decode_mk_supported(const flint_moe_shape& s) {
  return s.M <= kDecodeMaxTokens && 9 * s.H <= kStageBytes && 9 * s.I <= kStageBytes &&
         2 * s.H <= kStageBytes;
}

size_t decode_mk_ctr_bytes(const flint_moe_shape& s) {
  return (size_t)(C_N + s.E + s.H / 16) * 4;
}

size_t decode_mk_part_bytes(const flint_moe_shape& s) {
  const Geo G = make_geo(s.M, s.H, s.I, s.SI, s.E);
  return ((size_t)(s.SI / 8) * G.P_sg + (size_t)(s.H / 16) * G.P_sd) * 16 * 64 * 4;
}

cudaError_t launch_decode_mk(const MoEArgs& a, int* mk_ctr, float* mk_part, cudaStream_t st,
                             bool pdl) {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(moe_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(Smem));
  }
  MkArgs A{};
  A.a = a;
  A.G = make_geo(a.M, a.H, a.I, a.SI, a.E);
  A.ctr = mk_ctr;
  A.gu_done = A.ctr + C_N;
  A.down_cnt = A.gu_done + a.E;
  A.part_sg = mk_part;
  A.part_sd = A.part_sg + (size_t)(a.SI / 8) * A.G.P_sg * 16 * 64;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g_num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel, A);
}

}  // namespace flint
