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
// CTA: 8 consumer warps + 1 producer warp.  The producer copies each tile's
// weight rows (NVFP4 codes + E4M3 scales, or BF16 rows) into a 3-stage
// shared-memory ring with cp.async.bulk and stages x once; a tile's
// dependency wait happens after its weights have landed.  Consumer warps run
// independently: inside a tile, warp w takes n-tile (w mod nn) and every
// (8 / nn)-th 128-wide K slice, multiplies on the tensor cores (mma.sync
// m16n8k16, bf16 operands, fp32 accumulate) and leaves its partial in shared
// memory; the last warp to finish (shared counter) sums the partials in
// fixed warp order and applies the epilogue.  Completion is signalled with
// release adds; every wait is bounded (status FLINT_ERR_TIMEOUT on expiry).
#include "common.cuh"
#include "internal.h"

namespace flint {

namespace {

constexpr int kCW = 8;                    // consumer warps
constexpr int kThreads = (kCW + 1) * 32;  // + producer warp
constexpr int kStages = 3;
constexpr int kStageBytes = 32 * 1024;
constexpr int kXsBytes = 64 * 1024;       // staged x (M * H * 2 <= this)
constexpr int kSliceK = 128;
constexpr int kSfinRows = 64;             // shared intermediate rows per SFIN tile
constexpr int kCombineBlocks = 8;         // 16-row output blocks per COMBINE tile
constexpr unsigned long long kWaitNs = 2000000000ull;

enum : int { T_END = 0, T_ROUTER, T_SGU, T_TOPK, T_RGU, T_SFIN, T_SDN, T_RDN, T_COMBINE };

// counters (int32, workspace control block)
enum : int { C_WORK = 0, C_ROUTER = 1, C_ROUTED = 2, C_SGU = 3, C_SFIN = 4, C_EXIT = 5, C_N = 8 };

struct Tile {
  int type;
  int u, e;   // unique-expert slot, expert id (routed tiles)
  int row0;   // first intermediate / output row
  int part;   // K part (shared tiles)
  int s0, ns; // first K slice and slice count
};

struct Smem {
  uint8_t stage[kStages][kStageBytes];
  uint8_t xs[kXsBytes];
  float red[kStages][kCW][32][4];
  Tile info[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t xbar;
  int arr[kStages];
  int exit_arr;
  int cnt[kMaxE];
  int base[kMaxE];
};

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
  int* gu_done;    // [E]   RGU tiles done per routed-expert slot
  int* down_cnt;   // [H/16] SDN parts + RDN tiles done per output block
  float* part_sg;  // [SI/8][P_sg][16][64]
  float* part_sd;  // [H/16][P_sd][16][64]
};

namespace {

// Bounded wait (one lane) until *p >= target.
FLINT_DEV bool wait_ge(const int* p, int target, int* status) {
  const unsigned long long t0 = globaltimer_ns();
  for (int i = 0;; ++i) {
    if (ld_acquire(p) >= target) return true;
    if (i >= 16) {
      if (ld_acquire(status) != 0) return false;
      if (globaltimer_ns() - t0 > kWaitNs) {
        atomicCAS(status, 0, FLINT_ERR_TIMEOUT);
        return false;
      }
      __nanosleep(32);
    }
  }
}

// Warp-uniform bounded wait (lane 0 polls).
FLINT_DEV bool warp_wait_ge(const int* p, int target, int* status, int lane) {
  int ok = 1;
  if (lane == 0) ok = wait_ge(p, target, status);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

FLINT_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitNs) {
      atomicCAS(status, 0, FLINT_ERR_TIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------------------ tile list
FLINT_DEV Tile static_tile(const MoEArgs& a, const Geo& G, int idx) {
  Tile t{};
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

FLINT_DEV Tile dynamic_tile(const MoEArgs& a, const Geo& G, int d, int U) {
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
FLINT_DEV void issue_tile(const MoEArgs& a, const Geo& G, const Tile& t, uint8_t* buf,
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
      mbar_arrive_expect_tx(bar, 16 * pk * 2);
      if (G.P_sd == 1) {
        bulk_g2s(buf, a.shared_down + (size_t)t.row0 * SI, 16 * SI * 2, bar);
      } else {
        for (int i = 0; i < 16; ++i)
          bulk_g2s(buf + i * pk * 2, a.shared_down + (size_t)(t.row0 + i) * SI + t.s0 * kSliceK,
                   pk * 2, bar);
      }
      break;
    }
    case T_RDN: {
      const size_t r = (size_t)t.e * H + t.row0;
      mbar_arrive_expect_tx(bar, 16 * (I / 2) + 16 * (I / 16));
      bulk_g2s(buf, a.w2 + r * (I / 2), 16 * (I / 2), bar);
      bulk_g2s(buf + 16 * (I / 2), a.w2_sf + r * (I / 16), 16 * (I / 16), bar);
      break;
    }
    default:
      mbar_arrive(bar);  // tiles without weights
  }
}

// ------------------------------------------------------------ A operand
FLINT_DEV void a_frags_fp4(const uint8_t* cg, const uint8_t* cg8, const uint8_t* sg,
                           const uint8_t* sg8, int s, int t, uint32_t (&af)[4][2][4]) {
  const uint4 c0 = *reinterpret_cast<const uint4*>(cg + s * (kSliceK / 2) + 16 * t);
  const uint4 c1 = *reinterpret_cast<const uint4*>(cg8 + s * (kSliceK / 2) + 16 * t);
  const uint32_t s0 = *reinterpret_cast<const uint16_t*>(sg + s * (kSliceK / 16) + 2 * t);
  const uint32_t s1 = *reinterpret_cast<const uint16_t*>(sg8 + s * (kSliceK / 16) + 2 * t);
  const uint32_t sc0 = e4m3x2_to_bf16x2_x2p119(s0);
  const uint32_t sc1 = e4m3x2_to_bf16x2_x2p119(s1);
  const uint32_t wg[4] = {c0.x, c0.y, c0.z, c0.w};
  const uint32_t wg8[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t a = bf16x2_bcast(sc0, q >= 2);
    const uint32_t b = bf16x2_bcast(sc1, q >= 2);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      af[q][r][0] = bf16x2_mul(e2m1_pair(wg[q], 2 * r), a);
      af[q][r][1] = bf16x2_mul(e2m1_pair(wg8[q], 2 * r), b);
      af[q][r][2] = bf16x2_mul(e2m1_pair(wg[q], 2 * r + 1), a);
      af[q][r][3] = bf16x2_mul(e2m1_pair(wg8[q], 2 * r + 1), b);
    }
  }
}

FLINT_DEV void a_frags_bf16(const uint16_t* rg, const uint16_t* rg8, int s, int t,
                            uint32_t (&af)[4][2][4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 a = *reinterpret_cast<const uint4*>(rg + s * kSliceK + 32 * t + 8 * q);
    const uint4 b = *reinterpret_cast<const uint4*>(rg8 + s * kSliceK + 32 * t + 8 * q);
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

// 32 activations (16-bit) of one row at K offset koff + 32 t: smem or global.
FLINT_DEV void load_b(uint4 (&xb)[4], const uint16_t* row, bool smem, int koff, int t) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (!row) {
      xb[q] = make_uint4(0, 0, 0, 0);
    } else if (smem) {
      xb[q] = *reinterpret_cast<const uint4*>(row + koff + 32 * t + 8 * q);
    } else {
      xb[q] = ldg_cg_v4(row + koff + 32 * t + 8 * q);
    }
  }
}

FLINT_DEV void mma_slice(float (&acc)[4], const uint32_t (&af)[4][2][4], const uint4 (&xb)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    mma_bf16_16816(acc, af[q][0][0], af[q][0][1], af[q][0][2], af[q][0][3],
                   __byte_perm(xb[q].x, xb[q].z, 0x5410), __byte_perm(xb[q].x, xb[q].z, 0x7632));
    mma_bf16_16816(acc, af[q][1][0], af[q][1][1], af[q][1][2], af[q][1][3],
                   __byte_perm(xb[q].y, xb[q].w, 0x5410), __byte_perm(xb[q].y, xb[q].w, 0x7632));
  }
}

// ----------------------------------------------------------- routing
FLINT_DEV void topk_token(const MoEArgs& a, int t, int lane) {
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
    a.ws.tw[t * k + lane] = w;
    if (a.ids_out) a.ids_out[t * k + lane] = my_e;
    if (a.tw_out) a.tw_out[t * k + lane] = w;
  }
}

// Expert grouping of the M*k pairs (one warp): counts, offsets, routed
// experts, pairs stable-sorted by expert and the inverse map.
FLINT_DEV void group_pairs(const MoEArgs& a, Smem& S, int lane) {
  const int E = a.E, np = a.M * a.k;
  for (int e = lane; e < E; e += 32) S.cnt[e] = 0;
  __syncwarp();
  for (int p = lane; p < np; p += 32) atomicAdd(&S.cnt[ldg_cg_i32(a.ws.ids + p)], 1);
  __syncwarp();
  int run = 0, urun = 0;
  for (int b = 0; b < E; b += 32) {
    const int e = b + lane;
    const int c = e < E ? S.cnt[e] : 0, u = c > 0;
    int ic = c, iu = u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vc = __shfl_up_sync(0xffffffffu, ic, o), vu = __shfl_up_sync(0xffffffffu, iu, o);
      if (lane >= o) { ic += vc; iu += vu; }
    }
    if (e < E) {
      S.base[e] = run + ic - c;
      a.ws.e_cnt[e] = c;
      a.ws.e_off[e] = run + ic - c;
      if (u) a.ws.uniq[1 + urun + iu - u] = e;
    }
    run += __shfl_sync(0xffffffffu, ic, 31);
    urun += __shfl_sync(0xffffffffu, iu, 31);
  }
  if (lane == 0) { a.ws.e_off[E] = run; a.ws.uniq[0] = urun; }
  __syncwarp();
  for (int b = 0; b < np; b += 32) {
    const int p = b + lane;
    const int e = p < np ? ldg_cg_i32(a.ws.ids + p) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0) {
      const int pos = S.base[e] + rank;
      a.ws.sorted_pairs[pos] = p;
      a.ws.rowof[p] = pos;
    }
    __syncwarp();
    if (e >= 0 && rank == 0) S.base[e] += __popc(peers);
    __syncwarp();
  }
}

// Warp-level arrival at a tile: true for the last of the 8 warps.
FLINT_DEV bool tile_arrive(Smem& S, int st, int lane) {
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    __threadfence();  // this warp's global and shared writes before the count
    last = (atomicAdd(&S.arr[st], 1) == kCW - 1);
    if (last) {
      S.arr[st] = 0;
      __threadfence();
    }
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  return last != 0;
}

}  // namespace

// ======================================================================
__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(MkArgs A) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const MoEArgs& a = A.a;
  const Geo& G = A.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  int* status = a.ws.status;
  const int H = a.H, I = a.I, SI = a.SI, E = a.E, k = a.k, M = a.M;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
      S.arr[s] = 0;
    }
    mbar_init(&S.xbar, 1);
    S.exit_arr = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ======================================================= producer warp
  if (warp == kCW) {
    if (lane != 0) return;
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
      if (U < 0) U = wait_ge(&A.ctr[C_ROUTED], 1, status) ? ldg_cg_i32(a.ws.uniq) : 0;
      Tile tl = dynamic_tile(a, G, d, U);
      if (tl.type == T_RGU || tl.type == T_RDN) tl.e = ldg_cg_i32(a.ws.uniq + 1 + tl.u);
      S.info[st] = tl;
      issue_tile(a, G, tl, S.stage[st], &S.full[st]);
      ++n;
      if (tl.type == T_END) break;
    }
    return;
  }

  // ==================================================== consumer warps
  const int cw = warp;
  pdl_wait();
  pdl_launch_dependents();
  bool xs_ok = true;
  if (G.xs) xs_ok = __all_sync(0xffffffffu, mbar_wait(&S.xbar, 0, status));

  for (int n = 0; xs_ok; ++n) {
    const int st = n % kStages;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&S.full[st], (n / kStages) & 1, status));
    if (!ok) break;
    const Tile tl = S.info[st];
    if (tl.type == T_END) break;
    const uint8_t* buf = S.stage[st];

    // ---------------------------------------------------------- ROUTER
    if (tl.type == T_ROUTER) {
      // logits[t, e]: lane l owns h = 256 c + 8 l, partial over (c, i)
      // ascending with fmaf, then the xor butterfly 16, 8, 4, 2, 1
      const uint16_t* w = reinterpret_cast<const uint16_t*>(buf);
      for (int tok = cw; tok < M; tok += kCW) {
        const uint16_t* xr = G.xs ? reinterpret_cast<const uint16_t*>(S.xs) + (size_t)tok * H
                                  : a.x + (size_t)tok * H;
        float acc = 0.0f;
        for (int c = 0; 256 * c < H; ++c) {
          const int h = 256 * c + 8 * lane;
          if (h < H) {
            const uint4 xv = G.xs ? *reinterpret_cast<const uint4*>(xr + h) : ldg_cg_v4(xr + h);
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
      if (tile_arrive(S, st, lane) && lane == 0) {
        red_release_add(&A.ctr[C_ROUTER], 1);
        mbar_arrive(&S.empty[st]);
      }
      continue;
    }

    // ------------------------------------------------------------ TOPK
    if (tl.type == T_TOPK) {
      if (warp_wait_ge(&A.ctr[C_ROUTER], E, status, lane))
        for (int tok = cw; tok < M; tok += kCW) topk_token(a, tok, lane);
      if (tile_arrive(S, st, lane)) {
        group_pairs(a, S, lane);
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          st_release(&A.ctr[C_ROUTED], 1);
          mbar_arrive(&S.empty[st]);
        }
      }
      continue;
    }

    // ------------------------------------------------------------ SFIN
    if (tl.type == T_SFIN) {
      if (warp_wait_ge(&A.ctr[C_SGU], G.NSG, status, lane)) {
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
      if (tile_arrive(S, st, lane) && lane == 0) {
        red_release_add(&A.ctr[C_SFIN], 1);
        mbar_arrive(&S.empty[st]);
      }
      continue;
    }

    // --------------------------------------------------------- COMBINE
    if (tl.type == T_COMBINE) {
      const int U = ldg_cg_i32(a.ws.uniq);
      const int expect = U + (SI > 0 ? G.P_sd : 0);
      const int h_end = min(H, tl.row0 + kCombineBlocks * 16);
      bool ok2 = true;
      for (int hb = tl.row0 / 16; hb < h_end / 16 && ok2; ++hb)
        ok2 = warp_wait_ge(&A.down_cnt[hb], expect, status, lane);
      if (ok2) {
        const int nh = h_end - tl.row0;
        for (int idx = cw * 32 + lane; idx < nh * M; idx += kCW * 32) {
          const int tok = idx / nh, h = tl.row0 + idx % nh;
          float R = 0.0f;
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
            for (int pp = 0; pp < G.P_sd; ++pp)
              sum += ldg_cg_f32(part + ((size_t)pp * 16 + h % 16) * 64 + tok);
            ys = round_bf16(sum);
          }
          a.out[(size_t)tok * H + h] = (uint16_t)f32_to_bf16_bits(round_bf16(R) + ys);
        }
      }
      if (tile_arrive(S, st, lane) && lane == 0) mbar_arrive(&S.empty[st]);
      continue;
    }

    // ------------------------------------------------------ MMA tiles
    const bool fp4 = (tl.type == T_RGU || tl.type == T_RDN);
    int ntok = M, off = 0;
    if (fp4) {
      ntok = ldg_cg_i32(a.ws.e_cnt + tl.e);
      off = ldg_cg_i32(a.ws.e_off + tl.e);
    }
    const int nn = max(1, min((ntok + 7) / 8, kCW));  // n-tiles (ntok <= 64)
    const int nk = kCW / nn;                          // K groups
    const int nw = cw % nn, kw = cw / nn;
    const bool active = cw < nn * nk;

    bool dep_ok = true;
    if (tl.type == T_SDN) dep_ok = warp_wait_ge(&A.ctr[C_SFIN], G.NSF, status, lane);
    if (tl.type == T_RDN) dep_ok = warp_wait_ge(&A.gu_done[tl.u], I / 8, status, lane);

    if (active) {
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (dep_ok) {
        // activation row of this lane's token column (n = nw * 8 + g)
        const int n = nw * 8 + g;
        const uint16_t* brow = nullptr;
        bool bsm = false;
        if (n < ntok) {
          if (tl.type == T_RGU) {
            const int tok = ldg_cg_i32(a.ws.sorted_pairs + off + n) / k;
            brow = G.xs ? reinterpret_cast<const uint16_t*>(S.xs) + (size_t)tok * H : a.x + (size_t)tok * H;
            bsm = G.xs;
          } else if (tl.type == T_SGU) {
            brow = G.xs ? reinterpret_cast<const uint16_t*>(S.xs) + (size_t)n * H : a.x + (size_t)n * H;
            bsm = G.xs;
          } else if (tl.type == T_RDN) {
            brow = a.ws.act + (size_t)(off + n) * I;
          } else {
            brow = a.ws.sact + (size_t)n * SI;
          }
        }
        const uint8_t *cg = nullptr, *cg8 = nullptr, *sg = nullptr, *sg8 = nullptr;
        const uint16_t *rg = nullptr, *rg8 = nullptr;
        if (tl.type == T_RGU) {
          cg = buf + g * (H / 2);
          cg8 = buf + (8 + g) * (H / 2);
          sg = buf + 16 * (H / 2) + g * (H / 16);
          sg8 = buf + 16 * (H / 2) + (8 + g) * (H / 16);
        } else if (tl.type == T_RDN) {
          cg = buf + g * (I / 2);
          cg8 = buf + (8 + g) * (I / 2);
          sg = buf + 16 * (I / 2) + g * (I / 16);
          sg8 = buf + 16 * (I / 2) + (8 + g) * (I / 16);
        } else {
          const int pk = tl.ns * kSliceK;
          rg = reinterpret_cast<const uint16_t*>(buf) + g * pk;
          rg8 = reinterpret_cast<const uint16_t*>(buf) + (8 + g) * pk;
        }
        int s = kw;
        uint4 xb[4];
        if (s < tl.ns) load_b(xb, brow, bsm, (tl.s0 + s) * kSliceK, t);
        for (; s < tl.ns; s += nk) {
          uint32_t af[4][2][4];
          if (fp4) a_frags_fp4(cg, cg8, sg, sg8, s, t, af);
          else a_frags_bf16(rg, rg8, s, t, af);
          uint4 xn[4];
          if (s + nk < tl.ns) load_b(xn, brow, bsm, (tl.s0 + s + nk) * kSliceK, t);
          mma_slice(acc, af, xb);
#pragma unroll
          for (int q = 0; q < 4; ++q) xb[q] = xn[q];
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) S.red[st][cw][lane][i] = acc[i];
    }
    if (!tile_arrive(S, st, lane)) continue;

    // ---- last warp: fixed-order reduction over K groups + epilogue
    for (int nt = 0; nt < nn; ++nt) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float sum = S.red[st][nt][lane][i];
        for (int q = 1; q < nk; ++q) sum += S.red[st][q * nn + nt][lane][i];
        v[i] = sum;
      }
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
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      if (tl.type == T_RGU) red_release_add(&A.gu_done[tl.u], 1);
      else if (tl.type == T_SGU) red_release_add(&A.ctr[C_SGU], 1);
      else red_release_add(&A.down_cnt[tl.row0 / 16], 1);
      mbar_arrive(&S.empty[st]);
    }
  }

  // ---- exit: the last warp of the last CTA returns every counter to zero
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    __threadfence();
    last = (atomicAdd(&S.exit_arr, 1) == kCW - 1);
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  if (lane == 0) {
    __threadfence();
    last = (atomicAdd(&A.ctr[C_EXIT], 1) == (int)gridDim.x - 1);
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  for (int i = lane; i < C_N; i += 32)
    if (i != C_EXIT) A.ctr[i] = 0;
  for (int i = lane; i < E; i += 32) A.gu_done[i] = 0;
  for (int i = lane; i < H / 16; i += 32) A.down_cnt[i] = 0;
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    A.ctr[C_EXIT] = 0;
  }
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
