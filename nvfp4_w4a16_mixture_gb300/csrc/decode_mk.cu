// Decode megakernel: the whole MoE block for M <= kDecodeMaxTokens tokens in
// one persistent launch.
//
// Page "vllm.models.flint.ops.moe": the decode path is _router_kernel
// (router GEMV, top-k by the token's last program), _gate_up_gemv_kernel
// (per (token, expert) NVFP4 gate/up + SiLU * up) and _down_gemv_kernel
// (down GEMV over the top-k experts, weighted combine, shared-expert add),
// with the shared expert on an auxiliary stream.  Here the same steps run as
// work tiles of one kernel, chained by device-side counters, so the weight
// stream never drains between steps:
//
//   phase 1 (static, no dependencies; weights staged before the PDL wait)
//     ROUTER  one router row: logits of all tokens in a fixed fp32 order; the
//             last router tile runs top-k + expert grouping, then raises the
//             routing flag
//     SGU     shared expert gate/up: 8 intermediate rows (gate + up), a K part
//   phase 2 (dynamic, atomic work counter, decoded after the routing flag)
//     RGU     routed expert gate/up: expert u, 8 intermediate rows, all K
//     SDN     shared expert down: 16 output rows, a K part  (after all SGU)
//     RDN     routed expert down: expert u, 16 output rows  (after u's RGU)
//   the last tile of each 16-row output block forms
//     out = bf16(bf16(sum_j tw_j y_j) + ys) for every token.
//
// CTA: 8 consumer warps + 1 producer warp.  The producer copies each tile's
// weight rows (NVFP4 codes + E4M3 scales, or BF16 rows) into a 3-stage
// shared-memory ring with cp.async.bulk (mbarrier completion), running ahead
// of the consumers; a tile's dependency wait happens after its weights have
// landed.  Consumers split K across warps (128-wide slices), run mma.sync
// m16n8k16 (bf16, fp32 accumulate) with the weight rows as A and up to 8
// tokens per B tile, reduce in shared memory in warp order, and apply the
// tile's epilogue.  Deadlock freedom: every wait targets tiles of lower index,
// tiles are taken in index order and all counters are bounded waits.
#include "common.cuh"
#include "internal.h"

namespace flint {

namespace {

constexpr int kCW = 8;                       // consumer warps
constexpr int kThreads = (kCW + 1) * 32;     // + producer warp
constexpr int kStages = 3;
constexpr int kStageBytes = 32 * 1024;
constexpr int kNTP = 4;                      // 8-token n-tiles per pass
constexpr int kSliceK = 128;
constexpr int kBarConsumers = 1;             // named barrier id
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s bound on any wait

enum : int { T_END = 0, T_ROUTER = 1, T_SGU = 2, T_RGU = 3, T_SDN = 4, T_RDN = 5 };

struct Tile {
  int type;
  int u, e;        // unique-expert slot and expert id (routed tiles)
  int row0;        // first intermediate row (gate/up) or output row (down)
  int part;        // K part (shared tiles)
  int s0, ns;      // first K slice and slice count of this tile
};

struct Smem {
  uint8_t stage[kStages][kStageBytes];
  float red[kCW][kNTP][32][4];
  Tile info[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int flag;
  int stop;
  int cnt[kMaxE];
  int base[kMaxE];
};

FLINT_DEV unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait until *p >= target.  On timeout records FLINT_ERR_TIMEOUT in
// the status word; returns immediately once any error is recorded.
FLINT_DEV bool wait_ge(const int* p, int target, int* status) {
  const unsigned long long t0 = now_ns();
  for (int i = 0;; ++i) {
    if (ld_acquire(p) >= target) return true;
    if (i >= 32) {
      if (ld_acquire(status) != 0) return false;
      if (now_ns() - t0 > kWaitNs) {
        atomicCAS(status, 0, FLINT_ERR_TIMEOUT);
        return false;
      }
      __nanosleep(64);
    }
  }
}

FLINT_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > kWaitNs) {
      atomicCAS(status, 0, FLINT_ERR_TIMEOUT);
      return false;
    }
  }
}

FLINT_DEV void cbar() { named_bar(kBarConsumers, kCW * 32); }

// -------------------------------------------------------------- geometry
struct Geo {
  int nsl_H, nsl_I, nsl_SI;  // K slices of 128
  int P_sg, spp_sg;          // shared gate/up: K parts, slices per part
  int P_sd, spp_sd;          // shared down: K parts, slices per part
  int NR, NSG, N1;           // router tiles, shared gate/up tiles, phase-1 total
};

FLINT_DEV Tile static_tile(const MoEArgs& a, const Geo& G, int idx) {
  Tile t{};
  if (idx < G.NR) {
    t.type = T_ROUTER;
    t.e = idx;
    return t;
  }
  const int d = idx - G.NR;
  t.type = T_SGU;
  t.row0 = (d / G.P_sg) * 8;
  t.part = d % G.P_sg;
  t.s0 = t.part * G.spp_sg;
  t.ns = min(G.spp_sg, G.nsl_H - t.s0);
  return t;
}

FLINT_DEV Tile dynamic_tile(const MoEArgs& a, const Geo& G, int d, int U) {
  Tile t{};
  const int nrg = U * (a.I / 8);
  const int nsd = a.SI > 0 ? (a.H / 16) * G.P_sd : 0;
  const int nrd = U * (a.H / 16);
  if (d < nrg) {
    t.type = T_RGU;
    t.u = d / (a.I / 8);
    t.row0 = (d % (a.I / 8)) * 8;
    t.s0 = 0;
    t.ns = G.nsl_H;
  } else if (d < nrg + nsd) {
    const int dd = d - nrg;
    t.type = T_SDN;
    t.row0 = (dd / G.P_sd) * 16;
    t.part = dd % G.P_sd;
    t.s0 = t.part * G.spp_sd;
    t.ns = min(G.spp_sd, G.nsl_SI - t.s0);
  } else if (d < nrg + nsd + nrd) {
    const int dd = d - nrg - nsd;
    t.type = T_RDN;
    t.u = dd / (a.H / 16);
    t.row0 = (dd % (a.H / 16)) * 16;
    t.s0 = 0;
    t.ns = G.nsl_I;
  } else {
    t.type = T_END;
  }
  return t;
}

// Issue the bulk copies of a tile's weights into stage `buf`; returns bytes.
FLINT_DEV uint32_t issue_tile(const MoEArgs& a, const Geo& G, const Tile& t, uint8_t* buf,
                              uint64_t* bar) {
  const int H = a.H, I = a.I, SI = a.SI;
  uint32_t bytes = 0;
  switch (t.type) {
    case T_ROUTER: {
      bytes = H * 2;
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(buf, a.router_w + (size_t)t.e * H, bytes, bar);
      break;
    }
    case T_SGU: {
      const int pk = t.ns * kSliceK;  // K elements in this part
      bytes = 16 * pk * 2;
      mbar_arrive_expect_tx(bar, bytes);
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
      bytes = 16 * (H / 2) + 16 * (H / 16);
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(buf, a.w13 + rg * (H / 2), 8 * (H / 2), bar);
      bulk_g2s(buf + 8 * (H / 2), a.w13 + ru * (H / 2), 8 * (H / 2), bar);
      bulk_g2s(buf + 16 * (H / 2), a.w13_sf + rg * (H / 16), 8 * (H / 16), bar);
      bulk_g2s(buf + 16 * (H / 2) + 8 * (H / 16), a.w13_sf + ru * (H / 16), 8 * (H / 16), bar);
      break;
    }
    case T_SDN: {
      const int pk = t.ns * kSliceK;
      bytes = 16 * pk * 2;
      mbar_arrive_expect_tx(bar, bytes);
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
      bytes = 16 * (I / 2) + 16 * (I / 16);
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(buf, a.w2 + r * (I / 2), 16 * (I / 2), bar);
      bulk_g2s(buf + 16 * (I / 2), a.w2_sf + r * (I / 16), 16 * (I / 16), bar);
      break;
    }
    default:
      mbar_arrive(bar);
  }
  return bytes;
}

// ---------------------------------------------------------------- compute
// NVFP4 rows: cg / cg8 point at the codes of tile rows g and g + 8 (row
// stride irrelevant here), sg / sg8 at their scales; slice s of the tile.
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

// BF16 rows: rg / rg8 point at K element 0 of tile rows g and g + 8.
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

// acc[nt] += A(slice) * B(rows brow[nt], K offset koff of the activation row)
FLINT_DEV void mma_tiles(float (&acc)[kNTP][4], const uint32_t (&af)[4][2][4],
                         const uint16_t* const (&brow)[kNTP], int koff, int t, int ntiles) {
#pragma unroll
  for (int nt = 0; nt < kNTP; ++nt) {
    if (nt >= ntiles) break;
    uint4 xb[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      xb[q] = brow[nt] ? ldg_cg_v4(brow[nt] + koff + 32 * t + 8 * q) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      mma_bf16_16816(acc[nt], af[q][0][0], af[q][0][1], af[q][0][2], af[q][0][3],
                     __byte_perm(xb[q].x, xb[q].z, 0x5410), __byte_perm(xb[q].x, xb[q].z, 0x7632));
      mma_bf16_16816(acc[nt], af[q][1][0], af[q][1][1], af[q][1][2], af[q][1][3],
                     __byte_perm(xb[q].y, xb[q].w, 0x5410), __byte_perm(xb[q].y, xb[q].w, 0x7632));
    }
  }
}

FLINT_DEV void zero_acc(float (&acc)[kNTP][4]) {
#pragma unroll
  for (int nt = 0; nt < kNTP; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
}

FLINT_DEV void store_red(Smem& S, const float (&acc)[kNTP][4], int cw, int lane) {
#pragma unroll
  for (int nt = 0; nt < kNTP; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) S.red[cw][nt][lane][i] = acc[nt][i];
}

FLINT_DEV float red_sum(const Smem& S, int nt, int lane, int i) {
  float v = S.red[0][nt][lane][i];
#pragma unroll
  for (int w = 1; w < kCW; ++w) v += S.red[w][nt][lane][i];
  return v;
}

// --------------------------------------------------------- routing step
// Top-k of one token by one warp (keys: order-preserving bf16 bits << 8 |
// (E - 1 - e)); writes ids / tw (workspace and optional user copies).
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
    sum = sum + s;
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

// Expert grouping of the M*k pairs by one warp: counts, offsets, the list of
// routed experts, and the pairs stable-sorted by expert (rowof = inverse).
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

// out for the 16 output rows of block hb, all tokens (consumer threads).
FLINT_DEV void combine_block(const MoEArgs& a, int hb, int ctid) {
  const int H = a.H, k = a.k, h0 = hb * 16;
  for (int idx = ctid; idx < a.M * 16; idx += kCW * 32) {
    const int tt = idx >> 4, h = h0 + (idx & 15);
    float R = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int p = tt * k + j;
      const float w = ldg_cg_f32(a.ws.tw + p);
      const int row = ldg_cg_i32(a.ws.rowof + p);
      R = R + w * bf16_bits_to_f32(ldg_cg_u16(a.ws.y + (size_t)row * H + h));  // rank order
    }
    const float ys = a.SI > 0 ? bf16_bits_to_f32(ldg_cg_u16(a.ws.ys + (size_t)tt * H + h)) : 0.0f;
    a.out[(size_t)tt * H + h] = (uint16_t)f32_to_bf16_bits(round_bf16(R) + ys);
  }
}

}  // namespace

struct MkArgs {
  MoEArgs a;
  Geo G;
  int* ctr;       // [0] work, [1] router tiles done, [2] routing flag, [3] shared gate/up
                  // tiles done, [4] CTAs exited
  int* sg_cnt;    // [SI/8]   K parts done per shared gate/up tile
  int* sd_cnt;    // [H/16]   K parts done per shared down tile
  int* gu_done;   // [E]      gate/up tiles done per routed-expert slot
  int* down_cnt;  // [H/16]   down tiles done per output block
  float* part_sg; // [SI/8][P_sg][16][64]
  float* part_sd; // [H/16][P_sd][16][64]
};

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(MkArgs A) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const MoEArgs& a = A.a;
  const Geo& G = A.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  int* status = a.ws.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    fence_mbar_init();
    S.stop = 0;
  }
  __syncthreads();

  // ======================================================= producer warp
  if (warp == kCW) {
    if (lane != 0) return;
    int n = 0;  // tiles staged so far
    bool ok = true;
    auto put = [&](const Tile& tl) {
      const int st = n % kStages;
      if (n >= kStages && !mbar_wait(&S.empty[st], ((n / kStages) - 1) & 1, status)) ok = false;
      S.info[st] = tl;
      issue_tile(a, G, tl, S.stage[st], &S.full[st]);
      ++n;
    };
    int idx = blockIdx.x;
    // weights of the first static tiles do not depend on earlier grids
    for (; idx < G.N1 && n < kStages; idx += gridDim.x) put(static_tile(a, G, idx));
    pdl_wait();
    for (; idx < G.N1; idx += gridDim.x) put(static_tile(a, G, idx));
    int U = -1;
    for (;;) {
      const int st = n % kStages;
      if (!ok || (n >= kStages && !mbar_wait(&S.empty[st], ((n / kStages) - 1) & 1, status))) {
        // a bounded wait gave up (error recorded): tell the consumers to stop
        S.info[st].type = T_END;
        mbar_arrive(&S.full[st]);
        break;
      }
      const int d = atomicAdd(&A.ctr[0], 1);
      if (U < 0) {
        U = 0;
        if (wait_ge(&A.ctr[2], 1, status)) U = ldg_cg_i32(a.ws.uniq);
      }
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
  const int cw = warp, ctid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  const int H = a.H, I = a.I, SI = a.SI, E = a.E, k = a.k, M = a.M;

  for (int n = 0;; ++n) {
    const int st = n % kStages;
    // every consumer thread waits; the stop decision is made uniform
    if (!mbar_wait(&S.full[st], (n / kStages) & 1, status)) S.stop = 1;
    cbar();
    if (S.stop) break;
    const Tile tl = S.info[st];
    if (tl.type == T_END) break;
    const uint8_t* buf = S.stage[st];

    if (tl.type == T_ROUTER) {
      // logits[t, e] for every token; lane l owns h = 256 c + 8 l (c = 0..)
      const uint16_t* w = reinterpret_cast<const uint16_t*>(buf);
      for (int tok = cw; tok < M; tok += kCW) {
        const uint16_t* xr = a.x + (size_t)tok * H;
        float acc = 0.0f;
        for (int c = 0; 256 * c < H; ++c) {
          const int h = 256 * c + 8 * lane;
          if (h < H) {
            const uint4 xv = ldg_cg_v4(xr + h);
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
      cbar();
      if (ctid == 0) {
        mbar_arrive(&S.empty[st]);
        __threadfence();
        S.flag = (atomicAdd(&A.ctr[1], 1) == E - 1);
      }
      cbar();
      if (S.flag) {
        __threadfence();
        for (int tok = cw; tok < M; tok += kCW) topk_token(a, tok, lane);
        __threadfence();
        cbar();
        if (cw == 0) group_pairs(a, S, lane);
        __threadfence();
        cbar();
        if (ctid == 0) st_release(&A.ctr[2], 1);
      }
      continue;
    }

    // ---- MMA tiles: geometry of A rows g / g + 8 in the stage
    const bool fp4 = (tl.type == T_RGU || tl.type == T_RDN);
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

    // ---- dependencies (weights are already in the stage)
    int ntok = M, off = 0, cnt = 0;
    if (tl.type == T_RGU || tl.type == T_RDN) {
      cnt = ldg_cg_i32(a.ws.e_cnt + tl.e);
      off = ldg_cg_i32(a.ws.e_off + tl.e);
      ntok = cnt;
    }
    if (tl.type == T_SDN || tl.type == T_RDN) {
      if (ctid == 0) {
        if (tl.type == T_SDN) wait_ge(&A.ctr[3], SI / 8, status);
        else wait_ge(&A.gu_done[tl.u], I / 8, status);
      }
      cbar();
    }

    // ---- passes of up to 32 tokens
    for (int n0 = 0; n0 < ntok; n0 += kNTP * 8) {
      const int npass = min(ntok - n0, kNTP * 8);
      const int ntiles = (npass + 7) / 8;
      const uint16_t* brow[kNTP];
#pragma unroll
      for (int nt = 0; nt < kNTP; ++nt) {
        const int nn = n0 + nt * 8 + g;
        const uint16_t* p = nullptr;
        if (nt * 8 + g < npass) {
          if (tl.type == T_RGU) p = a.x + (size_t)(ldg_cg_i32(a.ws.sorted_pairs + off + nn) / k) * H;
          else if (tl.type == T_SGU) p = a.x + (size_t)nn * H;
          else if (tl.type == T_RDN) p = a.ws.act + (size_t)(off + nn) * I;
          else p = a.ws.sact + (size_t)nn * SI;
        }
        brow[nt] = p;
      }
      float acc[kNTP][4];
      zero_acc(acc);
      for (int s = cw; s < tl.ns; s += kCW) {
        uint32_t af[4][2][4];
        if (fp4) a_frags_fp4(cg, cg8, sg, sg8, s, t, af);
        else a_frags_bf16(rg, rg8, s, t, af);
        mma_tiles(acc, af, brow, (tl.s0 + s) * kSliceK, t, ntiles);
      }
      store_red(S, acc, cw, lane);
      cbar();
      if (ctid == 0 && n0 + kNTP * 8 >= ntok) mbar_arrive(&S.empty[st]);  // stage fully read
      if (cw < ntiles) {
        const int nt = cw;
        if (tl.type == T_RGU) {
          const float gs = a.w13_gs[tl.e];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int nn = nt * 8 + 2 * t + c;
            if (nn < npass) {
              const float gv = red_sum(S, nt, lane, c) * 128.0f * gs;
              const float uv = red_sum(S, nt, lane, 2 + c) * 128.0f * gs;
              a.ws.act[(size_t)(off + n0 + nn) * I + tl.row0 + g] =
                  (uint16_t)f32_to_bf16_bits(silu_approx(gv) * uv);
            }
          }
        } else if (tl.type == T_RDN) {
          const float gs2 = a.w2_gs[tl.e];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int nn = nt * 8 + 2 * t + (i & 1);
            if (nn < npass)
              a.ws.y[(size_t)(off + n0 + nn) * H + tl.row0 + g + (i >> 1) * 8] =
                  (uint16_t)f32_to_bf16_bits(red_sum(S, nt, lane, i) * 128.0f * gs2);
          }
        } else {
          // shared tiles: fp32 partial of this K part, [row][token]
          float* part = tl.type == T_SGU
                            ? A.part_sg + ((size_t)(tl.row0 / 8) * G.P_sg + tl.part) * 16 * 64
                            : A.part_sd + ((size_t)(tl.row0 / 16) * G.P_sd + tl.part) * 16 * 64;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int nn = nt * 8 + 2 * t + (i & 1);
            if (nn < npass) part[(g + (i >> 1) * 8) * 64 + n0 + nn] = red_sum(S, nt, lane, i);
          }
        }
      }
      cbar();
    }
    if (ntok == 0 && ctid == 0) mbar_arrive(&S.empty[st]);

    // ---- completion
    if (tl.type == T_RGU) {
      if (ctid == 0) {
        __threadfence();
        atomicAdd(&A.gu_done[tl.u], 1);
      }
      continue;
    }
    int hb = -1;  // output block that received a down tile
    if (tl.type == T_SGU || tl.type == T_SDN) {
      const bool sgu = tl.type == T_SGU;
      int* pc = sgu ? &A.sg_cnt[tl.row0 / 8] : &A.sd_cnt[tl.row0 / 16];
      const int P = sgu ? G.P_sg : G.P_sd;
      if (ctid == 0) {
        __threadfence();
        S.flag = (atomicAdd(pc, 1) == P - 1);
      }
      cbar();
      if (!S.flag) continue;
      __threadfence();
      if (ctid == 0) *pc = 0;
      const float* part = sgu ? A.part_sg + (size_t)(tl.row0 / 8) * P * 16 * 64
                              : A.part_sd + (size_t)(tl.row0 / 16) * P * 16 * 64;
      if (sgu) {
        for (int idx = ctid; idx < 8 * M; idx += kCW * 32) {
          const int r = idx / M, tok = idx % M;
          float gsum = 0.0f, usum = 0.0f;
          for (int pp = 0; pp < P; ++pp) {
            gsum += ldg_cg_f32(part + ((size_t)pp * 16 + r) * 64 + tok);
            usum += ldg_cg_f32(part + ((size_t)pp * 16 + 8 + r) * 64 + tok);
          }
          const float gS = round_bf16(gsum), uS = round_bf16(usum);
          a.ws.sact[(size_t)tok * SI + tl.row0 + r] = (uint16_t)f32_to_bf16_bits(silu_approx(gS) * uS);
        }
        cbar();
        if (ctid == 0) {
          __threadfence();
          atomicAdd(&A.ctr[3], 1);
        }
        continue;
      }
      for (int idx = ctid; idx < 16 * M; idx += kCW * 32) {
        const int r = idx / M, tok = idx % M;
        float sum = 0.0f;
        for (int pp = 0; pp < P; ++pp) sum += ldg_cg_f32(part + ((size_t)pp * 16 + r) * 64 + tok);
        a.ws.ys[(size_t)tok * H + tl.row0 + r] = (uint16_t)f32_to_bf16_bits(sum);
      }
      cbar();
      hb = tl.row0 / 16;
    } else {  // T_RDN
      hb = tl.row0 / 16;
    }
    // a down tile of output block hb is complete: last one combines
    if (ctid == 0) {
      __threadfence();
      const int expect = ldg_cg_i32(a.ws.uniq) + (SI > 0 ? 1 : 0);
      S.flag = (atomicAdd(&A.down_cnt[hb], 1) == expect - 1);
    }
    cbar();
    if (S.flag) {
      __threadfence();
      combine_block(a, hb, ctid);
    }
  }

  // ---- exit: the last CTA returns every counter to zero
  cbar();
  if (ctid == 0) {
    __threadfence();
    S.flag = (atomicAdd(&A.ctr[4], 1) == (int)gridDim.x - 1);
  }
  cbar();
  if (S.flag) {
    __threadfence();
    for (int i = ctid; i < 4; i += kCW * 32) A.ctr[i] = 0;
    for (int i = ctid; i < E; i += kCW * 32) A.gu_done[i] = 0;
    for (int i = ctid; i < H / 16; i += kCW * 32) { A.down_cnt[i] = 0; A.sd_cnt[i] = 0; }
    for (int i = ctid; i < SI / 8; i += kCW * 32) A.sg_cnt[i] = 0;
    cbar();
    if (ctid == 0) { __threadfence(); A.ctr[4] = 0; }
  }
}

// ---------------------------------------------------------------- launch
static int g_num_sms = 0;

static Geo make_geo(const MoEArgs& a) {
  Geo G{};
  G.nsl_H = a.H / kSliceK;
  G.nsl_I = a.I / kSliceK;
  G.nsl_SI = a.SI / kSliceK;
  const int max_sl_bf16 = kStageBytes / (16 * kSliceK * 2);  // slices of 16 BF16 rows per stage
  G.P_sg = (G.nsl_H + max_sl_bf16 - 1) / max_sl_bf16;
  G.spp_sg = (G.nsl_H + G.P_sg - 1) / G.P_sg;
  G.P_sg = (G.nsl_H + G.spp_sg - 1) / G.spp_sg;
  if (a.SI > 0) {
    G.P_sd = (G.nsl_SI + max_sl_bf16 - 1) / max_sl_bf16;
    G.spp_sd = (G.nsl_SI + G.P_sd - 1) / G.P_sd;
    G.P_sd = (G.nsl_SI + G.spp_sd - 1) / G.spp_sd;
  } else {
    G.P_sd = 1;
    G.spp_sd = 1;
  }
  G.NR = a.E;
  G.NSG = (a.SI / 8) * G.P_sg;
  G.N1 = G.NR + G.NSG;
  return G;
}

bool decode_mk_supported(const flint_moe_shape& s) {
  return s.M <= kDecodeMaxTokens && 9 * s.H <= kStageBytes && 9 * s.I <= kStageBytes &&
         2 * s.H <= kStageBytes;
}

size_t decode_mk_ctr_bytes(const flint_moe_shape& s) {
  return (size_t)(8 + s.SI / 8 + 2 * (s.H / 16) + s.E) * 4;
}

size_t decode_mk_part_bytes(const flint_moe_shape& s) {
  MoEArgs a{};
  a.H = s.H; a.I = s.I; a.SI = s.SI; a.E = s.E;
  const Geo G = make_geo(a);
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
  A.G = make_geo(a);
  A.ctr = mk_ctr;
  A.sg_cnt = A.ctr + 8;
  A.sd_cnt = A.sg_cnt + a.SI / 8;
  A.down_cnt = A.sd_cnt + a.H / 16;
  A.gu_done = A.down_cnt + a.H / 16;
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
