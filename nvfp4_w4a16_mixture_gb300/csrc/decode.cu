// Fallback decode kernels (few tokens, M <= 64) for shapes outside the
// main decode kernels' limits (decode2.cu: shared intermediate <= 1024,
// expert intermediate <= 2048, M * top_k <= 1024): NVFP4 gate/up + SiLU*up,
// and the down projection with the weighted combine and the shared-expert add.
//
// Page "vllm.models.flint.ops.moe": _gate_up_gemv_kernel
// (act[p] = silu(x[t] Wg[e]^T) * (x[t] Wu[e]^T), global scale on the fp32
// accumulator), _down_gemv_kernel (y_j = bf16(act W2[e_j]^T * gs),
// out = bf16(bf16(sum_j tw_j y_j) + shared)), and the module's Numerics rule.
//
// Layout of the work: expert-major.  Every routed expert that received at
// least one (token, slot) pair is streamed once per call, for all of its
// tokens.  One CTA (8 warps) owns a 16-row weight tile; the warps split K in
// 128-wide slices and the partial sums are reduced in shared memory in warp
// order.  The inner products run on the tensor cores (mma.sync m16n8k16,
// bf16 in, fp32 accumulate) with the weight rows as the 16-row A operand and
// up to 8 tokens per B tile, which keeps the dequantisation, not the
// multiply-adds, on the CUDA cores.
//
// Operand mapping inside a slice: thread (g = lane / 4, t = lane % 4) holds
// 32 consecutive K (16 code bytes) of rows g and g + 8 of the tile.  Each
// 8-code word yields four bf16x2 pairs (codes i, i + 4); the activation
// vector is permuted the same way, so every product pairs matching K.
// Dequantisation: each pair is built as e2m1 * 2^-126 (bit placement, exact)
// and multiplied by bf16(scale * 2^119), giving e2m1 * scale * 2^-7 exactly;
// the fp32 accumulator is multiplied back by 2^7 (exact).
#include "common.cuh"
#include "frag.cuh"
#include "internal.h"

namespace flint {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kNT = 8;  // 8-token n-tiles per pass (64 tokens)

FLINT_DEV void load_slice(Fp4Slice& d, const uint8_t* cg, const uint8_t* cg8, const uint8_t* sg,
                          const uint8_t* sg8, int s, int t) {
  d.c0 = ldg_nc_v4(cg + s * (kSliceK / 2) + 16 * t);
  d.c1 = ldg_nc_v4(cg8 + s * (kSliceK / 2) + 16 * t);
  d.s0 = ldg_nc_u16(sg + s * (kSliceK / 16) + 2 * t);
  d.s1 = ldg_nc_u16(sg8 + s * (kSliceK / 16) + 2 * t);
}

FLINT_DEV void load_slice(Bf16Slice& d, const uint16_t* rg, const uint16_t* rg8, int s, int t) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    d.r0[q] = ldg_nc_v4(rg + s * kSliceK + 32 * t + 8 * q);
    d.r1[q] = ldg_nc_v4(rg8 + s * kSliceK + 32 * t + 8 * q);
  }
}

// acc[nt] += A(slice s) * B, where B column g of n-tile nt is the 16-bit
// activation row brow[nt] (nullptr = zero column).
template <class Slice>
FLINT_DEV void mma_slice(float (&acc)[kNT][4], const Slice& d, int s, int t,
                         const uint16_t* const (&brow)[kNT], int ntiles) {
  uint32_t af[4][2][4];
  a_frags(d, af);
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    if (nt >= ntiles) break;
    uint4 xb[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      xb[q] = brow[nt] ? ldg_cg_v4(brow[nt] + s * kSliceK + 32 * t + 8 * q) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t b00 = __byte_perm(xb[q].x, xb[q].z, 0x5410);
      const uint32_t b01 = __byte_perm(xb[q].x, xb[q].z, 0x7632);
      const uint32_t b10 = __byte_perm(xb[q].y, xb[q].w, 0x5410);
      const uint32_t b11 = __byte_perm(xb[q].y, xb[q].w, 0x7632);
      mma_bf16_16816(acc[nt], af[q][0][0], af[q][0][1], af[q][0][2], af[q][0][3], b00, b01);
      mma_bf16_16816(acc[nt], af[q][1][0], af[q][1][1], af[q][1][2], af[q][1][3], b10, b11);
    }
  }
}

// Runs the K loop of one 16-row tile for one pass of up to 64 tokens and
// leaves the warp-ordered sum in red (per n-tile, lane, fragment).
template <class Slice, class Loader>
FLINT_DEV void tile_pass(float (&red)[kDecWarps][kNT][32][4], int nslice,
                         const uint16_t* const (&brow)[kNT], int ntiles, Slice& first,
                         bool first_loaded, Loader load) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = lane & 3;
  float acc[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
  Slice cur = first, nxt;
  int s = warp;
  if (s < nslice && !first_loaded) load(cur, s);
  for (; s < nslice; s += kDecWarps) {
    if (s + kDecWarps < nslice) load(nxt, s + kDecWarps);
    mma_slice(acc, cur, s, t, brow, ntiles);
    cur = nxt;
  }
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][nt][lane][i] = acc[nt][i];
  __syncthreads();
}

// Sum of the warps' partials for n-tile nt, lane, fragment i (warp order).
FLINT_DEV float red_sum(const float (&red)[kDecWarps][kNT][32][4], int nt, int lane, int i) {
  float v = red[0][nt][lane][i];
#pragma unroll
  for (int w = 1; w < kDecWarps; ++w) v += red[w][nt][lane][i];
  return v;
}

// ----------------------------------------------------------------------------
// Gate/up.  Items [0, ns_items): shared expert, 8 intermediate rows each
// (tile rows 0..7 = gate rows r0.., rows 8..15 = up rows SI + r0..).  Items
// after that: (routed expert u, 8 intermediate rows), u < U.
__global__ void __launch_bounds__(kDecThreads) gate_up_decode_kernel(MoEArgs a, int ns_items) {
  SpanGuard<kSpanGateUp> span_guard;
  __shared__ float red[kDecWarps][kNT][32][4];
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int warp = threadIdx.x >> 5;
  const int H = a.H, I = a.I, SI = a.SI, k = a.k;
  const int nslice = H / kSliceK;
  const int item = blockIdx.x;

  if (item < ns_items) {
    const int r0 = item * 8;
    const uint16_t* rg = a.shared_gu + (size_t)(r0 + g) * H;
    const uint16_t* rg8 = a.shared_gu + (size_t)(SI + r0 + g) * H;
    auto load = [&](Bf16Slice& d, int s) { load_slice(d, rg, rg8, s, t); };
    Bf16Slice first;
    if (warp < nslice) load(first, warp);  // weights: before the dependency wait
    pdl_wait();
    pdl_launch_dependents();
    for (int n0 = 0; n0 < a.M; n0 += kNT * 8) {
      const int ntok = min(a.M - n0, kNT * 8);
      const int ntiles = (ntok + 7) / 8;
      const uint16_t* brow[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = nt * 8 + g;
        brow[nt] = n < ntok ? a.x + (size_t)(n0 + n) * H : nullptr;
      }
      tile_pass(red, nslice, brow, ntiles, first, n0 == 0, load);
      if (warp < ntiles) {
        const int nt = warp;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int n = nt * 8 + 2 * t + c;
          if (n < ntok) {
            const float gs_ = round_bf16(red_sum(red, nt, lane, c));
            const float us_ = round_bf16(red_sum(red, nt, lane, 2 + c));
            const float v = silu_approx(gs_) * us_;
            a.ws.sact[(size_t)(n0 + n) * SI + r0 + g] = (uint16_t)f32_to_bf16_bits(v);
          }
        }
      }
      __syncthreads();
    }
    return;
  }

  pdl_wait();
  pdl_launch_dependents();
  const int ri = item - ns_items;
  const int ui = ri / (I / 8), rt = ri % (I / 8);
  const int U = ldg_cg_i32(a.ws.uniq);
  if (ui >= U) return;
  const int e = ldg_cg_i32(a.ws.uniq + 1 + ui);
  const int cnt = ldg_cg_i32(a.ws.e_cnt + e);
  const int off = ldg_cg_i32(a.ws.e_off + e);
  const int r0 = rt * 8;
  const size_t row_g = (size_t)e * 2 * I + r0 + g, row_u = row_g + I;
  const uint8_t* cg = a.w13 + row_g * (H / 2);
  const uint8_t* cg8 = a.w13 + row_u * (H / 2);
  const uint8_t* sg = a.w13_sf + row_g * (H / 16);
  const uint8_t* sg8 = a.w13_sf + row_u * (H / 16);
  auto load = [&](Fp4Slice& d, int s) { load_slice(d, cg, cg8, sg, sg8, s, t); };
  const float gs = a.w13_gs[e] * 128.0f;  // undo the 2^-7 of the operands, then gs
  Fp4Slice first;
  for (int n0 = 0; n0 < cnt; n0 += kNT * 8) {
    const int ntok = min(cnt - n0, kNT * 8);
    const int ntiles = (ntok + 7) / 8;
    const uint16_t* brow[kNT];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const int n = nt * 8 + g;
      brow[nt] = nullptr;
      if (n < ntok) {
        const int p = ldg_cg_i32(a.ws.sorted_pairs + off + n0 + n);
        brow[nt] = a.x + (size_t)(p / k) * H;
      }
    }
    tile_pass(red, nslice, brow, ntiles, first, false, load);
    if (warp < ntiles) {
      const int nt = warp;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int n = nt * 8 + 2 * t + c;
        if (n < ntok) {
          // (acc * 2^7) * gs == acc' * gs for the true accumulator acc'
          const float gv = red_sum(red, nt, lane, c) * 128.0f * a.w13_gs[e];
          const float uv = red_sum(red, nt, lane, 2 + c) * 128.0f * a.w13_gs[e];
          const float v = silu_approx(gv) * uv;
          a.ws.act[(size_t)(off + n0 + n) * I + r0 + g] = (uint16_t)f32_to_bf16_bits(v);
        }
      }
    }
    __syncthreads();
  }
  (void)gs;
}

// ----------------------------------------------------------------------------
// Down + combine.  Items [0, ns_items): shared expert, 16 output rows each;
// then (routed expert u, 16 output rows).  Each item writes its y / ys rows;
// the last item to finish an output row block (counter per block) forms
// out = bf16(bf16(sum_j tw_j y_j) + ys) for every token of that block.
__global__ void __launch_bounds__(kDecThreads) down_decode_kernel(MoEArgs a, int ns_items) {
  SpanGuard<kSpanDown> span_guard;
  __shared__ float red[kDecWarps][kNT][32][4];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int warp = threadIdx.x >> 5;
  const int H = a.H, I = a.I, SI = a.SI, k = a.k, M = a.M;
  const int hblocks = H / 16;
  const int item = blockIdx.x;
  int hb;

  if (item < ns_items) {
    hb = item;
    const int h0 = hb * 16;
    const int nslice = SI / kSliceK;
    const uint16_t* rg = a.shared_down + (size_t)(h0 + g) * SI;
    const uint16_t* rg8 = a.shared_down + (size_t)(h0 + 8 + g) * SI;
    auto load = [&](Bf16Slice& d, int s) { load_slice(d, rg, rg8, s, t); };
    Bf16Slice first;
    if (warp < nslice) load(first, warp);
    pdl_wait();
    pdl_launch_dependents();
    for (int n0 = 0; n0 < M; n0 += kNT * 8) {
      const int ntok = min(M - n0, kNT * 8);
      const int ntiles = (ntok + 7) / 8;
      const uint16_t* brow[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = nt * 8 + g;
        brow[nt] = n < ntok ? a.ws.sact + (size_t)(n0 + n) * SI : nullptr;
      }
      tile_pass(red, nslice, brow, ntiles, first, n0 == 0, load);
      if (warp < ntiles) {
        const int nt = warp;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = nt * 8 + 2 * t + (i & 1);
          const int h = h0 + g + (i >> 1) * 8;
          if (n < ntok)
            a.ws.ys[(size_t)(n0 + n) * H + h] = (uint16_t)f32_to_bf16_bits(red_sum(red, nt, lane, i));
        }
      }
      __syncthreads();
    }
  } else {
    const int ri = item - ns_items;
    const int ui = ri / hblocks;
    hb = ri % hblocks;
    const int h0 = hb * 16;
    // routing metadata is final: the gate/up grid released this grid only
    // after its own dependency wait, which follows the router's completion
    const int U = ldg_cg_i32(a.ws.uniq);
    if (ui >= U) {
      pdl_wait();
      return;
    }
    const int e = ldg_cg_i32(a.ws.uniq + 1 + ui);
    const int cnt = ldg_cg_i32(a.ws.e_cnt + e);
    const int off = ldg_cg_i32(a.ws.e_off + e);
    const int nslice = I / kSliceK;
    const size_t rg_ = (size_t)e * H + h0 + g, rg8_ = rg_ + 8;
    const uint8_t* cg = a.w2 + rg_ * (I / 2);
    const uint8_t* cg8 = a.w2 + rg8_ * (I / 2);
    const uint8_t* sg = a.w2_sf + rg_ * (I / 16);
    const uint8_t* sg8 = a.w2_sf + rg8_ * (I / 16);
    auto load = [&](Fp4Slice& d, int s) { load_slice(d, cg, cg8, sg, sg8, s, t); };
    Fp4Slice first;
    if (warp < nslice) load(first, warp);
    pdl_wait();
    pdl_launch_dependents();
    const float gs2 = a.w2_gs[e];
    for (int n0 = 0; n0 < cnt; n0 += kNT * 8) {
      const int ntok = min(cnt - n0, kNT * 8);
      const int ntiles = (ntok + 7) / 8;
      const uint16_t* brow[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = nt * 8 + g;
        brow[nt] = n < ntok ? a.ws.act + (size_t)(off + n0 + n) * I : nullptr;
      }
      tile_pass(red, nslice, brow, ntiles, first, n0 == 0, load);
      if (warp < ntiles) {
        const int nt = warp;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = nt * 8 + 2 * t + (i & 1);
          const int h = h0 + g + (i >> 1) * 8;
          if (n < ntok) {
            const float v = red_sum(red, nt, lane, i) * 128.0f * gs2;
            a.ws.y[(size_t)(off + n0 + n) * H + h] = (uint16_t)f32_to_bf16_bits(v);
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- last finisher of this output row block combines
  if (threadIdx.x == 0) {
    __threadfence();
    const int expect = ldg_cg_i32(a.ws.uniq) + (SI > 0 ? 1 : 0);
    const int old = atomicAdd(&a.ws.hblk_cnt[hb], 1);
    s_last = (old == expect - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) a.ws.hblk_cnt[hb] = 0;
  const int h0 = hb * 16;
  for (int idx = threadIdx.x; idx < M * 16; idx += blockDim.x) {
    const int tt = idx / 16, h = h0 + (idx & 15);
    float R = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int p = tt * k + j;
      const float w = ldg_cg_f32(a.ws.tw + p);
      const int row = ldg_cg_i32(a.ws.rowof + p);
      const float y = bf16_bits_to_f32(ldg_cg_u16(a.ws.y + (size_t)row * H + h));
      R = R + w * y;  // rank order j = 0 .. k-1
    }
    const float ys = SI > 0 ? bf16_bits_to_f32(ldg_cg_u16(a.ws.ys + (size_t)tt * H + h)) : 0.0f;
    a.out[(size_t)tt * H + h] = (uint16_t)f32_to_bf16_bits(round_bf16(R) + ys);
  }
}

// ----------------------------------------------------------------------------
static cudaError_t launch(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t st,
                          bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

static int max_routed_experts(const MoEArgs& a) { return a.M * a.k < a.E ? a.M * a.k : a.E; }

cudaError_t launch_decode_gate_up(const MoEArgs& a, cudaStream_t st, bool pdl) {
  int ns = a.SI / 8;
  const int items = ns + max_routed_experts(a) * (a.I / 8);
  MoEArgs aa = a;
  void* args[] = {&aa, &ns};
  return launch((const void*)gate_up_decode_kernel, dim3(items), dim3(kDecThreads), args, st, pdl);
}

cudaError_t launch_decode_down(const MoEArgs& a, cudaStream_t st, bool pdl) {
  int ns = a.SI > 0 ? a.H / 16 : 0;
  const int items = ns + max_routed_experts(a) * (a.H / 16);
  MoEArgs aa = a;
  void* args[] = {&aa, &ns};
  return launch((const void*)down_decode_kernel, dim3(items), dim3(kDecThreads), args, st, pdl);
}

FLINT_SPAN_SETTER(decode)

}  // namespace flint
