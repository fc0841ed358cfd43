// Decode MoE block on BF16 routed experts (at most 64 tokens).
//
// Page "vllm.models.flint.ops.moe": flint_moe_bf16_decode (with
// _gate_up_gemv_bf16_kernel and _down_gemv_bf16_kernel): the same routing as
// the NVFP4 block, then act = bf16(silu(g) * u) from the fp32 gate/up sums,
// y_e = bf16(acc) (no global scale), routed = bf16(sum_j tw_j y_j) in fp32
// in rank order, out = bf16(routed + shared) with the shared expert's output
// given.  The pages store the experts in a blocked order; this entry point
// takes them row-major: w13 [E, 2I, H] (gate rows, then up rows), w2 [E, H, I].
//
// After the router (which also groups the pairs by expert), a gate/up grid
// of (8 intermediate rows, routed expert) CTAs and a down grid of (16 output
// rows, routed expert) CTAs; the 8 warps of a CTA split over the expert's
// 8-token tiles and, when there are fewer tiles than warps, over K (kw warps
// per tile, their pairs added in warp order), and sum exactly (exact.cuh:
// weights and activations split per 128-K slice so that the high products
// chain exactly in the tensor cores, the rest in a compensation term, slices
// added with TwoSum),
// so both act and y are the roundings of the exact sums.  A combine
// kernel forms the outputs.  All launches are chained with programmatic
// dependent launch.  The weights are read straight from global memory (each
// row by the CTA's warps in turn, through L1 and L2): this path is exact and
// simple, not tuned for bandwidth.
#include "common.cuh"
#include "exact.cuh"
#include "frag.cuh"
#include "internal.h"

namespace flint {
namespace {

constexpr int kBfWarps = 8;  // token tiles of 8: an expert holds at most 64 tokens

// The 32 bf16 activations K 32 t .. 32 t + 31 of row p (nullptr: zeros).
FLINT_DEV void load_xcol(uint4 (&xb)[4], const uint16_t* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q) xb[q] = p ? ldg_cg_v4(p + 8 * q) : make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(kBfWarps * 32) bf16_gate_up_kernel(MoEArgs a, const uint16_t* w13) {
  SpanGuard<kSpanGateUp> span_guard;
  pdl_wait();  // the router's records are final
  pdl_launch_dependents();
  const int u = blockIdx.y;
  if (u >= ldg_cg_i32(a.ws.uniq)) return;
  const int* rec = a.ws.urec + (size_t)u * kUrecInts;
  const int e = ldg_cg_i32(rec), cnt = ldg_cg_i32(rec + 1), off = ldg_cg_i32(rec + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  __shared__ float4 red[kBfWarps * 64];
  const int ntiles = (cnt + 7) / 8;
  const int kw = max(1, kBfWarps / ntiles), tile = warp / kw, part = warp % kw;
  const bool active = tile < ntiles;
  const int H = a.H, I = a.I, k = a.k, r0 = 8 * blockIdx.x;
  const int nn = 8 * tile + g;  // this lane's token column
  const uint16_t* xrow = active && nn < cnt ? a.x + (size_t)(ldg_cg_i32(rec + 4 + nn) / k) * H : nullptr;
  const uint16_t* ra = w13 + ((size_t)e * 2 * I + r0 + g) * H;      // gate row r0 + g
  const uint16_t* rb = w13 + ((size_t)e * 2 * I + I + r0 + g) * H;  // up row r0 + g
  float S[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = part; active && s < H / kSliceK; s += kw) {
    uint4 xb[4];
    load_xcol(xb, xrow ? xrow + s * kSliceK + 32 * t : nullptr);
    slice_bf16_exact(S, C, ra + s * kSliceK + 32 * t, rb + s * kSliceK + 32 * t, xb);
  }
  if (kw > 1) {
    store_pair(red, warp, lane, S, C);
    __syncthreads();
    if (!active || part != 0) return;
    add_pairs(S, C, red, warp, kw, lane);
  } else if (!active) {
    return;
  }
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int tok = 8 * tile + 2 * t + cc;
    if (tok < cnt)
      a.ws.act[(size_t)(off + tok) * I + r0 + g] =
          (uint16_t)act_bits(__fadd_rn(S[cc], C[cc]), __fadd_rn(S[2 + cc], C[2 + cc]));
  }
}

__global__ void __launch_bounds__(kBfWarps * 32) bf16_down_kernel(MoEArgs a, const uint16_t* w2) {
  SpanGuard<kSpanDown> span_guard;
  pdl_wait();  // act is complete
  pdl_launch_dependents();
  // the cluster router's report on its f16 copy of x (unused here) goes
  // back to zero, as every launch leaves the workspace counters
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) a.ws.glob_cnt[1] = 0;
  const int u = blockIdx.y;
  if (u >= ldg_cg_i32(a.ws.uniq)) return;
  const int* rec = a.ws.urec + (size_t)u * kUrecInts;
  const int e = ldg_cg_i32(rec), cnt = ldg_cg_i32(rec + 1), off = ldg_cg_i32(rec + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  __shared__ float4 red[kBfWarps * 64];
  const int ntiles = (cnt + 7) / 8;
  const int kw = max(1, kBfWarps / ntiles), tile = warp / kw, part = warp % kw;
  const bool active = tile < ntiles;
  const int H = a.H, I = a.I, h0 = 16 * blockIdx.x;
  const int nn = 8 * tile + g;
  const uint16_t* arow = active && nn < cnt ? a.ws.act + (size_t)(off + nn) * I : nullptr;
  const uint16_t* ra = w2 + ((size_t)e * H + h0 + g) * I;
  const uint16_t* rb = w2 + ((size_t)e * H + h0 + 8 + g) * I;
  float S[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = part; active && s < I / kSliceK; s += kw) {
    uint4 xb[4];
    load_xcol(xb, arow ? arow + s * kSliceK + 32 * t : nullptr);
    slice_bf16_exact(S, C, ra + s * kSliceK + 32 * t, rb + s * kSliceK + 32 * t, xb);
  }
  if (kw > 1) {
    store_pair(red, warp, lane, S, C);
    __syncthreads();
    if (!active || part != 0) return;
    add_pairs(S, C, red, warp, kw, lane);
  } else if (!active) {
    return;
  }
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int tok = 8 * tile + 2 * t + cc;
    if (tok < cnt) {
      uint16_t* yrow = a.ws.y + (size_t)(off + tok) * H + h0;
      yrow[g] = (uint16_t)f32_to_bf16_bits(__fadd_rn(S[cc], C[cc]));
      yrow[8 + g] = (uint16_t)f32_to_bf16_bits(__fadd_rn(S[2 + cc], C[2 + cc]));
    }
  }
}

// out[t, h] = bf16(bf16(sum_j tw_j y[row(t, j), h]) + shared[t, h]), two
// columns per thread, the routed sum in fp32 in rank order.
__global__ void __launch_bounds__(256) bf16_combine_kernel(MoEArgs a, const uint16_t* shared_out) {
  SpanGuard<kSpanCombine> span_guard;
  pdl_wait();  // y is complete
  const int H = a.H, k = a.k;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)a.M * (H / 2)) return;
  const int tt = (int)(i / (H / 2)), h = 2 * (int)(i % (H / 2));
  float r0 = 0.0f, r1 = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int p = tt * k + j;
    const float w = ldg_cg_f32(a.ws.tw + p);
    const uint32_t y2 = *reinterpret_cast<const uint32_t*>(a.ws.y + (size_t)ldg_cg_i32(a.ws.rowof + p) * H + h);
    r0 = __fadd_rn(r0, __fmul_rn(w, bf16_bits_to_f32(y2 & 0xFFFFu)));
    r1 = __fadd_rn(r1, __fmul_rn(w, bf16_bits_to_f32(y2 >> 16)));
  }
  float s0 = 0.0f, s1 = 0.0f;
  if (shared_out) {
    const uint32_t s2 = *reinterpret_cast<const uint32_t*>(shared_out + (size_t)tt * H + h);
    s0 = bf16_bits_to_f32(s2 & 0xFFFFu);
    s1 = bf16_bits_to_f32(s2 >> 16);
  }
  const uint32_t o0 = f32_to_bf16_bits(__fadd_rn(round_bf16(r0), s0));
  const uint32_t o1 = f32_to_bf16_bits(__fadd_rn(round_bf16(r1), s1));
  *reinterpret_cast<uint32_t*>(a.out + (size_t)tt * H + h) = o0 | (o1 << 16);
}

cudaError_t launch_pdl_bf(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_bf16_experts(const MoEArgs& a, const uint16_t* w13, const uint16_t* w2,
                                const uint16_t* shared_out, cudaStream_t st) {
  cudaError_t err = route_cluster_supported(a) ? launch_route_cluster(a, st) : launch_route(a, true, st, true);
  if (err != cudaSuccess) return err;
  MoEArgs aa = a;
  const unsigned units = (unsigned)(a.M * a.k < a.E ? a.M * a.k : a.E);
  void* gu[] = {&aa, (void*)&w13};
  err = launch_pdl_bf((const void*)bf16_gate_up_kernel, dim3(a.I / 8, units), dim3(kBfWarps * 32), gu, st);
  if (err != cudaSuccess) return err;
  void* dn[] = {&aa, (void*)&w2};
  err = launch_pdl_bf((const void*)bf16_down_kernel, dim3(a.H / 16, units), dim3(kBfWarps * 32), dn, st);
  if (err != cudaSuccess) return err;
  void* cb[] = {&aa, (void*)&shared_out};
  const size_t n = (size_t)a.M * (a.H / 2);
  return launch_pdl_bf((const void*)bf16_combine_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), cb, st);
}

FLINT_SPAN_SETTER(bf16_experts)

}  // namespace flint
