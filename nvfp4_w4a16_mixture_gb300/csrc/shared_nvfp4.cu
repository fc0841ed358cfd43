// The MoE block with an NVFP4 shared expert.
//
// Page "vllm.models.flint.ops.moe": LLMoEWeights holds the shared expert as
// ModelOpt-packed NVFP4 gate/up and down weights with block scales and an
// fp32 global scale each, passed to the same kernels as the routed experts;
// so it follows their rule: g, u = fp32(sum) * gs_gu, sact = bf16(silu(g) *
// u), ys = bf16(fp32(sum) * gs_d), and out = bf16(bf16(routed) + ys).
//
// The routed part runs as the block without a shared expert, whose output is
// bf16(routed) exactly (bf16(bf16(R) + 0)); these kernels then form ys and
// replace each output o by bf16(o + ys), which is the block's rounding.
// Gate/up: CTA (8 intermediate rows, 64 tokens), its 8 warps split over the
// chunk's 8-token tiles and, when there are fewer tiles than warps, over K
// (kw warps per tile, their exact pairs added in warp order); every sum exact
// (exact.cuh slice_nvfp4_exact), act with the correctly rounded exp where it
// decides the rounding; down: CTA (16 output rows, 64 tokens) likewise.
// Weights are read straight from global memory.  Chained with programmatic
// dependent launch.
#include "common.cuh"
#include "exact.cuh"
#include "frag.cuh"
#include "internal.h"

namespace flint {
namespace {

constexpr int kShWarps = 8;

FLINT_DEV void load_col(uint4 (&xb)[4], const uint16_t* p) {
#pragma unroll
  for (int q = 0; q < 4; ++q) xb[q] = p ? ldg_cg_v4(p + 8 * q) : make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(kShWarps * 32) shared_nvfp4_gate_up_kernel(
    const uint16_t* __restrict__ x, const uint8_t* __restrict__ gu, const uint8_t* __restrict__ gu_sf,
    const float* __restrict__ gu_gs, int M, int H, int SI, uint16_t* __restrict__ sact) {
  SpanGuard<kSpanSharedGateUp> span_guard;
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float4 red[kShWarps * 64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int ntiles = (min(64, M - 64 * (int)blockIdx.y) + 7) / 8;
  const int kw = max(1, kShWarps / ntiles), tile = warp / kw, part = warp % kw;
  const bool active = tile < ntiles;
  const int t0 = 64 * blockIdx.y + 8 * tile;
  const int r0 = 8 * blockIdx.x;
  const int tok = t0 + g;
  const uint16_t* xrow = active && tok < M ? x + (size_t)tok * H : nullptr;
  const uint8_t* ca = gu + (size_t)(r0 + g) * (H / 2);
  const uint8_t* cb = gu + (size_t)(SI + r0 + g) * (H / 2);
  const uint8_t* sa = gu_sf + (size_t)(r0 + g) * (H / 16);
  const uint8_t* sb = gu_sf + (size_t)(SI + r0 + g) * (H / 16);
  float S[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = part; active && s < H / kSliceK; s += kw) {
    uint4 xb[4];
    load_col(xb, xrow ? xrow + s * kSliceK + 32 * t : nullptr);
    slice_nvfp4_exact(S, C, ca + s * (kSliceK / 2) + 16 * t, cb + s * (kSliceK / 2) + 16 * t,
                      *reinterpret_cast<const uint16_t*>(sa + s * (kSliceK / 16) + 2 * t),
                      *reinterpret_cast<const uint16_t*>(sb + s * (kSliceK / 16) + 2 * t), xb);
  }
  if (kw > 1) {
    store_pair(red, warp, lane, S, C);
    __syncthreads();
    if (!active || part != 0) return;
    add_pairs(S, C, red, warp, kw, lane);
  } else if (!active) {
    return;
  }
  const float gs = *gu_gs;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int tt = t0 + 2 * t + cc;
    if (tt < M) {
      // the slices summed the weights times 2^-7: scale back exactly, then
      // the global scale on the fp32 accumulator
      const float gv = __fmul_rn(__fadd_rn(S[cc], C[cc]) * 128.0f, gs);
      const float uv = __fmul_rn(__fadd_rn(S[2 + cc], C[2 + cc]) * 128.0f, gs);
      sact[(size_t)tt * SI + r0 + g] = (uint16_t)act_bits(gv, uv);
    }
  }
}

__global__ void __launch_bounds__(kShWarps * 32) shared_nvfp4_down_kernel(
    const uint16_t* __restrict__ sact, const uint8_t* __restrict__ dn, const uint8_t* __restrict__ dn_sf,
    const float* __restrict__ dn_gs, int M, int H, int SI, uint16_t* __restrict__ ys) {
  SpanGuard<kSpanSharedDown> span_guard;
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float4 red[kShWarps * 64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int ntiles = (min(64, M - 64 * (int)blockIdx.y) + 7) / 8;
  const int kw = max(1, kShWarps / ntiles), tile = warp / kw, part = warp % kw;
  const bool active = tile < ntiles;
  const int t0 = 64 * blockIdx.y + 8 * tile;
  const int h0 = 16 * blockIdx.x;
  const int tok = t0 + g;
  const uint16_t* arow = active && tok < M ? sact + (size_t)tok * SI : nullptr;
  const uint8_t* ca = dn + (size_t)(h0 + g) * (SI / 2);
  const uint8_t* cb = dn + (size_t)(h0 + 8 + g) * (SI / 2);
  const uint8_t* sa = dn_sf + (size_t)(h0 + g) * (SI / 16);
  const uint8_t* sb = dn_sf + (size_t)(h0 + 8 + g) * (SI / 16);
  float S[4] = {0.0f, 0.0f, 0.0f, 0.0f}, C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = part; active && s < SI / kSliceK; s += kw) {
    uint4 xb[4];
    load_col(xb, arow ? arow + s * kSliceK + 32 * t : nullptr);
    slice_nvfp4_exact(S, C, ca + s * (kSliceK / 2) + 16 * t, cb + s * (kSliceK / 2) + 16 * t,
                      *reinterpret_cast<const uint16_t*>(sa + s * (kSliceK / 16) + 2 * t),
                      *reinterpret_cast<const uint16_t*>(sb + s * (kSliceK / 16) + 2 * t), xb);
  }
  if (kw > 1) {
    store_pair(red, warp, lane, S, C);
    __syncthreads();
    if (!active || part != 0) return;
    add_pairs(S, C, red, warp, kw, lane);
  } else if (!active) {
    return;
  }
  const float gs = *dn_gs;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int tt = t0 + 2 * t + cc;
    if (tt < M) {
      ys[(size_t)tt * H + h0 + g] = (uint16_t)f32_to_bf16_bits(__fmul_rn(__fadd_rn(S[cc], C[cc]) * 128.0f, gs));
      ys[(size_t)tt * H + h0 + 8 + g] =
          (uint16_t)f32_to_bf16_bits(__fmul_rn(__fadd_rn(S[2 + cc], C[2 + cc]) * 128.0f, gs));
    }
  }
}

// out = bf16(out + ys), two elements per thread (out holds bf16(routed)).
__global__ void __launch_bounds__(256) shared_add_kernel(uint16_t* __restrict__ out,
                                                         const uint16_t* __restrict__ ys, size_t n2) {
  SpanGuard<kSpanSharedAdd> span_guard;
  pdl_wait();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n2) return;
  const uint32_t o = reinterpret_cast<const uint32_t*>(out)[i], y = reinterpret_cast<const uint32_t*>(ys)[i];
  const uint32_t lo = f32_to_bf16_bits(__fadd_rn(bf16_bits_to_f32(o & 0xFFFFu), bf16_bits_to_f32(y & 0xFFFFu)));
  const uint32_t hi = f32_to_bf16_bits(__fadd_rn(bf16_bits_to_f32(o >> 16), bf16_bits_to_f32(y >> 16)));
  reinterpret_cast<uint32_t*>(out)[i] = lo | (hi << 16);
}

cudaError_t launch_pdl_sh(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t st) {
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

cudaError_t launch_shared_nvfp4(const uint16_t* x, const uint8_t* gu, const uint8_t* gu_sf, const float* gu_gs,
                                const uint8_t* dn, const uint8_t* dn_sf, const float* dn_gs, int M, int H,
                                int SI, uint16_t* sact, uint16_t* ys, uint16_t* out, cudaStream_t st) {
  const unsigned chunks = (unsigned)((M + 63) / 64);
  void* a1[] = {&x, &gu, &gu_sf, &gu_gs, &M, &H, &SI, &sact};
  cudaError_t err = launch_pdl_sh((const void*)shared_nvfp4_gate_up_kernel, dim3(SI / 8, chunks),
                                  dim3(kShWarps * 32), a1, st);
  if (err != cudaSuccess) return err;
  void* a2[] = {&sact, &dn, &dn_sf, &dn_gs, &M, &H, &SI, &ys};
  err = launch_pdl_sh((const void*)shared_nvfp4_down_kernel, dim3(H / 16, chunks), dim3(kShWarps * 32), a2, st);
  if (err != cudaSuccess) return err;
  size_t n2 = (size_t)M * H / 2;
  void* a3[] = {&out, &ys, &n2};
  return launch_pdl_sh((const void*)shared_add_kernel, dim3((unsigned)((n2 + 255) / 256)), dim3(256), a3, st);
}

FLINT_SPAN_SETTER(shared_nvfp4)

}  // namespace flint
